// chunk_simt.cu -- chunked forward on CUDA cores (fp32 arithmetic), for fp32 inputs and for any
// supported shape that the tensor-core path does not cover.
//
// Chunked WY / UT form of the recurrence (burn-gdn2 0.1.5 docs: "chunked WY decomposition
// (training)"). For a chunk of C tokens entering with state S_n, with G_i the inclusive
// cumulative log-decay of the chunk (per key channel):
//     A_ij = sum_c b_i k_i k_j e^{G_i - G_j}   (j < i)        M_ij = sum_c q_i k_j e^{G_i - G_j}  (j <= i)
//     T    = (I + A)^{-1}   (unit lower triangular, forward substitution)
//     W    = T (b . k . e^{G}),   U~ = T (w . v)
//     U    = U~ - W S_n
//     O    = (q . e^{G}) S_n + M U
//     S_{n+1} = diag(e^{G_last}) S_n + (k . e^{G_last - G})^T U
//
// Two kernels:
//   factors (grid: chunks x heads, fully parallel) computes everything that does not depend on the
//           state and stores it in the workspace: W^T, (q . e^{G})^T, (k . e^{G_last - G})^T [d_k x C],
//           M [C x C], U~^T [d_v x C], e^{G_last} [d_k];
//   state   (grid: heads x 16-column slices of d_v, sequential over chunks) carries S_n and writes o.
// For the chunked backward the factor kernel writes the same quantities token-major ([C x d]) and adds
// channel-major copies of W and k . e^{G_last - G}; there the chains of backward_chunk.cu replace the
// state kernel.
// Padding: tokens past T read as zeros (k = q = b = v = w = 0, g = 0), which leaves S unchanged.
//
// Decay factors over the whole domain alpha in [0, 1] (g = log alpha in [-inf, 0]): g is first
// clamped at -100 (alpha = e^{-100} ~ 4e-44, which no fp32 result can tell from 0), so a full reset
// (g = -inf) stays finite. The exponent of every factor is then formed from 16-token blocks of the
// chunk: L_t = the inclusive prefix of g within t's block, S_B = the sum over block B. For tokens
// i >= j in blocks I >= J,
//     G_i - G_j = L_i - L_j + W_IJ,    W_IJ = S_J + sum_{J < B < I} S_B   (0 when I = J),
// so no exponent is the difference of two long prefixes: values stay small unless the factor itself
// is negligible, and no factor can overflow (every exponent is <= 0).
#include "common.cuh"

namespace gdn2 {

namespace {

__device__ int g_status_simt;

// 9 warps: the 528 pairs of A and M for C = 32 take at most two rounds of the block
constexpr int kFactorThreads = 288;

// kDK, kDV, kC: the sizes as compile-time constants, or 0 to take them from the arguments
template <typename Tin, int kDK, int kDV, int kC>
__global__ void __launch_bounds__(kFactorThreads) factors_simt_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                           const Tin* __restrict__ v, const Tin* __restrict__ g,
                                                           const Tin* __restrict__ b, const Tin* __restrict__ w,
                                                           float* __restrict__ ws, float* __restrict__ t_out, int T,
                                                           int Hk, int Hv, int dk_arg, int dv_arg, int C_arg,
                                                           int imajor) {
    const int dk = kDK ? kDK : dk_arg, dv = kDV ? kDV : dv_arg, C = kC ? kC : C_arg;
    extern __shared__ float smem[];
    const int n = blockIdx.x;                // chunk
    const int bh = blockIdx.y;               // bi * Hv + hv
    const int NC = gridDim.x;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    const int t0 = n * C;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int LD = dk + 1;
    const int LDQ = (dk > dv ? dk : dv) + 1;
    const int nb = C / 16;                   // 16-token blocks of the chunk
    float* sG = smem;                        // [C][LD]   g, then L: inclusive prefix within the 16-token block
    float* sK = sG + C * LD;                 // [C][LD]   k
    float* sBK = sK + C * LD;                // [C][LD]   b . k, later b . k . e^{G}
    float* sQ = sBK + C * LD;                // [C][LDQ]  q, later w . v
    float* sA = sQ + C * LDQ;                // [C][C+1]
    float* sT = sA + C * (C + 1);            // [C][C+1]
    float* sX = sQ;                          // [16][C] block products of the inverse (q is read out by then)
    float* sS = sT + C * (C + 1);            // [nb][dk]  block sums S_B
    float* sPre = sS + nb * dk;              // [nb][dk]  sum of the blocks before B (G at the start of B)
    float* sSuf = sPre + nb * dk;            // [nb][dk]  sum of the blocks after B
    float* sW = sSuf + nb * dk;              // [1 + nb(nb-1)/2][dk]  W_IJ (row 0: zeros, for I = J)

    const SimtWs L{dk, dv, C, imajor != 0};
    float* u = ws + ((size_t)bh * NC + n) * L.unit_floats();

    {   // w and v are read after the inverse: into L2 now, one 128-byte line per thread
        const int lines = (dv * (int)sizeof(Tin) + 127) / 128, per = 128 / (int)sizeof(Tin);
        for (int i = tid; i < 2 * C * lines; i += nt) {
            const int ten = i / (C * lines), t = (i / lines) % C, line = i % lines;
            if (t0 + t < T) {
                const Tin* base = ten ? v : w;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (((size_t)bi * T + t0 + t) * Hv + hv) * dv + line * per));
            }
        }
    }
    // eight consecutive channels per load (d_k, d_v are multiples of 16, so rows stay 16-byte aligned)
#pragma unroll 2
    for (int idx = tid; idx < C * dk / 8; idx += nt) {
        const int t = idx / (dk / 8), c = 8 * (idx - t * (dk / 8));
        const int tok = t0 + t;
        float gg[8], kk[8], bb[8], qq[8];
        if (tok < T) {
            const size_t kq_i = (((size_t)bi * T + tok) * Hk + hk) * dk + c;
            const size_t gb_i = (((size_t)bi * T + tok) * Hv + hv) * dk + c;
            Vec8<Tin>::load(g + gb_i, gg);
            Vec8<Tin>::load(b + gb_i, bb);
            Vec8<Tin>::load(k + kq_i, kk);
            Vec8<Tin>::load(q + kq_i, qq);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) gg[i] = kk[i] = bb[i] = qq[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sG[t * LD + c + i] = gg[i];
            sK[t * LD + c + i] = kk[i];
            sBK[t * LD + c + i] = bb[i] * kk[i];
            sQ[t * LDQ + c + i] = qq[i];
        }
    }
    __syncthreads();
    // per key channel: L (prefix within each 16-token block) of the clamped gates, the block sums,
    // the sums before / after each block and between block pairs, and the chunk decay e^{G_last}
    for (int c = tid; c < dk; c += nt) {
        for (int B = 0; B < nb; ++B) {
            float acc = 0.f;
            for (int t = 16 * B; t < 16 * B + 16; ++t) {
                acc += fmaxf(sG[t * LD + c], kGateFloor);
                sG[t * LD + c] = acc;
            }
            sS[B * dk + c] = acc;
        }
        float pre = 0.f;
        for (int B = 0; B < nb; ++B) {
            sPre[B * dk + c] = pre;
            pre += sS[B * dk + c];
        }
        float suf = 0.f;
        for (int B = nb - 1; B >= 0; --B) {
            sSuf[B * dk + c] = suf;
            suf += sS[B * dk + c];
        }
        sW[c] = 0.f;
        for (int I = 1; I < nb; ++I) {
            float z = 0.f;  // sum of the blocks strictly between J and I
            for (int J = I - 1; J >= 0; --J) {
                sW[(1 + I * (I - 1) / 2 + J) * dk + c] = sS[J * dk + c] + z;
                z += sS[J * dk + c];
            }
        }
        u[L.off_gam() + c] = __expf(pre);
    }
    __syncthreads();
    // erase interaction A (strictly lower) and causal q-k M (lower incl. diagonal): one thread per pair
    // (i, j <= i), the pairs numbered along the lower triangle so that no lane idles above the diagonal
    float* Mws = u + L.off_m();
    for (int p = tid; p < C * C; p += nt) {
        const int i = p / C, j = p - i * C;
        sT[i * (C + 1) + j] = 0.f;
        if (j > i) {
            sA[i * (C + 1) + j] = 0.f;
            Mws[p] = 0.f;
        }
    }
    for (int p = tid; p < C * (C + 1) / 2; p += nt) {
        int i = static_cast<int>((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= p) ++i;
        while (i * (i + 1) / 2 > p) --i;
        const int j = p - i * (i + 1) / 2;
        const int I = i >> 4, J = j >> 4;
        const float* wr = sW + (I == J ? 0 : 1 + I * (I - 1) / 2 + J) * dk;
        float a = 0.f, m = 0.f;
        for (int c = 0; c < dk; ++c) {
            const float e = __expf(sG[i * LD + c] - sG[j * LD + c] + wr[c]);  // G_i - G_j <= 0
            const float kj = sK[j * LD + c] * e;
            a = fmaf(sBK[i * LD + c], kj, a);
            m = fmaf(sQ[i * LDQ + c], kj, m);
        }
        sA[i * (C + 1) + j] = (j < i) ? a : 0.f;
        Mws[i * C + j] = m;
    }
    __syncthreads();
    // T = (I + A)^{-1} (unit lower triangular) by 16 x 16 blocks: each diagonal block by forward
    // substitution (thread = column), then the block rows r in order,
    //     T_rs = -T_rr X_rs,   X_rs = sum_{s <= l < r} A_rl T_ls   (blocks s < r)
    if (tid < C) {  // column j of its diagonal block, kept in registers
        const int j = tid, top = j & ~15, jl = j & 15;
        float tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) tc[r] = r == jl ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int l = 0; l < r; ++l) acc = fmaf(sA[(top + r) * (C + 1) + top + l], tc[l], acc);
            if (r > jl) tc[r] = -acc;  // rows above j stay 0, row j stays 1
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(top + r) * (C + 1) + j] = tc[r];
    }
    // decayed q and k ([d_k][C], or [C][d_k] when imajor) for the state kernel, by the threads that do not
    // solve; b . k . e^{G} in place
    for (int p = tid - C; p >= 0 && p < dk * C; p += nt - C) {
        int c, i;
        if (imajor) i = p / dk, c = p - i * dk;
        else c = p / C, i = p - c * C;
        const float Li = sG[i * LD + c];
        const int Bi = i >> 4;
        u[L.off_qbt() + p] = sQ[i * LDQ + c] * __expf(Li + sPre[Bi * dk + c]);                        // e^{G_i}
        u[L.off_kht() + p] = sK[i * LD + c] * __expf(sS[Bi * dk + c] - Li + sSuf[Bi * dk + c]);     // e^{G_last - G_i}
    }
    if (imajor)  // channel-major copy of k.e^{G_last-G}
        for (int p = tid - C; p >= 0 && p < dk * C; p += nt - C) {
            const int c = p / C, i = p - c * C, Bi = i >> 4;
            u[L.off_kht2() + p] = sK[i * LD + c] * __expf(sS[Bi * dk + c] - sG[i * LD + c] + sSuf[Bi * dk + c]);
        }
    __syncthreads();
    for (int r = 16; r < C; r += 16) {
        for (int p = tid; p < 16 * r; p += nt) {  // X: rows r .. r+15, columns 0 .. r-1
            const int ii = p / r, jj = p - ii * r;
            float acc = 0.f;
            for (int l = jj; l < r; ++l) acc = fmaf(sA[(r + ii) * (C + 1) + l], sT[l * (C + 1) + jj], acc);
            sX[p] = acc;
        }
        __syncthreads();
        for (int p = tid; p < 16 * r; p += nt) {
            const int ii = p / r, jj = p - ii * r;
            float acc = 0.f;
            for (int m2 = 0; m2 <= ii; ++m2) acc = fmaf(sT[(r + ii) * (C + 1) + r + m2], sX[m2 * r + jj], acc);
            sT[(r + ii) * (C + 1) + jj] = -acc;
        }
        __syncthreads();
    }
    for (int idx = tid; idx < C * dk; idx += nt) {
        const int t = idx / dk, c = idx - t * dk;
        sBK[t * LD + c] *= __expf(sG[t * LD + c] + sPre[(t >> 4) * dk + c]);
    }
#pragma unroll 2
    for (int idx = tid; idx < C * dv / 8; idx += nt) {
        const int t = idx / (dv / 8), c = 8 * (idx - t * (dv / 8));
        const int tok = t0 + t;
        float ww[8], vv[8];
        if (tok < T) {
            const size_t vw_i = (((size_t)bi * T + tok) * Hv + hv) * dv + c;
            Vec8<Tin>::load(w + vw_i, ww);
            Vec8<Tin>::load(v + vw_i, vv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) ww[i] = vv[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sQ[t * LDQ + c + i] = ww[i] * vv[i];
    }
    __syncthreads();
    // W = T X with X = b . k . e^{G}, and U~ = T (w . v), stored [C][d] when imajor, else transposed:
    // thread = channel c and the rows i, C-1-i together (four independent sums; the j loop runs to the
    // longer row, T being zero above its diagonal)
    {
        const int dm = dk > dv ? dk : dv;
        for (int p = tid; p < dm * (C / 2); p += nt) {
            const int ip = p / dm, c = p - ip * dm;
            const int i1 = ip, i2 = C - 1 - ip;
            const bool hw = c < dk, hu = c < dv;
            float w1 = 0.f, w2 = 0.f, u1 = 0.f, u2 = 0.f;
#pragma unroll 4
            for (int j = 0; j <= i2; ++j) {
                const float t1 = sT[i1 * (C + 1) + j], t2 = sT[i2 * (C + 1) + j];
                const float x = hw ? sBK[j * LD + c] : 0.f, y = hu ? sQ[j * LDQ + c] : 0.f;
                w1 = fmaf(t1, x, w1);
                w2 = fmaf(t2, x, w2);
                u1 = fmaf(t1, y, u1);
                u2 = fmaf(t2, y, u2);
            }
            if (hw) {
                u[L.off_wt() + (imajor ? (size_t)i1 * dk + c : (size_t)c * C + i1)] = w1;
                u[L.off_wt() + (imajor ? (size_t)i2 * dk + c : (size_t)c * C + i2)] = w2;
                if (imajor) {  // k is read out: W for its channel-major copy
                    sK[i1 * LD + c] = w1;
                    sK[i2 * LD + c] = w2;
                }
            }
            if (hu) {
                u[L.off_utt() + (imajor ? (size_t)i1 * dv + c : (size_t)c * C + i1)] = u1;
                u[L.off_utt() + (imajor ? (size_t)i2 * dv + c : (size_t)c * C + i2)] = u2;
            }
        }
    }
    if (imajor) {
        __syncthreads();
        for (int p = tid; p < dk * C; p += nt) {
            const int c = p / C, i = p - c * C;
            u[L.off_wt2() + p] = sK[i * LD + c];
        }
    }
    if (t_out)  // T = (I + A)^{-1} [C][C] for the gradients
        for (int p = tid; p < C * C; p += nt) {
            const int i = p / C, j = p - i * C;
            t_out[((size_t)bh * NC + n) * C * C + p] = sT[i * (C + 1) + j];
        }
}

constexpr int kSlice = 16;

template <typename Tin>
__global__ void __launch_bounds__(256) state_simt_kernel(const float* __restrict__ ws, const float* __restrict__ s0,
                                                         float* __restrict__ sT_out, Tin* __restrict__ o, int T,
                                                         int Hv, int dk, int dv, int C, int NC, float scale) {
    extern __shared__ float smem[];
    const int bh = blockIdx.x;
    const int bi = bh / Hv, hv = bh - bi * Hv;
    const int col0 = blockIdx.y * kSlice;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* sS = smem;                        // [dk][kSlice]
    float* sWT = sS + dk * kSlice;           // [dk][C]
    float* sQb = sWT + dk * C;               // [dk][C]
    float* sKh = sQb + dk * C;               // [dk][C]
    float* sM = sKh + dk * C;                // [C][C]
    float* sUt = sM + C * C;                 // [kSlice][C]
    float* sGam = sUt + kSlice * C;          // [dk]
    float* sU = sGam + dk;                   // [C][kSlice]
    float* sP = sU + C * kSlice;             // [C][kSlice]
    const SimtWs L{dk, dv, C};

    for (int p = tid; p < dk * kSlice; p += nt) {
        const int c = p / kSlice, j = p - c * kSlice;
        sS[p] = s0 ? s0[((size_t)bh * dk + c) * dv + col0 + j] : 0.f;
    }
    for (int n = 0; n < NC; ++n) {
        const float* u = ws + ((size_t)bh * NC + n) * L.unit_floats();
        __syncthreads();
        for (int p = tid; p < dk * C; p += nt) {
            sWT[p] = u[L.off_wt() + p];
            sQb[p] = u[L.off_qbt() + p];
            sKh[p] = u[L.off_kht() + p];
        }
        for (int p = tid; p < C * C; p += nt) sM[p] = u[L.off_m() + p];
        for (int p = tid; p < kSlice * C; p += nt) sUt[p] = u[L.off_utt() + (size_t)col0 * C + p];
        for (int p = tid; p < dk; p += nt) sGam[p] = u[L.off_gam() + p];
        __syncthreads();
        // U = U~ - W S_n ;  P = (q . e^{G}) S_n
        for (int p = tid; p < C * kSlice; p += nt) {
            const int i = p / kSlice, j = p - i * kSlice;
            float ws_ = 0.f, qs = 0.f;
            for (int c = 0; c < dk; ++c) {
                const float s = sS[c * kSlice + j];
                ws_ = fmaf(sWT[c * C + i], s, ws_);
                qs = fmaf(sQb[c * C + i], s, qs);
            }
            sU[p] = sUt[j * C + i] - ws_;
            sP[p] = qs;
        }
        __syncthreads();
        // O = P + M U ;  S_{n+1} = diag(e^{G_last}) S_n + K^^T U
        for (int p = tid; p < C * kSlice; p += nt) {
            const int i = p / kSlice, j = p - i * kSlice;
            const int tok = n * C + i;
            if (tok < T) {
                float acc = sP[p];
                for (int l = 0; l <= i; ++l) acc = fmaf(sM[i * C + l], sU[l * kSlice + j], acc);
                o[(((size_t)bi * T + tok) * Hv + hv) * dv + col0 + j] = from_f32<Tin>(scale * acc);
            }
        }
        for (int p = tid; p < dk * kSlice; p += nt) {
            const int c = p / kSlice, j = p - c * kSlice;
            float acc = sGam[c] * sS[p];
            for (int i = 0; i < C; ++i) acc = fmaf(sKh[c * C + i], sU[i * kSlice + j], acc);
            sS[p] = acc;
        }
    }
    __syncthreads();
    if (sT_out)
        for (int p = tid; p < dk * kSlice; p += nt) {
            const int c = p / kSlice, j = p - c * kSlice;
            sT_out[((size_t)bh * dk + c) * dv + col0 + j] = sS[p];
        }
}

size_t factors_smem(int dk, int dv, int C) {
    const int LD = dk + 1, LDQ = (dk > dv ? dk : dv) + 1, nb = C / 16;
    const size_t blk = (size_t)(3 * nb + 1 + nb * (nb - 1) / 2) * dk;  // S, before, after, W
    return sizeof(float) * ((size_t)3 * C * LD + (size_t)C * LDQ + 2 * (size_t)C * (C + 1) + blk);
}
size_t state_smem(int dk, int C) {
    return sizeof(float) * ((size_t)dk * kSlice + 3 * (size_t)dk * C + (size_t)C * C + (size_t)kSlice * C + dk +
                            2 * (size_t)C * kSlice);
}

template <typename Tin, int kDK, int kDV, int kC>
cudaError_t launch_factors_shape(const void* q, const void* k, const void* v, const void* g, const void* b,
                                 const void* w, const ChunkShape& sh, void* ws, float* t_out, int imajor,
                                 cudaStream_t s) {
    const size_t f_smem = factors_smem(sh.dk, sh.dv, sh.C);
    cudaError_t e = cudaFuncSetAttribute(factors_simt_kernel<Tin, kDK, kDV, kC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f_smem);
    if (e != cudaSuccess) return e;
    factors_simt_kernel<Tin, kDK, kDV, kC><<<dim3(sh.nchunks(), sh.B * sh.Hv), kFactorThreads, f_smem, s>>>(
        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
        static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), static_cast<float*>(ws),
        t_out, sh.T, sh.Hk, sh.Hv, sh.dk, sh.dv, sh.C, imajor);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_factors_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                             const ChunkShape& sh, void* ws, float* t_out, int imajor, cudaStream_t s) {
    if (sh.dk == 128 && sh.dv == 128 && sh.C == 32)
        return launch_factors_shape<Tin, 128, 128, 32>(q, k, v, g, b, w, sh, ws, t_out, imajor, s);
    if (sh.dk == 128 && sh.dv == 128 && sh.C == 64)
        return launch_factors_shape<Tin, 128, 128, 64>(q, k, v, g, b, w, sh, ws, t_out, imajor, s);
    return launch_factors_shape<Tin, 0, 0, 0>(q, k, v, g, b, w, sh, ws, t_out, imajor, s);
}

template <typename Tin>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     const float* s0, float* sT, void* o, const ChunkShape& sh, float scale, void* ws, cudaStream_t s) {
    const int NC = sh.nchunks();
    const size_t s_smem = state_smem(sh.dk, sh.C);
    cudaError_t e = launch_factors_t<Tin>(q, k, v, g, b, w, sh, ws, nullptr, 0, s);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(state_simt_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    state_simt_kernel<Tin><<<dim3(sh.B * sh.Hv, sh.dv / kSlice), 256, s_smem, s>>>(
        static_cast<const float*>(ws), s0, sT, static_cast<Tin*>(o), sh.T, sh.Hv, sh.dk, sh.dv, sh.C, NC, scale);
    return cudaGetLastError();
}

}  // namespace

size_t chunk_simt_workspace_bytes(const ChunkShape& sh, bool token_major) {
    const SimtWs L{sh.dk, sh.dv, sh.C, token_major};
    return sizeof(float) * L.unit_floats() * (size_t)sh.nchunks() * sh.B * sh.Hv;
}

cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, const void* g, const void* b,
                              const void* w, const float* s0, float* sT, void* o, const ChunkShape& sh, float scale,
                              gdn2_dtype dt, void* ws, cudaStream_t s) {
    if (dt == GDN2_BF16) return launch_t<__nv_bfloat16>(q, k, v, g, b, w, s0, sT, o, sh, scale, ws, s);
    return launch_t<float>(q, k, v, g, b, w, s0, sT, o, sh, scale, ws, s);
}

cudaError_t launch_factors_simt(const void* q, const void* k, const void* v, const void* g, const void* b,
                                const void* w, const ChunkShape& sh, gdn2_dtype dt, void* ws, float* t_out,
                                bool token_major, cudaStream_t s) {
    const int im = token_major ? 1 : 0;
    if (dt == GDN2_BF16) return launch_factors_t<__nv_bfloat16>(q, k, v, g, b, w, sh, ws, t_out, im, s);
    return launch_factors_t<float>(q, k, v, g, b, w, sh, ws, t_out, im, s);
}

int chunk_simt_read_clear_status(cudaStream_t) {
    (void)g_status_simt;
    return 0;  // no bounded waits in the SIMT kernels
}

}  // namespace gdn2

// backward_chunk.cu -- gradients of the GDN-2 core in chunked form, fp32 on CUDA cores (the recurrence
// of the burn-gdn2 0.1.5 docs, "Architecture", in the chunked WY form of its "chunked WY decomposition
// (training)" section), chunks of C = 32 tokens.
//
// Per chunk n, with the factors of the fp32 forward (chunk_simt.cu), S = S_n entering the chunk and
// S' = S_{n+1} leaving it:
//     U = T (U0 - K_bar S),  U0 = w.v,  K_bar = b.k.e^G,  W = T K_bar,  T = (I + A)^{-1}
//     O = Q_bar S + M U,     S' = G S + K^^T U,  G = diag(e^{G_last}),  Q_bar = q.e^G,  K^ = k.e^{G_last - G}
//     A_ts = sum_c b_t k_t k_s e^{G_t - G_s} (s < t),   M_ts = sum_c q_t k_s e^{G_t - G_s} (s <= t).
// Reverse mode, with dO~ = scale dO and dS' given:
//     dU  = M^T dO~ + K^ dS'                dS = G dS' + Q_bar^T dO~ - W^T dU      (the chain over chunks)
//     dQ_bar = dO~ S^T   dW = -dU S^T   dK^ = U dS'^T   dgamma = rowsum(dS' . S)   dM = tril(dO~ U^T)
//     dT = dU U0^T + dW K_bar^T   dU0 = T^T dU   dK_bar = T^T dW   dA = -strict_tril(T^T dT T^T)
// and through the elementwise factors to dq, dk, db, dg, dv, dw; the terms of A and M are taken pair
// by pair with e^{G_t - G_s} <= 1, so no factor can overflow whatever the decays.
//
// Four launches: the fp32 forward keeping T, S_n and U per chunk; the chain over chunks in reverse
// (adjoint_kernel: heads x 16-column slices, like the forward's state kernel); the local gradients of
// every (chunk, head) in parallel (grad_kernel); the sums of dq, dk over each key head's group.
#include <type_traits>

#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kD = 128;       // d_k = d_v
constexpr int kCb = 32;       // chunk of the backward
constexpr int kSl = 16;       // d_v columns per adjoint CTA
constexpr int kLD = kD + 1;   // padded row of [C][d] and [d][d] shared arrays
constexpr int kLC = kCb + 1;  // padded row of [C][C] shared arrays

// dS and dU over the chunks in reverse: dU_n = M_n^T dO~_n + K^_n dS_{n+1};
// dS_n = G_n dS_{n+1} + Q_bar_n^T dO~_n - W_n^T dU_n. Keeps dS_{n+1} and dU_n of every chunk.
template <typename Tin>
__global__ void __launch_bounds__(256) adjoint_kernel(const float* __restrict__ ws, const Tin* __restrict__ dO,
                                                      const float* __restrict__ dsT, float* __restrict__ ds0,
                                                      float* __restrict__ ds_save, float* __restrict__ du_save, int T,
                                                      int Hv, int NC, float scale) {
    extern __shared__ float smem[];
    const int bh = blockIdx.x, bi = bh / Hv, hv = bh - bi * Hv;
    const int col0 = blockIdx.y * kSl;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* sR = smem;                 // [kD][kSl] dS
    float* sWT = sR + kD * kSl;       // [kD][C]
    float* sQb = sWT + kD * kCb;      // [kD][C]
    float* sKh = sQb + kD * kCb;      // [kD][C]
    float* sM = sKh + kD * kCb;       // [C][C]
    float* sGam = sM + kCb * kCb;     // [kD]
    float* sDO = sGam + kD;           // [C][kSl]
    float* sDU = sDO + kCb * kSl;     // [C][kSl]
    const SimtWs L{kD, kD, kCb};

    for (int p = tid; p < kD * kSl; p += nt) {
        const int c = p / kSl, j = p - c * kSl;
        sR[p] = dsT ? dsT[((size_t)bh * kD + c) * kD + col0 + j] : 0.f;
    }
    for (int n = NC - 1; n >= 0; --n) {
        const float* u = ws + ((size_t)bh * NC + n) * L.unit_floats();
        __syncthreads();
        for (int p = tid; p < kD * kCb; p += nt) {
            sWT[p] = u[L.off_wt() + p];
            sQb[p] = u[L.off_qbt() + p];
            sKh[p] = u[L.off_kht() + p];
        }
        for (int p = tid; p < kCb * kCb; p += nt) sM[p] = u[L.off_m() + p];
        for (int p = tid; p < kD; p += nt) sGam[p] = u[L.off_gam() + p];
        for (int p = tid; p < kCb * kSl; p += nt) {
            const int i = p / kSl, j = p - i * kSl;
            const int tok = n * kCb + i;
            sDO[p] = tok < T ? scale * to_f32(dO[(((size_t)bi * T + tok) * Hv + hv) * kD + col0 + j]) : 0.f;
        }
        float* dsn = ds_save + ((size_t)bh * NC + n) * kD * kD;
        for (int p = tid; p < kD * kSl; p += nt) {
            const int c = p / kSl, j = p - c * kSl;
            dsn[(size_t)c * kD + col0 + j] = sR[p];  // dS_{n+1}
        }
        __syncthreads();
        float* dun = du_save + ((size_t)bh * NC + n) * kCb * kD;
        for (int p = tid; p < kCb * kSl; p += nt) {
            const int i = p / kSl, j = p - i * kSl;
            float acc = 0.f;
            for (int l = i; l < kCb; ++l) acc = fmaf(sM[l * kCb + i], sDO[l * kSl + j], acc);
            for (int c = 0; c < kD; ++c) acc = fmaf(sKh[c * kCb + i], sR[c * kSl + j], acc);
            sDU[p] = acc;
            dun[(size_t)i * kD + col0 + j] = acc;
        }
        __syncthreads();
        for (int p = tid; p < kD * kSl; p += nt) {
            const int c = p / kSl, j = p - c * kSl;
            float acc = sGam[c] * sR[p];
            for (int i = 0; i < kCb; ++i) {
                acc = fmaf(sQb[c * kCb + i], sDO[i * kSl + j], acc);
                acc = fmaf(-sWT[c * kCb + i], sDU[i * kSl + j], acc);
            }
            sR[p] = acc;
        }
    }
    __syncthreads();
    if (ds0)
        for (int p = tid; p < kD * kSl; p += nt) {
            const int c = p / kSl, j = p - c * kSl;
            ds0[((size_t)bh * kD + c) * kD + col0 + j] = sR[p];
        }
}

// The local gradients of one (chunk, head). Thread = channel c and the tokens t0, t0 + 2, .., t0 + 30.
template <typename Tin>
__global__ void __launch_bounds__(256) grad_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                   const Tin* __restrict__ v, const Tin* __restrict__ g,
                                                   const Tin* __restrict__ b, const Tin* __restrict__ w,
                                                   const Tin* __restrict__ dO, const float* __restrict__ ws,
                                                   const float* __restrict__ t_ws, const float* __restrict__ s_save,
                                                   const float* __restrict__ u_save, const float* __restrict__ ds_save,
                                                   const float* __restrict__ du_save, float* __restrict__ dq_ws,
                                                   float* __restrict__ dk_ws, Tin* __restrict__ dv, Tin* __restrict__ dg,
                                                   Tin* __restrict__ db, Tin* __restrict__ dw, int T, int Hk, int Hv,
                                                   float scale) {
    extern __shared__ float smem[];
    const int n = blockIdx.x, bh = blockIdx.y, NC = gridDim.x;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    const int tid = threadIdx.x;
    const int c = tid & (kD - 1), t0 = tid >> 7;
    constexpr int kM = kCb / 2;  // tokens per thread
    float* sG = smem;                 // [C][kLD] cumulative log-decay, later dG
    float* sQ = sG + kCb * kLD;       // q
    float* sK = sQ + kCb * kLD;       // k
    float* sBeta = sK + kCb * kLD;    // b.k
    float* sDO = sBeta + kCb * kLD;   // scale . do
    float* sU = sDO + kCb * kLD;      // U
    float* sDU = sU + kCb * kLD;      // dU
    float* sX = sDU + kCb * kLD;      // w.v, later K_bar
    float* sBig = sX + kCb * kLD;     // [kD][kLD]: dS_{n+1}, then S_n, then dW [C][kLD]
    float* sT = sBig + kD * kLD;      // [C][kLC]
    float* sM = sT + kCb * kLC;
    float* sdM = sM + kCb * kLC;
    float* sdT = sdM + kCb * kLC;
    float* sdA = sdT + kCb * kLC;
    float* sP = sdA + kCb * kLC;      // T^T dT, later the two halves of the dG_last sums
    const SimtWs L{kD, kD, kCb};
    const size_t unit = (size_t)bh * NC + n;

    // ---- inputs of the chunk
#pragma unroll 4
    for (int m = 0; m < kM; ++m) {
        const int t = t0 + 2 * m, tok = n * kCb + t;
        float qq = 0.f, kk = 0.f, bb = 0.f, gg = 0.f, oo = 0.f, uu0 = 0.f;
        if (tok < T) {
            const size_t kq = (((size_t)bi * T + tok) * Hk + hk) * kD + c;
            const size_t vh = (((size_t)bi * T + tok) * Hv + hv) * kD + c;
            qq = to_f32(q[kq]);
            kk = to_f32(k[kq]);
            bb = to_f32(b[vh]);
            gg = to_f32(g[vh]);
            oo = scale * to_f32(dO[vh]);
            uu0 = to_f32(w[vh]) * to_f32(v[vh]);
        }
        sQ[t * kLD + c] = qq;
        sK[t * kLD + c] = kk;
        sBeta[t * kLD + c] = bb * kk;
        sG[t * kLD + c] = gg;
        sDO[t * kLD + c] = oo;
        sX[t * kLD + c] = uu0;
        sU[t * kLD + c] = u_save[(unit * kCb + t) * kD + c];
        sDU[t * kLD + c] = du_save[(unit * kCb + t) * kD + c];
    }
    for (int p = tid; p < kCb * kCb; p += 256) {
        const int i = p / kCb, j = p - i * kCb;
        sT[i * kLC + j] = t_ws[unit * kCb * kCb + p];
        sM[i * kLC + j] = ws[unit * L.unit_floats() + L.off_m() + p];
    }
    const float* S = s_save + unit * kD * kD;
    const float* dS = ds_save + unit * kD * kD;
    float dgam = 0.f;  // rowsum(dS' . S) for channel c (threads below 128)
    if (tid < kD)
        for (int j = 0; j < kD; ++j) dgam = fmaf(dS[(size_t)c * kD + j], S[(size_t)c * kD + j], dgam);
    for (int p = tid; p < kD * kD; p += 256) sBig[(p >> 7) * kLD + (p & (kD - 1))] = dS[p];
    __syncthreads();
    if (tid < kD) {  // inclusive cumulative log-decay per channel
        float acc = 0.f;
        for (int t = 0; t < kCb; ++t) {
            acc += sG[t * kLD + c];
            sG[t * kLD + c] = acc;
        }
    }
    __syncthreads();
    const float Glast = sG[(kCb - 1) * kLD + c];
    // ---- dK^ = U dS'^T
    float dKh[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) dKh[m] = 0.f;
    for (int j = 0; j < kD; ++j) {
        const float x = sBig[c * kLD + j];
#pragma unroll
        for (int m = 0; m < kM; ++m) dKh[m] = fmaf(sU[(t0 + 2 * m) * kLD + j], x, dKh[m]);
    }
    __syncthreads();
    for (int p = tid; p < kD * kD; p += 256) sBig[(p >> 7) * kLD + (p & (kD - 1))] = S[p];
    __syncthreads();
    // ---- dQ_bar = dO~ S^T, dW = -dU S^T
    float dQb[kM], dW[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m) dQb[m] = dW[m] = 0.f;
    for (int j = 0; j < kD; ++j) {
        const float x = sBig[c * kLD + j];
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            dQb[m] = fmaf(sDO[(t0 + 2 * m) * kLD + j], x, dQb[m]);
            dW[m] = fmaf(-sDU[(t0 + 2 * m) * kLD + j], x, dW[m]);
        }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kM; ++m) sBig[(t0 + 2 * m) * kLD + c] = dW[m];  // dW [C][kLD]
    __syncthreads();
    // ---- dM = tril(dO~ U^T), dT = dU U0^T (then + dW K_bar^T)
    for (int p = tid; p < kCb * kCb; p += 256) {
        const int t = p / kCb, s = p - t * kCb;
        float am = 0.f, at = 0.f;
        for (int j = 0; j < kD; ++j) {
            am = fmaf(sDO[t * kLD + j], sU[s * kLD + j], am);
            at = fmaf(sDU[t * kLD + j], sX[s * kLD + j], at);
        }
        sdM[t * kLC + s] = s <= t ? am : 0.f;
        sdT[t * kLC + s] = at;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kM; ++m) {  // K_bar = b.k.e^G in place of w.v
        const int t = t0 + 2 * m;
        sX[t * kLD + c] = sBeta[t * kLD + c] * expf(sG[t * kLD + c]);
    }
    __syncthreads();
    for (int p = tid; p < kCb * kCb; p += 256) {
        const int t = p / kCb, s = p - t * kCb;
        float at = sdT[t * kLC + s];
        for (int j = 0; j < kD; ++j) at = fmaf(sBig[t * kLD + j], sX[s * kLD + j], at);
        sdT[t * kLC + s] = at;
    }
    __syncthreads();
    // ---- dU0 = T^T dU (-> dv, dw), dK_bar = T^T dW;  P = T^T dT
    float dKb[kM];
#pragma unroll 4
    for (int m = 0; m < kM; ++m) {
        const int t = t0 + 2 * m, tok = n * kCb + t;
        float du0 = 0.f, dkb = 0.f;
        for (int s = t; s < kCb; ++s) {
            const float ts = sT[s * kLC + t];
            du0 = fmaf(ts, sDU[s * kLD + c], du0);
            dkb = fmaf(ts, sBig[s * kLD + c], dkb);
        }
        dKb[m] = dkb;
        if (tok < T) {
            const size_t vh = (((size_t)bi * T + tok) * Hv + hv) * kD + c;
            dv[vh] = from_f32<Tin>(to_f32(w[vh]) * du0);
            dw[vh] = from_f32<Tin>(to_f32(v[vh]) * du0);
        }
    }
    for (int p = tid; p < kCb * kCb; p += 256) {
        const int t = p / kCb, s = p - t * kCb;
        float acc = 0.f;
        for (int r = t; r < kCb; ++r) acc = fmaf(sT[r * kLC + t], sdT[r * kLC + s], acc);
        sP[t * kLC + s] = acc;
    }
    __syncthreads();
    for (int p = tid; p < kCb * kCb; p += 256) {  // dA = -strict_tril(P T^T)
        const int t = p / kCb, s = p - t * kCb;
        float acc = 0.f;
        if (s < t)
            for (int r = 0; r <= s; ++r) acc = fmaf(sP[t * kLC + r], sT[s * kLC + r], acc);
        sdA[t * kLC + s] = -acc;
    }
    __syncthreads();
    // ---- the A and M terms pair by pair, then everything back to the inputs
    float dG[kM], dKhKh = 0.f;
#pragma unroll 2
    for (int m = 0; m < kM; ++m) {
        const int t = t0 + 2 * m, tok = n * kCb + t;
        const float Gt = sG[t * kLD + c];
        float X = 0.f, Y = sdM[t * kLC + t] * sK[t * kLD + c], Z = 0.f, V = sdM[t * kLC + t] * sQ[t * kLD + c];
        for (int s = 0; s < t; ++s) {
            const float e = expf(Gt - sG[s * kLD + c]);  // e^{G_t - G_s} <= 1
            const float ks = sK[s * kLD + c] * e;
            X = fmaf(sdA[t * kLC + s], ks, X);
            Y = fmaf(sdM[t * kLC + s], ks, Y);
        }
        for (int u = t + 1; u < kCb; ++u) {
            const float e = expf(sG[u * kLD + c] - Gt);  // e^{G_u - G_t} <= 1
            Z = fmaf(sdA[u * kLC + t], sBeta[u * kLD + c] * e, Z);
            V = fmaf(sdM[u * kLC + t], sQ[u * kLD + c] * e, V);
        }
        const float eG = expf(Gt), eH = expf(Glast - Gt);
        const float qq = sQ[t * kLD + c], kk = sK[t * kLD + c], be = sBeta[t * kLD + c];
        const float Qb = qq * eG, Kh = kk * eH, Kb = sX[t * kLD + c];
        const float dbeta = dKb[m] * eG + X;
        dG[m] = dQb[m] * Qb + dKb[m] * Kb - dKh[m] * Kh + be * X + qq * Y - kk * (Z + V);
        dKhKh = fmaf(dKh[m], Kh, dKhKh);
        if (tok < T) {
            const size_t vh = (((size_t)bi * T + tok) * Hv + hv) * kD + c;
            const float bb = to_f32(b[vh]);
            dq_ws[vh] = dQb[m] * eG + Y;
            dk_ws[vh] = dKh[m] * eH + Z + V + dbeta * bb;
            db[vh] = from_f32<Tin>(dbeta * kk);
        }
    }
    // dg_t = sum_{s >= t} dG_s + dG_last, dG_last = sum_t dK^.K^ + dgamma . e^{G_last}
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kM; ++m) sG[(t0 + 2 * m) * kLD + c] = dG[m];  // sG is no longer read
    sP[t0 * kD + c] = dKhKh;
    __syncthreads();
    if (tid < kD) {
        float run = sP[c] + sP[kD + c] + dgam * expf(Glast);  // dG_last
        for (int t = kCb - 1; t >= 0; --t) {
            run += sG[t * kLD + c];
            const int tok = n * kCb + t;
            if (tok < T) dg[(((size_t)bi * T + tok) * Hv + hv) * kD + c] = from_f32<Tin>(run);
        }
    }
}

// dq, dk of key head h_k = sums over the value heads of its group
template <typename Tout>
__global__ void __launch_bounds__(256) group_sum2_kernel(const float* __restrict__ dq_ws, const float* __restrict__ dk_ws,
                                                        Tout* __restrict__ dq, Tout* __restrict__ dk, long long rows,
                                                        int Hk, int Hv) {
    const int group = Hv / Hk;
    const long long n = rows * Hk * kD;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % kD);
        const long long rh = i / kD;
        const int hk = static_cast<int>(rh % Hk);
        const long long r = rh / Hk;
        float sq = 0.f, sk = 0.f;
        for (int m = 0; m < group; ++m) {
            const size_t src = ((static_cast<size_t>(r) * Hv) + hk * group + m) * kD + c;
            sq += dq_ws[src];
            sk += dk_ws[src];
        }
        dq[i] = from_f32<Tout>(sq);
        dk[i] = from_f32<Tout>(sk);
    }
}

struct ChunkBwdLayout {
    size_t simt, t, s, u, ds, du, dq, dk, total;
};
ChunkBwdLayout chunk_bwd_layout(int B, int T, int Hv) {
    const ChunkShape sh{B, T, 1, Hv, kD, kD, kCb};
    const size_t units = (size_t)sh.nchunks() * B * Hv, tok = (size_t)B * T * Hv * kD * 4;
    ChunkBwdLayout L;
    L.simt = 0;
    L.t = align_up(chunk_simt_workspace_bytes(sh), 256);
    L.s = align_up(L.t + units * kCb * kCb * 4, 256);
    L.u = align_up(L.s + units * kD * kD * 4, 256);
    L.ds = align_up(L.u + units * kCb * kD * 4, 256);
    L.du = align_up(L.ds + units * kD * kD * 4, 256);
    L.dq = align_up(L.du + units * kCb * kD * 4, 256);
    L.dk = align_up(L.dq + tok, 256);
    L.total = align_up(L.dk + tok, 256);
    return L;
}

template <typename Tin>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     const float* s0, const void* d_o, const float* dsT, void* dq, void* dk, void* dv, void* dg,
                     void* db, void* dw, float* ds0, int B, int T, int Hk, int Hv, float scale, uint8_t* ws,
                     cudaStream_t s) {
    const ChunkShape sh{B, T, Hk, Hv, kD, kD, kCb};
    const int NC = sh.nchunks();
    const ChunkBwdLayout L = chunk_bwd_layout(B, T, Hv);
    float* simt = reinterpret_cast<float*>(ws + L.simt);
    float* t_ws = reinterpret_cast<float*>(ws + L.t);
    float* s_save = reinterpret_cast<float*>(ws + L.s);
    float* u_save = reinterpret_cast<float*>(ws + L.u);
    float* ds_save = reinterpret_cast<float*>(ws + L.ds);
    float* du_save = reinterpret_cast<float*>(ws + L.du);
    float* dq_ws = reinterpret_cast<float*>(ws + L.dq);
    float* dk_ws = reinterpret_cast<float*>(ws + L.dk);
    cudaError_t e = launch_chunk_simt_saving(q, k, v, g, b, w, s0, sh, std::is_same<Tin, float>::value ? GDN2_F32 : GDN2_BF16,
                                             simt, t_ws, s_save, u_save, s);
    if (e != cudaSuccess) return e;
    const size_t a_smem = sizeof(float) * ((size_t)kD * kSl + 3 * (size_t)kD * kCb + kCb * kCb + kD + 2 * kCb * kSl);
    const size_t g_smem = sizeof(float) * (8 * (size_t)kCb * kLD + (size_t)kD * kLD + 6 * (size_t)kCb * kLC);
    e = cudaFuncSetAttribute(adjoint_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)a_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grad_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g_smem);
    if (e != cudaSuccess) return e;
    adjoint_kernel<Tin><<<dim3(B * Hv, kD / kSl), 256, a_smem, s>>>(simt, static_cast<const Tin*>(d_o), dsT, ds0,
                                                                    ds_save, du_save, T, Hv, NC, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    grad_kernel<Tin><<<dim3(NC, B * Hv), 256, g_smem, s>>>(
        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v), static_cast<const Tin*>(g),
        static_cast<const Tin*>(b), static_cast<const Tin*>(w), static_cast<const Tin*>(d_o), simt, t_ws, s_save, u_save,
        ds_save, du_save, dq_ws, dk_ws, static_cast<Tin*>(dv), static_cast<Tin*>(dg), static_cast<Tin*>(db),
        static_cast<Tin*>(dw), T, Hk, Hv, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long rows = (long long)B * T, nk = rows * Hk * kD;
    const int gs = static_cast<int>(nk / 256 + 1 < 4096 ? nk / 256 + 1 : 4096);
    group_sum2_kernel<Tin><<<gs, 256, 0, s>>>(dq_ws, dk_ws, static_cast<Tin*>(dq), static_cast<Tin*>(dk), rows, Hk, Hv);
    return cudaGetLastError();
}

}  // namespace

size_t backward_chunked_workspace_bytes(int B, int T, int Hv) { return chunk_bwd_layout(B, T, Hv).total; }

cudaError_t launch_backward_chunked(const void* q, const void* k, const void* v, const void* g, const void* b,
                                    const void* w, const float* s0, const void* d_o, const float* dsT, void* dq,
                                    void* dk, void* dv, void* dg, void* db, void* dw, float* ds0, int B, int T, int Hk,
                                    int Hv, float scale, gdn2_dtype dt, void* ws, cudaStream_t s) {
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if (dt == GDN2_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, g, b, w, s0, d_o, dsT, dq, dk, dv, dg, db, dw, ds0, B, T, Hk, Hv, scale,
                                       wsb, s);
    return launch_t<float>(q, k, v, g, b, w, s0, d_o, dsT, dq, dk, dv, dg, db, dw, ds0, B, T, Hk, Hv, scale, wsb, s);
}

}  // namespace gdn2

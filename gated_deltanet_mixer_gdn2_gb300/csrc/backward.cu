// backward.cu -- gradients of the GDN-2 core, exact, in recurrent form (the recurrence of the
// burn-gdn2 0.1.5 docs, "Architecture"):
//     S_t = (I - k_t (b_t . k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t . v_t)^T,  o_t = scale S_t^T q_t.
// With P = diag(alpha_t) S_{t-1}, beta = b_t . k_t, u = w_t . v_t, r = P^T beta, delta = u - r and
// G = dL/dS_t (from o_t and from S_{t+1}), reverse mode gives, per token:
//     x = G^T k,  dv = w . x,  dw = v . x,
//     dk = G delta + b . dbeta,  dbeta = -P x,  db = k . dbeta,
//     dg = alpha . rowsum((G - beta x^T) . S_{t-1}),  dq = scale (P do + k (delta . do)),
//     dL/dS_{t-1} = diag(alpha) (G - beta x^T) + scale q_{t-1} do_{t-1}^T.
// The walk back needs S_{t-1} for every t: the states at every kChk-th token are saved in a first
// forward sweep, and each stretch of kChk tokens is recomputed into a scratch buffer (L2-sized)
// before it is walked backward. The columns of S (and of its gradient) evolve independently, so two
// CTAs per (batch, value head) each hold 64 of the d_v columns of the fp32 state and its gradient in
// registers: warp w owns 8 columns, lane = 16 row groups x 2 column groups, 8 rows x 4 columns per
// thread. Column sums (over d_k) are in-thread plus shuffles; row sums (over d_v) go through shared
// memory and leave the CTA as fp32 partial sums (they are linear in the columns): a second kernel
// adds the two halves, and for q and k also the value heads of each key head's group, in a fixed
// order. Arithmetic is fp32.
#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kD = 128;
constexpr int kCols = 64;     // d_v columns per CTA
constexpr int kChk = 32;      // checkpoint interval = tokens recomputed at a time
constexpr int kThreads = 256;
constexpr int kParts = 2 * (kThreads / 32);  // row-sum partials per row inside a CTA: one per (warp, column group)

struct BwdArgs {
    const void *q, *k, *v, *g, *b, *w, *dout;
    const float* s0;      // nullable
    const float* dsT;     // nullable
    float* part;          // [4 sums][2 halves][B, T, H_v, 128] fp32: dq, dk, db, dg partial sums
    void *dv, *dg, *db, *dw;
    float* ds0;           // nullable
    float *ckpt, *scratch;
    int B, T, Hk, Hv;
    float scale;
};

constexpr int kBatch = 8;  // token vectors staged in shared memory at a time

// token vectors in shared memory (alpha = e^g, beta = b . k, u = w . v precomputed when staged)
struct Tok {
    float k[kD], q[kD], beta[kD], alpha[kD], u[kD], v[kD], w[kD], dO[kD], b[kD];
};

// Stage tokens t_lo .. t_lo + n - 1 into slots 0 .. n-1 (all loads of the batch issued together).
template <typename T>
__device__ void stage_tokens(const BwdArgs& a, int bi, int hv, int t_lo, int n, Tok* tk) {
    const int hk = hv / (a.Hv / a.Hk);
    const int i = threadIdx.x & (kD - 1);
    const bool low = threadIdx.x < kD;
    float r0[kBatch], r1[kBatch], r2[kBatch], r3[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        if (j >= n) break;
        const int t = t_lo + j;
        const size_t kq = ((static_cast<size_t>(bi) * a.T + t) * a.Hk + hk) * kD;
        const size_t vh = ((static_cast<size_t>(bi) * a.T + t) * a.Hv + hv) * kD;
        if (low) {
            r0[j] = to_f32(static_cast<const T*>(a.k)[kq + i]);
            r1[j] = to_f32(static_cast<const T*>(a.b)[vh + i]);
            r2[j] = to_f32(static_cast<const T*>(a.q)[kq + i]);
            r3[j] = to_f32(static_cast<const T*>(a.g)[vh + i]);
        } else {
            r0[j] = to_f32(static_cast<const T*>(a.v)[vh + i]);
            r1[j] = to_f32(static_cast<const T*>(a.w)[vh + i]);
            r2[j] = to_f32(static_cast<const T*>(a.dout)[vh + i]);
        }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        if (j >= n) break;
        Tok& x = tk[j];
        if (low) {
            x.k[i] = r0[j];
            x.b[i] = r1[j];
            x.beta[i] = r0[j] * r1[j];
            x.q[i] = r2[j];
            x.alpha[i] = expf(r3[j]);
        } else {
            x.v[i] = r0[j];
            x.w[i] = r1[j];
            x.u[i] = r0[j] * r1[j];
            x.dO[i] = r2[j];
        }
    }
}

// sum over the 16 row groups of a warp (lanes differing in bits 1..4)
__device__ __forceinline__ float col_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

// one forward token on this thread's 8 x 4 tile (c0: global d_v column)
__device__ __forceinline__ void forward_step(float (&S)[8][4], const Tok& tk, int r0, int c0) {
    float r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float al = tk.alpha[r0 + i], be = tk.beta[r0 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            S[i][j] *= al;
            r[j] = fmaf(be, S[i][j], r[j]);
        }
    }
    float d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = tk.u[c0 + j] - col_sum(r[j]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float kk = tk.k[r0 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) S[i][j] = fmaf(kk, d[j], S[i][j]);
    }
}

// ld: row stride of the stored matrix (kD for [d_k][d_v] states, kCols for this CTA's compact copies)
__device__ __forceinline__ void tile_load(float (&S)[8][4], const float* base, int ld, int r0, int c0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(base + (r0 + i) * ld + c0);
        S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
    }
}
__device__ __forceinline__ void tile_store(const float (&S)[8][4], float* base, int ld, int r0, int c0) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float4*>(base + (r0 + i) * ld + c0) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) backward_kernel(const __grid_constant__ BwdArgs a) {
    extern __shared__ float4 smem_f4[];
    float* smem = reinterpret_cast<float*>(smem_f4);
    Tok* tks = reinterpret_cast<Tok*>(smem);                       // [kBatch] staged tokens
    float* red = smem + kBatch * sizeof(Tok) / sizeof(float);      // [kParts][4 sums][128 rows]
    float* xcol = red + kParts * 4 * kD;                           // x = G^T k per column of this CTA [64]
    float* sdot = xcol + kCols;                                    // [kParts] partial delta . do

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 1, cg = lane & 1;
    const int r0 = 8 * rg, lc = 8 * warp + 4 * cg;  // first row; first column within the CTA's 64
    const int bh = blockIdx.x >> 1, hc = blockIdx.x & 1;
    const int c0 = kCols * hc + lc;                  // first column within d_v
    const int bi = bh / a.Hv, hv = bh - bi * a.Hv;
    const int nT = a.T;
    const int nchk = (nT + kChk - 1) / kChk;
    const size_t st = static_cast<size_t>(kD) * kCols;  // floats per compact [d_k][64] state copy
    float* ckpt = a.ckpt + static_cast<size_t>(blockIdx.x) * (nchk + 1) * st;
    float* scratch = a.scratch + static_cast<size_t>(blockIdx.x) * kChk * st;
    const size_t sbase = static_cast<size_t>(bh) * kD * kD;  // this head's [d_k][d_v] state

    // ---- forward sweep: save the state at every kChk-th token
    float S[8][4];
    if (a.s0) tile_load(S, a.s0 + sbase, kD, r0, c0);
    else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) S[i][j] = 0.f;
    }
    tile_store(S, ckpt, kCols, r0, lc);
    for (int tb = 0; tb < nT; tb += kBatch) {
        const int n = min(kBatch, nT - tb);
        __syncthreads();
        stage_tokens<T>(a, bi, hv, tb, n, tks);
        __syncthreads();
        for (int j = 0; j < n; ++j) {
            const int t = tb + j;
            forward_step(S, tks[j], r0, c0);
            if ((t + 1) % kChk == 0 && t + 1 < nT) tile_store(S, ckpt + static_cast<size_t>((t + 1) / kChk) * st, kCols, r0, lc);
        }
    }

    // ---- backward sweep
    float G[8][4];  // dL/dS after the token being processed (before its own readout term)
    if (a.dsT) tile_load(G, a.dsT + sbase, kD, r0, c0);
    else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) G[i][j] = 0.f;
    }
    const size_t nsum = static_cast<size_t>(a.B) * nT * a.Hv * kD;  // elements of one partial-sum array
    for (int c = nchk - 1; c >= 0; --c) {
        const int t0 = c * kChk, t1 = min(nT, t0 + kChk);
        // recompute the states before tokens t0 .. t1-1 into the scratch
        tile_load(S, ckpt + static_cast<size_t>(c) * st, kCols, r0, lc);
        for (int tb = t0; tb < t1; tb += kBatch) {
            const int n = min(kBatch, t1 - tb);
            __syncthreads();
            stage_tokens<T>(a, bi, hv, tb, n, tks);
            __syncthreads();
            for (int j = 0; j < n; ++j) {
                tile_store(S, scratch + static_cast<size_t>(tb + j - t0) * st, kCols, r0, lc);
                if (tb + j + 1 < t1) forward_step(S, tks[j], r0, c0);
            }
        }
        // walk back, kBatch tokens staged at a time (highest first); the state before the next token
        // is loaded from the scratch one token ahead
        float Sn[8][4];
        tile_load(Sn, scratch + static_cast<size_t>(t1 - 1 - t0) * st, kCols, r0, lc);
        for (int te = t1; te > t0; te -= kBatch) {
            const int tb = max(t0, te - kBatch), n = te - tb;
            __syncthreads();
            stage_tokens<T>(a, bi, hv, tb, n, tks);
            for (int j = n - 1; j >= 0; --j) {
                const int t = tb + j;
                const Tok& tk = tks[j];
                __syncthreads();  // staged tokens visible; the previous token's reductions have been read
                float (&Sp)[8][4] = S;  // state before token t
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) Sp[i][jj] = Sn[i][jj];
                if (t - 1 >= t0) tile_load(Sn, scratch + static_cast<size_t>(t - 1 - t0) * st, kCols, r0, lc);
                // G += scale q do^T (readout of token t)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float qs = a.scale * tk.q[r0 + i];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) G[i][jj] = fmaf(qs, tk.dO[c0 + jj], G[i][jj]);
                }
                // column sums: x = G^T k, r = P^T beta with P = alpha . S_prev
                float x[4] = {0.f, 0.f, 0.f, 0.f}, r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float kk = tk.k[r0 + i], pb = tk.alpha[r0 + i] * tk.beta[r0 + i];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        x[jj] = fmaf(G[i][jj], kk, x[jj]);
                        r[jj] = fmaf(Sp[i][jj], pb, r[jj]);
                    }
                }
                float dl[4];
                float sd = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    x[jj] = col_sum(x[jj]);
                    dl[jj] = tk.u[c0 + jj] - col_sum(r[jj]);
                    sd = fmaf(dl[jj], tk.dO[c0 + jj], sd);
                }
                if (rg == 0) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) xcol[lc + jj] = x[jj];
                    sdot[warp * 2 + cg] = sd;
                }
                // row sums over this thread's 4 columns: G delta, P x, P do, (G - beta x^T) . S_prev;
                // then G <- alpha (G - beta x^T), the gradient for the state before token t
                float* rd = red + (warp * 2 + cg) * 4 * kD;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = r0 + i;
                    const float al = tk.alpha[row], be = tk.beta[row];
                    float s_a = 0.f, s_c = 0.f, s_e = 0.f, s_f = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float p = al * Sp[i][jj];
                        s_a = fmaf(G[i][jj], dl[jj], s_a);
                        s_c = fmaf(p, x[jj], s_c);
                        s_e = fmaf(p, tk.dO[c0 + jj], s_e);
                        const float gm = fmaf(-be, x[jj], G[i][jj]);
                        s_f = fmaf(gm, Sp[i][jj], s_f);
                        G[i][jj] = al * gm;
                    }
                    rd[row] = s_a;
                    rd[kD + row] = s_c;
                    rd[2 * kD + row] = s_e;
                    rd[3 * kD + row] = s_f;
                }
                __syncthreads();
                const size_t vh = ((static_cast<size_t>(bi) * nT + t) * a.Hv + hv) * kD;
                if (tid < kD) {
                    // this half's share of dk, dq, db, dg (linear in the columns)
                    const int row = tid;
                    float s_a = 0.f, s_c = 0.f, s_e = 0.f, s_f = 0.f, s_d = 0.f;
#pragma unroll 4
                    for (int p = 0; p < kParts; ++p) {
                        const float* rp = red + p * 4 * kD;
                        s_a += rp[row];
                        s_c += rp[kD + row];
                        s_e += rp[2 * kD + row];
                        s_f += rp[3 * kD + row];
                        s_d += sdot[p];
                    }
                    const float kk = tk.k[row], bb = tk.b[row];
                    const float dbeta = -s_c;
                    float* pp = a.part + static_cast<size_t>(hc) * nsum + vh + row;
                    pp[0] = a.scale * (s_e + kk * s_d);  // dq
                    pp[2 * nsum] = s_a + bb * dbeta;     // dk
                    pp[4 * nsum] = kk * dbeta;           // db
                    pp[6 * nsum] = tk.alpha[row] * s_f;  // dg
                } else if (tid < kD + kCols) {
                    const int col = tid - kD, gc = kCols * hc + col;
                    const float xx = xcol[col];
                    static_cast<T*>(a.dv)[vh + gc] = from_f32<T>(tk.w[gc] * xx);
                    static_cast<T*>(a.dw)[vh + gc] = from_f32<T>(tk.v[gc] * xx);
                }
            }
        }
    }
    if (a.ds0) tile_store(G, a.ds0 + sbase, kD, r0, c0);
}

// dq, dk of key head h_k = sums over the two column halves and the value heads of its group; db, dg =
// sums over the two halves. part = [dq, dk, db, dg][half][B, T, H_v, 128].
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part, T* __restrict__ dq,
                                                     T* __restrict__ dk, T* __restrict__ db, T* __restrict__ dg,
                                                     long long rows, int Hk, int Hv) {
    const int group = Hv / Hk;
    const size_t nsum = static_cast<size_t>(rows) * Hv * kD;
    const long long nk = rows * Hk * kD, nv = rows * Hv * kD;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nk; i += stride) {
        const int c = static_cast<int>(i % kD);
        const long long rh = i / kD;
        const int hk = static_cast<int>(rh % Hk);
        const long long r = rh / Hk;
        float sq = 0.f, sk = 0.f;
        for (int m = 0; m < group; ++m) {
            const size_t src = ((static_cast<size_t>(r) * Hv) + hk * group + m) * kD + c;
            sq += part[src] + part[nsum + src];
            sk += part[2 * nsum + src] + part[3 * nsum + src];
        }
        dq[i] = from_f32<T>(sq);
        dk[i] = from_f32<T>(sk);
    }
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nv; i += stride) {
        db[i] = from_f32<T>(part[4 * nsum + i] + part[5 * nsum + i]);
        dg[i] = from_f32<T>(part[6 * nsum + i] + part[7 * nsum + i]);
    }
}

struct BwdLayout {
    size_t ckpt, scratch, part, total;
};
BwdLayout bwd_layout(int B, int T, int Hv) {
    const size_t ctas = static_cast<size_t>(B) * Hv * 2, st = static_cast<size_t>(kD) * kCols * 4;
    const size_t nchk = (T + kChk - 1) / kChk;
    BwdLayout L;
    L.ckpt = 0;
    L.scratch = align_up(ctas * (nchk + 1) * st, 256);
    L.part = align_up(L.scratch + ctas * kChk * st, 256);
    L.total = align_up(L.part + 8 * static_cast<size_t>(B) * T * Hv * kD * 4, 256);
    return L;
}

bool bwd_shape_ok(int B, int T, int Hk, int Hv, int dk, int dv) {
    // (batch, value head) is the second grid dimension of the per-chunk kernels (at most 65535)
    return B >= 0 && T >= 0 && Hk > 0 && Hv > 0 && Hv % Hk == 0 && dk == kD && dv == kD &&
           static_cast<long long>(B) * T * Hv < (1LL << 31) / kD && static_cast<long long>(B) * Hv <= 65535;
}
// The chunked form's shapes: bf16 (tensor cores) takes d_k and d_v of 64 or 128, fp32 128 only.
bool chunked_shape_ok(int B, int T, int Hk, int Hv, int dk, int dv, gdn2_dtype dt) {
    if (dt != GDN2_BF16) return bwd_shape_ok(B, T, Hk, Hv, dk, dv);
    return bwd_shape_ok(B, T, Hk, Hv, kD, kD) && (dk == 64 || dk == kD) && (dv == 64 || dv == kD);
}

}  // namespace
}  // namespace gdn2

using namespace gdn2;

namespace {

// Checks shared by both entry points; handles the empty sequence (dS0 = dS_T). Returns GDN2_OK with
// *done = false when the caller should launch.
gdn2_status check_and_trivial(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                              const float* initial_state, const void* d_o, const float* d_final_state, void* dq,
                              void* dk, void* dv, void* dg, void* db, void* dw, float* d_initial_state, int B, int T,
                              int Hk, int Hv, int d_k, int d_v, gdn2_dtype dt, void* workspace, size_t ws_bytes,
                              size_t need, cudaStream_t s, bool* done, bool chunked) {
    *done = true;
    if (dt != GDN2_F32 && dt != GDN2_BF16) return GDN2_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || d_k <= 0 || d_v <= 0 || Hv % Hk) return GDN2_ERR_INVALID_ARG;
    if (!(chunked ? chunked_shape_ok(B, T, Hk, Hv, d_k, d_v, dt) : bwd_shape_ok(B, T, Hk, Hv, d_k, d_v)))
        return GDN2_ERR_UNSUPPORTED;
    const size_t state_bytes = sizeof(float) * static_cast<size_t>(B) * Hv * d_k * d_v;
    if (B == 0 || T == 0) {  // no tokens: dS0 = dS_T
        if (d_initial_state && state_bytes) {
            if (!aligned16(d_initial_state)) return GDN2_ERR_MISALIGNED;
            const cudaError_t e = d_final_state ? cudaMemcpyAsync(d_initial_state, d_final_state, state_bytes,
                                                                  cudaMemcpyDeviceToDevice, s)
                                                : cudaMemsetAsync(d_initial_state, 0, state_bytes, s);
            if (e != cudaSuccess) return GDN2_ERR_CUDA;
        }
        return GDN2_OK;
    }
    const void* req[] = {q, k, v, g, b, w, d_o, dq, dk, dv, dg, db, dw};
    for (const void* p : req)
        if (!p) return GDN2_ERR_INVALID_ARG;
    for (const void* p : req)
        if (!aligned16(p)) return GDN2_ERR_MISALIGNED;
    if ((initial_state && !aligned16(initial_state)) || (d_final_state && !aligned16(d_final_state)) ||
        (d_initial_state && !aligned16(d_initial_state)))
        return GDN2_ERR_MISALIGNED;
    if (!workspace || ws_bytes < need) return GDN2_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GDN2_ERR_MISALIGNED;
    *done = false;
    return GDN2_OK;
}

}  // namespace

extern "C" {

size_t gdn2_backward_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, gdn2_dtype dt) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || !chunked_shape_ok(B, T, Hk, Hv, dk, dv, dt) || B == 0 || T == 0)
        return 0;
    return dt == GDN2_BF16 ? backward_tc_workspace_bytes(B, T, Hv, dk, dv) : backward_chunked_workspace_bytes(B, T, Hv);
}

gdn2_status gdn2_backward(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                          const float* initial_state, const void* d_o, const float* d_final_state, void* dq, void* dk,
                          void* dv, void* dg, void* db, void* dw, float* d_initial_state, int B, int T, int Hk, int Hv,
                          int d_k, int d_v, float scale, gdn2_dtype dt, void* workspace, size_t ws_bytes,
                          void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool done;
    const size_t need = gdn2_backward_workspace_size(B, T, Hk, Hv, d_k, d_v, dt);
    const gdn2_status st = check_and_trivial(q, k, v, g, b, w, initial_state, d_o, d_final_state, dq, dk, dv, dg, db,
                                             dw, d_initial_state, B, T, Hk, Hv, d_k, d_v, dt, workspace, ws_bytes, need,
                                             s, &done, true);
    if (done) return st;
    if (dt == GDN2_BF16)  // tensor cores: chunks of 64, bf16 operands, fp32 accumulators and state
        return launch_backward_tc(q, k, v, g, b, w, initial_state, d_o, d_final_state, dq, dk, dv, dg, db, dw,
                                  d_initial_state, B, T, Hk, Hv, d_k, d_v, scale, workspace, s,
                                  wait_limit_ns()) == cudaSuccess
                   ? GDN2_OK
                   : GDN2_ERR_CUDA;
    return launch_backward_chunked(q, k, v, g, b, w, initial_state, d_o, d_final_state, dq, dk, dv, dg, db, dw,
                                   d_initial_state, B, T, Hk, Hv, scale, dt, workspace, s) == cudaSuccess
               ? GDN2_OK
               : GDN2_ERR_CUDA;
}

size_t gdn2_backward_recurrent_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, gdn2_dtype dt) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || !bwd_shape_ok(B, T, Hk, Hv, dk, dv) || B == 0 || T == 0) return 0;
    return bwd_layout(B, T, Hv).total;
}

gdn2_status gdn2_backward_recurrent(const void* q, const void* k, const void* v, const void* g, const void* b,
                                    const void* w, const float* initial_state, const void* d_o,
                                    const float* d_final_state, void* dq, void* dk, void* dv, void* dg, void* db,
                                    void* dw, float* d_initial_state, int B, int T, int Hk, int Hv, int d_k, int d_v,
                                    float scale, gdn2_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool done;
    const size_t need = bwd_shape_ok(B, T, Hk, Hv, d_k, d_v) && B > 0 && T > 0 ? bwd_layout(B, T, Hv).total : 0;
    const gdn2_status st = check_and_trivial(q, k, v, g, b, w, initial_state, d_o, d_final_state, dq, dk, dv, dg, db,
                                             dw, d_initial_state, B, T, Hk, Hv, d_k, d_v, dt, workspace, ws_bytes, need,
                                             s, &done, false);
    if (done) return st;
    const BwdLayout L = bwd_layout(B, T, Hv);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    BwdArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.b = b; a.w = w; a.dout = d_o;
    a.s0 = initial_state; a.dsT = d_final_state;
    a.part = reinterpret_cast<float*>(ws + L.part);
    a.dv = dv; a.dg = dg; a.db = db; a.dw = dw; a.ds0 = d_initial_state;
    a.ckpt = reinterpret_cast<float*>(ws + L.ckpt);
    a.scratch = reinterpret_cast<float*>(ws + L.scratch);
    a.B = B; a.T = T; a.Hk = Hk; a.Hv = Hv; a.scale = scale;
    const size_t smem = kBatch * sizeof(Tok) + (kParts * 4 * kD + kCols + kParts) * sizeof(float);
    cudaError_t e;
    const long long rows = static_cast<long long>(B) * T;
    const long long n = rows * Hv * kD;
    const int gs = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    if (dt == GDN2_BF16) {
        e = cudaFuncSetAttribute(backward_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return GDN2_ERR_CUDA;
        backward_kernel<__nv_bfloat16><<<2 * B * Hv, kThreads, smem, s>>>(a);
        if (cudaGetLastError() != cudaSuccess) return GDN2_ERR_CUDA;
        combine_kernel<__nv_bfloat16><<<gs, 256, 0, s>>>(a.part, static_cast<__nv_bfloat16*>(dq),
                                                         static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(db),
                                                         static_cast<__nv_bfloat16*>(dg), rows, Hk, Hv);
    } else {
        e = cudaFuncSetAttribute(backward_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return GDN2_ERR_CUDA;
        backward_kernel<float><<<2 * B * Hv, kThreads, smem, s>>>(a);
        if (cudaGetLastError() != cudaSuccess) return GDN2_ERR_CUDA;
        combine_kernel<float><<<gs, 256, 0, s>>>(a.part, static_cast<float*>(dq), static_cast<float*>(dk),
                                                 static_cast<float*>(db), static_cast<float*>(dg), rows, Hk, Hv);
    }
    return cudaGetLastError() == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

}  // extern "C"

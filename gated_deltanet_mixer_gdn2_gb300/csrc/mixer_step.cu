// mixer_step.cu -- gdn2_mixer_decode_step: one decode token of the whole token mixer around the core,
// in one launch: ShortConv on the q, k, v projections with their carried conv states, L2 norm of q and
// k, the gate activations, the recurrent update of the core state, and the gated RMSNorm with the
// SiLU gate (burn-gdn2 0.1.5 docs, "Architecture": projections -> ShortConv -> L2-Norm -> Fused
// Recurrent -> Gated RMS Norm <- SiLU Gate; the llama.cpp GDN decode study, section 4, suggests fusing
// the conv and the gated norm into the delta-net kernel of a decode step).
//
// Per token the same operations as gdn2_mixer_prologue (T = 1), gdn2_recurrent_step and
// gdn2_mixer_epilogue in sequence:
//   q = L2norm(conv(xq)), k = L2norm(conv(xk)), v = conv(xv), conv(x)[c] = sum_j W[c][j] x_{-3+j}[c]
//   (x_0 the current token, x_{-3..-1} from the carried state, which then keeps x_{-2}, x_{-1}, x_0);
//   alpha = e^{-softplus(a_g)} = sigmoid(-a_g), b = sigmoid(a_b) (x 2 with negative eigenvalues),
//   w = sigmoid(a_w);
//   S' = diag(alpha) S, d = w.v - S'^T(b.k), S <- S' + k d^T, o = scale (S'^T q + (k.q) d);
//   y = o / sqrt(mean(o^2) + eps) * weight * silu(z).
// Two layouts, both with thread c on channel c of the per-head vectors and, for the state update, warp w
// on columns 16 w .. 16 w + 15 of the d_k x d_v fp32 state with lane = 8 row groups x 4 column groups
// (reductions over d_k in-thread, then across the row groups by shuffles, as the register decode
// kernel); the intermediate q, k, v, gates and o never leave the SM.
//   Up to 8 value heads per key head: one CTA per (batch row, value head), the CTAs of a key head's
//   group one thread-block cluster. Every load of the CTA (its state slice, the token vectors, the conv
//   states and weights, the gates) is issued at its start; each CTA computes q and k from the carried
//   conv states, and after a cluster barrier (all of them have read those states) the first CTA of
//   the cluster writes the new q and k conv states, so every conv state has one writer.
//   Larger groups: one CTA per (batch row, key head) computes q and k once, updates their conv states,
//   and runs the value heads of the group one after the other.
//   Many heads (d_k = d_v = 128, at least four value heads per SM): a persistent grid, each CTA a
//   contiguous run of (batch row, key head) units, so the value heads of a key head are processed by
//   one CTA one after another; a ring of shared-memory slots holds each head's state slab, token
//   vectors and carried conv states by bulk copy, loaded ahead of the head being computed, and the
//   updated state goes back through its slot by bulk copy. The last value head of a key head writes
//   the new q and k conv states: its siblings' copies of the old ones have all landed by then.
#include <cooperative_groups.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gdn2 {
namespace {

constexpr int kStepTaps = 4;
constexpr float kStepL2Eps = 1e-6f;
constexpr int kMaxClusterGroup = 8;  // portable cluster size

__device__ int g_status_step;
int g_step_sms = 0;

__device__ __forceinline__ float sigmoid_acc(float a) { return 1.f / (1.f + expf(-a)); }

// Sum of v over the 256 threads of the block; every thread gets the result. red: 8 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();  // red is free (its previous readers are done)
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w];
    return s;
}

// One channel of the causal conv: y = sum_j W[j] x_{-3+j}; the carried state moves one sample on.
template <typename T>
__device__ __forceinline__ float conv_channel(const T* x, const float* wt, float* state, size_t C, size_t ch,
                                              size_t bi) {
    const float cur = to_f32(x[0]);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f;
    float* sp = state ? state + bi * (kStepTaps - 1) * C + ch : nullptr;
    if (sp) {
        s0 = sp[0];
        s1 = sp[C];
        s2 = sp[2 * C];
    }
    const float4 w = *reinterpret_cast<const float4*>(wt + ch * kStepTaps);
    if (sp) {
        sp[0] = s1;
        sp[C] = s2;
        sp[2 * C] = cur;
    }
    return w.x * s0 + w.y * s1 + w.z * s2 + w.w * cur;
}

template <int DK, typename T>
__global__ void __launch_bounds__(256)
    mixer_step_kernel(const T* __restrict__ xq, const T* __restrict__ xk, const T* __restrict__ xv,
                      const float* __restrict__ cq, const float* __restrict__ ck, const float* __restrict__ cv,
                      const T* __restrict__ ag, const T* __restrict__ ab, const T* __restrict__ aw,
                      float* __restrict__ sq, float* __restrict__ sk, float* __restrict__ sv,
                      float* __restrict__ state, const T* __restrict__ z, const float* __restrict__ weight,
                      float eps, T* __restrict__ y, int Hk, int Hv, int dv, int neg_eigval, float scale) {
    __shared__ float s_q[DK], s_k[DK], s_a[DK], s_bk[DK];
    __shared__ float s_wv[128], s_o[128];
    __shared__ float s_red[8];
    constexpr int RPL = DK / 8;  // state rows per lane
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bi = blockIdx.x / Hk, hk = blockIdx.x - bi * Hk;
    const int G = Hv / Hk;

    // ---- q, k: conv (one thread per channel), L2 norm per head
    float qv = 0.f, kv = 0.f;
    if (tid < DK) {
        const size_t C = static_cast<size_t>(Hk) * DK, ch = static_cast<size_t>(hk) * DK + tid;
        const size_t xi = (static_cast<size_t>(bi) * Hk + hk) * DK + tid;
        qv = conv_channel(xq + xi, cq, sq, C, ch, bi);
        kv = conv_channel(xk + xi, ck, sk, C, ch, bi);
    }
    const float nq = rsqrtf(block_sum(qv * qv, s_red) + kStepL2Eps);
    const float nk = rsqrtf(block_sum(kv * kv, s_red) + kStepL2Eps);
    if (tid < DK) {
        s_q[tid] = qv * nq;
        s_k[tid] = kv * nk;
    }
    const float kq = block_sum(tid < DK ? (kv * nk) * (qv * nq) : 0.f, s_red);  // also publishes s_q, s_k

    for (int hv = hk * G; hv < hk * G + G; ++hv) {
        const size_t head = static_cast<size_t>(bi) * Hv + hv;
        // ---- per-head vectors: alpha, b.k over d_k; w.v (with v's conv) over d_v
        if (tid < DK) {
            const float a = to_f32(ag[head * DK + tid]), bb = to_f32(ab[head * DK + tid]);
            s_a[tid] = sigmoid_acc(-a);  // e^{-softplus(a)}
            s_bk[tid] = sigmoid_acc(bb) * (neg_eigval ? 2.f : 1.f) * s_k[tid];
        }
        if (tid < dv) {
            const size_t C = static_cast<size_t>(Hv) * dv, ch = static_cast<size_t>(hv) * dv + tid;
            const float vv = conv_channel(xv + head * dv + tid, cv, sv, C, ch, bi);
            s_wv[tid] = sigmoid_acc(to_f32(aw[head * dv + tid])) * vv;
        }
        __syncthreads();
        // ---- the recurrent update: warp w, columns 16 w .. 16 w + 15
        const int cg = lane & 3, rg = lane >> 2;
        const int col = 16 * warp + 4 * cg;
        if (16 * warp < dv) {
            float* S = state + head * DK * dv + col;
            float4 s[RPL];
#pragma unroll
            for (int i = 0; i < RPL; ++i) s[i] = *reinterpret_cast<const float4*>(S + static_cast<size_t>(rg + 8 * i) * dv);
            float4 rb = make_float4(0.f, 0.f, 0.f, 0.f), rq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                const int r = rg + 8 * i;
                const float a = s_a[r], bk = s_bk[r], qq = s_q[r];
                s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
                rb.x = fmaf(s[i].x, bk, rb.x); rb.y = fmaf(s[i].y, bk, rb.y);
                rb.z = fmaf(s[i].z, bk, rb.z); rb.w = fmaf(s[i].w, bk, rb.w);
                rq.x = fmaf(s[i].x, qq, rq.x); rq.y = fmaf(s[i].y, qq, rq.y);
                rq.z = fmaf(s[i].z, qq, rq.z); rq.w = fmaf(s[i].w, qq, rq.w);
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {  // the 8 row groups: lanes that differ in bits 2..4
                rb.x += __shfl_xor_sync(0xffffffffu, rb.x, off);
                rb.y += __shfl_xor_sync(0xffffffffu, rb.y, off);
                rb.z += __shfl_xor_sync(0xffffffffu, rb.z, off);
                rb.w += __shfl_xor_sync(0xffffffffu, rb.w, off);
                rq.x += __shfl_xor_sync(0xffffffffu, rq.x, off);
                rq.y += __shfl_xor_sync(0xffffffffu, rq.y, off);
                rq.z += __shfl_xor_sync(0xffffffffu, rq.z, off);
                rq.w += __shfl_xor_sync(0xffffffffu, rq.w, off);
            }
            const float4 d = make_float4(s_wv[col] - rb.x, s_wv[col + 1] - rb.y, s_wv[col + 2] - rb.z,
                                         s_wv[col + 3] - rb.w);
            if (rg == 0) {
                s_o[col] = scale * fmaf(kq, d.x, rq.x);
                s_o[col + 1] = scale * fmaf(kq, d.y, rq.y);
                s_o[col + 2] = scale * fmaf(kq, d.z, rq.z);
                s_o[col + 3] = scale * fmaf(kq, d.w, rq.w);
            }
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                const float kk = s_k[rg + 8 * i];
                s[i].x = fmaf(kk, d.x, s[i].x); s[i].y = fmaf(kk, d.y, s[i].y);
                s[i].z = fmaf(kk, d.z, s[i].z); s[i].w = fmaf(kk, d.w, s[i].w);
                *reinterpret_cast<float4*>(S + static_cast<size_t>(rg + 8 * i) * dv) = s[i];
            }
        }
        // ---- gated RMSNorm with the SiLU gate over d_v
        __syncthreads();  // s_o complete
        const float o_c = tid < dv ? s_o[tid] : 0.f;
        const float mean_sq = block_sum(o_c * o_c, s_red) / static_cast<float>(dv);
        if (tid < dv) {
            const float zz = to_f32(z[head * dv + tid]);
            y[head * dv + tid] = from_f32<T>(o_c * rsqrtf(mean_sq + eps) * weight[tid] * zz * sigmoid_acc(zz));
        }
        __syncthreads();  // the per-head shared vectors are rewritten by the next value head
    }
}

// One CTA per (batch row, value head); the G CTAs of a key head's group form one cluster (see the top).
template <int DK, typename T>
__global__ void __launch_bounds__(256, 2)
    mixer_step_cluster_kernel(const T* __restrict__ xq, const T* __restrict__ xk, const T* __restrict__ xv,
                              const float* __restrict__ cq, const float* __restrict__ ck, const float* __restrict__ cv,
                              const T* __restrict__ ag, const T* __restrict__ ab, const T* __restrict__ aw,
                              float* __restrict__ sq, float* __restrict__ sk, float* __restrict__ sv,
                              float* __restrict__ state, const T* __restrict__ z, const float* __restrict__ weight,
                              float eps, T* __restrict__ y, int Hk, int Hv, int dv, int neg_eigval, float scale) {
    __shared__ float s_q[DK], s_k[DK], s_a[DK], s_bk[DK];
    __shared__ float s_wv[128], s_o[128];
    __shared__ float s_red[8];
    constexpr int RPL = DK / 8;  // state rows per lane
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hv / Hk;
    const int rank = static_cast<int>(blockIdx.x % G), unit = blockIdx.x / G;
    const int bi = unit / Hk, hk = unit - bi * Hk, hv = hk * G + rank;
    const size_t head = static_cast<size_t>(bi) * Hv + hv;
    const int cg = lane & 3, rg = lane >> 2, col = 16 * warp + 4 * cg;
    const bool upd = 16 * warp < dv;

    // ---- every load first: the state slice, then the per-channel inputs
    float4 s[RPL];
    float* S = state + head * DK * dv + col;
    if (upd) {
#pragma unroll
        for (int i = 0; i < RPL; ++i) s[i] = *reinterpret_cast<const float4*>(S + static_cast<size_t>(rg + 8 * i) * dv);
    }
    const size_t Cqk = static_cast<size_t>(Hk) * DK, chqk = static_cast<size_t>(hk) * DK + tid;
    const size_t Cv = static_cast<size_t>(Hv) * dv, chv = static_cast<size_t>(hv) * dv + tid;
    float xq_c = 0.f, xk_c = 0.f, q3[3] = {0.f, 0.f, 0.f}, k3[3] = {0.f, 0.f, 0.f}, a_c = 0.f, b_c = 0.f;
    float4 wq = make_float4(0.f, 0.f, 0.f, 0.f), wk = wq, wv4 = wq;
    float xv_c = 0.f, v3[3] = {0.f, 0.f, 0.f}, w_c = 0.f, z_c = 0.f, wt_c = 0.f;
    if (tid < DK) {
        const size_t xi = (static_cast<size_t>(bi) * Hk + hk) * DK + tid;
        xq_c = to_f32(xq[xi]);
        xk_c = to_f32(xk[xi]);
        wq = *reinterpret_cast<const float4*>(cq + chqk * kStepTaps);
        wk = *reinterpret_cast<const float4*>(ck + chqk * kStepTaps);
        if (sq) {
            const float* sp = sq + static_cast<size_t>(bi) * (kStepTaps - 1) * Cqk + chqk;
            q3[0] = sp[0]; q3[1] = sp[Cqk]; q3[2] = sp[2 * Cqk];
        }
        if (sk) {
            const float* sp = sk + static_cast<size_t>(bi) * (kStepTaps - 1) * Cqk + chqk;
            k3[0] = sp[0]; k3[1] = sp[Cqk]; k3[2] = sp[2 * Cqk];
        }
        a_c = to_f32(ag[head * DK + tid]);
        b_c = to_f32(ab[head * DK + tid]);
    }
    if (tid < dv) {
        xv_c = to_f32(xv[head * dv + tid]);
        wv4 = *reinterpret_cast<const float4*>(cv + chv * kStepTaps);
        if (sv) {
            const float* sp = sv + static_cast<size_t>(bi) * (kStepTaps - 1) * Cv + chv;
            v3[0] = sp[0]; v3[1] = sp[Cv]; v3[2] = sp[2 * Cv];
        }
        w_c = to_f32(aw[head * dv + tid]);
        z_c = to_f32(z[head * dv + tid]);
        wt_c = weight[tid];
    }

    // ---- q, k: conv, L2 norm; gates; v conv
    const float qv = wq.x * q3[0] + wq.y * q3[1] + wq.z * q3[2] + wq.w * xq_c;
    const float kv = wk.x * k3[0] + wk.y * k3[1] + wk.z * k3[2] + wk.w * xk_c;
    const float nq = rsqrtf(block_sum(tid < DK ? qv * qv : 0.f, s_red) + kStepL2Eps);
    const float nk = rsqrtf(block_sum(tid < DK ? kv * kv : 0.f, s_red) + kStepL2Eps);
    if (tid < DK) {
        s_q[tid] = qv * nq;
        s_k[tid] = kv * nk;
        s_a[tid] = sigmoid_acc(-a_c);  // e^{-softplus(a)}
        s_bk[tid] = sigmoid_acc(b_c) * (neg_eigval ? 2.f : 1.f) * (kv * nk);
    }
    if (tid < dv) {
        const float vv = wv4.x * v3[0] + wv4.y * v3[1] + wv4.z * v3[2] + wv4.w * xv_c;
        s_wv[tid] = sigmoid_acc(w_c) * vv;
        if (sv) {  // this CTA's own value head: its conv state has no other reader
            float* sp = sv + static_cast<size_t>(bi) * (kStepTaps - 1) * Cv + chv;
            sp[0] = v3[1]; sp[Cv] = v3[2]; sp[2 * Cv] = xv_c;
        }
    }
    const float kq = block_sum(tid < DK ? (kv * nk) * (qv * nq) : 0.f, s_red);  // also publishes the vectors
    // every CTA of the group has read the q, k conv states before the first one moves them on
    cooperative_groups::this_cluster().sync();
    if (rank == 0 && tid < DK) {
        if (sq) {
            float* sp = sq + static_cast<size_t>(bi) * (kStepTaps - 1) * Cqk + chqk;
            sp[0] = q3[1]; sp[Cqk] = q3[2]; sp[2 * Cqk] = xq_c;
        }
        if (sk) {
            float* sp = sk + static_cast<size_t>(bi) * (kStepTaps - 1) * Cqk + chqk;
            sp[0] = k3[1]; sp[Cqk] = k3[2]; sp[2 * Cqk] = xk_c;
        }
    }

    // ---- the recurrent update: warp w, columns 16 w .. 16 w + 15
    if (upd) {
        float4 rb = make_float4(0.f, 0.f, 0.f, 0.f), rq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const int r = rg + 8 * i;
            const float a = s_a[r], bk = s_bk[r], qq = s_q[r];
            s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
            rb.x = fmaf(s[i].x, bk, rb.x); rb.y = fmaf(s[i].y, bk, rb.y);
            rb.z = fmaf(s[i].z, bk, rb.z); rb.w = fmaf(s[i].w, bk, rb.w);
            rq.x = fmaf(s[i].x, qq, rq.x); rq.y = fmaf(s[i].y, qq, rq.y);
            rq.z = fmaf(s[i].z, qq, rq.z); rq.w = fmaf(s[i].w, qq, rq.w);
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {  // the 8 row groups: lanes that differ in bits 2..4
            rb.x += __shfl_xor_sync(0xffffffffu, rb.x, off);
            rb.y += __shfl_xor_sync(0xffffffffu, rb.y, off);
            rb.z += __shfl_xor_sync(0xffffffffu, rb.z, off);
            rb.w += __shfl_xor_sync(0xffffffffu, rb.w, off);
            rq.x += __shfl_xor_sync(0xffffffffu, rq.x, off);
            rq.y += __shfl_xor_sync(0xffffffffu, rq.y, off);
            rq.z += __shfl_xor_sync(0xffffffffu, rq.z, off);
            rq.w += __shfl_xor_sync(0xffffffffu, rq.w, off);
        }
        const float4 d = make_float4(s_wv[col] - rb.x, s_wv[col + 1] - rb.y, s_wv[col + 2] - rb.z,
                                     s_wv[col + 3] - rb.w);
        if (rg == 0) {
            s_o[col] = scale * fmaf(kq, d.x, rq.x);
            s_o[col + 1] = scale * fmaf(kq, d.y, rq.y);
            s_o[col + 2] = scale * fmaf(kq, d.z, rq.z);
            s_o[col + 3] = scale * fmaf(kq, d.w, rq.w);
        }
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const float kk = s_k[rg + 8 * i];
            s[i].x = fmaf(kk, d.x, s[i].x); s[i].y = fmaf(kk, d.y, s[i].y);
            s[i].z = fmaf(kk, d.z, s[i].z); s[i].w = fmaf(kk, d.w, s[i].w);
            *reinterpret_cast<float4*>(S + static_cast<size_t>(rg + 8 * i) * dv) = s[i];
        }
    }
    // ---- gated RMSNorm with the SiLU gate over d_v
    __syncthreads();  // s_o complete
    const float o_c = tid < dv ? s_o[tid] : 0.f;
    const float mean_sq = block_sum(o_c * o_c, s_red) / static_cast<float>(dv);
    if (tid < dv) y[head * dv + tid] = from_f32<T>(o_c * rsqrtf(mean_sq + eps) * wt_c * z_c * sigmoid_acc(z_c));
}

// ---- persistent form ---------------------------------------------------------------------------

constexpr uint32_t kStepSmem = 232448;  // largest dynamic shared memory of one CTA

// Ring geometry: a slot is the fp32 state slab [128][128], then the head's token vectors (xq, xk, a_g,
// a_b, xv, a_w; 128 each) and the carried conv rows (q, k, v: 3 x 128 fp32 each).
template <typename T>
struct StepRing {
    static constexpr uint32_t vb = 128 * sizeof(T);
    static constexpr uint32_t slab = 128 * 128 * 4;
    static constexpr uint32_t conv_off = slab + 6 * vb;
    static constexpr uint32_t slot = (conv_off + 9 * 512 + 127) / 128 * 128;
    static constexpr uint32_t part_bytes = 8 * 2 * 128 * 4;  // [8 warps][r_b | r_q][128] fp32
    // per-head vectors q, k, alpha, b.k, w.v, o (fp32 [6][128]), reduction partials [16], the update's
    // cross-warp partials, mbarriers
    static constexpr uint32_t vecs_bytes = 6 * 512 + 16 * 4 + part_bytes;
    static constexpr int depth = (kStepSmem - vecs_bytes - 128) / slot > 4 ? 4 : (kStepSmem - vecs_bytes - 128) / slot;
    static constexpr uint32_t vecs_off = depth * slot;
    static constexpr uint32_t bar_off = vecs_off + vecs_bytes;
    static constexpr uint32_t total = bar_off + 8 * 4 + 16;
};

// Queue the copies of value head h = (batch row) * H_v + (value head) into a slot. Missing conv states
// (null) are not copied and read as zeros.
template <typename T>
__device__ __forceinline__ void step_issue(uint8_t* sl, uint64_t* bar, long long h, const float* state,
                                           const T* xq, const T* xk, const T* ag, const T* ab, const T* xv,
                                           const T* aw, const float* sq, const float* sk, const float* sv, int Hk,
                                           int Hv) {
    using R = StepRing<T>;
    const long long bi = h / Hv;
    const int hv = static_cast<int>(h - bi * Hv), hk = hv / (Hv / Hk);
    const int nconv = (sq ? 3 : 0) + (sk ? 3 : 0) + (sv ? 3 : 0);
    mbar_arrive_expect_tx(bar, R::slab + 6 * R::vb + 512 * nconv);
    bulk_load(sl, state + h * 16384, R::slab, bar);
    const size_t kq = (static_cast<size_t>(bi) * Hk + hk) * 128, vh = static_cast<size_t>(h) * 128;
    bulk_load(sl + R::slab + 0 * R::vb, xq + kq, R::vb, bar);
    bulk_load(sl + R::slab + 1 * R::vb, xk + kq, R::vb, bar);
    bulk_load(sl + R::slab + 2 * R::vb, ag + vh, R::vb, bar);
    bulk_load(sl + R::slab + 3 * R::vb, ab + vh, R::vb, bar);
    bulk_load(sl + R::slab + 4 * R::vb, xv + vh, R::vb, bar);
    bulk_load(sl + R::slab + 5 * R::vb, aw + vh, R::vb, bar);
    const size_t Cqk = static_cast<size_t>(Hk) * 128, Cv = static_cast<size_t>(Hv) * 128;
    uint8_t* cs = sl + R::conv_off;
    for (int j = 0; j < 3; ++j) {
        const size_t rq = (static_cast<size_t>(bi) * 3 + j) * Cqk + static_cast<size_t>(hk) * 128;
        if (sq) bulk_load(cs + (0 + j) * 512, sq + rq, 512, bar);
        if (sk) bulk_load(cs + (3 + j) * 512, sk + rq, 512, bar);
        if (sv) bulk_load(cs + (6 + j) * 512, sv + (static_cast<size_t>(bi) * 3 + j) * Cv + static_cast<size_t>(hv) * 128,
                          512, bar);
    }
}

// One CTA per SM, 256 threads: threads 0-127 take the q/k channels and the gates a_g, a_b; threads
// 128-255 the v channels, a_w, and the gated norm; for the state update warp w holds rows
// 16 w .. 16 w + 15 (conflict-free rows of the slot) and lane l columns 4 l .. 4 l + 3. The updated
// state goes back through its slot by bulk copy, and the slot is refilled once that copy has read it.
template <typename T>
__global__ void __launch_bounds__(256, 1)
    mixer_step_stream_kernel(const T* __restrict__ xq, const T* __restrict__ xk, const T* __restrict__ xv,
                             const float* __restrict__ cq, const float* __restrict__ ck,
                             const float* __restrict__ cv, const T* __restrict__ ag, const T* __restrict__ ab,
                             const T* __restrict__ aw, float* __restrict__ sq, float* __restrict__ sk,
                             float* __restrict__ sv, float* __restrict__ state, const T* __restrict__ z,
                             const float* __restrict__ weight, float eps, T* __restrict__ y, long long units, int Hk,
                             int Hv, int neg_eigval, float scale, long long wait_ns) {
    using R = StepRing<T>;
    constexpr int D = R::depth, P = D > 1 ? D - 1 : 1;
    extern __shared__ __align__(128) uint8_t smem_m[];
    float* s_q = reinterpret_cast<float*>(smem_m + R::vecs_off);
    float* s_k = s_q + 128;
    float* s_a = s_q + 256;
    float* s_bk = s_q + 384;
    float* s_wv = s_q + 512;
    float* s_o = s_q + 640;
    float* s_red = s_q + 768;  // [0..11] q.q, k.k, k.q per q/k warp; [12..15] o.o per v warp
    float* s_part = s_q + 784;   // the update's cross-warp partials
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_m + R::bar_off);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hv / Hk;
    const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    const long long h0 = u0 * G;
    const int count = static_cast<int>((u1 - u0) * G);
    const bool vside = tid >= 128;
    const int c = tid & 127;  // channel of this thread's side
    const float wt_c = vside ? weight[c] : 0.f;

    if (tid == 0) {
        for (int i = 0; i < D; ++i) mbar_init(full + i, 1);
        fence_mbar_init();
        for (int kk = 0; kk < P && kk < count; ++kk)
            step_issue<T>(smem_m + kk * R::slot, full + kk, h0 + kk, state, xq, xk, ag, ab, xv, aw, sq, sk, sv, Hk, Hv);
    }
    __syncthreads();

    // conv weights of the head (L2-resident: every batch row shares them), loaded one head ahead
    auto conv_w = [&](long long h) {
        const int hv = static_cast<int>(h % Hv);
        return vside ? *reinterpret_cast<const float4*>(cv + (static_cast<size_t>(hv) * 128 + c) * kStepTaps)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto conv_wq = [&](long long h, const float* wsrc) {
        const int hk = static_cast<int>(h % Hv) / G;
        return vside ? make_float4(0.f, 0.f, 0.f, 0.f)
                     : *reinterpret_cast<const float4*>(wsrc + (static_cast<size_t>(hk) * 128 + c) * kStepTaps);
    };
    float4 wv_n = make_float4(0.f, 0.f, 0.f, 0.f), wq_n = wv_n, wk_n = wv_n;
    float z_n = 0.f;  // the output gate of this thread's channel, one head ahead
    if (count > 0) {
        wv_n = conv_w(h0);
        wq_n = conv_wq(h0, cq);
        wk_n = conv_wq(h0, ck);
        if (vside) z_n = to_f32(z[static_cast<size_t>(h0) * 128 + c]);
    }

    int kk = 0;
    bool ok = true;
    for (; kk < count; ++kk) {
        const long long h = h0 + kk;
        const int bsel = kk % D;
        const uint32_t par = (kk / D) & 1;
        const long long bi = h / Hv;
        const int hv = static_cast<int>(h - bi * Hv), hk = hv / G, rank = hv - hk * G;
        const float4 wv4 = wv_n, wq = wq_n, wk = wk_n;
        const float z_c = z_n;
        if (kk + 1 < count) {
            wv_n = conv_w(h + 1);
            wq_n = conv_wq(h + 1, cq);
            wk_n = conv_wq(h + 1, ck);
            if (vside) z_n = to_f32(z[static_cast<size_t>(h + 1) * 128 + c]);
        }
        {  // every thread observes the slot's phase itself; one block vote decides
            const bool got = mbar_wait(full + bsel, par, wait_ns);
            if (!got) {
                atomicOr(&g_status_step, kStatusTimeout);
                mbar_wait(full + bsel, par, kDefaultWaitNs);
            }
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
        }
        uint8_t* sl = smem_m + bsel * R::slot;
        const T* V = reinterpret_cast<const T*>(sl + R::slab);
        const float* CS = reinterpret_cast<const float*>(sl + R::conv_off);

        // ---- prologue: conv of this side's channel; the partial sums of the two L2 norms and of k.q
        float xq_c = 0.f, xk_c = 0.f, q3[3] = {0.f, 0.f, 0.f}, k3[3] = {0.f, 0.f, 0.f}, qv = 0.f, kv = 0.f;
        float xv_c = 0.f, v3[3] = {0.f, 0.f, 0.f};
        if (!vside) {
            xq_c = to_f32(V[c]);
            xk_c = to_f32(V[128 + c]);
            if (sq) { q3[0] = CS[c]; q3[1] = CS[128 + c]; q3[2] = CS[256 + c]; }
            if (sk) { k3[0] = CS[384 + c]; k3[1] = CS[512 + c]; k3[2] = CS[640 + c]; }
            qv = wq.x * q3[0] + wq.y * q3[1] + wq.z * q3[2] + wq.w * xq_c;
            kv = wk.x * k3[0] + wk.y * k3[1] + wk.z * k3[2] + wk.w * xk_c;
            float a = qv * qv, b = kv * kv, e = kv * qv;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                b += __shfl_xor_sync(0xffffffffu, b, off);
                e += __shfl_xor_sync(0xffffffffu, e, off);
            }
            if (lane == 0) {
                s_red[3 * warp] = a;
                s_red[3 * warp + 1] = b;
                s_red[3 * warp + 2] = e;
            }
            // the raw conv outputs; the L2 norms are applied to the reductions over d_k below
            s_q[c] = qv;
            s_k[c] = kv;
            s_a[c] = sigmoid_acc(-to_f32(V[256 + c]));  // e^{-softplus(a)}
            s_bk[c] = sigmoid_acc(to_f32(V[384 + c])) * (neg_eigval ? 2.f : 1.f) * kv;
            if (rank == G - 1) {  // the key head's last value head: every sibling has its copy of the old states
                const size_t Cqk = static_cast<size_t>(Hk) * 128;
                const size_t base = static_cast<size_t>(bi) * (kStepTaps - 1) * Cqk + static_cast<size_t>(hk) * 128 + c;
                if (sq) { sq[base] = q3[1]; sq[base + Cqk] = q3[2]; sq[base + 2 * Cqk] = xq_c; }
                if (sk) { sk[base] = k3[1]; sk[base + Cqk] = k3[2]; sk[base + 2 * Cqk] = xk_c; }
            }
        } else {
            xv_c = to_f32(V[4 * 128 + c]);
            if (sv) { v3[0] = CS[768 + c]; v3[1] = CS[896 + c]; v3[2] = CS[1024 + c]; }
            const float vv = wv4.x * v3[0] + wv4.y * v3[1] + wv4.z * v3[2] + wv4.w * xv_c;
            s_wv[c] = sigmoid_acc(to_f32(V[5 * 128 + c])) * vv;
            if (sv) {  // this value head's own conv state: no other head reads it
                float* sp = sv + static_cast<size_t>(bi) * (kStepTaps - 1) * Hv * 128 + static_cast<size_t>(hv) * 128 + c;
                const size_t Cv = static_cast<size_t>(Hv) * 128;
                sp[0] = v3[1]; sp[Cv] = v3[2]; sp[2 * Cv] = xv_c;
            }
        }
        __syncthreads();
        const float qq = (s_red[0] + s_red[3]) + (s_red[6] + s_red[9]);
        const float kk2 = (s_red[1] + s_red[4]) + (s_red[7] + s_red[10]);
        const float kqr = (s_red[2] + s_red[5]) + (s_red[8] + s_red[11]);
        const float nq = rsqrtf(qq + kStepL2Eps), nk = rsqrtf(kk2 + kStepL2Eps);
        const float kq = (kqr * nk) * nq;

        // ---- the recurrent update: warp w, rows 16 w .. 16 w + 15; lane l, columns 4 l .. 4 l + 3. The
        // reductions over d_k go in-thread, then across the warps through a shared buffer.
        {
            float* red = s_part;  // [8][r_b | r_q][128]
            float* S = reinterpret_cast<float*>(sl) + 4 * lane;
            float4 st[16];
            float4 rb = make_float4(0.f, 0.f, 0.f, 0.f), rq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // rows 16 w + 4 j .. + 3: their scalars as one broadcast float4 each
                const int r0 = 16 * warp + 4 * j;
                const float4 a4 = *reinterpret_cast<const float4*>(s_a + r0);
                const float4 b4 = *reinterpret_cast<const float4*>(s_bk + r0);
                const float4 q4 = *reinterpret_cast<const float4*>(s_q + r0);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
                const float qv4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float4 t = *reinterpret_cast<const float4*>(S + (r0 + e) * 128);
                    const float a = av[e], bk = bv[e], qr = qv4[e];
                    t.x *= a; t.y *= a; t.z *= a; t.w *= a;
                    rb.x = fmaf(t.x, bk, rb.x); rb.y = fmaf(t.y, bk, rb.y); rb.z = fmaf(t.z, bk, rb.z); rb.w = fmaf(t.w, bk, rb.w);
                    rq.x = fmaf(t.x, qr, rq.x); rq.y = fmaf(t.y, qr, rq.y); rq.z = fmaf(t.z, qr, rq.z); rq.w = fmaf(t.w, qr, rq.w);
                    st[4 * j + e] = t;
                }
            }
            reinterpret_cast<float4*>(red + (2 * warp) * 128)[lane] = rb;
            reinterpret_cast<float4*>(red + (2 * warp + 1) * 128)[lane] = rq;
            __syncthreads();
            rb = make_float4(0.f, 0.f, 0.f, 0.f);
            rq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) {
                const float4 x = reinterpret_cast<const float4*>(red + (2 * w8) * 128)[lane];
                const float4 y4 = reinterpret_cast<const float4*>(red + (2 * w8 + 1) * 128)[lane];
                rb.x += x.x; rb.y += x.y; rb.z += x.z; rb.w += x.w;
                rq.x += y4.x; rq.y += y4.y; rq.z += y4.z; rq.w += y4.w;
            }
            // r_b = |k|^-1 S'^T (b . raw k), r_q = |q|^-1 S'^T raw q; the update adds raw k (|k|^-1 d)^T
            const float4 wv4c = *reinterpret_cast<const float4*>(s_wv + 4 * lane);
            const float4 d = make_float4(fmaf(-nk, rb.x, wv4c.x), fmaf(-nk, rb.y, wv4c.y), fmaf(-nk, rb.z, wv4c.z),
                                         fmaf(-nk, rb.w, wv4c.w));
            if (warp == 0)
                *reinterpret_cast<float4*>(s_o + 4 * lane) =
                    make_float4(scale * fmaf(kq, d.x, nq * rq.x), scale * fmaf(kq, d.y, nq * rq.y),
                                scale * fmaf(kq, d.z, nq * rq.z), scale * fmaf(kq, d.w, nq * rq.w));
            const float4 dn = make_float4(nk * d.x, nk * d.y, nk * d.z, nk * d.w);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r0 = 16 * warp + 4 * j;
                const float4 k4 = *reinterpret_cast<const float4*>(s_k + r0);
                const float kv4[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float4 t = st[4 * j + e];
                    const float kr = kv4[e];
                    t.x = fmaf(kr, dn.x, t.x); t.y = fmaf(kr, dn.y, t.y); t.z = fmaf(kr, dn.z, t.z); t.w = fmaf(kr, dn.w, t.w);
                    *reinterpret_cast<float4*>(S + (r0 + e) * 128) = t;
                }
            }
        }
        fence_proxy_async_smem();  // the slot's new state is read by the bulk copy below
        __syncthreads();           // o complete
        if (tid == 0) {
            bulk_store(state + h * 16384, sl, R::slab);
            bulk_commit();
            if (kk + P < count) {
                if (D > 1) bulk_wait_read<1>();  // the store of head kk-1 has read the slot it leaves
                else bulk_wait_read<0>();        // single slot: the store of head kk has read it
                const int nb = (kk + P) % D;
                step_issue<T>(smem_m + nb * R::slot, full + nb, h + P, state, xq, xk, ag, ab, xv, aw, sq, sk, sv, Hk,
                              Hv);
            }
        }
        // ---- gated RMSNorm with the SiLU gate over d_v (the v side's four warps)
        if (vside) {
            const float o_c = s_o[c];
            float e = o_c * o_c;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
            if (lane == 0) s_red[12 + warp - 4] = e;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const float ms = ((s_red[12] + s_red[13]) + (s_red[14] + s_red[15])) / 128.f;
            y[static_cast<size_t>(h) * 128 + c] = from_f32<T>(o_c * rsqrtf(ms + eps) * wt_c * z_c * sigmoid_acc(z_c));
        }
    }
    if (tid == 0) {
        if (!ok)  // drain the copies already issued for heads after kk
            for (int j = kk + 1; j < kk + P && j < count; ++j) mbar_wait(full + j % D, (j / D) & 1, kDefaultWaitNs);
        bulk_wait_all();
    }
    __syncthreads();
}

template <int DK, typename T>
cudaError_t launch_step(const void* xq, const void* xk, const void* xv, const float* cq, const float* ck,
                        const float* cv, const void* ag, const void* ab, const void* aw, float* sq, float* sk,
                        float* sv, float* state, const void* z, const float* weight, float eps, void* y, int B,
                        int Hk, int Hv, int dv, int neg_eigval, float scale, cudaStream_t s) {
    const int G = Hv / Hk;
    if (g_step_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&g_step_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            g_step_sms = 1;
    }
    if (DK == 128 && dv == 128 && static_cast<long long>(B) * Hv >= 4LL * g_step_sms) {
        using R = StepRing<T>;
        cudaError_t e = cudaFuncSetAttribute(mixer_step_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)R::total);
        if (e != cudaSuccess) return e;
        const long long units = static_cast<long long>(B) * Hk;
        const int grid = units < g_step_sms ? static_cast<int>(units) : g_step_sms;
        mixer_step_stream_kernel<T><<<grid, 256, R::total, s>>>(
            static_cast<const T*>(xq), static_cast<const T*>(xk), static_cast<const T*>(xv), cq, ck, cv,
            static_cast<const T*>(ag), static_cast<const T*>(ab), static_cast<const T*>(aw), sq, sk, sv, state,
            static_cast<const T*>(z), weight, eps, static_cast<T*>(y), units, Hk, Hv, neg_eigval, scale,
            wait_limit_ns());
        return cudaGetLastError();
    }
    if (G <= kMaxClusterGroup) {  // one CTA per value head, clusters of the key head's group
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(B) * Hv);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(G);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, mixer_step_cluster_kernel<DK, T>, static_cast<const T*>(xq),
                                  static_cast<const T*>(xk), static_cast<const T*>(xv), cq, ck, cv,
                                  static_cast<const T*>(ag), static_cast<const T*>(ab), static_cast<const T*>(aw),
                                  sq, sk, sv, state, static_cast<const T*>(z), weight, eps, static_cast<T*>(y), Hk,
                                  Hv, dv, neg_eigval, scale);
    }
    mixer_step_kernel<DK, T><<<static_cast<unsigned>(B) * Hk, 256, 0, s>>>(
        static_cast<const T*>(xq), static_cast<const T*>(xk), static_cast<const T*>(xv), cq, ck, cv,
        static_cast<const T*>(ag), static_cast<const T*>(ab), static_cast<const T*>(aw), sq, sk, sv, state,
        static_cast<const T*>(z), weight, eps, static_cast<T*>(y), Hk, Hv, dv, neg_eigval, scale);
    return cudaGetLastError();
}

}  // namespace

int step_read_clear_status(cudaStream_t s) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_step, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (v && cudaMemcpyToSymbolAsync(g_status_step, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    cudaStreamSynchronize(s);
    return v;
}

}  // namespace gdn2

using namespace gdn2;

extern "C" gdn2_status gdn2_mixer_decode_step(const void* xq, const void* xk, const void* xv, const float* conv_q,
                                              const float* conv_k, const float* conv_v, const void* ag,
                                              const void* ab, const void* aw, float* state_q, float* state_k,
                                              float* state_v, float* state, const void* z, const float* weight,
                                              float eps, void* y, int B, int Hk, int Hv, int dk, int dv,
                                              int neg_eigval, float scale, gdn2_dtype dt, void* stream) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || B < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk ||
        !(eps >= 0.f))
        return GDN2_ERR_INVALID_ARG;
    if (!(dk == 64 || dk == 128) || !(dv == 64 || dv == 128)) return GDN2_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hk >= (1LL << 31) || static_cast<long long>(B) * Hv * dk * dv >= (1LL << 46))
        return GDN2_ERR_UNSUPPORTED;
    if (B == 0) return GDN2_OK;
    const void* need[] = {xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state, z, weight, y};
    for (const void* p : need) {
        if (!p) return GDN2_ERR_INVALID_ARG;
        if (!aligned16(p)) return GDN2_ERR_MISALIGNED;
    }
    if ((state_q && !aligned16(state_q)) || (state_k && !aligned16(state_k)) || (state_v && !aligned16(state_v)))
        return GDN2_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dt == GDN2_BF16)
        e = dk == 128 ? launch_step<128, __nv_bfloat16>(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state_q,
                                                         state_k, state_v, state, z, weight, eps, y, B, Hk, Hv, dv,
                                                         neg_eigval, scale, s)
                      : launch_step<64, __nv_bfloat16>(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state_q,
                                                        state_k, state_v, state, z, weight, eps, y, B, Hk, Hv, dv,
                                                        neg_eigval, scale, s);
    else
        e = dk == 128 ? launch_step<128, float>(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state_q, state_k,
                                                 state_v, state, z, weight, eps, y, B, Hk, Hv, dv, neg_eigval, scale,
                                                 s)
                      : launch_step<64, float>(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state_q, state_k,
                                                state_v, state, z, weight, eps, y, B, Hk, Hv, dv, neg_eigval, scale,
                                                s);
    return e == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

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
#include <cooperative_groups.h>

#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kStepTaps = 4;
constexpr float kStepL2Eps = 1e-6f;
constexpr int kMaxClusterGroup = 8;  // portable cluster size

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

template <int DK, typename T>
cudaError_t launch_step(const void* xq, const void* xk, const void* xv, const float* cq, const float* ck,
                        const float* cv, const void* ag, const void* ab, const void* aw, float* sq, float* sk,
                        float* sv, float* state, const void* z, const float* weight, float eps, void* y, int B,
                        int Hk, int Hv, int dv, int neg_eigval, float scale, cudaStream_t s) {
    const int G = Hv / Hk;
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

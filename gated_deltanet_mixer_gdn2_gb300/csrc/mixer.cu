// mixer.cu -- the token-mixer operations around the GDN-2 core, fused into one pass over the tensors
// each reads: the prologue (ShortConv on q, k, v; L2 norm of q and k; gate activations) and the
// epilogue (gated RMSNorm with a SiLU gate).
//
// Sources: the burn-gdn2 0.1.5 docs ("Architecture": projections -> ShortConv -> L2-Norm -> core ->
// Gated RMS Norm <- SiLU Gate; configuration: depthwise conv before the recurrence, b x 2 for
// negative eigenvalues, norm_eps 1e-5) and the llama.cpp GDN decode study (conv kernel 4; the conv
// state keeps the previous 3 samples). Where they are silent:
//   ShortConv: depthwise causal, kernel 4, on q, k and v, no bias or activation:
//       y_t[c] = sum_j W[c][j] x_{t-3+j}[c], samples before the call taken from the carried state;
//   L2 norm: x / sqrt(sum x^2 + 1e-6) per (token, head);
//   gates: g = -softplus(a_g), b = sigmoid(a_b) (x 2 with negative eigenvalues), w = sigmoid(a_w);
//   epilogue: y = o / sqrt(mean(o^2) + eps) * weight * silu(z), per (token, value head).
// All of it is memory-bound: every element is read once and written once, in 16-byte vectors.
#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kTaps = 4;
constexpr int kTokBlock = 32;  // tokens walked by one lane group (the conv window stays in registers)
constexpr float kL2Eps = 1e-6f;

struct ConvJob {
    const void* x;
    const float* wt;     // [H * d][4]
    const float* state;  // [B][3][H * d] or null
    void* y;
    int H, d, l2;
};

struct PrologueArgs {
    ConvJob job[3];  // q, k, v
    const void* a[3];  // gate pre-activations g, b, w
    void* out[3];
    long long n8[3];   // 8-element vectors per gate tensor
    int B, T, neg_eigval;
};

__device__ __forceinline__ float sigmoid_f(float a) { return 1.f / (1.f + expf(-a)); }
__device__ __forceinline__ float softplus_f(float a) { return log1pf(expf(-fabsf(a))) + fmaxf(a, 0.f); }

// blockIdx.y = 0..2: conv job (q, k, v). A conv lane group of d/8 lanes owns one
// (batch row, head, block of kTokBlock tokens) at a time and walks its tokens with the 3 previous
// samples of its 8 channels in registers; the grid strides over the groups (a warp's groups move
// together, so the shuffles of the L2 norm always see the whole warp).
template <typename T>
__global__ void __launch_bounds__(256) prologue_kernel(const __grid_constant__ PrologueArgs args) {
    const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    {
        const ConvJob& jb = args.job[blockIdx.y];
        const int G = jb.d / 8;  // lanes per head (2..32, a power of two)
        const int nblk = (args.T + kTokBlock - 1) / kTokBlock;
        const long long groups = static_cast<long long>(args.B) * jb.H * nblk;
        const int lane = static_cast<int>(tid % G);
        const int C = jb.H * jb.d;
        const T* x = static_cast<const T*>(jb.x);
        T* y = static_cast<T*>(jb.y);
        for (long long grp = tid / G; grp - (threadIdx.x & 31) / G < groups; grp += nthreads / G) {
            const bool active = grp < groups;
            const long long gg = active ? grp : 0;
            const int blk = static_cast<int>(gg % nblk);
            const long long bh = gg / nblk;
            const int h = static_cast<int>(bh % jb.H);
            const int bi = static_cast<int>(bh / jb.H);
            const int c0 = h * jb.d + 8 * lane;
            float w[8][kTaps];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 t4 = *reinterpret_cast<const float4*>(jb.wt + (c0 + e) * kTaps);
                w[e][0] = t4.x; w[e][1] = t4.y; w[e][2] = t4.z; w[e][3] = t4.w;
            }
            const int t0 = blk * kTokBlock, t1 = min(t0 + kTokBlock, args.T);
            float prev[kTaps - 1][8];
#pragma unroll
            for (int j = 0; j < kTaps - 1; ++j) {
                const int t = t0 - (kTaps - 1) + j;
                if (t >= 0) {
                    Vec8<T>::load_ro(x + (static_cast<size_t>(bi) * args.T + t) * C + c0, prev[j]);
                } else if (jb.state) {
                    const float* sp = jb.state + (static_cast<size_t>(bi) * (kTaps - 1) + (kTaps - 1 + t)) * C + c0;
                    const float4 a = reinterpret_cast<const float4*>(sp)[0], b = reinterpret_cast<const float4*>(sp)[1];
                    prev[j][0] = a.x; prev[j][1] = a.y; prev[j][2] = a.z; prev[j][3] = a.w;
                    prev[j][4] = b.x; prev[j][5] = b.y; prev[j][6] = b.z; prev[j][7] = b.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) prev[j][e] = 0.f;
                }
            }
            const int n = active ? t1 - t0 : 0;
            const int trips = __reduce_max_sync(0xffffffffu, n);
#pragma unroll 4
            for (int i = 0; i < trips; ++i) {
                const int t = t0 + i;
                float cur[8], out[8];
                if (i < n) Vec8<T>::load_ro(x + (static_cast<size_t>(bi) * args.T + t) * C + c0, cur);
                else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) cur[e] = 0.f;
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    out[e] = w[e][0] * prev[0][e] + w[e][1] * prev[1][e] + w[e][2] * prev[2][e] + w[e][3] * cur[e];
                    ss += out[e] * out[e];
                    prev[0][e] = prev[1][e];
                    prev[1][e] = prev[2][e];
                    prev[2][e] = cur[e];
                }
                if (jb.l2) {
                    for (int off = 1; off < G; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                    const float r = rsqrtf(ss + kL2Eps);
#pragma unroll
                    for (int e = 0; e < 8; ++e) out[e] *= r;
                }
                if (i < n) Vec8<T>::store(y + (static_cast<size_t>(bi) * args.T + t) * C + c0, out);
            }
        }
    }
}

// gates: g = -softplus, b = sigmoid (x 2), w = sigmoid; blockIdx.y selects the tensor
template <typename T>
__global__ void __launch_bounds__(256) gates_kernel(const __grid_constant__ PrologueArgs args) {
    const int gi = blockIdx.y;
    const long long n8 = args.n8[gi];
    const T* src = static_cast<const T*>(args.a[gi]);
    T* dst = static_cast<T*>(args.out[gi]);
    const float mul = (gi == 1 && args.neg_eigval) ? 2.f : 1.f;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8; i += nthreads) {
        float a[8];
        Vec8<T>::load_ro(src + 8 * i, a);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = gi == 0 ? -softplus_f(a[e]) : sigmoid_f(a[e]) * mul;
        Vec8<T>::store(dst + 8 * i, a);
    }
}

// New conv state: the last 3 samples of [old state, x_0 .. x_{T-1}], one thread per channel.
template <typename Tx>
__global__ void __launch_bounds__(256) conv_state_kernel(const void* x, float* state, int B, int T, int C) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i >= static_cast<long long>(B) * C) return;
    const int bi = static_cast<int>(i / C), c = static_cast<int>(i % C);
    float* sp = state + static_cast<size_t>(bi) * (kTaps - 1) * C + c;
    float nw[kTaps - 1];
#pragma unroll
    for (int j = 0; j < kTaps - 1; ++j) {
        const int e = T + j;  // index into [old(3), x(T)]
        nw[j] = e < kTaps - 1 ? sp[e * C]
                              : to_f32(static_cast<const Tx*>(x)[(static_cast<size_t>(bi) * T + e - (kTaps - 1)) * C + c]);
    }
#pragma unroll
    for (int j = 0; j < kTaps - 1; ++j) sp[j * C] = nw[j];
}

// A lane group of d_v/8 lanes per (row, value head); the grid strides over the rows, a warp's
// groups together (the shuffles of the mean square see the whole warp).
template <typename T>
__global__ void __launch_bounds__(256) epilogue_kernel(const T* __restrict__ o, const T* __restrict__ z,
                                                      const float* __restrict__ weight, float eps, T* __restrict__ y,
                                                      long long rows, int dv) {
    const int G = dv / 8;
    const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x / G;
    const int lane = threadIdx.x % G;
    const float4 w0 = reinterpret_cast<const float4*>(weight + 8 * lane)[0];
    const float4 w1 = reinterpret_cast<const float4*>(weight + 8 * lane)[1];
    const float wt[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    for (long long r = tid / G; r - (threadIdx.x & 31) / G < rows; r += stride) {
        const bool active = r < rows;
        const size_t base = static_cast<size_t>(active ? r : 0) * dv + 8 * lane;
        float a[8], zz[8];
        Vec8<T>::load(o + base, a);   // y may alias o: plain loads
        Vec8<T>::load(z + base, zz);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += a[e] * a[e];
        for (int off = 1; off < G; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / dv + eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = a[e] * inv * wt[e] * (zz[e] * sigmoid_f(zz[e]));
        if (active) Vec8<T>::store(y + base, a);
    }
}

int persistent_blocks(long long lanes) {
    const long long want = (lanes + 255) / 256;
    return static_cast<int>(want < 152 * 32 ? (want < 1 ? 1 : want) : 152 * 32);
}

bool head_dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }

}  // namespace
}  // namespace gdn2

using namespace gdn2;

extern "C" {

gdn2_status gdn2_mixer_prologue(const void* xq, const void* xk, const void* xv, const float* conv_q,
                                const float* conv_k, const float* conv_v, const void* ag, const void* ab,
                                const void* aw, float* state_q, float* state_k, float* state_v, void* q, void* k,
                                void* v, void* g, void* b, void* w, int B, int T, int Hk, int Hv, int dk, int dv,
                                int neg_eigval, gdn2_dtype dt, void* stream) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 ||
        Hv % Hk)
        return GDN2_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDN2_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * T;
    if (rows * Hv * (dk > dv ? dk : dv) >= (1LL << 40) || static_cast<long long>(B) * Hv * dv * 3 >= (1LL << 40))
        return GDN2_ERR_UNSUPPORTED;
    if (rows == 0) return GDN2_OK;  // nothing to read; conv states unchanged
    const void* ptrs[] = {xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, q, k, v, g, b, w};
    for (const void* p : ptrs)
        if (!p) return GDN2_ERR_INVALID_ARG;
    for (const void* p : ptrs)
        if (!aligned16(p)) return GDN2_ERR_MISALIGNED;
    if ((state_q && !aligned16(state_q)) || (state_k && !aligned16(state_k)) || (state_v && !aligned16(state_v)))
        return GDN2_ERR_MISALIGNED;
    PrologueArgs a;
    a.job[0] = ConvJob{xq, conv_q, state_q, q, Hk, dk, 1};
    a.job[1] = ConvJob{xk, conv_k, state_k, k, Hk, dk, 1};
    a.job[2] = ConvJob{xv, conv_v, state_v, v, Hv, dv, 0};
    a.a[0] = ag; a.a[1] = ab; a.a[2] = aw;
    a.out[0] = g; a.out[1] = b; a.out[2] = w;
    a.n8[0] = a.n8[1] = rows * Hv * dk / 8;
    a.n8[2] = rows * Hv * dv / 8;
    a.B = B; a.T = T; a.neg_eigval = neg_eigval ? 1 : 0;
    const int nblk = static_cast<int>((T + kTokBlock - 1) / kTokBlock);
    long long lanes = 0;
    for (int j = 0; j < 3; ++j) {
        const long long l = static_cast<long long>(B) * a.job[j].H * nblk * (a.job[j].d / 8);
        lanes = l > lanes ? l : lanes;
    }
    // conv: one lane per 8 channels of a (row, head, token block), striding over the groups;
    // gates: one thread per 8 elements, striding
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(persistent_blocks(lanes), 3);
    const long long gate_n8 = a.n8[0] > a.n8[2] ? a.n8[0] : a.n8[2];
    const dim3 ggrid(static_cast<unsigned>(gate_n8 / 256 + 1 < 4096 ? gate_n8 / 256 + 1 : 4096), 3);
    if (dt == GDN2_BF16) {
        prologue_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
        gates_kernel<__nv_bfloat16><<<ggrid, 256, 0, s>>>(a);
    } else {
        prologue_kernel<float><<<grid, 256, 0, s>>>(a);
        gates_kernel<float><<<ggrid, 256, 0, s>>>(a);
    }
    if (cudaGetLastError() != cudaSuccess) return GDN2_ERR_CUDA;
    // the new conv states, after every read of the old ones
    float* states[3] = {state_q, state_k, state_v};
    const void* xs[3] = {xq, xk, xv};
    const int chans[3] = {Hk * dk, Hk * dk, Hv * dv};
    for (int j = 0; j < 3; ++j) {
        if (!states[j]) continue;
        const long long n = static_cast<long long>(B) * chans[j];
        const int gx = static_cast<int>((n + 255) / 256);
        if (dt == GDN2_BF16) conv_state_kernel<__nv_bfloat16><<<gx, 256, 0, s>>>(xs[j], states[j], B, T, chans[j]);
        else conv_state_kernel<float><<<gx, 256, 0, s>>>(xs[j], states[j], B, T, chans[j]);
        if (cudaGetLastError() != cudaSuccess) return GDN2_ERR_CUDA;
    }
    return GDN2_OK;
}

gdn2_status gdn2_mixer_epilogue(const void* o, const void* z, const float* weight, float eps, void* y, int B, int T,
                                int Hv, int dv, gdn2_dtype dt, void* stream) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || B < 0 || T < 0 || Hv <= 0 || dv <= 0 || !(eps >= 0.f))
        return GDN2_ERR_INVALID_ARG;
    if (!head_dim_ok(dv)) return GDN2_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * T * Hv;
    if (rows * dv >= (1LL << 40)) return GDN2_ERR_UNSUPPORTED;
    if (rows == 0) return GDN2_OK;
    if (!o || !z || !weight || !y) return GDN2_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(z) || !aligned16(weight) || !aligned16(y)) return GDN2_ERR_MISALIGNED;
    const int grid = persistent_blocks(rows * (dv / 8));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == GDN2_BF16)
        epilogue_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o),
                                                            static_cast<const __nv_bfloat16*>(z), weight, eps,
                                                            static_cast<__nv_bfloat16*>(y), rows, dv);
    else
        epilogue_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(o), static_cast<const float*>(z), weight,
                                                    eps, static_cast<float*>(y), rows, dv);
    return cudaGetLastError() == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

}  // extern "C"

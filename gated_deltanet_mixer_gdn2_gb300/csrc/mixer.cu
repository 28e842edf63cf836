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
// All of it is memory-bound: every element is read once and written once. The conv stages each
// (head, 128-token) tile in shared memory with asynchronous copies; the gates stream 16-byte vectors.
#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kTaps = 4;
constexpr int kConvTile = 128;  // tokens per conv tile (one CTA)
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

// The gate activations run at memory speed only with the hardware exponential and logarithm: the
// error of __expf / __logf / __fdividef (a few ulp at these arguments; 1 + e^{-a} stays below 2^116)
// stays far below the bf16 step of the outputs. log(1 + y) for y < 2^-10 is the series y - y^2/2 (next term y^3/3, below 2^-21 relative).
__device__ __forceinline__ float sigmoid_f(float a) { return __fdividef(1.f, 1.f + __expf(fminf(-a, 80.f))); }
__device__ __forceinline__ float softplus_f(float a) {
    const float y = __expf(-fabsf(a));
    return (y < 0x1p-10f ? y * (1.f - 0.5f * y) : __logf(1.f + y)) + fmaxf(a, 0.f);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// N consecutive elements (N = 4 or 8) <-> fp32, in 8-, 16- or 32-byte accesses
template <typename T, int N>
__device__ __forceinline__ void ld_vec(const T* p, float (&x)[N]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 f = reinterpret_cast<const float4*>(p)[i];
            x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
        }
    } else if constexpr (N == 8) {
        Vec8<T>::load(p, x);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    }
}
template <typename T, int N>
__device__ __forceinline__ void st_vec(T* p, const float (&x)[N]) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i)
            reinterpret_cast<float4*>(p)[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    } else if constexpr (N == 8) {
        Vec8<T>::store(p, x);
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = u;
    }
}

// ShortConv (+ L2 norm) on one tile: CTA = (job, batch row, head, kConvTile tokens). The tile and the
// 3 samples before it are copied to shared memory with asynchronous 16-byte copies (so the loads in
// flight cost no registers), then a lane group of d/N lanes (N channels per lane; one row per
// group) walks kConvTile / (256 / group) consecutive tokens with the window in registers. Samples
// before the first token come from the carried fp32 state (or are 0). tiles[j] = tiles of job j.
template <typename T, int N>
__global__ void __launch_bounds__(256) conv_tile_kernel(const __grid_constant__ PrologueArgs args, long long tiles0,
                                                        long long tiles1) {
    extern __shared__ __align__(16) uint8_t smem[];
    const long long tile = blockIdx.x;
    const int job = tile < tiles0 ? 0 : (tile < tiles0 + tiles1 ? 1 : 2);
    const long long tj = tile - (job == 0 ? 0 : (job == 1 ? tiles0 : tiles0 + tiles1));
    const ConvJob& jb = args.job[job];
    const int d = jb.d, C = jb.H * d, Tn = args.T;
    const int nblk = (Tn + kConvTile - 1) / kConvTile;
    const int blk = static_cast<int>(tj % nblk);
    const long long bh = tj / nblk;
    const int h = static_cast<int>(bh % jb.H), bi = static_cast<int>(bh / jb.H);
    const int t0 = blk * kConvTile;
    const T* x = static_cast<const T*>(jb.x) + static_cast<size_t>(bi) * Tn * C + h * d;
    T* y = static_cast<T*>(jb.y) + static_cast<size_t>(bi) * Tn * C + h * d;
    T* tl = reinterpret_cast<T*>(smem);  // row r = token t0 - 3 + r, d elements
    {
        const int cpr = d * static_cast<int>(sizeof(T)) / 16;  // 16-byte pieces per row
        for (int p = threadIdx.x; p < (kConvTile + 3) * cpr; p += 256) {
            const int r = p / cpr, c = p - r * cpr;
            const int t = t0 - 3 + r;
            if (t >= 0 && t < Tn) cp_async16(tl + r * d + c * (16 / sizeof(T)), x + static_cast<size_t>(t) * C + c * (16 / sizeof(T)));
        }
        cp_async_wait_all();
        __syncthreads();
    }
    const int G = d / N;  // lanes per row (a power of two, <= 32)
    const int lane = threadIdx.x & (G - 1), tg = threadIdx.x / G;
    const int tpt = kConvTile * G / 256;  // tokens per lane group
    const int c0 = N * lane;
    float w[N][kTaps];
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const float4 t4 = *reinterpret_cast<const float4*>(jb.wt + (h * d + c0 + e) * kTaps);
        w[e][0] = t4.x; w[e][1] = t4.y; w[e][2] = t4.z; w[e][3] = t4.w;
    }
    const int r0 = 3 + tg * tpt;  // tile row of the group's first token
    float prev[kTaps - 1][N];
#pragma unroll
    for (int j = 0; j < kTaps - 1; ++j) {
        const int t = t0 + r0 - 3 - 3 + j;  // token of window slot j
        if (t >= 0) {
            ld_vec<T, N>(tl + (r0 - 3 + j) * d + c0, prev[j]);
        } else if (jb.state) {
            const float* sp = jb.state + (static_cast<size_t>(bi) * (kTaps - 1) + (kTaps - 1 + t)) * C + h * d + c0;
            ld_vec<float, N>(sp, prev[j]);
        } else {
#pragma unroll
            for (int e = 0; e < N; ++e) prev[j][e] = 0.f;
        }
    }
#pragma unroll 2
    for (int i = 0; i < tpt; ++i) {
        const int t = t0 + r0 - 3 + i;
        float cur[N], out[N];
        ld_vec<T, N>(tl + (r0 + i) * d + c0, cur);  // rows past T hold stale data: never stored
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < N; ++e) {
            out[e] = w[e][0] * prev[0][e] + w[e][1] * prev[1][e] + w[e][2] * prev[2][e] + w[e][3] * cur[e];
            ss += out[e] * out[e];
            prev[0][e] = prev[1][e];
            prev[1][e] = prev[2][e];
            prev[2][e] = cur[e];
        }
        if (jb.l2) {
            for (int off = 1; off < G; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float rn = rsqrtf(ss + kL2Eps);
#pragma unroll
            for (int e = 0; e < N; ++e) out[e] *= rn;
        }
        if (t < Tn) st_vec<T, N>(y + static_cast<size_t>(t) * C + c0, out);
    }
}

// gates: g = -softplus, b = sigmoid (x 2), w = sigmoid; blockIdx.y selects the tensor. Bound by the
// two special-function operations per element about as much as by memory.
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
    // two rows per trip, all four loads issued before any arithmetic
    for (long long r = tid / G; r - (threadIdx.x & 31) / G < rows; r += 2 * stride) {
        float a[2][8], zz[2][8];
        bool active[2];
        size_t base[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const long long ru = r + u * stride;
            active[u] = ru < rows;
            base[u] = static_cast<size_t>(active[u] ? ru : 0) * dv + 8 * lane;
            Vec8<T>::load(o + base[u], a[u]);   // y may alias o: plain loads
            Vec8<T>::load(z + base[u], zz[u]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += a[u][e] * a[u][e];
            for (int off = 1; off < G; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss / dv + eps);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[u][e] = a[u][e] * inv * wt[e] * (zz[u][e] * sigmoid_f(zz[u][e]));
            if (active[u]) Vec8<T>::store(y + base[u], a[u]);
        }
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
    // conv: one CTA per (job, row, head, kConvTile tokens); gates: one thread per 8 elements, striding
    const long long nblk = (T + kConvTile - 1) / kConvTile;
    long long tiles[3];
    for (int j = 0; j < 3; ++j) tiles[j] = static_cast<long long>(B) * a.job[j].H * nblk;
    const long long ntiles = tiles[0] + tiles[1] + tiles[2];
    if (ntiles >= (1LL << 31)) return GDN2_ERR_UNSUPPORTED;
    const int dmax = dk > dv ? dk : dv;
    const size_t esz = dt == GDN2_BF16 ? 2 : 4;
    const size_t csmem = static_cast<size_t>(kConvTile + 3) * dmax * esz;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long gate_n8 = a.n8[0] > a.n8[2] ? a.n8[0] : a.n8[2];
    const dim3 ggrid(static_cast<unsigned>(gate_n8 / 256 + 1 < 4096 ? gate_n8 / 256 + 1 : 4096), 3);
    auto conv = [&](auto kernel) {
        if (csmem > 48 * 1024 &&
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(csmem)) !=
                cudaSuccess)
            return false;
        kernel<<<static_cast<unsigned>(ntiles), 256, csmem, s>>>(a, tiles[0], tiles[1]);
        return true;
    };
    bool ok;
    if (dt == GDN2_BF16) {
        ok = dmax == 256 ? conv(conv_tile_kernel<__nv_bfloat16, 8>) : conv(conv_tile_kernel<__nv_bfloat16, 4>);
        gates_kernel<__nv_bfloat16><<<ggrid, 256, 0, s>>>(a);
    } else {
        ok = dmax == 256 ? conv(conv_tile_kernel<float, 8>) : conv(conv_tile_kernel<float, 4>);
        gates_kernel<float><<<ggrid, 256, 0, s>>>(a);
    }
    if (!ok) return GDN2_ERR_CUDA;
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

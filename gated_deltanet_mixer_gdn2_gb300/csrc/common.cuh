// common.cuh -- internal definitions shared by the translation units of libgdn2.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/gdn2.h"

namespace gdn2 {

// Default budget of a bounded wait, in nanoseconds of polling.
constexpr long long kDefaultWaitNs = 2000000000LL;

// Device status bits (one word per translation unit, read and cleared by the host).
constexpr int kStatusTimeout = 1;

// Floor applied to the log-decay g by the chunked kernels: alpha = e^{-100} ~ 3.7e-44 is below
// every fp32 quantity those kernels form from it, so a full reset (g = -inf, alpha = 0) gives the
// same results while every cumulative sum of gates stays finite.
constexpr float kGateFloor = -100.f;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Eight consecutive elements of a token tensor as fp32 (16-byte aligned for bf16, 32 for fp32).
template <typename T>
struct Vec8;
template <>
struct Vec8<float> {
    __device__ static void load(const float* p, float (&x)[8]) {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    __device__ static void store(float* p, const float (&x)[8]) {
        reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    // through the read-only (non-coherent) path: only for data the kernel does not write
    __device__ static void load_ro(const float* p, float (&x)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};
template <>
struct Vec8<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16* p, float (&x)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float (&x)[8]) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
    // through the read-only (non-coherent) path: only for data the kernel does not write
    __device__ static void load_ro(const __nv_bfloat16* p, float (&x)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shapes of one chunked-forward call.
struct ChunkShape {
    int B, T, Hk, Hv, dk, dv, C;
    int nchunks() const { return (T + C - 1) / C; }
};

// Per-translation-unit status readers (defined next to the kernels).
int decode_read_clear_status(cudaStream_t s);
int step_read_clear_status(cudaStream_t s);
int chunk_simt_read_clear_status(cudaStream_t s);
int chunk_tc_read_clear_status(cudaStream_t s);

long long wait_limit_ns();

// Launchers (host side). Return cudaSuccess or the launch error.
cudaError_t launch_recurrent(const void* q, const void* k, const void* v, const void* g, const void* b,
                             const void* w, void* state, gdn2_dtype state_dt, const int* slots, int n_slots, void* o,
                             int B, int N, int Hk, int Hv, int dk, int dv, float scale, gdn2_dtype dt,
                             cudaStream_t s);

// Per-unit fp32 workspace of the CUDA-core chunked forward (chunk_simt.cu), also read by the chunked
// backward (backward_chunk.cu): W, q.e^G, k.e^{G_last-G} ([d_k][C], or token-major [C][d_k]), M [C][C],
// U~ ([d_v][C], or token-major [C][d_v]), e^{G_last} [d_k]; with both layouts (ext), channel-major
// copies of W and k.e^{G_last-G} [d_k][C] follow.
struct SimtWs {
    int dk, dv, C;
    bool ext = false;
    __host__ __device__ size_t unit_floats() const {
        size_t n = 3 * (size_t)dk * C + (size_t)C * C + (size_t)dv * C + dk;
        n = (n + 3) & ~size_t(3);
        return ext ? n + 2 * (size_t)dk * C : n;
    }
    __host__ __device__ size_t off_wt() const { return 0; }
    __host__ __device__ size_t off_qbt() const { return (size_t)dk * C; }
    __host__ __device__ size_t off_kht() const { return 2 * (size_t)dk * C; }
    __host__ __device__ size_t off_m() const { return 3 * (size_t)dk * C; }
    __host__ __device__ size_t off_utt() const { return 3 * (size_t)dk * C + (size_t)C * C; }
    __host__ __device__ size_t off_gam() const { return 3 * (size_t)dk * C + (size_t)C * C + (size_t)dv * C; }
    __host__ __device__ size_t off_wt2() const { return ((off_gam() + dk) + 3) & ~size_t(3); }
    __host__ __device__ size_t off_kht2() const { return off_wt2() + (size_t)dk * C; }
};

size_t chunk_simt_workspace_bytes(const ChunkShape& sh, bool token_major = false);
// The state-independent factors of every chunk into ws (layout SimtWs; token-major plus the
// channel-major copies of W and k.e^{G_last-G} when token_major), and, when t_out is given,
// T = (I + A)^{-1} per unit [C][C].
cudaError_t launch_factors_simt(const void* q, const void* k, const void* v, const void* g, const void* b,
                                const void* w, const ChunkShape& sh, gdn2_dtype dt, void* ws, float* t_out,
                                bool token_major, cudaStream_t s);
// Chunked backward (backward_chunk.cu): workspace bytes and the launches; d_k = d_v = 128.
size_t backward_chunked_workspace_bytes(int B, int T, int Hv);
cudaError_t launch_backward_chunked(const void* q, const void* k, const void* v, const void* g, const void* b,
                                    const void* w, const float* s0, const void* d_o, const float* dsT, void* dq,
                                    void* dk, void* dv, void* dg, void* db, void* dw, float* ds0, int B, int T, int Hk,
                                    int Hv, float scale, gdn2_dtype dt, void* ws, cudaStream_t s);
cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, const void* g, const void* b,
                              const void* w, const float* s0, float* sT, void* o, const ChunkShape& sh, float scale,
                              gdn2_dtype dt, void* ws, cudaStream_t s);

size_t chunk_tc_workspace_bytes(const ChunkShape& sh);
cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const void* g, const void* b,
                            const void* w, const float* s0, float* sT, void* o, const ChunkShape& sh, float scale,
                            void* ws, cudaStream_t s, long long wait_ns, void* s_save = nullptr,
                            void* u_save = nullptr);
// Tensor-core chunked backward (bf16, d_k and d_v 64 or 128, chunks of 64).
size_t backward_tc_workspace_bytes(int B, int T, int Hv, int dk, int dv);
cudaError_t launch_backward_tc(const void* q, const void* k, const void* v, const void* g, const void* b,
                               const void* w, const float* s0, const void* d_o, const float* dsT, void* dq, void* dk,
                               void* dv, void* dg, void* db, void* dw, float* ds0, int B, int T, int Hk, int Hv,
                               int d_k, int d_v, float scale, void* ws, cudaStream_t s, long long wait_ns);
int backward_tc_read_clear_status(cudaStream_t s);

}  // namespace gdn2

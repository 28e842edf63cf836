// tc_common.cuh -- pieces shared by the tensor-core chunk kernels (forward and backward): the
// workspace unit of the chunk factors, bounded mbarrier waits, tensor-memory and bulk-copy helpers,
// and the host-side tensor maps. Everything has internal linkage, so each translation unit that
// includes it gets its own device status word.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tma_map.cuh"

namespace gdn2 {
namespace {

__device__ int g_status_tc;

constexpr int kC = 64;
constexpr int kD = 128;

// workspace unit (one chunk of one value head), bytes
constexpr uint32_t kWsW = 0;         // -W = -T (b.k.e^G)    token-major [64][128] bf16
constexpr uint32_t kWsQb = 16384;    // q.e^G                token-major [64][128] bf16
constexpr uint32_t kWsKh = 32768;    // k.e^{G_last - G}     token-major [64][128] bf16
constexpr uint32_t kWsM = 49152;     // M = causal q-k       [64][64] bf16
constexpr uint32_t kWsT = 57344;     // T = (I + A)^{-1}      [64][64] bf16
constexpr uint32_t kWsGam = 65536;   // e^{G_last}           [128] fp32
constexpr uint32_t kWsUnit = 66048;

// ---------------------------------------------------------------------------------------------
// helpers

__device__ __forceinline__ void record_timeout() { atomicOr(&g_status_tc, kStatusTimeout); }

// CTA-uniform bounded wait: every thread polls with the caller's budget; a thread that gives up
// records the timeout and drains the barrier with the default budget (copies / MMAs in flight must
// land before the CTA releases its shared memory and TMEM). One block vote gives everyone the same
// outcome.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, long long limit_ns) {
    bool ok = mbar_wait(bar, parity, limit_ns);  // every thread observes the phase itself
    if (!ok) {
        record_timeout();
        mbar_wait(bar, parity, kDefaultWaitNs);
    }
    return __syncthreads_and(ok) != 0;
}



// 64 fp32 columns of this warp's TMEM lanes starting at column `col`.
__device__ __forceinline__ void tmem_ld64(uint32_t tmem_base, int warp, int col, float (&x)[64]) {
    uint32_t r[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        tmem_ld16(tmem_base + (static_cast<uint32_t>(32 * warp) << 16) + col + 16 * q, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) x[16 * q + i] = __uint_as_float(r[i]);
    }
}



__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

// Issue n16 x 16-column TMEM loads of this warp's lanes, then one wait.
template <int N16>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&x)[16 * N16]) {
    uint32_t r[N16][16];
#pragma unroll
    for (int q = 0; q < N16; ++q) tmem_ld16(taddr + 16 * q, r[q]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < N16; ++q)
#pragma unroll
        for (int i = 0; i < 16; ++i) x[16 * q + i] = __uint_as_float(r[q][i]);
}

__device__ __forceinline__ void tma_store_3d(const void* map, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}



// Bounded wait that also gives up as soon as another role has recorded a failure in *err.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, long long limit_ns,
                                                   volatile int* err) {
    if (limit_ns <= 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kWaitHintNs)) return true;
        if (*err) return false;
        if ((long long)(globaltimer_ns() - t0) > limit_ns) return false;
    }
}

__device__ __forceinline__ void note_failure(volatile int* err) {
    if (!*err) {
        record_timeout();
        *err = 1;
    }
}

// Warp-uniform wait: every lane observes the phase itself (bounded), and one vote makes the outcome
// the warp's; a lane that gave up records the timeout.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, long long limit_ns, volatile int* err) {
    const bool ok = mbar_wait_or_abort(bar, parity, limit_ns, err);
    if (!ok) note_failure(err);
    return __all_sync(0xffffffffu, ok) != 0;
}

// 32 fp32 values -> bf16 into four 16-byte chunks (c0..c0+3) of a 128-byte-swizzled row
__device__ __forceinline__ void st_row_bf16x32(uint8_t* tile, int row, int c0, const float* x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[8 * c + e];
        *reinterpret_cast<uint4*>(tile + row * 128 + (((c0 + c) ^ (row & 7)) << 4)) = pack8(y);
    }
}

// 64 fp32 values -> bf16, stored as eight 16-byte pieces at a 16-byte aligned global address
__device__ __forceinline__ void st_global_bf16x64(__nv_bfloat16* dst, const float* x) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[8 * c + e];
        d[c] = pack8(y);
    }
}

__device__ __forceinline__ void tma_store_4d(const void* map, const void* src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}


// ---------------------------------------------------------------------------------------------
// host: tensor maps

// token tensor [B, T, H, d] bf16 (d = 128 unless given) viewed as (d, H, T, B); box (64, 1, 64, 1)
bool token_map(CUtensorMap* m, const void* p, int B, int T, int H, int d = kD) {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)d * 2, (uint64_t)H * d * 2, (uint64_t)T * H * d * 2};
    const uint32_t box[4] = {64, 1, kC, 1};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// output [B, T, H, d_v] bf16 viewed as (d_v, H, T, B); box (64, 1, 32, 1), 128-byte swizzle
bool out_map(CUtensorMap* m, const void* p, int B, int T, int H, int dv) {
    const uint64_t dims[4] = {(uint64_t)dv, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)dv * 2, (uint64_t)H * dv * 2, (uint64_t)T * H * dv * 2};
    const uint32_t box[4] = {64, 1, 32, 1};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// workspace section viewed as (cols, rows, units); box (box_cols, box_rows, 1)
bool ws_map(CUtensorMap* m, const void* p, CUtensorMapDataType dt, int esize, int cols, int rows, int units,
            int box_cols, int box_rows, CUtensorMapSwizzle sw) {
    const uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)units};
    const uint64_t st[2] = {(uint64_t)cols * esize, kWsUnit};
    const uint32_t box[3] = {(uint32_t)box_cols, (uint32_t)box_rows, 1};
    return make_map(m, dt, 3, p, dims, st, box, sw);
}


}  // namespace
}  // namespace gdn2

// chunk_tc.cu -- chunked forward on the 5th-generation tensor cores (tcgen05 + TMA + TMEM), bf16
// inputs, d_k = d_v = 128, chunk C = 64.
//
// Same chunked WY / UT form as the SIMT path (burn-gdn2 0.1.5 docs: "chunked WY decomposition
// (training)"); per chunk of C tokens entering with state S_n, G_i = inclusive cumulative
// log-decay of the chunk per key channel:
//     A = tril_{-1}(K_bar K_til^T),  M = tril_0(Q_anc K_til^T)           [one M=128 MMA, stacked]
//         with K_bar = b.k.e^{G-a}, Q_anc = q.e^{G-a}, K_til = k.e^{a-G} and a per-channel anchor
//         a = (min G + max G)/2, so that every factor stays within e^{+-range/2}
//     T = (I + A)^{-1}                                                   [fp32, blocked forward substitution]
//     W^T = (b.k.e^{G})^T T^T,  U~^T = (w.v)^T T^T                        [two M=128 MMAs]
//     U = U~ - W S_n;  O = (q.e^{G}) S_n + M U;  S_{n+1} = e^{G_last} . S_n + (k.e^{G_last-G})^T U
//
// Kernel 1 "factors" (grid: chunks x heads; 128 threads; 2 CTAs/SM): TMA loads the six token
// tiles of one chunk, one pass over the chunk computes the decayed operands, tcgen05 forms A|M,
// CUDA cores invert (I + A), tcgen05 forms W^T and U~^T; results go to the workspace.
// Kernel 2 "state" (grid: heads x d_v halves; 128 threads; sequential over chunks): TMA double-
// buffers the chunk factors; the state slice lives in registers (fp32, one d_k row per thread =
// one TMEM lane) with a bf16 copy in shared memory as the MMA operand; per chunk two MMA rounds:
// [W; Q]·S_n -> U -> {[0; M]·U, K^^T·U}.
//
// Every barrier wait is bounded; on expiry the CTA records a timeout in the device status word,
// drains its own copies / MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gdn2 {

namespace {

__device__ int g_status_tc;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kSlice = 64;

// workspace unit (one chunk of one value head), bytes
constexpr uint32_t kWsWT = 0;        // W^T      [128][64] bf16
constexpr uint32_t kWsQbT = 16384;   // (q.e^G)^T [128][64] bf16
constexpr uint32_t kWsKhT = 32768;   // (k.e^{G_last-G})^T [128][64] bf16
constexpr uint32_t kWsM = 49152;     // M        [64][64]  bf16
constexpr uint32_t kWsUtT = 57344;   // U~^T     [128][64] fp32
constexpr uint32_t kWsGam = 90112;   // e^{G_last} [128] fp32
constexpr uint32_t kWsUnit = 91136;

// ---------------------------------------------------------------------------------------------
// helpers

__device__ __forceinline__ void record_timeout() { atomicOr(&g_status_tc, kStatusTimeout); }

// CTA-uniform bounded wait: thread 0 polls with the caller's budget; on failure it records the
// timeout and drains the barrier with the default budget (copies / MMAs in flight must land before
// the CTA releases its shared memory and TMEM). Everyone returns the same verdict.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, long long limit_ns, int* flag) {
    if (threadIdx.x == 0) {
        bool ok = mbar_wait(bar, parity, limit_ns);
        if (!ok) {
            record_timeout();
            mbar_wait(bar, parity, kDefaultWaitNs);
        }
        *flag = ok ? 1 : 0;
    }
    __syncthreads();
    const bool ok = *flag != 0;
    if (ok) mbar_wait(bar, parity, kDefaultWaitNs);  // completes at once; orders the async writes
    return ok;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_at(const uint8_t* base, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}
__device__ __forceinline__ void store_bf16(uint8_t* base, uint32_t off, float x) {
    *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(x);
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

// Write 64 values as one 128-byte bf16 row `row` of a 128B-swizzled tile at `tile`.
__device__ __forceinline__ void store_row_sw128(uint8_t* tile, int row, const float (&x)[64]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u;
        u.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
        u.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
        u.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
        u.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
        *reinterpret_cast<uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4)) = u;
    }
}

__device__ __forceinline__ void store_row_bf16_global(void* dst, const float (&x)[64], float scale) {
    uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u;
        u.x = pack_bf16x2(scale * x[8 * c + 0], scale * x[8 * c + 1]);
        u.y = pack_bf16x2(scale * x[8 * c + 2], scale * x[8 * c + 3]);
        u.z = pack_bf16x2(scale * x[8 * c + 4], scale * x[8 * c + 5]);
        u.w = pack_bf16x2(scale * x[8 * c + 6], scale * x[8 * c + 7]);
        p[c] = u;
    }
}

// ---------------------------------------------------------------------------------------------
// kernel 1: per-chunk factors

struct FactorMaps {
    CUtensorMap q, k, g, b, v, w;
};

namespace fs {  // shared-memory layout of the factor kernel (offsets from a 1024-aligned base)
constexpr uint32_t A1 = 0;        // [b.k.e^{G-a} ; q.e^{G-a}] 128 x 128, K-major, two 64-wide K blocks
constexpr uint32_t K = 32768;     // k -> k.e^{a-G} (64 x 128, K-major, two K blocks)
constexpr uint32_t G = 49152;     // g -> b.k.e^{G} (64 tokens x 128, MN-major for M = d_k)
constexpr uint32_t V = 65536;     // v -> w.v       (MN-major for M = d_v)
constexpr uint32_t W = 81920;     // w (then fp32 scratch for the blocked solve)
constexpr uint32_t T = 98304;     // T = (I + A)^{-1} bf16, 64 x 64, K-major (rows i, columns j)
constexpr uint32_t BAR = 106496;  // 2 mbarriers, TMEM base, flag
constexpr uint32_t TOTAL = BAR + 64;
constexpr uint32_t AF = 0;        // fp32 A [64][65] (aliases A1/K once A|M has been read)
constexpr uint32_t TF = 16640;    // fp32 T [64][65]
constexpr uint32_t PF = W;        // fp32 [3][16][16] partial products
constexpr int LDF = 65;
}  // namespace fs

__global__ void __launch_bounds__(128, 2)
    factors_tc_kernel(const __grid_constant__ FactorMaps maps, uint8_t* __restrict__ ws, int Hk, int Hv, int NC,
                      long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + fs::BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + fs::BAR + 16);
    int* flag = reinterpret_cast<int*>(sm + fs::BAR + 20);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, bh = blockIdx.y;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    uint8_t* unit = ws + (static_cast<size_t>(bh) * NC + n) * kWsUnit;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        mbar_arrive_expect_tx(bar_tma, 6 * 16384);
        const int t0 = n * kC;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + fs::A1 + kb * 16384 + 8192, &maps.q, 64 * kb, hk, t0, bi, bar_tma);
            tma_load_4d(sm + fs::A1 + kb * 16384, &maps.b, 64 * kb, hv, t0, bi, bar_tma);
            tma_load_4d(sm + fs::K + kb * 8192, &maps.k, 64 * kb, hk, t0, bi, bar_tma);
            tma_load_4d(sm + fs::G + kb * 8192, &maps.g, 64 * kb, hv, t0, bi, bar_tma);
            tma_load_4d(sm + fs::V + kb * 8192, &maps.v, 64 * kb, hv, t0, bi, bar_tma);
            tma_load_4d(sm + fs::W + kb * 8192, &maps.w, 64 * kb, hv, t0, bi, bar_tma);
        }
    }
    bool ok = cta_wait(bar_tma, 0, wait_ns, flag);
    if (ok) {
        // ---- one pass over the chunk per channel c (thread c): decayed operands, outputs
        const int c = tid;
        const int kb = c >> 6, cc = c & 63;
        uint8_t* pA1b = sm + fs::A1 + kb * 16384;
        uint8_t* pA1q = pA1b + 8192;
        uint8_t* pK = sm + fs::K + kb * 8192;
        uint8_t* pG = sm + fs::G + kb * 8192;
        uint8_t* pV = sm + fs::V + kb * 8192;
        uint8_t* pW = sm + fs::W + kb * 8192;
        float gmin = 0.f, gmax = 0.f, acc = 0.f;
        for (int t = 0; t < kC; ++t) {
            acc += bf16_at(pG, sw128_off(t, cc));
            gmin = (t == 0) ? acc : fminf(gmin, acc);
            gmax = (t == 0) ? acc : fmaxf(gmax, acc);
        }
        const float glast = acc;
        const float anc = 0.5f * (gmin + gmax);
        uint32_t qb_pack[4], kh_pack[4];
        float G = 0.f;
        for (int t = 0; t < kC; ++t) {
            const uint32_t off = sw128_off(t, cc);
            G += bf16_at(pG, off);
            const float e1 = __expf(G - anc);
            const float e2 = __expf(anc - G);
            const float eg = __expf(G);
            const float er = __expf(glast - G);
            const float kk = bf16_at(pK, off), qq = bf16_at(pA1q, off), bb = bf16_at(pA1b, off);
            const float vv = bf16_at(pV, off), ww = bf16_at(pW, off);
            store_bf16(pA1b, off, bb * kk * e1);
            store_bf16(pA1q, off, qq * e1);
            store_bf16(pK, off, kk * e2);
            store_bf16(pG, off, bb * kk * eg);
            store_bf16(pV, off, ww * vv);
            const float qb = qq * eg, kh = kk * er;
            const int slot = (t & 7) >> 1;
            if (t & 1) {
                qb_pack[slot] |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(qb))) << 16;
                kh_pack[slot] |= static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(kh))) << 16;
            } else {
                qb_pack[slot] = __bfloat16_as_ushort(__float2bfloat16_rn(qb));
                kh_pack[slot] = __bfloat16_as_ushort(__float2bfloat16_rn(kh));
            }
            if ((t & 7) == 7) {
                const int chunk = t >> 3;
                *reinterpret_cast<uint4*>(unit + kWsQbT + c * 128 + chunk * 16) =
                    make_uint4(qb_pack[0], qb_pack[1], qb_pack[2], qb_pack[3]);
                *reinterpret_cast<uint4*>(unit + kWsKhT + c * 128 + chunk * 16) =
                    make_uint4(kh_pack[0], kh_pack[1], kh_pack[2], kh_pack[3]);
            }
        }
        reinterpret_cast<float*>(unit + kWsGam)[c] = __expf(glast);
        fence_proxy_async_smem();
        __syncthreads();

        // ---- A | M = [K_bar ; Q_anc] K_til^T   (M = 128, N = 64, K = 128)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = smem_desc(sbase + fs::A1 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + fs::K + (s >> 2) * 8192 + (s & 3) * 32, 16, 1024, kSwizzle128B);
                mma_bf16(tmem, ad, bd, id, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, 0, wait_ns, flag);
    }
    if (ok) {
        tc_fence_after();
        float* AF = reinterpret_cast<float*>(sm + fs::AF);
        float* TF = reinterpret_cast<float*>(sm + fs::TF);
        float* PF = reinterpret_cast<float*>(sm + fs::PF);
        {
            float x[64];
            tmem_ld64(tmem, warp, 0, x);
            if (warp < 2) {
                const int i = 32 * warp + lane;
#pragma unroll
                for (int j = 0; j < 64; ++j) AF[i * fs::LDF + j] = (j < i) ? x[j] : 0.f;
            } else {
                const int i = 32 * (warp - 2) + lane;
#pragma unroll
                for (int j = 0; j < 64; ++j) x[j] = (j <= i) ? x[j] : 0.f;
                store_row_bf16_global(unit + kWsM + i * 128, x, 1.f);
            }
        }
        __syncthreads();
        // ---- T = (I + A)^{-1}: diagonal 16x16 blocks (one warp each), then block rows
        if (lane < 16) {
            const int base = 16 * warp, jj = lane;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = 0.f;
#pragma unroll
                for (int l = 0; l < i; ++l) s = fmaf(AF[(base + i) * fs::LDF + base + l], x[l], s);
                x[i] = (i == jj) ? 1.f : ((i < jj) ? 0.f : -s);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) TF[(base + i) * fs::LDF + base + jj] = x[i];
        }
        __syncthreads();
        for (int I = 1; I < 4; ++I) {
            for (int e = tid; e < I * 256; e += 128) {
                const int J = e >> 8, r = (e >> 4) & 15, cq = e & 15;
                float s = 0.f;
                for (int m = 16 * J; m < 16 * I; ++m) s = fmaf(AF[(16 * I + r) * fs::LDF + m], TF[m * fs::LDF + 16 * J + cq], s);
                PF[e] = s;
            }
            __syncthreads();
            for (int e = tid; e < I * 256; e += 128) {
                const int J = e >> 8, r = (e >> 4) & 15, cq = e & 15;
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) s = fmaf(TF[(16 * I + r) * fs::LDF + 16 * I + m], PF[(J << 8) + (m << 4) + cq], s);
                TF[(16 * I + r) * fs::LDF + 16 * J + cq] = -s;
            }
            __syncthreads();
        }
        for (int p = tid; p < 64 * 64; p += 128) {
            const int i = p >> 6, j = p & 63;
            store_bf16(sm + fs::T, sw128_off(i, j), (j <= i) ? TF[i * fs::LDF + j] : 0.f);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- W^T = (b.k.e^G)^T T^T and U~^T = (w.v)^T T^T   (M = 128, N = 64, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, true, false);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = smem_desc(sbase + fs::T + s * 32, 16, 1024, kSwizzle128B);
                const uint64_t a1 = smem_desc(sbase + fs::G + s * 2048, 8192, 1024, kSwizzle128B);
                const uint64_t a2 = smem_desc(sbase + fs::V + s * 2048, 8192, 1024, kSwizzle128B);
                mma_bf16(tmem + 64, a1, bd, id, s > 0);
                mma_bf16(tmem + 128, a2, bd, id, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, 1, wait_ns, flag);
        if (ok) {
            tc_fence_after();
            const int c = tid;
            float x[64];
            tmem_ld64(tmem, warp, 64, x);
            store_row_bf16_global(unit + kWsWT + c * 128, x, 1.f);
            tmem_ld64(tmem, warp, 128, x);
            float4* dst = reinterpret_cast<float4*>(unit + kWsUtT + c * 256);
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) dst[q4] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------------------------
// kernel 2: state chain + output

struct StateMaps {
    CUtensorMap wt, qbt, kht, m, utt;
};

namespace ss {
constexpr uint32_t A1 = 0;          // [W ; Q] MN-major: W^T tile, then (q.e^G)^T tile (16 KB each)
constexpr uint32_t A3 = 32768;      // (k.e^{G_last-G})^T, K-major (rows d_k, K = tokens)
constexpr uint32_t A2 = 49152;      // [0 ; M], K-major (rows 0..63 zero)
constexpr uint32_t UT = 65536;      // U~^T slice, fp32 [64 columns][64 tokens]
constexpr uint32_t GAM = 81920;     // e^{G_last} fp32 [128]
constexpr uint32_t STAGE = 82944;
constexpr uint32_t SBF = 2 * STAGE;         // S_n bf16 [128 rows d_k][64], MN-major B operand
constexpr uint32_t UBF = SBF + 16384;       // U bf16 [64 tokens][64], MN-major B operand
constexpr uint32_t BAR = UBF + 8192;        // full[2], mma, TMEM base, 3 flags
constexpr uint32_t TOTAL = BAR + 64;
constexpr uint32_t TX = 16384 * 3 + 8192 + 16384 + 512;
}  // namespace ss

__global__ void __launch_bounds__(128, 1)
    state_tc_kernel(const __grid_constant__ StateMaps maps, const uint8_t* __restrict__ ws,
                    const float* __restrict__ s0, float* __restrict__ sT_out, __nv_bfloat16* __restrict__ o, int T,
                    int Hv, int NC, float scale, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + ss::BAR);
    uint64_t* bar_mma = full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + ss::BAR + 24);
    int* flag = reinterpret_cast<int*>(sm + ss::BAR + 28);  // 3 slots: one per wait site, so that a
                                                            // slot is never rewritten before all read it

    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x, z = blockIdx.y;
    const int bi = bh / Hv, hv = bh - bi * Hv;
    const int r = tid;  // d_k row owned by this thread (= TMEM lane)

    if (tid == 0) {
        mbar_init(full, 1);
        mbar_init(full + 1, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    // zero rows 0..63 of the [0 ; M] operand in both stages
    for (int p = tid; p < 2 * 512; p += 128) {
        const int st = p >> 9, q16 = p & 511;
        reinterpret_cast<uint4*>(sm + st * ss::STAGE + ss::A2)[q16] = make_uint4(0, 0, 0, 0);
    }
    float S[64];
    {
        const float* src = s0 ? s0 + (static_cast<size_t>(bh) * kD + r) * kD + z * kSlice : nullptr;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            float4 t4 = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = t4.x;
            S[j + 1] = t4.y;
            S[j + 2] = t4.z;
            S[j + 3] = t4.w;
        }
        store_row_sw128(sm + ss::SBF, r, S);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto issue = [&](int n) {
        const int st = n & 1;
        uint8_t* sb = sm + st * ss::STAGE;
        const int u = bh * NC + n;
        mbar_arrive_expect_tx(full + st, ss::TX);
        tma_load_3d(sb + ss::A1, &maps.wt, 0, 0, u, full + st);
        tma_load_3d(sb + ss::A1 + 16384, &maps.qbt, 0, 0, u, full + st);
        tma_load_3d(sb + ss::A3, &maps.kht, 0, 0, u, full + st);
        tma_load_3d(sb + ss::A2 + 8192, &maps.m, 0, 0, u, full + st);
        tma_load_3d(sb + ss::UT, &maps.utt, 0, z * kSlice, u, full + st);
        bulk_load(sb + ss::GAM, ws + static_cast<size_t>(u) * kWsUnit + kWsGam, 512, full + st);
    };
    if (tid == 0 && NC > 0) issue(0);

    uint32_t mma_phase = 0;
    bool ok = true;
    int n = 0;
    for (; n < NC && ok; ++n) {
        const int st = n & 1;
        const uint32_t sb = sbase + st * ss::STAGE;
        if (tid == 0 && n + 1 < NC) issue(n + 1);
        ok = cta_wait(full + st, (n >> 1) & 1, wait_ns, flag + 0);
        if (!ok) break;
        // ---- D1 = [W ; Q] S_n   (M = 128, N = 64, K = 128; A and B MN-major)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = smem_desc(sb + ss::A1 + s * 2048, 16384, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + ss::SBF + s * 2048, 16384, 1024, kSwizzle128B);
                mma_bf16(tmem, ad, bd, id, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, mma_phase, wait_ns, flag + 1);
        mma_phase ^= 1;
        if (!ok) break;
        tc_fence_after();
        if (warp < 2) {  // U = U~ - W S_n for tokens i = 0..63
            const int i = tid;
            float x[64];
            tmem_ld64(tmem, warp, 0, x);
            const float* ut = reinterpret_cast<const float*>(sm + st * ss::STAGE + ss::UT);
#pragma unroll
            for (int j = 0; j < 64; ++j) x[j] = ut[j * 64 + i] - x[j];
            store_row_sw128(sm + ss::UBF, i, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- D1 += [0 ; M] U  and  D2 = K^^T U   (M = 128, N = 64, K = 64; A K-major, B MN-major)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = smem_desc(sbase + ss::UBF + s * 2048, 8192, 1024, kSwizzle128B);
                const uint64_t a2 = smem_desc(sb + ss::A2 + s * 32, 16, 1024, kSwizzle128B);
                const uint64_t a3 = smem_desc(sb + ss::A3 + s * 32, 16, 1024, kSwizzle128B);
                mma_bf16(tmem, a2, bd, id, 1);
                mma_bf16(tmem + 64, a3, bd, id, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, mma_phase, wait_ns, flag + 2);
        mma_phase ^= 1;
        if (!ok) break;
        tc_fence_after();
        if (warp >= 2) {  // O rows = tokens 0..63
            const int i = tid - 64;
            const int tok = n * kC + i;
            float x[64];
            tmem_ld64(tmem, warp, 0, x);
            if (tok < T)
                store_row_bf16_global(o + ((static_cast<size_t>(bi) * T + tok) * Hv + hv) * kD + z * kSlice, x, scale);
        }
        {
            float x[64];
            tmem_ld64(tmem, warp, 64, x);
            const float gam = reinterpret_cast<const float*>(sm + st * ss::STAGE + ss::GAM)[r];
#pragma unroll
            for (int j = 0; j < 64; ++j) S[j] = fmaf(gam, S[j], x[j]);
            store_row_sw128(sm + ss::SBF, r, S);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    if (!ok) {
        // drain the prefetch of the next chunk if it was issued
        if (tid == 0 && n + 1 < NC) mbar_wait(full + ((n + 1) & 1), ((n + 1) >> 1) & 1, kDefaultWaitNs);
    } else if (sT_out) {
        float* dst = sT_out + (static_cast<size_t>(bh) * kD + r) * kD + z * kSlice;
#pragma unroll
        for (int j = 0; j < 64; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------------------------
// UMMA layout self-test: one M=128, N=64 product with the operand layouts the kernels above use.

struct SelftestMaps {
    CUtensorMap a, b;
};

__global__ void __launch_bounds__(128, 1)
    selftest_umma_kernel(const __grid_constant__ SelftestMaps maps, int case_id, int soft,
                         const __nv_bfloat16* __restrict__ a_st, const __nv_bfloat16* __restrict__ b_st,
                         float* __restrict__ d_out, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint8_t* sA = sm;
    uint8_t* sB = sm + 32768;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 49152);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + 49152 + 16);
    int* flag = reinterpret_cast<int*>(sm + 49152 + 20);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // storage shapes (rows x cols) per case, see launch_selftest
    const int a_rows = (case_id == 0 || case_id == 2) ? 128 : (case_id == 1 ? 64 : 128);
    const int a_cols = (case_id == 3) ? 64 : 128;
    const int b_rows = (case_id == 0 || case_id == 1) ? 64 : (case_id == 2 ? 128 : 64);
    const int b_cols = (case_id == 0) ? 128 : 64;
    const bool a_mn = (case_id == 1 || case_id == 2);
    const bool b_mn = (case_id == 2 || case_id == 3);
    const int K = (case_id == 0 || case_id == 2) ? 128 : 64;

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // a storage of R rows x (64 * nb) columns becomes nb blocks of R x 128 B (block j = columns 64j..)
    bool ok = true;
    if (soft) {
        for (int p = tid; p < a_rows * a_cols; p += 128) {
            const int rr = p / a_cols, cc = p % a_cols;
            *reinterpret_cast<__nv_bfloat16*>(sA + (cc >> 6) * (a_rows * 128) + sw128_off(rr, cc & 63)) = a_st[p];
        }
        for (int p = tid; p < b_rows * b_cols; p += 128) {
            const int rr = p / b_cols, cc = p % b_cols;
            *reinterpret_cast<__nv_bfloat16*>(sB + (cc >> 6) * (b_rows * 128) + sw128_off(rr, cc & 63)) = b_st[p];
        }
        fence_proxy_async_smem();
        __syncthreads();
    } else {
        if (tid == 0) {
            mbar_arrive_expect_tx(bar, (a_rows * a_cols + b_rows * b_cols) * 2);
            for (int j = 0; j < a_cols / 64; ++j) tma_load_3d(sA + j * a_rows * 128, &maps.a, 64 * j, 0, 0, bar);
            for (int j = 0; j < b_cols / 64; ++j) tma_load_3d(sB + j * b_rows * 128, &maps.b, 64 * j, 0, 0, bar);
        }
        ok = cta_wait(bar, 0, wait_ns, flag);
    }
    if (ok) {
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64, a_mn, b_mn);
            for (int s = 0; s < K / 16; ++s) {
                // K-major: K blocks of 64 are separate R x 128 B regions; step 32 B inside a block.
                // MN-major: K rows are 128-byte rows; step 16 rows = 2048 B; LBO = next 64-wide MN block.
                const uint32_t aoff = a_mn ? s * 2048 : (s >> 2) * (a_rows * 128) + (s & 3) * 32;
                const uint32_t boff = b_mn ? s * 2048 : (s >> 2) * (b_rows * 128) + (s & 3) * 32;
                const uint64_t ad = smem_desc(sbase + aoff, a_mn ? a_rows * 128 : 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + 32768 + boff, b_mn ? b_rows * 128 : 16, 1024, kSwizzle128B);
                mma_bf16(tmem, ad, bd, id, s > 0);
            }
            mma_commit(bar + 1);
        }
        ok = cta_wait(bar + 1, 0, wait_ns, flag);
    }
    if (ok) {
        tc_fence_after();
        float x[64];
        tmem_ld64(tmem, warp, 0, x);
        for (int j = 0; j < 64; ++j) d_out[(32 * warp + lane) * 64 + j] = x[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------------------------------------
// host: tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    return f(m, dt, rank, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// token tensor [B, T, H, 128] bf16 viewed as (d, H, T, B); box (64, 1, 64, 1)
bool token_map(CUtensorMap* m, const void* p, int B, int T, int H) {
    const uint64_t dims[4] = {kD, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {kD * 2, (uint64_t)H * kD * 2, (uint64_t)T * H * kD * 2};
    const uint32_t box[4] = {64, 1, kC, 1};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// workspace section viewed as (cols, rows, units)
bool ws_map(CUtensorMap* m, const void* p, CUtensorMapDataType dt, int esize, int cols, int rows, int units,
            int box_rows, CUtensorMapSwizzle sw) {
    const uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)units};
    const uint64_t st[2] = {(uint64_t)cols * esize, kWsUnit};
    const uint32_t box[3] = {(uint32_t)cols, (uint32_t)box_rows, 1};
    return make_map(m, dt, 3, p, dims, st, box, sw);
}

}  // namespace

size_t chunk_tc_workspace_bytes(const ChunkShape& sh) {
    return static_cast<size_t>(kWsUnit) * sh.nchunks() * sh.B * sh.Hv;
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const void* g, const void* b,
                            const void* w, const float* s0, float* sT, void* o, const ChunkShape& sh, float scale,
                            void* ws, cudaStream_t s, long long wait_ns) {
    const int NC = sh.nchunks();
    FactorMaps fm;
    if (!token_map(&fm.q, q, sh.B, sh.T, sh.Hk) || !token_map(&fm.k, k, sh.B, sh.T, sh.Hk) ||
        !token_map(&fm.g, g, sh.B, sh.T, sh.Hv) || !token_map(&fm.b, b, sh.B, sh.T, sh.Hv) ||
        !token_map(&fm.v, v, sh.B, sh.T, sh.Hv) || !token_map(&fm.w, w, sh.B, sh.T, sh.Hv))
        return cudaErrorInvalidValue;
    const int units = NC * sh.B * sh.Hv;
    const uint8_t* wsb = static_cast<const uint8_t*>(ws);
    StateMaps sm_;
    if (!ws_map(&sm_.wt, wsb + kWsWT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, 128, units, 128,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
        !ws_map(&sm_.qbt, wsb + kWsQbT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, 128, units, 128,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
        !ws_map(&sm_.kht, wsb + kWsKhT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, 128, units, 128,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
        !ws_map(&sm_.m, wsb + kWsM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, 64, units, 64,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
        !ws_map(&sm_.utt, wsb + kWsUtT, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 64, 128, units, kSlice,
                CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    // The state kernel runs one CTA per SM, so it takes the whole 227 KB: operand descriptors can
    // then never reach past the CTA's own allocation.
    const size_t f_smem = fs::TOTAL + 1024, s_smem = 232448;
    static_assert(ss::TOTAL + 1024 <= 232448, "state kernel shared memory");
    cudaError_t e = cudaFuncSetAttribute(factors_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    factors_tc_kernel<<<dim3(NC, sh.B * sh.Hv), 128, f_smem, s>>>(fm, static_cast<uint8_t*>(ws), sh.Hk, sh.Hv, NC,
                                                                  wait_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    state_tc_kernel<<<dim3(sh.B * sh.Hv, kD / kSlice), 128, s_smem, s>>>(
        sm_, wsb, s0, sT, static_cast<__nv_bfloat16*>(o), sh.T, sh.Hv, NC, scale, wait_ns);
    return cudaGetLastError();
}

int chunk_tc_read_clear_status(cudaStream_t s) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_tc, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (v && cudaMemcpyToSymbolAsync(g_status_tc, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    cudaStreamSynchronize(s);
    return v;
}

cudaError_t launch_selftest_umma(int case_id, int soft, const void* a_st, const void* b_st, float* d_out,
                                 cudaStream_t s, long long wait_ns) {
    // storage (rows x cols): case 0: A 128x128 (M x K), B 64x128 (N x K)
    //                        case 1: A 64x128 (K x M),  B 64x64 (N x K)
    //                        case 2: A 128x128 (K x M), B 128x64 (K x N)
    //                        case 3: A 128x64 (M x K),  B 64x64 (K x N)
    static const int shp[4][4] = {{128, 128, 64, 128}, {64, 128, 64, 64}, {128, 128, 128, 64}, {128, 64, 64, 64}};
    if (case_id < 0 || case_id > 3) return cudaErrorInvalidValue;
    const int ar = shp[case_id][0], ac = shp[case_id][1], br = shp[case_id][2], bc = shp[case_id][3];
    SelftestMaps m;
    const uint64_t ad[3] = {(uint64_t)ac, (uint64_t)ar, 1}, as[2] = {(uint64_t)ac * 2, (uint64_t)ac * ar * 2};
    const uint64_t bdm[3] = {(uint64_t)bc, (uint64_t)br, 1}, bs[2] = {(uint64_t)bc * 2, (uint64_t)bc * br * 2};
    const uint32_t abox[3] = {64, (uint32_t)ar, 1}, bbox[3] = {64, (uint32_t)br, 1};
    if (!make_map(&m.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a_st, ad, as, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&m.b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b_st, bdm, bs, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const size_t smem = 102400;  // generous: every descriptor stays inside the allocation
    cudaError_t e = cudaFuncSetAttribute(selftest_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    selftest_umma_kernel<<<1, 128, smem, s>>>(m, case_id, soft, static_cast<const __nv_bfloat16*>(a_st),
                                              static_cast<const __nv_bfloat16*>(b_st), d_out, wait_ns);
    return cudaGetLastError();
}

}  // namespace gdn2

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
constexpr uint32_t kWsW = 0;         // W = T (b.k.e^G)      token-major [64][128] bf16
constexpr uint32_t kWsQb = 16384;    // q.e^G                token-major [64][128] bf16
constexpr uint32_t kWsKh = 32768;    // k.e^{G_last - G}     token-major [64][128] bf16
constexpr uint32_t kWsM = 49152;     // M = causal q-k       [64][64] bf16
constexpr uint32_t kWsT = 57344;     // T = (I + A)^{-1}      [64][64] bf16
constexpr uint32_t kWsGam = 65536;   // e^{G_last}           [128] fp32
constexpr uint32_t kWsUnit = 66048;

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


// ---------------------------------------------------------------------------------------------
// kernel 1: per-chunk factors

struct FactorMaps {
    CUtensorMap q, k, g, b;        // token tiles (loads)
    CUtensorMap m_st, t_st, w_st;  // workspace sections written with TMA stores
};

namespace fs {  // shared-memory layout of the factor kernel (offsets from a 1024-aligned base)
constexpr uint32_t A1 = 0;        // [b.k.e^{G-a} ; q.e^{G-a}] 128 x 128, K-major, two 64-wide K blocks
constexpr uint32_t K = 32768;     // k -> k.e^{a-G} (64 x 128, K-major, two K blocks)
constexpr uint32_t G = 49152;     // g -> b.k.e^{G} (64 tokens x 128: MN-major B operand, N = d_k)
constexpr uint32_t SGS = 65536;   // token-group sums fp32 [16][128]; later M staging [64][64] bf16
constexpr uint32_t BAR = 73728;   // 2 mbarriers, TMEM base, flag
constexpr uint32_t CST = BAR + 64;  // per-channel anchor a, e^{a}, e^{G_last - a} (fp32 [3][128])
constexpr uint32_t TOTAL = CST + 3 * 512;
// solve scratch (A1/K are dead once A|M has been read): fp32, 16-byte aligned rows of 68
constexpr int LDF = 68;
constexpr uint32_t AF = 0;                       // A [64][68]
constexpr uint32_t TF = 64 * LDF * 4;            // T [64][68]
constexpr uint32_t PF = 2 * 64 * LDF * 4;        // products [32][36]
constexpr int LDP = 36;
// T = (I + A)^{-1} as bf16 K-major [64][64]; its MMA reads 64 further rows (the first K-block of
// b.k.e^{G}, finite, result rows discarded)
constexpr uint32_t TB = 40960;
// W staging after the last MMA: two 128-byte-swizzled [64 tokens][64 channels] bf16 tiles
constexpr uint32_t WSTG = 0;
constexpr int kThreads = 256;
}  // namespace fs

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
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// sum_k L[k] R[k][c4..c4+3] (fp32 smem, 16-byte aligned rows)
template <int KN>
__device__ __forceinline__ float4 row_times(const float* Lrow, const float* R, int ldr, int c4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KN; ++k) {
        const float a = Lrow[k];
        const float4 b = *reinterpret_cast<const float4*>(R + k * ldr + c4);
        acc.x = fmaf(a, b.x, acc.x);
        acc.y = fmaf(a, b.y, acc.y);
        acc.z = fmaf(a, b.z, acc.z);
        acc.w = fmaf(a, b.w, acc.w);
    }
    return acc;
}

__global__ void __launch_bounds__(fs::kThreads, 2)
    factors_tc_kernel(const __grid_constant__ FactorMaps maps, uint8_t* __restrict__ ws, int Hk, int Hv, int NC,
                      long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + fs::BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + fs::BAR + 16);
    int* flag = reinterpret_cast<int*>(sm + fs::BAR + 20);
    float* s_anc = reinterpret_cast<float*>(sm + fs::CST);
    float* s_ea = s_anc + 128;
    float* s_ela = s_anc + 256;
    float* s_gs = reinterpret_cast<float*>(sm + fs::SGS);  // [16 token groups][128 channels]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, bh = blockIdx.y;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    const int unit_idx = bh * NC + n;
    uint8_t* unit = ws + static_cast<size_t>(unit_idx) * kWsUnit;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        mbar_arrive_expect_tx(bar_tma, 4 * 16384);
        const int t0 = n * kC;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_4d(sm + fs::A1 + kb * 16384 + 8192, &maps.q, 64 * kb, hk, t0, bi, bar_tma);
            tma_load_4d(sm + fs::A1 + kb * 16384, &maps.b, 64 * kb, hv, t0, bi, bar_tma);
            tma_load_4d(sm + fs::K + kb * 8192, &maps.k, 64 * kb, hk, t0, bi, bar_tma);
            tma_load_4d(sm + fs::G + kb * 8192, &maps.g, 64 * kb, hv, t0, bi, bar_tma);
        }
    }
    bool ok = cta_wait(bar_tma, 0, wait_ns, flag);
    if (ok) {
        // ---- elementwise pass. Thread = (channel chunk j: 8 channels, token group tg: 4 tokens);
        //      every shared-memory access is one 16-byte chunk of a 128-byte swizzled row.
        const int j = tid & 15, tg = tid >> 4;
        const int kb = j >> 3, cj = j & 7;
        uint8_t* pB = sm + fs::A1 + kb * 16384;
        uint8_t* pQ = pB + 8192;
        uint8_t* pK = sm + fs::K + kb * 8192;
        uint8_t* pG = sm + fs::G + kb * 8192;
        auto off = [&](int t) { return t * 128 + ((cj ^ (t & 7)) << 4); };
        float L[4][8];  // inclusive prefix of g within the token group
        {
            float x[8];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                unpack8(*reinterpret_cast<const uint4*>(pG + off(4 * tg + r)), x);
#pragma unroll
                for (int i = 0; i < 8; ++i) L[r][i] = (r ? L[r - 1][i] : 0.f) + x[i];
            }
            float4* dst = reinterpret_cast<float4*>(s_gs + tg * 128 + 8 * j);
            dst[0] = make_float4(L[3][0], L[3][1], L[3][2], L[3][3]);
            dst[1] = make_float4(L[3][4], L[3][5], L[3][6], L[3][7]);
        }
        __syncthreads();
        if (tid < 128) {  // exclusive prefix over the 16 token groups, per channel
            const int c = tid;
            float run = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float x = s_gs[q * 128 + c];
                s_gs[q * 128 + c] = run;
                run += x;
            }
            const float g0 = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16*>(sm + fs::G + (c >> 6) * 8192 + sw128_off(0, c & 63)));
            const float a = 0.5f * (g0 + run);  // G_0 and G_last bracket G when log-decays are <= 0
            s_anc[c] = a;
            s_ea[c] = __expf(a);
            s_ela[c] = __expf(run - a);
            reinterpret_cast<float*>(unit + kWsGam)[c] = __expf(run);
        }
        __syncthreads();
        {
            float pre[8], anc[8], ea[8], ela[8];
            {
                const float4* p4 = reinterpret_cast<const float4*>(s_gs + tg * 128 + 8 * j);
                const float4* a4 = reinterpret_cast<const float4*>(s_anc + 8 * j);
                const float4* e4 = reinterpret_cast<const float4*>(s_ea + 8 * j);
                const float4* l4 = reinterpret_cast<const float4*>(s_ela + 8 * j);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 pp = p4[h], aa = a4[h], ee = e4[h], ll = l4[h];
                    pre[4 * h] = pp.x; pre[4 * h + 1] = pp.y; pre[4 * h + 2] = pp.z; pre[4 * h + 3] = pp.w;
                    anc[4 * h] = aa.x; anc[4 * h + 1] = aa.y; anc[4 * h + 2] = aa.z; anc[4 * h + 3] = aa.w;
                    ea[4 * h] = ee.x; ea[4 * h + 1] = ee.y; ea[4 * h + 2] = ee.z; ea[4 * h + 3] = ee.w;
                    ela[4 * h] = ll.x; ela[4 * h + 1] = ll.y; ela[4 * h + 2] = ll.z; ela[4 * h + 3] = ll.w;
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * tg + r;
                const int o = off(t);
                float kk[8], qq[8], bb[8];
                unpack8(*reinterpret_cast<const uint4*>(pK + o), kk);
                unpack8(*reinterpret_cast<const uint4*>(pQ + o), qq);
                unpack8(*reinterpret_cast<const uint4*>(pB + o), bb);
                float o_kb[8], o_qa[8], o_kt[8], o_kg[8], qb[8], kh[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float Gi = pre[i] + L[r][i];
                    const float e1 = __expf(Gi - anc[i]);   // e^{G - a}
                    const float e2 = __expf(anc[i] - Gi);   // e^{a - G}
                    const float bk = bb[i] * kk[i];
                    o_kb[i] = bk * e1;
                    o_qa[i] = qq[i] * e1;
                    o_kt[i] = kk[i] * e2;
                    o_kg[i] = bk * (e1 * ea[i]);            // b.k.e^{G}
                    qb[i] = qq[i] * (e1 * ea[i]);            // q.e^{G}
                    kh[i] = kk[i] * (e2 * ela[i]);           // k.e^{G_last - G}
                }
                *reinterpret_cast<uint4*>(pB + o) = pack8(o_kb);
                *reinterpret_cast<uint4*>(pQ + o) = pack8(o_qa);
                *reinterpret_cast<uint4*>(pK + o) = pack8(o_kt);
                *reinterpret_cast<uint4*>(pG + o) = pack8(o_kg);   // in place of g (same thread, same chunk)
                // decayed q and k, token-major rows of 256 bytes: one 16-byte chunk per thread
                *reinterpret_cast<uint4*>(unit + kWsQb + t * 256 + j * 16) = pack8(qb);
                *reinterpret_cast<uint4*>(unit + kWsKh + t * 256 + j * 16) = pack8(kh);
            }
        }
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
        // T scratch starts at zero: the blocked solve below relies on its strictly upper blocks being 0
        for (int p = tid; p < 64 * fs::LDF / 4; p += fs::kThreads)
            reinterpret_cast<float4*>(TF)[p] = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            // warp w reads lanes 32(w%4).. and columns 32(w/4)..+31
            const int q4 = warp & 3, half = warp >> 2;
            float x[32];
            tmem_ld_cols<2>(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 32 * half, x);
            if (q4 < 2) {  // A rows, strictly lower
                const int i = 32 * q4 + lane;
                float4* dst = reinterpret_cast<float4*>(AF + i * fs::LDF + 32 * half);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) y[e] = (32 * half + 4 * c4 + e < i) ? x[4 * c4 + e] : 0.f;
                    dst[c4] = make_float4(y[0], y[1], y[2], y[3]);
                }
            } else {       // M rows, lower incl. diagonal, staged (128-byte swizzle) for a TMA store
                const int i = 32 * (q4 - 2) + lane;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] = (32 * half + 8 * c8 + e <= i) ? x[8 * c8 + e] : 0.f;
                    *reinterpret_cast<uint4*>(sm + fs::SGS + i * 128 + (((4 * half + c8) ^ (i & 7)) << 4)) = pack8(y);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&maps.m_st, sm + fs::SGS, 0, 0, unit_idx);
            bulk_commit();
        }
        // ---- T = (I + A)^{-1}, blocked: (1) the four 16x16 diagonal blocks by forward substitution
        //      (warps 0-3, one column per lane); (2) the two 16x16 blocks below them inside each
        //      32x32 diagonal block, T_{i+1,i} = -D_{i+1} A_{i+1,i} D_i; (3) the 32x32 block below
        //      the diagonal, T_10 = -T_11 A_10 T_00.
        if (warp < 4 && lane < 16) {
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
        if (tid < 128) {  // Y_i = A_{i+1,i} D_i for diagonal blocks i = 0, 2 (16 x 16 each, 4 columns per thread)
            const int blk = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
            const int i0 = 32 * blk;
            const float4 y = row_times<16>(AF + (i0 + 16 + r) * fs::LDF + i0, TF + i0 * fs::LDF + i0, fs::LDF, c4);
            *reinterpret_cast<float4*>(PF + (blk * 16 + r) * fs::LDP + c4) = y;
        }
        __syncthreads();
        if (tid < 128) {  // T_{i+1,i} = -D_{i+1} Y_i
            const int blk = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
            const int i1 = 32 * blk + 16;
            const float4 y = row_times<16>(TF + (i1 + r) * fs::LDF + i1, PF + (blk * 16) * fs::LDP, fs::LDP, c4);
            *reinterpret_cast<float4*>(TF + (i1 + r) * fs::LDF + i1 - 16 + c4) = make_float4(-y.x, -y.y, -y.z, -y.w);
        }
        __syncthreads();
        {  // X = A_10 T_00 (32 x 32; rows 32.., cols 0..31), one float4 per thread
            const int r = tid >> 3, c4 = (tid & 7) * 4;
            const float4 y = row_times<32>(AF + (32 + r) * fs::LDF, TF, fs::LDF, c4);
            *reinterpret_cast<float4*>(PF + r * fs::LDP + c4) = y;
        }
        __syncthreads();
        {  // T_10 = -T_11 X
            const int r = tid >> 3, c4 = (tid & 7) * 4;
            const float4 y = row_times<32>(TF + (32 + r) * fs::LDF + 32, PF, fs::LDP, c4);
            *reinterpret_cast<float4*>(TF + (32 + r) * fs::LDF + c4) = make_float4(-y.x, -y.y, -y.z, -y.w);
        }
        __syncthreads();
        for (int p = tid; p < 64 * 8; p += fs::kThreads) {  // bf16 T, K-major rows (one 16-byte chunk per item)
            const int i = p >> 3, c8 = p & 7;
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int jc = 8 * c8 + e;
                y[e] = (jc <= i) ? TF[i * fs::LDF + jc] : 0.f;
            }
            *reinterpret_cast<uint4*>(sm + fs::TB + i * 128 + ((c8 ^ (i & 7)) << 4)) = pack8(y);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- W = T (b.k.e^G), token-major, as rows 0..63 of [T ; X] (b.k.e^G)   (M = 128, N = 128, K = 64)
        if (tid == 0) {
            tma_store_3d(&maps.t_st, sm + fs::TB, 0, 0, unit_idx);
            bulk_commit();
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16(128, 128, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = smem_desc(sbase + fs::TB + s * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + fs::G + s * 2048, 8192, 1024, kSwizzle128B);
                mma_bf16(tmem, ad, bd, id, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, 1, wait_ns, flag);
        if (ok) {
            tc_fence_after();
            const int q4 = warp & 3, half = warp >> 2;
            if (q4 < 2) {  // token t = lane row; this thread's 64 channels -> swizzled W staging tile `half`
                const int t = 32 * q4 + lane;
                float x[64];
                tmem_ld_cols<4>(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 * half, x);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] = x[8 * c8 + e];
                    *reinterpret_cast<uint4*>(sm + fs::WSTG + half * 8192 + t * 128 + ((c8 ^ (t & 7)) << 4)) = pack8(y);
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_3d(&maps.w_st, sm + fs::WSTG, 0, 0, unit_idx);
                tma_store_3d(&maps.w_st, sm + fs::WSTG + 8192, 64, 0, unit_idx);
                bulk_commit();
            }
        }
    }
    if (tid == 0) bulk_wait_read_all();  // staging must be read out before the CTA releases its memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------------------------
// kernel 2: state chain + output

struct StateMaps {
    CUtensorMap w, qb, kh, m, t;   // workspace sections
    CUtensorMap v, wg;             // token tiles of v and of the write gate w
};

namespace ss {
// one pipeline stage (offsets inside the stage; every tile 1024-byte aligned)
constexpr uint32_t A1 = 0;          // [W ; Q]: two 64-wide K blocks of [128 rows][128 B], K-major
constexpr uint32_t KH = 32768;      // k.e^{G_last-G} token-major: MN-major A operand of K^^T (2 blocks)
constexpr uint32_t MM = 49152;      // M [64][64] K-major; as [X ; M] its first 64 rows are KH's 2nd block
constexpr uint32_t TT = 57344;      // T [64][64] K-major; as [T ; 0] it is followed by ...
constexpr uint32_t ZZ = 65536;      // ... 64 rows of zeros (written once)
constexpr uint32_t VV = 73728;      // v slice [64 tokens][64 columns] (128-byte swizzle)
constexpr uint32_t WW = 81920;      // w slice
constexpr uint32_t GAM = 90112;     // e^{G_last} fp32 [128]
constexpr uint32_t STAGE = 91136;
constexpr uint32_t TX = 3 * 16384 + 4 * 8192 + 512;   // bytes delivered per stage
constexpr uint32_t SBF = 2 * STAGE;         // S_n bf16 [128 rows d_k][64], MN-major B operand
constexpr uint32_t UBF = SBF + 16384;       // U bf16 [64 tokens][64], MN-major B operand
constexpr uint32_t WV = UBF + 8192;         // w.v bf16 [64 tokens][64], MN-major B operand
constexpr uint32_t BAR = WV + 8192;         // full[2], mma, TMEM base, 3 flags
constexpr uint32_t TOTAL = BAR + 64;
constexpr int kThreads = 256;
// TMEM columns: D1 (rows 0-63: U = T(w.v) - W S_n; rows 64-127: -(Q S_n + M U)) double-buffered at
// 0 and 128; D2 = K^^T U at 64.
__host__ __device__ constexpr uint32_t d1_col(int n) { return (n & 1) ? 128u : 0u; }
constexpr uint32_t kD2 = 64;
}  // namespace ss

// Write 32 values as half `half` (16-byte chunks 4*half .. 4*half+3) of 128-byte swizzled row `row`.
__device__ __forceinline__ void store_halfrow_sw128(uint8_t* tile, int row, int half, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = x[8 * c + e];
        *reinterpret_cast<uint4*>(tile + row * 128 + (((4 * half + c) ^ (row & 7)) << 4)) = pack8(y);
    }
}

__global__ void __launch_bounds__(ss::kThreads, 1)
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

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, half = warp >> 2;  // TMEM lane quarter, column half
    const int bh = blockIdx.x, z = blockIdx.y;
    const int bi = bh / Hv, hv = bh - bi * Hv;
    const int r = 32 * q4 + lane;  // d_k row of the state (= TMEM lane) owned by this thread
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;

    if (tid == 0) {
        mbar_init(full, 1);
        mbar_init(full + 1, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    for (int p = tid; p < 2 * 512; p += ss::kThreads) {  // the zero rows under T, both stages
        const int st = p >> 9, q16 = p & 511;
        reinterpret_cast<uint4*>(sm + st * ss::STAGE + ss::ZZ)[q16] = make_uint4(0, 0, 0, 0);
    }
    float S[32];  // S_n[r][32*half + j], fp32
    {
        const float* src = s0 ? s0 + (static_cast<size_t>(bh) * kD + r) * kD + z * kSlice + 32 * half : nullptr;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 t4 = src ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = t4.x;
            S[j + 1] = t4.y;
            S[j + 2] = t4.z;
            S[j + 3] = t4.w;
        }
        store_halfrow_sw128(sm + ss::SBF, r, half, S);
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
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            tma_load_3d(sb + ss::A1 + kb * 16384, &maps.w, 64 * kb, 0, u, full + st);
            tma_load_3d(sb + ss::A1 + kb * 16384 + 8192, &maps.qb, 64 * kb, 0, u, full + st);
            tma_load_3d(sb + ss::KH + kb * 8192, &maps.kh, 64 * kb, 0, u, full + st);
        }
        tma_load_3d(sb + ss::MM, &maps.m, 0, 0, u, full + st);
        tma_load_3d(sb + ss::TT, &maps.t, 0, 0, u, full + st);
        tma_load_4d(sb + ss::VV, &maps.v, z * kSlice, hv, n * kC, bi, full + st);
        tma_load_4d(sb + ss::WW, &maps.wg, z * kSlice, hv, n * kC, bi, full + st);
        bulk_load(sb + ss::GAM, ws + static_cast<size_t>(u) * kWsUnit + kWsGam, 512, full + st);
    };
    // O rows of chunk m (tokens 64m..64m+63): the D1 rows 64..127 it was accumulated in hold -O
    auto emit_o = [&](int m) {
        if (q4 < 2) return;
        const int i = 32 * (q4 - 2) + lane;
        const int tok = m * kC + i;
        float x[32];
        tmem_ld_cols<2>(tmem + lane_base + ss::d1_col(m) + 32 * half, x);
        if (tok < T) {
            uint4* dst = reinterpret_cast<uint4*>(o + ((static_cast<size_t>(bi) * T + tok) * Hv + hv) * kD +
                                                  z * kSlice + 32 * half);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = -scale * x[8 * c + e];
                dst[c] = pack8(y);
            }
        }
    };
    if (tid == 0 && NC > 0) issue(0);

    uint32_t mma_phase = 0;
    bool ok = true;
    int n = 0;
    for (; n < NC && ok; ++n) {
        const int st = n & 1;
        uint8_t* sbp = sm + st * ss::STAGE;
        const uint32_t sb = sbase + st * ss::STAGE;
        const uint32_t d1 = tmem + ss::d1_col(n);
        if (tid == 0 && n + 1 < NC) issue(n + 1);
        ok = cta_wait(full + st, (n >> 1) & 1, wait_ns, flag + 0);
        if (!ok) break;
        {  // w.v for this chunk's 64 x 64 slice: two 16-byte chunks per thread, same swizzled positions
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int item = tid + 256 * h2;  // 512 chunks = 64 rows x 8 chunks
                const uint32_t off = (item >> 3) * 128 + ((item & 7) << 4);
                float a[8], bw[8];
                unpack8(*reinterpret_cast<const uint4*>(sbp + ss::VV + off), a);
                unpack8(*reinterpret_cast<const uint4*>(sbp + ss::WW + off), bw);
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] *= bw[e];
                *reinterpret_cast<uint4*>(sm + ss::WV + off) = pack8(a);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- D1 = [T ; 0] (w.v)  then  D1 -= [W ; Q] S_n          (M = 128, N = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id0 = idesc_bf16(128, 64, false, true);
            constexpr uint32_t id1 = idesc_bf16(128, 64, false, true) | kNegateA;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = smem_desc(sb + ss::TT + s * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + ss::WV + s * 2048, 8192, 1024, kSwizzle128B);
                mma_bf16(d1, ad, bd, id0, s > 0);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t ad = smem_desc(sb + ss::A1 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSwizzle128B);
                const uint64_t bd = smem_desc(sbase + ss::SBF + s * 2048, 16384, 1024, kSwizzle128B);
                mma_bf16(d1, ad, bd, id1, 1);
            }
            mma_commit(bar_mma);
        }
        if (n > 0) emit_o(n - 1);  // previous chunk's output, overlapping these MMAs
        ok = cta_wait(bar_mma, mma_phase, wait_ns, flag + 1);
        mma_phase ^= 1;
        if (!ok) break;
        tc_fence_after();
        if (q4 < 2) {  // U rows = tokens 0..63, this thread's 32 columns
            float x[32];
            tmem_ld_cols<2>(d1 + lane_base + 32 * half, x);
            store_halfrow_sw128(sm + ss::UBF, r, half, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- D1 -= [X ; M] U (rows 0..63 are discarded)  and  D2 = K^^T U     (M = 128, N = 64, K = 64)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id2 = idesc_bf16(128, 64, false, true) | kNegateA;
            constexpr uint32_t id3 = idesc_bf16(128, 64, true, true);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bd = smem_desc(sbase + ss::UBF + s * 2048, 8192, 1024, kSwizzle128B);
                const uint64_t a2 = smem_desc(sb + ss::MM - 8192 + s * 32, 16, 1024, kSwizzle128B);
                const uint64_t a3 = smem_desc(sb + ss::KH + s * 2048, 8192, 1024, kSwizzle128B);
                mma_bf16(d1, a2, bd, id2, 1);
                mma_bf16(tmem + ss::kD2, a3, bd, id3, s > 0);
            }
            mma_commit(bar_mma);
        }
        ok = cta_wait(bar_mma, mma_phase, wait_ns, flag + 2);
        mma_phase ^= 1;
        if (!ok) break;
        tc_fence_after();
        {
            float x[32];
            tmem_ld_cols<2>(tmem + lane_base + ss::kD2 + 32 * half, x);
            const float gam = reinterpret_cast<const float*>(sbp + ss::GAM)[r];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) S[jj] = fmaf(gam, S[jj], x[jj]);
            store_halfrow_sw128(sm + ss::SBF, r, half, S);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    if (!ok) {
        // drain the prefetch of the next chunk if it was issued
        if (tid == 0 && n + 1 < NC) mbar_wait(full + ((n + 1) & 1), ((n + 1) >> 1) & 1, kDefaultWaitNs);
    } else {
        if (NC > 0) emit_o(NC - 1);
        if (sT_out) {
            float* dst = sT_out + (static_cast<size_t>(bh) * kD + r) * kD + z * kSlice + 32 * half;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
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
    const bool negate = (case_id == 4);  // case 4: case 0 with the A operand negated by the descriptor
    if (negate) case_id = 0;
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
            const uint32_t id = idesc_bf16(128, 64, a_mn, b_mn) | (negate ? kNegateA : 0u);
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

// workspace section viewed as (cols, rows, units); box (box_cols, box_rows, 1)
bool ws_map(CUtensorMap* m, const void* p, CUtensorMapDataType dt, int esize, int cols, int rows, int units,
            int box_cols, int box_rows, CUtensorMapSwizzle sw) {
    const uint64_t dims[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)units};
    const uint64_t st[2] = {(uint64_t)cols * esize, kWsUnit};
    const uint32_t box[3] = {(uint32_t)box_cols, (uint32_t)box_rows, 1};
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
    const int units = NC * sh.B * sh.Hv;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
    FactorMaps fm;
    if (!token_map(&fm.q, q, sh.B, sh.T, sh.Hk) || !token_map(&fm.k, k, sh.B, sh.T, sh.Hk) ||
        !token_map(&fm.g, g, sh.B, sh.T, sh.Hv) || !token_map(&fm.b, b, sh.B, sh.T, sh.Hv) ||
        !ws_map(&fm.m_st, wsb + kWsM, BF, 2, 64, 64, units, 64, 64, SW) ||
        !ws_map(&fm.t_st, wsb + kWsT, BF, 2, 64, 64, units, 64, 64, SW) ||
        !ws_map(&fm.w_st, wsb + kWsW, BF, 2, 128, 64, units, 64, 64, SW))
        return cudaErrorInvalidValue;
    StateMaps sm_;
    if (!ws_map(&sm_.w, wsb + kWsW, BF, 2, 128, 64, units, 64, 64, SW) ||
        !ws_map(&sm_.qb, wsb + kWsQb, BF, 2, 128, 64, units, 64, 64, SW) ||
        !ws_map(&sm_.kh, wsb + kWsKh, BF, 2, 128, 64, units, 64, 64, SW) ||
        !ws_map(&sm_.m, wsb + kWsM, BF, 2, 64, 64, units, 64, 64, SW) ||
        !ws_map(&sm_.t, wsb + kWsT, BF, 2, 64, 64, units, 64, 64, SW) ||
        !token_map(&sm_.v, v, sh.B, sh.T, sh.Hv) || !token_map(&sm_.wg, w, sh.B, sh.T, sh.Hv))
        return cudaErrorInvalidValue;

    // The state kernel runs one CTA per SM, so it takes the whole 227 KB: operand descriptors can
    // then never reach past the CTA's own allocation.
    const size_t f_smem = fs::TOTAL + 1024, s_smem = 232448;
    static_assert(ss::TOTAL + 1024 <= 232448, "state kernel shared memory");
    cudaError_t e = cudaFuncSetAttribute(factors_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    factors_tc_kernel<<<dim3(NC, sh.B * sh.Hv), fs::kThreads, f_smem, s>>>(fm, wsb, sh.Hk, sh.Hv, NC, wait_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    state_tc_kernel<<<dim3(sh.B * sh.Hv, kD / kSlice), ss::kThreads, s_smem, s>>>(
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
    static const int shp[5][4] = {{128, 128, 64, 128}, {64, 128, 64, 64}, {128, 128, 128, 64}, {128, 64, 64, 64},
                                  {128, 128, 64, 128}};
    if (case_id < 0 || case_id > 4) return cudaErrorInvalidValue;
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

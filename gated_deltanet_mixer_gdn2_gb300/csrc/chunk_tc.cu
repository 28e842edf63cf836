// chunk_tc.cu -- chunked forward on the 5th-generation tensor cores (tcgen05 + TMA + TMEM), bf16
// inputs, d_k = 128, d_v a multiple of 64 (up to 512), chunk C = 64.
//
// Same chunked WY / UT form as the SIMT path (burn-gdn2 0.1.5 docs: "chunked WY decomposition
// (training)"); per chunk of C tokens entering with state S_n, G_i = inclusive cumulative
// log-decay of the chunk per key channel:
//     A = tril_{-1}(K_bar K_til^T),  M = tril_0(Q_anc K_til^T)           [one M=128 MMA, stacked]
//         with K_bar = b.k.e^{G-a}, Q_anc = q.e^{G-a}, K_til = k.e^{a-G} and a per-channel anchor
//         a = (G_0 + G_last)/2, so that every factor stays within e^{+-range/2}
//     T = (I + A)^{-1}                                                   [fp32, blocked forward substitution]
//     W = T (b.k.e^{G})                                                  [M=128 MMA]
//     U = T (w.v) - W S_n;  O = (q.e^{G}) S_n + M U;  S_{n+1} = e^{G_last} . S_n + (k.e^{G_last-G})^T U
//
// Kernel 1 "factors" (grid: chunks x heads; 256 threads; 3 CTAs/SM): TMA loads q, k, g, b of one
// chunk, one pass computes the decayed operands, tcgen05 forms A|M, CUDA cores invert (I + A),
// tcgen05 forms W; -W, q.e^G, k.e^{G_last-G}, M, T and e^{G_last} go to the workspace.
// The gates are floored at kGateFloor (alpha = e^{-100}: a full reset, g = -inf, stays finite). A
// chunk in which some channel's log-decay spans more than kSpanAnchored cannot use one anchor per
// channel (its factors would leave bf16's range): kernel 1 lists it and kernel 1b "exact" forms that
// unit on CUDA cores with one factor e^{G_i - G_j} <= 1 per entry, so the whole domain alpha in
// [0, 1] is covered.
// Kernel 2 "state" (grid: 2 x batch x value heads; warp-specialised; sequential over chunks): the
// columns of S evolve independently, so each CTA runs the recurrence for 64 of the d_v columns with
// the fp32 state in registers, 128-row products over tokens or d_k, and the bf16 state and U as
// shared-memory operands.
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace gdn2 {

namespace {



// Largest per-channel span G_0 - G_last of the (floored) cumulative log-decay within one chunk that
// the anchored operands take: every factor then lies in [e^-60, e^60], far inside bf16's range
// (operands down to |x| ~ 1e-12 keep their value after the e^-60 scaling). Wider chunks go to the
// exact kernel.
constexpr float kSpanAnchored = 120.f;


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
constexpr uint32_t BAR = 73728;   // 2 mbarriers, TMEM base
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

// acc[i][c] += sum_{k = 4 g0}^{4 g1 - 1} L[i][k] R[k][c] for a 2 x 4 register tile (fp32 smem, 16-byte
// aligned rows ldl / ldr floats apart); k runs upwards, one FMA per term.
__device__ __forceinline__ void tile24_times(const float* L, int ldl, const float* R, int ldr, int g0, int g1,
                                             float (&acc)[2][4]) {
#pragma unroll 2
    for (int g = g0; g < g1; ++g) {
        float4 l[2], r[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) l[i] = *reinterpret_cast<const float4*>(L + i * ldl + 4 * g);
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = *reinterpret_cast<const float4*>(R + (4 * g + j) * ldr);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float a[4] = {l[i].x, l[i].y, l[i].z, l[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][0] = fmaf(a[j], r[j].x, acc[i][0]);
                acc[i][1] = fmaf(a[j], r[j].y, acc[i][1]);
                acc[i][2] = fmaf(a[j], r[j].z, acc[i][2]);
                acc[i][3] = fmaf(a[j], r[j].w, acc[i][3]);
            }
        }
    }
}
__device__ __forceinline__ void tile24_store(float* D, int ldd, const float (&acc)[2][4], float sgn) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
        *reinterpret_cast<float4*>(D + i * ldd) = make_float4(sgn * acc[i][0], sgn * acc[i][1], sgn * acc[i][2], sgn * acc[i][3]);
}

// T = (I + A)^{-1} for a strictly lower triangular 64 x 64 A (fp32 shared memory, rows LDF floats
// apart; T's scratch must hold zeros above its diagonal blocks on entry), by blocks: (1) the four
// 16x16 diagonal blocks by forward substitution (warps 0-3, one column per lane); (2) the two 16x16
// blocks below them inside each 32x32 diagonal block, T_{i+1,i} = -D_{i+1} A_{i+1,i} D_i; (3) the
// 32x32 block below the diagonal, T_10 = -T_11 A_10 T_00. Called by all 256 threads of the block;
// PF is a [32][LDP] fp32 scratch.
__device__ __forceinline__ void invert_unit_lower64(const float* AF, float* TF, float* PF, int warp, int lane) {
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
    // Products below run as 2 x 4 register tiles (each 16-byte load feeds 8 FMAs; 64 or 128 threads
    // share a product, which measured faster than 4 x 4 tiles on fewer threads or 1 x 4 on all 8
    // warps). A skipped k-range multiplies entries of a lower triangular factor that are exactly
    // zero, so bounds stay warp-uniform and the sums are unchanged.
    if (warp < 2) {  // Y_i = A_{i+1,i} D_i for diagonal blocks i = 0, 2 (warp = block, 2 x 4 tiles)
        const int i0 = 32 * warp, r0 = 2 * (lane >> 2), c0 = 4 * (lane & 3);
        float acc[2][4] = {};
        tile24_times(AF + (i0 + 16 + r0) * fs::LDF + i0, fs::LDF, TF + i0 * fs::LDF + i0 + c0, fs::LDF, 0, 4, acc);
        tile24_store(PF + (16 * warp + r0) * fs::LDP + c0, fs::LDP, acc, 1.f);
    }
    __syncthreads();
    if (warp < 2) {  // T_{i+1,i} = -D_{i+1} Y_i
        const int i1 = 32 * warp + 16, r0 = 2 * (lane >> 2), c0 = 4 * (lane & 3);
        float acc[2][4] = {};
        tile24_times(TF + (i1 + r0) * fs::LDF + i1, fs::LDF, PF + 16 * warp * fs::LDP + c0, fs::LDP, 0, 4, acc);
        tile24_store(TF + (i1 + r0) * fs::LDF + i1 - 16 + c0, fs::LDF, acc, -1.f);
    }
    __syncthreads();
    if (warp < 4) {  // X = A_10 T_00: warp w takes columns 8w.. (2 x 4 tiles)
        const int r0 = 2 * (lane >> 1), c0 = 8 * warp + 4 * (lane & 1);
        float acc[2][4] = {};
        tile24_times(AF + (32 + r0) * fs::LDF, fs::LDF, TF + c0, fs::LDF, 2 * warp, 8, acc);
        tile24_store(PF + r0 * fs::LDP + c0, fs::LDP, acc, 1.f);
    }
    __syncthreads();
    if (warp < 4) {  // T_10 = -T_11 X: warp w takes rows 8w.. (2 x 4 tiles)
        const int r0 = 8 * warp + 2 * (lane >> 3), c0 = 4 * (lane & 7);
        float acc[2][4] = {};
        tile24_times(TF + (32 + r0) * fs::LDF + 32, fs::LDF, PF + c0, fs::LDP, 0, 2 * (warp + 1), acc);
        tile24_store(TF + (32 + r0) * fs::LDF + c0, fs::LDF, acc, -1.f);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(fs::kThreads, 3)
    factors_tc_kernel(const __grid_constant__ FactorMaps maps, uint8_t* __restrict__ ws, int* __restrict__ exact_list,
                      int Hk, int Hv, int NC, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + fs::BAR);
    uint64_t* bar_mma = bar_tma + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + fs::BAR + 16);
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
    bool ok = cta_wait(bar_tma, 0, wait_ns);
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
                for (int i = 0; i < 8; ++i) L[r][i] = (r ? L[r - 1][i] : 0.f) + fmaxf(x[i], kGateFloor);
            }
            float4* dst = reinterpret_cast<float4*>(s_gs + tg * 128 + 8 * j);
            dst[0] = make_float4(L[3][0], L[3][1], L[3][2], L[3][3]);
            dst[1] = make_float4(L[3][4], L[3][5], L[3][6], L[3][7]);
        }
        __syncthreads();
        bool wide = false;  // this channel's log-decay spans more than the anchored form can hold
        if (tid < 128) {  // exclusive prefix over the 16 token groups, per channel
            const int c = tid;
            float part[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) part[q] = s_gs[q * 128 + c];  // all loads first
            float run = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                s_gs[q * 128 + c] = run;
                run += part[q];
            }
            const float g0 = fmaxf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                       sm + fs::G + (c >> 6) * 8192 + sw128_off(0, c & 63))),
                                   kGateFloor);
            const float a = 0.5f * (g0 + run);  // G_0 and G_last bracket G when log-decays are <= 0
            wide = g0 - run > kSpanAnchored;
            s_anc[c] = a;
            s_ea[c] = __expf(a);
            s_ela[c] = __expf(run - a);
            reinterpret_cast<float*>(unit + kWsGam)[c] = __expf(run);
        }
        // A channel whose log-decay spans more than kSpanAnchored would need factors beyond
        // e^{+-kSpanAnchored/2}: the exact kernel forms this unit instead (it is listed and skipped).
        const bool exact = __syncthreads_or(wide) != 0;
        if (exact && tid == 0) exact_list[1 + atomicAdd(exact_list, 1)] = unit_idx;
        if (exact) ok = false;
        if (!exact) {
        {
            // per channel: (G_{group start} - a) log2(e), e^{a}, e^{G_last - a}, as channel pairs
            uint64_t pa2[4], ea2[4], ela2[4];
            {
                const float4* p4 = reinterpret_cast<const float4*>(s_gs + tg * 128 + 8 * j);
                const float4* a4 = reinterpret_cast<const float4*>(s_anc + 8 * j);
                const float4* e4 = reinterpret_cast<const float4*>(s_ea + 8 * j);
                const float4* l4 = reinterpret_cast<const float4*>(s_ela + 8 * j);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 pp = p4[h], aa = a4[h], ee = e4[h], ll = l4[h];
                    pa2[2 * h] = f32x2((pp.x - aa.x) * kLog2e, (pp.y - aa.y) * kLog2e);
                    pa2[2 * h + 1] = f32x2((pp.z - aa.z) * kLog2e, (pp.w - aa.w) * kLog2e);
                    ea2[2 * h] = f32x2(ee.x, ee.y);
                    ea2[2 * h + 1] = f32x2(ee.z, ee.w);
                    ela2[2 * h] = f32x2(ll.x, ll.y);
                    ela2[2 * h + 1] = f32x2(ll.z, ll.w);
                }
            }
            const uint64_t log2e2 = f32x2(kLog2e, kLog2e);
            // each output is formed and stored before the next one, so that few values are live;
            // products run on channel pairs (packed fp32x2), bf16 inputs widen by shifts
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * tg + r;
                const int o = off(t);
                uint64_t e1[4], e2[4], kk[4], bk[4];
                uint32_t y[4];
                {
                    const uint4 ku = *reinterpret_cast<const uint4*>(pK + o);
                    const uint4 bu = *reinterpret_cast<const uint4*>(pB + o);
                    const uint32_t kw[4] = {ku.x, ku.y, ku.z, ku.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        // (G - a) log2(e) for channels 2i, 2i+1 of this token
                        const uint64_t d = fma_f32x2(f32x2(L[r][2 * i], L[r][2 * i + 1]), log2e2, pa2[i]);
                        float d0, d1;
                        f32x2_split(d, d0, d1);
                        e1[i] = f32x2(ex2_approx(d0), ex2_approx(d1));      // e^{G - a}
                        e2[i] = f32x2(ex2_approx(-d0), ex2_approx(-d1));    // e^{a - G}
                        kk[i] = bf16x2_widen(kw[i]);
                        bk[i] = mul_f32x2(bf16x2_widen(bw[i]), kk[i]);      // b.k
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint64_t kb_ = mul_f32x2(bk[i], e1[i]);       // b.k.e^{G-a}
                        y[i] = bf16x2_narrow(kb_);
                        bk[i] = mul_f32x2(kb_, ea2[i]);                     // b.k.e^{G}
                    }
                    *reinterpret_cast<uint4*>(pB + o) = make_uint4(y[0], y[1], y[2], y[3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] = bf16x2_narrow(bk[i]);
                    *reinterpret_cast<uint4*>(pG + o) = make_uint4(y[0], y[1], y[2], y[3]);  // in place of g
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kk[i] = mul_f32x2(kk[i], e2[i]);                        // k.e^{a-G}
                    y[i] = bf16x2_narrow(kk[i]);
                }
                *reinterpret_cast<uint4*>(pK + o) = make_uint4(y[0], y[1], y[2], y[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = bf16x2_narrow(mul_f32x2(kk[i], ela2[i]));  // k.e^{G_last - G}
                *reinterpret_cast<uint4*>(unit + kWsKh + t * 256 + j * 16) = make_uint4(y[0], y[1], y[2], y[3]);
                {
                    const uint4 qu = *reinterpret_cast<const uint4*>(pQ + o);
                    const uint32_t qw[4] = {qu.x, qu.y, qu.z, qu.w};
                    uint64_t qq[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qq[i] = mul_f32x2(bf16x2_widen(qw[i]), e1[i]);      // q.e^{G-a}
                        y[i] = bf16x2_narrow(qq[i]);
                    }
                    *reinterpret_cast<uint4*>(pQ + o) = make_uint4(y[0], y[1], y[2], y[3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] = bf16x2_narrow(mul_f32x2(qq[i], ea2[i]));  // q.e^{G}
                    // decayed q and k, token-major rows of 256 bytes: one 16-byte chunk per thread
                    *reinterpret_cast<uint4*>(unit + kWsQb + t * 256 + j * 16) = make_uint4(y[0], y[1], y[2], y[3]);
                }
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
        ok = cta_wait(bar_mma, 0, wait_ns);
        }
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
        invert_unit_lower64(AF, TF, PF, warp, lane);
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
        ok = cta_wait(bar_mma, 1, wait_ns);
        if (ok) {
            tc_fence_after();
            const int q4 = warp & 3, half = warp >> 2;
            if (q4 < 2) {  // token t = lane row; this thread's 64 channels -> swizzled W staging tile `half`
                const int t = 32 * q4 + lane;
#pragma unroll
                for (int c0 = 0; c0 < 2; ++c0) {
                    float x[32];
                    tmem_ld_cols<2>(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 * half + 32 * c0, x);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c8 = 4 * c0 + c4;
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = -x[8 * c4 + e];  // stored negated
                        *reinterpret_cast<uint4*>(sm + fs::WSTG + half * 8192 + t * 128 + ((c8 ^ (t & 7)) << 4)) = pack8(y);
                    }
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
// kernel 1b: exact factors of the units whose decay spans more than the anchored form holds
//
// Same outputs as the factor kernel (the workspace unit: -W, q.e^G, k.e^{G_last-G}, M, T, e^{G_last}),
// formed in fp32 on CUDA cores without any anchor: every entry of A and M takes its own factor
// e^{G_i - G_j} (i >= j, at most 1), every other factor is e^{G} or e^{G_last - G} (at most 1), so
// nothing can overflow whatever the decay, and a full reset (g = -inf, floored at kGateFloor) gives
// factors that are exactly or negligibly 0. A persistent grid walks the list the factor kernel
// wrote (count, then unit indices).

namespace xs {  // shared memory of the exact kernel (fp32 unless noted)
constexpr int LD = 132;                           // token rows of 128 channels, padded
constexpr uint32_t G = 0;                         // [64][LD] inclusive cumulative log-decay (floored)
constexpr uint32_t BK = G + 64 * LD * 4;          // [64][LD] b.k, later b.k.e^G
constexpr uint32_t Q = BK + 64 * LD * 4;          // [64][LD] q
constexpr uint32_t K = Q + 64 * LD * 4;           // [64][LD] k
constexpr uint32_t AF = K + 64 * LD * 4;          // [64][LDF] A (strictly lower)
constexpr uint32_t MF = AF + 64 * fs::LDF * 4;    // [64][LDF] M (lower incl. the diagonal)
constexpr uint32_t TF = MF + 64 * fs::LDF * 4;    // [64][LDF] T
constexpr uint32_t PF = TF + 64 * fs::LDF * 4;    // [32][LDP] inverse scratch
constexpr uint32_t TOTAL = PF + 32 * fs::LDP * 4;
constexpr int kThreads = 256;
}  // namespace xs

__global__ void __launch_bounds__(xs::kThreads, 1)
    factors_exact_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                         const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* __restrict__ b,
                         uint8_t* __restrict__ ws, const int* __restrict__ exact_list, int T, int Hk, int Hv, int NC,
                         int dk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    float* sG = reinterpret_cast<float*>(sm + xs::G);
    float* sBK = reinterpret_cast<float*>(sm + xs::BK);
    float* sQ = reinterpret_cast<float*>(sm + xs::Q);
    float* sK = reinterpret_cast<float*>(sm + xs::K);
    float* AF = reinterpret_cast<float*>(sm + xs::AF);
    float* MF = reinterpret_cast<float*>(sm + xs::MF);
    float* TF = reinterpret_cast<float*>(sm + xs::TF);
    float* PF = reinterpret_cast<float*>(sm + xs::PF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int count = exact_list[0];

    for (int li = blockIdx.x; li < count; li += gridDim.x) {
        const int unit_idx = exact_list[1 + li];
        const int bh = unit_idx / NC, n = unit_idx - bh * NC;
        const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
        uint8_t* unit = ws + static_cast<size_t>(unit_idx) * kWsUnit;
        __syncthreads();  // the previous unit's shared-memory readers are done
        // token tiles (zeros past T), 8 channels per item
        for (int p = tid; p < 64 * 16; p += xs::kThreads) {
            const int t = p >> 4, c = 8 * (p & 15), tok = n * kC + t;
            float gg[8], bb[8], kk[8], qq[8];
            if (tok < T && c < dk) {  // channels past d_k (d_k = 64) are zero: they leave the state unchanged
                const size_t kq = ((static_cast<size_t>(bi) * T + tok) * Hk + hk) * dk + c;
                const size_t gb = ((static_cast<size_t>(bi) * T + tok) * Hv + hv) * dk + c;
                unpack8(*reinterpret_cast<const uint4*>(g + gb), gg);
                unpack8(*reinterpret_cast<const uint4*>(b + gb), bb);
                unpack8(*reinterpret_cast<const uint4*>(k + kq), kk);
                unpack8(*reinterpret_cast<const uint4*>(q + kq), qq);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) gg[i] = bb[i] = kk[i] = qq[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                sG[t * xs::LD + c + i] = fmaxf(gg[i], kGateFloor);
                sBK[t * xs::LD + c + i] = bb[i] * kk[i];
                sK[t * xs::LD + c + i] = kk[i];
                sQ[t * xs::LD + c + i] = qq[i];
            }
        }
        for (int p = tid; p < 64 * fs::LDF; p += xs::kThreads) {
            AF[p] = 0.f;
            MF[p] = 0.f;
            TF[p] = 0.f;
        }
        __syncthreads();
        if (tid < 128) {  // inclusive cumulative log-decay of channel tid, and e^{G_last}
            float run = 0.f;
            for (int t = 0; t < kC; ++t) {
                run += sG[t * xs::LD + tid];
                sG[t * xs::LD + tid] = run;
            }
            reinterpret_cast<float*>(unit + kWsGam)[tid] = __expf(run);
        }
        __syncthreads();
        // A (j < i) and M (j <= i): one thread per pair, pairs numbered along the lower triangle
        for (int p = tid; p < kC * (kC + 1) / 2; p += xs::kThreads) {
            int i = static_cast<int>((sqrtf(8.f * p + 1.f) - 1.f) * 0.5f);
            while ((i + 1) * (i + 2) / 2 <= p) ++i;
            while (i * (i + 1) / 2 > p) --i;
            const int j = p - i * (i + 1) / 2;
            const float4* gi = reinterpret_cast<const float4*>(sG + i * xs::LD);
            const float4* gj = reinterpret_cast<const float4*>(sG + j * xs::LD);
            const float4* bki = reinterpret_cast<const float4*>(sBK + i * xs::LD);
            const float4* qi = reinterpret_cast<const float4*>(sQ + i * xs::LD);
            const float4* kj = reinterpret_cast<const float4*>(sK + j * xs::LD);
            float a = 0.f, m = 0.f;
#pragma unroll 4
            for (int c4 = 0; c4 < 32; ++c4) {
                const float4 Gi = gi[c4], Gj = gj[c4], B4 = bki[c4], Q4 = qi[c4], K4 = kj[c4];
                const float f0 = K4.x * __expf(Gi.x - Gj.x), f1 = K4.y * __expf(Gi.y - Gj.y);
                const float f2 = K4.z * __expf(Gi.z - Gj.z), f3 = K4.w * __expf(Gi.w - Gj.w);
                a = fmaf(B4.x, f0, fmaf(B4.y, f1, fmaf(B4.z, f2, fmaf(B4.w, f3, a))));
                m = fmaf(Q4.x, f0, fmaf(Q4.y, f1, fmaf(Q4.z, f2, fmaf(Q4.w, f3, m))));
            }
            if (j < i) AF[i * fs::LDF + j] = a;
            MF[i * fs::LDF + j] = m;
        }
        __syncthreads();
        invert_unit_lower64(AF, TF, PF, warp, lane);
        // b.k.e^{G}, then W = T (b.k.e^G): thread = (token row i, 4 channels), the row's T entries shared
        // by the warp
        for (int p = tid; p < 64 * 32; p += xs::kThreads) {
            const int t = p >> 5, c = 4 * (p & 31);
            float4* x = reinterpret_cast<float4*>(sBK + t * xs::LD + c);
            const float4 G4 = *reinterpret_cast<const float4*>(sG + t * xs::LD + c);
            float4 v = *x;
            v.x *= __expf(G4.x); v.y *= __expf(G4.y); v.z *= __expf(G4.z); v.w *= __expf(G4.w);
            *x = v;
        }
        __syncthreads();
        for (int p = tid; p < 64 * 16; p += xs::kThreads) {
            const int i = p >> 4, c = 8 * (p & 15);
            float acc[8] = {};
            for (int l = 0; l <= i; ++l) {
                const float tl = TF[i * fs::LDF + l];
                const float4 x0 = *reinterpret_cast<const float4*>(sBK + l * xs::LD + c);
                const float4 x1 = *reinterpret_cast<const float4*>(sBK + l * xs::LD + c + 4);
                acc[0] = fmaf(tl, x0.x, acc[0]); acc[1] = fmaf(tl, x0.y, acc[1]);
                acc[2] = fmaf(tl, x0.z, acc[2]); acc[3] = fmaf(tl, x0.w, acc[3]);
                acc[4] = fmaf(tl, x1.x, acc[4]); acc[5] = fmaf(tl, x1.y, acc[5]);
                acc[6] = fmaf(tl, x1.z, acc[6]); acc[7] = fmaf(tl, x1.w, acc[7]);
            }
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = -acc[e];  // stored negated
            *reinterpret_cast<uint4*>(unit + kWsW + i * 256 + c * 2) = pack8(y);
            // decayed q and k of the same token and channels
            float qb[8], kh[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float Gi = sG[i * xs::LD + c + e];
                qb[e] = sQ[i * xs::LD + c + e] * __expf(Gi);
                kh[e] = sK[i * xs::LD + c + e] * __expf(sG[(kC - 1) * xs::LD + c + e] - Gi);
            }
            *reinterpret_cast<uint4*>(unit + kWsQb + i * 256 + c * 2) = pack8(qb);
            *reinterpret_cast<uint4*>(unit + kWsKh + i * 256 + c * 2) = pack8(kh);
        }
        // M and T as bf16 [64][64] rows (zeros above their diagonals)
        for (int p = tid; p < 64 * 8; p += xs::kThreads) {
            const int i = p >> 3, c = 8 * (p & 7);
            float ym[8], yt[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ym[e] = (c + e <= i) ? MF[i * fs::LDF + c + e] : 0.f;
                yt[e] = (c + e <= i) ? TF[i * fs::LDF + c + e] : 0.f;
            }
            *reinterpret_cast<uint4*>(unit + kWsM + i * 128 + c * 2) = pack8(ym);
            *reinterpret_cast<uint4*>(unit + kWsT + i * 128 + c * 2) = pack8(yt);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// kernel 2: state chain + output

struct StateMaps {
    CUtensorMap w, qb, kh, m, t;   // workspace sections
    CUtensorMap v, wg;             // token tiles of v and of the write gate w
    CUtensorMap o_st;              // output, stored in [32 tokens][64 d_v] tiles (128-byte swizzle)
};

namespace ss {
// Shared memory (every tile 1024-byte aligned): two rings of two slots, "big" for what the products
// of chunk n read during step n, "pre" for what is used one step ahead (T and w.v), so each slot is
// released as soon as its last reader is done; the chunk decays have a ring of four of their own.
constexpr uint32_t A1 = 0;          // big: [-W ; Q] as a 128-row K-major A operand: two 64-wide d_k
                                    //      blocks of [128 rows (token)][128 B]
constexpr uint32_t KH = 32768;      // big: k.e^{G_last-G} token-major, two 64-wide d_k blocks
                                    //      (MN-major A operand, M = d_k)
constexpr uint32_t MM = 49152;      // big: M [64 tokens][64 tokens], K-major. The 8 KB before it are the
                                    //      upper half of the A operand of M U; those product rows fall on
                                    //      U rows that have been read already.
constexpr uint32_t BIG = 57344;     // big slot size
constexpr uint32_t TT = 0;          // pre: T [64][64] K-major followed by 8 KB of zeros: A operand [T ; 0]
constexpr uint32_t VV = 16384;      // pre: this CTA's 64 v columns [64 tokens][64]; w.v in place (MN-major B)
constexpr uint32_t WW = 24576;      // pre: the same columns of w
constexpr uint32_t PRE = 32768;     // pre slot size
constexpr uint32_t TX_BIG = 7 * 8192;
constexpr uint32_t TX_PRE = 3 * 8192;
constexpr uint32_t BIG0 = 0;
constexpr uint32_t PRE0 = 2 * BIG;
constexpr uint32_t SB = PRE0 + 2 * PRE;  // bf16 S_n [128 d_k][64 d_v] (MN-major B operand)
constexpr uint32_t UB = SB + 16384;      // bf16 U [64 tokens][64 d_v] (MN-major B operand)
constexpr uint32_t OST = UB + 8192;      // output staging [2 warps][32 tokens][64 d_v] bf16, 128-byte swizzle
constexpr uint32_t GAMC = OST + 8192;    // ring of e^{G_last}: [4 chunks][128] fp32, own barriers
constexpr uint32_t BAR = GAMC + 2048;    // mbarriers, TMEM base, error flag
constexpr uint32_t TOTAL = BAR + 256;
constexpr int kChainWarps = 4;           // warps 0-3: U and state read-outs, decay (64 columns each)
constexpr int kOutWarps = 4;             // warps 4-7: w.v; warps 6-7 also read the output
constexpr int kOutReaders = 2;
constexpr int kProducer = 8, kIssuer = 9;
constexpr int kThreads = 10 * 32;
// TMEM columns (lane = product row). D_UO[b] (b = chunk parity): lanes 0-63 hold U = T (w.v) - W S_n,
// lanes 64-127 O = Q S_n + M U. D_S receives K^T U (lane = d_k row).
constexpr uint32_t kDuo = 0, kDs = 128, kCols = 256;
}  // namespace ss

// The chunk recurrence for 64 of the d_v columns, d_v / 64 CTAs per (batch, value head): the columns of S
// evolve independently, so each CTA keeps its d_k x 64 slice of the state. Per chunk n, with the
// factors of the workspace,
//   U = T (w.v) - W S_n,   O = Q S_n + M U,   S_{n+1} = diag(e^{G_last}) S_n + K^T U.
// Every product has the 128 rows of M = 128: the token rows of [T ; 0], [-W ; Q] and [. ; M] put U and
// O into the two lane halves of one accumulator, and d_k is the row side of K^T U. The fp32 state
// stays in the registers of the four chain warps (one d_k row, all 64 columns per thread), where the
// decay is one scalar per row and K^T U is added from tensor memory; its bf16 copy and U are the B
// operands in shared memory. The dependent chain per chunk is
//   S_n -> [-W ; Q] S_n -> U -> + K^T U -> S_{n+1};
// w.v, T (w.v), M U, the decay and the output run beside it. Roles: a TMA warp keeps both slots of
// both rings in flight, an MMA warp issues (one lane), four chain warps read U and the state, four
// warps form w.v and two of them read the output. They hand over through mbarriers; every wait is
// bounded.
// kSave: the backward's form, which also keeps bf16 S_n and U_n of every chunk (s_save, u_save); the
// forward's form carries no save code in its chain.
template <bool kSave>
__global__ void __launch_bounds__(ss::kThreads, 1)
    state_tc_kernel(const __grid_constant__ StateMaps maps, const uint8_t* __restrict__ ws,
                    const float* __restrict__ s0, float* __restrict__ sT_out, int Hv, int dk, int dv, int NC,
                    float scale, __nv_bfloat16* __restrict__ s_save, __nv_bfloat16* __restrict__ u_save,
                    int write_o, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* full_big = reinterpret_cast<uint64_t*>(sm + ss::BAR);  // [2] big slot landed
    uint64_t* empty_big = full_big + 2;                              // [2] big slot consumed
    uint64_t* full_pre = full_big + 4;                               // [2] pre slot landed
    uint64_t* empty_pre = full_big + 6;                              // [2] pre slot consumed
    uint64_t* wv_ready = full_big + 8;                               // [2] w.v formed (per chunk parity)
    uint64_t* o_free = full_big + 10;                                // [2] O lanes of D_UO[b] read
    uint64_t* o_done = full_big + 12;                                // [2] O of D_UO[b] complete
    uint64_t* mma1_done = full_big + 14;                             // [-W ; Q] S_n complete
    uint64_t* s_done = full_big + 15;                                // K^T U complete
    uint64_t* u_ready = full_big + 16;                               // U written (2 warps)
    uint64_t* s_ready = full_big + 17;                               // bf16 S_n written (4 chain warps)
    uint64_t* drain = full_big + 18;
    uint64_t* gam_full = full_big + 19;                              // [4] e^{G_last} of chunk m landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + ss::BAR + 224);
    volatile int* err = reinterpret_cast<volatile int*>(sm + ss::BAR + 228);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslice = dv >> 6;                           // 64-column slices of d_v
    const int bh = blockIdx.x / nslice, hc = blockIdx.x - bh * nslice;  // (batch, value head), d_v slice
    const int bi = bh / Hv, hv = bh - bi * Hv;

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(full_big + i, 1);
        mbar_init(wv_ready, ss::kOutWarps);
        mbar_init(wv_ready + 1, ss::kOutWarps);
        mbar_init(o_free, ss::kOutReaders);
        mbar_init(o_free + 1, ss::kOutReaders);
        mbar_init(o_done, 1);
        mbar_init(o_done + 1, 1);
        mbar_init(mma1_done, 1);
        mbar_init(s_done, 1);
        mbar_init(u_ready, ss::kChainWarps / 2);
        mbar_init(s_ready, ss::kChainWarps);
        mbar_init(drain, 1);
        for (int i = 0; i < 4; ++i) mbar_init(gam_full + i, 1);
        *err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, ss::kCols);
        tmem_relinquish();
    }
    for (int p = tid; p < 2 * 512; p += ss::kThreads)  // the zero halves of [T ; 0] in both pre slots
        reinterpret_cast<uint4*>(sm + ss::PRE0 + (p >> 9) * ss::PRE + ss::TT + 8192)[p & 511] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == ss::kProducer) {
        // ================================ TMA warp ================================
        // order of need: pre(0), then big(m), pre(m+1)
        int big_issued = -1, pre_issued = -1;
        if (lane == 0) {
            auto issue_pre = [&](int m) -> bool {
                const int st = m & 1;
                if (m >= 2 && !mbar_wait_or_abort(empty_pre + st, ((m >> 1) + 1) & 1, wait_ns, err)) return false;
                uint8_t* sb = sm + ss::PRE0 + st * ss::PRE;
                const int u = bh * NC + m;
                mbar_arrive_expect_tx(full_pre + st, ss::TX_PRE);
                tma_load_3d(sb + ss::TT, &maps.t, 0, 0, u, full_pre + st);
                tma_load_4d(sb + ss::VV, &maps.v, 64 * hc, hv, m * kC, bi, full_pre + st);
                tma_load_4d(sb + ss::WW, &maps.wg, 64 * hc, hv, m * kC, bi, full_pre + st);
                // the decay of chunk m-4 has been applied once pre(m-2) was consumed
                mbar_arrive_expect_tx(gam_full + (m & 3), 512);
                bulk_load(sm + ss::GAMC + (m & 3) * 512, ws + static_cast<size_t>(u) * kWsUnit + kWsGam, 512,
                          gam_full + (m & 3));
                pre_issued = m;
                return true;
            };
            auto issue_big = [&](int m) -> bool {
                const int st = m & 1;
                if (m >= 2 && !mbar_wait_or_abort(empty_big + st, ((m >> 1) + 1) & 1, wait_ns, err)) return false;
                uint8_t* sb = sm + ss::BIG0 + st * ss::BIG;
                const int u = bh * NC + m;
                mbar_arrive_expect_tx(full_big + st, ss::TX_BIG);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_3d(sb + ss::A1 + kb * 16384, &maps.w, 64 * kb, 0, u, full_big + st);
                    tma_load_3d(sb + ss::A1 + kb * 16384 + 8192, &maps.qb, 64 * kb, 0, u, full_big + st);
                    tma_load_3d(sb + ss::KH + kb * 8192, &maps.kh, 64 * kb, 0, u, full_big + st);
                }
                tma_load_3d(sb + ss::MM, &maps.m, 0, 0, u, full_big + st);
                big_issued = m;
                return true;
            };
            bool go = NC > 0 && issue_pre(0);
            for (int m = 0; go && m < NC; ++m) go = issue_big(m) && (m + 1 >= NC || issue_pre(m + 1));
            if (!go && NC > 0) note_failure(err);
            // every load this warp issued has landed before the block releases its shared memory
            for (int m = big_issued - 1; m <= big_issued; ++m)
                if (m >= 0) mbar_wait(full_big + (m & 1), (m >> 1) & 1, kDefaultWaitNs);
            for (int m = pre_issued - 1; m <= pre_issued; ++m)
                if (m >= 0) mbar_wait(full_pre + (m & 1), (m >> 1) & 1, kDefaultWaitNs);
            for (int m = pre_issued - 3; m <= pre_issued; ++m)
                if (m >= 0) mbar_wait(gam_full + (m & 3), (m >> 2) & 1, kDefaultWaitNs);
        }
    } else if (warp == ss::kIssuer) {
        // ================================ MMA warp ================================
        // Tensor-pipe order per step n: [-W ; Q] S_n | K^T U (n) | M U (n) | T (w.v) (n+1): the
        // products off the chain run while the state is read out.
        if (lane == 0) {
            constexpr uint32_t id_k = idesc_bf16(128, 64, false, true);  // K-major A, MN-major B
            constexpr uint32_t id_s = idesc_bf16(128, 64, true, true);   // K^T U: MN-major A and B
            auto desc = [&](uint32_t off, uint32_t lbo) { return smem_desc(sbase + off, lbo, 1024, kSwizzle128B); };
            const uint64_t b_s = desc(ss::SB, 16384), b_u = desc(ss::UB, 8192);
            // D_UO[m&1] = [T ; 0] (w.v), once w.v of chunk m is formed and the output of chunk m-2 read
            auto mma0 = [&](int m) -> bool {
                const int st = m & 1, ph = (m >> 1) & 1;
                if (!mbar_wait_or_abort(wv_ready + st, ph, wait_ns, err) ||
                    !mbar_wait_or_abort(full_pre + st, ph, wait_ns, err) ||
                    !mbar_wait_or_abort(o_free + st, ph, wait_ns, err))
                    return false;
                tc_fence_after();
                const uint32_t pre = ss::PRE0 + st * ss::PRE;
                const uint64_t a = desc(pre + ss::TT, 16), b = desc(pre + ss::VV, 8192);
#pragma unroll
                for (int s = 0; s < 4; ++s)  // K = tokens
                    mma_bf16(tmem + ss::kDuo + 64 * st, a + (s * 32 >> 4), b + (s * 2048 >> 4), id_k, s > 0);
                mma_commit(empty_pre + st);
                return true;
            };
            bool run = NC > 0 && mma0(0);
            for (int n = 0; run && n < NC; ++n) {
                const int st = n & 1;
                const uint32_t big = ss::BIG0 + st * ss::BIG;
                if (!mbar_wait_or_abort(full_big + st, (n >> 1) & 1, wait_ns, err) ||
                    !mbar_wait_or_abort(s_ready, n & 1, wait_ns, err)) {
                    run = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint64_t a = desc(big + ss::A1, 16);
#pragma unroll
                    for (int s = 0; s < 8; ++s)  // K = d_k: two 64-wide blocks of 16 KB
                        mma_bf16(tmem + ss::kDuo + 64 * st, a + (((s >> 2) * 16384 + (s & 3) * 32) >> 4),
                                 b_s + (s * 2048 >> 4), id_k, 1);
                }
                mma_commit(mma1_done);
                if (!mbar_wait_or_abort(u_ready, n & 1, wait_ns, err)) {
                    run = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint64_t ak = desc(big + ss::KH, 8192), am = desc(big + ss::MM - 8192, 16);
#pragma unroll
                    for (int s = 0; s < 4; ++s)  // K = tokens
                        mma_bf16(tmem + ss::kDs, ak + (s * 2048 >> 4), b_u + (s * 2048 >> 4), id_s, s > 0);
                    mma_commit(s_done);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16(tmem + ss::kDuo + 64 * st, am + (s * 32 >> 4), b_u + (s * 2048 >> 4), id_k, 1);
                    mma_commit(o_done + st);
                    mma_commit(empty_big + st);
                }
                if (n + 1 < NC && !mma0(n + 1)) {
                    run = false;
                    break;
                }
            }
            if (!run && NC > 0) note_failure(err);
            // all issued MMAs complete before TMEM and shared memory are released
            mma_commit(drain);
            mbar_wait(drain, 0, kDefaultWaitNs);
        }
    } else if (warp >= ss::kChainWarps) {
        // ============== w.v (warps 4-7) and output read-out (warps 6-7) ==============
        const int q4 = warp & 3;                      // TMEM lane quarter
        const bool reader = q4 >= 2;                  // lanes 64-127: O rows = tokens 32 (q4 - 2) ..
        const int otid = tid - 32 * ss::kChainWarps;  // 0..127
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        uint8_t* stg = sm + ss::OST + (q4 & 1) * 4096;  // [32 tokens][64 d_v] bf16, 128-byte swizzle
        // w.v in place of v (both tiles carry the same swizzle, so the product is position-wise)
        auto take_pre = [&](int m) -> bool {
            const int st = m & 1;
            if (!warp_wait(full_pre + st, (m >> 1) & 1, wait_ns, err)) return false;
            uint8_t* sbp = sm + ss::PRE0 + st * ss::PRE;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = (otid + 128 * i) * 16;  // 512 chunks of 16 bytes
                float a[8], bw[8];
                unpack8(*reinterpret_cast<const uint4*>(sbp + ss::VV + off), a);
                unpack8(*reinterpret_cast<const uint4*>(sbp + ss::WW + off), bw);
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] *= bw[e];
                *reinterpret_cast<uint4*>(sbp + ss::VV + off) = pack8(a);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive1(wv_ready + st);
            return true;
        };
        bool ok = NC > 0;
        if (ok) {
            if (reader && lane == 0) {  // nothing to read before the first two chunks
                mbar_arrive1(o_free);
                mbar_arrive1(o_free + 1);
            }
            ok = take_pre(0) && (NC < 2 || take_pre(1));
        }
        for (int m = 0; ok && m < NC; ++m) {
            const int st = m & 1;
            if (reader) {
                if (!(ok = warp_wait(o_done + st, (m >> 1) & 1, wait_ns, err))) break;
                tc_fence_after();
                if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read the staging
                __syncwarp();
                float x[64];
                tmem_ld_cols<4>(tmem + lane_base + ss::kDuo + 64 * st, x);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive1(o_free + st);
#pragma unroll
                for (int j = 0; j < 64; ++j) x[j] *= scale;
#pragma unroll
                for (int h = 0; h < 2; ++h) st_row_bf16x32(stg, lane, 4 * h, x + 32 * h);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && write_o) {
                    // rows past T are clipped by the tensor map
                    tma_store_4d(&maps.o_st, stg, 64 * hc, hv, m * kC + 32 * (q4 - 2), bi);
                    bulk_commit();
                }
            }
            if (m + 2 < NC && !(ok = take_pre(m + 2))) break;
        }
        if (reader && lane == 0) bulk_wait_all();  // the output is written before the block retires
    } else {
        // ============= U and state read-outs, decay (warps 0-3) =============
        // Each thread keeps its row and the CTA's 64 columns of the fp32 state in registers, already
        // multiplied by the next chunk's decay; the tensor core only forms K^T U. One warp per TMEM
        // lane quarter: measured faster than two or four warps per quarter with fewer columns each,
        // since every extra warp is one more arrival on the barriers the MMA warp waits for.
        const int q4 = warp & 3;                    // TMEM lane quarter; all 64 columns
        const bool u_reader = q4 < 2;               // lanes 0-63 of D_UO hold U
        const int r = 32 * q4 + lane;               // d_k row of D_S (= TMEM lane); token row of U
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        auto arrive = [&](uint64_t* bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive1(bar);
        };
        auto decay = [&](int m, float (&x)[64]) -> bool {  // x = e^{G_last(m)} . x for this thread's row
            if (!warp_wait(gam_full + (m & 3), (m >> 2) & 1, wait_ns, err)) return false;
            const float gg = reinterpret_cast<const float*>(sm + ss::GAMC)[(m & 3) * 128 + r];
#pragma unroll
            for (int j = 0; j < 64; ++j) x[j] *= gg;
            return true;
        };
        uint8_t* sbt = sm + ss::SB;
        uint8_t* ubt = sm + ss::UB;
        // with d_k = 64 the rows 64..127 are zero padding: they start at 0 and stay there (their keys
        // are zero and their decay is 1), and are neither read from S0 nor written to S_T
        const bool real_row = r < dk;
        const size_t srow = (static_cast<size_t>(bh) * dk + (real_row ? r : 0)) * dv + 64 * hc;
        float sx[64];  // e^{G_last(n)} . S_n
        bool ok = NC > 0;
        if (ok) {
#pragma unroll
            for (int j4 = 0; j4 < 16; ++j4) {
                const float4 f = (s0 && real_row) ? reinterpret_cast<const float4*>(s0 + srow)[j4]
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                sx[4 * j4] = f.x;
                sx[4 * j4 + 1] = f.y;
                sx[4 * j4 + 2] = f.z;
                sx[4 * j4 + 3] = f.w;
            }
            st_row_bf16x32(sbt, r, 0, sx);
            st_row_bf16x32(sbt, r, 4, sx + 32);
            fence_proxy_async_smem();
            arrive(s_ready);
            if (kSave && s_save && real_row)
                st_global_bf16x64(s_save + (static_cast<size_t>(bh) * NC * dk + r) * dv + 64 * hc, sx);
            ok = decay(0, sx);
        }
        for (int n = 0; ok && n < NC; ++n) {
            const int st = n & 1;
            if (u_reader) {
                if (!(ok = warp_wait(mma1_done, n & 1, wait_ns, err))) break;
                tc_fence_after();
                float x[64];  // U: token row r, all 64 columns -> bf16 B operand
                tmem_ld_cols<4>(tmem + lane_base + ss::kDuo + 64 * st, x);
                st_row_bf16x32(ubt, r, 0, x);
                st_row_bf16x32(ubt, r, 4, x + 32);
                fence_proxy_async_smem();
                tc_fence_before();
                arrive(u_ready);
                if (kSave && u_save) st_global_bf16x64(u_save + ((static_cast<size_t>(bh) * NC + n) * kC + r) * dv + 64 * hc, x);
            }
            if (!(ok = warp_wait(s_done, n & 1, wait_ns, err))) break;
            tc_fence_after();
            {
                float x[64];  // K^T U: d_k row r, all 64 columns
                tmem_ld_cols<4>(tmem + lane_base + ss::kDs, x);
#pragma unroll
                for (int j = 0; j < 64; ++j) sx[j] += x[j];  // S_{n+1}
            }
            st_row_bf16x32(sbt, r, 0, sx);
            st_row_bf16x32(sbt, r, 4, sx + 32);
            fence_proxy_async_smem();
            tc_fence_before();
            arrive(s_ready);
            if (kSave && s_save && real_row && n + 1 < NC)
                st_global_bf16x64(s_save + ((static_cast<size_t>(bh) * NC + n + 1) * dk + r) * dv + 64 * hc, sx);
            if (n + 1 < NC) {
                if (!(ok = decay(n + 1, sx))) break;
            } else if (sT_out && real_row) {
                float4* dst = reinterpret_cast<float4*>(sT_out + srow);
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4)
                    dst[j4] = make_float4(sx[4 * j4], sx[4 * j4 + 1], sx[4 * j4 + 2], sx[4 * j4 + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ss::kCols);
}

// ---------------------------------------------------------------------------------------------
// UMMA layout self-test: one M=128 product with the operand layouts the kernels above use.

struct SelftestMaps {
    CUtensorMap a, b;
};

// Storage shapes (rows x cols of the row-major device arrays), N and K of each case; see
// gdn2_selftest_umma in the public header.
struct SelftestShape {
    int a_rows, a_cols, b_rows, b_cols, N, K;
    bool a_mn, b_mn, a_tmem;
};
__host__ __device__ constexpr SelftestShape selftest_shape(int c) {
    return c == 1   ? SelftestShape{64, 128, 64, 64, 64, 64, true, false, false}
           : c == 2 ? SelftestShape{128, 128, 128, 64, 64, 128, true, true, false}
           : c == 3 ? SelftestShape{128, 64, 64, 64, 64, 64, false, true, false}
           : c == 5 ? SelftestShape{128, 64, 64, 64, 64, 64, false, false, true}
           : c == 6 ? SelftestShape{128, 64, 64, 128, 128, 64, false, true, true}
           : c == 7 ? SelftestShape{128, 128, 128, 128, 128, 128, false, false, true}
                    : SelftestShape{128, 128, 64, 128, 64, 128, false, false, false};  // cases 0 and 4
}

__global__ void __launch_bounds__(128, 1)
    selftest_umma_kernel(const __grid_constant__ SelftestMaps maps, int case_id, int soft,
                         const __nv_bfloat16* __restrict__ a_st, const __nv_bfloat16* __restrict__ b_st,
                         float* __restrict__ d_out, long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const bool negate = (case_id == 4);  // case 4: case 0 with the A operand negated by the descriptor
    const SelftestShape sh = selftest_shape(case_id);
    uint8_t* sA = sm;
    uint8_t* sB = sm + 32768;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + 65536 + 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t kAcol = 128;  // TMEM column of an A operand held in tensor memory

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
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
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    if (sh.a_tmem) {  // row 32*warp + lane of A, K bf16 values packed two per column
        const uint32_t* src = reinterpret_cast<const uint32_t*>(a_st + (32 * warp + lane) * sh.a_cols);
        for (int c0 = 0; c0 < sh.a_cols / 2; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = src[c0 + i];
            tmem_st16(tmem + lane_base + kAcol + c0, r);
        }
        tmem_st_wait();
    }
    // a storage of R rows x (64 * nb) columns becomes nb blocks of R x 128 B (block j = columns 64j..)
    bool ok = true;
    if (soft) {
        if (!sh.a_tmem)
            for (int p = tid; p < sh.a_rows * sh.a_cols; p += 128) {
                const int rr = p / sh.a_cols, cc = p % sh.a_cols;
                *reinterpret_cast<__nv_bfloat16*>(sA + (cc >> 6) * (sh.a_rows * 128) + sw128_off(rr, cc & 63)) =
                    a_st[p];
            }
        for (int p = tid; p < sh.b_rows * sh.b_cols; p += 128) {
            const int rr = p / sh.b_cols, cc = p % sh.b_cols;
            *reinterpret_cast<__nv_bfloat16*>(sB + (cc >> 6) * (sh.b_rows * 128) + sw128_off(rr, cc & 63)) = b_st[p];
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    } else {
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(bar, ((sh.a_tmem ? 0 : sh.a_rows * sh.a_cols) + sh.b_rows * sh.b_cols) * 2);
            if (!sh.a_tmem)
                for (int j = 0; j < sh.a_cols / 64; ++j) tma_load_3d(sA + j * sh.a_rows * 128, &maps.a, 64 * j, 0, 0, bar);
            for (int j = 0; j < sh.b_cols / 64; ++j) tma_load_3d(sB + j * sh.b_rows * 128, &maps.b, 64 * j, 0, 0, bar);
        }
        ok = cta_wait(bar, 0, wait_ns);
    }
    if (ok) {
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, sh.N, sh.a_mn, sh.b_mn) | (negate ? kNegateA : 0u);
            for (int s = 0; s < sh.K / 16; ++s) {
                // K-major: K blocks of 64 are separate R x 128 B regions; step 32 B inside a block.
                // MN-major: K rows are 128-byte rows; step 16 rows = 2048 B; LBO = next 64-wide MN block.
                // Tensor memory: 16 K values are 8 columns.
                const uint32_t boff = sh.b_mn ? s * 2048 : (s >> 2) * (sh.b_rows * 128) + (s & 3) * 32;
                const uint64_t bd =
                    smem_desc(sbase + 32768 + boff, sh.b_mn ? sh.b_rows * 128 : 16, 1024, kSwizzle128B);
                if (sh.a_tmem) {
                    mma_bf16_ts(tmem, tmem + kAcol + 8 * s, bd, id, s > 0);
                } else {
                    const uint32_t aoff = sh.a_mn ? s * 2048 : (s >> 2) * (sh.a_rows * 128) + (s & 3) * 32;
                    const uint64_t ad = smem_desc(sbase + aoff, sh.a_mn ? sh.a_rows * 128 : 16, 1024, kSwizzle128B);
                    mma_bf16(tmem, ad, bd, id, s > 0);
                }
            }
            mma_commit(bar + 1);
        }
        ok = cta_wait(bar + 1, 0, wait_ns);
    }
    if (ok) {
        tc_fence_after();
        for (int c0 = 0; c0 < sh.N; c0 += 64) {
            float x[64];
            tmem_ld64(tmem, warp, c0, x);
            for (int j = 0; j < 64; ++j) d_out[(32 * warp + lane) * sh.N + c0 + j] = x[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

// Workspace: the 66 048-byte units, (batch . value head, chunk) order, then the list of units that
// the exact kernel forms: a count and up to one int32 index per unit.
size_t chunk_tc_workspace_bytes(const ChunkShape& sh) {
    const size_t units = static_cast<size_t>(sh.nchunks()) * sh.B * sh.Hv;
    return static_cast<size_t>(kWsUnit) * units + align_up(sizeof(int) * (units + 1), 256);
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const void* g, const void* b,
                            const void* w, const float* s0, float* sT, void* o, const ChunkShape& sh, float scale,
                            void* ws, cudaStream_t s, long long wait_ns, void* s_save, void* u_save) {
    const int NC = sh.nchunks();
    const int units = NC * sh.B * sh.Hv;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
    FactorMaps fm;
    // d_k = 64: the maps declare 64 channels, so the second 64-channel box of every tile reads as zeros
    if (!token_map(&fm.q, q, sh.B, sh.T, sh.Hk, sh.dk) || !token_map(&fm.k, k, sh.B, sh.T, sh.Hk, sh.dk) ||
        !token_map(&fm.g, g, sh.B, sh.T, sh.Hv, sh.dk) || !token_map(&fm.b, b, sh.B, sh.T, sh.Hv, sh.dk) ||
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
        !token_map(&sm_.v, v, sh.B, sh.T, sh.Hv, sh.dv) || !token_map(&sm_.wg, w, sh.B, sh.T, sh.Hv, sh.dv) ||
        !out_map(&sm_.o_st, o ? o : ws, sh.B, sh.T, sh.Hv, sh.dv))  // no output: a map that is never used
        return cudaErrorInvalidValue;

    // The state kernel runs one CTA per SM, so it takes the whole 227 KB: operand descriptors can
    // then never reach past the CTA's own allocation.
    const size_t f_smem = fs::TOTAL + 1024, x_smem = xs::TOTAL + 128, s_smem = 232448;
    static_assert(ss::TOTAL + 1024 <= 232448, "state kernel shared memory");
    static_assert(xs::TOTAL + 128 <= 232448, "exact factor kernel shared memory");
    cudaError_t e = cudaFuncSetAttribute(factors_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(factors_exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)x_smem);
    if (e != cudaSuccess) return e;
    const bool save = s_save || u_save;
    e = cudaFuncSetAttribute(save ? state_tc_kernel<true> : state_tc_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    int* exact_list = reinterpret_cast<int*>(wsb + static_cast<size_t>(kWsUnit) * units);
    if ((e = cudaMemsetAsync(exact_list, 0, sizeof(int), s)) != cudaSuccess) return e;
    factors_tc_kernel<<<dim3(NC, sh.B * sh.Hv), fs::kThreads, f_smem, s>>>(fm, wsb, exact_list, sh.Hk, sh.Hv, NC,
                                                                         wait_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    factors_exact_kernel<<<units < nsm ? units : nsm, xs::kThreads, x_smem, s>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(b), wsb, exact_list, sh.T, sh.Hk,
        sh.Hv, NC, sh.dk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto* state_kernel = save ? state_tc_kernel<true> : state_tc_kernel<false>;
    state_kernel<<<dim3((sh.dv / 64) * sh.B * sh.Hv), ss::kThreads, s_smem, s>>>(
        sm_, wsb, s0, sT, sh.Hv, sh.dk, sh.dv, NC, scale, static_cast<__nv_bfloat16*>(s_save),
        static_cast<__nv_bfloat16*>(u_save), o != nullptr, wait_ns);
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
    if (case_id < 0 || case_id > 7) return cudaErrorInvalidValue;
    const SelftestShape sh = selftest_shape(case_id);
    const int ar = sh.a_rows, ac = sh.a_cols, br = sh.b_rows, bc = sh.b_cols;
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

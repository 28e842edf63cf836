// backward_tc.cu -- gradients of the GDN-2 core in chunked form on the 5th-generation tensor cores
// (tcgen05 + TMA + TMEM): bf16 inputs, d_k and d_v 64 or 128, chunks of C = 64 (the recurrence of the
// burn-gdn2 0.1.5 docs, "Architecture", in the chunked WY form of its "chunked WY decomposition
// (training)" section).
//
// Per chunk n, with the factors that the forward's tensor-core kernels write to their workspace
// (-W, Q_bar = q.e^G, K^ = k.e^{G_last - G}, M, T, gamma = e^{G_last}), S = S_n, S' = S_{n+1}:
//     U = T U0 - W S,  U0 = w.v;   O = scale (Q_bar S + M U);   S' = diag(gamma) S + K^^T U.
// Reverse mode, with dO~ = scale dO:
//   the chain over chunks, in reverse:
//     dU = M^T dO~ + K^ dS'                 dS = diag(gamma) dS' + Q_bar^T dO~ - W^T dU
//   per chunk, given S, U, dS', dU:
//     dQ_bar = dO~ S^T   dW = -dU S^T   dK^ = U dS'^T   dM = tril(dO~ U^T)   dgamma = rowsum(dS' . S)
//     dT = dU U0^T + dW K_bar^T   dU0 = T^T dU   dK_bar = T^T dW   dA = -strict_tril(T^T dT T^T)
//   with K_bar = b.k.e^G, then the pair terms through A_ts = sum_c (b.k)_t k_s e^{G_t - G_s} and
//   M_ts = sum_c q_t k_s e^{G_t - G_s}, every exponential factor <= 1 (split at 8-token block edges),
//   and the chain rule through the elementwise factors to dq, dk, db, dg, dv, dw.
//
// Launches: the forward's factor kernels and its state kernel, which also keeps bf16 S_n and U_n of
// every chunk (chunk_tc.cu); rchain_tc_kernel, one CTA per (batch-head, 64 columns of d_v), the
// chain in reverse on the tensor cores (fp32 dS in registers), keeping bf16 dS_{n+1} and dU_n;
// grad_tc_kernel, one CTA per (chunk, head): every product on the tensor cores (the pair terms with
// one anchor per channel, or on CUDA cores in chunks whose log-decay spans too much for it) and the
// chain rule on CUDA cores; the sums of dq and dk over the value heads of each key head. A head size of
// 64 runs as 128 whose upper 64 channels (or columns) are zeros: the tensor maps declare the true size,
// so the upper boxes read as zeros, and only the true channels are written.
#include "common.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace gdn2 {
namespace {

// ---------------------------------------------------------------------------------------------
// the chain over chunks in reverse

struct RevMaps {
    CUtensorMap w, qb, kh, m;  // workspace sections of the forward factors
    CUtensorMap dout;          // token tiles of dO
};

namespace rs {
// Shared memory (tiles 1024-byte aligned): "big" slots hold what the two dependent products of step n
// read, "pre" slots what the products issued one step ahead read; two of each.
constexpr uint32_t KH = 0;      // big: K^ token-major, two 64-wide d_k blocks [64 tokens][128 B]: K-major A of
                                //      K^ dS' (its rows 64..127 are the next 8 KB: finite, their lanes unused)
constexpr uint32_t WN = 16384;  // big: -W token-major, two d_k blocks: MN-major A of (-W)^T dU (M = d_k)
constexpr uint32_t BIG = 32768;
constexpr uint32_t QB = 0;      // pre: Q_bar token-major, two d_k blocks: MN-major A of Q_bar^T dO~
constexpr uint32_t MM = 16384;  // pre: M [64 s][64 t]: MN-major A of M^T dO~ (M = t; the operand's second
                                //      64-wide block is the dO tile that follows: finite, lanes unused)
constexpr uint32_t DO = 24576;  // pre: this CTA's 64 columns of dO [64 tokens][128 B]; dO~ = scale dO in place
constexpr uint32_t PRE = 32768;
constexpr uint32_t TX_BIG = 32768, TX_PRE = 32768;
constexpr uint32_t BIG0 = 0, PRE0 = 2 * BIG;
constexpr uint32_t DSB = PRE0 + 2 * PRE;  // bf16 dS' [128 d_k][64 d_v] (MN-major B of K^ dS')
constexpr uint32_t DUB = DSB + 16384;     // bf16 dU [64 tokens][64 d_v] (MN-major B of (-W)^T dU)
constexpr uint32_t GAMC = DUB + 8192;     // ring of gamma: [4 chunks][128] fp32
constexpr uint32_t BAR = GAMC + 2048;
constexpr uint32_t TOTAL = BAR + 256;
constexpr int kChainWarps = 4;  // warps 0-3: dS in registers (one d_k row per thread); warps 0-1 also read dU
constexpr int kHelpWarps = 4;   // warps 4-7: dO~ = scale dO
constexpr int kProducer = 8, kIssuer = 9;
constexpr int kThreads = 10 * 32;
// TMEM columns: D_dU[b] (lanes 0-63 = tokens) at kDu + 64 b, D_dS[b] (lanes = d_k rows) at kDs + 64 b
constexpr uint32_t kDu = 0, kDs = 128, kCols = 256;
}  // namespace rs

// One CTA per (batch . value head, 64 columns of d_v), chunks from the last to the first. Per chunk n,
// with dS' = dS_{n+1} (fp32, registers of the chain warps):
//   dU = M^T dO~ + K^ dS'      (M^T dO~ issued one step ahead; K^ dS' waits for the bf16 dS')
//   dS_n = diag(gamma) dS' + Q_bar^T dO~ + (-W)^T dU   (Q_bar^T dO~ issued one step ahead)
// Every product has M = 128 (token-row products carry 64 discarded lanes). Kept per chunk: bf16 dS'
// and bf16 dU (this CTA's columns).
__global__ void __launch_bounds__(rs::kThreads, 1)
    rchain_tc_kernel(const __grid_constant__ RevMaps maps, const uint8_t* __restrict__ ws,
                     const float* __restrict__ dsT, float* __restrict__ ds0, __nv_bfloat16* __restrict__ ds_save,
                     __nv_bfloat16* __restrict__ du_save, int Hv, int NC, int dk, int dv, float scale,
                     long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* full_big = reinterpret_cast<uint64_t*>(sm + rs::BAR);  // [2]
    uint64_t* empty_big = full_big + 2;                              // [2]
    uint64_t* full_pre = full_big + 4;                               // [2]
    uint64_t* empty_pre = full_big + 6;                              // [2]
    uint64_t* do_ready = full_big + 8;                               // [2] dO~ formed
    uint64_t* du_done = full_big + 10;                               // dU complete
    uint64_t* ds_done = full_big + 11;                               // dS product complete
    uint64_t* ds_ready = full_big + 12;                              // bf16 dS' written (4 chain warps)
    uint64_t* du_ready = full_big + 13;                              // bf16 dU written (2 warps)
    uint64_t* drain = full_big + 14;
    uint64_t* gam_full = full_big + 15;                              // [4]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + rs::BAR + 160);
    volatile int* err = reinterpret_cast<volatile int*>(sm + rs::BAR + 164);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslice = dv >> 6;  // 64-column slices of d_v
    const int bh = blockIdx.x / nslice, hc = blockIdx.x - bh * nslice;
    const int bi = bh / Hv, hv = bh - bi * Hv;

    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(full_big + i, 1);
        mbar_init(do_ready, rs::kHelpWarps);
        mbar_init(do_ready + 1, rs::kHelpWarps);
        mbar_init(du_done, 1);
        mbar_init(ds_done, 1);
        mbar_init(ds_ready, rs::kChainWarps);
        mbar_init(du_ready, 2);
        mbar_init(drain, 1);
        for (int i = 0; i < 4; ++i) mbar_init(gam_full + i, 1);
        *err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, rs::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == rs::kProducer) {
        // ================================ TMA warp ================================
        int big_issued = -1, pre_issued = -1;
        if (lane == 0) {
            auto issue_pre = [&](int m) -> bool {
                const int st = m & 1;
                if (m >= 2 && !mbar_wait_or_abort(empty_pre + st, ((m >> 1) + 1) & 1, wait_ns, err)) return false;
                uint8_t* sb = sm + rs::PRE0 + st * rs::PRE;
                const int n = NC - 1 - m, u = bh * NC + n;
                mbar_arrive_expect_tx(full_pre + st, rs::TX_PRE);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) tma_load_3d(sb + rs::QB + kb * 8192, &maps.qb, 64 * kb, 0, u, full_pre + st);
                tma_load_3d(sb + rs::MM, &maps.m, 0, 0, u, full_pre + st);
                tma_load_4d(sb + rs::DO, &maps.dout, 64 * hc, hv, n * kC, bi, full_pre + st);
                // gamma of chunk m-4 has been applied once pre(m-2) was consumed
                mbar_arrive_expect_tx(gam_full + (m & 3), 512);
                bulk_load(sm + rs::GAMC + (m & 3) * 512, ws + static_cast<size_t>(u) * kWsUnit + kWsGam, 512,
                          gam_full + (m & 3));
                pre_issued = m;
                return true;
            };
            auto issue_big = [&](int m) -> bool {
                const int st = m & 1;
                if (m >= 2 && !mbar_wait_or_abort(empty_big + st, ((m >> 1) + 1) & 1, wait_ns, err)) return false;
                uint8_t* sb = sm + rs::BIG0 + st * rs::BIG;
                const int u = bh * NC + NC - 1 - m;
                mbar_arrive_expect_tx(full_big + st, rs::TX_BIG);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_3d(sb + rs::KH + kb * 8192, &maps.kh, 64 * kb, 0, u, full_big + st);
                    tma_load_3d(sb + rs::WN + kb * 8192, &maps.w, 64 * kb, 0, u, full_big + st);
                }
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
    } else if (warp == rs::kIssuer) {
        // ================================ MMA warp ================================
        if (lane == 0) {
            constexpr uint32_t id_mn = idesc_bf16(128, 64, true, true);   // MN-major A and B
            constexpr uint32_t id_k = idesc_bf16(128, 64, false, true);   // K-major A, MN-major B
            auto desc = [&](uint32_t off, uint32_t lbo) { return smem_desc(sbase + off, lbo, 1024, kSwizzle128B); };
            const uint64_t b_ds = desc(rs::DSB, 16384), b_du = desc(rs::DUB, 8192);
            // D_dU[m&1] = M^T dO~ and D_dS[m&1] = Q_bar^T dO~, once dO~ of chunk m is formed
            auto pre = [&](int m) -> bool {
                const int st = m & 1, ph = (m >> 1) & 1;
                if (!mbar_wait_or_abort(do_ready + st, ph, wait_ns, err) ||
                    !mbar_wait_or_abort(full_pre + st, ph, wait_ns, err))
                    return false;
                tc_fence_after();
                const uint32_t p = rs::PRE0 + st * rs::PRE;
                const uint64_t am = desc(p + rs::MM, 8192), aq = desc(p + rs::QB, 8192), bo = desc(p + rs::DO, 8192);
#pragma unroll
                for (int s = 0; s < 4; ++s)  // K = tokens
                    mma_bf16(tmem + rs::kDu + 64 * st, am + (s * 2048 >> 4), bo + (s * 2048 >> 4), id_mn, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + rs::kDs + 64 * st, aq + (s * 2048 >> 4), bo + (s * 2048 >> 4), id_mn, s > 0);
                mma_commit(empty_pre + st);
                return true;
            };
            bool run = NC > 0 && pre(0);
            for (int m = 0; run && m < NC; ++m) {
                const int st = m & 1;
                const uint32_t big = rs::BIG0 + st * rs::BIG;
                if (!mbar_wait_or_abort(full_big + st, (m >> 1) & 1, wait_ns, err) ||
                    !mbar_wait_or_abort(ds_ready, m & 1, wait_ns, err)) {
                    run = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint64_t a = desc(big + rs::KH, 16);
#pragma unroll
                    for (int s = 0; s < 8; ++s)  // K = d_k: two 64-wide blocks of 8 KB
                        mma_bf16(tmem + rs::kDu + 64 * st, a + (((s >> 2) * 8192 + (s & 3) * 32) >> 4),
                                 b_ds + (s * 2048 >> 4), id_k, 1);
                }
                mma_commit(du_done);
                if (!mbar_wait_or_abort(du_ready, m & 1, wait_ns, err)) {
                    run = false;
                    break;
                }
                tc_fence_after();
                {
                    const uint64_t a = desc(big + rs::WN, 8192);
#pragma unroll
                    for (int s = 0; s < 4; ++s)  // K = tokens
                        mma_bf16(tmem + rs::kDs + 64 * st, a + (s * 2048 >> 4), b_du + (s * 2048 >> 4), id_mn, 1);
                }
                mma_commit(ds_done);
                mma_commit(empty_big + st);
                if (m + 1 < NC && !pre(m + 1)) {
                    run = false;
                    break;
                }
            }
            if (!run && NC > 0) note_failure(err);
            mma_commit(drain);
            mbar_wait(drain, 0, kDefaultWaitNs);
        }
    } else if (warp >= rs::kChainWarps) {
        // ======================= dO~ = scale dO (warps 4-7) =======================
        const int htid = tid - 32 * rs::kChainWarps;
        for (int m = 0; m < NC; ++m) {
            const int st = m & 1;
            if (!warp_wait(full_pre + st, (m >> 1) & 1, wait_ns, err)) break;
            uint8_t* p = sm + rs::PRE0 + st * rs::PRE + rs::DO;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4* c = reinterpret_cast<uint4*>(p + (htid + 128 * i) * 16);
                float x[8];
                unpack8(*c, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= scale;
                *c = pack8(x);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive1(do_ready + st);
        }
    } else {
        // ==================== dS in registers, dU read-out (warps 0-3) ====================
        const int q4 = warp & 3;
        const bool u_reader = q4 < 2;                 // lanes 0-63 of D_dU hold dU
        const int r = 32 * q4 + lane;                 // d_k row of dS (= TMEM lane); token row of dU
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        auto arrive = [&](uint64_t* bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive1(bar);
        };
        uint8_t* dsb = sm + rs::DSB;
        uint8_t* dub = sm + rs::DUB;
        // with d_k = 64 the rows 64..127 are zero padding: they start at 0 and stay there (their keys are
        // zero and their decay is 1), and are neither read from dS_T nor written to dS_0
        const bool real_row = r < dk;
        const size_t srow = (static_cast<size_t>(bh) * dk + (real_row ? r : 0)) * dv + 64 * hc;
        float sx[64];  // dS' = dS_{n+1}
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
            const float4 f = (dsT && real_row) ? reinterpret_cast<const float4*>(dsT + srow)[j4]
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
            sx[4 * j4] = f.x;
            sx[4 * j4 + 1] = f.y;
            sx[4 * j4 + 2] = f.z;
            sx[4 * j4 + 3] = f.w;
        }
        bool ok = NC > 0;
        for (int m = 0; ok && m < NC; ++m) {
            const int st = m & 1;
            const size_t u = static_cast<size_t>(bh) * NC + (NC - 1 - m);
            st_row_bf16x32(dsb, r, 0, sx);
            st_row_bf16x32(dsb, r, 4, sx + 32);
            fence_proxy_async_smem();
            arrive(ds_ready);
            st_global_bf16x64(ds_save + (u * kD + r) * dv + 64 * hc, sx);
            if (!(ok = warp_wait(gam_full + (m & 3), (m >> 2) & 1, wait_ns, err))) break;
            {
                const float gg = reinterpret_cast<const float*>(sm + rs::GAMC)[(m & 3) * 128 + r];
#pragma unroll
                for (int j = 0; j < 64; ++j) sx[j] *= gg;
            }
            if (u_reader) {
                if (!(ok = warp_wait(du_done, m & 1, wait_ns, err))) break;
                tc_fence_after();
                float x[64];  // dU: token row r, this CTA's 64 columns
                tmem_ld_cols<4>(tmem + lane_base + rs::kDu + 64 * st, x);
                st_row_bf16x32(dub, r, 0, x);
                st_row_bf16x32(dub, r, 4, x + 32);
                fence_proxy_async_smem();
                tc_fence_before();
                arrive(du_ready);
                st_global_bf16x64(du_save + (u * kC + r) * dv + 64 * hc, x);
            }
            if (!(ok = warp_wait(ds_done, m & 1, wait_ns, err))) break;
            tc_fence_after();
            {
                float x[64];
                tmem_ld_cols<4>(tmem + lane_base + rs::kDs + 64 * st, x);
#pragma unroll
                for (int j = 0; j < 64; ++j) sx[j] += x[j];  // dS_n
            }
            tc_fence_before();
        }
        if (ok && ds0 && real_row) {
            float4* dst = reinterpret_cast<float4*>(ds0 + srow);
#pragma unroll
            for (int j4 = 0; j4 < 16; ++j4)
                dst[j4] = make_float4(sx[4 * j4], sx[4 * j4 + 1], sx[4 * j4 + 2], sx[4 * j4 + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, rs::kCols);
}

// ---------------------------------------------------------------------------------------------
// per-chunk gradients

struct GradMaps {
    CUtensorMap dout, v, w, q, k, g, b;  // token tiles (box 64 channels x 64 tokens)
    CUtensorMap du, u;                   // bf16 [units][64 tokens][128] saves (box 64 x 64)
    CUtensorMap s, ds;                   // bf16 [units][128 d_k][128 d_v] saves (box 64 x 128)
    CUtensorMap t;                       // T of the forward factors
    CUtensorMap dq_st, dk_st;            // fp32 [B][T][H_v][d_k] sums' inputs (store box 32 channels x 64 tokens)
    CUtensorMap db_st, dg_st;            // bf16 db, dg [B][T][H_v][d_k] (store box 64 channels x 64 tokens)
    CUtensorMap dv_st, dw_st;            // bf16 dv, dw [B][T][H_v][d_v] (store box 64 columns x 64 tokens)
};

namespace gs {
// Inputs (1024-byte aligned tiles, 128-byte swizzle, block j = columns 64j .. 64j+63):
constexpr uint32_t A1 = 0;        // [dO ; dU]: K-major A (K = d_v), block j at 16384 j: [128 rows][128 B]
constexpr uint32_t B1 = 32768;    // [S ; U ; U0]: K-major B (N = 256), block j at B1 + 32768 j: [256 rows][128 B]
constexpr uint32_t DS = 98304;    // dS': K-major B (N = 128), block j at DS + 16384 j
constexpr uint32_t WV = 131072;   // w, block j at WV + 8192 j
constexpr uint32_t TT = 147456;   // T [64][64] (8 KB) then 8 KB of zeros: the MN-major A operand [T^T ; 0]
constexpr uint32_t QT = 163840, KT = 180224, GT = 196608, BT = 212992;  // q, k, g, b, block j at +8192 j
constexpr uint32_t BAR = 229376;  // mbarriers, TMEM base; then G_last, anchors, dgamma
constexpr uint32_t TOTAL = BAR + 2048;
// Rooms reused once their first contents are consumed:
constexpr uint32_t GF = DS;                  // G fp32, two 16 KB halves of d_k
constexpr uint32_t KB = B1;                  // K_bar bf16 [64 s][128 B] x 2 (B of dW K_bar^T)
constexpr uint32_t VR = B1 + 32768;          // v again (U0 took its place), 2 blocks
constexpr uint32_t DW0 = B1 + 24576;         // dW bf16 blocks: rows 64..127 of A operands whose rows 0..63
constexpr uint32_t DW1 = B1 + 32768 + 24576;  //  are the U rows before them (finite, their lanes unused)
constexpr uint32_t DT = A1;                  // dT bf16 [64 t][64 s] (MN-major B)
constexpr uint32_t PM = A1 + 16384;          // P = T^T dT bf16 [64][64] (K-major A; rows 64.. = dU block 1)
constexpr uint32_t DAB = WV;                 // [dA ; dM] bf16 [128][64]: K-major A of [dA ; dM] K_til, and as
constexpr uint32_t DMB = WV + 8192;          //   two [64 u][64 s] tiles the MN-major A of dA^T B_a + dM^T Q_a
constexpr uint32_t XF = A1;                  // X, then dG (fp32 halves A1, A1 + 16384)
constexpr uint32_t YF = B1;                  // Y (halves B1, B1 + 16384)
constexpr uint32_t ZF = B1 + 32768;          // Z + V (halves B1 + 32768, B1 + 49152)
constexpr uint32_t KTA = B1 + 16384;         // anchored operands (bf16 [64 tokens][128 B] x 2): k.e^{a-G},
constexpr uint32_t BKA = B1 + 32768;         //   b.k.e^{G-a}, q.e^{G-a}; the second and third lie under Z + V,
constexpr uint32_t QA = B1 + 49152;          //   which is written once the product that reads them is done
constexpr uint32_t GL = BAR + 512;           // G_last fp32 [128]
constexpr uint32_t AN = BAR + 1024;          // per-channel anchor a fp32 [128]
constexpr uint32_t DGM = BAR + 1536;         // dgamma = rowsum(dS' . S) fp32 [128]
constexpr int kThreads = 512;  // 16 warps: four per tensor-memory lane quarter
// TMEM columns (lane = row of the product):
//   [0,128)   dO S^T (lanes 0-63: dQ_bar / scale) | dU S^T (lanes 64-127: -dW)
//   [128,192) dO U^T (lanes 0-63: dM / scale)     then dK_bar = T^T dW over [128,256) (lanes 0-63)
//   [192,256) dU U0^T + dW K_bar^T (lanes 64-127: dT)
//   [256,384) U dS'^T (lanes 0-63: dK^)
//   [384,512) T^T dU (lanes 0-63: dU0), then T^T dT over [384,448), (T^T dT) T^T over [448,512), then
//             [dA ; dM] K_til (lanes 0-63: X / e^{G-a}, lanes 64-127: Y / e^{G-a}), then
//             dA^T B_a + dM^T Q_a (lanes 0-63: (Z + V) e^{G-a})
constexpr uint32_t kCols = 512;
}  // namespace gs

// byte offset of fp32 element (t, c) of a [64][128] array kept as two [64][64] halves whose columns
// are XOR-swizzled by (t mod 32): conflict-free both for a warp over c (one t) and a warp over t (one c)
__device__ __forceinline__ uint32_t fidx(int t, int c) {
    return static_cast<uint32_t>(((c >> 6) * 4096 + t * 64 + ((c & 63) ^ (t & 31))) * 4);
}
// Largest per-channel span G_0 - G_last of the cumulative log-decay within one chunk for which the
// pair terms go to the tensor cores with one anchor a per channel: every factor e^{+-(G - a)} then lies
// in [e^-60, e^60] (the forward's factor kernel routes chunks by the same bound). Wider chunks take the
// pair terms on CUDA cores with factors e^{G_t - G_s} <= 1.
constexpr float kSpanPair = 120.f;

// One CTA per (chunk, batch . value head); 512 threads, one CTA per SM (the inputs fill shared memory).
__global__ void __launch_bounds__(gs::kThreads, 1)
    grad_tc_kernel(const __grid_constant__ GradMaps maps, int T, int Hk, int Hv, int d_k, int d_v, float scale,
                   long long wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + gs::BAR);  // copies a, b, v; products 1 .. 6, X|Y, Z+V
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + gs::BAR + 96);
    float* GLs = reinterpret_cast<float*>(sm + gs::GL);
    float* ANs = reinterpret_cast<float*>(sm + gs::AN);

    const int n = blockIdx.x, bh = blockIdx.y, NC = gridDim.x;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    const int u = bh * NC + n;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, h = warp >> 2;  // TMEM lane quarter, column quarter
    const int nvalid = min(kC, T - n * kC);

    if (tid == 0) {
        for (int i = 0; i < 9; ++i) mbar_init(bar + i, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, gs::kCols);
        tmem_relinquish();
    }
    for (int p = tid; p < 512; p += gs::kThreads)  // the zero half of [T^T ; 0]
        reinterpret_cast<uint4*>(sm + gs::TT + 8192)[p] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        mbar_arrive_expect_tx(bar + 0, 147456);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + gs::A1 + j * 16384, &maps.dout, 64 * j, hv, n * kC, bi, bar);
            tma_load_3d(sm + gs::A1 + j * 16384 + 8192, &maps.du, 64 * j, 0, u, bar);
            tma_load_3d(sm + gs::B1 + j * 32768, &maps.s, 64 * j, 0, u, bar);
            tma_load_3d(sm + gs::B1 + j * 32768 + 16384, &maps.u, 64 * j, 0, u, bar);
            tma_load_4d(sm + gs::B1 + j * 32768 + 24576, &maps.v, 64 * j, hv, n * kC, bi, bar);
            tma_load_3d(sm + gs::DS + j * 16384, &maps.ds, 64 * j, 0, u, bar);
            tma_load_4d(sm + gs::WV + j * 8192, &maps.w, 64 * j, hv, n * kC, bi, bar);
        }
        mbar_arrive_expect_tx(bar + 1, 73728);
        tma_load_3d(sm + gs::TT, &maps.t, 0, 0, u, bar + 1);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            tma_load_4d(sm + gs::QT + j * 8192, &maps.q, 64 * j, hk, n * kC, bi, bar + 1);
            tma_load_4d(sm + gs::KT + j * 8192, &maps.k, 64 * j, hk, n * kC, bi, bar + 1);
            tma_load_4d(sm + gs::GT + j * 8192, &maps.g, 64 * j, hv, n * kC, bi, bar + 1);
            tma_load_4d(sm + gs::BT + j * 8192, &maps.b, 64 * j, hv, n * kC, bi, bar + 1);
        }
    }
    auto desc = [&](uint32_t off, uint32_t lbo) { return smem_desc(sbase + off, lbo, 1024, kSwizzle128B); };
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);  // this warp's TMEM lanes
    bool v_issued = false, exact = false;
    bool ok = cta_wait(bar + 0, 0, wait_ns);

    // ---- U0 = w.v in place of v (both tiles carry the same swizzle)
    if (ok) {
#pragma unroll
        for (int i = 0; i < 1024 / gs::kThreads; ++i) {
            const int p = tid + gs::kThreads * i, j = p >> 9, o = (p & 511) * 16;
            uint4* vv = reinterpret_cast<uint4*>(sm + gs::B1 + j * 32768 + 24576 + o);
            float a[8], bw[8];
            unpack8(*vv, a);
            unpack8(*reinterpret_cast<const uint4*>(sm + gs::WV + j * 8192 + o), bw);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] *= bw[e];
            *vv = pack8(a);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P1: [dO ; dU] [S ; U ; U0]^T (N = 256), P2: [U ; U0] dS'^T (N = 128); K = d_v
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id1 = idesc_bf16(128, 256, false, false), id2 = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t ka = (s >> 2) * 16384 + (s & 3) * 32, kb = (s >> 2) * 32768 + (s & 3) * 32;
                mma_bf16(tmem, desc(gs::A1 + ka, 16), desc(gs::B1 + kb, 16), id1, s > 0);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t ka = (s >> 2) * 32768 + (s & 3) * 32, kb = (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tmem + 256, desc(gs::B1 + 16384 + ka, 16), desc(gs::DS + kb, 16), id2, s > 0);
            }
            mma_commit(bar + 3);
        }
        if (tid >= gs::kThreads - kD) {  // dgamma_c = sum over d_v of dS'[c][v] S[c][v] (same swizzle in both)
            const int c = tid - (gs::kThreads - kD);
            float acc = 0.f;
#pragma unroll 1
            for (int j = 0; j < 2; ++j)
#pragma unroll 2
                for (int p = 0; p < 8; ++p) {
                    float x[8], y[8];
                    const int o = c * 128 + ((p ^ (c & 7)) << 4);  // 8 lanes, 8 different 16-byte pieces
                    unpack8(*reinterpret_cast<const uint4*>(sm + gs::B1 + j * 32768 + o), x);
                    unpack8(*reinterpret_cast<const uint4*>(sm + gs::DS + j * 16384 + o), y);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc = fmaf(x[e], y[e], acc);
                }
            reinterpret_cast<float*>(sm + gs::DGM)[c] = acc;
        }
        ok = cta_wait(bar + 3, 0, wait_ns) && cta_wait(bar + 1, 0, wait_ns);
    }
    if (ok) {
        tc_fence_after();
        if (tid == 0) {  // v again, into the first room S has left
            v_issued = true;
            mbar_arrive_expect_tx(bar + 2, 16384);
#pragma unroll
            for (int j = 0; j < 2; ++j)
                tma_load_4d(sm + gs::VR + j * 8192, &maps.v, 64 * j, hv, n * kC, bi, bar + 2);
        }
        if (q4 >= 2) {  // dW = -(dU S^T): token row t, d_k columns 32h .. -> bf16 operand rows
            const int t = 32 * (q4 - 2) + lane;
            float x[32];
            tmem_ld_cols<2>(tl + 32 * h, x);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = -x[j];
            st_row_bf16x32(sm + ((h >> 1) ? gs::DW1 : gs::DW0), t, 4 * (h & 1), x);
        } else if (h < 2) {  // G (floored gates, inclusive sum over the chunk): thread = channel c
            const int c = 64 * h + 32 * q4 + lane;
            const uint32_t cb = (c >> 6) * 8192;
            float run = 0.f;
#pragma unroll 8
            for (int t = 0; t < kC; ++t) {
                run += fmaxf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::GT + cb + sw128_off(t, c & 63))),
                             kGateFloor);
                *reinterpret_cast<float*>(sm + gs::GF + fidx(t, c)) = run;
            }
            GLs[c] = run;
        }
        __syncthreads();
        {   // K_bar = b.k.e^G: thread = channel c, a quarter of the tokens
            const int c = tid & (kD - 1), t0 = 16 * (tid >> 7);
            const uint32_t cb = (c >> 6) * 8192;
#pragma unroll 4
            for (int t = t0; t < t0 + 16; ++t) {
                const uint32_t o = cb + sw128_off(t, c & 63);
                const float bk = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::BT + o)) *
                                 __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::KT + o));
                const float Gt = *reinterpret_cast<const float*>(sm + gs::GF + fidx(t, c));
                *reinterpret_cast<__nv_bfloat16*>(sm + gs::KB + o) = __float2bfloat16_rn(bk * __expf(Gt));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P4: dT += dW K_bar^T (K = d_k; rows 64..127 of the A operand), P5a: dU0 = T^T dU (K = tokens)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id4 = idesc_bf16(128, 64, false, false), id5 = idesc_bf16(128, 128, true, true);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t a = ((s >> 2) ? gs::DW1 : gs::DW0) - 8192 + (s & 3) * 32;
                mma_bf16(tmem + 192, desc(a, 16), desc(gs::KB + (s >> 2) * 8192 + (s & 3) * 32, 16), id4, 1);
            }
            const uint64_t at = desc(gs::TT, 8192), bu = desc(gs::A1 + 8192, 16384);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 384, at + (s * 2048 >> 4), bu + (s * 2048 >> 4), id5, s > 0);
            mma_commit(bar + 4);
        }
        ok = cta_wait(bar + 4, 0, wait_ns) && cta_wait(bar + 2, 0, wait_ns);
    }
    if (ok) {
        tc_fence_after();
        if (q4 < 2) {  // dU0 -> dv = w.dU0, dw = v.dU0: token row t, d_v columns 32h .., written in place
                       // of w and v (their last reader) for the bulk tensor stores below
            const int t = 32 * q4 + lane;
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                float x[16];
                tmem_ld_cols<1>(tl + 384 + 32 * h + 16 * q, x);
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int cc = 4 * h + 2 * q + c2;  // 16-byte piece of the row: 8 columns
                    const uint32_t so = (cc >> 3) * 8192 + t * 128 + (((cc & 7) ^ (t & 7)) << 4);
                    float wv[8], vv[8], ov[8], ow[8];
                    unpack8(*reinterpret_cast<const uint4*>(sm + gs::WV + so), wv);
                    unpack8(*reinterpret_cast<const uint4*>(sm + gs::VR + so), vv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        ov[e] = wv[e] * x[8 * c2 + e];
                        ow[e] = vv[e] * x[8 * c2 + e];
                    }
                    *reinterpret_cast<uint4*>(sm + gs::WV + so) = pack8(ov);
                    *reinterpret_cast<uint4*>(sm + gs::VR + so) = pack8(ow);
                }
            }
        } else if (h < 2) {  // dT: token row t, columns 32h .. -> bf16 [t][s] (MN-major B)
            const int t = 32 * (q4 - 2) + lane;
            float x[32];
            tmem_ld_cols<2>(tl + 192 + 32 * h, x);
            st_row_bf16x32(sm + gs::DT, t, 4 * h, x);
        }
        // dv and dw leave by bulk tensor stores (tokens past T and columns past d_v clipped by the maps);
        // their rooms are taken next, so the stores must have read them first
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                tma_store_4d(&maps.dv_st, sm + gs::WV + j * 8192, 64 * j, hv, n * kC, bi);
                tma_store_4d(&maps.dw_st, sm + gs::VR + j * 8192, 64 * j, hv, n * kC, bi);
            }
            bulk_commit();
            bulk_wait_read_all();
        }
        __syncthreads();  // w (now dv) is read: its room takes dA and dM
        if (q4 < 2 && h < 2) {  // dM = scale tril(dO U^T): token row t, columns 32h .. -> bf16 row
            const int t = 32 * q4 + lane;
            float x[32];
            tmem_ld_cols<2>(tl + 128 + 32 * h, x);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= t ? scale * x[j] : 0.f;
            st_row_bf16x32(sm + gs::DMB, t, 4 * h, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P5b: dK_bar = T^T dW, P6a: P = T^T dT (K = tokens)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id5 = idesc_bf16(128, 128, true, true), id6 = idesc_bf16(128, 64, true, true);
            const uint64_t at = desc(gs::TT, 8192), bw = desc(gs::DW0, gs::DW1 - gs::DW0), bt = desc(gs::DT, 8192);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tmem + 128, at + (s * 2048 >> 4), bw + (s * 2048 >> 4), id5, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tmem + 384, at + (s * 2048 >> 4), bt + (s * 2048 >> 4), id6, s > 0);
            mma_commit(bar + 5);
        }
        ok = cta_wait(bar + 5, 0, wait_ns);
    }
    if (ok) {
        tc_fence_after();
        if (q4 < 2 && h < 2) {  // P -> bf16 K-major rows
            const int t = 32 * q4 + lane;
            float x[32];
            tmem_ld_cols<2>(tl + 384 + 32 * h, x);
            st_row_bf16x32(sm + gs::PM, t, 4 * h, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P6b: P T^T (K = 64); while it runs, the per-channel anchors a = (G_0 + G_last) / 2, the span
        //      check and, for pair terms on the tensor cores, their operands K_til = k.e^{a-G},
        //      B_a = b.k.e^{G-a}, Q_a = q.e^{G-a} (X = E.([dA] K_til), Y = E.([dM] K_til),
        //      Z + V = (dA^T B_a + dM^T Q_a) / E with E = e^{G-a})
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id6 = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + 448, desc(gs::PM + s * 32, 16), desc(gs::TT + s * 32, 16), id6, s > 0);
            mma_commit(bar + 6);
        }
        float span = 0.f;
        if (tid < kD) {
            const float g0 = *reinterpret_cast<const float*>(sm + gs::GF + fidx(0, tid));
            ANs[tid] = 0.5f * (g0 + GLs[tid]);
            span = g0 - GLs[tid];
        }
        exact = __syncthreads_or(span > kSpanPair) != 0;
        if (!exact) {
            const int c = tid & (kD - 1), t0 = 16 * (tid >> 7);
            const float a = ANs[c];
            const uint32_t cb = (c >> 6) * 8192, cl = c & 63;
#pragma unroll 4
            for (int t = t0; t < t0 + 16; ++t) {
                const uint32_t o = cb + sw128_off(t, cl);
                const float Gt = *reinterpret_cast<const float*>(sm + gs::GF + fidx(t, c));
                const float e = __expf(Gt - a), ei = __expf(a - Gt);
                const float kk = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::KT + o));
                const float qq = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::QT + o));
                const float bb = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::BT + o));
                *reinterpret_cast<__nv_bfloat16*>(sm + gs::KTA + o) = __float2bfloat16_rn(kk * ei);
                *reinterpret_cast<__nv_bfloat16*>(sm + gs::BKA + o) = __float2bfloat16_rn(bb * kk * e);
                *reinterpret_cast<__nv_bfloat16*>(sm + gs::QA + o) = __float2bfloat16_rn(qq * e);
            }
        }
        ok = cta_wait(bar + 6, 0, wait_ns);
    }
    if (ok) {
        tc_fence_after();
        if (q4 < 2 && h < 2) {  // dA = -strict_tril(T^T dT T^T) -> bf16 row
            const int t = 32 * q4 + lane;
            float x[32];
            tmem_ld_cols<2>(tl + 448 + 32 * h, x);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 32 * h + j < t ? -x[j] : 0.f;
            st_row_bf16x32(sm + gs::DAB, t, 4 * h, x);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    if (ok && !exact) {
        if (tid == 0) {  // [dA ; dM] K_til: M = 128 (both halves used), K = tokens, N = d_k
            tc_fence_after();
            constexpr uint32_t id7 = idesc_bf16(128, 128, false, true);
            const uint64_t bk = desc(gs::KTA, 8192);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tmem + 384, desc(gs::DAB + s * 32, 16), bk + (s * 2048 >> 4), id7, s > 0);
            mma_commit(bar + 7);
        }
        ok = cta_wait(bar + 7, 0, wait_ns);
        if (ok) {
            tc_fence_after();
            {   // lanes 0-63: X / e^{G-a}, lanes 64-127: Y / e^{G-a}; token row t, channels 32h ..
                const int t = 32 * (q4 & 1) + lane;
                const uint32_t dst = q4 < 2 ? gs::XF : gs::YF;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float x[16];
                    tmem_ld_cols<1>(tl + 384 + 32 * h + 16 * q, x);
#pragma unroll
                    for (int j = 0; j < 16; ++j) *reinterpret_cast<float*>(sm + dst + fidx(t, 32 * h + 16 * q + j)) = x[j];
                }
            }
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {  // dA^T B_a + dM^T Q_a: M = 128 (rows 64.. discarded), K = 2 x 64 tokens, N = d_k
                tc_fence_after();
                constexpr uint32_t id8 = idesc_bf16(128, 128, true, true);
                const uint64_t ba = desc(gs::BKA, 8192), bq = desc(gs::QA, 8192);
                const uint64_t aa = desc(gs::DAB, 16384), am = desc(gs::DMB, 16384);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem + 384, aa + (s * 2048 >> 4), ba + (s * 2048 >> 4), id8, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tmem + 384, am + (s * 2048 >> 4), bq + (s * 2048 >> 4), id8, 1);
                mma_commit(bar + 8);
            }
            ok = cta_wait(bar + 8, 0, wait_ns);
        }
        if (ok) {
            tc_fence_after();
            if (q4 < 2) {  // (Z + V) e^{G-a}
                const int t = 32 * q4 + lane;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float x[16];
                    tmem_ld_cols<1>(tl + 384 + 32 * h + 16 * q, x);
#pragma unroll
                    for (int j = 0; j < 16; ++j) *reinterpret_cast<float*>(sm + gs::ZF + fidx(t, 32 * h + 16 * q + j)) = x[j];
                }
            }
            __syncthreads();
        }
    } else if (ok) {
        // ---- pair terms on CUDA cores (chunks wider than the anchored span), thread = channel c; side 0:
        //      X_t = sum_{s<t} dA_ts k_s e^{G_t-G_s},
        //      Y_t = sum_{s<=t} dM_ts k_s e^{G_t-G_s}; side 1: (Z+V)_s = sum_{u>s} dA_us (b.k)_u e^{G_u-G_s}
        //      + sum_{u>=s} dM_us q_u e^{G_u-G_s}. Tokens in blocks of 8; a pair in different blocks
        //      takes its factor as e^{G_t - G_r} e^{G_r - G_s} with r at the block edge.
        if (tid < 2 * kD) {
            const int c = tid & (kD - 1), side = tid >> 7;
            auto DA = [&](int t, int s2) {
                return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::DAB + sw128_off(t, s2)));
            };
            auto DM = [&](int t, int s2) {
                return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + gs::DMB + sw128_off(t, s2)));
            };
            const uint32_t cb = (c >> 6) * 8192, cl = c & 63;
            auto G = [&](int t) { return *reinterpret_cast<const float*>(sm + gs::GF + fidx(t, c)); };
            auto tok = [&](uint32_t tile, int t) {
                return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + tile + cb + sw128_off(t, cl)));
            };
#pragma unroll 1
            for (int blk = 0; blk < 8; ++blk) {
                const int t0 = 8 * blk;
                float Gb[8], A1v[8], A2v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) Gb[i] = G(t0 + i);
                if (side == 0) {
                    float kb[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        kb[i] = tok(gs::KT, t0 + i);
                        A1v[i] = 0.f;
                        A2v[i] = DM(t0 + i, t0 + i) * kb[i];
                    }
                    if (blk > 0) {
                        float ax[8], ay[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) ax[i] = ay[i] = 0.f;
                        const float Gr = Gb[0];
#pragma unroll 2
                        for (int s = 0; s < t0; ++s) {
                            const float ks = tok(gs::KT, s) * __expf(Gr - G(s));
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                ax[i] = fmaf(DA(t0 + i, s), ks, ax[i]);
                                ay[i] = fmaf(DM(t0 + i, s), ks, ay[i]);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float et = __expf(Gb[i] - Gr);
                            A1v[i] = fmaf(et, ax[i], A1v[i]);
                            A2v[i] = fmaf(et, ay[i], A2v[i]);
                        }
                    }
#pragma unroll
                    for (int i = 1; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < i; ++j) {
                            const float ks = kb[j] * __expf(Gb[i] - Gb[j]);
                            A1v[i] = fmaf(DA(t0 + i, t0 + j), ks, A1v[i]);
                            A2v[i] = fmaf(DM(t0 + i, t0 + j), ks, A2v[i]);
                        }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        *reinterpret_cast<float*>(sm + gs::XF + fidx(t0 + i, c)) = A1v[i];
                        *reinterpret_cast<float*>(sm + gs::YF + fidx(t0 + i, c)) = A2v[i];
                    }
                } else {
                    float xb[8], qb[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xb[i] = tok(gs::BT, t0 + i) * tok(gs::KT, t0 + i);
                        qb[i] = tok(gs::QT, t0 + i);
                        A1v[i] = 0.f;
                        A2v[i] = DM(t0 + i, t0 + i) * qb[i];
                    }
                    if (blk < 7) {
                        float az[8], av[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) az[i] = av[i] = 0.f;
                        const float Gr = Gb[7];
#pragma unroll 2
                        for (int uu = t0 + 8; uu < kC; ++uu) {
                            const float eu = __expf(G(uu) - Gr);
                            const float bu = tok(gs::BT, uu) * tok(gs::KT, uu) * eu, qu = tok(gs::QT, uu) * eu;
                            float av8[8], mv8[8];  // dA[u][t0 ..], dM[u][t0 ..]: one 16-byte piece of each row
                            unpack8(*reinterpret_cast<const uint4*>(sm + gs::DAB + sw128_off(uu, t0)), av8);
                            unpack8(*reinterpret_cast<const uint4*>(sm + gs::DMB + sw128_off(uu, t0)), mv8);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                az[i] = fmaf(av8[i], bu, az[i]);
                                av[i] = fmaf(mv8[i], qu, av[i]);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float es = __expf(Gr - Gb[i]);
                            A1v[i] = fmaf(es, az[i], A1v[i]);
                            A2v[i] = fmaf(es, av[i], A2v[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 7; ++i)
#pragma unroll
                        for (int j = i + 1; j < 8; ++j) {
                            const float e = __expf(Gb[j] - Gb[i]);
                            A1v[i] = fmaf(DA(t0 + j, t0 + i), xb[j] * e, A1v[i]);
                            A2v[i] = fmaf(DM(t0 + j, t0 + i), qb[j] * e, A2v[i]);
                        }
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float*>(sm + gs::ZF + fidx(t0 + i, c)) = A1v[i] + A2v[i];
                }
            }
        }
        __syncthreads();
    }
    if (ok) {
        // ---- back to the inputs, token row t (lanes 0-63), channels of half h:
        //      dq = dQ_bar e^G + Y; d(b.k) = dK_bar e^G + X; dk = dK^ e^{G_last-G} + Z + V + d(b.k) b;
        //      db = d(b.k) k; dG_t = dQ_bar q e^G + dK_bar K_bar - dK^ K^ + (b.k) X + q Y - k (Z+V) (into X's
        //      place) and E_t = dK^ K^ (the G_last part, into G's place). From the tensor cores X, Y and
        //      Z + V arrive without their anchor factors e^{+-(G-a)}, which are applied here.
        // The lanes 0-63 warps take channels 16h .. 16h+15 from tensor memory and copy those of channels
        // 64+16h .. for the lanes 64-127 warps, which cannot read those lanes, into rooms free by now.
        const uint32_t QS = gs::TT, KS = gs::WV, HS = gs::GT;  // fp32 [64 t][64], columns swizzled by t
        auto sidx = [](int t, int cc) { return static_cast<uint32_t>((t * 64 + (cc ^ (t & 31))) * 4); };
        if (q4 < 2) {
            const int t = 32 * q4 + lane;
            {
                const int cc0 = 16 * h;  // channel 64 + cc0 ..
                uint32_t rq[16], rk[16], rh[16];
                tmem_ld16(tl + 64 + cc0, rq);
                tmem_ld16(tl + 128 + 64 + cc0, rk);
                tmem_ld16(tl + 256 + 64 + cc0, rh);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    *reinterpret_cast<uint32_t*>(sm + QS + sidx(t, cc0 + e)) = rq[e];
                    *reinterpret_cast<uint32_t*>(sm + KS + sidx(t, cc0 + e)) = rk[e];
                    *reinterpret_cast<uint32_t*>(sm + HS + sidx(t, cc0 + e)) = rh[e];
                }
            }
        }
        __syncthreads();
        {
            const bool low = q4 < 2;
            const int t = 32 * (q4 & 1) + lane;
            {
                const int c0 = (low ? 0 : 64) + 16 * h;
                uint32_t rq[16], rk[16], rh[16];
                if (low) {
                    tmem_ld16(tl + c0, rq);
                    tmem_ld16(tl + 128 + c0, rk);
                    tmem_ld16(tl + 256 + c0, rh);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        rq[e] = *reinterpret_cast<const uint32_t*>(sm + QS + sidx(t, c0 - 64 + e));
                        rk[e] = *reinterpret_cast<const uint32_t*>(sm + KS + sidx(t, c0 - 64 + e));
                        rh[e] = *reinterpret_cast<const uint32_t*>(sm + HS + sidx(t, c0 - 64 + e));
                    }
                }
                float oq[16], ok_[16], ob[16], qv[16], kv[16], bv[16];
                {   // the 16 channels of q, k, b in token row t: two 16-byte pieces of each tile
                    const uint32_t cb = (c0 >> 6) * 8192 + t * 128;
                    const int p0 = (c0 & 63) >> 3;
#pragma unroll
                    for (int hp = 0; hp < 2; ++hp) {
                        const uint32_t o = cb + (((p0 + hp) ^ (t & 7)) << 4);
                        float y[8];
                        unpack8(*reinterpret_cast<const uint4*>(sm + gs::QT + o), y);
#pragma unroll
                        for (int e = 0; e < 8; ++e) qv[8 * hp + e] = y[e];
                        unpack8(*reinterpret_cast<const uint4*>(sm + gs::KT + o), y);
#pragma unroll
                        for (int e = 0; e < 8; ++e) kv[8 * hp + e] = y[e];
                        unpack8(*reinterpret_cast<const uint4*>(sm + gs::BT + o), y);
#pragma unroll
                        for (int e = 0; e < 8; ++e) bv[8 * hp + e] = y[e];
                    }
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int c = c0 + e;
                    float* xs = reinterpret_cast<float*>(sm + gs::XF + fidx(t, c));
                    float* gsl = reinterpret_cast<float*>(sm + gs::GF + fidx(t, c));
                    const float Gt = *gsl, eG = __expf(Gt), eH = __expf(GLs[c] - Gt);
                    const float qq = qv[e], kk = kv[e], bb = bv[e];
                    const float be = bb * kk;
                    const float dqb = scale * __uint_as_float(rq[e]), dkb = __uint_as_float(rk[e]),
                                dkh = __uint_as_float(rh[e]);
                    const float ea = exact ? 1.f : __expf(Gt - ANs[c]), eai = exact ? 1.f : __expf(ANs[c] - Gt);
                    const float x = ea * *xs, y = ea * *reinterpret_cast<const float*>(sm + gs::YF + fidx(t, c)),
                                zv = eai * *reinterpret_cast<const float*>(sm + gs::ZF + fidx(t, c));
                    const float dbeta = fmaf(dkb, eG, x);
                    const float E = dkh * kk * eH;
                    *xs = dqb * qq * eG + dkb * be * eG - E + be * x + qq * y - kk * zv;
                    *gsl = E;
                    oq[e] = fmaf(dqb, eG, y);
                    ok_[e] = fmaf(dkh, eH, zv) + dbeta * bb;
                    ob[e] = dbeta * kk;
                }
                // dq, dk, db leave through shared memory and bulk tensor stores (tokens past T and
                // channels past d_k are clipped by the tensor maps): the rooms of Y, Z + V and the copied
                // q / k / h columns are free once every thread has passed the barrier below
                __syncthreads();
                const int jq = c0 >> 5, cq = (c0 & 31) >> 2;  // fp32 box (32 channels) and its 16-byte chunk
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const uint32_t o = jq * 8192 + t * 128 + (((cq + f) ^ (t & 7)) << 4);
                    *reinterpret_cast<float4*>(sm + gs::YF + o) =
                        make_float4(oq[4 * f], oq[4 * f + 1], oq[4 * f + 2], oq[4 * f + 3]);
                    *reinterpret_cast<float4*>(sm + gs::ZF + o) =
                        make_float4(ok_[4 * f], ok_[4 * f + 1], ok_[4 * f + 2], ok_[4 * f + 3]);
                }
                const int jb = c0 >> 6, cb8 = (c0 & 63) >> 3;  // bf16 box (64 channels) and its chunk
                float y0[8], y1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    y0[e] = ob[e];
                    y1[e] = ob[8 + e];
                }
                *reinterpret_cast<uint4*>(sm + gs::TT + jb * 8192 + t * 128 + ((cb8 ^ (t & 7)) << 4)) = pack8(y0);
                *reinterpret_cast<uint4*>(sm + gs::TT + jb * 8192 + t * 128 + (((cb8 + 1) ^ (t & 7)) << 4)) = pack8(y1);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                tma_store_4d(&maps.dq_st, sm + gs::YF + j * 8192, 32 * j, hv, n * kC, bi);
                tma_store_4d(&maps.dk_st, sm + gs::ZF + j * 8192, 32 * j, hv, n * kC, bi);
            }
            tma_store_4d(&maps.db_st, sm + gs::TT, 0, hv, n * kC, bi);
            tma_store_4d(&maps.db_st, sm + gs::TT + 8192, 64, hv, n * kC, bi);
            bulk_commit();
        }
        // ---- dg_t = sum_{s >= t} dG_s + sum_s E_s + dgamma gamma (the gradient of G_last): thread = channel c
        //      and a quarter of the tokens; the quarters exchange their sums through the room g has left
        {
            const int c = tid & (kD - 1), hf = tid >> 7, t0 = 16 * hf;
            float* xs = reinterpret_cast<float*>(sm + gs::GT);  // [4 quarters][2 sums][128]
            float et = 0.f, sd = 0.f;
#pragma unroll 8
            for (int t = t0; t < t0 + 16; ++t) {
                et += *reinterpret_cast<const float*>(sm + gs::GF + fidx(t, c));
                sd += *reinterpret_cast<const float*>(sm + gs::XF + fidx(t, c));
            }
            xs[(2 * hf) * kD + c] = et;
            xs[(2 * hf + 1) * kD + c] = sd;
            __syncthreads();
            const float dgm = reinterpret_cast<const float*>(sm + gs::DGM)[c];
            const float off =
                fmaf(dgm, __expf(GLs[c]), (xs[c] + xs[2 * kD + c]) + (xs[4 * kD + c] + xs[6 * kD + c]));
            float run = 0.f;  // a quarter starts from the totals of the later ones
            for (int q = 3; q > hf; --q) run += xs[(2 * q + 1) * kD + c];
            // dg leaves through the room b has left (128-byte swizzled [64 t][64 c] blocks) and two bulk
            // tensor stores (tokens past T and channels past d_k clipped by the tensor map)
            uint8_t* dgs = sm + gs::BT + (c >> 6) * 8192 + 2 * (c & 7);
#pragma unroll 8
            for (int t = t0 + 15; t >= t0; --t) {
                run += *reinterpret_cast<const float*>(sm + gs::XF + fidx(t, c));
                *reinterpret_cast<__nv_bfloat16*>(dgs + t * 128 + ((((c & 63) >> 3) ^ (t & 7)) << 4)) =
                    __float2bfloat16_rn(run + off);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tma_store_4d(&maps.dg_st, sm + gs::BT, 0, hv, n * kC, bi);
            tma_store_4d(&maps.dg_st, sm + gs::BT + 8192, 64, hv, n * kC, bi);
            bulk_commit();
        }
    }
    if (tid == 0) {  // every copy issued has landed, and the stores have read their sources, before the
                     // block releases its shared memory
        mbar_wait(bar + 0, 0, kDefaultWaitNs);
        mbar_wait(bar + 1, 0, kDefaultWaitNs);
        if (v_issued) mbar_wait(bar + 2, 0, kDefaultWaitNs);
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, gs::kCols);
}

// dq, dk of key head h_k = sums over the value heads of its group, in a fixed order
__global__ void __launch_bounds__(256) group_sum_tc_kernel(const float* __restrict__ dq_ws,
                                                           const float* __restrict__ dk_ws,
                                                           __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
                                                           long long rows, int Hk, int Hv, int d) {
    const int group = Hv / Hk;
    const long long n4 = rows * Hk * (d / 4);
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c4 = static_cast<int>(i % (d / 4));
        const long long rh = i / (d / 4);
        const int hk = static_cast<int>(rh % Hk);
        const long long r = rh / Hk;
        float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
        for (int m = 0; m < group; ++m) {
            const size_t src = ((static_cast<size_t>(r) * Hv) + hk * group + m) * d + 4 * c4;
            const float4 a = *reinterpret_cast<const float4*>(dq_ws + src), b = *reinterpret_cast<const float4*>(dk_ws + src);
            sq.x += a.x; sq.y += a.y; sq.z += a.z; sq.w += a.w;
            sk.x += b.x; sk.y += b.y; sk.z += b.z; sk.w += b.w;
        }
        const size_t dst = static_cast<size_t>(i) * 4;
        reinterpret_cast<uint2*>(dq + dst)[0] = make_uint2(pack_bf16x2(sq.x, sq.y), pack_bf16x2(sq.z, sq.w));
        reinterpret_cast<uint2*>(dk + dst)[0] = make_uint2(pack_bf16x2(sk.x, sk.y), pack_bf16x2(sk.z, sk.w));
    }
}

struct TcBwdLayout {
    size_t fw, s, u, ds, du, dq, dk, total;
};
// Saves per (chunk, value head): S_n [d_k][d_v], U_n [64][d_v], dS_(n+1) [128][d_v] (rows past d_k are
// zeros), dU_n [64][d_v], bf16; then fp32 dq and dk per value head.
TcBwdLayout tc_bwd_layout(int B, int T, int Hv, int dk, int dv) {
    const ChunkShape sh{B, T, 1, Hv, dk, dv, kC};
    const size_t units = static_cast<size_t>(sh.nchunks()) * B * Hv, tok = static_cast<size_t>(B) * T * Hv * dk * 4;
    TcBwdLayout L;
    L.fw = 0;
    L.s = align_up(chunk_tc_workspace_bytes(sh), 1024);
    L.u = align_up(L.s + units * dk * dv * 2, 1024);
    L.ds = align_up(L.u + units * kC * dv * 2, 1024);
    L.du = align_up(L.ds + units * kD * dv * 2, 1024);
    L.dq = align_up(L.du + units * kC * dv * 2, 1024);
    L.dk = align_up(L.dq + tok, 1024);
    L.total = align_up(L.dk + tok, 1024);
    return L;
}

// bf16 saves [units][rows][cols] viewed as (cols, rows, units); box (64, box_rows, 1) (rows and columns
// past the saved ones read as zeros)
bool save_map(CUtensorMap* m, const void* p, int cols, int rows, int box_rows, size_t units) {
    const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), static_cast<uint64_t>(units)};
    const uint64_t st[2] = {static_cast<uint64_t>(cols) * 2, static_cast<uint64_t>(rows) * cols * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), 1};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

size_t backward_tc_workspace_bytes(int B, int T, int Hv, int dk, int dv) { return tc_bwd_layout(B, T, Hv, dk, dv).total; }

// [B][T][H][d] token rows (element size esize) as the target of bulk tensor stores: box of box_c
// channels (128 bytes, 128-byte swizzle) x 64 tokens of one head
static bool tok_store_map(CUtensorMap* m, const void* p, CUtensorMapDataType dt, int esize, int B, int T, int H,
                          int d, int box_c) {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t st[3] = {(uint64_t)d * esize, (uint64_t)H * d * esize, (uint64_t)T * H * d * esize};
    const uint32_t box[4] = {(uint32_t)box_c, 1, (uint32_t)kC, 1};
    return make_map(m, dt, 4, p, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_backward_tc(const void* q, const void* k, const void* v, const void* g, const void* b,
                               const void* w, const float* s0, const void* d_o, const float* dsT, void* dq, void* dk,
                               void* dv, void* dg, void* db, void* dw, float* ds0, int B, int T, int Hk, int Hv,
                               int d_k, int d_v, float scale, void* ws, cudaStream_t s, long long wait_ns) {
    const ChunkShape sh{B, T, Hk, Hv, d_k, d_v, kC};
    const int NC = sh.nchunks();
    const size_t units = static_cast<size_t>(NC) * B * Hv;
    const TcBwdLayout L = tc_bwd_layout(B, T, Hv, d_k, d_v);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    __nv_bfloat16* s_save = reinterpret_cast<__nv_bfloat16*>(wsb + L.s);
    __nv_bfloat16* u_save = reinterpret_cast<__nv_bfloat16*>(wsb + L.u);
    __nv_bfloat16* ds_save = reinterpret_cast<__nv_bfloat16*>(wsb + L.ds);
    __nv_bfloat16* du_save = reinterpret_cast<__nv_bfloat16*>(wsb + L.du);
    float* dq_ws = reinterpret_cast<float*>(wsb + L.dq);
    float* dk_ws = reinterpret_cast<float*>(wsb + L.dk);
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;

    // forward factors and the forward chain, keeping S_n and U_n (no output, no final state)
    cudaError_t e = launch_chunk_tc(q, k, v, g, b, w, s0, nullptr, nullptr, sh, scale, wsb + L.fw, s, wait_ns, s_save,
                                    u_save);
    if (e != cudaSuccess) return e;

    RevMaps rm;
    if (!ws_map(&rm.w, wsb + kWsW, BF, 2, 128, 64, static_cast<int>(units), 64, 64, SW) ||
        !ws_map(&rm.qb, wsb + kWsQb, BF, 2, 128, 64, static_cast<int>(units), 64, 64, SW) ||
        !ws_map(&rm.kh, wsb + kWsKh, BF, 2, 128, 64, static_cast<int>(units), 64, 64, SW) ||
        !ws_map(&rm.m, wsb + kWsM, BF, 2, 64, 64, static_cast<int>(units), 64, 64, SW) ||
        !token_map(&rm.dout, d_o, B, T, Hv, d_v))
        return cudaErrorInvalidValue;
    GradMaps gm;
    if (!token_map(&gm.dout, d_o, B, T, Hv, d_v) || !token_map(&gm.v, v, B, T, Hv, d_v) ||
        !token_map(&gm.w, w, B, T, Hv, d_v) || !token_map(&gm.q, q, B, T, Hk, d_k) ||
        !token_map(&gm.k, k, B, T, Hk, d_k) || !token_map(&gm.g, g, B, T, Hv, d_k) ||
        !token_map(&gm.b, b, B, T, Hv, d_k) || !save_map(&gm.du, du_save, d_v, kC, kC, units) ||
        !save_map(&gm.u, u_save, d_v, kC, kC, units) || !save_map(&gm.s, s_save, d_v, d_k, kD, units) ||
        !save_map(&gm.ds, ds_save, d_v, kD, kD, units) ||
        !ws_map(&gm.t, wsb + kWsT, BF, 2, 64, 64, static_cast<int>(units), 64, 64, SW) ||
        !tok_store_map(&gm.dq_st, dq_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, T, Hv, d_k, 32) ||
        !tok_store_map(&gm.dk_st, dk_ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, T, Hv, d_k, 32) ||
        !tok_store_map(&gm.db_st, db, BF, 2, B, T, Hv, d_k, 64) ||
        !tok_store_map(&gm.dg_st, dg, BF, 2, B, T, Hv, d_k, 64) ||
        !tok_store_map(&gm.dv_st, dv, BF, 2, B, T, Hv, d_v, 64) || !tok_store_map(&gm.dw_st, dw, BF, 2, B, T, Hv, d_v, 64))
        return cudaErrorInvalidValue;

    // Both kernels run one CTA per SM and take the whole 227 KB: operand descriptors can then never
    // reach past the CTA's own allocation.
    constexpr size_t kSmem = 232448;
    static_assert(rs::TOTAL + 1024 <= kSmem, "reverse chain shared memory");
    static_assert(gs::TOTAL + 1024 <= kSmem, "gradient kernel shared memory");
    if ((e = cudaFuncSetAttribute(rchain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem)) !=
        cudaSuccess)
        return e;
    rchain_tc_kernel<<<(d_v / 64) * B * Hv, rs::kThreads, kSmem, s>>>(rm, wsb + L.fw, dsT, ds0, ds_save, du_save, Hv,
                                                                       NC, d_k, d_v, scale, wait_ns);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    grad_tc_kernel<<<dim3(NC, B * Hv), gs::kThreads, kSmem, s>>>(
        gm, T, Hk, Hv, d_k, d_v, scale, wait_ns);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long rows = static_cast<long long>(B) * T, n4 = rows * Hk * (d_k / 4);
    const int gsz = static_cast<int>(n4 / 256 + 1 < 4096 ? n4 / 256 + 1 : 4096);
    group_sum_tc_kernel<<<gsz, 256, 0, s>>>(dq_ws, dk_ws, static_cast<__nv_bfloat16*>(dq),
                                            static_cast<__nv_bfloat16*>(dk), rows, Hk, Hv, d_k);
    return cudaGetLastError();
}

int backward_tc_read_clear_status(cudaStream_t s) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_tc, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (v && cudaMemcpyToSymbolAsync(g_status_tc, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    cudaStreamSynchronize(s);
    return v;
}

}  // namespace gdn2

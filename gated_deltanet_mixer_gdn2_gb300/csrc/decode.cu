// decode.cu -- the recurrent (token-by-token) mode against a persistent state, updated in place:
// gdn2_recurrent_step (one token, fp32 state) and gdn2_recurrent_update (N tokens per call, an
// optional slot map into a pool of states, fp32 or bf16 state storage).
//
// Recurrence (burn-gdn2 0.1.5 docs, "Architecture"), regrouped so that the state is read once and
// written once per call (the same decay -> erase-read -> delta -> rank-1 update -> readout order as
// the autoregressive GDN decode described in the llama.cpp GDN decode study):
//     S' = diag(alpha) S,  r_b = S'^T (b . k),  r_q = S'^T q,  d = w . v - r_b,
//     S  <- S' + k d^T,    o = scale * (r_q + (k . q) d)          [ = scale * S_new^T q ]
// With N tokens per call the state stays on chip between tokens; arithmetic is fp32 throughout, a
// bf16 state is widened on load and rounded (nearest even) once on store.
//
// Layout: state [rows, H_v, d_k, d_v] (d_v innermost), rows = batch or pool slots. The d_v columns
// evolve independently.
//   Register kernel: a warp owns 16 columns of one head across all d_k rows: lane = 8 row groups x
//   4 column groups, each lane holds d_k/8 rows x 4 columns. Reductions over d_k are in-thread, then
//   warp shuffles across the 8 row groups. No shared memory, no block barrier.
//   Streaming kernel (d_k = d_v = 128, up to 4 tokens per call, many heads): a persistent grid walks
//   the heads; each state slab is bulk-copied into a shared-memory ring with the call's token
//   vectors, so that the loads of the next heads are in flight while a head is computed. One token:
//   the updated slab goes back through its slot by bulk copy (one CTA per SM with 3 fp32 slots, or
//   two CTAs per SM with 3 bf16 slots each: a bf16 slab is half the bytes). Several tokens: two CTAs
//   per SM, the slab brought by tensor copies with the 128-byte swizzle (a warp then reads its 16
//   columns over 8 rows without bank conflicts), the state carried through the tokens in registers,
//   the slot refilled as soon as the state and the tokens' table are in registers, and the updated
//   state stored from registers.
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tma_map.cuh"

namespace gdn2 {

namespace {

__device__ int g_status_decode;

// ---- state element access: 4 consecutive columns ------------------------------------------------

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, c.x, c.y);
}
__device__ __forceinline__ void store4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), c = __floats2bfloat162_rn(x.z, x.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&c);
    *reinterpret_cast<uint2*>(p) = u;
}

// Columns c .. c + 3 of row r of a 128 x 128 slab stored as 128-byte-wide column boxes of 128 rows
// (16 KB each) with the 128-byte swizzle: within each 1024-byte group of 8 rows, the 16-byte chunk
// index of row r is XORed with r mod 8. c is a multiple of 4, so the 4 elements stay in one chunk.
template <typename TS>
__device__ __forceinline__ float4 load4_swizzled(const uint8_t* slab, int r, int c) {
    const int byte = c * static_cast<int>(sizeof(TS));
    const int bo = byte & 127;
    return load4(reinterpret_cast<const TS*>(slab + (byte >> 7) * 16384 + r * 128 +
                                             ((((bo >> 4) ^ (r & 7)) << 4) | (bo & 15))));
}

// state row of batch element bi: the slot map (when given) or bi itself; -1 = inactive
__device__ __forceinline__ int state_row(const int* slots, int n_slots, int bi) {
    if (!slots) return bi;
    const int s = slots[bi];
    return (s >= 0 && s < n_slots) ? s : -1;
}

// ---- register kernel ----------------------------------------------------------------------------

// MINB: blocks per SM the register budget is sized for. Launches of 2-warp CTAs over few heads take 1
// (their occupancy is set by the grid, and the d_k = 128 kernel then holds its state without
// spilling); 8-warp CTAs over many heads take 2.
template <int DK, typename Tin, typename TS, int MINB>
__global__ void __launch_bounds__(256, MINB)
    recurrent_reg_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                         const Tin* __restrict__ g, const Tin* __restrict__ b, const Tin* __restrict__ w,
                         TS* __restrict__ state, const int* __restrict__ slots, int n_slots, Tin* __restrict__ o,
                         int N, int Hk, int Hv, int dv, float scale) {
    constexpr int RPL = DK / 8;  // rows per lane
    const int head = blockIdx.x;
    const int bi = head / Hv;
    const int hv = head - bi * Hv;
    const int hk = hv / (Hv / Hk);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cg = lane & 3;
    const int rg = lane >> 2;
    const int col = blockIdx.y * (blockDim.x >> 1) + warp * 16 + cg * 4;  // 16 columns per warp
    if (col >= dv) return;  // whole warp exits together (dv is a multiple of 16)
    const int row = state_row(slots, n_slots, bi);
    if (row < 0) return;    // inactive batch row: nothing read or written

    TS* S = state + (static_cast<size_t>(row) * Hv + hv) * DK * dv + col;
    float4 s[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) s[i] = load4(S + static_cast<size_t>(rg + 8 * i) * dv);

    for (int t = 0; t < N; ++t) {
        const size_t tk = static_cast<size_t>(bi) * N + t;
        const Tin* qh = q + (tk * Hk + hk) * DK;
        const Tin* kh = k + (tk * Hk + hk) * DK;
        const Tin* gh = g + (tk * Hv + hv) * DK;
        const Tin* bh = b + (tk * Hv + hv) * DK;
        // w.v is loaded with the row scalars, before the reductions it waits for (at small batch the
        // token vectors are often not in L2, and a load after the shuffles would add a memory round
        // trip to the critical path)
        const Tin* vh = v + (tk * Hv + hv) * dv + col;
        const Tin* wh = w + (tk * Hv + hv) * dv + col;
        float wv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wv[c] = to_f32(wh[c]) * to_f32(vh[c]);

        float4 rb = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 rq = make_float4(0.f, 0.f, 0.f, 0.f);
        float kq = 0.f;
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const int r = rg + 8 * i;
            const float a = expf(to_f32(gh[r]));
            const float kk = to_f32(kh[r]);
            const float qq = to_f32(qh[r]);
            const float bk = to_f32(bh[r]) * kk;
            s[i].x *= a;
            s[i].y *= a;
            s[i].z *= a;
            s[i].w *= a;
            rb.x = fmaf(s[i].x, bk, rb.x);
            rb.y = fmaf(s[i].y, bk, rb.y);
            rb.z = fmaf(s[i].z, bk, rb.z);
            rb.w = fmaf(s[i].w, bk, rb.w);
            rq.x = fmaf(s[i].x, qq, rq.x);
            rq.y = fmaf(s[i].y, qq, rq.y);
            rq.z = fmaf(s[i].z, qq, rq.z);
            rq.w = fmaf(s[i].w, qq, rq.w);
            kq = fmaf(kk, qq, kq);
        }
        // sum over the 8 row groups: lanes that differ in bits 2..4
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            rb.x += __shfl_xor_sync(0xffffffffu, rb.x, off);
            rb.y += __shfl_xor_sync(0xffffffffu, rb.y, off);
            rb.z += __shfl_xor_sync(0xffffffffu, rb.z, off);
            rb.w += __shfl_xor_sync(0xffffffffu, rb.w, off);
            rq.x += __shfl_xor_sync(0xffffffffu, rq.x, off);
            rq.y += __shfl_xor_sync(0xffffffffu, rq.y, off);
            rq.z += __shfl_xor_sync(0xffffffffu, rq.z, off);
            rq.w += __shfl_xor_sync(0xffffffffu, rq.w, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }

        float4 d;
        d.x = wv[0] - rb.x;
        d.y = wv[1] - rb.y;
        d.z = wv[2] - rb.z;
        d.w = wv[3] - rb.w;

        if (rg == 0) {
            Tin* oh = o + (tk * Hv + hv) * dv + col;
            oh[0] = from_f32<Tin>(scale * fmaf(kq, d.x, rq.x));
            oh[1] = from_f32<Tin>(scale * fmaf(kq, d.y, rq.y));
            oh[2] = from_f32<Tin>(scale * fmaf(kq, d.z, rq.z));
            oh[3] = from_f32<Tin>(scale * fmaf(kq, d.w, rq.w));
        }
#pragma unroll
        for (int i = 0; i < RPL; ++i) {
            const float kk = to_f32(kh[rg + 8 * i]);  // re-read (L1) rather than hold d_k/8 registers
            s[i].x = fmaf(kk, d.x, s[i].x);
            s[i].y = fmaf(kk, d.y, s[i].y);
            s[i].z = fmaf(kk, d.z, s[i].z);
            s[i].w = fmaf(kk, d.w, s[i].w);
        }
    }
#pragma unroll
    for (int i = 0; i < RPL; ++i) store4(S + static_cast<size_t>(rg + 8 * i) * dv, s[i]);
}

// ---- streaming kernel (d_k = d_v = 128, up to kStreamTokens tokens per call) --------------------

constexpr int kStreamTokens = 4;
constexpr uint32_t kStreamSmemBlock = 232448;  // largest dynamic shared memory of one CTA
constexpr uint32_t kStreamSmemSM = 233472;     // shared memory of one SM (each resident CTA reserves 1 KB)

// Ring geometry for one (token type, state type, tokens per call, CTAs per SM): a slot holds a state
// slab and the call's token vectors; as many slots as fit in the CTA's share (at most 8). bf16 slabs
// are half the bytes: with two CTAs per SM, two heads are computed at once and each CTA still keeps
// two heads loading ahead.
template <typename Tin, typename TS, int NT, int CPS>
struct StreamRing {
    static constexpr uint32_t smem = CPS == 1 ? kStreamSmemBlock : (kStreamSmemSM / CPS - 1024) / 128 * 128;
    // one token: the cross-warp reduction buffer [8 warps][r_b | r_q][128] + [8] k.q
    static constexpr uint32_t red_bytes = NT > 1 ? 0 : (8 * 2 * 128 + 8) * 4;
    static constexpr uint32_t slab = 128 * 128 * sizeof(TS);
    static constexpr uint32_t tok = NT * 6 * 128 * sizeof(Tin);
    static constexpr uint32_t slot = (slab + tok + 127) / 128 * 128;
    // several tokens, per token: [64 d_k row pairs] (alpha, alpha', b.k, b.k') and (q, q', k, k') fp32,
    // two partial sums of k.q, then w.v of the 128 columns (float4 units)
    static constexpr uint32_t tab_f4 = 2 * 64 + 1 + 32;
    static constexpr uint32_t rows_bytes = NT > 1 ? NT * tab_f4 * 16 : 0;
    // several tokens: the slab comes by tensor copies with the 128-byte swizzle, whose shared-memory
    // tiles start on 1024-byte boundaries: the ring is placed on one (at most 1008 bytes of padding)
    static constexpr uint32_t align_pad = NT > 1 ? 1024 : 0;
    static constexpr uint32_t avail = smem - red_bytes - rows_bytes - 256 - align_pad;
    static constexpr int depth = avail / slot > 8 ? 8 : (int)(avail / slot);
    static constexpr uint32_t red_off = depth * slot;
    static constexpr uint32_t rows_off = red_off + red_bytes;
    static constexpr uint32_t bar_off = (rows_off + rows_bytes + 7) / 8 * 8;
};


// Queue the loads of head h into ring slot `slot`: its state slab and the N tokens' six vectors. An
// inactive head (slot map gives no row) completes the slot's barrier phase without loading. One token:
// the slab by one bulk copy (row-major). Several tokens: by tensor copies of 128-byte-wide column
// boxes over all 128 rows with the 128-byte swizzle (smap: [rows x H_v][128][128] of the state), so
// that the warps, each reading 16 columns over 8 rows at a time, read it without bank conflicts.
template <typename Tin, typename TS, int NT, int CPS>
__device__ __forceinline__ void stream_issue(uint8_t* smem_s, uint64_t* bar, int slot, int h, int N, const TS* state,
                                             const int* slots, int n_slots, const Tin* q, const Tin* k,
                                             const Tin* v, const Tin* g, const Tin* b, const Tin* w, int Hk, int Hv,
                                             const CUtensorMap* smap) {
    using R = StreamRing<Tin, TS, NT, CPS>;
    const int bi = h / Hv, hv = h - bi * Hv, hk = hv / (Hv / Hk);
    const int row = state_row(slots, n_slots, bi);
    if (row < 0) {
        mbar_arrive1(bar);
        return;
    }
    constexpr uint32_t vb = 128 * sizeof(Tin);
    mbar_arrive_expect_tx(bar, R::slab + 6 * vb * N);
    uint8_t* sl = smem_s + slot * R::slot;
    if (NT > 1) {
        constexpr int bc = 128 / sizeof(TS);  // columns per 128-byte box row
#pragma unroll
        for (int x = 0; x < 128 / bc; ++x) tma_load_3d(sl + x * 16384, smap, x * bc, 0, row * Hv + hv, bar);
    } else {
        bulk_load(sl, state + (static_cast<size_t>(row) * Hv + hv) * 16384, R::slab, bar);
    }
    for (int t = 0; t < N; ++t) {
        uint8_t* tk = sl + R::slab + t * 6 * vb;
        const size_t tt = static_cast<size_t>(bi) * N + t;
        const size_t kq = (tt * Hk + hk) * 128, gv = (tt * Hv + hv) * 128;
        bulk_load(tk + 0 * vb, q + kq, vb, bar);
        bulk_load(tk + 1 * vb, k + kq, vb, bar);
        bulk_load(tk + 2 * vb, g + gv, vb, bar);
        bulk_load(tk + 3 * vb, b + gv, vb, bar);
        bulk_load(tk + 4 * vb, v + gv, vb, bar);
        bulk_load(tk + 5 * vb, w + gv, vb, bar);
    }
}

// Persistent grid over the heads, one CTA per SM, 8 warps: a ring of state slabs (with the tokens of
// the call) keeps the next depth-1 heads loading and the previous head's store in flight while one
// head is updated. One token: thread (warp, lane) holds rows 16 warp .. 16 warp + 15 x columns
// 4 lane .. 4 lane + 3, and the reductions over d_k go in-thread, then across warps through a shared
// buffer (one block barrier). Several tokens: a warp holds 16 columns over all d_k rows, so the
// reductions stay inside the warp and the tokens run without block barriers; the per-row scalars of
// every token are tabulated once per head.
template <typename Tin, typename TS, int NT, int CPS>
__global__ void __launch_bounds__(256, CPS)
    recurrent_stream_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                            const Tin* __restrict__ g, const Tin* __restrict__ b, const Tin* __restrict__ w,
                            TS* __restrict__ state, const int* __restrict__ slots, int n_slots,
                            Tin* __restrict__ o, int nheads, int N, int Hk, int Hv, float scale, long long wait_ns,
                            const __grid_constant__ CUtensorMap smap) {
    using R = StreamRing<Tin, TS, NT, CPS>;
    static_assert(R::depth >= 1, "stream ring needs a slot");
    static_assert(R::align_pad + R::bar_off + 8 * 8 + 16 <= R::smem, "stream kernel shared memory");
    static_assert(NT == 1 || R::slot % 1024 == 0, "swizzled slabs start on 1024-byte boundaries");
    // ring slots; heads loading ahead. One token: the updated state goes back through its slot, so a
    // slot is refilled once the store of its head has read it (with a single slot the other CTA of the
    // SM covers that gap). Several tokens: a slot is refilled as soon as its head's state and tokens
    // are in registers and the table (the updated state goes from registers to global memory), so
    // every slot loads ahead.
    constexpr int D = R::depth, P = NT > 1 ? D : (D > 1 ? D - 1 : 1);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem_s = smem_raw + (R::align_pad ? (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u : 0u);
    float* red = reinterpret_cast<float*>(smem_s + R::red_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_s + R::bar_off);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, first = blockIdx.x;
    const int count = first < nheads ? (nheads - first + G - 1) / G : 0;

    if (tid == 0) {
        for (int i = 0; i < D; ++i) mbar_init(full + i, 1);
        fence_mbar_init();
        for (int kk = 0; kk < P && kk < count; ++kk)
            stream_issue<Tin, TS, NT, CPS>(smem_s, full + kk, kk, first + kk * G, N, state, slots, n_slots, q, k,
                                           v, g, b, w, Hk, Hv, &smap);
    }
    __syncthreads();

    int kk = 0;
    bool ok = true;
    for (; kk < count; ++kk) {
        const int h = first + kk * G;
        const int bsel = kk % D;
        const uint32_t par = (kk / D) & 1;
        const int bi = h / Hv, hv = h - bi * Hv;
        const int row = state_row(slots, n_slots, bi);

        {  // every thread observes the slot's phase itself; one block vote decides
            const bool got = mbar_wait(full + bsel, par, wait_ns);
            if (!got) {
                atomicOr(&g_status_decode, kStatusTimeout);
                mbar_wait(full + bsel, par, kDefaultWaitNs);
            }
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
        }

        if (NT == 1 && row >= 0) {
            // one token: lanes 0..15 take row 16 warp + lane's q, k, alpha, b.k and pass them round
            // the warp by shuffles; every lane its 4 columns of w.v
            const Tin* tk = reinterpret_cast<const Tin*>(smem_s + bsel * R::slot + R::slab);
            float q_r = 0.f, k_r = 0.f, a_r = 0.f, bk_r = 0.f;
            if (lane < 16) {
                const int rr = 16 * warp + lane;
                q_r = to_f32(tk[rr]);
                k_r = to_f32(tk[128 + rr]);
                a_r = expf(to_f32(tk[256 + rr]));
                bk_r = to_f32(tk[384 + rr]) * k_r;
            }
            float wv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) wv[c] = to_f32(tk[640 + 4 * lane + c]) * to_f32(tk[512 + 4 * lane + c]);
            TS* S = reinterpret_cast<TS*>(smem_s + bsel * R::slot);
            float4 s[16];
            float4 rb = make_float4(0.f, 0.f, 0.f, 0.f), rq = make_float4(0.f, 0.f, 0.f, 0.f);
            float kq = k_r * q_r;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float ai = __shfl_sync(0xffffffffu, a_r, i);
                const float bki = __shfl_sync(0xffffffffu, bk_r, i);
                const float qi = __shfl_sync(0xffffffffu, q_r, i);
                float4 t = load4(S + (16 * warp + i) * 128 + 4 * lane);
                t.x *= ai; t.y *= ai; t.z *= ai; t.w *= ai;
                s[i] = t;
                rb.x = fmaf(t.x, bki, rb.x); rb.y = fmaf(t.y, bki, rb.y); rb.z = fmaf(t.z, bki, rb.z); rb.w = fmaf(t.w, bki, rb.w);
                rq.x = fmaf(t.x, qi, rq.x); rq.y = fmaf(t.y, qi, rq.y); rq.z = fmaf(t.z, qi, rq.z); rq.w = fmaf(t.w, qi, rq.w);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);  // lanes 0..15 hold rows
            reinterpret_cast<float4*>(red + (warp * 2 + 0) * 128)[lane] = rb;
            reinterpret_cast<float4*>(red + (warp * 2 + 1) * 128)[lane] = rq;
            if (lane == 0) red[8 * 2 * 128 + warp] = kq;
            __syncthreads();
            rb = make_float4(0.f, 0.f, 0.f, 0.f);
            rq = make_float4(0.f, 0.f, 0.f, 0.f);
            kq = 0.f;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) {
                const float4 x = reinterpret_cast<const float4*>(red + (w8 * 2 + 0) * 128)[lane];
                const float4 y = reinterpret_cast<const float4*>(red + (w8 * 2 + 1) * 128)[lane];
                rb.x += x.x; rb.y += x.y; rb.z += x.z; rb.w += x.w;
                rq.x += y.x; rq.y += y.y; rq.z += y.z; rq.w += y.w;
                kq += red[8 * 2 * 128 + w8];
            }
            const float d0 = wv[0] - rb.x, d1 = wv[1] - rb.y, d2 = wv[2] - rb.z, d3 = wv[3] - rb.w;
            if (warp == 0) {
                Tin* oh = o + (static_cast<size_t>(bi) * Hv + hv) * 128 + 4 * lane;
                oh[0] = from_f32<Tin>(scale * fmaf(kq, d0, rq.x));
                oh[1] = from_f32<Tin>(scale * fmaf(kq, d1, rq.y));
                oh[2] = from_f32<Tin>(scale * fmaf(kq, d2, rq.z));
                oh[3] = from_f32<Tin>(scale * fmaf(kq, d3, rq.w));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float ki = __shfl_sync(0xffffffffu, k_r, i);
                float4 t = s[i];
                t.x = fmaf(ki, d0, t.x); t.y = fmaf(ki, d1, t.y); t.z = fmaf(ki, d2, t.z); t.w = fmaf(ki, d3, t.w);
                store4(S + (16 * warp + i) * 128 + 4 * lane, t);
            }
            fence_proxy_async_smem();
        }
        if (NT > 1 && row >= 0) {
            // Several tokens. Thread (warp, lane) holds columns 16 warp + 4 cq .. + 3 (cq = lane mod 4) of
            // the d_k row pairs (2p, 2p + 1), p = 8 j + rg (rg = lane / 4, j = 0..7): each fp32 pair of the
            // packed arithmetic is one column over two adjacent rows, so the per-row scalars come as
            // pairs from the table and the reductions over d_k are in-thread, then over the 8 row
            // groups of the warp by shuffles: no block barrier between tokens.
            const uint8_t* tkb = smem_s + bsel * R::slot + R::slab;
            float4* tab = reinterpret_cast<float4*>(smem_s + R::rows_off);
            const int rg = lane >> 2, cq = lane & 3, col = 16 * warp + 4 * cq;
            const uint8_t* S = smem_s + bsel * R::slot;
            uint64_t s[8][4];  // s[j][c]: column col + c, rows (2p, 2p + 1), p = 8 j + rg
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r0 = 2 * (8 * j + rg);
                const float4 x = load4_swizzled<TS>(S, r0, col), y = load4_swizzled<TS>(S, r0 + 1, col);
                s[j][0] = f32x2(x.x, y.x);
                s[j][1] = f32x2(x.y, y.y);
                s[j][2] = f32x2(x.z, y.z);
                s[j][3] = f32x2(x.w, y.w);
            }
            // the table, per token: [64 row pairs] (alpha, alpha', b.k, b.k'), [64] (q, q', k, k'), two
            // partial sums of k.q (one per 32 pairs) and w.v per column; thread tid fills pair and
            // column pair tid mod 64 of token tid / 64
            {
                const int t = tid >> 6, pr = tid & 63;
                if (t < N) {  // warp-uniform: a token spans two whole warps
                    const Tin* tk = reinterpret_cast<const Tin*>(tkb) + t * 6 * 128 + 2 * pr;
                    const float q0 = to_f32(tk[0]), q1 = to_f32(tk[1]), k0 = to_f32(tk[128]), k1 = to_f32(tk[129]);
                    const float a0 = expf(to_f32(tk[256])), a1 = expf(to_f32(tk[257]));
                    const float b0 = to_f32(tk[384]) * k0, b1 = to_f32(tk[385]) * k1;
                    float4* tt = tab + t * R::tab_f4;
                    tt[pr] = make_float4(a0, a1, b0, b1);
                    tt[64 + pr] = make_float4(q0, q1, k0, k1);
                    reinterpret_cast<float2*>(tt + 129)[pr] =
                        make_float2(to_f32(tk[640]) * to_f32(tk[512]), to_f32(tk[641]) * to_f32(tk[513]));
                    float kq = fmaf(k1, q1, k0 * q0);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
                    if (lane == 0) reinterpret_cast<float*>(tt + 128)[pr >> 5] = kq;
                }
            }
            fence_proxy_async_smem();  // the reads of the slot above come before the copy that refills it
            __syncthreads();
            if (tid == 0 && kk + D < count)
                stream_issue<Tin, TS, NT, CPS>(smem_s, full + bsel, bsel, first + (kk + D) * G, N, state, slots,
                                               n_slots, q, k, v, g, b, w, Hk, Hv, &smap);
            for (int t = 0; t < N; ++t) {
                const float4* tt = tab + t * R::tab_f4;
                uint64_t rb[4] = {0, 0, 0, 0}, rq[4] = {0, 0, 0, 0};  // +0.0f pairs (even-row, odd-row parts)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 ab = tt[8 * j + rg], qk = tt[64 + 8 * j + rg];
                    const uint64_t al = f32x2(ab.x, ab.y), bk = f32x2(ab.z, ab.w), qq = f32x2(qk.x, qk.y);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        s[j][c] = mul_f32x2(s[j][c], al);      // alpha
                        rb[c] = fma_f32x2(s[j][c], bk, rb[c]);  // b.k
                        rq[c] = fma_f32x2(s[j][c], qq, rq[c]);  // q
                    }
                }
                // v[0..3] = r_b, v[4..7] = r_q of columns col + 0..3, this row group's part; then a
                // reduce-scatter over the row groups (lane bits 4, 3, 2): row group rg ends with the
                // whole sum of value rg
                float v[8];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float lo, hi;
                    f32x2_split(rb[c], lo, hi);
                    v[c] = lo + hi;
                    f32x2_split(rq[c], lo, hi);
                    v[4 + c] = lo + hi;
                }
                const bool up4 = (rg & 4) != 0, up2 = (rg & 2) != 0, up1 = (rg & 1) != 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float keep = up4 ? v[4 + i] : v[i], give = up4 ? v[i] : v[4 + i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float keep = up2 ? v[2 + i] : v[i], give = up2 ? v[i] : v[2 + i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
                }
                {
                    const float keep = up1 ? v[1] : v[0], give = up1 ? v[0] : v[1];
                    v[0] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
                }
                // row groups 0..3: d of column col + rg; row groups 4..7 take it and write the output
                // of column col + rg - 4
                float dd = 0.f;
                if (rg < 4) dd = reinterpret_cast<const float*>(tt + 129)[col + rg] - v[0];
                const float dx = __shfl_xor_sync(0xffffffffu, dd, 16);
                if (rg >= 4) {
                    const float2 kqp = *reinterpret_cast<const float2*>(tt + 128);
                    const float kq = kqp.x + kqp.y;
                    o[((static_cast<size_t>(bi) * N + t) * Hv + hv) * 128 + col + rg - 4] =
                        from_f32<Tin>(scale * fmaf(kq, dx, v[0]));
                }
                uint64_t d2[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float dc = __shfl_sync(0xffffffffu, dd, 4 * c + cq);
                    d2[c] = f32x2(dc, dc);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 qk = tt[64 + 8 * j + rg];
                    const uint64_t kp = f32x2(qk.z, qk.w);
#pragma unroll
                    for (int c = 0; c < 4; ++c) s[j][c] = fma_f32x2(kp, d2[c], s[j][c]);
                }
            }
            TS* Sg = state + (static_cast<size_t>(row) * Hv + hv) * 16384;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r0 = 2 * (8 * j + rg);
                float x[4], y[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) f32x2_split(s[j][c], x[c], y[c]);
                store4(Sg + r0 * 128 + col, make_float4(x[0], x[1], x[2], x[3]));
                store4(Sg + (r0 + 1) * 128 + col, make_float4(y[0], y[1], y[2], y[3]));
            }
        }
        if (NT > 1) {
            if (row < 0) {  // an inactive head: nothing to read, the slot is free at once
                __syncthreads();  // every thread has passed its wait on the slot's barrier
                if (tid == 0 && kk + D < count)
                    stream_issue<Tin, TS, NT, CPS>(smem_s, full + bsel, bsel, first + (kk + D) * G, N, state,
                                                   slots, n_slots, q, k, v, g, b, w, Hk, Hv, &smap);
            }
            __syncthreads();  // the table is rewritten by the next head
            continue;
        }
        __syncthreads();
        if (tid == 0) {
            if (row >= 0)
                bulk_store(state + (static_cast<size_t>(row) * Hv + hv) * 16384, smem_s + bsel * R::slot, R::slab);
            bulk_commit();  // an empty group for an inactive head keeps the group count in step
            if (kk + P < count) {
                if (D > 1) bulk_wait_read<1>();  // the store of head kk-1 has finished reading the slot it leaves
                else bulk_wait_read<0>();        // single slot: the store of head kk has read it
                const int nb = (kk + P) % D;
                stream_issue<Tin, TS, NT, CPS>(smem_s, full + nb, nb, first + (kk + P) * G, N, state, slots, n_slots,
                                               q, k, v, g, b, w, Hk, Hv, &smap);
            }
        }
    }
    if (tid == 0) {
        if (!ok)  // drain the loads already issued for heads after kk
            for (int j = kk + 1; j < kk + P && j < count; ++j) mbar_wait(full + j % D, (j / D) & 1, kDefaultWaitNs);
        bulk_wait_all();
    }
    __syncthreads();
}

template <typename Tin, typename TS, int NT>
cudaError_t launch_stream(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                          TS* st, const int* slots, int n_slots, void* o, long long heads, int N, int Hk, int Hv,
                          float scale, int nsm, cudaStream_t s) {
    // Two CTAs per SM when each still gets a ring of three slots (bf16 state), or, with several tokens
    // per call (a head's compute is then long next to its copies), when each gets one slot at all.
    constexpr int depth2 = StreamRing<Tin, TS, NT, 2>::avail / StreamRing<Tin, TS, NT, 2>::slot;
    constexpr int CPS = (depth2 >= 3 || (NT > 1 && depth2 >= 1)) ? 2 : 1;
    using R = StreamRing<Tin, TS, NT, CPS>;
    cudaError_t e = cudaFuncSetAttribute(recurrent_stream_kernel<Tin, TS, NT, CPS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)R::smem);
    if (e != cudaSuccess) return e;
    // several tokens: the state pool as [rows x H_v][128 rows][128 columns], 128-byte-wide boxes of 128
    // rows, 128-byte swizzle (unused with one token)
    CUtensorMap smap = {};
    if (NT > 1) {
        const long long rows = slots ? n_slots : heads / Hv;  // an empty pool: no active head, map unused
        const uint64_t dims[3] = {128, 128, static_cast<uint64_t>(rows > 0 ? rows : 1) * Hv};
        const uint64_t strides[2] = {128 * sizeof(TS), 128 * 128 * sizeof(TS)};
        const uint32_t box[3] = {static_cast<uint32_t>(128 / sizeof(TS)), 128, 1};
        if (!make_map(&smap, sizeof(TS) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                      st, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    recurrent_stream_kernel<Tin, TS, NT, CPS><<<CPS * nsm, 256, R::smem, s>>>(
        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
        static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), st, slots, n_slots,
        static_cast<Tin*>(o), static_cast<int>(heads), N, Hk, Hv, scale, wait_limit_ns(), smap);
    return cudaGetLastError();
}

int g_num_sms = 0;

template <typename Tin, typename TS>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     void* state, const int* slots, int n_slots, void* o, int B, int N, int Hk, int Hv, int dk,
                     int dv, float scale, cudaStream_t s) {
    if (g_num_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            g_num_sms = 1;
    }
    const long long heads = static_cast<long long>(B) * Hv;
    TS* st = static_cast<TS*>(state);
    if (N <= kStreamTokens && dk == 128 && dv == 128 && heads >= 4LL * g_num_sms) {
        if (N == 1)
            return launch_stream<Tin, TS, 1>(q, k, v, g, b, w, st, slots, n_slots, o, heads, N, Hk, Hv, scale,
                                             g_num_sms, s);
        return launch_stream<Tin, TS, kStreamTokens>(q, k, v, g, b, w, st, slots, n_slots, o, heads, N, Hk, Hv,
                                                     scale, g_num_sms, s);
    }
    // register kernel: 8 warps (128 columns) per CTA when there are many heads, 2 warps (32
    // columns) otherwise so that small batches still spread over the SMs
    const int wpc = (heads * ((dv + 127) / 128) >= 4LL * g_num_sms) ? 8 : 2;
    const int cols = 16 * wpc;
    const dim3 grid(static_cast<unsigned>(heads), (dv + cols - 1) / cols);
    const dim3 block(32 * (dv >= cols ? wpc : dv / 16));
#define GDN2_DECODE_CASE(DKV)                                                                              \
    case DKV:                                                                                              \
        if (wpc == 8)                                                                                      \
            recurrent_reg_kernel<DKV, Tin, TS, 2><<<grid, block, 0, s>>>(                                  \
                static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),        \
                static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), st,    \
                slots, n_slots, static_cast<Tin*>(o), N, Hk, Hv, dv, scale);                               \
        else                                                                                               \
            recurrent_reg_kernel<DKV, Tin, TS, 1><<<grid, block, 0, s>>>(                                  \
                static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),        \
                static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), st,    \
                slots, n_slots, static_cast<Tin*>(o), N, Hk, Hv, dv, scale);                               \
        break;
    switch (dk) {
        GDN2_DECODE_CASE(16)
        GDN2_DECODE_CASE(32)
        GDN2_DECODE_CASE(64)
        GDN2_DECODE_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef GDN2_DECODE_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const void* q, const void* k, const void* v, const void* g, const void* b,
                             const void* w, void* state, gdn2_dtype state_dt, const int* slots, int n_slots, void* o,
                             int B, int N, int Hk, int Hv, int dk, int dv, float scale, gdn2_dtype dt,
                             cudaStream_t s) {
    if (dt == GDN2_BF16) {
        if (state_dt == GDN2_BF16)
            return launch_t<__nv_bfloat16, __nv_bfloat16>(q, k, v, g, b, w, state, slots, n_slots, o, B, N, Hk, Hv,
                                                           dk, dv, scale, s);
        return launch_t<__nv_bfloat16, float>(q, k, v, g, b, w, state, slots, n_slots, o, B, N, Hk, Hv, dk, dv,
                                              scale, s);
    }
    if (state_dt == GDN2_BF16)
        return launch_t<float, __nv_bfloat16>(q, k, v, g, b, w, state, slots, n_slots, o, B, N, Hk, Hv, dk, dv,
                                              scale, s);
    return launch_t<float, float>(q, k, v, g, b, w, state, slots, n_slots, o, B, N, Hk, Hv, dk, dv, scale, s);
}

int decode_read_clear_status(cudaStream_t s) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status_decode, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    const int zero = 0;
    if (v && cudaMemcpyToSymbolAsync(g_status_decode, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return -1;
    cudaStreamSynchronize(s);
    return v;
}

}  // namespace gdn2

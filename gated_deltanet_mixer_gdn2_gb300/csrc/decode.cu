// decode.cu -- gdn2_recurrent_step: one token against a persistent fp32 state, in place.
//
// Recurrence (burn-gdn2 0.1.5 docs, "Architecture"), regrouped so that the state is read once and
// written once (the same decay -> erase-read -> delta -> rank-1 update -> readout order as the
// autoregressive GDN decode described in the llama.cpp GDN decode study):
//     S' = diag(alpha) S,  r_b = S'^T (b . k),  r_q = S'^T q,  d = w . v - r_b,
//     S  <- S' + k d^T,    o = scale * (r_q + (k . q) d)          [ = scale * S_new^T q ]
//
// Layout: state [B, H_v, d_k, d_v] fp32 (d_v innermost). The d_v columns evolve independently, so
// a warp owns 16 columns of one head across all d_k rows: lane = 8 row groups x 4 column groups,
// each lane holds d_k/8 rows x 4 columns (one 128-bit load / store per row). Reductions over d_k
// are in-thread over the lane's rows, then warp shuffles across the 8 row groups. No shared
// memory, no block barrier; every state byte moves HBM -> registers -> HBM exactly once.
#include "common.cuh"
#include "ptx.cuh"

namespace gdn2 {

namespace {

__device__ int g_status_decode;

template <int DK, typename Tin>
__global__ void __launch_bounds__(256, 2)
    recurrent_step_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                          const Tin* __restrict__ g, const Tin* __restrict__ b, const Tin* __restrict__ w,
                          float* __restrict__ state, Tin* __restrict__ o, int Hk, int Hv, int dv, float scale) {
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

    float* S = state + static_cast<size_t>(head) * DK * dv + col;
    float4 s[RPL];
#pragma unroll
    for (int i = 0; i < RPL; ++i) s[i] = *reinterpret_cast<const float4*>(S + static_cast<size_t>(rg + 8 * i) * dv);

    const Tin* qh = q + (static_cast<size_t>(bi) * Hk + hk) * DK;
    const Tin* kh = k + (static_cast<size_t>(bi) * Hk + hk) * DK;
    const Tin* gh = g + (static_cast<size_t>(bi) * Hv + hv) * DK;
    const Tin* bh = b + (static_cast<size_t>(bi) * Hv + hv) * DK;

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

    const Tin* vh = v + (static_cast<size_t>(bi) * Hv + hv) * dv + col;
    const Tin* wh = w + (static_cast<size_t>(bi) * Hv + hv) * dv + col;
    float4 d;
    d.x = to_f32(wh[0]) * to_f32(vh[0]) - rb.x;
    d.y = to_f32(wh[1]) * to_f32(vh[1]) - rb.y;
    d.z = to_f32(wh[2]) * to_f32(vh[2]) - rb.z;
    d.w = to_f32(wh[3]) * to_f32(vh[3]) - rb.w;

    if (rg == 0) {
        Tin* oh = o + (static_cast<size_t>(bi) * Hv + hv) * dv + col;
        oh[0] = from_f32<Tin>(scale * fmaf(kq, d.x, rq.x));
        oh[1] = from_f32<Tin>(scale * fmaf(kq, d.y, rq.y));
        oh[2] = from_f32<Tin>(scale * fmaf(kq, d.z, rq.z));
        oh[3] = from_f32<Tin>(scale * fmaf(kq, d.w, rq.w));
    }
#pragma unroll
    for (int i = 0; i < RPL; ++i) {
        const float kk = to_f32(kh[rg + 8 * i]);  // re-read (L1) rather than hold d_k/8 registers
        float4 t = s[i];
        t.x = fmaf(kk, d.x, t.x);
        t.y = fmaf(kk, d.y, t.y);
        t.z = fmaf(kk, d.z, t.z);
        t.w = fmaf(kk, d.w, t.w);
        *reinterpret_cast<float4*>(S + static_cast<size_t>(rg + 8 * i) * dv) = t;
    }
}

// ---------------------------------------------------------------------------------------------
// Streaming variant for d_k = d_v = 128 and many heads: a persistent grid (one CTA per SM) walks
// the heads h = blockIdx.x, blockIdx.x + gridDim.x, ...; each 64 KB state slab (contiguous) is
// bulk-copied into a 3-deep shared-memory ring (cp.async.bulk, mbarrier completion), updated in
// place, and bulk-copied back. Loads for the next two heads and the store of the previous one are
// in flight while a head is computed. Warp w owns rows 16w..16w+15, lane l columns 4l..4l+3 (one
// 512-byte row per warp instruction); the d_k reductions finish across the 8 warps in shared memory.
constexpr int kRing = 3;
constexpr uint32_t kSlab = 128 * 128 * 4;
constexpr uint32_t kTokOff = kRing * kSlab;         // per ring slot: q, k, g, b, v, w (128 each)
constexpr uint32_t kTokSlot = 6 * 128 * 4;          // room for fp32 tokens
constexpr uint32_t kRed = kTokOff + kRing * kTokSlot;  // [8 warps][2][128] partial r_b, r_q + [8] k.q
constexpr uint32_t kStreamBar = kRed + 8 * 2 * 128 * 4 + 8 * 4;
constexpr uint32_t kStreamSmem = kStreamBar + 64;

__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(gdst)),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Queue the loads of head h into ring slot `slot`: its 64 KB state slab and its six token vectors.
template <typename Tin>
__device__ __forceinline__ void stream_issue(uint8_t* smem_s, uint64_t* bar, int slot, int h, const float* state,
                                             const Tin* q, const Tin* k, const Tin* v, const Tin* g, const Tin* b,
                                             const Tin* w, int Hk, int Hv) {
    const int bi = h / Hv, hv = h - bi * Hv, hk = hv / (Hv / Hk);
    constexpr uint32_t vb = 128 * sizeof(Tin);
    mbar_arrive_expect_tx(bar, kSlab + 6 * vb);
    bulk_load(smem_s + slot * kSlab, state + static_cast<size_t>(h) * 16384, kSlab, bar);
    uint8_t* tk = smem_s + kTokOff + slot * kTokSlot;
    const size_t kq = (static_cast<size_t>(bi) * Hk + hk) * 128, gv = (static_cast<size_t>(bi) * Hv + hv) * 128;
    bulk_load(tk + 0 * vb, q + kq, vb, bar);
    bulk_load(tk + 1 * vb, k + kq, vb, bar);
    bulk_load(tk + 2 * vb, g + gv, vb, bar);
    bulk_load(tk + 3 * vb, b + gv, vb, bar);
    bulk_load(tk + 4 * vb, v + gv, vb, bar);
    bulk_load(tk + 5 * vb, w + gv, vb, bar);
}

template <typename Tin>
__global__ void __launch_bounds__(256, 1)
    recurrent_step_stream_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                                 const Tin* __restrict__ g, const Tin* __restrict__ b, const Tin* __restrict__ w,
                                 float* __restrict__ state, Tin* __restrict__ o, int nheads, int Hk, int Hv,
                                 float scale, long long wait_ns) {
    extern __shared__ __align__(128) uint8_t smem_s[];
    float* red = reinterpret_cast<float*>(smem_s + kRed);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_s + kStreamBar);
    int* flag = reinterpret_cast<int*>(smem_s + kStreamBar + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, first = blockIdx.x;
    const int count = first < nheads ? (nheads - first + G - 1) / G : 0;

    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) mbar_init(full + i, 1);
        fence_mbar_init();
        for (int kk = 0; kk < 2 && kk < count; ++kk)
            stream_issue(smem_s, full + kk, kk, first + kk * G, state, q, k, v, g, b, w, Hk, Hv);
    }
    __syncthreads();

    int kk = 0;
    bool ok = true;
    for (; kk < count; ++kk) {
        const int h = first + kk * G;
        const int bsel = kk % kRing;
        const int bi = h / Hv, hv = h - bi * Hv;

        if (tid == 0) {
            const bool got = mbar_wait(full + bsel, (kk / kRing) & 1, wait_ns);
            if (!got) {
                atomicOr(&g_status_decode, kStatusTimeout);
                mbar_wait(full + bsel, (kk / kRing) & 1, kDefaultWaitNs);
            }
            *flag = got ? 1 : 0;
        }
        __syncthreads();
        if (!*flag) {
            ok = false;
            break;
        }
        mbar_wait(full + bsel, (kk / kRing) & 1, kDefaultWaitNs);

        // token vectors from the ring: lanes 0..15 take row 16*warp + lane's q, k, alpha, b.k;
        // every lane its 4 columns of w.v
        const Tin* tk = reinterpret_cast<const Tin*>(smem_s + kTokOff + bsel * kTokSlot);
        float q_r = 0.f, k_r = 0.f, a_r = 0.f, bk_r = 0.f;
        if (lane < 16) {
            const int row = 16 * warp + lane;
            q_r = to_f32(tk[row]);
            k_r = to_f32(tk[128 + row]);
            a_r = expf(to_f32(tk[256 + row]));
            bk_r = to_f32(tk[384 + row]) * k_r;
        }
        float wv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) wv[c] = to_f32(tk[640 + 4 * lane + c]) * to_f32(tk[512 + 4 * lane + c]);

        float* S = reinterpret_cast<float*>(smem_s + bsel * kSlab);
        float4 s[16];
        float4 rb = make_float4(0.f, 0.f, 0.f, 0.f), rq = make_float4(0.f, 0.f, 0.f, 0.f);
        float kq = k_r * q_r;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float ai = __shfl_sync(0xffffffffu, a_r, i);
            const float bki = __shfl_sync(0xffffffffu, bk_r, i);
            const float qi = __shfl_sync(0xffffffffu, q_r, i);
            float4 t = reinterpret_cast<const float4*>(S + (16 * warp + i) * 128)[lane];
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
            reinterpret_cast<float4*>(S + (16 * warp + i) * 128)[lane] = t;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_store(state + static_cast<size_t>(h) * 16384, S, kSlab);
            bulk_commit();
            if (kk + 2 < count) {
                bulk_wait_read<1>();  // the store of head kk-1 has finished reading its buffer
                const int nb = (kk + 2) % kRing;
                stream_issue(smem_s, full + nb, nb, first + (kk + 2) * G, state, q, k, v, g, b, w, Hk, Hv);
            }
        }
    }
    if (tid == 0) {
        if (!ok)  // drain the loads already issued for heads after kk
            for (int j = kk + 1; j < kk + 2 && j < count; ++j) mbar_wait(full + j % kRing, (j / kRing) & 1, kDefaultWaitNs);
        bulk_wait_all();
    }
    __syncthreads();
}

int g_num_sms = 0;

template <typename Tin>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     float* state, void* o, int B, int Hk, int Hv, int dk, int dv, float scale, cudaStream_t s) {
    if (g_num_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            g_num_sms = 1;
    }
    const long long heads = static_cast<long long>(B) * Hv;
    if (dk == 128 && dv == 128 && heads >= 4LL * g_num_sms) {
        cudaError_t e = cudaFuncSetAttribute(recurrent_step_stream_kernel<Tin>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
        if (e != cudaSuccess) return e;
        recurrent_step_stream_kernel<Tin><<<g_num_sms, 256, kStreamSmem, s>>>(
            static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),
            static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), state,
            static_cast<Tin*>(o), static_cast<int>(heads), Hk, Hv, scale, wait_limit_ns());
        return cudaGetLastError();
    }
    // register kernel: 8 warps (128 columns) per CTA when there are many heads, 2 warps (32
    // columns) otherwise so that small batches still spread over the SMs
    const int wpc = (heads * ((dv + 127) / 128) >= 4LL * g_num_sms) ? 8 : 2;
    const int cols = 16 * wpc;
    const dim3 grid(static_cast<unsigned>(heads), (dv + cols - 1) / cols);
    const dim3 block(32 * (dv >= cols ? wpc : dv / 16));
#define GDN2_DECODE_CASE(DKV)                                                                              \
    case DKV:                                                                                              \
        recurrent_step_kernel<DKV, Tin><<<grid, block, 0, s>>>(                                            \
            static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v),            \
            static_cast<const Tin*>(g), static_cast<const Tin*>(b), static_cast<const Tin*>(w), state,     \
            static_cast<Tin*>(o), Hk, Hv, dv, scale);                                                      \
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

cudaError_t launch_recurrent_step(const void* q, const void* k, const void* v, const void* g, const void* b,
                                  const void* w, float* state, void* o, int B, int Hk, int Hv, int dk, int dv,
                                  float scale, gdn2_dtype dt, cudaStream_t s) {
    if (dt == GDN2_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, g, b, w, state, o, B, Hk, Hv, dk, dv, scale, s);
    return launch_t<float>(q, k, v, g, b, w, state, o, B, Hk, Hv, dk, dv, scale, s);
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

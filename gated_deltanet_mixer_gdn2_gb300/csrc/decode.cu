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

namespace gdn2 {

namespace {

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
    const int col = blockIdx.y * 128 + warp * 16 + cg * 4;
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

template <typename Tin>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     float* state, void* o, int B, int Hk, int Hv, int dk, int dv, float scale, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(B) * Hv, (dv + 127) / 128);
    const dim3 block(dv >= 128 ? 256 : dv * 2);
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

int decode_read_clear_status(cudaStream_t) { return 0; }  // the decode kernel has no waits

}  // namespace gdn2

// backward_chunk.cu -- gradients of the GDN-2 core in chunked form, fp32 on CUDA cores (the recurrence
// of the burn-gdn2 0.1.5 docs, "Architecture", in the chunked WY form of its "chunked WY decomposition
// (training)" section), chunks of C = 32 tokens.
//
// Per chunk n, with the factors of the fp32 forward (chunk_simt.cu), S = S_n entering the chunk and
// S' = S_{n+1} leaving it:
//     U = T (U0 - K_bar S),  U0 = w.v,  K_bar = b.k.e^G,  W = T K_bar,  T = (I + A)^{-1}
//     O = Q_bar S + M U,     S' = G S + K^^T U,  G = diag(e^{G_last}),  Q_bar = q.e^G,  K^ = k.e^{G_last - G}
//     A_ts = sum_c b_t k_t k_s e^{G_t - G_s} (s < t),   M_ts = sum_c q_t k_s e^{G_t - G_s} (s <= t).
// Reverse mode, with dO~ = scale dO and dS' given:
//     dU  = M^T dO~ + K^ dS'                dS = G dS' + Q_bar^T dO~ - W^T dU      (the chain over chunks)
//     dQ_bar = dO~ S^T   dW = -dU S^T   dK^ = U dS'^T   dgamma = rowsum(dS' . S)   dM = tril(dO~ U^T)
//     dT = dU U0^T + dW K_bar^T   dU0 = T^T dU   dK_bar = T^T dW   dA = -strict_tril(T^T dT T^T)
// and through the elementwise factors to dq, dk, db, dg, dv, dw; every exponential factor of A and M is
// <= 1, so no factor can overflow whatever the decays.
//
// Four launches, all on the caller's stream: the state-independent factors of every chunk
// (factors_simt_kernel in token-major form, plus T); the chain over chunks forward (keeps S_n and U_n)
// and in reverse (keeps dS_{n+1} and dU_n) side by side in one launch (chains_kernel), each chain one
// CTA per (batch-head, 64 columns of d_v) with its state slice in registers; the per-token gradients of every (chunk, head) in parallel (grad_kernel,
// one 512-thread CTA per SM); the sums of dq, dk over each key head's group. Within a chunk the pair
// factors e^{G_t - G_s} of tokens in different 8-token blocks are split at a block edge into two
// factors <= 1.
#include <type_traits>

#include "common.cuh"

namespace gdn2 {
namespace {

constexpr int kD = 128;       // d_k = d_v
constexpr int kCb = 32;       // chunk of the backward

// ---- the two chains over chunks: one CTA of 512 threads per (batch-head, 64 columns of d_v), the
// 128 x 64 state slice in registers (4 x 4 per thread) with a copy in shared memory for the products
// that contract over d_k; the next chunk's factors arrive by cp.async while this chunk is processed.
constexpr int kCT = 512;        // threads of a chain CTA
constexpr int kSl = 64;         // d_v columns per chain CTA
constexpr int kLJ = kSl + 4;    // padded row of [*][64] slices
constexpr int kLW = kD + 4;     // padded row of [32][128] factor rows
constexpr int kLM = kCb + 4;    // padded row of [*][32] arrays (channel-major factors, M)

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void sts4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}
__device__ __forceinline__ float comp(float4 v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
// 16 bytes, or zeros when !valid (nothing is read then)
__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// waits until at most n of this thread's most recent groups are in flight (n folds to a constant when unrolled)
__device__ __forceinline__ void cp_async_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}
// four consecutive elements of a token tensor (global or shared) as fp32
template <typename Tin>
__device__ __forceinline__ float4 ld4_tok(const Tin* p) {
    if constexpr (sizeof(Tin) == 4) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
}
template <typename Tin>
__device__ __forceinline__ void st4_tok(Tin* p, float4 x) {
    if constexpr (sizeof(Tin) == 4) {
        *reinterpret_cast<float4*>(p) = x;
    } else {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&a);
        u.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = u;
    }
}

// Thread roles shared by both chains (16 warps). A shared load that every lane of a half-warp makes
// from one address costs half the wavefronts per value of one whose address differs per lane, so each
// product takes 8 values of one operand from half-warp-uniform addresses and 4 of the other per lane:
//  state products (out [128][64] += sum over the 32 tokens): warp w takes channels 8w .. 8w+7, lane
//    (kh = lane >> 4, jl = lane & 15) columns 4jl .. 4jl+3 over the tokens of parity kh; one exchange
//    adds the two parities and leaves rows 8w + 4kh .. +3 with the lane: its part of the state;
//  rows products (out [32][64], contraction over d_k): tokens 8(w & 3) .. +7, columns 4jl .. +3, d_k
//    slice ks = 2(w >> 2) + kh of 16 channels; one exchange adds the two slices of a warp, shared
//    memory the four warp groups (in a fixed order).
struct ChainRoles {
    int w, kh, jl, iset, ks;
    __device__ explicit ChainRoles(int tid) {
        w = tid >> 5;
        kh = (tid >> 4) & 1;
        jl = tid & 15;
        iset = w & 3;
        ks = 2 * (w >> 2) + kh;
    }
};

// a (8 rows x 4 columns) plus the other half-warp's a; rows 4kh .. 4kh+3 of the sum land in b
__device__ __forceinline__ void half_sum(const float (&a)[8][4], int kh, float (&b)[4][4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float lo = a[r][jj], hi = a[4 + r][jj];
            b[r][jj] = (kh ? hi : lo) + __shfl_xor_sync(0xffffffffu, kh ? lo : hi, 16);
        }
}

// a[r][jj] += x[r] * y[jj] for 8 x values given as two float4
__device__ __forceinline__ void outer8x4(float (&a)[8][4], float4 x0, float4 x1, float4 y) {
    const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        a[r][0] = fmaf(xs[r], y.x, a[r][0]);
        a[r][1] = fmaf(xs[r], y.y, a[r][1]);
        a[r][2] = fmaf(xs[r], y.z, a[r][2]);
        a[r][3] = fmaf(xs[r], y.w, a[r][3]);
    }
}

namespace fc {  // shared-memory map of the forward chain (floats)
constexpr int S = 0;                          // S_n [128][kLJ]
constexpr int U = S + kD * kLJ;               // U [32][kLJ]
constexpr int RED = U + kCb * kLJ;            // [4][32][64] partial rows products of the warp groups
constexpr int BUF = RED + 4 * kCb * kSl;      // two factor buffers
constexpr int WT = 0, KH = WT + kD * kLM, UT = KH + kCb * kLW, GAM = UT + kCb * kLJ, BUF_FLOATS = GAM + kD;
constexpr int TOTAL = BUF + 2 * BUF_FLOATS;
}  // namespace fc

// Forward chain keeping, for every chunk n, S_n (the state entering it) and U_n = U~_n - W_n S_n:
//     S_{n+1} = diag(e^{G_last}) S_n + K^_n^T U_n.
__device__ __forceinline__ void save_chain(const float* __restrict__ ws, const float* __restrict__ s0,
                                           float* __restrict__ s_save, float* __restrict__ u_save, int NC, int bh,
                                           int col0) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const SimtWs L{kD, kD, kCb, true};
    const ChainRoles R(tid);
    const int c_own = 8 * R.w + 4 * R.kh;  // first of the lane's four state rows
    auto prefetch = [&](int n, float* buf) {
        const float* u = ws + ((size_t)bh * NC + n) * L.unit_floats();
        for (int i = tid; i < kD * (kCb / 4); i += kCT) {  // W^T [d_k][C]
            const int r = i >> 3, c4 = 4 * (i & 7);
            cp_async16(buf + fc::WT + r * kLM + c4, u + L.off_wt2() + r * kCb + c4);
        }
        for (int i = tid; i < kCb * (kD / 4); i += kCT) {  // K^ [C][d_k]
            const int r = i >> 5, c4 = 4 * (i & 31);
            cp_async16(buf + fc::KH + r * kLW + c4, u + L.off_kht() + r * kD + c4);
        }
        {   // this CTA's columns of U~, and e^{G_last}
            const int r = tid >> 4, c4 = 4 * (tid & 15);
            cp_async16(buf + fc::UT + r * kLJ + c4, u + L.off_utt() + r * kD + col0 + c4);
        }
        if (tid < kD / 4) cp_async16(buf + fc::GAM + 4 * tid, u + L.off_gam() + 4 * tid);
        cp_async_commit();
    };
    float S[4][4];  // rows c_own + r, columns 4jl + jj of this CTA's slice
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + ((size_t)bh * kD + c_own + r) * kD + col0 + 4 * R.jl)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        S[r][0] = x.x; S[r][1] = x.y; S[r][2] = x.z; S[r][3] = x.w;
        sts4(sm + fc::S + (c_own + r) * kLJ + 4 * R.jl, x);
    }
    prefetch(0, sm + fc::BUF);
    cp_async_wait_all();
    __syncthreads();
    const int fi = tid >> 4, fj = 4 * (tid & 15);  // the (row, column quad) each thread finishes
    for (int n = 0; n < NC; ++n) {
        const float* buf = sm + fc::BUF + (n & 1) * fc::BUF_FLOATS;
        const size_t unit = (size_t)bh * NC + n;
#pragma unroll
        for (int r = 0; r < 4; ++r)  // S_n
            *reinterpret_cast<float4*>(s_save + (unit * kD + c_own + r) * kD + col0 + 4 * R.jl) =
                make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
        if (n + 1 < NC) prefetch(n + 1, sm + fc::BUF + ((n + 1) & 1) * fc::BUF_FLOATS);
        {   // W S_n over this lane's 16 channels
            float a[8][4] = {};
#pragma unroll 4
            for (int cc = 0; cc < 16; ++cc) {
                const int c = 16 * R.ks + cc;
                const float* wt = buf + fc::WT + c * kLM + 8 * R.iset;
                outer8x4(a, lds4(wt), lds4(wt + 4), lds4(sm + fc::S + c * kLJ + 4 * R.jl));
            }
            float b[4][4];
            half_sum(a, R.kh, b);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                sts4(sm + fc::RED + ((R.w >> 2) * kCb + 8 * R.iset + 4 * R.kh + r) * kSl + 4 * R.jl,
                     make_float4(b[r][0], b[r][1], b[r][2], b[r][3]));
        }
        __syncthreads();
        {   // U = U~ - W S_n
            float4 t = lds4(sm + fc::RED + fi * kSl + fj);
#pragma unroll
            for (int g2 = 1; g2 < 4; ++g2) {
                const float4 x = lds4(sm + fc::RED + (g2 * kCb + fi) * kSl + fj);
                t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
            }
            const float4 ut = lds4(buf + fc::UT + fi * kLJ + fj);
            const float4 uu = make_float4(ut.x - t.x, ut.y - t.y, ut.z - t.z, ut.w - t.w);
            sts4(sm + fc::U + fi * kLJ + fj, uu);
            *reinterpret_cast<float4*>(u_save + (unit * kCb + fi) * kD + col0 + fj) = uu;
        }
        __syncthreads();
        {   // S_{n+1} = diag(e^{G_last}) S_n + K^^T U
            float a[8][4] = {};
#pragma unroll 4
            for (int m = 0; m < kCb / 2; ++m) {
                const int i = 2 * m + R.kh;
                const float* kh = buf + fc::KH + i * kLW + 8 * R.w;
                outer8x4(a, lds4(kh), lds4(kh + 4), lds4(sm + fc::U + i * kLJ + 4 * R.jl));
            }
            float b[4][4];
            half_sum(a, R.kh, b);
            const float4 gm = lds4(buf + fc::GAM + c_own);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float gr = comp(gm, r);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) S[r][jj] = fmaf(gr, S[r][jj], b[r][jj]);
                sts4(sm + fc::S + (c_own + r) * kLJ + 4 * R.jl, make_float4(S[r][0], S[r][1], S[r][2], S[r][3]));
            }
        }
        cp_async_wait_all();
        __syncthreads();
    }
}

namespace ac {  // shared-memory map of the reverse chain (floats)
constexpr int R = 0;                          // dS_{n+1} [128][kLJ]
constexpr int DU = R + kD * kLJ;              // dU [32][kLJ]
constexpr int RED = DU + kCb * kLJ;           // [4][32][64] partial rows products of the warp groups
constexpr int BUF = RED + 4 * kCb * kSl;      // two buffers of factors and dO rows
constexpr int KHT = 0, QB = KHT + kD * kLM, W = QB + kCb * kLW, M = W + kCb * kLW, GAM = M + kCb * kLM,
              DO = GAM + kD, BUF_FLOATS = DO + kCb * kLJ;   // dO rows: 272 bytes each whatever the dtype
constexpr int TOTAL = BUF + 2 * BUF_FLOATS;
}  // namespace ac

// dS and dU over the chunks in reverse, with dO~ = scale dO:
//     dU_n = M_n^T dO~_n + K^_n dS_{n+1},   dS_n = diag(e^{G_last}) dS_{n+1} + Q_bar_n^T dO~_n - W_n^T dU_n,
// keeping dS_{n+1} and dU_n of every chunk and writing dS_0.
template <typename Tin>
__device__ __forceinline__ void adjoint_chain(const float* __restrict__ ws, const Tin* __restrict__ dO,
                                              const float* __restrict__ dsT, float* __restrict__ ds0,
                                              float* __restrict__ ds_save, float* __restrict__ du_save, int T, int Hv,
                                              int NC, float scale, int bh, int col0) {
    extern __shared__ __align__(16) float sm[];
    const int bi = bh / Hv, hv = bh - bi * Hv, tid = threadIdx.x;
    const SimtWs L{kD, kD, kCb, true};
    const ChainRoles R(tid);
    const int c_own = 8 * R.w + 4 * R.kh;
    constexpr int kPieces = kSl * (int)sizeof(Tin) / 16;  // 16-byte pieces of one dO row slice
    constexpr int kRowT = kLJ * 4 / (int)sizeof(Tin);      // dO row stride in elements
    auto prefetch = [&](int n, float* buf) {
        const float* u = ws + ((size_t)bh * NC + n) * L.unit_floats();
        for (int i = tid; i < kD * (kCb / 4); i += kCT) {  // K^^T [d_k][C]
            const int r = i >> 3, c4 = 4 * (i & 7);
            cp_async16(buf + ac::KHT + r * kLM + c4, u + L.off_kht2() + r * kCb + c4);
        }
        for (int i = tid; i < 2 * kCb * (kD / 4); i += kCT) {  // Q_bar, W [C][d_k]
            const int m = i >> 10, r = (i >> 5) & (kCb - 1), c4 = 4 * (i & 31);
            cp_async16(buf + (m ? ac::W : ac::QB) + r * kLW + c4, u + (m ? L.off_wt() : L.off_qbt()) + r * kD + c4);
        }
        if (tid < kCb * kCb / 4) {
            const int r = tid >> 3, c4 = 4 * (tid & 7);
            cp_async16(buf + ac::M + r * kLM + c4, u + L.off_m() + r * kCb + c4);
        } else if (tid < kCb * kCb / 4 + kD / 4) {
            const int c4 = 4 * (tid - kCb * kCb / 4);
            cp_async16(buf + ac::GAM + c4, u + L.off_gam() + c4);
        }
        if (tid < kCb * kPieces) {  // dO rows of the chunk, zeros past the end of the sequence
            const int r = tid / kPieces, pc = tid - r * kPieces, tok = n * kCb + r;
            const bool valid = tok < T;
            const Tin* src = dO + (((size_t)bi * T + (valid ? tok : 0)) * Hv + hv) * kD + col0 + pc * (16 / (int)sizeof(Tin));
            cp_async16_zfill(reinterpret_cast<char*>(buf + ac::DO + r * kLJ) + 16 * pc, src, valid);
        }
        cp_async_commit();
    };
    float G[4][4];  // dS_{n+1}: rows c_own + r, columns 4jl + jj of this CTA's slice
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float4 x = dsT ? *reinterpret_cast<const float4*>(dsT + ((size_t)bh * kD + c_own + r) * kD + col0 + 4 * R.jl)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        G[r][0] = x.x; G[r][1] = x.y; G[r][2] = x.z; G[r][3] = x.w;
        sts4(sm + ac::R + (c_own + r) * kLJ + 4 * R.jl, x);
    }
    prefetch(NC - 1, sm + ac::BUF + ((NC - 1) & 1) * ac::BUF_FLOATS);
    cp_async_wait_all();
    __syncthreads();
    const int fi = tid >> 4, fj = 4 * (tid & 15);
    for (int n = NC - 1; n >= 0; --n) {
        const float* buf = sm + ac::BUF + (n & 1) * ac::BUF_FLOATS;
        const Tin* sDO = reinterpret_cast<const Tin*>(buf + ac::DO);
        const size_t unit = (size_t)bh * NC + n;
#pragma unroll
        for (int r = 0; r < 4; ++r)  // dS_{n+1}
            *reinterpret_cast<float4*>(ds_save + (unit * kD + c_own + r) * kD + col0 + 4 * R.jl) =
                make_float4(G[r][0], G[r][1], G[r][2], G[r][3]);
        if (n > 0) prefetch(n - 1, sm + ac::BUF + ((n - 1) & 1) * ac::BUF_FLOATS);
        {   // K^ dS_{n+1} over this lane's 16 channels, M^T dO~ over its 4 tokens
            float a[8][4] = {};
#pragma unroll 4
            for (int cc = 0; cc < 16; ++cc) {
                const int c = 16 * R.ks + cc;
                const float* kt = buf + ac::KHT + c * kLM + 8 * R.iset;
                outer8x4(a, lds4(kt), lds4(kt + 4), lds4(sm + ac::R + c * kLJ + 4 * R.jl));
            }
#pragma unroll
            for (int ll = 0; ll < 4; ++ll) {  // M[l][i] = 0 for l < i
                const int l = 4 * R.ks + ll;
                const float* mr = buf + ac::M + l * kLM + 8 * R.iset;
                float4 ov = ld4_tok(sDO + l * kRowT + 4 * R.jl);
                ov = make_float4(scale * ov.x, scale * ov.y, scale * ov.z, scale * ov.w);
                outer8x4(a, lds4(mr), lds4(mr + 4), ov);
            }
            float b[4][4];
            half_sum(a, R.kh, b);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                sts4(sm + ac::RED + ((R.w >> 2) * kCb + 8 * R.iset + 4 * R.kh + r) * kSl + 4 * R.jl,
                     make_float4(b[r][0], b[r][1], b[r][2], b[r][3]));
        }
        __syncthreads();
        {   // dU
            float4 t = lds4(sm + ac::RED + fi * kSl + fj);
#pragma unroll
            for (int g2 = 1; g2 < 4; ++g2) {
                const float4 x = lds4(sm + ac::RED + (g2 * kCb + fi) * kSl + fj);
                t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
            }
            sts4(sm + ac::DU + fi * kLJ + fj, t);
            *reinterpret_cast<float4*>(du_save + (unit * kCb + fi) * kD + col0 + fj) = t;
        }
        __syncthreads();
        {   // dS_n = diag(e^{G_last}) dS_{n+1} + Q_bar^T dO~ - W^T dU
            float a[8][4] = {};
#pragma unroll 2
            for (int m = 0; m < kCb / 2; ++m) {
                const int i = 2 * m + R.kh;
                const float* qb = buf + ac::QB + i * kLW + 8 * R.w;
                const float* wr = buf + ac::W + i * kLW + 8 * R.w;
                float4 ov = ld4_tok(sDO + i * kRowT + 4 * R.jl);
                ov = make_float4(scale * ov.x, scale * ov.y, scale * ov.z, scale * ov.w);
                float4 dv = lds4(sm + ac::DU + i * kLJ + 4 * R.jl);
                dv = make_float4(-dv.x, -dv.y, -dv.z, -dv.w);
                outer8x4(a, lds4(qb), lds4(qb + 4), ov);
                outer8x4(a, lds4(wr), lds4(wr + 4), dv);
            }
            float b[4][4];
            half_sum(a, R.kh, b);
            const float4 gm = lds4(buf + ac::GAM + c_own);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float gr = comp(gm, r);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) G[r][jj] = fmaf(gr, G[r][jj], b[r][jj]);
                sts4(sm + ac::R + (c_own + r) * kLJ + 4 * R.jl, make_float4(G[r][0], G[r][1], G[r][2], G[r][3]));
            }
        }
        cp_async_wait_all();
        __syncthreads();
    }
    if (ds0)
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(ds0 + ((size_t)bh * kD + c_own + r) * kD + col0 + 4 * R.jl) =
                make_float4(G[r][0], G[r][1], G[r][2], G[r][3]);
}

// ---- grad_kernel: every per-token gradient of one (chunk, head), one CTA of 512 threads per SM
constexpr int kGT = 512;          // threads
constexpr int kLS = 132;          // padded row of its [*][128] arrays (16-byte aligned rows)
constexpr int kLQ = 36;           // padded row of its [32][32] arrays
constexpr int kSlot = kCb * kLS;  // one [32][128] array

namespace gk {  // shared-memory map (floats); arrays that are dead by the time another is written share room
constexpr int slot(int i) { return i * kSlot; }
constexpr int DS = 0, SS = kD * kLS;  // dS_{n+1}, S_n [128][kLS]: slots 0-3 and 4-7 while the big products run
constexpr int DKH = slot(0), DQB = slot(1), DW = slot(2), XX = slot(2), U0 = slot(3), KB = slot(3), G = slot(4),
              K = slot(5), BETA = slot(6), Q = slot(7);
constexpr int U = slot(8), DKB = slot(8), DU = slot(9), ZV = slot(9), DO = slot(10), YY = slot(10);
constexpr int TM = slot(11);                  // T [32][kLQ]
constexpr int DT = TM + kCb * kLQ;            // dT
constexpr int PP = DT + kCb * kLQ;            // T^T dT
constexpr int DA = PP + kCb * kLQ, DAT = DA + kCb * kLQ, DM = DAT + kCb * kLQ, DMT = DM + kCb * kLQ;
constexpr int DGP = DMT + kCb * kLQ;          // [128] rowsum(dS' . S)
constexpr int DGL = DGP + kD;                 // [4][128] partial sums of dK^ . K^
constexpr int DBT = DGL + 4 * kD;             // [4][128] sums of dG over each block of 8 tokens
constexpr int TOTAL = DBT + 4 * kD;
}  // namespace gk

// The local gradients of one (chunk n, batch-head bh), given S_n, dS_{n+1}, U, dU and T of the chunk:
//   1. dK^ = U dS'^T, dQ_bar = dO~ S^T, dW = -dU S^T, dgamma = rowsum(dS' . S)  (K = d_v, register tiles of
//      8 channels x 4 tokens; S and dS' arrive in eight 16-column groups that the products consume in order)
//   2. dM = tril(dO~ U^T), dT = dU U0^T + dW K_bar^T, dK_bar = T^T dW, dU0 = T^T dU (-> dv, dw)
//   3. P = T^T dT, dA = -strict_tril(P T^T)
//   4. the pair terms X, Y (thread = channel and block of 8 tokens t) and Z + V (block of 8 tokens s), each
//      factor e^{G_t - G_s} of two tokens in different blocks split at a block edge r between them into
//      e^{G_t - G_r} e^{G_r - G_s}, both <= 1, so the sums over the other block are plain products
//   5. dq, dk (fp32, per value head), db and dg = reverse cumulative sum of dG plus dG_last.
// Both chains in one launch: blockIdx.y < kD / kSl runs the backward chain on column slice blockIdx.y,
// the rest the forward chain (they only read the factors and write disjoint buffers, so they run side
// by side; the longer backward chain has the lower block indices and starts first).
template <typename Tin>
__global__ void __launch_bounds__(kCT, 1) chains_kernel(const float* __restrict__ ws, const float* __restrict__ s0,
                                                       float* __restrict__ s_save, float* __restrict__ u_save,
                                                       const Tin* __restrict__ dO, const float* __restrict__ dsT,
                                                       float* __restrict__ ds0, float* __restrict__ ds_save,
                                                       float* __restrict__ du_save, int T, int Hv, int NC, float scale) {
    constexpr int kSlices = kD / kSl;
    if (blockIdx.y < kSlices)
        adjoint_chain<Tin>(ws, dO, dsT, ds0, ds_save, du_save, T, Hv, NC, scale, blockIdx.x, blockIdx.y * kSl);
    else
        save_chain(ws, s0, s_save, u_save, NC, blockIdx.x, (blockIdx.y - kSlices) * kSl);
}

template <typename Tin>
__global__ void __launch_bounds__(kGT, 1) grad_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                      const Tin* __restrict__ v, const Tin* __restrict__ g,
                                                      const Tin* __restrict__ b, const Tin* __restrict__ w,
                                                      const Tin* __restrict__ dO, const float* __restrict__ t_ws,
                                                      const float* __restrict__ s_save, const float* __restrict__ u_save,
                                                      const float* __restrict__ ds_save,
                                                      const float* __restrict__ du_save, float* __restrict__ dq_ws,
                                                      float* __restrict__ dk_ws, Tin* __restrict__ dv,
                                                      Tin* __restrict__ dg, Tin* __restrict__ db, Tin* __restrict__ dw,
                                                      int T, int Hk, int Hv, float scale) {
    extern __shared__ __align__(16) float sm[];
    const int n = blockIdx.x, bh = blockIdx.y, NC = gridDim.x;
    const int bi = bh / Hv, hv = bh - bi * Hv, hk = hv / (Hv / Hk);
    const int tid = threadIdx.x;
    const size_t unit = (size_t)bh * NC + n;
    auto vrow = [&](int t) { return (((size_t)bi * T + n * kCb + t) * Hv + hv) * kD; };   // v-like token row
    auto krow = [&](int t) { return (((size_t)bi * T + n * kCb + t) * Hk + hk) * kD; };   // k-like token row
    const int nvalid = min(kCb, T - n * kCb);

    float4 do4[2];  // this thread's dO elements, in flight ahead of the copies
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int t = (tid >> 5) + 16 * pass;
        do4[pass] = t < nvalid ? ld4_tok(dO + vrow(t) + 4 * (tid & 31)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // ---- U, dU, T, then S and dS' in eight groups of 16 columns
    {
        const float* Ug = u_save + unit * kCb * kD;
        const float* DUg = du_save + unit * kCb * kD;
        for (int i = tid; i < kCb * kD / 4; i += kGT) {
            const int t = i >> 5, c4 = 4 * (i & 31);
            cp_async16(sm + gk::U + t * kLS + c4, Ug + t * kD + c4);
            cp_async16(sm + gk::DU + t * kLS + c4, DUg + t * kD + c4);
        }
        if (tid < kCb * kCb / 4) {
            const int r = tid >> 3, c4 = 4 * (tid & 7);
            cp_async16(sm + gk::TM + r * kLQ + c4, t_ws + unit * kCb * kCb + r * kCb + c4);
        }
    }
    const float* Sg = s_save + unit * kD * kD;
    const float* DSg = ds_save + unit * kD * kD;
    auto issue_block = [&](int jb) {  // columns 16jb .. 16jb+15 of S and dS'
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int id = tid + kGT * m;  // 2 matrices x 128 rows x 4 pieces of 16 bytes
            const int row = (id >> 2) & (kD - 1), c4 = 16 * jb + 4 * (id & 3);
            if (id < 512)
                cp_async16(sm + gk::DS + row * kLS + c4, DSg + row * kD + c4);
            else
                cp_async16(sm + gk::SS + row * kLS + c4, Sg + row * kD + c4);
        }
    };
#pragma unroll
    for (int jb = 0; jb < 8; ++jb) {  // all in flight at once (measured faster than a few groups ahead)
        issue_block(jb);
        cp_async_commit();  // group 0 also carries U, dU and T
    }
    {   // scaled dO, loaded before the copies were queued (zero past the end of the sequence)
        const int c4 = 4 * (tid & 31);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
            sts4(sm + gk::DO + ((tid >> 5) + 16 * pass) * kLS + c4,
                 make_float4(scale * do4[pass].x, scale * do4[pass].y, scale * do4[pass].z, scale * do4[pass].w));
    }

    // ---- 1. dK^ = U dS'^T (warps 0-3), dQ_bar = dO~ S^T (4-7), dW = -dU S^T (8-11), contraction over d_v:
    //      a quarter-warp takes 8 channels 4 apart (one shared address per quarter, the four quarters in
    //      different banks), its lanes 4 tokens each;
    //      warps 12-15 form rowsum(dS' . S)
    {
        const int warp = tid >> 5, lane = tid & 31, prod = warp >> 2;
        const int c0 = 32 * (warp & 3) + (lane >> 3), tq = lane & 7;  // channels c0 + 4i, tokens tq + 8i
        const float* Am = sm + (prod == 0 ? gk::DS : gk::SS) + c0 * kLS;
        const float* Bm = sm + (prod == 0 ? gk::U : prod == 1 ? gk::DO : gk::DU) + tq * kLS;
        float acc[8][4] = {};
        float dgam = 0.f;
#pragma unroll 1
        for (int jb = 0; jb < 8; ++jb) {  // kept rolled: the body is large (instruction-fetch stalls)
            cp_async_wait(7 - jb);  // groups 0 .. jb have landed
            __syncthreads();
            if (jb == 4) {  // the token inputs read after the products: into L2 now, one 128-byte line each
                constexpr int kLines = kD * (int)sizeof(Tin) / 128;  // lines per token row
                for (int i = tid; i < 6 * kCb * kLines; i += kGT) {
                    const int ten = i / (kCb * kLines), row = (i / kLines) % kCb, line = i % kLines;
                    if (row < nvalid) {
                        const Tin* base = ten == 0 ? w : ten == 1 ? v : ten == 2 ? g : ten == 3 ? b : ten == 4 ? k : q;
                        const size_t off = (ten >= 4 ? krow(row) : vrow(row)) + line * (128 / (int)sizeof(Tin));
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
                    }
                }
            }
            if (prod < 3) {
#pragma unroll
                for (int jq = 0; jq < 4; ++jq) {
                    const int j = 16 * jb + 4 * jq;
                    float4 av[8], bv[4];
#pragma unroll
                    for (int ci = 0; ci < 8; ++ci) av[ci] = lds4(Am + 4 * ci * kLS + j);
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) bv[ti] = lds4(Bm + 8 * ti * kLS + j);
#pragma unroll
                    for (int ci = 0; ci < 8; ++ci)
#pragma unroll
                        for (int ti = 0; ti < 4; ++ti) acc[ci][ti] = dot4(av[ci], bv[ti], acc[ci][ti]);
                }
            } else {
                const int c = tid - 3 * 128;
#pragma unroll
                for (int jq = 0; jq < 4; ++jq) {
                    const int j = 16 * jb + 4 * jq;
                    dgam = dot4(lds4(sm + gk::DS + c * kLS + j), lds4(sm + gk::SS + c * kLS + j), dgam);
                }
            }
        }
        __syncthreads();  // S, dS' read out: their room takes the per-token arrays
        if (prod < 3) {
            float* dst = sm + (prod == 0 ? gk::DKH : prod == 1 ? gk::DQB : gk::DW);
            const float sg = prod == 2 ? -1.f : 1.f;
#pragma unroll
            for (int ci = 0; ci < 8; ++ci)
#pragma unroll
                for (int ti = 0; ti < 4; ++ti) dst[(tq + 8 * ti) * kLS + c0 + 4 * ci] = sg * acc[ci][ti];
        } else {
            sm[gk::DGP + tid - 3 * 128] = dgam;
        }
    }
    {   // token inputs: U0 = w.v, g, k, b.k, q (zero past the end of the sequence)
        const int c4 = 4 * (tid & 31);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int t = (tid >> 5) + 16 * pass;
            float4 xw = make_float4(0.f, 0.f, 0.f, 0.f), xv = xw, xg = xw, xk = xw, xb = xw, xq = xw;
            if (t < nvalid) {
                xw = ld4_tok(w + vrow(t) + c4);
                xv = ld4_tok(v + vrow(t) + c4);
                xg = ld4_tok(g + vrow(t) + c4);
                xb = ld4_tok(b + vrow(t) + c4);
                xk = ld4_tok(k + krow(t) + c4);
                xq = ld4_tok(q + krow(t) + c4);
            }
            const int o = t * kLS + c4;
            sts4(sm + gk::U0 + o, make_float4(xw.x * xv.x, xw.y * xv.y, xw.z * xv.z, xw.w * xv.w));
            // gates floored as in the forward (a full reset keeps every cumulative sum finite)
            sts4(sm + gk::G + o, make_float4(fmaxf(xg.x, kGateFloor), fmaxf(xg.y, kGateFloor), fmaxf(xg.z, kGateFloor),
                                             fmaxf(xg.w, kGateFloor)));
            sts4(sm + gk::K + o, xk);
            sts4(sm + gk::BETA + o, make_float4(xb.x * xk.x, xb.y * xk.y, xb.z * xk.z, xb.w * xk.w));
            sts4(sm + gk::Q + o, xq);
        }
    }
    __syncthreads();

    // ---- 2. dM = tril(dO~ U^T) (threads 0-255), dT1 = dU U0^T (256-511): 2 x 2 tiles over d_v; warps 0-3 first
    //      form the cumulative log-decay G per channel
    if (tid < kD) {
        float acc = 0.f;
        for (int t = 0; t < kCb; ++t) {
            acc += sm[gk::G + t * kLS + tid];
            sm[gk::G + t * kLS + tid] = acc;
        }
    }
    const int prod = tid >> 8, tile = tid & 255;
    const int tp = tile >> 4, sp = tile & 15;  // tokens {tp, tp + 16} x {sp, sp + 16}
    float pt[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    {
        const float* A = sm + (prod ? gk::DU : gk::DO);
        const float* Bm = sm + (prod ? gk::U0 : gk::U);
#pragma unroll 4
        for (int j = 0; j < kD; j += 4) {
            const float4 a0 = lds4(A + tp * kLS + j), a1 = lds4(A + (tp + 16) * kLS + j);
            const float4 b0 = lds4(Bm + sp * kLS + j), b1 = lds4(Bm + (sp + 16) * kLS + j);
            pt[0][0] = dot4(a0, b0, pt[0][0]);
            pt[1][0] = dot4(a1, b0, pt[1][0]);
            pt[1][1] = dot4(a1, b1, pt[1][1]);
            if (prod) pt[0][1] = dot4(a0, b1, pt[0][1]);  // above the diagonal for dM
        }
    }
    if (prod == 0)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = tp + 16 * i, s2 = sp + 16 * j;
                const float x = s2 <= t ? pt[i][j] : 0.f;
                sm[gk::DM + t * kLQ + s2] = x;
                sm[gk::DMT + s2 * kLQ + t] = x;
            }
    __syncthreads();
    {   // K_bar = b.k.e^G in place of U0
        const int c4 = 4 * (tid & 31);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int o = ((tid >> 5) + 16 * pass) * kLS + c4;
            const float4 be = lds4(sm + gk::BETA + o), gg = lds4(sm + gk::G + o);
            sts4(sm + gk::KB + o, make_float4(be.x * __expf(gg.x), be.y * __expf(gg.y), be.z * __expf(gg.z),
                                              be.w * __expf(gg.w)));
        }
    }
    __syncthreads();

    // ---- dT = dT1 + dW K_bar^T (threads 256-511); dK_bar = T^T dW, dU0 = T^T dU -> dv, dw (threads 0-255)
    if (prod) {
#pragma unroll 4
        for (int c = 0; c < kD; c += 4) {
            const float4 a0 = lds4(sm + gk::DW + tp * kLS + c), a1 = lds4(sm + gk::DW + (tp + 16) * kLS + c);
            const float4 b0 = lds4(sm + gk::KB + sp * kLS + c), b1 = lds4(sm + gk::KB + (sp + 16) * kLS + c);
            pt[0][0] = dot4(a0, b0, pt[0][0]);
            pt[0][1] = dot4(a0, b1, pt[0][1]);
            pt[1][0] = dot4(a1, b0, pt[1][0]);
            pt[1][1] = dot4(a1, b1, pt[1][1]);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) sm[gk::DT + (tp + 16 * i) * kLQ + sp + 16 * j] = pt[i][j];
    } else {
        const int c0 = 4 * (tile & 31), tq = tile >> 5;  // tokens tq + 8i, i = 0..3
        float4 aKb[4], aU0[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) aKb[i] = aU0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sg = 0; sg < 4; ++sg)
#pragma unroll 4
            for (int ss = 0; ss < 8; ++ss) {
                const int s2 = 8 * sg + ss;
                const float4 w4 = lds4(sm + gk::DW + s2 * kLS + c0), u4 = lds4(sm + gk::DU + s2 * kLS + c0);
#pragma unroll
                for (int i = 0; i <= sg; ++i) {  // T[s][t] = 0 for t > s
                    const float tt = sm[gk::TM + s2 * kLQ + tq + 8 * i];
                    aKb[i].x = fmaf(tt, w4.x, aKb[i].x); aKb[i].y = fmaf(tt, w4.y, aKb[i].y);
                    aKb[i].z = fmaf(tt, w4.z, aKb[i].z); aKb[i].w = fmaf(tt, w4.w, aKb[i].w);
                    aU0[i].x = fmaf(tt, u4.x, aU0[i].x); aU0[i].y = fmaf(tt, u4.y, aU0[i].y);
                    aU0[i].z = fmaf(tt, u4.z, aU0[i].z); aU0[i].w = fmaf(tt, u4.w, aU0[i].w);
                }
            }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = tq + 8 * i;
            sts4(sm + gk::DKB + t * kLS + c0, aKb[i]);
            if (t < nvalid) {
                const float4 w4 = ld4_tok(w + vrow(t) + c0), v4 = ld4_tok(v + vrow(t) + c0);
                const float4 d = aU0[i];
                st4_tok(dv + vrow(t) + c0, make_float4(w4.x * d.x, w4.y * d.y, w4.z * d.z, w4.w * d.w));
                st4_tok(dw + vrow(t) + c0, make_float4(v4.x * d.x, v4.y * d.y, v4.z * d.z, v4.w * d.w));
            }
        }
    }
    __syncthreads();

    // ---- 3. P = T^T dT, dA = -strict_tril(P T^T): thread = row t and columns s, s + 16
    const int rt = tid >> 4, rs = tid & 15;
    {
        float p0 = 0.f, p1 = 0.f;
        for (int r = rt; r < kCb; ++r) {
            const float tt = sm[gk::TM + r * kLQ + rt];
            p0 = fmaf(tt, sm[gk::DT + r * kLQ + rs], p0);
            p1 = fmaf(tt, sm[gk::DT + r * kLQ + rs + 16], p1);
        }
        sm[gk::PP + rt * kLQ + rs] = p0;
        sm[gk::PP + rt * kLQ + rs + 16] = p1;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int s2 = rs + 16 * h;
        float a = 0.f;
        if (s2 < rt)
            for (int r = 0; r <= s2; ++r) a = fmaf(sm[gk::PP + rt * kLQ + r], sm[gk::TM + s2 * kLQ + r], a);
        sm[gk::DA + rt * kLQ + s2] = -a;
        sm[gk::DAT + s2 * kLQ + rt] = -a;
    }
    __syncthreads();

    // ---- 4. pair terms. Thread = channel c, half h: blocks {0, 3} (h = 0) or {1, 2}; side 0 forms X, Y of
    //      its blocks' tokens, side 1 forms Z + V
    {
        const int c = tid & (kD - 1), h = (tid >> 7) & 1, side = tid >> 8;
        const float* sG = sm + gk::G + c;
        const float* sK = sm + gk::K + c;
        const float* sB = sm + gk::BETA + c;
        const float* sQ = sm + gk::Q + c;
#pragma unroll 1
        for (int rep = 0; rep < 2; ++rep) {
            const int blk = h ? 1 + rep : 3 * rep;
            const int t0 = 8 * blk;
            float Gb[8], xb[8], A1[8], A2[8];
            if (side == 0) {  // X_t = sum_{s<t} dA_ts k_s e^{G_t-G_s};  Y_t = sum_{s<=t} dM_ts k_s e^{G_t-G_s}
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    Gb[i] = sG[(t0 + i) * kLS];
                    xb[i] = sK[(t0 + i) * kLS];
                    A1[i] = 0.f;
                    A2[i] = sm[gk::DM + (t0 + i) * kLQ + t0 + i] * xb[i];
                }
                if (blk > 0) {  // s in earlier blocks, split at r = t0: e^{G_t - G_r} e^{G_r - G_s}
                    float ax[8], ay[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) ax[i] = ay[i] = 0.f;
                    const float Gr = Gb[0];
#pragma unroll 2
                    for (int s2 = 0; s2 < t0; ++s2) {
                        const float ks = sK[s2 * kLS] * __expf(Gr - sG[s2 * kLS]);
                        const float4 a0 = lds4(sm + gk::DAT + s2 * kLQ + t0), a1 = lds4(sm + gk::DAT + s2 * kLQ + t0 + 4);
                        const float4 m0 = lds4(sm + gk::DMT + s2 * kLQ + t0), m1 = lds4(sm + gk::DMT + s2 * kLQ + t0 + 4);
                        ax[0] = fmaf(a0.x, ks, ax[0]); ax[1] = fmaf(a0.y, ks, ax[1]);
                        ax[2] = fmaf(a0.z, ks, ax[2]); ax[3] = fmaf(a0.w, ks, ax[3]);
                        ax[4] = fmaf(a1.x, ks, ax[4]); ax[5] = fmaf(a1.y, ks, ax[5]);
                        ax[6] = fmaf(a1.z, ks, ax[6]); ax[7] = fmaf(a1.w, ks, ax[7]);
                        ay[0] = fmaf(m0.x, ks, ay[0]); ay[1] = fmaf(m0.y, ks, ay[1]);
                        ay[2] = fmaf(m0.z, ks, ay[2]); ay[3] = fmaf(m0.w, ks, ay[3]);
                        ay[4] = fmaf(m1.x, ks, ay[4]); ay[5] = fmaf(m1.y, ks, ay[5]);
                        ay[6] = fmaf(m1.z, ks, ay[6]); ay[7] = fmaf(m1.w, ks, ay[7]);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float et = __expf(Gb[i] - Gr);
                        A1[i] = fmaf(et, ax[i], A1[i]);
                        A2[i] = fmaf(et, ay[i], A2[i]);
                    }
                }
#pragma unroll
                for (int i = 1; i < 8; ++i)  // s in the same block, s < t
#pragma unroll
                    for (int j = 0; j < i; ++j) {
                        const float ks = xb[j] * __expf(Gb[i] - Gb[j]);
                        A1[i] = fmaf(sm[gk::DA + (t0 + i) * kLQ + t0 + j], ks, A1[i]);
                        A2[i] = fmaf(sm[gk::DM + (t0 + i) * kLQ + t0 + j], ks, A2[i]);
                    }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    sm[gk::XX + (t0 + i) * kLS + c] = A1[i];
                    sm[gk::YY + (t0 + i) * kLS + c] = A2[i];
                }
            } else {  // Z_s = sum_{u>s} dA_us b_u k_u e^{G_u-G_s};  V_s = sum_{u>=s} dM_us q_u e^{G_u-G_s}
                float qb[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    Gb[i] = sG[(t0 + i) * kLS];
                    xb[i] = sB[(t0 + i) * kLS];
                    qb[i] = sQ[(t0 + i) * kLS];
                    A1[i] = 0.f;
                    A2[i] = sm[gk::DM + (t0 + i) * kLQ + t0 + i] * qb[i];
                }
                if (blk < 3) {  // u in later blocks, split at r = t0 + 7: e^{G_u - G_r} e^{G_r - G_s}
                    float az[8], av[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) az[i] = av[i] = 0.f;
                    const float Gr = Gb[7];
#pragma unroll 2
                    for (int u2 = t0 + 8; u2 < kCb; ++u2) {
                        const float eu = __expf(sG[u2 * kLS] - Gr);
                        const float bu = sB[u2 * kLS] * eu, qu = sQ[u2 * kLS] * eu;
                        const float4 a0 = lds4(sm + gk::DA + u2 * kLQ + t0), a1 = lds4(sm + gk::DA + u2 * kLQ + t0 + 4);
                        const float4 m0 = lds4(sm + gk::DM + u2 * kLQ + t0), m1 = lds4(sm + gk::DM + u2 * kLQ + t0 + 4);
                        az[0] = fmaf(a0.x, bu, az[0]); az[1] = fmaf(a0.y, bu, az[1]);
                        az[2] = fmaf(a0.z, bu, az[2]); az[3] = fmaf(a0.w, bu, az[3]);
                        az[4] = fmaf(a1.x, bu, az[4]); az[5] = fmaf(a1.y, bu, az[5]);
                        az[6] = fmaf(a1.z, bu, az[6]); az[7] = fmaf(a1.w, bu, az[7]);
                        av[0] = fmaf(m0.x, qu, av[0]); av[1] = fmaf(m0.y, qu, av[1]);
                        av[2] = fmaf(m0.z, qu, av[2]); av[3] = fmaf(m0.w, qu, av[3]);
                        av[4] = fmaf(m1.x, qu, av[4]); av[5] = fmaf(m1.y, qu, av[5]);
                        av[6] = fmaf(m1.z, qu, av[6]); av[7] = fmaf(m1.w, qu, av[7]);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float es = __expf(Gr - Gb[i]);
                        A1[i] = fmaf(es, az[i], A1[i]);
                        A2[i] = fmaf(es, av[i], A2[i]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 7; ++i)  // u in the same block, u > s
#pragma unroll
                    for (int j = i + 1; j < 8; ++j) {
                        const float e = __expf(Gb[j] - Gb[i]);
                        A1[i] = fmaf(sm[gk::DA + (t0 + j) * kLQ + t0 + i], xb[j] * e, A1[i]);
                        A2[i] = fmaf(sm[gk::DM + (t0 + j) * kLQ + t0 + i], qb[j] * e, A2[i]);
                    }
#pragma unroll
                for (int i = 0; i < 8; ++i) sm[gk::ZV + (t0 + i) * kLS + c] = A1[i] + A2[i];
            }
        }
    }
    __syncthreads();

    // ---- 5. back to the inputs: thread = channel c, block of 8 tokens; then dg_t = sum_{s >= t} dG_s +
    //      dG_last, dG_last = sum_t dK^.K^ + rowsum(dS'.S) e^{G_last}, from suffix sums inside each block
    //      plus the totals of the later blocks
    {
        const int c = tid & (kD - 1), blk = tid >> 7;
        const float Glast = sm[gk::G + (kCb - 1) * kLS + c];
        float dkk = 0.f, dGb[8], bb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * blk + i;
            bb[i] = t < nvalid ? to_f32(b[vrow(t) + c]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * blk + i, o = t * kLS + c;
            const float G = sm[gk::G + o], eG = __expf(G), eH = __expf(Glast - G);
            const float qq = sm[gk::Q + o], kk = sm[gk::K + o], be = sm[gk::BETA + o], kb = sm[gk::KB + o];
            const float dqb = sm[gk::DQB + o], dkb = sm[gk::DKB + o], dkh = sm[gk::DKH + o];
            const float x = sm[gk::XX + o], y = sm[gk::YY + o], zv = sm[gk::ZV + o];
            const float dbeta = fmaf(dkb, eG, x);
            dGb[i] = dqb * qq * eG + dkb * kb - dkh * kk * eH + be * x + qq * y - kk * zv;
            dkk = fmaf(dkh, kk * eH, dkk);
            if (t < nvalid) {
                const size_t vh = vrow(t) + c;
                dq_ws[vh] = fmaf(dqb, eG, y);
                dk_ws[vh] = fmaf(dkh, eH, zv) + dbeta * bb[i];
                db[vh] = from_f32<Tin>(dbeta * kk);
            }
        }
        float run = 0.f;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            run += dGb[i];
            dGb[i] = run;
        }
        sm[gk::DGL + blk * kD + c] = dkk;
        sm[gk::DBT + blk * kD + c] = run;
        __syncthreads();
        float off = (sm[gk::DGL + c] + sm[gk::DGL + kD + c]) + (sm[gk::DGL + 2 * kD + c] + sm[gk::DGL + 3 * kD + c]);
        off = fmaf(sm[gk::DGP + c], __expf(Glast), off);
        for (int b2 = 3; b2 > blk; --b2) off += sm[gk::DBT + b2 * kD + c];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * blk + i;
            if (t < nvalid) dg[vrow(t) + c] = from_f32<Tin>(dGb[i] + off);
        }
    }
}

// dq, dk of key head h_k = sums over the value heads of its group
template <typename Tout>
__global__ void __launch_bounds__(256) group_sum2_kernel(const float* __restrict__ dq_ws, const float* __restrict__ dk_ws,
                                                        Tout* __restrict__ dq, Tout* __restrict__ dk, long long rows,
                                                        int Hk, int Hv) {
    const int group = Hv / Hk;
    const long long n = rows * Hk * kD;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(i % kD);
        const long long rh = i / kD;
        const int hk = static_cast<int>(rh % Hk);
        const long long r = rh / Hk;
        float sq = 0.f, sk = 0.f;
        for (int m = 0; m < group; ++m) {
            const size_t src = ((static_cast<size_t>(r) * Hv) + hk * group + m) * kD + c;
            sq += dq_ws[src];
            sk += dk_ws[src];
        }
        dq[i] = from_f32<Tout>(sq);
        dk[i] = from_f32<Tout>(sk);
    }
}

struct ChunkBwdLayout {
    size_t simt, t, s, u, ds, du, dq, dk, total;
};
ChunkBwdLayout chunk_bwd_layout(int B, int T, int Hv) {
    const ChunkShape sh{B, T, 1, Hv, kD, kD, kCb};
    const size_t units = (size_t)sh.nchunks() * B * Hv, tok = (size_t)B * T * Hv * kD * 4;
    ChunkBwdLayout L;
    L.simt = 0;
    L.t = align_up(chunk_simt_workspace_bytes(sh, /*token_major=*/true), 256);
    L.s = align_up(L.t + units * kCb * kCb * 4, 256);
    L.u = align_up(L.s + units * kD * kD * 4, 256);
    L.ds = align_up(L.u + units * kCb * kD * 4, 256);
    L.du = align_up(L.ds + units * kD * kD * 4, 256);
    L.dq = align_up(L.du + units * kCb * kD * 4, 256);
    L.dk = align_up(L.dq + tok, 256);
    L.total = align_up(L.dk + tok, 256);
    return L;
}

template <typename Tin>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                     const float* s0, const void* d_o, const float* dsT, void* dq, void* dk, void* dv, void* dg,
                     void* db, void* dw, float* ds0, int B, int T, int Hk, int Hv, float scale, uint8_t* ws,
                     cudaStream_t s) {
    const ChunkShape sh{B, T, Hk, Hv, kD, kD, kCb};
    const int NC = sh.nchunks();
    const ChunkBwdLayout L = chunk_bwd_layout(B, T, Hv);
    float* simt = reinterpret_cast<float*>(ws + L.simt);
    float* t_ws = reinterpret_cast<float*>(ws + L.t);
    float* s_save = reinterpret_cast<float*>(ws + L.s);
    float* u_save = reinterpret_cast<float*>(ws + L.u);
    float* ds_save = reinterpret_cast<float*>(ws + L.ds);
    float* du_save = reinterpret_cast<float*>(ws + L.du);
    float* dq_ws = reinterpret_cast<float*>(ws + L.dq);
    float* dk_ws = reinterpret_cast<float*>(ws + L.dk);
    cudaError_t e = launch_factors_simt(q, k, v, g, b, w, sh, std::is_same<Tin, float>::value ? GDN2_F32 : GDN2_BF16,
                                        simt, t_ws, /*token_major=*/true, s);
    if (e != cudaSuccess) return e;
    const size_t c_smem = sizeof(float) * (size_t)fc::TOTAL, a_smem = sizeof(float) * (size_t)ac::TOTAL;
    const size_t ch_smem = c_smem > a_smem ? c_smem : a_smem;
    const size_t g_smem = sizeof(float) * (size_t)gk::TOTAL;
    e = cudaFuncSetAttribute(chains_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ch_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grad_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g_smem);
    if (e != cudaSuccess) return e;
    // the two chains side by side in one launch, on the caller's stream
    chains_kernel<Tin><<<dim3(B * Hv, 2 * (kD / kSl)), kCT, ch_smem, s>>>(
        simt, s0, s_save, u_save, static_cast<const Tin*>(d_o), dsT, ds0, ds_save, du_save, T, Hv, NC, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    grad_kernel<Tin><<<dim3(NC, B * Hv), kGT, g_smem, s>>>(
        static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v), static_cast<const Tin*>(g),
        static_cast<const Tin*>(b), static_cast<const Tin*>(w), static_cast<const Tin*>(d_o), t_ws, s_save, u_save,
        ds_save, du_save, dq_ws, dk_ws, static_cast<Tin*>(dv), static_cast<Tin*>(dg), static_cast<Tin*>(db),
        static_cast<Tin*>(dw), T, Hk, Hv, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long long rows = (long long)B * T, nk = rows * Hk * kD;
    const int gs = static_cast<int>(nk / 256 + 1 < 4096 ? nk / 256 + 1 : 4096);
    group_sum2_kernel<Tin><<<gs, 256, 0, s>>>(dq_ws, dk_ws, static_cast<Tin*>(dq), static_cast<Tin*>(dk), rows, Hk, Hv);
    return cudaGetLastError();
}

}  // namespace

size_t backward_chunked_workspace_bytes(int B, int T, int Hv) { return chunk_bwd_layout(B, T, Hv).total; }

cudaError_t launch_backward_chunked(const void* q, const void* k, const void* v, const void* g, const void* b,
                                    const void* w, const float* s0, const void* d_o, const float* dsT, void* dq,
                                    void* dk, void* dv, void* dg, void* db, void* dw, float* ds0, int B, int T, int Hk,
                                    int Hv, float scale, gdn2_dtype dt, void* ws, cudaStream_t s) {
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if (dt == GDN2_BF16)
        return launch_t<__nv_bfloat16>(q, k, v, g, b, w, s0, d_o, dsT, dq, dk, dv, dg, db, dw, ds0, B, T, Hk, Hv, scale,
                                       wsb, s);
    return launch_t<float>(q, k, v, g, b, w, s0, d_o, dsT, dq, dk, dv, dg, db, dw, ds0, B, T, Hk, Hv, scale, wsb, s);
}

}  // namespace gdn2

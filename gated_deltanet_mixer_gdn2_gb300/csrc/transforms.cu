// transforms.cu -- input transforms that let the GDN-2 core run neighbouring gated-delta variants.
//
// FG^2-GDN ("FG^2-GDN: Enhancing Long-Context Gated Delta Networks with Doubly Fine-Grained
// Control", section 2.A) gives every key channel its own learning rate beta_t in R^{d_k}, absorbed
// symmetrically into the key and the value:
//     k~ = sqrt(beta) . k,   v~ = sqrt(beta) . v,   S_t = (I - k~ k~^T) Diag(alpha_t) S_{t-1} + k~ v~^T.
// The GDN-2 core computes S_t = (I - k (b . k)^T) diag(alpha_t) S_{t-1} + k (w . v)^T, so FG^2-GDN is
// exactly the core with k <- sqrt(beta) . k, b <- 1 and w <- sqrt(beta) (which needs d_k = d_v).
// Since beta belongs to the value head while k belongs to the key head, the transformed key (and
// therefore q) is written per value head.
#include "common.cuh"

namespace gdn2 {
namespace {

// One thread per 8 consecutive channels of one (row, value head); grid-stride.
template <typename T>
__global__ void __launch_bounds__(256) fg2_inputs_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                         const T* __restrict__ beta, T* __restrict__ q_out,
                                                         T* __restrict__ k_out, T* __restrict__ b_out,
                                                         T* __restrict__ w_out, long long rows, int Hk, int Hv,
                                                         int d) {
    const int d8 = d / 8, group = Hv / Hk;
    const long long n = rows * Hv * d8;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c8 = static_cast<int>(i % d8);
        const long long rh = i / d8;
        const int hv = static_cast<int>(rh % Hv);
        const long long r = rh / Hv;
        const size_t src = (static_cast<size_t>(r) * Hk + hv / group) * d + 8 * c8;
        const size_t dst = static_cast<size_t>(rh) * d + 8 * c8;
        float x[8], y[8], one[8];
        Vec8<T>::load(beta + dst, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            x[e] = sqrtf(x[e]);  // sqrt(beta)
            one[e] = 1.f;
        }
        Vec8<T>::load(k + src, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] *= x[e];
        Vec8<T>::store(k_out + dst, y);
        Vec8<T>::store(w_out + dst, x);
        Vec8<T>::store(b_out + dst, one);
        Vec8<T>::load(q + src, y);
        Vec8<T>::store(q_out + dst, y);
    }
}

}  // namespace
}  // namespace gdn2

using namespace gdn2;

extern "C" gdn2_status gdn2_fg2_inputs(const void* q, const void* k, const void* beta, void* q_out, void* k_out,
                                       void* b_out, void* w_out, int B, int T, int Hk, int Hv, int d,
                                       gdn2_dtype dt, void* stream) {
    if ((dt != GDN2_F32 && dt != GDN2_BF16) || B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || d <= 0 || Hv % Hk)
        return GDN2_ERR_INVALID_ARG;
    if (d % 8) return GDN2_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * T;
    if (rows == 0) return GDN2_OK;
    if (rows * Hv * d >= (1LL << 46)) return GDN2_ERR_UNSUPPORTED;
    if (!q || !k || !beta || !q_out || !k_out || !b_out || !w_out) return GDN2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(beta) || !aligned16(q_out) || !aligned16(k_out) ||
        !aligned16(b_out) || !aligned16(w_out))
        return GDN2_ERR_MISALIGNED;
    const long long n = rows * Hv * (d / 8);
    const int grid = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == GDN2_BF16)
        fg2_inputs_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(beta), static_cast<__nv_bfloat16*>(q_out),
            static_cast<__nv_bfloat16*>(k_out), static_cast<__nv_bfloat16*>(b_out), static_cast<__nv_bfloat16*>(w_out),
            rows, Hk, Hv, d);
    else
        fg2_inputs_kernel<float><<<grid, 256, 0, s>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(beta),
            static_cast<float*>(q_out), static_cast<float*>(k_out), static_cast<float*>(b_out),
            static_cast<float*>(w_out), rows, Hk, Hv, d);
    return cudaGetLastError() == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

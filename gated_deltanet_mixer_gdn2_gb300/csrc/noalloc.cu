// noalloc.cu -- gdn2_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where device allocation is not available or not allowed -- a
// plugin inside a host application whose framework has already reserved the device memory and
// owns the allocator, or a latency-critical serving loop that must not call cudaMalloc / cudaFree
// (cudaFree synchronises the device; cudaMalloc can block and can fail once the memory is
// reserved). Such callers still own their inputs and outputs, but they cannot provide the
// workspace that gdn2_chunk_fwd asks for.
//
// What it does: the workspace lives in a file-scope __device__ array of kNoAllocBytes (32 MiB),
// which every GPU that loads the library holds until the process exits. Host code cannot use the
// array's name as a device address (it is a host-side stand-in), so the first call on each device
// asks the runtime for the array's device address with cudaGetSymbolAddress -- with that device
// current -- and caches it; that first call should therefore come before any stream capture. The
// address is then passed to the existing chunked-forward launchers like any workspace pointer.
// Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
//
// Sharing: every call uses the same array and the array keeps the last call's contents. Within a
// call the kernels write every workspace byte before they read it, except the tensor-core path's
// count of chunks for its exact kernel, which the launcher clears on the call's stream first; so
// the caller clears nothing. Calls whose kernels overlap on the GPU (different streams, or
// different host threads on one device) race on the array.
#include <mutex>

#include "common.cuh"

namespace gdn2 {
namespace {

constexpr size_t kNoAllocBytes = size_t(32) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
gdn2_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN2_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GDN2_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return GDN2_OK;
}

}  // namespace
}  // namespace gdn2

extern "C" gdn2_status gdn2_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                              const void* b, const void* w, const float* initial_state,
                                              float* final_state, void* o, int B, int T, int Hk, int Hv, int dk,
                                              int dv, int C, float scale, gdn2_dtype dt, void* stream) {
    const size_t need = gdn2_chunk_fwd_workspace_size(B, T, Hk, Hv, dk, dv, C, dt);
    if (need > gdn2::kNoAllocBytes) return GDN2_ERR_WORKSPACE;  // larger than the fixed scratch array
    if (need == 0)  // empty or unsupported problem: gdn2_chunk_fwd reports it without a workspace
        return gdn2_chunk_fwd(q, k, v, g, b, w, initial_state, final_state, o, B, T, Hk, Hv, dk, dv, C, scale,
                              dt, nullptr, 0, stream);
    void* scratch = nullptr;
    const gdn2_status st = gdn2::scratch_address(&scratch);
    if (st != GDN2_OK) return st;
    return gdn2_chunk_fwd(q, k, v, g, b, w, initial_state, final_state, o, B, T, Hk, Hv, dk, dv, C, scale, dt,
                          scratch, gdn2::kNoAllocBytes, stream);
}

// api.cu -- the extern "C" entry points of libgdn2.so: argument validation (all on the host,
// before anything is enqueued), kernel-family selection and status reporting.
#include <atomic>
#include <climits>

#include "common.cuh"

namespace gdn2 {

static std::atomic<long long> g_wait_ns{kDefaultWaitNs};

long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

cudaError_t launch_selftest_umma(int case_id, int soft, const void* a_st, const void* b_st, float* d_out,
                                 cudaStream_t s, long long wait_ns);

namespace {

// Tensor-core path: d_k = 128, or 64 run as 128 with zero channels; the state kernel runs one CTA per
// 64 columns of d_v.
bool tc_shape(const ChunkShape& sh, gdn2_dtype dt) {
    return dt == GDN2_BF16 && (sh.dk == 128 || sh.dk == 64) && sh.dv % 64 == 0 && sh.dv >= 64 && sh.dv <= 512 &&
           sh.C == 64;
}

bool simt_shape(const ChunkShape& sh) {
    auto okd = [](int d, int hi) { return d >= 16 && d <= hi && d % 16 == 0; };
    return okd(sh.dk, 128) && okd(sh.dv, 256) && (sh.C == 16 || sh.C == 32 || sh.C == 64);
}

// Resolve AUTO; returns GDN2_PATH_AUTO when the requested path cannot run this shape.
gdn2_path resolve(gdn2_path p, const ChunkShape& sh, gdn2_dtype dt) {
    switch (p) {
        case GDN2_PATH_AUTO:
            if (tc_shape(sh, dt)) return GDN2_PATH_TCGEN05;
            return simt_shape(sh) ? GDN2_PATH_SIMT : GDN2_PATH_AUTO;
        case GDN2_PATH_TCGEN05:
            return tc_shape(sh, dt) ? GDN2_PATH_TCGEN05 : GDN2_PATH_AUTO;
        case GDN2_PATH_SIMT:
            return simt_shape(sh) ? GDN2_PATH_SIMT : GDN2_PATH_AUTO;
    }
    return GDN2_PATH_AUTO;
}

bool dtype_ok(gdn2_dtype dt) { return dt == GDN2_F32 || dt == GDN2_BF16; }

// Sizes must keep every flat index and TMA coordinate well inside 64-bit / 32-bit ranges.
bool sizes_ok(long long B, long long T, long long Hk, long long Hv, long long dk, long long dv) {
    const long long lim = 1LL << 31;
    if (B >= lim || T >= lim || Hk >= lim || Hv >= lim) return false;
    const long long tok = B * T;
    if (tok >= lim) return false;
    const long long el = tok * (Hk > Hv ? Hk : Hv) * (dk > dv ? dk : dv);
    return el < (1LL << 46);
}

// The chunked kernels put (batch, value head) on the grid's second dimension (at most 65535).
bool grid_ok(long long B, long long Hv) { return B * Hv <= 65535; }

size_t ws_size(gdn2_path path, const ChunkShape& sh, gdn2_dtype dt) {
    if (sh.B <= 0 || sh.T <= 0) return 0;
    const gdn2_path p = resolve(path, sh, dt);
    if (p == GDN2_PATH_TCGEN05) return chunk_tc_workspace_bytes(sh);
    if (p == GDN2_PATH_SIMT) return chunk_simt_workspace_bytes(sh);
    return 0;
}

}  // namespace
}  // namespace gdn2

using namespace gdn2;

extern "C" {

const char* gdn2_status_string(gdn2_status s) {
    switch (s) {
        case GDN2_OK: return "ok";
        case GDN2_ERR_INVALID_ARG: return "invalid argument";
        case GDN2_ERR_UNSUPPORTED: return "unsupported shape, chunk size, dtype or path";
        case GDN2_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GDN2_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN2_ERR_CUDA: return "CUDA call failed";
        case GDN2_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    }
    return "unknown status";
}

int gdn2_version(void) { return 100; }

size_t gdn2_chunk_fwd_workspace_size_path(gdn2_path path, int B, int T, int Hk, int Hv, int dk, int dv, int C,
                                          gdn2_dtype dt) {
    if (!dtype_ok(dt) || B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || C <= 0 || Hv % Hk) return 0;
    if (!sizes_ok(B, T, Hk, Hv, dk, dv) || !grid_ok(B, Hv)) return 0;
    return ws_size(path, ChunkShape{B, T, Hk, Hv, dk, dv, C}, dt);
}

size_t gdn2_chunk_fwd_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, int C, gdn2_dtype dt) {
    return gdn2_chunk_fwd_workspace_size_path(GDN2_PATH_AUTO, B, T, Hk, Hv, dk, dv, C, dt);
}

gdn2_status gdn2_chunk_fwd_path(gdn2_path path, const void* q, const void* k, const void* v, const void* g,
                                const void* b, const void* w, const float* initial_state, float* final_state,
                                void* o, int B, int T, int Hk, int Hv, int dk, int dv, int C, float scale,
                                gdn2_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
    if (!dtype_ok(dt) || (path != GDN2_PATH_AUTO && path != GDN2_PATH_SIMT && path != GDN2_PATH_TCGEN05))
        return GDN2_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || C <= 0 || Hv % Hk)
        return GDN2_ERR_INVALID_ARG;
    if (!sizes_ok(B, T, Hk, Hv, dk, dv) || !grid_ok(B, Hv)) return GDN2_ERR_UNSUPPORTED;
    const ChunkShape sh{B, T, Hk, Hv, dk, dv, C};
    const gdn2_path p = resolve(path, sh, dt);
    if (p == GDN2_PATH_AUTO) return GDN2_ERR_UNSUPPORTED;
    if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
        return GDN2_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t state_bytes = sizeof(float) * (size_t)B * Hv * dk * dv;
    if (B == 0 || T == 0) {  // empty sequence: S_T = S_0
        if (final_state && state_bytes) {
            cudaError_t e = cudaSuccess;
            if (!initial_state) e = cudaMemsetAsync(final_state, 0, state_bytes, s);
            else if (initial_state != final_state)
                e = cudaMemcpyAsync(final_state, initial_state, state_bytes, cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return GDN2_ERR_CUDA;
        }
        return GDN2_OK;
    }
    if (!q || !k || !v || !g || !b || !w || !o) return GDN2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(b) || !aligned16(w) ||
        !aligned16(o))
        return GDN2_ERR_MISALIGNED;
    const size_t need = ws_size(p, sh, dt);
    if (!workspace || ws_bytes < need) return GDN2_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GDN2_ERR_MISALIGNED;
    const long long units = (long long)sh.nchunks() * B * Hv;
    if (units >= (1LL << 31)) return GDN2_ERR_UNSUPPORTED;

    cudaError_t e;
    if (p == GDN2_PATH_TCGEN05)
        e = launch_chunk_tc(q, k, v, g, b, w, initial_state, final_state, o, sh, scale, workspace, s, wait_limit_ns());
    else
        e = launch_chunk_simt(q, k, v, g, b, w, initial_state, final_state, o, sh, scale, dt, workspace, s);
    return e == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

gdn2_status gdn2_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                           const float* initial_state, float* final_state, void* o, int B, int T, int Hk, int Hv,
                           int dk, int dv, int C, float scale, gdn2_dtype dt, void* workspace, size_t ws_bytes,
                           void* stream) {
    return gdn2_chunk_fwd_path(GDN2_PATH_AUTO, q, k, v, g, b, w, initial_state, final_state, o, B, T, Hk, Hv, dk,
                               dv, C, scale, dt, workspace, ws_bytes, stream);
}

gdn2_status gdn2_recurrent_update(const void* q, const void* k, const void* v, const void* g, const void* b,
                                  const void* w, void* state, gdn2_dtype state_dt, const int32_t* slots, int n_slots,
                                  void* o, int B, int N, int Hk, int Hv, int dk, int dv, float scale, gdn2_dtype dt,
                                  void* stream) {
    if (!dtype_ok(dt) || !dtype_ok(state_dt)) return GDN2_ERR_INVALID_ARG;
    if (B < 0 || N < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk) return GDN2_ERR_INVALID_ARG;
    if (slots && n_slots < 0) return GDN2_ERR_INVALID_ARG;
    if (!(dk == 16 || dk == 32 || dk == 64 || dk == 128) || dv % 16 != 0 || dv > 512) return GDN2_ERR_UNSUPPORTED;
    if (!sizes_ok(B, N, Hk, Hv, dk, dv)) return GDN2_ERR_UNSUPPORTED;
    if (B == 0 || N == 0) return GDN2_OK;
    if (!q || !k || !v || !g || !b || !w || !state || !o) return GDN2_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(b) || !aligned16(w) ||
        !aligned16(state) || !aligned16(o) || (reinterpret_cast<uintptr_t>(slots) & 3u))
        return GDN2_ERR_MISALIGNED;
    const cudaError_t e = launch_recurrent(q, k, v, g, b, w, state, state_dt, slots, n_slots, o, B, N, Hk, Hv, dk,
                                           dv, scale, dt, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

gdn2_status gdn2_recurrent_step(const void* q, const void* k, const void* v, const void* g, const void* b,
                                const void* w, float* state, void* o, int B, int Hk, int Hv, int dk, int dv,
                                float scale, gdn2_dtype dt, void* stream) {
    return gdn2_recurrent_update(q, k, v, g, b, w, state, GDN2_F32, nullptr, 0, o, B, 1, Hk, Hv, dk, dv, scale, dt,
                                 stream);
}

gdn2_status gdn2_last_device_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN2_ERR_CUDA;
    const int a = chunk_tc_read_clear_status(s);
    const int b = chunk_simt_read_clear_status(s);
    const int c = decode_read_clear_status(s);
    const int d = backward_tc_read_clear_status(s);
    const int e = step_read_clear_status(s);
    if (a < 0 || b < 0 || c < 0 || d < 0 || e < 0) return GDN2_ERR_CUDA;
    return (a | b | c | d | e) ? GDN2_ERR_TIMEOUT : GDN2_OK;
}

void gdn2_set_wait_limit(long long ns) { g_wait_ns.store(ns < 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed); }

gdn2_status gdn2_selftest_umma(int case_id, int soft, const void* a_storage, const void* b_storage, float* d_out,
                               void* stream) {
    if (case_id < 0 || case_id > 7 || !a_storage || !b_storage || !d_out) return GDN2_ERR_INVALID_ARG;
    if (!aligned16(a_storage) || !aligned16(b_storage) || !aligned16(d_out)) return GDN2_ERR_MISALIGNED;
    const cudaError_t e = launch_selftest_umma(case_id, soft, a_storage, b_storage, d_out,
                                               static_cast<cudaStream_t>(stream), wait_limit_ns());
    return e == cudaSuccess ? GDN2_OK : GDN2_ERR_CUDA;
}

}  // extern "C"

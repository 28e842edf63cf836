/*
 * gdn2.h -- C ABI of libgdn2.so, the GB300 (sm_103a) Gated DeltaNet-2 token-mixer core.
 *
 * The operation (burn-gdn2 0.1.5 docs, "Architecture"): per batch element and value head, on a
 * matrix state S in R^{d_k x d_v},
 *
 *     S_t = (I - k_t (b_t . k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t . v_t)^T,    o_t = scale * S_t^T q_t
 *
 * where alpha_t = exp(g_t) is a per-key-channel decay, b_t the key-axis erase gate and w_t the
 * value-axis write gate ("." is the element-wise product; o_t reads the post-update state). The
 * same page names the two modes exported here: a chunked WY decomposition over a whole sequence
 * (training / prefill) and a token-by-token recurrent step on a persistent state (inference).
 *
 * Conventions shared by every entry point
 *   - Pointers: every tensor pointer is a DEVICE pointer to a caller-owned, contiguous, row-major
 *     buffer aligned to 16 bytes. The library never allocates, frees or keeps device memory.
 *   - Grouped heads: q and k belong to H_k key heads; g, b, v, w, o and the state to H_v value
 *     heads; H_v must be a multiple of H_k and value head h reads key head h / (H_v / H_k).
 *   - Token dtype: GDN2_F32 (float) or GDN2_BF16 (bfloat16) for q, k, v, g, b, w and o. States
 *     are always fp32. Arithmetic is fp32 (the bf16 chunked path feeds bf16 operands to the
 *     tensor cores with fp32 accumulation).
 *   - g is log(alpha) with alpha in [0, 1]: g <= 0, -inf included (a full reset of that key
 *     channel; not checked). b is the erase gate after its activation, with values in (0, 2) when
 *     negative eigenvalues are allowed (the caller doubles it); w is the write gate after its
 *     activation.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Every
 *     entry point only enqueues work: it returns without synchronising the host.
 *   - Errors: entry points never abort, trap or print. Argument errors are detected on the host
 *     before any work is enqueued and return a negative gdn2_status. A kernel that exceeds its
 *     bounded wait records GDN2_ERR_TIMEOUT in a device status word read by
 *     gdn2_last_device_status().
 */
#ifndef GDN2_H
#define GDN2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn2_status {
    GDN2_OK = 0,
    GDN2_ERR_INVALID_ARG = -1, /* null required pointer, non-positive size, H_v % H_k != 0     */
    GDN2_ERR_UNSUPPORTED = -2, /* shape / chunk size / dtype / path combination not built       */
    GDN2_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned                               */
    GDN2_ERR_WORKSPACE = -4,   /* workspace pointer null or smaller than required                */
    GDN2_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed (launch, attribute, symbol)  */
    GDN2_ERR_TIMEOUT = -6      /* a kernel gave up a bounded wait (device status word)           */
} gdn2_status;

typedef enum gdn2_dtype { GDN2_F32 = 0, GDN2_BF16 = 1 } gdn2_dtype;

/* Kernel family used by the chunked forward. AUTO picks TCGEN05 for bf16 with d_k = 128 or 64, d_v
 * a multiple of 64 (up to 512) and C = 64, and SIMT otherwise. */
typedef enum gdn2_path { GDN2_PATH_AUTO = 0, GDN2_PATH_SIMT = 1, GDN2_PATH_TCGEN05 = 2 } gdn2_path;

/* Human-readable name of a status code (static string, never NULL). */
const char* gdn2_status_string(gdn2_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gdn2_version(void);

/*
 * gdn2_chunk_fwd_workspace_size -- bytes of device workspace gdn2_chunk_fwd needs (AUTO path).
 * The chunked forward stores per-chunk factors (W, U~, decayed q and k, the causal q-k matrix, the
 * chunk decay) between its two kernels. Returns 0 for shapes the path does not support (and for
 * empty problems). Pure host function.
 */
size_t gdn2_chunk_fwd_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, int C,
                                     gdn2_dtype dt);
size_t gdn2_chunk_fwd_workspace_size_path(gdn2_path path, int B, int T, int Hk, int Hv, int dk,
                                          int dv, int C, gdn2_dtype dt);

/*
 * gdn2_chunk_fwd -- chunked forward over whole sequences (burn-gdn2 docs: "chunked WY
 * decomposition (training)"; chunk_size 64 by default in its configuration table).
 *
 *   q, k           [B, T, H_k, d_k]  dt
 *   v, w           [B, T, H_v, d_v]  dt
 *   g, b           [B, T, H_v, d_k]  dt
 *   initial_state  [B, H_v, d_k, d_v] fp32, may be NULL (zeros)
 *   final_state    [B, H_v, d_k, d_v] fp32, may be NULL (not written); may alias initial_state
 *   o              [B, T, H_v, d_v]  dt (output)
 *   C              chunk length: 64 on the tensor-core path; 16, 32 or 64 on the SIMT path
 *   workspace      device buffer of at least gdn2_chunk_fwd_workspace_size(...) bytes, 16-byte
 *                  aligned (GDN2_ERR_MISALIGNED otherwise); its contents on entry are ignored and
 *                  on return are unspecified, except as noted below for the TCGEN05 path
 *
 * T need not be a multiple of C (the last chunk is padded with tokens that leave the state
 * unchanged). T == 0 or B == 0 is valid: o is untouched and final_state receives initial_state (or
 * zeros). Supported: d_k a multiple of 16 in [16, 128] and d_v a multiple of 16 in [16, 256]
 * (SIMT, fp32 or bf16); bf16 with d_k = 128 or 64, d_v a multiple of 64 in [64, 512] and C = 64
 * (TCGEN05, which AUTO picks for those shapes; d_v = 256 is the configuration table's expand_v = 2
 * at head_dim 128; d_k = 64 runs as d_k = 128 whose upper 64 key channels are zero, so it costs
 * what d_k = 128 costs); B * H_v <= 65535 (GDN2_ERR_UNSUPPORTED beyond).
 *
 * Decay domain: any alpha in [0, 1] on both paths, including alpha = 0 (g = -inf) and decays that
 * forget a whole chunk. Both paths floor g at -100 (alpha = e^-100 ~ 4e-44, indistinguishable from
 * 0 in fp32) and form every decay factor so that it cannot overflow. On the TCGEN05 path a
 * (chunk, value head) whose per-channel log-decay spans more than 120 within the chunk (more than
 * about 1.9 per token on average) is formed by an exact CUDA-core kernel instead of the tensor-core
 * factor kernel: same results, slower for those chunks. Diagnostic: after the call completes, the
 * int32 at byte offset 66048 * ceil(T / 64) * B * H_v of the workspace holds the number of such
 * chunks.
 */
gdn2_status gdn2_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                           const void* b, const void* w, const float* initial_state,
                           float* final_state, void* o, int B, int T, int Hk, int Hv, int dk,
                           int dv, int C, float scale, gdn2_dtype dt, void* workspace,
                           size_t ws_bytes, void* stream);
gdn2_status gdn2_chunk_fwd_path(gdn2_path path, const void* q, const void* k, const void* v,
                                const void* g, const void* b, const void* w,
                                const float* initial_state, float* final_state, void* o, int B,
                                int T, int Hk, int Hv, int dk, int dv, int C, float scale,
                                gdn2_dtype dt, void* workspace, size_t ws_bytes, void* stream);

/*
 * gdn2_chunk_fwd_noalloc -- gdn2_chunk_fwd for callers that cannot allocate device memory. The
 * pages have no counterpart: this is a convenience of this library. Some callers cannot call
 * cudaMalloc -- a plugin whose host framework has reserved the device memory and owns the
 * allocator, or a serving loop that must not call cudaMalloc / cudaFree (cudaFree synchronises the
 * device; cudaMalloc can block or fail once memory is reserved) -- so they cannot provide the
 * workspace gdn2_chunk_fwd needs. This entry point takes the same arguments minus the workspace
 * and uses a fixed 32 MiB array in device memory that every GPU loading the library keeps until
 * the process exits. It allocates nothing.
 *   - Limit: problems whose workspace (gdn2_chunk_fwd_workspace_size) exceeds 33 554 432 bytes
 *     are rejected with GDN2_ERR_WORKSPACE before any work is enqueued (on the tensor-core path,
 *     one 66 048-byte unit per chunk and value head: at most 508 of them).
 *   - Set-up: the first call on a device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - Sharing: all calls share the array and it keeps the last call's contents (the call itself
 *     clears, on its stream, the one word that must start at zero); calls whose kernels overlap on
 *     the GPU race on it.
 * Other arguments, errors and results: as gdn2_chunk_fwd (AUTO path).
 */
gdn2_status gdn2_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                   const void* b, const void* w, const float* initial_state,
                                   float* final_state, void* o, int B, int T, int Hk, int Hv,
                                   int dk, int dv, int C, float scale, gdn2_dtype dt, void* stream);

/*
 * gdn2_recurrent_step -- one decode token against a persistent fp32 state, updated in place
 * (burn-gdn2 docs: token-by-token recurrent mode with persistent state; the same single fused
 * update that the llama.cpp GDN decode study describes for the scalar-beta rule).
 *
 *   q, k   [B, H_k, d_k] dt;   v, w [B, H_v, d_v] dt;   g, b [B, H_v, d_k] dt
 *   state  [B, H_v, d_k, d_v] fp32, read and written in place (read once, written once)
 *   o      [B, H_v, d_v] dt (output)
 *
 * Supported: d_k in {16, 32, 64, 128}; d_v a multiple of 16 up to 512. B == 0 is a no-op.
 */
gdn2_status gdn2_recurrent_step(const void* q, const void* k, const void* v, const void* g,
                                const void* b, const void* w, float* state, void* o, int B,
                                int Hk, int Hv, int dk, int dv, float scale, gdn2_dtype dt,
                                void* stream);

/*
 * gdn2_recurrent_update -- the recurrent mode for serving: N tokens per call against persistent
 * states, optionally addressed through a slot map into a pool, with fp32 or bf16 state storage.
 * The same per-token recurrence as gdn2_recurrent_step, applied to tokens 0..N-1 in order; the
 * state is read once and written once per call (it stays on chip between the call's tokens). This
 * serves the serving-side items the llama.cpp GDN decode study names: a recurrent state cache
 * whose entries are read and written every step, more than one token per step, and a bf16 state.
 *
 *   q, k    [B, N, H_k, d_k] dt;   v, w, o [B, N, H_v, d_v] dt;   g, b [B, N, H_v, d_k] dt
 *   state   slots == NULL: [B, H_v, d_k, d_v] of state_dt, row b for batch element b;
 *           slots != NULL: a pool [n_slots, H_v, d_k, d_v] of state_dt; batch element b uses pool
 *           row slots[b] (int32 device array of B entries). A slot outside [0, n_slots) marks the
 *           element inactive: its state, its o rows and every other pool row are left untouched.
 *           Active elements must name distinct slots (two elements on one slot race).
 *   state_dt  GDN2_F32, or GDN2_BF16: widened to fp32 on load, rounded to nearest even on store.
 *
 * Supported: d_k in {16, 32, 64, 128}; d_v a multiple of 16 up to 512. B == 0 or N == 0 is a no-op.
 * gdn2_recurrent_step(...) equals gdn2_recurrent_update(..., GDN2_F32, NULL, 0, ..., N = 1, ...).
 */
gdn2_status gdn2_recurrent_update(const void* q, const void* k, const void* v, const void* g,
                                  const void* b, const void* w, void* state, gdn2_dtype state_dt,
                                  const int32_t* slots, int n_slots, void* o, int B, int N,
                                  int Hk, int Hv, int dk, int dv, float scale, gdn2_dtype dt,
                                  void* stream);

/*
 * gdn2_last_device_status -- synchronises `stream`, then reads and clears the device status word
 * of the current device. Returns GDN2_OK, GDN2_ERR_TIMEOUT (a kernel gave up a bounded wait since
 * the last call) or GDN2_ERR_CUDA (the synchronisation itself failed).
 */
gdn2_status gdn2_last_device_status(void* stream);

/*
 * gdn2_set_wait_limit -- nanoseconds a kernel polls one barrier before it gives up and records
 * GDN2_ERR_TIMEOUT. Negative restores the default (two seconds). Applies to
 * launches enqueued after the call, process-wide. Zero makes every guarded wait give up at once;
 * the kernel then still drains its own copies and tensor-core work (with the default limit)
 * before it returns, so the device stays usable. Intended for tests of the error path.
 */
void gdn2_set_wait_limit(long long ns);

/*
 * gdn2_fg2_inputs -- FG^2-GDN as GDN-2 inputs ("FG^2-GDN: Enhancing Long-Context Gated Delta
 * Networks with Doubly Fine-Grained Control", section 2.A, "FG2-GDN: Tasa de Aprendizaje
 * Vectorial"). FG^2-GDN absorbs a per-channel learning rate beta_t (d values, >= 0) into key and
 * value, k~ = sqrt(beta) . k and v~ = sqrt(beta) . v, and updates
 *     S_t = (I - k~ k~^T) Diag(alpha_t) S_{t-1} + k~ v~^T.
 * That is the GDN-2 recurrence with k <- sqrt(beta) . k, b <- 1, w <- sqrt(beta) (d_k = d_v = d).
 * This call writes, for every value head h: q_out = q of key head floor(h * H_k / H_v),
 * k_out = sqrt(beta) . (that head's k), b_out = 1, w_out = sqrt(beta). Then run gdn2_chunk_fwd or
 * gdn2_recurrent_update with H_k = H_v on (q_out, k_out, v, g, b_out, w_out).
 *
 * q, k: [B, T, H_k, d]; beta: [B, T, H_v, d]; q_out, k_out, b_out, w_out: [B, T, H_v, d] (caller-
 * owned device buffers, distinct from the inputs); all of dtype dt. For decode tokens [B, H, d]
 * pass T = 1. d must be a multiple of 8; pointers 16-byte aligned. beta < 0 is not checked (its
 * square root is NaN). Asynchronous on `stream`.
 * Errors: GDN2_ERR_INVALID_ARG (dtype, sizes <= 0 or negative, H_v % H_k, null pointer),
 * GDN2_ERR_UNSUPPORTED (d % 8, too large), GDN2_ERR_MISALIGNED, GDN2_ERR_CUDA (launch failed).
 */
gdn2_status gdn2_fg2_inputs(const void* q, const void* k, const void* beta, void* q_out, void* k_out,
                            void* b_out, void* w_out, int B, int T, int Hk, int Hv, int d, gdn2_dtype dt,
                            void* stream);

/*
 * gdn2_mixer_prologue -- the token-mixer steps between the projections and the core, in one pass
 * (burn-gdn2 0.1.5 docs, "Architecture": projections -> ShortConv -> L2-Norm -> core; configuration
 * table: use_short_conv, allow_neg_eigval "b x 2"; llama.cpp GDN decode study, sections 1-2: conv
 * kernel 4, a carried state of the previous 3 samples):
 *   q = L2norm(conv(xq)), k = L2norm(conv(xk)), v = conv(xv), with the depthwise causal conv
 *       conv(x)_t[c] = sum_{j=0..3} W[c][j] x_{t-3+j}[c]   (samples before the call from the state)
 *       and L2norm(x) = x / sqrt(sum x^2 + 1e-6) per (token, head);
 *   g = -softplus(ag), b = sigmoid(ab) (x 2 when neg_eigval != 0), w = sigmoid(aw).
 * xq, xk: [B, T, H_k, d_k]; xv: [B, T, H_v, d_v]; ag, ab: [B, T, H_v, d_k]; aw: [B, T, H_v, d_v];
 * conv_q, conv_k: fp32 [H_k * d_k][4]; conv_v: fp32 [H_v * d_v][4] (tap 3 = current token).
 * state_q / state_k / state_v: fp32 conv states [B][3][channels] (x_{-3}, x_{-2}, x_{-1}), read and then
 * replaced by the last 3 samples of [state, x]; NULL = zeros in, nothing written. Outputs q, k, v, g,
 * b, w in the core's layout, token dtype dt; they must not overlap the inputs. d_k, d_v in
 * {16, 32, 64, 128, 256}; pointers 16-byte aligned. For decode tokens pass T = 1.
 * Errors: GDN2_ERR_INVALID_ARG (dtype, sizes, H_v % H_k, null required pointer), GDN2_ERR_UNSUPPORTED
 * (head size, too large), GDN2_ERR_MISALIGNED, GDN2_ERR_CUDA. Asynchronous on `stream`.
 */
gdn2_status gdn2_mixer_prologue(const void* xq, const void* xk, const void* xv, const float* conv_q,
                                const float* conv_k, const float* conv_v, const void* ag, const void* ab,
                                const void* aw, float* state_q, float* state_k, float* state_v, void* q, void* k,
                                void* v, void* g, void* b, void* w, int B, int T, int Hk, int Hv, int dk, int dv,
                                int neg_eigval, gdn2_dtype dt, void* stream);

/*
 * gdn2_mixer_epilogue -- gated RMSNorm with a SiLU gate after the core (burn-gdn2 0.1.5 docs,
 * "Architecture": Gated RMS Norm <- SiLU Gate; configuration table: norm_eps 1e-5):
 *   y = o / sqrt(mean_{d_v}(o^2) + eps) * weight * silu(z),  silu(z) = z / (1 + e^{-z}),
 * per (token, value head). o, z, y: [B, T, H_v, d_v] of dtype dt (y may alias o); weight: fp32
 * [d_v]. d_v in {16, 32, 64, 128, 256}; pointers 16-byte aligned. Errors as gdn2_mixer_prologue
 * (eps < 0 or NaN is GDN2_ERR_INVALID_ARG).
 */
gdn2_status gdn2_mixer_epilogue(const void* o, const void* z, const float* weight, float eps, void* y, int B,
                                int T, int Hv, int dv, gdn2_dtype dt, void* stream);

/*
 * gdn2_mixer_decode_step -- one decode token of the whole token mixer around the core in one launch
 * (burn-gdn2 0.1.5 docs, "Architecture": projections -> ShortConv -> L2-Norm -> Fused Recurrent ->
 * Gated RMS Norm <- SiLU Gate; the llama.cpp GDN decode study, section 4, suggests fusing the conv and
 * the gated norm into the delta-net step): the operations of gdn2_mixer_prologue (T = 1),
 * gdn2_recurrent_step and gdn2_mixer_epilogue in sequence, with q, k, v, the gates and o kept on chip.
 *   xq, xk            [B, H_k, d_k] dt  projections of the token (before the conv)
 *   xv                [B, H_v, d_v] dt
 *   conv_q, conv_k    fp32 [H_k * d_k][4]; conv_v fp32 [H_v * d_v][4] (tap 3 = current token)
 *   ag, ab            [B, H_v, d_k] dt  gate pre-activations (g = -softplus(ag), b = sigmoid(ab),
 *   aw                [B, H_v, d_v] dt   x 2 when neg_eigval != 0, w = sigmoid(aw))
 *   state_q, state_k  fp32 conv states [B][3][H_k * d_k]; state_v [B][3][H_v * d_v]: read, then
 *                     replaced by the last 3 samples; NULL = zeros in, nothing written
 *   state             fp32 core state [B, H_v, d_k, d_v], read and written in place
 *   z                 [B, H_v, d_v] dt  output gate; weight fp32 [d_v]; eps >= 0 (1e-5 in the pages)
 *   y                 [B, H_v, d_v] dt  output: gated RMSNorm of o = scale * S_new^T q
 * d_k and d_v in {64, 128}; pointers 16-byte aligned; y must not overlap the inputs. One CTA per
 * (batch row, key head) runs that key head's value heads in turn, so each conv state has one writer.
 * Errors: GDN2_ERR_INVALID_ARG (dtype, sizes, H_v % H_k, eps, null required pointer),
 * GDN2_ERR_UNSUPPORTED (head sizes), GDN2_ERR_MISALIGNED, GDN2_ERR_CUDA. B == 0 is a no-op.
 * Asynchronous on `stream`.
 */
gdn2_status gdn2_mixer_decode_step(const void* xq, const void* xk, const void* xv, const float* conv_q,
                                   const float* conv_k, const float* conv_v, const void* ag, const void* ab,
                                   const void* aw, float* state_q, float* state_k, float* state_v, float* state,
                                   const void* z, const float* weight, float eps, void* y, int B, int Hk, int Hv,
                                   int dk, int dv, int neg_eigval, float scale, gdn2_dtype dt, void* stream);

/*
 * gdn2_backward -- gradients of the core (dq, dk, dv, dg, db, dw and the initial state) for the
 * recurrence of the burn-gdn2 0.1.5 docs ("Architecture"), given the upstream gradient d_o of o
 * and optionally d_final_state of S_T: the gradients of sum(o * d_o) + sum(S_T * d_final_state).
 * Reverse mode of the chunked WY form of the same recurrence (burn-gdn2 0.1.5 docs, "chunked WY
 * decomposition (training)"): the state-independent factors of every chunk (with T = (I + A)^-1);
 * a forward chain that keeps each chunk's starting state S_n and its U; a reverse chain that keeps
 * dS_(n+1) and dU; one CTA per (chunk, batch, value head) that forms every per-token gradient of
 * its chunk from those; and a pass that adds the value heads of each key head for dq and dk in a
 * fixed order. The forward outputs are not needed.
 *   dt = GDN2_BF16: chunks of 64 tokens on the tensor cores (bf16 operands, fp32 accumulators and
 *   state): the factors and the forward chain are the chunked forward's, and the pair terms through
 *   A and M take one anchor per key channel, or CUDA cores with factors exp(G_t - G_s) <= 1 in chunks
 *   whose log-decay spans more than the anchors take.
 *   dt = GDN2_F32: chunks of 32 tokens in fp32 on CUDA cores; gates enter only as ratios
 *   exp(G_t - G_s) with t >= s.
 * Either way the whole decay domain g <= 0 (g = -inf included: gates are floored at -100) gives
 * finite gradients.
 * q, k, dq, dk: [B, T, H_k, d_k]; v, w, d_o, dv, dw: [B, T, H_v, d_v]; g, b, dg, db: [B, T, H_v, d_k]
 * (all dtype dt); initial_state, d_final_state, d_initial_state: fp32 [B, H_v, d_k, d_v] or NULL
 * (zeros / not written). dq and dk of a key head sum its value heads. bf16: d_k and d_v each 64 or
 * 128 (64 as zero-padded 128); fp32: d_k = d_v = 128; B * H_v <= 65535 (GDN2_ERR_UNSUPPORTED
 * otherwise). gdn2_backward_recurrent takes d_k = d_v = 128 only.
 * workspace: gdn2_backward_workspace_size(...) bytes of device memory, 16-byte aligned.
 * Errors: as gdn2_chunk_fwd. Asynchronous on `stream`: every launch goes to `stream` (the forward
 * and reverse chains over chunks run side by side inside one launch), the library holds no stream,
 * event or lock of its own, and the call can be captured in a CUDA graph.
 */
size_t gdn2_backward_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, gdn2_dtype dt);
gdn2_status gdn2_backward(const void* q, const void* k, const void* v, const void* g, const void* b, const void* w,
                          const float* initial_state, const void* d_o, const float* d_final_state, void* dq,
                          void* dk, void* dv, void* dg, void* db, void* dw, float* d_initial_state, int B, int T,
                          int Hk, int Hv, int dk_, int dv_, float scale, gdn2_dtype dt, void* workspace,
                          size_t ws_bytes, void* stream);

/*
 * gdn2_backward_recurrent -- the same gradients as gdn2_backward (same arguments, layouts and
 * errors) by exact reverse mode of the per-token recurrence in fp32, without the chunked form: a
 * forward sweep keeps the state at every 32nd token in the workspace, each stretch of 32 tokens is
 * recomputed and walked backward; two CTAs per (batch, value head), 64 columns of d_v each, whose
 * sums over d_v (for dq, dk, db, dg) a second kernel adds in a fixed order. Slower than the chunked
 * path; it shares none of its arithmetic and serves as an independent cross-check at lengths the
 * host reference cannot reach. workspace: gdn2_backward_recurrent_workspace_size(...) bytes.
 */
size_t gdn2_backward_recurrent_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, gdn2_dtype dt);
gdn2_status gdn2_backward_recurrent(const void* q, const void* k, const void* v, const void* g, const void* b,
                                    const void* w, const float* initial_state, const void* d_o,
                                    const float* d_final_state, void* dq, void* dk, void* dv, void* dg, void* db,
                                    void* dw, float* d_initial_state, int B, int T, int Hk, int Hv, int dk_,
                                    int dv_, float scale, gdn2_dtype dt, void* workspace, size_t ws_bytes,
                                    void* stream);

/*
 * gdn2_selftest_umma -- diagnostics: one tcgen05 product D[128][N] = A * B (bf16 in, fp32 out)
 * with the operand layouts the tensor-core chunked kernels use, so that a test can check them
 * against a host matrix product. The operands are row-major bf16 device arrays:
 *   case 0: A [128 (M)][128 (K)],  B [64 (N)][128 (K)]   (both K-major), N = 64
 *   case 1: A [64 (K)][128 (M)],   B [64 (N)][64 (K)]    (A MN-major, B K-major), N = 64
 *   case 2: A [128 (K)][128 (M)],  B [128 (K)][64 (N)]   (both MN-major), N = 64
 *   case 3: A [128 (M)][64 (K)],   B [64 (K)][64 (N)]    (A K-major, B MN-major), N = 64
 *   case 4: as case 0 with A negated through the instruction descriptor (D = -A * B)
 *   case 5: A [128 (M)][64 (K)] in tensor memory, B [64 (N)][64 (K)] K-major, N = 64
 *   case 6: A [128 (M)][64 (K)] in tensor memory, B [64 (K)][128 (N)] MN-major, N = 128
 *   case 7: A [128 (M)][128 (K)] in tensor memory, B [128 (N)][128 (K)] K-major, N = 128
 * soft = 0 stages the shared-memory operands with TMA (128-byte swizzle), soft = 1 with ordinary
 * stores using the same swizzle; an A operand in tensor memory is written with tcgen05.st.
 * d_out: [128][N] fp32 device array. Asynchronous on `stream`.
 */
gdn2_status gdn2_selftest_umma(int case_id, int soft, const void* a_storage, const void* b_storage,
                               float* d_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN2_H */

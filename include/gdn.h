/*
 * gdn.h -- C ABI of the chunked gated delta rule (Gated DeltaNet) operator
 * for NVIDIA GB300 (sm_103a).
 *
 * The operator.  For one sequence and one head, with a recurrent state S of
 * shape d_k x d_v (fp32), per token t:
 *     alpha_t = exp(g_t)                         (g_t <= 0, given in log space)
 *     S       <- alpha_t S                       (forget)
 *     v_old   =  S^T k_t                         (read what is stored for k_t)
 *     S       <- S + beta_t k_t (v_t - v_old)^T  (write the error, not the value)
 *     o_t     =  scale * S^T q_t                 (look up with the query)
 * Sources: "Research Sprint Day 1 - Verifying the flash-linear-attention
 * Gated DeltaNet kernel on GB10", section "The GDN update" (the loop);
 * "Research Sprint Day 2 - Rooflines", GDN update equation
 * S_t = S_{t-1}(alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T (the same
 * map on the transposed d_v x d_k state) and its GDN layer pseudocode step 5
 * (g kept in log space, accumulated as a cumsum); the cuLA issue #126
 * reproduction (scale = D^-0.5 passed to the kernel, fp32 (1,H,D,D) state,
 * caller-allocated out/final_state).  The library evaluates it chunk by chunk
 * (64 tokens), which reaches the same result in exact arithmetic.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates, frees or keeps a pointer after the call
 *     returns.  Scratch memory is the caller's `workspace`.
 *   - Tensors are contiguous, row-major, in the shapes given below.  bf16
 *     tensors (q, k, v, beta, out, d_out, dq, dk, dv, dbeta) are raw IEEE
 *     bfloat16 bit patterns (gdn_bf16) and must be 16-byte aligned; fp32
 *     tensors must be 16-byte aligned; cu_seqlens 4-byte aligned.
 *   - Dense inputs: q, k (B,T,H,d_k); v, out (B,T,H,d_v); g, beta (B,T,H);
 *     states (B,H,d_k,d_v) with state[n,h,i,j] = key i, value j.
 *   - Packed variable-length inputs (cu_seqlens != NULL): the tensors hold
 *     (1,T,H,.) with N = B sequences concatenated along T; cu_seqlens is a
 *     device int32 array of N+1 offsets, cu_seqlens[0] = 0,
 *     non-decreasing, cu_seqlens[N] = T.  The state starts afresh at each
 *     sequence (from initial_state[n] or zero); states are (N,H,d_k,d_v).
 *   - Supported sizes: d_k in {64, 128}; d_v in {64, 128, 256}; T >= 0;
 *     B >= 1 and H >= 1 (each at most 65535); B*T*H*max(d_k,d_v) < 2^40.
 *     Every g must be <= 0 (the
 *     documented domain: alpha = exp(g) in (0,1]).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *     Argument errors are found on the host and returned before any launch.
 *     Errors that only the device can see (malformed cu_seqlens, a bounded
 *     wait that ran out) are recorded in a per-device error word; the
 *     affected blocks write nothing.  Read and clear it with
 *     gdn_get_last_device_error().
 *   - Results are deterministic: the same inputs give bitwise-identical
 *     outputs on every launch (no atomics on data paths).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

/* IEEE bfloat16 stored as its 16-bit pattern. */
typedef uint16_t gdn_bf16;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null required pointer, negative/zero size, bad workspace */
    GDN_ERR_UNSUPPORTED = 2,   /* d_k / d_v outside the supported set, size too large */
    GDN_ERR_MISALIGNED = 3,    /* a tensor pointer is not 16-byte aligned */
    GDN_ERR_BAD_SEQLENS = 4,   /* device found cu_seqlens not 0 .. T non-decreasing */
    GDN_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up (kernel returned early) */
    GDN_ERR_CUDA = 6           /* a CUDA runtime call failed (launch, sync, copy) */
} gdn_status;

/* Chunk length used by the library (tokens per chunk). */
#define GDN_CHUNK 64

/* Human-readable name of a status code (static string, never NULL). */
GDN_API const char* gdn_status_string(gdn_status status);

/*
 * Bytes of device workspace gdn_chunk_fwd uses for these sizes: the bf16
 * hi/lo tiles of T = (I + A)^-1 of every chunk, 16 KB per chunk and head
 * (0 for unsupported sizes).  varlen != 0 when cu_seqlens will be given
 * (B is then the sequence count).
 */
GDN_API size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * Forward.  Reads q, k, v, g, beta (and initial_state, cu_seqlens when not
 * NULL); writes out (bf16, round-to-nearest-even) and, when final_state is
 * not NULL, the fp32 state after each sequence's last token.
 *   q, k          (B,T,H,d_k) bf16          v, out (B,T,H,d_v) bf16
 *   g             (B,T,H) fp32, log decay   beta   (B,T,H) bf16
 *   scale         readout scale (usually d_k^-0.5)
 *   initial_state (N,H,d_k,d_v) fp32 or NULL (zeros)
 *   cu_seqlens    NULL (dense) or device int32[N+1] (packed; N = B)
 *   final_state   (N,H,d_k,d_v) fp32 or NULL (not written)
 *   workspace     optional device scratch, 256-byte aligned.  With at least
 *                 gdn_chunk_fwd_workspace_size() bytes, every chunk's T is
 *                 formed first by a chunk-parallel kernel and the chunk chain
 *                 reads it (the faster route); with NULL or fewer bytes the
 *                 chunk chain forms T itself.  Both routes give the same
 *                 arithmetic.  A non-NULL workspace that is not 256-byte
 *                 aligned returns GDN_ERR_MISALIGNED.
 * Returns GDN_OK once the work is enqueued on `stream`.
 */
GDN_API gdn_status gdn_chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         gdn_bf16* out, float* final_state,
                         int B, int T, int H, int d_k, int d_v,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Token-serial forward: the same recurrence and arguments as gdn_chunk_fwd
 * (without a workspace), applied one token at a time ("Research Sprint Day 1",
 * section "The GDN update": decay, read v_old = S^T k, write the error
 * beta (v - v_old) along k, read out scale S^T q), with the fp32 state in
 * registers.  Meant for decode (a few tokens per call, state carried through
 * initial_state / final_state) and as a second GPU path for checks; for long
 * sequences gdn_chunk_fwd is much faster.  Same validation, layouts and error
 * behaviour as gdn_chunk_fwd; T = 0 copies initial_state (or zeros) to
 * final_state.
 */
GDN_API gdn_status gdn_recurrent_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                             const float* g, const gdn_bf16* beta, float scale,
                             const float* initial_state, const int32_t* cu_seqlens,
                             gdn_bf16* out, float* final_state,
                             int B, int T, int H, int d_k, int d_v, cudaStream_t stream);

/*
 * Token-serial forward of the per-channel-gate (KDA) variant that cuLA issue
 * #126 runs: g is (B, T, H, d_k) fp32, one log decay per key channel, and the
 * state update decays each key row of S by its own factor,
 * S <- diag(exp(g_t)) S; everything else (arguments, layouts, validation,
 * errors) is as gdn_recurrent_fwd.  gdn_kda_chunk_fwd below is the
 * chunked form of the same recurrence.
 */
GDN_API gdn_status gdn_kda_recurrent_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                 const float* g, const gdn_bf16* beta, float scale,
                                 const float* initial_state, const int32_t* cu_seqlens,
                                 gdn_bf16* out, float* final_state,
                                 int B, int T, int H, int d_k, int d_v, cudaStream_t stream);

/*
 * Bytes of the optional workspace of gdn_kda_chunk_fwd: T and P of every
 * chunk in fp32, 32 KB per chunk and head (0 for unsupported sizes).  varlen
 * as in gdn_chunk_fwd_workspace_size.
 */
GDN_API size_t gdn_kda_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * Chunked forward of the same per-channel-gate (KDA) recurrence: the sequence
 * is cut into chunks of 64 tokens, each chunk's gram A_ij = beta_i sum_c
 * k_ic k_jc exp(G_ic - G_jc) (j < i; G the per-channel running sum of g
 * inside the chunk) and causal score are formed with the decay inside the
 * sum over key channels, T = (I + A)^-1 by blocked forward substitution, and
 * the state passes from chunk to chunk, S <- diag(exp(G_n)) S +
 * (exp(G_n - G) o K)^T Delta.  All arithmetic fp32 on the CUDA cores; the
 * walk runs one thread block per (64 value columns, head, sequence).
 * Arguments, layouts, validation and errors as gdn_kda_recurrent_fwd (g is
 * (B, T, H, d_k) fp32, documented domain g <= 0), plus:
 *   workspace     optional device scratch, 256-byte aligned.  With at least
 *                 gdn_kda_chunk_fwd_workspace_size() bytes, every chunk's T
 *                 and P are formed first by a chunk-parallel kernel and the
 *                 walk reads them (the faster route: at d_k = 128 the walk
 *                 runs on the tensor cores over bf16 hi/lo operands); with
 *                 NULL or fewer bytes the walk forms them itself, fp32
 *                 throughout.  Both routes compute the same
 *                 algebra and agree within rounding.  A non-NULL workspace
 *                 that is not 256-byte aligned returns GDN_ERR_MISALIGNED.
 * Same result as the token-serial kernel up to fp32 rounding order.
 */
GDN_API gdn_status gdn_kda_chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                     const float* g, const gdn_bf16* beta, float scale,
                                     const float* initial_state, const int32_t* cu_seqlens,
                                     gdn_bf16* out, float* final_state,
                                     int B, int T, int H, int d_k, int d_v,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace gdn_kda_chunk_bwd needs for these sizes. */
GDN_API size_t gdn_kda_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * Backward of gdn_kda_chunk_fwd: the reverse mode of its chunk algebra,
 * chunk by chunk from the last, with the gradient w.r.t. each chunk's end
 * state carried backwards.  Arguments, layouts, validation and errors as
 * gdn_chunk_bwd, except that g and dg are (B, T, H, d_k) fp32: dg is the
 * gradient w.r.t. each token's per-channel log decay.  Four kernels: T and P
 * of every chunk (chunk-parallel, CUDA cores); the forward walk recording
 * each chunk's start state; the reverse walk of the state gradient (one
 * block per 64 value columns, head and sequence); the local gradients of
 * every chunk (chunk-parallel), which sum over the value columns once and
 * evaluate the decayed pair sums of the gram and the causal score once per
 * chunk.  At d_k = 128 the walks and the local gradients' products run on
 * the tensor cores (bf16 hi/lo operands, fp32 accumulation); at d_k = 64
 * everything is fp32 on the CUDA cores.  `workspace` (256-byte aligned, at least
 * gdn_kda_chunk_bwd_workspace_size() bytes, contents on entry ignored) holds
 * T and P and the per-chunk states and state gradients.  Every sum runs in a
 * fixed order: repeated calls give the same bits.
 */
GDN_API gdn_status gdn_kda_chunk_bwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                     const float* g, const gdn_bf16* beta, float scale,
                                     const float* initial_state, const int32_t* cu_seqlens,
                                     const gdn_bf16* d_out, const float* d_final_state,
                                     gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                                     gdn_bf16* dbeta, float* d_initial_state,
                                     int B, int T, int H, int d_k, int d_v,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Prologue: q/k L2 normalisation and the two gates from their raw inputs
 * ("Research Sprint Day 2 - Rooflines", GDN layer pseudocode steps 4 and 5),
 * producing the q, k, g, beta that gdn_chunk_fwd / gdn_chunk_bwd take.
 *   q_raw, k_raw  (rows, H, d_k) bf16; either may be NULL (then q / k must be
 *                 NULL too and that tensor is not touched)
 *   q, k          (rows, H, d_k) bf16 out: x / sqrt(|x|^2 + 1e-6) per row, in fp32, RNE
 *   a, b          (rows, H) fp32 raw gate inputs
 *   A_log, dt_bias (H) fp32; dt_bias may be NULL (zeros); A_log is required
 *                 for gate_mode 1
 *   gate_mode     1: g = -exp(A_log[h]) softplus(a + dt_bias[h])   (decay gate)
 *                 2: g = lower sigmoid(a + dt_bias[h])              (bounded gate,
 *                    fla issue #1550's CP2 test uses lower = -5)
 *   beta_scale    beta = beta_scale sigmoid(b) (2 allows negative eigenvalues)
 *   g             (rows, H) fp32 out;  beta (rows, H) bf16 out
 *   rows          tokens (B * T dense, total T packed);  d_k in {64, 128}
 * Returns GDN_OK once enqueued; GDN_ERR_INVALID_ARG for a bad mode, missing
 * pointer or inconsistent q/k pair, GDN_ERR_MISALIGNED for a pointer that is
 * not 16-byte aligned.
 */
GDN_API gdn_status gdn_prologue_fwd(const gdn_bf16* q_raw, const gdn_bf16* k_raw, const float* a,
                            const float* b, const float* A_log, const float* dt_bias,
                            int gate_mode, float lower, float beta_scale, gdn_bf16* q,
                            gdn_bf16* k, float* g, gdn_bf16* beta, int rows, int H, int d_k,
                            cudaStream_t stream);

/*
 * Reverse mode of gdn_prologue_fwd, from the gradients w.r.t. its outputs
 * (dq, dk, dg, dbeta, as gdn_chunk_bwd returns them): dq_raw, dk_raw (bf16),
 * da, db (fp32, (rows, H)) and the per-head sums dA_log, ddt_bias (fp32 (H),
 * each may be NULL; dA_log is not written for gate_mode 2).  With
 * r = (|x|^2 + 1e-6)^-1/2 and y = r x: dx = r (dy - y (y . dy)).  The per-head
 * sums run in a fixed order (deterministic).
 */
GDN_API gdn_status gdn_prologue_bwd(const gdn_bf16* q_raw, const gdn_bf16* k_raw, const float* a,
                            const float* b, const float* A_log, const float* dt_bias,
                            int gate_mode, float lower, float beta_scale, const gdn_bf16* dq,
                            const gdn_bf16* dk, const float* dg, const gdn_bf16* dbeta,
                            gdn_bf16* dq_raw, gdn_bf16* dk_raw, float* da, float* db,
                            float* dA_log, float* ddt_bias, int rows, int H, int d_k,
                            cudaStream_t stream);

/* Bytes of device workspace gdn_chunk_bwd needs for these sizes. */
GDN_API size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * Backward (reverse mode of gdn_chunk_fwd).  Given the forward inputs and the
 * upstream gradients d_out (B,T,H,d_v) bf16 and d_final_state
 * (N,H,d_k,d_v) fp32 or NULL (zero), writes
 *   dq, dk (B,T,H,d_k) bf16;  dv (B,T,H,d_v) bf16;
 *   dg (B,T,H) fp32 -- gradient w.r.t. the per-token g (not its cumsum);
 *   dbeta (B,T,H) bf16 -- gradient w.r.t. beta as passed;
 *   d_initial_state (N,H,d_k,d_v) fp32, or NULL (not written).
 * The chunk-start states and T tiles are recomputed into `workspace`
 * (256-byte aligned; contents on entry do not matter).
 * Returns GDN_OK once the work is enqueued on `stream`.
 */
GDN_API gdn_status gdn_chunk_bwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         const gdn_bf16* d_out, const float* d_final_state,
                         gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                         gdn_bf16* dbeta, float* d_initial_state,
                         int B, int T, int H, int d_k, int d_v,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Training route: a forward that keeps what the backward would otherwise
 * recompute, and the backward that reuses it.  fla issue #1550's validation
 * plan names both variants, retained and recomputed chunk states;
 * gdn_chunk_bwd recomputes them (no memory kept between the calls), this
 * route retains them (one T kernel and one chain pass fewer per step).
 *
 * Bytes of the saved-for-backward buffer for these sizes: every chunk's start
 * state (4 d_k d_v bytes per chunk and head, as bf16 hi/lo operand tiles),
 * then the T = (I + A)^-1 tiles (16 KB per chunk and head); 0 for unsupported
 * sizes.  At B=4, H=16, T=4096, d_k=d_v=128: 320 MiB.
 */
GDN_API size_t gdn_chunk_saved_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * gdn_chunk_fwd that also fills `saved` (device, 256-byte aligned, at least
 * gdn_chunk_saved_size() bytes; contents on entry do not matter): one chunk
 * chain writes out, final_state and every chunk's start state; the T tiles
 * come from the chunk-parallel kernel first.  out and final_state are
 * bitwise those of gdn_chunk_fwd.  Arguments, layouts and errors as
 * gdn_chunk_fwd, plus GDN_ERR_INVALID_ARG for a missing or short `saved` and
 * GDN_ERR_MISALIGNED for a misaligned one.
 */
GDN_API gdn_status gdn_chunk_fwd_save(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                              const float* g, const gdn_bf16* beta, float scale,
                              const float* initial_state, const int32_t* cu_seqlens,
                              gdn_bf16* out, float* final_state,
                              int B, int T, int H, int d_k, int d_v,
                              void* saved, size_t saved_bytes, cudaStream_t stream);

/* Bytes of device workspace gdn_chunk_bwd_saved needs: the per-chunk
 * end-state gradients (4 d_k d_v bytes per chunk and head). */
GDN_API size_t gdn_chunk_bwd_saved_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen);

/*
 * gdn_chunk_bwd from the buffer that gdn_chunk_fwd_save filled for the same
 * q, k, v, g, beta, initial_state and cu_seqlens (the caller keeps them
 * unchanged in between; nothing checks this).  It skips the T kernel and the
 * forward state pass: only the reverse chain of state gradients and the
 * chunk-parallel gradient pass run.  The initial state is not an argument
 * (the saved start states hold it).  Gradients are bitwise those of
 * gdn_chunk_bwd.  `saved` is only read; `workspace` (256-byte aligned, at
 * least gdn_chunk_bwd_saved_workspace_size() bytes) is scratch.  Errors as
 * gdn_chunk_bwd.
 */
GDN_API gdn_status gdn_chunk_bwd_saved(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                               const float* g, const gdn_bf16* beta, float scale,
                               const int32_t* cu_seqlens,
                               const gdn_bf16* d_out, const float* d_final_state,
                               gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                               gdn_bf16* dbeta, float* d_initial_state,
                               int B, int T, int H, int d_k, int d_v,
                               const void* saved, size_t saved_bytes,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device error word of
 * the current device: GDN_OK, GDN_ERR_BAD_SEQLENS or GDN_ERR_TIMEOUT
 * (GDN_ERR_CUDA if the synchronisation or the read itself failed).
 * The word is one per device, not one per stream: with library calls in
 * flight on several streams of the same device, the code returned (and
 * cleared) may come from another stream's call.  Callers that need to tell
 * their calls apart serialise them, or synchronise the device before
 * reading.  The first error recorded wins; later ones are dropped until the
 * word is cleared.
 */
GDN_API gdn_status gdn_get_last_device_error(cudaStream_t stream);

/*
 * Backward without any allocation: gdn_chunk_bwd with the same arguments
 * except the workspace, which comes from a device array built into the
 * library (GDN_NOALLOC_SCRATCH_BYTES bytes, held by every device that loads
 * the library until the process exits).  The pages have no counterpart; it
 * exists for callers that may not allocate device memory themselves (a
 * runtime that fixes its memory plan at start-up, a plugin whose host
 * framework owns all allocations), which therefore cannot supply a
 * workspace.  The caller still allocates and passes inputs and outputs.
 *   - Sizes whose workspace (gdn_chunk_bwd_workspace_size) exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES return GDN_ERR_UNSUPPORTED before any launch.
 *   - The first call on a device looks up the array's device address (a
 *     host-side runtime query); make that first call before any stream
 *     capture.
 *   - All calls in the process share the one array per device: calls whose
 *     work overlaps on the GPU (e.g. on two streams at once) race and give
 *     wrong results.  Serialise them.
 * Never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
GDN_API gdn_status gdn_chunk_bwd_noalloc(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         const gdn_bf16* d_out, const float* d_final_state,
                         gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                         gdn_bf16* dbeta, float* d_initial_state,
                         int B, int T, int H, int d_k, int d_v, cudaStream_t stream);

/*
 * Sequence split: gdn_chunk_fwd (dense inputs, no cu_seqlens) with every
 * sequence run as nseg segments of whole chunks, for long sequences with few
 * heads, where one chain per (sequence, head, value slice) leaves most of the
 * GPU idle.  cuLA issue #126 ("Hypothesis") describes the scheme: each
 * segment maps its start state affinely, S_end = M S_start + b, and the
 * carries compose in order.  Here b is a segment's end state from a zero
 * start and M its end state from the identity with zero values (both from
 * the chunk chain), the composition is fp32, and each segment then runs
 * from its true start.  Costs about three times the chain work of the
 * unsplit forward, in nseg times as many chains.
 *   nseg >= 1; more segments than chunks are clamped to one chunk each.
 *   workspace: device, 256-byte aligned, gdn_chunk_fwd_split_workspace_size()
 *   bytes (a few arrays of the inputs' and the states' sizes).
 * Outputs as gdn_chunk_fwd, to within rounding (not bitwise: the carries
 * change the order of the arithmetic).  Errors as gdn_chunk_fwd, plus
 * GDN_ERR_INVALID_ARG for nseg < 1 or a missing or short workspace and
 * GDN_ERR_UNSUPPORTED for B T >= 2^31.
 */
GDN_API size_t gdn_chunk_fwd_split_workspace_size(int B, int T, int H, int d_k, int d_v, int nseg);
GDN_API gdn_status gdn_chunk_fwd_split(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                               const float* g, const gdn_bf16* beta, float scale,
                               const float* initial_state, gdn_bf16* out, float* final_state,
                               int B, int T, int H, int d_k, int d_v, int nseg,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Peak probes: the denominators of a roofline, measured on the caller's GPU
 * in the same run as the operator ("Research Sprint Day 2 - Rooflines",
 * section "Rooflines": FLOP/s from 8192 x 8192 by 8192 x 8192 dense matmuls,
 * bandwidth from copying a 2 GB tensor).  Measurement tools, not part of
 * the operator; both are asynchronous on `stream`.
 *
 * gdn_probe_copy: dst[0 .. bytes) = src[0 .. bytes) with 16-byte vector
 * loads and stores (streaming cache hints).  bytes % 16 != 0 or a NULL
 * pointer (bytes > 0) returns GDN_ERR_INVALID_ARG; a pointer that is not
 * 16-byte aligned GDN_ERR_MISALIGNED.  The buffers must not overlap.
 */
GDN_API gdn_status gdn_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream);

/*
 * gdn_probe_gemm_bf16: C = A B^T on the tensor cores (tcgen05, fp32
 * accumulation in tensor memory, bf16 round-to-nearest-even output).
 *   A (M, K), B (N, K), C (M, N): bf16, row-major, 16-byte aligned.
 *   M % 128 == 0, N % 256 == 0, K % 64 == 0, each <= 65536, else
 *   GDN_ERR_UNSUPPORTED; non-positive sizes or NULL GDN_ERR_INVALID_ARG.
 * A bounded wait that gives up sets GDN_ERR_TIMEOUT in the device error word.
 */
GDN_API gdn_status gdn_probe_gemm_bf16(const gdn_bf16* A, const gdn_bf16* B, gdn_bf16* C, int M, int N, int K,
                                       cudaStream_t stream);

/*
 * gdn_chunk_fwd with a caller-chosen bound on the kernels' hand-off waits
 * (mbarrier waits between the warps of a CTA), for exercising failure
 * detection.  wait_limit counts polls (0 = the default; each poll may
 * suspend the thread until the awaited phase completes, so a small bound
 * alone rarely runs out).  With stall_first_wait != 0 the issuing warp of
 * every CTA first waits on a hand-off that nothing signals, so that wait
 * runs out: the CTA records GDN_ERR_TIMEOUT in the device error word (read
 * it with gdn_get_last_device_error), waits with the default bound for every
 * copy and tensor-core product it started, and leaves without writing its
 * final state, so the context stays usable.  Library bookkeeping with no
 * counterpart on the pages.  Takes a workspace of at least
 * gdn_chunk_fwd_workspace_size() bytes and d_k = 128 (the tile route this
 * test covers); otherwise GDN_ERR_UNSUPPORTED.  Other arguments and errors
 * as gdn_chunk_fwd.
 */
GDN_API gdn_status gdn_chunk_fwd_wait_limit(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                    const float* g, const gdn_bf16* beta, float scale,
                                    const float* initial_state, const int32_t* cu_seqlens,
                                    gdn_bf16* out, float* final_state,
                                    int B, int T, int H, int d_k, int d_v,
                                    void* workspace, size_t workspace_bytes, uint32_t wait_limit,
                                    int stall_first_wait, cudaStream_t stream);

/*
 * gdn_chunk_bwd_saved with a caller-chosen bound on the hand-off waits of the
 * chunk-parallel gradient pass (mbarrier waits between its epilogue warps and
 * its MMA-issuing warp), for exercising failure detection; the reverse chain
 * of state gradients keeps the default bound.  wait_limit counts polls (0 =
 * the default).  With stall_first_wait != 0 the epilogue warps of every CTA
 * first wait on a barrier that nothing signals, so that wait runs out: at the
 * next hand-off every warp of the CTA (the issuing warp included) leaves its
 * loop, the CTA waits with the default bound for every copy and product it
 * started, records GDN_ERR_TIMEOUT in the device error word (read it with
 * gdn_get_last_device_error) and writes no gradient of dq, dk, dv, dg or
 * dbeta, so the context stays usable.  Library bookkeeping with no
 * counterpart on the pages.  Other arguments and errors as
 * gdn_chunk_bwd_saved.
 */
GDN_API gdn_status gdn_chunk_bwd_saved_wait_limit(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                          const float* g, const gdn_bf16* beta, float scale,
                                          const int32_t* cu_seqlens,
                                          const gdn_bf16* d_out, const float* d_final_state,
                                          gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                                          gdn_bf16* dbeta, float* d_initial_state,
                                          int B, int T, int H, int d_k, int d_v,
                                          const void* saved, size_t saved_bytes,
                                          void* workspace, size_t workspace_bytes, uint32_t wait_limit,
                                          int stall_first_wait, cudaStream_t stream);

/*
 * Number of CUDA kernels this library has launched in this process so far
 * (all devices, all entry points).  Library bookkeeping with no counterpart
 * on the pages; lets a caller count the kernels inside a timed region.
 */
GDN_API uint64_t gdn_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */

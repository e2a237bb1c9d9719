/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) on one GB300 (sm_103a).
 *
 * The operation is the KDA recurrence of "[Paper Review] Kimi K3: Open Frontier
 * Intelligence" (baba9811.github.io), section "Kimi Delta Attention (KDA)".
 * Per sequence and head, with state S in R^{dk x dv}:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t,          alpha_t = exp(g_t) in (0, 1]^{dk}
 *
 * Diag(alpha_t) is the channel-wise forget gate applied to the prior state and
 * (I - beta_t k_t k_t^T) erases the key direction before the new pair is
 * written (same section).  The caller supplies g itself; the same section's
 * lower-bounded decay g = g_min * sigmoid(.) with g_min = -5 makes g lie in
 * [-5, 0], which is the precondition of the chunked tensor-core path.  There
 * is no 1/sqrt(dk) output scale: q and k are L2-normalised upstream.
 *
 * Layouts (row-major, tokens packed back to back, all buffers on the device):
 *   q, k, g     [T_total, H, dk]      v, out  [T_total, H, dv]
 *   beta        [T_total, H]          states  [N, H, dk, dv]  fp32, dv fastest
 * q, k, v, g, beta and out share one element type (kda_dtype); states are
 * always fp32.
 *
 * Ownership: the caller owns every buffer.  The library keeps no pointer past
 * the call and allocates no device memory; scratch comes from the caller's
 * workspace.
 * Streams: every call only enqueues work on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and returns without synchronising.  The split
 * tensor-core prefill (see kda_chunk_fwd) also runs its state kernels on a
 * helper stream of the library (one per device, highest priority), joined to
 * `stream` by events before and after, so work on `stream` stays ordered;
 * calls from several host threads serialise while they enqueue.
 * Errors: argument errors are detected on the host and returned before any
 * launch; launch failures return KDA_ERR_CUDA.  Errors found while kernels run
 * (a bounded wait that expired) are written to the optional device word
 * *dev_status (0 = fine), which the caller reads after synchronising.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID = -1,     /* null pointer, negative or inconsistent size      */
  KDA_ERR_UNSUPPORTED = -2, /* well-formed but not implemented (dims, dtype)    */
  KDA_ERR_CUDA = -3,        /* a CUDA runtime/driver call or a launch failed     */
  KDA_ERR_TIMEOUT = -4,     /* device: a bounded wait expired (via dev_status)  */
  KDA_ERR_ALIGNMENT = -5,   /* a buffer is not 16-byte aligned where required   */
  KDA_ERR_WORKSPACE = -6,   /* workspace missing or smaller than required       */
  KDA_ERR_SCRATCH_LIMIT = -7, /* more sequences than kda_chunk_fwd_noalloc holds */
  KDA_ERR_RANGE = -8         /* device: g outside [-5, 0] or beta outside [0, 1]
                                (kda_check_inputs; via dev_status)               */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef struct {
  int n_seqs;              /* N: sequences (prefill) or concurrent streams (decode) */
  long long total_tokens;  /* T_total: packed tokens; decode: must equal n_seqs     */
  int heads;               /* H                                                     */
  int dk, dv;              /* key / value head dims: each 64 or 128                 */
  int dtype;               /* kda_dtype of q, k, v, g, beta, out                    */
} kda_dims;

/*
 * Bytes of device workspace kda_chunk_fwd needs for these dims and chunk size
 * (0 when none is needed).  Never fails; returns 0 for invalid dims.
 */
KDA_API size_t kda_chunk_fwd_workspace_size(const kda_dims* dims, int chunk);

/*
 * Chunkwise prefill over packed variable-length sequences (the chunkwise
 * parallel form the same section names; the page's 16-token tiles inside a
 * chunk are what make it run on tensor cores).
 *
 *   q, k, v, g, beta  inputs, layouts above.
 *   init_state        [N, H, dk, dv] fp32 state entering each sequence, or NULL
 *                     for zeros.
 *   cu_seqlens        device int32 [N + 1]: sequence n owns tokens
 *                     [cu[n], cu[n+1]); cu[0] = 0, cu[N] = T_total, non-
 *                     decreasing (empty sequences pass init_state through).
 *                     NULL: N sequences of equal length T_total / N.
 *   out               [T_total, H, dv] outputs o_t (same dtype as v).
 *   final_state       [N, H, dk, dv] fp32 state after each sequence, or NULL.
 *                     May alias init_state.
 *   chunk             tokens per chunk: 16, 32 or 64.  Results agree across
 *                     chunk sizes up to rounding.
 *   workspace         device scratch of kda_chunk_fwd_workspace_size() bytes
 *                     (256-byte aligned), or NULL when that size is 0.
 *   dev_status        optional device int, set non-zero by a kernel whose
 *                     bounded wait expired (KDA_ERR_TIMEOUT); never cleared.
 *   stream            cudaStream_t to enqueue on.
 * Paths: bf16 with dk = dv = 128 runs on tcgen05 tensor cores (requires q,
 * k, v, g, out 16-byte aligned); a requested chunk of 16 or 32 tokens is
 * served there by 64-token chunks made of the same 16-token tiles (the chunk
 * size blocks the computation and does not change the result).  Every other
 * supported case runs the fp32 CUDA-core kernel that walks the recurrence.
 * On tensor cores, few
 * (sequence, head) pairs (N x H <= 304) or few sequences (N <= 32) run the
 * split form, given a workspace of kda_chunk_fwd_workspace_size() bytes: a
 * preparation kernel over every chunk at once, which writes a 66,048-byte
 * record per chunk into the workspace, then a state kernel per pair.  The
 * records fill at most 2 GiB when N x H <= 76 (windows of chunks then overlap
 * the state pass of one with the preparation of the next) and at most 32 GiB
 * otherwise; longer inputs run in windows with the state carried between
 * them.  When N x H fits the SMs in one wave but leaves fewer than half of
 * them free and every record fits, the chunks run as two windows: the state
 * pass of the first (most of the chunks) beside the preparation of the
 * second on the SMs it leaves free.  The helper streams this uses are the
 * library's own, joined to the caller's stream by events before the call
 * returns.
 * A smaller workspace that still holds the order array, N x H fp32 states and
 * one record per pair runs the split form in more, smaller windows; below
 * that, and otherwise, one fused kernel per pair runs.  The
 * environment variable KDA_CHUNK_PATH=fused|split overrides the choice.
 * Inputs with g outside [-5, 0] are outside the tensor-core path's contract;
 * kda_check_inputs (below) checks it on the device, and a KDA_DEBUG_BOUNDS
 * build of the library runs that check inside the call.
 */
KDA_API int kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                  const float* init_state, const int* cu_seqlens, void* out, float* final_state,
                  int chunk, const kda_dims* dims, void* workspace, size_t workspace_bytes,
                  int* dev_status, void* stream);

/*
 * kda_chunk_fwd that also writes prefix-cache checkpoints: the fp32 state of
 * every (sequence, head) after each `ckpt_interval` tokens of the sequence.
 * The serving description of the Kimi K3 architecture-atlas entry keeps KDA
 * state checkpoints at 512-token hash boundaries beside the MLA KV pages
 * ("KDA-aware prefix cache", also in the paper review's section
 * "Infrastructure: how to actually run trillion-scale").
 *
 *   checkpoints   fp32 [n_ckpt, H, dk, dv]: checkpoint j of sequence n (the
 *                 state after (j+1) * ckpt_interval tokens of it) is row
 *                 ckpt_offsets[n] + j.  A sequence of length L has
 *                 floor(L / ckpt_interval) checkpoints; the last one equals
 *                 final_state when L is a multiple of the interval.
 *   ckpt_offsets  device int32 [N + 1]: ckpt_offsets[n+1] - ckpt_offsets[n] =
 *                 floor(len_n / ckpt_interval), ckpt_offsets[0] = 0.
 *   ckpt_interval tokens between checkpoints: a positive multiple of 64.
 * Everything else, including results, is as kda_chunk_fwd.
 */
KDA_API int kda_chunk_fwd_checkpoints(const void* q, const void* k, const void* v,
                                      const void* g, const void* beta, const float* init_state,
                                      const int* cu_seqlens, void* out, float* final_state,
                                      int chunk, const kda_dims* dims, void* workspace,
                                      size_t workspace_bytes, int* dev_status, void* stream,
                                      float* checkpoints, const int* ckpt_offsets,
                                      int ckpt_interval);

/*
 * kda_chunk_fwd followed by KDA's output epilogue: head-wise RMSNorm of every
 * output row, then the input-dependent full-rank sigmoid gate ("[Paper
 * Review] Kimi K3: Open Frontier Intelligence", section "Kimi Delta Attention
 * (KDA)", paragraph "Full-rank gate"; the page lost the formula, read as
 *   out[t, h, :] = o / sqrt(mean(o^2) + eps) * norm_weight * sigmoid(gate[t, h, :])
 * with o the KDA output of token t, head h).
 *   gate         [T_total, H, dv] gate pre-activation (the full-rank projection
 *                of the hidden state, computed upstream), dtype of v, 16-byte
 *                aligned.
 *   norm_weight  fp32 [dv] RMSNorm scale (shared by the heads), device,
 *                16-byte aligned.
 *   eps          >= 0, added to the mean square.
 * Everything else, including final_state, is as kda_chunk_fwd.  The
 * CUDA-core recurrence and the split tensor-core form apply the epilogue
 * inside their kernels (from the fp32 outputs); after the fused tensor-core
 * kernel it runs as a pass over `out`.
 */
KDA_API int kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* init_state, const int* cu_seqlens,
                                const void* gate, const float* norm_weight, float eps, void* out,
                                float* final_state, int chunk, const kda_dims* dims,
                                void* workspace, size_t workspace_bytes, int* dev_status,
                                void* stream);

/*
 * Segment transitions, the building block of KDA context parallelism (the
 * paper review's infrastructure section: each segment's state transition is
 * computed locally and the segments are composed associatively).  For every
 * (sequence, head), with the sequences of cu_seqlens taken as segments:
 *   S_end = M S_0 + H  for every entry state S_0, where
 *   M [dk, dk] = the product over the segment's tokens of
 *                (I - beta_t k_t k_t^T) Diag(alpha_t)  (later tokens on the left)
 *   H [dk, dv] = the end state from S_0 = 0.
 * trans_M, trans_H: fp32 [N, H, dk, dk] and [N, H, dk, dv] (16-byte aligned).
 * Runs the split tensor-core form (bf16, dk = dv = 128, chunk 64, N <= 1024;
 * KDA_ERR_UNSUPPORTED otherwise) with a workspace of at least
 * kda_chunk_transition_workspace_size(dims) bytes.  No outputs are written.
 */
KDA_API size_t kda_chunk_transition_workspace_size(const kda_dims* dims);
KDA_API int kda_chunk_transition(const void* q, const void* k, const void* v, const void* g,
                                 const void* beta, const int* cu_seqlens, float* trans_M,
                                 float* trans_H, int chunk, const kda_dims* dims,
                                 void* workspace, size_t workspace_bytes, int* dev_status,
                                 void* stream);

/*
 * S_out[p] = M[p] S_in[p] + H[p] for p < pairs (fp32 on the device; H may be
 * NULL for no addend; dk, dv each 64 or 128).  With S_in = a later segment's
 * entry state this moves a state across a segment; with (M, H) = (M2, H2) and
 * S_in = H1 (then M1 with H = NULL) it composes (M2, H2) after (M1, H1).
 * S_out must not alias S_in or M.
 */
KDA_API int kda_transition_apply(const float* M, const float* H, const float* S_in,
                                 float* S_out, long long pairs, int dk, int dv, void* stream);

/*
 * Single-GPU KCP prefill: each of the N equal-length sequences (no
 * cu_seqlens: T_total / N tokens each) is cut into n_segments segments
 * (multiples of 64 tokens, the last ones shorter); every segment's transition
 * is computed at once, the segments' entry states follow from the composed
 * prefixes, and every segment then runs from its own entry state.  Results are
 * those of kda_chunk_fwd on the same inputs (up to rounding).  bf16,
 * dk = dv = 128, N * n_segments <= 1024; workspace of
 * kda_chunk_fwd_kcp_workspace_size(dims, n_segments) bytes.
 */
KDA_API size_t kda_chunk_fwd_kcp_workspace_size(const kda_dims* dims, int n_segments);
KDA_API int kda_chunk_fwd_kcp(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const float* init_state, void* out,
                              float* final_state, int n_segments, const kda_dims* dims,
                              void* workspace, size_t workspace_bytes, int* dev_status,
                              void* stream);

/*
 * KDA's input prologue, in one pass ("[Paper Review] Kimi K3: Open Frontier
 * Intelligence", section "Kimi Delta Attention (KDA)": queries and keys pass
 * through a short convolution and Swish and are L2-normalised; the log-decay
 * is the lower-bounded scaled sigmoid; the page lost both formulas, read as):
 *   q = L2norm(Swish(conv(q_pre, conv_q))),  k = L2norm(Swish(conv(k_pre, conv_k)))
 *   g = -5 sigmoid(exp(a_log[h]) z)
 * conv is depthwise and causal with 4 taps along each sequence, tap 3 on the
 * current token (out_t = sum_i w[i] x_{t-3+i}, nothing before the sequence's
 * first token); Swish(y) = y sigmoid(y); L2norm(y) = y / sqrt(sum(y^2) + 1e-6)
 * over a head's dk channels.
 *   q_pre, k_pre, z   [T_total, H, dk] pre-activations (dtype of dims), z the
 *                     decay logit
 *   conv_q, conv_k    fp32 [H, dk, 4];  a_log fp32 [H] (A_h)
 *   cu_seqlens        as kda_chunk_fwd (NULL: N equal-length sequences)
 *   q, k, g           [T_total, H, dk] outputs, ready for kda_chunk_fwd
 * dims->dv is not used.  All vectors 16-byte aligned.
 */
KDA_API int kda_prologue(const void* q_pre, const void* k_pre, const void* z,
                         const float* conv_q, const float* conv_k, const float* a_log,
                         const int* cu_seqlens, void* q, void* k, void* g, const kda_dims* dims,
                         void* stream);

/*
 * One recurrent decode step (the "dedicated kernels for KDA decode" of the
 * section "Infrastructure: how to actually run trillion-scale"; the state is
 * the fixed-size d_k x d_v cache object per head).  Every one of the N
 * sequences advances by one token: q, k, g [N, H, dk], v [N, H, dv],
 * beta [N, H].  `state` [N, H, dk, dv] fp32 is read and overwritten in place;
 * out [N, H, dv] receives o.  dims->total_tokens must equal dims->n_seqs.
 */
KDA_API int kda_decode_step(const void* q, const void* k, const void* v, const void* g, const void* beta,
                    float* state, void* out, const kda_dims* dims, int* dev_status, void* stream);

/*
 * kda_decode_step with the output epilogue of kda_chunk_fwd_gated applied to
 * out inside the decode kernel (gate [N, H, dv], norm_weight fp32 [dv], eps).
 */
KDA_API int kda_decode_step_gated(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const void* gate, const float* norm_weight,
                                  float eps, float* state, void* out, const kda_dims* dims,
                                  int* dev_status, void* stream);

/*
 * kda_chunk_fwd without a workspace, for callers that cannot allocate device
 * memory: for example a plugin inside an inference engine that owns every
 * device buffer and hands out only the tensors it planned, or a serving loop
 * that must not call cudaMalloc because it synchronises the device and
 * fragments a pool sized once at start-up.  The paper has no counterpart to
 * this entry point; it exists for those callers only.
 *
 * Arguments, layouts, checks and results are those of kda_chunk_fwd; bf16
 * with dk = dv = 128 always runs the fused tensor-core kernel (the split
 * form needs a workspace for its records).  The only
 * scratch (the longest-first order of the packed sequences) lives in a fixed
 * device array inside libkda.so that holds KDA_NOALLOC_MAX_SEQS entries
 * (256 KiB); every GPU that loads the library keeps it until the process
 * exits.  No call allocates or frees memory.
 *   - More than KDA_NOALLOC_MAX_SEQS sequences: returns KDA_ERR_SCRATCH_LIMIT
 *     before any launch.
 *   - Every call looks up the array's device address for the device
 *     current at the call (cudaGetSymbolAddress, which allocates nothing),
 *     so a new context on the device (after cudaDeviceReset) is handled.
 *     The first call on a device may load the library's device code there;
 *     make that first call before any stream capture.
 *   - All calls share the one array and each call rewrites the entries it
 *     uses before reading them, so nothing carries over between calls.  Calls
 *     that overlap on the GPU (different streams, no ordering between them)
 *     race on the array: order them on one stream or with events.
 */
#define KDA_NOALLOC_MAX_SEQS 65536
KDA_API int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* init_state,
                                  const int* cu_seqlens, void* out, float* final_state,
                                  int chunk, const kda_dims* dims, int* dev_status,
                                  void* stream);

typedef enum {
  KDA_ALGO_RECURRENT = 0,       /* CUDA-core recurrence                          */
  KDA_ALGO_TCGEN05 = 1,         /* fused tensor-core kernel, one CTA per pair    */
  KDA_ALGO_TCGEN05_SPLIT = 2    /* tensor-core preparation + state kernels       */
} kda_algo;

/*
 * Kernels one kda_chunk_fwd call launches on its stream for these dims, chunk
 * size and workspace size, with cu_seqlens given (varlen != 0) or not, on the
 * current device (the library's helper streams included): the length-order
 * kernel, then the split form's preparation and state kernels per window, or
 * one fused or token-recurrence kernel (N = 0 or H = 0: none).  A
 * KDA_DEBUG_BOUNDS build adds its range check when given a dev_status.
 * Returns the count (>= 0); a negative kda_status for invalid dims or chunk,
 * KDA_ERR_WORKSPACE where the call itself would fail for want of workspace
 * (packed sequences without room for the order array), or KDA_ERR_CUDA if
 * the device cannot be queried.
 */
KDA_API int kda_chunk_fwd_launch_count(const kda_dims* dims, int chunk, size_t workspace_bytes,
                                       int varlen);

/*
 * Which kernels kda_chunk_fwd runs for these dims and chunk size (given a
 * workspace of kda_chunk_fwd_workspace_size() bytes).  Returns a negative
 * kda_status for dims kda_chunk_fwd would reject.
 */
KDA_API int kda_chunk_fwd_algorithm(const kda_dims* dims, int chunk);

/*
 * Input precondition check.  The chunked tensor-core path relies on the
 * lower-bounded decay of "[Paper Review] Kimi K3: Open Frontier
 * Intelligence", section "Kimi Delta Attention (KDA)": g = g_min sigmoid(.)
 * with g_min = -5 keeps every g in [-5, 0], so a 16-token tile's log-decay
 * stays above -80 and its in-tile factors below e^80; beta lies in [0, 1].
 * This call enqueues one pass over g [T_total, H, dk] and beta [T_total, H]
 * (dtype and sizes from dims; g 16-byte aligned) and sets *dev_status
 * (device int, required) to KDA_ERR_RANGE if any g is outside [-5, 0] or any
 * beta outside [0, 1] (NaN counts as outside), unless *dev_status already
 * holds a non-zero code.  Nothing traps.  A library built with
 * KDA_DEBUG_BOUNDS defined runs this check inside every prefill and decode
 * call that is given a dev_status (kda_debug_bounds_build() returns 1 for
 * such a build, 0 otherwise).
 */
KDA_API int kda_check_inputs(const void* g, const void* beta, const kda_dims* dims,
                             int* dev_status, void* stream);
KDA_API int kda_debug_bounds_build(void);

/* Static description of a status code (never NULL). */
KDA_API const char* kda_status_string(int status);

/*
 * Failure-detection self-test (diagnostic).  Launches one small kernel that
 * runs the library's bounded mbarrier wait on a barrier nothing ever arrives
 * at, with a limit of `timeout_us` microseconds (1 .. 10,000,000) instead of
 * the kernels' 2 s; when the limit passes, the kernel stores KDA_ERR_TIMEOUT
 * into *dev_status (device int, caller-owned, required) and returns, leaving
 * the context usable.  Asynchronous on `stream`; returns KDA_ERR_INVALID for
 * a NULL dev_status or an out-of-range limit, KDA_ERR_CUDA if the launch
 * fails, KDA_OK otherwise.
 */
KDA_API int kda_debug_wait_timeout(int* dev_status, unsigned timeout_us, void* stream);

/*
 * Failure-detection self-test of the prefill kernels themselves (diagnostic).
 * Runs kda_chunk_fwd (bf16, dk = dv = 128, chunk 64, N equal-length
 * sequences, no cu_seqlens) with one copy deliberately never issued, so that
 * a production kernel's bounded wait (2 s) expires and its abort path runs:
 *   which = 1: the split form's state kernel, the first record of pair (0, 0);
 *   which = 2: the split form's preparation kernel, the first raw tiles of
 *              its first block;
 *   which = 3: the fused kernel, the first raw tiles of block (0, 0).
 * Every role of the affected block then gives up, waits (bounded) for its
 * copies and MMAs in flight, frees its TMEM and returns; *dev_status (device
 * int, required) receives KDA_ERR_TIMEOUT and the context stays usable.  The
 * outputs of the call are not meaningful.  Forms 1 and 2 need the split
 * form's workspace (kda_chunk_fwd_workspace_size), else KDA_ERR_WORKSPACE.
 */
KDA_API int kda_debug_chunk_fwd_withhold(int which, const void* q, const void* k, const void* v,
                                         const void* g, const void* beta,
                                         const float* init_state, void* out, float* final_state,
                                         const kda_dims* dims, void* workspace,
                                         size_t workspace_bytes, int* dev_status, void* stream);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

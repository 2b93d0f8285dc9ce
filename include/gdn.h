/*
 * gdn.h -- C ABI of the GatedDeltaNet layer library (libgdn.so), GB300 / sm_103a.
 *
 * The library computes one GatedDeltaNet linear-attention layer of a hybrid
 * Qwen3.5 decoder from its post-projection streams to the gated-normed output:
 * the "GatedDeltaNet" module with its "RMSNormGated" output norm, its
 * depthwise conv1d and softplus gate ("[Qwen3.5 MoE] Add hybrid decoder model
 * (GatedDeltaNet + full attention + MoE)", Summary: model.py and
 * parallelize.py bullets), over packed variable-length sequences described by
 * cu_seqlens ("Support Qwen35 SFT", XTuner changes: GatedDeltaNet in varlen
 * mode; "feat(models): dense Qwen3.5 custom attention", Summary: varlen
 * cu_seqlens, one packed row).  The pages name these pieces without formulas;
 * the library computes, per sequence n and value head h (query/key head
 * h' = h / (h_v / h_qk)), the gated delta rule of Yang et al., "Gated Delta
 * Networks" (ICLR 2025):
 *
 *   x^  = silu(conv1d_4(x)) for x in {q, k, v}   causal depthwise, width 4,
 *         conv_w[c][3] multiplies the current token, no bias, zero history at
 *         each sequence start (prefill) or the carried cache (decode)
 *   q^, k^ <- x / sqrt(sum x^2 + 1e-6)
 *   g_t = -exp(A_log[h]) softplus(a_t + dt_bias[h]),  beta_t = sigmoid(b_t)
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t = S_t q_t / sqrt(d_k)
 *   y_t = o_t / sqrt(mean(o_t^2) + 1e-6) * norm_w * silu(z_t)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensors are dense, row-major, token-major, caller-owned DEVICE memory
 *    on the current CUDA device; the library keeps no pointer after a call
 *    returns.  Stream tensors start on a 16-byte boundary.
 *  - Streams (dtype = io_dtype): q, k [T, h_qk, d_k]; v, z, out [T, h_v, d_v];
 *    a, b [T, h_v].  Parameters (always fp32): conv_w [Cc, 4] with
 *    Cc = 2 h_qk d_k + h_v d_v, channels ordered [q heads | k heads | v heads],
 *    each head-major then dim; A_log, dt_bias [h_v]; norm_w [d_v] (shared by
 *    all heads).
 *  - States (fp32): [N, h_v, d_k, d_v]; element [n][h][i][j] = S[j][i], i over
 *    d_k, j over d_v.
 *  - Supported shapes: 1 <= h_qk, h_v % h_qk == 0; d_k, d_v multiples of 16 in
 *    [16, 128].  The tensor-core prefill runs bf16 streams with
 *    d_k = d_v = 128; every other supported shape runs a token-sequential fp32
 *    kernel.  Anything else returns GDN_ERR_UNSUPPORTED.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous: they enqueue kernels and return without synchronising.
 *    With a caller-owned workspace (and the trace off) a prefill or decode
 *    call can be captured in a CUDA graph and replayed, the graph reading
 *    whatever values the captured buffers hold at replay time; calls on
 *    different streams with their own workspaces may run concurrently.
 *  - Errors.  Invalid arguments (NULL required pointer, non-positive size,
 *    misalignment, h_v not a multiple of h_qk, short workspace) return a status
 *    before anything is launched.  A failed launch returns GDN_ERR_CUDA.
 *    Problems only the device can see (cu_seqlens not non-decreasing within
 *    [0, T]; a bounded wait inside a kernel running out) are recorded in the
 *    workspace's status word and read back with gdn_workspace_status().  No
 *    entry point aborts, throws or traps.
 *  - Thread safety: entry points hold no global state and may be called from
 *    several host threads at once (with distinct workspaces); the one
 *    exception is gdn_prefill_noalloc, whose comment says how it shares state.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* NULL / non-positive / misaligned / inconsistent argument */
  GDN_ERR_UNSUPPORTED = 2,  /* valid but unsupported shape or dtype */
  GDN_ERR_WORKSPACE = 3,    /* workspace given but smaller than gdn_prefill_workspace_bytes() */
  GDN_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  GDN_ERR_DEVICE_CHECK = 5, /* device-side validation failed (bad cu_seqlens) */
  GDN_ERR_TIMEOUT = 6       /* a bounded device-side wait ran out */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

typedef struct {
  int32_t num_tokens; /* T: packed tokens (prefill) or batch size B (decode)      */
  int32_t num_seqs;   /* N: sequences in cu_seqlens (prefill); ignored by decode  */
  int32_t h_qk;       /* query/key heads                                          */
  int32_t h_v;        /* value heads, a multiple of h_qk                          */
  int32_t d_k;        /* query/key head dim                                       */
  int32_t d_v;        /* value head dim                                           */
  int32_t io_dtype;   /* gdn_dtype of the streams q, k, v, a, b, z, out, conv cache */
} gdn_dims;

/*
 * Bytes of device workspace gdn_prefill needs for `dims` (0 if dims is NULL or
 * invalid).  The workspace holds the device status word, the chunk schedule
 * (per sequence its first chunk, the order in which the state pass takes the
 * sequences, per chunk its tokens) and, on the chunked path, the operand
 * images the chunk preparation hands to the state pass (72.25 KiB per chunk
 * of 64 tokens and value head).  It is scratch: its contents need not be
 * preserved between calls, but a call's status word stays readable until the
 * next call that uses the same workspace.
 */
GDN_API size_t gdn_prefill_workspace_bytes(const gdn_dims *dims);

/*
 * Prefill: run the layer over N packed sequences of T tokens in total.
 *
 * cu_seqlens  int32 [N+1] on the device: sequence n owns tokens
 *             [cu_seqlens[n], cu_seqlens[n+1]); cu_seqlens[0] = 0,
 *             cu_seqlens[N] = T, non-decreasing (an empty sequence is allowed:
 *             its final state equals its initial state).
 * init_state  fp32 [N, h_v, d_k, d_v] or NULL (= zeros).
 * out         io_dtype [T, h_v, d_v]: y, rounded to nearest (even) for bf16.
 * final_state fp32 [N, h_v, d_k, d_v] or NULL (= not returned).  It may equal
 *             init_state (in-place update): each chain reads its state before
 *             it writes it.
 * workspace   device scratch of ws_bytes >= gdn_prefill_workspace_bytes(dims)
 *             bytes, 256-byte aligned; or NULL, in which case the library takes
 *             and returns stream-ordered memory (cudaMallocAsync /
 *             cudaFreeAsync) around the launch.
 * Returns a gdn_status.
 */
GDN_API int gdn_prefill(const gdn_dims *dims, const void *q, const void *k, const void *v, const void *a,
                const void *b, const void *z, const float *conv_w, const float *A_log,
                const float *dt_bias, const float *norm_w, const int32_t *cu_seqlens,
                const float *init_state, void *out, float *final_state, void *workspace,
                size_t ws_bytes, void *stream);

/*
 * Prefill that carries the conv history across calls: gdn_prefill plus an
 * initial conv history in and the conv history the call leaves out.
 *
 * The pages run the layer under context parallelism ("[Qwen3.5 MoE] Add
 * hybrid decoder model (GatedDeltaNet + full attention + MoE)", Summary:
 * parallelize.py bullet, TP/FSDP/CP/EP with a DTensor-safe depthwise conv1d;
 * "feat(models): dense Qwen3.5 custom attention", Summary: ring / Ulysses CP
 * substitution, and its E2E notes: CP hooks at cp = 2), where one sequence is
 * split into consecutive segments on different ranks.  The recurrence carries
 * across a split through init_state / final_state; the width-4 causal conv
 * also reads the three raw inputs before a segment's first token, which a
 * plain gdn_prefill takes as zeros.  With this entry point, running a sequence
 * as segments [t_0, t_1), [t_1, t_2), ... -- each call's init_state and
 * init_conv the previous call's final_state and final_conv -- gives the same
 * result as one call over the whole sequence (and the same for long prompts
 * prefilled piece by piece).
 *
 * init_conv   io_dtype [N, Cc, 3] or NULL (= zeros, a plain gdn_prefill): per
 *             sequence and conv channel (order [q | k | v], as conv_w) the raw
 *             inputs of the three tokens before the sequence's first token,
 *             oldest first -- the layout of the decode conv cache.
 * final_conv  io_dtype [N, Cc, 3] or NULL (= not returned): the same for the
 *             three tokens after the call (for a sequence shorter than three
 *             tokens, partly taken from init_conv).  It may equal init_conv
 *             (written after every read of it); it is also exactly the
 *             conv_state gdn_decode_step continues from.
 * Every other argument, the workspace and the errors are those of
 * gdn_prefill.  Returns a gdn_status.
 */
GDN_API int gdn_prefill_carry(const gdn_dims *dims, const void *q, const void *k, const void *v,
                              const void *a, const void *b, const void *z, const float *conv_w,
                              const float *A_log, const float *dt_bias, const float *norm_w,
                              const int32_t *cu_seqlens, const float *init_state, const void *init_conv,
                              void *out, float *final_state, void *final_conv, void *workspace,
                              size_t ws_bytes, void *stream);

/*
 * Segment-parallel prefill: the results of gdn_prefill, with more chains in
 * flight when there are few long sequences.
 *
 * The pages state no chunking; this follows from the recurrence above.  Over
 * a stretch of tokens the state map S_t = exp(g_t) S_{t-1} (I - beta_t k_t
 * k_t^T) + beta_t v_t k_t^T is affine in the state, so the state after a
 * stretch is S_out = S_in M + B: M the product of the tokens' linear parts
 * (per chunk of the tensor-core path, gamma_C I - W^T K~), B the state the
 * stretch leaves from zero.
 * Every sequence is cut into segments of seg_chunks chunks (64 tokens each);
 * one state pass runs, all at once, each sequence's first segment from its
 * initial state (with its outputs), every later segment from a zero state
 * (its B) and every middle segment on the identity (its M); a scan over each
 * sequence's segments, S_in(s + 1) = S_in(s) M_s + B_s, gives every segment's
 * true initial state; a second state pass runs the later segments from those
 * states, with their outputs and the final state.  The fp32 state is the
 * same; the results equal gdn_prefill's up to rounding order (the state
 * operands of the products are rounded to fp16 at different points).
 *
 * seg_chunks  chunks per segment, >= 1.  A sequence of S >= 2 segments takes
 *             3 - 3/S times the state-pass chunk steps of gdn_prefill, in
 *             fewer sequential steps: it pays when N * h_v chains leave most
 *             SMs idle.
 * Supported shapes: the chunked tensor-core shapes of gdn_prefill (bf16,
 * d_k = d_v = 128); others return GDN_ERR_UNSUPPORTED.
 * Every other argument, the workspace (of
 * gdn_prefill_segmented_workspace_bytes(dims, seg_chunks) bytes; the B, M and
 * start-state buffers add 192 KiB per segment and value head) and the errors
 * are those of gdn_prefill, including an in-place final_state.  Returns a
 * gdn_status.
 */
GDN_API size_t gdn_prefill_segmented_workspace_bytes(const gdn_dims *dims, int seg_chunks);
GDN_API int gdn_prefill_segmented(const gdn_dims *dims, const void *q, const void *k, const void *v,
                                  const void *a, const void *b, const void *z, const float *conv_w,
                                  const float *A_log, const float *dt_bias, const float *norm_w,
                                  const int32_t *cu_seqlens, const float *init_state, void *out,
                                  float *final_state, int seg_chunks, void *workspace, size_t ws_bytes,
                                  void *stream);

/*
 * Backward pass of gdn_prefill: the gradient, with respect to every input, of
 * the scalar loss  sum(dy * y) + sum(dfinal_state * final_state).
 *
 * The pages run the layer in training frameworks ("[Qwen3.5 MoE] Add hybrid
 * decoder model (GatedDeltaNet + full attention + MoE)", Summary; "Support
 * Qwen35 SFT"; "feat(models): dense Qwen3.5 custom attention", its E2E
 * training-throughput table) but state no backward; this is the chain rule of
 * the forward definitions above, in fp32 on the CUDA cores (the state's
 * gradient is carried token by token in reverse, each chain's state columns
 * split over CTAs of 32, the states recomputed from a checkpoint every 32
 * tokens).
 *
 * Inputs: dims, the forward's q, k, v, a, b, z, conv_w, A_log, dt_bias,
 *   norm_w, cu_seqlens and init_state (NULL = zeros), exactly as given to
 *   gdn_prefill; dy io_dtype [T, h_v, d_v]; dfinal_state fp32
 *   [N, h_v, d_k, d_v] or NULL (= 0).
 * Outputs (fp32, overwritten): dq, dk [T, h_qk, d_k]; dv, dz [T, h_v, d_v];
 *   da, db [T, h_v]; dconv_w [Cc, 4]; dA_log, ddt_bias [h_v]; dnorm_w [d_v];
 *   dinit_state [N, h_v, d_k, d_v] or NULL (= not returned).  The parameter
 *   gradients are sums over tokens and heads taken with atomic adds, so their
 *   last bits may differ from run to run.
 * workspace: gdn_prefill_backward_workspace_bytes(dims) bytes, 256-byte
 *   aligned, or NULL (stream-ordered allocation, as gdn_prefill).
 * Supported shapes and error behaviour as gdn_prefill (every supported shape
 * and both stream dtypes run this one kernel set).  Returns a gdn_status.
 */
GDN_API size_t gdn_prefill_backward_workspace_bytes(const gdn_dims *dims);
GDN_API int gdn_prefill_backward(const gdn_dims *dims, const void *q, const void *k, const void *v,
                                 const void *a, const void *b, const void *z, const float *conv_w,
                                 const float *A_log, const float *dt_bias, const float *norm_w,
                                 const int32_t *cu_seqlens, const float *init_state, const void *dy,
                                 const float *dfinal_state, float *dq, float *dk, float *dv, float *da, float *db,
                                 float *dz, float *dconv_w, float *dA_log, float *ddt_bias, float *dnorm_w,
                                 float *dinit_state, void *workspace, size_t ws_bytes, void *stream);

/*
 * Decode step: one new token for each of B = dims->num_tokens independent
 * sequences, against a carried state; the state and the conv cache are
 * updated in place.
 *
 * q, k, v, a, b, z  the B new tokens, layouts as above with T = B.
 * conv_state  io_dtype [B, Cc, 3], in/out: the raw (pre-conv) inputs of the
 *             three previous tokens of each sequence, oldest first; after the
 *             call it holds the last three including this token.
 * state       fp32 [B, h_v, d_k, d_v], in/out.
 * out         io_dtype [B, h_v, d_v].
 * Returns a gdn_status.
 */
GDN_API int gdn_decode_step(const gdn_dims *dims, const void *q, const void *k, const void *v,
                    const void *a, const void *b, const void *z, const float *conv_w,
                    const float *A_log, const float *dt_bias, const float *norm_w,
                    void *conv_state, float *state, void *out, void *stream);

/*
 * Prefill -> decode hand-off, for serving (an addition of this library: the
 * pages name varlen prefill and the layer, not a serving interface).
 *
 * gdn_conv_cache_from_prefill: the decode conv cache each sequence of a
 * prefill call leaves behind.  With the prefill's dims (num_tokens = T,
 * num_seqs = N), q, k, v and cu_seqlens, writes conv_cache io_dtype
 * [N, Cc, 3]: per sequence and conv channel (order [q | k | v], as conv_w)
 * the raw inputs of its last three tokens, oldest first, zero where the
 * sequence has fewer than three (the prefill's conv sees zeros before a
 * sequence start).  Together with the prefill's final_state this is exactly
 * what gdn_decode_step continues from.  An invalid cu_seqlens range gives
 * zeros for that sequence.  Returns a gdn_status (GDN_ERR_INVALID_ARG for null
 * pointers or num_seqs < 1).
 *
 * gdn_decode_step_slots: gdn_decode_step over pools of states and conv
 * caches, for paged / batched serving.  Sequence b of the batch reads and
 * updates entry slots[b] (int32, device) of conv_state [num_slots, Cc, 3] and
 * state [num_slots, h_v, d_k, d_v]; B = dims->num_tokens.  The slots of one
 * call must be distinct (two sequences on one entry race).  An entry outside
 * [0, num_slots) leaves every pool untouched, writes zeros to that sequence's
 * out rows and sets *device_status (device int, may be NULL) to
 * GDN_ERR_DEVICE_CHECK.  slots == NULL is gdn_decode_step (entry b).
 */
GDN_API int gdn_conv_cache_from_prefill(const gdn_dims *dims, const void *q, const void *k, const void *v,
                                        const int32_t *cu_seqlens, void *conv_cache, void *stream);
GDN_API int gdn_decode_step_slots(const gdn_dims *dims, const void *q, const void *k, const void *v,
                                  const void *a, const void *b, const void *z, const float *conv_w,
                                  const float *A_log, const float *dt_bias, const float *norm_w,
                                  void *conv_state, float *state, const int32_t *slots, int num_slots,
                                  void *out, int *device_status, void *stream);

/*
 * Read and clear the device status word of a prefill workspace.  Enqueued on
 * `stream` and waits for it (the one synchronising call of the library).
 * Writes GDN_OK, GDN_ERR_DEVICE_CHECK or GDN_ERR_TIMEOUT to *device_status
 * and returns GDN_OK, or returns GDN_ERR_INVALID_ARG / GDN_ERR_CUDA.
 */
GDN_API int gdn_workspace_status(void *workspace, void *stream, int *device_status);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot allocate.
 *
 * (An addition of this library; the pages have no counterpart.)
 *
 * Some callers cannot call cudaMalloc or hand out a workspace: an inference
 * engine whose memory planner owns all of HBM from start-up, a serving loop
 * that forbids allocation after warm-up (an allocation there can stall on the
 * driver or fail under memory pressure), or code running inside another
 * allocator's callback, where allocating would re-enter it.  This entry point
 * is gdn_prefill with the workspace taken from a fixed array of
 * GDN_NOALLOC_SCRATCH_BYTES in the library's own device memory; it calls no
 * cudaMalloc, cudaMallocAsync, cudaFree or other allocating routine.  The
 * caller still passes every input and output, with the meaning, layout and
 * error behaviour of gdn_prefill.
 *
 *  - Limit: problems whose gdn_prefill_workspace_bytes() exceeds
 *    GDN_NOALLOC_SCRATCH_BYTES are rejected with GDN_ERR_WORKSPACE before
 *    anything is launched.
 *  - The array is a device global of the library: every GPU that loads the
 *    library holds it until the process exits.  The first call on a device
 *    looks up its device address (cudaGetSymbolAddress, on the current
 *    device) and keeps it for later calls; make that first call before any
 *    stream capture.  A cudaDeviceReset() of that device invalidates the kept
 *    address (the reset context reloads the library's module elsewhere): a
 *    process that resets a device must not call this entry point on it again.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; each call clears the part that must start at zero.  Calls whose
 *    kernels overlap on the GPU (different streams, or different host threads
 *    without ordering) race on it: order them on one stream or serialise them.
 *  - The device status word of this entry point is not readable by the caller
 *    (gdn_workspace_status needs a caller-owned workspace).
 */
#define GDN_NOALLOC_SCRATCH_BYTES (8u << 20)
GDN_API int gdn_prefill_noalloc(const gdn_dims *dims, const void *q, const void *k, const void *v,
                                const void *a, const void *b, const void *z, const float *conv_w,
                                const float *A_log, const float *dt_bias, const float *norm_w,
                                const int32_t *cu_seqlens, const float *init_state, void *out,
                                float *final_state, void *stream);

/* Human-readable name of a gdn_status (never NULL). */
GDN_API const char *gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */

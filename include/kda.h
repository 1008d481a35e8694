/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) implementation of the Kimi
 * Delta Attention (KDA) recurrence.
 *
 * The operation ("Kimi (AI)", Wikipedia mirror, section "Kimi Delta
 * Attention (KDA)": the forget gating / predict / memory updating block, with
 * the output o_t = S_t q_t of the naive linear attention line before it):
 *
 *     S~_t = diag(alpha_t) S_{t-1}
 *     v~_t = S~_t k_t
 *     S_t  = S~_t + beta_t (v_t - v~_t) k_t^T
 *     o_t  = S_t q_t
 *
 * per (sequence, head).  S is d_v x d_k (a sum of v k^T outer products), so
 * alpha_t has d_v entries and scales the rows of S (value channels); beta_t
 * is one scalar per token and head.  No scale or normalisation is applied to
 * q or k and there is no output gate: the page has none.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Memory: every tensor argument is a DEVICE pointer owned by the caller.
 *   The library never allocates device memory, never frees caller memory and
 *   keeps no state between calls except a per-device cache of the SM count
 *   and the driver's tensor-map encoder entry point.
 * - Layouts are dense, row-major, last index fastest, no padding:
 *     q, k   [T][H][d_k]      v, o   [T][H][d_v]      (dtype: KDA_BF16 or KDA_FP32)
 *     alpha  [T][H][d_v] fp32, each in (0, 1]         beta   [T][H] fp32
 *     state  [N][H][d_v][d_k] fp32
 *   Every pointer must be 16-byte aligned.
 * - Stream: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  No call synchronises the host except
 *   kda_prefill_device_status, which says so.
 * - Errors: argument errors are returned synchronously and enqueue nothing.
 *   A failed kernel launch returns KDA_ERR_CUDA.  Errors that depend on device
 *   data are detected on the device and reported by kda_prefill_device_status:
 *   a malformed cu_seqlens (the kernels then write no output), or a decay too
 *   fast for the chunk form (see kda_prefill).
 *   No C++ exception crosses this interface.
 * - Alias rules: outputs must not overlap inputs, except that S_T may equal
 *   S0 exactly (in-place state update).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment, bad alias */
    KDA_ERR_UNSUPPORTED = 2,   /* sizes outside what the kernels implement (see each call) */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
    KDA_ERR_DEVICE_INPUT = 4,  /* device data invalid: cu_seqlens not 0-based, decreasing or past T */
    KDA_ERR_DEVICE_TIMEOUT = 5, /* a device-side wait hit its time limit; outputs are incomplete */
    KDA_ERR_DEVICE_RANGE = 6   /* device data outside the chunk form's range: alpha decays by more
                                  than a factor 1e30 within 16 tokens of one channel */
} kda_status;

typedef enum {
    KDA_BF16 = 0,   /* q, k, v, o stored as bfloat16 */
    KDA_FP32 = 1    /* q, k, v, o stored as float32 */
} kda_dtype;

/* Which prefill kernel runs.  AUTO picks the tensor-core kernel whenever the
 * shape qualifies (dtype KDA_BF16, d_k == 128, d_v a multiple of 128,
 * chunk == 64) and the portable chunk kernel otherwise; with the tensor-core
 * kernel it also splits the sequence axis (below) when the batch has fewer
 * (sequence, head, 128-channel block) chains than a third of the SMs, the
 * sequences average at least 2048 tokens per segment, and the workspace has
 * room for it. */
typedef enum {
    KDA_KERNEL_AUTO = 0,
    KDA_KERNEL_CHUNK_SIMT = 1,   /* fp32 CUDA-core chunk kernel: any supported shape */
    KDA_KERNEL_CHUNK_TC = 2,     /* tcgen05 / TMEM / TMA chunk kernel */
    /* the tensor-core kernel with the sequence axis split into M >= 2
     * segments of whole chunks: one pass runs segment 0 of every sequence
     * from S0 and, for segments 1..M-1, the segment from a zero state (its
     * output, final state and product of alpha) and its transition
     * prod (I - beta k k^T) applied to each token's q; a scan chains these
     * affine maps into each segment's initial state and S_T; a correction
     * adds each later segment's initial-state share to its output where it
     * can change the stored value.  Same results as KDA_KERNEL_CHUNK_TC up
     * to rounding.  Only for batches with few chains (those for which
     * kda_prefill_workspace_size_tokens exceeds kda_prefill_workspace_size),
     * whatever the sequence lengths. */
    KDA_KERNEL_CHUNK_TC_SPLIT = 3
} kda_prefill_kernel;

typedef void* kda_stream_t;   /* a cudaStream_t */

/* Layout of the forget gate for kda_prefill_gates. */
typedef enum {
    KDA_GATE_CHANNEL_F32 = 0,   /* alpha [T][H][d_v] fp32 in (0, 1] (kda_prefill's) */
    KDA_GATE_HEAD_F32 = 1,      /* alpha [T][H] fp32 in (0, 1]: one gate per token and
                                   head, the same for every value channel (the scalar
                                   gate of Gated DeltaNet) */
    KDA_GATE_CHANNEL_LOG_BF16 = 2   /* log alpha [T][H][d_v] bfloat16, <= 0: half the
                                       bytes of the fp32 gate */
} kda_gate_format;

/*
 * Bytes of device workspace kda_prefill needs for `num_seqs` sequences of H
 * heads with these sizes, without the sequence-axis split.  Returns 0 for
 * num_seqs < 0.  The workspace holds the varlen schedule (sequence order,
 * work counter, device error word) and a bitmap of the channels the
 * tensor-core kernel hands to the portable one (16 bytes per (sequence,
 * head, 128-channel block); see "Fast decay" at kda_prefill).  A smaller
 * workspace of at least the schedule's size is accepted; it reports
 * fast-decaying channels instead of recomputing them.  Its contents need no
 * initialisation and are overwritten by every call.
 */
size_t kda_prefill_workspace_size(int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                  int32_t chunk);

/*
 * kda_prefill_workspace_size for a batch of `total_tokens` tokens, with room
 * for the sequence-axis split where the kernel choice may take it (batches
 * with few (sequence, head, 128-channel block) chains on the current
 * device): its buffers, in the bitmap's place, hold each segment's states,
 * fp32 q-transforms of every token (total_tokens x H x d_k x 4 bytes) and
 * the zero-start outputs of later segments in fp32 (total_tokens x H x d_v x 4
 * bytes) and per-chunk decay factors (about total_tokens / 64 x H x d_v x 4 bytes).
 * Returns 0 for num_seqs < 0 or total_tokens < 0.  With a workspace of
 * kda_prefill_workspace_size bytes the split is not taken.
 */
size_t kda_prefill_workspace_size_tokens(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                         int32_t d_k, int32_t d_v, int32_t chunk);

/*
 * Chunkwise-parallel prefill over a packed (varlen) batch.  Runs the
 * recurrence above for every sequence n (tokens cu_seqlens[n] ..
 * cu_seqlens[n+1]-1) and head h, starting from S0[n][h] (zeros when S0 is
 * NULL); writes o for every token of every sequence and the final state S_T.
 * A zero-length sequence gives S_T[n] = S0[n] (zeros when S0 is NULL).
 * Tokens at or beyond cu_seqlens[num_seqs] are not read and their o is not
 * written.
 *
 *   q, k, v, alpha, beta  inputs, layouts above, T = total_tokens
 *   S0                    [N][H][d_v][d_k] fp32 or NULL
 *   cu_seqlens            device int32 [num_seqs+1]: cu[0] == 0,
 *                         non-decreasing, cu[num_seqs] <= total_tokens
 *                         (checked on the device -> KDA_ERR_DEVICE_INPUT)
 *   dtype                 storage type of q, k, v and o
 *   chunk                 tokens per chunk: 16, 32 or 64
 *   o                     output [T][H][d_v] (dtype)
 *   S_T                   output [N][H][d_v][d_k] fp32; may equal S0; may be
 *                         NULL only when num_seqs == 0
 *   workspace             device memory of kda_prefill_workspace_size_tokens
 *                         bytes (kda_prefill_workspace_size: no
 *                         sequence-axis split), 16-byte aligned; must not be
 *                         shared by calls that may run concurrently
 *
 * Supported: 1 <= H, 16 <= d_k <= 128 and d_k % 16 == 0, 1 <= d_v <= 1024
 * and d_v % 16 == 0, alpha in (0, 1].
 * num_seqs == 0 or total_tokens == 0 is a valid no-op apart from S_T = S0.
 *
 * Fast decay.  The chunk form divides by the running product of alpha within
 * a chunk, so it needs that product to stay above 1e-30.  The tensor-core
 * kernel hands every channel whose product over one of its 64-token chunks
 * falls below that to the portable kernel, which runs the channel again from
 * S0 (its S_T is left unwritten until then, so an in-place S0 survives) and
 * takes such chunks 16 tokens at a time.  This needs the workspace size
 * kda_prefill_workspace_size returns; with a smaller workspace, or when the
 * sequence axis is split, such a channel is reported instead.  A channel
 * whose alpha multiplies to less than 1e-30 over 16 tokens (a decay of more
 * than a factor 1e30 in 16 steps) is beyond the chunk form:
 * kda_prefill_device_status then returns KDA_ERR_DEVICE_RANGE, and o and S_T
 * of that sequence and head are not valid (all others are).
 */
kda_status kda_prefill(const void* q, const void* k, const void* v,
                       const float* alpha, const float* beta, const float* S0,
                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype, int32_t chunk,
                       void* o, float* S_T, void* workspace, size_t workspace_bytes,
                       kda_stream_t stream);

/* kda_prefill with an explicit kernel choice (for testing the kernels on one
 * shape).  Requesting KDA_KERNEL_CHUNK_TC or KDA_KERNEL_CHUNK_TC_SPLIT for a
 * shape the tensor-core kernel does not cover returns KDA_ERR_UNSUPPORTED;
 * KDA_KERNEL_CHUNK_TC_SPLIT with a workspace smaller than
 * kda_prefill_workspace_size_tokens returns KDA_ERR_INVALID_ARG. */
kda_status kda_prefill_ex(const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta, const float* S0,
                          const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype, int32_t chunk,
                          void* o, float* S_T, void* workspace, size_t workspace_bytes,
                          kda_prefill_kernel kernel, kda_stream_t stream);

/*
 * kda_prefill_ex with the forget gate in another layout (kda_gate_format):
 * `alpha` points to the gate in that layout; everything else as kda_prefill_ex.
 * The recurrence is the same with alpha_t[r] = alpha[t][h] (KDA_GATE_HEAD_F32)
 * or exp(log_alpha[t][h][r]) (KDA_GATE_CHANNEL_LOG_BF16).  Every shape
 * kda_prefill_ex supports; the sequence-axis split is not used with the two
 * new layouts (KDA_KERNEL_CHUNK_TC_SPLIT returns KDA_ERR_UNSUPPORTED).
 * KDA_GATE_CHANNEL_F32 is exactly kda_prefill_ex.
 */
kda_status kda_prefill_gates(const void* q, const void* k, const void* v, const void* alpha,
                             kda_gate_format gate_format, const float* beta, const float* S0,
                             const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                             int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                             int32_t chunk, void* o, float* S_T, void* workspace,
                             size_t workspace_bytes, kda_prefill_kernel kernel,
                             kda_stream_t stream);

/*
 * Whether `kernel` covers a prefill of this shape: KDA_OK if kda_prefill_ex
 * would accept it, KDA_ERR_UNSUPPORTED if not, KDA_ERR_INVALID_ARG for an
 * unknown enum value.  Host only; makes no CUDA call.
 */
kda_status kda_prefill_supported(kda_prefill_kernel kernel, int32_t H, int32_t d_k, int32_t d_v,
                                 kda_dtype dtype, int32_t chunk);

/*
 * Blocks until `stream` has finished the work enqueued so far, then returns
 * the device-side status a kda_prefill call on `workspace` recorded
 * (KDA_OK, KDA_ERR_DEVICE_INPUT, KDA_ERR_DEVICE_TIMEOUT or
 * KDA_ERR_DEVICE_RANGE), or KDA_ERR_CUDA if the copy fails.
 * This is the only call that synchronises the host.
 */
kda_status kda_prefill_device_status(const void* workspace, kda_stream_t stream);

/*
 * One step of the exchange that splits the sequence axis across devices (or
 * across calls).  Over a segment of tokens the recurrence is affine in the
 * state it starts from: S_end = diag(g) S_start P + R, with g the product of
 * alpha over the segment (per value channel), P the product of the segment's
 * (I - beta_t k_t k_t^T) factors in token order (d_k x d_k; the two commute
 * with the decay, which acts on the rows) and R the state the segment
 * reaches from zero ("Kimi (AI)", section "Kimi Delta Attention (KDA)": the
 * forget gating and memory updating lines, composed over the segment).  This
 * call applies such maps:
 *
 *     S_out[n][h] = diag(g[n][h]) S_in[n][h] P[n][h] + R[n][h]
 *
 *   S_in, R, S_out   [N][H][d_v][d_k] fp32; S_out may equal S_in
 *   g                [N][H][d_v] fp32
 *   P                [N][H][d_k][d_k] fp32
 *
 * kda_prefill itself gives each part of a segment's map: R is its S_T from
 * S0 = NULL; P is its S_T with v = 0, alpha = 1 and S0 = the identity (d_v =
 * d_k); g is any column of its S_T with k = 0 and S0 = all ones.  Supported:
 * d_k <= 128; arithmetic in fp32.
 */
kda_status kda_segment_combine(const float* S_in, const float* g, const float* P, const float* R,
                               int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                               float* S_out, kda_stream_t stream);

/*
 * Runs the device-side timeout path of the prefill kernels, so that a user can
 * see it work on their GPU.  Every wait inside the tensor-core prefill is
 * bounded: when one runs out, its warp records KDA_ERR_DEVICE_TIMEOUT in the
 * workspace and raises a flag that stops the CTA's other warps at their next
 * wait; each warp waits (bounded) for the copies and MMAs it issued, the CTA
 * frees its tensor memory and exits, and the context stays usable.  This call
 * enqueues one CTA that allocates tensor memory as the prefill kernel does,
 * waits with the limit `timeout_ns` on a barrier that nothing arrives on, and
 * on a second one with the prefill's own limit (2 s) until the flag stops it.
 * Afterwards kda_prefill_device_status(workspace) returns
 * KDA_ERR_DEVICE_TIMEOUT.  The pages have no counterpart to this call.
 *
 *   workspace   device memory of at least kda_prefill_workspace_size(0, ...)
 *               bytes, 16-byte aligned; its status word is overwritten
 *   timeout_ns  1e3 .. 1e9 (otherwise KDA_ERR_INVALID_ARG)
 */
kda_status kda_check_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t timeout_ns,
                                  kda_stream_t stream);

/* Largest num_seqs that kda_prefill_noalloc accepts. */
#define KDA_NOALLOC_MAX_SEQS 65536

/*
 * kda_prefill without a workspace argument.  The pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory: code
 * that runs inside a host program which owns every device allocation and
 * gives its extensions no scratch buffer, or serving code that must not
 * allocate once it is running, where an allocation can stall the device or
 * break a memory plan fixed in advance.
 *
 * Same arguments and results as kda_prefill, minus the workspace, except
 * that this call never splits the sequence axis (its scratch has no room for
 * the segment buffers): a batch with few long chains, such as one sequence
 * of 128K tokens with 32 heads, runs slower here than through kda_prefill
 * with a full workspace.  The scratch it needs lives in a device array built
 * into the library (about 768 KB on every GPU that loads it, held until the
 * process exits).  Every call looks up that array's address in the CUDA
 * context current at the call (cudaGetSymbolAddress, which allocates
 * nothing), so switching driver contexts or resetting the device between
 * calls is safe.  The first call in a context loads the library's device
 * code there; make that first call before any stream capture.  The call
 * itself allocates nothing.
 *
 * Every call shares the one array and leaves its contents behind; each call
 * clears what it needs cleared, but calls that overlap on the GPU (issued on
 * different streams with no ordering between them) race on it and must not
 * be made.  num_seqs > KDA_NOALLOC_MAX_SEQS returns KDA_ERR_UNSUPPORTED.
 * Channels whose decay is too fast for the tensor-core kernel's one-pass
 * chunks are redone by the portable kernel for batches of up to 16384
 * (sequence, head, 128-channel block) units; larger batches report such
 * channels as KDA_ERR_DEVICE_RANGE instead.
 * Device-detected input errors leave the outputs unwritten; they cannot be
 * queried afterwards, because kda_prefill_device_status needs a workspace.
 */
kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v,
                               const float* alpha, const float* beta, const float* S0,
                               const int32_t* cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                               kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                               kda_stream_t stream);

/*
 * One decode step for B sequences with one new token each, state updated in
 * place: for every (b, h), S[b][h] <- S_1 and o[b][h] <- S_1 q for the single
 * token (q[b][h], k[b][h], v[b][h], alpha[b][h], beta[b][h]).
 *
 *   q, k   [B][H][d_k] (dtype)     v, o  [B][H][d_v] (dtype)
 *   alpha  [B][H][d_v] fp32        beta  [B][H] fp32
 *   S      [B][H][d_v][d_k] fp32, read and overwritten
 *
 * Supported: d_k in {16, 32, 64, 128, 256}; 1 <= d_v <= 4096; B, H >= 1
 * (B == 0 is a valid no-op).
 */
kda_status kda_decode_step(const void* q, const void* k, const void* v,
                           const float* alpha, const float* beta, float* S,
                           int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                           void* o, kda_stream_t stream);

/* kda_decode_step with the forget gate in another layout (kda_gate_format):
 * alpha [B][H] fp32 (KDA_GATE_HEAD_F32) or log alpha [B][H][d_v] bf16
 * (KDA_GATE_CHANNEL_LOG_BF16); every shape kda_decode_step supports. */
kda_status kda_decode_step_gates(const void* q, const void* k, const void* v,
                                 const void* alpha, kda_gate_format gate_format,
                                 const float* beta, float* S, int32_t B, int32_t H,
                                 int32_t d_k, int32_t d_v, kda_dtype dtype, void* o,
                                 kda_stream_t stream);

/*
 * Bytes of device workspace kda_backward needs, or 0 for a shape it does not
 * support: for d_k = 128, about (total_tokens / 64 + num_seqs) x H x d_v x 768
 * bytes of per-chunk states and triangular factors, plus
 * 2 x d_v / 64 x total_tokens x H x d_k x 4 bytes of per-block partial sums.
 * Contents need no initialisation.
 */
size_t kda_backward_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                   int32_t d_k, int32_t d_v, int32_t chunk);

/*
 * Backward pass of kda_prefill: given dO = dL/do and dS_T = dL/dS_T for some
 * loss L of the outputs of kda_prefill on the same inputs, writes the
 * gradients of L with respect to every input.  The chain rule is taken
 * through the chunkwise form of the recurrence ("Kimi (AI)", section "Kimi
 * Delta Attention (KDA)": the three-line update and o_t = S_t q_t).  The
 * forward pass is recomputed inside the call: no state from kda_prefill is
 * needed.
 *
 *   q, k, v, alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k,
 *   d_v, dtype, chunk     as for kda_prefill (channel fp32 gate)
 *   d_o                   [T][H][d_v] (dtype): dL/do
 *   dS_T                  [N][H][d_v][d_k] fp32 or NULL (zeros): dL/dS_T
 *   dq, dk                outputs [T][H][d_k] fp32
 *   dv, dalpha            outputs [T][H][d_v] fp32
 *   dbeta                 output [T][H] fp32
 *   dS0                   output [N][H][d_v][d_k] fp32, or NULL (not written);
 *                         dL/dS0 (the gradient reaching S0 even when S0 is NULL)
 *   workspace             kda_backward_workspace_size bytes, 16-byte aligned,
 *                         not shared with calls that may run concurrently
 *
 * Gradients of tokens at or past cu_seqlens[num_seqs] are not written.  No
 * output may overlap an input or another output.  kda_prefill_device_status
 * on the same workspace reports device-detected input errors, which leave
 * every output unwritten.  The result is deterministic (no atomics).
 *
 * Supported: dtype KDA_BF16, d_k == 128, d_v a multiple of 64 up to 1024,
 * chunk == 64; alpha in (0, 1] with every product of alpha over one 64-token
 * chunk of one channel >= 1e-30 (the chunkwise reverse mode divides by it and
 * has no 16-token fallback; for d_v a multiple of 128 a chunk below it is
 * reported as KDA_ERR_DEVICE_RANGE).  Arithmetic is fp32.
 */
kda_status kda_backward(const void* q, const void* k, const void* v, const float* alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens,
                        int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype dtype, int32_t chunk, const void* d_o,
                        const float* dS_T, float* dq, float* dk, float* dv, float* dalpha,
                        float* dbeta, float* dS0, void* workspace, size_t workspace_bytes,
                        kda_stream_t stream);

/* Workspace for kda_backward_gates: kda_backward_workspace_size plus, for the
 * two non-channel layouts, 2 x total_tokens x H x d_v x 4 bytes (the gate per
 * channel and its gradient).  0 for an unsupported shape or layout. */
size_t kda_backward_gates_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t H,
                                         int32_t d_k, int32_t d_v, int32_t chunk,
                                         kda_gate_format gate_format);

/*
 * kda_backward with the forget gate in another layout (kda_gate_format), as
 * kda_prefill_gates takes it.  `dgate` is the gradient with respect to the
 * gate in its own layout, fp32: [T][H] for KDA_GATE_HEAD_F32 (the sum of the
 * per-channel gradients: one gate drives every channel of the head),
 * [T][H][d_v] with respect to log alpha for KDA_GATE_CHANNEL_LOG_BF16
 * (alpha times the per-channel gradient).  Everything else as kda_backward;
 * KDA_GATE_CHANNEL_F32 is exactly kda_backward.
 */
kda_status kda_backward_gates(const void* q, const void* k, const void* v, const void* alpha,
                              kda_gate_format gate_format, const float* beta, const float* S0,
                              const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                              int32_t chunk, const void* d_o, const float* dS_T, float* dq,
                              float* dk, float* dv, float* dgate, float* dbeta, float* dS0,
                              void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * The additive update of linear attention instead of the delta rule: the
 * predict step is dropped, so S_t = diag(alpha_t) S_{t-1} + beta_t v_t k_t^T
 * and o_t = S_t q_t.  With alpha = beta = 1 this is the page's naive linear
 * attention, S_t = S_{t-1} + v_t k_t^T, o_t = (sum_{i<=t} v_i k_i^T) q_t
 * ("Kimi (AI)", section "Kimi Delta Attention (KDA)", the line before the
 * three-line update).  Arguments, layouts and rules as kda_prefill_ex with the
 * per-channel fp32 gate; the chunk form is the delta rule's with the K S^T
 * term dropped and T = I.  Both chunk kernels take it (the tensor-core one for
 * the shapes it covers); KDA_KERNEL_CHUNK_TC_SPLIT returns KDA_ERR_UNSUPPORTED.
 */
kda_status kda_prefill_additive(const void* q, const void* k, const void* v, const float* alpha,
                                const float* beta, const float* S0, const int32_t* cu_seqlens,
                                int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                                int32_t d_v, kda_dtype dtype, int32_t chunk, void* o, float* S_T,
                                void* workspace, size_t workspace_bytes,
                                kda_prefill_kernel kernel, kda_stream_t stream);

/* One decode step of the additive update (kda_prefill_additive's recurrence):
 * arguments and shapes as kda_decode_step. */
kda_status kda_decode_step_additive(const void* q, const void* k, const void* v,
                                    const float* alpha, const float* beta, float* S, int32_t B,
                                    int32_t H, int32_t d_k, int32_t d_v, kda_dtype dtype,
                                    void* o, kda_stream_t stream);

/* Static description of a status code.  Never NULL. */
const char* kda_status_string(kda_status s);

/* Library ABI version, (major << 16) | minor. */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

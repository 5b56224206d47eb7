/*
 * kda.h -- C ABI of the GB300 Kimi Delta Attention (KDA) library (libkda_gb300.so).
 *
 * The operation (page "Kimi K3 im Detail", flozi.net, section "Sequenz-Mixing: KDA-Zustand
 * und globale MLA"): each KDA head keeps a recurrent matrix S in R^{d_k x d_v}.  For every
 * token t the old state is attenuated channel-wise by a retention vector, a scalar write gate
 * beta_t applies a delta-rule correction, and the query reads S_t^T q_t after that update:
 *
 *     S'  = diag(exp(clamp(g_t, -5, 0))) S_{t-1}          (decay over the key channels)
 *     S_t = S' + beta_t k_t (v_t - S'^T k_t)^T            (delta-rule write)
 *     o_t = S_t^T q_t                                     (read includes the current token)
 *
 * The floor -5 on the log-decay is the published bound of the same section; over a 16-token
 * tile the cumulative log-decay therefore stays >= -80, which keeps every exponential factor
 * of the chunked prefill inside the fp32/bf16 range.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller (the staged calls also take
 *     host buffers); the library allocates no memory and keeps no per-call state.  A compute
 *     call only validates its host-side arguments and enqueues kernels on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) of the current device, without
 *     synchronizing.  The exceptions are documented at their entry points: kda_device_status
 *     synchronizes `stream`, and the staged calls create two streams and four events per device
 *     on first use (the no-scratch variant one more event) and keep them.  Calls are
 *     thread-safe.
 *   - Layouts are row-major with the last index contiguous:
 *       q, k, g : [T_total, H, d_k]     v, out : [T_total, H, d_v]     beta : [T_total, H]
 *       states  : [N, H, d_k, d_v] fp32, S[i][j] with i = key channel, j = value channel.
 *   - `dtype` (kda_dtype) is the element type of q, k, v, g and beta; `out_dtype` that of out
 *     (fp32, the accumulation precision, or bf16).  States and checkpoints are always fp32 and
 *     all accumulation is fp32.  Rounding outputs to bf16 costs up to 2^-9 of the largest |o|,
 *     which on the synthetic workloads is ~3.5e-2 of RMS(o): fp32 outputs are the precise form.
 *   - Every pointer passed must be 16-byte aligned.
 *   - Return value: KDA_OK (0) or a kda_status code; nothing is enqueued on error.  Checks that
 *     need device data (monotone cu_seqlens, finite inputs) are not made.  A bounded device
 *     wait that expires, or a state index out of range, sets a sticky per-device error word
 *     that kda_device_status() reads.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad dtype or stride       */
    KDA_ERR_UNSUPPORTED_SHAPE = 2, /* head dimensions the kernels do not implement            */
    KDA_ERR_MISALIGNED = 3,        /* a pointer not 16-byte aligned                           */
    KDA_ERR_CUDA = 4,              /* a CUDA runtime call or kernel launch failed             */
    KDA_ERR_DEVICE_TIMEOUT = 5,    /* a bounded device-side wait expired (device error word)  */
    KDA_ERR_INDEX_RANGE = 6,       /* kda_state_copy met an index outside its slot range      */
    KDA_ERR_DEVICE_BOUNDS = 7      /* a device-side bounds check failed (library built with
                                      -DKDA_DEBUG, or kda_diag_bounds_check)                    */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/* ABI revision of this header; bumped on any incompatible change. */
#define KDA_ABI_VERSION 2
int kda_abi_version(void);

/* Human-readable name of a kda_status value (static storage, never NULL). */
const char *kda_status_string(int status);

/*
 * kda_prefill -- varlen chunked prefill.
 *
 * Defined by the section cited above: the tokens of a chunk are processed in parallel and the
 * recurrent state is handed from chunk to chunk (second paragraph); the prefix-reuse paragraph
 * (fourth paragraph) stores KDA states only at sparse checkpoints.
 *
 *   q, k, g, v, beta  inputs, layouts above, `dtype` elements.  May be NULL iff total_tokens==0.
 *   cu_seqlens        device int32 [n_seqs+1], cu_seqlens[0] = 0, non-decreasing,
 *                     cu_seqlens[n_seqs] = total_tokens.  Sequence n owns tokens
 *                     [cu_seqlens[n], cu_seqlens[n+1]); empty sequences are allowed.
 *                     May be NULL when n_seqs == 1 (one sequence of total_tokens).
 *   n_seqs, total_tokens, n_heads, d_k, d_v   sizes (n_seqs >= 0, total_tokens >= 0).
 *   init_state        fp32 [n_seqs, H, d_k, d_v] state before each sequence, or NULL = zeros.
 *                     May alias final_state (in-place resume).
 *   out               [total_tokens, H, d_v] outputs o_t, `out_dtype`.  Must not alias an input.
 *   final_state       fp32 [n_seqs, H, d_k, d_v] state after each sequence, or NULL.
 *   ckpt_stride       0 (no checkpoints) or a positive multiple of 32 (the tensor-core kernel
 *                     advances the state 32 tokens a step).  Sequence n of length
 *                     L_n emits floor(L_n / ckpt_stride) checkpoints: the state after its first
 *                     m*ckpt_stride tokens, m = 1..floor(L_n / ckpt_stride).
 *   ckpts             fp32 [sum_n floor(L_n / ckpt_stride), H, d_k, d_v]; slots are ordered by
 *                     sequence, then by position.  Required iff ckpt_stride > 0.
 *   stream            cudaStream_t to enqueue on.
 *
 * Supported head sizes: d_k = d_v = 128 for bf16 inputs (tensor-core chunked kernel); for fp32
 * inputs, and for bf16 inputs with other sizes, 1 <= d_k <= 128 and d_v a multiple of 32 up to 256 (per-token
 * CUDA-core kernel).  Errors: KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED_SHAPE,
 * KDA_ERR_MISALIGNED, KDA_ERR_CUDA.
 *
 * Value range of the tensor-core kernel: the state stays fp32, but the state products take the
 * new values V - K~S0 and a copy of the state as fp16 operands (full precision from 6.1e-5 to
 * 65504).  With q and k of unit norm and beta in [0, 1], v and init_state scaled by powers of two
 * from 2^-12 to 2^13 of unit variance (|v| up to about 4e4) keep the bf16-input bounds (outputs
 * 2e-2, states 1e-2 of RMS); at 2^14 (|v| ~ 8e4) the fp16 operands overflow and the outputs are not
 * finite, and at 2^-16 the fp16 subnormal range costs accuracy (outputs ~4e-2 of RMS).  Scale v
 * into that range (the recurrence is linear in v and the state) or use kda_prefill_recurrent,
 * which keeps every product in fp32.
 */
int kda_prefill(const void *q, const void *k, const void *v, const void *g, const void *beta,
                const int32_t *cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t n_heads,
                int32_t d_k, int32_t d_v, int32_t dtype, int32_t out_dtype, const float *init_state,
                void *out, float *final_state, int32_t ckpt_stride, float *ckpts, void *stream);

/*
 * kda_prefill_precise -- the same operation, arguments and errors as kda_prefill, with a smaller
 * output error on the tensor-core path (bf16 inputs, d_k = d_v = 128) at a higher cost.  The
 * largest rounding in kda_prefill's outputs is that of Aqk (the q.k products of a step, masked
 * lower-triangular) to fp16, the A operand of the product P = Aqk Bt.  Here Aqk is carried as
 * fp16(Aqk) plus its fp16 low part through two accumulating products, and P is rounded once.
 * On the T = 8192, 96-head workload this takes the largest output error from 1.6-1.7e-2 to
 * 0.9-1.1e-2 of RMS (three input draws) for about 1.09x the time; final states and checkpoints are
 * bit-identical to kda_prefill's.  Other dtypes and shapes run the per-token path, as in kda_prefill.  Same value range
 * as kda_prefill.
 */
int kda_prefill_precise(const void *q, const void *k, const void *v, const void *g,
                        const void *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                        int64_t total_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                        int32_t dtype, int32_t out_dtype, const float *init_state, void *out,
                        float *final_state, int32_t ckpt_stride, float *ckpts, void *stream);

/*
 * kda_prefill_recurrent -- the same operation and arguments as kda_prefill, always evaluated
 * token by token on CUDA cores (fp32 state in registers).  It is the path kda_prefill takes
 * for fp32 inputs; for bf16 it is a slower second evaluation used to cross-check the
 * tensor-core kernel.  Same errors as kda_prefill.
 */
int kda_prefill_recurrent(const void *q, const void *k, const void *v, const void *g,
                          const void *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                          int64_t total_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                          int32_t dtype, int32_t out_dtype, const float *init_state, void *out,
                          float *final_state, int32_t ckpt_stride, float *ckpts, void *stream);

/* Which kernel kda_prefill runs for these sizes: 1 = tensor-core chunked, 0 = per-token
 * CUDA-core, negative = a kda_status (unsupported / invalid). */
int kda_prefill_path(int32_t d_k, int32_t d_v, int32_t dtype);


/*
 * kda_decode -- one new token per sequence, state updated in place.
 *
 * The recurrence above at T = 1 (same section: the state has a fixed size and replaces a
 * per-token KV cache, so generating a token is one update of S).
 *
 *   q, k, g : [n_seqs, H, d_k]   v : [n_seqs, H, d_v]   beta : [n_seqs, H]   (`dtype`)
 *   state   : fp32 [n_seqs, H, d_k, d_v], read and overwritten in place with S_t.
 *   out     : [n_seqs, H, d_v] `out_dtype`, o_t = S_t^T q_t.
 * Supported: 1 <= d_k <= 128, d_v a multiple of 4 up to 128.  Errors as kda_prefill.
 */
int kda_decode(const void *q, const void *k, const void *v, const void *g, const void *beta,
               float *state, void *out, int32_t n_seqs, int32_t n_heads, int32_t d_k, int32_t d_v,
               int32_t dtype, int32_t out_dtype, void *stream);

/*
 * kda_state_copy -- copy whole per-sequence states (H x d_k x d_v fp32 each) between slot
 * arrays: dst[dst_idx[i]] = src[src_idx[i]] for i in [0, n).  This is the restore step of
 * prefix reuse (section cited above, fourth paragraph: a reused prefix restarts from a stored
 * KDA state at the same token boundary).
 *
 *   dst, src         fp32 slot arrays [n_dst_slots, H, d_k, d_v] and [n_src_slots, ...];
 *                    they may be the same array but copied slots must not overlap.
 *   dst_idx, src_idx device int64 [n] slot indices, or NULL for the identity i.
 *   An index outside [0, n_*_slots) skips that copy and sets the device error word to
 *   KDA_ERR_INDEX_RANGE.  Errors: KDA_ERR_INVALID_ARG, KDA_ERR_MISALIGNED, KDA_ERR_CUDA.
 */
int kda_state_copy(float *dst, const int64_t *dst_idx, int64_t n_dst_slots, const float *src,
                   const int64_t *src_idx, int64_t n_src_slots, int64_t n, int32_t n_heads,
                   int32_t d_k, int32_t d_v, void *stream);

/*
 * kda_premix -- the pre-mixer: the recurrence's inputs q, k, v, g, beta from the KDA projections.
 *
 * The section cited above gives the KDA projections a short convolution of width 4 (first
 * paragraph) and no formula; this call implements the plain reading, with q/k normalisation and
 * the gate functions of the recurrence's input range:
 *     y_t[c] = w[c][0] x_(t-3)[c] + w[c][1] x_(t-2)[c] + w[c][2] x_(t-1)[c] + w[c][3] x_t[c]
 *              (causal, depthwise, no activation; per tensor x in {xq, xk, xv})
 *     q_t = y^q_t / max(||y^q_t||_2, eps),  k_t likewise (per token and head),  v_t = y^v_t
 *     g_t = clamp(-softplus(a_t), -5, 0),   beta_t = 1 / (1 + exp(-b_t))
 * Tokens before a sequence's first token are its conv history: zeros, or three rows of `hist`
 * (the last three projected tokens of the prefix the sequence continues, e.g. after a prefix
 * restore or for a decode step packed as a one-token sequence).
 *
 *   xq, xk, xv, a     [total_tokens, H, d] `dtype` (bf16 or fp32) inputs.
 *   b                 [total_tokens, H] `dtype`.
 *   w                 fp32 [3, H*d, 4]: taps of the q, k and v filters, channel-major, tap 3
 *                     on the current token.
 *   hist              `dtype` [n_seqs, 3 (q, k, v), 3 (t-3, t-2, t-1), H*d], or NULL = zeros.
 *   cu_seqlens, n_seqs, total_tokens   as for kda_prefill.
 *   d                 8, 16, 32, 64, 128 or 256 (a head's channels).  eps > 0.
 *   q, k, v, g        [total_tokens, H, d] `dtype` outputs; beta [total_tokens, H] `dtype`.
 *                     They must not alias any input.
 * Arithmetic is fp32; bf16 outputs are rounded to nearest.  Errors: KDA_ERR_INVALID_ARG,
 * KDA_ERR_UNSUPPORTED_SHAPE (d), KDA_ERR_MISALIGNED, KDA_ERR_CUDA.
 */
int kda_premix(const void *xq, const void *xk, const void *xv, const void *a, const void *b,
               const float *w, const void *hist, const int32_t *cu_seqlens, int32_t n_seqs,
               int64_t total_tokens, int32_t n_heads, int32_t d, float eps, int32_t dtype, void *q,
               void *k, void *v, void *g, void *beta, void *stream);

/*
 * kda_output_gate -- the input-dependent output gate on the recurrence's output.
 *
 * The section cited above gives KDA an input-dependent output gate acting on the output of its
 * attention path (third paragraph) and no formula; this call implements the plain reading, an
 * elementwise sigmoid gate:  out[i] = o[i] / (1 + exp(-z[i])),  i in [0, n).
 *
 *   o, z, out         n elements each, dtypes o_dtype, z_dtype, out_dtype (kda_dtype).  `out`
 *                     may be `o` itself when out_dtype == o_dtype (in place); it must not be z.
 * Arithmetic is fp32.  Errors: KDA_ERR_INVALID_ARG, KDA_ERR_MISALIGNED, KDA_ERR_CUDA.
 */
int kda_output_gate(const void *o, int32_t o_dtype, const void *z, int32_t z_dtype, void *out,
                    int32_t out_dtype, int64_t n, void *stream);

/*
 * kda_prefill_staged -- kda_prefill from pinned host memory, with the copies overlapped.
 *
 * The same operation as kda_prefill (d_k = d_v = 128, no checkpoints) for inputs and outputs in
 * host memory.  The packed tokens are cut into chunks of `chunk_tokens`: chunk c's inputs are
 * copied host -> device on one internal stream, prefilled on `stream` (every sequence resumes
 * from its running state in final_state, as the recurrence hands the state on from token to
 * token), and its outputs moved device -> host on a second internal stream, so uploads,
 * prefills and downloads of neighbouring chunks overlap.  When chunk_tokens is a multiple of 32,
 * the last chunk is cut in halves (multiples of 32 tokens) down to at most 128 tokens, which
 * shortens the work left after the last upload.  Downloads into pinned host memory are SM
 * stores through its device mapping (a 64-block kernel beside the prefill); into other
 * host memory they are copies.  When the call returns, all of it is enqueued and `stream` is
 * ordered after the last download.
 *
 *   h_q, h_k, h_v, h_g, h_beta   pinned host inputs, layouts and `dtype` as for kda_prefill.
 *   h_cu_seqlens     HOST int32 [n_seqs + 1] (checked here: 0, non-decreasing, total_tokens),
 *                    or NULL when n_seqs == 1.
 *   init_state       device fp32 [n_seqs, H, 128, 128] or NULL (zeros); may alias final_state.
 *   d_q .. d_beta, d_out   device buffers of the inputs' / outputs' full size (staging).
 *   h_out            host [total_tokens, H, 128] outputs (`out_dtype`), pinned for speed
 *                    (pageable memory works, with copy-engine downloads).
 *   final_state      device fp32 [n_seqs, H, 128, 128] (required: it carries the states).
 *   d_scratch        device int32 [scratch_ints] for the chunks' sequence tables, at least
 *                    kda_prefill_staged_scratch(...) entries (0 for a single sequence).
 *   chunk_tokens     >= 1 (a multiple of 32 keeps a single sequence's arithmetic identical to
 *                    kda_prefill's).  When the tokens span more than one chunk, chunk_tokens x
 *                    n_heads x (2 for bf16, 4 for fp32) must be a multiple of 16, so that every
 *                    chunk's beta rows start 16-byte aligned (bf16: chunk_tokens x n_heads a
 *                    multiple of 8); otherwise KDA_ERR_INVALID_ARG and nothing is enqueued.
 *   stream           a stream of the current device (KDA_ERR_INVALID_ARG for another device's).
 * The first call on a device creates two non-blocking streams (uploads, downloads) and four
 * events, which later calls on that device reuse and which live until the process exits; calls
 * from several host threads take turns at enqueueing on them.
 * Errors: those of kda_prefill, KDA_ERR_INVALID_ARG (a bad host table, too little scratch, an
 * unaligned chunk size, another device's stream), KDA_ERR_CUDA (stream or event creation, copies).
 */
int kda_prefill_staged(const void *h_q, const void *h_k, const void *h_v, const void *h_g,
                       const void *h_beta, const int32_t *h_cu_seqlens, int32_t n_seqs,
                       int64_t total_tokens, int32_t n_heads, int32_t dtype, int32_t out_dtype,
                       const float *init_state, void *d_q, void *d_k, void *d_v, void *d_g,
                       void *d_beta, void *d_out, void *h_out, float *final_state,
                       int32_t *d_scratch, int64_t scratch_ints, int64_t chunk_tokens, void *stream);

/* Scratch entries (int32) kda_prefill_staged needs for these sequences and chunk size, or -1 for
 * invalid arguments.  Host-only. */
int64_t kda_prefill_staged_scratch(const int32_t *h_cu_seqlens, int32_t n_seqs, int64_t total_tokens,
                                   int64_t chunk_tokens);

/*
 * kda_prefill_staged_static -- kda_prefill_staged without caller scratch: the chunks' sequence
 * tables go to a fixed device array of the library (2^20 int32 entries per device, a file-scope
 * __device__ array), so the caller provides no scratch and the library allocates no memory.  Calls
 * share that array: each call's `stream` first waits for the previous call's last prefill, so
 * calls from several streams or threads are safe and run one after another on the device.  The
 * first call on a device creates the staged path's two copy streams and four events (shared with
 * kda_prefill_staged) and one event that orders calls on the array; later calls reuse them
 * (kda_diag_staged_handles counts them).
 * Arguments and errors as for kda_prefill_staged; KDA_ERR_INVALID_ARG also when the tables need
 * more than 2^20 entries (kda_prefill_staged_scratch tells).
 */
int kda_prefill_staged_static(const void *h_q, const void *h_k, const void *h_v, const void *h_g,
                              const void *h_beta, const int32_t *h_cu_seqlens, int32_t n_seqs,
                              int64_t total_tokens, int32_t n_heads, int32_t dtype, int32_t out_dtype,
                              const float *init_state, void *d_q, void *d_k, void *d_v, void *d_g,
                              void *d_beta, void *d_out, void *h_out, float *final_state,
                              int64_t chunk_tokens, void *stream);

/*
 * kda_cp_combine -- the scan of a context-parallel prefill.
 *
 * The recurrence above is affine in the state: per token S_t = A_t S_(t-1) + beta_t k_t v_t^T with
 * A_t = (I - beta_t k_t k_t^T) diag(exp(clamp(g_t, -5, 0))).  Over a segment of a sequence,
 * S_end = M S_start + S_loc, where S_loc is the segment's final state from a zero initial state
 * (a kda_prefill of the segment) and M = A_L ... A_1 is its final state when prefilled with v = 0
 * from the identity (a kda_prefill with d_v = d_k).  Splitting a sequence into segments lets
 * those two prefills run every segment side by side; this call turns their end states into each
 * segment's true initial state and each sequence's final state; kda_cp_correct then turns the two
 * prefills' outputs into the sequence's outputs (or one more kda_prefill of the segments from their
 * start states gives them).
 *
 * For every sequence n and head, over its segments j in [seq_seg[n], seq_seg[n+1]) (at least one;
 * the first prefilled from the sequence's own initial state, so S_loc(first) is its true end state):
 *     S_start(first + 1) = S_loc(first),   S_start(j + 1) = M(j) S_start(j) + S_loc(j).
 *   s_loc, m       fp32 [n_seg, H, d, d]: the segments' final states of the two prefills (m of a
 *                  sequence's first segment is not read).
 *   seq_seg        device int32 [n_seqs + 1], non-decreasing segment ranges per sequence.
 *   s_start        fp32 [n_seg, H, d, d]: written for every segment but the first of each sequence.
 *   final_state    fp32 [n_seqs, H, d, d] (M(last) S_start(last) + S_loc(last)) or NULL.
 *   d              128.  Outputs must not alias inputs.  Arithmetic is fp32.
 * Errors: KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED_SHAPE, KDA_ERR_MISALIGNED, KDA_ERR_CUDA.
 */
int kda_cp_combine(const float *s_loc, const float *m, const int32_t *seq_seg, int32_t n_seqs,
                   int32_t n_heads, int32_t d, float *s_start, float *final_state, void *stream);

/*
 * kda_cp_correct -- the outputs of a context-parallel prefill, without prefilling the segments a
 * third time.
 *
 * Within a segment the true state is S_t = P_t S_start + S_loc,t, with P_t = A_t ... A_1 the
 * segment's prefix map (the affine form of kda_cp_combine).  So the true output is
 *     o_t = S_t^T q_t = o_loc,t + S_start^T u_t,   u_t = P_t^T q_t,
 * where o_loc,t are the outputs of the segment prefilled from zeros and u_t the outputs of the
 * segment prefilled with v = 0 from the identity (the two kda_prefill calls whose final states
 * kda_cp_combine takes).  For every segment but those listed in skip_seg, this call adds
 * S_start(seg)^T u_t to out[t] for each of its tokens and heads, as one tensor-core product per
 * (segment, head): tf32 operands (S_start rounded to nearest, u read as tf32), fp32 accumulation
 * and addition.  List a sequence's first segment in skip_seg: prefilled from the sequence's own
 * initial state, its outputs are already the true ones.
 *   u            fp32 [total_tokens, H, d], 16-byte aligned: the identity prefill's outputs.
 *   s_start      fp32 [n_seg, H, d, d]: kda_cp_combine's segment start states (S[key][value]).
 *   cu_seg       device int32 [n_seg + 1]: the segments' token ranges in the packed token axis.
 *   skip_seg     device int32 [n_skip], increasing: the segments left as they are (NULL iff
 *                n_skip == 0).
 *   out          fp32 [total_tokens, H, d], updated in place; must alias neither u nor s_start.
 *   d            128.  Device tables are taken as they are (not validated on the host).
 * Errors: KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED_SHAPE, KDA_ERR_MISALIGNED, KDA_ERR_CUDA; a
 * bounded device wait that expired shows up as KDA_ERR_DEVICE_TIMEOUT in kda_device_status.
 */
int kda_cp_correct(const float *u, const float *s_start, const int32_t *cu_seg, int32_t n_seg,
                   const int32_t *skip_seg, int32_t n_skip, int64_t total_tokens, int32_t n_heads,
                   int32_t d, float *out, void *stream);

/*
 * kda_device_status -- synchronize `stream`, then read and clear the current device's sticky
 * error word (KDA_OK if no device-side error was recorded since the last read).  *status
 * receives the recorded kda_status.  Returns KDA_OK, or KDA_ERR_CUDA if the read failed.
 */
int kda_device_status(int32_t *status, void *stream);

/*
 * kda_diag_device_timeout -- failure-detection check.  Launches one CTA on `stream` whose bounded
 * device wait is on a barrier that nothing completes; after `timeout_cycles` SM clock cycles
 * (1 .. 4e9; 2e6 is about 1 ms) the wait gives up and records KDA_ERR_DEVICE_TIMEOUT in the device
 * error word, through the same wait routine every kernel of the library uses.  A following
 * kda_device_status() returns that code and clears it; the CUDA context stays usable.  The pages
 * have no counterpart: it exists so that a caller (or a test) can see an expired device wait
 * surface as an error status instead of a hang.
 * Errors: KDA_ERR_INVALID_ARG (cycles out of range), KDA_ERR_CUDA.
 */
int kda_diag_device_timeout(int64_t timeout_cycles, void *stream);

/*
 * kda_diag_bounds_check -- the device-side bounds check of a debug build, shown to work.  A library
 * compiled with -DKDA_DEBUG checks, inside the tensor-core prefill, every shared-memory pointer the
 * kernel's accessors take against the CTA's shared-memory window and every TMEM address against
 * the allocated columns and the lanes the executing warp may reach; a failed check skips the access
 * and records KDA_ERR_DEVICE_BOUNDS in the device error word (read by kda_device_status) and the
 * check's site number.  This call launches one thread that runs that check on an offset past its
 * window, without any access, so the same recording happens in every build.  *site receives the
 * site number of the first failed check since the last call (0 if none), after synchronizing
 * `stream`, and is cleared.  The pages have no counterpart.  Errors: KDA_ERR_INVALID_ARG (site
 * NULL), KDA_ERR_CUDA.
 */
int kda_diag_bounds_check(int32_t run_probe, int32_t *site, void *stream);

/*
 * kda_diag_staged_handles -- how many CUDA streams and events kda_prefill_staged and
 * kda_prefill_staged_static have created in this process so far (host only, no CUDA call).  The
 * first staged call on a device creates its two copy streams and four events, and the first static
 * call on a device its one table event; later calls reuse them, so the count stays put across
 * repeated calls.  The pages have no counterpart.  Errors: KDA_ERR_INVALID_ARG (created NULL).
 */
int kda_diag_staged_handles(int64_t *created);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */

/*
 * linattn.h -- C ABI of the GB300 (sm_103a) library for normalised causal
 * linear attention with a positive feature map and a recurrent S/z state.
 *
 * The method (sources cited by page title and section):
 *   [LA] "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention)
 *   [LC] "45. Linear Attention and Recurrent State | 线性注意力与递推状态" (datawhalechina, ch. 45)
 *
 *   phi(x)  = ELU(x) + 1  (x + 1 for x > 0, e^x otherwise)        [LA] "关键改写：让求和先发生"
 *   S_t     = alpha_t S_{t-1} + phi(k_t) v_t^T                     [LA] "公式里的每个维度",
 *   z_t     = alpha_t z_{t-1} + phi(k_t)                                "加一个门：让旧记忆逐渐淡出"
 *   y_t     = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)              [LA] "ε 是数值保护"
 * The state is updated before it is read, so y_t sees token t ([LA]
 * "每来一个 token，更新两个累加器"; [LC] TODO 3).  alpha_t == 1 is the ungated
 * form.  Prefill evaluates the recurrence chunk by chunk ([LA] "一个 chunk 的输出由
 * 两部分组成"); decode applies one step of it to a stored state ([LA]
 * "训练时，状态更新也能按块并行": the token recurrence suits decode).
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by the
 *    caller; all arrays are dense, row-major and contiguous.  The library keeps
 *    no pointer after a call returns and allocates no device memory.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream).  No call synchronises except la_last_device_status.
 *  - Errors are return codes.  Argument errors are detected on the host before
 *    anything is enqueued, and leave every output untouched.  LA_ERR_CUDA
 *    reports a failed launch or an earlier asynchronous CUDA error; kernels that
 *    give up waiting on an on-chip barrier record LA_ERR_TIMEOUT in a device
 *    status word that la_last_device_status reads.
 *  - Element types: q, k, v and y share `dtype` (BF16 or FP32).  States S, z and
 *    gates alpha are always FP32.  Arithmetic is FP32 with FP32 accumulation;
 *    on the BF16 path the features phi(q), phi(k) and the in-chunk score matrix
 *    enter the tensor cores as BF16.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_NULL = 1,        /* a required pointer is NULL                                      */
    LA_ERR_SHAPE = 2,       /* a size is < 1, out of range, or sizes disagree                    */
    LA_ERR_DTYPE = 3,       /* unknown element type                                            */
    LA_ERR_ALIGN = 4,       /* a pointer is not aligned as the chosen kernel requires           */
    LA_ERR_UNSUPPORTED = 5, /* a valid request that this build does not implement              */
    LA_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed                            */
    LA_ERR_TIMEOUT = 7,     /* a kernel gave up waiting on an on-chip barrier                   */
    LA_ERR_WORKSPACE = 8    /* workspace NULL or smaller than the entry point needs             */
} la_status;

typedef enum { LA_DTYPE_BF16 = 0, LA_DTYPE_FP32 = 1 } la_dtype;

/*
 * la_state_init -- S = 0, z = 0 (the empty history; [LA] "每来一个 token，更新两个累加器":
 * the state starts from S0 = 0, z0 = 0; [LC] the zero-initialised state and normaliser).
 *   S  device, FP32 [B,H,r,dv]  (row i = feature index, column j = value index)
 *   z  device, FP32 [B,H,r]
 * Requires B, H, r, dv >= 1.  Errors: LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_CUDA.
 */
la_status la_state_init(float *S, float *z, int B, int H, int r, int dv, la_stream_t stream);

/*
 * la_prefill_workspace_bytes -- device scratch that la_prefill_chunked needs for
 * these sizes on the current device.  It is non-zero only for the BF16 path
 * when B*H*(dv/64) CTAs would leave at least half of the device's SMs idle and
 * T is long enough (>= 2048 tokens): the kernel then splits every sequence
 * into segments that run in parallel ([LA] "门控递推为什么能做并行 scan？": the
 * per-token updates are affine maps of the state, so a segment's map (the
 * product A of its gates and the state dS, dz it writes from a zero state)
 * can be computed first, scanned, and each segment started from its state).
 * The scratch holds A, dS, dz per segment part and every segment's start
 * state: FP32, about 66 KB per head per entry at r = dv = 128.  The answer
 * depends on the device's SM count: ask with the device current that will run
 * the call.  Returns 0 for sizes the BF16 path does not support.
 */
size_t la_prefill_workspace_bytes(int B, int H, int T, int r, int dv, int chunk);

/*
 * la_prefill_chunked -- run T tokens of every (b, h) sequence through the
 * recurrence, starting from (S0, z0), and return every output y_t and the final
 * state ([LA] "一个 chunk 的输出由两部分组成": per chunk, the read of the carried
 * state Q~c Sprev plus the masked in-chunk product [(Q~c K~c^T) . M] Vc, the same
 * two parts for the denominator, and the hand-off Snext, znext; with a gate, each
 * term is scaled by the product of the gates between its write and its read).
 *
 *   q, k   device [B,H,T,r]  dtype          v, y   device [B,H,T,dv]  dtype
 *   alpha  device FP32 [B,H,T], 0 <= alpha <= 1, or NULL for alpha == 1.
 *          alpha_t scales the state carried into token t (alpha of the first
 *          token scales S0, z0).
 *   S0     device FP32 [B,H,r,dv] or NULL (zero);  z0 device FP32 [B,H,r] or NULL.
 *          S0 may equal S_out and z0 may equal z_out (in-place continuation).
 *   S_out  device FP32 [B,H,r,dv] final state;  z_out device FP32 [B,H,r].
 *   eps    added once to the whole denominator: y = num / (den + eps).
 *   chunk  chunk length in tokens, >= 1.  The result does not depend on it
 *          beyond rounding ([LA] "动手实验": chunk boundaries do not change the
 *          semantics), so the BF16 kernel computes in chunks of 64 tokens
 *          whatever value is given; the FP32 path runs token by token.
 *   workspace, workspace_bytes: device scratch of at least
 *          la_prefill_workspace_bytes(...) bytes, 256-byte aligned, owned by the
 *          caller and not read after the call's kernels finish (may be NULL
 *          when that is 0).  Calls sharing one workspace must be ordered.
 *
 * Kernels:
 *   BF16: tensor-core kernel (tcgen05 MMAs with TMEM accumulators, TMA tile
 *         loads), chunks of 64 tokens.  Requires r == 128, dv in {64, 128}, q, k,
 *         v, y, S_out 16-byte aligned.  With a workspace (see above) three launches:
 *         the state pass, the scan of segment start states, and the chunk
 *         kernel over all segments at once.
 *   FP32: exact FP32 token recurrence on CUDA cores (chunk is not used).
 *         Requires 1 <= r <= 256, 1 <= dv <= 256, 4-byte alignment.
 * T may be any length >= 1 (a final partial chunk is masked).
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE (B, H, T, r, dv or chunk < 1), LA_ERR_DTYPE,
 *         LA_ERR_ALIGN, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE, LA_ERR_CUDA.
 */
la_status la_prefill_chunked(const void *q, const void *k, const void *v, la_dtype dtype,
                             const float *alpha, const float *S0, const float *z0,
                             int B, int H, int T, int r, int dv, int chunk, float eps,
                             void *y, float *S_out, float *z_out,
                             void *workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * la_prefill_varlen_workspace_bytes -- device scratch that la_prefill_varlen needs
 * for a batch of B sequences, H heads and total_T tokens (total_T >= 0) on the
 * current device: the plan's tables and, when sequences can be split, their
 * segment states (0: the call needs none, dv = 64 with nothing to split).  It
 * depends on the sizes and the device's SM count only, not on the lengths, which
 * stay on the device.  Returns 0 for sizes la_prefill_varlen rejects.
 */
size_t la_prefill_varlen_workspace_bytes(int B, int H, int total_T, int r, int dv);

/*
 * la_prefill_varlen -- la_prefill_chunked for a batch of sequences of different
 * lengths packed one after another, e.g. the prompts of a serving batch, each
 * prefilled in large blocks and continuing from its own state ([LA]
 * "训练时，状态更新也能按块并行": token-by-token steps suit decode, prefill is
 * organised in chunks that hand the state on).  Sequence b is tokens cu_seqlens[b] ..
 * cu_seqlens[b+1]-1; it starts from S0[b], z0[b] and leaves its final state in
 * S_out[b], z_out[b] (an empty sequence copies S0, z0).
 *
 *   q, k       device BF16 [total_T, H, r]   (token-major: row t*H + h)
 *   v, y       device BF16 [total_T, H, dv]
 *   alpha      device FP32 [total_T, H] or NULL (alpha == 1)
 *   S0, z0     device FP32 [B, H, r, dv], [B, H, r] or NULL (zero); may alias S_out, z_out
 *   S_out, z_out  device FP32 [B, H, r, dv], [B, H, r]
 *   cu_seqlens device int32 [B + 1]: 0 = cu_seqlens[0] <= ... <= cu_seqlens[B] = total_T.
 *              The host cannot read it; a kernel finding a sequence outside
 *              [0, total_T] or of negative length skips it and records LA_ERR_SHAPE
 *              (read it with la_last_device_status).
 *   workspace  device scratch of la_prefill_varlen_workspace_bytes(B, H, total_T, r, dv)
 *              bytes, 256-byte aligned, owned by the caller and not read by the
 *              caller afterwards; may be NULL when that is 0.  Calls that may
 *              overlap in time need their own.
 * Long sequences are split into segments, as la_prefill_chunked splits a long T
 * ([LA] "门控递推为什么能做并行 scan？": a run of tokens composes into one affine map
 * of the state): a plan kernel reads the lengths and picks the segment length from
 * the batch's own chunk count, so that a long prompt among short ones no longer
 * holds up the batch; a state pass over the segments that end before a sequence's
 * last one and a scan give every segment its start state.  When no sequence is
 * long enough, or any sequence's bounds are invalid, nothing is split.  At dv = 128
 * with S0 16-byte aligned (or NULL), a sequence of at most 32 tokens (a short
 * continuation of one request, empty ones included) is walked token by token with
 * its state in registers (the walk of la_prefill_chunked), beside the others, on a
 * second stream of the library's (one per host thread and device, ordered against
 * `stream` by events): the first such call on a device from a host thread creates
 * it and must not be made inside a stream capture.
 * Requires BF16, r == 128, dv in {64, 128}, chunk >= 1 (computed in chunks of 64
 * tokens, as la_prefill_chunked); q, k, v, y, S_out 16-byte aligned.  total_T may be 0.
 * Rows of y outside every sequence are not written.
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_DTYPE, LA_ERR_ALIGN, LA_ERR_UNSUPPORTED
 *         (FP32 or other sizes), LA_ERR_WORKSPACE (workspace missing or too small),
 *         LA_ERR_CUDA.
 */
la_status la_prefill_varlen(const void *q, const void *k, const void *v, la_dtype dtype,
                            const float *alpha, const float *S0, const float *z0, const int *cu_seqlens,
                            int B, int H, int total_T, int r, int dv, int chunk, float eps,
                            void *y, float *S_out, float *z_out,
                            void *workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * la_prefill_chunked_noalloc -- la_prefill_chunked without caller scratch: the
 * workspace is a 32 MiB buffer compiled into the library (a static device array),
 * one per device for the whole process.  The pages have no counterpart; it is an
 * integration aid for callers that must not allocate device memory per call,
 * such as a serving loop that reserved its whole memory budget up front, or C
 * code without a caching allocator, where cudaMalloc/cudaFree would add
 * device-wide synchronisation and can fail under memory pressure.
 *   Arguments, results and errors are those of la_prefill_chunked, without
 *   workspace.  LA_ERR_WORKSPACE when la_prefill_workspace_bytes for these sizes
 *   exceeds the 32 MiB (the largest workspace la_prefill_workspace_bytes returns on
 *   devices with up to about 240 SMs).
 *   The first call on a device looks up the buffer's device address with that
 *   device current; make it before any stream capture.  The look-up is cached
 *   per device in an atomic, so first calls from several host threads are safe.
 *   Nothing in the buffer has to start at zero: a call writes every entry before
 *   reading it.  Calls that may overlap in time (other streams, other threads)
 *   race on the one buffer; the caller must serialise them.
 */
la_status la_prefill_chunked_noalloc(const void *q, const void *k, const void *v, la_dtype dtype,
                                     const float *alpha, const float *S0, const float *z0,
                                     int B, int H, int T, int r, int dv, int chunk, float eps,
                                     void *y, float *S_out, float *z_out, la_stream_t stream);

/*
 * la_decode_step -- one new token per (b, h), state updated in place:
 *   S <- alpha S + phi(k) v^T,  z <- alpha z + phi(k),  y = phi(q)^T S / (phi(q)^T z + eps)
 * ([LA] "公式里的每个维度" and "查询时，分子和分母一起读"; update before read).
 *   q, k   device [B,H,1,r] dtype;  v, y device [B,H,1,dv] dtype
 *   alpha  device FP32 [B,H] or NULL (alpha == 1)
 *   S      device FP32 [B,H,r,dv], read and overwritten;  z device FP32 [B,H,r], likewise.
 * Requires 1 <= r <= 256, 1 <= dv <= 256; 4-byte alignment (the r = dv = 128 fast
 * path is taken when S is 16-byte aligned).
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_DTYPE, LA_ERR_ALIGN, LA_ERR_UNSUPPORTED, LA_ERR_CUDA.
 */
la_status la_decode_step(const void *q, const void *k, const void *v, la_dtype dtype,
                         const float *alpha, float *S, float *z, int B, int H, int r, int dv,
                         float eps, void *y, la_stream_t stream);

/*
 * la_backward_workspace_bytes -- device scratch that la_prefill_backward needs for
 * these sizes on the current device, for any r, dv <= 128 and either dtype: the
 * FP32 per-token terms and one value per head (4 * B*H*(3T + 1) bytes), the maps
 * of the z_t pass (4 * B*H*ceil(T/128)*257 bytes), and, when B*H whole-head CTAs
 * would leave enough SMs idle and T is long enough, the two state passes of the
 * sequence-segmented tensor-core sweeps (forward and reversed: per head and part
 * or segment 4 * (128*128 + 128) bytes).  The size depends on the device's SM
 * count; it is 0 only for invalid sizes.
 */
size_t la_backward_workspace_bytes(int B, int H, int T);

/*
 * la_prefill_backward -- gradients of la_prefill_chunked's outputs for training.
 * Given dy = dL/dy and optionally dS_T = dL/dS_T, dz_T = dL/dz_T, returns
 * dL/dq, dL/dk, dL/dv, dL/dalpha, dL/dS0 and dL/dz0.  The pages give no backward
 * formula; this is the chain rule through the recurrence of [LA] "公式里的每个维度"
 * and "加一个门：让旧记忆逐渐淡出", with y_t = n_t / d_t:
 *   dn_t = dy_t / d_t,  dd_t = -(dy_t . y_t) / d_t,
 *   G_t = phi(q_t) dn_t^T + alpha_{t+1} G_{t+1},  g_t = dd_t phi(q_t) + alpha_{t+1} g_{t+1},
 *   dq_t = phi'(q_t) * (S_t dn_t + dd_t z_t),  dk_t = phi'(k_t) * (G_t v_t + g_t),
 *   dv_t = G_t^T phi(k_t),  dS0 = alpha_1 G_1,  dz0 = alpha_1 g_1,
 *   dalpha_u = (sum_{t >= u} (phi(q_t) . dq~_t - phi(k_t) . dk~_t) + <dS_T, S_T> + <dz_T, z_T>) / alpha_u
 * (dq~, dk~: the gradients before the phi' factor).
 *   q, k, v, alpha, S0, z0, eps: as passed to the forward call.
 *   y      device [B,H,T,dv] dtype: the forward's output (used for dd_t).
 *   dy     device [B,H,T,dv] dtype.
 *   dS_T, dz_T  device FP32 [B,H,r,dv], [B,H,r], or NULL (zero).
 *   dq, dk device [B,H,T,r] dtype;  dv_out device [B,H,T,dv] dtype.
 *   dalpha device FP32 [B,H,T], or NULL (not computed; ignored without alpha).
 *          Defined where alpha > 0 (it is the log-gate derivative over alpha).
 *   dS0, dz0  device FP32 [B,H,r,dv], [B,H,r] (written also when S0, z0 are NULL).
 *   workspace: >= la_backward_workspace_bytes device bytes, 16-byte aligned, owned by
 *          the caller; calls sharing it must be ordered.
 * Kernels: the z_t recurrence over segments of 128 tokens (maps, scan, products)
 * for d_t, one pass for dd_t, then the three gradients as causal linear
 * attentions over chunks of 64 tokens (dq forward in time, dk and dv in
 * reverse), then a reverse running sum for dalpha.  BF16 with r = dv = 128 runs
 * the three on the tensor cores (BF16 operands, FP32 accumulators and state), and
 * for few long sequences over sequence segments whose entering states a forward
 * and a reversed state pass compute ([LA] "门控递推为什么能做并行 scan？"); the
 * other shapes and FP32 run them as gated rank-1 recurrences in FP32 on the CUDA
 * cores.  With segments, the state passes run on a second stream of the library's
 * (one per host thread and device, ordered against `stream` by events), beside
 * the z pass and the dq sweep; the call's work is still complete, in order, on
 * `stream`.  The first call on a device from a host thread creates that stream
 * and must not be made inside a stream capture.  Requires r, dv in {32, 64, 128}, T >= 1, 16-byte aligned
 * token arrays (q, k, v, y, dy, dq, dk, dv_out), 4-byte aligned FP32 arrays
 * (dS_T 8-byte aligned).
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_DTYPE, LA_ERR_ALIGN, LA_ERR_UNSUPPORTED,
 *         LA_ERR_WORKSPACE, LA_ERR_CUDA.
 */
la_status la_prefill_backward(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                              const float *S0, const float *z0, int B, int H, int T, int r, int dv, float eps,
                              const void *y, const void *dy, const float *dS_T, const float *dz_T, void *dq,
                              void *dk, void *dv_out, float *dalpha, float *dS0, float *dz0, void *workspace,
                              size_t workspace_bytes, la_stream_t stream);

/*
 * la_backward_states_bytes -- bytes of the states buffer that la_prefill_chunked_save
 * can fill for la_prefill_backward_saved: the backward splits a sequence into
 * segments when few long sequences would leave SMs idle, and this is the state
 * [S | z] (FP32, 128 x 128 then 128) entering each segment of every (b, h).
 * 0 when the backward would not split (then there is nothing to keep).
 */
size_t la_backward_states_bytes(int B, int H, int T);

/*
 * la_prefill_chunked_save -- la_prefill_chunked that also keeps, for training, the
 * denominator of every output row: d_t = phi(q_t) . z_t + eps, the normaliser of
 * [LA] "公式里的每个维度" (y_t = phi(q_t)^T S_t / d_t), in FP32, and optionally the
 * states at which the backward's sequence segments start.
 * la_prefill_backward_saved takes them instead of recomputing them.
 *   d_out      device FP32 [B,H,T], 4-byte aligned, owned by the caller.
 *   states_out device buffer of la_backward_states_bytes(B, H, T) bytes, 16-byte
 *              aligned, or NULL (not kept).  Written for BF16 with r = dv = 128
 *              when that size is not 0; otherwise left untouched.
 *   Everything else as for la_prefill_chunked.
 * BF16: the chunk kernel's own denominator (the BF16 operands of its products,
 * FP32 accumulation), the one y was divided by, and its FP32 state; FP32: the
 * exact recurrence's denominator.
 * Errors: those of la_prefill_chunked; LA_ERR_NULL when d_out is NULL.
 */
la_status la_prefill_chunked_save(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                                  const float *S0, const float *z0, int B, int H, int T, int r, int dv, int chunk,
                                  float eps, void *y, float *S_out, float *z_out, float *d_out, float *states_out,
                                  void *workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * la_prefill_backward_saved -- la_prefill_backward with d_t taken from
 * la_prefill_chunked_save instead of recomputed: the z_t recurrence over the
 * sequence (three of the backward's launches) is skipped, and with states, the
 * forward state pass and scan of a segmented backward too.
 *   d      device FP32 [B,H,T] from la_prefill_chunked_save on the same inputs
 *          (eps is included in it, so there is no eps argument).
 *   states the states_out of that call, or NULL (recomputed when needed).
 *   Everything else as for la_prefill_backward.
 * Errors: those of la_prefill_backward; LA_ERR_NULL when d is NULL; LA_ERR_ALIGN
 *         when states is not 16-byte aligned.
 */
la_status la_prefill_backward_saved(const void *q, const void *k, const void *v, la_dtype dtype, const float *alpha,
                                    const float *S0, const float *z0, int B, int H, int T, int r, int dv,
                                    const void *y, const void *dy, const float *d, const float *states,
                                    const float *dS_T, const float *dz_T, void *dq, void *dk, void *dv_out,
                                    float *dalpha, float *dS0, float *dz0, void *workspace, size_t workspace_bytes,
                                    la_stream_t stream);

/*
 * la_delta_rule -- the delta-rule memory ([LA] "Delta rule：先读旧答案，再写误差"): a
 * state without the normaliser that, per token, reads its current answer for the
 * key, writes back beta times the error, and is then read by the query:
 *     p_t = S_{t-1}^T k_t,   S_t = S_{t-1} + beta_t k_t (v_t - p_t)^T,   y_t = S_t^T q_t
 * q and k are used as given (no feature map); the read follows the write, as in
 * the other entry points.  With a unit key and beta = 1 the memory returns v
 * exactly for that key; the error left on k after a step is (1 - beta |k|^2)
 * times the error before it, so the update contracts for 0 < beta |k|^2 < 2.
 *   q, k   device [B,H,T,r] dtype          v, y  device [B,H,T,dv] dtype
 *   beta   device FP32 [B,H,T] write strength, or NULL for beta == 1
 *   S0     device FP32 [B,H,r,dv] or NULL (zero); may equal S_out (in place)
 *   S_out  device FP32 [B,H,r,dv] final state
 * Kernel: the token recurrence in FP32 on CUDA cores (the pages give no block
 * algorithm for this rule, [LA] "训练时，状态更新也能按块并行"), the state in
 * registers, the value columns split over CTAs.  Requires r in {32, 64, 128, 256},
 * dv a multiple of 32, q, k, v, y 16-byte aligned, S0, S_out 8-byte aligned,
 * beta 4-byte aligned.  T may be 0 (S_out = S0; q, k, v, y may then be NULL and are not touched).
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE (B, H, r, dv < 1, T < 0), LA_ERR_DTYPE,
 *         LA_ERR_ALIGN, LA_ERR_UNSUPPORTED (other r or dv), LA_ERR_CUDA.
 */
la_status la_delta_rule(const void *q, const void *k, const void *v, la_dtype dtype, const float *beta,
                        const float *S0, int B, int H, int T, int r, int dv, void *y, float *S_out,
                        la_stream_t stream);

/*
 * la_delta_chunked_workspace_bytes -- bytes of device workspace la_delta_rule_chunked
 * needs for (B, H, T): 32 KB per chunk of 64 tokens per (b, h); 0 when T < 1.
 */
size_t la_delta_chunked_workspace_bytes(int B, int H, int T);

/*
 * la_delta_rule_chunked -- the memory of la_delta_rule, computed in chunks of 64
 * tokens on the tensor cores.  The pages give no block algorithm for this rule
 * ([LA] "训练时，状态更新也能按块并行"); this one follows from the update: for a
 * chunk with rows K, Q, V and the state S_prev before it, the written rows
 * V' = beta (V - K S) of the chunk's tokens solve (I + L) V' = diag(beta) X with
 * X = V - K S_prev and L = diag(beta) strictly-lower(K K^T), so
 *     V' = T X,  T = (I + L)^{-1} diag(beta),
 *     S_next = S_prev + K^T V',   Y = Q S_prev + (Q K^T masked causally, diagonal kept) V'.
 * The state chain evaluates V' as U - W S_prev with W = T K and U = T V, which
 * do not depend on the state.  The products take BF16 operands (q, k, v as
 * given, S_prev, W, T and V' rounded to BF16) with FP32 accumulation; U and the
 * state stay FP32 and T is solved in FP32.  Same arguments, layouts and ownership as
 * la_delta_rule, plus
 *   workspace  device buffer of >= la_delta_chunked_workspace_bytes(B, H, T) bytes,
 *              16-byte aligned, owned by the caller (may be NULL when T == 0);
 *              calls sharing it must be ordered.
 * Kernels: T, the masked scores (Q K^T) . M and -W of every chunk (one CTA per
 * chunk) into the workspace, then the state chain, one CTA per (b, h, 64-column
 * slice of v).  Requires dtype BF16,
 * r == 128, dv a multiple of 64, q, k, v, y, S0 and S_out 16-byte aligned, beta
 * 4-byte aligned.  T may be 0 (S_out = S0).
 * Errors: LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_DTYPE (not BF16), LA_ERR_ALIGN,
 *         LA_ERR_UNSUPPORTED (other r or dv), LA_ERR_WORKSPACE, LA_ERR_CUDA.
 */
la_status la_delta_rule_chunked(const void *q, const void *k, const void *v, la_dtype dtype, const float *beta,
                                const float *S0, int B, int H, int T, int r, int dv, void *y, float *S_out,
                                void *workspace, size_t workspace_bytes,
                                la_stream_t stream);

/*
 * la_last_device_status -- synchronise `stream`, then read and clear the device
 * status word of the current device: LA_OK, or LA_ERR_TIMEOUT when a kernel
 * gave up waiting on an on-chip barrier since the last read.  Returns
 * LA_ERR_CUDA when the synchronisation itself reports an error.
 */
la_status la_last_device_status(la_stream_t stream);

/* la_status_string -- a static, human-readable name for a status code. */
const char *la_status_string(la_status status);

/*
 * la_debug_wait_probe -- diagnostic: launches one block that waits on an
 * on-chip barrier that nothing ever completes, with a limit of `limit_ns`
 * nanoseconds (at most 1e9).  The wait runs out and records LA_ERR_TIMEOUT in the
 * device status word exactly as a stuck kernel would; the context stays usable.
 * Used to test the timeout path without faulting or hanging a GPU.
 */
la_status la_debug_wait_probe(unsigned long long limit_ns, la_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */

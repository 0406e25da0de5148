/*
 * still.h -- C ABI of libstill.so: one STILL intra-layer hybrid attention layer
 * (chunk-parallel prefill forward and bounded-memory decode step) on a GB300
 * (sm_103a).
 *
 * The method: "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient
 * LLM Linearization" (besthub.dev summary), with its companion write-ups
 * "STILL: Selecting Tokens for Intra-Layer Hybrid Attention to Linearize LLMs"
 * (roboind.com news page) and "NeurIPS 2026 | 层内混合注意力 ... STILL"
 * (shishifenxi.com).  Section names below are the headings of those pages.
 *
 * Conventions shared by every call
 *   - Tensors are dense, row-major, on the device unless stated otherwise.
 *     q, out: [B, Hq, N, d]; k, v: [B, Hkv, N, d]; query head h reads kv head
 *     h / G with G = Hq / Hkv (grouped-query attention).
 *   - still_bf16 is the raw 16-bit pattern of an IEEE bfloat16 value.
 *   - Wf: fp32 [d, d_f], one learned NP-Map matrix per layer, shared by q, k
 *     and all heads.
 *   - Routing parameters: W window slots, chunk length C, softmax budget m,
 *     T_max chunks that keep tokens; lambda = floor((m - W) / T_max) tokens kept
 *     per completed chunk (section "Content-Aware Routing with Fixed Budget").
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream).
 *     Argument errors are detected on the host and returned before anything
 *     is launched; launch failures return STILL_ERR_CUDA.  Errors found by a
 *     kernel (an index out of range) are written to a device status word
 *     (see still_read_status) and never trap.
 *   - Device pointers must be 16-byte aligned.  The caller owns all memory;
 *     the library keeps no device allocation between calls, apart from the
 *     fixed scratch array of still_prefill_noalloc.
 *   - Supported: d in {64, 128}, d_f in {64, 128}, 1 <= C <= 16384, W >= 0,
 *     m >= W, T_max >= 1, W >= 1 whenever lambda > 0.  N == 0 is a no-op.
 */
#ifndef STILL_H
#define STILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t still_bf16;
typedef struct CUstream_st *still_stream_t; /* the same handle as cudaStream_t */

typedef struct {
    int B, Hq, Hkv, N, d, d_f;
} still_shape;

typedef enum {
    STILL_OK = 0,
    STILL_ERR_INVALID_ARG = 1, /* null/misaligned pointer, inconsistent sizes   */
    STILL_ERR_UNSUPPORTED = 2, /* valid request outside the compiled shapes     */
    STILL_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
    STILL_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up            */
    STILL_ERR_BOUNDS = 5,      /* a kernel met an index outside its buffers     */
    STILL_ERR_WORKSPACE = 6    /* workspace smaller than still_prefill_workspace_size */
} still_status;

/*
 * Decode state of B sequences (all device memory, owned by the caller).  It is
 * the softmax KV cache of m slots per (sequence, kv head) plus the linear
 * recurrent state (section "Content-Aware Routing with Fixed Budget": W slots
 * for the sliding window, m - W for kept tokens, unkept tokens accumulated into
 * the linear-attention state, nothing re-scored or evicted).
 *   K, V        bf16  [B, Hkv, m, d]  slots 0..W-1: window ring, token j in
 *                                     slot j % W; slot W + c*lambda + r: the
 *                                     r-th kept token of chunk c.  While chunk
 *                                     c is unfinished its slots hold tokens of
 *                                     c that left the window and may still be
 *                                     among its top-lambda ("candidates").
 *   slot_pos    int32 [B, Hkv, m]     token position in the slot, -1 = empty
 *   slot_cnt    int32 [B, Hkv, m]     candidates: tokens of the chunk so far
 *                                     that outrank the candidate
 *   slot_score  fp32  [B, Hkv, m]     Self-Saliency score of the slot's token
 *   S           fp32  [B, Hkv, d_f, d] sum of phi(k) v^T over folded tokens
 *   z           fp32  [B, Hkv, d_f]   sum of phi(k) over folded tokens
 *   score_ring  fp32  [B, Hkv, C]     scores of the unfinished chunk (j % C)
 *   t           int64 [B, Hkv]        tokens absorbed so far
 *   status      int32 [1]             device status word (0 = fine)
 */
typedef struct {
    still_bf16 *K;
    still_bf16 *V;
    int32_t *slot_pos;
    int32_t *slot_cnt;
    float *slot_score;
    float *S;
    float *z;
    float *score_ring;
    int64_t *t;
    int32_t *status;
} still_decode_state;

/* Human-readable name of a status code (static string). */
const char *still_status_string(still_status s);

/* lambda = floor((m - W) / T_max), or -1 when the budget is invalid. */
int still_lambda(int W, int m, int T_max);

/*
 * Self-Saliency scores (section "Self-Saliency Score: Predicting Future
 * Utility from Local Context"; roboind "Highlight 2: Self-Absolute Score").
 * For each query head h and token t the window is keys [max(0, t-W+1), t];
 * a^diag is the softmax of q_t.k_j / sqrt(d) over the window, a^nodiag the
 * same without j = t, and Score = KL(a^nodiag || a^diag) in the closed form
 * -log(1 - p_t + 1e-6), p_t = a^diag_t.  The kv-head score is the mean over
 * the G query heads of the group.
 *   q [B,Hq,N,d] bf16, k [B,Hkv,N,d] bf16 -> scores fp32 [B,Hkv,N].
 * Requires W >= 1.
 */
still_status still_score(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, int W,
                         float *scores, still_stream_t stream);

/*
 * Routing metrics (section "Ablation Studies", routing metric comparison: the
 * fixed-budget selection run with other per-token scores in place of the
 * Self-Saliency Score).  Every metric yields one fp32 score per (sequence, kv
 * head, token), [B, Hkv, N]; a higher score ranks higher in the chunk's
 * top-lambda.  The pages name the metrics but print no formula; the readings:
 *   SELF_SALIENCY  the Self-Saliency Score, as still_score
 *   DIAGONAL       mean over the G query heads of p_t, the token's own weight in
 *                  the softmax over its causal window of W keys (a^diag_t)
 *   QK             mean over the G query heads of q_t . k_t / sqrt(d)
 *   KEY_NORM       ||k_t|| (two-norm over d)
 *   UNIFORM        1 at the lambda evenly spaced offsets floor((r + 1/2) C /
 *                  lambda), r < lambda, of every chunk, 0 elsewhere (every
 *                  offset when lambda >= C)
 *   RANDOM         SplitMix64 (Steele, Lea, Flood 2014) as a counter-based
 *                  generator: z = seed + (i + 1) * 0x9E3779B97F4A7C15, then its
 *                  published output mix, with i = (b Hkv + g) N + t; the score
 *                  is (z >> 40) * 2^-24 in [0, 1)
 */
typedef enum {
    STILL_METRIC_SELF_SALIENCY = 0,
    STILL_METRIC_DIAGONAL = 1,
    STILL_METRIC_QK = 2,
    STILL_METRIC_KEY_NORM = 3,
    STILL_METRIC_UNIFORM = 4,
    STILL_METRIC_RANDOM = 5
} still_metric;

/*
 * Scores of one routing metric.  q [B,Hq,N,d] bf16 (read by SELF_SALIENCY,
 * DIAGONAL and QK; may be NULL otherwise), k [B,Hkv,N,d] bf16 (read by all but
 * UNIFORM and RANDOM; may be NULL for those two) -> scores fp32 [B,Hkv,N].  W is
 * the window of SELF_SALIENCY and DIAGONAL (>= 1 for them); C, m and T_max
 * give UNIFORM its lambda and are checked as for still_select; seed is read by
 * RANDOM only.  An unknown metric returns STILL_ERR_INVALID_ARG.
 */
still_status still_score_metric(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, int W, int C,
                                int m, int T_max, still_metric metric, uint64_t seed, float *scores,
                                still_stream_t stream);

/*
 * Delayed chunk-level selection (section "Delayed Chunk-Level Selection for
 * Unified Training-Inference Parallelism"): each completed chunk c < T_max
 * (tokens [cC, cC + C), all < N) keeps its top-lambda tokens by score, an
 * exact tie going to the lower position; positions are written in ascending
 * order.  Rows of chunks that keep nothing (incomplete, or past the data) and
 * unused columns when lambda > C are -1.
 *   scores fp32 [B,Hkv,N] -> sel_idx int32 [B,Hkv,T_max,lambda].
 */
still_status still_select(const still_shape *shape, const float *scores, int W, int C, int m, int T_max,
                          int32_t *sel_idx, still_stream_t stream);

/*
 * NP-Map feature map (section "NP-Map: Norm-Preserving Feature Map"): the
 * learned map only chooses a direction and the input norm is put back,
 * phi(x) = ||x|| u / ||u||, u = softmax(x Wf) over the d_f features.
 *   x bf16 [rows, d], Wf fp32 [d, d_f] -> phi fp32 [rows, d_f].
 */
still_status still_npmap(const still_bf16 *x, long long rows, int d, const float *Wf, int d_f, float *phi,
                         still_stream_t stream);

/* Bytes of device workspace still_prefill needs for these sizes. */
size_t still_prefill_workspace_size(const still_shape *shape, int W, int C, int m, int T_max);

/*
 * Chunk-parallel prefill forward of one layer (sections "Content-Aware
 * Routing with Fixed Budget", "Delayed Chunk-Level Selection ...", "NP-Map"
 * and the shared normalisation of the two branches):
 *   SA(t) = {t-W < j <= t} U {j kept by chunk(j) < chunk(t), j <= t-W}
 *   LA(t) = {j <= t-W} minus SA(t)
 *   y_t = (sum_SA e^{s-c} v + phi(q)^T S_LA) / (sum_SA e^{s-c} + phi(q)^T z_LA)
 * with s = q.k / sqrt(d) and c = max over SA(t).
 *   out bf16 [B,Hq,N,d]; sel_idx int32 [B,Hkv,T_max,lambda] (nullable).
 *   workspace: device memory of still_prefill_workspace_size() bytes, or NULL
 *   to let the call take and release it stream-ordered (cudaMallocAsync).
 *   export_state (nullable): filled with the decode state after N tokens,
 *   identical to what N decode steps from an empty state would hold.
 */
still_status still_prefill(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                           const still_bf16 *v, const float *Wf, int W, int C, int m, int T_max,
                           still_bf16 *out, int32_t *sel_idx, void *workspace, size_t workspace_bytes,
                           const still_decode_state *export_state, still_stream_t stream);

/*
 * The prefill above with the chunk selection ranked by another routing metric
 * (see still_metric); everything after the scores is the same layer.  With
 * STILL_METRIC_SELF_SALIENCY it computes exactly what still_prefill does.  No
 * decode state is exported: the decode step ranks by the Self-Saliency Score.
 * workspace as for still_prefill (still_prefill_workspace_size bytes, or NULL).
 */
still_status still_prefill_routed(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                  const still_bf16 *v, const float *Wf, int W, int C, int m, int T_max,
                                  still_metric metric, uint64_t seed, still_bf16 *out, int32_t *sel_idx,
                                  void *workspace, size_t workspace_bytes, still_stream_t stream);

/*
 * The prefill above with a gate on the linear branch (section "NP-Map:
 * Norm-Preserving Feature Map": a gating mechanism raises the linear branch's
 * rank; the ablation loses 5.8 points without it).  The pages lost its
 * equation; the reading this library takes is a per-channel sigmoid gate on
 * the linear branch's numerator, the shared denominator ungated:
 *   y_t = (sum_SA e^{s-c} v + g_t * (phi(q)^T S_LA)) / (sum_SA e^{s-c} + phi(q)^T z_LA),
 *   g_t = 1 / (1 + exp(-a_t)) elementwise,
 * where a = gate, bf16 [B,Hq,N,d] (the layout of q), holds the pre-activation
 * of query head h at token t (the linear part of y includes the own-chunk and
 * lagged linear keys, gated alike).  A gate of +inf everywhere gives
 * still_prefill's layer.  Everything else -- routing, selection, workspace
 * (still_prefill_workspace_size bytes, or NULL) and the optional export of the
 * decode state -- is as for still_prefill.  The gate scales the output only:
 * the exported state is the ungated layer's, and still_decode_step_gated
 * continues the gated layer from it.
 */
still_status still_prefill_gated(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                 const still_bf16 *v, const still_bf16 *gate, const float *Wf, int W, int C, int m,
                                 int T_max, still_bf16 *out, int32_t *sel_idx, void *workspace,
                                 size_t workspace_bytes, const still_decode_state *export_state,
                                 still_stream_t stream);

/*
 * The decode step of the gated layer: still_decode_step with the gate
 * pre-activations of this step, gate_t bf16 [B,Hq,d] (the layout of q_t),
 *   y_t = (sum_SA e^{s-c} v + sigmoid(gate_t) * (phi(q)^T S + the linear keys' terms))
 *         / (sum_SA e^{s-c} + phi(q)^T z + the linear keys' weights).
 * Everything else is as for still_decode_step.  Only the staged decode kernel
 * carries the gate: states whose cache does not fit it (still_decode_step's
 * general path) return STILL_ERR_UNSUPPORTED.
 */
still_status still_decode_step_gated(const still_shape *shape, const still_decode_state *state, const still_bf16 *q_t,
                                     const still_bf16 *k_t, const still_bf16 *v_t, const still_bf16 *gate_t,
                                     const float *Wf, int W, int C, int m, int T_max, still_bf16 *out_t,
                                     still_stream_t stream);

/*
 * Backward pass of the layer (still_prefill's forward, ungated) with the
 * routing held fixed: given the selection sel_idx the forward made and the
 * upstream gradient dout = dL/dy, writes dL/dq, dL/dk, dL/dv and dL/dWf.
 * Section "Experiments" of "STILL: Content-Aware Intra-Layer Hybrid Attention
 * for Efficient LLM Linearization" trains through the layer; the selection is
 * a discrete choice and carries no gradient.  The stabiliser c_t (the row
 * maximum over the softmax keys) is part of the output -- the linear terms are
 * not scaled by it -- so its gradient goes to the logit of the key where the
 * maximum is attained (the lowest position among equal maxima).
 *   q, k, v, Wf   as for still_prefill (bf16 [B,H,N,d], fp32 [d,d_f])
 *   sel_idx       int32 [B,Hkv,T_max,lambda], the table still_prefill wrote
 *                 (-1 = no token); entries must be positions of completed
 *                 chunks c < T_max in ascending order within their chunk
 *   dout          bf16 [B,Hq,N,d]
 *   dq            fp32 [B,Hq,N,d]; dk, dv fp32 [B,Hkv,N,d]; dWf fp32 [d,d_f]:
 *                 overwritten (no accumulation into what they held)
 *   cmax_idx      nullable int32 [B,Hq,N]: the key position whose logit the
 *                 row maximum c_t took (the key that received c's gradient)
 *   workspace     still_backward_workspace_size() bytes, 16-byte aligned, or
 *                 NULL for a stream-ordered allocation inside the call
 * Supported: d == d_f in {64, 128}, G = Hq/Hkv in {1, 2, 4}, and lambda <= 128
 * when W < C (a kept key is then a linear key of the later queries of its own
 * chunk until the chunk completes); other shapes return STILL_ERR_UNSUPPORTED.  All device pointers 16-byte aligned.
 * The call is asynchronous on `stream`; dk, dv and dWf receive atomic
 * additions, so their low-order bits may differ between runs.
 */
size_t still_backward_workspace_size(const still_shape *shape, int W, int C, int m, int T_max);
still_status still_backward(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, const still_bf16 *v,
                            const float *Wf, int W, int C, int m, int T_max, const int32_t *sel_idx,
                            const still_bf16 *dout, float *dq, float *dk, float *dv, float *dWf, int32_t *cmax_idx,
                            void *workspace, size_t workspace_bytes, still_stream_t stream);

/*
 * The prefill above with its scratch memory taken from a fixed array inside
 * the library instead of a workspace argument.  The pages have no counterpart:
 * this entry point exists for callers that may not allocate device memory
 * while they run (an engine plug-in whose execution step must not allocate,
 * latency-critical code that cannot risk an allocation's synchronisation or
 * out-of-memory failure).  Inputs, outputs and the optional export state are
 * the caller's, exactly as for still_prefill.
 *   - The array holds still_prefill_noalloc_max_bytes() = 16 MiB; sizes whose
 *     still_prefill_workspace_size() exceeds it return STILL_ERR_WORKSPACE
 *     (and print why) without launching anything.
 *   - The call allocates and frees nothing.  The first call on a device looks
 *     up the array's device address (cudaGetSymbolAddress); make that first
 *     call before capturing a stream into a CUDA graph.
 *   - Every GPU that loads the library keeps the array until the process
 *     exits.  All calls on one GPU share it: calls that may overlap on the GPU
 *     (different streams without ordering between them) race on it and must
 *     not be issued.  Each call clears what has to start at zero itself.
 */
size_t still_prefill_noalloc_max_bytes(void);
still_status still_prefill_noalloc(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                   const still_bf16 *v, const float *Wf, int W, int C, int m, int T_max,
                                   still_bf16 *out, int32_t *sel_idx, const still_decode_state *export_state,
                                   still_stream_t stream);

/* Reset a decode state to "no token absorbed" (shape->N is ignored). */
still_status still_decode_state_init(const still_shape *shape, const still_decode_state *state, int W, int C,
                                     int m, int T_max, still_stream_t stream);

/*
 * One decode step for every sequence (the same routing and memory update as
 * the prefill, one token at a time): score the new token in its window; push
 * current-chunk candidates that fell out of the running top-lambda into (S,z);
 * move token t-W out of the window (into a slot or into (S,z)); attend over the
 * window and the kept slots with softmax plus phi(q)^T S; when the chunk
 * completes, keep its top-lambda.  shape->N is ignored.
 *   q_t bf16 [B,Hq,d], k_t, v_t bf16 [B,Hkv,d] -> out_t bf16 [B,Hq,d].
 */
still_status still_decode_step(const still_shape *shape, const still_decode_state *state,
                               const still_bf16 *q_t, const still_bf16 *k_t, const still_bf16 *v_t,
                               const float *Wf, int W, int C, int m, int T_max, still_bf16 *out_t,
                               still_stream_t stream);

/*
 * Failure-path testing.  The tensor-core prefill kernels bound every wait on
 * the device: a row warp waiting for a copy or a tensor-core result gives up
 * after a limit of clock cycles, writes STILL_ERR_TIMEOUT to the prefill's
 * status word (still_read_status on the first int32 of the workspace), lets
 * its block finish the copies and MMAs it already issued, and returns without
 * trapping.  This call sets that limit for kernels launched afterwards by
 * this process (cycles <= 0 restores the default of 4e9 cycles, about 2 s);
 * a limit far below a kernel's normal waiting time (a few hundred cycles)
 * makes the failure path run.  The outputs of a call that timed out are
 * undefined; the CUDA context stays usable.  Not for production use.
 */
void still_debug_set_wait_limit(long long cycles);

/* Synchronise `stream` and read a device status word (the one in a decode
 * state, or the first int32 of a prefill workspace). */
still_status still_read_status(const int32_t *status_word, still_stream_t stream, int32_t *host_value);

/*
 * Kernel timing for measurement: while enabled, every kernel the library
 * launches is bracketed by CUDA events on its stream.  still_timing_read
 * synchronises, returns per-kernel totals (name, launches, milliseconds) for
 * up to `max` kernels, clears the record and returns the number of kernels.
 */
typedef struct {
    char name[48];
    int launches;
    double ms;
} still_kernel_time;

void still_timing_enable(int on);
int still_timing_read(still_kernel_time *out, int max);

#ifdef __cplusplus
}
#endif

#endif /* STILL_H */

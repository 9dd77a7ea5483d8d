/*
 * switch_moe.h -- C ABI of the B300 (sm_103a) top-1 Switch MoE layer forward pass.
 *
 * The layer (pages cited by title, then section / equation):
 *   "042 · Switch Transformer：每个词只选一个专家" (wq-win.github.io), section 一:
 *       p(x) = softmax(W_r x), e*(x) = argmax_e p_e(x), y = p_{e*}(x) f_{e*}(x),
 *       capacity about (T/E) c, overflow tokens skip the expert and ride the residual;
 *   same page, section 二: L_aux = alpha E sum_e f_e P_e;
 *   same page, section 三: the pipeline (float32 router -> top-1 -> aux loss ->
 *       capacity truncation -> low-precision dispatch -> expert FFN -> gated combine),
 *       with "token representations, expert set, capacity factor, balance weight" in
 *       and "layer output and per-expert load statistics" out;
 *   "开源 AI 论文复现实验与代码解读 · 070" (zffjzz.top), section 核心思想与公式:
 *       Z = XW, f before truncation, P mean probability, C = ceil(cT/E), NumPy tie rule;
 *       section 官方代码阅读路线: slots by cumulative count in sequence order;
 *   "Switch Transformers ... - 中文验证版" (ai-papers.xuzou.cn), section 方法适配:
 *       float32 router inside, bfloat16 dispatch/combine;
 *   "混合专家" (world.lapla.si/zh/moe), section 专家里面是什么: d -> d_ff ReLU -> d with biases.
 *
 * Conventions for every call below
 *   - Ownership: the caller owns every pointer it passes (device memory unless
 *     a name ends in _host).  The handle owns only its internal workspace, which
 *     switch_create allocates and switch_destroy frees.  Nothing passed in is freed.
 *   - Execution: all calls except switch_get_stats, switch_sync_status and
 *     switch_stage_ms are asynchronous on the given stream.  Calls on one handle
 *     share its workspace: calls on one handle that overlap on the GPU race, so
 *     issue them on one stream (or serialise the streams).  The stream-ordered calls
 *     enqueue work only (no host synchronisation), so a CUDA graph may capture them
 *     and replay them on new contents of the same buffers (make one call before the
 *     capture).  With bfloat16 activations and more than two 64..256-expert router
 *     slices the router is a cooperative launch of one CTA per SM (two-CTA clusters
 *     for 256-expert slices): it starts once every SM can take one of its CTAs.
 *   - Errors: argument errors return at once (nothing is enqueued).  A kernel
 *     that finds an impossible state (a bounded wait that ran out, a debug bounds
 *     hit) sets a flag in the workspace; switch_get_stats / switch_sync_status
 *     report it.  Kernels never trap.
 *   - Layouts: row-major, dense.  N = G*T tokens, group-major ("16 sequences x 512"
 *     flattens sequence-major inside a group).  "act" = the config's dtype
 *     (float32 or bfloat16) for activations, expert weights and expert biases.
 *     The router weights and bias are always float32.
 *   - Alignment: every pointer must be 16-byte aligned; d_model * sizeof(act)
 *     and d_ff * sizeof(act) must be multiples of 16 bytes.
 */
#ifndef SWITCH_MOE_H
#define SWITCH_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SWITCH_API __attribute__((visibility("default")))
#else
#define SWITCH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SWITCH_OK = 0,
  SWITCH_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or config */
  SWITCH_ERR_UNSUPPORTED = 2,     /* valid but outside what this build implements */
  SWITCH_ERR_CUDA = 3,            /* a CUDA runtime call failed */
  SWITCH_ERR_DEVICE_TIMEOUT = 4,  /* a kernel's bounded wait ran out (flag set on device) */
  SWITCH_ERR_OOM = 5,             /* workspace allocation failed */
  SWITCH_ERR_DEVICE_BOUNDS = 6    /* a debug bounds check fired on the device */
} switch_status;

typedef enum { SWITCH_F32 = 0, SWITCH_BF16 = 1 } switch_dtype;

/* switch_config.flags */
#define SWITCH_FLAG_WRITE_PROBS   0x1u  /* route writes probs[N*E] (verification only) */
#define SWITCH_FLAG_WRITE_LOGITS  0x2u  /* route writes logits[N*E] (verification only) */
#define SWITCH_FLAG_DEBUG_BOUNDS  0x4u  /* kernels check slot/row/expert ranges */
#define SWITCH_FLAG_PROFILE       0x8u  /* switch_forward records per-stage CUDA events */
/* Top-2 routing (the variant on the 混合专家 page, section 路由器只开两条线): each token
 * goes to the experts of its two highest logits (ties to the lower index) with weights =
 * softmax over those two logits (they add to 1); capacity C = ceil(2 c T / E), twice the
 * top-1 capacity; a token's second choice takes a slot after its expert's kept first
 * choices of the group, in sequence order; f (and raw_count / accepted_count) count first
 * choices; a dropped choice's weight is not moved to the other.  Needs E >= 2. */
#define SWITCH_FLAG_TOP2          0x10u
/* Training: switch_forward keeps the dispatched rows, the hidden activations, the
 * expert outputs and the router logits in the workspace (unfused FFN and combine) for
 * switch_backward.  The workspace grows by float32 gradient scratch (2 E R d + E R d_ff +
 * N + N E floats, R = G min(C, T), plus the router's per-chunk partials, at most 64 M
 * floats) and, with bfloat16 and d, d_ff multiples of 128, by bfloat16 copies of the
 * backward's activations (E R (2 d + d_ff) bfloat16). */
#define SWITCH_FLAG_TRAINING      0x20u
/* Test only (fault injection on the host's request, no GPU fault): in the tensor-core
 * expert FFN, the first layer-1 tile of expert 0's first token chunk stores its part of h
 * but never publishes it, so the layer-2 tiles of that chunk wait on a count that nothing
 * completes.  Their bounded wait gives up after about a second of SM clock, sets the
 * device error word and carries on; switch_sync_status / switch_get_stats then return
 * SWITCH_ERR_DEVICE_TIMEOUT (and clear the word).  The outputs of such a call are
 * unspecified; the handle stays usable.  Has no effect where expert 0 receives no token
 * or the FFN runs on CUDA cores. */
#define SWITCH_FLAG_TEST_STALL    0x40u
/* Test only.  Outside training the tensor-core FFN drops each token chunk's hidden
 * activations from L2 once the chunk's last layer-2 tile has read them (no write-back
 * of scratch to DRAM), but only where they outgrow half of L2 and its tiles keep two
 * accumulator sets; this flag makes it do so for every shape, so small layers exercise
 * that path.  Results are unchanged. */
#define SWITCH_FLAG_TEST_DISCARD  0x80u

typedef struct {
  int G;                   /* routing groups; capacity and statistics are per group */
  int T;                   /* tokens per group */
  int d_model;             /* d */
  int d_ff;                /* expert hidden width */
  int E;                   /* experts, 1..2048 */
  double capacity_factor;  /* c; C = ceil(c*T/E), c*T/E snapped to an integer within 1e-9 */
  int capacity_override;   /* > 0: use this C instead */
  float alpha;             /* aux-loss weight (0.01 on the 042 page, section 二) */
  switch_dtype dtype;      /* act dtype */
  unsigned flags;          /* SWITCH_FLAG_* */
} switch_config;

typedef struct switch_layer* switch_handle;

/* Device buffers that switch_route fills (caller-owned).  Sizes in elements. */
typedef struct {
  int32_t* expert;          /* [N]   e*(x_t): the raw choice, also for dropped tokens   */
  int32_t* slot;            /* [N]   earlier tokens of the group that chose the same expert */
  uint8_t* keep;            /* [N]   1 when slot < C                                    */
  float* gate;              /* [N]   p_{t, expert_t}, never renormalised                */
  int32_t* row;             /* [N]   row of the token in its expert's block of xe, -1 if dropped */
  int32_t* raw_count;       /* [G*E] choices per expert before truncation               */
  int32_t* accepted_count;  /* [G*E] min(raw, C)                                        */
  float* P;                 /* [G*E] mean router probability per expert                 */
  float* balance;           /* [G]   unweighted E * sum_e f_e P_e                       */
  float* aux_loss_per_group;/* [G]   alpha * balance                                    */
  float* aux_loss;          /* [1]   mean over groups                                   */
  int32_t* expert_rows;     /* [E]   sum over groups of accepted_count (+ accepted2_count
                                     with SWITCH_FLAG_TOP2): rows of xe used              */
  float* probs;             /* [N*E] or NULL; written when SWITCH_FLAG_WRITE_PROBS      */
  float* logits;            /* [N*E] or NULL; written when SWITCH_FLAG_WRITE_LOGITS     */
  /* Router z-loss (ST-MoE, as restated on the 070 page, section 核心思想与公式):
   * L_z = (1/T) sum_t (log sum_e exp z_te)^2 over a group's T tokens, unweighted.
   * Either pointer may be NULL (not written). */
  float* z_loss_per_group;  /* [G]   L_z of each routing group                            */
  float* z_loss;            /* [1]   mean over groups                                     */
  /* Second choices (SWITCH_FLAG_TOP2 only, required then; ignored otherwise). */
  int32_t* expert2;         /* [N]   second choice                                        */
  int32_t* slot2;           /* [N]   kept first choices of that expert + earlier second choices */
  uint8_t* keep2;           /* [N]   1 when slot2 < C                                     */
  float* gate2;             /* [N]   its weight; gate + gate2 = 1 (gate is the first's)   */
  int32_t* row2;            /* [N]   row in the expert's block of xe, -1 if dropped       */
  int32_t* raw2_count;      /* [G*E] second choices per expert                            */
  int32_t* accepted2_count; /* [G*E] kept second choices per expert                       */
} switch_route_out;

/* Capacity C for cfg (host only, no GPU needed); -1 when cfg is invalid. */
SWITCH_API int64_t switch_capacity(const switch_config* cfg);

/* Rows per expert block of the dispatched buffer: G*C.  -1 when cfg is invalid. */
SWITCH_API int64_t switch_expert_block_rows(const switch_config* cfg);

SWITCH_API const char* switch_status_string(switch_status s);

/* Validate cfg, allocate the workspace on the current CUDA device, return a handle. */
SWITCH_API switch_status switch_create(const switch_config* cfg, switch_handle* out);
SWITCH_API switch_status switch_destroy(switch_handle h);

/*
 * Router + top-1 + slots + capacity mask + load statistics + aux loss.
 *   x   [N, d] act;  Wr [E, d] float32;  br [E] float32 or NULL (zero).
 * Logits are float32 (x cast up, then dot products with float32 accumulation);
 * ties go to the lowest expert index.  Measured against float64 dot products, the largest
 * logit error is ~1.5e-7 with float32 activations (CUDA cores) and grows with d on the
 * tensor-core path of bfloat16 activations: ~3.3e-9 d, or ~7.8e-9 d where more than 1024
 * experts and d <= 1024 let the three weight pieces share one accumulator (6.5e-6 at d = 768).
 * Writes every non-NULL field of *out
 * except probs/logits, which need their flags.  All fields other than
 * probs, logits and the z-loss are required, and with SWITCH_FLAG_TOP2 the
 * second-choice fields too.
 * With bfloat16 activations Wr may be NULL after switch_prepare_router on this handle:
 * the call then uses the prepared copy of the router weights (see there).  A non-NULL Wr
 * is read by this call, and the prepared copy is replaced by its split.
 */
SWITCH_API switch_status switch_route(switch_handle h, const void* x, const float* Wr, const float* br,
                           const switch_route_out* out, void* stream);

/*
 * Prepare the router weights once for calls that do not change them (inference).
 *   Wr [E, d] float32, read on `stream` by this call.
 * With bfloat16 activations the router multiplies on the tensor cores with W_r split into
 * three bfloat16 pieces (hi + mid + lo = w to within 2^-24 |w|).  Every switch_route,
 * switch_forward and switch_forward_host with a non-NULL Wr splits it again first (one
 * small kernel: 6 E d bytes written); after this call, passing Wr = NULL skips that step
 * and uses this split, until the next call with a non-NULL Wr replaces it.  The caller
 * must not change the weights in between without preparing again.
 * Returns SWITCH_ERR_UNSUPPORTED with float32 activations (the CUDA-core router reads Wr
 * itself), SWITCH_ERR_INVALID_ARG for a NULL handle or Wr.  Asynchronous on `stream`.
 * Not an operation of the method: a re-layout of the router weights kept on the handle.
 */
SWITCH_API switch_status switch_prepare_router(switch_handle h, const float* Wr, void* stream);

/*
 * Cap the CTAs of this handle's two persistent kernels, so that two handles working on two
 * batches on two streams run side by side on disjoint SMs: the router (bound by the
 * tensor cores) of one batch next to the expert FFN (bound by the weights' HBM bytes) of
 * the other.  Both kernels hold about 200 KB of shared memory, so each CTA takes an SM of
 * its own.
 *   route_ctas: CTAs of the tensor-core router; raised to the fewest that keep its expert
 *               slices waiting only on running CTAs (one cluster, or one CTA per slice).
 *               Routers whose slices meet in global memory then run as single CTAs, not
 *               CTA pairs: a pair needs two free SMs at once, while the other stream's
 *               kernels free them one at a time.
 *   ffn_ctas:   CTAs of the tensor-core expert FFN, at least 1 (2 where it runs on CTA pairs;
 *               rounded down to an even count there).
 * 0 restores the default (as many as the device holds).  Results do not depend on the caps:
 * only which CTA computes which tile changes.  Applies to later forward calls on the handle
 * (switch_route, switch_expert_ffn, switch_forward, switch_forward_host); the backward's
 * kernels are not capped.
 * Returns SWITCH_ERR_INVALID_ARG for a NULL handle or a negative cap.  Not an operation of the
 * method: a scheduling knob of this library.
 */
SWITCH_API switch_status switch_set_sm_budget(switch_handle h, int route_ctas, int ffn_ctas);

/*
 * Dispatch gather: xe[e, row_t, :] = x_t for every kept token t with expert e
 * (with SWITCH_FLAG_TOP2 also xe[expert2_t, row2_t, :] = x_t for kept second
 * choices); every other row of xe is zero.  xe is [E, G*C, d] act: expert e's block holds
 * its kept tokens group by group in sequence order.
 */
SWITCH_API switch_status switch_dispatch(switch_handle h, const void* x, const switch_route_out* r,
                              void* xe, void* stream);

/*
 * Expert FFN on each expert's first expert_rows[e] rows of xe:
 *   ye[e, i, :] = ReLU(xe[e, i, :] W1[e]^T + b1[e]) W2[e]^T + b2[e]
 * W1 [E, d_ff, d], b1 [E, d_ff] or NULL, W2 [E, d, d_ff], b2 [E, d] or NULL (act).
 * bfloat16: products on the tensor cores with float32 accumulation; the hidden
 * activation is rounded to bfloat16, and so is ye.  Rows of ye past
 * expert_rows[e] are left unspecified.
 */
SWITCH_API switch_status switch_expert_ffn(switch_handle h, const void* xe, const void* W1, const void* b1,
                                const void* W2, const void* b2, const int32_t* expert_rows,
                                void* ye, void* stream);

/*
 * Combine: y_t = gate_t * ye[expert_t, row_t, :] for kept tokens, 0 for dropped
 * ones (with SWITCH_FLAG_TOP2 plus gate2_t * ye[expert2_t, row2_t, :] for a kept
 * second choice), plus x_residual_t when x_residual is not NULL.  The gate is used as is
 * (no renormalisation).  y [N, d] act.
 */
SWITCH_API switch_status switch_combine(switch_handle h, const void* ye, const switch_route_out* r,
                             const void* x_residual, void* y, void* stream);

/*
 * The whole layer: route, dispatch, expert FFN, combine, on one stream.
 * Same arguments and results as the four calls above; the dispatched buffer,
 * the hidden activations and the expert outputs live in the workspace.
 * x_residual may be NULL.
 */
SWITCH_API switch_status switch_forward(switch_handle h, const void* x, const float* Wr, const float* br,
                             const void* W1, const void* b1, const void* W2, const void* b2,
                             const switch_route_out* r, const void* x_residual, void* y,
                             void* stream);

/*
 * The whole layer (as switch_forward) with the activations in HOST memory:
 * x_host [N, d] act is copied to the device, the layer runs, and y [N, d] act
 * and the aux loss are copied back to y_host and aux_loss_host (may be NULL).
 * Weights and the route results r are device buffers, as in switch_forward;
 * residual != 0 adds the layer input x to y.  Page-locked host buffers
 * (cudaHostAlloc / cudaHostRegister) let the copies run asynchronously;
 * pageable ones work, but their copies block the calling thread.
 *
 * Streams: the copy in runs on a copy stream of the handle and is NOT ordered
 * after earlier work on `stream` (it only reads x_host, which the caller has
 * filled); the layer runs on `stream`; the copy out runs on a second copy
 * stream of the handle.  The handle keeps two staging slots that alternate
 * between calls, so one call's copies overlap the previous or next call's
 * layer.  Completion:
 *   done_event == NULL: `stream` waits for the copy out, so the results are in
 *     place once `stream` has reached the end of this call;
 *   done_event != NULL (a cudaEvent_t the caller created): it is recorded after
 *     the copy out and `stream` does not wait; the results are in place once
 *     the event has completed.
 * The copy in is issued in four pieces of at least 1 MiB (one large host-to-device copy
 * was measured slower than a few pieces on some PCIe hosts of B300 machines).
 * The first call allocates the staging buffers (4 * N * d act elements) and
 * creates the copy streams, so it is not for use under stream capture.
 * Returns SWITCH_ERR_INVALID_ARG for NULL x_host / y_host with N > 0, else as
 * switch_forward.  The pages' layer is device-resident; moving activations
 * between host and device has no counterpart there.
 */
SWITCH_API switch_status switch_forward_host(switch_handle h, const void* x_host, const float* Wr,
                                  const float* br, const void* W1, const void* b1, const void* W2,
                                  const void* b2, const switch_route_out* r, int residual,
                                  void* y_host, float* aux_loss_host, void* done_event, void* stream);

/*
 * Backward of the top-1 layer (SWITCH_FLAG_TRAINING; top-2 returns
 * SWITCH_ERR_UNSUPPORTED): float32 gradients of
 *   L = sum(dy * y) + w_aux * aux_loss + w_z * z_loss
 * for the inputs of the last switch_forward on this handle, whose route results `r`
 * (and the workspace's saved activations) it reads.  The choices, slots and capacity
 * mask are held fixed; the router's gradient flows through the chosen expert's gate
 * probability (Switch Transformers card, section 方法适配) and through P in the aux loss,
 * not through the hard counts f (070 page, section 核心思想与公式); the z-loss through the
 * log-sum-exp.  residual != 0: y included x (dx gets dy too).
 *   x [N, d] act, Wr [E, d] f32, W1 [E, d_ff, d], W2 [E, d, d_ff] act, dy [N, d] act.
 *   Outputs (float32, caller-owned): dx [N, d], dWr [E, d], dbr [E], dW1 [E, d_ff, d],
 *   db1 [E, d_ff], dW2 [E, d, d_ff], db2 [E, d]; dbr, db1, db2 may be NULL.
 * With bfloat16 and d, d_ff multiples of 128 the expert products run on the tensor cores
 * (dye, dh, dxe and the weight gradients pass through bfloat16; float32 accumulation), and
 * so do the router's products dW_r = dz^T x and dz W_r when E is a multiple of 64 (dz and
 * W_r as bfloat16 hi + lo pieces, ~2^-16 relative); otherwise on CUDA cores in float32.
 */
SWITCH_API switch_status switch_backward(switch_handle h, const void* x, const float* Wr, const void* W1,
                              const void* W2, const switch_route_out* r, const void* dy, float w_aux,
                              float w_z, int residual, float* dx, float* dWr, float* dbr, float* dW1,
                              float* db1, float* dW2, float* db2, void* stream);

/*
 * Synchronise `stream`, then copy the aux loss, the [G*E] raw and accepted counts
 * and the number of dropped tokens of the route results `r` to the host
 * (any _host pointer may be NULL).  Returns the device error flag's status
 * (SWITCH_ERR_DEVICE_TIMEOUT / SWITCH_ERR_DEVICE_BOUNDS) if set, and clears it.
 */
SWITCH_API switch_status switch_get_stats(switch_handle h, const switch_route_out* r, void* stream,
                               float* aux_loss_host, int32_t* raw_host,
                               int32_t* accepted_host, int64_t* dropped_host);

/* Synchronise `stream` and return the device error flag's status (then clear it). */
SWITCH_API switch_status switch_sync_status(switch_handle h, void* stream);

/*
 * With SWITCH_FLAG_PROFILE: synchronise and return the elapsed milliseconds of
 * each stage of the last switch_forward: ms[0] route, ms[1] dispatch,
 * ms[2] FFN first layer, ms[3] FFN second layer, ms[4] combine.  n >= 5.
 */
SWITCH_API switch_status switch_stage_ms(switch_handle h, float* ms, int n);

/*
 * Expert parallelism: regroup the rows an expert-owning rank receives.  The Switch
 * Transformers card (ai-papers.xuzou.cn, 方法适配) shards the experts over the cores and
 * moves tokens with an all-to-all before the expert FFN and another after it.  With W ranks,
 * this rank owning El experts, every source rank s sends the blocks [El][R][row] of its
 * dispatched buffer for those experts (R = the source's expert block rows, G*C); counts
 * [W][El] int32 (device) holds the valid rows of each block (the source's expert_rows).
 *   inverse = 0: src = chunks [W][El][R][row] (as received), dst = packed [El][W*R][row]:
 *                dst[e][off(s, e) + i] = src[s][e][i] for i < counts[s][e], with
 *                off(s, e) = counts[0][e] + ... + counts[s-1][e] (sources in rank order);
 *                rows_out (device [El] int32, may be NULL) gets sum_s counts[s][e], the row
 *                counts for switch_expert_ffn on the packed buffer.
 *   inverse = 1: src = packed, dst = chunks: dst[s][e][i] = src[e][off(s, e) + i] (the
 *                expert outputs back into per-source chunks for the return all-to-all);
 *                rows_out must be NULL.
 * Rows past the counts are not written.  row bytes: a multiple of 16; src and dst 16-byte
 * aligned, not overlapping; a count outside 0 .. R counts as zero.  Asynchronous on
 * `stream`; argument errors return SWITCH_ERR_INVALID_ARG.
 */
SWITCH_API switch_status switch_ep_regroup(const void* src, void* dst, const int32_t* counts, int32_t* rows_out,
                                           int W, int El, int R, int row_bytes, int inverse, void* stream);

/* Number of kernels the last switch_forward on this handle launched. */
SWITCH_API int switch_last_launch_count(switch_handle h);

/*
 * switch_route without a handle, for callers that cannot allocate device memory once
 * they are running: code inside a CUDA graph that is already instantiated, a real-time
 * loop or driver where cudaMalloc could block or fail, an allocator-less embedding.
 * (No page of the method has a counterpart: it is a packaging choice of this library.)
 *
 * Same arguments and outputs as switch_route, with the config in place of a handle.
 * The routing kernels' scratch (split router weights, per-tile statistics, scan state,
 * error word) is one fixed 32 MiB device array inside the library, which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated: no cudaMalloc,
 * no cudaFree, no allocating library call; the call enqueues one cudaMemsetAsync of 16
 * bytes (clearing the error word and a counter) and the routing kernels on `stream`.
 *   - Every call looks up the array's device address in the current device's context
 *     (cudaGetSymbolAddress), so a call after a context reset (cudaDeviceReset) uses the
 *     new address.  The first call on a device also loads the library's device code there;
 *     make that first call before any stream capture.
 *   - Every call on a device shares the array and leaves its contents behind: two calls
 *     whose kernels overlap on the GPU (different streams, or concurrent graphs) race and
 *     give wrong results.  Serialise them.
 *   - A configuration whose scratch needs more than 32 MiB returns SWITCH_ERR_UNSUPPORTED.
 *     The scratch is about (12 E + 4) G ceil(T/128) + 6 E d + 4 E G C bytes (d rounded up to a
 *     multiple of 64, E up to the next multiple of the router's experts per CTA) with bfloat16
 *     activations (all five named workloads fit; 65536 tokens x 2048 experts needs 22 MiB),
 *     plus 4 G T E bytes of logits with float32 activations.  Invalid arguments return
 *     SWITCH_ERR_INVALID_ARG.
 *   - Device-side flags (a bounded wait that ran out, non-finite logits) stay in the array
 *     and are not reported; use switch_route on a handle when they are needed.
 *   - SWITCH_FLAG_TOP2 returns SWITCH_ERR_UNSUPPORTED (top-2 routing uses a logits buffer
 *     that only a handle's workspace holds).
 */
SWITCH_API switch_status switch_route_static(const switch_config* cfg, const void* x, const float* Wr,
                                  const float* br, const switch_route_out* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SWITCH_MOE_H */

/*
 * kda.h -- C ABI of libkda.so: the Kimi Delta Attention (KDA) decode and
 * spec-verify core of a Kimi-K3 layer on one GB300 GPU (sm_103a).
 *
 * One step runs, for every request r and head h, from the packed bf16
 * projection row to the gated-RMSNorm bf16 core output:
 *   1. split the row into q|k|v | out-gate | f_a | beta
 *      ("...cutedsl.kda.prepared" page, PreparedKda._operands);
 *   2. causal depthwise short conv of the q/k/v channels against the slot's
 *      conv window, SiLU, bf16 ("...mono.attention.kda" page, K1 docstring,
 *      kda_conv);
 *   3. z = f_b . f_a (bf16), g = lb * sigmoid(exp(A_log[h]) * (z + dt_bias)),
 *      beta = sigmoid(beta_logit) (K1 docstring, kda_gates: "f_b MFMA +
 *      lower-bound gate");
 *   4. q^ = q / |q| * 128^-0.5, k^ = k / |k| (l2norm, eps 1e-6 inside the root);
 *   5. gated delta rule on the 128 x 128 fp32 state:
 *      S <- diag(e^g) S;  S <- S + beta k^ (v - S^T k^)^T;  o = S^T q^
 *      (K1 docstring, kda_recur: "a state a token written");
 *   6. gated RMSNorm of bf16 o with the fp32 o_norm weight times
 *      sigmoid(out-gate) -> bf16 core_out (K1 docstring, kda_norm;
 *      PreparedKda.__init__: fp32 norm weight, eps = o_norm.eps).
 *
 * Layouts (D = 128 H, C = 3 D conv channels, W = conv width, SL = W - 1):
 *   projected   bf16 [rows, pitch], pitch >= 4D + 128 + H elements:
 *               cols [0,3D) q|k|v, [3D,4D) out-gate, [4D,4D+128) f_a,
 *               [4D+128, 4D+128+H) beta logits.
 *   conv_state  bf16 [pool, C, SL] (conv_dim_first = 1) or [pool, SL, C];
 *               each window holds the last SL inputs, oldest first.
 *   state_pool  fp32 [pool, H, 128 (v), 128 (k)]: one contiguous 64 KiB block
 *               per (slot, head), k contiguous within a 512-byte v row (bf16
 *               and 32 KiB / 256-byte rows after kda_set_state_dtype(BF16)).
 *   out         bf16 [rows, D].
 * Decode: L = 1, accepted = NULL, row b reads and writes slot slots[b].
 * Verify: rows = R L request-major (row = r L + t), slots [R, L] contiguous,
 *   accepted [R] in 1..L; request r starts from slot slots[r, accepted[r]-1]
 *   and after token t stores its state and conv window into slots[r, t]
 *   (PreparedKda.run: rows = batch // tokens, accepted[:rows]).
 * A slot of -1 in slots[r, 0] marks a padding request: no cache is read or
 *   written and its out rows are zero.  Duplicate slots within one step are
 *   undefined behaviour.
 *
 * All pointers passed to kda_step are DEVICE pointers on the device that was
 * current when the handle was prepared; the caller keeps ownership of every
 * buffer and keeps it alive until the step has completed on its stream.
 *
 * Thread safety: one handle may be used from one host thread at a time.
 * Steps enqueued on different streams against the same caches race.
 *
 * Around the core: kda_linear computes the layer's projections y = x . W^T
 * (in_proj in front of the step, o_proj after it), and kda_layer_plan_create
 * records in_proj -> step -> o_proj on fixed buffers as one CUDA graph.
 */
#ifndef KDA_H
#define KDA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kda_handle kda_handle;

/* Return codes. */
#define KDA_OK 0
#define KDA_EINVAL (-1) /* an argument is invalid; nothing was enqueued   */
#define KDA_ECUDA (-2)  /* a CUDA call or a launch failed                 */

/* Device error bits, accumulated in the handle's device error word and
 * returned (then cleared) by kda_check. */
#define KDA_ERR_SLOT 1u     /* a slot outside [0, pool) other than a padding -1: request skipped */
#define KDA_ERR_ACCEPTED 2u /* accepted[r] outside 1..L: request skipped                         */
#define KDA_ERR_TIMEOUT 4u  /* a bounded wait (about 1 s) for the start state gave up: see below */
#define KDA_ERR_DUPLICATE 8u /* KDA_DEBUG builds only: two rows of the step write the same slot    */

/* KDA_ERR_TIMEOUT: the step reads a (request, head)'s start state in two
 * halves of 64 v rows, each warp waiting (about 1 s at most) for the half it
 * needs.  A warp that gives up writes none of its state rows; the warps whose
 * copies landed may already have written theirs to slots[r, t] (decode:
 * slots[b]).  The out rows of a CTA that saw a wait give up are not written
 * (decode of two rows or more serves rows 2p and 2p + 1 of a head in one CTA,
 * so both rows' out stay unwritten), and the conv
 * windows, stored before the state is needed, are.  Treat the requests' caches
 * as undefined after a timeout. */

/* Decode of two rows or more (L = 1, rows >= 2, one CTA a (request, head))
 * runs rows 2p and 2p + 1 of a head in one CTA: the rows share their load
 * round trips and the head's f_b; with a bf16 pool their two 32 KiB states sit
 * side by side, with an fp32 pool the second row's halves are loaded into the
 * one 64 KiB state buffer as the first row's passes free them.  Each row's
 * results are those of one row a CTA. */

/* Maximum verify tokens per request. */
#define KDA_MAX_TOKENS 8

/*
 * kda_prepare -- copy the layer's weights into handle-owned device buffers,
 * re-laying out the conv weight [3D, 1, W] so that each channel's W taps sit
 * right-aligned in four bf16 (one 8-byte word a channel), as PreparedKda.__init__
 * re-lays its conv weight out once for its kernel (decode_conv_weight,
 * "...cutedsl.kda.prepared" page), and taking the Euclidean norm of each f_b
 * row.
 *
 *   heads             H >= 1 (D = 128 H)
 *   conv_width        W in 2..4
 *   conv_w            device bf16 [3D, 1, W]
 *   bias              device bf16 [3D], or NULL for no conv bias
 *   f_b               device bf16 [D, 128]
 *   A_log             device fp32 [H]
 *   dt_bias           device fp32 [D]
 *   o_norm            device fp32 [128] (shared by all heads)
 *   gate_lower_bound  lb < 0 of the gate (the model's gate_lower_bound)
 *   eps               o_norm epsilon (> 0)
 *   out               receives the handle
 *
 * Synchronous on the device that is current.  The source buffers may be
 * freed once it returns.  Returns KDA_OK, KDA_EINVAL (NULL pointer, heads < 1,
 * W outside 2..4, eps <= 0, a misaligned pointer) or KDA_ECUDA.
 */
int kda_prepare(int heads, int conv_width, const void* conv_w, const void* bias, const void* f_b,
                const float* A_log, const float* dt_bias, const float* o_norm,
                float gate_lower_bound, float eps, kda_handle** out);

/*
 * kda_step -- enqueue one decode or verify step on `cuda_stream` (a
 * cudaStream_t; NULL = the legacy default stream) without a host sync.
 *
 *   projected       device bf16 [rows, pitch]                 (read)
 *   rows, pitch     rows >= 0, a multiple of L; pitch >= 4D + 128 + H
 *   conv_state      device bf16 windows, see layouts          (read + written)
 *   conv_dim_first  1: [pool, 3D, W-1]; 0: [pool, W-1, 3D]
 *   state_pool      device fp32 (or bf16, see kda_set_state_dtype) [pool, H, 128, 128],
 *                   16-byte aligned (read + written)
 *   pool_slots      pool size (slots)
 *   slots           device int32 [rows]
 *   L               1..KDA_MAX_TOKENS tokens per request
 *   accepted        device int32 [rows / L] for verify, NULL for decode (L must be 1)
 *   out             device bf16 [rows, D], 8-byte aligned     (written)
 *
 * rows = 0 enqueues nothing.  Returns KDA_OK, KDA_EINVAL (NULL handle or
 * buffer, bad sizes, L outside 1..8, rows % L != 0, L > 1 without accepted,
 * misalignment) or KDA_ECUDA (launch failure).  Bad slot / accepted VALUES
 * are found on the device: they set KDA_ERR_* bits in the handle's error
 * word and the request is skipped (nothing written for it); they never trap.
 */
int kda_step(kda_handle* handle, const void* projected, long long rows, long long pitch,
             void* conv_state, int conv_dim_first, float* state_pool, long long pool_slots,
             const int* slots, int L, const int* accepted, void* out, void* cuda_stream);

/*
 * kda_check -- synchronise `cuda_stream`, then read and clear the handle's
 * device error word into *device_flags (may be NULL).  Returns KDA_OK,
 * KDA_EINVAL (NULL handle) or KDA_ECUDA (the stream reported an error).
 */
int kda_check(kda_handle* handle, void* cuda_stream, unsigned* device_flags);

/*
 * kda_set_gate_mode -- choose the decay gate the handle's steps compute.  The
 * K1 page names a "lower-bound gate" and PreparedKda takes gate_lower_bound
 * (lb) without giving the formula, so both forms it admits are offered:
 *   KDA_GATE_SIGMOID  (default)  g = lb * sigmoid(e^{A_log[h]} (z + dt_bias[c])), in (lb, 0)
 *   KDA_GATE_SOFTPLUS            g = max(-e^{A_log[h]} softplus(z + dt_bias[c]), lb), in [lb, 0)
 * Applies to steps enqueued after the call.  Returns KDA_OK, or KDA_EINVAL
 * for a NULL handle or an unknown mode.  No CUDA call.
 */
#define KDA_GATE_SIGMOID 0
#define KDA_GATE_SOFTPLUS 1
int kda_set_gate_mode(kda_handle* handle, int mode);

/*
 * kda_set_state_dtype -- the storage type of the state pool the handle's
 * steps read and write (the layout stays [pool, H, 128 (v), 128 (k)]):
 *   KDA_STATE_F32  (default)  fp32, 64 KiB a (slot, head)
 *   KDA_STATE_BF16            bf16, 32 KiB a (slot, head): the step widens the
 *                             start state exactly, computes in fp32 and rounds
 *                             each stored state to bf16 (nearest even); half
 *                             the state bytes, at bf16 precision of the cache
 * For KDA_STATE_BF16 pass the bf16 pool as kda_step's state_pool (same
 * 16-byte alignment rule).  Applies to steps enqueued (and plans
 * made) after the call.  Returns KDA_OK, or KDA_EINVAL for a NULL handle or an unknown
 * type.  No CUDA call.
 */
#define KDA_STATE_F32 0
#define KDA_STATE_BF16 1
int kda_set_state_dtype(kda_handle* handle, int dtype);

/*
 * kda_set_v_split -- how many CTAs share one (request, head) of a step: 1
 * (default), or 2 in a thread-block cluster, each owning 64 of the 128 v rows
 * of the state (one recurrence pass, half the state copy and half the
 * outputs; both run the conv, the gates and the l2norm, and they swap their
 * halves of o through distributed shared memory for the RMSNorm).  The K1
 * page splits a head's state rows over several workers (8 v-chunks of 16
 * rows); here the split is a launch option, and on GB300 it is slower on every
 * workload measured (the halves repeat the prologue, and the doubled grid of
 * three-per-SM CTAs needs more waves), so it is off unless asked for.  It
 * applies to the window-first conv layout (conv_dim_first = 1); the other
 * layout always runs one CTA.  Decode under v_split 2 runs one row a cluster
 * instead of two rows a CTA.  Results are the same either
 * way.  Applies to steps enqueued (and plans made) after the call.  Returns
 * KDA_OK, or KDA_EINVAL for a NULL handle or another value.  No CUDA call.
 */
int kda_set_v_split(kda_handle* handle, int v_split);

/*
 * Launch plans.  A plan records one kda_step, with exactly these arguments,
 * as a CUDA graph (captured once on a private stream and instantiated), so
 * that each later step is a single graph launch: the analogue of the
 * per-shape prepared executables of PreparedKda (prepare_caches / run on the
 * "...cutedsl.kda.prepared" page), for small batches where the launch costs
 * as much as the kernel.  The pointers, sizes and the handle's gate mode are
 * fixed when the plan is made; the buffers' contents may change between
 * launches (write the next step's inputs into the same buffers).  The
 * buffers and the handle must outlive the plan.
 *
 * kda_plan_create -- arguments as kda_step (no stream).  Returns KDA_OK and
 *   *plan, KDA_EINVAL (the arguments kda_step rejects, or plan == NULL) or
 *   KDA_ECUDA.
 * kda_plan_launch -- enqueue the recorded step on cuda_stream (NULL = the
 *   legacy default stream).  Returns KDA_OK, KDA_EINVAL (NULL plan) or KDA_ECUDA.
 * kda_plan_destroy -- free the plan (NULL is a no-op).
 */
typedef struct kda_plan kda_plan;
int kda_plan_create(kda_handle* handle, const void* projected, long long rows, long long pitch,
                    void* conv_state, int conv_dim_first, float* state_pool, long long pool_slots,
                    const int* slots, int L, const int* accepted, void* out, kda_plan** plan);
int kda_plan_launch(kda_plan* plan, void* cuda_stream);

/*
 * kda_layer_plan_create -- one decode / verify step of the whole layer as a
 * CUDA graph: in_proj (kda_linear: x [rows, hidden] (row stride ldx) .
 * w_in [pitch, hidden]^T -> projected [rows, pitch]), kda_step (projected ->
 * core_out [rows, D], the caches updated as by kda_step), o_proj (kda_linear:
 * core_out . w_o [hidden, D]^T -> y [rows, hidden], row stride ldy).  The K1
 * page's gemv stage in front of kda_pre and the K2a page's o_proj after it,
 * without the all-reduce.  projected and core_out are the caller's
 * intermediate buffers (contiguous); every pointer is the caller's, must stay
 * valid while the plan exists, and is read or written at each launch; the
 * handle's gate mode and state dtype at creation are baked in.  pdl is a
 * mask of the edges launched as programmatic dependents (the kernel may start
 * while the previous one finishes; it loads what does not depend on its
 * predecessor, then waits for it before reading its output):
 * KDA_PDL_STEP (in_proj -> kda_step), KDA_PDL_O_PROJ (kda_step -> o_proj);
 * 0 = plain stream order.  Validation and error codes as kda_step and
 * kda_linear; launch with kda_plan_launch, free with kda_plan_destroy.
 */
#define KDA_PDL_STEP 1
#define KDA_PDL_O_PROJ 2
int kda_layer_plan_create(kda_handle* handle, const void* x, long long rows, long long ldx, long long hidden,
                          const void* w_in, void* projected, long long pitch, void* conv_state, int conv_dim_first,
                          float* state_pool, long long pool_slots, const int* slots, int L, const int* accepted,
                          void* core_out, const void* w_o, void* y, long long ldy, int pdl, kda_plan** plan);
void kda_plan_destroy(kda_plan* plan);

/*
 * kda_linear -- the layer's projections around the core: y = x . W^T with
 * x [rows, K] (row stride ldx), W [N, K] row-major (a torch Linear weight:
 * out_features x in_features), y [rows, N] (row stride ldy); bf16 in and out
 * (nearest even), fp32 accumulation.  in_proj (x [rows, 7168] -> the packed
 * projection row, the K1 page's gemv in front of kda_pre) and o_proj
 * (core_out [rows, D] -> [rows, 7168], the K2a page's GEMV after the core)
 * are both this product.  Device pointers; x and W 16-byte aligned with
 * ldx % 8 == 0, y 2-byte aligned; K a multiple of 8 (16-byte rows).  x, W and y are the
 * caller's and are not retained; y must not overlap x or W.
 * Enqueued on cuda_stream with no host sync.  Returns KDA_OK (rows = 0
 * launches nothing), KDA_EINVAL or KDA_ECUDA.
 */
int kda_linear(const void* x, long long rows, long long ldx, const void* w, long long N, long long K, void* y,
               long long ldy, void* cuda_stream);

/*
 * kda_linear_check -- synchronise `cuda_stream`, then read and clear the
 * projections' device error bits into *device_flags: KDA_ERR_TIMEOUT if a
 * kda_linear launch since the last check gave up waiting (about a second) for
 * its own bulk copies, in which case that launch's y is not meaningful.
 * Returns KDA_OK, KDA_EINVAL (device_flags NULL) or KDA_ECUDA.
 */
int kda_linear_check(void* cuda_stream, unsigned* device_flags);

/* kda_destroy -- free the handle's device buffers (synchronises the device). NULL is a no-op. */
void kda_destroy(kda_handle* handle);

/* kda_strerror -- a static string for a return code. */
const char* kda_strerror(int code);

/*
 * kda_launch_info -- the launch shape kda_step uses for L tokens (one CTA per
 * (request, head), fp32 state pool, window-first conv cache): threads per
 * CTA, dynamic shared memory bytes per CTA and the resident CTAs per SM the
 * occupancy calculator reports (each output pointer may be NULL).  A decode of
 * two rows or more runs two rows of one head a CTA in a second kernel with the
 * same threads and residency and a little more shared memory (the second row's
 * norms and gates); L = 1 reports the one-row kernel.  Returns
 * KDA_OK, KDA_EINVAL (L outside 1..KDA_MAX_TOKENS) or KDA_ECUDA.  Needs a
 * current CUDA device when ctas_per_sm is not NULL.
 */
int kda_launch_info(int L, int* threads, int* smem_bytes, int* ctas_per_sm);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */

/*
 * moe.h -- C ABI of the GB300 (sm_103a) local Mixture-of-Experts forward and
 * its first-order backward.
 *
 * The pipeline follows the ruDNN user guide ("ruDNN Benutzerhandbuch"),
 * section 3 "MoE-Workflow": router logits -> FP32 softmax / top-k ->
 * capacity-free dispatch -> bias-free SwiGLU experts -> weighted combine.
 * The staged calls mirror section 6 "MoE aufrufen" (route, dispatch,
 * forward_dispatched, combine) and the fused call mirrors
 * SwiGluExperts::forward in the ruDNN 0.1.25 source view of src/moe/experts.rs.
 *
 * Conventions for every call
 *   - Tensors are caller-owned, dense, row-major DEVICE pointers on the
 *     current CUDA device (unless a parameter says "host").  Floating-point
 *     tensors other than logits/weights must be 16-byte aligned; workspaces
 *     must be 256-byte aligned.  The library never allocates device memory
 *     during a call and never frees caller memory.
 *   - Work is enqueued on `stream` and the call returns without waiting for
 *     the device (except moe_get_device_status, which synchronises that
 *     stream).  Calls are therefore capturable in a CUDA graph, except
 *     moe_get_device_status, moe_forward_host with pageable memory and the
 *     moe_host_pipeline_* calls (which own their streams).
 *   - Shapes are element counts.  T = tokens, E = experts, k = top_k,
 *     H = hidden size, I = expert intermediate size, N = T*k dispatched rows.
 *   - Every call returns a moe_status.  On any status other than MOE_OK,
 *     nothing was enqueued, and moe_last_error() returns a message for the
 *     calling thread.  T == 0 is valid and enqueues nothing.
 *   - Limits: 1 <= E <= 1024, 1 <= k <= min(E, 64), N < 2^31, H and I in
 *     [1, 2^20].  Outside them MOE_ERR_UNSUPPORTED (k outside [1, E] is
 *     MOE_ERR_INVALID_ARG, as the routing contract requires 1 <= top_k <= E).
 *   - There is no CPU fallback: every step runs in this library's CUDA kernels.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad top_k, small workspace, misalignment */
    MOE_ERR_SHAPE = 2,          /* dimension zero or mismatched, element count overflow */
    MOE_ERR_DTYPE = 3,          /* dtype not F32/F16/BF16 or operands disagree */
    MOE_ERR_UNSUPPORTED = 4,    /* outside the stated limits */
    MOE_ERR_CUDA = 5,           /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_INVALID_INDEX = 6,  /* device-side: an expert index >= E reached dispatch */
    MOE_ERR_DEVICE_TIMEOUT = 7  /* device-side: a bounded wait inside a kernel gave up */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_F16 = 1, MOE_BF16 = 2 } moe_dtype;

typedef struct moe_experts* moe_experts_t;

/* Message for the last failing call on this thread ("" if none).  The
 * pointer stays valid until the next call on the same thread. */
const char* moe_last_error(void);

/* Static name of a status code. */
const char* moe_status_string(moe_status status);

/* ------------------------------------------------------------------------
 * Routing.  ruDNN Benutzerhandbuch, section 4 "Routing-Vertrag".
 *
 * For each of the T rows of `logits` [T,E] (dtype F32, F16 or BF16, any
 * element alignment): softmax over all E experts in FP32; the top_k experts
 * by logit (ties go to the lower expert id; +0 and -0 are equal), listed in
 * descending weight; weights = the selected softmax values, divided by their
 * FP32 sum (added in slot order) when `renormalize` is non-zero, then rounded
 * to the logits dtype (round to nearest even).  A row holding a NaN, a +inf,
 * or only -inf entries gets idx = 0..top_k-1 and NaN weights.
 *
 *   idx          out [T,top_k] uint32 (device)
 *   weights      out [T,top_k] in the logits dtype (device)
 *   weights_f32  out [T,top_k] float, the same weights before the final
 *                rounding (device; may be NULL)
 * ---------------------------------------------------------------------- */
moe_status moe_route(const void* logits, moe_dtype logits_dtype, int64_t T, int64_t E,
                     int32_t top_k, int renormalize, uint32_t* idx, void* weights,
                     float* weights_f32, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Sigmoid group-limited routing.  ruDNN Benutzerhandbuch, section 10
 * "Gruppenbeschraenktes Sigmoid-MoE-Routing" (GroupRoutingOptions).
 *
 * Per row: scores s_e = sigmoid(logit_e); corrected scores c_e = s_e +
 * bias_e (bias: optional FP32 [E] device array; it only affects the
 * selection); the E experts form `groups` contiguous groups of E/groups; a
 * group scores max c over its experts, or the sum of its two largest c when
 * group_top_two != 0; the `selected_groups` best groups are kept and top_k
 * experts are chosen among their experts by c.  Ties go to the lower id.
 * Selection runs in FP32 with the correctly rounded FP32 sigmoid.  Weights
 * are s of the chosen experts, divided by their FP32 sum (slot order) when
 * renormalize != 0, times scale, rounded to the logits dtype; idx lists the
 * chosen experts in descending c.  A row holding a NaN logit (or NaN
 * corrected score) gets idx = 0..top_k-1 and NaN weights.
 * Rules (MOE_ERR_INVALID_ARG unless noted): 1 <= E <= 1024
 * (MOE_ERR_UNSUPPORTED above), 1 <= groups <= 128, E % groups == 0,
 * 1 <= selected_groups <= groups, 1 <= top_k <= 64 and top_k <=
 * selected_groups * E/groups, group_top_two needs E/groups >= 2, scale
 * finite and > 0.  Outputs as for moe_route.
 * With F16/BF16 logits the sigmoid is read from a device table of all 65536
 * patterns.  The first such call on a device enqueues the table's fill on
 * its stream, and later calls on other streams wait for that fill (a stream
 * event, no host synchronisation).  A stream being captured into a CUDA
 * graph gets a fill of its own in the graph.
 * ---------------------------------------------------------------------- */
typedef struct {
    int32_t top_k;
    int32_t groups;
    int32_t selected_groups;
    int32_t group_top_two;
    int32_t renormalize;
    float scale;
} moe_group_routing_options;

moe_status moe_route_sigmoid_grouped(const void* logits, moe_dtype logits_dtype, int64_t T,
                                     int64_t E, const float* bias,
                                     const moe_group_routing_options* options, uint32_t* idx,
                                     void* weights, float* weights_f32, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Dispatch.  ruDNN Benutzerhandbuch, section 5 "Expertengewichte und
 * Verteilung" (no token dropped; a stored map restores token order) and
 * the DispatchedTokens invariant in src/moe/experts.rs ("complete, monotone
 * expert segments without token dropping").
 *
 * Slot s = t*top_k + j holds expert idx[t,j].  Rows are grouped into
 * contiguous per-expert segments: offsets[e]..offsets[e+1] holds expert e's
 * slots in ascending s (a stable sort of the slots by expert id, so the
 * result is bit-reproducible).  For dispatched row r:
 *   perm[r] = s, row_experts[r] = e, x_disp[r,:] = x[s / top_k, :].
 *
 *   idx          in  [T,top_k] uint32 (device)
 *   x            in  [T,H] (device; may be NULL, then x_disp must be NULL)
 *   offsets      out [E+1] uint32;  row_experts, perm  out [T*top_k] uint32
 *   x_disp       out [T*top_k, H] in x's dtype (may be NULL)
 *   workspace    device scratch of moe_dispatch_workspace_size() bytes; its
 *                first word receives the device status (see
 *                moe_get_device_status).
 * An index >= E is not dispatched (no out-of-bounds access): offsets[E] then
 * counts only valid slots, the unused tail of perm/row_experts is set to
 * 0xFFFFFFFF and the device status becomes MOE_ERR_INVALID_INDEX.
 * ---------------------------------------------------------------------- */
size_t moe_dispatch_workspace_size(int64_t T, int64_t E, int32_t top_k);
moe_status moe_dispatch(const uint32_t* idx, int64_t T, int64_t E, int32_t top_k,
                        const void* x, moe_dtype x_dtype, int64_t H,
                        uint32_t* offsets, uint32_t* row_experts, uint32_t* perm,
                        void* x_disp, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* Dispatch for callers that can neither allocate device memory nor lend
 * this library a workspace, for example a layer plugin inside an inference
 * engine that only receives the layer's own tensors, or a serving loop that
 * fixed its memory plan at start-up and must not trigger cudaMalloc later
 * (an allocation can synchronise the whole device).  The pages have no
 * counterpart to this call: it exists for those callers only.
 *
 * Same arguments, results and ordering as moe_dispatch, without the
 * workspace.  The dispatch scratch (chunk counts and bases) lives in a fixed
 * 2 MiB device array inside the library, which every GPU that loads the
 * library holds until the process exits.  Problems needing more scratch than
 * that (dispatch scratch = 4*ceil(T/256)*(2E+1) bytes, rounded up; e.g.
 * T <= 65,280 at E = 1024, T <= ~1M at E = 64) get MOE_ERR_UNSUPPORTED with a
 * message.  The call allocates nothing.
 *
 * The first call in a CUDA context (for runtime-API callers: the first call
 * on each device) looks up the array's device address with that device
 * current and caches it under the context's unique id; make that first call
 * before any stream capture.  A context created later on the same device
 * (after cudaDeviceReset, or a driver-API context) gets its own lookup.  All calls share the array and it keeps the last call's contents;
 * nothing in it needs clearing because each call writes every entry it reads.
 * Calls whose kernels overlap on the GPU (unordered streams) race on the
 * array and give wrong results.  There is no device status word: an index
 * >= E shows up as offsets[E] < T*top_k and 0xFFFFFFFF at the tail of perm. */
moe_status moe_dispatch_noalloc(const uint32_t* idx, int64_t T, int64_t E, int32_t top_k,
                                const void* x, moe_dtype x_dtype, int64_t H,
                                uint32_t* offsets, uint32_t* row_experts, uint32_t* perm,
                                void* x_disp, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Experts.  SwiGluExperts::new in src/moe/experts.rs and the user guide,
 * section 5: bias-free gate and up [E,I,H], down [E,H,I], one float dtype,
 * one device, every dimension non-zero.
 *
 * The handle does not own the weights: they must stay alive and unchanged
 * while the handle is used.  It records shapes and prebuilt TMA descriptors
 * and is reusable across batches.  Errors: MOE_ERR_DTYPE for a bad dtype,
 * MOE_ERR_SHAPE for a zero dimension or an element-count overflow,
 * MOE_ERR_INVALID_ARG for null or misaligned pointers or pointers that are
 * not device memory of one device.
 * ---------------------------------------------------------------------- */
moe_status moe_experts_create(const void* gate, const void* up, const void* down,
                              moe_dtype dtype, int64_t E, int64_t I, int64_t H,
                              moe_experts_t* out);
void moe_experts_destroy(moe_experts_t experts);

/* SwiGluExperts::forward_dispatched_with_strategy in src/moe/experts.rs:
 * for each dispatched row r of expert e (offsets[e] <= r < offsets[e+1]):
 *   g = x_disp[r] . W_gate[e]^T, u = x_disp[r] . W_up[e]^T,
 *   h = silu(g) * u  (rounded to the weight dtype),
 *   expert_out[r] = h . W_down[e]^T  (FP32 accumulation, stored in the
 *   weight dtype).
 * x_disp [N,H] and expert_out [N,H] are in the weight dtype; offsets [E+1]
 * on the device (never read by the host), non-decreasing with offsets[E] <=
 * N.  Rows at or beyond offsets[E] are not written.  The call checks the
 * offsets on the device: an entry below its predecessor or above N is
 * clamped (to the predecessor, or to N) and MOE_ERR_INVALID_INDEX is set in
 * the workspace status word (moe_get_device_status); the outputs are then
 * undefined, and no access leaves the buffers.  workspace:
 * moe_experts_workspace_size(experts, N) bytes. */
size_t moe_experts_workspace_size(moe_experts_t experts, int64_t N);
moe_status moe_experts_forward(moe_experts_t experts, const void* x_disp, int64_t N,
                               const uint32_t* offsets, void* expert_out,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Combine.  User guide, section 6: the dispatch map restores token order and
 * the expert outputs are summed with the routing weights:
 *   y[t,:] = sum_{j=0..k-1} weights[t,j] * expert_out[r(t,j), :]
 * where r(t,j) is the row with perm[r] = t*k+j; the sum runs in ascending j
 * with FP32 accumulation and is rounded once to `dtype`.  A slot that no row
 * holds makes y[t,:] NaN.
 *   expert_out [T*k, H] and y [T,H] in `dtype`; weights [T,k] in
 *   `weights_dtype`; perm [T*k] uint32.  workspace:
 *   moe_combine_workspace_size(T, k) bytes.
 * ---------------------------------------------------------------------- */
size_t moe_combine_workspace_size(int64_t T, int32_t top_k);
moe_status moe_combine(const void* expert_out, moe_dtype dtype, const uint32_t* perm,
                       const void* weights, moe_dtype weights_dtype, int64_t T,
                       int32_t top_k, int64_t H, void* y, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Fused forward.  SwiGluExperts::forward in src/moe/experts.rs: route ->
 * dispatch -> experts -> combine for precomputed logits, all on `stream`
 * with no host synchronisation.  x [T,H] and y [T,H] in the weight dtype;
 * logits [T,E] in F32/F16/BF16.  The down projection's epilogue multiplies
 * each row by its routing weight and stores it at its token slot; a final
 * pass sums each token's k slots in ascending j.  Results equal the staged
 * calls up to the rounding of the weighted slot values.
 * workspace: moe_forward_workspace_size(...) bytes (intermediates live there;
 * see moe_forward_layout).
 * ---------------------------------------------------------------------- */
size_t moe_forward_workspace_size(moe_experts_t experts, int64_t T, int32_t top_k,
                                  moe_dtype logits_dtype);
moe_status moe_forward(moe_experts_t experts, const void* x, const void* logits,
                       moe_dtype logits_dtype, int64_t T, int32_t top_k, int renormalize,
                       void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* SwiGluExperts::forward_sigmoid_grouped in src/moe/experts.rs: the fused
 * forward with moe_route_sigmoid_grouped as its routing step (user guide,
 * section 10).  Same buffers and workspace as moe_forward with
 * top_k = options->top_k (moe_forward_workspace_size applies). */
moe_status moe_forward_sigmoid_grouped(moe_experts_t experts, const void* x, const void* logits,
                                       moe_dtype logits_dtype, int64_t T, const float* bias,
                                       const moe_group_routing_options* options, void* y,
                                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Same as moe_forward, and records CUDA events on `stream` at the stage
 * boundaries: events[0] before routing, [1] after routing, [2] after
 * dispatch, [3] after the gate/up projection, [4] after the down projection,
 * [5] after the combine.  `events` holds n_events (>= 6) cudaEvent_t handles
 * created by the caller, or NULL for a boundary that is not to be recorded
 * (each record sits between two kernels of the forward, so record only the
 * boundaries you need); the library records them and nothing else. */
moe_status moe_forward_timed(moe_experts_t experts, const void* x, const void* logits,
                             moe_dtype logits_dtype, int64_t T, int32_t top_k, int renormalize,
                             void* y, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream, void* const* events, int n_events);

/* Same computation with HOST buffers: x_host [T,H], logits_host [T,E] and
 * y_host [T,H] live in host memory (page-locked memory makes the copies
 * asynchronous).  The call enqueues the host-to-device copies into staging
 * space inside the workspace, the forward, and the device-to-host copy of y;
 * the caller synchronises `stream` before reading y_host.  workspace:
 * moe_forward_host_workspace_size(...) bytes. */
size_t moe_forward_host_workspace_size(moe_experts_t experts, int64_t T, int32_t top_k,
                                       moe_dtype logits_dtype);
moe_status moe_forward_host(moe_experts_t experts, const void* x_host, const void* logits_host,
                            moe_dtype logits_dtype, int64_t T, int32_t top_k, int renormalize,
                            void* y_host, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Pipelined host-buffer forward for a stream of batches (serving).  Not a
 * call of the pages: their forward takes device tensors (user guide
 * section 6); this overlaps the host copies of consecutive batches with the
 * forward of the batch between them.
 *   - The pipeline owns `depth` (2..4) device staging slots for x, logits and
 *     y, one host-to-device and one device-to-host stream, and CUDA events.
 *     Its device memory is the caller's workspace of
 *     moe_host_pipeline_workspace_size(...) bytes (256-byte aligned), which
 *     must outlive the pipeline.  The forward itself runs on `stream`, given
 *     at creation.
 *   - moe_host_pipeline_submit(p, x_host, logits_host, y_host, T), T <= T_max:
 *     enqueues the copy of x and logits into the next slot (after that slot's
 *     previous forward has consumed it), the forward on `stream`, and the copy
 *     of y back to y_host (after the forward).  It returns without waiting.
 *     Host buffers should be pinned for the copies to overlap; they must stay
 *     valid, and y_host unread, until moe_host_pipeline_sync returns.
 *   - moe_host_pipeline_sync waits for every submitted batch.
 *   - moe_host_pipeline_destroy synchronises and frees the streams and events.
 * Results are bitwise those of moe_forward on the same batch.  The device
 * status word is the one at the start of the workspace.
 * Errors: a NULL handle, output or pipeline, depth outside 2..4, a bad dtype
 * or workspace -> MOE_ERR_INVALID_ARG / MOE_ERR_DTYPE (nothing created);
 * T outside 0..=T_max in submit -> MOE_ERR_SHAPE (nothing enqueued; T == 0 is
 * a no-op); stream or event creation failure -> MOE_ERR_CUDA.  A pipeline is
 * used from one host thread at a time.  destroy(NULL) is a no-op. */
typedef struct moe_host_pipeline* moe_host_pipeline_t;
size_t moe_host_pipeline_workspace_size(moe_experts_t experts, int64_t T_max, int32_t top_k,
                                        moe_dtype logits_dtype, int depth);
moe_status moe_host_pipeline_create(moe_experts_t experts, int64_t T_max, int32_t top_k,
                                    moe_dtype logits_dtype, int renormalize, int depth,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream,
                                    moe_host_pipeline_t* out);
moe_status moe_host_pipeline_submit(moe_host_pipeline_t pipeline, const void* x_host,
                                    const void* logits_host, void* y_host, int64_t T);
moe_status moe_host_pipeline_sync(moe_host_pipeline_t pipeline);
moe_status moe_host_pipeline_destroy(moe_host_pipeline_t pipeline);

/* Byte offsets of the intermediates moe_forward leaves in its workspace, so
 * that a caller can inspect them after the stream has finished:
 *   idx [T,k] u32, weights [T,k] logits dtype, offsets [E+1] u32,
 *   perm [T*k] u32, x_disp [T*k,H], h [T*k,I], slots [T*k,H] (weighted
 *   expert outputs at token-slot order), slot_row [T*k] u32 (the dispatched
 *   row of slot t*k+j, the inverse of perm; written only when a row of x is
 *   a whole number of 16-byte vectors).  Returns MOE_ERR_INVALID_ARG for a
 *   null handle or output. */
typedef struct {
    size_t idx, weights, offsets, perm, x_disp, h, slots, slot_row, total;
} moe_forward_layout_t;
moe_status moe_forward_layout(moe_experts_t experts, int64_t T, int32_t top_k,
                              moe_dtype logits_dtype, moe_forward_layout_t* out);

/* Reads the device status word at the start of `workspace` after
 * synchronising `stream`: MOE_OK, MOE_ERR_INVALID_INDEX (dispatch met an
 * index >= E, or a staged expert call met offsets that are not
 * non-decreasing within N) or MOE_ERR_DEVICE_TIMEOUT (a kernel's bounded wait
 * expired and the kernel returned early; its outputs are undefined).
 * MOE_ERR_CUDA if the synchronisation itself fails. */
moe_status moe_get_device_status(const void* workspace, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * First-order training backward.  ruDNN Benutzerhandbuch, section 12
 * "MoE-Training erster Ordnung", and ExpertTrainingCache::backward in
 * src/moe/experts.rs.  All calls are deterministic (fixed summation orders).
 * ---------------------------------------------------------------------- */

/* Combine backward: for the row r holding slot s = t*top_k + j (perm[r] = s),
 *   dexpert[r,:] = weights[s] * dy[t,:]            ([T*k, H], in `dtype`)
 *   dweights[s]  = sum_h expert_out[r,h] * dy[t,h] ([T,k], FP32)
 * Rows holding no slot (perm[r] = 0xFFFFFFFF, or any entry >= T*top_k) get
 * dexpert = 0; slots held by no row get NaN. */
moe_status moe_combine_backward(const void* expert_out, moe_dtype dtype, const uint32_t* perm,
                                const void* weights, moe_dtype weights_dtype, const void* dy,
                                int64_t T, int32_t top_k, int64_t H, void* dexpert,
                                float* dweights, cudaStream_t stream);

/* Dispatch backward: dx[t,:] = sum_j dinput[r(t,j),:] (ascending j, FP32
 * accumulation, rounded once to `dtype`), without routing weights.  A slot no
 * row holds makes dx[t,:] NaN.  workspace: moe_combine_workspace_size(T, k). */
moe_status moe_dispatch_backward(const void* dinput, moe_dtype dtype, const uint32_t* perm,
                                 int64_t T, int32_t top_k, int64_t H, void* dx, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/* Expert backward for dispatched rows x_disp [N,H] (as for
 * moe_experts_forward) and the gradient of the expert outputs dout [N,H]:
 *   g = x W_gate^T, u = x W_up^T (recomputed), a = silu(g) u,
 *   da = dout W_down, dg = da u silu'(g), du = da silu(g),
 *   dinput = dg W_gate + du W_up        ([N,H], weight dtype)
 *   ddown = sum_r dout_r^T a_r, dgate = sum_r dg_r^T x_r, dup = sum_r du_r^T x_r
 * (FP32 [E,H,I], [E,I,H], [E,I,H]; experts without rows get zeros).
 * FP32 accumulation throughout.  offsets as for moe_experts_forward, checked
 * and clamped on the device in the same way (MOE_ERR_INVALID_INDEX in the
 * workspace status word).  workspace:
 * moe_experts_backward_workspace_size(experts, N) bytes (enough for every
 * strategy of moe_experts_backward_with_strategy). */
size_t moe_experts_backward_workspace_size(moe_experts_t experts, int64_t N);
moe_status moe_experts_backward(moe_experts_t experts, const void* x_disp, int64_t N,
                                const uint32_t* offsets, const void* dout, void* dinput,
                                float* dgate, float* dup, float* ddown, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* The same backward with an explicit strategy (section 12: the expert backward
 * takes Scalar, Auto or TensorCore, independently of the forward's strategy;
 * moe_experts_backward above is Scalar, the pages' default).
 *   MOE_BWD_SCALAR      FP32 CUDA-core kernels; g, u, a, dg, du kept in FP32.
 *   MOE_BWD_TENSOR_CORE tcgen05 kernels, F16/BF16 experts only (otherwise
 *                       MOE_ERR_UNSUPPORTED, nothing enqueued).  As in the
 *                       pages' training cache, a, dg and du are held in the
 *                       weight dtype and are the 16-bit operands of dinput and
 *                       of the weight gradients; g and u stay FP32.  FP32
 *                       accumulation; weight gradients FP32.
 *   MOE_BWD_AUTO        TENSOR_CORE where the experts support it, else SCALAR
 *                       (a capability choice only: errors are returned).
 * The tensor-core path's waits are bounded; a timeout sets the device status
 * word to MOE_ERR_DEVICE_TIMEOUT (moe_get_device_status on the workspace). */
enum { MOE_BWD_SCALAR = 0, MOE_BWD_AUTO = 1, MOE_BWD_TENSOR_CORE = 2 };
moe_status moe_experts_backward_with_strategy(moe_experts_t experts, const void* x_disp, int64_t N,
                                              const uint32_t* offsets, const void* dout,
                                              void* dinput, float* dgate, float* dup, float* ddown,
                                              int strategy, void* workspace,
                                              size_t workspace_bytes, cudaStream_t stream);

/* Router weights of a fixed selection idx [T,k] (section 12
 * selected_router_weights), FP32 [T,k]: scoring 0 = softmax over all E,
 * 1 = sigmoid of the selected logits; divided by their sum when renormalize
 * != 0; times scale (finite, > 0).  Repeated indices gather; an index >= E
 * makes the row NaN.  1 <= top_k <= min(E, 64). */
moe_status moe_router_weights(const void* logits, moe_dtype logits_dtype, const uint32_t* idx,
                              int64_t T, int64_t E, int32_t top_k, int scoring, int renormalize,
                              float scale, float* weights, cudaStream_t stream);

/* Gradient of those weights with respect to the logits (section 12
 * selected_router_backward): dlogits [T,E] in the logits dtype from FP32
 * dweights [T,k]; the selection itself is not differentiated.  An index >= E
 * makes the row NaN. */
moe_status moe_router_backward(const void* logits, moe_dtype logits_dtype, const uint32_t* idx,
                               const float* dweights, int64_t T, int64_t E, int32_t top_k,
                               int scoring, int renormalize, float scale, void* dlogits,
                               cudaStream_t stream);

/* Diagnostics (no counterpart on the pages): exercises the failure path of
 * the bounded waits inside this library's kernels.  Enqueues one small kernel
 * that waits on a barrier nothing completes; after limit_ms (1..2000) the
 * wait gives up, the kernel writes MOE_ERR_DEVICE_TIMEOUT into the status
 * word at the start of `workspace` (>= 256 bytes, 256-byte aligned, device)
 * and returns normally.  moe_get_device_status(workspace, stream) then
 * reports MOE_ERR_DEVICE_TIMEOUT and the CUDA context stays usable. */
moe_status moe_selftest_bounded_wait(void* workspace, uint32_t limit_ms, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

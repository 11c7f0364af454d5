/*
 * gclip.h -- global L2-norm gradient clipping on one GB300 GPU (sm_103a).
 *
 * The operation.  "Grow a language model: gradient clipping"
 * (unhomeschool.com, Russian), section "Mathematics": treat every gradient
 * element of every parameter as one vector g; norm = sqrt(sum g_i^2); if
 * norm <= max_norm the gradients pass unchanged, otherwise each element is
 * multiplied by max_norm / norm.  "Gradient Clipping" (paweldubiel.com
 * glossary), section "Mechanism and details": the same piecewise rule for a
 * threshold c > 0, with the comparison strict.  The clip runs once per
 * optimizer step, after gradient accumulation, averaging and loss-scale
 * unscaling (glossary, "Order changes the result"; "Grow a language model:
 * backprop", section "Accumulation across microbatches") and before the AdamW
 * moments and weights are updated (clipping page, "Order matters: Pre-Adam").
 *
 * The library works in place on the caller's gradient buffers, on the device,
 * asynchronously on the caller's stream.  It never synchronises the host with
 * the device inside clip_grad_norm and never allocates there: every buffer is
 * allocated once in clip_create (the backprop page, section "Cost of general
 * frameworks": buffers are preallocated at start-up, never reallocated).
 *
 * Return codes are synchronous, host-side checks of the arguments and of the
 * CUDA launch.  Results that depend on the data (the norm, the nonfinite
 * flag, the decision, a timeout of the single-launch variant's grid barrier)
 * are written to device memory and never returned by these calls.
 */
#ifndef GCLIP_H
#define GCLIP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define GCLIP_OK 0
#define GCLIP_ERR_INVALID_ARG 1  /* a host-side argument check failed      */
#define GCLIP_ERR_OOM 2          /* device or host allocation failed       */
#define GCLIP_ERR_CUDA 3         /* a CUDA runtime call or launch failed   */
#define GCLIP_ERR_UNSUPPORTED 4  /* the device cannot run the request      */
#define GCLIP_ERR_TOO_LARGE 5    /* more than the fixed scratch can hold   */

/* ---- values written to clip_result_t.status on the device -------------- */
#define GCLIP_STATUS_OK 0
#define GCLIP_STATUS_TIMEOUT 1   /* single-launch variant: a CTA gave up
                                    waiting at the grid barrier; see
                                    clip_reset */

/* ---- element formats of a gradient tensor ------------------------------ */
#define GCLIP_F32 0              /* IEEE binary32                          */
#define GCLIP_F16 1              /* IEEE binary16                          */
#define GCLIP_BF16 2             /* bfloat16 (upper half of a binary32)    */

/* ---- clip decisions (clip_result_t.decision) --------------------------- */
#define GCLIP_DECISION_PASS 0    /* norm <= max_norm: only the unscale (if
                                    inv_scale != 1) was written            */
#define GCLIP_DECISION_CLIP 1    /* norm > max_norm: every element scaled  */
#define GCLIP_DECISION_SKIP 2    /* nonfinite: no element was written      */

/* ---- execution variants (clip_set_variant) ----------------------------- */
#define GCLIP_VARIANT_SPLIT 0       /* the clipping page's three steps
                                       ("ANDREA's three-kernel pipeline")
                                       in two launches: partial sums with
                                       the final reduction done by the last
                                       block to finish, then the scaling,
                                       with one block per chunk after a
                                       call that wrote and as the claiming
                                       wave of SPLIT_WAVE after one that did
                                       not (see clip_grad_norm)             */
#define GCLIP_VARIANT_PERSISTENT 1  /* all three steps in one cooperative
                                       launch: the last block to finish
                                       reduces, the others wait for it on a
                                       bounded grid barrier, then scale     */
#define GCLIP_VARIANT_SPLIT_TMA 2   /* as SPLIT, with chunks staged through
                                       shared memory by bulk (TMA) copies  */
#define GCLIP_VARIANT_PERSISTENT_TMA 3  /* as PERSISTENT, staged by bulk
                                       (TMA) copies                         */
#define GCLIP_VARIANT_SPLIT_WAVE 4  /* as SPLIT, with the scaling done by one
                                       resident wave of blocks that claim
                                       chunks from a counter: slower by
                                       about 1.5% when every element is
                                       written, faster when nothing is
                                       (few blocks to retire)               */
#define GCLIP_VARIANT_THREE_KERNEL 5  /* the clipping page's pipeline as
                                       written: one block per chunk writes
                                       that chunk's sum of squares, one
                                       block reduces them and decides, one
                                       block per chunk scales (three
                                       launches)                            */

/* One gradient tensor: `numel` elements of format `dtype`, contiguous, in
 * device memory at `ptr` (aligned to the element size).  `reserved` must be
 * 0.  Tensors of one handle must not overlap. */
typedef struct {
    void *ptr;
    int64_t numel;
    int32_t dtype;
    int32_t reserved;
} clip_tensor_desc_t;

/* The device-resident record of the last call on a handle.  The multiplier
 * that was applied to every element x is coef_hi + coef_lo (a float-float
 * pair; the product x * inv_scale * max_norm / norm for CLIP, x * inv_scale
 * for PASS).  sumsq_hi + sumsq_lo is the sum of squares of the unscaled
 * gradients (the double-precision total rounded to a float-float pair, so
 * it underflows for sums below about 1e-38 even where the norm does not). */
typedef struct {
    float norm;          /* global norm of the unscaled gradients (fp32)   */
    int32_t nonfinite;   /* 1 if an element is NaN/inf or the sum of
                            squares exceeds the largest finite fp32 value  */
    int32_t decision;    /* GCLIP_DECISION_*                               */
    int32_t status;      /* GCLIP_STATUS_*                                 */
    float coef_hi;
    float coef_lo;
    float sumsq_hi;
    float sumsq_lo;
    uint32_t calls;      /* completed calls on this handle (wraps)         */
    int32_t reserved;
} clip_result_t;

/* One entry of the chunk table: a run of one tensor, handled by one thread
 * block: at most GCLIP_CHUNK_BYTES, plus, for the first chunk of a tensor,
 * the fewer than 16 bytes that precede the tensor's first 16-byte boundary. */
typedef struct {
    uint64_t addr;       /* device address of the first element            */
    uint32_t numel;      /* elements in this chunk                         */
    uint32_t meta;       /* bits 0-7: dtype; bits 8-31: tensor index       */
} clip_chunk_t;

#define GCLIP_CHUNK_BYTES 32768
#define GCLIP_MAX_TENSORS (1 << 24)

typedef struct gclip_handle *clip_handle_t;

/* clip_create -- plan the clip of one fixed set of gradient tensors.
 *
 * Source: the clipping page, section "ANDREA's three-kernel pipeline": the
 * work is cut into fragments, one thread block per fragment, hundreds of
 * blocks across all tensors of very different shapes (section "Why computing
 * the grad norm needs three kernels": embedding 8449x768 next to layer norm
 * [768]).  This call builds that fragment (chunk) table once, on the host,
 * uploads it, and allocates the per-chunk scratch of partial sums and the
 * result record on the current CUDA device, and one small pinned host word
 * (the write hint of GCLIP_VARIANT_SPLIT).  It is the only call that
 * allocates, apart from the attach calls.
 *
 * descs, n_tensors: host array of the gradient tensors, in the order their
 *   squares are summed; copied, so the array may be freed on return.  The
 *   tensors themselves stay owned by the caller, who must keep them
 *   allocated, at the same addresses, until clip_destroy.
 * out: receives the new handle (owned by the caller; free with clip_destroy).
 * Returns GCLIP_OK; GCLIP_ERR_INVALID_ARG if out is NULL, n_tensors < 0 or
 *   > GCLIP_MAX_TENSORS, descs is NULL with n_tensors > 0, a numel is < 0, a
 *   dtype is unknown, reserved != 0, ptr is NULL or misaligned for a
 *   non-empty tensor, or two non-empty tensors overlap; GCLIP_ERR_OOM or
 *   GCLIP_ERR_CUDA from the device.  *out is untouched on error. */
int clip_create(const clip_tensor_desc_t *descs, int32_t n_tensors,
                clip_handle_t *out);

/* clip_grad_norm -- clip the handle's gradients in place by their global
 * L2 norm.
 *
 * Source: the clipping page, section "Mathematics" (norm, strict test,
 * factor max_norm / norm) and section "ANDREA's three-kernel pipeline"
 * (partial sums of squares per fragment into a scratch buffer, one reduction
 * to a scalar and its square root, one scaling pass); the glossary page,
 * "Mechanism and details" (c > 0) and "Order changes the result" (unscale
 * before the threshold); the backprop page, "Accumulation across
 * microbatches" (average by 1/n_microbatches).
 *
 * Each element x is read in its own format and widened to fp32; the norm is
 * that of y = x * inv_scale, so inv_scale = 1 / (loss_scale * n_microbatches)
 * folds the unscale and the average into the clip.  If any element is NaN or
 * infinite (or the sum of squares overflows fp32) the decision is SKIP and no
 * element is written (the glossary, "Shorten the arrow": a nonfinite value
 * stops the update).  Otherwise, if norm > max_norm, every element becomes
 * x * inv_scale * max_norm / norm (CLIP); else x * inv_scale (PASS), and when
 * that multiplier is exactly 1 nothing is written at all.  Results are rounded
 * to nearest-even into the tensor's own format.
 *
 * The sum is taken in a fixed order (per chunk, then over chunks) with
 * float-float accumulators, so the norm is bit-identical from run to run and
 * between the SPLIT, SPLIT_WAVE and PERSISTENT variants (the two TMA variants
 * share another fixed order, THREE_KERNEL a third).  Squares are fp32, in two
 * bins: a 16-byte vector whose fp32 sum of unscaled squares is below 2^-100
 * (every element's unscaled magnitude below 2^-50) is summed again scaled by
 * a power of two, so that its squares neither underflow nor lose precision;
 * the bins are combined in double.  The norm is therefore
 * accurate to about one fp32 ulp for gradients of any magnitude down to the
 * smallest fp32 values (below about 1e-40, where the fp32 norm itself is
 * subnormal, it is accurate to an fp32 ulp of that range).
 *
 * With GCLIP_VARIANT_SPLIT the shape of the scaling launch follows the
 * decision of the last call on this handle that has completed when this one
 * is enqueued: the norm pass's last block writes whether it will write into
 * a small pinned host word (allocated by clip_create), which this call reads
 * without waiting.  After a clip that wrote, one block per chunk, of which
 * the first resident wave loads its chunks while the norm pass finishes;
 * after one that wrote nothing, one resident wave of blocks (few blocks to
 * retire).
 * Both give the same results bit for bit; a wrong guess costs time only.  A
 * call captured in a CUDA graph keeps the shape chosen at capture.
 *
 * max_norm: threshold c, finite and > 0.  inv_scale: finite and > 0.
 * out_norm: device float, may be NULL; receives the norm (fp32).
 * out_nonfinite_flag: device int32, may be NULL; receives 0 or 1.
 * stream: a cudaStream_t of the handle's device (NULL = legacy default).
 * Asynchronous: returns after enqueueing.  Calls on one handle must not
 * overlap on the device (they share the scratch).
 * Returns GCLIP_OK; GCLIP_ERR_INVALID_ARG for a NULL handle or a bad
 *   max_norm / inv_scale (nothing is enqueued then); GCLIP_ERR_CUDA if a
 *   launch failed. */
int clip_grad_norm(clip_handle_t h, float max_norm, float inv_scale,
                   float *out_norm, int32_t *out_nonfinite_flag, void *stream);

/* clip_grad_norm_profiled -- clip_grad_norm that also records four CUDA
 * events (cudaEvent_t handles created by the caller on the handle's device)
 * on `stream`: events[0] before the first launch, events[1] and events[2]
 * after the norm pass (partial sums and final reduction, one launch; with
 * GCLIP_VARIANT_THREE_KERNEL events[1] after the per-chunk sums and
 * events[2] after the final reduction), events[3] after the scaling pass.  With the single-launch variant the one
 * launch lies between events[2] and events[3], and events[1] and events[2]
 * are recorded with events[0].  Programmatic dependent launch is not used in
 * this mode, so the launches do not overlap their neighbours; it is meant
 * for measuring each step of the clip, with the same arithmetic and results
 * as clip_grad_norm.  Returns as clip_grad_norm, and GCLIP_ERR_INVALID_ARG
 * for NULL events. */
int clip_grad_norm_profiled(clip_handle_t h, float max_norm, float inv_scale,
                            float *out_norm, int32_t *out_nonfinite_flag,
                            void *stream, void *const *events);

/* clip_destroy -- wait for the handle's device work, free its device memory
 * and the handle.  NULL is accepted and ignored.  Returns GCLIP_OK, or
 * GCLIP_ERR_CUDA if the device reported an error while finishing. */
int clip_destroy(clip_handle_t h);

/* clip_set_variant -- choose one of the GCLIP_VARIANT_* values for later
 * calls (GCLIP_VARIANT_SPLIT is the default).  SPLIT, SPLIT_WAVE and
 * PERSISTENT compute bit-identical norms and outputs, and so do SPLIT_TMA and
 * PERSISTENT_TMA; THREE_KERNEL sums each chunk on its own first.  The three
 * groups sum in different (fixed) orders, so their norms can differ in the
 * last bits.  Returns GCLIP_ERR_INVALID_ARG for an unknown variant,
 * GCLIP_ERR_UNSUPPORTED if the device cannot launch cooperative kernels. */
int clip_set_variant(clip_handle_t h, int32_t variant);

/* clip_get_variant -- the variant in use, or -1 for a NULL handle. */
int32_t clip_get_variant(clip_handle_t h);

/* clip_result_device -- device address of the handle's clip_result_t,
 * valid until clip_destroy; NULL for a NULL handle.  Stream-ordered reads of
 * it after a call see that call's record. */
const clip_result_t *clip_result_device(clip_handle_t h);

/* clip_read_result -- copy the record to host memory `out`, synchronising
 * `stream` (inspection and tests; not for the training loop).  Returns
 * GCLIP_ERR_INVALID_ARG for NULL arguments, GCLIP_ERR_CUDA on failure. */
int clip_read_result(clip_handle_t h, clip_result_t *out, void *stream);

/* clip_last_status -- enqueue on `stream` a copy of the status word of the
 * handle's record (GCLIP_STATUS_OK, or GCLIP_STATUS_TIMEOUT after a
 * single-launch call whose grid barrier gave up) into the device int32 at
 * d_out, in stream order after the calls before it; no host sync, no
 * allocation.  The same word is clip_result_device(h)->status.  Returns
 * GCLIP_OK, GCLIP_ERR_INVALID_ARG (NULL handle or d_out) or GCLIP_ERR_CUDA. */
int clip_last_status(clip_handle_t h, int32_t *d_out, void *stream);

/* clip_reset -- enqueue a clear of the handle's grid-barrier words and of
 * the status in its record.  Needed only after a call reported
 * GCLIP_STATUS_TIMEOUT, whose gradients are then in an unspecified state
 * (some chunks may have been scaled).  Returns GCLIP_OK or GCLIP_ERR_*. */
int clip_reset(clip_handle_t h, void *stream);

/* clip_num_chunks -- chunks in the handle's table (-1 for NULL). */
int64_t clip_num_chunks(clip_handle_t h);

/* clip_persistent_grid -- thread blocks of the single-launch variant on this
 * handle's device (-1 for NULL). */
int32_t clip_persistent_grid(clip_handle_t h);

/* clip_tma_grid -- thread blocks of the TMA variants on this handle's
 * device (-1 for NULL). */
int32_t clip_tma_grid(clip_handle_t h);

/* clip_plan -- host-only: validate `descs` exactly as clip_create does and
 * write the chunk table it would build into `out` (capacity entries, may be
 * NULL to count).  Chunks follow tensor order; within a tensor they are
 * consecutive and sized as clip_chunk_t states, and every chunk after a
 * tensor's first starts on a 16-byte boundary.  Empty tensors get no chunk.
 * *n_chunks receives the count.  Touches no device.  Returns GCLIP_OK,
 * GCLIP_ERR_INVALID_ARG (as clip_create, or capacity too small for a
 * non-NULL out). */
int clip_plan(const clip_tensor_desc_t *descs, int32_t n_tensors,
              clip_chunk_t *out, int64_t capacity, int64_t *n_chunks);

/* clip_status_string -- a static English description of a return code. */
const char *clip_status_string(int32_t code);

/* clip_set_l2_keep -- how many bytes at the end of the norm pass (the
 * chunks the scaling pass visits first) are read with an L2 evict_last
 * policy, so that the scaling pass finds them in L2 instead of HBM.  The
 * default is 0 (off): on the ANDREA-120M fp32 set the hint moved ~50 MB of
 * the scaling pass's reads into L2 but did not shorten the clip.  Rounded
 * down to whole chunks.  The other chunks are read with evict_first, except
 * in sets that fit in half of the device's L2, which are read with the normal
 * policy so that a set clipped again soon is still in L2.  Affects timing
 * only, never results.  Returns GCLIP_OK or GCLIP_ERR_INVALID_ARG (NULL
 * handle, negative bytes). */
int clip_set_l2_keep(clip_handle_t h, int64_t bytes);

/* clip_debug_barrier -- test hook for the single-launch variant's bounded
 * grid barrier.  extra_arrivals > 0 makes the barrier wait for that many
 * more thread blocks than exist, so it cannot complete and every block must
 * give up after timeout_ns (0 keeps the default of one second), write
 * GCLIP_STATUS_TIMEOUT and return without writing gradients.  The library
 * clears the barrier words around such a call.  extra_arrivals = 0 restores
 * normal operation.  Returns GCLIP_OK or GCLIP_ERR_INVALID_ARG. */
int clip_debug_barrier(clip_handle_t h, int32_t extra_arrivals,
                       int64_t timeout_ns);

/* ---- fused clip + AdamW ---------------------------------------------------
 *
 * Source: the clipping page, section "Order matters: Pre-Adam": the clip runs
 * before the AdamW moments m, v and the weights are updated, so a spike never
 * reaches m and v; section "Adjacent activities": AdamW keeps m and v.  The
 * backprop page, section "Optimizer state": one m and one v per weight, and
 * section "Accumulation across microbatches": zero_grads() after the step.
 * The pages do not write the update out; it is the published AdamW with
 * decoupled weight decay and bias correction, on g^ = x * multiplier (the
 * clipped, unscaled gradient of clip_grad_norm):
 *   m = beta1 m + (1 - beta1) g^;  v = beta2 v + (1 - beta2) g^^2
 *   w = w (1 - lr wd) - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 * Fusing it makes the clip's scaling pass unnecessary: the clipped gradient
 * is formed in registers, never stored. */

/* The optimizer state of one gradient tensor: fp32 device arrays with the
 * tensor's numel, each aligned to 4 bytes (16 bytes, like the gradient,
 * lets the kernel use vector access).  Owned by the caller. */
typedef struct {
    float *w;
    float *m;
    float *v;
} clip_adamw_state_t;

typedef struct {
    float lr;            /* >= 0 */
    float beta1;         /* in [0, 1) */
    float beta2;         /* in [0, 1) */
    float eps;           /* > 0 */
    float weight_decay;  /* >= 0, decoupled */
    int32_t zero_grads;  /* nonzero: write +0 to every gradient element after
                            use (not on SKIP) */
} clip_adamw_params_t;

/* clip_attach_adamw -- give the handle the optimizer state of its tensors,
 * states[i] for descriptor i (n_tensors must equal the handle's count;
 * empty tensors may have NULL pointers).  Checks alignment and that no two
 * arrays (weights, moments, gradients) overlap; copies a table of pointers to
 * the device (the only allocation, at attach time).  May be called again to
 * replace the state.  Returns GCLIP_OK, GCLIP_ERR_INVALID_ARG, GCLIP_ERR_OOM
 * or GCLIP_ERR_CUDA. */
int clip_attach_adamw(clip_handle_t h, const clip_adamw_state_t *states,
                      int32_t n_tensors);

/* clip_grad_norm_adamw -- the clip of clip_grad_norm (norm, nonfinite flag,
 * decision; max_norm, inv_scale, out_norm, out_nonfinite_flag and stream as
 * there), then, unless the decision is SKIP, one AdamW step of optimizer
 * step number `step` (1-based) on every element, with g^ = x * the clip's
 * multiplier.  The gradients are read, not rewritten (set to +0 if
 * p->zero_grads).  On SKIP nothing at all is written except the record,
 * out_norm and out_nonfinite_flag.  Always runs as two launches (the split
 * variant's norm pass, then the AdamW pass), whatever clip_set_variant chose.
 * Asynchronous, no allocation.  Returns GCLIP_OK; GCLIP_ERR_INVALID_ARG
 * (NULL handle or p, no state attached, bad max_norm / inv_scale, lr < 0,
 * beta outside [0, 1), eps <= 0, weight_decay < 0, step < 1, or any of them
 * not finite); GCLIP_ERR_CUDA if a launch failed. */
int clip_grad_norm_adamw(clip_handle_t h, float max_norm, float inv_scale,
                         const clip_adamw_params_t *p, int64_t step,
                         float *out_norm, int32_t *out_nonfinite_flag,
                         void *stream);

/* clip_adamw_step -- one AdamW step of optimizer step number `step`
 * (1-based) on the attached state with the gradients as they are: the second
 * launch of clip_grad_norm_adamw alone, with multiplier 1 and no norm pass.
 * For an update that follows a clip already made by clip_grad_norm (the
 * clipping page, "Order matters: Pre-Adam": clip, then AdamW), and the
 * unfused counterpart the fused call is measured against.  For fp32
 * gradients, clip_grad_norm followed by this call gives w, m and v bit for
 * bit equal to clip_grad_norm_adamw (the in-place clip stores exactly the
 * fp32 value the fused pass forms in registers); for fp16/bf16 gradients
 * the clipped values are rounded to the gradient's format first.  Nonfinite
 * gradients are not checked: they reach the moments as they are.  The
 * gradients are read, and set to +0 if p->zero_grads.  Asynchronous, no
 * allocation, nothing written to the record.  Returns GCLIP_OK (also for a
 * set with no elements); GCLIP_ERR_INVALID_ARG (NULL handle or p, no state
 * attached, a hyperparameter or step out of range as for
 * clip_grad_norm_adamw); GCLIP_ERR_CUDA if the launch failed. */
int clip_adamw_step(clip_handle_t h, const clip_adamw_params_t *p, int64_t step,
                    void *stream);

/* ---- per-tensor clipping -------------------------------------------------
 *
 * Source: the clipping page, section "Per-Tensor or Global": each gradient
 * tensor clipped by its own norm, the simpler alternative that distorts the
 * relative scales between tensors (the global clip above is what the page
 * uses); the glossary page, "Shorten the arrow, keep the direction": a limit
 * per layer is a different constraint. */

/* clip_grad_norm_per_tensor -- for every tensor t of the handle on its own:
 * norm_t of its unscaled elements, and x <- x * inv_scale * (norm_t > max_norm
 * ? max_norm / norm_t : 1), nothing written when that multiplier is 1 or
 * when tensor t holds a NaN/inf (that tensor alone is skipped).  Empty
 * tensors have norm 0.  out_norms, out_nonfinite_flags: device arrays of one
 * entry per tensor, each may be NULL.  The per-tensor records go to the
 * handle (clip_read_per_tensor).  Three launches (chunk sums; one block per
 * tensor, which decides and lists the chunks to rewrite; one wave of blocks
 * scaling the listed chunks); asynchronous, no allocation.  Consecutive
 * per-tensor calls on one handle must be issued in stream order (the chunk
 * list is the handle's).  Returns GCLIP_OK,
 * GCLIP_ERR_INVALID_ARG (NULL handle, bad max_norm / inv_scale) or
 * GCLIP_ERR_CUDA. */
int clip_grad_norm_per_tensor(clip_handle_t h, float max_norm, float inv_scale,
                              float *out_norms, int32_t *out_nonfinite_flags,
                              void *stream);

/* clip_read_per_tensor -- copy the first n per-tensor records of the last
 * clip_grad_norm_per_tensor call to host memory `out`, synchronising
 * `stream`.  Returns GCLIP_OK, GCLIP_ERR_INVALID_ARG (n < 0 or more than the
 * handle's tensors, NULL arguments) or GCLIP_ERR_CUDA. */
int clip_read_per_tensor(clip_handle_t h, clip_result_t *out, int32_t n, void *stream);

/* ---- out-of-place clip into fp32 ----------------------------------------
 *
 * For fp16/bf16 gradients kept under loss scaling: the unscaled values
 * (the glossary page, "Order changes the result": unscale before the
 * threshold) are often below binary16's normal range, where an in-place
 * result can only keep a few bits.  This writes the clipped, unscaled
 * gradients as fp32 into separate buffers (master gradients) and leaves the
 * originals as they were. */

/* clip_attach_f32_out -- outs[i] receives descriptor i's result: an fp32
 * device array of the same numel, aligned to 4 bytes (16 lets the kernel
 * use vector stores), not overlapping any gradient or other output.  Empty
 * tensors may have NULL.  Copies a table of pointers to the device (the only
 * allocation).  Returns GCLIP_OK, GCLIP_ERR_INVALID_ARG, GCLIP_ERR_OOM or
 * GCLIP_ERR_CUDA. */
int clip_attach_f32_out(clip_handle_t h, float *const *outs, int32_t n_tensors);

/* clip_grad_norm_to_f32 -- the norm, flag and decision of clip_grad_norm;
 * then, unless the decision is SKIP, every element x is written to its
 * output as x * multiplier (inv_scale * max_norm / norm, or inv_scale)
 * rounded once to fp32, even when the multiplier is 1.  The gradients are
 * only read.  Two launches (the split norm pass, then the conversion),
 * whatever clip_set_variant chose; asynchronous, no allocation.  Returns
 * GCLIP_OK; GCLIP_ERR_INVALID_ARG (NULL handle, no outputs attached, bad
 * max_norm / inv_scale); GCLIP_ERR_CUDA. */
int clip_grad_norm_to_f32(clip_handle_t h, float max_norm, float inv_scale,
                          float *out_norm, int32_t *out_nonfinite_flag,
                          void *stream);

/* ------------------------------------------------------------------------
 * Accumulation epilogue.  "Grow a language model: backprop" (unhomeschool.com,
 * Vietnamese), section "Accumulation across microbatches": with several
 * microbatches per step the backward kernels add (+=) into the gradient
 * buffers, which hold the running sum; the glossary page, section "Order
 * changes the result", clips only after the whole effective batch is in.
 * These two calls fold the last microbatch's += into the clip's norm pass:
 * the pass that reads the gradients to square them also adds the addend and
 * writes the sum back, so the sum costs no read of its own. */

/* clip_attach_addend -- addends[i] is added into descriptor i's gradient by
 * clip_grad_norm_accumulate: a device array of the same numel and format
 * (dtype), aligned to the element size (the same offset within 16 bytes as
 * its gradient lets the kernel use vector loads), not overlapping any
 * gradient or other addend.  Empty tensors may have NULL.  The arrays stay
 * owned by the caller and are only read.  Copies a table of pointers to the
 * device (the only allocation); a new call replaces the table.  Returns
 * GCLIP_OK, GCLIP_ERR_INVALID_ARG (NULL handle, count different from the
 * handle's tensors, NULL, misaligned or overlapping arrays), GCLIP_ERR_OOM
 * or GCLIP_ERR_CUDA. */
int clip_attach_addend(clip_handle_t h, const void *const *addends, int32_t n_tensors);

/* clip_grad_norm_accumulate -- every gradient element x becomes x + a (its
 * addend element), the sum rounded once to nearest even in the gradient's
 * format and stored in place; then the clip of clip_grad_norm on the sums:
 * the same norm, flag, decision and outputs, bit for bit, as adding the
 * addends with the format's own addition and then calling clip_grad_norm
 * with the split variant.  The sums are stored whatever the decision: on
 * SKIP (a nonfinite sum) the gradients hold the unscaled, unclipped sums.
 * Two launches (the norm pass with the addition, then the scaling: by the
 * claiming wave under GCLIP_VARIANT_SPLIT_WAVE, else one block per chunk);
 * asynchronous, no allocation.  Returns
 * GCLIP_OK; GCLIP_ERR_INVALID_ARG (NULL handle, no addends attached, bad
 * max_norm / inv_scale); GCLIP_ERR_CUDA. */
int clip_grad_norm_accumulate(clip_handle_t h, float max_norm, float inv_scale,
                              float *out_norm, int32_t *out_nonfinite_flag,
                              void *stream);

/* clip_grad_norm_flat_noalloc -- the same clip for one contiguous gradient
 * buffer, for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for the library's
 * users.  Some callers cannot call cudaMalloc or hold a handle: code whose
 * device memory is all owned by another allocator (a framework's caching
 * allocator, or a fixed arena sized at start-up) and must not take memory
 * from the driver in the middle of a run, where an allocation can fail or
 * stall the device at an arbitrary point; and plug-in or callback interfaces
 * that get a buffer and a stream but no create/destroy hooks in which to set
 * up and free a handle.  This call asks for no memory from anyone: its
 * scratch (the per-chunk partial sums and the result record) lives in one
 * fixed array compiled into the library, GCLIP_NOALLOC_SCRATCH_BYTES long,
 * which every GPU that loads the library holds until the process exits.
 *
 * grads: `numel` elements of format `dtype` in device memory of the current
 *   device, contiguous, aligned to the element size; clipped in place by the
 *   three launches of GCLIP_VARIANT_THREE_KERNEL, with the buffer cut into
 *   the chunks clip_create cuts a single tensor into.  The norm, record and
 *   outputs are bit-identical to clip_grad_norm on a handle made of this one
 *   tensor with GCLIP_VARIANT_THREE_KERNEL, and agree with the default
 *   variant within the parity tolerances (that variant sums the same chunks
 *   in another fixed order).
 * max_norm, inv_scale, out_norm, out_nonfinite_flag, stream: as for
 *   clip_grad_norm; the stream must belong to the current device.
 * Limit: the buffer may span at most GCLIP_NOALLOC_MAX_CHUNKS chunks of
 *   GCLIP_CHUNK_BYTES (2 GiB of gradients: 536,870,912 fp32 or 1,073,741,824
 *   fp16/bf16 elements, a little less when the buffer does not start on a
 *   16-byte boundary); a larger buffer returns GCLIP_ERR_TOO_LARGE and
 *   nothing is enqueued.
 * Set-up: the first call on each device looks up the device address of the
 *   scratch array and the device's L2 size (with that device current) and
 *   may load the library's device code there; make that first call before
 *   any stream capture.  The address is kept for the life of the process:
 *   after cudaDeviceReset on a device, which unloads the library's device
 *   code there, this call must not be used on that device again.
 * Sharing: every call, on every stream, uses the same scratch array and it
 *   keeps the last call's contents.  Calls that overlap on the device race
 *   with each other and give wrong results: serialise them (one stream, or
 *   events).  Nothing needs clearing between calls: every partial sum a call
 *   reads is first written by that call; only the record's call counter is
 *   carried over from call to call.  The record is not readable through the
 *   handle functions; use out_norm and out_nonfinite_flag.
 * Returns GCLIP_OK; GCLIP_ERR_INVALID_ARG (bad dtype, negative numel, NULL or
 *   misaligned grads with numel > 0, bad max_norm / inv_scale);
 *   GCLIP_ERR_TOO_LARGE; GCLIP_ERR_CUDA (no current device, the scratch could
 *   not be located, or a launch failed).  Allocates nothing. */
#define GCLIP_NOALLOC_MAX_CHUNKS 65536
#define GCLIP_NOALLOC_SCRATCH_BYTES (GCLIP_NOALLOC_MAX_CHUNKS * 16 + 256)
int clip_grad_norm_flat_noalloc(void *grads, int64_t numel, int32_t dtype,
                                float max_norm, float inv_scale,
                                float *out_norm, int32_t *out_nonfinite_flag,
                                void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GCLIP_H */

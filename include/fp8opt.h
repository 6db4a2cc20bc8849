/*
 * libfp8opt: the scaled FP8 cast and the FP8-state AdamW step of the MS-AMP
 * mixed-precision scheme, as hand-written CUDA kernels for one GB300 (sm_103a).
 *
 * Where the operations come from:
 *   - MS-AMP documentation, "Optimization Level" page, O1 paragraph and level
 *     table: weight gradients are kept in FP8 (the cast below).
 *   - Same page, O2 paragraph and table row: the Adam/AdamW first moment is
 *     kept in FP8 and the second moment in FP16, with FP16 weights.
 *   - Same page, O3 paragraph and table row: an FP16 master weight plus an
 *     FP8 regular weight used for forward/backward.
 *   - MS-AMP README, "Usage": the GradScaler loop (scaler.scale(loss).backward(),
 *     scaler.step(optimizer)) and the recognised optimizers (torch.optim.Adam,
 *     torch.optim.AdamW).
 *   - TransformerEngine issue #131 ("FP8 questions"): the two FP8 formats
 *     E4M3 and E5M2, each used in its own place, never cast into one another.
 *
 * Formats: E4M3 and E5M2 are the OCP 8-bit floating-point formats (E4M3:
 * bias 7, max 448, no infinity, NaN = 0x7F/0xFF; E5M2: bias 15, max 57344,
 * +-inf = 0x7C/0xFC).  FP16 buffers hold IEEE binary16 bit patterns, BF16
 * buffers bfloat16 bit patterns.  Every encode rounds to nearest, ties to even,
 * and saturates finite overflow to +-max; a NaN encodes as 0x7F, an infinity
 * as 0x7F in E4M3 and as the signed infinity code in E5M2.
 *
 * Memory: every pointer in an item or parameter record is a DEVICE pointer
 * owned by the caller; the library never frees or keeps them beyond the call's
 * stream work.  The library owns a per-(device, stream) workspace (tensor
 * tables, chunk tables, amax slots, the found_inf word) that it allocates on
 * first use and grows when a longer list arrives; fp8opt_release() frees all
 * of it.  The workspace also caches the tensor tables of the last list seen on
 * each stream, so repeating a call with the same list uploads nothing.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 * work of a call is ordered on that stream; the calls return before the GPU
 * finishes unless the caller asks for found_inf on the host.  Calls on one
 * stream must come from one host thread at a time; calls on different streams
 * use different workspaces and may run concurrently.
 *
 * CUDA graphs: a call may be captured into a CUDA graph (stream capture) once
 * the same tensor list has run on that stream, so that its tables and
 * workspace exist; a list not yet seen on the stream is refused under capture
 * (FP8OPT_ERR_ARG).  The graph then refers to that stream's workspace, which
 * is frozen: later calls on the stream must use the lists already there (a
 * new list is refused with FP8OPT_ERR_ARG, a larger workspace fails with
 * FP8OPT_ERR_CUDA, "operation not permitted"), so other lists belong on other
 * streams; fp8opt_release_stream() or fp8opt_release() frees it (after the
 * graph is destroyed).  A
 * captured call
 * zeroes its per-tensor slots as part of the captured work, so every replay
 * is a fresh call on the buffers' current contents.  Host outputs (found_inf,
 * the host norm) wait for the stream and cannot be captured: pass NULL and use
 * the device outputs.  What a capture fixes: the records, and the step's
 * scalars (lr, the bias corrections of `step`, inv_loss_scale, the clip
 * threshold); the cast and the reduction have none, so their replays are
 * exactly new calls.  The *_dev step calls read lr, inv_loss_scale and the
 * step count from device memory instead (fp8opt_step_state), so one captured
 * graph of them serves every step of a training loop.
 *
 * Errors: every entry point returns FP8OPT_OK (0) or a negative status.  On an
 * argument error nothing is launched and no output is touched.  On a CUDA
 * error the CUDA error text is kept for fp8opt_last_error().
 */
#ifndef FP8OPT_H
#define FP8OPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define FP8OPT_API __attribute__((visibility("default")))
#else
#define FP8OPT_API
#endif

/* FP8 formats. */
#define FP8OPT_E4M3 0
#define FP8OPT_E5M2 1

/* Element types accepted by the cast. */
#define FP8OPT_F32  0
#define FP8OPT_BF16 1
#define FP8OPT_F16  2

/* Status codes. */
#define FP8OPT_OK               0
#define FP8OPT_ERR_ARG         (-1)  /* null pointer, n < 0, numel < 0, step < 1,
                                        nonzero reserved field, incomplete O3
                                        record */
#define FP8OPT_ERR_UNSUPPORTED (-2)  /* unknown format or element type */
#define FP8OPT_ERR_CUDA        (-4)  /* a CUDA call failed; see fp8opt_last_error */
#define FP8OPT_ERR_LIMIT       (-5)  /* a size above a fixed maximum (the
                                        no-allocation entry point's limits) */

/* One tensor of a scaled cast. */
typedef struct {
    const void *src;   /* numel elements of type `dtype`, contiguous */
    int64_t numel;     /* >= 0; 0 is allowed (amax 0, scale 1) */
    int32_t dtype;     /* FP8OPT_F32, FP8OPT_BF16 or FP8OPT_F16 */
    int32_t reserved;  /* must be 0 */
    uint8_t *codes;    /* out: numel FP8 codes */
    float *amax;       /* out: one fp32, max |x| (NaN above inf above finite;
                          a NaN amax is written as 0x7FC00000) */
    float *scale;      /* out: one fp32, fp8_max / amax, or 1.0 when amax is 0
                          or not finite or the quotient is not finite */
} fp8opt_cast_item;

/*
 * fp8_cast_scaled: per-tensor just-in-time scaled cast of a tensor list to FP8
 * (MS-AMP O1: weight gradients from a wider type to FP8).
 *
 * For each item: amax = max |x|; scale = fp8_max / amax (one IEEE fp32
 * division; fp8_max 448 for E4M3, 57344 for E5M2); code[i] = encode(x[i] *
 * scale) with one fp32 round-to-nearest product.  One launch covers the whole
 * list (two passes over the data: amax, then encode).
 *
 * items: host array of n records; n >= 0; fmt: FP8OPT_E4M3 or FP8OPT_E5M2;
 * stream: cudaStream_t.  Source buffers may be unaligned (a scalar path takes
 * them); the output buffers may not overlap the inputs.
 */
FP8OPT_API int fp8_cast_scaled(const fp8opt_cast_item *items, int n, int fmt, void *stream);

/* One tensor of the AdamW step.  O2 when w8, w8_scale and w8_amax are all
 * NULL; O3 when w8_scale and w8_amax are set, with w8 set too unless numel is
 * 0 (an empty tensor's buffer may have a NULL address). */
typedef struct {
    int64_t numel;         /* >= 0 */
    const uint8_t *g;      /* numel gradient codes (format g_fmt), as written by
                              fp8_cast_scaled; may hold loss-scaled values */
    const float *g_scale;  /* one fp32: the scale the codes were encoded with */
    int32_t g_fmt;         /* FP8OPT_E4M3 or FP8OPT_E5M2 */
    int32_t reserved;      /* must be 0 */
    uint8_t *m;            /* in/out: first moment, numel E4M3 codes */
    float *m_scale;        /* in/out: one fp32, its scale (1.0 for m = 0) */
    uint16_t *v;           /* in/out: second moment, numel FP16 */
    uint16_t *w;           /* in/out: O2 weight, or O3 master weight, FP16 */
    uint8_t *w8;           /* O3 out: numel E4M3 codes of the master, else NULL */
    float *w8_scale;       /* O3 out: one fp32, its scale, else NULL */
    float *w8_amax;        /* O3 out: one fp32, max |master|, else NULL */
    float *v_bound;        /* in/out: one fp32 for a scaled second moment
                              (v then holds FP16 of v * 2^14 / v_bound; start
                              at 0 with v = 0), or NULL for plain FP16 v */
} fp8opt_param;

/*
 * fp8_adamw_step: one multi-tensor AdamW step with FP8 first moment and FP16
 * second moment (MS-AMP O2), with FP16 master and FP8 weight copy for O3
 * records, and the GradScaler inf/NaN skip.
 *
 * Per element, in fp32, each operation rounded once (fma: product and sum
 * rounded once together), in this order:
 *   g = decode(g_code) * k,               k = inv_loss_scale / g_scale
 *   m = fma(beta1, decode(m_code) * (1 / m_scale_old), (1 - beta1) * g)
 *   v = fma(beta2, v_old, (1 - beta2) * (g * g))
 *   u = m / fma(sqrt(v), inv_sbc2, eps)
 *   w = fma(-step_size, u, w_old * (1 - lr * wd))
 * with step_size = lr / (1 - beta1^step) and inv_sbc2 = 1 / sqrt(1 -
 * beta2^step) evaluated in double and rounded to fp32 once: torch.optim.AdamW's
 * update (decoupled decay, eps after the bias-corrected root) with the bias
 * corrections folded into two scalars.  The first moment is stored as
 * E4M3 with the new scale 448 / amax(m) of this step; v and w are stored as
 * FP16 (round to nearest even, overflow to inf).  For O3 records, the FP16
 * master's amax gives w8_scale = 448 / w8_amax and w8 = encode(master *
 * w8_scale).
 *
 * Scaled second moment (v_bound set): plain FP16 cannot hold the (1 -
 * beta2) g^2 of small gradients (about 1e-13 at g ~ 1e-5; FP16's smallest
 * subnormal is 6e-8), so v is kept relative to a per-tensor bound B on max v:
 * B_new = fma(beta2, B_old, (1 - beta2) * gmax * gmax) with gmax = max |g| of
 * this step; v_old = FP16 * (B_old * 2^-14), and v is stored as FP16 of v *
 * (2^14 / B_new) (1.0 when B_new is 0 or not finite), so the stored values
 * stay below about 2^14 * (1 + 2^-10).  The bound is written only when the
 * step is taken.
 *
 * found_inf: if any unscaled g of any record is not finite, nothing is
 * written (no code, no state, no scale) and found_inf is 1; the caller then
 * lowers its loss scale and does not advance `step`, like a GradScaler.
 *
 * params: host array of n records; step >= 1.  found_inf: host int, may be
 * NULL; when set the call waits for the stream and writes 0 or 1.
 * found_inf_dev: device uint32, may be NULL; when set the kernels write 0 or 1
 * there without a host round trip.  stream: cudaStream_t.  A record's buffers
 * must not overlap another record's.  Returns a status; found_inf is a result,
 * not an error.
 */
FP8OPT_API int fp8_adamw_step(const fp8opt_param *params, int n, float lr, float beta1,
                   float beta2, float eps, float wd, int64_t step,
                   float inv_loss_scale, int *found_inf,
                   uint32_t *found_inf_dev, void *stream);

/* Limits of fp8_cast_scaled_noalloc: tensors per call, and chunks of 32768
 * elements per call (an empty tensor counts as one chunk). */
#define FP8OPT_NOALLOC_MAX_TENSORS 1024
#define FP8OPT_NOALLOC_MAX_CHUNKS  65536

/*
 * fp8_cast_scaled_noalloc: fp8_cast_scaled for callers that must not allocate
 * device memory.  No counterpart in the MS-AMP pages: it exists for callers
 * such as runtimes whose pool allocator owns all device memory, or services
 * that must not stall on or fail from an allocation mid-step.
 * fp8_cast_scaled allocates its workspace on first use; this entry point
 * instead keeps its tensor table, chunk table and amax slots in one fixed
 * array compiled into the library (about 1.1 MB per device, present on every
 * device that loads the library, until the process exits), and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Same arguments, same results and same errors as fp8_cast_scaled, plus
 * FP8OPT_ERR_LIMIT (nothing launched) when n exceeds
 * FP8OPT_NOALLOC_MAX_TENSORS or the list needs more than
 * FP8OPT_NOALLOC_MAX_CHUNKS chunks.  The first call on each device sets the
 * entry point up for that device (it looks up the array's device address).
 * Each call copies its tables from host arrays that the next call refills, so
 * a stream that is capturing a CUDA graph is refused with FP8OPT_ERR_ARG and
 * nothing enqueued.  All calls on a device share the one array, which keeps
 * the previous call's contents; each call clears what it needs zeroed, but
 * calls whose GPU work overlaps (on different streams, or from different host
 * threads) race on the array: order them.
 */
FP8OPT_API int fp8_cast_scaled_noalloc(const fp8opt_cast_item *items, int n,
                                       int fmt, void *stream);

/*
 * fp8_adam_step: as fp8_adamw_step, but Adam with L2 weight decay (the
 * README's other recognised optimizer, torch.optim.Adam with weight_decay):
 * each unscaled gradient becomes g = fma(wd, w_old, g) before the moments
 * (found_inf is still decided on the unscaled g), and the weight is not
 * decayed (w = fma(-step_size, u, w_old)).  Its first pass also reads w:
 * 2 bytes more per parameter.  Same arguments, results and errors otherwise.
 */
FP8OPT_API int fp8_adam_step(const fp8opt_param *params, int n, float lr,
                             float beta1, float beta2, float eps, float wd,
                             int64_t step, float inv_loss_scale, int *found_inf,
                             uint32_t *found_inf_dev, void *stream);

/*
 * fp8_cast_adamw_step: fp8_cast_scaled(grads, n, fmt) followed by
 * fp8_adamw_step(params, n, ...) on the codes it wrote, in one call and with
 * one pass fewer over memory: the encode pass of the cast also computes the
 * step's first pass (found_inf and the amax of the new first moment) from the
 * codes it has just produced.  Results, found_inf semantics and errors are
 * those of the two calls made in turn (MS-AMP O1 gradient cast, then the
 * O2/O3 step with the GradScaler skip).
 *
 * params[i] must take grads[i]'s output: params[i].g == grads[i].codes,
 * params[i].g_scale == grads[i].scale, the same numel, and g_fmt == fmt;
 * otherwise FP8OPT_ERR_ARG and nothing is launched.  Other arguments as for
 * the two calls.  With BF16 gradients an O2 step moves 17 bytes per parameter
 * instead of 18.
 */
FP8OPT_API int fp8_cast_adamw_step(const fp8opt_cast_item *grads,
                                   const fp8opt_param *params, int n, int fmt,
                                   float lr, float beta1, float beta2, float eps,
                                   float wd, int64_t step, float inv_loss_scale,
                                   int *found_inf, uint32_t *found_inf_dev,
                                   void *stream);

/*
 * Device-resident step values for the *_dev calls (the graph-replayable form
 * of the step: a captured call reads these at replay time, where the other
 * step calls fix lr, the step's bias corrections and inv_loss_scale at
 * capture).  Device memory, 8-byte aligned, owned by the caller:
 *   lr              learning rate of the next step;
 *   inv_loss_scale  1 / the GradScaler loss scale of the next step;
 *   step            steps taken so far (>= 0).  A call computes the bias
 *                   corrections of t = step + 1, in the arithmetic of
 *                   fp8_adamw_step, and stores t back unless found_inf skips
 *                   the step (GradScaler semantics: a skipped step does not
 *                   count).
 * The host reads none of these: values the host entry points would refuse
 * (step < 0, a non-finite lr) are not checked.
 */
typedef struct {
  float lr;
  float inv_loss_scale;
  int64_t step;
} fp8opt_step_state;

/*
 * fp8_adam_step_dev: fp8_adamw_step (l2 = 0) or fp8_adam_step (l2 = 1) with lr,
 * inv_loss_scale and the step count read from *state on the device (see
 * fp8opt_step_state), so that the call can be captured once into a CUDA graph
 * and replayed every step.  Results are bit-identical to the host-scalar call
 * with the same values.  found_inf goes to found_inf_dev (device, may be
 * NULL); there is no host output.  beta1, beta2, eps and wd are fixed per
 * call as in fp8_adamw_step.  Errors: as fp8_adamw_step, plus FP8OPT_ERR_ARG
 * when state is NULL or misaligned or l2 is not 0 or 1.
 */
FP8OPT_API int fp8_adam_step_dev(const fp8opt_param *params, int n, float beta1,
                                 float beta2, float eps, float wd, int l2,
                                 fp8opt_step_state *state,
                                 uint32_t *found_inf_dev, void *stream);

/*
 * fp8_cast_adamw_step_dev: fp8_cast_adamw_step with lr, inv_loss_scale and the
 * step count read from *state on the device, as fp8_adam_step_dev (AdamW
 * only).  Arguments, results and errors otherwise those of
 * fp8_cast_adamw_step, with found_inf in found_inf_dev only.
 */
FP8OPT_API int fp8_cast_adamw_step_dev(const fp8opt_cast_item *grads,
                                       const fp8opt_param *params, int n,
                                       int fmt, float beta1, float beta2,
                                       float eps, float wd,
                                       fp8opt_step_state *state,
                                       uint32_t *found_inf_dev, void *stream);

/*
 * fp8_cast_adam_step_clipped_dev: fp8_cast_adam_step_clipped with lr,
 * inv_loss_scale and the step count read from *state on the device, as
 * fp8_adam_step_dev: the capturable form of the clipped (and Adam-L2) fused
 * step.  max_grad_norm is fixed per call like the betas.  The norm goes to
 * grad_norm_dev (device float, may be NULL) and found_inf to found_inf_dev
 * (may be NULL); there are no host outputs.  Arguments, results and errors
 * otherwise those of fp8_cast_adam_step_clipped, plus FP8OPT_ERR_ARG when
 * state is NULL or misaligned.
 */
FP8OPT_API int fp8_cast_adam_step_clipped_dev(
    const fp8opt_cast_item *grads, const fp8opt_param *params, int n, int fmt,
    float beta1, float beta2, float eps, float wd, int l2, float max_grad_norm,
    fp8opt_step_state *state, float *grad_norm_dev, uint32_t *found_inf_dev,
    void *stream);

/*
 * fp8_grad_norm: the global L2 norm of the unscaled gradient of a step call
 * (the quantity torch.nn.utils.clip_grad_norm_ clips; the run script's
 * --clip-grad), without a step.  Element i of record t is g = decode(g code)
 * * k_t with k_t = inv_loss_scale / g_scale, the step's own factor.  The norm
 * is sqrt(sum over t, in record order, of fl64(k_t^2 * fl64(S_t))), where
 * S_t = sum of decode(code)^2 over record t is taken exactly (every code value
 * is a multiple of 2^-16, so S_t is an integer count of 2^-32; the library
 * sums it in 128-bit integers), each sum over records is rounded to double,
 * and the root is correctly rounded.  The result does not depend on the
 * kernel schedule.  If some g is not finite (found_inf, the step's test) the
 * norm is +inf.
 *
 * Reads only the records' g, g_scale, g_fmt and numel (one byte per element);
 * the other fields must still be valid (same checks as fp8_adamw_step).
 * norm: host double, may be NULL (when set, the call waits for the stream);
 * norm_dev: device fp32, may be NULL; found_inf: host int, may be NULL.
 */
FP8OPT_API int fp8_grad_norm(const fp8opt_param *params, int n,
                             float inv_loss_scale, double *norm, float *norm_dev,
                             int *found_inf, void *stream);

/*
 * fp8_adam_step_clipped: fp8_adamw_step (l2 = 0) or fp8_adam_step (l2 = 1)
 * with the unscaled gradient clipped to a global L2 norm of max_grad_norm, as
 * torch.nn.utils.clip_grad_norm_ does between GradScaler.unscale_ and the
 * optimizer step.  The norm is fp8_grad_norm's; the clip coefficient is
 * c = max_grad_norm / (norm + 1e-6) in double, rounded to fp32, applied when
 * it is below 1 by multiplying every record's factor: k_t' = fl32(k_t * c).
 * found_inf is decided on the unclipped gradient, as the norm's +inf.  With
 * max_grad_norm <= 0 nothing is clipped (the step equals the unclipped one and
 * the norm is still reported).  One extra pass over the gradient codes (1 byte
 * per element) precedes the step.
 *
 * grad_norm: host double, may be NULL; grad_norm_dev: device fp32, may be
 * NULL.  Other arguments, results and errors as fp8_adamw_step; also
 * FP8OPT_ERR_ARG for l2 not 0 or 1, or a NaN max_grad_norm.
 */
FP8OPT_API int fp8_adam_step_clipped(const fp8opt_param *params, int n, float lr,
                                     float beta1, float beta2, float eps,
                                     float wd, int64_t step,
                                     float inv_loss_scale, int l2,
                                     float max_grad_norm, double *grad_norm,
                                     float *grad_norm_dev, int *found_inf,
                                     uint32_t *found_inf_dev, void *stream);

/*
 * Sharded steps.  When each of several ranks (one per GPU) owns the optimizer
 * state of a disjoint part of the tensor list (ZeRO-1 style; a tensor may be
 * cut into element ranges, pieces, on several ranks), a step needs
 * exchanges between ranks: found_inf must be combined (every rank skips if
 * any rank saw a non-finite gradient), with clipping the global norm taken
 * over all ranks' tensors, and for a cut tensor its per-tensor maxima
 * (the amax of the new first moment, max |g|, the new master's amax)
 * combined over its pieces.  The calls below split the step at those
 * exchanges; the caller runs the collectives (e.g. NCCL) between them.  On
 * one rank they give exactly fp8_adamw_step / fp8_adam_step /
 * fp8_adam_step_clipped.
 *
 * fp8_grad_norm_terms: for each of the n records, term_t = fl64(k_t^2 *
 * fl64(S_t)) with S_t the exact sum of squared code values (fp8_grad_norm's
 * definition), written to terms_dev[t] (device doubles); found_dev (device
 * uint32, may be NULL) receives this rank's found_inf.  A rank places its
 * terms at its records' positions of a vector of all records, zero elsewhere;
 * summing those vectors over ranks (any order: each position has one nonzero
 * addend) reproduces every term exactly.
 *
 * fp8_clip_coef: from the n terms of all records (in record order), norm =
 * sqrt(sum of terms in order) (+inf if *found_dev is nonzero; found_dev may be
 * NULL), written to norm_dev (device double, may be NULL), and the clip
 * coefficient (fp8_adam_step_clipped's) to clip_dev (device fp32): 1 when
 * max_grad_norm <= 0 or the norm is within it.
 *
 * fp8_adam_step_begin: the step's first pass over this rank's records
 * (found_inf, and the amax of each new first moment); found_dev (device
 * uint32, may be NULL) receives this rank's found_inf.  clip_dev: a device
 * fp32 clip coefficient (from fp8_clip_coef) or NULL for none; it scales the
 * gradient the moments see, while found_inf is still decided on the unclipped
 * gradient (GradScaler unscales, and finds any inf, before the norm is
 * clipped), so a gradient that overflows fp32 when unscaled skips the step
 * even where the clip coefficient would bring it back in range.
 * maxima_out (device uint32[2n], may be NULL): each record's per-tensor
 * maxima of this step, [0, n) the amax of the new first moment and [n, 2n)
 * max |g| (0 without a scaled second moment), as fp32 bits (NaN as
 * 0x7FC00000; the bits of these non-negative values order like the values,
 * NaN above +inf).
 *
 * fp8_adam_step_finish: the rest of the step (update and O3 weight copy) of
 * the same records, skipped when this rank's found_inf or *found_in_dev (the
 * value combined over ranks; may be NULL) is nonzero; found_dev (may be NULL)
 * receives the combined flag.  maxima_in (device uint32[2n], may be NULL):
 * the maxima to use instead of this rank's own, in maxima_out's layout.  A
 * record that is a piece of a tensor cut across ranks (an element range, with
 * the tensor's scales and bound) gives the whole tensor's result on its
 * elements when maxima_in holds the MAX over the pieces' maxima_out.
 * master_amax_out (device uint32[n], may be NULL): the amax of each O3
 * record's new FP16 master (fp32 bits); when it is given the O3 weight copy
 * does not run here but in fp8_adam_step_copy, which must follow, so that
 * the pieces' master amax can be combined first.  It must follow
 * fp8_adam_step_begin on the same stream with the same records and the same
 * hyperparameters, with no other step, cast or norm call on that stream in
 * between; otherwise FP8OPT_ERR_ARG and nothing is launched.
 *
 * fp8_adam_step_copy: the O3 weight copy of the records of the preceding
 * fp8_adam_step_finish (called with master_amax_out) from the given master
 * amax master_amax_in (device uint32[n], fp32 bits: w8_scale = 448 / amax,
 * with the cast's guards); skipped with the step.  Otherwise FP8OPT_ERR_ARG
 * and nothing is launched.
 *
 * Arguments otherwise as fp8_adamw_step; l2: 0 AdamW, 1 Adam with L2 decay.
 * None of these calls waits for the stream.
 */
FP8OPT_API int fp8_grad_norm_terms(const fp8opt_param *params, int n,
                                   float inv_loss_scale, double *terms_dev,
                                   uint32_t *found_dev, void *stream);
FP8OPT_API int fp8_clip_coef(const double *terms_dev, int n,
                             const uint32_t *found_dev, float max_grad_norm,
                             double *norm_dev, float *clip_dev, void *stream);
FP8OPT_API int fp8_adam_step_begin(const fp8opt_param *params, int n, float lr,
                                   float beta1, float beta2, float eps, float wd,
                                   int64_t step, float inv_loss_scale, int l2,
                                   const float *clip_dev, uint32_t *found_dev,
                                   uint32_t *maxima_out, void *stream);
FP8OPT_API int fp8_adam_step_finish(const fp8opt_param *params, int n, float lr,
                                    float beta1, float beta2, float eps,
                                    float wd, int64_t step,
                                    float inv_loss_scale, int l2,
                                    const float *clip_dev,
                                    const uint32_t *found_in_dev,
                                    uint32_t *found_dev,
                                    const uint32_t *maxima_in,
                                    uint32_t *master_amax_out, void *stream);
FP8OPT_API int fp8_adam_step_copy(const fp8opt_param *params, int n,
                                  const uint32_t *master_amax_in, void *stream);

/* Most shards one fp8_reduce_scaled call takes. */
#define FP8OPT_MAX_SHARDS 64

/* One tensor of a local FP8 reduction: k shards of numel codes each. */
typedef struct {
    const uint8_t *src;       /* k shards: shard j is the numel codes at
                                 src + j * stride (the call's in_fmt) */
    int64_t numel;            /* >= 0; 0 is allowed (amax 0, scale 1) */
    int64_t stride;           /* codes from one shard to the next, >= numel */
    const float *src_scale;   /* k fp32: shard j was encoded with scale
                                 src_scale[j], so its values are code * (1 /
                                 src_scale[j]); may be NULL when numel is 0 */
    uint8_t *codes;           /* out: numel codes of the result (out_fmt); may
                                 be the address of one of the shards (an
                                 in-place reduction), may not overlap them
                                 otherwise */
    float *amax;              /* out: one fp32, max |y| (as the cast's amax) */
    float *scale;             /* out: one fp32, fp8_max(out_fmt) / amax, with
                                 the cast's guards */
} fp8opt_reduce_item;

/*
 * fp8_reduce_scaled: local reduction of k FP8 shards per tensor, the
 * arithmetic half of an FP8 all-reduce (MS-AMP O1: weight gradients and their
 * AllReduce communication in FP8), e.g. the receive side of a reduce-scatter
 * or the k-way sum of gradient shards gathered on one GPU.
 *
 * Per element, in fp32 with every product and sum rounded on its own:
 *   y = (((x_0 + x_1) + x_2) + ... + x_{k-1}) * post,
 *   x_j = decode(code_j) * r_j,   r_j = 1 / src_scale[j] (one division)
 * then, per tensor, the cast of y exactly as fp8_cast_scaled casts an fp32
 * tensor: amax = max |y|, scale = fp8_max / amax, code = encode(y * scale).
 * post = 1 gives the sum, 1 / k the mean.  A NaN or infinite x_j, or an
 * overflowing sum, gives a non-finite y that takes the cast's non-finite codes.
 *
 * items: host array of n records; 1 <= k <= FP8OPT_MAX_SHARDS; in_fmt and
 * out_fmt: FP8OPT_E4M3 or FP8OPT_E5M2.  16-byte-aligned src and codes with a
 * stride that is a multiple of 16 take the vector path; other buffers a
 * scalar path.  Bytes per element: 2k + 1 (two passes over the shards).
 */
FP8OPT_API int fp8_reduce_scaled(const fp8opt_reduce_item *items, int n, int k,
                                 int in_fmt, int out_fmt, float post,
                                 void *stream);

/*
 * fp8_cast_adam_step_clipped: fp8_cast_scaled(grads, n, fmt) followed by
 * fp8_adam_step_clipped(params, n, ...) on the codes it wrote, in one call:
 * the cast's encode pass also sums the exact squares of the codes it writes
 * and decides found_inf, so the gradient norm costs no pass of its own (BF16
 * gradients, O2: 2 + 3 + 2 + 11 = 18 bytes per parameter, against 19 for the
 * two calls).  l2: 0 AdamW, 1 Adam with L2 decay; max_grad_norm <= 0 clips
 * nothing (the norm is still reported).  With max_grad_norm <= 0 and neither
 * grad_norm nor grad_norm_dev there is no norm to take: the cast's encode
 * pass is then fused with the step's first pass as in fp8_cast_adamw_step
 * (Adam with L2 decay, O2: 2 + 6 + 11 = 19 bytes per parameter, the first
 * pass reading the FP16 weights for the decay term).  Results, found_inf
 * semantics and
 * errors are those of the two calls made in turn; params[i] must take
 * grads[i]'s output as for fp8_cast_adamw_step.
 */
FP8OPT_API int fp8_cast_adam_step_clipped(const fp8opt_cast_item *grads,
                                          const fp8opt_param *params, int n,
                                          int fmt, float lr, float beta1,
                                          float beta2, float eps, float wd,
                                          int64_t step, float inv_loss_scale,
                                          int l2, float max_grad_norm,
                                          double *grad_norm, float *grad_norm_dev,
                                          int *found_inf, uint32_t *found_inf_dev,
                                          void *stream);

/*
 * fp8_reduce_scaled_norm: fp8_reduce_scaled, whose encode pass also sums the
 * exact squares of the codes it writes, so that the reduced gradients' norm
 * terms come without a pass of their own: terms_dev[t] (device doubles, one
 * per item) = fp8_grad_norm_terms' term of item t's output codes with the
 * factor k_t = inv_loss_scale / (item t's output scale), and found_dev
 * (device uint32, may be NULL) = whether some code value times k_t is not
 * finite.  For the sharded step's exchange (see fp8_grad_norm_terms); same
 * arguments and errors as fp8_reduce_scaled otherwise.
 */
FP8OPT_API int fp8_reduce_scaled_norm(const fp8opt_reduce_item *items, int n,
                                      int k, int in_fmt, int out_fmt, float post,
                                      float inv_loss_scale, double *terms_dev,
                                      uint32_t *found_dev, void *stream);

/*
 * fp8_reduce_scaled_begin and fp8_reduce_scaled_finish: fp8_reduce_scaled
 * split at its one per-tensor quantity, the amax of the reduced values, for
 * a tensor reduced in pieces on several ranks (each rank reduces an element
 * range of every shard; the MS-AMP "Optimization Level" page's O3 paragraph
 * names ZeRO, which cuts the optimizer's work across data-parallel ranks).
 *
 * begin: the amax pass; amax_bits_dev[i] (device uint32[n]) receives item i's
 * amax as fp32 bits (NaN as 0x7FC00000; the bits of these non-negative values
 * order like the values).  The caller combines the pieces of a tensor by MAX
 * (e.g. an all-reduce of int32 maxima over ranks).
 *
 * finish: the encode pass with item i's amax taken from amax_bits_dev[i] (the
 * combined value): codes, amax and scale exactly as fp8_reduce_scaled writes
 * them for that amax, so the pieces of a tensor give its whole codes.
 * limbs_dev (device int64[4n], may be NULL): item i's exact sum of the
 * squared values of its output codes (fp8_grad_norm_terms' S, units of
 * 2^-32) as four 32-bit limbs, low first (limbs_dev[4i + j] < 2^32), which a
 * SUM over fewer than 2^31 ranks keeps exact; with it, found_dev (device
 * uint32, may be NULL) receives whether some output code times
 * inv_loss_scale / scale is not finite (the step's test).  found_dev without
 * limbs_dev is FP8OPT_ERR_ARG.
 *
 * fp8_norm_terms_from_limbs: terms_dev[t] (device doubles) = the norm term
 * fl64(k_t^2 * fl64(S_t * 2^-32)) of tensor t from its limbs (limbs_dev[4t ..
 * 4t + 3], possibly summed over ranks: each below 2^63, the top one below
 * 2^32) and k_t = inv_loss_scale / scale_t, scale_t = fp8_max(fmt) / amax_t
 * with the cast's guards (amax_bits_dev[t]); the terms fp8_clip_coef sums.
 *
 * Arguments otherwise as fp8_reduce_scaled / fp8_reduce_scaled_norm.
 */
FP8OPT_API int fp8_reduce_scaled_begin(const fp8opt_reduce_item *items, int n,
                                       int k, int in_fmt, float post,
                                       uint32_t *amax_bits_dev, void *stream);
FP8OPT_API int fp8_reduce_scaled_finish(const fp8opt_reduce_item *items, int n,
                                        int k, int in_fmt, int out_fmt,
                                        float post, const uint32_t *amax_bits_dev,
                                        float inv_loss_scale, int64_t *limbs_dev,
                                        uint32_t *found_dev, void *stream);
FP8OPT_API int fp8_norm_terms_from_limbs(const int64_t *limbs_dev,
                                         const uint32_t *amax_bits_dev, int n,
                                         int fmt, float inv_loss_scale,
                                         double *terms_dev, void *stream);

/* Text of a status code (static storage). */
FP8OPT_API const char *fp8opt_strerror(int status);

/* Detail of the last failing call on this host thread (static or thread-local
 * storage, valid until the next call on the thread). */
FP8OPT_API const char *fp8opt_last_error(void);

/* Per-kernel timing (off by default).  While it is on, every kernel the
 * library launches is bracketed by two CUDA events recorded on the call's
 * stream, so a caller can measure each kernel's device time inside its own
 * timed region.  fp8opt_timing_enable(1) clears the record and starts
 * recording; fp8opt_timing_enable(0) stops.  fp8opt_timing_read waits for the
 * recorded events and returns, for one kernel name ("cast_amax",
 * "cast_encode", "step_amax", "step_update", "step_w8", "cast_step_amax",
 * "reduce_amax", "reduce_encode", "grad_norm", "grad_norm_terms", "clip_coef",
 * "found"), the launches
 * recorded since enabling and their summed duration in milliseconds.  Returns
 * FP8OPT_ERR_ARG for an unknown name or NULL outputs. */
FP8OPT_API int fp8opt_timing_enable(int on);
FP8OPT_API int fp8opt_timing_read(const char *kernel, int *launches,
                                  double *total_ms);

/* Frees every workspace the library holds, on every device.  The caller must
 * make sure no call's work is still running. */
FP8OPT_API void fp8opt_release(void);

/* Frees the workspace of one stream (on the current device), e.g. after the
 * CUDA graphs captured on it are destroyed, so that the stream takes any
 * tensor list again.  The caller must make sure no work that uses it is
 * still running. */
FP8OPT_API void fp8opt_release_stream(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8OPT_H */

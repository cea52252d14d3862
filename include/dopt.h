/*
 * dopt: the ZeRO-1 distributed-optimizer step over a contiguous flat
 * gradient/parameter buffer, on one GPU, with D data-parallel ranks held as
 * D replica buffers in device memory.
 *
 * The operations follow the Megatron-LM distributed-optimizer page
 * ("04 · 分布式优化器"):
 *   - the flat buffer cut into buckets, each bucket split into D equal
 *     contiguous ranges, rank r owning range r (§2, §3);
 *   - Range and the four ranges of every (param, rank) piece (§4.1);
 *   - the bucket-wise reduce-scatter of the grads, scaled first (§4.2, §5);
 *   - the shard going to fp32 main grads, Adam on the shard, the write-back
 *     of the updated shard into the param buffer (§4.3);
 *   - the all-gather of the params (§4.4).
 *
 * Conventions
 *   - Every call returns DOPT_OK (0) or a negative DOPT_E_* code; the text
 *     of the last error on the calling thread is dopt_last_error().
 *   - Device buffers belong to the caller.  The library owns a dopt_layout
 *     and its device tables and frees both in dopt_layout_free.
 *   - dopt_step and dopt_gather are asynchronous on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).  They check their
 *     arguments on the host before anything is queued, report launch errors
 *     through cudaGetLastError, and never allocate or synchronise.  Faults
 *     inside a kernel surface at the caller's next synchronisation.
 *   - The step, all-reduce, gather, norm and finalize kernels are launched
 *     as programmatic dependents of the kernel before them on the stream
 *     (the counted step's kernel of its counter kernel, the clipped step's
 *     passes of the launch before each): when that kernel
 *     lets its dependents start early (as the library's own kernels do),
 *     their CTAs may become resident during its last wave and look up their
 *     runs, but they read no grad, state or param, and write nothing,
 *     before it has completed.  (The clipped step's second pass loads
 *     master/m/v before its norm pass completes: neither of the call's
 *     earlier kernels writes them, and the call's first launch is
 *     stream-ordered, so everything queued before the call has completed
 *     by then.)  Stream order is unchanged for everything else (copies,
 *     events, kernels that do not let dependents start).
 *   - Buffer-indexed arrays hold one element per position of the padded
 *     buffer (padded_numel elements).  Padding positions belong to no param;
 *     the step neither reads nor writes them in any buffer.
 */
#ifndef DOPT_H
#define DOPT_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DOPT_OK 0
#define DOPT_E_ARG (-1)    /* invalid argument (null, out of range) */
#define DOPT_E_LAYOUT (-2) /* a bucket does not divide by R (distributed-optimizer
                              page, §4.1 and §5) */
#define DOPT_E_ALIGN (-3)  /* a device pointer is not 16-byte aligned */
#define DOPT_E_CUDA (-4)   /* a CUDA runtime call failed */
#define DOPT_E_STATE (-5)  /* the layout has no device tables on this device */
#define DOPT_E_NOMEM (-6)  /* host allocation failed */

/* Largest number of simulated data-parallel ranks. */
#define DOPT_MAX_D 64

/* Range(start, end): the half-open interval [start, end)
 * (distributed-optimizer page, §4.1). */
typedef struct {
    int64_t start;
    int64_t end;
} dopt_range;

/*
 * One (param, rank) piece: the part of a param that falls in one rank's
 * range of its bucket, with the four ranges of the distributed-optimizer
 * page, §4.1:
 *   gbuf_world            the piece's range in the whole flat buffer
 *   gbuf_world_in_bucket  the same, relative to the start of its bucket
 *   gbuf_local            the same, relative to the start of the rank's range
 *   param                 the same, relative to the start of the param
 * All four have the same length; they differ by a translation.
 */
typedef struct {
    dopt_range gbuf_world;
    dopt_range gbuf_world_in_bucket;
    dopt_range gbuf_local;
    dopt_range param;
    int32_t param_id;
    int32_t bucket_id;
    int32_t rank;
    int32_t reserved;
} dopt_piece;

/*
 * Layout parameters, in the order of the boundary's own statement of them
 * (D, bucket_elems, pad_unit), so that a caller who sets just those three
 * positionally gets one instance and a zero reserved word:
 *   D             simulated data-parallel ranks (replica buffers),
 *                 1..DOPT_MAX_D
 *   bucket_elems  a bucket is closed as soon as its unpadded element count
 *                 reaches bucket_elems; 0 puts all params in one bucket
 *                 (distributed-optimizer page, §2)
 *   pad_unit      every bucket is padded at its end to a multiple of
 *                 R * pad_unit elements (>= 1), R = D / instances (§4.1, §5:
 *                 a bucket must divide by the rank count)
 *   instances     distributed-optimizer instances (distributed-optimizer
 *                 page, §5, num_distributed_optimizer_instances); 0 or 1: one
 *                 instance.  D must divide by it.  The ranks form
 *                 `instances` groups of R = D / instances consecutive ranks;
 *                 each bucket is split into R ranges, rank r of every group
 *                 owning range r; the grads are reduced inside each group in
 *                 rank order and the groups' sums are then added in group
 *                 order (the all-reduce across instances).
 *   reserved      must be 0
 */
typedef struct {
    int32_t D;
    int64_t bucket_elems;
    int32_t pad_unit;
    int32_t instances;
    int32_t reserved;
} dopt_layout_cfg;

/*
 * AdamW hyper-parameters.  grad_scale is the gradient scaling factor applied
 * to every replica's grads before the reduction (distributed-optimizer
 * page, §5).
 * Valid ranges: lr >= 0, 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0,
 * weight_decay >= 0, grad_scale finite.
 */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    float grad_scale;
} dopt_adam_cfg;

/*
 * Gradient element type of the replica buffers.  DOPT_FP16 is IEEE
 * binary16 (the tutorial's mixed-precision section and the ZeRO page's
 * state table list FP16 grads next to BF16): widened exactly; where a
 * reduced grad goes back into the grad type (DOPT_STEP_ROUND_GRAD, the
 * all-reduce) it is rounded to nearest even and overflows to Inf beyond
 * 65504.
 */
typedef enum { DOPT_BF16 = 0, DOPT_FP32 = 1, DOPT_FP16 = 2 } dopt_dtype;

/* dopt_step flags. */
#define DOPT_STEP_GATHER 1u /* fuse the all-gather: write all D replicas */
/*
 * The grad replicas are pinned host buffers (cudaHostAlloc, or
 * cudaHostRegister'ed) that the device reads in place over the host link,
 * instead of device buffers: no staging copy and no device memory for the
 * grads.  Each pointer is resolved with cudaPointerGetAttributes; anything
 * that is not registered host memory with a device mapping is refused with
 * DOPT_E_ARG before any launch.  Accepted by dopt_step, dopt_step_buckets,
 * dopt_step_allreduce (which then writes the host buffers) and
 * dopt_step_clipped.
 */
#define DOPT_STEP_HOST_GRADS 2u
/*
 * Round each reduced grad to the grad type before clipping and Adam (bf16
 * and fp16: nearest even; fp32 grads are unchanged), as when the
 * reduce-scatter writes into the grad buffer and the optimizer copies the
 * shard from there (distributed-optimizer page, §4.2-§4.3).  main_grad_out /
 * main_grad then hold the rounded values and the clipped step's norm is
 * taken over them.  Without the flag the fp32 sum feeds Adam directly.
 * Accepted by every step entry point.
 */
#define DOPT_STEP_ROUND_GRAD 4u
/*
 * The param replicas hold IEEE fp16 instead of bf16: the write-back rounds
 * the fp32 master to fp16 (nearest even, Inf beyond 65504).  The all-gather
 * copies 16-bit values and is the same for both types.
 */
#define DOPT_STEP_PARAMS_FP16 16u
/*
 * The param replicas may be pinned host buffers (cudaHostAlloc, or
 * cudaHostRegister'ed, with a device mapping) that the write-back and
 * all-gather store into in place over the host link, each replica either
 * that or device memory: a caller that needs one replica of the updated
 * params on the host gets it without a device copy and a separate transfer.
 * Each pointer is resolved with cudaPointerGetAttributes; anything that is
 * neither device memory nor registered host memory with a device mapping is
 * refused with DOPT_E_ARG before any launch.  Accepted by every step entry
 * point (the pages store params on the devices; this is an addition of the
 * library for callers whose grads and params cross the host link).
 */
#define DOPT_STEP_HOST_PARAMS 64u
/*
 * Read each tile's grads and master/m/v through shared memory: one thread
 * of every CTA issues 1-D bulk copies (the SM's TMA unit, from this
 * GPU's own memory into that CTA's shared memory; no cluster multicast),
 * and the CTA computes from shared memory once they complete.  The results
 * are those of the default path (128-bit vector loads into registers), bit
 * for bit.  The pages suggest staging bucket tiles this way; the library
 * keeps it as a measured alternative, not the default.  Accepted by
 * dopt_step, dopt_step_buckets and dopt_step_counted, for layouts with one
 * instance and D in {1, 2, 4, 8, 16} and device grads (DOPT_E_ARG
 * otherwise).  A CTA whose copies do not complete within 2 s skips its
 * tile and is counted (dopt_stage_timeouts) instead of hanging.
 */
#define DOPT_STEP_STAGE 32u

typedef struct dopt_layout dopt_layout;

/*
 * Build the flat-buffer layout and its four-way range map
 * (distributed-optimizer page, §2, §3, §4.1, §5).
 *
 *   param_sizes[n_params]  element count of each param (>= 0), in buffer
 *                          order; params sit at consecutive offsets.
 *   wd_mask[n_params]      nullable; nonzero where the param takes weight
 *                          decay (NULL: every param does).
 *   cfg                    D, bucket_elems, pad_unit, instances (see
 *                          dopt_layout_cfg).
 *   out                    receives a new layout; free it with
 *                          dopt_layout_free.
 *
 * Buckets are greedy: params are appended to the open bucket, which closes
 * as soon as its unpadded count reaches bucket_elems; a param never spans
 * two buckets; each bucket is padded to a multiple of R * pad_unit, and rank
 * r (of each instance) owns [start + r*S, start + (r+1)*S) of it with
 * S = size / R, R = D / instances.  Pieces carry the rank inside the
 * instance (0..R-1).
 * Host only: makes no CUDA call.  Errors: DOPT_E_ARG, DOPT_E_NOMEM.
 */
int dopt_build_range_map(const int64_t *param_sizes, int32_t n_params, const uint8_t *wd_mask,
                         const dopt_layout_cfg *cfg, dopt_layout **out);

/*
 * Sizes of a layout: the padded length of the flat buffer (distributed-
 * optimizer page, §2: every param's grads in one contiguous buffer, each
 * bucket padded so that it divides by the rank count, §4.1 and §5), the
 * bucket count (§2) and the piece count (§4.1: one piece per (param, rank)
 * overlap).  Any output pointer may be NULL.  Host only.  Errors: DOPT_E_ARG
 * (NULL layout).
 */
int dopt_layout_query(const dopt_layout *layout, int64_t *padded_numel, int32_t *n_buckets,
                      int32_t *n_pieces);

/*
 * Copy the bucket ranges, padding included, in buffer order, into
 * buckets[n_buckets] (caller-owned host array; distributed-optimizer page,
 * §2: the flat buffer cut into buckets; §3: each bucket split into equal
 * contiguous rank ranges).  Host only.  Errors: DOPT_E_ARG (NULL argument).
 */
int dopt_layout_buckets(const dopt_layout *layout, dopt_range *buckets);

/*
 * Copy the pieces into pieces[n_pieces] (caller-owned host array), sorted by
 * (bucket, rank, gbuf_world.start): for every param and every rank range it
 * overlaps, the four ranges of the distributed-optimizer page, §4.1
 * (gbuf_world, gbuf_world_in_bucket, gbuf_local, param; see dopt_piece).
 * Host only.  Errors: DOPT_E_ARG (NULL argument).
 */
int dopt_layout_pieces(const dopt_layout *layout, dopt_piece *pieces);

/*
 * Copy each param's full range [offset, offset + size) in the flat buffer
 * into params[n_params] (caller-owned host array, in the order the params
 * were given): the param's place in the contiguous buffer of the
 * distributed-optimizer page, §2, from which the §4.1 ranges of its pieces
 * are cut.  Params sit at consecutive offsets inside their bucket; padding
 * follows the last param of a bucket.  Host only.  Errors: DOPT_E_ARG (NULL
 * argument).
 */
int dopt_layout_param_offsets(const dopt_layout *layout, dopt_range *params);

/* The same call as dopt_layout_param_offsets, under its earlier name. */
int dopt_layout_param_ranges(const dopt_layout *layout, dopt_range *params);

/*
 * Copy the layout's kernel tables to the current CUDA device: the owned
 * runs of the buffer (stretches of the §4.1 pieces of the distributed-
 * optimizer page with one owner rank and one weight-decay flag, merged) and
 * a per-tile index into them.  Allocates device memory once; must precede
 * dopt_step / dopt_gather on that device and any stream capture.  Calling
 * it again on the same device is a no-op; on another device it moves the
 * tables there.  Synchronous.  Errors: DOPT_E_ARG, DOPT_E_CUDA.
 */
int dopt_layout_to_device(dopt_layout *layout);

/* Free a layout (the range map of dopt_build_range_map) and its device
 * tables.  NULL is ignored.  Library bookkeeping: the pages have no
 * counterpart. */
void dopt_layout_free(dopt_layout *layout);

/*
 * One distributed-optimizer step for all D simulated ranks, fused into one
 * kernel launch over the whole buffer (distributed-optimizer page, §4.2-§4.4):
 *
 *   for every owned element i (rank q owns it, param p holds it):
 *     g      = fp32 sum over r = 0..D-1, in rank order, of
 *              grad_scale * float(grad_replicas[r][i])   (each op rounded);
 *              with several instances, the rank-order sum inside each
 *              instance, then those sums in instance order
 *     m      = beta1*m + (1-beta1)*g
 *     v      = beta2*v + (1-beta2)*(g*g)
 *     w      = w * (1 - lr*weight_decay)          (only if p decays)
 *     w      = w - step_size * (m / (sqrt(v)/bc2_sqrt + eps))
 *     param_replicas[r][i] = bf16_rne(w)   for every r (DOPT_STEP_GATHER;
 *                                          fp16_rne(w) with DOPT_STEP_PARAMS_FP16)
 *                                          or, without the flag, for the
 *                                          replica of rank q in every
 *                                          instance
 *     main_grad_out[i] = g                 (when main_grad_out is not NULL)
 *   with step_size = lr / (1 - beta1^step), bc2_sqrt = sqrt(1 - beta2^step)
 *   and the scalars (1-beta1), (1-beta2), (1-lr*wd), step_size, bc2_sqrt
 *   evaluated in double on the host and rounded to float once.  Every fp32
 *   multiply, add, divide and square root is rounded on its own (no fused
 *   multiply-add).
 *
 *   layout          built by dopt_build_range_map, tables on this device
 *   cfg             AdamW hyper-parameters (host pointer)
 *   step            1-based step count t
 *   grad_replicas   host array of D device pointers, each padded_numel
 *                   elements of grad_dtype; read only
 *   master, exp_avg, exp_avg_sq
 *                   device fp32, padded_numel elements each, buffer-indexed
 *                   (the union of all D ranks' shards); updated in place
 *   param_replicas  host array of D device pointers, bf16 (fp16 with
 *                   DOPT_STEP_PARAMS_FP16), padded_numel each
 *   flags           DOPT_STEP_GATHER, DOPT_STEP_HOST_GRADS, DOPT_STEP_ROUND_GRAD,
 *                   DOPT_STEP_PARAMS_FP16
 *   main_grad_out   nullable device fp32[padded_numel]: the reduce-scattered
 *                   fp32 main grad of every owned element
 *   stream          CUDA stream to launch on
 *
 * Every device pointer must be 16-byte aligned (DOPT_E_ALIGN otherwise).
 * The D grad replicas must not overlap any output.  Errors: DOPT_E_ARG,
 * DOPT_E_ALIGN, DOPT_E_STATE, DOPT_E_CUDA.
 */
int dopt_step(const dopt_layout *layout, const dopt_adam_cfg *cfg, int64_t step,
              const void *const *grad_replicas, dopt_dtype grad_dtype, float *master,
              float *exp_avg, float *exp_avg_sq, void *const *param_replicas, uint32_t flags,
              float *main_grad_out, cudaStream_t stream);

/*
 * The step over the contiguous bucket range [first_bucket, first_bucket +
 * n_buckets) only, one launch.  The per-bucket form of the distributed
 * optimizer page's pipeline (§2, §4.2: each bucket's reduce-scatter starts
 * as soon as the bucket is full, so its update can follow on its own): the
 * caller may launch the buckets one by one, on one or several streams, in
 * any order; together they give exactly dopt_step's result, since every
 * element belongs to one bucket.  Arguments otherwise as dopt_step (buffers
 * are still whole-buffer pointers).  n_buckets = 0 is a no-op.
 * Errors: as dopt_step, and DOPT_E_ARG for a range outside the layout.
 */
int dopt_step_buckets(const dopt_layout *layout, const dopt_adam_cfg *cfg, int64_t step,
                      int32_t first_bucket, int32_t n_buckets, const void *const *grad_replicas,
                      dopt_dtype grad_dtype, float *master, float *exp_avg, float *exp_avg_sq,
                      void *const *param_replicas, uint32_t flags, float *main_grad_out,
                      cudaStream_t stream);

/*
 * Step counter in device memory for dopt_step_counted: 64 bytes, 16-byte
 * aligned, owned by the caller, zeroed by the caller before first use.
 *   next_step  1-based number of the step the next dopt_step_counted launch
 *              takes.  The caller sets it (to 1, or to the step to resume
 *              at); every such launch reads it on the device and adds one.
 *   status     written by every launch: 0, or DOPT_COUNTER_BAD_STEP when
 *              next_step was outside 1 .. 2^62; such a launch changes
 *              nothing else (not the counter, the state or the params).
 *   scratch    the library's: the two Adam scalars that depend on the step
 *              number, for the step last taken, and a copy of the status.
 *   exact_steps, undecided_steps
 *              diagnostics of the device's evaluation of those two scalars
 *              (see dopt_step_counted): the steps whose scalars needed the
 *              slow exact evaluation, and the steps where even that could
 *              not tell which float pow(beta, t) leads to.  The library only
 *              adds to them.
 */
typedef struct {
    int64_t next_step;
    int32_t status;
    int32_t reserved;
    float scratch[4];
    uint32_t exact_steps;
    uint32_t undecided_steps;
    uint32_t reserved2[6];
} dopt_step_counter;

#define DOPT_COUNTER_BAD_STEP 1

/*
 * dopt_step with the step number taken from a counter in device memory
 * instead of a host argument, and the counter advanced on the device.  A
 * kernel of four threads reads counter->next_step = t, evaluates the step's
 * two scalars that depend on t into counter->scratch and stores t + 1; then
 * the step kernel of dopt_step runs with those scalars.  dopt_step takes
 * beta^t from the C library's pow; the device has none, so it computes
 * beta^t by binary powering with a bound on its error, and evaluates each
 * scalar at both ends of the interval where pow's result must lie (pow is
 * within 0.52 ulp of the exact power).  When the two ends give the same
 * float it is dopt_step's float.  Otherwise (rarely) it evaluates beta^t
 * again in double-double and the scalar at every double within 0.52 ulp of
 * that value, and counts the step in counter->exact_steps; if those still
 * give two floats, it takes the one of the nearest double and counts the
 * step in counter->undecided_steps (the only case in which the counted
 * step may differ from dopt_step, by one float ulp of a scalar).  The first kernel is launched as a
 * programmatic dependent of the kernel before it on the stream: it may start
 * early, but it reads the final counter and writes only after that kernel
 * has completed.  The launches and
 * their arguments do not depend on t, so a sequence captured once (a CUDA
 * graph) replays every later step.  The pages describe no such counter:
 * it is an addition of this library for graph replay.
 *   counter  device dopt_step_counter (see there); read and written by the
 *            device only, in stream order
 * Other arguments, the arithmetic and the errors as dopt_step, plus
 * DOPT_E_ARG for a NULL counter and DOPT_E_ALIGN for a misaligned one.  A
 * bad next_step is reported in counter->status, not by the return value.
 */
int dopt_step_counted(const dopt_layout *layout, const dopt_adam_cfg *cfg,
                      dopt_step_counter *counter, const void *const *grad_replicas,
                      dopt_dtype grad_dtype, float *master, float *exp_avg, float *exp_avg_sq,
                      void *const *param_replicas, uint32_t flags, float *main_grad_out,
                      cudaStream_t stream);

/*
 * The all-reduce of the grads on its own (distributed-optimizer page, §5,
 * force_all_reduce: all ranks keep the whole reduced grad, e.g. to save full weight grads;
 * distributed-training tutorial, "AllReduce" = reduce-scatter followed by
 * all-gather).  For every owned element i:
 *     g = fp32 sum over r in rank order of grad_scale * float(grad_replicas[r][i])
 *     grad_replicas[r][i] = g rounded to the grad type (bf16, fp16: nearest
 *                           even)
 * for every r, in place.  Padding is not written.
 *   grad_replicas  host array of D device pointers (16-byte aligned),
 *                  padded_numel elements of grad_dtype each; read and written
 * Asynchronous on `stream`.  Errors: DOPT_E_ARG, DOPT_E_ALIGN, DOPT_E_STATE,
 * DOPT_E_CUDA.
 */
int dopt_allreduce(const dopt_layout *layout, void *const *grad_replicas, dopt_dtype grad_dtype,
                   float grad_scale, cudaStream_t stream);

/*
 * dopt_step with force_all_reduce (distributed-optimizer page, §5): the
 * same step, one launch, which also writes the reduced grad of every owned element into every grad
 * replica, as dopt_allreduce does (the Adam update uses the fp32 reduced
 * grad, unchanged).  grad_replicas are read and then written.  Arguments and
 * errors otherwise as dopt_step.
 */
int dopt_step_allreduce(const dopt_layout *layout, const dopt_adam_cfg *cfg, int64_t step,
                        void *const *grad_replicas, dopt_dtype grad_dtype, float *master,
                        float *exp_avg, float *exp_avg_sq, void *const *param_replicas,
                        uint32_t flags, float *main_grad_out, cudaStream_t stream);

/*
 * The all-gather of the params on its own (distributed-optimizer page,
 * §4.4): for every rank q and every element q owns, copy param_replicas[q][i] into every other
 * replica of q's instance.  Padding is not copied.  param_replicas: host
 * array of D device pointers to 16-bit params (bf16 or fp16: the copy does
 * not look at the values), 16-byte aligned.  Asynchronous on `stream`.
 * Errors: DOPT_E_ARG, DOPT_E_ALIGN, DOPT_E_STATE, DOPT_E_CUDA.
 */
int dopt_gather(const dopt_layout *layout, void *const *param_replicas, cudaStream_t stream);

/* Bytes of device workspace that dopt_step_clipped needs (16-byte aligned). */
#define DOPT_CLIP_WORKSPACE_BYTES 16384

/*
 * dopt_step_clipped flag: skip the update when any owned element's reduced
 * grad (after DOPT_STEP_ROUND_GRAD's rounding, when set) is Inf or NaN.
 * The first launch counts such elements; when the count is not 0 the
 * second launch stores nothing (master, exp_avg, exp_avg_sq and every param
 * replica keep their values), the coefficient is reported as NaN, and the
 * count is reported in the dopt_clip_report.  The pages give no rule for
 * non-finite grads (the tutorial's §8.2 only notes that FP16 overflows
 * easily); this is the usual mixed-precision practice of dropping a step
 * whose grads overflowed.  Refused (DOPT_E_ARG) by every other entry point.
 */
#define DOPT_STEP_SKIP_NONFINITE 8u

/*
 * What dopt_step_clipped reports through norm_out.  Without
 * DOPT_STEP_SKIP_NONFINITE only norm and coef are written (norm_out may
 * then point to just 2 floats); with it, the whole 16-byte report.
 */
typedef struct {
    float norm;         /* global norm of the reduced grads */
    float coef;         /* clipping coefficient; NaN when the step was skipped */
    uint64_t nonfinite; /* owned elements whose reduced grad is Inf or NaN */
} dopt_clip_report;

/*
 * The step with global grad-norm clipping (distributed-training tutorial,
 * §8.3: the norm sqrt(sum ||g||^2) over every rank's shard is needed before
 * the optimizer update).  Two passes over memory on `stream` (four
 * launches: a one-CTA reset of the workspace, the first pass, a one-CTA
 * finalize kernel, the second pass):
 *
 *   1. the fused reduce-scatter writes every owned element's reduced fp32
 *      grad g (as in dopt_step) into main_grad, and the global
 *      norm^2 = sum of g^2 over all owned elements is accumulated (fp32
 *      squares summed per 8 elements, then in fp64 within each CTA, the
 *      CTAs' partials added exactly and rounded once, so the result does
 *      not depend on the grid or on the order of the CTAs); the coefficient
 *      c = min(1, max_norm / (norm + 1e-6)) is evaluated in fp64 and rounded
 *      to float;
 *   2. the AdamW step, write-back and (with DOPT_STEP_GATHER) all-gather of
 *      dopt_step, with g replaced by fl(g * c).
 *
 *   max_norm    > 0, finite
 *   main_grad   device fp32[padded_numel], written: the reduced grads
 *               before clipping (padding untouched)
 *   workspace   device, DOPT_CLIP_WORKSPACE_BYTES, 16-byte aligned, owned by
 *               the caller; holds the exact sum of squares between the
 *               launches (zeroed by the call itself); calls that share a
 *               workspace must not overlap on the GPU
 *   norm_out    nullable device pointer, 8-byte aligned, to a
 *               dopt_clip_report: norm and c (and, with
 *               DOPT_STEP_SKIP_NONFINITE, the count of non-finite reduced
 *               grads)
 *   flags       as in dopt_step, plus DOPT_STEP_SKIP_NONFINITE
 *   other arguments as in dopt_step.
 *
 * The norm's fp32 squares and pairwise sums differ from an exact sum by at
 * most a few units in the 24th bit, so c is within ~2e-7 relative of the
 * exactly rounded coefficient.  Errors: as dopt_step.
 */
int dopt_step_clipped(const dopt_layout *layout, const dopt_adam_cfg *cfg, int64_t step,
                      float max_norm, const void *const *grad_replicas, dopt_dtype grad_dtype,
                      float *master, float *exp_avg, float *exp_avg_sq,
                      void *const *param_replicas, uint32_t flags, float *main_grad,
                      void *workspace, float *norm_out, cudaStream_t stream);

/* Size of the static device scratch behind dopt_step_clipped_noalloc. */
#define DOPT_NOALLOC_SCRATCH_BYTES 16384

/*
 * dopt_step_clipped with the step number taken from, and advanced in, a
 * device counter, as dopt_step_counted does for dopt_step: the counter
 * kernel, then the launches of dopt_step_clipped, whose step pass takes
 * the two step-dependent scalars and the status from the counter.  The
 * launches do not depend on the step number, so a captured sequence replays
 * every later step.  With a bad next_step (see dopt_step_counter) the norm
 * pass still writes main_grad and norm_out; master, exp_avg, exp_avg_sq and
 * the params are not written.  A step that DOPT_STEP_SKIP_NONFINITE skips
 * is not counted: next_step is left as it was before the call.  The pages
 * describe no such counter: it is an
 * addition of this library for graph replay.  Arguments and errors as
 * dopt_step_clipped, plus those of dopt_step_counted for `counter`.
 */
int dopt_step_clipped_counted(const dopt_layout *layout, const dopt_adam_cfg *cfg,
                              dopt_step_counter *counter, float max_norm,
                              const void *const *grad_replicas, dopt_dtype grad_dtype,
                              float *master, float *exp_avg, float *exp_avg_sq,
                              void *const *param_replicas, uint32_t flags, float *main_grad,
                              void *workspace, float *norm_out, cudaStream_t stream);

/*
 * dopt_step_clipped for callers that cannot allocate device memory on the
 * step's path.  The pages have no counterpart: this entry point exists for
 * such callers, not for the method.
 *
 * Who needs it: code whose device memory belongs to a framework's caching
 * allocator (a raw cudaMalloc would bypass that allocator's budget and
 * bookkeeping), and training loops that cannot take the device-wide
 * synchronisation that cudaFree, and a cudaMalloc that has to grow the
 * heap, can cause.  Such a caller cannot hand dopt_step_clipped a fresh
 * workspace, so this variant keeps the norm pass's scratch (the exact sum
 * of squares, norm and coefficient) in a file-scope
 * `static __device__` array of DOPT_NOALLOC_SCRATCH_BYTES inside the
 * library.  Every GPU that loads the library holds that array until the
 * process exits.
 *
 * The entry point calls no cudaMalloc, cudaFree or other allocating
 * routine.  The caller still passes all inputs and outputs (main_grad
 * included), and the layout's device tables must already be on the device
 * (dopt_layout_to_device, which allocates, belongs to set-up).
 *
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and remembers it for the
 * life of the process; make that first call on each device before any
 * stream capture.  A cudaDeviceReset of that device destroys the array
 * with the context, and the remembered address is then stale: after a
 * reset, do not call this entry point again in the same process.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Each call zeroes what must start at zero (the
 * accumulator, the special-value bits and the non-finite count, with a
 * one-CTA kernel launched on `stream` before the norm pass); the rest is
 * overwritten before it is read.  Calls whose executions overlap on the GPU
 * (other streams, other layouts, other threads) race on the array: the
 * caller must order them.
 *
 * Size: the norm pass uses a fixed 1,856 bytes of the array, whatever the
 * buffer size.
 *
 * Arguments, results and errors otherwise as dopt_step_clipped (without
 * `workspace`, and without DOPT_STEP_SKIP_NONFINITE, which it refuses).
 */
int dopt_step_clipped_noalloc(const dopt_layout *layout, const dopt_adam_cfg *cfg, int64_t step,
                              float max_norm, const void *const *grad_replicas,
                              dopt_dtype grad_dtype, float *master, float *exp_avg,
                              float *exp_avg_sq, void *const *param_replicas, uint32_t flags,
                              float *main_grad, float *norm_out, cudaStream_t stream);

/* Device-side checks (library infrastructure for testing; the pages have
 * no counterpart): a test build of the library, compiled with
 * DOPT_DEVICE_CHECKS defined; built by build(checked=True) as
 * libdopt_checked.so).  In that build every kernel checks, before each
 * vector or element access, that the index lies inside the buffers (all of
 * a launch's buffers are padded_numel long) and that a vector starts on an
 * 8-element boundary; a failed check sets its DOPT_CHECK_* bit, records the
 * first bad element index and skips the access instead of making it.
 * These are the kernels' own guards against a wrong run table or index
 * arithmetic; valid inputs never fail them.
 *
 * Reads the current device's record: *flags (DOPT_CHECK_* bits, 0 if no
 * check failed) and *first_bad (the first failing element index, -1 if
 * none); with reset != 0 it then clears the record.  Synchronous (it waits
 * for the device's work to finish).  Errors: DOPT_E_ARG (NULL output),
 * DOPT_E_STATE in a build without the checks (the product library),
 * DOPT_E_CUDA. */
#define DOPT_CHECK_INDEX 1u /* an element or vector index outside the buffers */
#define DOPT_CHECK_ALIGN 2u /* a vector not on an 8-element boundary */
int dopt_device_checks(int reset, uint32_t *flags, int64_t *first_bad);

/* Count of staged CTAs (DOPT_STEP_STAGE) on the current device whose bulk
 * copies did not complete within their time limit, so that they skipped
 * their tile; with reset != 0 the count is then cleared.  0 unless a bulk
 * copy failed to complete.  Library infrastructure: the pages have no
 * counterpart.  Synchronous.  Errors: DOPT_E_ARG (NULL count), DOPT_E_CUDA. */
int dopt_stage_timeouts(int reset, uint32_t *count);

/* Test build only (DOPT_DEVICE_CHECKS, libdopt_checked.so): every staged CTA
 * launched after this call on the current device expects `extra_bytes`
 * more from its bulk copies than they deliver, so its 2 s wait runs out
 * and it takes the failure path described at DOPT_STEP_STAGE (counted by
 * dopt_stage_timeouts, its tile left untouched, a second bounded wait,
 * about 4 s in all) without any fault; 0 restores normal staging.
 * 0 <= extra_bytes <= 65536.  Library infrastructure for testing the
 * bounded wait: the pages have no counterpart.  Synchronous.  Errors:
 * DOPT_E_STATE in the product build (which has no such hook), DOPT_E_ARG,
 * DOPT_E_CUDA. */
int dopt_stage_wait_test(uint32_t extra_bytes);

/*
 * The HBM bandwidth of a mix of streams, for measurement: one launch over
 * n_vectors 16-byte vectors, one per thread, that reads vector i of each of
 * the `reads` read buffers and writes the XOR of them with a seed made of i
 * to vector i of each of the `writes` write buffers, with the streaming
 * 128-bit loads and stores of the step kernels.  Timing it (the caller's
 * CUDA events) gives the ceiling of a read/write mix (the step at D reads
 * D + 6 and writes D + 6 16-byte vectors per 8 elements: equal read and
 * write streams), against which the step kernels are measured.  Buffers:
 * device, 16-byte aligned, n_vectors * 16 bytes each, owned by the caller;
 * with no write stream, a thread whose XOR equals one fixed 128-bit pattern
 * stores it into read buffer 0 (this keeps the loads from being optimised
 * away).  0 <= reads, writes <= 16, not both 0.  Library
 * infrastructure for measurement: the pages have no counterpart.
 * Asynchronous on `stream`.  Errors: DOPT_E_ARG, DOPT_E_ALIGN, DOPT_E_CUDA.
 */
int dopt_stream_probe(int32_t reads, int32_t writes, const void *const *read_buffers,
                      void *const *write_buffers, int64_t n_vectors, cudaStream_t stream);

/* Text of the last error raised on the calling thread ("" if none).
 * Library infrastructure: the pages have no counterpart. */
const char *dopt_last_error(void);

/* Library version string.  Library infrastructure: the pages have no
 * counterpart. */
const char *dopt_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DOPT_H */

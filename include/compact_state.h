/*
 * compact_state.h -- C ABI of the fused multi-tensor AdamW step for GB300.
 *
 * One call, adamw_step(), runs one AdamW optimizer step over a whole list of
 * parameter tensors in a single persistent kernel launch. Moment state is kept
 * as fp32, compact bf16, or block-wise 8-bit codes (signed linear, linear with
 * an unsigned second moment, or a dynamic-exponent codebook).
 *
 * What the step computes is the AdamW update of "Fused Optimizers and State
 * Precision" (xuujii.github.io ai-infra-kb M041), section 02, for every element
 * of every tensor that has a gradient, with t the tensor's own step count:
 *
 *     t = t + 1
 *     m = beta1*m + (1-beta1)*g
 *     v = beta2*v + (1-beta2)*g*g
 *     theta = theta*(1-lr*wd) - lr * (m/(1-beta1^t)) / (sqrt(v/(1-beta2^t)) + eps)
 *
 * with g = stored_grad * inv_scale (the grad-scaler unscale of the Apex
 * FusedAdam capturable path, Apex fused-optimizers guide section 4.3). The bias
 * corrections are per-tensor scalars; m_hat and v_hat are never stored
 * (section 04). The theta update uses the freshly updated moments before they
 * are re-encoded (section 05: decode -> update -> re-encode).
 *
 * Contract (sections 02, 03, 06 of the same page):
 *   - every parameter group has its own lr, betas, eps and weight decay;
 *   - a tensor without a gradient this step (grad=None) is not touched at all:
 *     no decay, no moment update, no step advance; a zero gradient IS a full
 *     update;
 *   - when *found_inf != 0 the whole step is a no-op: params, moments, scales
 *     and step counts are left bit-identical.
 *
 * Conventions for every function:
 *   - Return value 0 (CS_OK) on success, a negative CS_ERR_* code otherwise;
 *     adamw_strerror() names it. No function aborts or throws across the ABI.
 *   - "device" pointers are CUDA global-memory addresses on the device that was
 *     current when the plan was created; "host" pointers are ordinary memory.
 *   - The caller owns every buffer it passes (params, grads, moments, scales,
 *     step counters, inv_scale, found_inf); they must outlive the plan. The
 *     plan owns only its own device tables, freed by adamw_plan_destroy().
 *   - Only adamw_plan_create / adamw_plan_destroy allocate or free device
 *     memory. adamw_step() allocates nothing, never synchronises the host and
 *     is asynchronous on the given stream.
 *   - A plan must not be stepped concurrently on two streams.
 */
#ifndef COMPACT_STATE_H
#define COMPACT_STATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;              /* cudaStream_t is `struct CUstream_st *` */

/* ---- status codes ------------------------------------------------------ */
#define CS_OK                    0
#define CS_ERR_INVALID_ARGUMENT (-1)  /* null/negative/out-of-range argument   */
#define CS_ERR_UNSUPPORTED      (-2)  /* unknown dtype or state kind          */
#define CS_ERR_MISALIGNED       (-3)  /* pointer not aligned to its element   */
#define CS_ERR_LIMIT            (-4)  /* too many tensors / groups / elements */
#define CS_ERR_CUDA             (-5)  /* a CUDA runtime call failed           */
#define CS_ERR_OUT_OF_MEMORY    (-6)  /* host or device allocation failed     */
#define CS_ERR_HYPERPARAM       (-7)  /* beta outside [0,1), non-finite lr... */
#define CS_ERR_WRONG_DEVICE     (-8)  /* current device is not the plan's     */

/* ---- element types ----------------------------------------------------- */
#define CS_DTYPE_F32   0         /* params / grads                          */
#define CS_DTYPE_BF16  1
#define CS_DTYPE_F16   2

#define CS_STATE_F32   0         /* two fp32 moments per element            */
#define CS_STATE_BF16  1         /* two bf16 moments per element (RNE)      */
#define CS_STATE_INT8  2         /* two int8 codes per element + two fp32
                                    scales per 256-element block            */
/* 8-bit variants ("Fused Optimizers and State Precision", section 05: real
 * 8-bit optimizers may use other codebooks than the uniform teaching codec).
 * Same layout as CS_STATE_INT8: one byte per element per moment, one fp32
 * scale per 256-element block per moment.                                   */
#define CS_STATE_INT8_UV 3       /* m as CS_STATE_INT8; v unsigned: codes
                                    0..255, scale = max|v| / 255            */
#define CS_STATE_DYN8  4         /* dynamic-exponent codebook (dynamic tree
                                    quantization): m signed map (sign bit,
                                    base-10 exponent as leading zeros,
                                    indicator bit, linear fraction), v the
                                    unsigned map; scale = block max|x|; the
                                    code is the nearest table value        */

/* adamw_tensor_t.flags */
#define CS_TENSOR_STATE_F32  1   /* in an 8-bit plan, keep fp32 moments for
                                    this tensor (m, v: numel fp32 values, no
                                    scales): the selective high precision
                                    section 05 cites for small tensors      */

#define CS_INT8_BLOCK        256     /* elements per int8 scale block       */
#define CS_MAX_GROUPS        64      /* parameter groups per step           */
#define CS_MAX_TENSORS       245760  /* tensors per plan                    */

/* ---- one parameter group's hyper-parameters (host memory, per step) ---- */
typedef struct adamw_group_t {
    float lr;            /* learning rate, finite                            */
    float beta1;         /* in [0, 1)                                        */
    float beta2;         /* in [0, 1)                                        */
    float eps;           /* finite, > 0, added outside the square root      */
    float weight_decay;  /* decoupled decay: theta *= 1 - lr*weight_decay    */
} adamw_group_t;

/* ---- one parameter tensor (host memory, read by adamw_plan_create) ----- */
typedef struct adamw_tensor_t {
    void       *param;   /* device, numel elements of param_dtype, in place  */
    const void *grad;    /* device, numel elements of param_dtype (stored,
                            i.e. still multiplied by the loss scale)         */
    void       *m;       /* device, first moment: numel fp32 / bf16 values,
                            or numel 8-bit codes for the 8-bit kinds
                            (CS_STATE_INT8 / _INT8_UV / _DYN8), or numel fp32
                            values for a CS_TENSOR_STATE_F32 tensor          */
    void       *v;       /* device, second moment, same layout as m          */
    float      *m_scale; /* device, 8-bit kinds only: ceil(numel/256) fp32
                            scales of m, one per 256-element block of the
                            tensor's flat order (else ignored, may be NULL)  */
    float      *v_scale; /* device, 8-bit kinds only: scales of v            */
    int64_t     numel;   /* elements, >= 0 (0: no buffer is touched, but the
                            step count still advances when it has a grad)    */
    int32_t     param_dtype;  /* CS_DTYPE_*; grad has the same dtype         */
    int32_t     group;        /* index into the per-step group table         */
    float      *master;  /* device, optional fp32 master weights (numel
                            values) of a CS_DTYPE_BF16 / CS_DTYPE_F16 param,
                            or NULL. With a master the step reads the master,
                            not param; it stores the new value to the master
                            and its round-to-nearest-even to param, in the
                            same pass (the Apex fused-optimizers guide,
                            FusedAdam master_weights, sections 4.2 and 4.3).
                            The caller initialises it, usually to param's
                            exact fp32 value. A master on an fp32 param is
                            CS_ERR_INVALID_ARGUMENT.                       */
    int32_t     flags;   /* CS_TENSOR_* bits (0: none). CS_TENSOR_STATE_F32
                            outside an 8-bit plan is CS_ERR_INVALID_ARGUMENT */
} adamw_tensor_t;

/* Moments start at zero: the caller zero-fills m and v (and, for int8, the
 * codes and the scales) before the first step. Pointers need only be aligned
 * to their element size; when every buffer of a tensor is also aligned to
 * four elements the kernel uses vector loads for it.                        */

typedef struct adamw_plan adamw_plan_t;

typedef struct adamw_plan_info_t {
    int64_t n_units;        /* work units in the device queue               */
    int64_t total_numel;    /* sum of numel over the plan's tensors          */
    int64_t device_bytes;   /* device memory owned by the plan               */
    int32_t n_tensors;
    int32_t state_kind;
    int32_t unit_elems;     /* elements per work unit                        */
    int32_t grid_blocks;    /* CTAs of the persistent launch                 */
    int32_t block_threads;  /* threads per CTA                               */
    int32_t device;         /* CUDA device ordinal of the plan               */
} adamw_plan_info_t;

/*
 * adamw_plan_create -- validate a tensor list and upload its descriptor and
 * work-unit tables to the current device, once per parameter set.
 *   tensors     host array [n_tensors], read only during the call.
 *   n_tensors   1 .. CS_MAX_TENSORS.
 *   state_kind  CS_STATE_*; one kind for all tensors of the plan.
 *   unit_elems  elements per work unit; 0 picks the default (49152). Must be
 *               a positive multiple of 256 otherwise.
 *   out_plan    host out-parameter; set to NULL on failure.
 * Allocates device memory (descriptors 64 B/tensor, units 16 B/unit,
 * a 4 B/tensor commit counter, two scheduler words, an error word and 16 KB
 * of partial sums for adamw_grad_prologue).
 * Synchronous.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_UNSUPPORTED, CS_ERR_MISALIGNED,
 * CS_ERR_LIMIT, CS_ERR_OUT_OF_MEMORY, CS_ERR_CUDA.
 */
int adamw_plan_create(const adamw_tensor_t *tensors, int32_t n_tensors,
                      int32_t state_kind, int32_t unit_elems,
                      adamw_plan_t **out_plan);

/*
 * adamw_step -- one fused AdamW step over every tensor of the plan, enqueued
 * on `stream` as one kernel launch.
 *   groups        host array [n_groups] (copied into the launch; may be freed
 *                 on return). Every tensor's group must be < n_groups.
 *   n_groups      1 .. CS_MAX_GROUPS.
 *   grad_present  host bitmask [ceil(n_tensors/32)] (copied into the launch):
 *                 bit (i % 32) of word (i / 32) set means tensor i has a
 *                 gradient this step. NULL means every tensor has one.
 *   step          device int32 [n_tensors]: per-tensor step counts. The kernel
 *                 uses t = step[i] + 1 and stores t back only for tensors it
 *                 updated, and only when the step is not skipped.
 *   inv_scale     device fp32 scalar multiplied into every gradient; NULL = 1.
 *   found_inf     device fp32 scalar; nonzero (or NaN) skips the whole step.
 *                 NULL = 0.
 *   stream        CUDA stream (NULL = legacy default stream).
 * Allocates nothing, does not synchronise, can be captured in a CUDA graph
 * (the group table and bitmask are captured by value). The kernel is launched
 * with programmatic dependent launch: it may start on SMs that the previous
 * kernel on the stream has left (when that kernel allows it, as this step and
 * adamw_grad_prologue do), but it touches no buffer until the work before it
 * on the stream has completed and its writes are visible.
 * Errors (nothing is enqueued): CS_ERR_INVALID_ARGUMENT, CS_ERR_HYPERPARAM,
 * CS_ERR_LIMIT, CS_ERR_WRONG_DEVICE; CS_ERR_CUDA if the launch fails.
 */
int adamw_step(adamw_plan_t *plan, const adamw_group_t *groups, int32_t n_groups,
               const uint32_t *grad_present, int32_t *step,
               const float *inv_scale, const float *found_inf,
               struct CUstream_st *stream);

/*
 * adamw_grad_prologue -- the gradient checks that precede the update, in one
 * pass over every present gradient of the plan, on the device: unscale,
 * non-finite check, global L2 norm and clip factor ("Fused Optimizers and
 * State Precision", section 06: unscale, check for non-finite values and clip
 * before updating; the Apex FusedAdam capturable path, section 4.3, and
 * FusedLAMB's global gradient norm, section 5.3).
 *   grad_present   as for adamw_step (host bitmask, NULL = all present).
 *   inv_scale      device fp32 scalar multiplied into every gradient; NULL = 1.
 *   max_norm       clip threshold; <= 0 disables clipping; must be finite.
 *   found_inf_out  device fp32: 1 if any g*inv_scale (fp32) of a present
 *                  tensor is NaN or infinite, else 0.
 *   grad_norm_out  device fp32 (NULL allowed): sqrt(sum (g*inv_scale)^2) over
 *                  present tensors; NaN when found_inf_out is 1.
 *   scale_out      device fp32: inv_scale * min(1, max_norm/(norm + 1e-6)),
 *                  or inv_scale when not clipping or when found_inf_out is 1.
 * Passing found_inf_out and scale_out to adamw_step as its found_inf and
 * inv_scale runs unscale, check, clip and update in that order with no host
 * sync. Squares are summed in fp32 with compensation per thread and in fp64
 * across blocks, in a fixed order (the result does not depend on timing).
 * Asynchronous on `stream`, allocates nothing. Must not overlap another
 * prologue of the same plan.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_HYPERPARAM (non-finite max_norm),
 * CS_ERR_WRONG_DEVICE, CS_ERR_CUDA.
 */
int adamw_grad_prologue(adamw_plan_t *plan, const uint32_t *grad_present,
                        const float *inv_scale, float max_norm, float *found_inf_out,
                        float *grad_norm_out, float *scale_out, struct CUstream_st *stream);

/*
 * adamw_plan_set_grads -- replace the gradient pointers of every tensor (for
 * frameworks that reallocate gradients between steps).
 *   grads   host array [n_tensors] of device pointers (NULL allowed only for
 *           tensors with numel 0); alignment rules as at creation.
 *   stream  the stream later steps use; the table update is ordered on it.
 * Copies through a plan-owned pinned staging buffer; it waits on the host only
 * if the previous call's copy has not yet left that buffer.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_MISALIGNED, CS_ERR_CUDA.
 */
int adamw_plan_set_grads(adamw_plan_t *plan, const void *const *grads,
                         struct CUstream_st *stream);

/*
 * adamw_plan_error -- read and clear the plan's device error word (host out).
 * Every wait inside the step kernel is bounded (2 s by default). A wait that
 * runs out sets a bit here and that CTA winds down without touching its
 * remaining tiles; nothing traps and the CUDA context stays usable. Bits:
 * 1 a compute warp gave up waiting for a tile, 2 the producer gave up waiting
 * for a tile's compute, 4 the producer gave up waiting for its own loads,
 * 8 the unit fetcher gave up waiting for the producer.
 * 0 means every step since the last call ran to completion. A nonzero read
 * also clears the plan's work queue and commit counters, which a step that
 * gave up leaves behind, so the next step starts clean (the steps that gave up
 * are not redone). Synchronises the device.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_WRONG_DEVICE, CS_ERR_CUDA.
 */
int adamw_plan_error(adamw_plan_t *plan, uint32_t *out_flags);

/*
 * adamw_plan_set_debug -- test hook for later steps of this plan: the bound
 * on every wait in nanoseconds (0 restores the 2 s default; at most 60 s) and
 * debug flags. Flag 1 leaves the first tile of the queue's first unit
 * unsignalled, so that the bounded waits of the CTA holding it run out and
 * report through adamw_plan_error. Normal use never calls it.
 * Errors: CS_ERR_INVALID_ARGUMENT (unknown flag or bound above 60 s).
 */
int adamw_plan_set_debug(adamw_plan_t *plan, uint64_t wait_ns, uint32_t flags);

/* adamw_plan_info -- fill *out (host) with the plan's sizes and launch shape. */
int adamw_plan_info(const adamw_plan_t *plan, adamw_plan_info_t *out);

/* adamw_plan_destroy -- synchronise the device and free the plan's tables.
 * NULL is accepted. The caller's buffers are untouched.                      */
int adamw_plan_destroy(adamw_plan_t *plan);

/*
 * adamw_state_bytes -- bytes of optimizer state for a tensor list, host only:
 * moments (8 / 4 / 2 bytes per element for fp32 / bf16 / the 8-bit kinds),
 * plus for the 8-bit kinds two fp32 scales per 256-element block of each
 * tensor, plus a 4-byte step counter per tensor. A tensor whose flags hold
 * CS_TENSOR_STATE_F32 (8-bit kinds only, as in adamw_plan_create) counts 8
 * bytes per element and no scales. Section 05's payload ledger; the ApexW
 * Unsloth benchmark page's 185.501 / 92.751 / 47.101 MB for its LoRA set
 * follow from it.
 *   numels  host array [n_tensors]; flags host array [n_tensors] of
 *           adamw_tensor_t.flags values, or NULL (all 0); out: host int64.
 * Errors: CS_ERR_INVALID_ARGUMENT (negative size, unknown flag, fp32 flag
 * outside an 8-bit kind), CS_ERR_UNSUPPORTED.
 */
int adamw_state_bytes(const int64_t *numels, const int32_t *flags, int32_t n_tensors,
                      int32_t state_kind, int64_t *out_bytes);

/*
 * adamw_build_units -- the work-unit cut before the queue's tail is re-cut
 * (see adamw_build_queue), computed on the host only (no CUDA call), for
 * inspection and tests. Units are (tensor, start, len) with start a multiple
 * of unit_elems, len <= unit_elems, covering each tensor exactly once,
 * ordered longest first; a tensor with numel 0 has one unit of len 0.
 *   numels      host [n_tensors];  unit_elems as for adamw_plan_create.
 *   tensor_out, start_out, len_out  host arrays of capacity `cap` (may be NULL
 *               when cap is 0, to query the count).
 *   n_units_out host int64: the number of units (always written).
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_LIMIT (cap too small: nothing but
 * *n_units_out written).
 */
int adamw_build_units(const int64_t *numels, int32_t n_tensors, int32_t unit_elems,
                      int32_t *tensor_out, int64_t *start_out, int32_t *len_out,
                      int64_t cap, int64_t *n_units_out);

/*
 * adamw_build_queue -- the exact work queue adamw_plan_create builds for a
 * state kind on a GPU with `ctas` persistent CTAs (its SM count), on the host
 * only. It is adamw_build_units' cut, after which the units holding the last
 * two waves' worth of elements (2 * ctas * unit_elems) are re-cut into
 * pieces of four tiles (12288 elements for fp32/bf16 moments, 16384 for the
 * 8-bit kinds, never more than unit_elems); for the 8-bit kinds the units
 * holding the last ctas such pieces' worth are cut again into two-tile
 * pieces (8192). All are kept longest first, so CTAs that take units
 * dynamically finish close together. Starts stay multiples of 256.
 * Arguments and outputs as adamw_build_units, plus state_kind (CS_STATE_*)
 * and ctas (>= 1).
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_UNSUPPORTED (state kind),
 * CS_ERR_LIMIT (cap too small: nothing but *n_units_out written).
 */
int adamw_build_queue(const int64_t *numels, int32_t n_tensors, int32_t state_kind,
                      int32_t unit_elems, int32_t ctas, int32_t *tensor_out,
                      int64_t *start_out, int32_t *len_out, int64_t cap,
                      int64_t *n_units_out);

/*
 * adamw_shard_ranges -- the part of every tensor that rank `rank` of `world`
 * updates in a ZeRO-style sharded step, computed on the host only (no CUDA
 * call). "Fused Optimizers and State Precision", section 06: sharding
 * (ZeRO / FSDP) decides which rank owns which state, the fused optimizer how
 * the local state is updated, and the two compose. Because the update is
 * elementwise (and blockwise for the 8-bit kinds), a step over every rank's
 * part equals the step over the whole list.
 * Layout: the tensors end to end in one flat buffer, each padded to a whole
 * number of 256-element blocks (CS_INT8_BLOCK); the flat buffer is cut into
 * `world` equal shards of shard_elems = ceil(blocks / world) * 256 elements
 * (the last shards may hold padding only); rank r owns the flat elements
 * [r * shard_elems, (r + 1) * shard_elems). Tensor i's part is its elements
 * [lo[i], hi[i]): lo is a multiple of 256 and hi a multiple of 256 or numel,
 * so no 8-bit scale block is split between ranks; lo == hi == 0 when the rank
 * owns none of it.
 *   numels           host [n_tensors], each >= 0.
 *   world, rank      1 <= world, 0 <= rank < world.
 *   lo_out, hi_out   host int64 [n_tensors].
 *   offset_out       host int64 [n_tensors] or NULL: each tensor's first
 *                    element in the flat buffer (a multiple of 256).
 *   shard_elems_out  host int64 or NULL: elements per shard; the padded flat
 *                    buffer holds world * shard_elems.
 * A rank steps a plan whose tensor i is the slice [lo[i], hi[i]) of every
 * buffer (param, reduced grad, m, v; scales from block lo[i] / 256), empty
 * slices included: every rank then keeps the step counts of every tensor
 * and advances them identically, given the same grad_present mask and the
 * same (all-reduced) found_inf.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_LIMIT (a tensor above 2^40).
 */
int adamw_shard_ranges(const int64_t *numels, int32_t n_tensors, int32_t world, int32_t rank,
                       int64_t *lo_out, int64_t *hi_out, int64_t *offset_out,
                       int64_t *shard_elems_out);

/*
 * adamw_step_noalloc -- one fused AdamW step that allocates nothing. The pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * call cudaMalloc: an allocator or memory pool that runs the step from its own
 * callbacks and must not re-enter the device allocator, or a runtime that
 * hands all device memory to its own pool at start-up.
 *   Arguments as adamw_plan_create's tensors/state_kind plus adamw_step's
 *   groups/grad_present/step/inv_scale/found_inf/stream; every buffer is the
 *   caller's. Work units are CS_NOALLOC_UNIT elements, cut and ordered like a
 *   default plan's units but without a plan's re-cut of the queue's tail
 *   (adamw_build_units gives the cut), so results equal adamw_step's on the
 *   same inputs; only the balance of the last units across CTAs differs.
 * Scratch: one file-scope device array of fixed size (descriptors, units,
 * tickets, scheduler and error words; about 1.3 MB), held by every GPU that
 * loads the library until the process exits. Limits: at most
 * CS_NOALLOC_MAX_TENSORS tensors, CS_NOALLOC_MAX_UNITS work units (3.2e9
 * elements at full units) and CS_MAX_GROUPS groups; beyond them it returns
 * CS_ERR_LIMIT without touching the device.
 * The first call on a device resolves the array's device address there (with
 * that device current); make that first call before any stream capture. A
 * call on a stream that is being captured returns CS_ERR_INVALID_ARGUMENT:
 * each call uploads its tables from host staging that the next call rewrites.
 * Every call shares the array and rewrites it: calls that overlap on the GPU
 * race, so order them (one stream, or events). Calls are serialised on the
 * host. No cudaMalloc, cudaFree or other allocating routine is called.
 * A bounded wait that runs out inside the kernel (see adamw_plan_error) sets a
 * bit in the array's error word, which later calls do not clear: read it with
 * adamw_noalloc_error.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_UNSUPPORTED, CS_ERR_MISALIGNED,
 * CS_ERR_HYPERPARAM, CS_ERR_LIMIT, CS_ERR_CUDA.
 */
#define CS_NOALLOC_MAX_TENSORS 4096
#define CS_NOALLOC_MAX_UNITS   65536
#define CS_NOALLOC_UNIT        49152
int adamw_step_noalloc(const adamw_tensor_t *tensors, int32_t n_tensors, int32_t state_kind,
                       const adamw_group_t *groups, int32_t n_groups,
                       const uint32_t *grad_present, int32_t *step,
                       const float *inv_scale, const float *found_inf,
                       struct CUstream_st *stream);

/*
 * adamw_noalloc_error -- read and clear the error word of adamw_step_noalloc
 * on the current device (host out): the bits of adamw_plan_error, collected
 * over every no-allocation step since the last read. 0 means they all ran to
 * completion. A nonzero value means some step gave up part of its work (its
 * step counts may have advanced for tensors it did not finish); the next call
 * starts with a clean queue either way. Synchronises the device; allocates
 * nothing.
 * Errors: CS_ERR_INVALID_ARGUMENT, CS_ERR_LIMIT (device ordinal >= 64),
 * CS_ERR_CUDA.
 */
int adamw_noalloc_error(uint32_t *out_flags);

/*
 * adamw_noalloc_set_debug -- test hook for later adamw_step_noalloc calls in
 * this process: the bound on every wait and the debug flags, with the meaning
 * of adamw_plan_set_debug. Normal use never calls it.
 * Errors: CS_ERR_INVALID_ARGUMENT (unknown flag or bound above 60 s).
 */
int adamw_noalloc_set_debug(uint64_t wait_ns, uint32_t flags);

/* adamw_strerror -- static string naming a status code (never NULL). */
const char *adamw_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* COMPACT_STATE_H */

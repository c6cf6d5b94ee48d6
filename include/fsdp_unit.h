/*
 * fsdp_unit.h -- C ABI of the GB300 per-unit FSDP cycle.
 *
 * One FSDP unit (a group of parameters gathered and freed together) is sharded
 * over N data-parallel ranks.  The ranks are virtual: their shard buffers all
 * live in the memory of the one GPU that was current when the unit was
 * created, and every "collective" is a memory-bound kernel on that GPU.
 *
 * Sources (page title, then section):
 *  [FSDP]   "PyTorch FSDP: Experiences on Scaling Fully Sharded Data Parallel"
 *  [HOOD]   "FSDP Under The Hood: ZeRO-3 The PyTorch Way"
 *  [ARCH]   "FSDP Architecture"
 *  [NOTE]   "FSDP (Fully Sharded Data Parallel)" concept note
 *
 * Conventions shared by every call
 *  - Return value: FSDP_OK (0) or a negative FSDP_E_* code.  Arguments are
 *    checked on the host before anything is enqueued; a call that fails its
 *    checks changes nothing.  fsdp_last_error() gives a one-line reason for
 *    the calling thread's most recent failure.  No call aborts or traps.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Calls that enqueue GPU work return without waiting.
 *  - Device: a unit belongs to the device that was current at creation; every
 *    call makes that device current for its duration and restores the
 *    caller's device afterwards.
 *  - Pointers named *_dev are device pointers (or managed memory) that the
 *    caller owns and keeps alive until the enqueued work has finished.  The
 *    library never keeps a caller pointer after a call returns.
 *  - Hot-path buffers (gradients, the gathered output) must be 16-byte
 *    aligned (FSDP_E_ALIGN otherwise).  Gradients that are all 32-byte aligned
 *    (as allocations from cudaMalloc or torch are) are read with 32-byte
 *    vector loads; if any is only 16-byte aligned, that call's reduction
 *    reads every gradient with 16-byte loads (same results).
 *  - Element types: fp32 is IEEE binary32; bf16 is stored as uint16_t bit
 *    patterns (the upper half of the binary32 pattern).
 *  - A unit is not thread-safe; distinct units are independent.
 */
#ifndef FSDP_UNIT_H
#define FSDP_UNIT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FSDP_API __attribute__((visibility("default")))
#else
#define FSDP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define FSDP_OK             0
#define FSDP_E_INVALID_ARG (-1)  /* bad shape, count, enum, null pointer   */
#define FSDP_E_OOM         (-2)  /* device or host allocation failed        */
#define FSDP_E_CUDA        (-3)  /* a CUDA runtime call or launch failed    */
#define FSDP_E_STATE       (-4)  /* call not valid in the unit's state      */
#define FSDP_E_ALIGN       (-5)  /* a buffer is not aligned as required     */
#define FSDP_E_CAPACITY    (-6)  /* caller's output array is too small      */

/* ---- enums ------------------------------------------------------------ */
/* FLAT: the FSDP1 FlatParameter.  All parameters are flattened (row-major)
 *   and concatenated in the order given; rank k owns the contiguous elements
 *   floor(kP/N) .. floor((k+1)P/N)-1, no padding ([ARCH], the GPU-k boundary
 *   formula; [FSDP] section 3.2.1 and Figure 3 for flatten + concatenate).
 * DIM0: FSDP2 per-parameter Shard(0).  Each parameter is chunked along dim 0
 *   with torch.chunk semantics: ceil(m/N) rows per chunk, the last chunk
 *   short, trailing ranks empty when there are fewer chunks than ranks
 *   ([NOTE] "FSDP1 vs FSDP2"; [HOOD] section 2).  A rank's shard is its chunks
 *   of every parameter, concatenated in parameter order. */
#define FSDP_LAYOUT_FLAT 0
#define FSDP_LAYOUT_DIM0 1
/* FLAT_PADDED: the FlatParameter as [FSDP] section 3.2.1 / Figure 3 builds it:
 *   right-padded to a multiple of N and cut into N equal chunks of ceil(P/N)
 *   elements; rank k owns [min(k*c, P), min((k+1)*c, P)) followed by zero
 *   padding up to c elements (at most N-1 padding elements in all). */
#define FSDP_LAYOUT_FLAT_PADDED 2

#define FSDP_DTYPE_F32  0
#define FSDP_DTYPE_BF16 1

/* where the all-gather reads from */
#define FSDP_GATHER_FROM_MASTER 0  /* fp32 master shard, cast to bf16 while gathering */
#define FSDP_GATHER_FROM_SHADOW 1  /* bf16 shadow shard (RNE(master) when read), copied */

/* per-rank state a unit owns */
#define FSDP_STATE_PARAM      0  /* fp32 sharded master parameters           */
#define FSDP_STATE_GRAD       1  /* fp32 gradient shard (reduce-scatter out) */
#define FSDP_STATE_EXP_AVG    2  /* fp32 AdamW first moment m                */
#define FSDP_STATE_EXP_AVG_SQ 3  /* fp32 AdamW second moment v               */
#define FSDP_STATE_SHADOW     4  /* bf16 copy of the master shard            */

/* kernels the profiler times */
#define FSDP_KERNEL_SHARD_IN       0
#define FSDP_KERNEL_GATHER         1
#define FSDP_KERNEL_REDUCE_SCATTER 2
#define FSDP_KERNEL_ADAMW          3
#define FSDP_KERNEL_REDUCE_ADAMW   4   /* fused reduce-scatter + AdamW (fsdp_step) */
#define FSDP_KERNEL_COUNT          5

/* bits of a unit's kernel status word (fsdp_kernel_status) */
#define FSDP_KSTATUS_WAIT_TIMEOUT  1   /* a kernel gave up waiting for its own copies into
                                          shared memory; its outputs are incomplete      */
#define FSDP_KSTATUS_DRAIN_TIMEOUT 2   /* after that, a wait for its remaining copies ran out
                                          too: copies may have landed in shared memory after
                                          the kernel ended, so nothing computed around that
                                          launch can be trusted                             */

/* ---- plain structs ------------------------------------------------------ */
typedef struct fsdp_unit fsdp_unit;   /* opaque; one FlatParamHandle ([FSDP] section 4.2) */

/* torch.optim.AdamW's hyper-parameters, as doubles (the update itself runs
 * in fp32; see fsdp_adamw_step). */
typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
} fsdp_adamw_hp;

typedef struct {
    int layout;                /* FSDP_LAYOUT_FLAT, _DIM0 or _FLAT_PADDED                  */
    int num_ranks;             /* N: ranks a parameter is sharded over (the sharding
                                  factor F of [FSDP] 3.2.2), 1 .. 1024                     */
    int grad_dtype;            /* dtype of the full gradient buffers: F32 or BF16         */
    int reshard_after_forward; /* nonzero: fsdp_step gathers twice ([FSDP] 5.4)           */
    int replicas;              /* hybrid sharding ([FSDP] 3.2.2): R >= 1 replication
                                  groups; the data-parallel world is W = N*R ranks and a
                                  reduce-scatter takes W gradients.  0 is read as 1.
                                  N*R <= 1024.                                             */
    int reduce_dtype;          /* F32 (default) or BF16 ([FSDP] 4.4: reductions in the
                                  low precision); BF16 requires replicas == 1              */
    int gather_source;         /* FSDP_GATHER_FROM_MASTER (default) or _FROM_SHADOW        */
    int fuse_reduce_adamw;     /* nonzero: fsdp_step runs its reduce-scatter and AdamW as
                                  one pass per element (the gradient shard is written and
                                  used without being read back); results are identical   */
} fsdp_unit_config;

/* Options of fsdp_reduce_scatter_ex; all-zero means a plain reduce-scatter. */
typedef struct {
    int accumulate;            /* nonzero: add the result to the existing gradient
                                  shard (gradient accumulation with communication,
                                  [FSDP] 3.3.4) instead of overwriting it               */
    double inv_scale;          /* 0 or 1: no unscale; otherwise the reduced gradient is
                                  multiplied by fp32(inv_scale) before accumulation
                                  (loss-scale removal, [FSDP] 4.4 sharded grad scaler)  */
    int32_t* found_nonfinite_dev; /* optional device int32: set to 1 if any written
                                  gradient value is inf or NaN, else 0 (the global
                                  overflow decision: an OR over every rank's shard)   */
} fsdp_rs_options;

/* One contiguous piece of a rank's shard. */
typedef struct {
    int32_t rank;        /* owning virtual rank                                        */
    int32_t param;       /* parameter index (DIM0); -1 for FLAT (may span parameters)  */
    int64_t global_off;  /* first element in the unsharded flat buffer                 */
    int64_t shard_off;   /* first element within the rank's packed shard (no padding)  */
    int64_t arena_off;   /* first element within the rank's device arena (with pads)   */
    int64_t len;         /* element count, >= 1                                        */
} fsdp_segment;

/* Parameter shapes are passed as `nparams`, `ndims[nparams]` (0..8; a 0-d
 * parameter is one element) and `dims`, all parameters' dims concatenated
 * (sum of ndims entries, each >= 0).  The unit's element count P must be >= 1. */

/* ---- layout (host only; no GPU needed) --------------------------------- */

/* The layout the unit would use: P (total elements), the number of segments,
 * and the segments themselves (rank-major, in each rank's storage order).
 * `segs` may be NULL to query the count only; otherwise `cap` bounds the
 * number written (FSDP_E_CAPACITY if too small, with *nsegs set).
 * Arena offsets place global index i and its arena slot at the same
 * remainder modulo 32 elements. */
FSDP_API int fsdp_plan_layout(int nparams, const int* ndims, const int64_t* dims,
                     int layout, int num_ranks,
                     int64_t* numel, int64_t* nsegs,
                     fsdp_segment* segs, int64_t cap);

/* ---- lifetime ----------------------------------------------------------- */

/* Create a unit on the current device.  Allocates and zero-fills the N ranks'
 * state (master, gradient shard, m, v: 4 bytes per owned element each; bf16
 * shadow: 2 bytes; plus up to 31 alignment pad elements per segment) and a
 * small device tile table.  Synchronous.  ([FSDP] section 3.2.1: the
 * FlatParameter owns the storage of its shards.) */
FSDP_API int fsdp_unit_create(int nparams, const int* ndims, const int64_t* dims,
                     const fsdp_unit_config* cfg, fsdp_unit** out);

/* Optional provider of the unit's device memory (library infrastructure; the
 * pages have no counterpart), for
 * fsdp_unit_create_with_allocator (so that, for instance, a framework's
 * caching allocator owns and accounts for the rank arenas).  alloc(bytes,
 * ctx) returns a block of device memory on the current device, aligned to at
 * least 256 bytes, or NULL; free(ptr, ctx) takes back a block alloc returned.
 * The library calls them on the calling thread from
 * fsdp_unit_create_with_allocator (every buffer the unit owns),
 * fsdp_adamw_device_steps (its step table and counters) and
 * fsdp_unit_destroy (all of them, after the device has synchronised), and on
 * a failure in those calls for the blocks it already obtained.  The struct is
 * copied; ctx must stay valid until the unit is destroyed. */
typedef struct {
    void* (*alloc)(size_t bytes, void* ctx);
    void (*free)(void* ptr, void* ctx);
    void* ctx;
} fsdp_allocator;

/* fsdp_unit_create with the unit's device memory taken from `alloc` (NULL:
 * cudaMalloc, as fsdp_unit_create).  Errors besides fsdp_unit_create's:
 * FSDP_E_INVALID_ARG if alloc or free is NULL; FSDP_E_OOM if alloc returns
 * NULL; FSDP_E_ALIGN if it returns a block not aligned to 256 bytes (the
 * block is freed at once).  Every block obtained is freed on failure. */
FSDP_API int fsdp_unit_create_with_allocator(int nparams, const int* ndims, const int64_t* dims,
                     const fsdp_unit_config* cfg, const fsdp_allocator* alloc,
                     fsdp_unit** out);

/* Free everything the unit owns.  Synchronises the unit's device first.
 * NULL is accepted. */
FSDP_API int fsdp_unit_destroy(fsdp_unit* unit);

/* ---- the per-unit cycle --------------------------------------------------- */

/* Shard-in (FlatParameter construction, [FSDP] section 3.2.1): copy the full
 * fp32 parameters into the N ranks' master shards per the layout, zero the
 * gradient shards and m, v, set the bf16 shadow to the rounded master, and
 * reset the step count to 0.  `params_dev[p]` is parameter p, contiguous
 * row-major fp32 (may be NULL for a parameter with zero elements). */
FSDP_API int fsdp_load_params(fsdp_unit* unit, const float* const* params_dev, void* stream);

/* All-gather with the param_dtype cast ([FSDP] section 3.2.1 "communication
 * layout": the gathered buffer is the shards concatenated in rank order, i.e.
 * the unsharded FlatParameter; [FSDP] section 4.4: one fp32 -> bf16 cast per
 * gather).  Writes out_bf16_dev[i] = RNE_bf16(master[i]) for all i in [0, P):
 * one buffer, since every virtual rank's result is the same.  Rounding is
 * IEEE round-to-nearest-even; NaN stays NaN.  With gather_source
 * FSDP_GATHER_FROM_SHADOW the same bytes are copied from the bf16 shadow
 * shards (which hold RNE(master) whenever they are read; see fsdp_adamw_step):
 * the gather then moves bf16, as when the collective runs in the low precision
 * ([FSDP] 4.4). */
FSDP_API int fsdp_allgather(fsdp_unit* unit, uint16_t* out_bf16_dev, void* stream);

/* Reduce-scatter ([ARCH] backward step 3: sum the ranks' gradients and give
 * rank k only the slice of its shard; [HOOD] section 3: fp32 reduction).
 * `grads_dev` is a HOST array of W = N*replicas device pointers; pointer r is
 * data-parallel rank r's full unsharded gradient, P elements of the unit's
 * grad_dtype.  With replicas R, rank r = i*N + k is rank k of sharding group i.
 * For every element, with g_r upcast exactly to fp32:
 *   fp32 reduce:  acc_i = g_{iN} + g_{iN+1} + ... + g_{iN+N-1}   (left fold)
 *                 tot   = acc_0 + acc_1 + ... + acc_{R-1}         (left fold)
 *                 grad_shard = tot / W                            (IEEE division)
 *     (R = 1 is the plain rank-order fold; the grouping is [FSDP] 3.2.2's
 *     decomposition: reduce-scatter inside each sharding group, then all-reduce
 *     across groups.)
 *   bf16 reduce:  every input rounded to bf16, every partial sum and the
 *     division by N rounded to bf16 (RNE), the result widened to fp32.
 * The gradient shards are overwritten. */
FSDP_API int fsdp_reduce_scatter(fsdp_unit* unit, const void* const* grads_dev, void* stream);

/* The same reduction followed, per element and in this order, by the
 * optional unscale (x * fp32(inv_scale)) and accumulation (shard + x), and the
 * optional found-non-finite flag over the values written.  `opt` may be NULL. */
FSDP_API int fsdp_reduce_scatter_ex(fsdp_unit* unit, const void* const* grads_dev,
                                    const fsdp_rs_options* opt, void* stream);

/* Zero every rank's gradient shard (before the first accumulated micro-batch). */
FSDP_API int fsdp_zero_grad(fsdp_unit* unit, void* stream);

/* Local AdamW on every rank's shard ([ARCH]: each GPU updates its own shard
 * from its own gradient and optimizer-state shards, no communication; [HOOD]
 * appendix: torch.optim.AdamW).  Increments the step count t, then for every
 * owned element, in fp32 with one rounding per operation:
 *     p = p * fp32(1 - lr*wd)
 *     m = fp32(beta1)*m + fp32(1-beta1)*g
 *     v = fp32(beta2)*v + fp32(1-beta2)*(g*g)
 *     p = p - fp32(lr/(1-beta1^t)) * (m / (sqrt(v / fp32(1-beta2^t)) + fp32(eps)))
 *     shadow = RNE_bf16(p)
 * The scalar constants are formed in double on the host and rounded once.
 * The bf16 shadow holds RNE_bf16(p) whenever it is read: the update stores it
 * when the unit gathers from the shadow (gather_source FSDP_GATHER_FROM_SHADOW);
 * otherwise the store is skipped (2 bytes per element less) and the next read
 * of the shadow (a gather from it, fsdp_get_state, fsdp_read_global or
 * fsdp_read_arena of FSDP_STATE_SHADOW) first recomputes it on that call's
 * stream.
 * The step count advances when the launch is enqueued; if a kernel of this
 * unit later reports a status bit (fsdp_kernel_status), the count no longer
 * matches the state and the unit must be reloaded. */
FSDP_API int fsdp_adamw_step(fsdp_unit* unit, const fsdp_adamw_hp* hp, void* stream);

/* One unit step ([ARCH] the per-unit cycle; [FSDP] section 5.4): gather into
 * out_bf16_dev (forward), gather again when reshard_after_forward is set
 * (backward), reduce-scatter `grads_dev`, AdamW.  Same arguments and rules as
 * the individual calls; all four are checked before any is enqueued.  With
 * fuse_reduce_adamw the last two run as one kernel with the same results;
 * when W x gradient bytes <= 100 (bf16 gradients with W <= 50, fp32 with
 * W <= 25) that kernel stages its inputs in shared memory with bounded waits
 * (see fsdp_kernel_status: a raised bit means this step's update was
 * incomplete while the step count advanced, and the unit must be reloaded). */
FSDP_API int fsdp_step(fsdp_unit* unit, const void* const* grads_dev, uint16_t* out_bf16_dev,
              const fsdp_adamw_hp* hp, void* stream);

/* Change how fsdp_step runs on an existing unit: gather_source
 * (FSDP_GATHER_FROM_MASTER or _FROM_SHADOW) and fuse_reduce_adamw, as in
 * fsdp_unit_config.  Results do not depend on either choice (the shadow holds
 * RNE(master) whenever it is read, and the fused kernel performs the same
 * operations), only the bytes moved do.  Takes effect for calls enqueued
 * afterwards. */
FSDP_API int fsdp_unit_set_step_options(fsdp_unit* unit, int gather_source, int fuse_reduce_adamw);

/* ---- reduce-scatter without device allocation ------------------------------ */
/* Library infrastructure: the pages have no counterpart.
 *
 * Some callers cannot allocate device memory: a custom operator or plug-in
 * inside a host framework that owns all of the GPU's memory through its own
 * pool and forbids side allocations, or a process that has given nearly all
 * of HBM to shards and optimizer state so that one more cudaMalloc would fail
 * (and a cudaFree would stall every stream of the device).  Creating a unit
 * allocates its arenas and work tables, so such a caller cannot use
 * fsdp_reduce_scatter.  This entry point performs the same reduce-scatter for
 * the FLAT layout with no unit and no allocation of any kind: the caller
 * passes the inputs and the output, and the one scratch buffer it needs (the
 * kernel's table of work tiles) is a fixed array in the library's device
 * image, FSDP_NOALLOC_MAX_TILES tiles of 24 bytes (768 KiB), which every GPU
 * that loads the library holds until the process exits.
 *
 * grads_dev: HOST array of num_ranks (1..1024) device pointers, each rank's
 *   full gradient of `numel` elements of `grad_dtype` (F32 or BF16), 32-byte
 *   aligned.
 * out_dev: `numel` fp32 elements, 32-byte aligned: rank k's gradient shard is
 *   written to out_dev[floor(k*numel/N) .. floor((k+1)*numel/N)), so the buffer
 *   holds every rank's shard back to back, in rank order.  Each element is the
 *   rank-order fp32 left fold divided by N, bit for bit what
 *   fsdp_reduce_scatter writes for a FLAT unit of the same numel and N.
 * Size limit: the work must fit the scratch, that is, the pieces of rank
 *   ranges cut at multiples of 8192 elements number at most
 *   FSDP_NOALLOC_MAX_TILES; numel <= 8192 * (32769 - num_ranks) always fits.
 *   Larger sizes return FSDP_E_INVALID_ARG with the needed and available tile
 *   counts in fsdp_last_error(), before anything is enqueued.
 * The first call on each device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *   first call before any stream capture begins.
 * Every call shares the one scratch table, and each call rewrites the part it
 *   uses (a stream-ordered copy on `stream`, then the kernel), so calls in one
 *   stream's order are safe; calls that may overlap on the GPU (other streams,
 *   other threads, no ordering between them) race on the table and must not
 *   be issued.  Errors: FSDP_E_INVALID_ARG, FSDP_E_ALIGN, FSDP_E_CUDA. */
#define FSDP_NOALLOC_MAX_TILES 32768
FSDP_API int fsdp_reduce_scatter_flat_noalloc(const void* const* grads_dev, int num_ranks, int grad_dtype,
                                              int64_t numel, float* out_dev, void* stream);

/* ---- state access (tests, checkpoint / resume) --------------------------- */
/* Library infrastructure: the pages describe the sharded state ([FSDP] 3.2.1,
 * the FlatParameter owns its shards) but no access calls; these expose it per
 * rank, in unsharded order, and with the pads, for checkpoints and checks. */

/* Copy rank `rank`'s packed shard of state `which` (pads excluded; fp32, or
 * bf16 for FSDP_STATE_SHADOW) to `dst`, or from `src` into the unit.  dst/src
 * may be device or host memory (cudaMemcpyAsync with cudaMemcpyDefault; use
 * pinned host memory for asynchrony).  Size = the rank's shard length.
 * Setting FSDP_STATE_PARAM also recomputes that rank's shadow as RNE(master).
 * Reading (or setting) FSDP_STATE_SHADOW first enqueues, on `stream`, the
 * recomputation of a shadow that AdamW left stale (see fsdp_adamw_step); so do
 * fsdp_read_global and fsdp_read_arena. */
FSDP_API int fsdp_get_state(const fsdp_unit* unit, int which, int rank, void* dst, void* stream);
FSDP_API int fsdp_set_state(fsdp_unit* unit, int which, int rank, const void* src, void* stream);

/* Copy elements [begin, begin+count) of state `which` in unsharded (global)
 * order to `dst` (device or host). */
FSDP_API int fsdp_read_global(const fsdp_unit* unit, int which, int64_t begin, int64_t count,
                     void* dst, void* stream);

/* Copy rank `rank`'s whole device arena of state `which`, alignment pads and
 * layout padding included (arena_len elements, see fsdp_memory_report /
 * fsdp_segment.arena_off), to `dst`; with dst NULL only *arena_len is set.
 * For integrity checks: every element
 * outside the rank's segments is zero from creation and must stay zero; a
 * non-zero pad means some kernel wrote outside its segment. */
FSDP_API int fsdp_read_arena(const fsdp_unit* unit, int which, int rank, void* dst, int64_t* arena_len,
                             void* stream);

/* Device-side AdamW step counter, for replaying a captured CUDA graph
 * (library infrastructure; the pages have no counterpart).
 * Normally the step count t lives on the host and each AdamW launch carries
 * its bias-correction constants, so a captured launch would replay the same
 * step forever.  This call forms, on the host and with the same formulas as
 * fsdp_adamw_step, the fp32 constants of the next `count` steps (t+1 ..
 * t+count, count <= 2^24) into a device table owned by the unit, and switches
 * the unit to device-step mode: every AdamW launch (fsdp_adamw_step, fsdp_step)
 * then takes the constants of the step its device counter names, and a one-
 * thread kernel queued after it advances the counter, so replays step
 * correctly and give the same results as normal calls.  `hp` is fixed for the
 * table (the `hp` given to later calls is checked but not used).  A step that
 * finds the table used up changes nothing and sets the status that
 * fsdp_adamw_device_status reports.  Allocates (on the first call or when
 * count grows) and synchronises `stream`: call it before capturing.  count 0
 * leaves the mode and makes the host step count equal the device's.
 * fsdp_load_params also leaves the mode. */
FSDP_API int fsdp_adamw_device_steps(fsdp_unit* unit, const fsdp_adamw_hp* hp, int64_t count, void* stream);

/* In device-step mode: the step count reached on the device and whether a
 * step found the table used up (synchronises `stream`).  Otherwise the host
 * step count and 0. */
FSDP_API int fsdp_adamw_device_status(fsdp_unit* unit, int64_t* step, int32_t* exhausted, void* stream);

/* AdamW step count t (0 after load).  In device-step mode this host copy
 * counts enqueued steps only; graph replays advance the device counter. */
FSDP_API int fsdp_get_step_count(const fsdp_unit* unit, int64_t* t);
FSDP_API int fsdp_set_step_count(fsdp_unit* unit, int64_t t);

/* ---- introspection --------------------------------------------------------- */

/* The unit's element count P and the configuration it was created with
 * (replicas normalised to >= 1). */
FSDP_API int fsdp_unit_info(const fsdp_unit* unit, int64_t* numel, fsdp_unit_config* cfg);

/* The unit's segments (same contract as fsdp_plan_layout). */
FSDP_API int fsdp_unit_segments(const fsdp_unit* unit, fsdp_segment* segs, int64_t cap, int64_t* nsegs);

/* Steady-state bytes held for rank `rank` ([ARCH] memory breakdown: 4 bytes
 * of parameters, 4 of gradient and 8 of Adam state per owned element), the
 * bf16 shadow (2 per owned element) and the pads of all five (the padded
 * layout's chunk padding plus alignment padding).  Under hybrid sharding this
 * is one replica's copy; each of the R replicas holds the same. */
FSDP_API int fsdp_memory_report(const fsdp_unit* unit, int rank, int64_t* param_bytes,
                       int64_t* grad_bytes, int64_t* adam_bytes, int64_t* shadow_bytes,
                       int64_t* pad_bytes);

/* ---- kernel status ---------------------------------------------------------- */

/* Library infrastructure (the pages have no counterpart).
 * Kernels that wait on their own asynchronous copies (the shared-memory
 * staged fused reduce-scatter + AdamW of fsdp_step, and the staged
 * reduce-scatter that serves hybrid sharding, accumulation, unscaling and the
 * non-finite flag when W x gradient bytes <= 100) bound every wait; a wait
 * that runs out raises a FSDP_KSTATUS_* bit in the unit's device status word,
 * and the kernel returns with its outputs incomplete instead of hanging.
 * fsdp_kernel_status synchronises `stream`, stores the word in *flags
 * (0: nothing raised) and clears it.  The word starts at 0 at creation.
 * Reading a raised bit also blocks the unit: after FSDP_KSTATUS_WAIT_TIMEOUT
 * the gradient shards, master, m and v may be partly updated and the step
 * count has advanced past an incomplete update, so fsdp_allgather,
 * fsdp_reduce_scatter(_ex), fsdp_zero_grad, fsdp_adamw_step and fsdp_step
 * return FSDP_E_STATE until fsdp_load_params reloads the unit; after
 * FSDP_KSTATUS_DRAIN_TIMEOUT every call but fsdp_unit_destroy and the
 * read-only queries is refused (destroy and recreate the unit).  Calls
 * enqueued before the word is read are not refused: read it before trusting
 * any result that followed the launch in question. */
FSDP_API int fsdp_kernel_status(fsdp_unit* unit, int32_t* flags, void* stream);

/* Library infrastructure (the pages have no counterpart).
 * The bound of every wait of this unit's staged kernels: `seconds` in
 * [1e-6, 60] (10 s until set).  withhold_next arms a one-shot test of the
 * give-up path (0: none): in the next reduce-scatter or fused fsdp_step
 * launch of this unit, if it is one of the shared-memory staged kernels,
 * CTA 0 arms the barrier of its first stage but issues none of that stage's
 * copies, so that wait runs out exactly as for a copy that never arrives.
 * With 1 the kernel raises FSDP_KSTATUS_WAIT_TIMEOUT, waits for its other
 * copies and returns with its outputs incomplete; with 2 its drain also
 * waits on the withheld stage, runs out again and raises
 * FSDP_KSTATUS_DRAIN_TIMEOUT as well (no copy is in flight, so nothing lands
 * late).  The launch touches no memory a normal launch would not (it reads
 * and writes less).  The next launch of either kind consumes the request. */
FSDP_API int fsdp_unit_set_wait_limit(fsdp_unit* unit, double seconds, int withhold_next);

/* Library infrastructure (the pages have no counterpart).
 * Self-test of the bounded wait on the current device: one CTA waits on an
 * mbarrier that nothing completes, gives up after `limit_seconds` (1e-3 ..
 * 10), and reports through a status word like the staged kernel does.
 * Synchronous on `stream`; *timed_out is 1 when the wait ran out and the
 * status came back (the expected outcome), and the context stays usable. */
FSDP_API int fsdp_selftest_bounded_wait(double limit_seconds, int32_t* timed_out, void* stream);

/* ---- profiling ------------------------------------------------------------- */
/* Library infrastructure (the pages have no counterpart). */

/* While enabled, every kernel the unit launches is bracketed by CUDA events
 * recorded on its launch stream (launches on a stream that is being captured
 * into a CUDA graph are not timed).  fsdp_profile_read waits for the recorded
 * events and returns, for one FSDP_KERNEL_* kind, the summed device time in
 * milliseconds and the launch count since the last reset.  Disabling keeps
 * the records; fsdp_profile_reset drops them. */
FSDP_API int fsdp_profile_enable(fsdp_unit* unit, int on);
FSDP_API int fsdp_profile_read(fsdp_unit* unit, int kernel, double* total_ms, int64_t* launches);
FSDP_API int fsdp_profile_reset(fsdp_unit* unit);

/* ---- host-resident buffers -------------------------------------------------- */
/* Library infrastructure (the pages have no counterpart). */

/* Device address of pinned (page-locked, mapped) host memory, e.g. from
 * cudaHostAlloc or a pinned torch tensor.  Gradient buffers given to
 * fsdp_reduce_scatter / fsdp_step may live there: the reduce-scatter then reads
 * them straight over the host link, with no staging copy.  Returns
 * FSDP_E_INVALID_ARG if `host` is not pinned, mapped host memory. */
FSDP_API int fsdp_host_device_pointer(const void* host, void** dev);

/* ---- errors -------------------------------------------------------------- */
/* Library infrastructure (the pages have no counterpart). */
FSDP_API const char* fsdp_strerror(int code);
FSDP_API const char* fsdp_last_error(void);    /* calling thread's latest failure reason */

#ifdef __cplusplus
}
#endif
#endif /* FSDP_UNIT_H */

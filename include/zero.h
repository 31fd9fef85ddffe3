/*
 * zero.h -- C ABI of the GB300 (sm_103a) sharded mixed-precision AdamW step.
 *
 * The data-parallel hot path of ZeRO as described on the page "Zero Redundancy
 * Optimizer (ZeRO) and Fully Sharded Data Parallelism (FSDP): Mathematical
 * Foundations of Memory Partitioning, Communication Complexity, and Overlapped
 * Execution" (llms.blog), sections "ZeRO-Stage 1/2/3", "Execution Flow for
 * ZeRO-1", "ZeRO-3 / FSDP Layer Execution Lifecycle" and "FSDP-1: FlatParameter
 * and Module-Level Wrapping".
 *
 * The N_d data-parallel ranks are emulated inside one GPU: every rank's 16-bit
 * gradient contribution is a separate device buffer.  For each shard a bound
 * rank owns, one fused kernel
 *   (1) reduces the N_d contributions in fp32, r ascending, and multiplies by
 *       inv = fp32(1 / (N_d * loss_scale))   [the reduce-scatter's reduction],
 *   (2) ORs a global non-finite flag           [dynamic loss-scale skip],
 *   (3) applies AdamW to the fp32 master/m/v of the shard,
 *   (4) casts the new weight to bf16/fp16 into the all-gather destination.
 *
 * Conventions
 *  - Every call returns a zero_status_t; no exception or abort crosses the ABI.
 *    On an error, zero_last_error() (thread-local) describes it.
 *  - The plan owns host tables and a few scalars only.  ALL device memory
 *    (state, contributions, 16-bit buffers, workspace) is owned by the caller
 *    and is never freed by the library.  The library allocates no device memory.
 *  - Calls that take a `stream` (a cudaStream_t passed as void*) are
 *    asynchronous on it, except zero_set_scaler, zero_read_state,
 *    zero_step_host_finish and zero_step_finish with a result pointer, which
 *    synchronise it.  The skip decision, the applied-step count t, the current
 *    ping-pong half and the loss scale live on the device (in the workspace),
 *    so a training loop enqueues step after step without waiting for the host.
 *    Issue every call of one plan on one stream (or order the streams
 *    yourself).
 *  - Device pointers must be aligned to their element size (2 B for 16-bit
 *    data, 4 B for fp32, 16 B for the workspace); otherwise ZERO_EALIGN.  The
 *    128-bit vector path is used when every base pointer is 16-byte aligned and
 *    every stream of a launch has the same element phase modulo 8 (always true
 *    for the state layout below when bucket_elems is a multiple of 8); other
 *    launches use the scalar path of the same kernel.
 *  - Kernels never trap or assert.  The only waits are those of the bulk-staged step and
 *    gather kernels (zero_set_option, ZERO_OPT_STAGING / ZERO_OPT_GATHER_STAGING) on their
 *    shared-memory barriers; each is bounded in time (ZERO_OPT_WAIT_LIMIT_NS) and one that
 *    runs out is reported as ZERO_ETIMEOUT.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZERO_OK = 0,
    ZERO_EINVAL = 1,  /* invalid argument (null pointer, bad stage, size, rank ...) */
    ZERO_EALIGN = 2,  /* a pointer is not aligned to its element size */
    ZERO_ECUDA = 3,   /* a CUDA runtime call failed */
    ZERO_ESTATE = 4,  /* call out of order (e.g. finish before every bucket was stepped) */
    ZERO_ERANGE = 5,  /* a size beyond a documented limit */
    ZERO_ETIMEOUT = 6, /* a bounded wait inside a kernel ran out; the step was discarded */
    ZERO_ENOMEM = 7   /* a host resource (memory, a worker thread) could not be obtained; the
                         call changed nothing it had not finished */
} zero_status_t;

enum { ZERO_BF16 = 0, ZERO_FP16 = 1 };

/* Largest supported N_d (contribution pointers travel in the kernel parameters). */
#define ZERO_MAX_RANKS 128

typedef struct zero_plan zero_plan_t;

/* AdamW hyperparameters (decoupled weight decay, bias-corrected moments), plus the optional
 * global gradient norm: max_grad_norm > 0 clips the averaged, unscaled gradient g by
 * fp32(min(1, max_grad_norm / (norm + 1e-6))), norm = sqrt(sum of fp32(g*g) in double), which
 * needs zero_grad_norm (or zero_grad_norm_host) over every bucket/unit of the step first;
 * flags & ZERO_REPORT_GRAD_NORM computes the norm inside the fused pass for reporting (no
 * clipping, no extra pass). */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    double max_grad_norm;    /* 0: no clipping */
    int64_t flags;           /* ZERO_REPORT_GRAD_NORM */
} zero_hyper_t;

#define ZERO_REPORT_GRAD_NORM 1

/* Dynamic loss scale (kept on the device once set with zero_set_scaler).  On a step whose
 * reduced gradient holds inf/nan the step is skipped and scale = max(scale * backoff_factor,
 * min_scale); after growth_interval consecutive applied steps scale *= growth_factor. */
typedef struct {
    double scale;
    double growth_factor;
    double backoff_factor;
    double min_scale;
    int64_t growth_interval;
    int64_t good_steps;      /* applied steps since the last change of scale (initial value) */
} zero_scaler_t;

typedef struct {
    int64_t n_tensors;
    int64_t n_units;         /* FSDP units (stage 3); 1 for stages 1/2 */
    int64_t n_buckets;       /* reduce-scatter buckets (stages 1/2); n_units for stage 3 */
    int64_t phi;             /* sum of tensor sizes */
    int64_t phi_pad;         /* sum of padded unit sizes = length of the global flat index space */
    int64_t shard;           /* elements each rank owns: sum over units of phi_pad_u / N_d */
    int64_t max_contrib_elems; /* elements every contribution buffer must hold for the largest
                                  bucket (stages 1/2) or unit (stage 3) */
    int64_t max_unit_pad;    /* largest padded unit (stage 3 gather destination length) */
    int64_t workspace_bytes; /* device workspace the caller provides (zero_bind): 256 bytes of
                                step state and a table of Adam bias corrections */
    int32_t n_d;
    int32_t stage;
    int32_t dtype16;
    int32_t reserved;
    int64_t host_staging_bytes; /* each of the two device staging areas zero_bind_host_staging
                                   takes: N_d areas of max_contrib_elems 16-bit elements, each
                                   rounded up to a multiple of 8 elements */
} zero_plan_info_t;

/* Table selectors for zero_plan_tables (all entries int64, row-major). */
enum {
    ZERO_TABLE_TENSOR_OFFSET = 0,  /* 1 col: global flat offset of each tensor */
    ZERO_TABLE_UNITS = 1,          /* 7 cols: first tensor, tensor count, numel, numel_pad,
                                      shard size S_u, global base, rank-local shard base */
    ZERO_TABLE_SHARD_SEGMENTS = 2, /* 6 cols: rank, unit, tensor (-1 = padding), offset in the
                                      tensor (or the padding), rank-local shard offset, length;
                                      ordered by rank, unit, flat position */
    ZERO_TABLE_BUCKET_SEGMENTS = 3,/* 5 cols: bucket, rank, flat start, rank-local shard offset,
                                      length; ordered by bucket, rank (stages 1/2) */
    ZERO_TABLE_STATE_LAYOUT = 4,   /* 4 cols: rank, unit, element offset of the unit's shard in the
                                      rank's state buffers, length (physical layout, see zero_bind) */
    ZERO_TABLE_PARAM_CHUNKS = 5    /* per-parameter plans, 10 cols: rank, unit, tensor, first row,
                                      owned rows, cols, chunk rows, offset of the owned rows in the
                                      unit's gradient buffer, logical and physical offset of the
                                      local shard in the rank's state; ordered rank, unit, tensor */
};

/* Device-resident step state, read back by zero_read_state / zero_step_finish. */
typedef struct {
    int32_t skipped;         /* 1: the last finished step saw inf/nan and was not applied */
    int32_t current;         /* current half (0/1) of every ping-pong pair */
    int64_t t;               /* applied steps so far */
    double scale;            /* loss scale of the next step */
    int64_t good_steps;      /* applied steps since the last change of scale */
    int64_t skipped_total;   /* skipped steps so far */
    int64_t finished;        /* finished steps (applied + skipped) */
    double grad_norm;        /* global gradient norm of the last finished step, -1 if not computed */
} zero_step_result_t;

/* Per-rank bytes.  logical[s][c]: stage s in (DDP, ZeRO-1, ZeRO-2, ZeRO-3), component c in
 * (16-bit params, 16-bit grads, fp32 optimizer state) at phi_pad -- the closed forms of
 * section "Static Memory Allocation" and the stage equations M(ZeRO-1/2/3). */
typedef struct {
    int64_t logical[4][3];
    int64_t logical_total[4];
    int64_t logical_ddp_fp32_grads;  /* the 18-Phi variant with fp32 gradient buffers */
    int64_t physical_state_bytes;    /* per bound rank: master/m/v, both ping-pong copies */
    int64_t physical_param16_bytes;  /* stages 1/2: flat buffer; stage 3: one rank's shard */
    int64_t physical_contrib_bytes;  /* N_d contribution buffers of the largest bucket/unit */
    int64_t physical_gather_bytes;   /* stage 3: largest full-unit buffer */
    int64_t workspace_bytes;
} zero_mem_report_t;

/* Elements sent (= received) per rank per step, sections "Standard Ring-AllReduce
 * Communication Analysis", "ZeRO-1 and ZeRO-2 Communication Volume", "ZeRO-3 and FSDP
 * Communication Volume".  One ring collective over phi_pad moves (N_d-1)/N_d * phi_pad. */
typedef struct {
    int64_t per_collective;   /* (N_d - 1) * shard */
    int64_t ddp;              /* all-reduce = scatter-reduce + all-gather */
    int64_t zero1;            /* reduce-scatter + all-gather */
    int64_t zero2;
    int64_t zero3;            /* forward all-gather + backward all-gather + reduce-scatter */
    int64_t this_stage;       /* the entry for the plan's stage */
    int64_t bytes_per_elem;   /* 2 (16-bit) */
    int64_t collectives_per_step; /* reduce-scatters + all-gathers issued per step by this plan */
} zero_comm_report_t;

/* Build the flat-buffer partition ("FSDP-1: FlatParameter": tensors flattened in the given
 * order, each unit padded at its tail to a multiple of N_d and sliced into N_d equal shards).
 *   tensor_sizes[n_tensors]  element counts (>= 0)
 *   stage                    1, 2 or 3
 *   bucket_elems             stages 1/2: reduce-scatter bucket size in elements (0 = one
 *                            bucket); stage 3: must be 0
 *   unit_first[n_units]      stage 3: first tensor of each unit, strictly increasing, starting
 *                            at 0 (NULL / 0 = one unit); stages 1/2: must be NULL / 0
 *   dtype16                  ZERO_BF16 or ZERO_FP16
 * On success *out owns host memory only; release it with zero_plan_destroy. */
zero_status_t zero_plan_create(const int64_t* tensor_sizes, int64_t n_tensors, int n_d, int stage,
                               int64_t bucket_elems, const int64_t* unit_first, int64_t n_units,
                               int dtype16, zero_plan_t** out);

/* FSDP-2 per-parameter sharding ("FSDP-2: Per-Parameter Sharding via DTensor (fully_shard)":
 * each tensor sharded along its leading dimension, Shard(0), without flattening).  Tensor t has
 * dim0[t] rows of tensor_sizes[t] / dim0[t] elements; rank r owns rows
 * [r*c, min((r+1)*c, dim0[t])), c = ceil(dim0[t] / N_d), and holds a local shard of c rows per
 * tensor (rows past the tensor are padding, never touched).  Stage-3 semantics otherwise: units
 * group tensors for the gather, each unit's gradient buffer is its tensors concatenated without
 * padding (phi_pad == phi), zero_bind takes a 16-bit shard per rank, zero_gather_layer rebuilds
 * a unit (info.max_unit_pad elements).  Tables: ZERO_TABLE_UNITS and ZERO_TABLE_PARAM_CHUNKS. */
zero_status_t zero_plan_create_per_param(const int64_t* tensor_sizes, const int64_t* dim0,
                                         int64_t n_tensors, int n_d, const int64_t* unit_first,
                                         int64_t n_units, int dtype16, zero_plan_t** out);

/* Fill *out with the partition's sizes ("FSDP-1: FlatParameter": phi, phi_pad, the shard,
 * buckets and units) and the buffer sizes the caller allocates (contributions, gather
 * destination, workspace; see zero_plan_info_t).  Host-only; ZERO_EINVAL on NULL. */
zero_status_t zero_plan_info(const zero_plan_t* plan, zero_plan_info_t* out);

/* Element count of rank `rank`'s state buffers (master, m, v; and stage 3's 16-bit shard).
 * The layout places each unit's shard at an offset congruent, modulo 8, to the unit-local
 * start of that shard, so the fp32 state, the 16-bit contributions and the 16-bit output
 * share one 128-bit vector phase.  Unused gap elements are never read or written. */
zero_status_t zero_rank_state_elems(const zero_plan_t* plan, int rank, int64_t* elems);

/* Copy table `which` of the partition ("FSDP-1: FlatParameter": tensor offsets, units,
 * shard and bucket segments, state layout, per-parameter chunks) into dst (capacity `cap`
 * int64 values).  *n_rows receives the row count; if the table does not fit, nothing is
 * written and ZERO_ERANGE is returned. */
zero_status_t zero_plan_tables(const zero_plan_t* plan, int which, int64_t* dst, int64_t cap,
                               int64_t* n_rows);

/* Bind rank `rank`'s device buffers ("Static Memory Allocation": the 12 bytes of fp32
 * master/m/v per parameter a rank keeps for its shard; caller-owned, each of
 * zero_rank_state_elems elements):
 *   master[2], m[2], v[2]  fp32 ping-pong pairs; index 0 holds the current state at bind time
 *   shard16                stage 3: the rank's 16-bit parameter shard; else NULL
 *   full16                 stages 1/2: the flat 16-bit parameter buffer (phi_pad elements),
 *                          shared by every rank (all replicas are identical); else NULL
 *   workspace              device memory of info.workspace_bytes, 16-byte aligned: the step
 *                          state (non-finite flag, current half, t, loss scale) and the bias
 *                          corrections; plan-wide: every bind must pass the same pointer
 * The first bind synchronously initialises the workspace (t = 0, half 0 current, scale 1).
 * Bind every rank before the first step.  Only bound ranks are updated by zero_step. */
zero_status_t zero_bind(zero_plan_t* plan, int rank, float* const master[2], float* const m[2],
                        float* const v[2], void* shard16, void* full16, void* workspace);

/* Stage 3 ("ZeRO-3 / FSDP Layer Execution Lifecycle": every rank holds only its shard of the
 * 16-bit parameters): register the 16-bit shard of a rank whose optimizer runs elsewhere, so
 * that zero_gather_layer can reconstruct full units.  The buffer follows that rank's layout. */
zero_status_t zero_bind_peer(zero_plan_t* plan, int rank, const void* shard16);

/* Dynamic loss scaling (not on the pages, which name fp16/bf16 mixed precision only; the
 * skip-and-back-off scheme of mixed-precision training).  Set (cfg != NULL) or disable
 * (cfg == NULL: scale fixed at 1) the dynamic loss scale: writes
 * cfg->scale and cfg->good_steps into the device state and keeps the growth/back-off settings.
 * Not inside an open step.  Synchronises `stream`. */
zero_status_t zero_set_scaler(zero_plan_t* plan, const zero_scaler_t* cfg, void* stream);

/* One fused reduce + AdamW + cast over every bound rank's part of bucket / unit `which`
 * ("Execution Flow for ZeRO-1" steps 2-4: reduce-scatter of the averaged gradient, update of
 * the owned shard, 16-bit write into the all-gather destination; "ZeRO-Stage 2": one call per
 * bucket as gradients are produced; "ZeRO-3 / FSDP Layer Execution Lifecycle": one per unit).
 *   grad_contribs[n_contribs]  n_contribs == N_d device pointers; contribution r holds rank r's
 *                              16-bit gradient for the whole range of the bucket (stages 1/2:
 *                              [b*B, min((b+1)*B, phi_pad)); which = -1: all of [0, phi_pad))
 *                              or of the unit (stage 3: phi_pad_u elements, padding zero).
 *                              Only the bound ranks' shard slices are read.
 *   hyper                      AdamW hyperparameters (identical for every call of one step);
 *                              betas in [0, 1)
 * The step index t + 1, the loss scale and the current half are read on the device.  A step
 * is the sequence of calls that covers every bucket (or unit) exactly once, ended by
 * zero_step_finish.  New state is written to the non-current half of each ping-pong pair.
 * The first call with new betas copies a bias-correction table into the workspace. */
zero_status_t zero_step(zero_plan_t* plan, const void* const* grad_contribs, int64_t n_contribs,
                        int64_t which, const zero_hyper_t* hyper, void* stream);

/* Gradient-norm pre-pass of bucket / unit `which` (same contributions as zero_step): adds the
 * bound ranks' sum of fp32(g*g) to the step's norm on the device, reading only the 16-bit
 * contributions (2 N_d bytes per element).  Needed before the first zero_step of a step that
 * clips (hyper->max_grad_norm > 0); call it for every bucket/unit, before any zero_step. */
zero_status_t zero_grad_norm(zero_plan_t* plan, const void* const* grad_contribs,
                             int64_t n_contribs, int64_t which, void* stream);

/* End the step on the device: a re-cast kernel (which does nothing unless the flag is set)
 * rewrites the 16-bit parameters of a skipped step from the unchanged master, and its last
 * block to finish commits: it either makes the new state current (t += 1, loss-scale growth)
 * or keeps the old one (loss-scale back-off), and clears the flag.  With out == NULL the call
 * only enqueues this work; with out != NULL it also synchronises `stream` and reads the
 * state. */
zero_status_t zero_step_finish(zero_plan_t* plan, void* stream, zero_step_result_t* out);

/* Read the device-resident step state (synchronises `stream`).  zero_read_state and
 * zero_step_finish (out != NULL) return ZERO_ETIMEOUT, with *out filled, when a wait of a
 * bulk-staged kernel (step or gather) ran out since the state was last read: every step
 * finished since then was discarded (state, t, loss scale and counters unchanged; 16-bit
 * parameters rewritten from the current master).  Reading the state clears the condition. */
zero_status_t zero_read_state(zero_plan_t* plan, void* stream, zero_step_result_t* out);

/* Execution options of a plan (not inside an open step; values are checked here):
 *   ZERO_OPT_STAGING        which step kernel zero_step launches.  ZERO_STAGING_BULK: per block
 *                           a producer warp stages the contribution slices and the fp32 state
 *                           tile by tile into a ring of shared-memory buffers with 1-D
 *                           cp.async.bulk copies (the TMA engine) completing on mbarriers, and
 *                           four consumer warps reduce and update from shared memory.
 *                           ZERO_STAGING_REGISTER_LOADS: every thread loads them with 128-bit
 *                           register loads.  ZERO_STAGING_AUTO (default): the staged kernel where
 *                           its ring gives two resident blocks per SM with tiles of at least 512
 *                           elements, or three with 512-element tiles (on GB300 with the default
 *                           geometry: N_d = 4-11, 13-20 and 22-50, where it measured faster at all
 *                           but N_d = 10, 11 and 33), register loads elsewhere.  All give
 *                           identical results, bit for bit.  Launches whose streams do not
 *                           share one 16-byte phase use the scalar register-load path either
 *                           way, and so do steps that report the gradient norm from the fused
 *                           pass (ZERO_REPORT_GRAD_NORM without clipping).
 *   ZERO_OPT_WAIT_LIMIT_NS  bound on each barrier wait of the bulk-staged kernels, in ns of
 *                           %globaltimer (default 1e9; 0 gives up at the first wait that does
 *                           not succeed at once).  A wait that runs out sets the plan's error
 *                           word, its block drains its own copies in flight and returns.
 *   ZERO_OPT_BULK_TILE      elements per staged tile, a multiple of 8 in [8, 8192]; 0 (default):
 *                           the largest multiple of 512 up to 2048 with tile * (2 N_d + 12)
 *                           bytes within 53.5 KB; 512 while that is within 56 KB (N_d <= 50);
 *                           a power of two below 512 beyond.
 *   ZERO_OPT_BULK_STAGES    ring depth in [2, 16]; 0 (default): 2 (two blocks per SM).
 *   ZERO_OPT_GATHER_STAGING which kernel zero_gather_layer launches.  ZERO_STAGING_AUTO
 *                           (default) and ZERO_STAGING_BULK: one lane per block copies chunks
 *                           of the shards through a ring of shared-memory entries with 1-D
 *                           cp.async.bulk loads (completing on mbarriers) and bulk stores,
 *                           the loads two chunks ahead of the stores; ZERO_STAGING_REGISTER_LOADS:
 *                           128-bit register copies.  Gathers whose copies do not share one
 *                           16-byte phase, and plans without a bound workspace (which holds the
 *                           error word), use register loads either way.  Identical results.
 *   ZERO_OPT_GATHER_CHUNK   elements per bulk copy of the staged gather, a multiple of 8 in
 *                           [8, 32768]; 0 (default): 16384 (32 KB).
 *   ZERO_OPT_GATHER_STAGES  its ring entries in [3, 32]; 0 (default): 4 (a 128 KB ring).
 * A geometry whose ring does not fit one block's shared memory gives ZERO_ERANGE and leaves
 * the earlier one in place. */
enum {
    ZERO_OPT_STAGING = 0,
    ZERO_OPT_WAIT_LIMIT_NS = 1,
    ZERO_OPT_BULK_TILE = 2,
    ZERO_OPT_BULK_STAGES = 3,
    ZERO_OPT_LAST_STEP_KERNEL = 4,  /* read only: the step kernel of the last zero_step launch
                                       (1 staged, 0 register loads, -1 none yet) */
    ZERO_OPT_GATHER_STAGING = 5,
    ZERO_OPT_GATHER_CHUNK = 6,
    ZERO_OPT_GATHER_STAGES = 7,
    ZERO_OPT_HOST_PIPELINE = 8,     /* zero_step_host: 1 (default) copies the next call's
                                       gradients while this call's step runs; 0 runs each call's
                                       host->device copies, step and device->host copies one
                                       after another, after the previous call's (for measuring
                                       what the overlap hides) */
    ZERO_OPT_HOST_H2D_BYTES = 9,    /* read only: bytes zero_step_host copied host->device in
                                       the last step finished by zero_step_host_finish */
    ZERO_OPT_HOST_D2H_BYTES = 10,   /* read only: bytes copied device->host in that step (the
                                       updated 16-bit parameters, re-copies after a skip
                                       included) */
    ZERO_OPT_LAST_GATHER_IN_STEP = 11, /* read only: 1 if the last zero_step_gather_next
                                       streamed its gather inside the step launch, 0 if the
                                       gather ran as a launch of its own, -1 none yet */
    ZERO_OPT_OFFLOAD_DEFER = 12,    /* offloaded plans: 0 (default) zero_offload_step reduces its
                                       contributions into host memory in stream order; 1 it only
                                       runs the non-finite flag pass, and zero_offload_finish,
                                       once every call's flag is known, streams the reductions
                                       (a skipped step skips them) while the host threads update
                                       each group as it lands.  With 1 the contributions of every
                                       call must stay unchanged until zero_offload_finish
                                       returns. */
    ZERO_OPT_UNIT_ORDER = 13        /* stage 3, zero_step_units_overlapped: 0 (default) steps the
                                       units first to last, each unit's gather prefetching the
                                       next one (a forward pass's order); 1 last to first, each
                                       prefetching the one before it (a backward pass's order,
                                       in which the gradients arrive).  Same results. */
};
enum { ZERO_STAGING_REGISTER_LOADS = 0, ZERO_STAGING_BULK = 1, ZERO_STAGING_AUTO = 2 };
zero_status_t zero_set_option(zero_plan_t* plan, int option, int64_t value);

/* Read an option (the tile, stages, chunk and entries in effect when left at 0), or
 * ZERO_OPT_LAST_STEP_KERNEL. */
zero_status_t zero_get_option(const zero_plan_t* plan, int option, int64_t* value);

/* Overwrite the device-resident step state, e.g. when resuming from a checkpoint whose fp32
 * master/m/v were saved from the half `in->current` after `in->t` applied steps.  Clears the
 * non-finite flag.  Not inside an open step.  Synchronises `stream`. */
zero_status_t zero_restore_state(zero_plan_t* plan, const zero_step_result_t* in, void* stream);

/* Stage 3 all-gather of unit `unit` ("ZeRO-3 / FSDP Layer Execution Lifecycle"): copies the
 * N_d 16-bit shards (bound or peer ranks) into full_unit16 (phi_pad_u elements, padding
 * included), asynchronously on `stream` with the kernel ZERO_OPT_GATHER_STAGING selects.  The
 * unit stays "gathered" until zero_release_layer.  A barrier wait of the staged gather that
 * runs out leaves the unit incomplete and sets the plan's error word (see zero_read_state). */
zero_status_t zero_gather_layer(zero_plan_t* plan, int64_t unit, void* full_unit16, void* stream);

/* zero_step of stage-3 unit `unit` and zero_gather_layer of unit `next_unit` into next_full16
 * (max_unit_pad elements suffice) in one launch where possible ("Overlapping Computation and
 * Communication Streams": the next unit's all-gather runs while this unit is reduced and
 * updated; "ZeRO-3 / FSDP Layer Execution Lifecycle").  When the bulk-staged step kernel runs
 * the unit and the gather's copy list fits its parameter block (32 copies, or 256 when the
 * call has more than 32 work items), each block's producer warp streams gather chunks through
 * its shared-memory ring after its last tile; otherwise the gather follows as its own launch
 * on `stream` (ZERO_OPT_LAST_GATHER_IN_STEP tells which).  Results are those of the two calls
 * made one after the other.  unit must name one unit (not -1) and next_unit must differ from
 * it (the step writes unit's shards), else ZERO_EINVAL; next_full16 must not overlap any buffer
 * of the plan.  The errors of zero_step and of zero_gather_layer; next_unit stays gathered
 * until zero_release_layer. */
zero_status_t zero_step_gather_next(zero_plan_t* plan, const void* const* grad_contribs,
                                    int64_t n_contribs, int64_t unit, const zero_hyper_t* hyper,
                                    int64_t next_unit, void* next_full16, void* stream);

/* A whole stage-3 step with the all-gather overlapped ("Overlapping Computation and
 * Communication Streams"): for every unit u in order (ZERO_OPT_UNIT_ORDER: first to last,
 * or last to first), `comm_stream` gathers u into gather_bufs[i % 2] (i = its position in that
 * order; each buffer max_unit_pad elements) while `compute_stream` runs the fused step of the
 * unit before it; unit u's step waits only for its own gather (the point where a layer's
 * backward would consume W_u), and a buffer is re-filled only after the step that followed
 * its gather has been enqueued past it.  comm_stream == NULL: one stream; the first unit in
 * the order is gathered on its own, then each unit's step and the next unit's gather run as
 * zero_step_gather_next (one launch each where possible).  Ends with zero_step_finish on `compute_stream` (out as
 * there).  unit_contribs: n_units * N_d pointers, unit-major (unit u's N_d contributions at
 * [u * N_d]).  With max_grad_norm > 0 a norm pre-pass over every unit runs first on
 * compute_stream.  Stage 3 only; two given streams must differ. */
zero_status_t zero_step_units_overlapped(zero_plan_t* plan, const void* const* unit_contribs,
                                         int64_t n_ptrs, void* const* gather_bufs,
                                         const zero_hyper_t* hyper, void* compute_stream,
                                         void* comm_stream, zero_step_result_t* out);

/* ---- ZeRO-Offload ("ZeRO-Offload Mechanics": the optimizer step runs on the host CPU over
 * fp32 state in host memory; gradients go to the host, updated parameters come back). ----
 * Bind rank `rank` with host-resident state: master/m/v (host memory, zero_rank_state_elems
 * floats each, updated in place by CPU threads), grad_host (pinned, same length: the GPU
 * writes the averaged fp32 gradient there over NVLink-C2C), param16_host (pinned, 16-bit:
 * the CPU writes the new parameters there before they are copied back).  shard16 / full16 /
 * workspace as for zero_bind.  A plan's bound ranks are either all offloaded or all on the
 * GPU; bind every rank before the first step. */
zero_status_t zero_bind_offload(zero_plan_t* plan, int rank, float* master, float* m, float* v,
                                float* grad_host, void* param16_host, void* shard16, void* full16,
                                void* workspace);

/* Offloaded counterpart of zero_step ("ZeRO-Offload Mechanics": gradients to the host, the
 * optimizer step on the CPU): reduces bucket / unit `which` on the GPU (same
 * contributions, scaling and non-finite flag) and writes the averaged gradient into the bound
 * ranks' grad_host.  It first runs the reduction for the non-finite flag alone (no writes),
 * then the writing reduction in groups of segments of at least 4M elements, an event after
 * each group.  Clipping (max_grad_norm > 0) needs zero_grad_norm over every bucket/unit
 * first (ZERO_ESTATE otherwise); the finish then scales each gradient by the coefficient
 * min(1, max_grad_norm / (norm + 1e-6)), formed in double as the GPU step forms it and
 * rounded once to fp32.  ZERO_REPORT_GRAD_NORM is refused (ZERO_EINVAL): with clipping the
 * norm is reported anyway. */
zero_status_t zero_offload_step(zero_plan_t* plan, const void* const* grad_contribs,
                                int64_t n_contribs, int64_t which, const zero_hyper_t* hyper,
                                void* stream);

/* End an offloaded step.  Once the step's last flag pass is done, the step state is read on
 * a side stream.  Then `threads` CPU threads (kept by the plan from step to step, asleep in
 * between, ended by zero_plan_destroy) apply AdamW to the host state with the same fp32
 * operation order as the GPU kernel, each group of segments as soon as its gradient has
 * landed.  Finished ranges of 16-bit parameters are copied to the all-gather destination on
 * `stream` while the rest is still being updated.  If the flag is set, the call waits for
 * every gradient and re-casts the unchanged master instead.  Then the commit kernel updates
 * t / the loss scale.  Returns when the host update is complete (the copies and the commit
 * are enqueued on `stream`); out as for zero_step_finish. */
zero_status_t zero_offload_finish(zero_plan_t* plan, int threads, void* stream,
                                  zero_step_result_t* out);

/* ---- Steps fed from host memory ("Execution Flow for ZeRO-1" steps 2-4 with the gradients
 * and the all-gather's result in host memory; "Overlapping Computation and Communication
 * Streams": the transfer of the next bucket runs while the current one is reduced and
 * updated). ----
 * Bind two device staging areas of bytes_each bytes (caller-owned device memory, each at
 * least info.host_staging_bytes, 16-byte aligned, not overlapping) for zero_step_host.  Area
 * k of a call holds rank r's contribution at byte offset r * P, P = bytes_each / N_d rounded
 * down to a multiple of 16.  info.host_staging_bytes gives P room for the largest bucket or
 * unit; bucket -1 on a plan of several buckets or units needs P >= 2 * (its range), i.e.
 * areas of N_d * 2 * R bytes, R = phi_pad rounded up to a multiple of 8 (stages 1/2).  Not inside an open step; bind every rank
 * first.  ZERO_ERANGE if bytes_each < info.host_staging_bytes; ZERO_EINVAL if the areas
 * overlap or are not device memory of the plan's device. */
zero_status_t zero_bind_host_staging(zero_plan_t* plan, void* const staging[2], int64_t bytes_each);

/* zero_step for bucket / unit `which` with host buffers:
 *   host_contribs[n_contribs]  n_contribs == N_d pointers to pinned host memory (cudaHostAlloc
 *                              or cudaHostRegister), laid out like zero_step's contributions
 *                              (the bucket's or unit's range); only the slices the bound ranks
 *                              read are copied
 *   host_out16                 pinned host memory of the same range length: receives the
 *                              updated 16-bit parameters of every element the bound ranks own
 *                              in the range (all ranks bound: the whole range, i.e. what the
 *                              all-gather delivers), at the element's offset in the range
 * The library copies the slices into staging area (call count mod 2) on its own copy stream
 * once the step that last read that area is done, runs zero_step on `stream` after the copies,
 * and copies the 16-bit results to host_out16 on a second stream of its own after the step.
 * With ZERO_OPT_HOST_PIPELINE = 1 (default) the copies of the next call therefore run while
 * this call's step does; a call that is the step's only call (bucket -1, or the plan's one
 * bucket) is cut into pieces of its range instead (at least 2^24 elements each, at most 8),
 * each piece's step launch and copy back running while the next piece is copied in.
 * Asynchronous: host_contribs must stay unchanged and host_out16 is
 * not final until zero_step_host_finish returns.  ZERO_REPORT_GRAD_NORM is allowed; clipping
 * (max_grad_norm > 0) needs the norm pre-pass of every bucket/unit first (zero_grad_norm_host,
 * or zero_grad_norm on device copies), as zero_step does.  ZERO_ESTATE without bound staging;
 * ZERO_ERANGE (nothing enqueued) if the call's range does not fit a rank's part of the areas;
 * ZERO_EINVAL for NULL or unpinned host pointers and the argument errors of zero_step. */
zero_status_t zero_step_host(zero_plan_t* plan, const void* const* host_contribs,
                             int64_t n_contribs, int64_t which, const zero_hyper_t* hyper,
                             void* host_out16, void* stream);

/* zero_grad_norm with host buffers: copies the slices of bucket / unit `which` the bound ranks
 * read from pinned host memory (host_contribs as for zero_step_host) into the next staging
 * area, in the same rotation and order as zero_step_host, and runs the norm pre-pass on
 * `stream` over them.  For clipped steps fed from host memory: every bucket's norm call first,
 * then the zero_step_host calls, which copy the gradients again (twice the host-to-device
 * bytes of an unclipped step; the counters of ZERO_OPT_HOST_H2D_BYTES include both).  The
 * errors of zero_grad_norm, and those of zero_step_host for the staging and host pointers. */
zero_status_t zero_grad_norm_host(zero_plan_t* plan, const void* const* host_contribs,
                                  int64_t n_contribs, int64_t which, void* stream);

/* End a step that had zero_step_host calls: zero_step_finish on `stream`, then wait for every
 * device->host copy; if the step was skipped (or discarded, ZERO_ETIMEOUT) the re-cast 16-bit
 * parameters are copied to each call's host_out16 again.  Always synchronises; out (may be
 * NULL) and the return value as for zero_step_finish with a result pointer.  A step with host
 * calls must end here (zero_step_finish returns ZERO_ESTATE for it). */
zero_status_t zero_step_host_finish(zero_plan_t* plan, void* stream, zero_step_result_t* out);

/* Release after use ("ZeRO-3 / FSDP Layer Execution Lifecycle": the full parameters of a unit
 * are freed once its forward or backward is done): mark unit `unit`'s gathered buffer free;
 * the caller may reuse its memory.  ZERO_ESTATE if the unit is not gathered. */
zero_status_t zero_release_layer(zero_plan_t* plan, int64_t unit);

/* Fill *out with the per-rank memory accounting of the plan (the closed forms of "Static
 * Memory Allocation" and the stage equations, at phi_pad, plus this emulation's physical
 * bytes; see zero_mem_report_t).  Host-only; ZERO_EINVAL on NULL arguments. */
zero_status_t zero_memory_report(const zero_plan_t* plan, zero_mem_report_t* out);

/* Fill *out with the elements each rank sends per step under DDP and ZeRO-1/2/3 ("Standard
 * Ring-AllReduce Communication Analysis", "ZeRO-1 and ZeRO-2 Communication Volume", "ZeRO-3
 * and FSDP Communication Volume"; see zero_comm_report_t).  Host-only; ZERO_EINVAL on NULL. */
zero_status_t zero_comm_report(const zero_plan_t* plan, zero_comm_report_t* out);

/* ---------------------------------------------------------------------------------------
 * No-allocation variant of the fused step (the pages have no counterpart of this call).
 *
 * For callers that cannot allocate device memory themselves: code that runs inside a host
 * framework which has reserved the GPU's memory for its own pool, or latency-critical loops
 * that cannot afford cudaMalloc/cudaFree (which may synchronise the whole device).  Such a
 * caller cannot provide the workspace zero_bind needs.  This call needs no plan and no
 * workspace: it runs the same fused reduce + AdamW + cast kernel over ONE flat range and keeps
 * the kernel's scratch (the 4-byte non-finite flag) in a library-owned static device array of
 * ZERO_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads the library holds that array until
 * the process exits.  The library allocates nothing here: no cudaMalloc, no cudaFree.
 *
 *   grad_contribs[n_d]   device pointers, n elements of 16-bit gradient each
 *   master_in/m_in/v_in  fp32 state read (n elements); not modified
 *   master_out/m_out/v_out  fp32 state written (n elements); must not alias the inputs
 *   out16                16-bit parameters written (n elements), even when the flag is set
 *   hyper                AdamW hyperparameters; max_grad_norm and flags must be 0 here
 *   t                    1-based index of the step being applied (bias correction)
 *   loss_scale           gradients are multiplied by 1 / (n_d * loss_scale)
 *   *nonfinite           receives 1 if any reduced gradient element is inf/nan, else 0
 * The call enqueues its work on `stream` and then synchronises `stream` to read the flag.
 *
 * Set-up: the first call on each device (in each CUDA context: a device reset makes a new
 * one) looks up the array's device address, with that device current, and caches it.  All
 * calls share the one array: the flag is cleared at the start of every call, and calls that
 * overlap on the GPU (different streams, threads or processes sharing the library) race on it.
 * Limits: n_d <= ZERO_MAX_RANKS (else ZERO_ERANGE); the call uses 4 of the
 * ZERO_NOALLOC_SCRATCH_BYTES bytes whatever n and n_d are.
 * --------------------------------------------------------------------------------------- */
#define ZERO_NOALLOC_SCRATCH_BYTES 256

zero_status_t zero_step_range_noalloc(const void* const* grad_contribs, int n_d, int64_t n,
                                      int dtype16, const float* master_in, const float* m_in,
                                      const float* v_in, float* master_out, float* m_out,
                                      float* v_out, void* out16, const zero_hyper_t* hyper,
                                      int64_t t, double loss_scale, void* stream,
                                      int32_t* nonfinite);

/* Text of the last error of the calling thread (empty if none); valid until its next call. */
const char* zero_last_error(void);

/* Release a plan: its host tables, and the CUDA events, side stream and host worker threads
 * it created on first use (the caller's device memory is not touched).  Not while work the
 * plan enqueued may still use them: synchronise its streams first.  NULL is ignored. */
void zero_plan_destroy(zero_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_H */

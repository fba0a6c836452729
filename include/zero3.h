/*
 * zero3.h -- C ABI of the ZeRO-3 sharded mixed-precision AdamW hot path.
 *
 * One GPU emulates N_d data-parallel ranks: every rank's local gradients,
 * fp32 optimizer-state shard and bf16 parameter shard are separate device
 * buffers, and the "collectives" are the reads and writes the kernels make
 * across them.  No call here talks to another GPU.
 *
 * Conventions
 *  - Every call returns a zero3_status; nothing aborts, throws or exits.
 *  - Device buffers are owned by the caller (allocated with any CUDA
 *    allocator) and passed as raw pointers; every device pointer must be
 *    16-byte aligned (ZERO3_EINVAL otherwise).  Element offsets inside
 *    buffers need no alignment: the kernels handle any phase.
 *  - Arrays of per-rank pointers (grads[], master[], ...) are HOST arrays of
 *    n_ranks device pointers.  The library reads them during the call only.
 *    A rank whose shard does not meet the requested flat range may pass NULL
 *    for its state pointers (this is how one device holds only rank 0).
 *  - Compute calls are asynchronous on the given stream.  A kernel fault is
 *    reported as ZERO3_ECUDA by a later call or by zero3_sync.
 *  - Kernels are launched with programmatic stream serialization: one may be
 *    scheduled while the previous kernel of its stream is still draining,
 *    but every thread waits for the previous grids to complete, and their
 *    writes to be visible, before it touches memory.  Plain stream order
 *    therefore holds for the data, whatever kernel (this library's or
 *    another's) comes before or after.  The compute calls (steps,
 *    reduce-scatter, all-gathers, quantization) can be captured in a CUDA
 *    graph; the fetch, release and coordinator calls keep host-side state
 *    (status, references, events) that a replay would not repeat, so they
 *    are issued directly.
 *  - A plan is owned by the library: created by zero3_partition, released by
 *    zero3_plan_destroy.  Calls on one plan must not run concurrently from
 *    several host threads.
 *
 * Citations name the web page (title or site) and its section.
 *  [baike]   "DeepSpeed ZeRO-3", baike.kuaisou.com/zh/1104615
 *  [111qqz]  "ddp-to-zero-memory-sharding", 111qqz.com/2026/10/ddp-to-zero-memory-sharding
 *  [cnhsyj]  ZERO tutorial, cnhsyj.com/news/20093
 *  [hotelren] "DeepSpeed Zero-3 的参数分区与按需访问机制", hotelren.com/news/4329759
 *  [compass] "ZeRO-1/2/3（Zero Redundancy Optimizer 三階段）",
 *            compassingai.com/zh-hant/concept/zero-stages
 */
#ifndef ZERO3_H
#define ZERO3_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* zero3_stream;

typedef enum zero3_status {
    ZERO3_OK = 0,
    ZERO3_EINVAL = 1, /* bad argument: NULL/misaligned pointer, bad range, size, id */
    ZERO3_ESTATE = 2, /* call not allowed in the submodule's current state */
    ZERO3_ECUDA = 3,  /* CUDA runtime error, including an earlier asynchronous fault */
    ZERO3_ENOMEM = 4, /* host allocation failed */
    ZERO3_EIO = 5     /* checkpoint file missing, short, or written for another partition */
} zero3_status;

typedef enum zero3_dtype { ZERO3_BF16 = 0, ZERO3_F32 = 1 } zero3_dtype;

/* Parameter status of a submodule ([hotelren], ZeroParamStatus state machine). */
enum { ZERO3_NOT_AVAILABLE = 0, ZERO3_INFLIGHT = 1, ZERO3_AVAILABLE = 2 };

#define ZERO3_MAX_RANKS 64

typedef struct zero3_plan zero3_plan;

/* AdamW hyper-parameters ([cnhsyj] section 3.1, optimizer block: lr, betas,
 * eps, weight_decay).  Doubles; the library derives the binary32 step
 * scalars from them once per call. */
typedef struct zero3_adamw_hparams {
    double lr, beta1, beta2, eps, weight_decay;
} zero3_adamw_hparams;

typedef struct zero3_plan_info {
    int32_t n_ranks;        /* N_d */
    int32_t n_submodules;   /* max(submodule id) + 1 */
    int64_t n_tensors;
    int64_t n_partitioned;  /* tensors with numel >= threshold */
    int64_t n_persistent;   /* tensors with numel <  threshold */
    int64_t psi_p;          /* partitioned elements */
    int64_t psi_pad;        /* psi_p rounded up to a multiple of N_d */
    int64_t shard_len;      /* S = psi_pad / N_d */
    int64_t psi_s;          /* persistent elements */
    int64_t persistence_threshold;
    int64_t reduce_bucket_size;
    int64_t n_buckets;
} zero3_plan_info;

typedef struct zero3_tensor_info {
    int64_t numel;
    int64_t offset;       /* flat offset (partitioned) or offset in the persistent buffer */
    int32_t persistent;   /* 1 = unpartitioned, resident on every rank */
    int32_t submodule;
    int32_t first_rank;   /* owners of the tensor's first and last element; -1 if persistent or empty */
    int32_t last_rank;
    int64_t n_segments;   /* pieces of the tensor, one per owning rank */
} zero3_tensor_info;

/* The part of a partitioned tensor owned by one rank: elements
 * [tensor_off, tensor_off+len) of the tensor live at [shard_off, shard_off+len)
 * of rank `rank`'s shard. */
typedef struct zero3_segment {
    int32_t rank;
    int32_t reserved;
    int64_t shard_off;
    int64_t tensor_off;
    int64_t len;
} zero3_segment;

/* The unpartitioned (persistent) group: one resident copy of its fp32
 * master/m/v and bf16 parameters (psi_s elements each) plus every rank's
 * local bf16 gradient of it.  `grads` is a host array of n_ranks device
 * pointers. */
typedef struct zero3_persist_state {
    const uint16_t* const* grads;
    float* master;
    float* m;
    float* v;
    uint16_t* param;
} zero3_persist_state;

/* ------------------------------------------------------------------ plan */

/* Flatten, classify, pad and shard a parameter list (host only, no GPU).
 *  - Tensor t is persistent iff numels[t] < persistence_threshold; persistent
 *    tensors stay unpartitioned on every rank ([hotelren], 小参数驻留, default
 *    1e5; [cnhsyj] section 3.2, stage3_param_persistence_threshold).
 *  - The other tensors are concatenated in list order into one flat buffer,
 *    zero-padded to a multiple of N_d and cut into N_d contiguous shards of
 *    S elements; rank r owns flat [r*S, (r+1)*S) ([cnhsyj] section 2.1: GPU0
 *    keeps the first Ψ/Nd parameters, GPU1 the next; [111qqz] section
 *    "ZeRO-3：参数为什么也可以分片": one layer's weights spread over all GPUs).
 *  - Reduce buckets are consecutive ranges of reduce_bucket_size flat
 *    elements ([cnhsyj] sections 3.1 and 3.3, reduce_bucket_size).
 * numels: n_tensors element counts (>= 0).  submodule_of: n_tensors ids >= 0,
 * or NULL for "tensor t is submodule t".  n_ranks in [1, ZERO3_MAX_RANKS];
 * persistence_threshold >= 0; reduce_bucket_size >= 1.
 * On success *out receives a new plan.  EINVAL on bad arguments, ENOMEM. */
zero3_status zero3_partition(const int64_t* numels, const int32_t* submodule_of, int64_t n_tensors,
                             int32_t n_ranks, int64_t persistence_threshold,
                             int64_t reduce_bucket_size, zero3_plan** out);

zero3_status zero3_plan_info_get(const zero3_plan* plan, zero3_plan_info* info);

/* Per-tensor placement.  EINVAL if t is out of range. */
zero3_status zero3_plan_tensor(const zero3_plan* plan, int64_t t, zero3_tensor_info* info);

/* Copies up to `cap` segments of tensor t into out (may be NULL when cap is
 * 0) and the total count into *n. */
zero3_status zero3_plan_segments(const zero3_plan* plan, int64_t t, zero3_segment* out,
                                 int64_t cap, int64_t* n);

/* Flat range [*flat_lo, *flat_hi) of reduce bucket b. */
zero3_status zero3_plan_bucket(const zero3_plan* plan, int64_t b, int64_t* flat_lo,
                               int64_t* flat_hi);

/* Member count and total elements of submodule k (the size of the buffer
 * zero3_fetch_submodule writes). */
zero3_status zero3_plan_submodule(const zero3_plan* plan, int32_t k, int64_t* n_tensors,
                                  int64_t* numel);

/* Frees the plan and its per-submodule events.  NULL is a no-op. */
void zero3_plan_destroy(zero3_plan* plan);

/* ------------------------------------------------------------ training step
 * Addressing shared by the calls below:
 *  - [flat_lo, flat_hi) is a range of the padded flat buffer, 0 <= flat_lo
 *    <= flat_hi <= psi_pad (a bucket, or everything).  Flat index f is
 *    processed by its owner r = f / S at local index i = f - r*S.
 *  - grads[q] (q = 0..N_d-1) is rank q's local bf16 gradient: the gradient
 *    of flat index f is grads[q][f - grads_origin], so a caller may pass
 *    buffers that hold only a bucket (grads_origin = bucket start).
 *    grads_origin <= flat_lo is required.  Padding entries must be zero.
 *  - master[r], m[r], v[r]: rank r's fp32 state shard, S elements, indexed
 *    by local index.  sparam[r]: rank r's bf16 parameter shard, S elements.
 *  - full: the flat bf16 parameter buffer, psi_pad elements.
 *  - t: 1-based step count for the bias correction.
 */

/* Gradient reduce-scatter ([111qqz] section "ZeRO-2：梯度为什么也可以分片",
 * worked example G0=[2,6], G1=[4,10] -> rank 0 [3], rank 1 [8]; [compass]
 * Stage 3 mechanism, ReduceScatter).  For every f in the range:
 *   g = (sum over q = 0..N_d-1 in that order of f32(grads[q][f])) * f32(1/N_d)
 * accumulated in binary32, written to shard_grad[r][i] as ZERO3_F32 (exact
 * value) or ZERO3_BF16 (rounded to nearest even). */
zero3_status zero3_reduce_scatter(const zero3_plan* plan, const uint16_t* const* grads,
                                  int64_t grads_origin, int64_t flat_lo, int64_t flat_hi,
                                  void* const* shard_grad, zero3_dtype out_dtype,
                                  zero3_stream stream);

/* AdamW on each rank's own fp32 slice ([111qqz] section
 * "ZeRO-1：Optimizer States 为什么可以分片": elementwise-independent updates;
 * [compass] Stage 1 mechanism: update the fp32 slice and write it back to the
 * 2-byte parameter slice).  Per element, one binary32 operation at a time,
 * rounded to nearest even, no fused multiply-add:
 *   p = p*decay; m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g);
 *   d = sqrt(v)*inv_sqrt_bc2 + eps; p = p - step_size*(m/d); sparam = bf16(p)
 * with decay = f32(1-lr*wd), step_size = f32(lr/(1-b1^t)),
 * inv_sqrt_bc2 = f32(1/sqrt(1-b2^t)).  g is read from shard_grad[r][i]
 * (grad_dtype).  Does not write `full`. */
zero3_status zero3_adamw_step(const zero3_plan* plan, const zero3_adamw_hparams* hp, int64_t t,
                              const void* const* shard_grad, zero3_dtype grad_dtype,
                              float* const* master, float* const* m, float* const* v,
                              uint16_t* const* sparam, int64_t flat_lo, int64_t flat_hi,
                              zero3_stream stream);

/* Parameter all-gather ([111qqz] section "ZeRO-1": shards [9] and [18]
 * gather to [9, 18]; [compass] Stage 1 mechanism, AllGather):
 * full[r*S + i] = sparam[r][i] for every flat index in the range. */
zero3_status zero3_allgather(const zero3_plan* plan, const uint16_t* const* sparam,
                             uint16_t* full, int64_t flat_lo, int64_t flat_hi,
                             zero3_stream stream);

/* The fused ZeRO-3 step: reduce-scatter, AdamW, bf16 cast into the shard and
 * all-gather into `full`, one pass over the range with the reduced gradient
 * kept in registers ([baike] section 原理, flowchart E -> F -> A).
 * Results equal zero3_reduce_scatter(F32) + zero3_adamw_step(F32) +
 * zero3_allgather bit for bit.  If persist is not NULL the persistent group is
 * also updated (same arithmetic, DDP style, on its single resident copy),
 * whatever the range.  When every rank's persist->grads[q] lies at one common
 * element offset from grads[q] (e.g. each rank's gradient buffer holds the
 * flat gradients followed by the persistent group's, as one buffer of
 * psi_pad + psi_s elements), the group is one more span of the same kernel
 * launch and may have any element alignment; otherwise it is a second
 * launch and its gradient pointers must be 16-byte aligned. */
zero3_status zero3_step(const zero3_plan* plan, const zero3_adamw_hparams* hp, int64_t t,
                        const uint16_t* const* grads, int64_t grads_origin,
                        float* const* master, float* const* m, float* const* v,
                        uint16_t* const* sparam, uint16_t* full,
                        const zero3_persist_state* persist,
                        int64_t flat_lo, int64_t flat_hi, zero3_stream stream);

/* The ZeRO-1 / ZeRO-2 step: parameters are not partitioned and every rank
 * keeps the full 2-byte parameters ([compass] Stage 1 and Stage 2
 * mechanisms; [111qqz] sections "ZeRO-1" and "ZeRO-2").  Same reduce-scatter
 * and AdamW on each rank's fp32 shard as zero3_step, then the updated bf16
 * values are written into EVERY rank's full copy: params[q][f] for all
 * q = 0..N_d-1 and every flat f in the range (the all-gather that restores
 * consistency after the sharded update).  params: host array of N_d device
 * pointers, each psi_pad bf16 elements.  Stages 1 and 2 share this step;
 * they differ in the gradient memory a rank keeps (see zero3_memory_bytes).
 * Per element it moves 2*N_d + 24 + 2*N_d bytes.  Create the plan with
 * persistence threshold 0 (the threshold is a stage-3 setting); persistent
 * tensors, if any, are updated by zero3_persistent_step. */
zero3_status zero3_step_stage12(const zero3_plan* plan, const zero3_adamw_hparams* hp, int64_t t,
                                const uint16_t* const* grads, int64_t grads_origin,
                                float* const* master, float* const* m, float* const* v,
                                uint16_t* const* params, int64_t flat_lo, int64_t flat_hi,
                                zero3_stream stream);

/* ----------------------------------------------------- qwZ (ZeRO++)
 * The parameter all-gather sends int8 or int4 codes instead of bf16 values
 * ([compass] section ZeRO++: qwZ quantizes the weights of the all-gather to
 * int8/int4 to cut the communicated volume).  The pages give no block size
 * or scale format; this library fixes: symmetric integers of `bits` = 8 or 4
 * bits (qmax = 127 or 7), one fp32 scale per ZERO3_QWZ_BLOCK = 256
 * consecutive elements of a rank's shard (local indices [256b, 256b+256); a
 * shard's last block may be shorter),
 *   absmax = max |x|, x = f32(bf16 parameter);  scale = absmax / qmax;
 *   code = round-half-even(x * (qmax / absmax)), 0 when absmax = 0;
 * and the receiver writes bf16_rne(code * scale).  Layout per rank r:
 * codes[r] [ceil(S * bits / 8)] bytes (int8: one byte per element; int4: two
 * per byte, element 2j in the low nibble, two's complement), scales[r] fp32
 * [ceil(S/256)] (host arrays of N_d device pointers, 16-byte aligned).  Any
 * other `bits` is ZERO3_EINVAL.  Quantizing calls need ranges that cover whole
 * blocks of every shard they touch: each rank's local range must start on a
 * multiple of 256 and end on one or at S (else ZERO3_EINVAL). */
#define ZERO3_QWZ_BLOCK 256

/* zero3_step whose all-gather output is the quantized wire format: writes
 * master/m/v and sparam like zero3_step, and codes/scales of the updated
 * shard instead of `full` (the receiving side is zero3_allgather_qwz). */
zero3_status zero3_step_qwz(const zero3_plan* plan, const zero3_adamw_hparams* hp, int64_t t,
                            const uint16_t* const* grads, int64_t grads_origin,
                            float* const* master, float* const* m, float* const* v,
                            uint16_t* const* sparam, int32_t bits, int8_t* const* codes,
                            float* const* scales, const zero3_persist_state* persist,
                            int64_t flat_lo, int64_t flat_hi, zero3_stream stream);

/* Quantizes existing bf16 shards into codes/scales (e.g. at initialisation). */
zero3_status zero3_quantize_shards(const zero3_plan* plan, const uint16_t* const* sparam,
                                   int32_t bits, int8_t* const* codes, float* const* scales,
                                   int64_t flat_lo, int64_t flat_hi, zero3_stream stream);

/* The quantized all-gather: full[r*S + i] = bf16_rne(code_r(i) *
 * scales[r][i / 256]) for every flat index in the range (any range). */
zero3_status zero3_allgather_qwz(const zero3_plan* plan, int32_t bits, const int8_t* const* codes,
                                 const float* const* scales, uint16_t* full, int64_t flat_lo,
                                 int64_t flat_hi, zero3_stream stream);

/* Update of the unpartitioned group alone ([hotelren], 小参数驻留: small
 * parameters stay resident and are not partitioned): the same fixed-order
 * sum times 1/N_d of the ranks' gradients and the same AdamW as above on the
 * one resident copy; param = bf16(master). */
zero3_status zero3_persistent_step(const zero3_plan* plan, const zero3_adamw_hparams* hp,
                                   int64_t t, const zero3_persist_state* persist,
                                   zero3_stream stream);

/* Writes bf16(master) into sparam (and into full when full is not NULL) over
 * the range, and param = bf16(master) for the persistent group when persist
 * is not NULL ([compass] Stage 1 mechanism: fp32 master written back to the
 * 2-byte parameters).  Used at initialisation and after loading states. */
zero3_status zero3_cast_params(const zero3_plan* plan, const float* const* master,
                               uint16_t* const* sparam, uint16_t* full,
                               const zero3_persist_state* persist,
                               int64_t flat_lo, int64_t flat_hi, zero3_stream stream);

/* --------------------------------------------------------- submodule fetch */

/* Gathers submodule k's parameters into `out` before its forward or backward
 * ([baike] section 原理: gather before forward, release the non-local part,
 * gather again for backward; [compass] "ZeRO Stage 3 的 AllGather 與釋放機制").
 * Layout of out: the member tensors in list order, each complete; element
 * tensor_off of a partitioned tensor comes from sparam[owner] (see
 * zero3_plan_segments), persistent tensors from persist_param (psi_s bf16).
 * State machine ([hotelren], ZeroParamStatus): NOT_AVAILABLE -> launch the
 * gather, INFLIGHT, reference count 1; INFLIGHT/AVAILABLE -> reference count
 * + 1 and no new gather (out must equal the first call's out, else
 * ZERO3_ESTATE).  The gather completes in stream order; the status turns
 * AVAILABLE when zero3_submodule_status or zero3_submodule_wait observe it.
 * sparam[r] may be NULL for ranks that own no element of submodule k. */
zero3_status zero3_fetch_submodule(zero3_plan* plan, int32_t k, const uint16_t* const* sparam,
                                   const uint16_t* persist_param, uint16_t* out,
                                   zero3_stream stream);

/* Several fetches in one call, their gathers packed into shared launches
 * ([cnhsyj] section 3.1, allgather_bucket_size: many small gathers are
 * aggregated into a few large ones; [hotelren], minimal ZeRO-3 config,
 * allgather_bucket_size 5e8).  The result equals n calls
 * zero3_fetch_submodule(ks[i], ..., outs[i]) in list order: every submodule
 * keeps its own ZeroParamStatus transitions, reference count and event, and a
 * submodule listed twice, or already fetched, only gains a reference and must
 * name the same output (ZERO3_ESTATE otherwise).  The gathers of the
 * submodules that were NOT_AVAILABLE run as launches of up to 512 pieces
 * (one piece per tensor segment), so a bucket of many small submodules costs
 * a few launches instead of one per submodule.
 * ks: host array of n submodule ids; outs: host array of n device pointers
 * (16-byte aligned, each holding its submodule's elements; outputs of
 * different submodules must not overlap).  Everything is checked before
 * anything is launched or any state changes: EINVAL (bad id, NULL or
 * misaligned pointer, n < 0), ESTATE, ECUDA, ENOMEM. */
zero3_status zero3_fetch_submodules(zero3_plan* plan, const int32_t* ks, int32_t n,
                                    const uint16_t* const* sparam, const uint16_t* persist_param,
                                    uint16_t* const* outs, zero3_stream stream);

/* Drops one reference; at zero the submodule returns to NOT_AVAILABLE (its
 * gathered copy may be reused by the caller).  ZERO3_ESTATE if the submodule
 * is NOT_AVAILABLE. */
zero3_status zero3_release_submodule(zero3_plan* plan, int32_t k);

/* Current status (ZERO3_NOT_AVAILABLE / INFLIGHT / AVAILABLE); an INFLIGHT
 * gather whose work has finished is reported (and recorded) AVAILABLE. */
zero3_status zero3_submodule_status(zero3_plan* plan, int32_t k, int32_t* status);

/* Blocks the host until submodule k's gather has finished; marks AVAILABLE. */
zero3_status zero3_submodule_wait(zero3_plan* plan, int32_t k);

/* ------------------------------------------------- prefetching coordinator
 * Gathers the submodules that come next while the current one computes
 * ([hotelren]: fetch_sub_module starts collecting later layers' parameters
 * before the current layer has finished; [cnhsyj] section 3.2 and
 * [hotelren], tuning list: stage3_prefetch_bucket_size,
 * stage3_max_live_parameters, stage3_max_reuse_distance).
 *  - Gathers run on prefetch_stream into a caller-owned arena (bf16,
 *    16-byte aligned, arena_elems >= the largest submodule rounded up to a
 *    multiple of 8); each gathered copy occupies a whole number of 8-element
 *    units so that it starts 16-byte aligned.  The compute stream waits on a
 *    submodule's ready event before its first use, so a fetch never blocks
 *    the host.  Ranges of the arena are reused only after the compute stream
 *    has passed the release of their previous contents.
 *  - Order: `trace` (n_trace submodule ids) is the fetch order of one step;
 *    with n_trace = 0 the order of the first step is recorded (no prefetch
 *    during it) and used from the next step on.  A fetch that departs from
 *    the order disables prefetching until the next step (counted in
 *    trace_misses) and the new order is adopted.
 *  - Budgets (elements): at most prefetch_bucket_size gathered ahead of use
 *    (0 disables prefetching), at most max_live_parameters gathered at once;
 *    a submodule whose next use comes within max_reuse_distance gathered
 *    elements stays gathered after its release.  When the arena or the live
 *    budget is exhausted, unreferenced copies are dropped, farthest next use
 *    first; ZERO3_ENOMEM when only referenced copies remain.
 *  - Status per submodule follows the ZeroParamStatus machine
 *    (NOT_AVAILABLE, INFLIGHT, AVAILABLE).
 *  - sparam (n_ranks device pointers) and persist_param are read at every
 *    gather; their contents change only through the optimizer step, after
 *    which the caller calls zero3_coordinator_next_step.
 *  - compute_stream and prefetch_stream must differ; the coordinator records
 *    events on both and never synchronises the host.
 *  - Prefetches go out in batches: all submodules that fit the budgets at a
 *    fetch are gathered by one zero3_fetch_submodules-style call (a few
 *    launches of up to 512 pieces), with one wait for the arena ranges they
 *    reuse; the compute stream waits on a ready event only if it has not
 *    already waited on a later one of the prefetch stream. */
typedef struct zero3_coordinator zero3_coordinator;

typedef struct zero3_prefetch_config {
    int64_t prefetch_bucket_size;  /* stage3_prefetch_bucket_size */
    int64_t max_live_parameters;   /* stage3_max_live_parameters */
    int64_t max_reuse_distance;    /* stage3_max_reuse_distance */
} zero3_prefetch_config;

typedef struct zero3_coordinator_stats {
    int64_t steps;           /* zero3_coordinator_next_step calls */
    int64_t gathers;         /* gathers issued (ahead of use or on demand) */
    int64_t prefetched;      /* gathers issued ahead of use */
    int64_t prefetch_hits;   /* fetches served by a gather issued ahead */
    int64_t reuse_hits;      /* fetches served by a copy kept after release */
    int64_t evictions;       /* unreferenced copies dropped for room */
    int64_t trace_misses;    /* fetches that departed from the order */
    int64_t gathered_elems;
    int64_t peak_live_elems;
    int64_t live_elems;
    int64_t gather_calls;    /* batches issued (each gathers one or more submodules) */
    int64_t gather_launches; /* kernel launches of those batches */
    int64_t compute_waits;   /* waits of the compute stream on a ready event */
} zero3_coordinator_stats;

/* EINVAL: NULL plan/cfg/out, negative sizes, equal streams, arena smaller
 * than the largest submodule, max_live below it, a trace id out of range, a
 * NULL or misaligned source shard or arena. */
zero3_status zero3_coordinator_create(zero3_plan* plan, const int32_t* trace, int64_t n_trace,
                                      const uint16_t* const* sparam,
                                      const uint16_t* persist_param, uint16_t* arena,
                                      int64_t arena_elems, const zero3_prefetch_config* cfg,
                                      zero3_stream compute_stream, zero3_stream prefetch_stream,
                                      zero3_coordinator** out);

/* Takes a reference to submodule k's gathered parameters (layout as
 * zero3_fetch_submodule) and issues the next prefetches.  *out points into
 * the arena and is valid for work enqueued on compute_stream until the
 * matching release. */
zero3_status zero3_coordinator_fetch(zero3_coordinator* c, int32_t k, uint16_t** out);

/* Drops a reference (ESTATE if k holds none). */
zero3_status zero3_coordinator_release(zero3_coordinator* c, int32_t k);

zero3_status zero3_coordinator_status(zero3_coordinator* c, int32_t k, int32_t* status);

/* Call after the optimizer step has been enqueued on compute_stream: drops
 * every gathered copy (they predate the update), orders later gathers after
 * the step, adopts the recorded order if needed and prefetches the start of
 * the next step.  ESTATE if a reference is still held. */
zero3_status zero3_coordinator_next_step(zero3_coordinator* c);

zero3_status zero3_coordinator_get_stats(const zero3_coordinator* c,
                                         zero3_coordinator_stats* stats);

/* Frees the coordinator's events; the arena stays the caller's.  Work already
 * enqueued keeps running. */
void zero3_coordinator_destroy(zero3_coordinator* c);

/* ------------------------------------------------------------ checkpoints
 * Each partition is saved and restored by itself ([cnhsyj] section 4.3:
 * save_checkpoint / load_checkpoint write and read every partition), or the
 * weights are gathered into complete 16-bit tensors on save ([hotelren],
 * stage3_gather_16bit_weights_on_model_save; [baike] section 应用).
 * A file is a 48-byte little-endian header
 *   char magic[8] = "ZERO3CKP"; uint32 version = 1; uint32 kind (1 shard,
 *   2 persistent group, 3 16-bit weights, 4 fp32 weights); int32 rank (-1 when
 *   not a shard); int32 n_ranks; int64 element count; int64 step t;
 *   uint64 fingerprint = FNV-1a 64 (offset basis 14695981039346656037,
 *   prime 1099511628211) over the bytes of the int64 values n_ranks,
 *   persistence threshold, tensor count, then every tensor's element count
 * followed by raw little-endian arrays (a shard: fp32 master, m, v of S
 * elements each; the persistent group likewise with psi_s elements).
 * Loading checks every header field against the plan and the arguments, and
 * the file's size against exactly header + arrays, and returns ZERO3_EIO on
 * any mismatch (a short file and one with trailing bytes included); nothing
 * is written to device memory before these checks have passed, so a
 * rejected file leaves the destination buffers as they were.  Saving writes
 * "<path>.tmp.<pid>", flushes it to disk (fsync) and renames it over `path`
 * only when every byte has been written; on any error the temporary file is
 * removed and an existing file at `path` is left unchanged.  Calls are
 * synchronous (they synchronise `stream`); device pointers need no alignment
 * except `full` (16 bytes).  The library stages through a 16 MiB host buffer
 * that it allocates and frees per call. */

/* Writes rank `rank`'s fp32 master, m and v shards (S elements each) and the
 * step count t. */
zero3_status zero3_save_shard(const zero3_plan* plan, int32_t rank, int64_t t, const float* master,
                              const float* m, const float* v, const char* path,
                              zero3_stream stream);

/* Restores a shard written by zero3_save_shard for the same rank and
 * partition; *t receives the saved step count.  After loading every rank,
 * zero3_cast_params rebuilds the bf16 shards and the full buffer. */
zero3_status zero3_load_shard(const zero3_plan* plan, int32_t rank, int64_t* t, float* master,
                              float* m, float* v, const char* path, zero3_stream stream);

/* Same for the persistent group's fp32 master, m and v (psi_s each);
 * persist->grads and persist->param are not used. */
zero3_status zero3_save_persistent(const zero3_plan* plan, int64_t t,
                                   const zero3_persist_state* persist, const char* path,
                                   zero3_stream stream);
zero3_status zero3_load_persistent(const zero3_plan* plan, int64_t* t,
                                   const zero3_persist_state* persist, const char* path,
                                   zero3_stream stream);

/* Consolidated 16-bit weights: every tensor in list order, complete, as bf16
 * (partitioned tensors read from the all-gathered `full` buffer, persistent
 * ones from persist_param).  Element count in the header = psi_p + psi_s. */
zero3_status zero3_save_16bit_weights(const zero3_plan* plan, const uint16_t* full,
                                      const uint16_t* persist_param, const char* path,
                                      zero3_stream stream);

/* Offline merge of partition-wise checkpoints into complete fp32 weights
 * ([baike] section 应用: save the shard weights, then merge them with the
 * accompanying script).  Host only, no GPU: reads the fp32 master array of
 * the N_d shard files (shard_paths[r] written by zero3_save_shard for rank r)
 * and of the persistent file (NULL allowed when psi_s = 0), and writes kind 4
 * with every tensor complete, in list order, as fp32.  All inputs are
 * validated (headers, ranks, partition, equal step counts) before the output
 * is created; ZERO3_EIO otherwise.  Memory use is one 16 MiB buffer. */
zero3_status zero3_merge_shards(const zero3_plan* plan, const char* const* shard_paths,
                                const char* persistent_path, const char* out_path);

/* ------------------------------------------------------------- accounting */

/* Model-state bytes per rank, 2-byte params and grads plus 12 bytes of Adam
 * state per parameter ([baike] section 原理, (2+2+K)Ψ/N_d with K = 12;
 * [compass] section 三階段記憶體公式彙總): stage 0 16Ψ, stage 1 4Ψ+12Ψ/N_d,
 * stage 2 2Ψ+14Ψ/N_d, stage 3 16Ψ/N_d.  EINVAL for other stages or n_d < 1. */
zero3_status zero3_memory_bytes(int32_t stage, double psi, int32_t n_d, double* bytes_per_rank);

/* Model-state bytes one rank holds for this plan: zero3_memory_bytes on the
 * padded partitioned elements (psi_pad) plus the persistent group, which every
 * rank keeps whole at 2 + 2 + 12 bytes per element. */
zero3_status zero3_plan_memory_bytes(const zero3_plan* plan, int32_t stage, double* bytes_per_rank);

/* Elements sent per rank per step by ring collectives ([111qqz] section
 * "为什么 ZeRO-2 的通信量和 DDP 接近", V = (N-1)/N * S; [compass] section
 * 通訊量對比): 2Ψ(N_d-1)/N_d for stages 0-2, 3Ψ(N_d-1)/N_d for stage 3. */
zero3_status zero3_comm_elems(int32_t stage, double psi, int32_t n_d, double* elems_per_rank);

/* ------------------------------------------------------------------ misc */

/* cudaStreamSynchronize(stream); returns ZERO3_ECUDA on any pending fault. */
zero3_status zero3_sync(zero3_stream stream);

/* Static text for a status code. */
const char* zero3_status_string(zero3_status s);

#ifdef __cplusplus
}
#endif

#endif /* ZERO3_H */

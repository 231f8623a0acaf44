/*
 * zero_gb300.h -- C ABI of the GB300 (sm_103a) ZeRO optimizer step.
 *
 * One call performs one data-parallel optimizer step for M emulated ranks whose bf16
 * gradient replicas sit in one GPU's HBM:
 *
 *   (1) reduce-scatter: owner r of every bucket receives the average over ranks of its
 *       slice, summed in fp32 in rank order 0..M-1 from +0 and multiplied by (float)(1/M)
 *       ("CS336 2026 Lecture 8" notes, Slide 8: all-reduce = reduce-scatter + all-gather;
 *       Slide 20 step 2; "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 reduce_scatter_sum);
 *   (2) optional clipping by the global L2 norm of the averaged gradient;
 *   (3) AdamW with bias correction and decoupled weight decay on each owner's shard of
 *       fp32 master / m / v, the 16 bytes/param mixed-precision ledger of Lecture 8
 *       Slide 17 (Slide 20 step 3; "并行训练优化…" 2.2.1 step 3);
 *   (4) all-gather of the updated bf16 parameters into the full, unpadded parameter buffer
 *       (Slide 20 step 4; "并行训练优化…" 1.2.2 all_gather, 2.2.6 for ZeRO-3).
 * ZeRO stages 1, 2 and 3 (Lecture 8 Slides 19-26; "并行训练优化…" 2.2.1-2.2.6) run the same
 * arithmetic and differ only in which buffers persist between steps.
 *
 * Conventions shared by every entry point:
 *  - Return value: ZERO_OK (0) or a negative ZERO_ERR_* code; nothing else crosses the ABI.
 *    zero_strerror() gives the text. No call aborts or throws.
 *  - Memory: the library allocates no device memory. The caller allocates every device
 *    buffer in the sizes zero_plan() reports and keeps it alive while a context uses it;
 *    the context only borrows the pointers. A pointer that a call passes to the kernels
 *    must be device memory of the context's GPU (or managed memory); anything else is
 *    refused with ZERO_ERR_INVALID_ARG before work is enqueued. The context owns host
 *    tables, CUDA events for optional kernel timing, and nothing else.
 *  - Streams: work is enqueued on the caller's stream (a cudaStream_t passed as void*; NULL
 *    is the legacy default stream). Calls return once the work is enqueued; only zero_init,
 *    zero_last_norm(), zero_sync_status(), zero_check_report() and zero_kernel_times() wait
 *    for the stream.
 *  - Device: the context binds to the device that holds its buffers; calls make it current
 *    for their duration and restore the caller's current device.
 *  - Threads: a context must not be used from two threads at once. Different contexts are
 *    independent.
 *
 * Flat layout (all lane counts are elements, not bytes):
 *  Tensors are packed in declared order into buckets; a bucket is filled greedily up to
 *  bucket_bytes of bf16 gradient and never splits a tensor (a larger tensor gets a bucket
 *  of its own; bucket_bytes = 0 means a single bucket). Bucket b with n_b real lanes is
 *  padded to M * S_b lanes, S_b = ceil(n_b / (M * ZERO_ALIGN)) * ZERO_ALIGN, and occupies
 *  padded lanes [off_b, off_b + M * S_b); rank r owns [off_b + r * S_b, off_b + (r+1) * S_b).
 *  (With hybrid sharding, M here and below is the group size K = M / groups.)
 *  Real lanes of bucket b are [off_b, off_b + n_b). npad = sum of M * S_b.
 *  The unpadded index of real lane o of bucket b is o - off_b + (sum of n over earlier
 *  buckets). Padding lanes of gradient buffers are ignored (read as +0); padding lanes of
 *  master / m / v stay exactly 0; padding never reaches the unpadded parameter buffer.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------- */
#define ZERO_OK                 0
#define ZERO_ERR_INVALID_ARG   -1  /* null pointer, out-of-range value, bad enum; a
                                      pointer that the kernels would use which is not
                                      device memory of the context's GPU (or managed
                                      memory): host memory is refused, never dereferenced */
#define ZERO_ERR_MISALIGNED    -2  /* a device pointer is not 16-byte aligned           */
#define ZERO_ERR_SIZE_MISMATCH -3  /* a required buffer is missing for this config       */
#define ZERO_ERR_STAGE         -4  /* stage not 1/2/3, or not the context's stage        */
#define ZERO_ERR_NONFINITE     -5  /* the last clipped step saw a non-finite norm and
                                      left the state untouched                           */
#define ZERO_ERR_CUDA          -6  /* a CUDA runtime call failed; see zero_last_cuda_error */
#define ZERO_ERR_BAD_CONTEXT   -7  /* null, destroyed or unknown context                 */
#define ZERO_ERR_NOT_COMPUTED  -8  /* the requested value was not computed (no clipping)  */
#define ZERO_ERR_TOO_LARGE     -9  /* a count over a fixed limit: buckets for
                                      zero_grad_norm_noalloc (ZERO_NOALLOC_MAX_BUCKETS),
                                      schedule entries (ZERO_MAX_SCHEDULE)                */
#define ZERO_ERR_DEVICE       -10  /* checked build: a kernel rejected an out-of-bounds
                                      index (and skipped the access); see zero_check_report */
#define ZERO_ERR_SCHEDULE     -11  /* scheduled steps: a call that needs the host step count
                                      while a schedule is installed, a scheduled call with
                                      none, or a step past the schedule's last entry        */

#define ZERO_ALIGN       64  /* shard length granule in lanes: 128 B of bf16, 256 B of fp32 */
#define ZERO_MAX_RANKS   64  /* largest rank count M (emulated ranks, or processes)       */
#define ZERO_NOALLOC_MAX_BUCKETS 2048  /* bucket-table rows zero_grad_norm_noalloc can hold  */
#define ZERO_MAX_SCHEDULE 1024  /* entries of one step schedule (zero_set_schedule), kept in
                                   the scratch buffer (40 bytes each)                       */

/* gather modes (zero_config.gather) */
#define ZERO_GATHER_FUSED  0  /* the AdamW epilogue writes each owner's bf16 values straight
                                 into the full parameter buffer (in-place all-gather)      */
#define ZERO_GATHER_SHARDS 1  /* stage 3 only: the epilogue writes the persistent padded bf16
                                 shards; a gather kernel then copies them into the full
                                 buffer (also available on its own: zero_gather)           */

/* averaged-gradient handling when clipping (zero_hyper.ghat_mode) */
#define ZERO_GHAT_AUTO        0  /* MATERIALIZE when M > 4 and a ghat buffer exists, else
                                    RECOMPUTE (fewer bytes in each case)                   */
#define ZERO_GHAT_MATERIALIZE 1  /* pass 1 writes the fp32 averaged gradient; pass 2 reads it:
                                    2M + 34 bytes per lane                                 */
#define ZERO_GHAT_RECOMPUTE   2  /* pass 1 only sums squares; pass 2 re-reads the M bf16
                                    gradients: 4M + 26 bytes per lane, no ghat buffer      */

/* state arrays for zero_get_state */
#define ZERO_STATE_MASTER 0
#define ZERO_STATE_M      1
#define ZERO_STATE_V      2
#define ZERO_STATE_GHAT   3

/* kernels reported by zero_kernel_times, in this order */
#define ZERO_K_RS_NORM      0  /* reduce-scatter + squared-norm partials (+ ghat write)   */
#define ZERO_K_NORM_FINAL   1  /* one CTA: norm, clip scale, non-finite flag              */
#define ZERO_K_ADAMW        2  /* AdamW from the materialized averaged gradient           */
#define ZERO_K_RS_ADAMW     3  /* fused reduce-scatter + AdamW (+ all-gather epilogue)     */
#define ZERO_K_GATHER       4  /* bf16 shards -> full unpadded buffer                     */
#define ZERO_K_INIT         5  /* state initialisation                                    */
#define ZERO_K_STEP_BEGIN   6  /* scheduled steps: one thread, counter and scalars         */
#define ZERO_NUM_KERNELS    7

typedef struct zero_ctx zero_ctx; /* opaque, library-owned */

/* Layout and persistence choices, fixed for the life of a context. */
typedef struct {
    int32_t M;            /* data-parallel ranks, 1..ZERO_MAX_RANKS: emulated on this
                             device, or the job's processes when sharded = 1                */
    int32_t stage;        /* ZeRO stage: 1, 2 or 3                                        */
    int64_t bucket_bytes; /* bf16 gradient bytes per bucket; 0 = one bucket              */
    int32_t gather;       /* ZERO_GATHER_FUSED or ZERO_GATHER_SHARDS (stage 3 only)       */
    int32_t groups;       /* hybrid sharding ("CS231n Lecture 11" 4.4): 0 or 1 = none; G > 1
                             splits the M ranks into G groups of K = M / G. The state is
                             sharded over the K ranks of a group (the layout is planned for K
                             owners) and each group holds a replica of it, of which the
                             device keeps one copy; rank q = grp * K + k. The average sums
                             each group's K gradients in order, then the G group sums in
                             order, then multiplies by (float)(1/M). M % G must be 0.        */
    int32_t sharded;      /* 0: all M ranks are emulated on this device (the default).
                             1: process per rank: this context is rank `rank` of a job of M
                             processes, one per GPU, and holds only that rank's part of the
                             state; see "Process-per-rank mode" below.                      */
    int32_t rank;         /* sharded mode: this process's rank, 0..M-1 (owner of shard `rank`
                             of every bucket); unused otherwise                              */
} zero_config;

/* Hyper-parameters of one step. */
typedef struct {
    double lr;            /* >= 0                                                         */
    double beta1, beta2;  /* in [0, 1)                                                    */
    double eps;           /* > 0                                                          */
    double weight_decay;  /* >= 0, decoupled: p <- p * (1 - lr * weight_decay)           */
    double max_grad_norm; /* > 0 when clip != 0                                           */
    int32_t clip;         /* 1: scale the averaged gradient by max_grad_norm / norm when
                             norm > max_grad_norm; 0: no clipping and no norm             */
    int32_t ghat_mode;    /* ZERO_GHAT_*; only used when clip != 0                         */
} zero_hyper;

/* Sizes reported by zero_plan (elements, and bytes for each caller-allocated buffer). */
typedef struct {
    int64_t npad;               /* padded flat length (lanes)                              */
    int64_t n;                  /* real parameters (sum of numel)                          */
    int64_t n_buckets;
    int64_t shard_len;          /* lanes owned by one rank (sum of S_b)                     */
    int64_t bytes_master;       /* fp32 npad                                               */
    int64_t bytes_m;            /* fp32 npad                                               */
    int64_t bytes_v;            /* fp32 npad                                               */
    int64_t bytes_ghat;         /* fp32 npad: averaged-gradient workspace; optional        */
    int64_t bytes_param_full;   /* bf16 n                                                  */
    int64_t bytes_param_shards; /* bf16 npad with ZERO_GATHER_SHARDS, else 0               */
    int64_t bytes_grad_each;    /* bf16 npad: each of the M gradient buffers               */
    int64_t bytes_scratch;      /* status word, norm partials, bucket table, per-bucket
                                   sums, the step schedule and per-bucket norm partials
                                   (9,728 bytes per bucket)                                 */
} zero_sizes;

/* Device buffers borrowed by a context. All 16-byte aligned (torch allocations are). */
typedef struct {
    void* master;       /* fp32 [npad], owner-sharded flat layout; required                */
    void* m;            /* fp32 [npad]; required                                           */
    void* v;            /* fp32 [npad]; required                                           */
    void* ghat;         /* fp32 [npad]; optional (NULL: clipped steps use RECOMPUTE)       */
    void* param_full;   /* bf16 [n], unpadded tensor-order concatenation; required         */
    void* param_shards; /* bf16 [npad]; required with ZERO_GATHER_SHARDS, else NULL        */
    void* scratch;      /* bytes_scratch; required                                         */
} zero_buffers;

/* Host only, no CUDA call. Computes the layout of n_tensors tensors of numel[i] elements
 * (numel[i] >= 0, at least one > 0) and the buffer sizes. Errors: INVALID_ARG, STAGE. */
int zero_plan(const zero_config* cfg, const int64_t* numel, int64_t n_tensors, zero_sizes* out);

/* Host only. Writes the padded start lane of each tensor (tensor_off[n_tensors]) and, if
 * bucket_table is not NULL, four int64 per bucket: {off_b, n_b, S_b, first tensor}
 * (bucket_table[4 * n_buckets]). A gradient for tensor i goes to lanes
 * [tensor_off[i], tensor_off[i] + numel[i]) of each rank's buffer. */
int zero_plan_layout(const zero_config* cfg, const int64_t* numel, int64_t n_tensors,
                     int64_t* tensor_off, int64_t* bucket_table);

/* Creates a context over the caller's buffers and initialises the state on `stream`:
 * master = master_init scattered into the padded layout (padding 0), m = v = 0, t = 0,
 * param_full = bf16(master_init) (and param_shards = bf16(master) with ZERO_GATHER_SHARDS).
 * master_init: device fp32 [n], unpadded, read during this call's kernels only. Unlike the
 * step calls, zero_init waits for `stream` before returning (its host-side bucket table must
 * outlive the upload). Errors: INVALID_ARG, STAGE, MISALIGNED, SIZE_MISMATCH, CUDA. On error
 * *out is NULL. */
int zero_init(zero_ctx** out, const zero_config* cfg, const int64_t* numel, int64_t n_tensors,
              const zero_buffers* bufs, const void* master_init, void* stream);

/* One optimizer step (steps (1)-(4) above), asynchronous on `stream`.
 * grads: M device pointers, grads[r] = rank r's bf16 gradient [npad] in the padded layout,
 * 16-byte aligned, read-only and borrowed until the stream passes this step.
 * stage must equal the context's stage. Increments the step count t (bias correction uses
 * the new t) even if the device later skips the update for a non-finite norm.
 * Errors: BAD_CONTEXT, INVALID_ARG, STAGE, MISALIGNED, SIZE_MISMATCH, CUDA. */
int zero_step(zero_ctx* ctx, const void* const* grads, int stage, const zero_hyper* hyper,
              void* stream);

/* ZeRO-2 per-bucket streaming ("CS336 2026 Lecture 8" Slide 23; "并行训练优化、MoE扩展与系统瓶颈"
 * 2.2.4: each layer's gradient is reduce-scattered as soon as it is produced and the full
 * gradient is then freed). zero_reduce_bucket reduce-scatters bucket `bucket` into the
 * persistent fp32 averaged-gradient shard (the ghat buffer, required) and keeps the
 * bucket's sum of squares; grads_b[r] points at rank r's slice of that bucket (M * S_b bf16
 * lanes in the padded layout, 16-byte aligned), which the caller may free or reuse once the
 * stream has passed the call. When every bucket has been reduced, zero_apply performs the
 * rest of the step: the global norm from the per-bucket sums (and the clip scale if
 * hyper->clip), AdamW on all owner shards from the averaged gradient, the all-gather; it
 * increments t. All calls of one step must be ordered on one stream (they share the norm
 * partials). Bytes per lane: 2M + 4 in the reductions, 30 in the update.
 * Errors: BAD_CONTEXT, INVALID_ARG (bad bucket, or zero_apply before every bucket was
 * reduced), MISALIGNED, SIZE_MISMATCH (no ghat buffer), STAGE, CUDA. */
int zero_reduce_bucket(zero_ctx* ctx, int64_t bucket, const void* const* grads_b, void* stream);
int zero_apply(zero_ctx* ctx, int stage, const zero_hyper* hyper, void* stream);

/* ZeRO-2 per-bucket step without clipping. Same sources as zero_reduce_bucket: each
 * bucket's gradient is reduce-scattered as soon as it exists and then freed. Nothing global
 * stands between a bucket's reduce-scatter and its owners' update when there is no norm to
 * wait for. So this call does both for bucket `bucket` in one pass: reduce-scatter, AdamW
 * on the owners' shards of that bucket, and the bucket's bf16 parameters (with
 * ZERO_GATHER_SHARDS: the shards, then the bucket's all-gather into param_full). That moves
 * 2M + 26 bytes per lane, with no averaged-gradient round trip and no ghat buffer.
 * grads_b as in zero_reduce_bucket. Every bucket takes step t + 1. The step is complete,
 * and t advances, when each bucket has been stepped once, in any order.
 * hyper->clip must be 0: a clipped step needs every bucket's norm first, which is what
 * zero_reduce_bucket + zero_apply do. A step must use one form. While some but not all
 * buckets have been stepped, zero_step, zero_reduce_bucket and a second call for the same
 * bucket return INVALID_ARG.
 * Errors: BAD_CONTEXT, INVALID_ARG, MISALIGNED, STAGE, SCHEDULE (a schedule is installed),
 * CUDA. */
int zero_step_bucket(zero_ctx* ctx, int64_t bucket, const void* const* grads_b, int stage,
                     const zero_hyper* hyper, void* stream);

/* zero_step with host-resident data: enqueues the copy of each pinned host gradient
 * host_grads[r] (bf16 [npad]) into the device buffer dev_grads[r], the step, and the copy
 * of the full bf16 parameters into the pinned host buffer host_params (bf16 [n]), all on
 * `stream`. Host buffers must stay valid until the stream passes the step. */
int zero_step_host(zero_ctx* ctx, const void* const* host_grads, void* const* dev_grads, int stage,
                   const zero_hyper* hyper, void* host_params, void* stream);

/* zero_step_host with the copies overlapped across steps: the host-to-device copies go on
 * copy_stream (a second stream of the caller), the step's kernels and the copy of the
 * parameters back to host_params on `stream`. The library orders them with its own CUDA
 * events: the kernels wait for this call's copies, and a copy into a set of device gradient
 * buffers (identified by dev_grads[0]; at most 8 distinct sets whose last step is still
 * pending: a set whose step has finished is forgotten when a new one needs the room) waits
 * until the previous step that read that set is done. A caller alternating two device sets lets the copies of step
 * k+1 run while step k computes and returns its parameters; with one set, only the
 * parameter copy overlaps. The host buffers must stay valid, and host_params unread, until
 * `stream` has passed the call. Errors as zero_step_host; INVALID_ARG also when the two
 * streams are the same. */
int zero_step_host_overlapped(zero_ctx* ctx, const void* const* host_grads, void* const* dev_grads,
                              int stage, const zero_hyper* hyper, void* host_params, void* stream,
                              void* copy_stream);

/* ---- Process-per-rank mode (zero_config.sharded = 1) ----------------------------------
 * The same step split across M processes, one per GPU, each holding only its own part
 * ("CS336 2026 Lecture 8" Slides 8 and 20: reduce-scatter the gradients to their owners,
 * each owner updates its shard, all-gather the parameters; "并行训练优化、MoE扩展与系统瓶颈"
 * 1.2.2 reduce_scatter_sum / all_gather and 2.2.1-2.2.6; "并行策略总览：六个维度各切什么、
 * 怎么通信", the per-card volumes of the reduce-scatter and all-gather; "CS231n Lecture 11"
 * 4.3-4.4). Rank r = zero_config.rank owns lanes [off_b + r*S_b, off_b + (r+1)*S_b) of every
 * bucket b of the flat layout above: its "shard", shard_len lanes, the concatenation of these
 * slices in bucket order (local lane base_b + j is global lane off_b + r*S_b + j, base_b the
 * sum of S over earlier buckets). The library's kernels read and write this device's buffers
 * only; the caller moves data between processes with its own collectives (torch.distributed
 * over NCCL, or gloo through host memory), at three points of a step:
 *   (1) the exchange that feeds the reduce-scatter. Gradients travel as bf16 bytes and are
 *       summed at the owner in fp32, rank order 0..M-1 from +0, so the result is the
 *       emulated step's bit for bit (a collective that reduced in bf16, or in another order,
 *       would not be). Per bucket, an all-to-all of the bucket's M slices:
 *         recv[off_b + q*S_b + j] = grad_q[off_b + r*S_b + j],   0 <= q < M, 0 <= j < S_b,
 *       i.e. all_to_all_single(recv[off_b : off_b + M*S_b], grad[off_b : off_b + M*S_b])
 *       with equal splits. recv is bf16 [npad] ("the exchange layout"). With one rank per
 *       group (M = 1, or K = 1 with hybrid sharding) the rank's own gradient is already in
 *       the exchange layout and may be passed wherever recv is asked for; the shard is then
 *       the whole padded layout, lane for lane, so param_full may be the param_shards
 *       buffer itself and (3) is the identity.
 *   (2) with clipping, one fp64 per rank: each rank's sum of squares of its averaged shard
 *       (zero_rank_sumsq), gathered in rank order into a device array of M doubles on every
 *       rank (all_gather). Every rank then forms the same norm in the same order.
 *   (3) the all-gather of the updated bf16 shards: per bucket,
 *         all_gather(param_full[off_b : off_b + M*S_b], param_shards[base_b : base_b + S_b]).
 *       With ZeRO-3 the same call into a transient buffer of M*S_b lanes gives bucket b's
 *       parameters, in tensor order, in its first n_b lanes (the per-module gather).
 * Hybrid sharding (groups = G > 1, M = G*K processes, rank q = grp*K + k owns shard k of a
 * layout planned for K owners, replicated across the G groups): (1) runs inside each group
 * (an all-to-all among its K ranks, source index k' in place of q); zero_rank_partial then
 * sums the K slices in order into an fp32 group partial; the partials of shard k are
 * all-gathered across the G groups in group order (among ranks k, K + k, ...) into
 * parts[G * shard_len]; the step sums them in group order and multiplies by (float)(1/M)
 * -- the all-reduce across groups, in a fixed order. (2) gathers the K sums of one group.
 * Streamed bucket by bucket, each bucket goes through the same steps on its own region:
 * zero_rank_partial_bucket, the cross-group all-gather of that bucket's partials, then
 * zero_rank_step_bucket or zero_rank_reduce_bucket.
 *
 * Buffers in this mode (zero_plan reports these sizes when cfg->sharded = 1):
 *   master, m, v  fp32 [shard_len]: this rank's shard of the state (required)
 *   ghat          fp32 [shard_len]: averaged-gradient workspace (optional, as above)
 *   param_shards  bf16 [shard_len]: this rank's updated bf16 shard, the all-gather's send
 *                 buffer (required; the persistent parameters at stage 3)
 *   param_full    bf16 [npad]: the full parameters in the padded layout, tensor i at lanes
 *                 [tensor_off[i], tensor_off[i] + numel[i]) like the gradients (the
 *                 all-gather's receive buffer; required at stages 1 and 2, may be NULL at
 *                 stage 3, where the caller gathers into its own transient buffers)
 *   scratch       bytes_scratch
 * bytes_grad_each is 2 * npad: this rank's gradient, and the exchange buffer recv.
 * zero_init takes the full unpadded master_init [n] (the same on every rank), initialises
 * this rank's shard, its bf16 shard and all of param_full (padding 0), with no collective.
 * The gather field has no effect: the owner always writes param_shards.
 * Calls of the emulated mode that would touch other ranks' data (zero_step, zero_step_host*,
 * the per-bucket and scheduled forms, zero_gather*) return INVALID_ARG on such a context.
 * zero_get_state copies this rank's shard (its `rank` argument must name the shard this
 * context owns: cfg->rank, or cfg->rank % K with hybrid sharding);
 * zero_save_state writes this rank's real lanes of the unpadded vectors and leaves the other
 * lanes untouched (the ranks' outputs are disjoint; summing zero-filled outputs across
 * ranks, or across one group, gives the whole state); zero_load_state reads the whole
 * unpadded vectors. */

/* Without clipping, the whole update of this rank's shard in one fused pass, one launch over
 * every bucket of the shard: reduce-scatter from the exchanged slices (rank-ordered fp32 sum
 * x (float)(1/M)), AdamW, the bf16 shard into param_shards. With clipping: zero_rank_sumsq
 * first, then the gathered sums, then this call. Increments t.
 *  src        flat mode: bf16 recv [npad] in the exchange layout (read-only, borrowed until
 *             the stream passes the call); hybrid mode: fp32 parts [G * shard_len], the
 *             gathered group partials of this shard, group grp at [grp * shard_len]. May be
 *             NULL when the clipped form is the materialized one (the update then reads the
 *             average from the ghat buffer)
 *  sumsq_all  clipping only (else NULL): device fp64 [P], P = M (flat) or K (hybrid), entry i
 *             = the value zero_rank_sumsq wrote on rank i (of this group); the same on every
 *             rank, so every rank computes the same norm and clip scale
 * The materialized / recomputed choice of the clipped form is the one zero_rank_sumsq made.
 * Errors: BAD_CONTEXT, INVALID_ARG (not a sharded context, missing sumsq_all, clipping
 * without a preceding zero_rank_sumsq), STAGE, MISALIGNED, SIZE_MISMATCH, CUDA. */
int zero_rank_step(zero_ctx* ctx, const void* src, const double* sumsq_all, int stage,
                   const zero_hyper* hyper, void* stream);

/* Per-bucket form of zero_rank_step without clipping: the update of bucket `bucket`'s slice
 * of this rank's shard, from src, of which only the bucket's region is read. Flat mode: src
 * is the exchange buffer (the region is lanes [off_b, off_b + M*S_b)). Hybrid mode: src is
 * the gathered group partials, fp32 [G * shard_len] as for zero_rank_step (the region is
 * lanes [grp * shard_len + base_b, +S_b) of each group grp). So the call may follow that
 * bucket's collectives while later buckets are still in flight: the ZeRO-2 pattern of
 * reducing each bucket as soon as its gradients exist ("CS336 2026 Lecture 8" Slide 23;
 * "并行训练优化、MoE扩展与系统瓶颈" 2.2.4). Every bucket takes step t + 1; the step is
 * complete, and t advances, once every bucket has been stepped, in any order. Until then
 * zero_rank_step, zero_rank_sumsq and a second call for the same bucket return INVALID_ARG.
 * Errors: BAD_CONTEXT, INVALID_ARG (not a sharded context, clipping, bad bucket), STAGE,
 * MISALIGNED, CUDA. */
int zero_rank_step_bucket(zero_ctx* ctx, int64_t bucket, const void* src, int stage,
                          const zero_hyper* hyper, void* stream);

/* Clipping, first pass: averages this rank's shard from src (as in zero_rank_step) and writes
 * the fp64 sum of squares over its real lanes to *sumsq (device, 8-byte aligned). Under
 * ZERO_GHAT_MATERIALIZE (or AUTO choosing it) the fp32 average also goes to the ghat buffer,
 * and zero_rank_step reads it instead of src. hyper->clip must be 1.
 * src NULL (after zero_rank_reduce_bucket of every bucket): *sumsq = the sum of the buckets'
 * sums, and zero_rank_step then updates from the ghat buffer (materialized form).
 * Errors: BAD_CONTEXT, INVALID_ARG (also: src NULL before every bucket was reduced, or src
 * given while some were), MISALIGNED, SIZE_MISMATCH, CUDA. */
int zero_rank_sumsq(zero_ctx* ctx, const void* src, const zero_hyper* hyper, double* sumsq,
                    void* stream);

/* Clipped ZeRO-2 streaming: reduces bucket `bucket`'s slice of this rank's shard from src
 * (as for zero_rank_step_bucket: the exchange buffer, or in hybrid mode the gathered group
 * partials; only the bucket's region is read) as soon as its collectives have landed: the
 * average into the ghat buffer (required) and the bucket's sum of squares kept by the
 * context. Once every bucket is reduced, zero_rank_sumsq(src = NULL) gives the
 * rank's sum for the all-gather of sums, and zero_rank_step(src = NULL, sums) updates the
 * shard from the ghat buffer ("CS336 2026 Lecture 8" Slide 23; "并行训练优化、MoE扩展与系统
 * 瓶颈" 2.2.4: each bucket is reduce-scattered as its gradients appear; clipping needs every
 * bucket's norm before the update). A bucket reduced twice keeps its last reduction.
 * Errors: BAD_CONTEXT, INVALID_ARG, SIZE_MISMATCH (no ghat buffer), MISALIGNED, CUDA. */
int zero_rank_reduce_bucket(zero_ctx* ctx, int64_t bucket, const void* src, void* stream);

/* Hybrid mode only: the group partial of this rank's shard, part[j] = the K exchanged bf16
 * slices of local lane j summed in fp32 in order from +0 (no scaling; padding lanes 0), from
 * recv (bf16 [npad], the exchange layout of this rank's group) into part (fp32 [shard_len]).
 * Errors: BAD_CONTEXT, INVALID_ARG (not a hybrid sharded context), MISALIGNED, CUDA. */
int zero_rank_partial(zero_ctx* ctx, const void* recv, void* part, void* stream);

/* Hybrid mode, per bucket: the group partial of bucket `bucket`'s slice only (local lanes
 * [base_b, base_b + S_b) of part, from the bucket's region of recv), so that a bucket's
 * partial can cross the groups while later buckets are still being exchanged. Arguments and
 * errors as zero_rank_partial; INVALID_ARG also for a bucket outside [0, n_buckets). */
int zero_rank_partial_bucket(zero_ctx* ctx, int64_t bucket, const void* recv, void* part, void* stream);

/* Steps whose scalars live on the device, for capture in a CUDA graph. The pages define no
 * interface for this. It serves training loops that capture whole steps as CUDA graphs and
 * replay them. A captured launch keeps the arguments it was captured with. The per-step
 * scalars of AdamW (lr and the bias corrections of step t, Loshchilov & Hutter's decoupled
 * weight decay with Kingma & Ba's corrections) therefore cannot travel as launch arguments.
 *
 * zero_set_schedule uploads them for the next `count` steps. Entry i serves step t + 1 + i,
 * t being the step count at the call. The host forms them exactly as zero_step does, so a
 * scheduled step is bit-identical to zero_step with the same hyper-parameters.
 *   per_step  host array of `count` zero_hyper, one per step (schedules of lr, betas, eps,
 *             weight_decay or max_grad_norm). `clip` and `ghat_mode` must be equal in all
 *             entries, since they choose the kernels a graph fixes.
 *   count     entries; 0 (per_step NULL) leaves scheduled mode.
 * The entries go to the scratch buffer (at most ZERO_MAX_SCHEDULE; a longer run uploads
 * the next schedule when one ends). The call synchronises `stream` and must not be
 * captured.
 *
 * zero_step_scheduled, zero_apply_scheduled and zero_step_bucket_scheduled are zero_step,
 * zero_apply and zero_step_bucket without hyper-parameters. Their first launch is one thread (ZERO_K_STEP_BEGIN). It advances a
 * step counter kept on the device and copies that step's entry into the status word, which
 * the update kernels read. They enqueue kernel launches only, so they can be captured, and
 * every replay is the next step. A step past the last entry changes no state and leaves
 * the counter where it was. It sets a sticky flag, so later steps skip too, and
 * zero_sync_status returns ZERO_ERR_SCHEDULE. A new schedule clears the flag and continues
 * from the last step that ran.
 *
 * A captured graph borrows the context's buffers like the calls it captured: it must not
 * be replayed after zero_destroy or once those buffers are freed.
 * While a schedule is installed, the device counts the steps. zero_get_step synchronises
 * the device and reads that count. zero_step, zero_apply, zero_step_host*, zero_set_step
 * and zero_load_state return ZERO_ERR_SCHEDULE, as do the scheduled calls when no schedule
 * is installed. Status queries (zero_last_norm, zero_sync_status, zero_check_report)
 * synchronise the whole device, since replays may run on any stream.
 * Errors: BAD_CONTEXT, INVALID_ARG (count < 0, per_step NULL with count > 0, a bad entry,
 * entries with unequal clip or ghat_mode), TOO_LARGE (count > ZERO_MAX_SCHEDULE),
 * SIZE_MISMATCH (materialize without a ghat buffer), STAGE, MISALIGNED, SCHEDULE, CUDA. */
int zero_set_schedule(zero_ctx* ctx, const zero_hyper* per_step, int64_t count, void* stream);
int zero_step_scheduled(zero_ctx* ctx, const void* const* grads, int stage, void* stream);
int zero_apply_scheduled(zero_ctx* ctx, int stage, void* stream);
/* zero_step_bucket with the scalars from the schedule (whose entries must not clip); the
 * first bucket of each step also launches ZERO_K_STEP_BEGIN. */
int zero_step_bucket_scheduled(zero_ctx* ctx, int64_t bucket, const void* const* grads_b, int stage,
                               void* stream);

/* Device pointer of the full bf16 parameters [n] (valid until the next step). */
int zero_params(zero_ctx* ctx, void** full_bf16);

/* Stage 3 with ZERO_GATHER_SHARDS: all-gathers bucket `bucket` (or every bucket when -1)
 * from the persistent bf16 shards into dst (device bf16 [n], unpadded; NULL = param_full).
 * Errors: BAD_CONTEXT, INVALID_ARG (bucket out of range or no shards), CUDA. */
int zero_gather(zero_ctx* ctx, int64_t bucket, void* dst, void* stream);

/* ZeRO-3 per-module gather ("CS336 2026 Lecture 8" Slides 24-26: parameters are gathered
 * just before a module's forward / backward and freed after; "CS231n Lecture 11" 4.3: the
 * next block's weights are prefetched while the current one computes). With
 * ZERO_GATHER_SHARDS, writes bucket `bucket`'s n_b bf16 parameters, in tensor order, to the
 * transient device buffer dst[0 .. n_b) (2-byte aligned), on `stream`; running it on a side
 * stream one bucket ahead is the prefetch. Errors: BAD_CONTEXT, INVALID_ARG, MISALIGNED,
 * CUDA. */
int zero_gather_bucket(zero_ctx* ctx, int64_t bucket, void* dst, void* stream);

/* Bucket `bucket`'s first unpadded parameter index and its parameter count (host only). */
int zero_bucket_info(zero_ctx* ctx, int64_t bucket, int64_t* uoff, int64_t* n);

/* Copies rank `rank`'s shard of state array `which` (ZERO_STATE_*), shard_len fp32 values in
 * bucket order, into the device buffer dst. GHAT needs a ghat buffer and holds the
 * averaged gradient of the last step that materialized it. */
int zero_get_state(zero_ctx* ctx, int which, int rank, void* dst, void* stream);

/* Waits for the last step's stream; returns its global gradient norm and clip scale.
 * Errors: NOT_COMPUTED when the last step did not clip (or no step yet). */
int zero_last_norm(zero_ctx* ctx, double* norm, float* scale);

/* Waits for the last step's stream and returns ZERO_OK, ZERO_ERR_NONFINITE (update
 * skipped), ZERO_ERR_SCHEDULE (a scheduled step found no entry), ZERO_ERR_DEVICE (checked
 * build: a bounds check failed) or ZERO_ERR_CUDA. */
int zero_sync_status(zero_ctx* ctx);

/* Checked builds (compiled with -DZERO_CHECKED; zero_checked_build() returns 1) test every
 * global index of every kernel against its buffer before the access, record the first
 * failure and skip the access instead of trapping, so the context stays usable. This stands
 * in for a memory checker. zero_check_report waits for the last step's stream and returns
 * the first failing check site (0 = none) and the index it rejected; in normal builds the
 * tests are compiled out and the site is always 0. */
int zero_check_report(zero_ctx* ctx, int64_t* site, int64_t* index);
int zero_checked_build(void);

/* Checkpoint form of the optimizer state: the real lanes of fp32 master, m and v as unpadded
 * vectors of n values in tensor order. This form does not depend on the rank count, bucket
 * size or stage, so a state saved by one context loads into another with a different M
 * (resharding, elastic restart; "CS336 2026 Lecture 8" Slide 67 lists checkpointing and
 * elastic restart among the needs at scale).
 * zero_save_state: device fp32 [n] outputs; any of the three may be NULL (not written).
 * zero_load_state: device fp32 [n] inputs, read during this call's kernel; m and v may be
 * NULL (zeros); also rebuilds the bf16 parameters (and shards) from the master and sets the
 * step counter to t. Both are asynchronous on `stream`. Errors: BAD_CONTEXT, INVALID_ARG,
 * CUDA. */
int zero_save_state(zero_ctx* ctx, void* master, void* m, void* v, void* stream);
int zero_load_state(zero_ctx* ctx, const void* master, const void* m, const void* v, int64_t t,
                    void* stream);

/* Step counter (number of steps taken). zero_set_step restores it from a checkpoint. */
int zero_get_step(zero_ctx* ctx, int64_t* t);
int zero_set_step(zero_ctx* ctx, int64_t t);

/* Per-kernel timing with CUDA events on the launching stream (off by default). When on,
 * every launch is bracketed by two events (up to 65,536 launches between two calls of
 * zero_kernel_times; later ones run untimed). zero_kernel_times waits for them and writes the
 * summed milliseconds and launch counts of each ZERO_K_* kernel since the last call (each
 * array ZERO_NUM_KERNELS long; either may be NULL), then resets the sums. */
int zero_set_timing(zero_ctx* ctx, int on);
int zero_kernel_times(zero_ctx* ctx, double* ms, int64_t* launches);

/* Launch configuration of the fused step kernel: CTAs in the grid and threads per CTA as
 * launched (fewer threads with one source, M = 1). */
int zero_launch_shape(zero_ctx* ctx, int* ctas, int* threads);

/* Caps the grid of every streaming kernel at `ctas` CTAs (0 = no cap, the default: as many
 * as the GPU holds). Results do not depend on the grid except the norm's summation order;
 * small and odd grids exist to test the index arithmetic. */
int zero_set_max_ctas(zero_ctx* ctx, int ctas);

/* Launch overlap of the per-bucket kernels: those of zero_step_bucket (the fused
 * reduce-scatter + AdamW of one bucket), of zero_reduce_bucket (one bucket's reduce-scatter
 * and sum of squares) and of zero_gather_bucket / zero_gather (one bucket's all-gather).
 * The pages stream buckets one after another (ZeRO-2 reduce-scatter as gradients appear,
 * "CS336 2026 Lecture 8" Slides 23 and 26; ZeRO-3 per-module gather with prefetch, Slides
 * 24-26); each such launch is short (tens of microseconds), so the ramp-up and tail of every
 * launch cost a visible share. Overlap uses programmatic dependent launch: the kernel is
 * launched with programmatic stream serialization and may start while the kernel before it
 * on the stream is still finishing.
 *  ZERO_OVERLAP_NONE     ordinary launches (the default). Every per-bucket launch then pays
 *                        its ramp-up and tail in full. Measured on GB300: the ZeRO-2 streamed
 *                        GPT-2-small step (9 buckets) 0.860 ms = 89% of the copy peak against
 *                        0.758 ms (101%) with ZERO_OVERLAP_BUCKETS; its clipped reduce-then-
 *                        apply form 1.11 ms (83% on its real bytes) against 0.942 (97%); the
 *                        4B layout's 129 per-bucket gathers 3.80 ms (69%) against 2.39 ms
 *                        (101%) with BUCKETS and four prefetch buffers. Callers that stream
 *                        buckets should choose ZERO_OVERLAP_BUCKETS (after checking its
 *                        condition below) or ZERO_OVERLAP_LAUNCH, which is always safe.
 *  ZERO_OVERLAP_LAUNCH   each per-bucket kernel waits for the preceding kernel to complete,
 *                        its writes visible, before its first memory access; only the
 *                        launch itself overlaps. Correct whatever precedes the call.
 *  ZERO_OVERLAP_BUCKETS  as LAUNCH, except that a per-bucket kernel that directly follows a
 *                        per-bucket kernel of the same kind from this context on the same
 *                        stream does its work at once and waits for its predecessor only
 *                        before it exits: a fused bucket step or a bucket reduction after
 *                        another bucket of the same step (not the first bucket of a step, not
 *                        a bucket reduced a second time), a gather after a gather into a
 *                        disjoint destination. It still completes after its predecessor, so
 *                        stream order holds for whatever is enqueued later. The library
 *                        decides this from its own launches; the caller guarantees the rest:
 *                        the kernel that the caller enqueues on the stream directly before
 *                        such a call must not write what the call reads (gradient slices;
 *                        the parameter shards) nor access what it writes. Work ordered by an
 *                        event wait (cudaStreamWaitEvent) is not affected: that dependency is
 *                        kept whole.
 * zero_step_bucket_scheduled always launches ordinary kernels. Under either overlap mode each
 * bucket reduction keeps its norm partials in a region of the scratch buffer of its own
 * (zero_plan sizes the scratch for it). With overlap, per-kernel event timing
 * (zero_set_timing) brackets launches that may run concurrently; time the whole sequence
 * instead. Errors: BAD_CONTEXT, INVALID_ARG. */
#define ZERO_OVERLAP_NONE    0
#define ZERO_OVERLAP_LAUNCH  1
#define ZERO_OVERLAP_BUCKETS 2
int zero_set_launch_overlap(zero_ctx* ctx, int mode);

/* Releases the context (not the caller's buffers). Waits for nothing. */
int zero_destroy(zero_ctx* ctx);

/* Text of a status code; never NULL. */
const char* zero_strerror(int status);

/* CUDA error code of the last ZERO_ERR_CUDA on this thread (0 if none). */
int zero_last_cuda_error(void);

/* Global L2 norm of the averaged gradient and its clip scale, without any allocation.
 *
 * This entry point has no counterpart in the pages; it exists for callers that cannot
 * allocate device memory -- code running where cudaMalloc is not allowed or not possible
 * (inside an allocator or memory-manager callback, under a host runtime that owns every
 * device allocation and hands out only fixed buffers, or in tools that must not change the
 * process's memory footprint). It computes what a clipped zero_step computes first: the
 * norm over real lanes of the rank-ordered fp32 average of the M bf16 gradients, and
 * scale = max_grad_norm / norm when norm > max_grad_norm, else 1.
 *
 * It takes no context and no scratch buffer: its scratch (status word, per-CTA partial
 * sums, bucket table: 98,560 bytes) is a fixed array inside the library image, which every
 * GPU that loads the library holds until the process exits. It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *  grads         M device pointers, bf16 [npad] each in the padded layout, 16-byte aligned,
 *                all on one device (the device of grads[0] runs the call)
 *  M             1..ZERO_MAX_RANKS
 *  bucket_table  host array, 4 int64 per bucket {off_b, n_b, S_b, unused} as written by
 *                zero_plan_layout; buckets must tile [0, npad) from lane 0
 *  n_buckets     1..ZERO_NOALLOC_MAX_BUCKETS; more returns ZERO_ERR_TOO_LARGE
 *  norm_out      device double (8-byte aligned) on that device, receives the norm
 *  scale_out     device float (4-byte aligned) on that device, receives the clip scale
 *  stream        NULL or a stream of that device
 * A gradient or output that is not device memory of that device, or a stream of another
 * device, returns INVALID_ARG before anything is enqueued.
 * Asynchronous on `stream`. The first call on a device also does that device's set-up
 * (looks up the fixed array's device address and the launch shapes of every M); make that
 * first call before any stream capture. The set-up is kept for the life of the process:
 * after cudaDeviceReset of a device the entry point must not be used on it again. All calls
 * share the one array, which keeps the last call's contents; nothing in it has to start at
 * zero (every value a call reads is written earlier in the same call). Calls whose work
 * overlaps on the GPU -- on different streams, or from different threads -- race on the
 * array and must be serialised by the caller. In the bounds-checked build
 * (zero_checked_build() == 1) the call clears the array's status word first, waits for its
 * stream at the end and returns ZERO_ERR_DEVICE if a bounds check failed.
 * Errors: INVALID_ARG, MISALIGNED, TOO_LARGE, CUDA, DEVICE (checked build). */
int zero_grad_norm_noalloc(const void* const* grads, int M, const int64_t* bucket_table,
                           int64_t n_buckets, double max_grad_norm, double* norm_out,
                           float* scale_out, void* stream);

/* Training-state bytes per parameter held by one rank: param + grad + optimizer bytes, of
 * which ZeRO stage 1 shards the optimizer part over M ranks, stage 2 also the gradient,
 * stage 3 everything ("CS336 2026 Lecture 8" Slides 17-28; stage 0 = plain data parallel).
 * Returns a negative value for invalid arguments. Host only. */
double zero_state_bytes_per_param(int stage, int M, double param_bytes, double grad_bytes,
                                  double optim_bytes);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_GB300_H */

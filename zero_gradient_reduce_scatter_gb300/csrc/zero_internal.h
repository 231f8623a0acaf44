// Internal declarations shared by the host API (zero_api.cpp) and the kernels
// (zero_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "zero_gb300.h"

namespace zg {

// One bucket of the flat layout, as the kernels see it (32 bytes).
//   padded lanes [off, end) with end = off + M * S; real lanes [off, off + n);
//   the real lane o maps to unpadded index o - off + uoff.
struct Bucket {
    int64_t off;
    int64_t n;
    int64_t end;
    int64_t uoff;
};

// Step constants of AdamW, formed on the host in double and rounded once to float.
struct AdamConsts {
    float b1, b2, c1, c2, step, isb, decay, eps;
};

// One entry of a device-resident schedule: the scalars of one step (scheduled steps).
struct ScheduleEntry {
    AdamConsts k;
    double max_norm;  // clip threshold of the step
};

// Device status word at the start of the scratch buffer. Written by the norm-finalise
// kernel (norm, scale, flags) and by the step-begin kernel of scheduled steps (counter and
// this step's scalars); read by the update kernels and, after a synchronisation, by the host.
struct Status {
    double sumsq;   // sum of squared averaged gradient over real lanes
    double norm;    // sqrt(sumsq)
    float scale;    // clip scale applied to the averaged gradient
    int32_t flags;  // kFlagNonfinite | kFlagSchedule | kFlagBounds
    int64_t bad_site;   // checked builds: first failing bounds check (0 = none) ...
    int64_t bad_index;  // ... and the index it rejected
    int64_t t_dev;        // scheduled steps: the step count, advanced on the device
    int64_t sched_base;   // step served by schedule entry 0
    int64_t sched_count;  // entries in the schedule
    AdamConsts cur;       // scheduled steps: the scalars of the running step ...
    double cur_max_norm;  // ... and its clip threshold
    int64_t reserved[3];
};
static_assert(sizeof(Status) == 128, "status word is 128 bytes");

constexpr int32_t kFlagNonfinite = 1;
constexpr int32_t kFlagSchedule = 2;  // a scheduled step found no entry: it and later ones skip (sticky)
constexpr int32_t kFlagBounds = 4;    // checked builds: an index failed its bounds check (sticky)

// Everything a streaming kernel needs; passed by value (kernel parameter space).
struct StepArgs {
    const uint16_t* grads[ZERO_MAX_RANKS];  // M bf16 gradient buffers, padded layout
    float* master;
    float* m;
    float* v;
    float* ghat;          // fp32 averaged gradient (materialized mode) or nullptr
    uint16_t* out;        // param_full (unpadded) or param_shards (padded)
    const Bucket* buckets;
    int64_t nb;
    int64_t nvec;         // npad / 8: work items of 8 lanes (16 B of bf16)
    int64_t vbeg, vend;   // vec range of the norm pass and the fused kernel (the layout, or one bucket)
    int64_t gbase;        // norm pass: lane at which grads[r] starts (0, or the bucket's first lane)
    int64_t gext;         // norm pass: lanes in each gradient buffer; fused kernel: end lane of
                          // the gradients (which it addresses by absolute lane); bounds checks
    int64_t npad;         // padded lanes (bounds checks)
    int64_t n;            // unpadded parameters (bounds checks)
    int32_t M;
    float inv_M;          // (float)(1.0 / M)
    int32_t out_shards;   // 1: `out` is the padded shard buffer; 0: the unpadded full buffer
    int32_t groups;       // hybrid sharding: M ranks in `groups` groups (1 = none)
    AdamConsts k;
    Status* status;
    double* partials;     // one fp64 partial sum of squares per CTA of the norm pass
    int32_t pdl;          // PdlMode of kernels launched with programmatic stream serialization
    int32_t part_cap;     // partial sums `partials` holds (0: kMaxPartials; bounds checks)
    int64_t b_first;      // the launch's lanes lie in buckets [b_first, b_end) (b_end 0: all):
    int64_t b_end;        // its threads search only those for their first bucket
};

// Programmatic dependent launch of the per-bucket kernels (zero_set_launch_overlap).
enum PdlMode : int32_t {
    kPdlNone = 0,       // ordinary launch
    kPdlWaitFirst = 1,  // waits for the preceding kernel before its first memory access
    kPdlWaitLast = 2,   // works at once; waits for the preceding kernel before exiting
    kPdlTriggerWait = 3,  // lets the next kernel launch at once, then waits like kPdlWaitFirst
};

// Launch shapes and load paths of the streaming kernels, chosen by measurement on GB300
// (threads per CTA; CTAs per SM, 0 = as many as fit; how gradients are loaded). Measured
// on the full 4B (M = 4) and 1.3B (M = 8) workloads: the fused reduce-scatter + AdamW
// kernel and the AdamW-from-average kernel run best with 16 warps per SM (one 512-thread
// CTA; 24 warps per SM lost ~8%), the read-only norm pass with 32 warps per SM, and the
// norm pass that also writes the average with as many 256-thread CTAs as fit.
enum LoadPath : int {
    kLoadEvictFirst = 0,  // ld.global.cs: streaming, evict-first in L1 and L2
    kLoadNonCoherent = 1, // ld.global.nc.L1::no_allocate: read-only path, no L1 allocation
    kLoadReadOnly = 2,    // ld.global.nc: read-only (texture) path
};
constexpr int kThreadsRsNormOnly = 1024;   // norm pass, averaged gradient kept in registers
constexpr int kThreadsRsNormWrite = 256;  // norm pass that also writes the averaged gradient
constexpr int kThreadsRsAdamw = 512;
// The one-source fused kernel (M = 1) launches fewer threads into the same one CTA per SM:
// 14 warps per SM ran it at 96-98% of the copy peak against 92-94% with 16, and 12, 10 and
// 24 warps were slower again (A/B runs, each on one GPU); with more sources 14 warps lost.
constexpr int kThreadsRsAdamwOne = 448;
constexpr int rs_adamw_threads(int M) { return M == 1 ? kThreadsRsAdamwOne : kThreadsRsAdamw; }
constexpr int kThreadsAdamw = 512;
constexpr int kThreadsGather = 256;
constexpr int kThreadsInit = 256;
constexpr int kCtasPerSmRsNormOnly = 0;
constexpr int kCtasPerSmRsNormWrite = 0;
constexpr int kCtasPerSmRsAdamw = 0;
constexpr int kCtasPerSmAdamw = 1;
constexpr int kGradLoadRsNorm = kLoadReadOnly;
constexpr int kGradLoadRsAdamw = kLoadReadOnly;
// Cache policies of the fp32 state and averaged-gradient accesses, per kernel.
enum CachePolicy : int {
    kCacheStreaming = 0,  // ld/st.global.cs: evict-first
    kCacheDefault = 1,    // plain ld/st.global
    kCacheAllLevels = 2,  // ld.global.ca (loads only; stores as kCacheDefault)
    kCacheGlobal = 3,     // ld/st.global.cg: L2 only
};
// Chosen by a sweep of all load x store combinations on GB300 (full 4B, 1.3B, ragged and
// GPT-2-small workloads, two runs each on one GPU). The fused kernel: plain loads and stores
// 25.23 ms per 4B step against 25.53 with evict-first ones (ld.ca + st.cg within noise);
// evict-first loads with plain stores lost 10%. AdamW from the average: ld.ca loads and plain
// stores 9.55 ms per 1.3B step against 9.73; the same pair cost the fused kernel 5%, so each
// kernel takes its own. The averaged-gradient store of the norm pass: no policy mattered.
constexpr int kStateLoadRsAdamw = kCacheDefault;
constexpr int kStateStoreRsAdamw = kCacheDefault;
constexpr int kStateLoadAdamw = kCacheAllLevels;
constexpr int kGhatLoadAdamw = kCacheAllLevels;
constexpr int kStateStoreAdamw = kCacheDefault;
constexpr int kGhatStoreRsNorm = kCacheStreaming;
// The gather's 16-byte shard loads and parameter stores: plain ones ran the full-range
// gather of the 4B layout at 6.77-6.78 TB/s against 6.57-6.58 with evict-first ones (.ca /
// .cg pairs 6.76); the per-bucket launches were the same under every pair (4.66-4.69 TB/s).
constexpr int kGatherLoad = kCacheDefault;
constexpr int kGatherStore = kCacheDefault;
constexpr int kThreads = 256;         // CTA size of the single-CTA norm finalise

// Scratch layout (bytes from the scratch base; every part 256-byte aligned).
constexpr int kMaxPartials = 4096;    // largest grid of the norm pass
constexpr int64_t kScratchStatus = 0;
constexpr int64_t kScratchPartials = 256;
constexpr int64_t kScratchBuckets = kScratchPartials + 8 * kMaxPartials;
// One fp64 sum of squares per bucket (per-bucket streaming) follows the bucket table.
inline int64_t scratch_bucket_sums(int64_t n_buckets) { return (kScratchBuckets + 32 * n_buckets + 255) / 256 * 256; }
// The step schedule (scheduled steps, ZERO_MAX_SCHEDULE entries) follows the bucket sums.
inline int64_t scratch_schedule(int64_t n_buckets) {
    return (scratch_bucket_sums(n_buckets) + 8 * n_buckets + 255) / 256 * 256;
}
// Per-bucket norm partials (zero_reduce_bucket with launch overlap: one region of
// kBucketPartials per bucket, so that the reductions of consecutive buckets never share one)
// follow the schedule.
constexpr int kBucketPartials = 1216;  // the largest grid of that norm pass on GB300: 152 SMs x 8 CTAs of 256 threads
inline int64_t scratch_bucket_partials(int64_t n_buckets) {
    return (scratch_schedule(n_buckets) + (int64_t)sizeof(ScheduleEntry) * ZERO_MAX_SCHEDULE + 255) / 256 * 256;
}
inline int64_t scratch_bytes(int64_t n_buckets) {
    return (scratch_bucket_partials(n_buckets) + 8 * (int64_t)kBucketPartials * n_buckets + 255) / 256 * 256;
}

// Kernel variants, used as keys of the per-context launch-shape cache.
enum KernelVariant : int {
    kVarRsNormWrite = 0,  // reduce-scatter + norm partials + write ghat
    kVarRsNormOnly,       // reduce-scatter + norm partials
    kVarAdamw,            // AdamW from ghat
    kVarRsAdamwScaled,    // fused, applies the device clip scale
    kVarRsAdamwPlain,     // fused, no clipping
    kVarGather,
    kVarInit,
    // process-per-rank mode: sources in the exchange layout (X) or fp32 group partials (F);
    // their register use differs from the plain kernels', so their grids are their own
    kVarRsNormWriteX,
    kVarRsNormOnlyX,
    kVarRsAdamwScaledX,
    kVarRsAdamwPlainX,
    kVarRsNormWriteF,
    kVarRsNormOnlyF,
    kVarRsAdamwScaledF,
    kVarRsAdamwPlainF,
    kNumVariants
};

// Records a CUDA error for zero_last_cuda_error() and returns ZERO_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Threads per CTA of a kernel variant, and its CTAs-per-SM cap (0 = occupancy limit).
int variant_threads(int variant);
int variant_ctas_per_sm_cap(int variant);

// Largest number of CTAs of `variant` (for rank count M, hybrid-sharding groups) resident
// on one SM.
cudaError_t variant_blocks_per_sm(int variant, int M, int groups, int* blocks);

// Launchers: `grid` CTAs of variant_threads(variant) threads on `stream`.
// a.pdl != kPdlNone (write_ghat only): launched with programmatic stream serialization.
cudaError_t launch_rs_norm(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s);
// sched: the clip threshold is the running scheduled step's (st->cur_max_norm), not max_norm.
cudaError_t launch_norm_final(Status* st, const double* partials, int nparts, double max_norm,
                              int clip, bool sched, cudaStream_t s);
// One CTA: *out = sum of partials[0 .. nparts) in a fixed order.
cudaError_t launch_sum_partials(const double* partials, int nparts, double* out, cudaStream_t s,
                                int pdl = kPdlNone);
// sched: the AdamW scalars are the running scheduled step's (st->cur), not a.k.
cudaError_t launch_adamw(const StepArgs& a, bool sched, int grid, cudaStream_t s);
// The norm pass and the fused step over fp32 sources: a.M fp32 buffers a.grads[r] (cast),
// summed in order (process-per-rank hybrid sharding, the group partials). Launch shapes as
// the bf16 variants of the generic rank count.
cudaError_t launch_rs_norm_f32src(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s);
cudaError_t launch_rs_adamw_f32src(const StepArgs& a, bool apply_scale, int grid, cudaStream_t s);
// The same over sources in the exchange layout of the process-per-rank mode: a.grads[0] is
// the exchange buffer (gext lanes), a.M sources, a.buckets the rank's own table; one launch
// covers every bucket of the shard.
cudaError_t launch_rs_norm_exchange(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s);
cudaError_t launch_rs_adamw_exchange(const StepArgs& a, bool apply_scale, int grid, cudaStream_t s);
// a.pdl != kPdlNone (plain, unscheduled form only): launched with programmatic stream
// serialization in that mode.
cudaError_t launch_rs_adamw(const StepArgs& a, bool apply_scale, bool sched, int grid, cudaStream_t s);
// Scheduled steps. Install: counter = t, entry 0 serves step t + 1, `count` entries, the
// schedule flag cleared. Begin (one thread, first launch of every scheduled step): advance
// the counter and copy its entry into the status word, or raise kFlagSchedule.
cudaError_t launch_schedule_install(Status* st, int64_t t, int64_t count, cudaStream_t s);
cudaError_t launch_step_begin(Status* st, const ScheduleEntry* table, cudaStream_t s);
// out[d] = bf16 parameter of unpadded index u0 + d, d < count, from the padded shards
// (out needs only 2-byte alignment).
// pdl != kPdlNone: launched with programmatic stream serialization in that mode. The
// indices lie in buckets [b_first, b_end) (b_end 0: all buckets).
cudaError_t launch_gather(const uint16_t* shards, uint16_t* out, const Bucket* buckets, int64_t nb,
                          int64_t npad, int64_t u0, int64_t count, Status* st, int grid, cudaStream_t s,
                          int pdl = kPdlNone, int64_t b_first = 0, int64_t b_end = 0);
// State from unpadded fp32 vectors (m_init / v_init may be null: zeros), plus bf16 copies.
cudaError_t launch_init(const float* master_init, const float* m_init, const float* v_init,
                        float* master, float* m, float* v, uint16_t* full, uint16_t* shards,
                        const Bucket* buckets, int64_t nb, int64_t npad, int64_t n, Status* st, int grid,
                        cudaStream_t s);
// Real lanes of master / m / v into unpadded vectors (any output may be null).
cudaError_t launch_save(const float* master, const float* m, const float* v, float* out_master,
                        float* out_m, float* out_v, const Bucket* buckets, int64_t nb, int64_t npad,
                        int64_t n, Status* st, int grid, cudaStream_t s);

}  // namespace zg

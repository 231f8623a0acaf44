// zero_api.cpp -- host side of the C ABI declared in include/zero_gb300.h: the flat-layout
// planner, argument validation, step orchestration and optional per-kernel event timing.
// All arithmetic of the step runs in the kernels of zero_kernels.cu; this file only forms
// the per-step scalars and launches.
//
// Built with -ffp-contract=off so the step scalars are plain IEEE double operations.

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include <cuda_runtime.h>

#include "zero_gb300.h"
#include "zero_internal.h"

struct zero_ctx {
    zero_config cfg;
    int device;
    int sm_count;
    // layout
    std::vector<int64_t> numel;
    std::vector<int64_t> tensor_off;
    std::vector<zg::Bucket> buckets;  // host copy of the device table
    int64_t npad, n, shard_len;
    // borrowed device buffers
    zero_buffers bufs;
    // pointers passed to later calls that were found to be this GPU's memory (dev_ptr_ok)
    mutable std::unordered_set<uintptr_t> dev_ok;
    zg::Status* status;
    double* partials;
    zg::Bucket* dev_buckets;
    // step state
    int64_t t;
    int last_clip;
    cudaStream_t last_stream;
    int stepped;
    // per-bucket streaming (zero_reduce_bucket / zero_apply)
    double* bucket_sums;          // device: one fp64 sum of squares per bucket
    double* bucket_partials;      // device: kBucketPartials norm partials per bucket (launch overlap)
    std::vector<char> reduced;    // host: buckets reduced since the last zero_apply
    int64_t n_reduced = 0;
    std::vector<char> bucket_done;  // host: buckets updated by zero_step_bucket in this step
    int64_t n_bucket_done = 0;
    // launch shapes, per kernel variant (0 = not computed yet), and an optional cap
    int grid[zg::kNumVariants];
    int max_ctas;
    // timing
    int timing;
    struct TimedLaunch {
        int kernel;
        cudaEvent_t start, stop;
    };
    std::vector<TimedLaunch> events;  // pool; the first `n_timed` are in use
    size_t n_timed;
    // overlapped host steps: per device gradient set, "its last step has read it"
    struct GradSet {
        const void* key;        // dev_grads[0] of the set
        cudaEvent_t consumed;
        bool recorded;
    };
    std::vector<GradSet> grad_sets;
    cudaEvent_t h2d_done = nullptr;
    // scheduled steps (zero_set_schedule): the table of per-step scalars (in the scratch
    // buffer); while active, the step count lives in the device status word
    zg::ScheduleEntry* dev_sched = nullptr;
    bool sched_active = false;
    int sched_clip = 0;
    int sched_mode = ZERO_GHAT_RECOMPUTE;
    // launch overlap (zero_set_launch_overlap): the library's kernel launches are counted;
    // after a per-bucket launch that a successor may overlap, its count, stream, kind
    // (ZERO_K_RS_ADAMW or ZERO_K_GATHER) and, for a gather, the destination bytes
    int overlap = ZERO_OVERLAP_NONE;
    uint64_t seq = 0;
    uint64_t chain_seq = ~0ull;
    cudaStream_t chain_stream = nullptr;
    int chain_kind = -1;
    uintptr_t chain_lo = 0, chain_hi = 0;
    // process-per-rank mode (cfg.sharded): this rank owns shard `owner` of every bucket; its
    // shard is a layout of its own (`local`: per bucket {base_b, real lanes of the slice,
    // base_b + S_b, unpadded index of the slice's first lane}, on the device at dev_local);
    // npad / buckets / dev_buckets stay the global layout
    int owner = 0;
    std::vector<zg::Bucket> local;
    zg::Bucket* dev_local = nullptr;
    bool rank_reduced = false;          // zero_rank_sumsq ran and zero_rank_step has not
    int rank_mode = ZERO_GHAT_RECOMPUTE;  // the clipped form zero_rank_sumsq chose
};

namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

int zg::record_cuda_error(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return ZERO_ERR_CUDA;
}

namespace {

std::mutex g_live_mu;
std::unordered_set<const zero_ctx*> g_live;  // contexts not yet destroyed

int cuda_fail(cudaError_t e) { return zg::record_cuda_error(e); }

bool live(const zero_ctx* c) {
    std::lock_guard<std::mutex> lk(g_live_mu);
    return c && g_live.count(c);
}

// Makes `dev` current for the lifetime of the guard and restores the caller's device.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------------------
// Planner. Tensors in declared order; a new bucket opens before a non-empty tensor that
// would push a non-empty bucket past bucket_bytes of bf16 gradient; each bucket is padded
// to a multiple of M * ZERO_ALIGN lanes.
// ---------------------------------------------------------------------------------------
struct Layout {
    std::vector<int64_t> tensor_off;
    std::vector<int64_t> first_tensor;
    std::vector<zg::Bucket> buckets;
    int64_t npad = 0, n = 0, shard_len = 0;
};

// Ranks that share one copy of the sharded state: K = M without hybrid sharding, M / groups with.
int shard_count(const zero_config* cfg) { return cfg->groups > 1 ? cfg->M / cfg->groups : cfg->M; }

int check_config(const zero_config* cfg) {
    if (!cfg) return ZERO_ERR_INVALID_ARG;
    if (cfg->stage < 1 || cfg->stage > 3) return ZERO_ERR_STAGE;
    if (cfg->M < 1 || cfg->M > ZERO_MAX_RANKS) return ZERO_ERR_INVALID_ARG;
    if (cfg->bucket_bytes < 0 || cfg->groups < 0) return ZERO_ERR_INVALID_ARG;
    if (cfg->groups > 1 && cfg->M % cfg->groups != 0) return ZERO_ERR_INVALID_ARG;
    if (cfg->sharded != 0 && cfg->sharded != 1) return ZERO_ERR_INVALID_ARG;
    if (cfg->sharded && (cfg->rank < 0 || cfg->rank >= cfg->M)) return ZERO_ERR_INVALID_ARG;
    if (cfg->gather != ZERO_GATHER_FUSED && cfg->gather != ZERO_GATHER_SHARDS) return ZERO_ERR_INVALID_ARG;
    if (cfg->sharded) return ZERO_OK;  // the gather mode has no effect in process-per-rank mode
    if (cfg->gather == ZERO_GATHER_SHARDS && cfg->stage != 3) return ZERO_ERR_STAGE;
    return ZERO_OK;
}

int make_layout(const zero_config* cfg, const int64_t* numel, int64_t n_tensors, Layout* L) {
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!numel || n_tensors <= 0) return ZERO_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (numel[i] < 0 || numel[i] > (int64_t(1) << 40)) return ZERO_ERR_INVALID_ARG;
        total += numel[i];
    }
    if (total <= 0 || total > (int64_t(1) << 42)) return ZERO_ERR_INVALID_ARG;

    const int64_t M = shard_count(cfg), cap = cfg->bucket_bytes;  // owners per copy of the state
    L->tensor_off.assign((size_t)n_tensors, 0);
    std::vector<int64_t> bucket_real;  // real lanes per bucket
    int64_t open_bytes = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        const int64_t bytes = 2 * numel[i];
        const bool fresh = bucket_real.empty() ||
                           (cap > 0 && bytes > 0 && open_bytes > 0 && open_bytes + bytes > cap);
        if (fresh) {
            L->first_tensor.push_back(i);
            bucket_real.push_back(0);
            open_bytes = 0;
        }
        L->tensor_off[(size_t)i] = bucket_real.back();  // relative; made absolute below
        bucket_real.back() += numel[i];
        open_bytes += bytes;
    }
    const int64_t granule = M * ZERO_ALIGN;
    int64_t off = 0, uoff = 0, shard = 0;
    for (size_t b = 0; b < bucket_real.size(); ++b) {
        const int64_t nb = bucket_real[b];
        const int64_t S = (nb + granule - 1) / granule * ZERO_ALIGN;
        L->buckets.push_back(zg::Bucket{off, nb, off + M * S, uoff});
        off += M * S;
        uoff += nb;
        shard += S;
    }
    for (size_t b = 0; b < bucket_real.size(); ++b) {
        const int64_t last = (b + 1 < bucket_real.size()) ? L->first_tensor[b + 1] : n_tensors;
        for (int64_t i = L->first_tensor[b]; i < last; ++i) L->tensor_off[(size_t)i] += L->buckets[b].off;
    }
    L->npad = off;
    L->n = uoff;
    L->shard_len = shard;
    return ZERO_OK;
}

// Process-per-rank mode: the rank's own bucket table follows the regular scratch parts.
int64_t local_table_offset(int64_t n_buckets) { return zg::scratch_bytes(n_buckets); }

int64_t scratch_size(const zero_config* cfg, int64_t n_buckets) {
    const int64_t base = zg::scratch_bytes(n_buckets);
    return cfg->sharded ? base + (32 * n_buckets + 255) / 256 * 256 : base;
}

void fill_sizes(const zero_config* cfg, const Layout& L, zero_sizes* s) {
    s->npad = L.npad;
    s->n = L.n;
    s->n_buckets = (int64_t)L.buckets.size();
    s->shard_len = L.shard_len;
    s->bytes_grad_each = 2 * L.npad;
    s->bytes_scratch = scratch_size(cfg, (int64_t)L.buckets.size());
    if (cfg->sharded) {  // one rank's shard of the state; the full parameters padded
        s->bytes_master = s->bytes_m = s->bytes_v = 4 * L.shard_len;
        s->bytes_ghat = 4 * L.shard_len;
        s->bytes_param_full = 2 * L.npad;
        s->bytes_param_shards = 2 * L.shard_len;
        return;
    }
    s->bytes_master = s->bytes_m = s->bytes_v = 4 * L.npad;
    s->bytes_ghat = 4 * L.npad;
    s->bytes_param_full = 2 * L.n;
    s->bytes_param_shards = (cfg->gather == ZERO_GATHER_SHARDS) ? 2 * L.npad : 0;
}

// Process-per-rank mode: owner k's slice of every bucket as a layout of its own. Slice b
// starts at local lane base_b (its position in the shard), holds S_b lanes of which the
// first min(max(n_b - k * S_b, 0), S_b) are real, and its lane j is unpadded index
// uoff_b + k * S_b + j (clamped to the bucket's end for a slice of padding only).
std::vector<zg::Bucket> local_table(const std::vector<zg::Bucket>& global, int K, int k) {
    std::vector<zg::Bucket> out;
    int64_t base = 0;
    for (const zg::Bucket& e : global) {
        const int64_t S = (e.end - e.off) / K;
        const int64_t first = std::min((int64_t)k * S, e.n);
        const int64_t real = std::min(std::max(e.n - (int64_t)k * S, (int64_t)0), S);
        out.push_back(zg::Bucket{base, real, base + S, e.uoff + first});
        base += S;
    }
    return out;
}

// ---------------------------------------------------------------------------------------
// Per-step scalars of AdamW (double, rounded once to float).
// ---------------------------------------------------------------------------------------
zg::AdamConsts adam_consts(const zero_hyper* h, int64_t t) {
    const double bc1 = 1.0 - std::pow(h->beta1, (double)t);
    const double bc2 = 1.0 - std::pow(h->beta2, (double)t);
    zg::AdamConsts k;
    k.b1 = (float)h->beta1;
    k.b2 = (float)h->beta2;
    k.c1 = (float)(1.0 - h->beta1);
    k.c2 = (float)(1.0 - h->beta2);
    k.step = (float)(h->lr / bc1);
    k.isb = (float)(1.0 / std::sqrt(bc2));
    k.decay = (float)(1.0 - h->lr * h->weight_decay);
    k.eps = (float)h->eps;
    return k;
}

int check_hyper(const zero_hyper* h) {
    if (!h) return ZERO_ERR_INVALID_ARG;
    if (!(std::isfinite(h->lr) && h->lr >= 0.0)) return ZERO_ERR_INVALID_ARG;
    if (!(h->beta1 >= 0.0 && h->beta1 < 1.0 && h->beta2 >= 0.0 && h->beta2 < 1.0)) return ZERO_ERR_INVALID_ARG;
    if (!(std::isfinite(h->eps) && h->eps > 0.0)) return ZERO_ERR_INVALID_ARG;
    if (!(std::isfinite(h->weight_decay) && h->weight_decay >= 0.0)) return ZERO_ERR_INVALID_ARG;
    if (h->clip != 0 && h->clip != 1) return ZERO_ERR_INVALID_ARG;
    if (h->clip && !(std::isfinite(h->max_grad_norm) && h->max_grad_norm > 0.0)) return ZERO_ERR_INVALID_ARG;
    if (h->ghat_mode < ZERO_GHAT_AUTO || h->ghat_mode > ZERO_GHAT_RECOMPUTE) return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

// Grid of a streaming kernel: every SM filled with as many CTAs as fit, no more CTAs than
// work items, at most kMaxPartials (the norm pass writes one partial per CTA).
int grid_for(zero_ctx* c, int variant, int64_t work_items) {
    if (c->grid[variant] == 0) {
        int per_sm = 0;
        // the exchange-layout kernels of a hybrid context read the K slices of its group
        const bool group_sources = c->cfg.groups > 1 && variant >= zg::kVarRsNormWriteX && variant <= zg::kVarRsAdamwPlainX;
        const int m = group_sources ? shard_count(&c->cfg) : c->cfg.M;
        if (zg::variant_blocks_per_sm(variant, m, c->cfg.groups > 1 ? c->cfg.groups : 1, &per_sm) !=
                cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        int g = per_sm * c->sm_count;
        if (g > zg::kMaxPartials) g = zg::kMaxPartials;
        c->grid[variant] = g;
    }
    const int threads = zg::variant_threads(variant);
    int64_t need = (work_items + threads - 1) / threads;
    if (need < 1) need = 1;
    int g = c->grid[variant];
    if (c->max_ctas > 0 && c->max_ctas < g) g = c->max_ctas;
    return (int)(need < g ? need : g);
}

// Event timing around one launch. At most kMaxTimedLaunches launches are recorded between two
// zero_kernel_times calls; later launches run untimed.
constexpr size_t kMaxTimedLaunches = 1 << 16;

struct Timed {
    zero_ctx* c;
    cudaStream_t s;
    size_t slot = SIZE_MAX;  // index into c->events (an index stays valid if the pool grows)
    Timed(zero_ctx* ctx, int kernel, cudaStream_t stream) : c(ctx), s(stream) {
        ++c->seq;  // every kernel launch of the library passes through here
        if (!c->timing || c->n_timed >= kMaxTimedLaunches) return;
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;  // a graph replays no host timing
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return;
        if (c->n_timed == c->events.size()) {
            zero_ctx::TimedLaunch tl{kernel, nullptr, nullptr};
            if (cudaEventCreate(&tl.start) != cudaSuccess) return;
            if (cudaEventCreate(&tl.stop) != cudaSuccess) {
                cudaEventDestroy(tl.start);
                return;
            }
            c->events.push_back(tl);
        }
        slot = c->n_timed++;
        c->events[slot].kernel = kernel;
        cudaEventRecord(c->events[slot].start, s);
    }
    ~Timed() {
        if (slot != SIZE_MAX) cudaEventRecord(c->events[slot].stop, s);
    }
};

zg::StepArgs base_args(zero_ctx* c) {
    zg::StepArgs a;
    std::memset(&a, 0, sizeof a);
    a.master = (float*)c->bufs.master;
    a.m = (float*)c->bufs.m;
    a.v = (float*)c->bufs.v;
    a.ghat = (float*)c->bufs.ghat;
    const bool shards = c->cfg.gather == ZERO_GATHER_SHARDS;
    a.out = (uint16_t*)(shards ? c->bufs.param_shards : c->bufs.param_full);
    a.out_shards = shards ? 1 : 0;
    a.buckets = c->dev_buckets;
    a.nb = (int64_t)c->buckets.size();
    a.nvec = c->npad / 8;
    a.vbeg = 0;
    a.vend = a.nvec;
    a.gbase = 0;
    a.gext = c->npad;
    a.npad = c->npad;
    a.n = c->n;
    a.M = c->cfg.M;
    a.inv_M = (float)(1.0 / (double)c->cfg.M);
    a.groups = c->cfg.groups > 1 ? c->cfg.groups : 1;
    a.status = c->status;
    a.partials = c->partials;
    return a;
}

// Programmatic-launch mode of a per-bucket kernel of `kind` about to be launched on s.
// It may overlap its predecessor (wait last) only under ZERO_OVERLAP_BUCKETS, when the
// caller allows it for this launch and the library's previous kernel launch was a
// per-bucket launch of the same kind on the same stream, with nothing launched since.
int pdl_mode(const zero_ctx* c, int kind, cudaStream_t s, bool may_overlap) {
    if (c->overlap == ZERO_OVERLAP_NONE) return zg::kPdlNone;
    if (c->overlap == ZERO_OVERLAP_BUCKETS && may_overlap && c->chain_seq == c->seq && c->chain_stream == s &&
        c->chain_kind == kind)
        return zg::kPdlWaitLast;
    return zg::kPdlWaitFirst;
}

// After a per-bucket launch: a successor of the same kind may overlap it.
void note_chain(zero_ctx* c, int kind, cudaStream_t s, uintptr_t lo = 0, uintptr_t hi = 0) {
    c->chain_seq = c->seq;
    c->chain_stream = s;
    c->chain_kind = kind;
    c->chain_lo = lo;
    c->chain_hi = hi;
}

// out[0 .. count) = parameters of unpadded indices [u0, u0 + count). may_overlap: the
// launch may overlap a directly preceding gather into a disjoint destination.
// b_first / b_end: the buckets the indices lie in (b_end 0: any).
int gather_range(zero_ctx* c, int64_t u0, int64_t count, uint16_t* out, cudaStream_t s, bool may_overlap = false,
                 int64_t b_first = 0, int64_t b_end = 0) {
    const int grid = grid_for(c, zg::kVarGather, count / 8 + 2);
    const uintptr_t lo = reinterpret_cast<uintptr_t>(out), hi = lo + 2 * (uintptr_t)(count > 0 ? count : 0);
    const bool disjoint = hi <= c->chain_lo || lo >= c->chain_hi;
    const int pdl = pdl_mode(c, ZERO_K_GATHER, s, may_overlap && disjoint);
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_GATHER, s);
        e = zg::launch_gather((const uint16_t*)c->bufs.param_shards, out, c->dev_buckets, (int64_t)c->buckets.size(),
                              c->npad, u0, count, c->status, grid, s, pdl, b_first, b_end);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (count > 0 && pdl != zg::kPdlNone) note_chain(c, ZERO_K_GATHER, s, lo, hi);
    return ZERO_OK;
}

// State from unpadded fp32 vectors (m_init / v_init may be null: zeros) and the bf16
// parameters: init and checkpoint load. Emulated mode: one kernel over the whole layout.
// Process-per-rank mode: one over this rank's shard (state and bf16 shard), then one over the
// global layout that writes only the padded full parameters (padding 0), if there are any.
cudaError_t launch_state_in(zero_ctx* c, const float* master, const float* m, const float* v, cudaStream_t s) {
    const int64_t nb = (int64_t)c->buckets.size();
    if (!c->cfg.sharded) {
        const int grid = grid_for(c, zg::kVarInit, c->npad);
        Timed tm(c, ZERO_K_INIT, s);
        return zg::launch_init(master, m, v, (float*)c->bufs.master, (float*)c->bufs.m, (float*)c->bufs.v,
                               (uint16_t*)c->bufs.param_full, (uint16_t*)c->bufs.param_shards, c->dev_buckets, nb,
                               c->npad, c->n, c->status, grid, s);
    }
    cudaError_t e;
    {
        const int grid = grid_for(c, zg::kVarInit, c->shard_len);
        Timed tm(c, ZERO_K_INIT, s);
        e = zg::launch_init(master, m, v, (float*)c->bufs.master, (float*)c->bufs.m, (float*)c->bufs.v, nullptr,
                            (uint16_t*)c->bufs.param_shards, c->dev_local, nb, c->shard_len, c->n, c->status, grid, s);
    }
    if (e == cudaSuccess && c->bufs.param_full) {
        const int grid = grid_for(c, zg::kVarInit, c->npad);
        Timed tm(c, ZERO_K_INIT, s);
        e = zg::launch_init(master, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                            (uint16_t*)c->bufs.param_full, c->dev_buckets, nb, c->npad, c->n, c->status, grid, s);
    }
    return e;
}

}  // namespace

extern "C" {

int zero_plan(const zero_config* cfg, const int64_t* numel, int64_t n_tensors, zero_sizes* out) {
    if (!out) return ZERO_ERR_INVALID_ARG;
    Layout L;
    int rc = make_layout(cfg, numel, n_tensors, &L);
    if (rc) return rc;
    fill_sizes(cfg, L, out);
    return ZERO_OK;
}

int zero_plan_layout(const zero_config* cfg, const int64_t* numel, int64_t n_tensors, int64_t* tensor_off,
                     int64_t* bucket_table) {
    if (!tensor_off) return ZERO_ERR_INVALID_ARG;
    Layout L;
    int rc = make_layout(cfg, numel, n_tensors, &L);
    if (rc) return rc;
    std::memcpy(tensor_off, L.tensor_off.data(), sizeof(int64_t) * (size_t)n_tensors);
    if (bucket_table) {
        for (size_t b = 0; b < L.buckets.size(); ++b) {
            const zg::Bucket& e = L.buckets[b];
            bucket_table[4 * b + 0] = e.off;
            bucket_table[4 * b + 1] = e.n;
            bucket_table[4 * b + 2] = (e.end - e.off) / shard_count(cfg);
            bucket_table[4 * b + 3] = L.first_tensor[b];
        }
    }
    return ZERO_OK;
}

int zero_init(zero_ctx** out, const zero_config* cfg, const int64_t* numel, int64_t n_tensors,
              const zero_buffers* bufs, const void* master_init, void* stream) {
    if (!out) return ZERO_ERR_INVALID_ARG;
    *out = nullptr;
    Layout L;
    int rc = make_layout(cfg, numel, n_tensors, &L);
    if (rc) return rc;
    if (!bufs || !master_init) return ZERO_ERR_INVALID_ARG;
    if (!bufs->master || !bufs->m || !bufs->v || !bufs->scratch) return ZERO_ERR_SIZE_MISMATCH;
    if (cfg->sharded) {
        // the rank's bf16 shard always; the full parameters unless ZeRO-3 gathers on demand
        if (!bufs->param_shards || (cfg->stage < 3 && !bufs->param_full)) return ZERO_ERR_SIZE_MISMATCH;
    } else {
        if (!bufs->param_full) return ZERO_ERR_SIZE_MISMATCH;
        if (cfg->gather == ZERO_GATHER_SHARDS && !bufs->param_shards) return ZERO_ERR_SIZE_MISMATCH;
    }
    const void* must_align[] = {bufs->master, bufs->m, bufs->v, bufs->ghat, bufs->param_full, bufs->param_shards,
                                bufs->scratch, master_init};
    for (const void* p : must_align)
        if (p && !aligned16(p)) return ZERO_ERR_MISALIGNED;

    // The device that holds the buffers.
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, bufs->master);
    if (e != cudaSuccess) return cuda_fail(e);
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return ZERO_ERR_INVALID_ARG;
    const int dev = attr.device;
    DeviceGuard guard(dev);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);

    zero_ctx* c = new (std::nothrow) zero_ctx();
    if (!c) return ZERO_ERR_INVALID_ARG;
    c->cfg = *cfg;
    c->device = dev;
    c->sm_count = sms;
    c->numel.assign(numel, numel + n_tensors);
    c->tensor_off = L.tensor_off;
    c->buckets = L.buckets;
    c->npad = L.npad;
    c->n = L.n;
    c->shard_len = L.shard_len;
    c->bufs = *bufs;
    if (cfg->gather != ZERO_GATHER_SHARDS && !cfg->sharded) c->bufs.param_shards = nullptr;
    char* scratch = (char*)bufs->scratch;
    if (cfg->sharded) {
        const int K = shard_count(cfg);
        c->owner = cfg->rank % K;
        c->local = local_table(L.buckets, K, c->owner);
        c->dev_local = (zg::Bucket*)(scratch + local_table_offset((int64_t)L.buckets.size()));
    }
    c->status = (zg::Status*)(scratch + zg::kScratchStatus);
    c->partials = (double*)(scratch + zg::kScratchPartials);
    c->dev_buckets = (zg::Bucket*)(scratch + zg::kScratchBuckets);
    c->bucket_sums = (double*)(scratch + zg::scratch_bucket_sums((int64_t)L.buckets.size()));
    c->dev_sched = (zg::ScheduleEntry*)(scratch + zg::scratch_schedule((int64_t)L.buckets.size()));
    c->bucket_partials = (double*)(scratch + zg::scratch_bucket_partials((int64_t)L.buckets.size()));
    c->reduced.assign(L.buckets.size(), 0);
    c->bucket_done.assign(L.buckets.size(), 0);
    c->t = 0;
    c->last_clip = 0;
    c->last_stream = (cudaStream_t)stream;
    c->stepped = 0;
    std::memset(c->grid, 0, sizeof c->grid);
    c->max_ctas = 0;
    c->timing = 0;
    c->n_timed = 0;

    cudaStream_t s = (cudaStream_t)stream;
    zg::Status zero_status;
    std::memset(&zero_status, 0, sizeof zero_status);
    zero_status.scale = 1.0f;
    // Pageable-source copies: the runtime stages the host data before returning.
    e = cudaMemcpyAsync(c->status, &zero_status, sizeof zero_status, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(c->dev_buckets, c->buckets.data(), sizeof(zg::Bucket) * c->buckets.size(),
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && cfg->sharded)
        e = cudaMemcpyAsync(c->dev_local, c->local.data(), sizeof(zg::Bucket) * c->local.size(),
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_state_in(c, (const float*)master_init, nullptr, nullptr, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // host tables above must outlive the copies
    if (e != cudaSuccess) {
        delete c;
        return cuda_fail(e);
    }
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        g_live.insert(c);
    }
    *out = c;
    return ZERO_OK;
}

// Which clipped form a step takes (ZERO_GHAT_MATERIALIZE or ZERO_GHAT_RECOMPUTE).
static int resolve_ghat_mode(const zero_ctx* c, const zero_hyper* h, int* mode) {
    *mode = ZERO_GHAT_RECOMPUTE;
    if (!h->clip) return ZERO_OK;
    int m = h->ghat_mode;
    if (m == ZERO_GHAT_AUTO) m = (c->cfg.M > 4 && c->bufs.ghat) ? ZERO_GHAT_MATERIALIZE : ZERO_GHAT_RECOMPUTE;
    if (m == ZERO_GHAT_MATERIALIZE && !c->bufs.ghat) return ZERO_ERR_SIZE_MISMATCH;
    *mode = m;
    return ZERO_OK;
}

// A pointer that a call hands to the context's kernels: device memory of the context's GPU,
// or managed memory. Checked with cudaPointerGetAttributes once per pointer value, then
// remembered, so that steps over the same buffers pay a set lookup. A host pointer, or one
// of another GPU, is refused (INVALID_ARG) instead of faulting in a kernel.
static bool dev_ptr_ok(const zero_ctx* c, const void* p) {
    const uintptr_t key = (uintptr_t)p;
    if (c->dev_ok.count(key)) return true;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // the non-sticky error of an unknown pointer
        return false;
    }
    const bool ok = attr.type == cudaMemoryTypeManaged ||
                    (attr.type == cudaMemoryTypeDevice && attr.device == c->device);
    if (!ok) return false;
    if (c->dev_ok.size() >= 4096) c->dev_ok.clear();
    c->dev_ok.insert(key);
    return true;
}

static int check_grads(const zero_ctx* c, const void* const* grads) {
    if (!grads) return ZERO_ERR_INVALID_ARG;
    for (int r = 0; r < c->cfg.M; ++r) {
        if (!grads[r]) return ZERO_ERR_INVALID_ARG;
        if (!aligned16(grads[r])) return ZERO_ERR_MISALIGNED;
        if (!dev_ptr_ok(c, grads[r])) return ZERO_ERR_INVALID_ARG;
    }
    return ZERO_OK;
}

// The kernels of one whole step: reduce-scatter (+ norm and clip), AdamW, all-gather.
// sched: the scalars come from the device schedule (k_step_begin ran first), not a.k.
static int launch_step(zero_ctx* c, const zg::StepArgs& a, int clip, int mode, double max_norm, bool sched,
                       cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (clip) {
        const bool write = mode == ZERO_GHAT_MATERIALIZE;
        const int g1 = grid_for(c, write ? zg::kVarRsNormWrite : zg::kVarRsNormOnly, a.nvec);
        {
            Timed tm(c, ZERO_K_RS_NORM, s);
            e = zg::launch_rs_norm(a, write, g1, s);
        }
        if (e == cudaSuccess) {
            Timed tm(c, ZERO_K_NORM_FINAL, s);
            e = zg::launch_norm_final(c->status, c->partials, g1, max_norm, 1, sched, s);
        }
        if (e == cudaSuccess) {
            if (write) {
                const int g3 = grid_for(c, zg::kVarAdamw, a.nvec);
                Timed tm(c, ZERO_K_ADAMW, s);
                e = zg::launch_adamw(a, sched, g3, s);
            } else {
                const int g4 = grid_for(c, zg::kVarRsAdamwScaled, a.nvec);
                Timed tm(c, ZERO_K_RS_ADAMW, s);
                e = zg::launch_rs_adamw(a, true, sched, g4, s);
            }
        }
    } else {
        const int g4 = grid_for(c, zg::kVarRsAdamwPlain, a.nvec);
        Timed tm(c, ZERO_K_RS_ADAMW, s);
        e = zg::launch_rs_adamw(a, false, sched, g4, s);
    }
    if (e == cudaSuccess && c->cfg.gather == ZERO_GATHER_SHARDS) {
        const int rc = gather_range(c, 0, c->n, (uint16_t*)c->bufs.param_full, s);  // the all-gather
        if (rc) return rc;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    c->last_clip = clip;
    c->last_stream = s;
    c->stepped = 1;
    return ZERO_OK;
}

static int launch_step_begin(zero_ctx* c, cudaStream_t s) {
    Timed tm(c, ZERO_K_STEP_BEGIN, s);
    const cudaError_t e = zg::launch_step_begin(c->status, c->dev_sched, s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e);
}

int zero_step(zero_ctx* c, const void* const* grads, int stage, const zero_hyper* h, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    if (c->n_reduced || c->n_bucket_done) return ZERO_ERR_INVALID_ARG;  // a per-bucket step is in progress
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    int rc = check_hyper(h);
    if (rc) return rc;
    if ((rc = check_grads(c, grads))) return rc;
    int mode;
    if ((rc = resolve_ghat_mode(c, h, &mode))) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;

    c->t += 1;
    zg::StepArgs a = base_args(c);
    for (int r = 0; r < c->cfg.M; ++r) a.grads[r] = (const uint16_t*)grads[r];
    a.k = adam_consts(h, c->t);
    return launch_step(c, a, h->clip, mode, h->max_grad_norm, false, s);
}

int zero_step_scheduled(zero_ctx* c, const void* const* grads, int stage, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (!c->sched_active) return ZERO_ERR_SCHEDULE;
    if (c->n_reduced || c->n_bucket_done) return ZERO_ERR_INVALID_ARG;
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    int rc = check_grads(c, grads);
    if (rc) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    zg::StepArgs a = base_args(c);
    for (int r = 0; r < c->cfg.M; ++r) a.grads[r] = (const uint16_t*)grads[r];
    if ((rc = launch_step_begin(c, s))) return rc;
    return launch_step(c, a, c->sched_clip, c->sched_mode, 0.0, true, s);
}

int zero_reduce_bucket(zero_ctx* c, int64_t bucket, const void* const* grads_b, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    const int64_t nb = (int64_t)c->buckets.size();
    if (bucket < 0 || bucket >= nb || !grads_b) return ZERO_ERR_INVALID_ARG;
    if (!c->bufs.ghat) return ZERO_ERR_SIZE_MISMATCH;
    if (c->n_bucket_done) return ZERO_ERR_INVALID_ARG;  // a zero_step_bucket step is in progress
    for (int r = 0; r < c->cfg.M; ++r) {
        if (!grads_b[r]) return ZERO_ERR_INVALID_ARG;
        if (!aligned16(grads_b[r])) return ZERO_ERR_MISALIGNED;
        if (!dev_ptr_ok(c, grads_b[r])) return ZERO_ERR_INVALID_ARG;
    }
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    const zg::Bucket& e = c->buckets[(size_t)bucket];
    zg::StepArgs a = base_args(c);
    for (int r = 0; r < c->cfg.M; ++r) a.grads[r] = (const uint16_t*)grads_b[r];
    a.vbeg = e.off / 8;
    a.vend = e.end / 8;
    a.gbase = e.off;
    a.gext = e.end - e.off;
    a.b_first = bucket;
    a.b_end = bucket + 1;
    int g1 = grid_for(c, zg::kVarRsNormWrite, a.vend - a.vbeg);
    double* parts = c->partials;
    int sum_pdl = zg::kPdlNone;
    if (c->overlap != ZERO_OVERLAP_NONE) {
        // launch overlap: the bucket's partials in a region of its own, so that the next
        // bucket's reduction may run while this bucket's sum is still being formed; the
        // reduction may overlap its predecessor when it follows the previous bucket's
        // reduction of this step (a bucket reduced twice in one step waits)
        if (g1 > zg::kBucketPartials) g1 = zg::kBucketPartials;
        parts = c->bucket_partials + (size_t)bucket * zg::kBucketPartials;
        a.partials = parts;
        a.part_cap = zg::kBucketPartials;
        a.pdl = pdl_mode(c, ZERO_K_RS_NORM, s, c->n_reduced > 0 && !c->reduced[(size_t)bucket]);
        sum_pdl = c->overlap == ZERO_OVERLAP_BUCKETS ? zg::kPdlTriggerWait : zg::kPdlWaitFirst;
    }
    cudaError_t err;
    {
        Timed tm(c, ZERO_K_RS_NORM, s);
        err = zg::launch_rs_norm(a, true, g1, s);
    }
    if (err == cudaSuccess) {
        Timed tm(c, ZERO_K_NORM_FINAL, s);
        err = zg::launch_sum_partials(parts, g1, c->bucket_sums + bucket, s, sum_pdl);
    }
    if (err != cudaSuccess) return cuda_fail(err);
    if (c->overlap != ZERO_OVERLAP_NONE) note_chain(c, ZERO_K_RS_NORM, s);
    if (!c->reduced[(size_t)bucket]) c->n_reduced += 1;
    c->reduced[(size_t)bucket] = 1;
    return ZERO_OK;
}

// One bucket of a ZeRO-2 fused per-bucket step (zero_step_bucket[_scheduled]).
static int step_one_bucket(zero_ctx* c, int64_t bucket, const void* const* grads_b, const zero_hyper* h,
                           cudaStream_t s) {
    const bool sched = h == nullptr;
    const zg::Bucket& e = c->buckets[(size_t)bucket];
    zg::StepArgs a = base_args(c);
    // The fused kernel addresses gradients by absolute lane: rebase each bucket buffer so that
    // lane o of the bucket lands on grads_b[r][o - off] (address arithmetic only; the kernel
    // touches lanes [off, end) alone).
    for (int r = 0; r < c->cfg.M; ++r)
        a.grads[r] = (const uint16_t*)((uintptr_t)grads_b[r] - (uintptr_t)(2 * e.off));
    a.vbeg = e.off / 8;
    a.vend = e.end / 8;
    a.gext = e.end;
    a.b_first = bucket;
    a.b_end = bucket + 1;
    if (!sched) a.k = adam_consts(h, c->t + 1);  // every bucket of the step takes step t + 1
    int rc;
    if (sched && c->n_bucket_done == 0 && (rc = launch_step_begin(c, s))) return rc;  // once per step
    const int g4 = grid_for(c, zg::kVarRsAdamwPlain, a.vend - a.vbeg);
    // launch overlap: buckets after the first of a step may overlap the bucket before;
    // scheduled steps launch as ordinary kernels
    a.pdl = sched ? zg::kPdlNone : pdl_mode(c, ZERO_K_RS_ADAMW, s, c->n_bucket_done > 0);
    cudaError_t err;
    {
        Timed tm(c, ZERO_K_RS_ADAMW, s);
        err = zg::launch_rs_adamw(a, false, sched, g4, s);
    }
    if (err != cudaSuccess) return cuda_fail(err);
    if (a.pdl != zg::kPdlNone) note_chain(c, ZERO_K_RS_ADAMW, s);
    if (c->cfg.gather == ZERO_GATHER_SHARDS) {  // the bucket's all-gather
        rc = gather_range(c, e.uoff, e.n, (uint16_t*)c->bufs.param_full + e.uoff, s, false, bucket, bucket + 1);
        if (rc) return rc;
    }
    c->bucket_done[(size_t)bucket] = 1;
    c->last_stream = s;
    if (++c->n_bucket_done == (int64_t)c->buckets.size()) {  // the step is complete
        std::fill(c->bucket_done.begin(), c->bucket_done.end(), 0);
        c->n_bucket_done = 0;
        if (!sched) c->t += 1;
        c->last_clip = 0;
        c->stepped = 1;
    }
    return ZERO_OK;
}

static int check_step_bucket(const zero_ctx* c, int64_t bucket, const void* const* grads_b, int stage) {
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    if (bucket < 0 || bucket >= (int64_t)c->buckets.size() || !grads_b) return ZERO_ERR_INVALID_ARG;
    if (c->n_reduced || c->bucket_done[(size_t)bucket]) return ZERO_ERR_INVALID_ARG;
    for (int r = 0; r < c->cfg.M; ++r) {
        if (!grads_b[r]) return ZERO_ERR_INVALID_ARG;
        if (!aligned16(grads_b[r])) return ZERO_ERR_MISALIGNED;
        if (!dev_ptr_ok(c, grads_b[r])) return ZERO_ERR_INVALID_ARG;
    }
    return ZERO_OK;
}

int zero_step_bucket(zero_ctx* c, int64_t bucket, const void* const* grads_b, int stage, const zero_hyper* h,
                     void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    int rc = check_hyper(h);
    if (rc) return rc;
    // clipping needs every bucket's norm before any update: zero_reduce_bucket + zero_apply
    if (h->clip) return ZERO_ERR_INVALID_ARG;
    if ((rc = check_step_bucket(c, bucket, grads_b, stage))) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    return step_one_bucket(c, bucket, grads_b, h, (cudaStream_t)stream);
}

int zero_step_bucket_scheduled(zero_ctx* c, int64_t bucket, const void* const* grads_b, int stage, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (!c->sched_active) return ZERO_ERR_SCHEDULE;
    if (c->sched_clip) return ZERO_ERR_INVALID_ARG;
    int rc = check_step_bucket(c, bucket, grads_b, stage);
    if (rc) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    return step_one_bucket(c, bucket, grads_b, nullptr, (cudaStream_t)stream);
}

// The rest of a streamed step once every bucket is reduced: norm (+ clip), AdamW, all-gather.
static int launch_apply(zero_ctx* c, const zg::StepArgs& a, int clip, double max_norm, bool sched, cudaStream_t s) {
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_NORM_FINAL, s);
        e = zg::launch_norm_final(c->status, c->bucket_sums, (int)c->buckets.size(), max_norm, clip, sched, s);
    }
    if (e == cudaSuccess) {
        const int g3 = grid_for(c, zg::kVarAdamw, a.nvec);
        Timed tm(c, ZERO_K_ADAMW, s);
        e = zg::launch_adamw(a, sched, g3, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (c->cfg.gather == ZERO_GATHER_SHARDS) {
        const int rc = gather_range(c, 0, c->n, (uint16_t*)c->bufs.param_full, s);
        if (rc) return rc;
    }
    std::fill(c->reduced.begin(), c->reduced.end(), 0);
    c->n_reduced = 0;
    c->last_clip = clip;
    c->last_stream = s;
    c->stepped = 1;
    return ZERO_OK;
}

static int check_apply(const zero_ctx* c, int stage) {
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    if (!c->bufs.ghat) return ZERO_ERR_SIZE_MISMATCH;
    for (char r : c->reduced)
        if (!r) return ZERO_ERR_INVALID_ARG;  // every bucket must be reduced first
    return ZERO_OK;
}

int zero_apply(zero_ctx* c, int stage, const zero_hyper* h, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    int rc = check_hyper(h);
    if (rc) return rc;
    if ((rc = check_apply(c, stage))) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    c->t += 1;
    zg::StepArgs a = base_args(c);
    a.k = adam_consts(h, c->t);
    return launch_apply(c, a, h->clip, h->max_grad_norm, false, s);
}

int zero_apply_scheduled(zero_ctx* c, int stage, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (!c->sched_active) return ZERO_ERR_SCHEDULE;
    int rc = check_apply(c, stage);
    if (rc) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    zg::StepArgs a = base_args(c);
    if ((rc = launch_step_begin(c, s))) return rc;
    return launch_apply(c, a, c->sched_clip, 0.0, true, s);
}

// The device step counter of scheduled mode (synchronises the device).
static int read_device_step(zero_ctx* c, int64_t* t) {
    zg::Status st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&st, c->status, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    *t = st.t_dev;
    return ZERO_OK;
}

int zero_set_schedule(zero_ctx* c, const zero_hyper* h, int64_t count, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (count < 0 || (count > 0 && !h)) return ZERO_ERR_INVALID_ARG;
    if (count > ZERO_MAX_SCHEDULE) return ZERO_ERR_TOO_LARGE;
    int mode = ZERO_GHAT_RECOMPUTE;
    for (int64_t i = 0; i < count; ++i) {
        int rc = check_hyper(&h[i]);
        if (rc) return rc;
        if (h[i].clip != h[0].clip || h[i].ghat_mode != h[0].ghat_mode) return ZERO_ERR_INVALID_ARG;
        if (i == 0 && (rc = resolve_ghat_mode(c, &h[0], &mode))) return rc;
    }
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cap != cudaStreamCaptureStatusNone) return ZERO_ERR_INVALID_ARG;
    if (c->sched_active) {  // continue from the last step that ran
        int64_t t = 0;
        const int rc = read_device_step(c, &t);
        if (rc) return rc;
        c->t = t;
    }
    std::vector<zg::ScheduleEntry> tab((size_t)count);
    for (int64_t i = 0; i < count; ++i) {
        tab[(size_t)i].k = adam_consts(&h[i], c->t + 1 + i);
        tab[(size_t)i].max_norm = h[i].clip ? h[i].max_grad_norm : 0.0;
    }
    if (count > 0)
        e = cudaMemcpyAsync(c->dev_sched, tab.data(), (size_t)count * sizeof(zg::ScheduleEntry),
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = zg::launch_schedule_install(c->status, c->t, count, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the host table must outlive the copy
    if (e != cudaSuccess) return cuda_fail(e);
    c->sched_active = count > 0;
    c->sched_clip = count > 0 ? h[0].clip : 0;
    c->sched_mode = mode;
    c->last_stream = s;
    // launch shapes now, outside any capture
    for (int v = 0; v < zg::kNumVariants; ++v) grid_for(c, v, 1);
    return ZERO_OK;
}

int zero_step_host(zero_ctx* c, const void* const* host_grads, void* const* dev_grads, int stage,
                   const zero_hyper* h, void* host_params, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    if (!host_grads || !dev_grads || !host_params) return ZERO_ERR_INVALID_ARG;
    for (int r = 0; r < c->cfg.M; ++r)
        if (!host_grads[r] || !dev_grads[r]) return ZERO_ERR_INVALID_ARG;
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    int rc = check_hyper(h);
    if (rc) return rc;
    if ((rc = check_grads(c, (const void* const*)dev_grads))) return rc;  // before any copy
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t gbytes = (size_t)(2 * c->npad);
    for (int r = 0; r < c->cfg.M; ++r) {
        cudaError_t e = cudaMemcpyAsync(dev_grads[r], host_grads[r], gbytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    rc = zero_step(c, (const void* const*)dev_grads, stage, h, stream);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(host_params, c->bufs.param_full, (size_t)(2 * c->n), cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e);
}

int zero_save_state(zero_ctx* c, void* master, void* m, void* v, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!master && !m && !v) return ZERO_ERR_INVALID_ARG;
    for (const void* p : {(const void*)master, (const void*)m, (const void*)v})
        if (p && !dev_ptr_ok(c, p)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    // process-per-rank mode: this rank's real lanes only, through its own table
    const int64_t lanes = c->cfg.sharded ? c->shard_len : c->npad;
    const int grid = grid_for(c, zg::kVarInit, lanes);
    cudaError_t e = zg::launch_save((const float*)c->bufs.master, (const float*)c->bufs.m, (const float*)c->bufs.v,
                                    (float*)master, (float*)m, (float*)v,
                                    c->cfg.sharded ? c->dev_local : c->dev_buckets, (int64_t)c->buckets.size(),
                                    lanes, c->n, c->status, grid, s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e);
}

int zero_load_state(zero_ctx* c, const void* master, const void* m, const void* v, int64_t t, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    if (!master || t < 0) return ZERO_ERR_INVALID_ARG;
    for (const void* p : {master, m, v})
        if (p && !dev_ptr_ok(c, p)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    const cudaError_t e = launch_state_in(c, (const float*)master, (const float*)m, (const float*)v, s);
    if (e != cudaSuccess) return cuda_fail(e);
    c->t = t;
    c->rank_reduced = false;
    if (c->cfg.sharded) {  // a loaded state starts a fresh step
        std::fill(c->reduced.begin(), c->reduced.end(), 0);
        c->n_reduced = 0;
        std::fill(c->bucket_done.begin(), c->bucket_done.end(), 0);
        c->n_bucket_done = 0;
    }
    return ZERO_OK;
}

int zero_step_host_overlapped(zero_ctx* c, const void* const* host_grads, void* const* dev_grads, int stage,
                              const zero_hyper* h, void* host_params, void* stream, void* copy_stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    if (!host_grads || !dev_grads || !host_params || copy_stream == stream) return ZERO_ERR_INVALID_ARG;
    for (int r = 0; r < c->cfg.M; ++r)
        if (!host_grads[r] || !dev_grads[r]) return ZERO_ERR_INVALID_ARG;
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    int rc = check_hyper(h);
    if (rc) return rc;
    if ((rc = check_grads(c, (const void* const*)dev_grads))) return rc;  // before any copy
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream, cs = (cudaStream_t)copy_stream;
    cudaError_t e = cudaSuccess;
    if (!c->h2d_done) {
        e = cudaEventCreateWithFlags(&c->h2d_done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    zero_ctx::GradSet* set = nullptr;
    for (auto& g : c->grad_sets)
        if (g.key == dev_grads[0]) set = &g;
    if (!set && c->grad_sets.size() >= 8) {
        // forget sets whose last reading step has finished: nothing to wait for there
        std::vector<zero_ctx::GradSet> keep;
        for (auto& g : c->grad_sets) {
            if (g.recorded && cudaEventQuery(g.consumed) == cudaSuccess) cudaEventDestroy(g.consumed);
            else keep.push_back(g);
        }
        c->grad_sets.swap(keep);
    }
    if (!set) {
        if (c->grad_sets.size() >= 8) return ZERO_ERR_INVALID_ARG;  // a handful of buffer sets at most
        zero_ctx::GradSet g{dev_grads[0], nullptr, false};
        e = cudaEventCreateWithFlags(&g.consumed, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
        c->grad_sets.push_back(g);
        set = &c->grad_sets.back();
    }
    // the copy may overwrite this device set only after the last step that read it
    if (set->recorded && (e = cudaStreamWaitEvent(cs, set->consumed, 0)) != cudaSuccess) return cuda_fail(e);
    const size_t gbytes = (size_t)(2 * c->npad);
    for (int r = 0; r < c->cfg.M; ++r) {
        e = cudaMemcpyAsync(dev_grads[r], host_grads[r], gbytes, cudaMemcpyHostToDevice, cs);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if ((e = cudaEventRecord(c->h2d_done, cs)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(s, c->h2d_done, 0)) != cudaSuccess) return cuda_fail(e);
    rc = zero_step(c, (const void* const*)dev_grads, stage, h, stream);
    if (rc) return rc;
    if ((e = cudaEventRecord(set->consumed, s)) != cudaSuccess) return cuda_fail(e);
    set->recorded = true;
    // on the kernels' stream: the next step's kernels rewrite the parameters after this copy
    e = cudaMemcpyAsync(host_params, c->bufs.param_full, (size_t)(2 * c->n), cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------------------
// Process-per-rank mode. The kernels are the emulated mode's, run over this rank's shard
// (the local table) with the exchanged slices as their M sources.
// ---------------------------------------------------------------------------------------
static bool hybrid(const zero_ctx* c) { return c->cfg.groups > 1; }

// Arguments of a kernel over this rank's shard; the caller sets the sources.
static zg::StepArgs rank_args(zero_ctx* c) {
    zg::StepArgs a = base_args(c);
    a.out = (uint16_t*)c->bufs.param_shards;  // the owner's bf16 shard, the all-gather's send buffer
    a.out_shards = 1;
    a.buckets = c->dev_local;
    a.nvec = c->shard_len / 8;
    a.vbeg = 0;
    a.vend = a.nvec;
    a.gbase = 0;
    a.gext = c->shard_len;
    a.npad = c->shard_len;
    a.groups = 1;
    return a;
}

// The exchange buffer as the sources of one launch over the whole shard: `count` sources,
// bucket b's slice of source q at lanes [count * base_b + q * S_b, +S_b) (the kernels find it
// from the rank's own table).
static void exchange_sources(const zero_ctx* c, zg::StepArgs& a, const void* recv, int count) {
    a.grads[0] = (const uint16_t*)recv;
    a.M = count;
    a.gext = c->npad;  // lanes of the exchange buffer
}

// Restricts a launch over the shard to bucket b's slice: local lanes [base_b, base_b + S_b).
static void one_bucket(const zero_ctx* c, zg::StepArgs& a, int64_t b) {
    const zg::Bucket& L = c->local[(size_t)b];
    a.vbeg = L.off / 8;
    a.vend = L.end / 8;
    a.b_first = b;
    a.b_end = b + 1;
}

// Hybrid mode: the G gathered fp32 group partials of this shard, group grp at [grp * shard_len].
static void part_sources(const zero_ctx* c, zg::StepArgs& a, const void* parts) {
    for (int grp = 0; grp < c->cfg.groups; ++grp)
        a.grads[grp] = (const uint16_t*)((const float*)parts + (size_t)grp * (size_t)c->shard_len);
    a.M = c->cfg.groups;
}

static int check_rank_ctx(const zero_ctx* c) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!c->cfg.sharded) return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

// The group partial of the whole shard (bucket < 0) or of one bucket's slice.
static int rank_partial(zero_ctx* c, int64_t bucket, const void* recv, void* part, void* stream) {
    int rc = check_rank_ctx(c);
    if (rc) return rc;
    if (!hybrid(c) || !recv || !part || bucket >= (int64_t)c->buckets.size()) return ZERO_ERR_INVALID_ARG;
    if (!aligned16(recv) || !aligned16(part)) return ZERO_ERR_MISALIGNED;
    if (!dev_ptr_ok(c, recv) || !dev_ptr_ok(c, part)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    // the group's K slices summed in order from +0, unscaled (x 1 is exact), into `part`; the
    // pass's partial sums of squares are not used
    zg::StepArgs a = rank_args(c);
    exchange_sources(c, a, recv, shard_count(&c->cfg));
    if (bucket >= 0) one_bucket(c, a, bucket);
    a.inv_M = 1.0f;
    a.ghat = (float*)part;
    const int g1 = grid_for(c, zg::kVarRsNormWriteX, a.vend - a.vbeg);
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_RS_NORM, s);
        e = zg::launch_rs_norm_exchange(a, true, g1, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    c->last_stream = s;
    return ZERO_OK;
}

int zero_rank_partial(zero_ctx* c, const void* recv, void* part, void* stream) {
    return rank_partial(c, -1, recv, part, stream);
}

int zero_rank_partial_bucket(zero_ctx* c, int64_t bucket, const void* recv, void* part, void* stream) {
    if (bucket < 0) return ZERO_ERR_INVALID_ARG;
    return rank_partial(c, bucket, recv, part, stream);
}

int zero_rank_sumsq(zero_ctx* c, const void* src, const zero_hyper* h, double* sumsq, void* stream) {
    int rc = check_rank_ctx(c);
    if (rc) return rc;
    if (c->n_bucket_done) return ZERO_ERR_INVALID_ARG;  // a per-bucket step is in progress
    if ((rc = check_hyper(h))) return rc;
    if (!h->clip || !sumsq) return ZERO_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(sumsq) & 7u) return ZERO_ERR_MISALIGNED;
    if (!dev_ptr_ok(c, sumsq)) return ZERO_ERR_INVALID_ARG;
    const int64_t nb = (int64_t)c->buckets.size();
    if (!src) {  // every bucket reduced by zero_rank_reduce_bucket: the sum of their sums
        if (c->n_reduced != nb) return ZERO_ERR_INVALID_ARG;
        DeviceGuard guard(c->device);
        if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
        cudaStream_t s = (cudaStream_t)stream;
        cudaError_t e;
        {
            Timed tm(c, ZERO_K_NORM_FINAL, s);
            e = zg::launch_sum_partials(c->bucket_sums, (int)nb, sumsq, s);
        }
        if (e != cudaSuccess) return cuda_fail(e);
        std::fill(c->reduced.begin(), c->reduced.end(), 0);
        c->n_reduced = 0;
        c->rank_reduced = true;
        c->rank_mode = ZERO_GHAT_MATERIALIZE;
        c->last_stream = s;
        return ZERO_OK;
    }
    if (c->n_reduced) return ZERO_ERR_INVALID_ARG;  // a per-bucket reduction is in progress
    if (!aligned16(src)) return ZERO_ERR_MISALIGNED;
    int mode;
    if ((rc = resolve_ghat_mode(c, h, &mode))) return rc;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    const bool write = mode == ZERO_GHAT_MATERIALIZE;
    // one pass over the whole shard: from the gathered group partials (hybrid) or from the
    // exchange buffer (flat)
    zg::StepArgs a = rank_args(c);
    if (hybrid(c)) part_sources(c, a, src);
    else exchange_sources(c, a, src, c->cfg.M);
    const int g1 = grid_for(c, hybrid(c) ? (write ? zg::kVarRsNormWriteF : zg::kVarRsNormOnlyF)
                                         : (write ? zg::kVarRsNormWriteX : zg::kVarRsNormOnlyX),
                            a.nvec);
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_RS_NORM, s);
        e = hybrid(c) ? zg::launch_rs_norm_f32src(a, write, g1, s) : zg::launch_rs_norm_exchange(a, write, g1, s);
    }
    if (e == cudaSuccess) {
        Timed tm(c, ZERO_K_NORM_FINAL, s);
        e = zg::launch_sum_partials(c->partials, g1, sumsq, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    c->rank_reduced = true;
    c->rank_mode = mode;
    c->last_stream = s;
    return ZERO_OK;
}

int zero_rank_step(zero_ctx* c, const void* src, const double* sumsq_all, int stage, const zero_hyper* h,
                   void* stream) {
    int rc = check_rank_ctx(c);
    if (rc) return rc;
    if (c->n_bucket_done || c->n_reduced) return ZERO_ERR_INVALID_ARG;  // a per-bucket step is in progress
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    if ((rc = check_hyper(h))) return rc;
    const int clip = h->clip;
    if (clip && (!sumsq_all || !c->rank_reduced)) return ZERO_ERR_INVALID_ARG;
    const int mode = clip ? c->rank_mode : ZERO_GHAT_RECOMPUTE;
    const bool from_ghat = clip && mode == ZERO_GHAT_MATERIALIZE;  // the sources are not read again
    if (!from_ghat && !src) return ZERO_ERR_INVALID_ARG;
    if (src && !aligned16(src)) return ZERO_ERR_MISALIGNED;
    if (clip && (reinterpret_cast<uintptr_t>(sumsq_all) & 7u)) return ZERO_ERR_MISALIGNED;
    if ((src && !dev_ptr_ok(c, src)) || (clip && !dev_ptr_ok(c, sumsq_all))) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    c->t += 1;
    const zg::AdamConsts k = adam_consts(h, c->t);
    cudaError_t e = cudaSuccess;
    if (clip) {  // every rank sums the same P values in the same order: the same norm and scale
        const int P = hybrid(c) ? shard_count(&c->cfg) : c->cfg.M;
        Timed tm(c, ZERO_K_NORM_FINAL, s);
        e = zg::launch_norm_final(c->status, sumsq_all, P, h->max_grad_norm, 1, false, s);
    }
    if (e == cudaSuccess && from_ghat) {
        zg::StepArgs a = rank_args(c);
        a.k = k;
        const int g3 = grid_for(c, zg::kVarAdamw, a.nvec);
        Timed tm(c, ZERO_K_ADAMW, s);
        e = zg::launch_adamw(a, false, g3, s);
    } else if (e == cudaSuccess) {  // the fused pass, one launch over the whole shard
        zg::StepArgs a = rank_args(c);
        if (hybrid(c)) part_sources(c, a, src);
        else exchange_sources(c, a, src, c->cfg.M);
        a.k = k;
        const int g4 = grid_for(c, hybrid(c) ? (clip ? zg::kVarRsAdamwScaledF : zg::kVarRsAdamwPlainF)
                                             : (clip ? zg::kVarRsAdamwScaledX : zg::kVarRsAdamwPlainX),
                                a.nvec);
        Timed tm(c, ZERO_K_RS_ADAMW, s);
        e = hybrid(c) ? zg::launch_rs_adamw_f32src(a, clip != 0, g4, s)
                      : zg::launch_rs_adamw_exchange(a, clip != 0, g4, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    c->rank_reduced = false;
    c->last_clip = clip;
    c->last_stream = s;
    c->stepped = 1;
    return ZERO_OK;
}

int zero_rank_reduce_bucket(zero_ctx* c, int64_t bucket, const void* src, void* stream) {
    int rc = check_rank_ctx(c);
    if (rc) return rc;
    const int64_t nb = (int64_t)c->buckets.size();
    if (!src || bucket < 0 || bucket >= nb) return ZERO_ERR_INVALID_ARG;
    if (!c->bufs.ghat) return ZERO_ERR_SIZE_MISMATCH;
    if (c->n_bucket_done || c->rank_reduced) return ZERO_ERR_INVALID_ARG;
    if (!aligned16(src)) return ZERO_ERR_MISALIGNED;
    if (!dev_ptr_ok(c, src)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    // the bucket's average into the ghat shard, its sum of squares into its slot: from the
    // exchange buffer (flat) or the gathered group partials (hybrid)
    zg::StepArgs a = rank_args(c);
    if (hybrid(c)) part_sources(c, a, src);
    else exchange_sources(c, a, src, c->cfg.M);
    one_bucket(c, a, bucket);
    const int g1 = grid_for(c, hybrid(c) ? zg::kVarRsNormWriteF : zg::kVarRsNormWriteX, a.vend - a.vbeg);
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_RS_NORM, s);
        e = hybrid(c) ? zg::launch_rs_norm_f32src(a, true, g1, s) : zg::launch_rs_norm_exchange(a, true, g1, s);
    }
    if (e == cudaSuccess) {
        Timed tm(c, ZERO_K_NORM_FINAL, s);
        e = zg::launch_sum_partials(c->partials, g1, c->bucket_sums + bucket, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    if (!c->reduced[(size_t)bucket]) c->n_reduced += 1;
    c->reduced[(size_t)bucket] = 1;
    c->last_stream = s;
    return ZERO_OK;
}

int zero_rank_step_bucket(zero_ctx* c, int64_t bucket, const void* src, int stage, const zero_hyper* h,
                          void* stream) {
    int rc = check_rank_ctx(c);
    if (rc) return rc;
    if (stage != c->cfg.stage) return ZERO_ERR_STAGE;
    if ((rc = check_hyper(h))) return rc;
    const int64_t nb = (int64_t)c->buckets.size();
    if (h->clip || !src || bucket < 0 || bucket >= nb) return ZERO_ERR_INVALID_ARG;
    if (c->rank_reduced || c->n_reduced || c->bucket_done[(size_t)bucket]) return ZERO_ERR_INVALID_ARG;
    if (!aligned16(src)) return ZERO_ERR_MISALIGNED;
    if (!dev_ptr_ok(c, src)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    zg::StepArgs a = rank_args(c);
    if (hybrid(c)) part_sources(c, a, src);
    else exchange_sources(c, a, src, c->cfg.M);
    one_bucket(c, a, bucket);
    a.k = adam_consts(h, c->t + 1);  // every bucket of the step takes step t + 1
    const int g4 = grid_for(c, hybrid(c) ? zg::kVarRsAdamwPlainF : zg::kVarRsAdamwPlainX, a.vend - a.vbeg);
    cudaError_t e;
    {
        Timed tm(c, ZERO_K_RS_ADAMW, s);
        e = hybrid(c) ? zg::launch_rs_adamw_f32src(a, false, g4, s) : zg::launch_rs_adamw_exchange(a, false, g4, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    c->bucket_done[(size_t)bucket] = 1;
    c->last_stream = s;
    if (++c->n_bucket_done == nb) {  // the step is complete
        std::fill(c->bucket_done.begin(), c->bucket_done.end(), 0);
        c->n_bucket_done = 0;
        c->t += 1;
        c->last_clip = 0;
        c->stepped = 1;
    }
    return ZERO_OK;
}

int zero_params(zero_ctx* c, void** full_bf16) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!full_bf16) return ZERO_ERR_INVALID_ARG;
    *full_bf16 = c->bufs.param_full;
    return ZERO_OK;
}

int zero_gather(zero_ctx* c, int64_t bucket, void* dst, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->cfg.gather != ZERO_GATHER_SHARDS) return ZERO_ERR_INVALID_ARG;
    const int64_t nb = (int64_t)c->buckets.size();
    if (bucket < -1 || bucket >= nb) return ZERO_ERR_INVALID_ARG;
    if (dst && !aligned16(dst)) return ZERO_ERR_MISALIGNED;
    if (dst && !dev_ptr_ok(c, dst)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    uint16_t* out = (uint16_t*)(dst ? dst : c->bufs.param_full);
    int64_t u0 = 0, count = c->n;
    if (bucket >= 0) {
        u0 = c->buckets[(size_t)bucket].uoff;
        count = c->buckets[(size_t)bucket].n;
    }
    return gather_range(c, u0, count, out + u0, (cudaStream_t)stream, true, bucket >= 0 ? bucket : 0,
                        bucket >= 0 ? bucket + 1 : 0);
}

int zero_gather_bucket(zero_ctx* c, int64_t bucket, void* dst, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->cfg.sharded) return ZERO_ERR_INVALID_ARG;  // emulated mode only
    if (c->cfg.gather != ZERO_GATHER_SHARDS || !dst) return ZERO_ERR_INVALID_ARG;
    if (bucket < 0 || bucket >= (int64_t)c->buckets.size()) return ZERO_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dst) & 1u) return ZERO_ERR_MISALIGNED;
    if (!dev_ptr_ok(c, dst)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    const zg::Bucket& e = c->buckets[(size_t)bucket];
    return gather_range(c, e.uoff, e.n, (uint16_t*)dst, (cudaStream_t)stream, true, bucket, bucket + 1);
}

int zero_bucket_info(zero_ctx* c, int64_t bucket, int64_t* uoff, int64_t* n) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (bucket < 0 || bucket >= (int64_t)c->buckets.size() || !uoff || !n) return ZERO_ERR_INVALID_ARG;
    *uoff = c->buckets[(size_t)bucket].uoff;
    *n = c->buckets[(size_t)bucket].n;
    return ZERO_OK;
}

int zero_get_state(zero_ctx* c, int which, int rank, void* dst, void* stream) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!dst || rank < 0 || rank >= shard_count(&c->cfg)) return ZERO_ERR_INVALID_ARG;
    const float* src = nullptr;
    switch (which) {
        case ZERO_STATE_MASTER: src = (const float*)c->bufs.master; break;
        case ZERO_STATE_M: src = (const float*)c->bufs.m; break;
        case ZERO_STATE_V: src = (const float*)c->bufs.v; break;
        case ZERO_STATE_GHAT: src = (const float*)c->bufs.ghat; break;
        default: return ZERO_ERR_INVALID_ARG;
    }
    if (!src) return ZERO_ERR_SIZE_MISMATCH;
    if (!dev_ptr_ok(c, dst)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaStream_t s = (cudaStream_t)stream;
    float* d = (float*)dst;
    if (c->cfg.sharded) {  // the shard is contiguous on this rank
        if (rank != c->owner) return ZERO_ERR_INVALID_ARG;
        const cudaError_t ce =
            cudaMemcpyAsync(d, src, sizeof(float) * (size_t)c->shard_len, cudaMemcpyDeviceToDevice, s);
        return ce == cudaSuccess ? ZERO_OK : cuda_fail(ce);
    }
    for (const zg::Bucket& e : c->buckets) {
        const int64_t S = (e.end - e.off) / shard_count(&c->cfg);
        cudaError_t ce = cudaMemcpyAsync(d, src + e.off + rank * S, sizeof(float) * (size_t)S,
                                         cudaMemcpyDeviceToDevice, s);
        if (ce != cudaSuccess) return cuda_fail(ce);
        d += S;
    }
    return ZERO_OK;
}

static int read_status(zero_ctx* c, zg::Status* out) {
    DeviceGuard guard(c->device);
    ++c->seq;  // enqueues stream work: no later per-bucket launch overlaps what came before
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    cudaError_t e;
    if (c->sched_active) {  // replays of captured steps may run on any stream
        e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaMemcpy(out, c->status, sizeof *out, cudaMemcpyDeviceToHost);
    } else {
        e = cudaMemcpyAsync(out, c->status, sizeof *out, cudaMemcpyDeviceToHost, c->last_stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
    }
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e);
}

int zero_last_norm(zero_ctx* c, double* norm, float* scale) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!norm || !scale) return ZERO_ERR_INVALID_ARG;
    if (!c->stepped || !c->last_clip) return ZERO_ERR_NOT_COMPUTED;
    zg::Status st;
    int rc = read_status(c, &st);
    if (rc) return rc;
    *norm = st.norm;
    *scale = st.scale;
    return ZERO_OK;
}

int zero_sync_status(zero_ctx* c) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    zg::Status st;
    int rc = read_status(c, &st);
    if (rc) return rc;
    if (st.flags & zg::kFlagBounds) return ZERO_ERR_DEVICE;
    if (st.flags & zg::kFlagSchedule) return ZERO_ERR_SCHEDULE;
    if (c->stepped && c->last_clip && (st.flags & zg::kFlagNonfinite)) return ZERO_ERR_NONFINITE;
    return ZERO_OK;
}

int zero_check_report(zero_ctx* c, int64_t* site, int64_t* index) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!site || !index) return ZERO_ERR_INVALID_ARG;
    zg::Status st;
    int rc = read_status(c, &st);
    if (rc) return rc;
    *site = st.bad_site;
    *index = st.bad_index;
    return ZERO_OK;
}

int zero_checked_build(void) {
#ifdef ZERO_CHECKED
    return 1;
#else
    return 0;
#endif
}

int zero_get_step(zero_ctx* c, int64_t* t) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (!t) return ZERO_ERR_INVALID_ARG;
    if (c->sched_active) {
        DeviceGuard guard(c->device);
        if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
        return read_device_step(c, t);
    }
    *t = c->t;
    return ZERO_OK;
}

int zero_set_step(zero_ctx* c, int64_t t) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (c->sched_active) return ZERO_ERR_SCHEDULE;
    if (t < 0) return ZERO_ERR_INVALID_ARG;
    c->t = t;
    return ZERO_OK;
}

int zero_set_timing(zero_ctx* c, int on) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    c->timing = on ? 1 : 0;
    return ZERO_OK;
}

int zero_kernel_times(zero_ctx* c, double* ms, int64_t* launches) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    DeviceGuard guard(c->device);
    if (!guard.ok) return cuda_fail(cudaErrorInvalidDevice);
    double acc[ZERO_NUM_KERNELS] = {0};
    int64_t cnt[ZERO_NUM_KERNELS] = {0};
    for (size_t i = 0; i < c->n_timed; ++i) {
        zero_ctx::TimedLaunch& tl = c->events[i];
        cudaError_t e = cudaEventSynchronize(tl.stop);
        float t = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, tl.start, tl.stop);
        if (e != cudaSuccess) {
            c->n_timed = 0;
            return cuda_fail(e);
        }
        acc[tl.kernel] += (double)t;
        cnt[tl.kernel] += 1;
    }
    c->n_timed = 0;
    for (int k = 0; k < ZERO_NUM_KERNELS; ++k) {
        if (ms) ms[k] = acc[k];
        if (launches) launches[k] = cnt[k];
    }
    return ZERO_OK;
}

int zero_set_launch_overlap(zero_ctx* c, int mode) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (mode < ZERO_OVERLAP_NONE || mode > ZERO_OVERLAP_BUCKETS) return ZERO_ERR_INVALID_ARG;
    c->overlap = mode;
    c->chain_seq = ~0ull;  // nothing launched so far may be overlapped
    return ZERO_OK;
}

int zero_set_max_ctas(zero_ctx* c, int ctas) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (ctas < 0) return ZERO_ERR_INVALID_ARG;
    c->max_ctas = ctas;
    return ZERO_OK;
}

int zero_launch_shape(zero_ctx* c, int* ctas, int* threads) {
    if (!live(c)) return ZERO_ERR_BAD_CONTEXT;
    if (ctas) *ctas = grid_for(c, zg::kVarRsAdamwPlain, c->npad / 8);
    if (threads) *threads = zg::rs_adamw_threads(c->cfg.M);  // as launched
    return ZERO_OK;
}

int zero_destroy(zero_ctx* c) {
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        if (!c || !g_live.count(c)) return ZERO_ERR_BAD_CONTEXT;
        g_live.erase(c);
    }
    {
        // A context may be released while some stream is being captured into a CUDA graph
        // in global mode (for example when a garbage collector runs during the capture).
        // Releasing events is harmless to any capture, so this thread relaxes its capture
        // mode around the releases and restores it afterwards.
        cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
        const bool exchanged = cudaThreadExchangeStreamCaptureMode(&mode) == cudaSuccess;
        {
            DeviceGuard guard(c->device);
            for (auto& tl : c->events) {
                cudaEventDestroy(tl.start);
                cudaEventDestroy(tl.stop);
            }
            for (auto& g : c->grad_sets) cudaEventDestroy(g.consumed);
            if (c->h2d_done) cudaEventDestroy(c->h2d_done);
        }
        if (exchanged) cudaThreadExchangeStreamCaptureMode(&mode);
    }
    delete c;
    return ZERO_OK;
}

const char* zero_strerror(int status) {
    switch (status) {
        case ZERO_OK: return "ok";
        case ZERO_ERR_INVALID_ARG: return "invalid argument";
        case ZERO_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case ZERO_ERR_SIZE_MISMATCH: return "a buffer this configuration needs is missing";
        case ZERO_ERR_STAGE: return "stage must be 1, 2 or 3 and match the context";
        case ZERO_ERR_NONFINITE: return "non-finite gradient norm: the update was skipped";
        case ZERO_ERR_CUDA: return "CUDA runtime error (see zero_last_cuda_error)";
        case ZERO_ERR_BAD_CONTEXT: return "null, destroyed or unknown context";
        case ZERO_ERR_NOT_COMPUTED: return "value not computed by the last step";
        case ZERO_ERR_TOO_LARGE: return "layout exceeds the fixed scratch of zero_grad_norm_noalloc";
        case ZERO_ERR_DEVICE: return "a device-side bounds check failed (checked build); see zero_check_report";
        case ZERO_ERR_SCHEDULE:
            return "scheduled steps: no schedule installed, a host-step call while one is, or a step past its end";
        default: return "unknown status";
    }
}

int zero_last_cuda_error(void) { return g_last_cuda_error; }

double zero_state_bytes_per_param(int stage, int M, double param_bytes, double grad_bytes, double optim_bytes) {
    if (M < 1 || param_bytes < 0 || grad_bytes < 0 || optim_bytes < 0) return -1.0;
    switch (stage) {
        case 0: return param_bytes + grad_bytes + optim_bytes;
        case 1: return param_bytes + grad_bytes + optim_bytes / M;
        case 2: return param_bytes + (grad_bytes + optim_bytes) / M;
        case 3: return (param_bytes + grad_bytes + optim_bytes) / M;
        default: return -1.0;
    }
}

}  // extern "C"

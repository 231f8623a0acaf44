/*
 * zero_oracle.c -- plain, slow CPU oracle of the data-parallel ZeRO optimizer step:
 *   M rank-local bf16 gradient replicas -> reduce-scatter (rank-ordered fp32 sum, x 1/M)
 *   -> global gradient L2 norm and clip scale -> mixed-precision AdamW on each owner's
 *   shard -> all-gather of the updated bf16 parameters.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the package smoke check and the benchmark's
 * CPU-baseline / reference leg load this library. The GPU path never calls it, and the two
 * share no code, header, table or constant generator. Everything here is written for a
 * reader to check by eye against its sources: plain loops, one element at a time, no
 * blocking, no vectorisation, no reordering.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math (no FMA contraction, IEEE float).
 *
 * Sources, by page title and section:
 *  [L8]  "CS336 2026 Lecture 8: Parallelism Basics 与大模型并行训练" (hqhq1025.github.io
 *        ai-course-notes): Slide 8 (all-reduce = reduce-scatter + all-gather), Slide 15 (DP
 *        gradient average), Slide 17 (16 bytes/param mixed-precision Adam), Slides 19-21
 *        (ZeRO-1 four-step lifecycle), Slides 22-23 (ZeRO-2), Slides 24-26 (ZeRO-3 / FSDP).
 *  [EQ]  "并行训练优化、MoE扩展与系统瓶颈" (equinox-blog.pages.dev, CS336 notes): 1.2.2
 *        (reduce_scatter_sum / all_gather decomposition), 2.1 (DDP all_reduce AVG),
 *        2.2.1 (ZeRO-1 steps), 2.2.4 (ZeRO-2 pseudocode), 2.2.6 (ZeRO-3 pseudocode).
 *  [JZ]  "并行策略总览：六个维度各切什么、怎么通信" (blog.javazero.top), section
 *        "数据并行：切 batch" (gradient-average identity; ZeRO: computation unchanged, only
 *        where W and g are stored changes) and its collective-volume table.
 *  [231] "CS231n Lecture 11: Large-Scale Distributed Training" notes (fqmmm.github.io),
 *        4.1 (DP loss/gradient average over M GPUs), 4.3 (FSDP).
 *
 * The pages fix the structure of the step but print no optimizer formula, clip rule or
 * padding rule. This file takes these readings (each one is the plainest published form):
 *  - average = fp32 sum over ranks in order 0..M-1, starting from +0.0f, then one
 *    multiplication by inv_M = (float)(1/M)  ([EQ] 2.1 uses ReduceOp.AVG; [JZ] divides by N);
 *  - AdamW = Adam with bias correction (Kingma & Ba 2015) and decoupled weight decay applied
 *    to the previous parameter (Loshchilov & Hutter 2019), eps added after the square root;
 *    fp32 master / m / v, bf16 parameter copy (the 16 B/param ledger of [L8] Slide 17);
 *  - gradient clipping by global L2 norm (Pascanu et al. 2013): the norm of the averaged
 *    gradient, summed in fp64 in ascending flat order; scale = c/norm only when norm > c;
 *    a non-finite norm skips the update;
 *  - padding per bucket to a multiple of M*A lanes; padding lanes are zero everywhere,
 *    are excluded from the norm and never reach the unpadded parameter buffer;
 *  - buckets are filled greedily in declared tensor order, never splitting a tensor;
 *  - bf16 = IEEE round-to-nearest-even of the fp32 value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Hyper-parameters of one optimizer step.                                               */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay, max_grad_norm;
    int32_t clip; /* 1: clip by global norm at max_grad_norm; 0: no clipping */
    int32_t reserved;
} orc_hyper;

/* ------------------------------------------------------------------------------------ */
/* bf16 <-> fp32. bf16 is the upper half of an IEEE binary32.                            */
/* ------------------------------------------------------------------------------------ */
static float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16; /* widening is exact */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest, ties-to-even, of the 32-bit pattern to its upper 16 bits. Adding
 * 0x7FFF (+1 when the kept half is odd) carries into bit 16 exactly when the dropped half
 * is above one half-ulp, or equal to it with an odd kept half. A carry out of the largest
 * finite exponent lands on the infinity pattern, as IEEE rounding requires. NaN maps to the
 * quiet NaN 0x7FC0. */
static uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)0x7FC0u;
    uint32_t keep_odd = (u >> 16) & 1u;
    u += 0x7FFFu + keep_odd;
    return (uint16_t)(u >> 16);
}

void orc_bf16_rne_array(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

void orc_bf16_to_f32_array(const uint16_t* x, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(x[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Flat layout: buckets and owner shards.                                                */
/* [L8] Slide 23 / [JZ] DP section: gradients travel in buckets; a bucket is reduce-     */
/* scattered so that rank r owns slice r of it ([L8] Slide 8, [EQ] 1.2.2).               */
/*                                                                                       */
/* Bucket b holds tensors b_first[b] .. b_first[b+1]-1 contiguously, n_b real lanes,     */
/* padded to M*S_b lanes with S_b = ceil(n_b / (M*A)) * A. Bucket b starts at padded     */
/* lane b_off[b]; rank r owns lanes [b_off + r*S_b, b_off + (r+1)*S_b). A lane o of      */
/* bucket b is real iff o - b_off[b] < n_b.                                              */
/* Returns the padded length npad (sum of M*S_b).                                        */
/* ------------------------------------------------------------------------------------ */
int64_t orc_plan(int32_t M, int64_t A, int64_t bucket_bytes, const int64_t* numel, int64_t T,
                 int64_t* b_first, int64_t* b_off, int64_t* b_n, int64_t* b_S, int64_t* t_off,
                 int64_t* n_buckets)
{
    int64_t nb = 0;
    int64_t cur_bytes = 0; /* bf16 gradient bytes in the open bucket */
    for (int64_t t = 0; t < T; ++t) {
        int64_t bytes = 2 * numel[t];
        int open_new = (nb == 0) ||
                       (bucket_bytes > 0 && bytes > 0 && cur_bytes > 0 && cur_bytes + bytes > bucket_bytes);
        if (open_new) {
            b_first[nb] = t;
            b_n[nb] = 0;
            nb += 1;
            cur_bytes = 0;
        }
        t_off[t] = b_n[nb - 1]; /* position inside the bucket; made absolute below */
        b_n[nb - 1] += numel[t];
        cur_bytes += bytes;
    }
    int64_t off = 0;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t unit = (int64_t)M * A;
        b_S[b] = ((b_n[b] + unit - 1) / unit) * A;
        b_off[b] = off;
        off += (int64_t)M * b_S[b];
    }
    b_first[nb] = T;
    for (int64_t b = 0; b < nb; ++b)
        for (int64_t t = b_first[b]; t < b_first[b + 1]; ++t) t_off[t] += b_off[b];
    *n_buckets = nb;
    return off;
}

/* Per-rank shard length: the rank's slices of all buckets, concatenated in bucket order. */
static int64_t orc_shard_len(int64_t nb, const int64_t* b_S)
{
    int64_t s = 0;
    for (int64_t b = 0; b < nb; ++b) s += b_S[b];
    return s;
}

/* ------------------------------------------------------------------------------------ */
/* Gradient average of one lane over the M emulated ranks ([L8] Slide 15; [EQ] 2.1       */
/* all_reduce with ReduceOp.AVG; [JZ] DP identity grad = (1/N) sum_i g_i; [231] 4.1).    */
/* With G > 1 (hybrid sharding, [231] 4.4: M = G x K ranks, sharded inside each group of  */
/* K, replicated across the G groups), rank q = grp*K + k: each group's K values are      */
/* summed in order (the reduce-scatter inside the group), then the G group sums in order  */
/* (the all-reduce across groups), then the one multiplication by 1/M.                    */
/* ------------------------------------------------------------------------------------ */
static float orc_rank_average_grouped(int32_t M, int32_t G, const uint16_t* const* g, int64_t o)
{
    float inv_M = (float)(1.0 / (double)M);
    if (G <= 1) {
        float acc = 0.0f; /* +0: a sum of -0 replicas is +0 */
        for (int32_t r = 0; r < M; ++r) acc = acc + orc_bf16_to_f32(g[r][o]);
        return acc * inv_M;
    }
    int32_t K = M / G;
    float acc = 0.0f;
    for (int32_t grp = 0; grp < G; ++grp) {
        float part = 0.0f;
        for (int32_t k = 0; k < K; ++k) part = part + orc_bf16_to_f32(g[grp * K + k][o]);
        acc = acc + part;
    }
    return acc * inv_M;
}

static float orc_rank_average(int32_t M, const uint16_t* const* g, int64_t o)
{
    return orc_rank_average_grouped(M, 1, g, o);
}

/* ------------------------------------------------------------------------------------ */
/* Reduce-scatter ([L8] Slide 20 step 2; [EQ] 2.2.1 step 2, reduce_scatter_sum): owner r  */
/* receives, for each lane of its shard, the average over ranks. Padding lanes get +0.    */
/* grads[q] is rank q's full padded gradient; ghat[r] is owner r's shard. K owners, M     */
/* ranks in G groups (K = M, G = 1 without hybrid sharding).                              */
/* ------------------------------------------------------------------------------------ */
static void orc_rs(int32_t K, int32_t M, int32_t G, int64_t nb, const int64_t* b_off, const int64_t* b_n,
                   const int64_t* b_S, const uint16_t* const* grads, float* const* ghat)
{
    for (int32_t r = 0; r < K; ++r) {
        int64_t base = 0; /* start of bucket b's slice inside rank r's shard */
        for (int64_t b = 0; b < nb; ++b) {
            for (int64_t j = 0; j < b_S[b]; ++j) {
                int64_t in_bucket = (int64_t)r * b_S[b] + j;
                int64_t o = b_off[b] + in_bucket;
                ghat[r][base + j] = (in_bucket < b_n[b]) ? orc_rank_average_grouped(M, G, grads, o) : 0.0f;
            }
            base += b_S[b];
        }
    }
}

void orc_reduce_scatter(int32_t M, int64_t nb, const int64_t* b_off, const int64_t* b_n,
                        const int64_t* b_S, const uint16_t* const* grads, float* const* ghat)
{
    orc_rs(M, M, 1, nb, b_off, b_n, b_S, grads, ghat);
}

/* ------------------------------------------------------------------------------------ */
/* Global L2 norm of the averaged gradient, squares summed in fp64 in ascending flat     */
/* order over real lanes (the flat order visits bucket, then owner, then lane). In a     */
/* multi-GPU run this is one scalar all-reduce of the per-owner partial sums.            */
/* ------------------------------------------------------------------------------------ */
double orc_global_sumsq(int32_t M, int64_t nb, const int64_t* b_n, const int64_t* b_S,
                        const float* const* ghat)
{
    double acc = 0.0;
    int64_t base = 0;
    for (int64_t b = 0; b < nb; ++b) {
        for (int32_t r = 0; r < M; ++r) {
            for (int64_t j = 0; j < b_S[b]; ++j) {
                if ((int64_t)r * b_S[b] + j < b_n[b]) {
                    double x = (double)ghat[r][base + j];
                    acc += x * x;
                }
            }
        }
        base += b_S[b];
    }
    return acc;
}

/* The same sum taken straight from the rank gradients, over flat lanes [o0, o0+len), for
 * workloads whose averaged gradient is too large to hold on the host. grads[q] points at
 * lane o0 of rank q. Continuing from acc over consecutive chunks gives the very same
 * sequence of fp64 additions as orc_global_sumsq over the whole layout. */
double orc_sumsq_chunk(double acc, int32_t M, const uint16_t* const* grads, int64_t o0,
                       int64_t len, int64_t nb, const int64_t* b_off, const int64_t* b_n)
{
    if (nb <= 0) return acc;
    int64_t b = 0;
    for (int64_t i = 0; i < len; ++i) {
        int64_t o = o0 + i;
        while (b + 1 < nb && o >= b_off[b + 1]) ++b;
        while (b > 0 && o < b_off[b]) --b;
        if (o - b_off[b] < b_n[b]) {
            double x = (double)orc_rank_average(M, grads, i);
            acc += x * x;
        }
    }
    return acc;
}

/* Clip scale from the global norm: c / norm when norm exceeds c, else exactly 1. */
float orc_clip_scale(double norm, double max_grad_norm)
{
    if (norm > max_grad_norm) return (float)(max_grad_norm / norm);
    return 1.0f;
}

/* ------------------------------------------------------------------------------------ */
/* AdamW, fp32 state ([L8] Slide 17: fp32 master, Adam m and v beside the bf16 copy).     */
/* Step-constant scalars are formed in double and rounded once to float.                  */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    float b1, b2, c1, c2, step_size, inv_sqrt_bc2, decay, eps;
} orc_adamw_consts;

static orc_adamw_consts orc_adamw_scalars(const orc_hyper* h, int64_t t)
{
    orc_adamw_consts k;
    double bc1 = 1.0 - pow(h->beta1, (double)t); /* bias corrections of step t */
    double bc2 = 1.0 - pow(h->beta2, (double)t);
    k.b1 = (float)h->beta1;
    k.b2 = (float)h->beta2;
    k.c1 = (float)(1.0 - h->beta1);
    k.c2 = (float)(1.0 - h->beta2);
    k.step_size = (float)(h->lr / bc1);
    k.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    k.decay = (float)(1.0 - h->lr * h->weight_decay);
    k.eps = (float)h->eps;
    return k;
}

/* One lane: g = s*ghat; m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
 * p <- p (1 - lr wd) - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps). */
static void orc_adamw_lane(float ghat, float s, float* p, float* m, float* v,
                           const orc_adamw_consts* k)
{
    float g = s * ghat;
    float m1 = k->b1 * (*m) + k->c1 * g;
    float v1 = k->b2 * (*v) + k->c2 * (g * g);
    float den = sqrtf(v1) * k->inv_sqrt_bc2 + k->eps;
    float p1 = (*p) * k->decay - k->step_size * (m1 / den);
    *m = m1;
    *v = v1;
    *p = p1;
}

/* AdamW over one flat array of n lanes (an owner's shard, or a full replica). */
void orc_adamw(int64_t n, const float* ghat, float s, float* p, float* m, float* v,
               const orc_hyper* h, int64_t t)
{
    orc_adamw_consts k = orc_adamw_scalars(h, t);
    for (int64_t i = 0; i < n; ++i) orc_adamw_lane(ghat[i], s, &p[i], &m[i], &v[i], &k);
}

/* ------------------------------------------------------------------------------------ */
/* Initial state. master_init is the unpadded fp32 parameter vector (N values); m_init and */
/* v_init are the unpadded Adam moments, or NULL for zeros (a fresh start). Every rank's   */
/* optimizer state is its shard of the padded layout; padding lanes are 0.               */
/* Stages 1 and 2 keep a full bf16 replica per rank (N values); stage 3 keeps a bf16      */
/* shard per rank ([L8] Slides 19, 22, 24; [EQ] 2.2.1, 2.2.3, 2.2.5).                     */
/* ------------------------------------------------------------------------------------ */
void orc_init(int32_t M, int32_t stage, int64_t nb, const int64_t* b_n, const int64_t* b_S,
              const float* master_init, const float* m_init, const float* v_init,
              float* const* master, float* const* mom, float* const* var, uint16_t* const* param)
{
    int64_t slen = orc_shard_len(nb, b_S);
    for (int32_t r = 0; r < M; ++r) {
        int64_t base = 0, ubase = 0;
        for (int64_t b = 0; b < nb; ++b) {
            for (int64_t j = 0; j < b_S[b]; ++j) {
                int64_t in_bucket = (int64_t)r * b_S[b] + j;
                int real = in_bucket < b_n[b];
                int64_t u = ubase + in_bucket;
                master[r][base + j] = real ? master_init[u] : 0.0f;
                mom[r][base + j] = (real && m_init) ? m_init[u] : 0.0f;
                var[r][base + j] = (real && v_init) ? v_init[u] : 0.0f;
            }
            base += b_S[b];
            ubase += b_n[b];
        }
        if (stage == 3) {
            for (int64_t i = 0; i < slen; ++i) param[r][i] = orc_f32_to_bf16(master[r][i]);
        } else {
            for (int64_t u = 0; u < ubase; ++u) param[r][u] = orc_f32_to_bf16(master_init[u]);
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* All-gather ([L8] Slide 20 step 4; [EQ] 1.2.2 all_gather, 2.2.1 step 4): receiver q      */
/* gets every owner r's bf16 shard at its unpadded place; padding never leaves the owner.  */
/* shard_bf16[r] is owner r's bf16 shard; dst is q's full buffer (N values).               */
/* ------------------------------------------------------------------------------------ */
static void orc_all_gather(int32_t M, int64_t nb, const int64_t* b_n, const int64_t* b_S,
                           const uint16_t* const* shard_bf16, uint16_t* dst)
{
    for (int32_t r = 0; r < M; ++r) {
        int64_t base = 0, ubase = 0;
        for (int64_t b = 0; b < nb; ++b) {
            for (int64_t j = 0; j < b_S[b]; ++j) {
                int64_t in_bucket = (int64_t)r * b_S[b] + j;
                if (in_bucket < b_n[b]) dst[ubase + in_bucket] = shard_bf16[r][base + j];
            }
            base += b_S[b];
            ubase += b_n[b];
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* One ZeRO step over M separate rank structures.                                         */
/*  grads[q]   rank q's bf16 gradient, padded layout (npad lanes)                         */
/*  master/mom/var/ghat[r]  owner r's fp32 shards (shard_len lanes)                        */
/*  param[r]   stage 1/2: rank r's full bf16 replica (N); stage 3: its bf16 shard          */
/*  full_out   N bf16 values: the parameters every rank holds after the all-gather         */
/*  t          1-based step index used for bias correction                                */
/* Returns 0, or 1 when clipping is on and the norm is not finite (state left untouched), */
/* or -1 when the M gathered replicas disagree.                                           */
/* ------------------------------------------------------------------------------------ */
/* The step of one sharding group: K owners (and K receivers of the all-gather); the    */
/* average runs over M ranks in G groups.                                                 */
static int orc_step_core(int32_t K, int32_t Mtot, int32_t G, int32_t stage, int64_t nb, const int64_t* b_off,
                         const int64_t* b_n, const int64_t* b_S, const uint16_t* const* grads,
                         float* const* master, float* const* mom, float* const* var,
                         float* const* ghat, uint16_t* const* param, uint16_t* full_out,
                         const orc_hyper* h, int64_t t, double* norm_out, float* scale_out)
{
    const int32_t M = K; /* owners and receivers of this group */
    int64_t slen = orc_shard_len(nb, b_S);
    int64_t N = 0;
    for (int64_t b = 0; b < nb; ++b) N += b_n[b];

    /* (2) reduce-scatter: every owner receives the averaged gradient of its shard. */
    orc_rs(K, Mtot, G, nb, b_off, b_n, b_S, grads, ghat);

    /* norm and clip scale */
    double norm = sqrt(orc_global_sumsq(M, nb, b_n, b_S, (const float* const*)ghat));
    *norm_out = norm;
    float s = 1.0f;
    int skipped = 0;
    if (h->clip) {
        if (!isfinite(norm)) skipped = 1;
        else s = orc_clip_scale(norm, h->max_grad_norm);
    }
    *scale_out = s;

    /* (3) each owner updates its shard with its own optimizer state. */
    uint16_t** shard_bf16 = (uint16_t**)malloc(sizeof(uint16_t*) * (size_t)M);
    for (int32_t r = 0; r < M; ++r) {
        if (!skipped) orc_adamw(slen, ghat[r], s, master[r], mom[r], var[r], h, t);
        if (stage == 3) {
            if (!skipped)
                for (int64_t i = 0; i < slen; ++i) param[r][i] = orc_f32_to_bf16(master[r][i]);
            shard_bf16[r] = param[r]; /* the persistent bf16 shard */
        } else {
            shard_bf16[r] = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(slen > 0 ? slen : 1));
            for (int64_t i = 0; i < slen; ++i) shard_bf16[r][i] = orc_f32_to_bf16(master[r][i]);
        }
    }

    /* (4) all-gather: every rank rebuilds the full parameters from all owners. */
    int rc = skipped ? 1 : 0;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(N > 0 ? N : 1));
    for (int32_t q = 0; q < M; ++q) {
        uint16_t* dst = (stage == 3) ? tmp : param[q];
        if (!(stage != 3 && skipped)) orc_all_gather(M, nb, b_n, b_S, (const uint16_t* const*)shard_bf16, dst);
        if (q == 0) memcpy(full_out, dst, sizeof(uint16_t) * (size_t)N);
        else if (memcmp(full_out, dst, sizeof(uint16_t) * (size_t)N) != 0) rc = -1;
    }
    free(tmp);
    if (stage != 3)
        for (int32_t r = 0; r < M; ++r) free(shard_bf16[r]);
    free(shard_bf16);
    return rc;
}

int orc_zero_step(int32_t M, int32_t stage, int64_t nb, const int64_t* b_off,
                  const int64_t* b_n, const int64_t* b_S, const uint16_t* const* grads,
                  float* const* master, float* const* mom, float* const* var,
                  float* const* ghat, uint16_t* const* param, uint16_t* full_out,
                  const orc_hyper* h, int64_t t, double* norm_out, float* scale_out)
{
    return orc_step_core(M, M, 1, stage, nb, b_off, b_n, b_S, grads, master, mom, var, ghat, param, full_out,
                         h, t, norm_out, scale_out);
}

/* ------------------------------------------------------------------------------------ */
/* Hybrid sharded data parallelism ([231] 4.4): M = G x K ranks; the state is sharded over */
/* the K ranks of each group (the layout b_off / b_S is planned for K owners) and every   */
/* group holds a replica of it. The rank structures are G x K: structure grp*K + k is     */
/* owner k of group grp. Each group runs the ZeRO step on the average over all M ranks    */
/* (reduce-scatter inside the group, all-reduce of the shard across groups); the G        */
/* replicas must agree. Returns 0, 1 (skipped, non-finite norm) or -1 (replicas differ).  */
/* ------------------------------------------------------------------------------------ */
int orc_hsdp_step(int32_t G, int32_t K, int32_t stage, int64_t nb, const int64_t* b_off,
                  const int64_t* b_n, const int64_t* b_S, const uint16_t* const* grads,
                  float* const* master, float* const* mom, float* const* var,
                  float* const* ghat, uint16_t* const* param, uint16_t* full_out,
                  const orc_hyper* h, int64_t t, double* norm_out, float* scale_out)
{
    int64_t N = 0;
    for (int64_t b = 0; b < nb; ++b) N += b_n[b];
    uint16_t* other = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(N > 0 ? N : 1));
    int rc = 0;
    for (int32_t grp = 0; grp < G; ++grp) {
        double norm;
        float s;
        uint16_t* dst = grp == 0 ? full_out : other;
        int r = orc_step_core(K, G * K, G, stage, nb, b_off, b_n, b_S, grads, master + grp * K, mom + grp * K,
                              var + grp * K, ghat + grp * K, param + grp * K, dst, h, t, &norm, &s);
        if (grp == 0) {
            *norm_out = norm;
            *scale_out = s;
            rc = r;
        } else if (r != rc || memcmp(dst, full_out, sizeof(uint16_t) * (size_t)N) != 0 ||
                   !(norm == *norm_out || (norm != norm && *norm_out != *norm_out)) || s != *scale_out) {
            rc = -1;
        }
    }
    free(other);
    return rc;
}

/* ------------------------------------------------------------------------------------ */
/* Naive data parallelism ([L8] Slides 15-16; [EQ] 2.1 pseudocode): every rank holds the  */
/* full unpadded state, all-reduces (averages) the full gradient and runs the same AdamW  */
/* on all N lanes. grads[q] is rank q's UNPADDED gradient (N values). The replicas must   */
/* agree; ZeRO must reproduce them exactly ([L8] Slide 19: "mathematically still data     */
/* parallel"; [JZ]: the computation does not change, only where W and g are stored).      */
/* Returns 0, 1 (non-finite norm, skipped) or -1 (replicas disagree).                      */
/* ------------------------------------------------------------------------------------ */
int orc_naive_dp_step_groups(int32_t M, int32_t G, int64_t N, const uint16_t* const* grads,
                             float* const* master, float* const* mom, float* const* var,
                             uint16_t* const* param, const orc_hyper* h, int64_t t, double* norm_out,
                             float* scale_out)
{
    float* gbar = (float*)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1));
    int rc = 0;
    for (int32_t q = 0; q < M; ++q) {
        for (int64_t u = 0; u < N; ++u) gbar[u] = orc_rank_average_grouped(M, G, grads, u); /* all-reduce */
        double acc = 0.0;
        for (int64_t u = 0; u < N; ++u) acc += (double)gbar[u] * (double)gbar[u];
        double norm = sqrt(acc);
        float s = 1.0f;
        int skipped = 0;
        if (h->clip) {
            if (!isfinite(norm)) skipped = 1;
            else s = orc_clip_scale(norm, h->max_grad_norm);
        }
        if (!skipped) {
            orc_adamw(N, gbar, s, master[q], mom[q], var[q], h, t);
            for (int64_t u = 0; u < N; ++u) param[q][u] = orc_f32_to_bf16(master[q][u]);
        }
        if (q == 0) {
            *norm_out = norm;
            *scale_out = s;
            rc = skipped;
        } else if (memcmp(master[q], master[0], sizeof(float) * (size_t)N) != 0 ||
                   memcmp(param[q], param[0], sizeof(uint16_t) * (size_t)N) != 0) {
            rc = -1;
        }
    }
    free(gbar);
    return rc;
}

int orc_naive_dp_step(int32_t M, int64_t N, const uint16_t* const* grads, float* const* master,
                      float* const* mom, float* const* var, uint16_t* const* param,
                      const orc_hyper* h, int64_t t, double* norm_out, float* scale_out)
{
    return orc_naive_dp_step_groups(M, 1, N, grads, master, mom, var, param, h, t, norm_out, scale_out);
}

/* ------------------------------------------------------------------------------------ */
/* Per-lane trajectories for sampled checks of large layouts. For L sampled lanes and K   */
/* consecutive steps starting at step index t0:                                          */
/*   g[(k*M + r)*L + i]  rank r's bf16 gradient at lane i in step k                      */
/*   real[i]             1 for a real lane, 0 for a padding lane (gradient treated as 0) */
/*   scale[k], apply[k]  the clip scale of step k and whether step k updates (0 = the    */
/*                       step was skipped for a non-finite norm)                         */
/*   p/m/v[i]            in: state before the first step; out: after the last            */
/*   bf[i]               out: the bf16 parameter                                         */
/*   ghat_out[k*L + i]   out (may be NULL): the averaged gradient of step k               */
/* ------------------------------------------------------------------------------------ */
void orc_lane_steps(int32_t M, int64_t L, int32_t K, const uint16_t* g, const uint8_t* real,
                    const float* scale, const uint8_t* apply, const orc_hyper* h, int64_t t0,
                    float* p, float* m, float* v, uint16_t* bf, float* ghat_out)
{
    const uint16_t** rows = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)M);
    for (int32_t k = 0; k < K; ++k) {
        orc_adamw_consts c = orc_adamw_scalars(h, t0 + k);
        for (int32_t r = 0; r < M; ++r) rows[r] = g + ((int64_t)k * M + r) * L;
        for (int64_t i = 0; i < L; ++i) {
            float gh = real[i] ? orc_rank_average(M, rows, i) : 0.0f;
            if (ghat_out) ghat_out[(int64_t)k * L + i] = gh;
            if (apply[k]) orc_adamw_lane(gh, scale[k], &p[i], &m[i], &v[i], &c);
        }
    }
    for (int64_t i = 0; i < L; ++i) bf[i] = orc_f32_to_bf16(p[i]);
    free(rows);
}

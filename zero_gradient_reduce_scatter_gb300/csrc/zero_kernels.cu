// zero_kernels.cu -- sm_103a kernels of the ZeRO optimizer step.
//
// Everything here is HBM-bandwidth bound: per lane the step moves 2M bytes of bf16
// gradient, 12 bytes of fp32 state in and 12 out, and 2 bytes of bf16 parameter out, for
// about 10 flops. There is no contraction, so no tensor cores: the kernels are grid-stride
// streams of 16-byte vector accesses with evict-first cache hints, one "vec" of 8 lanes
// (16 B of bf16, 32 B of fp32) per thread per iteration, grids of (SMs x resident CTAs).
//
// Reduction order is fixed so that results are bit-identical to a plain CPU evaluation:
// the M rank values of a lane are added in rank order 0..M-1 to a +0.0f accumulator,
// multiplied once by (float)(1/M), and every AdamW operation is an explicitly rounded
// IEEE operation (__fadd_rn, __fmul_rn, __fsqrt_rn, __fdiv_rn), so nvcc cannot contract
// any of them into an FMA.
//
// Sources: "CS336 2026 Lecture 8" notes, Slides 8 and 19-26 (reduce-scatter, owner update,
// all-gather; ZeRO stages); "并行训练优化、MoE扩展与系统瓶颈" 1.2.2 and 2.2.1-2.2.6.

#include <cuda_bf16.h>

#include <utility>

#include "zero_internal.h"

namespace zg {
namespace {

// ---------------------------------------------------------------------------------------
// Checked builds (-DZERO_CHECKED): before each global access group the kernels test the
// index against the bounds of its buffer; a failing test records (site, index) in the
// status word, raises kFlagBounds and skips the access -- no trap, the context stays usable.
// Normal builds compile the tests to `true`, i.e. to nothing.
// ---------------------------------------------------------------------------------------
#ifdef ZERO_CHECKED
__device__ __noinline__ bool zg_bounds_fail(Status* st, int site, int64_t idx) {
    if (atomicCAS(reinterpret_cast<unsigned long long*>(&st->bad_site), 0ull, (unsigned long long)site) == 0ull)
        st->bad_index = idx;
    atomicOr(&st->flags, kFlagBounds);
    return false;
}
#define ZG_OK(st, cond, site, idx) ((cond) ? true : zg_bounds_fail((st), (site), (int64_t)(idx)))
#else
#define ZG_OK(st, cond, site, idx) true
#endif
// check sites
enum : int {
    kSiteGradNorm = 1, kSiteGhatWrite, kSitePartial, kSiteStepLanes, kSiteParamFull, kSiteGhatRead,
    kSiteGatherSrc, kSiteGatherOut, kSiteInit, kSiteSave, kSiteFinalCount
};

// ---------------------------------------------------------------------------------------
// bf16 helpers: bf16 is the upper half of a binary32, so widening is a shift.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two bf16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Streaming (evict-first) vector accesses.
__device__ __forceinline__ uint4 ld_u4(const uint16_t* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
// Read-only path without L1 allocation, for gradients no kernel writes.
__device__ __forceinline__ uint4 ld_u4_nc(const uint16_t* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}
template <int PATH>
__device__ __forceinline__ uint4 ld_grad(const uint16_t* p) {
    if constexpr (PATH == kLoadNonCoherent) return ld_u4_nc(p);
    else if constexpr (PATH == kLoadReadOnly) return __ldg(reinterpret_cast<const uint4*>(p));
    else return ld_u4(p);
}
// fp32 vector accesses under a cache policy (CachePolicy; chosen per kernel by measurement).
template <int P>
__device__ __forceinline__ float4 ld_f4(const float* p) {
    const float4* q = reinterpret_cast<const float4*>(p);
    if constexpr (P == kCacheStreaming) return __ldcs(q);
    else if constexpr (P == kCacheAllLevels) return __ldca(q);
    else if constexpr (P == kCacheGlobal) return __ldcg(q);
    else return *q;
}
// 16-byte bf16 accesses under a cache policy (the gather's).
template <int P>
__device__ __forceinline__ uint4 ld_u4p(const uint16_t* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    if constexpr (P == kCacheStreaming) return __ldcs(q);
    else if constexpr (P == kCacheAllLevels) return __ldca(q);
    else if constexpr (P == kCacheGlobal) return __ldcg(q);
    else return *q;
}
template <int P>
__device__ __forceinline__ void st_u4p(uint16_t* p, uint4 x) {
    uint4* q = reinterpret_cast<uint4*>(p);
    if constexpr (P == kCacheStreaming) __stcs(q, x);
    else if constexpr (P == kCacheGlobal) __stcg(q, x);
    else *q = x;
}
template <int P>
__device__ __forceinline__ void st_f4(float* p, float4 x) {
    float4* q = reinterpret_cast<float4*>(p);
    if constexpr (P == kCacheStreaming) __stcs(q, x);
    else if constexpr (P == kCacheGlobal) __stcg(q, x);
    else *q = x;
}
__device__ __forceinline__ void st_u4(uint16_t* p, uint4 x) { __stcs(reinterpret_cast<uint4*>(p), x); }

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch (kernels launched with programmatic stream serialization,
// which may start while the kernel before them on the stream is still running).
// kPdlWaitFirst: griddepcontrol.wait (the preceding grid complete, its writes visible)
// before any memory access, then let the next such kernel launch. kPdlWaitLast: let the
// next kernel launch at once, do the work, and wait only before exiting, so that the
// kernel still completes after its predecessor. kPdlTriggerWait: let the next kernel launch
// at once, then wait before any memory access (for a kernel whose successor does not depend
// on it). The destructor runs the exit wait on every return path. ON = false compiles to
// nothing (the kernels of ordinary launches).
// ---------------------------------------------------------------------------------------
template <bool ON>
struct PdlScope {
    const int32_t mode;
    __device__ __forceinline__ explicit PdlScope(int32_t m) : mode(ON ? m : (int32_t)kPdlNone) {
        if (ON && mode == kPdlWaitFirst) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (ON && mode != kPdlNone) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (ON && mode == kPdlTriggerWait) asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    __device__ __forceinline__ ~PdlScope() {
        if (ON && mode == kPdlWaitLast) asm volatile("griddepcontrol.wait;" ::: "memory");
    }
};

// ---------------------------------------------------------------------------------------
// Bucket cursor: which bucket a (non-decreasing) lane index falls in.
// ---------------------------------------------------------------------------------------
struct Cursor {
    const Bucket* tab;
    int64_t nb;
    int64_t b;
    Bucket e;

    // Last bucket whose padded start is <= lane (empty buckets share their successor's start),
    // searched among buckets [first, end) (end <= 0: all); a launch over one bucket passes
    // just that one, and its threads then need no search of the table.
    __device__ __forceinline__ void init(const Bucket* t, int64_t n, int64_t lane, int64_t first = 0,
                                         int64_t end = 0) {
        tab = t;
        nb = n;
        int64_t lo = first, hi = (end > 0 ? end : n) - 1;
        while (lo < hi) {
            int64_t mid = (lo + hi + 1) >> 1;
            if (tab[mid].off <= lane) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
        e = tab[b];
    }
    __device__ __forceinline__ void seek(int64_t lane) {
        while (lane >= e.end && b + 1 < nb) {
            ++b;
            e = tab[b];
        }
    }
    // Real lanes of the vec starting at lane o (0..8).
    __device__ __forceinline__ int nreal(int64_t o) const {
        int64_t r = e.off + e.n - o;
        return r <= 0 ? 0 : (r >= 8 ? 8 : (int)r);
    }
};

// ---------------------------------------------------------------------------------------
// Reduce-scatter of one vec: acc[i] = sum over ranks (in order) of the bf16 values at
// gradient index g (the lane, less the first lane of the gradient buffers).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void add8(float acc[8], uint4 q) {
    acc[0] = __fadd_rn(acc[0], bf_lo(q.x));
    acc[1] = __fadd_rn(acc[1], bf_hi(q.x));
    acc[2] = __fadd_rn(acc[2], bf_lo(q.y));
    acc[3] = __fadd_rn(acc[3], bf_hi(q.y));
    acc[4] = __fadd_rn(acc[4], bf_lo(q.z));
    acc[5] = __fadd_rn(acc[5], bf_hi(q.z));
    acc[6] = __fadd_rn(acc[6], bf_lo(q.w));
    acc[7] = __fadd_rn(acc[7], bf_hi(q.w));
}

// Hybrid sharding: rank q = grp * K + k; each group's K values summed in order (the
// reduce-scatter inside the group), then the group sums in order (the all-reduce of the
// shard across groups). The ranks are loaded four at a time across group boundaries, so
// small groups do not serialise the load latency; a group's partial sum (from +0) is added
// to the total when its last rank has been added.
template <int PATH>
__device__ __forceinline__ void rank_sum_grouped(const StepArgs& a, int64_t g, float acc[8]) {
    const int K = a.M / a.groups;
    float part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) part[i] = 0.0f;
    int kin = 0;
    auto take = [&](uint4 q) {
        add8(part, q);
        if (++kin == K) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[i] = __fadd_rn(acc[i], part[i]);
                part[i] = 0.0f;
            }
            kin = 0;
        }
    };
    int r = 0;
    for (; r + 4 <= a.M; r += 4) {
        const uint4 q0 = ld_grad<PATH>(a.grads[r] + g), q1 = ld_grad<PATH>(a.grads[r + 1] + g);
        const uint4 q2 = ld_grad<PATH>(a.grads[r + 2] + g), q3 = ld_grad<PATH>(a.grads[r + 3] + g);
        take(q0);
        take(q1);
        take(q2);
        take(q3);
    }
    for (; r < a.M; ++r) take(ld_grad<PATH>(a.grads[r] + g));
}

// The same order with a compile-time rank count: all MT loads are issued first (as in the
// plain kernels), then the values are added group by group.
template <int MT, int PATH>
__device__ __forceinline__ void rank_sum_grouped_fixed(const StepArgs& a, int64_t g, float acc[8]) {
    constexpr int CH = MT < 8 ? MT : 8;  // loads in flight at once (bounds the registers)
    uint4 q[CH];
    const int K = MT / a.groups;
    float part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) part[i] = 0.0f;
    int kin = 0;
#pragma unroll
    for (int r = 0; r < MT; ++r) {
        if (r % CH == 0) {
#pragma unroll
            for (int j = 0; j < CH; ++j) q[j] = ld_grad<PATH>(a.grads[r + j] + g);
        }
        add8(part, q[r % CH]);
        // branch-free group flush: compute, then select (a branch here would keep the
        // compiler from issuing later loads early)
        const bool last = ++kin == K;
        kin = last ? 0 : kin;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float t = __fadd_rn(acc[i], part[i]);
            acc[i] = last ? t : acc[i];
            part[i] = last ? 0.0f : part[i];
        }
    }
}

// fp32 sources (process-per-rank hybrid sharding: the G group partials of this rank's
// shard, gathered across groups): a.M sources, each read as fp32 at lane g, added in source
// order -- the all-reduce across groups in a fixed order.
__device__ __forceinline__ void rank_sum_f32(const StepArgs& a, int64_t g, float acc[8]) {
    for (int r = 0; r < a.M; ++r) {
        const float* p = reinterpret_cast<const float*>(a.grads[r]) + g;
        const float4 x0 = __ldg(reinterpret_cast<const float4*>(p)), x1 = __ldg(reinterpret_cast<const float4*>(p + 4));
        acc[0] = __fadd_rn(acc[0], x0.x);
        acc[1] = __fadd_rn(acc[1], x0.y);
        acc[2] = __fadd_rn(acc[2], x0.z);
        acc[3] = __fadd_rn(acc[3], x0.w);
        acc[4] = __fadd_rn(acc[4], x1.x);
        acc[5] = __fadd_rn(acc[5], x1.y);
        acc[6] = __fadd_rn(acc[6], x1.z);
        acc[7] = __fadd_rn(acc[7], x1.w);
    }
}

// Exchange-layout sources (process-per-rank mode): a.grads[0] is the exchange buffer, in
// which source q's slice of local bucket e sits at lanes [M*e.off + q*S, +S), S = e.end - e.off
// (the bucket's global start is M times its local start). So local lane g of bucket e reads
// source q at g + (M-1)*e.off + q*S, and one launch covers every bucket of the shard.
template <int MT, int PATH>
__device__ __forceinline__ void rank_sum_exchange(const StepArgs& a, const Bucket& e, int64_t g, float acc[8]) {
    const int M = MT > 0 ? MT : a.M;
    const int64_t S = e.end - e.off;
    const uint16_t* p = a.grads[0] + g + (int64_t)(M - 1) * e.off;
    if constexpr (MT > 0) {
        uint4 q[MT];
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_grad<PATH>(p + r * S);
#pragma unroll
        for (int r = 0; r < MT; ++r) add8(acc, q[r]);
    } else {
        int r = 0;
        for (; r + 4 <= M; r += 4) {
            uint4 q0 = ld_grad<PATH>(p + r * S), q1 = ld_grad<PATH>(p + (r + 1) * S);
            uint4 q2 = ld_grad<PATH>(p + (r + 2) * S), q3 = ld_grad<PATH>(p + (r + 3) * S);
            add8(acc, q0);
            add8(acc, q1);
            add8(acc, q2);
            add8(acc, q3);
        }
        for (; r < M; ++r) add8(acc, ld_grad<PATH>(p + r * S));
    }
}

// Where the sources of a kernel live (a compile-time choice, so the plain kernels are
// unchanged): M bf16 buffers addressed by lane, M fp32 buffers addressed by lane, or the
// exchange buffer of the process-per-rank mode.
enum SrcMode : int { kSrcRanks = 0, kSrcF32 = 1, kSrcExchange = 2 };

// Checked builds: lane g's eight sources lie inside the source buffers (exchange layout: the
// farthest source lane of bucket e is below M * e.end).
template <int SRC>
__device__ __forceinline__ bool src_in_range(const StepArgs& a, const Bucket& e, int64_t g) {
    if constexpr (SRC == kSrcExchange) return g >= e.off && g + 8 <= e.end && (int64_t)a.M * e.end <= a.gext;
    else return g >= 0 && g + 8 <= a.gext;
}

// GROUPED selects the hybrid-sharding order at compile time, so the plain kernels carry no
// branch that would keep the compiler from issuing the state loads beside the gradient loads.
// SRC: the sources (SrcMode); e is the bucket of lane g (used by the exchange layout).
template <int MT, int PATH, bool GROUPED, int SRC = kSrcRanks>
__device__ __forceinline__ void rank_sum(const StepArgs& a, const Bucket& e, int64_t g, float acc[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;  // +0: a sum of -0 replicas is +0
    if constexpr (SRC == kSrcF32) {
        rank_sum_f32(a, g, acc);
    } else if constexpr (SRC == kSrcExchange) {
        rank_sum_exchange<MT, PATH>(a, e, g, acc);
    } else if constexpr (GROUPED && MT > 0) {
        rank_sum_grouped_fixed<MT, PATH>(a, g, acc);
    } else if constexpr (GROUPED) {
        rank_sum_grouped<PATH>(a, g, acc);
    } else if constexpr (MT > 0) {
        uint4 q[MT];
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_grad<PATH>(a.grads[r] + g);
#pragma unroll
        for (int r = 0; r < MT; ++r) add8(acc, q[r]);
    } else {
        int r = 0;
        for (; r + 4 <= a.M; r += 4) {
            uint4 q0 = ld_grad<PATH>(a.grads[r] + g), q1 = ld_grad<PATH>(a.grads[r + 1] + g);
            uint4 q2 = ld_grad<PATH>(a.grads[r + 2] + g), q3 = ld_grad<PATH>(a.grads[r + 3] + g);
            add8(acc, q0);
            add8(acc, q1);
            add8(acc, q2);
            add8(acc, q3);
        }
        for (; r < a.M; ++r) add8(acc, ld_grad<PATH>(a.grads[r] + g));
    }
}

// Averaged gradient of the vec; padding lanes are +0 whatever the buffers hold.
__device__ __forceinline__ void average8(const float acc[8], float inv_M, int nreal, float gh[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) gh[i] = (i < nreal) ? __fmul_rn(acc[i], inv_M) : 0.0f;
}

// ---------------------------------------------------------------------------------------
// AdamW of one lane (decoupled weight decay, bias correction; eps after the square root).
// ---------------------------------------------------------------------------------------
template <bool SCALE>
__device__ __forceinline__ void adam_lane(float gh, float s, float& p, float& m, float& v,
                                          const AdamConsts& k) {
    const float g = SCALE ? __fmul_rn(s, gh) : gh;
    const float m1 = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.c1, g));
    const float v1 = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.c2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(v1), k.isb), k.eps);
    p = __fsub_rn(__fmul_rn(p, k.decay), __fmul_rn(k.step, __fdiv_rn(m1, den)));
    m = m1;
    v = v1;
}

template <bool SCALE>
__device__ __forceinline__ void adam_vec(const float gh[8], float s, float p[8], float m[8], float v[8],
                                         const AdamConsts& k) {
#pragma unroll
    for (int i = 0; i < 8; ++i) adam_lane<SCALE>(gh[i], s, p[i], m[i], v[i], k);
}

__device__ __forceinline__ void unpack(float4 a, float4 b, float x[8]) {
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <int P>
__device__ __forceinline__ void load_state(const StepArgs& a, int64_t o, float p[8], float m[8], float v[8]) {
    float4 p0 = ld_f4<P>(a.master + o), p1 = ld_f4<P>(a.master + o + 4);
    float4 m0 = ld_f4<P>(a.m + o), m1 = ld_f4<P>(a.m + o + 4);
    float4 v0 = ld_f4<P>(a.v + o), v1 = ld_f4<P>(a.v + o + 4);
    unpack(p0, p1, p);
    unpack(m0, m1, m);
    unpack(v0, v1, v);
}

template <int P>
__device__ __forceinline__ void store_state(const StepArgs& a, int64_t o, const float p[8], const float m[8],
                                            const float v[8]) {
    st_f4<P>(a.master + o, make_float4(p[0], p[1], p[2], p[3]));
    st_f4<P>(a.master + o + 4, make_float4(p[4], p[5], p[6], p[7]));
    st_f4<P>(a.m + o, make_float4(m[0], m[1], m[2], m[3]));
    st_f4<P>(a.m + o + 4, make_float4(m[4], m[5], m[6], m[7]));
    st_f4<P>(a.v + o, make_float4(v[0], v[1], v[2], v[3]));
    st_f4<P>(a.v + o + 4, make_float4(v[4], v[5], v[6], v[7]));
}

// ---------------------------------------------------------------------------------------
// All-gather epilogue: the owner writes its updated bf16 values either into its padded
// shard (ZeRO-3 shard mode) or straight to their place in the unpadded full buffer.
// The unpadded address of a vec is shifted by the padding of earlier buckets, so its
// alignment is that of (u0 mod 8): the widest aligned stores are used.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void store_params(const StepArgs& a, const Cursor& c, int64_t o, int nreal,
                                             const float p[8]) {
    const uint32_t w0 = pack_bf16x2(p[0], p[1]), w1 = pack_bf16x2(p[2], p[3]);
    const uint32_t w2 = pack_bf16x2(p[4], p[5]), w3 = pack_bf16x2(p[6], p[7]);
    if (a.out_shards) {
        st_u4(a.out + o, make_uint4(w0, w1, w2, w3));
        return;
    }
    if (nreal <= 0) return;
    const int64_t u0 = o - c.e.off + c.e.uoff;
    if (!ZG_OK(a.status, u0 >= 0 && u0 + nreal <= a.n, kSiteParamFull, u0)) return;
    uint16_t* dst = a.out + u0;
    if (nreal == 8) {
        const int al = (int)(u0 & 7);
        if (al == 0) {
            st_u4(dst, make_uint4(w0, w1, w2, w3));
        } else if (al == 4) {
            __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w0, w1));
            __stcs(reinterpret_cast<uint2*>(dst + 4), make_uint2(w2, w3));
        } else if ((al & 1) == 0) {
            unsigned int* d = reinterpret_cast<unsigned int*>(dst);
            __stcs(d, w0);
            __stcs(d + 1, w1);
            __stcs(d + 2, w2);
            __stcs(d + 3, w3);
        } else {
            unsigned short* d = reinterpret_cast<unsigned short*>(dst);
            __stcs(d + 0, (unsigned short)(w0 & 0xFFFF));
            __stcs(d + 1, (unsigned short)(w0 >> 16));
            __stcs(d + 2, (unsigned short)(w1 & 0xFFFF));
            __stcs(d + 3, (unsigned short)(w1 >> 16));
            __stcs(d + 4, (unsigned short)(w2 & 0xFFFF));
            __stcs(d + 5, (unsigned short)(w2 >> 16));
            __stcs(d + 6, (unsigned short)(w3 & 0xFFFF));
            __stcs(d + 7, (unsigned short)(w3 >> 16));
        }
        return;
    }
    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < nreal) dst[i] = (uint16_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFFF);
}

// ---------------------------------------------------------------------------------------
// Squared-norm accumulation. Each square is split exactly as x*x = p + err (p the rounded
// product, err = fma(x, x, -p), the two-product of Dekker 1971); the p are summed with
// Kahan's (1965) compensated fp32 summation and the tiny err terms plainly. A thread's
// total is formed in fp64, and threads and CTAs are combined in fp64 in a fixed order.
// ---------------------------------------------------------------------------------------
struct SumSq {
    float s = 0.0f, c = 0.0f, e = 0.0f;
    __device__ __forceinline__ void add_square(float x) {
        const float p = __fmul_rn(x, x);
        e = __fadd_rn(e, __fmaf_rn(x, x, -p));
        const float y = __fsub_rn(p, c);
        const float t = __fadd_rn(s, y);
        c = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
    }
    __device__ __forceinline__ void add8(const float g[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) add_square(g[i]);
    }
    __device__ __forceinline__ double value() const { return ((double)s - (double)c) + (double)e; }
};

// Sum over the CTA in a fixed order; the result is valid in thread 0.
template <int THREADS>
__device__ __forceinline__ double block_sum(double x) {
    __shared__ double warp_sums[THREADS / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xFFFFFFFFu, x, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_sums[warp] = x;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) t += warp_sums[w];
    }
    return t;
}

// ---------------------------------------------------------------------------------------
// K1: reduce-scatter + per-CTA partial sums of squares (+ write of the fp32 average).
// ---------------------------------------------------------------------------------------
template <int MT, bool WRITE, bool GROUPED = false, int THREADS = WRITE ? kThreadsRsNormWrite : kThreadsRsNormOnly,
          bool PDL = false, int SRC = kSrcRanks>
__global__ void __launch_bounds__(THREADS) k_rs_norm(const StepArgs a) {
    const PdlScope<PDL> pdl(a.pdl);
    SumSq acc;
    const int64_t stride = (int64_t)gridDim.x * THREADS;
    int64_t vi = a.vbeg + (int64_t)blockIdx.x * THREADS + threadIdx.x;
    if (vi < a.vend) {
        Cursor c;
        c.init(a.buckets, a.nb, vi * 8, a.b_first, a.b_end);
        for (; vi < a.vend; vi += stride) {
            const int64_t o = vi * 8;
            c.seek(o);
            float sum[8], gh[8];
            if (!ZG_OK(a.status, src_in_range<SRC>(a, c.e, o - a.gbase), kSiteGradNorm, o)) continue;
            rank_sum<MT, kGradLoadRsNorm, GROUPED, SRC>(a, c.e, o - a.gbase, sum);
            average8(sum, a.inv_M, c.nreal(o), gh);
            if (WRITE && ZG_OK(a.status, o + 8 <= a.npad, kSiteGhatWrite, o)) {
                st_f4<kGhatStoreRsNorm>(a.ghat + o, make_float4(gh[0], gh[1], gh[2], gh[3]));
                st_f4<kGhatStoreRsNorm>(a.ghat + o + 4, make_float4(gh[4], gh[5], gh[6], gh[7]));
            }
            acc.add8(gh);
        }
    }
    const double t = block_sum<THREADS>(acc.value());
    if (threadIdx.x == 0 && ZG_OK(a.status, blockIdx.x < (a.part_cap > 0 ? a.part_cap : kMaxPartials), kSitePartial,
                                  blockIdx.x))
        a.partials[blockIdx.x] = t;
}

// ---------------------------------------------------------------------------------------
// K2: one CTA. Global norm = sqrt(sum of partials); clip scale c / norm when norm > c.
// A non-finite norm raises the flag that makes the update kernels skip the step.
// ---------------------------------------------------------------------------------------
// Fixed-order fp64 sum of n partials by one CTA; the result is valid in thread 0.
__device__ __forceinline__ double cta_sum_partials(const double* partials, int n) {
    __shared__ double sm[kThreads];
    double x = 0.0;
    for (int i = threadIdx.x; i < n; i += kThreads) x += partials[i];
    sm[threadIdx.x] = x;
    __syncthreads();
    for (int h = kThreads / 2; h > 0; h >>= 1) {
        if (threadIdx.x < h) sm[threadIdx.x] += sm[threadIdx.x + h];
        __syncthreads();
    }
    return sm[0];
}

__global__ void __launch_bounds__(kThreads) k_norm_final(Status* st, const double* partials, int nparts,
                                                         double max_norm, int clip, int sched) {
    if (!ZG_OK(st, nparts <= kMaxPartials, kSiteFinalCount, nparts)) return;
    const double sumsq = cta_sum_partials(partials, nparts);
    if (threadIdx.x == 0) {
        if (sched) max_norm = st->cur_max_norm;
        const double norm = sqrt(sumsq);
        const bool finite = isfinite(norm);
        st->sumsq = sumsq;
        st->norm = norm;
        st->flags = (st->flags & (kFlagBounds | kFlagSchedule)) | ((clip && !finite) ? kFlagNonfinite : 0);
        st->scale = (clip && finite && norm > max_norm) ? (float)(max_norm / norm) : 1.0f;
    }
}

// ---------------------------------------------------------------------------------------
// Scheduled steps: the scalars of AdamW come from a device table that the host filled ahead,
// indexed by a step counter kept on the device, so that a launch sequence captured once
// (a CUDA graph) performs a different step at every replay.
// ---------------------------------------------------------------------------------------
__global__ void k_schedule_install(Status* st, int64_t t, int64_t count) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    st->t_dev = t;
    st->sched_base = t + 1;
    st->sched_count = count;
    st->flags &= ~kFlagSchedule;
}

// A step with no entry changes nothing but the flag; the counter stays at the last step run.
__global__ void k_step_begin(Status* st, const ScheduleEntry* table) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const int64_t t = st->t_dev + 1;
    const int64_t i = t - st->sched_base;
    if ((st->flags & kFlagSchedule) || table == nullptr || i < 0 || i >= st->sched_count) {
        st->flags |= kFlagSchedule;
        return;
    }
    st->t_dev = t;
    st->cur = table[i].k;
    st->cur_max_norm = table[i].max_norm;
}

// Per-bucket streaming: the sum of one bucket's CTA partials into the bucket's slot.
template <bool PDL>
__global__ void __launch_bounds__(kThreads) k_sum_partials(const double* partials, int nparts, double* out,
                                                           int32_t pdl_mode) {
    const PdlScope<PDL> pdl(pdl_mode);
    const double t = cta_sum_partials(partials, nparts);
    if (threadIdx.x == 0) *out = t;
}

// ---------------------------------------------------------------------------------------
// K3: AdamW from the materialized fp32 average (clipped, two-pass form).
// ---------------------------------------------------------------------------------------
template <bool SCHED>
__global__ void __launch_bounds__(kThreadsAdamw) k_adamw(const StepArgs a) {
    if (a.status->flags & (SCHED ? (kFlagNonfinite | kFlagSchedule) : kFlagNonfinite)) return;
    const float s = a.status->scale;
    // scheduled steps read their scalars from the status word where they are used
    const AdamConsts& k = SCHED ? a.status->cur : a.k;
    const int64_t stride = (int64_t)gridDim.x * kThreadsAdamw;
    int64_t vi = (int64_t)blockIdx.x * kThreadsAdamw + threadIdx.x;
    if (vi >= a.nvec) return;
    Cursor c;
    c.init(a.buckets, a.nb, vi * 8);
    for (; vi < a.nvec; vi += stride) {
        const int64_t o = vi * 8;
        c.seek(o);
        float gh[8], p[8], m[8], v[8];
        if (!ZG_OK(a.status, o + 8 <= a.npad, kSiteGhatRead, o)) continue;
        const float4 g0 = ld_f4<kGhatLoadAdamw>(a.ghat + o), g1 = ld_f4<kGhatLoadAdamw>(a.ghat + o + 4);
        load_state<kStateLoadAdamw>(a, o, p, m, v);
        unpack(g0, g1, gh);
        adam_vec<true>(gh, s, p, m, v, k);
        store_state<kStateStoreAdamw>(a, o, p, m, v);
        store_params(a, c, o, c.nreal(o), p);
    }
}

// ---------------------------------------------------------------------------------------
// K4: fused reduce-scatter + AdamW + all-gather epilogue: the averaged gradient never
// leaves registers. SCALE applies the clip scale computed by K2 (recompute form). Runs over
// vecs [vbeg, vend): the whole layout, or one bucket (ZeRO-2 per-bucket steps).
// ---------------------------------------------------------------------------------------
template <int MT, bool SCALE, bool GROUPED = false, bool SCHED = false, bool PDL = false, int SRC = kSrcRanks>
__global__ void __launch_bounds__(kThreadsRsAdamw) k_rs_adamw(const StepArgs a) {
    const PdlScope<PDL> pdl(a.pdl);
    float s = 1.0f;
    if (SCALE) {
        if (a.status->flags & (SCHED ? (kFlagNonfinite | kFlagSchedule) : kFlagNonfinite)) return;
        s = a.status->scale;
    } else if (SCHED) {
        if (a.status->flags & kFlagSchedule) return;
    }
    // scheduled steps copy their scalars from the status word into registers at the start
    // (with plain state accesses the clipped M = 4 kernel ran 1.7% faster this way than when
    // it read them where they are used)
    const AdamConsts k = SCHED ? a.status->cur : a.k;
    // the launched block size, rs_adamw_threads(M): only the one-source instance (MT = 1) is
    // launched for M = 1 (ByM), and it takes fewer threads
    constexpr int kT = MT == 1 ? kThreadsRsAdamwOne : kThreadsRsAdamw;
    const int64_t stride = (int64_t)gridDim.x * kT;
    int64_t vi = a.vbeg + (int64_t)blockIdx.x * kT + threadIdx.x;
    if (vi >= a.vend) return;
    Cursor c;
    c.init(a.buckets, a.nb, vi * 8, a.b_first, a.b_end);
    for (; vi < a.vend; vi += stride) {
        const int64_t o = vi * 8;
        c.seek(o);
        float sum[8], gh[8], p[8], m[8], v[8];
        if constexpr (MT == 1) {
            // one source: too few loads in flight per thread to cover the memory latency at one
            // CTA per SM, so the next iteration's state lines are prefetched into L2 (the state
            // arrays hold every lane below vend * 8, so the addresses are in range)
            const int64_t on = o + stride * 8;
            if (on < a.vend * 8) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.master + on));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.m + on));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.v + on));
            }
        }
        if (!ZG_OK(a.status, o + 8 <= a.npad && src_in_range<SRC>(a, c.e, o), kSiteStepLanes, o)) continue;
        // state loads first: neutral for the plain kernel, +10% for the grouped one (measured)
        load_state<kStateLoadRsAdamw>(a, o, p, m, v);
        rank_sum<MT, kGradLoadRsAdamw, GROUPED, SRC>(a, c.e, o, sum);  // grads[r] is addressed by absolute lane
        const int nr = c.nreal(o);
        average8(sum, a.inv_M, nr, gh);
        adam_vec<SCALE>(gh, s, p, m, v, k);
        store_state<kStateStoreRsAdamw>(a, o, p, m, v);
        store_params(a, c, o, nr, p);
    }
}

// ---------------------------------------------------------------------------------------
// K5: all-gather of the padded bf16 shards into the unpadded full buffer, over unpadded
// indices [u_begin, u_end). Work item: 8 destination elements (one 16-byte store). When
// its source run is unaligned by k elements, two aligned 16-byte loads are spliced.
// ---------------------------------------------------------------------------------------
// Last bucket among [first, end) whose unpadded start is <= u (end <= 0: all buckets;
// buckets are never empty for a valid plan).
__device__ __forceinline__ int64_t bucket_of_unpadded(const Bucket* tab, int64_t nb, int64_t u, int64_t first,
                                                      int64_t end) {
    int64_t lo = first, hi = (end > 0 ? end : nb) - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (tab[mid].uoff <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint4 splice(uint4 A, uint4 B, int k) {
    const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
    switch (k) {
        case 1: return make_uint4(__byte_perm(w[0], w[1], 0x5432), __byte_perm(w[1], w[2], 0x5432),
                                  __byte_perm(w[2], w[3], 0x5432), __byte_perm(w[3], w[4], 0x5432));
        case 2: return make_uint4(w[1], w[2], w[3], w[4]);
        case 3: return make_uint4(__byte_perm(w[1], w[2], 0x5432), __byte_perm(w[2], w[3], 0x5432),
                                  __byte_perm(w[3], w[4], 0x5432), __byte_perm(w[4], w[5], 0x5432));
        case 4: return make_uint4(w[2], w[3], w[4], w[5]);
        case 5: return make_uint4(__byte_perm(w[2], w[3], 0x5432), __byte_perm(w[3], w[4], 0x5432),
                                  __byte_perm(w[4], w[5], 0x5432), __byte_perm(w[5], w[6], 0x5432));
        case 6: return make_uint4(w[3], w[4], w[5], w[6]);
        case 7: return make_uint4(__byte_perm(w[3], w[4], 0x5432), __byte_perm(w[4], w[5], 0x5432),
                                  __byte_perm(w[5], w[6], 0x5432), __byte_perm(w[6], w[7], 0x5432));
        default: return A;
    }
}

// out[d] = shards[lane of unpadded index u0 + d] for d in [0, count). Work item: one
// 16-byte-aligned slot of 8 output elements (a0 = the output's misalignment in elements);
// slots wholly inside the range whose source run lies in one bucket take one aligned
// 16-byte store (the source run spliced from two aligned loads when it is unaligned);
// edge slots go element by element. Each thread finds its first bucket once and then walks
// forward (its indices only grow).
struct UCursor {
    const Bucket* tab;
    int64_t nb, b;
    Bucket e;
    __device__ __forceinline__ void init(const Bucket* t, int64_t n, int64_t u, int64_t first, int64_t end) {
        tab = t;
        nb = n;
        b = bucket_of_unpadded(t, n, u, first, end);
        e = tab[b];
    }
    __device__ __forceinline__ void seek(int64_t u) {
        while (u >= e.uoff + e.n && b + 1 < nb) {
            ++b;
            e = tab[b];
        }
    }
};

template <bool PDL>
__global__ void __launch_bounds__(kThreadsGather) k_gather(const uint16_t* __restrict__ shards,
                                                     uint16_t* __restrict__ out, const Bucket* tab, int64_t nb,
                                                     int64_t npad, int64_t u0, int64_t count, Status* st,
                                                     int64_t b_first, int64_t b_end, int32_t pdl_mode) {
    const PdlScope<PDL> pdl(pdl_mode);
    const int64_t a0 = (int64_t)((reinterpret_cast<uintptr_t>(out) >> 1) & 7);
    const int64_t nslots = (count + a0 + 7) >> 3;
    const int64_t stride = (int64_t)gridDim.x * kThreadsGather;
    int64_t w = (int64_t)blockIdx.x * kThreadsGather + threadIdx.x;
    if (w >= nslots) return;
    UCursor c;
    c.init(tab, nb, u0 + (w * 8 - a0 > 0 ? w * 8 - a0 : 0), b_first, b_end);
    for (; w < nslots; w += stride) {
        const int64_t d0 = w * 8 - a0;  // first output element of the slot (may be < 0)
        if (d0 >= 0 && d0 + 8 <= count) {
            const int64_t u = u0 + d0;
            c.seek(u);
            if (u + 8 <= c.e.uoff + c.e.n) {
                const int64_t src = u - c.e.uoff + c.e.off;
                const int k = (int)(src & 7);
                const uint16_t* base = shards + (src - k);
                if (!ZG_OK(st, src >= 0 && src + 8 <= npad, kSiteGatherSrc, src)) continue;
                if (k == 0) {
                    st_u4p<kGatherStore>(out + d0, ld_u4p<kGatherLoad>(base));
                    continue;
                }
                if (src - k + 8 < npad) {
                    st_u4p<kGatherStore>(out + d0, splice(ld_u4p<kGatherLoad>(base), ld_u4p<kGatherLoad>(base + 8), k));
                    continue;
                }
            }
        }
        for (int i = 0; i < 8; ++i) {
            const int64_t d = d0 + i;
            if (d < 0 || d >= count) continue;
            const int64_t uu = u0 + d;
            c.seek(uu);
            const int64_t lane = uu - c.e.uoff + c.e.off;
            if (!ZG_OK(st, lane >= 0 && lane < npad && uu - c.e.uoff < c.e.n, kSiteGatherSrc, lane)) continue;
            out[d] = shards[lane];
        }
    }
}

// ---------------------------------------------------------------------------------------
// State in: master (and optionally m, v; zeros when null) from unpadded vectors scattered
// into the padded layout (padding 0), plus the bf16 copies of the parameters. One lane per
// thread (not a hot kernel). Serves initialisation and checkpoint loading. Any output may be
// null (the padded full parameters of the process-per-rank mode are written alone).
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsInit) k_init(const float* __restrict__ init, const float* __restrict__ m_init,
                                                   const float* __restrict__ v_init, float* master, float* m,
                                                   float* v, uint16_t* full, uint16_t* shards, const Bucket* tab,
                                                   int64_t nb, int64_t npad, int64_t n, Status* st) {
    const int64_t stride = (int64_t)gridDim.x * kThreadsInit;
    int64_t o = (int64_t)blockIdx.x * kThreadsInit + threadIdx.x;
    if (o >= npad) return;
    Cursor c;
    c.init(tab, nb, o);
    for (; o < npad; o += stride) {
        c.seek(o);
        const bool real = o < c.e.off + c.e.n;
        const int64_t u = o - c.e.off + c.e.uoff;
        if (!ZG_OK(st, !real || (u >= 0 && u < n), kSiteInit, u)) continue;
        const float x = real ? init[u] : 0.0f;
        if (master) master[o] = x;
        if (m) m[o] = (real && m_init) ? m_init[u] : 0.0f;
        if (v) v[o] = (real && v_init) ? v_init[u] : 0.0f;
        const uint16_t h = to_bf16(x);
        if (shards) shards[o] = h;
        if (real && full) full[u] = h;
    }
}

// State out: the real lanes of master, m and v gathered into unpadded vectors (the layout-
// independent form a checkpoint keeps, loadable under any rank count or bucket size).
__global__ void __launch_bounds__(kThreadsInit) k_save(const float* __restrict__ master, const float* __restrict__ m,
                                                   const float* __restrict__ v, float* out_master, float* out_m,
                                                   float* out_v, const Bucket* tab, int64_t nb, int64_t npad,
                                                   int64_t n, Status* st) {
    const int64_t stride = (int64_t)gridDim.x * kThreadsInit;
    int64_t o = (int64_t)blockIdx.x * kThreadsInit + threadIdx.x;
    if (o >= npad) return;
    Cursor c;
    c.init(tab, nb, o);
    for (; o < npad; o += stride) {
        c.seek(o);
        if (o >= c.e.off + c.e.n) continue;
        const int64_t u = o - c.e.off + c.e.uoff;
        if (!ZG_OK(st, u >= 0 && u < n, kSiteSave, u)) continue;
        if (out_master) out_master[u] = master[o];
        if (out_m) out_m[u] = m[o];
        if (out_v) out_v[u] = v[o];
    }
}

// ---------------------------------------------------------------------------------------
// Dispatch on the rank count: fully unrolled variants for M in {1, 2, 4, 8, 16}, a generic
// loop otherwise.
// ---------------------------------------------------------------------------------------
template <template <int> class F>
struct ByM {
    static auto get(int M, int groups = 1) {
        if (groups > 1) {  // hybrid sharding: grouped kernels, encoded as F<-M> (F<-64>: generic M)
            switch (M) {
                case 4: return F<-4>::fn();
                case 8: return F<-8>::fn();
                case 16: return F<-16>::fn();
                default: return F<-64>::fn();
            }
        }
        switch (M) {
            case 1: return F<1>::fn();
            case 2: return F<2>::fn();
            case 4: return F<4>::fn();
            case 8: return F<8>::fn();
            case 16: return F<16>::fn();
            default: return F<0>::fn();
        }
    }
};

// A negative MT stands for the grouped (hybrid-sharding) kernel of rank count -MT, with -64
// for the generic (runtime rank count) one.
constexpr int grouped_mt(int mt) { return mt == -64 ? 0 : -mt; }
template <int MT> struct RsNormWrite {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_norm<grouped_mt(MT), true, true>;
        else return &k_rs_norm<MT, true>;
    }
};
template <int MT> struct RsNormWritePdl {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_norm<grouped_mt(MT), true, true, kThreadsRsNormWrite, true>;
        else return &k_rs_norm<MT, true, false, kThreadsRsNormWrite, true>;
    }
};
template <int MT> struct RsNormOnly {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_norm<grouped_mt(MT), false, true>;
        else return &k_rs_norm<MT, false>;
    }
};
template <int MT> struct RsAdamwScaled {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_adamw<grouped_mt(MT), true, true>;
        else return &k_rs_adamw<MT, true>;
    }
};
template <int MT> struct RsAdamwPlain {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_adamw<grouped_mt(MT), false, true>;
        else return &k_rs_adamw<MT, false>;
    }
};
template <int MT> struct RsAdamwPlainPdl {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_adamw<grouped_mt(MT), false, true, false, true>;
        else return &k_rs_adamw<MT, false, false, false, true>;
    }
};
template <int MT> struct RsAdamwScaledSched {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_adamw<grouped_mt(MT), true, true, true>;
        else return &k_rs_adamw<MT, true, false, true>;
    }
};
template <int MT> struct RsAdamwPlainSched {
    static auto fn() {
        if constexpr (MT < 0) return &k_rs_adamw<grouped_mt(MT), false, true, true>;
        else return &k_rs_adamw<MT, false, false, true>;
    }
};

// Process-per-rank mode, sources in the exchange layout (flat mode; no grouped variants).
template <int MT> struct RsNormWriteX {
    static auto fn() { return &k_rs_norm<MT < 0 ? 0 : MT, true, false, kThreadsRsNormWrite, false, kSrcExchange>; }
};
template <int MT> struct RsNormOnlyX {
    static auto fn() { return &k_rs_norm<MT < 0 ? 0 : MT, false, false, kThreadsRsNormOnly, false, kSrcExchange>; }
};
template <int MT> struct RsAdamwScaledX {
    static auto fn() { return &k_rs_adamw<MT < 0 ? 0 : MT, true, false, false, false, kSrcExchange>; }
};
template <int MT> struct RsAdamwPlainX {
    static auto fn() { return &k_rs_adamw<MT < 0 ? 0 : MT, false, false, false, false, kSrcExchange>; }
};

const void* variant_fn(int variant, int M, int groups) {
    switch (variant) {
        case kVarRsNormWrite: return (const void*)ByM<RsNormWrite>::get(M, groups);
        case kVarRsNormOnly: return (const void*)ByM<RsNormOnly>::get(M, groups);
        case kVarAdamw: return (const void*)&k_adamw<false>;
        case kVarRsAdamwScaled: return (const void*)ByM<RsAdamwScaled>::get(M, groups);
        case kVarRsAdamwPlain: return (const void*)ByM<RsAdamwPlain>::get(M, groups);
        case kVarGather: return (const void*)&k_gather<false>;
        case kVarInit: return (const void*)&k_init;
        case kVarRsNormWriteX: return (const void*)ByM<RsNormWriteX>::get(M);
        case kVarRsNormOnlyX: return (const void*)ByM<RsNormOnlyX>::get(M);
        case kVarRsAdamwScaledX: return (const void*)ByM<RsAdamwScaledX>::get(M);
        case kVarRsAdamwPlainX: return (const void*)ByM<RsAdamwPlainX>::get(M);
        case kVarRsNormWriteF: return (const void*)&k_rs_norm<0, true, false, kThreadsRsNormWrite, false, kSrcF32>;
        case kVarRsNormOnlyF: return (const void*)&k_rs_norm<0, false, false, kThreadsRsNormOnly, false, kSrcF32>;
        case kVarRsAdamwScaledF: return (const void*)&k_rs_adamw<0, true, false, false, false, kSrcF32>;
        case kVarRsAdamwPlainF: return (const void*)&k_rs_adamw<0, false, false, false, false, kSrcF32>;
        default: return nullptr;
    }
}

// Launch with programmatic stream serialization (see PdlScope).
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*fn)(P...), int grid, int threads, cudaStream_t s, A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, std::forward<A>(args)...);
}

}  // namespace

int variant_threads(int variant) {
    switch (variant) {
        case kVarRsNormWrite:
        case kVarRsNormWriteX:
        case kVarRsNormWriteF: return kThreadsRsNormWrite;
        case kVarRsNormOnly:
        case kVarRsNormOnlyX:
        case kVarRsNormOnlyF: return kThreadsRsNormOnly;
        case kVarAdamw: return kThreadsAdamw;
        case kVarRsAdamwScaled:
        case kVarRsAdamwPlain:
        case kVarRsAdamwScaledX:
        case kVarRsAdamwPlainX:
        case kVarRsAdamwScaledF:
        case kVarRsAdamwPlainF: return kThreadsRsAdamw;
        case kVarGather: return kThreadsGather;
        case kVarInit: return kThreadsInit;
        default: return kThreads;
    }
}

int variant_ctas_per_sm_cap(int variant) {
    switch (variant) {
        case kVarRsNormWrite:
        case kVarRsNormWriteX:
        case kVarRsNormWriteF: return kCtasPerSmRsNormWrite;
        case kVarRsNormOnly:
        case kVarRsNormOnlyX:
        case kVarRsNormOnlyF: return kCtasPerSmRsNormOnly;
        case kVarAdamw: return kCtasPerSmAdamw;
        case kVarRsAdamwScaled:
        case kVarRsAdamwPlain:
        case kVarRsAdamwScaledX:
        case kVarRsAdamwPlainX:
        case kVarRsAdamwScaledF:
        case kVarRsAdamwPlainF: return kCtasPerSmRsAdamw;
        default: return 0;
    }
}

cudaError_t variant_blocks_per_sm(int variant, int M, int groups, int* blocks) {
    const void* fn = variant_fn(variant, M, groups);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, variant_threads(variant), 0);
    const int cap = variant_ctas_per_sm_cap(variant);
    if (e == cudaSuccess && cap > 0 && *blocks > cap) *blocks = cap;
    return e;
}

cudaError_t launch_rs_norm(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s) {
    if (write_ghat && a.pdl != kPdlNone)
        return launch_pdl(ByM<RsNormWritePdl>::get(a.M, a.groups), grid, kThreadsRsNormWrite, s, a);
    if (write_ghat) ByM<RsNormWrite>::get(a.M, a.groups)<<<grid, kThreadsRsNormWrite, 0, s>>>(a);
    else ByM<RsNormOnly>::get(a.M, a.groups)<<<grid, kThreadsRsNormOnly, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_norm_f32src(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s) {
    if (write_ghat) k_rs_norm<0, true, false, kThreadsRsNormWrite, false, kSrcF32><<<grid, kThreadsRsNormWrite, 0, s>>>(a);
    else k_rs_norm<0, false, false, kThreadsRsNormOnly, false, kSrcF32><<<grid, kThreadsRsNormOnly, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_adamw_f32src(const StepArgs& a, bool apply_scale, int grid, cudaStream_t s) {
    if (apply_scale) k_rs_adamw<0, true, false, false, false, kSrcF32><<<grid, kThreadsRsAdamw, 0, s>>>(a);
    else k_rs_adamw<0, false, false, false, false, kSrcF32><<<grid, kThreadsRsAdamw, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_norm_exchange(const StepArgs& a, bool write_ghat, int grid, cudaStream_t s) {
    if (write_ghat) ByM<RsNormWriteX>::get(a.M)<<<grid, kThreadsRsNormWrite, 0, s>>>(a);
    else ByM<RsNormOnlyX>::get(a.M)<<<grid, kThreadsRsNormOnly, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_adamw_exchange(const StepArgs& a, bool apply_scale, int grid, cudaStream_t s) {
    const int threads = rs_adamw_threads(a.M);
    if (apply_scale) ByM<RsAdamwScaledX>::get(a.M)<<<grid, threads, 0, s>>>(a);
    else ByM<RsAdamwPlainX>::get(a.M)<<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_norm_final(Status* st, const double* partials, int nparts, double max_norm, int clip,
                              bool sched, cudaStream_t s) {
    k_norm_final<<<1, kThreads, 0, s>>>(st, partials, nparts, max_norm, clip, sched ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_schedule_install(Status* st, int64_t t, int64_t count, cudaStream_t s) {
    k_schedule_install<<<1, 32, 0, s>>>(st, t, count);
    return cudaGetLastError();
}

cudaError_t launch_step_begin(Status* st, const ScheduleEntry* table, cudaStream_t s) {
    k_step_begin<<<1, 32, 0, s>>>(st, table);
    return cudaGetLastError();
}

cudaError_t launch_sum_partials(const double* partials, int nparts, double* out, cudaStream_t s, int pdl) {
    if (pdl != kPdlNone) return launch_pdl(&k_sum_partials<true>, 1, kThreads, s, partials, nparts, out, (int32_t)pdl);
    k_sum_partials<false><<<1, kThreads, 0, s>>>(partials, nparts, out, (int32_t)kPdlNone);
    return cudaGetLastError();
}

cudaError_t launch_adamw(const StepArgs& a, bool sched, int grid, cudaStream_t s) {
    if (sched) k_adamw<true><<<grid, kThreadsAdamw, 0, s>>>(a);
    else k_adamw<false><<<grid, kThreadsAdamw, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_adamw(const StepArgs& a, bool apply_scale, bool sched, int grid, cudaStream_t s) {
    const int threads = rs_adamw_threads(a.M);
    if (sched) {
        if (apply_scale) ByM<RsAdamwScaledSched>::get(a.M, a.groups)<<<grid, threads, 0, s>>>(a);
        else ByM<RsAdamwPlainSched>::get(a.M, a.groups)<<<grid, threads, 0, s>>>(a);
    } else if (apply_scale) {
        ByM<RsAdamwScaled>::get(a.M, a.groups)<<<grid, threads, 0, s>>>(a);
    } else if (a.pdl != kPdlNone) {
        return launch_pdl(ByM<RsAdamwPlainPdl>::get(a.M, a.groups), grid, threads, s, a);
    } else {
        ByM<RsAdamwPlain>::get(a.M, a.groups)<<<grid, threads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* shards, uint16_t* out, const Bucket* buckets, int64_t nb, int64_t npad,
                          int64_t u0, int64_t count, Status* st, int grid, cudaStream_t s, int pdl,
                          int64_t b_first, int64_t b_end) {
    if (count <= 0) return cudaSuccess;
    if (pdl != kPdlNone)
        return launch_pdl(&k_gather<true>, grid, kThreadsGather, s, shards, out, buckets, nb, npad, u0, count, st,
                          b_first, b_end, (int32_t)pdl);
    k_gather<false><<<grid, kThreadsGather, 0, s>>>(shards, out, buckets, nb, npad, u0, count, st, b_first, b_end,
                                                    (int32_t)kPdlNone);
    return cudaGetLastError();
}

cudaError_t launch_init(const float* master_init, const float* m_init, const float* v_init, float* master, float* m,
                        float* v, uint16_t* full, uint16_t* shards, const Bucket* buckets, int64_t nb, int64_t npad,
                        int64_t n, Status* st, int grid, cudaStream_t s) {
    if (npad <= 0) return cudaSuccess;
    k_init<<<grid, kThreadsInit, 0, s>>>(master_init, m_init, v_init, master, m, v, full, shards, buckets, nb, npad, n,
                                         st);
    return cudaGetLastError();
}

cudaError_t launch_save(const float* master, const float* m, const float* v, float* out_master, float* out_m,
                        float* out_v, const Bucket* buckets, int64_t nb, int64_t npad, int64_t n, Status* st, int grid,
                        cudaStream_t s) {
    if (npad <= 0) return cudaSuccess;
    k_save<<<grid, kThreadsInit, 0, s>>>(master, m, v, out_master, out_m, out_v, buckets, nb, npad, n, st);
    return cudaGetLastError();
}

}  // namespace zg

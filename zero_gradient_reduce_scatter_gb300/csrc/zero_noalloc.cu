// zero_noalloc.cu -- zero_grad_norm_noalloc: the global gradient norm and clip scale of the
// averaged gradient, for callers that cannot allocate device memory.
//
// The regular path keeps its status word, per-CTA partial sums and bucket table in the
// caller's `scratch` buffer. Some callers cannot provide one: code that runs where device
// allocation is not allowed or not possible (an allocator callback, a host runtime that
// owns all device memory and hands out only fixed buffers, a tool that must not change the
// process's memory footprint). For them this entry point uses a fixed scratch array that
// is part of the library image instead: every GPU that loads the library holds it until
// the process exits.

#include <cstdint>
#include <cstring>
#include <mutex>

#include "zero_internal.h"

namespace {

// Largest bucket table the fixed scratch holds (larger layouts are rejected).
constexpr int64_t kNoallocMaxBuckets = 2048;
constexpr int64_t kNoallocBytes = zg::kScratchBuckets + 32 * kNoallocMaxBuckets;  // 98,560 bytes

// The fixed scratch: status word, per-CTA partials, bucket table (same layout as the
// caller-provided scratch of the regular path). Host code must not use this name as an
// address; it uses the per-device address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices];       // device address of g_noalloc_scratch, per device
int g_grid[kMaxDevices][ZERO_MAX_RANKS + 1];  // grid of the norm pass, per device and M

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

int fail(cudaError_t e) { return zg::record_cuda_error(e); }

// Set-up, once per device, with that device current: the scratch array's device address
// and the launch grid for every rank count 1..ZERO_MAX_RANKS (same rule as the regular path,
// so both sum in the same order). All of it happens in the device's first call, so no later
// call, whatever its M, queries the runtime.
int setup(int dev, int M, void** addr, int* grid_cap) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail(e);
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(e);
        for (int m = 1; m <= ZERO_MAX_RANKS; ++m) {
            int per_sm = 0;
            e = zg::variant_blocks_per_sm(zg::kVarRsNormOnly, m, 1, &per_sm);
            if (e != cudaSuccess) return fail(e);
            const int g = (per_sm < 1 ? 1 : per_sm) * sms;
            g_grid[dev][m] = g > zg::kMaxPartials ? zg::kMaxPartials : g;
        }
        g_addr[dev] = p;  // last: set-up is complete once the address is published
    }
    *addr = g_addr[dev];
    *grid_cap = g_grid[dev][M];
    return ZERO_OK;
}

// A pointer the call may hand to its kernels: device (or managed) memory on device `dev`.
bool on_device(const void* p, int dev) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error of an unknown pointer
        return false;
    }
    if (attr.type == cudaMemoryTypeManaged) return true;
    return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}

// Up to 64 bucket-table rows, passed by value, written into the fixed scratch.
struct TableChunk {
    zg::Bucket row[64];
    int64_t first;
    int64_t count;
};

__global__ void k_write_table(zg::Bucket* table, const TableChunk c) {
    if (threadIdx.x < c.count) table[c.first + threadIdx.x] = c.row[threadIdx.x];
}

__global__ void k_copy_result(const zg::Status* st, double* norm_out, float* scale_out) {
    *norm_out = st->norm;
    *scale_out = st->scale;
}

}  // namespace

extern "C" int zero_grad_norm_noalloc(const void* const* grads, int M, const int64_t* bucket_table,
                                      int64_t n_buckets, double max_grad_norm, double* norm_out,
                                      float* scale_out, void* stream) {
    if (!grads || !bucket_table || !norm_out || !scale_out) return ZERO_ERR_INVALID_ARG;
    if (M < 1 || M > ZERO_MAX_RANKS || n_buckets < 1) return ZERO_ERR_INVALID_ARG;
    if (n_buckets > kNoallocMaxBuckets) return ZERO_ERR_TOO_LARGE;
    if (!(max_grad_norm > 0.0) || max_grad_norm != max_grad_norm) return ZERO_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(norm_out) & 7u) || (reinterpret_cast<uintptr_t>(scale_out) & 3u))
        return ZERO_ERR_MISALIGNED;
    for (int r = 0; r < M; ++r) {
        if (!grads[r]) return ZERO_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(grads[r]) & 15u) return ZERO_ERR_MISALIGNED;
    }
    // The table must tile the padded layout contiguously from lane 0, in vecs of 8 lanes
    // (S is bounded before any product is formed, so no sum or product overflows).
    int64_t off = 0;
    for (int64_t b = 0; b < n_buckets; ++b) {
        const int64_t o = bucket_table[4 * b], n = bucket_table[4 * b + 1], S = bucket_table[4 * b + 2];
        if (o != off || S < 0 || n < 0 || S > (INT64_MAX - off) / M) return ZERO_ERR_INVALID_ARG;
        if (n > M * S || (M * S) % 8 != 0) return ZERO_ERR_INVALID_ARG;
        off += M * S;
    }
    const int64_t npad = off;

    // The device is the one that holds the gradients: every gradient and both outputs must
    // be device memory there (a pointer to another GPU's memory, or to host memory, is
    // refused rather than read across devices), and so must the stream, if one is given.
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, grads[0]);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ZERO_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return ZERO_ERR_INVALID_ARG;
    int dev = attr.device;
    if (attr.type == cudaMemoryTypeManaged && cudaGetDevice(&dev) != cudaSuccess) return ZERO_ERR_INVALID_ARG;
    if (dev < 0 || dev >= kMaxDevices) return ZERO_ERR_INVALID_ARG;
    for (int r = 1; r < M; ++r)
        if (!on_device(grads[r], dev)) return ZERO_ERR_INVALID_ARG;
    if (!on_device(norm_out, dev) || !on_device(scale_out, dev)) return ZERO_ERR_INVALID_ARG;
    DeviceGuard guard(dev);
    if (!guard.ok) return fail(cudaErrorInvalidDevice);
    if (stream) {  // with `dev` current, so that the special stream handles resolve to it
        int sdev = -1;
        if (cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess || sdev != dev) {
            cudaGetLastError();
            return ZERO_ERR_INVALID_ARG;
        }
    }
    void* base = nullptr;
    int grid_cap = 0;
    int rc = setup(dev, M, &base, &grid_cap);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    char* scratch = (char*)base;
    zg::Status* status = (zg::Status*)(scratch + zg::kScratchStatus);
    double* partials = (double*)(scratch + zg::kScratchPartials);
    zg::Bucket* table = (zg::Bucket*)(scratch + zg::kScratchBuckets);

    // Bucket table into the fixed scratch, 64 rows per launch (kernel arguments carry the
    // rows, so no host staging buffer or host-to-device copy is involved).
    TableChunk chunk;
    int64_t uoff = 0;
    for (int64_t b0 = 0; b0 < n_buckets; b0 += 64) {
        chunk.first = b0;
        chunk.count = (n_buckets - b0) < 64 ? (n_buckets - b0) : 64;
        for (int64_t i = 0; i < chunk.count; ++i) {
            const int64_t* row = bucket_table + 4 * (b0 + i);
            chunk.row[i] = zg::Bucket{row[0], row[1], row[0] + M * row[2], uoff};
            uoff += row[1];
        }
        k_write_table<<<1, 64, 0, s>>>(table, chunk);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail(e);
    }

    zg::StepArgs a;
    std::memset(&a, 0, sizeof a);
    for (int r = 0; r < M; ++r) a.grads[r] = (const uint16_t*)grads[r];
    a.buckets = table;
    a.nb = n_buckets;
    a.nvec = npad / 8;
    a.vbeg = 0;
    a.vend = a.nvec;
    a.gbase = 0;
    a.gext = npad;
    a.npad = npad;
    a.n = uoff;
    a.M = M;
    a.inv_M = (float)(1.0 / (double)M);
    a.groups = 1;
    a.status = status;
    a.partials = partials;
    int64_t need = (a.nvec + zg::kThreadsRsNormOnly - 1) / zg::kThreadsRsNormOnly;
    if (need < 1) need = 1;
    const int grid = (int)(need < grid_cap ? need : grid_cap);
    // Every partial the finalise kernel reads is written by this call's norm pass, and the
    // status word is written whole, so nothing in the scratch has to be cleared first. The
    // bounds-checked build is the exception: its failed-check record is sticky, so each
    // call starts from a cleared status word (a memset of the fixed array, no allocation).
#ifdef ZERO_CHECKED
    e = cudaMemsetAsync(status, 0, sizeof(zg::Status), s);
    if (e != cudaSuccess) return fail(e);
#endif
    e = zg::launch_rs_norm(a, false, grid, s);
    if (e == cudaSuccess) e = zg::launch_norm_final(status, partials, grid, max_grad_norm, 1, false, s);
    if (e == cudaSuccess) {
        k_copy_result<<<1, 1, 0, s>>>(status, norm_out, scale_out);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return fail(e);
#ifdef ZERO_CHECKED
    // checked build only: wait, and report a failed bounds check of this call
    zg::Status st;
    e = cudaMemcpyAsync(&st, status, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(e);
    if (st.flags & zg::kFlagBounds) return ZERO_ERR_DEVICE;
#endif
    return ZERO_OK;
}

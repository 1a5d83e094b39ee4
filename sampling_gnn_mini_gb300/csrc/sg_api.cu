// C ABI entry points for status, graph and cache handles, and the read probe.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(api)

namespace sgi {

static thread_local std::string t_last_error;

sg_status fail(sg_status s, const char* fmt, ...) {
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

sg_status cuda_fail(cudaError_t e, const char* what) {
    return fail(e == cudaErrorMemoryAllocation ? SG_ERR_OOM : SG_ERR_CUDA, "%s: %s (%s)", what,
                cudaGetErrorString(e), cudaGetErrorName(e));
}

int num_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// SG_FAULT_INJECT=alloc:N makes the N-th owned allocation fail (N >= 1).
static long long inject_alloc_at() {
    static long long at = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* v = getenv("SG_FAULT_INJECT");
        if (v && strncmp(v, "alloc:", 6) == 0) {
            char* end = nullptr;
            const long long n = strtoll(v + 6, &end, 10);
            if (end != v + 6 && n >= 1) at = n;
        }
    });
    return at;
}

cudaError_t dev_alloc(void** p, size_t bytes) {
    static std::atomic<long long> count{0};
    *p = nullptr;
    const long long at = inject_alloc_at();
    if (at > 0 && ++count == at) return cudaErrorMemoryAllocation;
    return cudaMalloc(p, bytes);
}

bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace sgi

using namespace sgi;

// ------------------------------------------------------------------ kernels
namespace {

// Graph validation: offsets start at 0, never decrease, end at m; every
// index in [0, n).  Sets bit 1 (offsets) or bit 2 (indices) of *bad.
template <typename Off>
__global__ void k_validate_indptr(const Off* indptr, int64_t n, int64_t m, unsigned* bad, unsigned long long* maxdeg) {
    unsigned long long local_max = 0;
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n; v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t a = (int64_t)indptr[v], b = (int64_t)indptr[v + 1];
        if (b < a) atomicOr(bad, 1u);
        else if ((unsigned long long)(b - a) > local_max) local_max = (unsigned long long)(b - a);
        if (v == 0 && a != 0) atomicOr(bad, 1u);
        if (v == n - 1 && b != m) atomicOr(bad, 1u);
    }
    for (int d = 16; d > 0; d >>= 1) {
        unsigned long long o = __shfl_xor_sync(0xffffffffu, local_max, d);
        local_max = o > local_max ? o : local_max;
    }
    if ((threadIdx.x & 31) == 0) atomicMax(maxdeg, local_max);
}

__global__ void k_validate_indices(const int32_t* idx, int64_t m, int64_t n, unsigned* bad) {
    bool b = false;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < m; e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t u = idx[e];
        b |= (u < 0) || ((int64_t)u >= n);
    }
    if (__any_sync(0xffffffffu, b) && (threadIdx.x & 31) == 0) atomicOr(bad, 2u);
}

// Fill cache slot s with feature row ranked[s] (or row s when ranked is NULL)
// and record slot_of[node] = s (when there is a slot map).  One 16-byte
// vector per thread step.
__global__ void k_cache_fill(const int32_t* ranked, int64_t n_cache, int64_t n_nodes, const uint4* src,
                             int64_t row_vecs, uint4* cache, int32_t* slot_of) {
    const int64_t total = n_cache * row_vecs;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s = t / row_vecs, c = t - s * row_vecs;
        const int64_t g = ranked ? (int64_t)ranked[s] : s;
        if (g < 0 || g >= n_nodes) {
            if (c == 0) dev_err(ERR_INDEX);
            continue;
        }
        cache[s * row_vecs + c] = src[g * row_vecs + c];
        if (c == 0 && slot_of) slot_of[g] = (int32_t)s;
    }
}

__global__ void k_cache_check_distinct(const int32_t* ranked, int64_t n_cache, const int32_t* slot_of, unsigned* bad) {
    for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s < n_cache; s += (int64_t)gridDim.x * blockDim.x) {
        const int32_t g = ranked[s];
        if (slot_of[g] != (int32_t)s) atomicOr(bad, 1u);
    }
}

// Reads the rows of the host table that the cache does not hold once, in
// order, so that the device's first-access work on the table happens here
// and not inside the first gathers.  Measured on GB300 with a 57 GB table:
// without it the first gathers of 100K misses took 40-600 ms and reached
// their steady time (~1.2 ms) only after ~25 batches; after it, the first
// gather took 1.5 ms.  One 16-byte vector of every 64 KB page was not
// enough.  The read runs at the link's rate (~200 GB/s).
__global__ void k_host_touch(const uint4* __restrict__ host, int64_t nvec, unsigned* sink) {
    uint32_t acc = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (; t + 3 * stride < nvec; t += 4 * stride) {
        const uint4 a = __ldcs(host + t), b = __ldcs(host + t + stride), c = __ldcs(host + t + 2 * stride),
                    d = __ldcs(host + t + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; t < nvec; t += stride) {
        const uint4 a = __ldcs(host + t);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (acc == 0x9E3779B9u) atomicXor(sink, acc);  // keeps the loads live; almost never taken
}

// Streams bytes with 16-byte loads and folds them into one word (read probe).
__global__ void k_read_probe(const uint4* __restrict__ src, int64_t nvec, uint32_t* sink) {
    uint32_t acc = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (; t + 3 * stride < nvec; t += 4 * stride) {
        uint4 a = __ldcs(src + t), b = __ldcs(src + t + stride), c = __ldcs(src + t + 2 * stride),
              d = __ldcs(src + t + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; t < nvec; t += stride) {
        uint4 a = __ldcs(src + t);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (acc == 0x9E3779B9u) atomicXor(sink, acc);  // keeps the loads live; almost never taken
}

// Philox throughput: each thread evaluates consecutive counter blocks.
__global__ void k_hash_probe(int64_t n_calls, uint32_t k0, uint32_t k1, uint32_t* sink) {
    uint32_t acc = 0;
    for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n_calls; q += (int64_t)gridDim.x * blockDim.x) {
        const uint4 w = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), 1u, 0u), k0, k1);
        acc += w.x ^ w.y ^ w.z ^ w.w;
    }
    if (acc == 0x9E3779B9u) atomicXor(sink, acc);
}

// Bounded-wait probe: n_tiles blocks take tiles in order from *counter and
// run the decoupled look-back of the library's single-pass scans on status,
// tile t contributing t + 1; out[t] = its exclusive prefix.  The block that
// takes tile `silent` leaves without publishing, so the look-back of every
// later tile that reaches it waits spin_limit polls, gives up and reports
// ERR_TIMEOUT.  Every wait is bounded; nothing else is outstanding.
__global__ void __launch_bounds__(32) k_wait_probe(unsigned long long* status, unsigned* counter, int32_t silent,
                                                   int32_t spin_limit, int32_t* out) {
    __shared__ int tile_sh;
    if (threadIdx.x == 0) tile_sh = (int)atomicAdd(counter, 1u);
    __syncwarp();
    const int t = tile_sh;
    if (t == silent) return;
    bool late = false;
    const int32_t x = chain_lookback(status, t, 0, t + 1, &late, spin_limit);
    if (threadIdx.x == 0) {
        out[t] = x;
        if (late) dev_err(ERR_TIMEOUT);
    }
}

}  // namespace

// ------------------------------------------------------------------- status
extern "C" int32_t sg_version(void) { return 100; }

extern "C" int32_t sg_last_error(char* buf, size_t n) {
    const std::string& s = t_last_error;
    if (buf && n) {
        size_t k = s.size() < n - 1 ? s.size() : n - 1;
        memcpy(buf, s.data(), k);
        buf[k] = 0;
    }
    return (int32_t)s.size();
}

extern "C" sg_status sg_stream_check(sg_stream_t stream) {
    cudaStream_t s = (cudaStream_t)stream;
    SG_CUDA(cudaStreamSynchronize(s));
    unsigned w = fetch_err_api(s) | fetch_err_sampler(s) | fetch_err_gather(s) | fetch_err_aggregate(s) |
               fetch_err_update(s) | fetch_err_recode(s) |
               fetch_err_dyncache(s) | fetch_err_match(s);
    if (w & 0x80000000u) return fail(SG_ERR_CUDA, "sg_stream_check: could not read the device error word");
    if (w & ERR_INDEX) return fail(SG_ERR_INVALID_INDEX, "a kernel met a node ID or index out of range");
    if (w & ERR_CAPACITY) return fail(SG_ERR_CAPACITY, "a device table or buffer bound was exceeded");
    if (w & ERR_ARG) return fail(SG_ERR_INVALID_ARG, "a repeated seed / prefix ID was found on the device");
    if (w & ERR_TIMEOUT) return fail(SG_ERR_TIMEOUT, "a bounded device wait gave up");
    return SG_OK;
}

// -------------------------------------------------------------------- graph
extern "C" sg_status sg_graph_load(const void* h_indptr, int32_t offset_bits, const int32_t* h_indices,
                                   int64_t n_nodes, int64_t n_edges, sg_graph** out) {
    if (!out) return fail(SG_ERR_INVALID_ARG, "sg_graph_load: out is NULL");
    *out = nullptr;
    if (!h_indptr || (n_edges > 0 && !h_indices)) return fail(SG_ERR_INVALID_ARG, "sg_graph_load: NULL array");
    if (offset_bits != 32 && offset_bits != 64) return fail(SG_ERR_INVALID_ARG, "sg_graph_load: offset_bits must be 32 or 64");
    if (n_nodes <= 0 || n_nodes > 2147483647LL) return fail(SG_ERR_INVALID_ARG, "sg_graph_load: n_nodes out of range");
    if (n_edges < 0) return fail(SG_ERR_INVALID_ARG, "sg_graph_load: n_edges < 0");
    if (offset_bits == 32 && n_edges > 2147483647LL)
        return fail(SG_ERR_INVALID_ARG, "sg_graph_load: int32 offsets cannot hold %lld edges", (long long)n_edges);
    sg_graph* g = new (std::nothrow) sg_graph();
    if (!g) return fail(SG_ERR_OOM, "sg_graph_load: host allocation");
    g->n_nodes = n_nodes;
    g->n_edges = n_edges;
    g->offset_bits = offset_bits;
    const size_t ob = offset_bits / 8;
    cudaError_t e = dev_alloc(&g->indptr, (size_t)(n_nodes + 1) * ob);
    if (e == cudaSuccess) e = dev_alloc((void**)&g->indices, (size_t)(n_edges > 0 ? n_edges : 1) * sizeof(int32_t));
    void* scratch = nullptr;
    if (e == cudaSuccess) e = dev_alloc(&scratch, 64);
    if (e == cudaSuccess) e = cudaMemcpy(g->indptr, h_indptr, (size_t)(n_nodes + 1) * ob, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && n_edges > 0)
        e = cudaMemcpy(g->indices, h_indices, (size_t)n_edges * sizeof(int32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(scratch, 0, 64);
    unsigned bad = 0;
    unsigned long long maxdeg = 0;
    if (e == cudaSuccess) {
        unsigned* d_bad = (unsigned*)scratch;
        unsigned long long* d_max = (unsigned long long*)((char*)scratch + 8);
        const int blocks = num_sms() * 4;
        if (offset_bits == 32)
            k_validate_indptr<int32_t><<<blocks, 256>>>((const int32_t*)g->indptr, n_nodes, n_edges, d_bad, d_max);
        else
            k_validate_indptr<int64_t><<<blocks, 256>>>((const int64_t*)g->indptr, n_nodes, n_edges, d_bad, d_max);
        if (n_edges > 0) k_validate_indices<<<blocks, 256>>>(g->indices, n_edges, n_nodes, d_bad);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaMemcpy(&bad, d_bad, 4, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(&maxdeg, d_max, 8, cudaMemcpyDeviceToHost);
    }
    if (scratch) cudaFree(scratch);
    if (e != cudaSuccess) {
        sg_status s = cuda_fail(e, "sg_graph_load");
        sg_graph_destroy(g);
        return s;
    }
    if (bad) {
        sg_graph_destroy(g);
        return fail(SG_ERR_INVALID_ARG, (bad & 1u) ? "sg_graph_load: offsets must start at 0, not decrease and end at n_edges"
                                                   : "sg_graph_load: an index is outside [0, n_nodes)");
    }
    g->max_degree = (int64_t)maxdeg;
    *out = g;
    return SG_OK;
}

extern "C" sg_status sg_graph_destroy(sg_graph* g) {
    if (!g) return SG_OK;
    if (g->indptr) cudaFree(g->indptr);
    if (g->indices) cudaFree(g->indices);
    delete g;
    return SG_OK;
}

extern "C" sg_status sg_graph_info(const sg_graph* g, int64_t* n_nodes, int64_t* n_edges, int32_t* offset_bits,
                                   int64_t* max_degree) {
    if (!g) return fail(SG_ERR_INVALID_ARG, "sg_graph_info: NULL graph");
    if (n_nodes) *n_nodes = g->n_nodes;
    if (n_edges) *n_edges = g->n_edges;
    if (offset_bits) *offset_bits = g->offset_bits;
    if (max_degree) *max_degree = g->max_degree;
    return SG_OK;
}

extern "C" sg_status sg_graph_copy_out(const sg_graph* g, void* h_indptr, int32_t* h_indices) {
    if (!g || !h_indptr || (g->n_edges > 0 && !h_indices)) return fail(SG_ERR_INVALID_ARG, "sg_graph_copy_out: NULL argument");
    SG_CUDA(cudaMemcpy(h_indptr, g->indptr, (size_t)(g->n_nodes + 1) * (g->offset_bits / 8), cudaMemcpyDeviceToHost));
    if (g->n_edges > 0)
        SG_CUDA(cudaMemcpy(h_indices, g->indices, (size_t)g->n_edges * sizeof(int32_t), cudaMemcpyDeviceToHost));
    return SG_OK;
}

// -------------------------------------------------------------------- cache
extern "C" sg_status sg_cache_build(const void* h_feat, const void* d_feat, int32_t dtype, int64_t n_nodes, int32_t dim,
                                    const int32_t* h_ranked, int64_t n_cache, sg_cache** out, sg_stream_t stream) {
    if (!out) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: out is NULL");
    *out = nullptr;
    if (dtype != SG_F32 && dtype != SG_BF16) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: dtype");
    if (n_nodes <= 0 || n_nodes > 2147483647LL || dim <= 0) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: shape");
    if (n_cache < 0 || n_cache > n_nodes) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: n_cache outside [0, n_nodes]");
    const int64_t row_bytes = (int64_t)dim * (dtype == SG_F32 ? 4 : 2);
    if (row_bytes % 16) return fail(SG_ERR_UNSUPPORTED, "sg_cache_build: row bytes (%lld) must be a multiple of 16", (long long)row_bytes);
    if (!h_feat && !d_feat) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: no feature table");
    if (!h_feat && n_cache < n_nodes) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: uncached rows need the host table");
    cudaStream_t s = (cudaStream_t)stream;

    // A device-usable address for the host table (zero-copy reads of misses).
    const void* host_dev = nullptr;
    if (h_feat) {
        void* dp = nullptr;
        if (cudaHostGetDevicePointer(&dp, const_cast<void*>(h_feat), 0) == cudaSuccess && dp) {
            host_dev = dp;
        } else {
            cudaGetLastError();
            int dev = 0, pageable = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
            if (is_device_ptr(h_feat)) host_dev = h_feat;
            else if (pageable) host_dev = h_feat;
            else return fail(SG_ERR_INVALID_ARG, "sg_cache_build: host table is not pinned and the device cannot read pageable memory");
        }
        if (((uintptr_t)host_dev) % 16) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: host table must be 16-byte aligned");
    }
    if (d_feat && ((uintptr_t)d_feat) % 16) return fail(SG_ERR_INVALID_ARG, "sg_cache_build: d_feat must be 16-byte aligned");

    sg_cache* c = new (std::nothrow) sg_cache();
    if (!c) return fail(SG_ERR_OOM, "sg_cache_build: host allocation");
    c->n_nodes = n_nodes;
    c->dim = dim;
    c->dtype = dtype;
    c->row_bytes = row_bytes;
    c->n_cache = n_cache;
    c->host_rows = host_dev;
    // Tables of 32 GiB and more: misses can be read grouped by 2 MB region
    // (sg_gather with a workspace).  Measured on GB300 with random 512-byte
    // rows: a 16 GB pinned table reads at ~208 GB/s in any order, a 60 GB one
    // at ~10 GB/s in random order and ~40 GB/s grouped by region.
    if (host_dev && n_cache < n_nodes && n_nodes * row_bytes >= (int64_t(32) << 30)) {
        int32_t shift = 0;
        while ((int64_t(row_bytes) << (shift + 1)) <= (int64_t(2) << 20)) ++shift;
        c->region_shift = shift > 0 ? shift : 1;
        c->n_regions = ((n_nodes - 1) >> c->region_shift) + 1;
    }
    int32_t* d_ranked = nullptr;
    unsigned* d_bad = nullptr;
    // with a ranked list, a slot map; without, the ID range [0, n_cache)
    cudaError_t e = h_ranked ? dev_alloc((void**)&c->slot_of, (size_t)n_nodes * sizeof(int32_t)) : cudaSuccess;
    if (e == cudaSuccess && n_cache > 0) e = dev_alloc(&c->rows, (size_t)n_cache * (size_t)row_bytes);
    if (e == cudaSuccess && h_ranked && n_cache > 0) e = dev_alloc((void**)&d_ranked, (size_t)n_cache * sizeof(int32_t));
    if (e == cudaSuccess) e = dev_alloc((void**)&d_bad, 2 * sizeof(unsigned));  // flag, touch sink
    if (e == cudaSuccess) e = cudaMemsetAsync(d_bad, 0, sizeof(unsigned), s);
    if (e == cudaSuccess && c->slot_of) e = cudaMemsetAsync(c->slot_of, 0xFF, (size_t)n_nodes * sizeof(int32_t), s);
    if (e == cudaSuccess && d_ranked)
        e = cudaMemcpyAsync(d_ranked, h_ranked, (size_t)n_cache * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && n_cache > 0) {
        const int blocks = num_sms() * 8;
        k_cache_fill<<<blocks, 256, 0, s>>>(d_ranked, n_cache, n_nodes, (const uint4*)(d_feat ? d_feat : host_dev),
                                             row_bytes / 16, (uint4*)c->rows, c->slot_of);
        e = cudaGetLastError();
        if (e == cudaSuccess && d_ranked) {
            k_cache_check_distinct<<<blocks, 256, 0, s>>>(d_ranked, n_cache, c->slot_of, d_bad);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess && host_dev && n_cache < n_nodes) {
        // an ID-range cache never reads rows below n_cache from the host table
        const int64_t first = h_ranked ? 0 : n_cache;
        k_host_touch<<<num_sms() * 8, 256, 0, s>>>((const uint4*)((const char*)host_dev + first * row_bytes),
                                                   (n_nodes - first) * row_bytes / 16, d_bad + 1);
        e = cudaGetLastError();
    }
    unsigned bad = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&bad, d_bad, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (d_ranked) cudaFree(d_ranked);
    if (d_bad) cudaFree(d_bad);
    if (e != cudaSuccess) {
        sg_status st = cuda_fail(e, "sg_cache_build");
        sg_cache_destroy(c);
        return st;
    }
    unsigned w = fetch_err_api(s);
    if (bad || (w & ERR_INDEX)) {
        sg_cache_destroy(c);
        return fail(SG_ERR_INVALID_ARG, "sg_cache_build: ranked node IDs must be distinct and in [0, n_nodes)");
    }
    *out = c;
    return SG_OK;
}

extern "C" sg_status sg_cache_destroy(sg_cache* c) {
    if (!c) return SG_OK;
    dyn_cache_free(c);
    if (c->rows) cudaFree(c->rows);
    if (c->slot_of) cudaFree(c->slot_of);
    delete c;
    return SG_OK;
}

extern "C" sg_status sg_cache_info(const sg_cache* c, int64_t* n_nodes, int32_t* dim, int32_t* dtype, int64_t* n_cache,
                                   const int32_t** d_slot_of) {
    if (!c) return fail(SG_ERR_INVALID_ARG, "sg_cache_info: NULL cache");
    if (n_nodes) *n_nodes = c->n_nodes;
    if (dim) *dim = c->dim;
    if (dtype) *dtype = c->dtype;
    if (n_cache) *n_cache = c->n_cache;
    if (d_slot_of) *d_slot_of = c->slot_of;
    return SG_OK;
}

// ---------------------------------------------------------------- read probe
extern "C" sg_status sg_read_probe(const void* d_src, int64_t bytes, uint32_t* d_sink, sg_stream_t stream) {
    if (!d_src || !d_sink || bytes <= 0 || bytes % 16 || ((uintptr_t)d_src) % 16)
        return fail(SG_ERR_INVALID_ARG, "sg_read_probe: need a 16-byte aligned source and a multiple of 16 bytes");
    const int blocks = num_sms() * 8;
    k_read_probe<<<blocks, 256, 0, (cudaStream_t)stream>>>((const uint4*)d_src, bytes / 16, d_sink);
    SG_CHECK_LAUNCH("k_read_probe");
    return SG_OK;
}

extern "C" sg_status sg_wait_probe(int32_t n_tiles, int32_t silent_tile, int32_t spin_limit, void* d_workspace,
                                   size_t workspace_bytes, int32_t* d_out, sg_stream_t stream) {
    if (n_tiles <= 0 || n_tiles > 4096 || spin_limit <= 0 || spin_limit > kLookbackSpins || !d_out || !d_workspace)
        return fail(SG_ERR_INVALID_ARG, "sg_wait_probe: need 1..4096 tiles, a spin limit in 1..%d and buffers",
                    kLookbackSpins);
    const size_t need = sg_wait_probe_workspace(n_tiles);
    if (workspace_bytes < need || ((uintptr_t)d_workspace) % 256)
        return fail(SG_ERR_INVALID_ARG, "sg_wait_probe: workspace needs %zu bytes, 256-byte aligned", need);
    cudaStream_t s = (cudaStream_t)stream;
    unsigned long long* status = (unsigned long long*)d_workspace;
    unsigned* counter = (unsigned*)(status + n_tiles);
    SG_CUDA(cudaMemsetAsync(d_workspace, 0, need, s));
    k_wait_probe<<<n_tiles, 32, 0, s>>>(status, counter, silent_tile, spin_limit, d_out);
    SG_CHECK_LAUNCH("k_wait_probe");
    return SG_OK;
}

extern "C" size_t sg_wait_probe_workspace(int32_t n_tiles) {
    if (n_tiles <= 0) return 0;
    return (size_t)n_tiles * sizeof(unsigned long long) + 256;
}

extern "C" sg_status sg_hash_probe(int64_t n_calls, uint64_t seed, uint32_t* d_sink, sg_stream_t stream) {
    if (n_calls <= 0 || !d_sink) return fail(SG_ERR_INVALID_ARG, "sg_hash_probe: need n_calls > 0 and a sink");
    const int blocks = num_sms() * 8;
    k_hash_probe<<<blocks, 256, 0, (cudaStream_t)stream>>>(n_calls, (uint32_t)(seed & 0xFFFFFFFFull),
                                                           (uint32_t)(seed >> 32), d_sink);
    SG_CHECK_LAUNCH("k_hash_probe");
    return SG_OK;
}

// Feature gather through the HBM hot-node cache (GARDEN page, Section II-B,
// Fig. 2: Nfeat-Selecting reads cached rows from GPU memory and misses from
// pinned host memory over the host link, zero-copy).
//
// Layout: a feature row is row_bytes = dim * element size, a multiple of 16,
// so it moves as row_vecs 16-byte vectors.  The work is flattened over
// (row, vector) so that consecutive threads copy consecutive 16-byte pieces
// of the output: output stores are fully coalesced and each source row is
// read as a contiguous run, from the cache or from the host table.  Every
// thread keeps kUnroll (8) independent 16-byte loads in flight before it
// stores, which the latency of host-link reads needs.  Source rows are read
// with the streaming hint (each is used once here); the output is stored
// with the default policy, so that the first aggregation hop, which reads it
// next, finds part of it in L2.
//
// Hit test: with a slot map (a cache built from a ranked list), slot_of[g];
// without one (an ID-range cache, hot nodes recoded to the smallest IDs),
// node g is cached in slot g exactly when g < n_cache, and no map is read.
// A static miss is then looked up in the dynamic cache, when there is one
// (counted as a hit when found there).
//
// Large host tables (32 GiB and more) with a workspace: random zero-copy
// reads there lose most of their rate to address translation (measured on
// GB300, 512-byte rows: ~208 GB/s from a 16 GB pinned table in any order,
// ~10 GB/s from a 60 GB one in random order, ~40 GB/s grouped by 2 MB
// region).  So k_gather leaves the misses out and counts them per region;
// k_region_scan turns the counts into offsets, k_region_scatter lists the
// missed rows region by region (any order within a region), and
// k_gather_list copies them in list order.
#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(gather)

using namespace sgi;

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr int kListUnroll = 8;      // loads in flight a thread of k_gather_list
constexpr int kListBlocksPerSm = 8;

// cache slot of node g, or -1 when it is read from the host table
__device__ __forceinline__ int64_t slot_for(const int32_t* __restrict__ slot_of, int64_t n_cache, int32_t g) {
    if (slot_of) return __ldg(slot_of + g);
    return (int64_t)g < n_cache ? (int64_t)g : -1;
}

// The optional dynamic cache beside the static one: a static miss g is read
// from dyn_rows[dyn_slot[g]] when that slot is not -1.
struct DynView {
    const int32_t* slot;
    const uint4* rows;
};

// Optional reuse of the previous batch's rows (FastGL explainer page,
// "Match-Reorder"): row i with pos[i] >= 0 is copied from prev[pos[i]], the
// previous batch's gathered features still resident in HBM, and counted in
// *reused instead of hits or misses.
struct ReuseView {
    const int32_t* pos;
    const uint4* prev;
    unsigned long long* reused;
};

__global__ void __launch_bounds__(kThreads) k_gather(const int32_t* __restrict__ ids, const int32_t* __restrict__ d_n,
                                                     const int32_t* __restrict__ d_first,
                                                     int64_t n_cap, const int32_t* __restrict__ slot_of, int64_t n_cache,
                                                     int64_t n_nodes,
                                                     const uint4* __restrict__ cache, const uint4* __restrict__ host,
                                                     int32_t row_vecs, int64_t step_rows, int32_t step_rem,
                                                     uint4* __restrict__ out, sg_gather_stats* __restrict__ stats,
                                                     uint32_t* __restrict__ region_cnt, int32_t region_shift,
                                                     DynView dyn, ReuseView reuse) {
    pdl_start();
    int64_t n = n_cap;
    if (d_n) {
        const int64_t dn = *d_n;
        n = dn < n_cap ? (dn < 0 ? 0 : dn) : n_cap;
    }
    int64_t first = 0;
    if (d_first) {
        const int64_t df = *d_first;
        first = df < 0 ? 0 : (df < n ? df : n);
    }
    const int64_t total = n * row_vecs;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // (i, c) = (row, vector) of flat index t, advanced by the grid stride
    // without a division: stride = step_rows * row_vecs + step_rem.
    int64_t t = first * row_vecs + blockIdx.x * (int64_t)kThreads + threadIdx.x;
    int64_t i = t / row_vecs;
    int32_t c = (int32_t)(t - i * row_vecs);
    unsigned long long hits = 0, misses = 0, reused = 0;
    while (t < total) {
        uint4 v[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            dst[u] = -1;
            if (t < total) {
                const int32_t g = __ldg(ids + i);
                const int32_t rp = reuse.pos ? __ldg(reuse.pos + i) : -1;
                dst[u] = t;
                if (rp >= 0) {
                    v[u] = __ldcs(reuse.prev + (int64_t)rp * row_vecs + c);
                    reused += (c == 0);
                } else if (g < 0 || (int64_t)g >= n_nodes) {
                    if (c == 0) dev_err(ERR_INDEX);
                    v[u] = make_uint4(0, 0, 0, 0);
                } else {
                    const int64_t s = slot_for(slot_of, n_cache, g);
                    const int32_t ds = (s < 0 && dyn.slot) ? __ldg(dyn.slot + g) : -1;
                    if (s >= 0) {
                        v[u] = __ldcs(cache + (int64_t)s * row_vecs + c);
                        hits += (c == 0);
                    } else if (ds >= 0) {
                        v[u] = __ldcs(dyn.rows + (int64_t)ds * row_vecs + c);
                        hits += (c == 0);
                    } else if (region_cnt) {  // left for k_gather_list
                        if (c == 0) atomicAdd(region_cnt + (g >> region_shift), 1u);
                        dst[u] = -1;
                        misses += (c == 0);
                    } else {
                        v[u] = __ldcs(host + (int64_t)g * row_vecs + c);
                        misses += (c == 0);
                    }
                }
            }
            t += stride;
            i += step_rows;
            c += step_rem;
            if (c >= row_vecs) {
                c -= row_vecs;
                ++i;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dst[u] >= 0) out[dst[u]] = v[u];
    }
    if (stats) {
        hits = warp_sum(hits);
        misses = warp_sum(misses);
        if (lane_id() == 0 && (hits | misses)) {
            atomicAdd(&stats->hits, hits);
            atomicAdd(&stats->misses, misses);
        }
    }
    if (reuse.reused) {
        reused = warp_sum(reused);
        if (lane_id() == 0 && reused) atomicAdd(reuse.reused, reused);
    }
}

// Rows [first, n) of the call, from the device counts (as k_gather).
__device__ __forceinline__ void gather_range(const int32_t* d_n, const int32_t* d_first, int64_t n_cap, int64_t& first,
                                             int64_t& n) {
    n = n_cap;
    if (d_n) {
        const int64_t dn = *d_n;
        n = dn < n_cap ? (dn < 0 ? 0 : dn) : n_cap;
    }
    first = 0;
    if (d_first) {
        const int64_t df = *d_first;
        first = df < 0 ? 0 : (df < n ? df : n);
    }
}

// Exclusive scan of the n_regions miss counts in place (one block); the
// total goes to cnt[n_regions].  The counts are staged through shared memory
// with coalesced loads and stores (kScanSmemMax of them at most); each thread
// then scans a contiguous run of the staged copy.
constexpr int kScanThreads = 1024;
constexpr int64_t kScanSmemMax = 54 * 1024;  // counts staged in shared memory (216 KB)
__global__ void __launch_bounds__(kScanThreads) k_region_scan(uint32_t* __restrict__ cnt, int64_t n_regions) {
    pdl_start();
    extern __shared__ uint32_t staged[];
    __shared__ uint32_t sh[kScanThreads];
    const bool smem = n_regions <= kScanSmemMax;
    uint32_t* src = smem ? staged : cnt;
    if (smem) {
        for (int64_t r = threadIdx.x; r < n_regions; r += kScanThreads) staged[r] = cnt[r];
        __syncthreads();
    }
    const int64_t per = (n_regions + kScanThreads - 1) / kScanThreads;
    const int64_t a = min((int64_t)threadIdx.x * per, n_regions), b = min(a + per, n_regions);
    uint32_t sum = 0;
    for (int64_t r = a; r < b; ++r) sum += src[r];
    sh[threadIdx.x] = sum;
    __syncthreads();
    for (int d = 1; d < kScanThreads; d <<= 1) {  // inclusive scan of the run totals
        const uint32_t x = threadIdx.x >= (unsigned)d ? sh[threadIdx.x - d] : 0u;
        __syncthreads();
        sh[threadIdx.x] += x;
        __syncthreads();
    }
    uint32_t run = sh[threadIdx.x] - sum;
    for (int64_t r = a; r < b; ++r) {
        const uint32_t k = src[r];
        src[r] = run;
        run += k;
    }
    if (threadIdx.x == kScanThreads - 1) cnt[n_regions] = sh[kScanThreads - 1];
    if (smem) {
        __syncthreads();
        for (int64_t r = threadIdx.x; r < n_regions; r += kScanThreads) cnt[r] = staged[r];
    }
}

// Lists the missed rows i in [first, n) by region: list[pos] = i, pos taken
// from the region's offset.
__global__ void __launch_bounds__(kThreads) k_region_scatter(const int32_t* __restrict__ ids,
                                                             const int32_t* __restrict__ d_n,
                                                             const int32_t* __restrict__ d_first, int64_t n_cap,
                                                             const int32_t* __restrict__ slot_of, int64_t n_cache,
                                                             int64_t n_nodes,
                                                             uint32_t* __restrict__ cnt, int32_t region_shift,
                                                             int32_t* __restrict__ list, DynView dyn,
                                                             const int32_t* __restrict__ reuse_pos) {
    pdl_start();
    int64_t first, n;
    gather_range(d_n, d_first, n_cap, first, n);
    for (int64_t i = first + blockIdx.x * (int64_t)kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        const int32_t g = __ldg(ids + i);
        if (g < 0 || (int64_t)g >= n_nodes) continue;
        if (reuse_pos && __ldg(reuse_pos + i) >= 0) continue;
        if (slot_for(slot_of, n_cache, g) >= 0) continue;
        if (dyn.slot && __ldg(dyn.slot + g) >= 0) continue;
        const uint32_t pos = atomicAdd(cnt + (g >> region_shift), 1u);
        if ((int64_t)pos < n_cap) list[pos] = (int32_t)i;
        else dev_err(ERR_CAPACITY);
    }
}

// Copies the listed rows from the host table, flattened over (entry,
// vector) with kListUnroll loads in flight a thread, in list order, at full
// occupancy (eight blocks an SM).  Reads of rows not read before are bound by
// address translation, and more requests in flight help: in the benchmark on
// the 57 GB Billion-edge table (CUDA events, each gather reading new rows),
// 8 loads x 8 blocks an SM gave 1.37 ms a step at the median against 1.38
// (16 x 4), 1.39 (8 x 4) and 1.53 (16 x 1).  (Re-reading rows just read runs
// several times faster; such repeated reads are not what a batch does.)
__global__ void __launch_bounds__(kThreads, kListBlocksPerSm) k_gather_list(const int32_t* __restrict__ list,
                                                          const uint32_t* __restrict__ total,
                                                          const int32_t* __restrict__ ids,
                                                          const uint4* __restrict__ host, int32_t row_vecs,
                                                          int64_t n_cap, uint4* __restrict__ out) {
    pdl_start();
    int64_t m = *total;
    if (m > n_cap) m = n_cap;
    const int64_t work = m * row_vecs;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // piece t of the list is vector t % row_vecs of entry t / row_vecs; a
    // thread loads kListUnroll pieces a grid stride apart, then stores them
    for (int64_t t0 = blockIdx.x * (int64_t)kThreads + threadIdx.x; t0 < work; t0 += stride * kListUnroll) {
        uint4 v[kListUnroll];
#pragma unroll
        for (int u = 0; u < kListUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < work) {
                const int64_t j = t / row_vecs;
                v[u] = __ldcs(host + (int64_t)__ldg(ids + __ldg(list + j)) * row_vecs + (t - j * row_vecs));
            }
        }
#pragma unroll
        for (int u = 0; u < kListUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < work) {
                const int64_t j = t / row_vecs;
                out[(int64_t)__ldg(list + j) * row_vecs + (t - j * row_vecs)] = v[u];
            }
        }
    }
}

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" size_t sg_gather_workspace(const sg_cache* c, int64_t n_cap) {
    if (!c || c->region_shift <= 0 || n_cap <= 0) return 0;
    return a256((size_t)(c->n_regions + 1) * sizeof(uint32_t)) + a256((size_t)n_cap * sizeof(int32_t));
}

namespace {
sg_status gather_impl(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                      const int32_t* d_first, void* d_out, sg_gather_stats* d_stats, void* d_workspace,
                      size_t workspace_bytes, ReuseView reuse, sg_stream_t stream) {
    if (!c) return fail(SG_ERR_INVALID_ARG, "sg_gather: NULL cache");
    if (n_cap < 0) return fail(SG_ERR_INVALID_ARG, "sg_gather: n_cap < 0");
    if (n_cap == 0) return SG_OK;
    if (!d_ids || !d_out) return fail(SG_ERR_INVALID_ARG, "sg_gather: NULL ids or out");
    if (((uintptr_t)d_out) % 16) return fail(SG_ERR_INVALID_ARG, "sg_gather: out must be 16-byte aligned");
    if (c->n_cache < c->n_nodes && !c->host_rows)
        return fail(SG_ERR_INVALID_ARG, "sg_gather: cache has no host table for misses");
    const int64_t row_vecs = c->row_bytes / 16;
    const int64_t work = n_cap * row_vecs;
    int64_t blocks = cdiv(work, (int64_t)kThreads * kUnroll);
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const int64_t stride = blocks * kThreads;
    cudaStream_t s = (cudaStream_t)stream;
    // misses grouped by host-table region (large tables, with a workspace)
    const size_t need = sg_gather_workspace(c, n_cap);
    const bool by_region = d_workspace && need > 0;
    if (by_region && workspace_bytes < need)
        return fail(SG_ERR_INVALID_ARG, "sg_gather: workspace needs %zu bytes", need);
    if (by_region && ((uintptr_t)d_workspace) % 256)
        return fail(SG_ERR_INVALID_ARG, "sg_gather: workspace must be 256-byte aligned");
    uint32_t* cnt = by_region ? (uint32_t*)d_workspace : nullptr;
    int32_t* list = by_region ? (int32_t*)((char*)d_workspace + a256((size_t)(c->n_regions + 1) * sizeof(uint32_t)))
                              : nullptr;
    if (by_region) SG_CUDA(cudaMemsetAsync(cnt, 0, (size_t)(c->n_regions + 1) * sizeof(uint32_t), s));
    DynView dyn;
    dyn.slot = c->dyn ? c->dyn->slot : nullptr;
    dyn.rows = c->dyn ? (const uint4*)c->dyn->rows : nullptr;
    SG_CUDA(launch_pdl(k_gather, dim3((unsigned)blocks), dim3(kThreads), 0, s, d_ids, d_n, d_first,
                       n_cap, c->slot_of, c->n_cache, c->n_nodes, (const uint4*)c->rows, (const uint4*)c->host_rows,
                       (int32_t)row_vecs, stride / row_vecs, (int32_t)(stride % row_vecs), (uint4*)d_out, d_stats,
                       cnt, c->region_shift, dyn, reuse));
    if (!by_region) return SG_OK;
    const size_t scan_smem = c->n_regions <= kScanSmemMax ? (size_t)c->n_regions * sizeof(uint32_t) : 0;
    if (scan_smem > 48 * 1024) {
        static bool attr_set[64] = {false};  // per device
        int dev = 0;
        SG_CUDA(cudaGetDevice(&dev));
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            SG_CUDA(cudaFuncSetAttribute(k_region_scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kScanSmemMax * sizeof(uint32_t))));
            attr_set[dev] = true;
        }
    }
    SG_CUDA(launch_pdl(k_region_scan, dim3(1), dim3(kScanThreads), scan_smem, s, cnt, c->n_regions));
    int64_t sblocks = cdiv(n_cap, (int64_t)kThreads);
    if (sblocks > cap) sblocks = cap;
    SG_CUDA(launch_pdl(k_region_scatter, dim3((unsigned)sblocks), dim3(kThreads), 0, s, d_ids, d_n, d_first, n_cap,
                       c->slot_of, c->n_cache, c->n_nodes, cnt, c->region_shift, list, dyn, reuse.pos));
    int64_t lblocks = cdiv(work, (int64_t)kThreads * kListUnroll);
    const int64_t lcap = (int64_t)num_sms() * kListBlocksPerSm;
    if (lblocks > lcap) lblocks = lcap;
    if (lblocks < 1) lblocks = 1;
    SG_CUDA(launch_pdl(k_gather_list, dim3((unsigned)lblocks), dim3(kThreads), 0, s, (const int32_t*)list,
                       (const uint32_t*)(cnt + c->n_regions), d_ids, (const uint4*)c->host_rows, (int32_t)row_vecs,
                       n_cap, (uint4*)d_out));
    return SG_OK;
}
}  // namespace

extern "C" sg_status sg_gather(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                               const int32_t* d_first, void* d_out, sg_gather_stats* d_stats, void* d_workspace,
                               size_t workspace_bytes, sg_stream_t stream) {
    ReuseView none = {nullptr, nullptr, nullptr};
    return gather_impl(c, d_ids, n_cap, d_n, d_first, d_out, d_stats, d_workspace, workspace_bytes, none, stream);
}

extern "C" sg_status sg_gather_reuse(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                                     const int32_t* d_first, const int32_t* d_pos, const void* d_prev_rows,
                                     void* d_out, sg_gather_stats* d_stats, unsigned long long* d_reused,
                                     void* d_workspace, size_t workspace_bytes, sg_stream_t stream) {
    if (!d_pos || !d_prev_rows) return fail(SG_ERR_INVALID_ARG, "sg_gather_reuse: NULL match positions or rows");
    if (((uintptr_t)d_prev_rows) % 16) return fail(SG_ERR_INVALID_ARG, "sg_gather_reuse: rows must be 16-byte aligned");
    ReuseView r = {d_pos, (const uint4*)d_prev_rows, d_reused};
    return gather_impl(c, d_ids, n_cap, d_n, d_first, d_out, d_stats, d_workspace, workspace_bytes, r, stream);
}

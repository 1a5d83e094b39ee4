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
#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(gather)

using namespace sgi;

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) k_gather(const int32_t* __restrict__ ids, const int32_t* __restrict__ d_n,
                                                     const int32_t* __restrict__ d_first,
                                                     int64_t n_cap, const int32_t* __restrict__ slot_of, int64_t n_nodes,
                                                     const uint4* __restrict__ cache, const uint4* __restrict__ host,
                                                     int32_t row_vecs, int64_t step_rows, int32_t step_rem,
                                                     uint4* __restrict__ out, sg_gather_stats* __restrict__ stats) {
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
    unsigned long long hits = 0, misses = 0;
    while (t < total) {
        uint4 v[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            dst[u] = -1;
            if (t < total) {
                const int32_t g = __ldg(ids + i);
                dst[u] = t;
                if (g < 0 || (int64_t)g >= n_nodes) {
                    if (c == 0) dev_err(ERR_INDEX);
                    v[u] = make_uint4(0, 0, 0, 0);
                } else {
                    const int32_t s = __ldg(slot_of + g);
                    if (s >= 0) {
                        v[u] = __ldcs(cache + (int64_t)s * row_vecs + c);
                        hits += (c == 0);
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
}

}  // namespace

extern "C" sg_status sg_gather(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                               const int32_t* d_first, void* d_out, sg_gather_stats* d_stats, sg_stream_t stream) {
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
    SG_CUDA(launch_pdl(k_gather, dim3((unsigned)blocks), dim3(kThreads), 0, (cudaStream_t)stream, d_ids, d_n, d_first,
                       n_cap, c->slot_of, c->n_nodes, (const uint4*)c->rows, (const uint4*)c->host_rows,
                       (int32_t)row_vecs, stride / row_vecs, (int32_t)(stride % row_vecs), (uint4*)d_out, d_stats));
    return SG_OK;
}

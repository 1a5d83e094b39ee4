// Match and reorder of consecutive batches (FastGL explainer page,
// "Match-Reorder"): consecutive sampled subgraphs share many nodes, so a
// batch copies the features of the nodes it shares with the previous batch
// from that batch's rows, still resident in HBM, and ships only the rest
// (sg_gather_reuse); a group of batches is ordered so that each follows the
// one it overlaps most (nearest overlap first).
//
// Both use a caller-owned direct map over the node IDs, idle when all ones
// (match: the previous batch's position of a node) or all zeros (overlap:
// a bit per batch of the group); each call leaves it idle again.
#include <string.h>

#include "sg_internal.cuh"

SGI_ERROR_WORD(match)

using namespace sgi;

namespace {

constexpr int kNT = 256;
constexpr int kMaxGroup = 32;

__device__ __forceinline__ int64_t count_of(const int32_t* d_n, int64_t cap) {
    if (!d_n) return cap;
    const int64_t v = *d_n;
    return v < 0 ? 0 : (v < cap ? v : cap);
}

// map[prev[i]] = i
__global__ void k_match_mark(const int32_t* __restrict__ prev, int64_t cap, const int32_t* __restrict__ d_n,
                             int32_t* __restrict__ map, int64_t n_nodes) {
    const int64_t n = count_of(d_n, cap);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = prev[i];
        if (v < 0 || (int64_t)v >= n_nodes) dev_err(ERR_INDEX);
        else map[v] = (int32_t)i;
    }
}

// pos[j] = map[cur[j]] (-1 when absent); *matched += the found count
__global__ void __launch_bounds__(kNT) k_match_lookup(const int32_t* __restrict__ cur, int64_t cap,
                                                      const int32_t* __restrict__ d_n,
                                                      const int32_t* __restrict__ map, int64_t n_nodes,
                                                      int32_t* __restrict__ pos, int32_t* __restrict__ matched) {
    const int64_t n = count_of(d_n, cap);
    int32_t found = 0;
    for (int64_t j = blockIdx.x * (int64_t)kNT + threadIdx.x; j < n; j += (int64_t)gridDim.x * kNT) {
        const int32_t v = cur[j];
        int32_t p = -1;
        if (v < 0 || (int64_t)v >= n_nodes) dev_err(ERR_INDEX);
        else p = map[v];
        pos[j] = p;
        found += p >= 0;
    }
    found = warp_sum(found);
    if (matched && lane_id() == 0 && found) atomicAdd(matched, found);
}

// map[prev[i]] = -1 (back to idle)
__global__ void k_match_clear(const int32_t* __restrict__ prev, int64_t cap, const int32_t* __restrict__ d_n,
                              int32_t* __restrict__ map, int64_t n_nodes) {
    const int64_t n = count_of(d_n, cap);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = prev[i];
        if (v >= 0 && (int64_t)v < n_nodes) map[v] = -1;
    }
}

struct Group {
    const int32_t* ids;
    int64_t off[kMaxGroup + 1];
    int32_t G;
};

// list a sets bit a of mask[v] for its nodes
__global__ void k_ov_mark(Group g, uint32_t* __restrict__ mask, int64_t n_nodes) {
    const int64_t total = g.off[g.G];
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int a = 0;
        while (a + 1 < g.G && g.off[a + 1] <= i) ++a;
        const int32_t v = g.ids[i];
        if (v < 0 || (int64_t)v >= n_nodes) dev_err(ERR_INDEX);
        else atomicOr(mask + v, 1u << a);
    }
}

// O[b][a] += 1 for every node of list b whose mask has bit a; a block sums
// into shared counters first
__global__ void __launch_bounds__(kNT) k_ov_count(Group g, const uint32_t* __restrict__ mask, int64_t n_nodes,
                                                  unsigned long long* __restrict__ O) {
    __shared__ unsigned int cnt[kMaxGroup * kMaxGroup];
    const int GG = g.G * g.G;
    for (int t = threadIdx.x; t < GG; t += kNT) cnt[t] = 0;
    __syncthreads();
    const int64_t total = g.off[g.G];
    for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < total; i += (int64_t)gridDim.x * kNT) {
        int b = 0;
        while (b + 1 < g.G && g.off[b + 1] <= i) ++b;
        const int32_t v = g.ids[i];
        if (v < 0 || (int64_t)v >= n_nodes) continue;
        uint32_t m = mask[v];
        while (m) {
            const int a = __ffs(m) - 1;
            m &= m - 1;
            atomicAdd(&cnt[b * g.G + a], 1u);
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < GG; t += kNT)
        if (cnt[t]) atomicAdd(O + t, (unsigned long long)cnt[t]);
}

__global__ void k_ov_clear(Group g, uint32_t* __restrict__ mask, int64_t n_nodes) {
    const int64_t total = g.off[g.G];
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = g.ids[i];
        if (v >= 0 && (int64_t)v < n_nodes) mask[v] = 0;
    }
}

int grid_for(int64_t n) {
    int64_t b = cdiv(n, kNT);
    const int64_t cap = (int64_t)num_sms() * 8;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

}  // namespace

extern "C" sg_status sg_match(const int32_t* d_prev, int64_t prev_cap, const int32_t* d_prev_n, const int32_t* d_cur,
                              int64_t cur_cap, const int32_t* d_cur_n, int32_t* d_map, int64_t n_nodes,
                              int32_t* d_pos, int32_t* d_matched, sg_stream_t stream) {
    if (prev_cap < 0 || cur_cap < 0 || n_nodes <= 0) return fail(SG_ERR_INVALID_ARG, "sg_match: sizes out of range");
    if ((prev_cap > 0 && !d_prev) || (cur_cap > 0 && (!d_cur || !d_pos)) || !d_map)
        return fail(SG_ERR_INVALID_ARG, "sg_match: NULL array");
    cudaStream_t s = (cudaStream_t)stream;
    if (prev_cap > 0) k_match_mark<<<grid_for(prev_cap), kNT, 0, s>>>(d_prev, prev_cap, d_prev_n, d_map, n_nodes);
    if (cur_cap > 0)
        k_match_lookup<<<grid_for(cur_cap), kNT, 0, s>>>(d_cur, cur_cap, d_cur_n, d_map, n_nodes, d_pos, d_matched);
    if (prev_cap > 0) k_match_clear<<<grid_for(prev_cap), kNT, 0, s>>>(d_prev, prev_cap, d_prev_n, d_map, n_nodes);
    SG_CHECK_LAUNCH("sg_match");
    return SG_OK;
}

extern "C" sg_status sg_overlap(const int32_t* d_ids, const int64_t* h_off, int32_t n_lists, uint32_t* d_mask,
                                int64_t n_nodes, unsigned long long* d_overlap, sg_stream_t stream) {
    if (n_lists < 1 || n_lists > kMaxGroup || !h_off || !d_mask || !d_overlap || n_nodes <= 0)
        return fail(SG_ERR_INVALID_ARG, "sg_overlap: 1..%d lists, offsets, mask and output needed", kMaxGroup);
    Group g;
    memset(&g, 0, sizeof(g));
    g.ids = d_ids;
    g.G = n_lists;
    for (int a = 0; a <= n_lists; ++a) {
        g.off[a] = h_off[a];
        if (a > 0 && h_off[a] < h_off[a - 1]) return fail(SG_ERR_INVALID_ARG, "sg_overlap: offsets must not decrease");
    }
    if (h_off[0] != 0) return fail(SG_ERR_INVALID_ARG, "sg_overlap: offsets must start at 0");
    cudaStream_t s = (cudaStream_t)stream;
    SG_CUDA(cudaMemsetAsync(d_overlap, 0, (size_t)n_lists * n_lists * sizeof(unsigned long long), s));
    const int64_t total = g.off[n_lists];
    if (total == 0) return SG_OK;
    if (!d_ids) return fail(SG_ERR_INVALID_ARG, "sg_overlap: NULL IDs");
    k_ov_mark<<<grid_for(total), kNT, 0, s>>>(g, d_mask, n_nodes);
    k_ov_count<<<grid_for(total), kNT, 0, s>>>(g, d_mask, n_nodes, d_overlap);
    k_ov_clear<<<grid_for(total), kNT, 0, s>>>(g, d_mask, n_nodes);
    SG_CHECK_LAUNCH("sg_overlap");
    return SG_OK;
}

extern "C" sg_status sg_greedy_order(const unsigned long long* h_overlap, int32_t n_lists, int32_t first,
                                     int32_t* h_order) {
    if (!h_overlap || !h_order || n_lists < 1 || n_lists > 1024 || first < 0 || first >= n_lists)
        return fail(SG_ERR_INVALID_ARG, "sg_greedy_order: 1..1024 lists and a first list in range");
    unsigned char taken[1024];
    memset(taken, 0, sizeof(taken));
    h_order[0] = first;
    taken[first] = 1;
    for (int32_t k = 1; k < n_lists; ++k) {
        const int32_t last = h_order[k - 1];
        int32_t best = -1;
        for (int32_t b = 0; b < n_lists; ++b) {
            if (taken[b]) continue;
            if (best < 0 || h_overlap[(int64_t)last * n_lists + b] > h_overlap[(int64_t)last * n_lists + best]) best = b;
        }
        h_order[k] = best;
        taken[best] = 1;
    }
    return SG_OK;
}

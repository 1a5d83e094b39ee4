// The bounded dynamic cache beside the static feature cache (GARDEN page,
// Section IV-B, "Adaptive Dynamic Feature Caching", Eq. (5)-(6)).
//
// Scores follow Eq. (5) over the nodes each batch misses in the static
// cache, in the windowed fixed-point form (gamma = g / 2^16, 8 fractional
// bits): batch j of a window of T batches adds W_j = gamma^(T-1-j) (Q8) to
// A[v] for each of its static misses v (integer atomics, so the sum does not
// depend on their order); at the end of the window
//   S[v] = (S[v] * gamma^T >> 16) + A[v],  A[v] = 0
// and the k_dyn nodes of largest S (ties by ascending ID, S > 0 only) become
// the dynamic set (Eq. (6), the Top-K).  The set is found by radix selection,
// not by ranking every node: four passes of 8-bit histograms over the nonzero
// scores (the first folded into the update of S) give the k_dyn-th largest
// score T and how many nodes scoring exactly T are still needed, r; four more
// over the IDs of the nodes scoring T give the r-th smallest of those IDs, I.
// The set is then {S > T} plus {S = T, ID <= I}, or every node with S > 0
// when there are no more than k_dyn of them.  Nodes that stay keep their slot;
// leaving nodes free theirs, and only the entering nodes' rows are copied
// from the host table.  The gather looks a static miss up in the dynamic
// slot map before reading the host table.
#include <string.h>

#include <new>

#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(dyncache)

using namespace sgi;

namespace {

constexpr int kNT = 256;
constexpr int32_t kKeep = 1 << 30;  // slot tag: the node stays in the new set

__device__ __forceinline__ bool static_hit(const int32_t* slot_of, int64_t n_cache, int32_t v) {
    return slot_of ? slot_of[v] >= 0 : (int64_t)v < n_cache;
}

// A[v] += w for every static miss v among the batch's n nodes
__global__ void __launch_bounds__(kNT) k_dyn_accumulate(const int32_t* __restrict__ ids, int64_t n_cap,
                                                        const int32_t* __restrict__ d_n,
                                                        const int32_t* __restrict__ slot_of, int64_t n_cache,
                                                        int64_t n_nodes, uint32_t w, uint32_t* __restrict__ A) {
    int64_t n = n_cap;
    if (d_n) n = min((int64_t)max(*d_n, 0), n_cap);
    for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < n; i += (int64_t)gridDim.x * kNT) {
        const int32_t v = ids[i];
        if (v < 0 || (int64_t)v >= n_nodes) {
            dev_err(ERR_INDEX);
            continue;
        }
        if (!static_hit(slot_of, n_cache, v)) atomicAdd(A + v, w);
    }
}

// The selection state in d->sel: a 256-bin histogram, then the parameters.
constexpr int kHist = 0;
constexpr int kMode = 256;   // kSelect, or kAll when every nonzero score is in the set
constexpr int kSPre = 257;   // the score bits chosen so far (T after four passes)
constexpr int kSNeed = 258;  // rank, descending, of the k_dyn-th score within them
constexpr int kIPre = 259;   // the ID bits chosen so far (I after four passes)
constexpr int kINeed = 260;  // rank, ascending, of the r-th tie ID within them
constexpr int kSelWords = 512;
constexpr uint32_t kSelect = 1, kAll = 2;

// Adds a block's shared histogram into the selection histogram.
__device__ __forceinline__ void flush_hist(const uint32_t* h, uint32_t* sel) {
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += kNT)
        if (h[i]) atomicAdd(sel + kHist + i, h[i]);
}

// S = (S * G >> 16) + A, A = 0; the nonzero scores binned by their top byte
// (the selection's first pass)
__global__ void __launch_bounds__(kNT) k_dyn_fold(uint32_t* __restrict__ S, uint32_t* __restrict__ A, int64_t n,
                                                  uint32_t G, uint32_t* __restrict__ sel) {
    __shared__ uint32_t h[256];
    for (int i = threadIdx.x; i < 256; i += kNT) h[i] = 0;
    __syncthreads();
    for (int64_t v = blockIdx.x * (int64_t)kNT + threadIdx.x; v < n; v += (int64_t)gridDim.x * kNT) {
        const uint32_t s = (uint32_t)(((uint64_t)S[v] * G) >> 16) + A[v];
        S[v] = s;
        A[v] = 0;
        if (s) atomicAdd(&h[s >> 24], 1u);
    }
    flush_hist(h, sel);
}

// Score pass p = 1..3: nonzero scores whose top 8p bits are the chosen
// prefix, binned by their next byte.
__global__ void __launch_bounds__(kNT) k_sel_score_hist(const uint32_t* __restrict__ S, int64_t n, int p,
                                                        uint32_t* __restrict__ sel) {
    if (sel[kMode] != kSelect) return;
    __shared__ uint32_t h[256];
    for (int i = threadIdx.x; i < 256; i += kNT) h[i] = 0;
    __syncthreads();
    const uint32_t pre = sel[kSPre];
    const int sh = 32 - 8 * p;
    for (int64_t v = blockIdx.x * (int64_t)kNT + threadIdx.x; v < n; v += (int64_t)gridDim.x * kNT) {
        const uint32_t s = S[v];
        if (s && (s >> sh) == pre) atomicAdd(&h[(s >> (sh - 8)) & 255u], 1u);
    }
    flush_hist(h, sel);
}

// After score pass p: the bin holding the score of descending rank need
// (the k_dyn-th largest at p = 0) joins the prefix and need drops by the
// counts of the bins above it.  At p = 0, no more than k_dyn nonzero scores
// select them all.  The histogram is cleared for the next pass.
__global__ void k_sel_score_pick(uint32_t* __restrict__ sel, int p, int64_t k) {
    if (threadIdx.x != 0) return;
    uint32_t* h = sel + kHist;
    if (p == 0) {
        uint64_t tot = 0;
        for (int b = 0; b < 256; ++b) tot += h[b];
        sel[kMode] = tot <= (uint64_t)k ? kAll : kSelect;
        sel[kSPre] = 0;
        sel[kSNeed] = (uint32_t)k;
    }
    if (sel[kMode] == kSelect) {
        uint32_t need = sel[kSNeed];
        int b = 255;
        for (; b > 0 && h[b] < need; --b) need -= h[b];
        sel[kSPre] = (sel[kSPre] << 8) | (uint32_t)b;
        sel[kSNeed] = need;
    }
    for (int b = 0; b < 256; ++b) h[b] = 0;
}

// ID pass q = 0..3 over the nodes scoring T: IDs whose top 8q bits are the
// chosen prefix, binned by their next byte.
__global__ void __launch_bounds__(kNT) k_sel_id_hist(const uint32_t* __restrict__ S, int64_t n, int q,
                                                     uint32_t* __restrict__ sel) {
    if (sel[kMode] != kSelect) return;
    __shared__ uint32_t h[256];
    for (int i = threadIdx.x; i < 256; i += kNT) h[i] = 0;
    __syncthreads();
    const uint32_t T = sel[kSPre], pre = sel[kIPre];
    const int sh = 32 - 8 * q;
    for (int64_t v = blockIdx.x * (int64_t)kNT + threadIdx.x; v < n; v += (int64_t)gridDim.x * kNT) {
        const uint32_t id = (uint32_t)v;
        if (S[v] == T && (q == 0 || (id >> sh) == pre)) atomicAdd(&h[(id >> (sh - 8)) & 255u], 1u);
    }
    flush_hist(h, sel);
}

// After ID pass q: the bin holding the tie ID of ascending rank need (r at
// q = 0) joins the prefix.
__global__ void k_sel_id_pick(uint32_t* __restrict__ sel, int q) {
    if (threadIdx.x != 0) return;
    uint32_t* h = sel + kHist;
    if (sel[kMode] == kSelect) {
        if (q == 0) {
            sel[kIPre] = 0;
            sel[kINeed] = sel[kSNeed];
        }
        uint32_t need = sel[kINeed];
        int b = 0;
        for (; b < 255 && h[b] < need; ++b) need -= h[b];
        sel[kIPre] = (sel[kIPre] << 8) | (uint32_t)b;
        sel[kINeed] = need;
    }
    for (int b = 0; b < 256; ++b) h[b] = 0;
}

// The new set is {S > T} u {S = T, ID <= I} (or {S > 0}, see k_sel_score_pick).
// A node of it that holds a slot is tagged to keep it; the others are listed
// as entering.  cnt[0] counts them.
__global__ void __launch_bounds__(kNT) k_dyn_mark(const uint32_t* __restrict__ S, int64_t n,
                                                  const uint32_t* __restrict__ sel, int32_t* __restrict__ slot,
                                                  int32_t* __restrict__ enter, int32_t* __restrict__ cnt) {
    const bool all = sel[kMode] == kAll;
    const uint32_t T = sel[kSPre], I = sel[kIPre];
    for (int64_t v = blockIdx.x * (int64_t)kNT + threadIdx.x; v < n; v += (int64_t)gridDim.x * kNT) {
        const uint32_t s = S[v];
        const bool in = all ? s > 0u : (s > T || (s == T && (uint32_t)v <= I));
        if (!in) continue;
        if (slot[v] >= 0) slot[v] |= kKeep;
        else enter[atomicAdd(cnt, 1)] = (int32_t)v;
    }
}

// Slots whose node left are freed (listed in cnt[1]); kept nodes lose the tag.
__global__ void k_dyn_evict(int32_t* __restrict__ nodes, int64_t k, int32_t* __restrict__ slot,
                            int32_t* __restrict__ free_slots, int32_t* __restrict__ cnt) {
    for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s < k; s += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = nodes[s];
        if (v >= 0 && (slot[v] & kKeep)) {
            slot[v] &= ~kKeep;
            continue;
        }
        if (v >= 0) {
            slot[v] = -1;
            nodes[s] = -1;
        }
        free_slots[atomicAdd(cnt + 1, 1)] = (int32_t)s;
    }
}

// Entering node i takes free slot i; its row is copied from the host table
// (flattened over (entry, 16-byte vector)).
__global__ void __launch_bounds__(kNT) k_dyn_admit(const int32_t* __restrict__ enter,
                                                   const int32_t* __restrict__ free_slots,
                                                   const int32_t* __restrict__ cnt, int32_t* __restrict__ nodes,
                                                   int32_t* __restrict__ slot, const uint4* __restrict__ host,
                                                   int64_t row_vecs, uint4* __restrict__ rows) {
    const int64_t m = cnt[0] < cnt[1] ? cnt[0] : cnt[1];
    for (int64_t t = blockIdx.x * (int64_t)kNT + threadIdx.x; t < m * row_vecs; t += (int64_t)gridDim.x * kNT) {
        const int64_t i = t / row_vecs, c = t - i * row_vecs;
        const int32_t v = enter[i], s = free_slots[i];
        if (c == 0) {
            nodes[s] = v;
            slot[v] = s;
        }
        rows[(int64_t)s * row_vecs + c] = __ldcs(host + (int64_t)v * row_vecs + c);
    }
}

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

void dyn_free(sg_dyn* d) {
    if (!d) return;
    cudaFree(d->rows);
    cudaFree(d->slot);
    cudaFree(d->nodes);
    cudaFree(d->S);
    cudaFree(d->A);
    cudaFree(d->sel);
    cudaFree(d->lists);
    delete d;
}

}  // namespace

namespace sgi {
void dyn_cache_free(sg_cache* c) {
    if (c && c->dyn) {
        dyn_free(c->dyn);
        c->dyn = nullptr;
    }
}
}  // namespace sgi

extern "C" sg_status sg_dyn_cache_create(sg_cache* c, int64_t k_dyn, uint32_t gamma_q16, int32_t t_update,
                                         sg_stream_t stream) {
    if (!c) return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_create: NULL cache");
    if (c->dyn) return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_create: the cache has a dynamic cache already");
    if (!c->host_rows || c->n_cache >= c->n_nodes)
        return fail(SG_ERR_UNSUPPORTED, "sg_dyn_cache_create: the cache holds every row (no host table to supplement)");
    if (k_dyn <= 0 || k_dyn > c->n_nodes - c->n_cache || k_dyn >= kKeep)
        return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_create: k_dyn must be in [1, uncached rows]");
    if (gamma_q16 == 0 || gamma_q16 > 65536 || t_update < 1 || t_update > kDynMaxWindow)
        return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_create: gamma_q16 in [1, 65536], t_update in [1, %d]",
                    kDynMaxWindow);
    sg_dyn* d = new (std::nothrow) sg_dyn();
    if (!d) return fail(SG_ERR_OOM, "sg_dyn_cache_create: host allocation");
    d->k_dyn = k_dyn;
    d->T = t_update;
    d->W[t_update - 1] = 256;
    for (int j = t_update - 1; j > 0; --j) d->W[j - 1] = (uint32_t)(((uint64_t)d->W[j] * gamma_q16) >> 16);
    uint64_t G = gamma_q16;
    for (int i = 1; i < t_update; ++i) G = (G * gamma_q16) >> 16;
    d->G_T = (uint32_t)G;
    const int64_t n = c->n_nodes;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = dev_alloc(&d->rows, (size_t)k_dyn * c->row_bytes);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->slot, (size_t)n * 4);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->nodes, (size_t)k_dyn * 4);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->S, (size_t)n * 4);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->A, (size_t)n * 4);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->sel, (size_t)kSelWords * 4);
    if (e == cudaSuccess) e = dev_alloc((void**)&d->lists, a256((size_t)(2 * k_dyn + 8) * 4));
    if (e == cudaSuccess) e = cudaMemsetAsync(d->slot, 0xFF, (size_t)n * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d->nodes, 0xFF, (size_t)k_dyn * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d->S, 0, (size_t)n * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d->A, 0, (size_t)n * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d->sel, 0, (size_t)kSelWords * 4, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        sg_status st = cuda_fail(e, "sg_dyn_cache_create");
        dyn_free(d);
        return st;
    }
    c->dyn = d;
    return SG_OK;
}

extern "C" sg_status sg_dyn_cache_batch(sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                                        sg_stream_t stream) {
    if (!c || !c->dyn) return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_batch: no dynamic cache");
    if (n_cap < 0 || (n_cap > 0 && !d_ids)) return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_batch: bad IDs");
    sg_dyn* d = c->dyn;
    cudaStream_t s = (cudaStream_t)stream;
    const int cap = num_sms() * 8;
    if (n_cap > 0) {
        const int64_t b = min(cdiv(n_cap, kNT), (int64_t)cap);
        k_dyn_accumulate<<<(unsigned)b, kNT, 0, s>>>(d_ids, n_cap, d_n, c->slot_of, c->n_cache, c->n_nodes,
                                                      d->W[d->j], d->A);
        SG_CHECK_LAUNCH("k_dyn_accumulate");
    }
    if (++d->j < d->T) return SG_OK;
    // end of the window: Eq. (5) folded in, then Eq. (6)
    d->j = 0;
    const int64_t n = c->n_nodes, k = d->k_dyn;
    int32_t* enter = d->lists;
    int32_t* free_slots = d->lists + k;
    int32_t* cnt = d->lists + 2 * k;
    k_dyn_fold<<<cap, kNT, 0, s>>>(d->S, d->A, n, d->G_T, d->sel);
    SG_CHECK_LAUNCH("k_dyn_fold");
    k_sel_score_pick<<<1, 32, 0, s>>>(d->sel, 0, k);
    for (int p = 1; p < 4; ++p) {
        k_sel_score_hist<<<cap, kNT, 0, s>>>(d->S, n, p, d->sel);
        k_sel_score_pick<<<1, 32, 0, s>>>(d->sel, p, k);
    }
    for (int q = 0; q < 4; ++q) {
        k_sel_id_hist<<<cap, kNT, 0, s>>>(d->S, n, q, d->sel);
        k_sel_id_pick<<<1, 32, 0, s>>>(d->sel, q);
    }
    SG_CHECK_LAUNCH("k_sel_id_pick");
    SG_CUDA(cudaMemsetAsync(cnt, 0, 8 * sizeof(int32_t), s));
    const int kb = (int)min(cdiv(k, kNT), (int64_t)cap);
    k_dyn_mark<<<cap, kNT, 0, s>>>(d->S, n, d->sel, d->slot, enter, cnt);
    k_dyn_evict<<<kb, kNT, 0, s>>>(d->nodes, k, d->slot, free_slots, cnt);
    const int64_t rv = c->row_bytes / 16;
    k_dyn_admit<<<(unsigned)min(cdiv(k * rv, kNT), (int64_t)cap), kNT, 0, s>>>(
        enter, free_slots, cnt, d->nodes, d->slot, (const uint4*)c->host_rows, rv, (uint4*)d->rows);
    SG_CHECK_LAUNCH("k_dyn_admit");
    return SG_OK;
}

extern "C" sg_status sg_dyn_cache_info(const sg_cache* c, int64_t* k_dyn, int32_t* window_pos, uint32_t* h_score,
                                       int32_t* h_nodes, sg_stream_t stream) {
    if (!c || !c->dyn) return fail(SG_ERR_INVALID_ARG, "sg_dyn_cache_info: no dynamic cache");
    if (k_dyn) *k_dyn = c->dyn->k_dyn;
    if (window_pos) *window_pos = c->dyn->j;
    cudaStream_t s = (cudaStream_t)stream;
    if (h_score)
        SG_CUDA(cudaMemcpyAsync(h_score, c->dyn->S, (size_t)c->n_nodes * 4, cudaMemcpyDeviceToHost, s));
    if (h_nodes)
        SG_CUDA(cudaMemcpyAsync(h_nodes, c->dyn->nodes, (size_t)c->dyn->k_dyn * 4, cudaMemcpyDeviceToHost, s));
    SG_CUDA(cudaStreamSynchronize(s));
    return SG_OK;
}

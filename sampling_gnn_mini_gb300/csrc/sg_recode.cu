// Cache presampling and node recoding (GARDEN page, Section IV-A and IV-B):
//  - sg_access_stats: the full-link access statistics of Eq. (4) over the
//    output of a presampling sampler_run, added into a per-node score;
//  - sg_rank_by_score: nodes ordered by descending score, ties by ascending
//    ID (a stable LSD radix sort of the complemented scores, 8 bits a pass);
//  - sg_graph_renumber: the graph with the node of rank r renamed r, so that
//    the hot nodes hold the smallest IDs and a cache of the top C rows is hit
//    exactly when ID < C (the ID-range hit test of Section IV-A).
//
// Layouts: scores are uint32 [n]; order[r] is the old ID of rank r and
// rank_of[v] the new ID of old node v.  The radix sort keeps 4096 items a
// block; the digit histograms are laid out digit-major ([256][blocks]) so
// that one exclusive scan gives every (digit, block) its output offset.
#include <string.h>

#include <new>

#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(recode)

using namespace sgi;

namespace {

constexpr int kNT = 256;
constexpr int kItems = 16;               // items a thread, in rounds of kNT
constexpr int kTile = kNT * kItems;      // 4096 items a block
constexpr int kDigits = 256;
constexpr int kScanThreads = 1024;

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// --------------------------------------------------------------- statistics
struct StatsArgs {
    const int32_t* unique;
    const int32_t* counts;
    int64_t n_cap;       // capacity of unique
    int32_t H, K;
    uint32_t omega[SG_MAX_HOPS];
    uint32_t w_in;
    uint32_t* score;
    int64_t n_nodes;
};

// Node i of the concatenated V_H lists belongs to mini-batch k with local ID
// j = i - U_k; it is in V_h^k exactly when j < |V_h^k| (V_h is a prefix).
__global__ void __launch_bounds__(kNT) k_access_stats(StatsArgs a) {
    __shared__ int32_t sz[SG_MAX_SUB][SG_MAX_HOPS + 1];
    __shared__ int64_t base[SG_MAX_SUB + 1];
    const int H = a.H, K = a.K;
    for (int t = threadIdx.x; t < K * (H + 1); t += kNT) {
        const int k = t / (H + 1), h = t - k * (H + 1);
        sz[k][h] = a.counts[(2 * H + 1) * (1 + k) + h];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t acc = 0;
        for (int k = 0; k < K; ++k) {
            base[k] = acc;
            acc += sz[k][H];
        }
        base[K] = acc;
    }
    __syncthreads();
    const int64_t n = base[K] < a.n_cap ? base[K] : a.n_cap;
    for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < n; i += (int64_t)gridDim.x * kNT) {
        int k = 0;
        while (k + 1 < K && base[k + 1] <= i) ++k;
        const int64_t j = i - base[k];
        uint32_t w = a.w_in;
#pragma unroll 1
        for (int l = 1; l <= H; ++l) w += a.omega[l - 1] * (uint32_t)((j < sz[k][l]) + (j < sz[k][l - 1]));
        const int32_t v = a.unique[i];
        if (v < 0 || (int64_t)v >= a.n_nodes) {
            dev_err(ERR_INDEX);
            continue;
        }
        atomicAdd(a.score + v, w);
    }
}

// in-degree: deg[u] += 1 for every CSR position naming u
__global__ void k_in_degree(const int32_t* __restrict__ indices, int64_t m, int64_t n, uint32_t* __restrict__ deg) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < m; e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t u = indices[e];
        if (u >= 0 && (int64_t)u < n) atomicAdd(deg + u, 1u);
        else dev_err(ERR_INDEX);
    }
}

// ------------------------------------------------------------ radix sort
// Digit histogram of block b's tile.  A first pass reads the keys as
// ~score[v] with v = init[i] (or i without an initial order).
__global__ void __launch_bounds__(kNT) k_radix_hist(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ score,
                                                    const int32_t* __restrict__ init, int64_t n, int shift,
                                                    uint32_t* __restrict__ hist, int64_t nb) {
    __shared__ uint32_t h[kDigits];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t i0 = (int64_t)blockIdx.x * kTile;
#pragma unroll 4
    for (int r = 0; r < kItems; ++r) {
        const int64_t i = i0 + r * kNT + threadIdx.x;
        if (i < n) {
            const uint32_t key = score ? ~score[init ? init[i] : i] : keys[i];
            atomicAdd(&h[(key >> shift) & 0xFF], 1u);
        }
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * nb + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter of block b's tile: item r*kNT + t of the tile goes to
// offs[digit][b] + (items of the tile before it with the same digit).  Within
// a round, a warp ranks its lanes by digit with match_any; the warps' counts
// per digit are turned into offsets by one thread per digit.
__global__ void __launch_bounds__(kNT) k_radix_scatter(const uint32_t* __restrict__ keys_in,
                                                       const uint32_t* __restrict__ score,
                                                       const int32_t* __restrict__ vals_in, int64_t n, int shift,
                                                       const uint32_t* __restrict__ offs, int64_t nb,
                                                       uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out) {
    __shared__ uint32_t run[kDigits];
    __shared__ uint32_t wcnt[kNT / 32][kDigits];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    run[threadIdx.x] = offs[(int64_t)threadIdx.x * nb + blockIdx.x];
    const int64_t i0 = (int64_t)blockIdx.x * kTile;
    for (int r = 0; r < kItems; ++r) {
        const int64_t i = i0 + r * kNT + threadIdx.x;
        const bool valid = i < n;
        uint32_t key = 0;
        int32_t val = 0;
        if (valid) {
            val = vals_in ? vals_in[i] : (int32_t)i;
            key = score ? ~score[val] : keys_in[i];
        }
        const uint32_t d = valid ? (key >> shift) & 0xFF : 0x100u + (uint32_t)lane;  // invalid lanes match none
#pragma unroll
        for (int w = 0; w < kNT / 32; ++w) wcnt[w][threadIdx.x] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, d);
        const uint32_t rank = __popc(peers & lanemask_lt());
        if (valid && rank == 0) wcnt[warp][d] = __popc(peers);
        __syncthreads();
        {
            uint32_t acc = run[threadIdx.x];
#pragma unroll
            for (int w = 0; w < kNT / 32; ++w) {
                const uint32_t c = wcnt[w][threadIdx.x];
                wcnt[w][threadIdx.x] = acc;
                acc += c;
            }
            run[threadIdx.x] = acc;
        }
        __syncthreads();
        if (valid) {
            const uint32_t pos = wcnt[warp][d] + rank;
            if (keys_out) keys_out[pos] = key;
            vals_out[pos] = val;
        }
        __syncthreads();
    }
}

// rank_of[order[r]] = r; order must be a permutation (checked).
__global__ void k_rank_scatter(const int32_t* __restrict__ order, int64_t n, int32_t* __restrict__ rank_of) {
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < n; r += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = order[r];
        if (v < 0 || (int64_t)v >= n) dev_err(ERR_INDEX);
        else rank_of[v] = (int32_t)r;
    }
}

// ------------------------------------------------------- exclusive scan
// Three passes over n items in chunks of kTile: chunk totals, one block over
// the totals, then each chunk scanned from its base.  In place is allowed.
template <typename T>
__global__ void __launch_bounds__(kNT) k_scan_reduce(const T* __restrict__ in, int64_t n, T* __restrict__ part) {
    __shared__ T red[kNT / 32 + 1];
    const int64_t i0 = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
    T s = 0;
    for (int q = 0; q < kItems; ++q)
        if (i0 + q < n) s += in[i0 + q];
    const T t = block_sum<kNT, T>(s, red);
    if (threadIdx.x == 0) part[blockIdx.x] = t;
}

template <typename T>
__global__ void __launch_bounds__(kScanThreads) k_scan_partials(T* __restrict__ part, int64_t m, T* __restrict__ total) {
    __shared__ T sh[kScanThreads];
    const int64_t per = (m + kScanThreads - 1) / kScanThreads;
    const int64_t a = min((int64_t)threadIdx.x * per, m), b = min(a + per, m);
    T sum = 0;
    for (int64_t r = a; r < b; ++r) sum += part[r];
    sh[threadIdx.x] = sum;
    __syncthreads();
    for (int d = 1; d < kScanThreads; d <<= 1) {
        const T x = threadIdx.x >= (unsigned)d ? sh[threadIdx.x - d] : T(0);
        __syncthreads();
        sh[threadIdx.x] += x;
        __syncthreads();
    }
    T run = sh[threadIdx.x] - sum;
    for (int64_t r = a; r < b; ++r) {
        const T k = part[r];
        part[r] = run;
        run += k;
    }
    if (threadIdx.x == kScanThreads - 1 && total) *total = sh[kScanThreads - 1];
}

template <typename T>
__global__ void __launch_bounds__(kNT) k_scan_down(const T* in, int64_t n, const T* __restrict__ part, T* out) {
    __shared__ T red[kNT / 32 + 1];
    const int64_t i0 = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
    T v[kItems];
    T s = 0;
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
        v[q] = (i0 + q < n) ? in[i0 + q] : T(0);
        s += v[q];
    }
    T tot;
    T run = block_excl_scan<kNT, T>(s, red, tot) + part[blockIdx.x];
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
        if (i0 + q < n) out[i0 + q] = run;
        run += v[q];
    }
}

template <typename T>
size_t scan_scratch(int64_t n) {
    return a256((size_t)((n + kTile - 1) / kTile + 1) * sizeof(T));
}

template <typename T>
sg_status scan_excl(const T* in, T* out, int64_t n, T* total, void* scratch, cudaStream_t s) {
    if (n <= 0) return SG_OK;
    const int64_t nb = (n + kTile - 1) / kTile;
    T* part = (T*)scratch;
    k_scan_reduce<T><<<(unsigned)nb, kNT, 0, s>>>(in, n, part);
    k_scan_partials<T><<<1, kScanThreads, 0, s>>>(part, nb, total);
    k_scan_down<T><<<(unsigned)nb, kNT, 0, s>>>(in, n, part, out);
    SG_CHECK_LAUNCH("scan");
    return SG_OK;
}

struct RankLayout {
    int64_t nb;
    size_t keys0, keys1, vals, order1, hist, scan, total;
};

RankLayout rank_layout(int64_t n) {
    RankLayout L;
    L.nb = (n + kTile - 1) / kTile;
    size_t o = 0;
    L.keys0 = o;
    o += a256((size_t)n * 4);
    L.keys1 = o;
    o += a256((size_t)n * 4);
    L.vals = o;
    o += a256((size_t)n * 4);
    L.order1 = o;  // the order by the tie key, when there is one
    o += a256((size_t)n * 4);
    L.hist = o;
    o += a256((size_t)kDigits * L.nb * 4);
    L.scan = o;
    o += scan_scratch<uint32_t>((int64_t)kDigits * L.nb);
    L.total = o;
    return L;
}

// ------------------------------------------------------------ renumbering
// degree of the new row r (the old row order[r]) at out[r]; out[n] = 0, so
// that an exclusive scan over n + 1 entries gives the new offsets
template <typename Off>
__global__ void k_new_degrees(const Off* __restrict__ indptr, const int32_t* __restrict__ order,
                              const int32_t* __restrict__ rank_of, int64_t n, Off* __restrict__ out,
                              unsigned* __restrict__ bad) {
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r <= n; r += (int64_t)gridDim.x * blockDim.x) {
        if (r == n) {
            out[n] = 0;
            continue;
        }
        const int32_t v = order[r];
        if (v < 0 || (int64_t)v >= n || rank_of[v] != (int32_t)r) {  // not a permutation with its inverse
            atomicOr(bad, 1u);
            out[r] = 0;
            continue;
        }
        out[r] = indptr[v + 1] - indptr[v];
    }
}

// New row r, position for position: a warp per row, neighbours renamed.
template <typename Off>
__global__ void __launch_bounds__(kNT) k_copy_rows(const Off* __restrict__ indptr, const int32_t* __restrict__ indices,
                                                   const int32_t* __restrict__ order, const int32_t* __restrict__ rank_of,
                                                   int64_t n, const Off* __restrict__ new_indptr,
                                                   int32_t* __restrict__ new_indices) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kNT / 32);
    for (int64_t r = blockIdx.x * (int64_t)(kNT / 32) + (threadIdx.x >> 5); r < n; r += warps) {
        const int32_t v = order[r];
        if (v < 0 || (int64_t)v >= n) continue;  // reported by k_new_degrees
        const int64_t a = (int64_t)indptr[v], deg = (int64_t)indptr[v + 1] - a, b = (int64_t)new_indptr[r];
        if ((int64_t)new_indptr[r + 1] - b != deg) continue;  // order was not a permutation (reported)
        for (int64_t j = lane; j < deg; j += 32) new_indices[b + j] = __ldg(rank_of + __ldg(indices + a + j));
    }
}

template <typename Off>
sg_status renumber_impl(const sg_graph* g, const int32_t* order, const int32_t* rank_of, sg_graph* out, cudaStream_t s) {
    const int64_t n = g->n_nodes;
    void* scratch = nullptr;
    unsigned* bad = nullptr;
    cudaError_t e = dev_alloc(&scratch, scan_scratch<Off>(n + 1) + 256);
    if (e != cudaSuccess) return cuda_fail(e, "sg_graph_renumber: scratch");
    bad = (unsigned*)((char*)scratch + scan_scratch<Off>(n + 1));
    sg_status st = SG_OK;
    const int blocks = num_sms() * 8;
    Off* nip = (Off*)out->indptr;
    if ((e = cudaMemsetAsync(bad, 0, sizeof(unsigned), s)) != cudaSuccess) st = cuda_fail(e, "sg_graph_renumber");
    if (st == SG_OK) {
        k_new_degrees<Off><<<blocks, kNT, 0, s>>>((const Off*)g->indptr, order, rank_of, n, nip, bad);
        if ((e = cudaGetLastError()) != cudaSuccess) st = cuda_fail(e, "k_new_degrees");
    }
    if (st == SG_OK) st = scan_excl<Off>(nip, nip, n + 1, (Off*)nullptr, scratch, s);
    if (st == SG_OK) {
        k_copy_rows<Off><<<blocks, kNT, 0, s>>>((const Off*)g->indptr, g->indices, order, rank_of, n, nip,
                                                out->indices);
        if ((e = cudaGetLastError()) != cudaSuccess) st = cuda_fail(e, "k_copy_rows");
    }
    unsigned h_bad = 0;
    if (st == SG_OK && (e = cudaMemcpyAsync(&h_bad, bad, sizeof(unsigned), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        st = cuda_fail(e, "sg_graph_renumber");
    if (st == SG_OK && (e = cudaStreamSynchronize(s)) != cudaSuccess) st = cuda_fail(e, "sg_graph_renumber");
    cudaFree(scratch);
    if (st == SG_OK && h_bad)
        st = fail(SG_ERR_INVALID_ARG, "sg_graph_renumber: order and rank_of must be inverse permutations of [0, n)");
    return st;
}

}  // namespace

// ------------------------------------------------------------------- ABI
extern "C" sg_status sg_access_stats(const sg_blocks* blocks, int64_t unique_cap, int32_t n_hops, int32_t n_sub,
                                     const uint32_t* h_omega, uint32_t w_in, uint32_t* d_score, int64_t n_nodes,
                                     sg_stream_t stream) {
    if (!blocks || !blocks->unique || !blocks->counts || !d_score || !h_omega)
        return fail(SG_ERR_INVALID_ARG, "sg_access_stats: NULL argument");
    if (n_hops < 1 || n_hops > SG_MAX_HOPS || n_sub < 1 || n_sub > SG_MAX_SUB || unique_cap < 0 || n_nodes <= 0)
        return fail(SG_ERR_INVALID_ARG, "sg_access_stats: sizes out of range");
    if (unique_cap == 0) return SG_OK;
    StatsArgs a;
    memset(&a, 0, sizeof(a));
    a.unique = blocks->unique;
    a.counts = blocks->counts;
    a.n_cap = unique_cap;
    a.H = n_hops;
    a.K = n_sub;
    for (int l = 0; l < n_hops; ++l) a.omega[l] = h_omega[l];
    a.w_in = w_in;
    a.score = d_score;
    a.n_nodes = n_nodes;
    int64_t blocks_n = cdiv(unique_cap, kNT);
    if (blocks_n > (int64_t)num_sms() * 8) blocks_n = (int64_t)num_sms() * 8;
    k_access_stats<<<(unsigned)blocks_n, kNT, 0, (cudaStream_t)stream>>>(a);
    SG_CHECK_LAUNCH("k_access_stats");
    return SG_OK;
}

extern "C" size_t sg_rank_workspace(int64_t n_nodes) {
    if (n_nodes <= 0 || n_nodes > 2147483647LL) return 0;
    return rank_ws_bytes(n_nodes);
}

namespace sgi {
size_t rank_ws_bytes(int64_t n) { return rank_layout(n).total; }

// Four LSD passes of 8 bits over the complemented keys of `score` (ascending
// key = descending score), stable, starting from the order `init` (or the
// IDs); the values end in d_order.  Pass 0 gathers the keys through the
// values and writes keys0 / tmp, pass 1 keys1 / order, pass 2 keys0 / tmp,
// pass 3 the values alone into order.
sg_status radix_by(const uint32_t* score, const int32_t* init, int64_t n_nodes, int32_t* d_order, char* ws,
                   const RankLayout& L, cudaStream_t s) {
    uint32_t* keys[2] = {(uint32_t*)(ws + L.keys0), (uint32_t*)(ws + L.keys1)};
    int32_t* vals[2] = {(int32_t*)(ws + L.vals), d_order};
    uint32_t* hist = (uint32_t*)(ws + L.hist);
    for (int p = 0; p < 4; ++p) {
        const int shift = 8 * p;
        const uint32_t* kin = p == 0 ? nullptr : keys[(p + 1) & 1];
        const int32_t* vin = p == 0 ? init : vals[(p + 1) & 1];
        uint32_t* kout = p == 3 ? nullptr : keys[p & 1];
        int32_t* vout = vals[p & 1];
        k_radix_hist<<<(unsigned)L.nb, kNT, 0, s>>>(kin, p == 0 ? score : nullptr, p == 0 ? init : nullptr, n_nodes,
                                                    shift, hist, L.nb);
        sg_status st = scan_excl<uint32_t>(hist, hist, (int64_t)kDigits * L.nb, (uint32_t*)nullptr, ws + L.scan, s);
        if (st != SG_OK) return st;
        k_radix_scatter<<<(unsigned)L.nb, kNT, 0, s>>>(kin, p == 0 ? score : nullptr, vin, n_nodes, shift, hist,
                                                       L.nb, kout, vout);
        SG_CHECK_LAUNCH("k_radix_scatter");
    }
    return SG_OK;
}

// Nodes by descending score, then descending tie key (when given), then
// ascending ID: a stable sort by the tie key, then a stable sort of that
// order by the score.
sg_status rank_scores2(const uint32_t* d_score, const uint32_t* d_tie, int64_t n_nodes, int32_t* d_order,
                       void* d_workspace, cudaStream_t s) {
    const RankLayout L = rank_layout(n_nodes);
    char* ws = (char*)d_workspace;
    if (!d_tie) return radix_by(d_score, nullptr, n_nodes, d_order, ws, L, s);
    int32_t* first = (int32_t*)(ws + L.order1);
    sg_status st = radix_by(d_tie, nullptr, n_nodes, first, ws, L, s);
    if (st != SG_OK) return st;
    return radix_by(d_score, first, n_nodes, d_order, ws, L, s);
}

sg_status rank_scores(const uint32_t* d_score, int64_t n_nodes, int32_t* d_order, void* d_workspace, cudaStream_t s) {
    return rank_scores2(d_score, nullptr, n_nodes, d_order, d_workspace, s);
}
}  // namespace sgi

extern "C" sg_status sg_rank_by_score(const uint32_t* d_score, const uint32_t* d_tie, int64_t n_nodes, int32_t* d_order,
                                      int32_t* d_rank_of, void* d_workspace, size_t workspace_bytes,
                                      sg_stream_t stream) {
    if (n_nodes <= 0 || n_nodes > 2147483647LL) return fail(SG_ERR_INVALID_ARG, "sg_rank_by_score: n_nodes out of range");
    if (!d_score || !d_order || !d_workspace) return fail(SG_ERR_INVALID_ARG, "sg_rank_by_score: NULL argument");
    const size_t need = rank_ws_bytes(n_nodes);
    if (workspace_bytes < need || ((uintptr_t)d_workspace) % 256)
        return fail(SG_ERR_INVALID_ARG, "sg_rank_by_score: workspace needs %zu bytes, 256-byte aligned", need);
    cudaStream_t s = (cudaStream_t)stream;
    sg_status st = rank_scores2(d_score, d_tie, n_nodes, d_order, d_workspace, s);
    if (st != SG_OK) return st;
    if (d_rank_of) {
        k_rank_scatter<<<num_sms() * 8, kNT, 0, s>>>(d_order, n_nodes, d_rank_of);
        SG_CHECK_LAUNCH("k_rank_scatter");
    }
    return SG_OK;
}

extern "C" sg_status sg_graph_in_degree(const sg_graph* g, uint32_t* d_deg, sg_stream_t stream) {
    if (!g || !d_deg) return fail(SG_ERR_INVALID_ARG, "sg_graph_in_degree: NULL argument");
    cudaStream_t s = (cudaStream_t)stream;
    SG_CUDA(cudaMemsetAsync(d_deg, 0, (size_t)g->n_nodes * sizeof(uint32_t), s));
    if (g->n_edges > 0) {
        k_in_degree<<<num_sms() * 8, kNT, 0, s>>>(g->indices, g->n_edges, g->n_nodes, d_deg);
        SG_CHECK_LAUNCH("k_in_degree");
    }
    return SG_OK;
}

extern "C" sg_status sg_graph_renumber(const sg_graph* g, const int32_t* d_order, const int32_t* d_rank_of,
                                       sg_graph** out, sg_stream_t stream) {
    if (!out) return fail(SG_ERR_INVALID_ARG, "sg_graph_renumber: out is NULL");
    *out = nullptr;
    if (!g || !d_order || !d_rank_of) return fail(SG_ERR_INVALID_ARG, "sg_graph_renumber: NULL argument");
    sg_graph* ng = new (std::nothrow) sg_graph();
    if (!ng) return fail(SG_ERR_OOM, "sg_graph_renumber: host allocation");
    ng->n_nodes = g->n_nodes;
    ng->n_edges = g->n_edges;
    ng->offset_bits = g->offset_bits;
    ng->max_degree = g->max_degree;
    const size_t ob = g->offset_bits / 8;
    cudaError_t e = dev_alloc(&ng->indptr, (size_t)(g->n_nodes + 1) * ob);
    if (e == cudaSuccess) e = dev_alloc((void**)&ng->indices, (size_t)(g->n_edges > 0 ? g->n_edges : 1) * sizeof(int32_t));
    sg_status st = e == cudaSuccess ? SG_OK : cuda_fail(e, "sg_graph_renumber");
    if (st == SG_OK)
        st = g->offset_bits == 64 ? renumber_impl<int64_t>(g, d_order, d_rank_of, ng, (cudaStream_t)stream)
                                  : renumber_impl<int32_t>(g, d_order, d_rank_of, ng, (cudaStream_t)stream);
    if (st != SG_OK) {
        sg_graph_destroy(ng);
        return st;
    }
    *out = ng;
    return SG_OK;
}

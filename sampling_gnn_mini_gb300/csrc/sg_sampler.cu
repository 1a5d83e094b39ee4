// Multi-hop neighbour sampling and relabel into per-hop blocks.
//
// What is computed (GARDEN page, "GARDEN: Efficient GPU-Accelerated
// Billion-Scale GNN Training via Caching-Sampling-Batching Co-Design"):
//  - Section II-B / Fig. 1: hop h takes V_{h-1} as its dst set and forms
//    V_h = V_{h-1} u N_h(V_{h-1}); seeds are V_0.
//  - Section IV-C: fixed-fanout uniform sampling; a node with degree <= fanout
//    keeps all neighbours ("full node"), otherwise a uniform subset is drawn
//    ("random node") without altering the sampling distribution.  The draw is
//    the bottom-f positions by the key (Philox word, position).
//  - Section IV-D: mini-batches of a super-batch are stored back to back with a
//    BatchPtr; dedup goes through a GPU hash table; node classification is
//    turned into index arithmetic by a flag + exclusive scan (no atomics on the
//    placement), generalised here from two classes to four degree bins.
//  - FastGL explainer page, "Fused-Map": the hash insert and the local-ID
//    bookkeeping share one pass; here the insert records the minimum edge
//    position per node (atomicMin), so the numbering is the deterministic
//    first-occurrence order instead of the atomic arrival order.
//
// Per hop the kernels are:
//   dst_count  c_v = min(deg, f) and the degree bin of every dst row
//   dst_scan   block row pointer (exclusive scan of c_v) and bin order
//              (largest rows first), per mini-batch edge offsets
//   sample     one warp per dst row in bin order: copy a full row, or hash
//              every position of a random row with Philox, keep the positions
//              under a threshold as candidates, and pick the f smallest keys
//              exactly; each emitted neighbour is inserted in the table
//   flag       is edge e the first occurrence of its node in this hop?
//   assign     local IDs of new nodes = |V_{h-1}^k| + rank of first occurrence
//   map        src ID of every edge
#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(sampler)

using namespace sgi;

namespace {

constexpr int kNT = 256;            // threads of the segmented scan kernels
constexpr int kSampleNT = 256;      // threads of the sample kernel (8 warps)
constexpr int kCandCap = 256;       // candidate slots per warp
constexpr int kMaxSeg = 1024;       // blocks of a segmented pass
constexpr uint32_t kEmpty = 0xFFFFFFFFu;

// bins: 0 full row, 1 random deg <= 256, 2 random deg <= 4096, 3 random larger
__device__ __forceinline__ int degree_bin(int64_t deg, int f) {
    if (deg <= f) return 0;
    if (deg <= 256) return 1;
    if (deg <= 4096) return 2;
    return 3;
}

struct SubPtr {
    int32_t v[SG_MAX_SUB + 1];
};

// Where the counts of hop h live (see sg_blocks in sg.h).
struct CountsLayout {
    int H;
    __host__ __device__ __forceinline__ int tot_n(int h) const { return h; }
    __host__ __device__ __forceinline__ int tot_e(int h) const { return H + h; }
    __host__ __device__ __forceinline__ int sub_n(int k, int h) const { return (2 * H + 1) * (1 + k) + h; }
    __host__ __device__ __forceinline__ int sub_e(int k, int h) const { return (2 * H + 1) * (1 + k) + H + h; }
};

__device__ __forceinline__ uint32_t slot_hash(int32_t key, int logT) {
    return ((uint32_t)key * 0x9E3779B1u) >> (32 - logT);
}

// Open addressing with linear probing; slots are {key, value} pairs, both
// 0xFFFFFFFF when empty.  Records min(value) for the key and returns the slot
// index (relative to `tab`), or -1 when the table is full.  *was_present tells
// whether the key was already in the table.
__device__ __forceinline__ int table_insert(uint2* tab, int logT, int32_t key, uint32_t val, bool* was_present) {
    const uint32_t mask = (1u << logT) - 1u;
    uint32_t s = slot_hash(key, logT);
    for (uint32_t probe = 0; probe <= mask; ++probe) {
        const uint32_t prev = atomicCAS(&tab[s].x, kEmpty, (uint32_t)key);
        if (prev == kEmpty || prev == (uint32_t)key) {
            atomicMin(&tab[s].y, val);
            if (was_present) *was_present = (prev == (uint32_t)key);
            return (int)s;
        }
        s = (s + 1) & mask;
    }
    dev_err(ERR_CAPACITY);
    return -1;
}

// index k with sp[k] <= x < sp[k+1] over a non-decreasing sp[0..K]; for ties
// (empty mini-batches) the last k with sp[k] <= x.
__device__ __forceinline__ int find_sub(const int32_t* sp, int K, int64_t x) {
    int lo = 0, hi = K;  // answer in [0, K-1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)sp[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename Off>
__device__ __forceinline__ int64_t row_start(const Off* indptr, int32_t v) { return (int64_t)indptr[v]; }

// Loads the per-mini-batch sizes of hop h into shared memory as an exclusive
// prefix: pre[k] = sum_{k'<k} counts[sub_n(k', h)], pre[K] = total.
__device__ void load_prefix_sub_n(const int32_t* counts, CountsLayout L, int K, int h, int32_t* pre) {
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int k = 0; k < K; ++k) {
            pre[k] = acc;
            acc += counts[L.sub_n(k, h)];
        }
        pre[K] = acc;
    }
    __syncthreads();
}

// ----------------------------------------------------------------- seeds
// Seeds take local IDs 0..B_k-1 of their mini-batch.  A repeated seed inside
// one mini-batch or an ID out of range is reported through the error word.
__global__ void k_seed_init(const int32_t* __restrict__ seeds, int32_t n_seeds, SubPtr bptr, int K, int64_t n_nodes,
                            uint2* table, int logT, int32_t* ustr, int64_t capU, int32_t* counts, CountsLayout L) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) counts[L.tot_n(0)] = n_seeds;
        for (int k = threadIdx.x; k < K; k += blockDim.x) counts[L.sub_n(k, 0)] = bptr.v[k + 1] - bptr.v[k];
    }
    if (i >= n_seeds) return;
    const int k = find_sub(bptr.v, K, i);
    const int32_t l = i - bptr.v[k];
    const int32_t s = seeds[i];
    ustr[(int64_t)k * capU + l] = s;  // later passes skip an ID out of range
    if (s < 0 || (int64_t)s >= n_nodes) {
        dev_err(ERR_INDEX);
        return;
    }
    bool present = false;
    if (table_insert(table + ((int64_t)k << logT), logT, s, (uint32_t)l, &present) < 0) return;
    if (present) dev_err(ERR_ARG);
}

// --------------------------------------------------------------- dst_count
struct HopArgs {
    const void* indptr;
    const int32_t* indices;
    int64_t n_nodes;
    int K, logT, h, fanout;
    int64_t capU;
    uint32_t key0, key1;
    const uint64_t* d_seed;  // when not NULL, the key is read from here
    uint32_t lambda_num;     // expected candidates per random row (threshold)
    int32_t pos_base;        // value of edge e in the table = pos_base + e
    CountsLayout L;
    int32_t* counts;
    int32_t* ustr;
    uint2* table;
    int32_t* dst_gid;
    uint8_t* dbin;
    int32_t* order;
    int32_t* bindptr;
    int32_t* bidx;
    int32_t* epre;           // [K+1] edge offset of each mini-batch in this hop
    int32_t* enbr;
    int32_t* eslot;
    uint8_t* eflag;
    int32_t* bsum;           // [kMaxSeg * 8]
    int G_d, G_e;
};

template <typename Off>
__global__ void __launch_bounds__(kNT) k_dst_count(HopArgs a) {
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ int32_t red[kNT / 32 + 1];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);
    const int64_t T = pre[a.K];
    int64_t lo, hi;
    segment_of(T, blockIdx.x, gridDim.x, lo, hi);
    const Off* indptr = (const Off*)a.indptr;
    int32_t csum = 0, nb[4] = {0, 0, 0, 0};
    for (int64_t r = lo + threadIdx.x; r < hi; r += kNT) {
        const int k = find_sub(pre, a.K, r);
        const int32_t v = a.ustr[(int64_t)k * a.capU + (r - pre[k])];
        int64_t deg = 0;
        if (v >= 0 && (int64_t)v < a.n_nodes) deg = (int64_t)indptr[v + 1] - (int64_t)indptr[v];
        else dev_err(ERR_INDEX);
        const int32_t c = (int32_t)(deg < a.fanout ? deg : a.fanout);
        const int b = degree_bin(deg, a.fanout);
        a.dst_gid[r] = v;
        a.dbin[r] = (uint8_t)b;
        a.bindptr[r] = c;  // row length for now; dst_scan turns it into offsets
        csum += c;
        nb[b]++;
    }
    int32_t t;
    t = block_sum<kNT>(csum, red);
    if (threadIdx.x == 0) a.bsum[blockIdx.x * 8 + 0] = t;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        t = block_sum<kNT>(nb[b], red);
        if (threadIdx.x == 0) a.bsum[blockIdx.x * 8 + 1 + b] = t;
    }
}

// ---------------------------------------------------------------- dst_scan
__global__ void __launch_bounds__(kNT) k_dst_scan(HopArgs a) {
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ unsigned long long red64[kNT / 32 + 1];
    __shared__ int32_t carry[5], base[4], total_c;
    load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);
    const int64_t T = pre[a.K];
    // prefixes over earlier blocks and totals over all blocks
    int32_t my[5] = {0, 0, 0, 0, 0}, all[5] = {0, 0, 0, 0, 0};
    for (int b = threadIdx.x; b < (int)gridDim.x; b += kNT) {
#pragma unroll
        for (int q = 0; q < 5; ++q) {
            const int32_t x = a.bsum[b * 8 + q];
            all[q] += x;
            if (b < (int)blockIdx.x) my[q] += x;
        }
    }
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        const int32_t s1 = block_sum<kNT>(my[q], red);
        const int32_t s2 = block_sum<kNT>(all[q], red);
        if (threadIdx.x == 0) {
            carry[q] = s1;
            if (q == 0) total_c = s2;
            else my[q] = s2;  // thread 0 keeps the bin totals
        }
    }
    if (threadIdx.x == 0) {
        // bin order: largest rows first (bin 3, 2, 1, then full rows)
        base[3] = 0;
        base[2] = my[4];
        base[1] = my[4] + my[3];
        base[0] = my[4] + my[3] + my[2];
    }
    __syncthreads();
    int64_t lo, hi;
    segment_of(T, blockIdx.x, gridDim.x, lo, hi);
    for (int64_t t0 = lo; t0 < hi; t0 += kNT) {
        const int64_t r = t0 + threadIdx.x;
        const bool in = r < hi;
        const int32_t c = in ? a.bindptr[r] : 0;
        const int b = in ? (int)a.dbin[r] : 0;
        int32_t tc;
        const int32_t ex = block_excl_scan<kNT>(c, red, tc);
        const unsigned long long bits = in ? (1ull << (16 * b)) : 0ull;
        unsigned long long tb;
        const unsigned long long exb = block_excl_scan<kNT>(bits, red64, tb);
        if (in) {
            const int32_t off = carry[0] + ex;
            a.bindptr[r] = off;
            const int32_t rank = (int32_t)((exb >> (16 * b)) & 0xFFFFull);
            a.order[base[b] + carry[1 + b] + rank] = (int32_t)r;
            // edge offset of every mini-batch whose first dst row is r
            int k = find_sub(pre, a.K, r);
            while (k >= 0 && pre[k] == r) {
                a.epre[k] = off;
                --k;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            carry[0] += tc;
#pragma unroll
            for (int q = 0; q < 4; ++q) carry[1 + q] += (int32_t)((tb >> (16 * q)) & 0xFFFFull);
        }
        __syncthreads();
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.bindptr[T] = total_c;
        a.counts[a.L.tot_e(a.h)] = total_c;
        for (int k = a.K; k >= 0 && pre[k] == T; --k) a.epre[k] = total_c;
    }
}

// ------------------------------------------------------------------ sample
__device__ __forceinline__ void emit_edge(const HopArgs& a, uint2* tab, int64_t e, int32_t u) {
    a.enbr[e] = u;
    const int s = table_insert(tab, a.logT, u, (uint32_t)(a.pos_base + e), nullptr);
    a.eslot[e] = s < 0 ? -1 : (int32_t)((int64_t)(tab - a.table) + s);
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long x) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, x, d);
        x = o < x ? o : x;
    }
    return x;
}

// Exact bottom-f by f passes of a warp-wide minimum over all positions
// (rarely used: only when the threshold filter cannot hold or find f keys).
template <typename Off>
__device__ void sample_exact(const HopArgs& a, uint2* tab, int32_t v, int64_t start, int64_t deg, int64_t out0,
                             int32_t* cj) {
    const unsigned lane = lane_id();
    const int f = a.fanout;
    unsigned long long prev = 0;
    for (int s = 0; s < f; ++s) {
        unsigned long long best = ~0ull;
        for (int64_t base = 0; base < deg; base += 128) {
            const int64_t q = (base >> 2) + lane;
            if (4 * q < deg) {
                const uint4 w = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)v, (uint32_t)a.h, 0u), a.key0, a.key1);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int64_t j = 4 * q + t;
                    if (j < deg) {
                        const unsigned long long key = ((unsigned long long)ws[t] << 32) | (unsigned long long)j;
                        if ((s == 0 || key > prev) && key < best) best = key;
                    }
                }
            }
        }
        best = warp_min_u64(best);
        if (lane == 0) cj[s] = (int32_t)(best & 0xFFFFFFFFull);
        prev = best;
    }
    __syncwarp();
    // list the f positions in ascending order (rank among distinct values)
    for (int i = lane; i < f; i += 32) {
        const int32_t x = cj[i];
        int rank = 0;
        for (int t = 0; t < f; ++t) rank += cj[t] < x;
        const int32_t u = a.indices[start + x];
        emit_edge(a, tab, out0 + rank, u);
    }
    __syncwarp();
}

template <typename Off>
__global__ void __launch_bounds__(kSampleNT) k_sample(HopArgs a) {
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ uint32_t cand_r[kSampleNT / 32][kCandCap];
    __shared__ int32_t cand_j[kSampleNT / 32][kCandCap];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);
    const int64_t T = pre[a.K];
    const unsigned lane = lane_id();
    const int wib = threadIdx.x >> 5;
    uint32_t* cr = cand_r[wib];
    int32_t* cj = cand_j[wib];
    const Off* indptr = (const Off*)a.indptr;
    const int f = a.fanout;
    const int64_t nwarps = (int64_t)gridDim.x * (kSampleNT / 32);
    if (a.d_seed) {
        const uint64_t sd = *a.d_seed;
        a.key0 = (uint32_t)(sd & 0xFFFFFFFFull);
        a.key1 = (uint32_t)(sd >> 32);
    }
    for (int64_t i = blockIdx.x * (int64_t)(kSampleNT / 32) + wib; i < T; i += nwarps) {
        const int32_t r = a.order[i];
        const int32_t v = a.dst_gid[r];
        if (v < 0 || (int64_t)v >= a.n_nodes) continue;  // reported by dst_count
        const int64_t start = (int64_t)indptr[v];
        const int64_t deg = (int64_t)indptr[v + 1] - start;
        const int64_t out0 = a.bindptr[r];
        const int k = find_sub(pre, a.K, r);
        uint2* tab = a.table + ((int64_t)k << a.logT);
        if (deg <= f) {  // full node: every neighbour, in row order
            for (int64_t t = lane; t < deg; t += 32) emit_edge(a, tab, out0 + t, a.indices[start + t]);
            continue;
        }
        // random node: candidates are the positions whose key is <= tau
        const unsigned long long lam = a.lambda_num;
        unsigned long long tau64 = (lam << 32) / (unsigned long long)deg;
        uint32_t tau = tau64 > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)tau64;
        bool done = false;
        for (int attempt = 0; attempt < 3 && !done; ++attempt) {
            int n = 0;
            bool overflow = false;
            for (int64_t base = 0; base < deg; base += 128) {
                const int64_t q = (base >> 2) + lane;
                uint4 w = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
                if (4 * q < deg)
                    w = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)v, (uint32_t)a.h, 0u), a.key0, a.key1);
                const int64_t j0 = 4 * q;
                const bool p0 = j0 + 0 < deg && w.x <= tau;
                const bool p1 = j0 + 1 < deg && w.y <= tau;
                const bool p2 = j0 + 2 < deg && w.z <= tau;
                const bool p3 = j0 + 3 < deg && w.w <= tau;
                const unsigned m0 = __ballot_sync(0xffffffffu, p0), m1 = __ballot_sync(0xffffffffu, p1);
                const unsigned m2 = __ballot_sync(0xffffffffu, p2), m3 = __ballot_sync(0xffffffffu, p3);
                const unsigned lt = lanemask_lt();
                const int before = __popc(m0 & lt) + __popc(m1 & lt) + __popc(m2 & lt) + __popc(m3 & lt);
                const int tot = __popc(m0) + __popc(m1) + __popc(m2) + __popc(m3);
                if (n + tot > kCandCap) {
                    overflow = true;
                    break;
                }
                int p = n + before;  // candidates stay in ascending position order
                if (p0) { cr[p] = w.x; cj[p] = (int32_t)(j0 + 0); ++p; }
                if (p1) { cr[p] = w.y; cj[p] = (int32_t)(j0 + 1); ++p; }
                if (p2) { cr[p] = w.z; cj[p] = (int32_t)(j0 + 2); ++p; }
                if (p3) { cr[p] = w.w; cj[p] = (int32_t)(j0 + 3); ++p; }
                n += tot;
            }
            __syncwarp();
            if (overflow) break;
            if (n < f) {  // too few under the threshold: widen it and retry
                tau = tau > 0x3FFFFFFFu ? 0xFFFFFFFFu : (tau << 2) | 3u;
                __syncwarp();
                continue;
            }
            // exact bottom-f among the candidates: rank by (key, position)
            int sel_before = 0;
            for (int c0 = 0; c0 < n; c0 += 32) {
                const int ci = c0 + lane;
                bool sel = false;
                if (ci < n) {
                    const uint32_t ri = cr[ci];
                    int rank = 0;
                    for (int t = 0; t < n; ++t) {
                        const uint32_t rt = cr[t];
                        rank += (rt < ri) || (rt == ri && t < ci);
                    }
                    sel = rank < f;
                }
                const unsigned m = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    const int o = sel_before + __popc(m & lanemask_lt());
                    emit_edge(a, tab, out0 + o, a.indices[start + cj[ci]]);
                }
                sel_before += __popc(m);
            }
            __syncwarp();
            done = true;
        }
        if (!done) sample_exact<Off>(a, tab, v, start, deg, out0, cj);
    }
}

// -------------------------------------------------------------------- flag
__global__ void __launch_bounds__(kNT) k_flag(HopArgs a) {
    __shared__ int32_t red[kNT / 32 + 1];
    const int64_t E = a.epre[a.K];
    int64_t lo, hi;
    segment_of(E, blockIdx.x, gridDim.x, lo, hi);
    int32_t cnt = 0;
    for (int64_t e = lo + threadIdx.x; e < hi; e += kNT) {
        const int32_t s = a.eslot[e];
        const bool first = s >= 0 && a.table[s].y == (uint32_t)(a.pos_base + e);
        a.eflag[e] = first;
        cnt += first;
    }
    const int32_t t = block_sum<kNT>(cnt, red);
    if (threadIdx.x == 0) a.bsum[blockIdx.x] = t;
}

// ------------------------------------------------------------------ assign
__global__ void __launch_bounds__(kNT) k_assign(HopArgs a) {
    __shared__ int32_t npre[SG_MAX_SUB + 1];   // |V_{h-1}^k| prefix
    __shared__ int32_t ep[SG_MAX_SUB + 1];     // edge offset of each mini-batch
    __shared__ int32_t fpre[SG_MAX_SUB + 1];   // first occurrences before ep[k]
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ int32_t carry;
    const int K = a.K;
    load_prefix_sub_n(a.counts, a.L, K, a.h - 1, npre);
    for (int k = threadIdx.x; k <= K; k += kNT) ep[k] = a.epre[k];
    __syncthreads();
    const int64_t E = ep[K];
    const int G = gridDim.x;
    const int64_t seglen = (E + G - 1) / G;
    // fpre[k] = number of flags in [0, ep[k]): whole blocks before the one
    // holding ep[k], plus the part of that block's segment before ep[k]
    for (int k = threadIdx.x >> 5; k <= K; k += kNT / 32) {
        const int64_t ek = ep[k];
        const int bk = seglen > 0 ? (int)(ek / seglen) : 0;
        int32_t s = 0;
        for (int b = lane_id(); b < bk && b < G; b += 32) s += a.bsum[b];
        const int64_t seg0 = (int64_t)bk * seglen;
        for (int64_t e = seg0 + lane_id(); e < ek; e += 32) s += a.eflag[e];
        s = warp_sum(s);
        if (lane_id() == 0) fpre[k] = s;
    }
    int32_t mine = 0;
    for (int b = threadIdx.x; b < (int)blockIdx.x; b += kNT) mine += a.bsum[b];
    mine = block_sum<kNT>(mine, red);
    if (threadIdx.x == 0) carry = mine;
    __syncthreads();
    int64_t lo, hi;
    segment_of(E, blockIdx.x, G, lo, hi);
    for (int64_t t0 = lo; t0 < hi; t0 += kNT) {
        const int64_t e = t0 + threadIdx.x;
        const int32_t fl = e < hi ? (int32_t)a.eflag[e] : 0;
        int32_t tot;
        const int32_t ex = block_excl_scan<kNT>(fl, red, tot);
        if (fl) {
            const int32_t rank = carry + ex;
            const int k = find_sub(ep, K, e);
            const int64_t lid = (int64_t)a.counts[a.L.sub_n(k, a.h - 1)] + (rank - fpre[k]);
            if (lid >= a.capU) {
                dev_err(ERR_CAPACITY);
            } else {
                a.table[a.eslot[e]].y = (uint32_t)lid;
                a.ustr[(int64_t)k * a.capU + lid] = a.enbr[e];
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        int32_t tot_n = 0;
        for (int k = 0; k < K; ++k) {
            const int32_t nk = (npre[k + 1] - npre[k]) + (fpre[k + 1] - fpre[k]);
            a.counts[a.L.sub_n(k, a.h)] = nk;
            a.counts[a.L.sub_e(k, a.h)] = ep[k + 1] - ep[k];
            tot_n += nk;
        }
        a.counts[a.L.tot_n(a.h)] = tot_n;
    }
}

// --------------------------------------------------------------------- map
__global__ void __launch_bounds__(kNT) k_map(HopArgs a) {
    __shared__ int32_t ep[SG_MAX_SUB + 1];
    __shared__ int32_t spre[SG_MAX_SUB + 1];
    for (int k = threadIdx.x; k <= a.K; k += kNT) ep[k] = a.epre[k];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h, spre);
    const int64_t E = ep[a.K];
    for (int64_t e = blockIdx.x * (int64_t)kNT + threadIdx.x; e < E; e += (int64_t)gridDim.x * kNT) {
        const int32_t s = a.eslot[e];
        int32_t out = -1;
        if (s >= 0) {
            const int k = a.K == 1 ? 0 : find_sub(ep, a.K, e);
            out = spre[k] + (int32_t)a.table[s].y;
        }
        a.bidx[e] = out;
    }
}

// ----------------------------------------------------------------- compact
// Lays the mini-batches' V_H regions out back to back.
__global__ void k_compact(const int32_t* ustr, int64_t capU, int K, const int32_t* counts, CountsLayout L, int H,
                          int32_t* unique) {
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    load_prefix_sub_n(counts, L, K, H, pre);
    const int64_t n = pre[K];
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int k = find_sub(pre, K, i);
        unique[i] = ustr[(int64_t)k * capU + (i - pre[k])];
    }
}

// ------------------------------------------------------ standalone relabel
__global__ void k_relabel_insert(const int32_t* __restrict__ ids, int64_t n_ids, uint2* table, int logT, int32_t pos_base,
                                 int32_t* enbr, int32_t* eslot, int32_t* epre) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        epre[0] = 0;
        epre[1] = (int32_t)n_ids;
    }
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_ids; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t u = ids[i];
        enbr[i] = u;
        if (u < 0) {
            dev_err(ERR_INDEX);
            eslot[i] = -1;
            continue;
        }
        eslot[i] = table_insert(table, logT, u, (uint32_t)(pos_base + i), nullptr);
    }
}

// ------------------------------------------------------------------- host
struct Plan {
    int K, H;
    int32_t bptr[SG_MAX_SUB + 1];
    int32_t fan[SG_MAX_HOPS];
    int64_t nb_tot[SG_MAX_HOPS + 1], eb_tot[SG_MAX_HOPS];
    int64_t capU;      // per mini-batch bound on |V_H^k|
    int logT;          // table slots per mini-batch = 2^logT
    int64_t nb_max, eb_max;
    // workspace offsets
    size_t o_table, o_ustr, o_gid, o_dbin, o_order, o_enbr, o_eslot, o_eflag, o_bsum, o_epre, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

sg_status make_plan(const sg_graph* g, int32_t n_seeds, const int32_t* h_bptr, int32_t n_sub, const int32_t* h_fan,
                    int32_t n_hops, Plan* p) {
    if (!g) return fail(SG_ERR_INVALID_ARG, "sampler: NULL graph");
    if (n_hops < 1 || n_hops > SG_MAX_HOPS) return fail(SG_ERR_INVALID_ARG, "sampler: n_hops must be 1..%d", SG_MAX_HOPS);
    if (!h_fan) return fail(SG_ERR_INVALID_ARG, "sampler: NULL fanouts");
    if (n_seeds < 0) return fail(SG_ERR_INVALID_ARG, "sampler: n_seeds < 0");
    const int K = h_bptr ? n_sub : 1;
    if (K < 1 || K > SG_MAX_SUB) return fail(SG_ERR_INVALID_ARG, "sampler: n_sub must be 1..%d", SG_MAX_SUB);
    p->K = K;
    p->H = n_hops;
    if (h_bptr) {
        if (h_bptr[0] != 0 || h_bptr[K] != n_seeds) return fail(SG_ERR_INVALID_ARG, "sampler: batch_ptr must run 0..n_seeds");
        for (int k = 0; k <= K; ++k) {
            if (k > 0 && h_bptr[k] < h_bptr[k - 1]) return fail(SG_ERR_INVALID_ARG, "sampler: batch_ptr decreases");
            p->bptr[k] = h_bptr[k];
        }
    } else {
        p->bptr[0] = 0;
        p->bptr[1] = n_seeds;
    }
    for (int h = 0; h < n_hops; ++h) {
        if (h_fan[h] < 1 || h_fan[h] > SG_MAX_FANOUT)
            return fail(SG_ERR_INVALID_ARG, "sampler: fanout %d outside 1..%d", h_fan[h], SG_MAX_FANOUT);
        p->fan[h] = h_fan[h];
    }
    const int64_t N = g->n_nodes, maxdeg = g->max_degree;
    for (int h = 0; h <= n_hops; ++h) p->nb_tot[h] = 0;
    for (int h = 0; h < n_hops; ++h) p->eb_tot[h] = 0;
    p->capU = 1;
    for (int k = 0; k < K; ++k) {
        int64_t nb = p->bptr[k + 1] - p->bptr[k];
        p->nb_tot[0] += nb;
        for (int h = 1; h <= n_hops; ++h) {
            const int64_t f = p->fan[h - 1] < maxdeg ? p->fan[h - 1] : maxdeg;
            const int64_t eb = nb * f;
            nb = nb + eb < N ? nb + eb : N;
            p->eb_tot[h - 1] += eb;
            p->nb_tot[h] += nb;
        }
        if (nb > p->capU) p->capU = nb;
    }
    p->nb_max = 1;
    p->eb_max = 1;
    for (int h = 0; h < n_hops; ++h) {
        if (p->nb_tot[h] > p->nb_max) p->nb_max = p->nb_tot[h];
        if (p->eb_tot[h] > p->eb_max) p->eb_max = p->eb_tot[h];
    }
    // table values hold local IDs (< capU) and edge positions capU + e
    if (p->capU + p->eb_max >= 2147483647LL || p->nb_tot[n_hops] >= 2147483647LL)
        return fail(SG_ERR_UNSUPPORTED, "sampler: a mini-batch this large needs 64-bit local IDs");
    int logT = 6;
    while (((int64_t)1 << logT) < 2 * p->capU) ++logT;
    p->logT = logT;
    size_t o = 0;
    p->o_table = o; o = align256(o + (size_t)K * ((size_t)1 << logT) * sizeof(uint2));
    p->o_ustr = o;  o = align256(o + (K > 1 ? (size_t)K * (size_t)p->capU * 4 : 0));
    p->o_gid = o;   o = align256(o + (size_t)p->nb_max * 4);
    p->o_dbin = o;  o = align256(o + (size_t)p->nb_max);
    p->o_order = o; o = align256(o + (size_t)p->nb_max * 4);
    p->o_enbr = o;  o = align256(o + (size_t)p->eb_max * 4);
    p->o_eslot = o; o = align256(o + (size_t)p->eb_max * 4);
    p->o_eflag = o; o = align256(o + (size_t)p->eb_max);
    p->o_bsum = o;  o = align256(o + (size_t)kMaxSeg * 8 * 4);
    p->o_epre = o;  o = align256(o + (size_t)(SG_MAX_SUB + 1) * 4);
    p->total = o;
    return SG_OK;
}

int seg_blocks(int64_t bound, int64_t per_block) {
    int64_t b = cdiv(bound, per_block);
    if (b < 1) b = 1;
    if (b > kMaxSeg) b = kMaxSeg;
    return (int)b;
}

uint32_t lambda_for(int f) {
    // expected candidates per random row: f + 4 sqrt(f) + 16 keeps fewer than f
    // (a retry) or more than the warp's 256 slots (the exact path) rare
    double lam = f + 4.0 * __builtin_sqrt((double)f) + 16.0;
    return (uint32_t)lam;
}

}  // namespace

extern "C" sg_status sg_sampler_bounds(const sg_graph* g, int32_t n_seeds, const int32_t* h_batch_ptr, int32_t n_sub,
                                       const int32_t* h_fanouts, int32_t n_hops, sg_sample_bounds* out) {
    if (!out) return fail(SG_ERR_INVALID_ARG, "sg_sampler_bounds: out is NULL");
    Plan p;
    sg_status st = make_plan(g, n_seeds, h_batch_ptr, n_sub, h_fanouts, n_hops, &p);
    if (st != SG_OK) return st;
    for (int h = 0; h <= SG_MAX_HOPS; ++h) out->max_nodes[h] = h <= n_hops ? p.nb_tot[h] : 0;
    for (int h = 0; h < SG_MAX_HOPS; ++h) out->max_edges[h] = h < n_hops ? p.eb_tot[h] : 0;
    out->counts_len = (int64_t)(2 * n_hops + 1) * (1 + p.K);
    out->workspace_bytes = p.total;
    return SG_OK;
}

extern "C" sg_status sg_sampler_run(const sg_graph* g, const int32_t* d_seeds, int32_t n_seeds, const int32_t* h_batch_ptr,
                                    int32_t n_sub, const int32_t* h_fanouts, int32_t n_hops, uint64_t seed,
                                    const uint64_t* d_seed, void* d_workspace, size_t workspace_bytes,
                                    const sg_blocks* out, sg_stream_t stream) {
    Plan p;
    sg_status st = make_plan(g, n_seeds, h_batch_ptr, n_sub, h_fanouts, n_hops, &p);
    if (st != SG_OK) return st;
    if (!out || !out->unique || !out->counts) return fail(SG_ERR_INVALID_ARG, "sg_sampler_run: output arrays missing");
    for (int h = 0; h < n_hops; ++h)
        if (!out->indptr[h] || !out->idx[h]) return fail(SG_ERR_INVALID_ARG, "sg_sampler_run: block arrays of hop %d missing", h + 1);
    if (n_seeds > 0 && !d_seeds) return fail(SG_ERR_INVALID_ARG, "sg_sampler_run: NULL seeds");
    if (!d_workspace || workspace_bytes < p.total)
        return fail(SG_ERR_INVALID_ARG, "sg_sampler_run: workspace needs %zu bytes", p.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_sampler_run: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d_workspace;
    const int K = p.K, H = p.H;
    CountsLayout L{H};
    HopArgs a;
    a.indptr = g->indptr;
    a.indices = g->indices;
    a.n_nodes = g->n_nodes;
    a.K = K;
    a.logT = p.logT;
    a.capU = p.capU;
    a.key0 = (uint32_t)(seed & 0xFFFFFFFFull);
    a.key1 = (uint32_t)(seed >> 32);
    a.d_seed = d_seed;
    a.pos_base = (int32_t)p.capU;
    a.L = L;
    a.counts = out->counts;
    a.ustr = K > 1 ? (int32_t*)(ws + p.o_ustr) : out->unique;
    a.table = (uint2*)(ws + p.o_table);
    a.dst_gid = (int32_t*)(ws + p.o_gid);
    a.dbin = (uint8_t*)(ws + p.o_dbin);
    a.order = (int32_t*)(ws + p.o_order);
    a.enbr = (int32_t*)(ws + p.o_enbr);
    a.eslot = (int32_t*)(ws + p.o_eslot);
    a.eflag = (uint8_t*)(ws + p.o_eflag);
    a.bsum = (int32_t*)(ws + p.o_bsum);
    a.epre = (int32_t*)(ws + p.o_epre);

    SG_CUDA(cudaMemsetAsync(a.table, 0xFF, (size_t)K * ((size_t)1 << p.logT) * sizeof(uint2), s));
    SubPtr bp;
    for (int k = 0; k <= K; ++k) bp.v[k] = p.bptr[k];
    {
        const int blocks = n_seeds > 0 ? (int)cdiv(n_seeds, 256) : 1;
        k_seed_init<<<blocks, 256, 0, s>>>(d_seeds, n_seeds, bp, K, g->n_nodes, a.table, p.logT, a.ustr, p.capU,
                                           out->counts, L);
        SG_CHECK_LAUNCH("k_seed_init");
    }
    const int sms = num_sms();
    for (int h = 1; h <= H; ++h) {
        a.h = h;
        a.fanout = p.fan[h - 1];
        a.lambda_num = lambda_for(a.fanout);
        a.bindptr = out->indptr[h - 1];
        a.bidx = out->idx[h - 1];
        const int64_t nb = p.nb_tot[h - 1], eb = p.eb_tot[h - 1];
        a.G_d = seg_blocks(nb, 2048);
        a.G_e = seg_blocks(eb, 4096);
        if (g->offset_bits == 32) k_dst_count<int32_t><<<a.G_d, kNT, 0, s>>>(a);
        else k_dst_count<int64_t><<<a.G_d, kNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_dst_count");
        k_dst_scan<<<a.G_d, kNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_dst_scan");
        int64_t sb = cdiv(nb, kSampleNT / 32);
        if (sb > (int64_t)sms * 8) sb = (int64_t)sms * 8;
        if (sb < 1) sb = 1;
        if (g->offset_bits == 32) k_sample<int32_t><<<(unsigned)sb, kSampleNT, 0, s>>>(a);
        else k_sample<int64_t><<<(unsigned)sb, kSampleNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_sample");
        k_flag<<<a.G_e, kNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_flag");
        k_assign<<<a.G_e, kNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_assign");
        int64_t mb = cdiv(eb, kNT * 4);
        if (mb > (int64_t)sms * 8) mb = (int64_t)sms * 8;
        if (mb < 1) mb = 1;
        k_map<<<(unsigned)mb, kNT, 0, s>>>(a);
        SG_CHECK_LAUNCH("k_map");
    }
    if (K > 1) {
        int64_t cb = cdiv(p.nb_tot[H], 256);
        if (cb > (int64_t)sms * 8) cb = (int64_t)sms * 8;
        if (cb < 1) cb = 1;
        k_compact<<<(unsigned)cb, 256, 0, s>>>(a.ustr, p.capU, K, out->counts, L, H, out->unique);
        SG_CHECK_LAUNCH("k_compact");
    }
    return SG_OK;
}

// ------------------------------------------------------ standalone relabel
namespace {
struct RelabelPlan {
    int logT;
    int64_t capU;
    size_t o_table, o_enbr, o_eslot, o_eflag, o_bsum, o_epre, o_counts, total;
};

bool relabel_plan(int64_t n_prefix, int64_t n_ids, RelabelPlan* p) {
    if (n_prefix < 0 || n_ids < 0 || n_prefix + 2 * n_ids >= 2147483647LL) return false;
    p->capU = n_prefix + n_ids + 1;
    int logT = 6;
    while (((int64_t)1 << logT) < 2 * p->capU) ++logT;
    p->logT = logT;
    size_t o = 0;
    p->o_table = o; o = align256(o + ((size_t)1 << logT) * sizeof(uint2));
    p->o_enbr = o; o = align256(o + (size_t)(n_ids + 1) * 4);
    p->o_eslot = o; o = align256(o + (size_t)(n_ids + 1) * 4);
    p->o_eflag = o; o = align256(o + (size_t)(n_ids + 1));
    p->o_bsum = o; o = align256(o + (size_t)kMaxSeg * 8 * 4);
    p->o_epre = o; o = align256(o + (size_t)(SG_MAX_SUB + 1) * 4);
    p->o_counts = o; o = align256(o + 16 * 4);
    p->total = o;
    return true;
}
}  // namespace

extern "C" size_t sg_relabel_workspace(int64_t n_prefix, int64_t n_ids) {
    RelabelPlan p;
    return relabel_plan(n_prefix, n_ids, &p) ? p.total : 0;
}

extern "C" sg_status sg_relabel(const int32_t* d_ids, int64_t n_ids, const int32_t* d_prefix, int64_t n_prefix,
                                int32_t* d_unique, int32_t* d_local, int32_t* d_n_unique, void* d_workspace,
                                size_t workspace_bytes, sg_stream_t stream) {
    RelabelPlan p;
    if (!relabel_plan(n_prefix, n_ids, &p)) return fail(SG_ERR_INVALID_ARG, "sg_relabel: sizes out of range");
    if ((n_ids > 0 && (!d_ids || !d_local)) || (n_prefix > 0 && !d_prefix) || !d_unique || !d_n_unique)
        return fail(SG_ERR_INVALID_ARG, "sg_relabel: NULL array");
    if (!d_workspace || workspace_bytes < p.total) return fail(SG_ERR_INVALID_ARG, "sg_relabel: workspace needs %zu bytes", p.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_relabel: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d_workspace;
    CountsLayout L{1};
    HopArgs a;
    a.indptr = nullptr;
    a.indices = nullptr;
    a.n_nodes = 2147483647LL;
    a.K = 1;
    a.logT = p.logT;
    a.capU = p.capU;
    a.key0 = a.key1 = 0;
    a.d_seed = nullptr;
    a.lambda_num = 0;
    a.pos_base = (int32_t)p.capU;
    a.L = L;
    a.counts = (int32_t*)(ws + p.o_counts);
    a.ustr = d_unique;
    a.table = (uint2*)(ws + p.o_table);
    a.dst_gid = nullptr;
    a.dbin = nullptr;
    a.order = nullptr;
    a.enbr = (int32_t*)(ws + p.o_enbr);
    a.eslot = (int32_t*)(ws + p.o_eslot);
    a.eflag = (uint8_t*)(ws + p.o_eflag);
    a.bsum = (int32_t*)(ws + p.o_bsum);
    a.epre = (int32_t*)(ws + p.o_epre);
    a.h = 1;
    a.fanout = 1;
    a.bindptr = nullptr;
    a.bidx = d_local;
    SG_CUDA(cudaMemsetAsync(a.table, 0xFF, ((size_t)1 << p.logT) * sizeof(uint2), s));
    SubPtr bp;
    bp.v[0] = 0;
    bp.v[1] = (int32_t)n_prefix;
    const int sms = num_sms();
    k_seed_init<<<n_prefix > 0 ? (int)cdiv(n_prefix, 256) : 1, 256, 0, s>>>(d_prefix, (int32_t)n_prefix, bp, 1, a.n_nodes,
                                                                          a.table, p.logT, a.ustr, p.capU, a.counts, L);
    SG_CHECK_LAUNCH("k_seed_init");
    int64_t ib = cdiv(n_ids, 256);
    if (ib > (int64_t)sms * 8) ib = (int64_t)sms * 8;
    if (ib < 1) ib = 1;
    k_relabel_insert<<<(unsigned)ib, 256, 0, s>>>(d_ids, n_ids, a.table, p.logT, a.pos_base, a.enbr, a.eslot, a.epre);
    SG_CHECK_LAUNCH("k_relabel_insert");
    a.G_e = seg_blocks(n_ids, 4096);
    k_flag<<<a.G_e, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_flag");
    k_assign<<<a.G_e, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_assign");
    k_map<<<(unsigned)ib, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_map");
    SG_CUDA(cudaMemcpyAsync(d_n_unique, a.counts + L.tot_n(1), sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    return SG_OK;
}

// ------------------------------------------- relabel without allocation
// The scratch of sg_relabel_noalloc: a static device array, so callers that
// cannot allocate device memory still get a relabel.  Host code must not use
// the array's name as an address; the device address is looked up once per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_relabel_scratch[SG_RELABEL_NOALLOC_SCRATCH_BYTES];

#include <mutex>

namespace {
std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};

sg_status relabel_scratch_address(void** out) {
    int dev = 0;
    SG_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(SG_ERR_UNSUPPORTED, "sg_relabel_noalloc: device ordinal %d >= 64", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_relabel_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e, "sg_relabel_noalloc: cudaGetSymbolAddress of the static scratch");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SG_OK;
}
}  // namespace

extern "C" sg_status sg_relabel_noalloc(const int32_t* d_ids, int64_t n_ids, const int32_t* d_prefix, int64_t n_prefix,
                                        int32_t* d_unique, int32_t* d_local, int32_t* d_n_unique, sg_stream_t stream) {
    if (n_ids < 0 || n_prefix < 0) return fail(SG_ERR_INVALID_ARG, "sg_relabel_noalloc: negative size");
    if (n_ids + n_prefix > SG_RELABEL_NOALLOC_MAX_IDS)
        return fail(SG_ERR_INVALID_ARG,
                    "sg_relabel_noalloc: n_prefix + n_ids = %lld exceeds the static scratch limit of %d IDs; "
                    "use sg_relabel with a caller workspace",
                    (long long)(n_ids + n_prefix), SG_RELABEL_NOALLOC_MAX_IDS);
    RelabelPlan p;
    if (!relabel_plan(n_prefix, n_ids, &p) || p.total > SG_RELABEL_NOALLOC_SCRATCH_BYTES)
        return fail(SG_ERR_INVALID_ARG, "sg_relabel_noalloc: sizes out of range");
    if ((n_ids > 0 && (!d_ids || !d_local)) || (n_prefix > 0 && !d_prefix) || !d_unique || !d_n_unique)
        return fail(SG_ERR_INVALID_ARG, "sg_relabel_noalloc: NULL array");
    void* scratch = nullptr;
    sg_status st = relabel_scratch_address(&scratch);
    if (st != SG_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)scratch;
    CountsLayout L{1};
    HopArgs a;
    a.indptr = nullptr;
    a.indices = nullptr;
    a.n_nodes = 2147483647LL;
    a.K = 1;
    a.logT = p.logT;
    a.capU = p.capU;
    a.key0 = a.key1 = 0;
    a.d_seed = nullptr;
    a.lambda_num = 0;
    a.pos_base = (int32_t)p.capU;
    a.L = L;
    a.counts = (int32_t*)(ws + p.o_counts);
    a.ustr = d_unique;
    a.table = (uint2*)(ws + p.o_table);
    a.dst_gid = nullptr;
    a.dbin = nullptr;
    a.order = nullptr;
    a.enbr = (int32_t*)(ws + p.o_enbr);
    a.eslot = (int32_t*)(ws + p.o_eslot);
    a.eflag = (uint8_t*)(ws + p.o_eflag);
    a.bsum = (int32_t*)(ws + p.o_bsum);
    a.epre = (int32_t*)(ws + p.o_epre);
    a.h = 1;
    a.fanout = 1;
    a.bindptr = nullptr;
    a.bidx = d_local;
    // the array keeps the previous call's contents: the table must start empty
    SG_CUDA(cudaMemsetAsync(a.table, 0xFF, ((size_t)1 << p.logT) * sizeof(uint2), s));
    SubPtr bp;
    bp.v[0] = 0;
    bp.v[1] = (int32_t)n_prefix;
    const int sms = num_sms();
    k_seed_init<<<n_prefix > 0 ? (int)cdiv(n_prefix, 256) : 1, 256, 0, s>>>(d_prefix, (int32_t)n_prefix, bp, 1, a.n_nodes,
                                                                          a.table, p.logT, a.ustr, p.capU, a.counts, L);
    SG_CHECK_LAUNCH("k_seed_init");
    int64_t ib = cdiv(n_ids, 256);
    if (ib > (int64_t)sms * 8) ib = (int64_t)sms * 8;
    if (ib < 1) ib = 1;
    k_relabel_insert<<<(unsigned)ib, 256, 0, s>>>(d_ids, n_ids, a.table, p.logT, a.pos_base, a.enbr, a.eslot, a.epre);
    SG_CHECK_LAUNCH("k_relabel_insert");
    a.G_e = seg_blocks(n_ids, 4096);
    k_flag<<<a.G_e, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_flag");
    k_assign<<<a.G_e, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_assign");
    k_map<<<(unsigned)ib, kNT, 0, s>>>(a);
    SG_CHECK_LAUNCH("k_map");
    SG_CUDA(cudaMemcpyAsync(d_n_unique, a.counts + L.tot_n(1), sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    return SG_OK;
}

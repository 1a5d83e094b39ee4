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
//    BatchPtr; dedup goes through GPU hash tables; node classification is
//    turned into index arithmetic (here: degree bins that order the work).
//    A node that appears in several mini-batches of the super-batch is
//    sampled once per hop and its sample copied to the others.
//  - FastGL explainer page, "Fused-Map": there one atomic pass builds the
//    table and hands out local IDs in arrival order.  Here the insert pass
//    keeps the minimum edge position per node (atomicMin) and one flag + scan
//    pass turns that into the deterministic first-occurrence numbering.
//
// The workspace holds, per mini-batch, a direct map from node ID to the
// smallest edge position that names it (then to its local ID); it and the
// scan states arrive all-ones and every run leaves them so (k_cleanup).  Per
// hop h three kernels run (four for a super-batch):
//   k_rows     one pass over the dst rows V_{h-1}: c_v = min(deg, f), the
//              block row pointer by a single-pass exclusive scan (decoupled
//              look-back), per-row metadata and the rows' degree bins (work
//              order, largest first).  For hop 1 it also places the seeds;
//              for later hops it also maps the previous hop's edges.
//   k_sample   rows by bin, handed out by counters: a block per row longer
//              than 4096, a warp per other long row, an 8-lane group per
//              short row; full rows are copied, random rows hashed with
//              Philox; keys under a threshold are candidates (a shared-memory
//              pool) and the f smallest are picked exactly; every emitted
//              neighbour records its edge position in its mini-batch's map
//              (atomicMin keeps the first occurrence)
//   k_copy     (super-batch only) rows whose node another row samples copy it
//   k_relabel  first-occurrence flags, ranked by a single-pass scan per
//              mini-batch: new local IDs into the map and into V_h
// then k_finish maps the last hop's edges (and lays a super-batch out) and
// k_cleanup restores the workspace.
#include <string.h>

#include <mutex>

#include "sg_internal.cuh"
#include "sg_objects.cuh"

SGI_ERROR_WORD(sampler)

using namespace sgi;

namespace {

constexpr int kNT = 256;             // threads of every sampler kernel (8 warps)
constexpr int kTile = 1024;          // rows / edges per scan tile (4 per thread)
constexpr int kUnitQueues = 8;      // k_sample's warp units come from this many counters
constexpr int kCtrWords = 32 + 32 * kUnitQueues;  // counters of one hop (see HopArgs::ctr)
constexpr int kGroupLambdaMax = 64;  // short random rows go to 8-lane groups when f + 2 sqrt(f) + 4 <= this
constexpr uint32_t kEmpty = 0xFFFFFFFFu;

struct SubPtr {
    int32_t v[SG_MAX_SUB + 1];
};

// Where the counts live (see sg_blocks in sg.h).
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
    int lo = 0, hi = K;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)sp[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

// pre[k] = sum_{k'<k} counts[sub_n(k', h)], pre[K] = total (shared memory).
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

// ------------------------------------------------------------------ seeds
// Seeds take local IDs 0..B_k-1 of their mini-batch.  A repeated seed inside
// one mini-batch or an ID out of range is reported through the error word.
__global__ void k_seed_init(const int32_t* __restrict__ seeds, int32_t n_seeds, SubPtr bptr, int K, int64_t n_nodes,
                            uint2* table, int logT, int32_t* ustr, int64_t capU, int32_t* counts, CountsLayout L) {
    pdl_start();
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

// ---------------------------------------------------------------- hop args
// What k_sample needs of a row, written into its degree bin by k_rows so that
// a unit of work is one record load: the row's CSR start and degree, its
// node, its index in V_{h-1} and its first edge in the block.
struct __align__(16) BinRec {
    int32_t start_lo, start_hi, deg, v;
    int32_t r, out0, pad0, pad1;
};

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
    // this hop's rows
    struct BinRec* brec;     // the four degree bins (see bin_slot)
    int64_t bin_cap;         // capacity of one half of brec (rows of the hop's bound)
    uint32_t* ctr;           // [0] row tiles, [1] edge tiles, [2..9] bin sizes, [10] block rows, [32 + 32 q] unit queue q
    unsigned long long* row_status;
    unsigned long long* edge_status;
    int32_t* bindptr;
    int32_t* epre;           // [K+1] edge offset of each mini-batch in this hop
    int32_t* enbr;
    int32_t* eslot;          // standalone relabel: table slot of each id
    uint32_t* pos_of;        // sampler: direct map, [K][n_nodes] first position / local ID
    const int32_t* prev_enbr;
    // super-batch owner rows
    uint2* utab;
    int logU;
    int32_t* rslot;
    // the previous hop's edges (mapped by k_rows)
    int32_t* prev_bidx;
    const int32_t* prev_epre;
    const int32_t* prev_eslot;
    int map_blocks;
};

// Entry i of bin b.  Bins 2j and 2j+1 share quarter j of brec (the even bin
// from its start, the odd one from its end), so the eight bins of a hop take
// four row capacities.
__device__ __forceinline__ BinRec* bin_slot(const HopArgs& a, int b, int64_t i) {
    const int64_t half = (int64_t)(b >> 1) * a.bin_cap;
    return a.brec + half + ((b & 1) ? a.bin_cap - 1 - i : i);
}

__device__ __forceinline__ BinRec load_rec(const BinRec* p) {
    const int4 x = reinterpret_cast<const int4*>(p)[0], y = reinterpret_cast<const int4*>(p)[1];
    BinRec rc;
    rc.start_lo = x.x;
    rc.start_hi = x.y;
    rc.deg = x.z;
    rc.v = x.w;
    rc.r = y.x;
    rc.out0 = y.y;
    rc.pad0 = rc.pad1 = 0;
    return rc;
}

// bins: 0 full row, 1 small random row (8-lane groups), 2..4 random rows up
// to 1024, 2048 and 4096 positions (a warp each), 5..7 up to 8192, 16384 and
// longer (a block each).  Work goes out longest first (bins 7..5, then 4..2,
// then 1 and 0), so that no long row is started last.
constexpr int kBins = 8;
__device__ __forceinline__ int degree_bin(int64_t deg, int f, bool group_ok) {
    if (deg <= f) return 0;
    if (deg <= 256 && group_ok) return 1;
    if (deg <= 1024) return 2;
    if (deg <= 2048) return 3;
    if (deg <= 4096) return 4;
    if (deg <= 8192) return 5;
    if (deg <= 16384) return 6;
    return 7;
}

// Edge e of the previous hop gets its src row (mini-batch offset + local ID).
// spre holds the prefix of the mini-batches' node counts of that hop.
__device__ void map_prev_edges(const HopArgs& a, int blk, int nblk, int32_t* ep, const int32_t* spre) {
    const int K = a.K;
    for (int k = threadIdx.x; k <= K; k += kNT) ep[k] = a.prev_epre[k];
    __syncthreads();
    const int64_t E = ep[K];
    for (int64_t e = (int64_t)blk * kNT + threadIdx.x; e < E; e += (int64_t)nblk * kNT) {
        const int k = K == 1 ? 0 : find_sub(ep, K, e);
        int32_t out = -1;
        if (a.pos_of) {
            out = spre[k] + (int32_t)a.pos_of[(int64_t)k * a.n_nodes + a.prev_enbr[e]];
        } else {
            const int32_t s = a.prev_eslot[e];
            if (s >= 0) out = spre[k] + (int32_t)a.table[s].y;
        }
        a.prev_bidx[e] = out;
    }
}

// In seed mode (hop 1) the rows are the seeds themselves, in the given order
// (V_0 of every mini-batch, back to back): each is also placed, with local
// ID = its index inside its mini-batch, in that mini-batch's table and V_0.
template <typename Off>
__global__ void __launch_bounds__(kNT) k_rows(HopArgs a, int seed_mode, const int32_t* __restrict__ seeds,
                                              SubPtr bptr) {
    pdl_start();
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ int32_t ep[SG_MAX_SUB + 1];
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ int32_t s_tile, s_excl, s_bcnt[kBins], s_bbase[kBins];
    if (seed_mode) {
        for (int k = threadIdx.x; k <= a.K; k += kNT) pre[k] = bptr.v[k];
        __syncthreads();
        if (blockIdx.x == 0)
            for (int k = threadIdx.x; k < a.K; k += kNT) a.counts[a.L.sub_n(k, 0)] = pre[k + 1] - pre[k];
    } else {
        load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);  // V_{h-1} per mini-batch
    }
    const int64_t T = pre[a.K];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.counts[a.L.tot_n(a.h - 1)] = (int32_t)T;
        if (T == 0) {
            a.bindptr[0] = 0;
            a.counts[a.L.tot_e(a.h)] = 0;
            for (int k = 0; k <= a.K; ++k) a.epre[k] = 0;
        }
    }
    if ((int)blockIdx.x < a.map_blocks) {  // the previous hop's edges
        map_prev_edges(a, blockIdx.x, a.map_blocks, ep, pre);
        return;
    }
    const Off* indptr = (const Off*)a.indptr;
    const int f = a.fanout;
    const bool group_ok = a.lambda_num <= (uint32_t)kGroupLambdaMax;
    const int64_t n_tiles = (T + kTile - 1) / kTile;
    // blocks past the tile count leave at once; the others take tiles in
    // order (one each unless the grid is smaller than the tile count)
    const int64_t row_block = (int64_t)blockIdx.x - a.map_blocks;
    const int64_t row_grid = (int64_t)gridDim.x - a.map_blocks;
    if (row_block >= n_tiles) return;
    for (int iter = 0;; ++iter) {
        if (iter > 0 && row_grid >= n_tiles) break;
        if (threadIdx.x == 0) s_tile = (int32_t)(atomicAdd(a.ctr + 0, 1u) + 1u);
        __syncthreads();
        const int64_t tile = s_tile;
        if (tile >= n_tiles) break;
        const int64_t r0 = tile * kTile + (int64_t)threadIdx.x * 4;
        int32_t c[4], dg[4], vv[4];
        int64_t st[4];
        int b[4], kq[4];
        int32_t mysum = 0;
        // the four rows' nodes, then their CSR bounds, each set loaded at
        // once; the side effects (seed placement, owner table) come after
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t r = r0 + q;
            kq[q] = 0;
            vv[q] = -1;
            if (r < T) {
                kq[q] = find_sub(pre, a.K, r);
                vv[q] = seed_mode ? seeds[r] : a.ustr[(int64_t)kq[q] * a.capU + (r - pre[kq[q]])];
            }
        }
        int64_t en[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            st[q] = 0;
            en[q] = 0;
            if (r0 + q < T && vv[q] >= 0 && (int64_t)vv[q] < a.n_nodes) {
                st[q] = (int64_t)indptr[vv[q]];
                en[q] = (int64_t)indptr[vv[q] + 1];
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t r = r0 + q;
            c[q] = 0;
            b[q] = -1;
            dg[q] = 0;
            if (r < T) {
                const int k = kq[q];
                const int32_t v = vv[q];
                const bool ok = v >= 0 && (int64_t)v < a.n_nodes;
                if (seed_mode) {
                    const int32_t l = (int32_t)(r - pre[k]);
                    a.ustr[(int64_t)k * a.capU + l] = v;
                    if (ok) {
                        const uint32_t old = atomicMin(a.pos_of + (int64_t)k * a.n_nodes + v, (uint32_t)l);
                        if (old != kEmpty) dev_err(ERR_ARG);  // a repeated seed in one mini-batch
                    }
                }
                if (!ok) dev_err(ERR_INDEX);
                const int64_t deg = en[q] - st[q];
                c[q] = (int32_t)(deg < f ? deg : f);
                b[q] = degree_bin(deg, f, group_ok);
                dg[q] = (int32_t)deg;
                if (a.utab) {  // super-batch: the first row of a node samples it
                    a.rslot[r] = ok ? table_insert(a.utab, a.logU, v, (uint32_t)r, nullptr) : -1;
                }
            }
            mysum += c[q];
        }
        int32_t tile_total;
        const int32_t ex = block_excl_scan<kNT>(mysum, red, tile_total);
        if (threadIdx.x < 32) {
            bool late = false;
            const int32_t x = chain_lookback(a.row_status, (int)tile, 0, tile_total, &late);
            if (threadIdx.x == 0) s_excl = x;
            if (late && threadIdx.x == 0) dev_err(ERR_TIMEOUT);
        }
        // bin sizes of the tile, then one global atomic per bin
        if (threadIdx.x < kBins) s_bcnt[threadIdx.x] = 0;
        __syncthreads();
        int brank[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) brank[q] = b[q] >= 0 ? atomicAdd(&s_bcnt[b[q]], 1) : 0;
        __syncthreads();
        if (threadIdx.x < kBins)
            s_bbase[threadIdx.x] =
                s_bcnt[threadIdx.x] ? (int32_t)(atomicAdd(a.ctr + 2 + threadIdx.x, (uint32_t)s_bcnt[threadIdx.x]) + 1u) : 0;
        __syncthreads();
        int32_t off = s_excl + ex;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t r = r0 + q;
            if (r < T) {
                a.bindptr[r] = off;
                int k = find_sub(pre, a.K, r);
                while (k >= 0 && pre[k] == r) {  // first row of mini-batch k (and of empty ones before it)
                    a.epre[k] = off;
                    --k;
                }
                if (b[q] >= 0) {
                    int4* d = reinterpret_cast<int4*>(bin_slot(a, b[q], s_bbase[b[q]] + brank[q]));
                    d[0] = make_int4((int32_t)(uint32_t)st[q], (int32_t)(st[q] >> 32), dg[q], vv[q]);
                    d[1] = make_int4((int32_t)r, off, 0, 0);
                }
            }
            off += c[q];
        }
        if (tile == n_tiles - 1 && threadIdx.x == kNT - 1) {
            const int32_t E = s_excl + tile_total;
            a.bindptr[T] = E;
            a.counts[a.L.tot_e(a.h)] = E;
            for (int k = a.K; k >= 0 && pre[k] == T; --k) a.epre[k] = E;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ sample
// Key threshold keeping about lam of deg positions as candidates; any value
// gives the same sample (the filter only decides how many keys are ranked).
__device__ __forceinline__ uint32_t threshold_for(uint32_t lam, int64_t deg) {
    const float t = (float)lam * 4294967296.0f / (float)deg;
    return t >= 4294967040.0f ? 0xFFFFFFFFu : (uint32_t)t;
}

// Edge e of a mini-batch gets node u: recorded, and the node's entry in the
// mini-batch's direct map `pos` keeps the smallest position (no reply is
// waited for).
__device__ __forceinline__ void emit_edge(const HopArgs& a, uint32_t* pos, int64_t e, int32_t u) {
    a.enbr[e] = u;
    atomicMin(pos + u, (uint32_t)(a.pos_base + e));
}

__device__ __forceinline__ unsigned long long min_u64_xor(unsigned long long x, unsigned mask, int width) {
    for (int d = width >> 1; d > 0; d >>= 1) {
        const unsigned long long o = __shfl_xor_sync(mask, x, d, width);
        x = o < x ? o : x;
    }
    return x;
}

// Exact bottom-f by f passes of a group-wide minimum over all positions;
// used only when the threshold filter cannot hold or find f keys.  A group is
// W lanes (8 or 32) named by `mask`; cj has room for f entries.
template <int W>
__device__ void sample_exact(const HopArgs& a, uint32_t* tab, uint32_t k0, uint32_t k1, int32_t v, int64_t start,
                             int64_t deg, int64_t out0, int32_t* cj, unsigned mask, int gl) {
    const int f = a.fanout;
    unsigned long long prev = 0;
    for (int s = 0; s < f; ++s) {
        unsigned long long best = ~0ull;
        for (int64_t base = 0; base < deg; base += 4 * W) {
            const int64_t q = (base >> 2) + gl;
            if (4 * q < deg) {
                const uint4 w = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)v, (uint32_t)a.h, 0u), k0, k1);
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
        best = min_u64_xor(best, mask, W);
        if (gl == 0) cj[s] = (int32_t)(best & 0xFFFFFFFFull);
        prev = best;
    }
    __syncwarp(mask);
    for (int i = gl; i < f; i += W) {  // list the f positions in ascending order
        const int32_t x = cj[i];
        int rank = 0;
        for (int t = 0; t < f; ++t) rank += cj[t] < x;
        emit_edge(a, tab, out0 + rank, a.indices[start + x]);
    }
    __syncwarp(mask);
}

// Candidates: a pool holds the key (Philox word) and the row position of
// every candidate in two arrays, keys[] and pos[], filled in arbitrary order.
constexpr int kWarpPool = 512;                      // candidates of a warp
constexpr int kGroupPool = kWarpPool / 4;           // of an 8-lane group
constexpr int kBlockPool = kWarpPool * (kNT / 32);  // of a block (rows longer than 4096)
constexpr int kWarpSel = 256;                       // picked positions of a warp (f <= 256)
constexpr int kGroupSel = kWarpSel / 4;             // of an 8-lane group (f + 2 sqrt(f) + 4 <= 64)

struct Pool {
    uint32_t* keys;  // room for cap entries, 16-byte aligned, cap a multiple of 4
    uint32_t* pos;
    uint32_t* sel;   // room for f entries
    int* n;          // fill count (shared)
    int cap;
};

// Adds one candidate; past cap the entry is dropped, and the caller sees the
// overflow as *n > cap.
__device__ __forceinline__ void push_cand(const Pool& p, uint32_t key, uint32_t j) {
    const int s = atomicAdd(p.n, 1);
    if (s < p.cap) {
        p.keys[s] = key;
        p.pos[s] = j;
    }
}

// The positions of counter block q (4q .. 4q+3, those below deg) whose key is
// at most tau.  4q < deg holds.
__device__ __forceinline__ void filter_block(const uint4& w, uint32_t q, uint32_t deg, uint32_t tau, const Pool& p) {
    const uint32_t j0 = 4u * q, rem = deg - j0;
    if (w.x <= tau) push_cand(p, w.x, j0);
    if (w.y <= tau && rem > 1u) push_cand(p, w.y, j0 + 1u);
    if (w.z <= tau && rem > 2u) push_cand(p, w.z, j0 + 2u);
    if (w.w <= tau && rem > 3u) push_cand(p, w.w, j0 + 3u);
}

// Hashes every position of row v by `nthr` threads (this one is number t):
// each step takes counter blocks t and t + nthr of the next 2 * nthr, as two
// independent Philox chains.
__device__ __forceinline__ void hash_row(const HopArgs& a, uint32_t k0, uint32_t k1, int32_t v, uint32_t deg,
                                         uint32_t tau, const Pool& p, uint32_t t, uint32_t nthr) {
    const uint32_t qn = (deg + 3u) >> 2;
    for (uint32_t qb = 0; qb < qn; qb += 2u * nthr) {
        const uint32_t qa = qb + t, qc = qa + nthr;
        const uint4 wa = philox4x32_10(make_uint4(qa, (uint32_t)v, (uint32_t)a.h, 0u), k0, k1);
        const uint4 wc = philox4x32_10(make_uint4(qc, (uint32_t)v, (uint32_t)a.h, 0u), k0, k1);
        if (qa < qn) filter_block(wa, qa, deg, tau, p);
        if (qc < qn) filter_block(wc, qc, deg, tau, p);
    }
}

__device__ __forceinline__ uint32_t widen(uint32_t tau) { return tau > 0x3FFFFFFFu ? 0xFFFFFFFFu : (tau << 2) | 3u; }

// A group of threads that picks together: W lanes of a warp named by a mask,
// or the whole block.
struct LaneGroup {
    unsigned mask;
    __device__ void sync() const { __syncwarp(mask); }
    __device__ bool any(bool x) const { return __any_sync(mask, x); }
};
struct BlockGroup {
    __device__ void sync() const { __syncthreads(); }
    __device__ bool any(bool x) const { return __syncthreads_or(x) != 0; }
};

// The f smallest of the n pool candidates (f <= n <= cap) by (key, position),
// emitted in position order.  A candidate's rank is the number of keys below
// its own (16-byte loads of four keys at a time); a candidate of rank r < f
// puts its position in sel[r].  Two equal keys below the f-th get the same
// rank, so some slot is claimed twice; then the ranks are taken again with the
// position as tie-break.  The output slot of sel[r] is the number of picks at
// smaller positions.  The group is `nthr` threads (this one is number t).
template <typename Grp>
__device__ __forceinline__ void pick_emit(const HopArgs& a, uint32_t* tab, const Pool& p, int n, int64_t start,
                                          int64_t out0, int t, int nthr, const Grp& grp) {
    const int f = a.fanout;
    const int n4 = (n + 3) & ~3;
    for (int i = n + t; i < n4; i += nthr) p.keys[i] = 0xFFFFFFFFu;  // never below a real key
    for (int i = t; i < f; i += nthr) p.sel[i] = 0xFFFFFFFFu;        // no position is this large
    grp.sync();
    const uint4* k4 = reinterpret_cast<const uint4*>(p.keys);
    bool tie = false;
    for (int i = t; i < n; i += nthr) {
        const uint32_t x = p.keys[i];
        int rank = 0;
#pragma unroll 2
        for (int s = 0; s < (n4 >> 2); ++s) {
            const uint4 k = k4[s];
            rank += (k.x < x) + (k.y < x) + (k.z < x) + (k.w < x);
        }
        if (rank < f && atomicExch(&p.sel[rank], p.pos[i]) != 0xFFFFFFFFu) tie = true;
    }
    grp.sync();
    if (grp.any(tie)) {  // equal keys: rank by (key, position)
        for (int i = t; i < n; i += nthr) {
            const uint32_t x = p.keys[i], j = p.pos[i];
            int rank = 0;
            for (int s = 0; s < n; ++s) rank += (p.keys[s] < x) || (p.keys[s] == x && p.pos[s] < j);
            if (rank < f) p.sel[rank] = j;
        }
        grp.sync();
    }
    for (int r = t; r < f; r += nthr) {
        const uint32_t j = p.sel[r];
        int slot = 0;
        for (int q = 0; q < f; ++q) slot += p.sel[q] < j;
        emit_edge(a, tab, out0 + slot, a.indices[start + j]);
    }
    grp.sync();
}

// One random row by a group of W lanes (W = 8 or 32) named by `mask`: keys at
// most tau become candidates (about lambda of them), and the f smallest are
// emitted.  With fewer than f candidates tau widens (twice at most); when the
// pool overflows or two widenings do not suffice, the exact path runs.
template <int W>
__device__ void sample_random_row(const HopArgs& a, uint32_t* tab, uint32_t k0, uint32_t k1, int32_t v, int64_t start,
                                  uint32_t deg, int64_t out0, const Pool& p, unsigned mask, int gl) {
    const int f = a.fanout;
    const LaneGroup grp{mask};
    uint32_t tau = threshold_for(a.lambda_num, deg);
    for (int attempt = 0; attempt < 3; ++attempt) {
        if (gl == 0) *p.n = 0;
        __syncwarp(mask);
        hash_row(a, k0, k1, v, deg, tau, p, (uint32_t)gl, W);
        __syncwarp(mask);
        const int n = *p.n;
        __syncwarp(mask);
        if (n > p.cap) break;
        if (n < f) {
            tau = widen(tau);
            continue;
        }
        pick_emit(a, tab, p, n, start, out0, gl, W, grp);
        return;
    }
    sample_exact<W>(a, tab, k0, k1, v, start, deg, out0, (int32_t*)p.sel, mask, gl);
}

// One row of the frontier (its bin record), by a group of W lanes.
template <int W>
__device__ void sample_row(const HopArgs& a, const BinRec& rc, const int32_t* pre, uint32_t k0, uint32_t k1,
                           const Pool& p, unsigned mask, int gl) {
    const int32_t v = rc.v, r = rc.r;
    const int64_t deg = rc.deg;
    if (v < 0 || (int64_t)v >= a.n_nodes || deg == 0) return;
    if (a.utab && (a.rslot[r] < 0 || (int32_t)a.utab[a.rslot[r]].y != r)) return;  // another row samples this node
    const int64_t start = (int64_t)(uint32_t)rc.start_lo | ((int64_t)rc.start_hi << 32);
    const int64_t out0 = rc.out0;
    uint32_t* tab = a.pos_of + (int64_t)(a.K == 1 ? 0 : find_sub(pre, a.K, r)) * a.n_nodes;
    if (deg <= a.fanout) {  // full node: every neighbour, in row order
        for (int64_t t = gl; t < deg; t += W) emit_edge(a, tab, out0 + t, a.indices[start + t]);
        return;
    }
    sample_random_row<W>(a, tab, k0, k1, v, start, (uint32_t)deg, out0, p, mask, gl);
}

// Four short random rows at once, one per 8-lane group of the warp (the steps
// of sample_random_row).  Every loop runs to the warp-wide maximum trip count
// with per-group predicates, so the groups stay converged: diverged groups
// would take turns.  A group whose pool overflows, keeps fewer than f keys or
// holds equal keys finishes alone (rare).
__device__ void sample_rows_x4(const HopArgs& a, const BinRec& rc, bool valid, const int32_t* pre, uint32_t k0,
                               uint32_t k1, const Pool& p, unsigned gmask, int gl) {
    const int f = a.fanout;
    int32_t v = 0;
    uint32_t deg = 0;
    int64_t start = 0, out0 = 0;
    uint32_t* tab = a.pos_of;
    if (valid) {
        const int32_t r = rc.r;
        v = rc.v;
        deg = (uint32_t)rc.deg;
        valid = v >= 0 && (int64_t)v < a.n_nodes && (int64_t)deg > f;
        if (valid && a.utab && (a.rslot[r] < 0 || (int32_t)a.utab[a.rslot[r]].y != r)) valid = false;
        start = (int64_t)(uint32_t)rc.start_lo | ((int64_t)rc.start_hi << 32);
        out0 = rc.out0;
        tab = a.pos_of + (int64_t)(a.K == 1 ? 0 : find_sub(pre, a.K, r)) * a.n_nodes;
    }
    const uint32_t tau = valid ? threshold_for(a.lambda_num, deg) : 0u;
    const uint32_t qn = valid ? (deg + 3u) >> 2 : 0u;
    const uint32_t max_steps = __reduce_max_sync(0xffffffffu, (qn + 15u) >> 4);
    if (gl == 0) *p.n = 0;
    __syncwarp();
    for (uint32_t st = 0; st < max_steps; ++st) {
        const uint32_t qa = st * 16u + (uint32_t)gl, qc = qa + 8u;
        const uint4 wa = philox4x32_10(make_uint4(qa, (uint32_t)v, (uint32_t)a.h, 0u), k0, k1);
        const uint4 wc = philox4x32_10(make_uint4(qc, (uint32_t)v, (uint32_t)a.h, 0u), k0, k1);
        if (qa < qn) filter_block(wa, qa, deg, tau, p);
        if (qc < qn) filter_block(wc, qc, deg, tau, p);
    }
    __syncwarp();
    const int n = *p.n;
    bool ok = valid && n >= f && n <= p.cap;
    const int n_max = (int)__reduce_max_sync(0xffffffffu, ok ? (unsigned)n : 0u);
    const int n4 = (n_max + 3) & ~3;  // the same padded length for every group
    if (ok) {
        for (int i = n + gl; i < n4; i += 8) p.keys[i] = 0xFFFFFFFFu;
        for (int i = gl; i < f; i += 8) p.sel[i] = 0xFFFFFFFFu;
    }
    __syncwarp();
    const uint4* k4 = reinterpret_cast<const uint4*>(p.keys);
    bool tie = false;
    for (int i0 = 0; i0 < n_max; i0 += 8) {
        const int i = i0 + gl;
        const bool in = ok && i < n;
        const uint32_t x = in ? p.keys[i] : 0u;
        int rank = 0;
#pragma unroll 2
        for (int s = 0; s < (n4 >> 2); ++s) {
            const uint4 k = k4[s];
            rank += (k.x < x) + (k.y < x) + (k.z < x) + (k.w < x);
        }
        if (in && rank < f && atomicExch(&p.sel[rank], p.pos[i]) != 0xFFFFFFFFu) tie = true;
    }
    __syncwarp();
    if (ok && __any_sync(gmask, tie)) ok = false;  // equal keys: this group takes the general path
    for (int r0 = 0; r0 < f; r0 += 8) {
        const int rr = r0 + gl;
        if (ok && rr < f) {
            const uint32_t j = p.sel[rr];
            int slot = 0;
            for (int q = 0; q < f; ++q) slot += p.sel[q] < j;
            emit_edge(a, tab, out0 + slot, a.indices[start + j]);
        }
    }
    __syncwarp();
    if (valid && !ok) sample_random_row<8>(a, tab, k0, k1, v, start, deg, out0, p, gmask, gl);
    __syncwarp();
}

// A random row longer than 4096 by the whole block (the same steps as
// sample_random_row, with 256 threads and the block's pool).
__device__ void sample_big_row(const HopArgs& a, const BinRec& rc, const int32_t* pre, uint32_t k0, uint32_t k1,
                               const Pool& p) {
    const int32_t v = rc.v, r = rc.r;
    const int64_t deg = rc.deg;
    if (v < 0 || (int64_t)v >= a.n_nodes || deg <= a.fanout) return;
    if (a.utab && (a.rslot[r] < 0 || (int32_t)a.utab[a.rslot[r]].y != r)) return;
    const int64_t start = (int64_t)(uint32_t)rc.start_lo | ((int64_t)rc.start_hi << 32);
    const int64_t out0 = rc.out0;
    uint32_t* tab = a.pos_of + (int64_t)(a.K == 1 ? 0 : find_sub(pre, a.K, r)) * a.n_nodes;
    const int f = a.fanout;
    uint32_t tau = threshold_for(a.lambda_num, deg);
    const BlockGroup grp;
    for (int attempt = 0; attempt < 3; ++attempt) {
        if (threadIdx.x == 0) *p.n = 0;
        __syncthreads();
        hash_row(a, k0, k1, v, (uint32_t)deg, tau, p, threadIdx.x, kNT);
        __syncthreads();
        const int n = *p.n;
        __syncthreads();
        if (n > p.cap) break;
        if (n < f) {
            tau = widen(tau);
            continue;
        }
        pick_emit(a, tab, p, n, start, out0, (int)threadIdx.x, kNT, grp);
        return;
    }
    if (threadIdx.x < 32) sample_exact<32>(a, tab, k0, k1, v, start, deg, out0, (int32_t*)p.sel, 0xffffffffu, (int)lane_id());
    __syncthreads();
}

// Rows by bin, largest first, handed out by counters so that no SM is left
// with a long tail: blocks take the rows of bins 7, 6 and 5 one at a time,
// then warps take units (a row of bins 4, 3 or 2; four bin 1 rows, one per
// 8-lane group; or sixteen full rows).  The grid is at most what fits on the
// GPU at once.
__global__ void __launch_bounds__(kNT, 4) k_sample(HopArgs a) {
    pdl_start();
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ __align__(16) uint32_t s_key[kBlockPool];
    __shared__ uint32_t s_pos[kBlockPool];
    __shared__ uint32_t s_sel[kWarpSel * (kNT / 32)];
    __shared__ int s_n[kNT / 8];
    __shared__ int s_item;
    load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);
    uint32_t k0 = a.key0, k1 = a.key1;
    if (a.d_seed) {
        const uint64_t sd = *a.d_seed;
        k0 = (uint32_t)(sd & 0xFFFFFFFFull);
        k1 = (uint32_t)(sd >> 32);
    }
    // the counters start at all-ones, so a count is the word + 1
    // bin sizes (row counts fit in 32 bits); b7, b76 and bblk are prefixes of
    // the block bins in work order, w4, w43 and u2 those of the warp bins
    const int32_t n0 = (int32_t)(a.ctr[2] + 1u), n1 = (int32_t)(a.ctr[3] + 1u);
    const int32_t b7 = (int32_t)(a.ctr[9] + 1u), b76 = b7 + (int32_t)(a.ctr[8] + 1u), bblk = b76 + (int32_t)(a.ctr[7] + 1u);
    const int32_t w4 = (int32_t)(a.ctr[6] + 1u), w43 = w4 + (int32_t)(a.ctr[5] + 1u), u2 = w43 + (int32_t)(a.ctr[4] + 1u);
    const Pool bpool{s_key, s_pos, s_sel, &s_n[0], kBlockPool};
    for (;;) {
        if (threadIdx.x == 0) s_item = (int)(atomicAdd(a.ctr + 10, 1u) + 1u);
        __syncthreads();
        const int64_t i = s_item;
        __syncthreads();
        if (i >= bblk) break;
        const BinRec* slot = i < b7 ? bin_slot(a, 7, i) : (i < b76 ? bin_slot(a, 6, i - b7) : bin_slot(a, 5, i - b76));
        sample_big_row(a, load_rec(slot), pre, k0, k1, bpool);
    }
    // units: the warp rows of bins 4, 3, 2 (u2 of them), then four bin 1 rows
    // a unit, then sixteen full rows a unit
    const int32_t u1 = (n1 + 3) / 4, u0 = (n0 + 15) / 16;
    const int32_t units = u2 + u1 + u0;
    auto warp_slot = [&](int32_t uu) {
        return uu < w4 ? bin_slot(a, 4, uu) : (uu < w43 ? bin_slot(a, 3, uu - w4) : bin_slot(a, 2, uu - w43));
    };
    const unsigned lane = lane_id();
    const int wib = threadIdx.x >> 5;
    const int g = (int)(lane >> 3), gl = (int)(lane & 7);
    const unsigned gmask = 0xFFu << (8 * g);
    const Pool wpool{s_key + wib * kWarpPool, s_pos + wib * kWarpPool, s_sel + wib * kWarpSel, &s_n[4 * wib], kWarpPool};
    const Pool gpool{s_key + wib * kWarpPool + g * kGroupPool, s_pos + wib * kWarpPool + g * kGroupPool,
                     s_sel + wib * kWarpSel + g * kGroupSel, &s_n[4 * wib + g], kGroupPool};
    // Units come from kUnitQueues counters, each in its own 128-byte line:
    // queue q hands out units q, q + kUnitQueues, ... to the warps w with
    // w mod kUnitQueues = q, so no single counter takes every warp's atomics.
    // The next unit is reserved while this one runs only when units are
    // plentiful (more than two per warp left); near the end of a queue a warp
    // takes its next unit once it is done, so that no unit waits behind a busy
    // warp while others are idle.
    auto unit_rec = [&](int32_t uu, BinRec& rc) {
        rc.v = -1;
        if (uu < u2) {
            rc = load_rec(warp_slot(uu));
        } else if (uu < u2 + u1) {
            const int32_t i = (uu - u2) * 4 + g;
            if (i < n1) rc = load_rec(bin_slot(a, 1, i));
        }
    };
    const int32_t n_warps = (int32_t)(gridDim.x * (kNT / 32));
    // this warp's queue and its next unit (lane 0 only)
    auto take = [&]() -> uint32_t {
        const uint32_t q = (blockIdx.x * (kNT / 32) + (threadIdx.x >> 5)) % kUnitQueues;
        return (atomicAdd(a.ctr + 32 + 32 * q, 1u) + 1u) * kUnitQueues + q;
    };
    uint32_t nxt = 0;
    if (lane == 0) nxt = take();
    int32_t u = (int32_t)__shfl_sync(0xffffffffu, nxt, 0);
    while (u < units) {
        const bool ahead = u + 2 * n_warps < units;
        if (ahead && lane == 0) nxt = take();
        BinRec rec;
        unit_rec(u, rec);
        if (u < u2) {
            sample_row<32>(a, rec, pre, k0, k1, wpool, 0xffffffffu, (int)lane);
        } else if (u < u2 + u1) {
            const int32_t i = (u - u2) * 4 + g;
            sample_rows_x4(a, rec, i < n1, pre, k0, k1, gpool, gmask, gl);
        } else {
            for (int t = 0; t < 4; ++t) {
                const int32_t i = (u - u2 - u1) * 16 + 4 * t + g;
                if (i < n0) sample_row<8>(a, load_rec(bin_slot(a, 0, i)), pre, k0, k1, gpool, gmask, gl);
            }
        }
        __syncwarp();
        if (!ahead && lane == 0) nxt = take();
        u = (int32_t)__shfl_sync(0xffffffffu, nxt, 0);
    }
}

// --------------------------------------------------------------------- copy
// Super-batch: a row whose node was sampled by an earlier row (its owner)
// copies the owner's neighbours into its own edge range and inserts them into
// its own mini-batch's table at its own positions.
__global__ void __launch_bounds__(kNT) k_copy(HopArgs a) {
    pdl_start();
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h - 1, pre);
    const int64_t T = pre[a.K];
    const int64_t nwarps = (int64_t)gridDim.x * (kNT / 32);
    const unsigned lane = lane_id();
    for (int64_t r = (blockIdx.x * (int64_t)kNT + threadIdx.x) / 32; r < T; r += nwarps) {
        const int32_t s = a.rslot[r];
        if (s < 0) continue;
        const int32_t owner = (int32_t)a.utab[s].y;
        if (owner == (int32_t)r || owner < 0 || (int64_t)owner >= T) continue;
        const int64_t o = a.bindptr[r], c = a.bindptr[r + 1] - o, so = a.bindptr[owner];
        uint32_t* tab = a.pos_of + (int64_t)find_sub(pre, a.K, r) * a.n_nodes;
        for (int64_t t = lane; t < c; t += 32) emit_edge(a, tab, o + t, a.enbr[so + t]);
    }
}

// ----------------------------------------------------------------- relabel
// First-occurrence flags and new local IDs; one scan chain per mini-batch.
__global__ void __launch_bounds__(kNT) k_relabel(HopArgs a) {
    pdl_start();
    __shared__ int32_t ep[SG_MAX_SUB + 1];
    __shared__ int32_t tpre[SG_MAX_SUB + 1];
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ int32_t s_tile, s_excl;
    const int K = a.K;
    for (int k = threadIdx.x; k <= K; k += kNT) ep[k] = a.epre[k];
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int k = 0; k <= K; ++k) {
            tpre[k] = acc;
            if (k < K) acc += (ep[k + 1] - ep[k] + kTile - 1) / kTile;
        }
        tpre[K] = acc;
    }
    __syncthreads();
    if (blockIdx.x == 0) {  // mini-batches without edges keep V_{h-1}
        for (int k = threadIdx.x; k < K; k += kNT) {
            a.counts[a.L.sub_e(k, a.h)] = ep[k + 1] - ep[k];
            if (ep[k + 1] == ep[k]) a.counts[a.L.sub_n(k, a.h)] = a.counts[a.L.sub_n(k, a.h - 1)];
        }
    }
    const int n_tiles = tpre[K];
    if ((int)blockIdx.x >= n_tiles) return;  // see k_rows
    for (int iter = 0;; ++iter) {
        if (iter > 0 && (int)gridDim.x >= n_tiles) break;
        if (threadIdx.x == 0) s_tile = (int32_t)(atomicAdd(a.ctr + 1, 1u) + 1u);
        __syncthreads();
        const int t = s_tile;
        if (t >= n_tiles) break;
        const int k = find_sub(tpre, K, t);
        const int32_t n_prev = a.counts[a.L.sub_n(k, a.h - 1)];  // needed after the scan; loaded now
        const int64_t e_end = ep[k + 1];
        const int64_t e0 = ep[k] + (int64_t)(t - tpre[k]) * kTile + (int64_t)threadIdx.x * 4;
        bool fl[4];
        int32_t mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t e = e0 + q;
            fl[q] = false;
            if (e < e_end) {
                if (a.pos_of) {
                    fl[q] = a.pos_of[(int64_t)k * a.n_nodes + a.enbr[e]] == (uint32_t)(a.pos_base + e);
                } else {
                    const int32_t s = a.eslot[e];
                    fl[q] = s >= 0 && a.table[s].y == (uint32_t)(a.pos_base + e);
                }
            }
            mine += fl[q];
        }
        int32_t tile_total;
        const int32_t ex = block_excl_scan<kNT>(mine, red, tile_total);
        if (threadIdx.x < 32) {
            bool late = false;
            const int32_t x = chain_lookback(a.edge_status, t, tpre[k], tile_total, &late);
            if (threadIdx.x == 0) s_excl = x;
            if (late && threadIdx.x == 0) dev_err(ERR_TIMEOUT);
        }
        __syncthreads();
        int32_t rank = s_excl + ex;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (fl[q]) {
                const int64_t e = e0 + q;
                const int64_t lid = (int64_t)n_prev + rank;
                if (lid >= a.capU) {
                    dev_err(ERR_CAPACITY);
                } else {
                    const int32_t u = a.enbr[e];
                    if (a.pos_of) a.pos_of[(int64_t)k * a.n_nodes + u] = (uint32_t)lid;
                    else a.table[a.eslot[e]].y = (uint32_t)lid;
                    a.ustr[(int64_t)k * a.capU + lid] = u;
                }
                ++rank;
            }
        }
        if (t == tpre[k + 1] - 1 && threadIdx.x == 0) a.counts[a.L.sub_n(k, a.h)] = n_prev + s_excl + tile_total;
        __syncthreads();
    }
}

// ------------------------------------------------------------------ finish
// Maps the last hop's edges, writes the last total and, for a super-batch,
// lays the mini-batches' V_H back to back.
__global__ void __launch_bounds__(kNT) k_finish(HopArgs a, int32_t* unique_out) {
    pdl_start();
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    __shared__ int32_t ep[SG_MAX_SUB + 1];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h, pre);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.counts[a.L.tot_n(a.h)] = pre[a.K];
    map_prev_edges(a, blockIdx.x, gridDim.x, ep, pre);
    if (unique_out) {
        const int64_t n = pre[a.K];
        for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < n; i += (int64_t)gridDim.x * kNT) {
            const int k = find_sub(pre, a.K, i);
            unique_out[i] = a.ustr[(int64_t)k * a.capU + (i - pre[k])];
        }
    }
}

// ----------------------------------------------------------------- cleanup
// Leaves the workspace ready for the next call: every node of V_H gets its
// direct-map entry back to empty, and the scan states and counters of all
// hops are reset (all-ones).
__global__ void __launch_bounds__(kNT) k_cleanup(HopArgs a, uint32_t* reset, int64_t reset_words) {
    pdl_start();
    __shared__ int32_t pre[SG_MAX_SUB + 1];
    load_prefix_sub_n(a.counts, a.L, a.K, a.h, pre);
    const int64_t n = pre[a.K];
    const int64_t stride = (int64_t)gridDim.x * kNT;
    for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < n; i += stride) {
        const int k = a.K == 1 ? 0 : find_sub(pre, a.K, i);
        const int32_t u = a.ustr[(int64_t)k * a.capU + (i - pre[k])];
        if (u >= 0 && (int64_t)u < a.n_nodes) a.pos_of[(int64_t)k * a.n_nodes + u] = kEmpty;
    }
    for (int64_t i = blockIdx.x * (int64_t)kNT + threadIdx.x; i < reset_words; i += stride) reset[i] = kEmpty;
}

// ------------------------------------------------------ standalone relabel
__global__ void k_relabel_insert(const int32_t* __restrict__ ids, int64_t n_ids, uint2* table, int logT, int32_t pos_base,
                                 int32_t* enbr, int32_t* eslot, int32_t* epre) {
    pdl_start();
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
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int pow2_log(int64_t atleast) {
    int l = 6;
    while (((int64_t)1 << l) < atleast) ++l;
    return l;
}

struct Plan {
    int K, H;
    int32_t bptr[SG_MAX_SUB + 1];
    int32_t fan[SG_MAX_HOPS];
    int64_t nb_tot[SG_MAX_HOPS + 1], eb_tot[SG_MAX_HOPS];
    int64_t capU;      // per mini-batch bound on |V_H^k|
    int logU[SG_MAX_HOPS];
    int64_t nb_max, eb_max;
    // workspace: [o_pos, o_rest) persists between calls (all-ones when idle:
    // set by sg_sampler_workspace_init, restored by every run's cleanup);
    // [o_utab[0], o_scratch) is set to all-ones per call (super-batch only);
    // the rest is scratch
    size_t o_pos, o_zero, o_rstat[SG_MAX_HOPS], o_estat[SG_MAX_HOPS], o_ctr, o_rest;
    size_t o_utab[SG_MAX_HOPS], o_scratch;
    size_t o_ustr, o_rslot, o_bins, o_enbr[2], o_epre, total;
};

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
    if (maxdeg > 2147483647LL) return fail(SG_ERR_UNSUPPORTED, "sampler: rows longer than 2^31 - 1 entries");
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
    // map values hold local IDs (< capU) and edge positions capU + e
    if (p->capU + p->eb_max >= 2147483647LL || p->nb_tot[n_hops] >= 2147483647LL)
        return fail(SG_ERR_UNSUPPORTED, "sampler: a mini-batch this large needs 64-bit local IDs");
    size_t o = 0;
    p->o_pos = o;
    o = align256(o + (size_t)K * (size_t)N * 4);
    p->o_zero = o;
    for (int h = 0; h < n_hops; ++h) {
        p->o_rstat[h] = o;
        o = align256(o + (size_t)(p->nb_tot[h] / kTile + 2) * 8);
        p->o_estat[h] = o;
        o = align256(o + (size_t)(p->eb_tot[h] / kTile + K + 2) * 8);
    }
    p->o_ctr = o;
    o = align256(o + (size_t)n_hops * kCtrWords * 4);
    p->o_rest = o;
    for (int h = 0; h < n_hops; ++h) {
        p->logU[h] = K > 1 ? pow2_log(2 * p->nb_tot[h]) : 0;
        p->o_utab[h] = o;
        if (K > 1) o = align256(o + ((size_t)1 << p->logU[h]) * sizeof(uint2));
    }
    p->o_scratch = o;
    p->o_ustr = o;
    o = align256(o + (K > 1 ? (size_t)K * (size_t)p->capU * 4 : 0));
    p->o_rslot = o;
    o = align256(o + (K > 1 ? (size_t)p->nb_max * 4 : 0));
    p->o_bins = o;
    o = align256(o + (size_t)(kBins / 2) * (size_t)p->nb_max * sizeof(BinRec));
    for (int i = 0; i < 2; ++i) {  // edge arrays alternate between hops (k_rows maps the previous hop's)
        p->o_enbr[i] = o;
        o = align256(o + (size_t)p->eb_max * 4);
    }
    p->o_epre = o;
    o = align256(o + (size_t)(n_hops + 1) * (SG_MAX_SUB + 1) * 4);
    p->total = o;
    return SG_OK;
}

uint32_t lambda_for(int f) {
    // expected candidates per random row: f + 2 sqrt(f) + 4 keeps a retry
    // (fewer than f pass, about 1% of rows) cheap and the candidate set small
    double lam = f + 2.0 * __builtin_sqrt((double)f) + 4.0;
    return (uint32_t)lam;
}

// Blocks of k_sample that fit on the GPU at once (its grid hands out work by
// counters, so more blocks would only wait).
int64_t resident_sample_blocks(int sms) {
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_sample, kNT, 0) != cudaSuccess || n < 1) n = 1;
        per_sm = n;
    }
    return (int64_t)per_sm * sms;
}

int64_t clamp_blocks(int64_t want, int64_t cap) {
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    return want;
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

extern "C" sg_status sg_sampler_workspace_init(const sg_graph* g, int32_t n_seeds, const int32_t* h_batch_ptr,
                                               int32_t n_sub, const int32_t* h_fanouts, int32_t n_hops,
                                               void* d_workspace, size_t workspace_bytes, sg_stream_t stream) {
    Plan p;
    sg_status st = make_plan(g, n_seeds, h_batch_ptr, n_sub, h_fanouts, n_hops, &p);
    if (st != SG_OK) return st;
    if (!d_workspace || workspace_bytes < p.total)
        return fail(SG_ERR_INVALID_ARG, "sg_sampler_workspace_init: workspace needs %zu bytes", p.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_sampler_workspace_init: workspace must be 256-byte aligned");
    SG_CUDA(cudaMemsetAsync((char*)d_workspace + p.o_pos, 0xFF, p.o_rest - p.o_pos, (cudaStream_t)stream));
    return SG_OK;
}

extern "C" sg_status sg_sampler_run(const sg_graph* g, const int32_t* d_seeds, int32_t n_seeds, const int32_t* h_batch_ptr,
                                    int32_t n_sub, const int32_t* h_fanouts, int32_t n_hops, uint64_t seed,
                                    const uint64_t* d_seed, void* d_workspace, size_t workspace_bytes,
                                    const sg_blocks* out, const sg_event_t* h_hop_events, sg_stream_t stream) {
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
    const int sms = num_sms();
    CountsLayout L{H};
    HopArgs a;
    memset(&a, 0, sizeof(a));
    a.indptr = g->indptr;
    a.indices = g->indices;
    a.n_nodes = g->n_nodes;
    a.K = K;
    a.capU = p.capU;
    a.key0 = (uint32_t)(seed & 0xFFFFFFFFull);
    a.key1 = (uint32_t)(seed >> 32);
    a.d_seed = d_seed;
    a.pos_base = (int32_t)p.capU;
    a.L = L;
    a.counts = out->counts;
    a.ustr = K > 1 ? (int32_t*)(ws + p.o_ustr) : out->unique;
    a.pos_of = (uint32_t*)(ws + p.o_pos);
    a.brec = (BinRec*)(ws + p.o_bins);
    a.bin_cap = p.nb_max;
    a.rslot = K > 1 ? (int32_t*)(ws + p.o_rslot) : nullptr;
    int32_t* epre_all = (int32_t*)(ws + p.o_epre);

    // the direct map, scan states and counters arrive all-ones (left so by
    // sg_sampler_workspace_init or the previous run); the owner tables of a
    // super-batch are cleared here
    if (K > 1) SG_CUDA(cudaMemsetAsync(ws + p.o_utab[0], 0xFF, p.o_scratch - p.o_utab[0], s));
    SubPtr bp;
    for (int k = 0; k <= K; ++k) bp.v[k] = p.bptr[k];
    const int64_t cap_blocks = (int64_t)sms * 8;
    const int64_t sample_blocks = resident_sample_blocks(sms);
    for (int h = 1; h <= H; ++h) {
        const int cur = (h - 1) & 1, prv = h & 1;
        a.h = h;
        a.fanout = p.fan[h - 1];
        a.lambda_num = lambda_for(a.fanout);
        a.bindptr = out->indptr[h - 1];
        a.epre = epre_all + (size_t)h * (SG_MAX_SUB + 1);
        a.enbr = (int32_t*)(ws + p.o_enbr[cur]);
        a.ctr = (uint32_t*)(ws + p.o_ctr) + (size_t)(h - 1) * kCtrWords;
        a.row_status = (unsigned long long*)(ws + p.o_rstat[h - 1]);
        a.edge_status = (unsigned long long*)(ws + p.o_estat[h - 1]);
        a.utab = K > 1 ? (uint2*)(ws + p.o_utab[h - 1]) : nullptr;
        a.logU = p.logU[h - 1];
        // the previous hop's edges are mapped inside this hop's row pass
        a.prev_bidx = h > 1 ? out->idx[h - 2] : nullptr;
        a.prev_epre = h > 1 ? epre_all + (size_t)(h - 1) * (SG_MAX_SUB + 1) : nullptr;
        a.prev_enbr = h > 1 ? (const int32_t*)(ws + p.o_enbr[prv]) : nullptr;
        const int64_t nb = p.nb_tot[h - 1], eb = p.eb_tot[h - 1];
        a.map_blocks = h > 1 ? (int)clamp_blocks(cdiv(p.eb_tot[h - 2], kNT * 8), cap_blocks) : 0;
        const int64_t row_blocks = clamp_blocks(cdiv(nb, kTile), cap_blocks);
        const int seed_mode = h == 1;
        if (g->offset_bits == 32)
            SG_CUDA(launch_pdl(k_rows<int32_t>, dim3((unsigned)(a.map_blocks + row_blocks)), dim3(kNT), 0, s, a,
                               seed_mode, d_seeds, bp));
        else
            SG_CUDA(launch_pdl(k_rows<int64_t>, dim3((unsigned)(a.map_blocks + row_blocks)), dim3(kNT), 0, s, a,
                               seed_mode, d_seeds, bp));
        SG_CUDA(launch_pdl(k_sample, dim3((unsigned)clamp_blocks(cdiv(nb, kNT / 32), sample_blocks)), dim3(kNT), 0, s, a));
        if (K > 1) {
            SG_CUDA(launch_pdl(k_copy, dim3((unsigned)clamp_blocks(cdiv(nb, kNT / 32), cap_blocks)), dim3(kNT), 0, s, a));
        }
        SG_CUDA(launch_pdl(k_relabel, dim3((unsigned)clamp_blocks(cdiv(eb, kTile) + K, cap_blocks)), dim3(kNT), 0, s, a));
        // one mini-batch: V_h is final in `unique` (and its size in sub_n(0, h))
        if (K == 1 && h_hop_events && h_hop_events[h - 1])
            SG_CUDA(cudaEventRecord((cudaEvent_t)h_hop_events[h - 1], s));
    }
    // the last hop's edges, the last total and the super-batch layout
    a.prev_bidx = out->idx[H - 1];
    a.prev_epre = epre_all + (size_t)H * (SG_MAX_SUB + 1);
    a.prev_enbr = (const int32_t*)(ws + p.o_enbr[(H - 1) & 1]);
    a.h = H;
    const int64_t fin = p.eb_tot[H - 1] > p.nb_tot[H] ? p.eb_tot[H - 1] : p.nb_tot[H];
    SG_CUDA(launch_pdl(k_finish, dim3((unsigned)clamp_blocks(cdiv(fin, kNT * 4), cap_blocks)), dim3(kNT), 0, s, a,
                       K > 1 ? out->unique : nullptr));
    const int64_t reset_words = (int64_t)(p.o_rest - p.o_zero) / 4;
    const int64_t clean = p.nb_tot[H] > reset_words ? p.nb_tot[H] : reset_words;
    SG_CUDA(launch_pdl(k_cleanup, dim3((unsigned)clamp_blocks(cdiv(clean, kNT * 4), cap_blocks)), dim3(kNT), 0, s, a,
                       (uint32_t*)(ws + p.o_zero), reset_words));
    if (K > 1 && h_hop_events)  // a super-batch's `unique` is laid out by k_finish
        for (int h = 1; h <= H; ++h)
            if (h_hop_events[h - 1]) SG_CUDA(cudaEventRecord((cudaEvent_t)h_hop_events[h - 1], s));
    return SG_OK;
}

// ------------------------------------------------------ standalone relabel
namespace {
struct RelabelPlan {
    int logT;
    int64_t capU;
    size_t o_table, o_zero, o_estat, o_ctr, o_rest, o_enbr, o_eslot, o_epre, o_counts, total;
};

bool relabel_plan(int64_t n_prefix, int64_t n_ids, RelabelPlan* p) {
    if (n_prefix < 0 || n_ids < 0 || n_prefix + 2 * n_ids >= 2147483647LL) return false;
    p->capU = n_prefix + n_ids + 1;
    p->logT = pow2_log(2 * p->capU);
    size_t o = 0;
    p->o_table = o;
    o = align256(o + ((size_t)1 << p->logT) * sizeof(uint2));
    p->o_zero = o;
    p->o_estat = o;
    o = align256(o + (size_t)(n_ids / kTile + 3) * 8);
    p->o_ctr = o;
    o = align256(o + 8 * 4);
    p->o_rest = o;
    p->o_enbr = o;
    o = align256(o + (size_t)(n_ids + 1) * 4);
    p->o_eslot = o;
    o = align256(o + (size_t)(n_ids + 1) * 4);
    p->o_epre = o;
    o = align256(o + (size_t)(SG_MAX_SUB + 1) * 4);
    p->o_counts = o;
    o = align256(o + 16 * 4);
    p->total = o;
    return true;
}

// Runs the standalone relabel with its scratch at ws (layout of relabel_plan).
sg_status relabel_launch(const RelabelPlan& p, char* ws, const int32_t* d_ids, int64_t n_ids, const int32_t* d_prefix,
                         int64_t n_prefix, int32_t* d_unique, int32_t* d_local, int32_t* d_n_unique, cudaStream_t s) {
    CountsLayout L{1};
    HopArgs a;
    memset(&a, 0, sizeof(a));
    a.n_nodes = 2147483647LL;
    a.K = 1;
    a.logT = p.logT;
    a.capU = p.capU;
    a.pos_base = (int32_t)p.capU;
    a.L = L;
    a.counts = (int32_t*)(ws + p.o_counts);
    a.ustr = d_unique;
    a.table = (uint2*)(ws + p.o_table);
    a.enbr = (int32_t*)(ws + p.o_enbr);
    a.eslot = (int32_t*)(ws + p.o_eslot);
    a.epre = (int32_t*)(ws + p.o_epre);
    a.ctr = (uint32_t*)(ws + p.o_ctr);
    a.edge_status = (unsigned long long*)(ws + p.o_estat);
    a.h = 1;
    a.fanout = 1;
    // the scratch may hold a previous call's contents: the table, the scan
    // state and the counter are reset (all-ones bytes) before use; everything
    // else is written before it is read
    SG_CUDA(cudaMemsetAsync(ws + p.o_table, 0xFF, p.o_rest - p.o_table, s));
    SubPtr bp;
    bp.v[0] = 0;
    bp.v[1] = (int32_t)n_prefix;
    const int sms = num_sms();
    SG_CUDA(launch_pdl(k_seed_init, dim3(n_prefix > 0 ? (int)cdiv(n_prefix, 256) : 1), dim3(256), 0, s, d_prefix,
                       (int32_t)n_prefix, bp, 1, a.n_nodes, a.table, p.logT, a.ustr, p.capU, a.counts, L));
    const int64_t ib = clamp_blocks(cdiv(n_ids, 256), (int64_t)sms * 8);
    SG_CUDA(launch_pdl(k_relabel_insert, dim3((unsigned)ib), dim3(256), 0, s, d_ids, n_ids, a.table, p.logT, a.pos_base,
                       a.enbr, a.eslot, a.epre));
    SG_CUDA(launch_pdl(k_relabel, dim3((unsigned)clamp_blocks(cdiv(n_ids, kTile) + 1, (int64_t)sms * 8)), dim3(kNT), 0, s, a));
    a.prev_bidx = d_local;
    a.prev_epre = a.epre;
    a.prev_eslot = a.eslot;
    SG_CUDA(launch_pdl(k_finish, dim3((unsigned)ib), dim3(kNT), 0, s, a, nullptr));
    SG_CUDA(cudaMemcpyAsync(d_n_unique, a.counts + L.tot_n(1), sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    return SG_OK;
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
    return relabel_launch(p, (char*)d_workspace, d_ids, n_ids, d_prefix, n_prefix, d_unique, d_local, d_n_unique,
                          (cudaStream_t)stream);
}

// ------------------------------------------- relabel without allocation
// The scratch of sg_relabel_noalloc: a static device array, so callers that
// cannot allocate device memory still get a relabel.  Host code must not use
// the array's name as an address; the device address is looked up once per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_relabel_scratch[SG_RELABEL_NOALLOC_SCRATCH_BYTES];

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
    return relabel_launch(p, (char*)scratch, d_ids, n_ids, d_prefix, n_prefix, d_unique, d_local, d_n_unique,
                          (cudaStream_t)stream);
}

/*
 * CPU ORACLE for the mini-batch pipeline of sampling-based GNN training.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this file.  It shares no code,
 * header, table or constant with the CUDA library; every definition below is
 * written out again here from its source.
 *
 * Plain, slow and direct: every step follows its definition in order,
 * floating-point sums are taken in double precision, and the only parallelism
 * is OpenMP over independent rows (each row's result does not depend on the
 * others, so the output is the same for any thread count).
 *
 * What is computed (GARDEN page, "Efficient GPU-Accelerated Billion-Scale GNN
 * Training via Caching-Sampling-Batching Co-Design"):
 *   sampling   - Section II-B and Fig. 1 (layer-wise blocks, V_l = V_{l-1} u
 *                N_l(V_{l-1})), Section IV-C (fixed-fanout uniform sampling;
 *                a node whose degree is at most the fanout keeps all of its
 *                neighbours; the sampling distribution is not altered)
 *   relabel    - Section IV-D (hash-table dedup of sampled node IDs); the local
 *                numbering is first occurrence, seeds first
 *   gather     - Section II-B, Fig. 2 (Nfeat-Selecting: cached rows from GPU
 *                memory, misses from host memory; residency does not change
 *                the rows)
 *   aggregate  - Section II-A, Eq. (1) with AGGREGATE = mean; the backward
 *                pass is the transpose of the same linear map
 * Readings where the pages leave a step open:
 *   - the uniform sample of k out of deg neighbour positions is the k
 *     positions with the smallest keys (r, j), r = one 32-bit word of
 *     Philox4x32-10 (Salmon et al., SC'11) with counter (j/4, v, hop, 0) and
 *     key (seed low, seed high), word j mod 4; j is the position in the CSR
 *     row and v the global node ID; ties in r go to the lower j
 *   - the sample of a row is listed in ascending position order
 *   - every node of V_{h-1} (seeds and earlier hops' nodes included) is
 *     sampled at hop h, with that hop's number in the hash
 *   - new nodes of a hop are numbered in order of first occurrence in the
 *     hop's edge list, which is ordered by (dst local ID, position)
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ Philox */
/* Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11, Section 4.2).  One round maps the
 * counter (c0,c1,c2,c3) under round key (k0,k1) to
 *   (hi(B*c2) ^ c1 ^ k0,  lo(B*c2),  hi(A*c0) ^ c3 ^ k1,  lo(A*c0))
 * with multipliers A = 0xD2511F53, B = 0xCD9E8D57; the key is bumped by the
 * Weyl constants (0x9E3779B9, 0xBB67AE85) between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t pa = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t pb = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)pb;
        uint32_t n2 = (uint32_t)(pa >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)pa;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* sampling key r(seed, hop, v, j) */
uint32_t orc_sample_key(uint64_t seed, int32_t hop, int32_t v, int64_t j) {
    uint32_t ctr[4] = {(uint32_t)(j / 4), (uint32_t)v, (uint32_t)hop, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    return w[j % 4];
}

/* ---------------------------------------------------------------- sampling */
typedef struct { uint32_t r; int64_t j; } orc_keyed;

static int cmp_keyed(const void* a, const void* b) {
    const orc_keyed* x = (const orc_keyed*)a;
    const orc_keyed* y = (const orc_keyed*)b;
    if (x->r != y->r) return x->r < y->r ? -1 : 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/* Sample of node v at hop `hop` with fanout f: writes the chosen row
 * positions in ascending order to pos_out (room for min(deg, f)) and returns
 * their number, or -1 on allocation failure. */
int64_t orc_sample_positions(const int64_t* indptr, int32_t v, int32_t fanout, int32_t hop,
                             uint64_t seed, int64_t* pos_out) {
    int64_t deg = indptr[v + 1] - indptr[v];
    if (deg <= fanout) {                        /* full node: every neighbour */
        for (int64_t j = 0; j < deg; j++) pos_out[j] = j;
        return deg;
    }
    orc_keyed* keys = (orc_keyed*)malloc((size_t)deg * sizeof(orc_keyed));
    if (!keys) return -1;
    for (int64_t j = 0; j < deg; j++) {        /* random node: key every position */
        keys[j].r = orc_sample_key(seed, hop, v, j);
        keys[j].j = j;
    }
    qsort(keys, (size_t)deg, sizeof(orc_keyed), cmp_keyed);
    for (int64_t t = 0; t < fanout; t++) pos_out[t] = keys[t].j;  /* the f smallest */
    free(keys);
    qsort(pos_out, (size_t)fanout, sizeof(int64_t), cmp_i64);      /* listed by position */
    return fanout;
}

/* Multi-hop sampling plus relabel for one mini-batch.
 *   indptr[n_nodes+1] (int64), indices[m]      CSR graph
 *   seeds[n_seeds]                             distinct global IDs (V_0)
 *   fanouts[n_hops]                            fanouts[h-1] is the fanout of hop h
 * Outputs (caller-allocated, capacities given):
 *   unique[cap_unique]     V_H as global IDs; V_h is its prefix of length hop_off[h]
 *   hop_off[n_hops+1]      |V_0|, |V_1|, ..., |V_H|
 *   edge_off[n_hops+1]     hop h's edges are [edge_off[h-1], edge_off[h]) of the edge arrays
 *   indptr_off[n_hops+1]   hop h's block row pointer is blk_indptr[indptr_off[h-1] ...]
 *   blk_indptr             per hop: |V_{h-1}|+1 entries, local to the hop's edges
 *   blk_idx[cap_edges]     local src ID of each edge (index into V_h)
 *   nbr[cap_edges]         global ID of each sampled neighbour
 *   pos[cap_edges]         its position in the dst's CSR row
 * Returns 0, or -1 (bad input or allocation), -2 (a capacity is too small). */
int orc_sampler_run(const int64_t* indptr, const int32_t* indices, int64_t n_nodes,
                    const int32_t* seeds, int32_t n_seeds, const int32_t* fanouts, int32_t n_hops,
                    uint64_t seed,
                    int32_t* unique, int64_t cap_unique, int64_t* hop_off,
                    int64_t* edge_off, int64_t* indptr_off, int64_t* blk_indptr, int64_t cap_indptr,
                    int32_t* blk_idx, int32_t* nbr, int64_t* pos, int64_t cap_edges) {
    if (n_seeds < 0 || n_hops < 0 || n_seeds > cap_unique) return -2;
    int32_t* lid_of = (int32_t*)malloc((size_t)n_nodes * sizeof(int32_t));
    if (!lid_of) return -1;
    for (int64_t v = 0; v < n_nodes; v++) lid_of[v] = -1;
    int64_t n_cur = 0;
    for (int32_t i = 0; i < n_seeds; i++) {                 /* seeds take 0..B-1 */
        int32_t s = seeds[i];
        if (s < 0 || s >= n_nodes || lid_of[s] >= 0) { free(lid_of); return -1; }
        lid_of[s] = (int32_t)n_cur;
        unique[n_cur++] = s;
    }
    hop_off[0] = n_cur;
    edge_off[0] = 0;
    indptr_off[0] = 0;
    int rc = 0;
    for (int32_t h = 1; h <= n_hops && rc == 0; h++) {
        int32_t f = fanouts[h - 1];
        int64_t n_dst = n_cur;                              /* V_{h-1} = unique[0, n_dst) */
        int64_t e0 = edge_off[h - 1];
        int64_t* bp = blk_indptr + indptr_off[h - 1];
        if (indptr_off[h - 1] + n_dst + 1 > cap_indptr) { rc = -2; break; }
        /* sizes: c_v = min(deg, f) */
        bp[0] = 0;
        for (int64_t d = 0; d < n_dst; d++) {
            int32_t v = unique[d];
            int64_t deg = indptr[v + 1] - indptr[v];
            bp[d + 1] = bp[d] + (deg < f ? deg : f);
        }
        int64_t n_e = bp[n_dst];
        if (e0 + n_e > cap_edges) { rc = -2; break; }
        /* the sample of every dst (independent rows) */
        int failed = 0;
        #pragma omp parallel for schedule(dynamic, 64) reduction(|:failed)
        for (int64_t d = 0; d < n_dst; d++) {
            int32_t v = unique[d];
            int64_t* p = pos + e0 + bp[d];
            int64_t c = orc_sample_positions(indptr, v, f, h, seed, p);
            if (c < 0) { failed = 1; continue; }
            for (int64_t t = 0; t < c; t++) nbr[e0 + bp[d] + t] = indices[indptr[v] + p[t]];
        }
        if (failed) { rc = -1; break; }
        /* relabel: new nodes in order of first occurrence in the edge list */
        for (int64_t e = 0; e < n_e; e++) {
            int32_t u = nbr[e0 + e];
            if (lid_of[u] < 0) {
                if (n_cur >= cap_unique) { rc = -2; break; }
                lid_of[u] = (int32_t)n_cur;
                unique[n_cur++] = u;
            }
            blk_idx[e0 + e] = lid_of[u];
        }
        hop_off[h] = n_cur;
        edge_off[h] = e0 + n_e;
        indptr_off[h] = indptr_off[h - 1] + n_dst + 1;
    }
    free(lid_of);
    return rc;
}

/* Standalone relabel: IDs already numbered (prefix, local IDs 0..n_prefix-1)
 * keep their number; the other IDs of `ids` are numbered n_prefix, n_prefix+1,
 * ... in order of first occurrence.  unique[] receives the prefix followed by
 * the new IDs (room for n_prefix + n_ids), local[i] the number of ids[i].
 * Returns the number of unique IDs, or -1 on bad input. */
int64_t orc_relabel(const int32_t* ids, int64_t n_ids, const int32_t* prefix, int64_t n_prefix,
                    int32_t* unique, int32_t* local) {
    int64_t max_id = -1;
    for (int64_t i = 0; i < n_ids; i++) { if (ids[i] < 0) return -1; if (ids[i] > max_id) max_id = ids[i]; }
    for (int64_t i = 0; i < n_prefix; i++) { if (prefix[i] < 0) return -1; if (prefix[i] > max_id) max_id = prefix[i]; }
    int32_t* lid_of = (int32_t*)malloc((size_t)(max_id + 1 > 0 ? max_id + 1 : 1) * sizeof(int32_t));
    if (!lid_of) return -1;
    for (int64_t v = 0; v <= max_id; v++) lid_of[v] = -1;
    int64_t n = 0;
    for (int64_t i = 0; i < n_prefix; i++) {
        if (lid_of[prefix[i]] >= 0) { free(lid_of); return -1; }   /* prefix must be distinct */
        lid_of[prefix[i]] = (int32_t)n;
        unique[n++] = prefix[i];
    }
    for (int64_t i = 0; i < n_ids; i++) {
        int32_t u = ids[i];
        if (lid_of[u] < 0) { lid_of[u] = (int32_t)n; unique[n++] = u; }
        local[i] = lid_of[u];
    }
    free(lid_of);
    return n;
}

/* ------------------------------------------------------------------ gather */
/* out row i = feature row ids[i], byte for byte, whatever is cached. */
void orc_gather(const void* feat, int64_t row_bytes, const int32_t* ids, int64_t n, void* out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        memcpy((char*)out + i * row_bytes, (const char*)feat + (int64_t)ids[i] * row_bytes, (size_t)row_bytes);
}

/* --------------------------------------------------------------- aggregate */
static double load_elem(const void* h, int dtype, int64_t k) {
    if (dtype == 0) return (double)((const float*)h)[k];
    uint32_t b = (uint32_t)((const uint16_t*)h)[k] << 16;   /* bf16 -> fp32 is exact */
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* Mean aggregation (Eq. (1), AGGREGATE = mean) over one block:
 *   out[v,:] = (1/c_v) * sum over the block's edges e of row v of h[idx[e],:]
 * with c_v = indptr[v+1] - indptr[v] and out[v,:] = 0 when c_v = 0.
 * h: n_src x dim (dtype 0 fp32, 1 bf16); out and absmean: n_dst x dim doubles;
 * absmean[v,:] = (1/c_v) * sum |h[idx[e],:]| (the scale of the fp error). */
void orc_aggregate_fwd(const int64_t* indptr, const int32_t* idx, int64_t n_dst,
                       const void* h, int dtype, int32_t dim, double* out, double* absmean) {
    #pragma omp parallel for schedule(dynamic, 64)
    for (int64_t v = 0; v < n_dst; v++) {
        int64_t c = indptr[v + 1] - indptr[v];
        for (int32_t k = 0; k < dim; k++) {
            double s = 0.0, a = 0.0;
            for (int64_t e = indptr[v]; e < indptr[v + 1]; e++) {
                double x = load_elem(h, dtype, (int64_t)idx[e] * dim + k);
                s += x;
                a += x < 0 ? -x : x;
            }
            out[v * dim + k] = c > 0 ? s / (double)c : 0.0;
            if (absmean) absmean[v * dim + k] = c > 0 ? a / (double)c : 0.0;
        }
    }
}

/* Backward of the mean aggregation (the transpose map):
 *   gsrc[u,:] = sum over edges (v -> u) of the block of gdst[v,:] / c_v
 * for u < n_src, zero for a u that no edge names.  Accumulated in the edge
 * order of the block.  absmean has the same form with |gdst|. */
void orc_aggregate_bwd(const int64_t* indptr, const int32_t* idx, int64_t n_dst, int64_t n_src,
                       const void* gdst, int dtype, int32_t dim, double* gsrc, double* absmean) {
    memset(gsrc, 0, (size_t)n_src * (size_t)dim * sizeof(double));
    if (absmean) memset(absmean, 0, (size_t)n_src * (size_t)dim * sizeof(double));
    for (int64_t v = 0; v < n_dst; v++) {
        int64_t c = indptr[v + 1] - indptr[v];
        for (int64_t e = indptr[v]; e < indptr[v + 1]; e++) {
            int64_t u = idx[e];
            for (int32_t k = 0; k < dim; k++) {
                double g = load_elem(gdst, dtype, v * dim + k) / (double)c;
                gsrc[u * dim + k] += g;
                if (absmean) absmean[u * dim + k] += g < 0 ? -g : g;
            }
        }
    }
}

/* SAGE UPDATE of one layer (GARDEN page, Section II-A, Eq. (2) with UPDATE a
 * learnable map of the node's previous state and its aggregated message;
 * GraphSAGE's form: a linear layer over the concatenation, then ReLU):
 *   y[r][o]   = sum_{k<d} W[o][k] h[r][k] + sum_{k<d} W[o][d+k] m[r][k]
 *   out[r][o] = y[r][o] > 0 ? y[r][o] : 0
 * for r < n, o < d_out, with W of d_out rows of 2d.  h holds the dst rows'
 * own previous states, m their mean-aggregated messages.  Sums in fp64, in k
 * order; absum[r][o] is the sum of |terms| (the tolerance scale). */
void orc_sage_fwd(const void* h, const void* m, int dtype, const void* W, int wtype, int64_t n, int32_t d,
                  int32_t d_out, double* y, double* out, double* absum) {
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < n; r++) {
        for (int32_t o = 0; o < d_out; o++) {
            double s = 0.0, a = 0.0;
            for (int32_t k = 0; k < 2 * d; k++) {
                double z = k < d ? load_elem(h, dtype, r * d + k) : load_elem(m, dtype, r * d + (k - d));
                double t = load_elem(W, wtype, (int64_t)o * 2 * d + k) * z;
                s += t;
                a += t < 0 ? -t : t;
            }
            y[r * d_out + o] = s;
            out[r * d_out + o] = s > 0 ? s : 0.0;
            if (absum) absum[r * d_out + o] = a;
        }
    }
}

/* Backward of orc_sage_fwd for the loss gradient g = dL/dout [n x d_out]
 * (ReLU's derivative is 1 where y > 0, else 0, y from the forward):
 *   dy[r][o] = g[r][o] * (y[r][o] > 0)
 *   dW[o][k] = sum_r dy[r][o] z[r][k]          z = [h | m], k < 2d
 *   dh[r][k] = sum_o dy[r][o] W[o][k]          k < d
 *   dm[r][k] = sum_o dy[r][o] W[o][d + k]      k < d
 * Sums in fp64 (dW in r order, dh and dm in o order); the absum arrays hold
 * the sums of |terms|. */
void orc_sage_bwd(const void* h, const void* m, int dtype, const void* W, int wtype, const double* y,
                  const void* g, int gtype, int64_t n, int32_t d, int32_t d_out, double* dW, double* absum_dW,
                  double* dh, double* dm, double* absum_dz) {
    #pragma omp parallel for schedule(dynamic, 4)
    for (int32_t o = 0; o < d_out; o++) {
        for (int32_t k = 0; k < 2 * d; k++) {
            double s = 0.0, a = 0.0;
            for (int64_t r = 0; r < n; r++) {
                if (!(y[r * d_out + o] > 0)) continue;
                double z = k < d ? load_elem(h, dtype, r * d + k) : load_elem(m, dtype, r * d + (k - d));
                double t = load_elem(g, gtype, r * d_out + o) * z;
                s += t;
                a += t < 0 ? -t : t;
            }
            dW[(int64_t)o * 2 * d + k] = s;
            if (absum_dW) absum_dW[(int64_t)o * 2 * d + k] = a;
        }
    }
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < n; r++) {
        for (int32_t k = 0; k < 2 * d; k++) {
            double s = 0.0, a = 0.0;
            for (int32_t o = 0; o < d_out; o++) {
                if (!(y[r * d_out + o] > 0)) continue;
                double t = load_elem(g, gtype, r * d_out + o) * load_elem(W, wtype, (int64_t)o * 2 * d + k);
                s += t;
                a += t < 0 ? -t : t;
            }
            if (k < d) dh[r * d + k] = s;
            else dm[r * d + (k - d)] = s;
            if (absum_dz) absum_dz[r * 2 * d + k] = a;
        }
    }
}

/* ------------------------------------------------- cache presampling (NEXT) */
/* Full-link access statistics of one sampled mini-batch (GARDEN page, Section
 * IV-B, Eq. (4)): every node v of the batch adds
 *   W_feat(v) = w_in * 1(v in V_in) + sum_{l=1..L} omega_l * (1(v in V_src^(l)) + 1(v in V_dst^(l)))
 * to score[v].  Layer l is hop l of the sample: its src nodes are V_l and its
 * dst nodes V_{l-1}; the input nodes V_in are V_L, the nodes whose features
 * are gathered.  The nodes of V_h are the first hop_off[h] entries of unique.
 * Readings: the page gives no values for the layer weights omega_l, so they
 * are inputs (integers, so that sums are exact and independent of order);
 * w_in = 1, omega = 0 is the plain count of gathered appearances. */
void orc_access_stats(const int32_t* unique, const int64_t* hop_off, int32_t n_hops, const uint32_t* omega,
                      uint32_t w_in, uint32_t* score) {
    int64_t n_in = hop_off[n_hops];
    for (int64_t i = 0; i < n_in; i++) {
        uint32_t w = w_in;  /* every node of the batch is an input node */
        for (int32_t l = 1; l <= n_hops; l++) {
            int in_src = i < hop_off[l];      /* v in V_l     */
            int in_dst = i < hop_off[l - 1];  /* v in V_{l-1} */
            w += omega[l - 1] * (uint32_t)(in_src + in_dst);
        }
        score[unique[i]] += w;
    }
}

/* Nodes by descending score, ties by ascending ID: order[r] is the node of
 * rank r and rank_of[v] the rank of node v (the new ID a node gets when hot
 * nodes are recoded to the smallest IDs, GARDEN page Section IV-A). */
static const uint32_t* g_rank_score;
static int cmp_rank(const void* a, const void* b) {
    int32_t u = *(const int32_t*)a, v = *(const int32_t*)b;
    if (g_rank_score[u] != g_rank_score[v]) return g_rank_score[u] > g_rank_score[v] ? -1 : 1;
    return (u > v) - (u < v);
}

void orc_rank_by_score(const uint32_t* score, int64_t n, int32_t* order, int32_t* rank_of) {
    for (int64_t v = 0; v < n; v++) order[v] = (int32_t)v;
    g_rank_score = score;
    qsort(order, (size_t)n, sizeof(int32_t), cmp_rank);
    for (int64_t r = 0; r < n; r++) rank_of[order[r]] = (int32_t)r;
}

/* The graph with node order[r] renamed r (GARDEN page, Section IV-A: compact
 * IDs for high-frequency nodes): new row r is old row order[r], position for
 * position, with every neighbour u written as rank_of[u]. */
void orc_graph_renumber(const int64_t* indptr, const int32_t* indices, int64_t n, const int32_t* order,
                        const int32_t* rank_of, int64_t* new_indptr, int32_t* new_indices) {
    new_indptr[0] = 0;
    for (int64_t r = 0; r < n; r++) {
        int64_t v = order[r];
        int64_t deg = indptr[v + 1] - indptr[v];
        for (int64_t j = 0; j < deg; j++) new_indices[new_indptr[r] + j] = rank_of[indices[indptr[v] + j]];
        new_indptr[r + 1] = new_indptr[r] + deg;
    }
}

/* ------------------------------------------------ dynamic cache (NEXT) */
/* Adaptive dynamic feature caching (GARDEN page, Section IV-B, Eq. (5)-(6)).
 * Eq. (5): Score(v, t) = gamma * Score(v, t-1) + (occurrences of v among the
 * batch-t nodes B_t).  Readings:
 *   - B_t are the nodes of batch t that the static cache does not hold (the
 *     page's Dynamic-Cache serves only accesses the static cache misses);
 *   - the score is kept in fixed point and evaluated at the end of each
 *     update window of T batches (Eq. (6) reads it only there): with
 *     gamma = g / 2^16 and 8 fractional bits,
 *       W_{T-1} = 2^8,  W_{j-1} = (W_j * g) >> 16      (gamma^{T-1-j} in Q8)
 *       G_1 = g,        G_{i+1} = (G_i * g) >> 16       (gamma^T in Q16)
 *     batch j of the window (0 <= j < T) adds W_j to A[v] for each of its
 *     occurrences of v in B_j, and at the window's end
 *       S[v] = ((S[v] * G_T) >> 16) + A[v],  A[v] = 0,
 *     which is Eq. (5) applied T times, rounded down to the fixed point;
 *     every sum is an integer, so the result is exact and order-free.
 * orc_dyn_weights fills W[0..T) and returns G_T. */
uint32_t orc_dyn_weights(uint32_t g, int32_t T, uint32_t* W) {
    W[T - 1] = 256;
    for (int32_t j = T - 1; j > 0; j--) W[j - 1] = (uint32_t)(((uint64_t)W[j] * g) >> 16);
    uint64_t G = g;
    for (int32_t i = 1; i < T; i++) G = (G * g) >> 16;
    return (uint32_t)G;
}

/* batch j of the window: A[v] += w for every node v of the batch (local
 * order, n entries of unique) that the static cache does not hold */
void orc_dyn_accumulate(const int32_t* unique, int64_t n, const uint8_t* static_cached, uint32_t w, uint32_t* A) {
    for (int64_t i = 0; i < n; i++) {
        int32_t v = unique[i];
        if (!static_cached[v]) A[v] += w;
    }
}

/* end of a window: S = (S * G_T >> 16) + A, A = 0; then Eq. (6): the k_dyn
 * nodes of largest S (ties by ascending ID), only nodes with S > 0, into
 * dyn[]; returns how many were chosen */
int64_t orc_dyn_update(uint32_t* S, uint32_t* A, int64_t n_nodes, uint32_t G_T, int64_t k_dyn, int32_t* dyn) {
    for (int64_t v = 0; v < n_nodes; v++) {
        S[v] = (uint32_t)(((uint64_t)S[v] * G_T) >> 16) + A[v];
        A[v] = 0;
    }
    int32_t* order = (int32_t*)malloc((size_t)(n_nodes > 0 ? n_nodes : 1) * sizeof(int32_t));
    int32_t* rank = (int32_t*)malloc((size_t)(n_nodes > 0 ? n_nodes : 1) * sizeof(int32_t));
    if (!order || !rank) { free(order); free(rank); return -1; }
    orc_rank_by_score(S, n_nodes, order, rank);
    int64_t c = 0;
    for (int64_t r = 0; r < n_nodes && c < k_dyn; r++) {
        if (S[order[r]] == 0) break;
        dyn[c++] = order[r];
    }
    free(order);
    free(rank);
    return c;
}

/* -------------------------------------------- match and reorder (NEXT) */
/* FastGL explainer page ("Match-Reorder"): consecutive sampled subgraphs
 * share many nodes, so a batch reuses the features of the previous batch
 * still resident on the GPU, and a group of batches is ordered so that each
 * follows the one it overlaps most.
 * Match: pos[j] = the position of cur[j] in prev (prev holds distinct IDs),
 * or -1 when cur[j] is not there; returns the number matched. */
int64_t orc_match(const int32_t* prev, int64_t n_prev, const int32_t* cur, int64_t n_cur, int64_t n_nodes,
                  int32_t* pos) {
    int32_t* at = (int32_t*)malloc((size_t)(n_nodes > 0 ? n_nodes : 1) * sizeof(int32_t));
    if (!at) return -1;
    for (int64_t v = 0; v < n_nodes; v++) at[v] = -1;
    for (int64_t i = 0; i < n_prev; i++) at[prev[i]] = (int32_t)i;
    int64_t m = 0;
    for (int64_t j = 0; j < n_cur; j++) {
        pos[j] = at[cur[j]];
        m += pos[j] >= 0;
    }
    free(at);
    return m;
}

/* Overlap matrix of G node lists (list a = ids[off[a] .. off[a+1]), each with
 * distinct IDs): O[a*G + b] = |list a intersect list b| (the diagonal is the
 * list's size). */
int orc_overlap(const int32_t* ids, const int64_t* off, int32_t G, int64_t n_nodes, int64_t* O) {
    uint8_t* in = (uint8_t*)malloc((size_t)(n_nodes > 0 ? n_nodes : 1));
    if (!in) return -1;
    for (int32_t a = 0; a < G; a++) {
        memset(in, 0, (size_t)n_nodes);
        for (int64_t i = off[a]; i < off[a + 1]; i++) in[ids[i]] = 1;
        for (int32_t b = 0; b < G; b++) {
            int64_t c = 0;
            for (int64_t i = off[b]; i < off[b + 1]; i++) c += in[ids[i]];
            O[(int64_t)a * G + b] = c;
        }
    }
    free(in);
    return 0;
}

/* Greedy order (nearest overlap first): start at batch `first`, then
 * repeatedly take the batch not yet taken that overlaps most with the last
 * one taken (ties: the lowest index). */
void orc_greedy_order(const int64_t* O, int32_t G, int32_t first, int32_t* order) {
    uint8_t taken[1024];
    memset(taken, 0, sizeof(taken));
    order[0] = first;
    taken[first] = 1;
    for (int32_t k = 1; k < G; k++) {
        int32_t last = order[k - 1], best = -1;
        for (int32_t b = 0; b < G; b++) {
            if (taken[b]) continue;
            if (best < 0 || O[(int64_t)last * G + b] > O[(int64_t)last * G + best]) best = b;
        }
        order[k] = best;
        taken[best] = 1;
    }
}

/* In-degree of every node: the number of CSR positions that name it (how
 * often uniform neighbour sampling can reach it). */
void orc_in_degree(const int32_t* indices, int64_t m, int64_t n, uint32_t* deg) {
    for (int64_t v = 0; v < n; v++) deg[v] = 0;
    for (int64_t e = 0; e < m; e++) deg[indices[e]]++;
}

/* Ranking with a second key: descending score, then descending tie key,
 * then ascending ID.  Reading: Eq. (4) gives no score to the nodes the
 * presampled batches never reach (and equal scores to many others); their
 * in-degree, the chance uniform neighbour sampling reaches them, orders
 * them (GARDEN page, Section IV-A: hot nodes first). */
static const uint32_t* g_rank_tie;
static int cmp_rank2(const void* a, const void* b) {
    int32_t u = *(const int32_t*)a, v = *(const int32_t*)b;
    if (g_rank_score[u] != g_rank_score[v]) return g_rank_score[u] > g_rank_score[v] ? -1 : 1;
    if (g_rank_tie[u] != g_rank_tie[v]) return g_rank_tie[u] > g_rank_tie[v] ? -1 : 1;
    return (u > v) - (u < v);
}

void orc_rank_by_score_tie(const uint32_t* score, const uint32_t* tie, int64_t n, int32_t* order, int32_t* rank_of) {
    for (int64_t v = 0; v < n; v++) order[v] = (int32_t)v;
    g_rank_score = score;
    g_rank_tie = tie;
    qsort(order, (size_t)n, sizeof(int32_t), cmp_rank2);
    for (int64_t r = 0; r < n; r++) rank_of[order[r]] = (int32_t)r;
}

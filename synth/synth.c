/*
 * Seeded synthetic inputs for the mini-batch pipeline: a Chung-Lu power-law
 * CSR graph, N(0,1) node features and the seed nodes of each mini-batch.
 *
 * This module produces INPUTS only.  It holds none of the pipeline's own
 * arithmetic (no sampling hash, no relabel, no aggregation), so both the CUDA
 * path and the CPU oracle can consume what it makes without sharing code.
 * Its random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014), used here as a
 * counter-based generator: draw(seed, stream, i) = mix(base(seed,stream) +
 * (i+1)*golden).  The sampler's own hash is a different generator (Philox).
 *
 * Graph recipe (stand-in for the power-law graphs the GARDEN and FastGL pages
 * measure on, which are not available here):
 *   w(x) = w_max * (1 + x/i0)^(-1/(gamma-1)),  x in [0, N)
 *   node rank i has expected degree  wbar_i = integral of w over [i, i+1)
 *   i0 is bisected so that the mean of wbar equals the target mean degree
 *   M = round(N*mean) edge slots; slot s draws a source rank and a target rank
 *   independently from the density w (closed-form inverse CDF)
 *   ranks are mapped to node IDs by a keyed Feistel permutation, so an ID does
 *   not encode its degree
 *   self-loops and repeated (u,v) pairs are dropped; every row is sorted.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN64 0x9E3779B97F4A7C15ull

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* i-th output of the SplitMix64 stream whose state starts at base(seed, stream) */
static inline uint64_t draw(uint64_t seed, uint64_t stream, uint64_t i) {
    uint64_t base = sm_mix(seed * GOLDEN64 + sm_mix(stream + 0x5851F42D4C957F2Dull));
    return sm_mix(base + (i + 1) * GOLDEN64);
}

uint64_t synth_draw(uint64_t seed, uint64_t stream, uint64_t i) { return draw(seed, stream, i); }

int synth_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- Feistel */
/* A keyed bijection of [0, n): a balanced 4-round Feistel network on the
 * smallest even bit width 2^k >= n, with cycle walking back into [0, n). */
typedef struct { uint64_t key; int64_t n; int half; uint64_t mask; } feistel_t;

static feistel_t feistel_make(uint64_t key, int64_t n) {
    feistel_t f;
    int k = 2;
    while (((int64_t)1 << k) < n) k++;
    if (k & 1) k++;
    f.key = key; f.n = n; f.half = k / 2; f.mask = (1ull << f.half) - 1ull;
    return f;
}

static inline uint64_t feistel_once(const feistel_t* f, uint64_t x) {
    uint64_t l = x >> f->half, r = x & f->mask;
    for (int round = 0; round < 4; round++) {
        uint64_t t = l ^ (draw(f->key, 1000 + (uint64_t)round, r) & f->mask);
        l = r; r = t;
    }
    return (l << f->half) | r;
}

static inline int64_t feistel_apply(const feistel_t* f, int64_t i) {
    uint64_t x = (uint64_t)i;
    do { x = feistel_once(f, x); } while ((int64_t)x >= f->n);
    return (int64_t)x;
}

int64_t synth_perm(uint64_t key, int64_t n, int64_t i) {
    feistel_t f = feistel_make(key, n);
    return feistel_apply(&f, i);
}

/* -------------------------------------------------------------- Chung-Lu */
typedef struct { double n, wmax, a, i0, total; } cl_t;

/* integral of w over [0, x) */
static double cl_W(const cl_t* c, double x) {
    if (fabs(c->a - 1.0) < 1e-12) return c->wmax * c->i0 * log1p(x / c->i0);
    return c->wmax * c->i0 / (1.0 - c->a) * (pow(1.0 + x / c->i0, 1.0 - c->a) - 1.0);
}

/* inverse of cl_W */
static double cl_Winv(const cl_t* c, double u) {
    if (fabs(c->a - 1.0) < 1e-12) return c->i0 * expm1(u / (c->wmax * c->i0));
    double base = 1.0 + u * (1.0 - c->a) / (c->wmax * c->i0);
    if (base <= 0.0) return c->n;
    return c->i0 * (pow(base, 1.0 / (1.0 - c->a)) - 1.0);
}

static int cl_setup(cl_t* c, int64_t n, double mean, double gamma, double wmax) {
    if (n <= 0 || mean <= 0.0 || gamma <= 1.0 || wmax <= mean) return -1;
    c->n = (double)n; c->wmax = wmax; c->a = 1.0 / (gamma - 1.0);
    double lo = -30.0, hi = 40.0; /* natural log of i0 */
    for (int it = 0; it < 200; it++) {
        double mid = 0.5 * (lo + hi);
        c->i0 = exp(mid);
        double m = cl_W(c, c->n) / c->n;
        if (m < mean) lo = mid; else hi = mid;
    }
    c->i0 = exp(0.5 * (lo + hi));
    c->total = cl_W(c, c->n);
    return 0;
}

/* rank drawn for slot s on the given stream (1: source, 2: target) */
static inline int64_t cl_rank(const cl_t* c, uint64_t seed, uint64_t stream, int64_t s) {
    double u = (double)(draw(seed, stream, (uint64_t)s) >> 11) * (1.0 / 9007199254740992.0);
    double x = cl_Winv(c, u * c->total);
    int64_t i = (int64_t)x;
    if (i < 0) i = 0;
    if (i >= (int64_t)c->n) i = (int64_t)c->n - 1;
    return i;
}

double synth_chung_lu_i0(int64_t n, double mean, double gamma, double wmax) {
    cl_t c;
    if (cl_setup(&c, n, mean, gamma, wmax)) return -1.0;
    return c.i0;
}

/* expected degree of rank i (integral of w over [i, i+1)) */
double synth_chung_lu_weight(int64_t n, double mean, double gamma, double wmax, int64_t i) {
    cl_t c;
    if (cl_setup(&c, n, mean, gamma, wmax)) return -1.0;
    return cl_W(&c, (double)(i + 1)) - cl_W(&c, (double)i);
}

typedef struct {
    int64_t n, m;
    int64_t* indptr;
    int32_t* indices;
} synth_graph;

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Builds the graph; returns NULL on bad parameters or allocation failure. */
synth_graph* synth_graph_build(int64_t n, double mean, double gamma, double wmax, uint64_t seed) {
    cl_t c;
    if (n <= 0 || n > 2147483647LL) return NULL;
    if (cl_setup(&c, n, mean, gamma, wmax)) return NULL;
    int64_t slots = (int64_t)llround((double)n * mean);
    feistel_t perm = feistel_make(seed ^ 0xC0FFEEull, n);

    int64_t* cnt = (int64_t*)calloc((size_t)n + 1, sizeof(int64_t));
    if (!cnt) return NULL;
    /* pass 1: out-degree of every source before dedup */
    #pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < slots; s++) {
        int64_t u = feistel_apply(&perm, cl_rank(&c, seed, 1, s));
        __atomic_fetch_add(&cnt[u], 1, __ATOMIC_RELAXED);
    }
    int64_t* start = (int64_t*)malloc(((size_t)n + 1) * sizeof(int64_t));
    if (!start) { free(cnt); return NULL; }
    start[0] = 0;
    for (int64_t u = 0; u < n; u++) start[u + 1] = start[u] + cnt[u];
    int32_t* adj = (int32_t*)malloc((size_t)(slots > 0 ? slots : 1) * sizeof(int32_t));
    if (!adj) { free(cnt); free(start); return NULL; }
    memcpy(cnt, start, (size_t)n * sizeof(int64_t)); /* cnt becomes the fill cursor */
    /* pass 2: place targets (order inside a row is fixed by the sort below) */
    #pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < slots; s++) {
        int64_t u = feistel_apply(&perm, cl_rank(&c, seed, 1, s));
        int64_t v = feistel_apply(&perm, cl_rank(&c, seed, 2, s));
        int64_t p = __atomic_fetch_add(&cnt[u], 1, __ATOMIC_RELAXED);
        adj[p] = (int32_t)v;
    }
    /* pass 3: sort rows, drop self-loops and repeats */
    #pragma omp parallel for schedule(dynamic, 4096)
    for (int64_t u = 0; u < n; u++) {
        int32_t* row = adj + start[u];
        int64_t d = start[u + 1] - start[u], w = 0;
        if (d > 1) qsort(row, (size_t)d, sizeof(int32_t), cmp_i32);
        for (int64_t k = 0; k < d; k++) {
            if (row[k] == (int32_t)u) continue;
            if (w > 0 && row[w - 1] == row[k]) continue;
            row[w++] = row[k];
        }
        cnt[u] = w;
    }
    synth_graph* g = (synth_graph*)malloc(sizeof(synth_graph));
    if (!g) { free(cnt); free(start); free(adj); return NULL; }
    g->n = n;
    g->indptr = (int64_t*)malloc(((size_t)n + 1) * sizeof(int64_t));
    if (!g->indptr) { free(g); free(cnt); free(start); free(adj); return NULL; }
    g->indptr[0] = 0;
    for (int64_t u = 0; u < n; u++) g->indptr[u + 1] = g->indptr[u] + cnt[u];
    g->m = g->indptr[n];
    g->indices = (int32_t*)malloc((size_t)(g->m > 0 ? g->m : 1) * sizeof(int32_t));
    if (!g->indices) { free(g->indptr); free(g); free(cnt); free(start); free(adj); return NULL; }
    #pragma omp parallel for schedule(dynamic, 4096)
    for (int64_t u = 0; u < n; u++)
        memcpy(g->indices + g->indptr[u], adj + start[u], (size_t)cnt[u] * sizeof(int32_t));
    free(cnt); free(start); free(adj);
    return g;
}

int64_t synth_graph_n(const synth_graph* g) { return g->n; }
int64_t synth_graph_m(const synth_graph* g) { return g->m; }
int64_t* synth_graph_indptr(const synth_graph* g) { return g->indptr; }
int32_t* synth_graph_indices(const synth_graph* g) { return g->indices; }
void synth_graph_free(synth_graph* g) {
    if (!g) return;
    free(g->indptr); free(g->indices); free(g);
}

/* -------------------------------------------------------------- features */
static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b; memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

/* Rows [row0, row0+nrows) of the N x dim feature table: N(0,1) by Box-Muller
 * on a pair of 24-bit uniforms drawn for (row, column pair).
 * dtype 0 = fp32, 1 = bf16 (fp32 value rounded to nearest even). */
static void feature_row(int64_t v, int32_t dim, int32_t dtype, uint64_t seed, void* out_row) {
    int64_t pairs = (dim + 1) / 2;
    for (int64_t p = 0; p < pairs; p++) {
        uint64_t x = draw(seed, 3, (uint64_t)(v * pairs + p));
        float u1 = (float)((x >> 40) + 1) * (1.0f / 16777216.0f);
        float u2 = (float)(x & 0xFFFFFFull) * (1.0f / 16777216.0f);
        float rad = sqrtf(-2.0f * logf(u1));
        float z[2];
        z[0] = rad * cosf(6.28318530717958647692f * u2);
        z[1] = rad * sinf(6.28318530717958647692f * u2);
        for (int t = 0; t < 2; t++) {
            int64_t col = 2 * p + t;
            if (col >= dim) break;
            if (dtype == 0) ((float*)out_row)[col] = z[t];
            else ((uint16_t*)out_row)[col] = f32_to_bf16_rne(z[t]);
        }
    }
}

int synth_features(int64_t row0, int64_t nrows, int32_t dim, int32_t dtype, uint64_t seed, void* out) {
    if (dim <= 0 || nrows < 0 || (dtype != 0 && dtype != 1)) return -1;
    size_t rb = (size_t)dim * (dtype == 0 ? 4 : 2);
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; r++) feature_row(row0 + r, dim, dtype, seed, (char*)out + (size_t)r * rb);
    return 0;
}

/* Rows of the table in a given order: output row r is node ids[r]'s row (a
 * table laid out for recoded node IDs). */
int synth_features_rows(const int32_t* ids, int64_t nrows, int32_t dim, int32_t dtype, uint64_t seed, void* out) {
    if (dim <= 0 || nrows < 0 || (dtype != 0 && dtype != 1)) return -1;
    size_t rb = (size_t)dim * (dtype == 0 ? 4 : 2);
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; r++) feature_row(ids[r], dim, dtype, seed, (char*)out + (size_t)r * rb);
    return 0;
}

/* ------------------------------------------------------------ seed nodes */
/* Training mask: node v is a training node when draw(seed, 4, v) < p * 2^64
 * (p >= 1 keeps every node).  The epoch order walks a keyed permutation of
 * [0, N) and keeps training nodes; batch b is entries [b*B, (b+1)*B) of that
 * order.  Writes up to B distinct node IDs; returns how many were written. */
int32_t synth_batch_seeds(int64_t n, double p_mask, uint64_t seed, int64_t epoch, int64_t batch,
                          int32_t bsize, int32_t* out) {
    if (n <= 0 || bsize <= 0 || batch < 0) return 0;
    feistel_t perm = feistel_make(seed ^ (0xE90C0000ull + (uint64_t)epoch), n);
    uint64_t thr = 0;
    int all = p_mask >= 1.0;
    if (!all) thr = (uint64_t)(p_mask * 18446744073709551616.0);
    int64_t want_lo = batch * (int64_t)bsize, want_hi = want_lo + bsize, seen = 0;
    int32_t w = 0;
    for (int64_t i = 0; i < n && seen < want_hi; i++) {
        int64_t v = feistel_apply(&perm, i);
        if (!all && draw(seed, 4, (uint64_t)v) >= thr) continue;
        if (seen >= want_lo) out[w++] = (int32_t)v;
        seen++;
    }
    return w;
}

/* The whole epoch order of the training nodes (the sequence synth_batch_seeds
 * slices), in one pass: writes up to cap IDs, returns how many. */
int64_t synth_epoch_order(int64_t n, double p_mask, uint64_t seed, int64_t epoch, int32_t* out, int64_t cap) {
    if (n <= 0 || cap < 0) return 0;
    feistel_t perm = feistel_make(seed ^ (0xE90C0000ull + (uint64_t)epoch), n);
    uint64_t thr = 0;
    int all = p_mask >= 1.0;
    if (!all) thr = (uint64_t)(p_mask * 18446744073709551616.0);
    int64_t w = 0;
    for (int64_t i = 0; i < n && w < cap; i++) {
        int64_t v = feistel_apply(&perm, i);
        if (!all && draw(seed, 4, (uint64_t)v) >= thr) continue;
        out[w++] = (int32_t)v;
    }
    return w;
}

/* number of training nodes under the mask above */
int64_t synth_mask_count(int64_t n, double p_mask, uint64_t seed) {
    if (p_mask >= 1.0) return n;
    uint64_t thr = (uint64_t)(p_mask * 18446744073709551616.0);
    int64_t c = 0;
    #pragma omp parallel for reduction(+:c)
    for (int64_t v = 0; v < n; v++) c += draw(seed, 4, (uint64_t)v) < thr;
    return c;
}

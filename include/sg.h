/*
 * sg.h - C ABI of the GB300 mini-batch pipeline for sampling-based GNN
 * training: multi-hop neighbour sampling, ID dedup + relabel into per-hop
 * blocks, feature gather through an HBM hot-node cache, and mean
 * aggregation forward and backward.
 *
 * The operations follow the GARDEN page ("GARDEN: Efficient GPU-Accelerated
 * Billion-Scale GNN Training via Caching-Sampling-Batching Co-Design"):
 * Section II-A Eq. (1)-(2) (message passing; AGGREGATE = mean here), Section
 * II-B and Fig. 1 (layer-wise blocks: V_l = V_{l-1} u N_l(V_{l-1}), seeds are
 * the output nodes, V_k the input nodes), Section II-B Fig. 2 (Nfeat-Cache in
 * GPU memory, misses read zero-copy from pinned host memory), Section IV-C
 * (fixed-fanout uniform sampling; degree <= fanout keeps every neighbour),
 * Section IV-D (super-batch of K mini-batches with a BatchPtr and a GPU hash
 * table for dedup).  The sync-free ID map follows the FastGL explainer page
 * ("Fused-Map").
 *
 * Conventions
 *  - Every call returns sg_status (SG_OK = 0).  No exception crosses the ABI.
 *    sg_last_error() gives a message for the calling thread's last failure.
 *  - Pointers named d_* are device memory (or managed / device-accessible
 *    memory) of the current CUDA device; h_* are host memory.  Every buffer is
 *    OWNED BY THE CALLER except what sits behind an opaque handle (sg_graph,
 *    sg_cache), which the library owns and frees in the matching *_destroy.
 *  - Device work is asynchronous on the caller's stream (sg_stream_t is a
 *    cudaStream_t; NULL is the legacy default stream).  Calls return before the
 *    work finishes; no call synchronises the stream unless it says so.
 *  - Bad arguments found on the host return SG_ERR_INVALID_ARG at once.
 *    Problems found by a kernel (a node ID out of range, a full hash table,
 *    a repeated seed) set a sticky device error word; sg_stream_check()
 *    synchronises the stream, reads and clears it.
 *  - Memory the library owns (behind sg_graph and sg_cache) is allocated in
 *    sg_graph_load and sg_cache_build only; a failed allocation returns
 *    SG_ERR_OOM and leaves nothing allocated.  With the environment variable
 *    SG_FAULT_INJECT=alloc:N (read once per process) the N-th such allocation
 *    fails in that way without reaching the CUDA runtime, so callers can test
 *    their out-of-memory handling.
 *  - Every device-side wait (the look-back of the single-pass scans, the
 *    mbarrier waits of the copy-engine and tensor-core kernels) is bounded;
 *    a wait that gives up sets SG_ERR_TIMEOUT in the device error word.
 *  - Sizes that depend on the data (|V_h|, E_h) stay on the device.  Calls that
 *    consume them take a host-side CAPACITY plus an optional device pointer to
 *    the actual count (d_n / d_dims), so a whole mini-batch can run, and be
 *    captured in a CUDA graph, without a host synchronisation.
 */
#ifndef SG_H
#define SG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t sg_status;
#define SG_OK 0
#define SG_ERR_INVALID_ARG 1    /* a host-side argument is invalid */
#define SG_ERR_INVALID_INDEX 2  /* a kernel met a node ID / index out of range */
#define SG_ERR_CAPACITY 3       /* a table or buffer bound was exceeded */
#define SG_ERR_OOM 4            /* the library could not allocate memory it owns */
#define SG_ERR_CUDA 5           /* a CUDA runtime call failed (message has the name) */
#define SG_ERR_TIMEOUT 6        /* a bounded device wait gave up */
#define SG_ERR_UNSUPPORTED 7    /* valid request this build does not support */

#define SG_F32 0                /* IEEE binary32 */
#define SG_BF16 1               /* bfloat16, stored as uint16 bit patterns */

#define SG_MAX_HOPS 8
#define SG_MAX_SUB 64           /* mini-batches per super-batch */
#define SG_MAX_FANOUT 256

typedef void* sg_stream_t;      /* cudaStream_t */
typedef void* sg_event_t;       /* cudaEvent_t */

typedef struct sg_graph sg_graph;
typedef struct sg_cache sg_cache;

/* Library version (major*10000 + minor*100 + patch). */
int32_t sg_version(void);

/* Copies the calling thread's last error message into buf (NUL-terminated,
 * truncated to n bytes); returns the full message length. */
int32_t sg_last_error(char* buf, size_t n);

/* Synchronises `stream`, then reads and clears the device error word that the
 * library's kernels set.  Returns SG_OK, SG_ERR_INVALID_INDEX, SG_ERR_CAPACITY,
 * SG_ERR_INVALID_ARG (repeated seed in one mini-batch), SG_ERR_TIMEOUT (a
 * bounded device wait gave up) or SG_ERR_CUDA. */
sg_status sg_stream_check(sg_stream_t stream);

/* ------------------------------------------------------------------ graph */
/* Loads a CSR graph into HBM (one-time, synchronous).  Row v lists the
 * neighbours that node v aggregates from (the GARDEN page's N(u), Section
 * II-A); sampling takes positions of this row.
 *   h_indptr    host, n_nodes+1 offsets, int32 (offset_bits = 32) or int64
 *               (offset_bits = 64); must start at 0, be non-decreasing and end
 *               at n_edges.  int32 offsets need n_edges < 2^31.
 *   h_indices   host, n_edges int32 node IDs in [0, n_nodes).
 *   n_nodes     1 .. 2^31-1.
 * The library copies both arrays (it keeps the offset width given) and
 * validates them on the GPU; invalid input returns SG_ERR_INVALID_ARG and no
 * handle.  *out receives a handle freed by sg_graph_destroy. */
sg_status sg_graph_load(const void* h_indptr, int32_t offset_bits, const int32_t* h_indices,
                        int64_t n_nodes, int64_t n_edges, sg_graph** out);

/* Frees the graph's device memory (synchronous).  NULL is a no-op. */
sg_status sg_graph_destroy(sg_graph* g);

/* Shape of a loaded graph; any out pointer may be NULL. */
sg_status sg_graph_info(const sg_graph* g, int64_t* n_nodes, int64_t* n_edges, int32_t* offset_bits,
                        int64_t* max_degree);

/* Copies a loaded graph's CSR back to host memory (synchronous): h_indptr
 * gets n_nodes + 1 offsets of the graph's offset width, h_indices n_edges
 * int32 IDs; for example to keep a recoded graph (sg_graph_renumber). */
sg_status sg_graph_copy_out(const sg_graph* g, void* h_indptr, int32_t* h_indices);

/* ---------------------------------------------------------------- sampling */
/* Worst-case sizes of one sampler_run, so the caller can preallocate.
 * Counts are totals over the n_sub mini-batches of a super-batch. */
typedef struct sg_sample_bounds {
    int64_t max_nodes[SG_MAX_HOPS + 1];  /* bound on sum_k |V_h^k|, h = 0..H */
    int64_t max_edges[SG_MAX_HOPS];      /* bound on sum_k E_h^k, index h-1 */
    int64_t counts_len;                  /* int32 entries of sg_blocks.counts */
    size_t workspace_bytes;              /* device workspace sampler_run needs (see
                                            sg_sampler_workspace_init) */
} sg_sample_bounds;

/*   h_batch_ptr  host, n_sub+1 non-decreasing offsets into the seed array
 *                (GARDEN page Section IV-D "BatchPtr"); NULL means n_sub = 1
 *                with n_seeds seeds.
 *   h_fanouts    host, n_hops fanouts; h_fanouts[h-1] is the fanout of hop h,
 *                hop 1 being the hop next to the seeds; 1..SG_MAX_FANOUT. */
sg_status sg_sampler_bounds(const sg_graph* g, int32_t n_seeds, const int32_t* h_batch_ptr, int32_t n_sub,
                            const int32_t* h_fanouts, int32_t n_hops, sg_sample_bounds* out);

/* Output of sg_sampler_run: caller-allocated DEVICE arrays sized by
 * sg_sampler_bounds.  With K = n_sub mini-batches laid back to back:
 *   unique     [max_nodes[H]]  global IDs: mini-batch k's V_H^k occupies
 *              unique[U_k, U_k + |V_H^k|), U_k = sum_{k'<k} |V_H^k'|; inside
 *              it, its seeds come first (in the order given) and V_h^k is the
 *              prefix of length |V_h^k|.
 *   counts     [counts_len] int32, written on the device:
 *                counts[h]           = sum_k |V_h^k|     (h = 0..H)
 *                counts[H+1+h-1]     = sum_k E_h^k       (h = 1..H)
 *                counts[(2H+1)(1+k) + h]       = |V_h^k|
 *                counts[(2H+1)(1+k) + H+1+h-1] = E_h^k
 *   indptr[h-1] [max_nodes[h-1]+1] block CSR of hop h over dst rows: mini-
 *              batch k's dst d (its local ID, d < |V_{h-1}^k|) is row
 *              D_k + d with D_k = sum_{k'<k} |V_{h-1}^k'|.
 *   idx[h-1]   [max_edges[h-1]] src row of each edge: mini-batch k's local
 *              src ID s (< |V_h^k|) is stored as S_k + s with
 *              S_k = sum_{k'<k} |V_h^k'|.
 * For K = 1 this is the plain per-batch block list: idx holds local IDs into
 * V_h and rows are the local IDs of V_{h-1}.  A hop-h block maps H_h (rows in
 * V_h order) to H_{h-1}, so aggregate_fwd can run hop H .. 1 on these arrays
 * directly, with d_dims = counts + (h-1). */
typedef struct sg_blocks {
    int32_t* unique;
    int32_t* counts;
    int32_t* indptr[SG_MAX_HOPS];
    int32_t* idx[SG_MAX_HOPS];
} sg_blocks;

/* Prepares a sampler workspace (sizes as in sg_sampler_bounds): clears its
 * persistent part once.  Asynchronous on `stream`. */
sg_status sg_sampler_workspace_init(const sg_graph* g, int32_t n_seeds, const int32_t* h_batch_ptr, int32_t n_sub,
                                    const int32_t* h_fanouts, int32_t n_hops, void* d_workspace,
                                    size_t workspace_bytes, sg_stream_t stream);

/* Multi-hop sampling plus relabel (GARDEN page Section II-B and Fig. 1;
 * Section IV-C; Section IV-D; FastGL explainer "Fused-Map").
 * Hop h = 1..H samples every node v of V_{h-1}: with deg = the length of
 * v's CSR row and f = h_fanouts[h-1], all positions when deg <= f, otherwise
 * the f positions j with the smallest keys (r, j), where r is word (j mod 4)
 * of Philox4x32-10 (Salmon et al., SC'11) with counter (j/4, v, h, 0) and key
 * (seed & 0xffffffff, seed >> 32); positions are listed in ascending order.
 * This is a uniform sample without replacement, identical on every device and
 * on the CPU.  The sampled neighbours not yet in V_{h-1}^k join V_h^k in order
 * of first occurrence in the hop's edge list, ordered by (dst, position).
 * A super-batch (n_sub = K > 1) gives exactly the K results of K separate
 * calls with the same seed; each distinct node is sampled once per hop.
 *   d_seeds      device, n_seeds int32; seeds of one mini-batch must be
 *                distinct (else the device error word reports
 *                SG_ERR_INVALID_ARG) and in [0, n_nodes).
 *   h_batch_ptr  host, as in sg_sampler_bounds.
 *   seed / d_seed  the hash seed; when d_seed (device, one uint64) is not
 *                NULL it overrides `seed` and is read when the kernels run, so
 *                a captured CUDA graph can be replayed with a new seed.
 *   d_workspace  device workspace of at least bounds.workspace_bytes, 256-byte
 *                aligned, prepared once by sg_sampler_workspace_init for this
 *                graph and these sizes.  Part of it persists: a direct map
 *                with one 32-bit entry per node and mini-batch (the first
 *                position of each sampled node, then its local ID) that every
 *                run leaves cleared for the next.  Hand the same workspace to
 *                no other call in between, and do not run two calls on it at
 *                once.
 *   h_hop_events  host array of n_hops event handles (an entry may be NULL),
 *                or NULL.  Entry h-1 is recorded on `stream` as soon as the
 *                node list of hop h is final, so that work on V_h (such as
 *                gathering its feature rows) can start on another stream
 *                while later hops are sampled.  With n_sub = 1, at that
 *                point unique[0, |V_h|) and counts[(2H+1) + h] (= |V_h|) are
 *                final (counts[h] and the block arrays are not yet); with
 *                n_sub > 1 every entry is recorded at the end of the call.
 * Asynchronous on `stream`; no host synchronisation inside. */
sg_status sg_sampler_run(const sg_graph* g, const int32_t* d_seeds, int32_t n_seeds, const int32_t* h_batch_ptr,
                         int32_t n_sub, const int32_t* h_fanouts, int32_t n_hops, uint64_t seed,
                         const uint64_t* d_seed, void* d_workspace, size_t workspace_bytes, const sg_blocks* out,
                         const sg_event_t* h_hop_events, sg_stream_t stream);

/* Standalone dedup + relabel (the step sampler_run fuses; FastGL explainer
 * "Fused-Map", GARDEN page Section IV-D hash-table dedup).
 *   d_prefix    device, n_prefix distinct IDs that keep local IDs 0..n_prefix-1
 *   d_ids       device, n_ids IDs (non-negative int32)
 * Output (device): d_unique[0 .. n_unique) = the prefix, then every ID of
 * d_ids not in the prefix in order of first occurrence; d_local[i] = local ID
 * of d_ids[i]; *d_n_unique (device int32) = n_unique.
 *   d_unique    room for n_prefix + n_ids entries
 *   workspace   sg_relabel_workspace(n_prefix, n_ids) bytes, 256-byte aligned
 * A repeated prefix ID sets the device error word (SG_ERR_INVALID_ARG). */
size_t sg_relabel_workspace(int64_t n_prefix, int64_t n_ids);
sg_status sg_relabel(const int32_t* d_ids, int64_t n_ids, const int32_t* d_prefix, int64_t n_prefix,
                     int32_t* d_unique, int32_t* d_local, int32_t* d_n_unique, void* d_workspace,
                     size_t workspace_bytes, sg_stream_t stream);

/* Relabel that allocates nothing, for callers that cannot call cudaMalloc or
 * hand the library a workspace: a plugin or kernel-launch hook inside another
 * framework whose memory is owned by that framework's allocator, a process
 * with a fixed device-memory budget, or a code path where an allocation would
 * synchronise the device.  The pages have no counterpart of this call; it is
 * an interface convenience of this library.
 * Same inputs, outputs and result as sg_relabel, but its scratch is a static
 * device array of SG_RELABEL_NOALLOC_SCRATCH_BYTES (11 MiB) inside the library,
 * which every GPU that loads the library keeps until the process exits.
 *   n_prefix + n_ids  at most SG_RELABEL_NOALLOC_MAX_IDS (262,144); larger
 *                     requests return SG_ERR_INVALID_ARG (use sg_relabel).
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any CUDA stream capture.
 * Every call on a device shares the one array: calls whose GPU work overlaps
 * (on different streams) race and give wrong results; serialise them.  The
 * array's previous contents are never relied on (the hash table is cleared
 * at the start of each call). */
#define SG_RELABEL_NOALLOC_MAX_IDS 262144
#define SG_RELABEL_NOALLOC_SCRATCH_BYTES (11u << 20)
sg_status sg_relabel_noalloc(const int32_t* d_ids, int64_t n_ids, const int32_t* d_prefix, int64_t n_prefix,
                             int32_t* d_unique, int32_t* d_local, int32_t* d_n_unique, sg_stream_t stream);

/* ------------------------------------------------------------------- cache */
/* Builds the HBM feature cache (GARDEN page Section II-B Fig. 2, Nfeat-Cache;
 * one-time, synchronous on `stream`).
 *   h_feat        host feature table, n_nodes x dim, row-major, dtype SG_F32 or
 *                 SG_BF16.  It must stay valid while the cache lives: rows not
 *                 cached are read from it zero-copy.  Pinned memory
 *                 (cudaHostAlloc / cudaHostRegister) is required unless the
 *                 device can access pageable memory.  May be NULL when
 *                 n_cache = n_nodes and d_feat gives the rows.
 *   d_feat        optional device copy of the whole table to fill the cache
 *                 from (NULL: read the rows from h_feat).
 *   h_ranked      host, n_cache distinct node IDs; h_ranked[s] goes to cache
 *                 slot s, and a map of n_nodes int32 slots says where each
 *                 node is.  NULL caches the ID range [0, n_cache) with slot =
 *                 ID and no map: the hit test is ID < n_cache (GARDEN page
 *                 Section IV-A, hot nodes recoded to the smallest IDs; see
 *                 sg_graph_renumber).  That is also the form for a whole
 *                 table (n_cache = n_nodes).
 * The library allocates n_cache rows (plus the slot map with h_ranked) in HBM. */
sg_status sg_cache_build(const void* h_feat, const void* d_feat, int32_t dtype, int64_t n_nodes, int32_t dim,
                         const int32_t* h_ranked, int64_t n_cache, sg_cache** out, sg_stream_t stream);

/* Frees the cache's device memory (synchronous).  NULL is a no-op. */
sg_status sg_cache_destroy(sg_cache* c);

/* Device view of a cache (for callers that want to inspect it); *d_slot_of
 * is NULL for an ID-range cache (built without h_ranked). */
sg_status sg_cache_info(const sg_cache* c, int64_t* n_nodes, int32_t* dim, int32_t* dtype, int64_t* n_cache,
                        const int32_t** d_slot_of);

typedef struct sg_gather_stats {
    unsigned long long hits;     /* rows read from the HBM cache */
    unsigned long long misses;   /* rows read zero-copy from host memory */
} sg_gather_stats;

/* Feature gather through the cache (GARDEN page Section II-B, Nfeat-
 * Selecting): for first <= i < n, out row i = feature row d_ids[i], byte for
 * byte, taken from the HBM cache when the node is cached, else read zero-copy
 * from the host table.
 *   d_ids     device, n_cap node IDs
 *   d_n       device int32 count (n = *d_n <= n_cap) or NULL (n = n_cap)
 *   d_first   device int32 first row (0 <= first, clamped to n) or NULL (0);
 *             with it a list can be gathered in two parts, the first while
 *             the rest of the list is still being produced
 *   d_out     device, n_cap x dim in the cache's dtype (other rows untouched)
 *   d_stats   device, accumulated (+=) hit/miss counters, or NULL
 *   d_workspace, workspace_bytes
 *             device scratch of sg_gather_workspace(c, n_cap) bytes (256-byte
 *             aligned; one per gather in flight), or NULL.  With it, and a
 *             host table large enough that sg_gather_workspace is non-zero,
 *             the misses are read grouped by 2 MB region of the host table
 *             (a counting sort of the missed rows by region) instead of in
 *             row order: on a table of tens of GB, random zero-copy reads
 *             lose most of their rate to address translation, and reads of
 *             one region in a row share it.  The output is the same either
 *             way.
 * An ID out of range sets the device error word and its row is zero-filled. */
sg_status sg_gather(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                    const int32_t* d_first, void* d_out, sg_gather_stats* d_stats, void* d_workspace,
                    size_t workspace_bytes, sg_stream_t stream);

/* sg_gather with reuse of the previous batch's rows (FastGL explainer page,
 * "Match-Reorder": consecutive sampled subgraphs share many nodes, so the
 * features a batch shares with the previous one are copied from that
 * batch's gathered rows, still in HBM, and only the rest is shipped):
 *   d_pos        device int32 [n_cap]: for row i, the row of d_prev_rows that
 *                holds node d_ids[i] (sg_match), or -1
 *   d_prev_rows  device, the previous batch's gathered rows (same row size),
 *                16-byte aligned; it must not overlap d_out
 *   d_reused     device, accumulated (+=) count of rows copied from it, or
 *                NULL; d_stats counts the other rows as with sg_gather
 * Other arguments and the result as sg_gather: out row i = feature row
 * d_ids[i], byte for byte. */
sg_status sg_gather_reuse(const sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                          const int32_t* d_first, const int32_t* d_pos, const void* d_prev_rows, void* d_out,
                          sg_gather_stats* d_stats, unsigned long long* d_reused, void* d_workspace,
                          size_t workspace_bytes, sg_stream_t stream);

/* Match (FastGL explainer page, "Match-Reorder"): d_pos[j] = the position of
 * node d_cur[j] in d_prev (whose IDs are distinct), or -1.  Counts: the
 * lists hold prev_cap / cur_cap entries, *d_prev_n / *d_cur_n of them when
 * those device pointers are not NULL.  d_map: device int32 [n_nodes],
 * caller-owned scratch that must be all -1 (bytes 0xFF) on entry and is all
 * -1 again when the call's work is done.  d_matched: device int32,
 * accumulated (+=) number of matches, or NULL.  IDs outside [0, n_nodes) set
 * the device error word.  Asynchronous on `stream`. */
sg_status sg_match(const int32_t* d_prev, int64_t prev_cap, const int32_t* d_prev_n, const int32_t* d_cur,
                   int64_t cur_cap, const int32_t* d_cur_n, int32_t* d_map, int64_t n_nodes, int32_t* d_pos,
                   int32_t* d_matched, sg_stream_t stream);

/* Overlap matrix of a group of node lists (the Reorder step): list a is
 * d_ids[h_off[a] .. h_off[a+1]) (distinct IDs within a list), 1..32 lists;
 * d_overlap (device uint64 [n_lists x n_lists]) gets |list a ^ list b| at
 * [a * n_lists + b] (the diagonal is a list's size).  d_mask: device uint32
 * [n_nodes] scratch, all zero on entry and again after the call's work.
 * Asynchronous on `stream`. */
sg_status sg_overlap(const int32_t* d_ids, const int64_t* h_off, int32_t n_lists, uint32_t* d_mask, int64_t n_nodes,
                     unsigned long long* d_overlap, sg_stream_t stream);

/* Greedy order of a group (nearest overlap first; host only): h_order[0] =
 * first, then each next list is the one not yet taken that overlaps most
 * with the last one taken (ties: the lowest index).  h_overlap: host
 * n_lists x n_lists as from sg_overlap; 1..1024 lists. */
sg_status sg_greedy_order(const unsigned long long* h_overlap, int32_t n_lists, int32_t first, int32_t* h_order);

/* Bytes of the workspace sg_gather uses to read the misses of up to n_cap
 * rows grouped by host-table region; 0 when the cache has no host table or
 * the table is small enough (under 32 GiB) that row order reads as fast. */
size_t sg_gather_workspace(const sg_cache* c, int64_t n_cap);

/* Bounded dynamic cache beside the static one (GARDEN page, Section IV-B,
 * "Adaptive Dynamic Feature Caching", Eq. (5)-(6)).  It holds k_dyn more rows
 * in HBM, chosen among the nodes the static cache misses by a decayed count
 * of their recent accesses, and sg_gather serves a static miss from it when
 * it can (counted as a hit).  Rows are byte-identical to the table's, so a
 * gather's output does not depend on it.
 * Scores (Eq. (5), read in windows of t_update batches and in fixed point):
 * with gamma = gamma_q16 / 2^16 in (0, 1], batch j of a window (0-based)
 * adds W_j = gamma^(t_update-1-j) (8 fractional bits, computed as
 * W_{T-1} = 256, W_{j-1} = W_j * gamma_q16 >> 16) to A[v] for each of its
 * nodes v that the static cache misses; after the window's last batch
 *   S[v] = (S[v] * gamma^T >> 16) + A[v],  A[v] = 0
 * (gamma^T in Q16 by repeated multiplication, rounded down each time), and
 * the dynamic set becomes the k_dyn nodes of largest S > 0, ties by
 * ascending ID (Eq. (6)).  Nodes that stay keep their slot; only entering
 * nodes' rows are copied from the host table.  All sums are integers: the
 * scores and the set are deterministic.
 *   sg_dyn_cache_create  attaches the dynamic cache to c (which must leave
 *                 rows to the host table); freed with the cache.  Synchronous.
 *   sg_dyn_cache_batch   adds one batch's nodes (device IDs, n_cap entries,
 *                 *d_n of them when d_n is not NULL; e.g. the sampler's unique
 *                 array and its count of V_H) and, after every t_update-th
 *                 call, updates the set.  Asynchronous on `stream`; order it
 *                 after the gathers of the batch and before the next batch's
 *                 gathers (the update changes the slots they read).  It
 *                 keeps the window position on the host, so a captured CUDA
 *                 graph would replay one position only.
 *   sg_dyn_cache_info    k_dyn, the position in the window and, into host
 *                 arrays when not NULL, the scores S [n_nodes] and the node in
 *                 each slot [k_dyn] (-1: free); synchronises `stream`. */
sg_status sg_dyn_cache_create(sg_cache* c, int64_t k_dyn, uint32_t gamma_q16, int32_t t_update, sg_stream_t stream);
sg_status sg_dyn_cache_batch(sg_cache* c, const int32_t* d_ids, int64_t n_cap, const int32_t* d_n,
                             sg_stream_t stream);
sg_status sg_dyn_cache_info(const sg_cache* c, int64_t* k_dyn, int32_t* window_pos, uint32_t* h_score,
                            int32_t* h_nodes, sg_stream_t stream);

/* -------------------------------------------------------------- aggregate */
/* Mean aggregation over one block (GARDEN page Section II-A Eq. (1) with
 * AGGREGATE = mean):
 *   out[v,:] = (1/c_v) * sum_{e in row v} h[idx[e],:],  c_v = row length,
 *   out[v,:] = 0 when c_v = 0,                          for v < n_dst.
 * Sums are accumulated in fp32.  dtype_in/dtype_out: SG_F32 -> SG_F32, or
 * SG_BF16 -> SG_BF16 (round to nearest even) / SG_F32.
 *   d_indptr  device int32 [n_dst_cap+1], d_idx device int32 [E]
 *   d_h       device [n_src_cap x dim]; d_out device [n_dst_cap x dim]
 *   d_dims    device int32[2] = {n_dst, n_src} (each <= its cap) or NULL
 * An idx outside [0, n_src) sets the device error word (the edge is skipped). */
sg_status sg_aggregate_fwd(const int32_t* d_indptr, const int32_t* d_idx, int32_t n_dst_cap, int32_t n_src_cap,
                           const int32_t* d_dims, const void* d_h, int32_t dtype_in, int32_t dim, void* d_out,
                           int32_t dtype_out, sg_stream_t stream);

/* Workspace of sg_aggregate_bwd for a block with these capacities. */
size_t sg_aggregate_bwd_workspace(int32_t n_dst_cap, int32_t n_src_cap, int64_t n_edge_cap);

/* Backward of the mean aggregation (the transpose of the map above):
 *   gsrc[u,:] = sum over edges e = (v -> u) of gdst[v,:] / c_v,  u < n_src,
 * zero for a u no edge names.  The block is transposed in the workspace (a
 * sort of the edges by (src, edge), so the summation order is fixed and the
 * result deterministic), then each src row is one fp32 sum: no float atomics.
 *   d_gdst   device [n_dst_cap x dim]; d_gsrc device [n_src_cap x dim]
 *   n_edge_cap  capacity bound on E = indptr[n_dst]
 * dtypes as in sg_aggregate_fwd. */
sg_status sg_aggregate_bwd(const int32_t* d_indptr, const int32_t* d_idx, int32_t n_dst_cap, int32_t n_src_cap,
                           int64_t n_edge_cap, const int32_t* d_dims, const void* d_gdst, int32_t dtype_in,
                           int32_t dim, void* d_gsrc, int32_t dtype_out, void* d_workspace, size_t workspace_bytes,
                           sg_stream_t stream);

/* Transposed blocks of one sampler_run output, for the backward pass:
 * caller-allocated DEVICE arrays, hop h at index h-1:
 *   tptr[h-1]  [max_nodes[h] + 2] row pointer over the src rows of hop h
 *   tdst[h-1]  [max_edges[h-1]]   dst row of each edge, edges of a src row in
 *                                 ascending (dst, position) order
 *   tw[h-1]    [max_edges[h-1]]   1 / c_dst (fp32) */
typedef struct sg_transposed {
    int32_t* tptr[SG_MAX_HOPS];
    int32_t* tdst[SG_MAX_HOPS];
    float* tw[SG_MAX_HOPS];
} sg_transposed;

/* Workspace of sg_transpose_blocks (max_nodes / max_edges as returned by
 * sg_sampler_bounds); 0 on bad arguments. */
size_t sg_transpose_workspace(const int64_t* max_nodes, const int64_t* max_edges, int32_t n_hops);

/* Transposes every block of `blocks` (the output of sg_sampler_run with these
 * bounds) in one set of launches; the counts are read on the device.  The
 * transposed blocks feed sg_aggregate_bwd_t and do not depend on features, so
 * the call can run on a second stream while gather and forward proceed.
 * Edges of one src row are ordered by edge index: the result is deterministic. */
sg_status sg_transpose_blocks(const sg_blocks* blocks, const int64_t* max_nodes, const int64_t* max_edges,
                              int32_t n_hops, const sg_transposed* out, void* d_workspace, size_t workspace_bytes,
                              sg_stream_t stream);

/* Backward of the mean aggregation over a transposed block (see
 * sg_aggregate_bwd): gsrc[u,:] = sum_p tw[p] * gdst[tdst[p],:] for u < n_src.
 *   d_dims  device int32[2] = {n_dst, n_src} of the FORWARD block, or NULL */
sg_status sg_aggregate_bwd_t(const int32_t* d_tptr, const int32_t* d_tdst, const float* d_tw, int32_t n_src_cap,
                             int32_t n_dst_cap, const int32_t* d_dims, const void* d_gdst, int32_t dtype_in,
                             int32_t dim, void* d_gsrc, int32_t dtype_out, sg_stream_t stream);

/* ------------------------------------- cache presampling and node recoding */
/* Full-link access statistics (GARDEN page Section IV-B, Eq. (4)) of one
 * sampler_run output, for ranking nodes before the cache is built: every node
 * v of every mini-batch adds
 *   W_feat(v) = w_in + sum_{l=1..H} omega[l-1] * (1(v in V_l) + 1(v in V_{l-1}))
 * to d_score[v] (layer l's src nodes are V_l, its dst nodes V_{l-1}; every
 * node of the output is an input node, V_in = V_H).  The page leaves the
 * layer weights open; they are integers here, so the sums are exact and
 * do not depend on the order of the atomic adds.  w_in = 1, omega = 0 counts
 * gathered appearances.  Sums wrap modulo 2^32.
 *   blocks, unique_cap  the sampler output and the capacity of its unique
 *                       array (bounds.max_nodes[H]); counts are read on the
 *                       device
 *   h_omega      host, n_hops weights
 *   d_score      device uint32 [n_nodes], accumulated (+=)
 * A node ID outside [0, n_nodes) sets the device error word. */
sg_status sg_access_stats(const sg_blocks* blocks, int64_t unique_cap, int32_t n_hops, int32_t n_sub,
                          const uint32_t* h_omega, uint32_t w_in, uint32_t* d_score, int64_t n_nodes,
                          sg_stream_t stream);

/* Nodes ordered by descending score, then (when d_tie is not NULL) by
 * descending tie key, then by ascending ID: d_order[r] (device int32
 * [n_nodes]) is the node of rank r and, when d_rank_of is not NULL,
 * d_rank_of[v] (device int32 [n_nodes]) the rank of node v.  d_score and
 * d_tie: device uint32 [n_nodes].  Presampled statistics leave most nodes of
 * a large graph without a score; their in-degree (sg_graph_in_degree), the
 * chance that uniform neighbour sampling reaches them, is the natural tie
 * key.  Stable radix sorts; the result is deterministic.  Workspace:
 * sg_rank_workspace(n_nodes) bytes, 256-byte aligned (0 on bad sizes). */
size_t sg_rank_workspace(int64_t n_nodes);
sg_status sg_rank_by_score(const uint32_t* d_score, const uint32_t* d_tie, int64_t n_nodes, int32_t* d_order,
                           int32_t* d_rank_of, void* d_workspace, size_t workspace_bytes, sg_stream_t stream);

/* In-degree of every node of a graph: d_deg[u] (device uint32 [n_nodes]) =
 * the number of CSR positions naming u.  Asynchronous on `stream`. */
sg_status sg_graph_in_degree(const sg_graph* g, uint32_t* d_deg, sg_stream_t stream);

/* Recodes a graph's nodes (GARDEN page Section IV-A: the allocator gives the
 * high-frequency nodes compact IDs): the new graph's row r is the old row
 * d_order[r], position for position, with every neighbour u written as
 * d_rank_of[u].  With the order of sg_rank_by_score the hot nodes take the
 * smallest IDs, so an ID-range cache (sg_cache_build without h_ranked) of
 * the top C rows is hit exactly when ID < C, and the rows a batch misses
 * sit in a compact, rank-ordered part of the host table.  The caller lays the
 * feature table out in the new order (new row r = old row d_order[r]) and
 * maps seed IDs through d_rank_of.  Sampling the new graph is sampling a
 * graph like any other: the hash takes the new IDs.
 *   d_order, d_rank_of  device int32 [n_nodes], inverse permutations of
 *               [0, n_nodes) (checked: SG_ERR_INVALID_ARG otherwise)
 * One-time and synchronous on `stream`; *out receives a new handle (same
 * offset width) freed by sg_graph_destroy. */
sg_status sg_graph_renumber(const sg_graph* g, const int32_t* d_order, const int32_t* d_rank_of, sg_graph** out,
                            sg_stream_t stream);

/* ----------------------------------------------------- SAGE UPDATE (GEMM) */
/* The UPDATE of one GraphSAGE layer (GARDEN page Section II-A, Eq. (2); the
 * linear layer over the concatenation of a node's previous state and its
 * mean-aggregated message, then ReLU; hidden width 128 as in Section VI-A):
 *   y[r, o]   = sum_{k<d} W[o, k] h[r, k] + sum_{k<d} W[o, d + k] m[r, k]
 *   out[r, o] = max(y[r, o], 0)          r < n, o < d_out
 * on the tensor cores (fp32 inputs as tf32, bf16 inputs as bf16; fp32
 * accumulation).
 *   d_h       device [n_cap x dim], the dst rows' previous states (in a
 *             pipeline: the first n_dst rows of H_h, since V_{h-1} is a
 *             prefix of V_h)
 *   d_m       device [n_cap x dim], their aggregated messages (the output of
 *             sg_aggregate_fwd for the block)
 *   d_W       device [d_out x 2 dim] row-major, same dtype as d_h and d_m
 *   dtype     SG_F32 or SG_BF16 (of d_h, d_m and d_W)
 *   d_n       device int32 count (n = *d_n <= n_cap) or NULL (n = n_cap)
 *   dim       dim * element size a multiple of 16 bytes
 *   d_out     128
 *   d_out_act device [n_cap x d_out] fp32: rows r < n written
 *   d_y       device [n_cap x d_out] fp32 pre-activations, or NULL
 * All arrays 16-byte aligned; nothing is allocated. */
sg_status sg_sage_fwd(const void* d_h, const void* d_m, const void* d_W, int32_t dtype, int32_t n_cap,
                      const int32_t* d_n, int32_t dim, int32_t d_out, float* d_out_act, float* d_y,
                      sg_stream_t stream);

/* Backward of sg_sage_fwd for the loss gradient d_g = dL/dout (GraphSAGE's
 * layer as above; ReLU'(0) = 0):
 *   dY = g * (y > 0)
 *   dW[o, k]   = sum_{r<n} dY[r, o] z[r, k]         z = [h | m]
 *   dh[r, k]   = sum_o dY[r, o] W[o, k]             k < dim
 *   dm[r, k]   = sum_o dY[r, o] W[o, dim + k]
 * on the tensor cores (operands as in sg_sage_fwd; for bf16 inputs dY is
 * rounded to bf16).  dW sums over rows in a fixed order of splits, so the
 * result is deterministic.
 *   d_y, d_g  device [n_cap x d_out] fp32 (d_y: the forward's pre-activation)
 *   d_dW      device [d_out x 2 dim] fp32
 *   d_dh,d_dm device [n_cap x dim] fp32, rows r < n written
 *   d_workspace  device scratch of sg_sage_bwd_workspace(n_cap, dim, dtype)
 *             bytes, 256-byte aligned
 * Other arguments as in sg_sage_fwd. */
sg_status sg_sage_bwd(const void* d_h, const void* d_m, const void* d_W, int32_t dtype, int32_t n_cap,
                      const int32_t* d_n, int32_t dim, int32_t d_out, const float* d_y, const float* d_g, float* d_dW,
                      float* d_dh, float* d_dm, void* d_workspace, size_t workspace_bytes, sg_stream_t stream);

/* Bytes of the workspace of sg_sage_bwd; 0 on bad arguments. */
size_t sg_sage_bwd_workspace(int32_t n_cap, int32_t dim, int32_t dtype);

/* ------------------------------------------------------------ measurement */
/* Streams `bytes` of device-accessible memory at d_src with 16-byte loads
 * (a read roofline probe: HBM when d_src is device memory, the host link when
 * it is pinned host memory) and folds them into *d_sink (device uint32).
 * bytes must be a multiple of 16 and d_src 16-byte aligned. */
sg_status sg_read_probe(const void* d_src, int64_t bytes, uint32_t* d_sink, sg_stream_t stream);

/* Evaluates n_calls Philox4x32-10 blocks (the sampler's hash, counters
 * 0..n_calls-1 under `seed`) across the whole GPU and folds the outputs into
 * *d_sink (device uint32): the integer-throughput roofline of sampling. */
sg_status sg_hash_probe(int64_t n_calls, uint64_t seed, uint32_t* d_sink, sg_stream_t stream);

/* Exercises the bounded wait of the library's single-pass scans (decoupled
 * look-back) so that callers can check their timeout handling: n_tiles
 * blocks (1..4096) take tiles in order and each computes the exclusive
 * prefix of the values t + 1 over the tiles before it, written to d_out[t]
 * (device int32 [n_tiles]; t(t+1)/2 when every tile publishes).  The block
 * that takes tile `silent_tile` (or none, when it is outside [0, n_tiles))
 * exits without publishing, so every later tile's look-back that reaches it
 * polls spin_limit (1..2^22) times, gives up and sets SG_ERR_TIMEOUT in the
 * device error word, which the next sg_stream_check reports; the stream and
 * the library stay usable.  d_out[t] for t < silent_tile is exact; later
 * entries are not defined.  d_workspace: sg_wait_probe_workspace(n_tiles)
 * bytes, 256-byte aligned, cleared by the call.  No page defines this call:
 * it is a diagnostic of this library. */
size_t sg_wait_probe_workspace(int32_t n_tiles);
sg_status sg_wait_probe(int32_t n_tiles, int32_t silent_tile, int32_t spin_limit, void* d_workspace,
                        size_t workspace_bytes, int32_t* d_out, sg_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SG_H */

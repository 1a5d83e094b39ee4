// Opaque handle layouts shared by the library's translation units.
#pragma once

#include <stdint.h>

struct sg_graph {
    int64_t n_nodes = 0;
    int64_t n_edges = 0;
    int32_t offset_bits = 32;   // width of indptr entries (32 or 64)
    int64_t max_degree = 0;
    void* indptr = nullptr;     // device, n_nodes + 1 offsets
    int32_t* indices = nullptr; // device, n_edges
};

// The bounded dynamic cache beside the static one (GARDEN page, Section IV-B,
// Eq. (5)-(6)); see sg_dyncache.cu.
constexpr int kDynMaxWindow = 4096;
struct sg_dyn {
    int64_t k_dyn = 0;           // slots
    int32_t T = 1;               // batches per update window
    int32_t j = 0;               // batches of the current window so far
    uint32_t W[kDynMaxWindow];   // Q8 weight of batch j of a window
    uint32_t G_T = 0;            // gamma^T in Q16
    void* rows = nullptr;        // device, k_dyn x row_bytes
    int32_t* slot = nullptr;     // device, n_nodes: dynamic slot of a node or -1
    int32_t* nodes = nullptr;    // device, k_dyn: node in each slot or -1
    uint32_t* S = nullptr;       // device, n_nodes: scores (Q8)
    uint32_t* A = nullptr;       // device, n_nodes: the window's weighted counts
    uint32_t* sel = nullptr;     // device, 512 words: the Top-K selection (histogram, then its parameters)
    int32_t* lists = nullptr;    // device, 2 k_dyn + 8: new nodes, free slots, counters
};

struct sg_cache {
    int64_t n_nodes = 0;
    int32_t dim = 0;
    int32_t dtype = 0;
    int64_t row_bytes = 0;
    int64_t n_cache = 0;
    void* rows = nullptr;            // device, n_cache x row_bytes (slot order)
    int32_t* slot_of = nullptr;      // device, n_nodes: slot of a cached node, else -1; NULL: slot = ID for ID < n_cache
    const void* host_rows = nullptr; // device-usable address of the host table (may be NULL)
    int32_t region_shift = 0;        // log2 rows of a 2 MB host-table region; 0: misses read in row order
    int64_t n_regions = 0;           // regions of the host table when region_shift > 0
    sg_dyn* dyn = nullptr;           // optional dynamic cache (sg_dyn_cache_create)
};

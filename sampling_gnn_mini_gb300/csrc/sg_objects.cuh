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
};

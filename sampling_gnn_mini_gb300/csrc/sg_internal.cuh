// Internal helpers of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sg.h"

namespace sgi {

// ------------------------------------------------------------ host status
sg_status fail(sg_status s, const char* fmt, ...);
sg_status cuda_fail(cudaError_t e, const char* what);
int num_sms();             // SMs of the current device (cached per device)
bool is_device_ptr(const void* p);

#define SG_CUDA(call)                                                   \
    do {                                                                \
        cudaError_t sg_e_ = (call);                                     \
        if (sg_e_ != cudaSuccess) return ::sgi::cuda_fail(sg_e_, #call); \
    } while (0)

#define SG_CHECK_LAUNCH(what) SG_CUDA(cudaGetLastError())

// --------------------------------------------------------- device errors
// Each translation unit owns one sticky error word; sg_stream_check ORs them.
enum : unsigned { ERR_INDEX = 1u, ERR_CAPACITY = 2u, ERR_ARG = 4u, ERR_TIMEOUT = 8u };

// Each .cu file instantiates SGI_ERROR_WORD(tag): a static device word plus a
// host function that fetches and clears it.
#define SGI_ERROR_WORD(tag)                                                          \
    static __device__ unsigned int g_err_word;                                       \
    static __device__ __forceinline__ void dev_err(unsigned f) { atomicOr(&g_err_word, f); } \
    namespace sgi {                                                                  \
    unsigned fetch_err_##tag(cudaStream_t s) {                                       \
        unsigned v = 0, z = 0;                                                       \
        if (cudaMemcpyFromSymbolAsync(&v, g_err_word, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) \
            return 0x80000000u;                                                      \
        if (cudaMemcpyToSymbolAsync(g_err_word, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) \
            return 0x80000000u;                                                      \
        if (cudaStreamSynchronize(s) != cudaSuccess) return 0x80000000u;            \
        return v;                                                                    \
    }                                                                                \
    }

unsigned fetch_err_sampler(cudaStream_t);
unsigned fetch_err_gather(cudaStream_t);
unsigned fetch_err_aggregate(cudaStream_t);
unsigned fetch_err_api(cudaStream_t);
unsigned fetch_err_update(cudaStream_t);
unsigned fetch_err_recode(cudaStream_t);
unsigned fetch_err_dyncache(cudaStream_t);
unsigned fetch_err_match(cudaStream_t);

// ------------------------------------------------------------- ranking
// Nodes by descending 32-bit score, ties by ascending ID, into order[n]
// (sg_rank_by_score without argument checks); workspace of rank_ws_bytes(n)
// bytes, 256-byte aligned.
size_t rank_ws_bytes(int64_t n);
sg_status rank_scores(const uint32_t* score, int64_t n, int32_t* order, void* ws, cudaStream_t s);

// Frees a cache's dynamic cache, if any (sg_cache_destroy).
void dyn_cache_free(::sg_cache* c);

// ------------------------------------------------- allocation (owned memory)
// Every device allocation the library owns goes through dev_alloc.  With the
// environment variable SG_FAULT_INJECT=alloc:N (read once per process) the
// N-th such allocation fails as if the device were out of memory, without
// calling the CUDA runtime, so the OOM paths can be exercised on any host.
cudaError_t dev_alloc(void** p, size_t bytes);

// ------------------------------------------------------ dependent launches
// Kernels of the per-batch path are launched with programmatic stream
// serialization: a kernel may be scheduled while the previous kernel of the
// stream still runs, and griddepcontrol.wait holds it until that kernel has
// completed and its writes are visible.  Every such kernel calls pdl_start()
// first, before any early return, so a grid never completes ahead of the
// kernel before it (which keeps the usual stream order for the kernels after
// it).  No kernel triggers early: the next grid is scheduled as this one's
// blocks exit.
__device__ __forceinline__ void pdl_start() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------ arithmetic
__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 products whose halves are
// mixed with the other counter words and the round key; the key advances by
// the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_lo = 0xD2511F53u * c.x, a_hi = __umulhi(0xD2511F53u, c.x);
        const uint32_t b_lo = 0xCD9E8D57u * c.z, b_hi = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(b_hi ^ c.y ^ k0, b_lo, a_hi ^ c.w ^ k1, a_lo);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// ------------------------------------------------------------ warp / block
__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ unsigned lanemask_lt() { return (1u << lane_id()) - 1u; }

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T x) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, d);
        if ((int)lane_id() >= d) x += y;
    }
    return x;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(0xffffffffu, x, d);
    return x;
}

// Exclusive scan over a block of NT threads; every thread gets the block total.
// `sh` needs NT/32 + 1 entries; the call contains __syncthreads.
template <int NT, typename T>
__device__ __forceinline__ T block_excl_scan(T x, T* sh, T& total) {
    const int w = threadIdx.x >> 5;
    T inc = warp_incl_scan(x);
    if (lane_id() == 31) sh[w] = inc;
    __syncthreads();
    if (w == 0) {
        T v = (lane_id() < NT / 32) ? sh[lane_id()] : T(0);
        T s = warp_incl_scan(v);
        if (lane_id() < NT / 32) sh[lane_id()] = s - v;
        if (lane_id() == NT / 32 - 1) sh[NT / 32] = s;
    }
    __syncthreads();
    T r = sh[w] + inc - x;
    total = sh[NT / 32];
    __syncthreads();
    return r;
}

template <int NT, typename T>
__device__ __forceinline__ T block_sum(T x, T* sh) {
    T t;
    block_excl_scan<NT, T>(x, sh, t);
    return t;
}

// ------------------------------------------------- single-pass scan chains
// Tile status words: (state << 32) | value, state 1 aggregate, 2 inclusive
// prefix, anything else (a zeroed or all-ones word) empty.  A block publishes its tile's aggregate, then walks back
// over its predecessors until one has an inclusive prefix (decoupled
// look-back).  Tiles are handed out in increasing order by an atomic counter,
// so every predecessor belongs to a block that is already running; each wait
// is still bounded (kLookbackSpins polls), and *timed_out reports a wait that
// gave up.
constexpr int kLookbackSpins = 1 << 22;

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Exclusive prefix of tile t in the chain whose first tile is t0.  Called by
// all 32 lanes of one warp: the warp reads 32 predecessors at once, adds the
// aggregates up to the closest inclusive prefix, and moves the window back by
// 32 only while none is inclusive.  A predecessor still empty after
// spin_limit polls counts as an inclusive zero and sets *timed_out.
__device__ __forceinline__ int32_t chain_lookback(unsigned long long* status, int t, int t0, int32_t agg,
                                                  bool* timed_out, int spin_limit = kLookbackSpins) {
    const int lane = (int)lane_id();
    if (t == t0) {
        if (lane == 0) st_release(status + t, (2ull << 32) | (uint32_t)agg);
        return 0;
    }
    if (lane == 0) st_release(status + t, (1ull << 32) | (uint32_t)agg);
    int32_t excl = 0;
    for (int top = t - 1;; top -= 32) {
        const int p = top - lane;
        unsigned long long s = 2ull << 32;  // before the chain: an inclusive zero
        if (p >= t0) {
            int spins = 0;
            while (true) {
                s = ld_acquire(status + p);
                if ((s >> 32) == 1 || (s >> 32) == 2 || ++spins >= spin_limit) break;
                __nanosleep(32);
            }
            if ((s >> 32) != 1 && (s >> 32) != 2) {
                *timed_out = true;
                s = 2ull << 32;
            }
        }
        const unsigned incl = __ballot_sync(0xffffffffu, (s >> 32) == 2);
        const int first = incl ? __ffs(incl) - 1 : 31;
        excl += warp_sum(lane <= first ? (int32_t)(uint32_t)s : 0);
        if (incl) break;
    }
    if (lane == 0) st_release(status + t, (2ull << 32) | (uint32_t)(excl + agg));
    *timed_out = __any_sync(0xffffffffu, *timed_out);
    return excl;
}

// Contiguous segment [lo, hi) of n items owned by block b of g.
__device__ __forceinline__ void segment_of(int64_t n, int b, int g, int64_t& lo, int64_t& hi) {
    const int64_t len = (n + g - 1) / g;
    lo = (int64_t)b * len;
    hi = lo + len;
    if (lo > n) lo = n;
    if (hi > n) hi = n;
}

}  // namespace sgi

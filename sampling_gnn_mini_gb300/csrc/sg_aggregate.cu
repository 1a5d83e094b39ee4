// Mean aggregation over a sampled block, forward and backward (GARDEN page,
// Section II-A, Eq. (1) with AGGREGATE = mean; the backward map is its
// transpose).
//
// Both directions are one row-split sparse x dense product, y[r] = s_r *
// sum_{p in row r} w_p * x[col[p]]:
//   forward   rows = dst, col = src, w = 1,      s_r = 1 / c_r
//   backward  rows = src, col = dst, w = 1/c_dst, s_r = 1
// over the transposed block.  A group of LPR lanes owns one output row and
// keeps it in fp32 registers (VPL 16-byte vectors per lane), so every input
// row is read once per edge with coalesced 16-byte loads and every output row
// is written once (the FastGL explainer's Memory-Aware aggregation keeps
// partial sums on chip for the same reason).  No float atomics are used: the
// transpose is built by a sort of the edges by (src, edge index), so the
// summation order, and the result, are fixed.
#include <cuda_bf16.h>
#include <string.h>

#include "sg_internal.cuh"

SGI_ERROR_WORD(aggregate)

using namespace sgi;

namespace {

constexpr int kNT = 256;
constexpr int kWarpSortCap = 256;   // longest segment a warp sorts in shared memory
constexpr int kBlockSortCap = 4096; // longest segment a block sorts in shared memory
constexpr int kLongRow = 16;        // SpMM rows longer than this are summed by a whole warp

enum { DT_F32 = 0, DT_BF16 = 1, DT_BF16_F32 = 2 };  // input -> output types

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat16 x = __float2bfloat16_rn(a), y = __float2bfloat16_rn(b);
    return (uint32_t)__bfloat16_as_ushort(x) | ((uint32_t)__bfloat16_as_ushort(y) << 16);
}

template <int DT>
struct Elems { static constexpr int n = DT == DT_F32 ? 4 : 8; };

template <int DT>
__device__ __forceinline__ void fma_vec(float* acc, const uint4& v, float w) {
    if (DT == DT_F32) {
        acc[0] = fmaf(w, __uint_as_float(v.x), acc[0]);
        acc[1] = fmaf(w, __uint_as_float(v.y), acc[1]);
        acc[2] = fmaf(w, __uint_as_float(v.z), acc[2]);
        acc[3] = fmaf(w, __uint_as_float(v.w), acc[3]);
    } else {
        acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
        acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
        acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
        acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
        acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
        acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
        acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
        acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
    }
}

template <int DT>
__device__ __forceinline__ void add_vec(float* acc, const uint4& v) {
    if (DT == DT_F32) {
        acc[0] += __uint_as_float(v.x);
        acc[1] += __uint_as_float(v.y);
        acc[2] += __uint_as_float(v.z);
        acc[3] += __uint_as_float(v.w);
    } else {
        acc[0] += bf16_lo(v.x);
        acc[1] += bf16_hi(v.x);
        acc[2] += bf16_lo(v.y);
        acc[3] += bf16_hi(v.y);
        acc[4] += bf16_lo(v.z);
        acc[5] += bf16_hi(v.z);
        acc[6] += bf16_lo(v.w);
        acc[7] += bf16_hi(v.w);
    }
}

// Stores vector vi of output row r from acc (already scaled).
template <int DT>
__device__ __forceinline__ void store_vec(void* y, int64_t r, int32_t row_vecs, int vi, const float* a) {
    if (DT == DT_F32) {
        uint4* o = (uint4*)y + r * row_vecs + vi;
        *o = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
    } else if (DT == DT_BF16) {
        uint4* o = (uint4*)y + r * row_vecs + vi;
        *o = make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]), pack_bf16(a[6], a[7]));
    } else {
        uint4* o = (uint4*)y + (r * row_vecs + vi) * 2;
        o[0] = make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
        o[1] = make_uint4(__float_as_uint(a[4]), __float_as_uint(a[5]), __float_as_uint(a[6]), __float_as_uint(a[7]));
    }
}

// Adds to acc the edges of chunks lo + (first + k * stride) * LPR, k = 0, 1,
// ..., of row [lo, hi) (a chunk is LPR consecutive edges), for the group of
// LPR lanes named by gmask (this lane is gl): each lane holds VPL 16-byte
// vectors of the row (vector gl + p * LPR) and keeps UE edges in flight.
// With `pre` the column (and weight) of this lane's edge of the first chunk
// were loaded already (pcol, pw).
template <int LPR, int VPL, int DT, bool WEIGHTED>
__device__ __forceinline__ void accumulate_chunks(float (&acc)[VPL][Elems<DT>::n], int32_t lo, int32_t hi, int first,
                                                  int stride, const int32_t* __restrict__ col,
                                                  const float* __restrict__ w, int32_t n_cols,
                                                  const uint4* __restrict__ x, int32_t row_vecs, unsigned gmask,
                                                  int gl, bool pre = false, int32_t pcol = -1, float pw = 1.f) {
    constexpr int UE = VPL >= 8 ? 1 : (VPL == 4 ? 2 : 4);  // edges in flight per lane
    for (int32_t c0 = lo + first * LPR; c0 < hi; c0 += stride * LPR) {
        const int32_t my_e = c0 + gl;
        int32_t my_col = -1;
        float my_w = 1.f;
        if (pre && c0 == lo) {
            my_col = pcol;
            my_w = pw;
        } else if (my_e < hi) {
            my_col = __ldg(col + my_e);
            if (WEIGHTED) my_w = __ldg(w + my_e);
        }
        const int cnt = min(LPR, hi - c0);
        for (int t0 = 0; t0 < cnt; t0 += UE) {
            uint4 buf[UE][VPL];
            float wt[UE];
            bool ok[UE];
#pragma unroll
            for (int u = 0; u < UE; ++u) {
                const int t = t0 + u;
                const int32_t cu = __shfl_sync(gmask, my_col, t < cnt ? t : 0, LPR);
                wt[u] = WEIGHTED ? __shfl_sync(gmask, my_w, t < cnt ? t : 0, LPR) : 1.f;
                ok[u] = t < cnt && cu >= 0 && cu < n_cols;
                if (t < cnt && !ok[u] && gl == 0) dev_err(ERR_INDEX);
                const uint4* xr = x + (int64_t)(ok[u] ? cu : 0) * row_vecs;
#pragma unroll
                for (int p = 0; p < VPL; ++p) {
                    const int vi = gl + p * LPR;
                    buf[u][p] = (ok[u] && vi < row_vecs) ? __ldg(xr + vi) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < UE; ++u) {
                if (!ok[u]) continue;
#pragma unroll
                for (int p = 0; p < VPL; ++p) {
                    if (WEIGHTED) fma_vec<DT>(acc[p], buf[u][p], wt[u]);
                    else add_vec<DT>(acc[p], buf[u][p]);
                }
            }
        }
    }
}

// Scales and stores output row r from the group's accumulators (the mean
// multiplies by 1 / c: within one rounding of the quotient).
template <int LPR, int VPL, int DT, bool WEIGHTED>
__device__ __forceinline__ void store_row(const float (&acc)[VPL][Elems<DT>::n], int64_t r, int32_t c, void* y,
                                          int32_t row_vecs, int gl) {
    constexpr int EPV = Elems<DT>::n;
    const float rc = WEIGHTED ? 1.f : (c > 0 ? __frcp_rn((float)c) : 0.f);
#pragma unroll
    for (int p = 0; p < VPL; ++p) {
        const int vi = gl + p * LPR;
        if (vi >= row_vecs) continue;
        float o[EPV];
#pragma unroll
        for (int q = 0; q < EPV; ++q) o[q] = WEIGHTED ? acc[p][q] : acc[p][q] * rc;
        store_vec<DT>(y, r, row_vecs, vi, o);
    }
}

// Row r = [rlo, rhi), longer than kLongRow edges, summed by the whole warp:
// the warp's 32 / LPR groups take every (32 / LPR)-th chunk of the row and
// their sums are added in a fixed order (xor shuffles by LPR, 2 LPR, ...), so
// the result does not depend on which warp sums the row.
template <int LPR, int VPL, int DT, bool WEIGHTED>
__device__ __forceinline__ void long_row(int64_t r, int32_t rlo, int32_t rhi, const int32_t* __restrict__ col,
                                         const float* __restrict__ w, int32_t n_cols, const uint4* __restrict__ x,
                                         int32_t row_vecs, void* __restrict__ y) {
    constexpr int EPV = Elems<DT>::n;
    constexpr int SG = 32 / LPR;
    const unsigned lane = lane_id();
    const int gl = lane % LPR, sg = (int)(lane / LPR);
    const unsigned gmask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << (lane - gl));
    float acc[VPL][EPV];
#pragma unroll
    for (int p = 0; p < VPL; ++p)
#pragma unroll
        for (int q = 0; q < EPV; ++q) acc[p][q] = 0.f;
    accumulate_chunks<LPR, VPL, DT, WEIGHTED>(acc, rlo, rhi, sg, SG, col, w, n_cols, x, row_vecs, gmask, gl);
#pragma unroll
    for (int d = LPR; d < 32; d <<= 1)
#pragma unroll
        for (int p = 0; p < VPL; ++p)
#pragma unroll
            for (int q = 0; q < EPV; ++q) acc[p][q] += __shfl_xor_sync(0xffffffffu, acc[p][q], d);
    if (sg == 0) store_row<LPR, VPL, DT, WEIGHTED>(acc, r, rhi - rlo, y, row_vecs, gl);
}

// Rows longer than kLongRow edges among the rows of this warp's groups (group
// g owns rows g, g + groups, ...), found by a pass over their bounds ahead of
// the other rows and summed one at a time by the whole warp.
template <int LPR, int VPL, int DT, bool WEIGHTED>
__device__ __forceinline__ void long_rows(const int32_t* __restrict__ ptr, const int32_t* __restrict__ col,
                                          const float* __restrict__ w, int64_t n_rows, int32_t n_cols,
                                          const uint4* __restrict__ x, int32_t row_vecs, void* __restrict__ y,
                                          int64_t gid, int64_t groups) {
    const unsigned lane = lane_id();
    const int gl = lane % LPR, sg = (int)(lane / LPR);
    constexpr int kAhead = 4;  // row bounds of this many rounds are loaded together
    for (int64_t base0 = gid - sg; base0 < n_rows; base0 += kAhead * groups) {
      int32_t lob[kAhead], hib[kAhead];
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
          const int64_t rr = base0 + u * groups + sg;
          lob[u] = 0;
          hib[u] = 0;
          if (rr < n_rows) {
              lob[u] = ptr[rr];
              hib[u] = ptr[rr + 1];
          }
      }
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        const int64_t base = base0 + u * groups;
        const int32_t lo = lob[u], hi = hib[u];
        unsigned longs = __ballot_sync(0xffffffffu, gl == 0 && hi - lo > kLongRow);
        while (longs) {
            const int src = __ffs(longs) - 1;
            longs &= longs - 1;
            const int32_t rlo = __shfl_sync(0xffffffffu, lo, src), rhi = __shfl_sync(0xffffffffu, hi, src);
            long_row<LPR, VPL, DT, WEIGHTED>(base + src / LPR, rlo, rhi, col, w, n_cols, x, row_vecs, y);
        }
      }
    }
}

// y[r] = scale_r * sum_p w_p x[col[p]] for r < n_rows (see the file comment).
// WEIGHTED = false: w_p = 1 and scale_r = 1 / row length (forward mean).
// WEIGHTED = true:  w_p = w[p] and scale_r = 1 (backward over the transpose).
// A warp holds 32 / LPR groups, and group g of the grid owns rows g, g +
// groups, ...; every group sums its rows alone, in edge order.  Rows longer
// than kLongRow edges (hubs of a transposed block) are summed by a whole warp
// instead (long_row), so a long row is no longer a serial tail.  With
// long_cap > 0 a group that meets one appends it to a list in shared memory
// (long_cap entries: at least the rows of the block's groups) and the block's
// warps sum the list once every group is done; with long_cap = 0 a pass over
// the bounds finds them first.  Three blocks fit on an SM for fp32 rows, two
// for bf16 (twice the accumulators).
template <int LPR, int VPL, int DT, bool WEIGHTED>
__global__ void __launch_bounds__(kNT, DT == DT_F32 ? 3 : 2)
    k_spmm(const int32_t* __restrict__ ptr, const int32_t* __restrict__ col, const float* __restrict__ w,
           int32_t n_rows_cap, const int32_t* __restrict__ d_rows, int32_t n_cols_cap,
           const int32_t* __restrict__ d_cols, const uint4* __restrict__ x, int32_t row_vecs, void* __restrict__ y,
           int32_t long_cap) {
    extern __shared__ int32_t s_long[];  // long_cap row indices
    __shared__ int32_t s_nlong;
    pdl_start();
    constexpr int EPV = Elems<DT>::n;
    constexpr int SG = 32 / LPR;  // groups per warp
    const int64_t n_rows = d_rows ? (int64_t)min(*d_rows, n_rows_cap) : n_rows_cap;
    const int32_t n_cols = d_cols ? min(*d_cols, n_cols_cap) : n_cols_cap;
    const unsigned lane = lane_id();
    const int gl = lane % LPR;
    // the LPR lanes of a group share a row (and so every loop trip count);
    // shuffles name only them, so groups of one warp proceed independently
    const unsigned gmask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << (lane - gl));
    const int64_t groups = (int64_t)gridDim.x * (kNT / LPR);
    const int64_t gid = (blockIdx.x * (int64_t)kNT + threadIdx.x) / LPR;
    const bool defer = SG > 1 && long_cap > 0;  // the same in every thread
    if (defer) {
        if (threadIdx.x == 0) s_nlong = 0;
        __syncthreads();
    } else if (SG > 1) {
        long_rows<LPR, VPL, DT, WEIGHTED>(ptr, col, w, n_rows, n_cols, x, row_vecs, y, gid, groups);
    }
    // the rows of this group.  Row bounds are loaded two rows ahead and the
    // first chunk's columns one row ahead, so a row's feature loads start
    // without waiting for its indices.
    int64_t r = gid;
    int32_t lo1 = 0, hi1 = 0, lo2 = 0, hi2 = 0;  // bounds of rows r and r + groups
    if (r < n_rows) {
        lo1 = ptr[r];
        hi1 = ptr[r + 1];
    }
    if (r + groups < n_rows) {
        lo2 = ptr[r + groups];
        hi2 = ptr[r + groups + 1];
    }
    int32_t c1 = -1;  // this lane's first-chunk column (and weight) of row r
    float w1 = 1.f;
    if (lo1 + gl < hi1) {
        c1 = __ldg(col + lo1 + gl);
        if (WEIGHTED) w1 = __ldg(w + lo1 + gl);
    }
    for (; r < n_rows; r += groups) {
        const int32_t lo = lo1, hi = hi1, fc = c1;
        const float fw = w1;
        lo1 = lo2;
        hi1 = hi2;
        c1 = -1;
        w1 = 1.f;
        if (r + groups < n_rows && lo1 + gl < hi1) {
            c1 = __ldg(col + lo1 + gl);
            if (WEIGHTED) w1 = __ldg(w + lo1 + gl);
        }
        if (r + 2 * groups < n_rows) {
            lo2 = ptr[r + 2 * groups];
            hi2 = ptr[r + 2 * groups + 1];
        }
        if (SG > 1 && hi - lo > kLongRow) {
            if (defer && gl == 0) {
                const int32_t k = atomicAdd(&s_nlong, 1);
                if (k < long_cap) s_long[k] = (int32_t)r;
                else dev_err(ERR_CAPACITY);
            }
            continue;
        }
        float acc[VPL][EPV];
#pragma unroll
        for (int p = 0; p < VPL; ++p)
#pragma unroll
            for (int q = 0; q < EPV; ++q) acc[p][q] = 0.f;
        accumulate_chunks<LPR, VPL, DT, WEIGHTED>(acc, lo, hi, 0, 1, col, w, n_cols, x, row_vecs, gmask, gl, true, fc, fw);
        store_row<LPR, VPL, DT, WEIGHTED>(acc, r, hi - lo, y, row_vecs, gl);
    }
    if (defer) {
        __syncthreads();
        const int32_t n_long = min(s_nlong, long_cap);
        for (int32_t i = (int32_t)(threadIdx.x / 32); i < n_long; i += kNT / 32) {
            const int32_t rr = s_long[i];
            long_row<LPR, VPL, DT, WEIGHTED>(rr, ptr[rr], ptr[rr + 1], col, w, n_cols, x, row_vecs, y);
        }
    }
}

// ------------------------------------------------------- copy-engine SpMM
// The same product with the feature rows brought into shared memory by the
// copy engine: one cp.async.bulk per edge moves a whole source row and
// completes on the mbarrier of its slot.  A warp owns a contiguous range of
// rows, so its edges are one run of the CSR, and walks the run in stages of
// C edges.  A ring of kTmaStages stage buffers keeps kTmaStages - 1 stages of
// copies in flight ahead of the one being summed (columns load one stage
// before their copies are issued); lane v adds up vectors v, v + 32, ... of
// the current row and rows end where the edge index reaches the next row
// pointer (32 row pointers in a register, the next 32 already loading).  The
// parity each slot's mbarrier is next waited on is kept in a bitmask (the same
// in every lane), so stages that leave slots unused keep no stale phase.
// Every wait on an mbarrier is bounded: a wait that gives up sets the error
// word (SG_ERR_TIMEOUT), and the warp then waits (bounded) for its copies
// still in flight before it exits.
constexpr int kTmaWarps = 4;        // warps per block
constexpr int kTmaStages = 6;       // stage buffers per warp
constexpr int kTmaStageMax = 8;     // edges per stage at most (slots per warp <= 48)
constexpr int kTmaSpins = 1 << 16;  // polls of one mbarrier before giving up
constexpr int kTmaRowsMax = 4096;   // forward blocks up to this many rows take this path

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// true once the phase of the given parity has completed; false after
// kTmaSpins polls
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (int i = 0; i < kTmaSpins; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
// bytes (a multiple of 16) from 16-byte aligned global src to shared dst,
// completing on bar
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Shared memory of one warp: kTmaStages * C slots of row_bytes, then as many
// mbarriers, weights and validity flags.
__host__ __device__ __forceinline__ size_t tma_warp_bytes(int C, int row_bytes) {
    return (size_t)kTmaStages * C * row_bytes + (size_t)kTmaStages * C * (8 + 4 + 4);
}

template <int VPL, int DT, bool WEIGHTED>
__global__ void __launch_bounds__(32 * kTmaWarps) k_spmm_tma(
    const int32_t* __restrict__ ptr, const int32_t* __restrict__ col, const float* __restrict__ w, int32_t n_rows_cap,
    const int32_t* __restrict__ d_rows, int32_t n_cols_cap, const int32_t* __restrict__ d_cols,
    const uint4* __restrict__ x, int32_t row_vecs, int32_t C, void* __restrict__ y) {
    pdl_start();
    constexpr int EPV = Elems<DT>::n;
    constexpr int NS = kTmaStages;
    extern __shared__ __align__(16) unsigned char tsm[];
    const int64_t n_rows = d_rows ? (int64_t)min(*d_rows, n_rows_cap) : n_rows_cap;
    const int32_t n_cols = d_cols ? min(*d_cols, n_cols_cap) : n_cols_cap;
    const int lane = (int)lane_id();
    const int wib = threadIdx.x >> 5;
    const int row_bytes = row_vecs * 16;
    const int S = NS * C;  // slots
    unsigned char* base = tsm + (size_t)wib * tma_warp_bytes(C, row_bytes);
    uint4* slots = (uint4*)base;
    uint64_t* bars = (uint64_t*)(base + (size_t)S * row_bytes);
    float* sw = (float*)(bars + S);
    int32_t* sval = (int32_t*)(sw + S);
    for (int i = lane; i < S; i += 32) mbar_init(bars + i);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    __syncwarp();

    const int64_t n_warps = (int64_t)gridDim.x * kTmaWarps;
    const int64_t per = (n_rows + n_warps - 1) / n_warps;
    const int64_t ra = min(((int64_t)blockIdx.x * kTmaWarps + wib) * per, n_rows);
    const int64_t rb = min(ra + per, n_rows);
    if (ra >= rb) return;
    const int32_t E0 = ptr[ra], E1 = ptr[rb];
    const int32_t n_st = (E1 - E0 + C - 1) / C;
    uint64_t phase = 0;    // bit i: parity of slot i's next completion
    uint64_t pending = 0;  // bit i: a copy into slot i was issued and not yet waited on

    // columns (and weights) of stage s are held by lanes k < C (edge E0 + s C + k)
    auto load_col = [&](int32_t s, int32_t& c, float& wt) {
        const int32_t e = E0 + s * C + lane;
        c = -1;
        wt = 0.f;
        if (lane < C && s < n_st && e < E1) {
            c = __ldg(col + e);
            if (WEIGHTED) wt = __ldg(w + e);
        }
    };
    auto issue = [&](int32_t s, int32_t c, float wt) {
        if (s >= n_st) return;
        const int grp = s % NS;
        const int n_e = min(C, E1 - (E0 + s * C));
        pending |= ((1ull << n_e) - 1ull) << (grp * C);
        if (lane < n_e) {
            const int slot = grp * C + lane;
            uint64_t* bar = bars + slot;
            if (c >= 0 && c < n_cols) {
                sval[slot] = 1;
                if (WEIGHTED) sw[slot] = wt;
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // earlier reads of the slot first
                mbar_expect_tx(bar, (uint32_t)row_bytes);
                bulk_copy(slots + (size_t)slot * row_vecs, x + (int64_t)c * row_vecs, (uint32_t)row_bytes, bar);
            } else {
                dev_err(ERR_INDEX);
                sval[slot] = 0;
                mbar_arrive(bar);
            }
        }
    };
    // stages 0 .. NS-2 (at most 40 edges): their columns in two loads a lane
    {
        const int span = (NS - 1) * C;
        int32_t ca = -1, cb = -1;
        float wa = 0.f, wb = 0.f;
        if (lane < span && E0 + lane < E1) {
            ca = __ldg(col + E0 + lane);
            if (WEIGHTED) wa = __ldg(w + E0 + lane);
        }
        if (lane + 32 < span && E0 + lane + 32 < E1) {
            cb = __ldg(col + E0 + lane + 32);
            if (WEIGHTED) wb = __ldg(w + E0 + lane + 32);
        }
        for (int s = 0; s < NS - 1; ++s) {
            const int src = s * C + lane;  // this lane's edge of stage s, as a position of the first span
            const int32_t c_lo = __shfl_sync(0xffffffffu, ca, src & 31), c_hi = __shfl_sync(0xffffffffu, cb, src & 31);
            const float w_lo = __shfl_sync(0xffffffffu, wa, src & 31), w_hi = __shfl_sync(0xffffffffu, wb, src & 31);
            issue(s, src < 32 ? c_lo : c_hi, src < 32 ? w_lo : w_hi);
        }
    }
    int32_t cn;
    float wn;
    load_col(NS - 1, cn, wn);

    // row ends: lane i of pcur holds ptr[pb + i]; pnext the next 32
    int64_t pb = ra + 1;
    int32_t pcur = pb + lane <= rb ? ptr[pb + lane] : E1;
    int32_t pnext = pb + 32 + lane <= rb ? ptr[pb + 32 + lane] : E1;
    int64_t r = ra;
    int32_t rstart = E0;
    int32_t rend = __shfl_sync(0xffffffffu, pcur, 0);
    float acc[VPL][EPV];
#pragma unroll
    for (int p = 0; p < VPL; ++p)
#pragma unroll
        for (int q = 0; q < EPV; ++q) acc[p][q] = 0.f;
    auto finish_row = [&]() {
        const int32_t cnt = rend - rstart;
        const float rc = WEIGHTED ? 1.f : (cnt > 0 ? __frcp_rn((float)cnt) : 0.f);
#pragma unroll
        for (int p = 0; p < VPL; ++p) {
            const int vi = lane + 32 * p;
            if (vi < row_vecs) {
                float o[EPV];
#pragma unroll
                for (int q = 0; q < EPV; ++q) o[q] = WEIGHTED ? acc[p][q] : acc[p][q] * rc;
                store_vec<DT>(y, r, row_vecs, vi, o);
            }
#pragma unroll
            for (int q = 0; q < EPV; ++q) acc[p][q] = 0.f;
        }
        ++r;
        rstart = rend;
        if (r + 1 - pb == 32) {
            pb += 32;
            pcur = pnext;
            pnext = pb + 32 + lane <= rb ? ptr[pb + 32 + lane] : E1;
        }
        rend = r < rb ? __shfl_sync(0xffffffffu, pcur, (int)((r + 1 - pb) & 31)) : E1;
    };

    bool failed = false;
    for (int32_t st = 0; st < n_st; ++st) {
        issue(st + NS - 1, cn, wn);  // into the buffer that stage st - 1 has freed
        load_col(st + NS, cn, wn);
        const int grp = st % NS;
        const int32_t e0 = E0 + st * C;
        const int n_e = min(C, E1 - e0);
        bool ok = true;
        for (int k = 0; k < n_e; ++k) ok &= mbar_wait(bars + grp * C + k, (uint32_t)((phase >> (grp * C + k)) & 1ull));
        if (!__all_sync(0xffffffffu, ok)) {  // (this stage's slots stay pending for the drain below)
            if (lane == 0) dev_err(ERR_TIMEOUT);
            failed = true;
            break;
        }
        const uint64_t used = ((1ull << n_e) - 1ull) << (grp * C);
        phase ^= used;
        pending &= ~used;
        for (int k = 0; k < n_e; ++k) {
            while (e0 + k >= rend) finish_row();
            const int slot = grp * C + k;
            if (!sval[slot]) continue;
            const float wt = WEIGHTED ? sw[slot] : 1.f;
            const uint4* sb = slots + (size_t)slot * row_vecs;
#pragma unroll
            for (int p = 0; p < VPL; ++p) {
                const int vi = lane + 32 * p;
                if (vi < row_vecs) {
                    const uint4 v = sb[vi];
                    if (WEIGHTED) fma_vec<DT>(acc[p], v, wt);
                    else add_vec<DT>(acc[p], v);
                }
            }
        }
        __syncwarp();
    }
    if (failed) {  // let this warp's copies in flight land before it exits (bounded)
        for (int i = lane; i < S; i += 32)
            if ((pending >> i) & 1ull) (void)mbar_wait(bars + i, (uint32_t)((phase >> i) & 1ull));
        return;
    }
    while (r < rb) finish_row();
}

// Element-wise variant for rows whose byte size is not a multiple of 16 or is
// larger than 4 KB: a warp per row, lanes over the elements.
__global__ void __launch_bounds__(kNT) k_spmm_scalar(const int32_t* __restrict__ ptr, const int32_t* __restrict__ col,
                                                     const float* __restrict__ w, int32_t n_rows_cap,
                                                     const int32_t* __restrict__ d_rows, int32_t n_cols_cap,
                                                     const int32_t* __restrict__ d_cols, const void* __restrict__ x,
                                                     int32_t dim, int dt, void* __restrict__ y) {
    pdl_start();
    const int64_t n_rows = d_rows ? (int64_t)min(*d_rows, n_rows_cap) : n_rows_cap;
    const int32_t n_cols = d_cols ? min(*d_cols, n_cols_cap) : n_cols_cap;
    const int64_t warps = (int64_t)gridDim.x * (kNT / 32);
    for (int64_t r = (blockIdx.x * (int64_t)kNT + threadIdx.x) / 32; r < n_rows; r += warps) {
        const int32_t lo = ptr[r], hi = ptr[r + 1];
        for (int32_t k = lane_id(); k < dim; k += 32) {
            float acc = 0.f;
            for (int32_t p = lo; p < hi; ++p) {
                const int32_t cu = col[p];
                if (cu < 0 || cu >= n_cols) {
                    if (k == 0) dev_err(ERR_INDEX);
                    continue;
                }
                const int64_t at = (int64_t)cu * dim + k;
                const float v = dt == DT_F32 ? ((const float*)x)[at]
                                             : __uint_as_float((uint32_t)((const uint16_t*)x)[at] << 16);
                acc = w ? fmaf(w[p], v, acc) : acc + v;
            }
            const float o = w ? acc : (hi > lo ? __fdiv_rn(acc, (float)(hi - lo)) : 0.f);
            const int64_t at = r * dim + k;
            if (dt == DT_BF16) ((__nv_bfloat16*)y)[at] = __float2bfloat16_rn(o);
            else ((float*)y)[at] = o;
        }
    }
}

// --------------------------------------------------------------- transpose
// The backward pass needs each block's edges grouped by src row, in edge
// order inside a group.  All blocks of a set (the hops of one mini-batch) are
// transposed by the same five launches; blockIdx.y selects the block.
//   k_tcount   edges per src row (integer atomics: the counts are exact)
//   k_tscan    row pointer of the transposed block (single-pass look-back)
//   k_tscatter every edge into its src segment (order fixed by the sort)
//   k_tsort    short segments sorted by edge index by one warp; long ones listed
//   k_tsort_long  long segments sorted by a block (bitonic network)
// The outputs per edge are the dst row and the weight 1 / c_dst.
struct TSet {
    int nb;
    const int32_t* indptr[SG_MAX_HOPS];
    const int32_t* idx[SG_MAX_HOPS];
    int32_t n_dst_cap[SG_MAX_HOPS], n_src_cap[SG_MAX_HOPS];
    const int32_t* dims[SG_MAX_HOPS];          // device {n_dst, n_src} or NULL
    int32_t* tcnt[SG_MAX_HOPS];                // [n_src_cap + 1], zeroed
    int32_t* tptr[SG_MAX_HOPS];                // [n_src_cap + 1] output
    int32_t* tkey[SG_MAX_HOPS];                // [edges] scratch
    int32_t* dst_of[SG_MAX_HOPS];              // [edges] scratch
    int32_t* tdst[SG_MAX_HOPS];                // [edges] output
    float* tw[SG_MAX_HOPS];                    // [edges] output
    unsigned long long* status[SG_MAX_HOPS];   // scan chain, zeroed
    int32_t* long_list[SG_MAX_HOPS];           // [n_src_cap]
    uint32_t* ctr;                             // [2 * SG_MAX_HOPS]: tile counter, long count; zeroed
};

__device__ __forceinline__ int32_t set_n_dst(const TSet& t, int b) {
    return t.dims[b] ? min(t.dims[b][0], t.n_dst_cap[b]) : t.n_dst_cap[b];
}
__device__ __forceinline__ int32_t set_n_src(const TSet& t, int b) {
    return t.dims[b] ? min(t.dims[b][1], t.n_src_cap[b]) : t.n_src_cap[b];
}

__global__ void k_tcount(TSet t) {
    pdl_start();
    const int b = blockIdx.y;
    const int32_t E = t.indptr[b][set_n_dst(t, b)];
    const int32_t n_src = set_n_src(t, b);
    const int32_t* idx = t.idx[b];
    int32_t* tcnt = t.tcnt[b];
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < E; e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t u = idx[e];
        if (u >= 0 && u < n_src) atomicAdd(tcnt + u, 1);
        else dev_err(ERR_INDEX);
    }
}

constexpr int kTTile = 1024;  // entries per scan tile (4 per thread)

// Exclusive scan of tcnt[0, n_src] into tptr[0, n_src] (tptr[n_src] = E).
__global__ void __launch_bounds__(kNT) k_tscan(TSet t) {
    pdl_start();
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ int32_t s_tile, s_excl;
    const int b = blockIdx.y;
    const int64_t n = (int64_t)set_n_src(t, b) + 1;
    const int64_t n_tiles = (n + kTTile - 1) / kTTile;
    if ((int64_t)blockIdx.x >= n_tiles) return;
    for (int iter = 0;; ++iter) {
        if (iter > 0 && (int64_t)gridDim.x >= n_tiles) break;
        if (threadIdx.x == 0) s_tile = (int32_t)atomicAdd(t.ctr + 2 * b, 1u);
        __syncthreads();
        const int64_t tile = s_tile;
        if (tile >= n_tiles) break;
        const int64_t i0 = tile * kTTile + (int64_t)threadIdx.x * 4;
        int32_t v[4], mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q] = i0 + q < n ? t.tcnt[b][i0 + q] : 0;
            mine += v[q];
        }
        int32_t total;
        const int32_t ex = block_excl_scan<kNT>(mine, red, total);
        if (threadIdx.x < 32) {
            bool late = false;
            const int32_t x = chain_lookback(t.status[b], (int)tile, 0, total, &late);
            if (threadIdx.x == 0) {
                s_excl = x;
                if (late) dev_err(ERR_TIMEOUT);
            }
        }
        __syncthreads();
        int32_t run = s_excl + ex;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (i0 + q < n) t.tptr[b][i0 + q] = run;
            run += v[q];
        }
        __syncthreads();
    }
}

// Places every edge in its src segment and records the edge's dst row.
__global__ void k_tscatter(TSet t) {
    pdl_start();
    const int b = blockIdx.y;
    const int32_t n_dst = set_n_dst(t, b), n_src = set_n_src(t, b);
    const int32_t* indptr = t.indptr[b];
    const int32_t* idx = t.idx[b];
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t v = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; v < n_dst; v += warps) {
        const int32_t lo = indptr[v], hi = indptr[v + 1];
        for (int32_t e = lo + (int32_t)lane_id(); e < hi; e += 32) {
            const int32_t u = idx[e];
            t.dst_of[b][e] = (int32_t)v;
            if (u < 0 || u >= n_src) continue;
            const int32_t p = t.tptr[b][u] + atomicSub(t.tcnt[b] + u, 1) - 1;
            t.tkey[b][p] = e;
        }
    }
}

__device__ __forceinline__ void emit_transposed(const int32_t* indptr, const int32_t* dst_of, int32_t e, int32_t p,
                                                int32_t* tdst, float* tw) {
    const int32_t v = dst_of[e];
    tdst[p] = v;
    tw[p] = 1.0f / (float)(indptr[v + 1] - indptr[v]);
}

// Sorts each src segment by edge index.  Segments up to kWarpSortCap are
// ranked by one warp; longer ones go to the block's list for k_tsort_long.
__global__ void __launch_bounds__(kNT) k_tsort(TSet t) {
    pdl_start();
    __shared__ int32_t sk[kNT / 32][kWarpSortCap];
    const int b = blockIdx.y;
    const int32_t n_src = set_n_src(t, b);
    const int32_t* tptr = t.tptr[b];
    const int32_t* tkey = t.tkey[b];
    const int32_t* dst_of = t.dst_of[b];
    const int32_t* indptr = t.indptr[b];
    const int wib = threadIdx.x >> 5;
    const unsigned lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (kNT / 32);
    for (int64_t u = blockIdx.x * (int64_t)(kNT / 32) + wib; u < n_src; u += warps) {
        const int32_t lo = tptr[u], len = tptr[u + 1] - lo;
        if (len == 0) continue;
        if (len <= 32) {
            const int32_t key = (int)lane < len ? tkey[lo + lane] : 0x7FFFFFFF;
            int rank = 0;
            for (int q = 0; q < len; ++q) rank += __shfl_sync(0xffffffffu, key, q) < key;
            if ((int)lane < len) emit_transposed(indptr, dst_of, key, lo + rank, t.tdst[b], t.tw[b]);
        } else if (len <= kWarpSortCap) {
            int32_t* sw = sk[wib];
            for (int q = lane; q < len; q += 32) sw[q] = tkey[lo + q];
            __syncwarp();
            for (int i = lane; i < len; i += 32) {
                const int32_t key = sw[i];
                int rank = 0;
                for (int q = 0; q < len; ++q) rank += sw[q] < key;
                emit_transposed(indptr, dst_of, key, lo + rank, t.tdst[b], t.tw[b]);
            }
            __syncwarp();
        } else if (lane == 0) {
            t.long_list[b][atomicAdd(t.ctr + 2 * b + 1, 1u)] = (int32_t)u;
        }
    }
}

// Ascending sort of keys[0, len) by one block: a bitonic network in which every
// comparator puts the smaller key first (the first step of each merge stage
// compares mirrored positions), so positions >= len act as +infinity and need
// no storage.  Works on shared or global memory.
__device__ void block_bitonic_sort(int32_t* keys, int32_t len) {
    int32_t P = 1;
    while (P < len) P <<= 1;
    for (int32_t k = 2; k <= P; k <<= 1) {
        for (int32_t i = threadIdx.x; i < P / 2; i += blockDim.x) {
            const int32_t half = k >> 1;
            const int32_t lo = (i / half) * k + (i % half);
            const int32_t hi = (i / half) * k + (k - 1 - (i % half));
            if (hi < len) {
                const int32_t x = keys[lo], y = keys[hi];
                if (y < x) { keys[lo] = y; keys[hi] = x; }
            }
        }
        __syncthreads();
        for (int32_t j = k >> 2; j > 0; j >>= 1) {
            for (int32_t i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int32_t lo = (i / j) * (2 * j) + (i % j);
                const int32_t hi = lo + j;
                if (hi < len) {
                    const int32_t x = keys[lo], y = keys[hi];
                    if (y < x) { keys[lo] = y; keys[hi] = x; }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kNT) k_tsort_long(TSet t) {
    pdl_start();
    __shared__ int32_t sk[kBlockSortCap];
    const int b = blockIdx.y;
    const int32_t n = (int32_t)t.ctr[2 * b + 1];
    for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t u = t.long_list[b][i];
        const int32_t lo = t.tptr[b][u], len = t.tptr[b][u + 1] - lo;
        int32_t* keys;
        if (len <= kBlockSortCap) {
            for (int32_t q = threadIdx.x; q < len; q += blockDim.x) sk[q] = t.tkey[b][lo + q];
            keys = sk;
        } else {
            keys = t.tkey[b] + lo;  // long segment: sort in place in global memory
        }
        __syncthreads();
        block_bitonic_sort(keys, len);
        for (int32_t q = threadIdx.x; q < len; q += blockDim.x)
            emit_transposed(t.indptr[b], t.dst_of[b], keys[q], lo + q, t.tdst[b], t.tw[b]);
        __syncthreads();
    }
}

// ------------------------------------------------------------------- host
int dt_code(int32_t in, int32_t out) {
    if (in == SG_F32 && out == SG_F32) return DT_F32;
    if (in == SG_BF16 && out == SG_BF16) return DT_BF16;
    if (in == SG_BF16 && out == SG_F32) return DT_BF16_F32;
    return -1;
}

constexpr int kLongListBytes = 16384;  // shared-memory list of long rows a block, at most

// k_spmm with LPR = L, VPL = V, no more groups than rows.  Forward: a grid
// of what fits on the GPU at once, and the long-row list when the rows of a
// block's groups fit kLongListBytes.  Backward (weighted, the transposed
// blocks, whose hubs make long rows common): up to 8 blocks an SM in waves
// and the pass over the bounds, which start the long rows first (measured
// faster there: a list summed at the end of a block leaves a tail).
template <int L, int V, int DT, bool WGT>
sg_status launch_spmm_lv(cudaStream_t s, const int32_t* ptr, const int32_t* col, const float* w, int32_t nr,
                         const int32_t* dr, int32_t nc, const int32_t* dc, const void* x, int32_t rv, void* y) {
    static int per_sm = 0;  // resident blocks an SM with the largest list (occupancy calculator, once)
    if (per_sm == 0) {
        int p = 0;
        SG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p, k_spmm<L, V, DT, WGT>, kNT, kLongListBytes));
        per_sm = p > 0 ? p : 1;
    }
    int64_t blocks = (int64_t)(WGT ? 8 : per_sm) * num_sms();
    const int64_t need = cdiv((int64_t)nr * L, kNT);
    if (blocks > need) blocks = need;
    if (blocks < 1) blocks = 1;
    int32_t long_cap = 0;
    if (!WGT && L < 32) {
        const int64_t per_block = kNT / L;  // groups
        const int64_t cap = per_block * cdiv((int64_t)nr, blocks * per_block);
        if (cap * (int64_t)sizeof(int32_t) <= kLongListBytes) long_cap = (int32_t)cap;
    }
    SG_CUDA(launch_pdl(k_spmm<L, V, DT, WGT>, dim3((unsigned)blocks), dim3(kNT), (size_t)long_cap * sizeof(int32_t), s,
                       ptr, col, w, nr, dr, nc, dc, (const uint4*)x, rv, y, long_cap));
    return SG_OK;
}

template <int DT, bool WGT>
sg_status launch_vec(int lpr, int vpl, cudaStream_t s, const int32_t* ptr, const int32_t* col, const float* w,
                     int32_t nr, const int32_t* dr, int32_t nc, const int32_t* dc, const void* x, int32_t rv, void* y) {
#define SG_SPMM(L, V) return launch_spmm_lv<L, V, DT, WGT>(s, ptr, col, w, nr, dr, nc, dc, x, rv, y)
    if (lpr == 4 && vpl == 1) SG_SPMM(4, 1);
    if (lpr == 4 && vpl == 2) SG_SPMM(4, 2);
    if (lpr == 4) SG_SPMM(4, 4);
    if (lpr == 8) SG_SPMM(8, 4);
    if (lpr == 16) SG_SPMM(16, 4);
    if (vpl == 4) SG_SPMM(32, 4);
    SG_SPMM(32, 8);
#undef SG_SPMM
}

template <int VPL, int DT, bool WGT>
sg_status launch_tma_t(int64_t n_rows_cap, size_t smem, cudaStream_t s, const int32_t* ptr, const int32_t* col,
                       const float* w, int32_t nr, const int32_t* dr, int32_t nc, const int32_t* dc, const void* x,
                       int32_t rv, int32_t C, void* y) {
    static size_t smem_set = 0;  // the kernel's dynamic shared-memory limit, raised once per size
    if (smem > smem_set) {
        SG_CUDA(cudaFuncSetAttribute(k_spmm_tma<VPL, DT, WGT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        smem_set = smem;
    }
    int per_sm = 0;
    SG_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_spmm_tma<VPL, DT, WGT>, 32 * kTmaWarps, smem));
    if (per_sm < 1) return fail(SG_ERR_UNSUPPORTED, "aggregate: rows of %d bytes do not fit the copy-engine path", rv * 16);
    int64_t blocks = cdiv(n_rows_cap, kTmaWarps);  // a warp per row at most
    const int64_t cap = (int64_t)per_sm * num_sms();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    SG_CUDA(launch_pdl(k_spmm_tma<VPL, DT, WGT>, dim3((unsigned)blocks), dim3(32 * kTmaWarps), smem, s, ptr, col, w, nr,
                       dr, nc, dc, (const uint4*)x, rv, C, y));
    return SG_OK;
}

// The copy-engine SpMM for rows of row_vecs (<= 256) 16-byte vectors.
template <int DT, bool WGT>
sg_status launch_tma(const int32_t* ptr, const int32_t* col, const float* w, int32_t n_rows_cap,
                     const int32_t* d_rows, int32_t n_cols_cap, const int32_t* d_cols, const void* x, int32_t row_vecs,
                     void* y, cudaStream_t s) {
    const int row_bytes = row_vecs * 16;
    int C = 4096 / row_bytes;  // edges a stage: about 4 KB of rows, 2..8
    if (C > kTmaStageMax) C = kTmaStageMax;
    if (C < 2) C = 2;
    const size_t smem = (size_t)kTmaWarps * tma_warp_bytes(C, row_bytes);
    const int vpl = row_vecs <= 32 ? 1 : (row_vecs <= 64 ? 2 : (row_vecs <= 128 ? 4 : 8));
    if (vpl == 1) return launch_tma_t<1, DT, WGT>(n_rows_cap, smem, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, row_vecs, C, y);
    if (vpl == 2) return launch_tma_t<2, DT, WGT>(n_rows_cap, smem, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, row_vecs, C, y);
    if (vpl == 4) return launch_tma_t<4, DT, WGT>(n_rows_cap, smem, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, row_vecs, C, y);
    return launch_tma_t<8, DT, WGT>(n_rows_cap, smem, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, row_vecs, C, y);
}

// Runs y = A x for the row-split CSR (ptr, col, w) with n_rows rows.
sg_status run_spmm(const int32_t* ptr, const int32_t* col, const float* w, int32_t n_rows_cap, const int32_t* d_rows,
                   int32_t n_cols_cap, const int32_t* d_cols, const void* x, int32_t dtype_in, int32_t dim, void* y,
                   int32_t dtype_out, cudaStream_t s) {
    const int dt = dt_code(dtype_in, dtype_out);
    if (dt < 0) return fail(SG_ERR_UNSUPPORTED, "aggregate: dtype pair (%d -> %d) not supported", dtype_in, dtype_out);
    if (n_rows_cap <= 0) return SG_OK;
    const int64_t row_bytes = (int64_t)dim * (dtype_in == SG_F32 ? 4 : 2);
    const int64_t row_vecs = row_bytes / 16;
    const bool vec_ok = row_bytes % 16 == 0 && row_vecs <= 256 && ((uintptr_t)x % 16 == 0) && ((uintptr_t)y % 16 == 0);
    const int sms = num_sms();
    if (!vec_ok) {
        int64_t blocks = cdiv(n_rows_cap, kNT / 32);
        if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
        SG_CUDA(launch_pdl(k_spmm_scalar, dim3((unsigned)blocks), dim3(kNT), 0, s, ptr, col, w, n_rows_cap, d_rows,
                           n_cols_cap, d_cols, x, dim, dt == DT_F32 ? DT_F32 : (dt == DT_BF16 ? DT_BF16 : DT_BF16_F32), y));
        return SG_OK;
    }
    // a row goes to a group of LPR lanes holding VPL vectors each: small
    // groups put several rows of one warp in flight (rows of sampled blocks
    // are short, so latency, not bandwidth, limits a lone row)
    int lpr, vpl;
    if (row_vecs <= 16) {
        lpr = 4;
        vpl = row_vecs <= 4 ? 1 : (row_vecs <= 8 ? 2 : 4);
    } else if (row_vecs <= 32) {
        lpr = 8;
        vpl = 4;
    } else if (row_vecs <= 64) {
        lpr = 16;
        vpl = 4;
    } else {
        lpr = 32;
        vpl = row_vecs <= 128 ? 4 : 8;
    }
    // forward blocks of few rows (the hop next to the seeds): the copy-engine
    // path, whose warps keep several stages of whole rows in flight; larger
    // blocks: the register path (the copy engine moved 400-byte rows at only
    // ~1.6 TB/s there, against ~3.5 TB/s for k_spmm on the 52K-row hop)
    if (w == nullptr && n_rows_cap <= kTmaRowsMax) {
        if (dt == DT_F32) return launch_tma<DT_F32, false>(ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y, s);
        if (dt == DT_BF16) return launch_tma<DT_BF16, false>(ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y, s);
        return launch_tma<DT_BF16_F32, false>(ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y, s);
    }
    const bool wgt = w != nullptr;
    const int32_t rv = (int32_t)row_vecs;
    if (dt == DT_F32) return wgt ? launch_vec<DT_F32, true>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y)
                                 : launch_vec<DT_F32, false>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y);
    if (dt == DT_BF16) return wgt ? launch_vec<DT_BF16, true>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y)
                                  : launch_vec<DT_BF16, false>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y);
    return wgt ? launch_vec<DT_BF16_F32, true>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y)
               : launch_vec<DT_BF16_F32, false>(lpr, vpl, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, rv, y);
}

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of a transpose set: zeroed region first (counts, scan chains,
// counters), then scratch.  Outputs (tptr, tdst, tw) may live in the
// workspace (sg_aggregate_bwd) or in caller arrays (sg_transpose_blocks).
struct TLayout {
    size_t o_tcnt[SG_MAX_HOPS], o_status[SG_MAX_HOPS], o_ctr, zero_end;
    size_t o_tkey[SG_MAX_HOPS], o_dst[SG_MAX_HOPS], o_long[SG_MAX_HOPS];
    size_t o_tptr[SG_MAX_HOPS], o_tdst[SG_MAX_HOPS], o_tw[SG_MAX_HOPS], total;
};

TLayout t_layout(int nb, const int64_t* n_src_cap, const int64_t* n_edge_cap, bool outputs_inside) {
    TLayout L;
    size_t o = 0;
    for (int b = 0; b < nb; ++b) {
        const size_t ns = (size_t)(n_src_cap[b] > 0 ? n_src_cap[b] : 0) + 1;
        L.o_tcnt[b] = o;
        o = a256(o + ns * 4);
        L.o_status[b] = o;
        o = a256(o + (ns / kTTile + 2) * 8);
    }
    L.o_ctr = o;
    o = a256(o + 2 * SG_MAX_HOPS * 4);
    L.zero_end = o;
    for (int b = 0; b < nb; ++b) {
        const size_t ns = (size_t)(n_src_cap[b] > 0 ? n_src_cap[b] : 0) + 1;
        const size_t ne = (size_t)(n_edge_cap[b] > 0 ? n_edge_cap[b] : 1);
        L.o_tkey[b] = o;
        o = a256(o + ne * 4);
        L.o_dst[b] = o;
        o = a256(o + ne * 4);
        L.o_long[b] = o;
        o = a256(o + ns * 4);
        if (outputs_inside) {
            L.o_tptr[b] = o;
            o = a256(o + (ns + 1) * 4);
            L.o_tdst[b] = o;
            o = a256(o + ne * 4);
            L.o_tw[b] = o;
            o = a256(o + ne * 4);
        }
    }
    L.total = o;
    return L;
}

// Launches the five transpose kernels for the set.
sg_status run_transpose(TSet& t, const int64_t* n_dst_cap, const int64_t* n_src_cap, const int64_t* n_edge_cap,
                        char* ws, const TLayout& L, cudaStream_t s) {
    const int sms = num_sms();
    const int nb = t.nb;
    t.ctr = (uint32_t*)(ws + L.o_ctr);
    int64_t max_e = 1, max_src = 1, max_dst = 1;
    for (int b = 0; b < nb; ++b) {
        t.tcnt[b] = (int32_t*)(ws + L.o_tcnt[b]);
        t.status[b] = (unsigned long long*)(ws + L.o_status[b]);
        t.tkey[b] = (int32_t*)(ws + L.o_tkey[b]);
        t.dst_of[b] = (int32_t*)(ws + L.o_dst[b]);
        t.long_list[b] = (int32_t*)(ws + L.o_long[b]);
        if (n_edge_cap[b] > max_e) max_e = n_edge_cap[b];
        if (n_src_cap[b] > max_src) max_src = n_src_cap[b];
        if (n_dst_cap[b] > max_dst) max_dst = n_dst_cap[b];
    }
    SG_CUDA(cudaMemsetAsync(ws, 0, L.zero_end, s));
    auto grid = [&](int64_t work, int64_t per_block) {
        int64_t g = cdiv(work, per_block);
        if (g > (int64_t)sms * 8) g = (int64_t)sms * 8;
        if (g < 1) g = 1;
        return dim3((unsigned)g, (unsigned)nb, 1);
    };
    SG_CUDA(launch_pdl(k_tcount, grid(max_e, 256 * 4), dim3(256), 0, s, t));
    SG_CUDA(launch_pdl(k_tscan, grid(max_src + 1, kTTile), dim3(kNT), 0, s, t));
    SG_CUDA(launch_pdl(k_tscatter, grid(max_dst, 8), dim3(256), 0, s, t));
    SG_CUDA(launch_pdl(k_tsort, grid(max_src, kNT / 32), dim3(kNT), 0, s, t));
    SG_CUDA(launch_pdl(k_tsort_long, dim3((unsigned)sms, (unsigned)nb, 1), dim3(kNT), 0, s, t));
    return SG_OK;
}

}  // namespace

extern "C" sg_status sg_aggregate_fwd(const int32_t* d_indptr, const int32_t* d_idx, int32_t n_dst_cap, int32_t n_src_cap,
                                      const int32_t* d_dims, const void* d_h, int32_t dtype_in, int32_t dim, void* d_out,
                                      int32_t dtype_out, sg_stream_t stream) {
    if (n_dst_cap < 0 || n_src_cap < 0 || dim <= 0) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_fwd: bad sizes");
    if (n_dst_cap == 0) return SG_OK;
    if (!d_indptr || !d_out || (!d_h && n_src_cap > 0)) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_fwd: NULL array");
    return run_spmm(d_indptr, d_idx, nullptr, n_dst_cap, d_dims, n_src_cap, d_dims ? d_dims + 1 : nullptr, d_h, dtype_in,
                    dim, d_out, dtype_out, (cudaStream_t)stream);
}

extern "C" size_t sg_aggregate_bwd_workspace(int32_t n_dst_cap, int32_t n_src_cap, int64_t n_edge_cap) {
    (void)n_dst_cap;
    const int64_t ns = n_src_cap, ne = n_edge_cap;
    return t_layout(1, &ns, &ne, true).total;
}

extern "C" sg_status sg_aggregate_bwd(const int32_t* d_indptr, const int32_t* d_idx, int32_t n_dst_cap, int32_t n_src_cap,
                                      int64_t n_edge_cap, const int32_t* d_dims, const void* d_gdst, int32_t dtype_in,
                                      int32_t dim, void* d_gsrc, int32_t dtype_out, void* d_workspace,
                                      size_t workspace_bytes, sg_stream_t stream) {
    if (n_dst_cap < 0 || n_src_cap < 0 || dim <= 0 || n_edge_cap < 0 || n_edge_cap > 2147483647LL)
        return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: bad sizes");
    if (n_src_cap == 0) return SG_OK;
    if (!d_indptr || !d_gsrc || !d_workspace || (n_dst_cap > 0 && (!d_gdst || !d_idx)))
        return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: NULL array");
    if (dt_code(dtype_in, dtype_out) < 0) return fail(SG_ERR_UNSUPPORTED, "sg_aggregate_bwd: dtype pair not supported");
    const int64_t nd = n_dst_cap, ns = n_src_cap, ne = n_edge_cap;
    const TLayout L = t_layout(1, &ns, &ne, true);
    if (workspace_bytes < L.total) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: workspace needs %zu bytes", L.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d_workspace;
    TSet t;
    memset(&t, 0, sizeof(t));
    t.nb = 1;
    t.indptr[0] = d_indptr;
    t.idx[0] = d_idx;
    t.n_dst_cap[0] = n_dst_cap;
    t.n_src_cap[0] = n_src_cap;
    t.dims[0] = d_dims;
    t.tptr[0] = (int32_t*)(ws + L.o_tptr[0]);
    t.tdst[0] = (int32_t*)(ws + L.o_tdst[0]);
    t.tw[0] = (float*)(ws + L.o_tw[0]);
    sg_status st = run_transpose(t, &nd, &ns, &ne, ws, L, s);
    if (st != SG_OK) return st;
    return run_spmm(t.tptr[0], t.tdst[0], t.tw[0], n_src_cap, d_dims ? d_dims + 1 : nullptr, n_dst_cap, d_dims, d_gdst,
                    dtype_in, dim, d_gsrc, dtype_out, s);
}

extern "C" size_t sg_transpose_workspace(const int64_t* max_nodes, const int64_t* max_edges, int32_t n_hops) {
    if (!max_nodes || !max_edges || n_hops < 1 || n_hops > SG_MAX_HOPS) return 0;
    int64_t ns[SG_MAX_HOPS], ne[SG_MAX_HOPS];
    for (int h = 0; h < n_hops; ++h) {
        ns[h] = max_nodes[h + 1];
        ne[h] = max_edges[h];
    }
    return t_layout(n_hops, ns, ne, false).total;
}

extern "C" sg_status sg_transpose_blocks(const sg_blocks* blocks, const int64_t* max_nodes, const int64_t* max_edges,
                                         int32_t n_hops, const sg_transposed* out, void* d_workspace,
                                         size_t workspace_bytes, sg_stream_t stream) {
    if (!blocks || !blocks->counts || !max_nodes || !max_edges || !out || n_hops < 1 || n_hops > SG_MAX_HOPS)
        return fail(SG_ERR_INVALID_ARG, "sg_transpose_blocks: bad arguments");
    int64_t nd[SG_MAX_HOPS], ns[SG_MAX_HOPS], ne[SG_MAX_HOPS];
    TSet t;
    memset(&t, 0, sizeof(t));
    t.nb = n_hops;
    for (int h = 0; h < n_hops; ++h) {
        nd[h] = max_nodes[h];
        ns[h] = max_nodes[h + 1];
        ne[h] = max_edges[h];
        if (nd[h] < 0 || ns[h] < 0 || ne[h] < 0 || ns[h] > 2147483646LL || ne[h] > 2147483647LL || nd[h] > 2147483646LL)
            return fail(SG_ERR_INVALID_ARG, "sg_transpose_blocks: sizes of hop %d out of range", h + 1);
        if (!blocks->indptr[h] || !blocks->idx[h] || !out->tptr[h] || !out->tdst[h] || !out->tw[h])
            return fail(SG_ERR_INVALID_ARG, "sg_transpose_blocks: arrays of hop %d missing", h + 1);
        t.indptr[h] = blocks->indptr[h];
        t.idx[h] = blocks->idx[h];
        t.n_dst_cap[h] = (int32_t)nd[h];
        t.n_src_cap[h] = (int32_t)ns[h];
        t.dims[h] = blocks->counts + h;  // {sum_k |V_{h-1}^k|, sum_k |V_h^k|}
        t.tptr[h] = out->tptr[h];
        t.tdst[h] = out->tdst[h];
        t.tw[h] = out->tw[h];
    }
    const TLayout L = t_layout(n_hops, ns, ne, false);
    if (!d_workspace || workspace_bytes < L.total)
        return fail(SG_ERR_INVALID_ARG, "sg_transpose_blocks: workspace needs %zu bytes", L.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_transpose_blocks: workspace must be 256-byte aligned");
    return run_transpose(t, nd, ns, ne, (char*)d_workspace, L, (cudaStream_t)stream);
}

extern "C" sg_status sg_aggregate_bwd_t(const int32_t* d_tptr, const int32_t* d_tdst, const float* d_tw, int32_t n_src_cap,
                                        int32_t n_dst_cap, const int32_t* d_dims, const void* d_gdst, int32_t dtype_in,
                                        int32_t dim, void* d_gsrc, int32_t dtype_out, sg_stream_t stream) {
    if (n_src_cap < 0 || n_dst_cap < 0 || dim <= 0) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd_t: bad sizes");
    if (n_src_cap == 0) return SG_OK;
    if (!d_tptr || !d_gsrc || (n_dst_cap > 0 && (!d_tdst || !d_tw || !d_gdst)))
        return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd_t: NULL array");
    return run_spmm(d_tptr, d_tdst, d_tw, n_src_cap, d_dims ? d_dims + 1 : nullptr, n_dst_cap, d_dims, d_gdst, dtype_in, dim,
                    d_gsrc, dtype_out, (cudaStream_t)stream);
}

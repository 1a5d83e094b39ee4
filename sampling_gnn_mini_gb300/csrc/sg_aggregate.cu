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

#include "sg_internal.cuh"

SGI_ERROR_WORD(aggregate)

using namespace sgi;

namespace {

constexpr int kNT = 256;
constexpr int kMaxSeg = 1024;
constexpr int kWarpSortCap = 256;   // longest segment a warp sorts in shared memory
constexpr int kBlockSortCap = 4096; // longest segment a block sorts in shared memory

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

// y[r] = scale_r * sum_p w_p x[col[p]] for r < n_rows (see the file comment).
// WEIGHTED = false: w_p = 1 and scale_r = 1 / row length (forward mean).
// WEIGHTED = true:  w_p = w[p] and scale_r = 1 (backward over the transpose).
template <int LPR, int VPL, int DT, bool WEIGHTED>
__global__ void __launch_bounds__(kNT) k_spmm(const int32_t* __restrict__ ptr, const int32_t* __restrict__ col,
                                              const float* __restrict__ w, int32_t n_rows_cap,
                                              const int32_t* __restrict__ d_rows, int32_t n_cols_cap,
                                              const int32_t* __restrict__ d_cols, const uint4* __restrict__ x,
                                              int32_t row_vecs, void* __restrict__ y) {
    constexpr int EPV = Elems<DT>::n;
    constexpr int UE = VPL >= 4 ? 1 : (VPL == 2 ? 2 : 4);  // edges in flight per lane
    const int64_t n_rows = d_rows ? (int64_t)min(*d_rows, n_rows_cap) : n_rows_cap;
    const int32_t n_cols = d_cols ? min(*d_cols, n_cols_cap) : n_cols_cap;
    const unsigned lane = lane_id();
    const int gl = lane % LPR;
    // the LPR lanes of a group share a row (and so every loop trip count);
    // shuffles name only them, so groups of one warp proceed independently
    const unsigned gmask = LPR == 32 ? 0xffffffffu : (((1u << LPR) - 1u) << (lane - gl));
    const int64_t groups = (int64_t)gridDim.x * (kNT / LPR);
    for (int64_t r = (blockIdx.x * (int64_t)kNT + threadIdx.x) / LPR; r < n_rows; r += groups) {
        const int32_t lo = ptr[r], hi = ptr[r + 1];
        float acc[VPL][EPV];
#pragma unroll
        for (int p = 0; p < VPL; ++p)
#pragma unroll
            for (int q = 0; q < EPV; ++q) acc[p][q] = 0.f;
        for (int32_t c0 = lo; c0 < hi; c0 += LPR) {
            const int32_t my_e = c0 + gl;
            int32_t my_col = -1;
            float my_w = 1.f;
            if (my_e < hi) {
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
        const int32_t c = hi - lo;
#pragma unroll
        for (int p = 0; p < VPL; ++p) {
            const int vi = gl + p * LPR;
            if (vi >= row_vecs) continue;
            float o[EPV];
#pragma unroll
            for (int q = 0; q < EPV; ++q) {
                if (WEIGHTED) o[q] = acc[p][q];
                else o[q] = c > 0 ? __fdiv_rn(acc[p][q], (float)c) : 0.f;
            }
            store_vec<DT>(y, r, row_vecs, vi, o);
        }
    }
}

// Element-wise variant for rows whose byte size is not a multiple of 16 or is
// larger than 4 KB: a warp per row, lanes over the elements.
__global__ void __launch_bounds__(kNT) k_spmm_scalar(const int32_t* __restrict__ ptr, const int32_t* __restrict__ col,
                                                     const float* __restrict__ w, int32_t n_rows_cap,
                                                     const int32_t* __restrict__ d_rows, int32_t n_cols_cap,
                                                     const int32_t* __restrict__ d_cols, const void* __restrict__ x,
                                                     int32_t dim, int dt, void* __restrict__ y) {
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
// Edge count of the block from its row pointer.
__device__ __forceinline__ int32_t block_edges(const int32_t* indptr, int32_t n_dst_cap, const int32_t* dims) {
    const int32_t n_dst = dims ? min(dims[0], n_dst_cap) : n_dst_cap;
    return indptr[n_dst];
}

__global__ void k_tcount(const int32_t* __restrict__ indptr, const int32_t* __restrict__ idx, int32_t n_dst_cap,
                         int32_t n_src_cap, const int32_t* dims, int32_t* tcnt) {
    const int32_t E = block_edges(indptr, n_dst_cap, dims);
    const int32_t n_src = dims ? min(dims[1], n_src_cap) : n_src_cap;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < E; e += (int64_t)gridDim.x * blockDim.x) {
        const int32_t u = idx[e];
        if (u >= 0 && u < n_src) atomicAdd(tcnt + u, 1);
        else dev_err(ERR_INDEX);
    }
}

// Segmented exclusive scan of in[0, n) into out[0, n), n = (dims ? dims[1] :
// cap) + 1: pass 1 writes one sum per block, pass 2 adds the sums of earlier
// blocks and scans the block's segment in tiles.
__global__ void __launch_bounds__(kNT) k_scan_sums(const int32_t* in, int32_t cap, const int32_t* dims, int32_t* bsum) {
    __shared__ int32_t red[kNT / 32 + 1];
    const int64_t n = (int64_t)(dims ? min(dims[1], cap) : cap) + 1;
    int64_t lo, hi;
    segment_of(n, blockIdx.x, gridDim.x, lo, hi);
    int32_t s = 0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += kNT) s += in[i];
    s = block_sum<kNT>(s, red);
    if (threadIdx.x == 0) bsum[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kNT) k_scan_write(const int32_t* in, int32_t cap, const int32_t* dims,
                                                    const int32_t* bsum, int32_t* out) {
    __shared__ int32_t red[kNT / 32 + 1];
    __shared__ int32_t carry;
    const int64_t n = (int64_t)(dims ? min(dims[1], cap) : cap) + 1;
    int32_t pre = 0;
    for (int b = threadIdx.x; b < (int)blockIdx.x; b += kNT) pre += bsum[b];
    pre = block_sum<kNT>(pre, red);
    if (threadIdx.x == 0) carry = pre;
    __syncthreads();
    int64_t lo, hi;
    segment_of(n, blockIdx.x, gridDim.x, lo, hi);
    for (int64_t t0 = lo; t0 < hi; t0 += kNT) {
        const int64_t i = t0 + threadIdx.x;
        const int32_t v = i < hi ? in[i] : 0;
        int32_t tot;
        const int32_t ex = block_excl_scan<kNT>(v, red, tot);
        if (i < hi) out[i] = carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
}

// Places every edge in its src segment (order inside a segment is fixed by
// the sort that follows) and records the edge's dst row.
__global__ void k_tscatter(const int32_t* __restrict__ indptr, const int32_t* __restrict__ idx, int32_t n_dst_cap,
                           int32_t n_src_cap, const int32_t* dims, const int32_t* __restrict__ tptr, int32_t* tcnt,
                           int32_t* tkey, int32_t* dst_of) {
    const int32_t n_dst = dims ? min(dims[0], n_dst_cap) : n_dst_cap;
    const int32_t n_src = dims ? min(dims[1], n_src_cap) : n_src_cap;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t v = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; v < n_dst; v += warps) {
        const int32_t lo = indptr[v], hi = indptr[v + 1];
        for (int32_t e = lo + (int32_t)lane_id(); e < hi; e += 32) {
            const int32_t u = idx[e];
            dst_of[e] = (int32_t)v;
            if (u < 0 || u >= n_src) continue;
            const int32_t p = tptr[u] + atomicSub(tcnt + u, 1) - 1;
            tkey[p] = e;
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
// ranked by one warp; longer ones go to a list for k_tsort_long.
__global__ void __launch_bounds__(kNT) k_tsort(const int32_t* __restrict__ indptr, int32_t n_src_cap, const int32_t* dims,
                                               const int32_t* __restrict__ tptr, const int32_t* __restrict__ tkey,
                                               const int32_t* __restrict__ dst_of, int32_t* tdst, float* tw,
                                               int32_t* long_list, int32_t* long_count) {
    __shared__ int32_t sk[kNT / 32][kWarpSortCap];
    const int32_t n_src = dims ? min(dims[1], n_src_cap) : n_src_cap;
    const int wib = threadIdx.x >> 5;
    const unsigned lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (kNT / 32);
    for (int64_t u = blockIdx.x * (int64_t)(kNT / 32) + wib; u < n_src; u += warps) {
        const int32_t lo = tptr[u], len = tptr[u + 1] - lo;
        if (len == 0) continue;
        if (len <= 32) {
            const int32_t key = (int)lane < len ? tkey[lo + lane] : 0x7FFFFFFF;
            int rank = 0;
            for (int t = 0; t < len; ++t) rank += __shfl_sync(0xffffffffu, key, t) < key;
            if ((int)lane < len) emit_transposed(indptr, dst_of, key, lo + rank, tdst, tw);
        } else if (len <= kWarpSortCap) {
            int32_t* s = sk[wib];
            for (int t = lane; t < len; t += 32) s[t] = tkey[lo + t];
            __syncwarp();
            for (int i = lane; i < len; i += 32) {
                const int32_t key = s[i];
                int rank = 0;
                for (int t = 0; t < len; ++t) rank += s[t] < key;
                emit_transposed(indptr, dst_of, key, lo + rank, tdst, tw);
            }
            __syncwarp();
        } else if (lane == 0) {
            long_list[atomicAdd(long_count, 1)] = (int32_t)u;
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
            const int32_t a = (i / half) * k + (i % half);
            const int32_t b = (i / half) * k + (k - 1 - (i % half));
            if (b < len) {
                const int32_t x = keys[a], y = keys[b];
                if (y < x) { keys[a] = y; keys[b] = x; }
            }
        }
        __syncthreads();
        for (int32_t j = k >> 2; j > 0; j >>= 1) {
            for (int32_t i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int32_t a = (i / j) * (2 * j) + (i % j);
                const int32_t b = a + j;
                if (b < len) {
                    const int32_t x = keys[a], y = keys[b];
                    if (y < x) { keys[a] = y; keys[b] = x; }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kNT) k_tsort_long(const int32_t* __restrict__ indptr, const int32_t* __restrict__ tptr,
                                                    int32_t* tkey, const int32_t* __restrict__ dst_of, int32_t* tdst,
                                                    float* tw, const int32_t* long_list, const int32_t* long_count) {
    __shared__ int32_t sk[kBlockSortCap];
    const int32_t n = *long_count;
    for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int32_t u = long_list[i];
        const int32_t lo = tptr[u], len = tptr[u + 1] - lo;
        int32_t* keys;
        if (len <= kBlockSortCap) {
            for (int32_t t = threadIdx.x; t < len; t += blockDim.x) sk[t] = tkey[lo + t];
            keys = sk;
        } else {
            keys = tkey + lo;  // long segment: sort in place in global memory
        }
        __syncthreads();
        block_bitonic_sort(keys, len);
        for (int32_t t = threadIdx.x; t < len; t += blockDim.x) emit_transposed(indptr, dst_of, keys[t], lo + t, tdst, tw);
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

template <int DT, bool WGT>
sg_status launch_vec(int lpr, int vpl, int blocks, cudaStream_t s, const int32_t* ptr, const int32_t* col, const float* w,
                     int32_t nr, const int32_t* dr, int32_t nc, const int32_t* dc, const void* x, int32_t rv, void* y) {
#define SG_SPMM(L, V) k_spmm<L, V, DT, WGT><<<blocks, kNT, 0, s>>>(ptr, col, w, nr, dr, nc, dc, (const uint4*)x, rv, y)
    if (lpr == 4) SG_SPMM(4, 1);
    else if (lpr == 8) SG_SPMM(8, 1);
    else if (lpr == 16) SG_SPMM(16, 1);
    else if (vpl == 1) SG_SPMM(32, 1);
    else if (vpl == 2) SG_SPMM(32, 2);
    else if (vpl == 4) SG_SPMM(32, 4);
    else SG_SPMM(32, 8);
#undef SG_SPMM
    SG_CHECK_LAUNCH("k_spmm");
    return SG_OK;
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
        k_spmm_scalar<<<(unsigned)blocks, kNT, 0, s>>>(ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, dim,
                                                      dt == DT_F32 ? DT_F32 : (dt == DT_BF16 ? DT_BF16 : DT_BF16_F32), y);
        SG_CHECK_LAUNCH("k_spmm_scalar");
        return SG_OK;
    }
    int lpr = 32, vpl = 1;
    if (row_vecs <= 4) lpr = 4;
    else if (row_vecs <= 8) lpr = 8;
    else if (row_vecs <= 16) lpr = 16;
    else vpl = row_vecs <= 32 ? 1 : (row_vecs <= 64 ? 2 : (row_vecs <= 128 ? 4 : 8));
    int64_t blocks = cdiv((int64_t)n_rows_cap * lpr, kNT);
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    const bool wgt = w != nullptr;
    if (dt == DT_F32) return wgt ? launch_vec<DT_F32, true>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y)
                                 : launch_vec<DT_F32, false>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y);
    if (dt == DT_BF16) return wgt ? launch_vec<DT_BF16, true>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y)
                                  : launch_vec<DT_BF16, false>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y);
    return wgt ? launch_vec<DT_BF16_F32, true>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y)
               : launch_vec<DT_BF16_F32, false>(lpr, vpl, (int)blocks, s, ptr, col, w, n_rows_cap, d_rows, n_cols_cap, d_cols, x, (int32_t)row_vecs, y);
}

struct BwdLayout {
    size_t o_tcnt, o_tptr, o_tkey, o_dst, o_tdst, o_tw, o_bsum, o_long, total;
};

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

BwdLayout bwd_layout(int32_t n_dst_cap, int32_t n_src_cap, int64_t n_edge_cap) {
    (void)n_dst_cap;
    BwdLayout L;
    const size_t ns = (size_t)(n_src_cap > 0 ? n_src_cap : 0) + 2, ne = (size_t)(n_edge_cap > 0 ? n_edge_cap : 1);
    size_t o = 0;
    L.o_tcnt = o; o = a256(o + (ns + 1) * 4);  // + the long-segment counter
    L.o_tptr = o; o = a256(o + ns * 4);
    L.o_tkey = o; o = a256(o + ne * 4);
    L.o_dst = o;  o = a256(o + ne * 4);
    L.o_tdst = o; o = a256(o + ne * 4);
    L.o_tw = o;   o = a256(o + ne * 4);
    L.o_bsum = o; o = a256(o + (size_t)kMaxSeg * 4);
    L.o_long = o; o = a256(o + ns * 4);
    L.total = o;
    return L;
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
    return bwd_layout(n_dst_cap, n_src_cap, n_edge_cap).total;
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
    const BwdLayout L = bwd_layout(n_dst_cap, n_src_cap, n_edge_cap);
    if (workspace_bytes < L.total) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: workspace needs %zu bytes", L.total);
    if (((uintptr_t)d_workspace) % 256) return fail(SG_ERR_INVALID_ARG, "sg_aggregate_bwd: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)d_workspace;
    int32_t* tcnt = (int32_t*)(ws + L.o_tcnt);
    int32_t* long_count = tcnt + (n_src_cap + 2);
    int32_t* tptr = (int32_t*)(ws + L.o_tptr);
    int32_t* tkey = (int32_t*)(ws + L.o_tkey);
    int32_t* dst_of = (int32_t*)(ws + L.o_dst);
    int32_t* tdst = (int32_t*)(ws + L.o_tdst);
    float* tw = (float*)(ws + L.o_tw);
    int32_t* bsum = (int32_t*)(ws + L.o_bsum);
    int32_t* long_list = (int32_t*)(ws + L.o_long);
    const int sms = num_sms();
    SG_CUDA(cudaMemsetAsync(tcnt, 0, ((size_t)n_src_cap + 3) * 4, s));
    if (n_dst_cap > 0) {
        int64_t eb = cdiv(n_edge_cap > 0 ? n_edge_cap : 1, 256);
        if (eb > (int64_t)sms * 8) eb = (int64_t)sms * 8;
        k_tcount<<<(unsigned)eb, 256, 0, s>>>(d_indptr, d_idx, n_dst_cap, n_src_cap, d_dims, tcnt);
        SG_CHECK_LAUNCH("k_tcount");
    }
    int64_t gs = cdiv((int64_t)n_src_cap + 1, 2048);
    if (gs > kMaxSeg) gs = kMaxSeg;
    if (gs < 1) gs = 1;
    k_scan_sums<<<(unsigned)gs, kNT, 0, s>>>(tcnt, n_src_cap, d_dims, bsum);
    SG_CHECK_LAUNCH("k_scan_sums");
    k_scan_write<<<(unsigned)gs, kNT, 0, s>>>(tcnt, n_src_cap, d_dims, bsum, tptr);
    SG_CHECK_LAUNCH("k_scan_write");
    if (n_dst_cap > 0) {
        int64_t wb = cdiv(n_dst_cap, 8);
        if (wb > (int64_t)sms * 8) wb = (int64_t)sms * 8;
        k_tscatter<<<(unsigned)wb, 256, 0, s>>>(d_indptr, d_idx, n_dst_cap, n_src_cap, d_dims, tptr, tcnt, tkey, dst_of);
        SG_CHECK_LAUNCH("k_tscatter");
    }
    int64_t sb = cdiv(n_src_cap, kNT / 32);
    if (sb > (int64_t)sms * 8) sb = (int64_t)sms * 8;
    if (sb < 1) sb = 1;
    k_tsort<<<(unsigned)sb, kNT, 0, s>>>(d_indptr, n_src_cap, d_dims, tptr, tkey, dst_of, tdst, tw, long_list, long_count);
    SG_CHECK_LAUNCH("k_tsort");
    k_tsort_long<<<(unsigned)sms, kNT, 0, s>>>(d_indptr, tptr, tkey, dst_of, tdst, tw, long_list, long_count);
    SG_CHECK_LAUNCH("k_tsort_long");
    return run_spmm(tptr, tdst, tw, n_src_cap, d_dims ? d_dims + 1 : nullptr, n_dst_cap, d_dims, d_gdst, dtype_in, dim,
                    d_gsrc, dtype_out, s);
}

// SAGE UPDATE of one layer as a dense product on the tensor cores (GARDEN
// page, Section II-A, Eq. (2): a node's new state from its previous state and
// its aggregated message; GraphSAGE's form, a linear layer over the
// concatenation followed by ReLU, hidden width 128 as in Section VI-A):
//   y[r, o]   = sum_{k<d} W[o, k] h[r, k] + sum_{k<d} W[o, d + k] m[r, k]
//   out[r, o] = max(y[r, o], 0)
// for r < n rows (the dst nodes of a block), o < 128.
//
// One CTA computes a 128 x 128 tile of y with tcgen05.mma (cta_group::1,
// M = 128, N = 128): fp32 inputs as kind::tf32, bf16 inputs as kind::f16,
// fp32 accumulation in tensor memory.  The concatenation is never
// materialised: the K loop runs over the tiles of h, then those of m, each
// with the matching half of W, all four through their own TMA tensor maps
// (128-byte swizzle; columns past d are zero-filled by the copy engine).
// Warp roles: lane 0 of warp 0 issues the TMA loads into a ring of kStages
// stages, lane 0 of warp 1 issues the MMAs (warp 1 also allocates and frees
// the tensor memory), and all four warps read the accumulator back
// (tcgen05.ld, 32 rows each) for the ReLU epilogue.  Every mbarrier wait is
// bounded; a wait that gives up sets the error word (SG_ERR_TIMEOUT) and the
// CTA stops issuing work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include "sg_internal.cuh"

SGI_ERROR_WORD(update)

using namespace sgi;

namespace {

constexpr int kThreads = 128;          // 4 warps
constexpr int kBM = 128;               // rows of a tile
constexpr int kBN = 128;               // outputs (the hidden width)
constexpr int kTileBytes = 128;        // K bytes of a stage (one 128-byte swizzle row)
constexpr int kStages = 3;            // 96 KB of ring: two CTAs an SM (their epilogues overlap the other's loads)
constexpr int kStageA = kBM * kTileBytes;  // 16 KB
constexpr int kStageB = kBN * kTileBytes;  // 16 KB
constexpr int kSmemTiles = kStages * (kStageA + kStageB);
constexpr int kSpins = 1 << 22;        // polls of one mbarrier before giving up

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// true once the phase of the given parity has completed; false after kSpins polls
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (int i = 0; i < kSpins; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// 2-D tiled TMA load of the box at (x = column, y = row) into shared memory,
// completing on bar
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzle layout: rows of 128 bytes, groups of 8 rows 1024 bytes apart (the
// stride offset), tile base 1024-byte aligned (base offset 0).  Fields: start
// address >> 4 in bits 0-13, leading offset >> 4 in bits 16-29 (unused by
// swizzled K-major layouts; 1), stride offset >> 4 in bits 32-45, the fixed
// value 1 in bits 46-47, layout (2 = 128-byte swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::tf32 / kind::f16: D fp32
// (bits 4-5 = 1), A and B formats (bits 7-9, 10-12: 2 = tf32, 1 = bf16),
// both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_format) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((uint32_t)(kBN >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_issue(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate, bool tf32) {
    if (tf32) {
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// arrives once on bar when every MMA this thread issued so far has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 lanes (lane i: row 32w + i)
__device__ __forceinline__ void tmem_load_32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The four operand maps: A = [h | m] by halves, B = W by halves (its columns
// [0, d) and [d, 2d)).
struct UpdateMaps {
    CUtensorMap h, m, wh, wm;
};

template <bool TF32>
__global__ void __launch_bounds__(kThreads, 2)
    k_sage_fwd(const __grid_constant__ UpdateMaps maps, int32_t n_cap, const int32_t* __restrict__ d_n, int32_t kt_half,
               float* __restrict__ out, float* __restrict__ y) {
    extern __shared__ uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_base;
    pdl_start();
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    const int32_t n = d_n ? min(max(*d_n, 0), n_cap) : n_cap;
    const int32_t row0 = (int32_t)blockIdx.x * kBM;
    if (row0 >= n) return;  // the same in every thread, before any barrier
    uint8_t* tiles = dsm + ((1024 - (smem_addr(dsm) & 1023)) & 1023);  // 1024-byte aligned stages
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 1) {  // 128 fp32 columns of tensor memory: the 128 x 128 accumulator
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&tmem_base)),
                     "r"(kBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = tmem_base;
    const int n_k = 2 * kt_half;
    constexpr int kBK = kTileBytes / (TF32 ? 4 : 2);  // K elements of a stage
    if (warp == 0 && lane == 0) {
        // TMA producer: stage s takes K tile kt of A (h, then m) and of B
        int issued = 0;
        for (int kt = 0; kt < n_k; ++kt) {
            const int s = kt % kStages;
            if (kt >= kStages && !mbar_wait(&empty[s], (uint32_t)((kt / kStages) - 1) & 1u)) {
                dev_err(ERR_TIMEOUT);
                break;
            }
            uint8_t* a = tiles + s * (kStageA + kStageB);
            const bool second = kt >= kt_half;
            const int32_t x = (second ? kt - kt_half : kt) * kBK;
            mbar_expect_tx(&full[s], kStageA + kStageB);
            tma_load_2d(a, second ? &maps.m : &maps.h, x, row0, &full[s]);
            tma_load_2d(a + kStageA, second ? &maps.wm : &maps.wh, x, 0, &full[s]);
            ++issued;
        }
        // every load issued has landed before this thread moves on (on the
        // normal path the MMA issuer waited for them already)
        for (int k = issued - kStages < 0 ? 0 : issued - kStages; k < issued; ++k)
            if (!mbar_wait(&full[k % kStages], (uint32_t)(k / kStages) & 1u)) dev_err(ERR_TIMEOUT);
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: kTileBytes / 32 MMAs of K = 32 bytes per stage
        const uint32_t idesc = instr_desc(TF32 ? 2u : 1u);
        for (int kt = 0; kt < n_k; ++kt) {
            const int s = kt % kStages;
            if (!mbar_wait(&full[s], (uint32_t)(kt / kStages) & 1u)) {
                dev_err(ERR_TIMEOUT);
                break;
            }
            tmem_fence_after();
            const uint32_t a = smem_addr(tiles + s * (kStageA + kStageB)), b = a + kStageA;
#pragma unroll
            for (int kk = 0; kk < kTileBytes / 32; ++kk)
                mma_issue(tmem, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc,
                          (uint32_t)((kt | kk) != 0), TF32);
            mma_commit(&empty[s]);  // frees stage s once these MMAs have read it
        }
        mma_commit(&done);  // the accumulator is final once every MMA issued has completed
    }
    __syncwarp();
    // epilogue: warp w reads rows 32w .. 32w + 31 of the tile from tensor memory
    const bool ok = mbar_wait(&done, 0);
    if (!ok && lane == 0) dev_err(ERR_TIMEOUT);
    tmem_fence_after();
    const int32_t r = row0 + warp * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        float v[32];
        tmem_load_32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        if (ok && r < n) {
            float4* o = reinterpret_cast<float4*>(out + (size_t)r * kBN + c0);
            float4* yo = y ? reinterpret_cast<float4*>(y + (size_t)r * kBN + c0) : nullptr;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 t = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                if (yo) yo[q] = t;
                o[q] = make_float4(fmaxf(t.x, 0.f), fmaxf(t.y, 0.f), fmaxf(t.z, 0.f), fmaxf(t.w, 0.f));
            }
        }
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 1) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kBN) : "memory");
    }
}

// ------------------------------------------------------------ backward
// The backward products in the same form as the forward (both operands
// K-major, D = A B^T with B given as N rows of K):
//   dZ = dY W       A = dY  [n x 128],  B = W^T [2d x 128]  (N tiles of 128 over 2d)
//   dW = dY^T Z     A = dY^T [128 x n], B = Z^T [2d x n]    (K = rows, split over CTAs)
// with dY = g * (y > 0).  The transposed operands are written first by
// k_transpose (columns past n up to the next K tile are zeros, so a K tile
// never reads stale workspace).  A split of dW writes its partial 128 x 2d
// tile; k_split_sum adds the partials in split order, so the result does not
// depend on scheduling.
enum { EPI_DZ = 0, EPI_SPLIT = 1 };

struct GemmMaps {
    CUtensorMap a, b;
};

template <bool TF32, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
    k_sage_gemm(const __grid_constant__ GemmMaps maps, int32_t m_cap, const int32_t* __restrict__ d_m_rows,
                int32_t k_cap, const int32_t* __restrict__ d_k, int32_t n_cols, int32_t split_col, float* __restrict__ o0,
                float* __restrict__ o1, int32_t ld1) {
    extern __shared__ uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_base;
    pdl_start();
    constexpr int kBK = kTileBytes / (TF32 ? 4 : 2);
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
    const int32_t m_rows = d_m_rows ? min(max(*d_m_rows, 0), m_cap) : m_cap;
    const int32_t k_len = d_k ? min(max(*d_k, 0), k_cap) : k_cap;
    const int32_t row0 = (int32_t)blockIdx.x * kBM, col0 = (int32_t)blockIdx.y * kBN;
    if (EPI == EPI_DZ && row0 >= m_rows) return;  // the same in every thread, before any barrier
    // this CTA's K tiles: all of them, or split blockIdx.z of gridDim.z
    const int32_t n_kt = (k_len + kBK - 1) / kBK;
    const int32_t per = (n_kt + (int32_t)gridDim.z - 1) / (int32_t)gridDim.z;
    const int32_t kt0 = min(n_kt, (int32_t)blockIdx.z * per), kt1 = min(n_kt, kt0 + per);
    const int n_k = kt1 - kt0;
    if (EPI == EPI_SPLIT && n_k == 0) {
        // a split with no K tiles: its partial tile is zero, and no MMA, copy
        // or barrier is needed (the same in every thread)
        float* dst = o0 + (size_t)blockIdx.z * kBM * ld1 + (size_t)(warp * 32 + lane) * ld1 + col0;
        for (int j = 0; j < kBN && col0 + j < n_cols; ++j) dst[j] = 0.f;
        return;
    }
    uint8_t* tiles = dsm + ((1024 - (smem_addr(dsm) & 1023)) & 1023);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(&tmem_base)),
                     "r"(kBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = tmem_base;
    if (warp == 0 && lane == 0) {
        int issued = 0;
        for (int i = 0; i < n_k; ++i) {
            const int s = i % kStages;
            if (i >= kStages && !mbar_wait(&empty[s], (uint32_t)((i / kStages) - 1) & 1u)) {
                dev_err(ERR_TIMEOUT);
                break;
            }
            uint8_t* a = tiles + s * (kStageA + kStageB);
            const int32_t x = (kt0 + i) * kBK;
            mbar_expect_tx(&full[s], kStageA + kStageB);
            tma_load_2d(a, &maps.a, x, row0, &full[s]);
            tma_load_2d(a + kStageA, &maps.b, x, col0, &full[s]);
            ++issued;
        }
        for (int k = issued - kStages < 0 ? 0 : issued - kStages; k < issued; ++k)
            if (!mbar_wait(&full[k % kStages], (uint32_t)(k / kStages) & 1u)) dev_err(ERR_TIMEOUT);
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = instr_desc(TF32 ? 2u : 1u);
        for (int i = 0; i < n_k; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(&full[s], (uint32_t)(i / kStages) & 1u)) {
                dev_err(ERR_TIMEOUT);
                break;
            }
            tmem_fence_after();
            const uint32_t a = smem_addr(tiles + s * (kStageA + kStageB)), b = a + kStageA;
#pragma unroll
            for (int kk = 0; kk < kTileBytes / 32; ++kk)
                mma_issue(tmem, smem_desc_sw128(a + kk * 32), smem_desc_sw128(b + kk * 32), idesc,
                          (uint32_t)((i | kk) != 0), TF32);
            mma_commit(&empty[s]);
        }
        mma_commit(&done);
    }
    __syncwarp();
    const bool ok = mbar_wait(&done, 0);
    if (!ok && lane == 0) dev_err(ERR_TIMEOUT);
    tmem_fence_after();
    const int32_t r = row0 + warp * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        float v[32];
        tmem_load_32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        if (!ok) continue;
        if (EPI == EPI_DZ) {
            // columns [0, split_col) to o0 (row stride split_col), the rest to o1 (row stride ld1)
            if (r >= m_rows) continue;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int32_t c = col0 + c0 + j;
                if (c >= n_cols) break;
                if (c < split_col) o0[(size_t)r * split_col + c] = v[j];
                else o1[(size_t)r * ld1 + (c - split_col)] = v[j];
            }
        } else {
            // the partial tile of split z
            float* dst = o0 + (size_t)blockIdx.z * kBM * ld1 + (size_t)r * ld1 + col0 + c0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + c0 + j < n_cols) dst[j] = v[j];
        }
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 1) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kBN) : "memory");
    }
}

// dY = g * (y > 0), in the operand type (fp32, or bf16 rounded to nearest)
template <typename T>
__global__ void __launch_bounds__(256) k_relu_grad(const float* __restrict__ g, const float* __restrict__ y,
                                                   int32_t n_cap, const int32_t* __restrict__ d_n, T* __restrict__ dy) {
    pdl_start();
    const int64_t n = d_n ? min(max(*d_n, 0), n_cap) : n_cap;
    const int64_t total = n * kBN;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = y[i] > 0.f ? g[i] : 0.f;
        if constexpr (sizeof(T) == 4) dy[i] = v;
        else dy[i] = __float2bfloat16_rn(v);
    }
}

// dst[c * dst_ld + dst_row0 + r] = src[r * src_ld + c] for r < rows, c < cols
// (rows from the device count when given), and zeros at r in [rows, pad_to)
// so that the last K tile of the transposed operand reads no stale data.
template <typename T>
__global__ void __launch_bounds__(256) k_transpose(const T* __restrict__ src, int32_t rows_cap,
                                                   const int32_t* __restrict__ d_rows, int32_t cols, int32_t src_ld,
                                                   T* __restrict__ dst, int32_t dst_ld, int32_t pad_unit) {
    pdl_start();
    __shared__ T tile[32][33];
    const int32_t rows = d_rows ? min(max(*d_rows, 0), rows_cap) : rows_cap;
    const int32_t pad_to = min(((rows + pad_unit - 1) / pad_unit) * pad_unit, dst_ld);
    const int32_t r0 = (int32_t)blockIdx.x * 32, c0 = (int32_t)blockIdx.y * 32;
    if (r0 >= pad_to) return;
    const int tx = (int)(threadIdx.x & 31), ty = (int)(threadIdx.x >> 5);  // 32 x 8 threads
    for (int i = ty; i < 32; i += 8) {
        const int32_t r = r0 + i, c = c0 + tx;
        tile[i][tx] = (r < rows && c < cols) ? src[(size_t)r * src_ld + c] : T(0.f);
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int32_t c = c0 + i, r = r0 + tx;
        if (c < cols && r < pad_to) dst[(size_t)c * dst_ld + r] = tile[tx][i];
    }
}

// dW[o, k] = sum over splits z (in order) of part[z][o][k]
__global__ void __launch_bounds__(256) k_split_sum(const float* __restrict__ part, int32_t splits, int32_t ld,
                                                   int32_t cols, float* __restrict__ dW) {
    pdl_start();
    const int64_t total = (int64_t)kBM * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = i / cols, k = i - o * cols;
        float s = 0.f;
        for (int32_t z = 0; z < splits; ++z) s += part[((size_t)z * kBM + o) * ld + k];
        dW[i] = s;
    }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
        else
            cudaGetLastError();
    }
    return fn;
}

// Map of a row-major [rows x cols] matrix (row stride in bytes), loaded in
// boxes of kTileBytes x 128 rows with the 128-byte swizzle; reads past the
// matrix fill zeros.
bool make_map(CUtensorMap* map, const void* base, bool tf32, uint64_t cols, uint64_t rows, uint64_t stride_bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const uint32_t elem = tf32 ? 4 : 2;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(kTileBytes / elem), (cuuint32_t)kBM};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool TF32>
sg_status launch_fwd(const UpdateMaps& maps, int32_t n_cap, const int32_t* d_n, int32_t kt_half, float* out, float* y,
                     cudaStream_t s) {
    const size_t smem = (size_t)kSmemTiles + 1024;
    static bool attr = false;
    if (!attr) {
        SG_CUDA(cudaFuncSetAttribute(k_sage_fwd<TF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr = true;
    }
    const unsigned blocks = (unsigned)((n_cap + kBM - 1) / kBM);
    SG_CUDA(launch_pdl(k_sage_fwd<TF32>, dim3(blocks), dim3(kThreads), smem, s, maps, n_cap, d_n, kt_half, out, y));
    return SG_OK;
}

}  // namespace

extern "C" sg_status sg_sage_fwd(const void* d_h, const void* d_m, const void* d_W, int32_t dtype, int32_t n_cap,
                                 const int32_t* d_n, int32_t dim, int32_t d_out, float* d_out_act, float* d_y,
                                 sg_stream_t stream) {
    if (dtype != SG_F32 && dtype != SG_BF16) return fail(SG_ERR_UNSUPPORTED, "sg_sage_fwd: dtype");
    if (n_cap < 0 || dim <= 0) return fail(SG_ERR_INVALID_ARG, "sg_sage_fwd: bad sizes");
    if (d_out != kBN) return fail(SG_ERR_UNSUPPORTED, "sg_sage_fwd: d_out must be %d", kBN);
    if (n_cap == 0) return SG_OK;
    const bool tf32 = dtype == SG_F32;
    const int64_t elem = tf32 ? 4 : 2;
    if ((dim * elem) % 16) return fail(SG_ERR_UNSUPPORTED, "sg_sage_fwd: rows of %lld bytes are not a multiple of 16",
                                       (long long)(dim * elem));
    if (!d_h || !d_m || !d_W || !d_out_act) return fail(SG_ERR_INVALID_ARG, "sg_sage_fwd: NULL array");
    if (((uintptr_t)d_h | (uintptr_t)d_m | (uintptr_t)d_W | (uintptr_t)d_out_act | (uintptr_t)d_y) % 16)
        return fail(SG_ERR_INVALID_ARG, "sg_sage_fwd: arrays must be 16-byte aligned");
    UpdateMaps maps;
    memset(&maps, 0, sizeof(maps));
    const uint64_t row = (uint64_t)dim * elem;
    const char* w = (const char*)d_W;
    if (!make_map(&maps.h, d_h, tf32, dim, n_cap, row) || !make_map(&maps.m, d_m, tf32, dim, n_cap, row) ||
        !make_map(&maps.wh, w, tf32, dim, kBN, 2 * row) || !make_map(&maps.wm, w + row, tf32, dim, kBN, 2 * row))
        return fail(SG_ERR_CUDA, "sg_sage_fwd: tensor map encoding failed");
    const int32_t kt_half = (int32_t)((row + kTileBytes - 1) / kTileBytes);
    cudaStream_t s = (cudaStream_t)stream;
    return tf32 ? launch_fwd<true>(maps, n_cap, d_n, kt_half, d_out_act, d_y, s)
                : launch_fwd<false>(maps, n_cap, d_n, kt_half, d_out_act, d_y, s);
}

namespace {

constexpr int kSplits = 64;  // K splits of the dW product
constexpr int kPadK = 64;    // columns of a transposed operand are padded to this (>= a K tile)

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

struct BwdLayout {
    size_t dy, dyt, zt, wt, part, total;
    int64_t ld;  // columns of the transposed operands (rows n_cap padded)
};

BwdLayout bwd_layout(int64_t n_cap, int64_t dim, int64_t elem) {
    BwdLayout L;
    L.ld = ((n_cap + kPadK - 1) / kPadK) * kPadK;
    size_t o = 0;
    L.dy = o;
    o += a256((size_t)n_cap * kBN * elem);
    L.dyt = o;
    o += a256((size_t)kBN * L.ld * elem);
    L.zt = o;
    o += a256((size_t)2 * dim * L.ld * elem);
    L.wt = o;
    o += a256((size_t)2 * dim * kBN * elem);
    L.part = o;
    o += a256((size_t)kSplits * kBM * 2 * dim * sizeof(float));
    L.total = o;
    return L;
}

template <bool TF32, int EPI>
sg_status launch_gemm(const GemmMaps& maps, dim3 grid, int32_t m_cap, const int32_t* d_m, int32_t k_cap,
                      const int32_t* d_k, int32_t n_cols, int32_t split_col, float* o0, float* o1, int32_t ld1,
                      cudaStream_t s) {
    const size_t smem = (size_t)kSmemTiles + 1024;
    static bool attr = false;
    if (!attr) {
        SG_CUDA(cudaFuncSetAttribute(k_sage_gemm<TF32, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr = true;
    }
    SG_CUDA(launch_pdl(k_sage_gemm<TF32, EPI>, grid, dim3(kThreads), smem, s, maps, m_cap, d_m, k_cap, d_k, n_cols,
                       split_col, o0, o1, ld1));
    return SG_OK;
}

template <typename T, bool TF32>
sg_status run_bwd(const T* h, const T* m, const T* W, int32_t n_cap, const int32_t* d_n, int32_t dim, const float* y,
                  const float* g, float* dW, float* dh, float* dm, char* ws, const BwdLayout& L, cudaStream_t s) {
    const int64_t elem = sizeof(T);
    constexpr int32_t kBK = kTileBytes / (TF32 ? 4 : 2);
    T* dy = (T*)(ws + L.dy);
    T* dyt = (T*)(ws + L.dyt);
    T* zt = (T*)(ws + L.zt);
    T* wt = (T*)(ws + L.wt);
    float* part = (float*)(ws + L.part);
    const int32_t ld = (int32_t)L.ld, two_d = 2 * dim;
    int64_t eb = cdiv((int64_t)n_cap * kBN, 256);
    if (eb > (int64_t)num_sms() * 8) eb = (int64_t)num_sms() * 8;
    if (eb < 1) eb = 1;
    SG_CUDA(launch_pdl(k_relu_grad<T>, dim3((unsigned)eb), dim3(256), 0, s, g, y, n_cap, d_n, dy));
    const unsigned rb = (unsigned)cdiv((int64_t)ld, 32);
    SG_CUDA(launch_pdl(k_transpose<T>, dim3(rb, (unsigned)cdiv(kBN, 32)), dim3(256), 0, s, (const T*)dy, n_cap, d_n,
                       (int32_t)kBN, (int32_t)kBN, dyt, ld, kBK));
    SG_CUDA(launch_pdl(k_transpose<T>, dim3(rb, (unsigned)cdiv(dim, 32)), dim3(256), 0, s, h, n_cap, d_n, dim, dim, zt,
                       ld, kBK));
    SG_CUDA(launch_pdl(k_transpose<T>, dim3(rb, (unsigned)cdiv(dim, 32)), dim3(256), 0, s, m, n_cap, d_n, dim, dim,
                       zt + (size_t)dim * ld, ld, kBK));
    SG_CUDA(launch_pdl(k_transpose<T>, dim3((unsigned)cdiv(kBN, 32), (unsigned)cdiv(two_d, 32)), dim3(256), 0, s, W,
                       (int32_t)kBN, (const int32_t*)nullptr, two_d, two_d, wt, (int32_t)kBN, 1));
    GemmMaps dz, dw;
    memset(&dz, 0, sizeof(dz));
    memset(&dw, 0, sizeof(dw));
    if (!make_map(&dz.a, dy, TF32, kBN, n_cap, (uint64_t)kBN * elem) ||
        !make_map(&dz.b, wt, TF32, kBN, two_d, (uint64_t)kBN * elem) ||
        !make_map(&dw.a, dyt, TF32, ld, kBN, (uint64_t)ld * elem) ||
        !make_map(&dw.b, zt, TF32, ld, two_d, (uint64_t)ld * elem))
        return fail(SG_ERR_CUDA, "sg_sage_bwd: tensor map encoding failed");
    const unsigned n_tiles = (unsigned)cdiv(two_d, kBN);
    sg_status st = launch_gemm<TF32, EPI_DZ>(dz, dim3((unsigned)cdiv(n_cap, kBM), n_tiles, 1), n_cap, d_n, kBN, nullptr,
                                             two_d, dim, dh, dm, dim, s);
    if (st != SG_OK) return st;
    st = launch_gemm<TF32, EPI_SPLIT>(dw, dim3(1, n_tiles, kSplits), kBM, nullptr, n_cap, d_n, two_d, 0, part, nullptr,
                                      two_d, s);
    if (st != SG_OK) return st;
    int64_t sb = cdiv((int64_t)kBM * two_d, 256);
    if (sb > (int64_t)num_sms() * 4) sb = (int64_t)num_sms() * 4;
    SG_CUDA(launch_pdl(k_split_sum, dim3((unsigned)sb), dim3(256), 0, s, (const float*)part, (int32_t)kSplits, two_d,
                       two_d, dW));
    return SG_OK;
}

}  // namespace

extern "C" size_t sg_sage_bwd_workspace(int32_t n_cap, int32_t dim, int32_t dtype) {
    if (n_cap <= 0 || dim <= 0 || (dtype != SG_F32 && dtype != SG_BF16)) return 0;
    return bwd_layout(n_cap, dim, dtype == SG_F32 ? 4 : 2).total;
}

extern "C" sg_status sg_sage_bwd(const void* d_h, const void* d_m, const void* d_W, int32_t dtype, int32_t n_cap,
                                 const int32_t* d_n, int32_t dim, int32_t d_out, const float* d_y, const float* d_g,
                                 float* d_dW, float* d_dh, float* d_dm, void* d_workspace, size_t workspace_bytes,
                                 sg_stream_t stream) {
    if (dtype != SG_F32 && dtype != SG_BF16) return fail(SG_ERR_UNSUPPORTED, "sg_sage_bwd: dtype");
    if (n_cap < 0 || dim <= 0) return fail(SG_ERR_INVALID_ARG, "sg_sage_bwd: bad sizes");
    if (d_out != kBN) return fail(SG_ERR_UNSUPPORTED, "sg_sage_bwd: d_out must be %d", kBN);
    const int64_t elem = dtype == SG_F32 ? 4 : 2;
    if ((dim * elem) % 16) return fail(SG_ERR_UNSUPPORTED, "sg_sage_bwd: rows of %lld bytes are not a multiple of 16",
                                       (long long)(dim * elem));
    if (!d_h || !d_m || !d_W || !d_y || !d_g || !d_dW || !d_dh || !d_dm || !d_workspace)
        return fail(SG_ERR_INVALID_ARG, "sg_sage_bwd: NULL array");
    if (((uintptr_t)d_h | (uintptr_t)d_m | (uintptr_t)d_W) % 16 || ((uintptr_t)d_workspace) % 256)
        return fail(SG_ERR_INVALID_ARG, "sg_sage_bwd: arrays must be 16-byte aligned, the workspace 256-byte aligned");
    const BwdLayout L = bwd_layout(n_cap > 0 ? n_cap : 1, dim, elem);
    if (workspace_bytes < L.total) return fail(SG_ERR_INVALID_ARG, "sg_sage_bwd: workspace needs %zu bytes", L.total);
    cudaStream_t s = (cudaStream_t)stream;
    if (n_cap == 0) {  // no rows: dW = 0
        SG_CUDA(cudaMemsetAsync(d_dW, 0, (size_t)kBN * 2 * dim * sizeof(float), s));
        return SG_OK;
    }
    if (dtype == SG_F32)
        return run_bwd<float, true>((const float*)d_h, (const float*)d_m, (const float*)d_W, n_cap, d_n, dim, d_y, d_g,
                                    d_dW, d_dh, d_dm, (char*)d_workspace, L, s);
    return run_bwd<__nv_bfloat16, false>((const __nv_bfloat16*)d_h, (const __nv_bfloat16*)d_m,
                                         (const __nv_bfloat16*)d_W, n_cap, d_n, dim, d_y, d_g, d_dW, d_dh, d_dm,
                                         (char*)d_workspace, L, s);
}

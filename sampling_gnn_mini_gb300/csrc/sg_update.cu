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
constexpr int kStages = 4;
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
__global__ void __launch_bounds__(kThreads, 1)
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

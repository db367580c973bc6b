// Peak probes, measured in the same run as the operator: a large-tensor copy
// (HBM bandwidth) and a dense bf16 GEMM on the tensor cores (bf16 FLOP/s).
// "Research Sprint Day 2 - Rooflines", section "Rooflines", benchmarks its
// hardware the same way: FLOP/s with 8192 x 8192 by 8192 x 8192 dense
// matmuls, bandwidth by copying a 2 GB tensor.  These are measurement tools,
// not part of the operator.
//
// GEMM: C[M][N] (bf16, row-major) = A[M][K] . B[N][K]^T, both operands
// row-major along K (K-major), fp32 accumulation in tensor memory.  Persistent
// CTAs (one per SM) walk 128 x 256 output tiles; per CTA one warp issues the
// TMA loads of 64-wide K slabs into a 4-stage ring, one warp issues
// tcgen05.mma (M = 128, N = 256, K = 16) into one of two TMEM accumulators,
// and four warps drain the other accumulator (tcgen05.ld -> bf16 -> global)
// while the next tile's products run.  Every wait is bounded; a wait that
// gives up records GDN_ERR_TIMEOUT and the CTA drains what it issued.
#include <cuda.h>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

using namespace sm100;
using namespace tc;

// ------------------------------------------------------------------ copy

__global__ void __launch_bounds__(512) gdn_probe_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                             size_t n16) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // four 16-byte loads in flight per thread
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcs(src + i);
        const uint4 b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride);
        const uint4 d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// ------------------------------------------------------------------ GEMM

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStagesG = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageG = kABytes + kBBytes;
constexpr int kThreadsG = 192;           // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kAccCols = kBN;       // fp32 accumulator columns per buffer
constexpr uint32_t kTmemColsG = 2 * kAccCols;

// barrier slots
constexpr int bFull = 0;                 // [kStagesG] stage loaded (TMA bytes)
constexpr int bEmpty = kStagesG;         // [kStagesG] stage read by the MMAs
constexpr int bTFull = 2 * kStagesG;     // [2] accumulator ready for the epilogue
constexpr int bTEmpty = bTFull + 2;      // [2] accumulator drained (4 epilogue warps)
constexpr int bDrain = bTEmpty + 2;      // every issued MMA completed (abort path)
constexpr int kBarsG = bDrain + 1;

constexpr int oBarG = kStagesG * kStageG;
constexpr int oMiscG = oBarG + kBarsG * 8;   // TMEM slot, abort flag, load counters
constexpr int kAllocG = oMiscG + 16 + 1024;
static_assert(kAllocG <= 232448, "shared memory");

struct GemmArgs {
    uint16_t* C;
    int M, N, K;
    int* err;
    uint32_t wait_limit;
};

// Output tile t of the grouped raster: groups of 8 row blocks, the column
// block fastest within a group column, so one wave of CTAs reads a few row
// blocks of A against a band of B that together fit in L2.
__device__ __forceinline__ void tile_coords(int t, int mt, int nt, int& m0, int& n0) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * nt;
    const int g = t / per_group;
    const int first_m = g * kGroup;
    const int gm = min(kGroup, mt - first_m);
    const int r = t - g * per_group;
    m0 = (first_m + r % gm) * kBM;
    n0 = (r / gm) * kBN;
}

__global__ void __launch_bounds__(kThreadsG, 1)
    gdn_probe_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const GemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBarG);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMiscG);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oMiscG + 4);
    volatile int* loads_issued = reinterpret_cast<volatile int*>(sm + oMiscG + 8);
    volatile int* loads_used = reinterpret_cast<volatile int*>(sm + oMiscG + 12);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = p.M / kBM, nt = p.N / kBN, ntiles = mt * nt;
    const int kblocks = p.K / kBK;
    const uint32_t wl = p.wait_limit;

    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), kTmemColsG);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesG; ++s) {
            mbar_init(bar(bFull + s), 1);
            mbar_init(bar(bEmpty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(bTFull + b), 1);
            mbar_init(bar(bTEmpty + b), 4);
        }
        mbar_init(bar(bDrain), 1);
        fence_mbar_init();
        *abort_flag = 0;
        *loads_issued = 0;
        *loads_used = 0;
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- TMA producer ----
        if (elect_one()) {
            int g = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
                int m0, n0;
                tile_coords(t, mt, nt, m0, n0);
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int s = g % kStagesG;
                    if (g >= kStagesG && !mbar_wait(bar(bEmpty + s), ((g / kStagesG) & 1) ^ 1, wl)) {
                        *abort_flag = 1;
                        break;
                    }
                    uint8_t* st = sm + s * kStageG;
                    mbar_arrive_expect_tx(bar(bFull + s), kStageG);
                    tma_load_2d(smem_u32(st), &tmap_a, kb * kBK, m0, bar(bFull + s));
                    tma_load_2d(smem_u32(st + kABytes), &tmap_b, kb * kBK, n0, bar(bFull + s));
                    *loads_issued = g + 1;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (elect_one()) {
            constexpr uint32_t id = idesc(kFmtBf16, 0, 0, kBM, kBN);
            int g = 0, i = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x, ++i) {
                const int b = i & 1;
                if (i >= 2 && !mbar_wait(bar(bTEmpty + b), ((i >> 1) & 1) ^ 1, wl)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + b * kAccCols;
                bool ok = true;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int s = g % kStagesG;
                    if (!mbar_wait(bar(bFull + s), (g / kStagesG) & 1, wl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sm + s * kStageG);
                    const uint32_t b0 = a0 + kABytes;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // K-major SW128 slabs: 16 K elements = 32 bytes along the row,
                        // 8-row groups 1024 bytes apart
                        mma_bf16(acc, desc_sw128(a0 + k * 32, 0, 1024), desc_sw128(b0 + k * 32, 0, 1024), id,
                                 (kb | k) != 0);
                    }
                    mma_commit(bar(bEmpty + s));  // the stage is free once these products complete
                    *loads_used = g + 1;
                }
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
                mma_commit(bar(bTFull + b));
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = tile rows ----
        const int sub = warp & 3;
        const int row = 32 * sub + lane;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int b = i & 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(bTFull + b), (i >> 1) & 1, wl));
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            int m0, n0;
            tile_coords(t, mt, nt, m0, n0);
            uint16_t* crow = p.C + static_cast<long long>(m0 + row) * p.N + n0;
            const uint32_t base = tmem + (static_cast<uint32_t>(32 * sub) << 16) + b * kAccCols;
#pragma unroll 1
            for (int c = 0; c < kBN; c += 32) {
                float v[32];
                tmem_ld16(base + c, v);
                tmem_ld16(base + c + 16, v + 16);
                tmem_ld_wait();
                uint4 w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
                uint4* dst = reinterpret_cast<uint4*>(crow + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = w[q];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bTEmpty + b));
        }
    }

    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) record_error(p.err, kErrTimeout);
        if (warp == 1) {
            // every product issued so far completes before the TMEM is freed
            if (elect_one()) {
                mma_commit(bar(bDrain));
                mbar_wait(bar(bDrain), 0, wl);
            }
            __syncwarp();
        }
        if (threadIdx.x == 0) {
            // loads issued but never consumed land before the CTA exits
            for (int g = *loads_used; g < *loads_issued; ++g)
                mbar_wait(bar(bFull + g % kStagesG), (g / kStagesG) & 1, wl);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemColsG);
}

// 2-D view {K (inner), rows} of a row-major bf16 [rows][K] operand, box
// {64, box_rows}: 64 K elements = one 128-byte swizzled row per slab row.
bool make_operand_map(CUtensorMap* m, const uint16_t* base, int rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

cudaError_t launch_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
    const size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    gdn_probe_copy_kernel<<<4 * sms, 512, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
    return cudaGetLastError();
}

cudaError_t launch_probe_gemm(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, int* err,
                              cudaStream_t stream) {
    CUtensorMap ma, mb;
    if (!make_operand_map(&ma, A, M, K, kBM) || !make_operand_map(&mb, B, N, K, kBN)) return cudaErrorInvalidValue;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(gdn_probe_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAllocG);
    if (e != cudaSuccess) return e;
    GemmArgs a{C, M, N, K, err, kDefaultWaitLimit};
    const int ntiles = (M / kBM) * (N / kBN);
    gdn_probe_gemm_kernel<<<min(sms, ntiles), kThreadsG, kAllocG, stream>>>(ma, mb, a);
    return cudaGetLastError();
}

}  // namespace gdn

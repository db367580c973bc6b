// Helpers shared by the tensor-core kernels: operand-tile writes (bf16 hi/lo
// split into 128-byte-swizzled rows), TMEM row loads, decay exponentials,
// named barriers and the TMA tensor maps of q/k.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

namespace gdn {
namespace tc {

using namespace sm100;

constexpr int kTile64 = 64 * 128;        // 64 rows x 128 bytes (64 bf16)
constexpr int kRegionBytes = 128 * 128;  // [K rows 0-63 ; Q rows 64-127] x 128 bytes
constexpr int kDk = 128;                 // key width of the tiles

// Bytes to add to the dynamic shared-memory base for 1024-byte alignment.
// Offsetting the shared array itself (rather than rounding its address as an
// integer) lets the compiler keep using shared-memory loads and stores.
__device__ __forceinline__ uint32_t smem_align_pad(const uint8_t* base) {
    return (1024u - (smem_u32(base) & 1023u)) & 1023u;
}

// bar.sync on a named barrier for `count` threads
__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo_elem));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi_elem));
    return a | (b << 16);
}

// Two fp32 -> packed bf16x2 (round to nearest even), element a in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Two values split as x = hi + lo (both bf16, packed in pairs).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = cvt_bf16x2(a, b);
    lo = cvt_bf16x2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

// One 16-byte chunk (8 values, columns 8*ch .. 8*ch+7) of a split row.
__device__ __forceinline__ void store_split_chunk(uint8_t* tile_hi, uint8_t* tile_lo, int row, int ch,
                                                  const float* x8) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_bf16x2(x8[2 * e], x8[2 * e + 1], h[e], l[e]);
    const uint32_t off = sw128_offset(row, ch * 16);
    *reinterpret_cast<uint4*>(tile_hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(tile_lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Half a split row: 32 values, columns 32*hf .. 32*hf+31.
__device__ __forceinline__ void store_split_half(uint8_t* tile_hi, uint8_t* tile_lo, int row, int hf,
                                                 const float* x) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) store_split_chunk(tile_hi, tile_lo, row, 4 * hf + ch, x + 8 * ch);
}

// Half rows of M = 64 accumulators, every lane busy: lane l of warp w holds
// row 16w + (l & 15), columns 32*(l >> 4) .. +31 (no wait).
__device__ __forceinline__ int m64_half_row(int warp, int lane) { return warp * 16 + (lane & 15); }
__device__ __forceinline__ void ld_half32_nowait(uint32_t tmem, int sub, uint32_t col, float* v) {
    tmem_ld_pair32(tmem + (static_cast<uint32_t>(sub * 32) << 16) + col, v);
}
__device__ __forceinline__ void ld_half32(uint32_t tmem, int sub, uint32_t col, float* v) {
    ld_half32_nowait(tmem, sub, col, v);
    tmem_ld_wait();
}

constexpr float kLog2e = 1.4426950408889634f;

// exp(x) for x <= 0 as 2^(x log2 e) by the PTX instruction ex2.approx.ftz.f32
// (relative error about 2^-22 per the PTX ISA reference; results below the
// normal range flush to zero, i.e. decays under 1e-38 are dropped).
__device__ __forceinline__ float exp_nonpos(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * kLog2e));
    return y;
}

// Unpack 8 bf16 (one uint4) into fp32.
__device__ __forceinline__ void unpack8(const uint4& raw, float* out) {
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        out[2 * m] = __uint_as_float(w4[m] << 16);
        out[2 * m + 1] = __uint_as_float(w4[m] & 0xffff0000u);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D view {d (inner), head, token row} of a (rows, H, 128) bf16 tensor; box
// {64, 1, 64} = 64 token rows x 128 bytes, 128-byte swizzled.
inline bool make_qk_map(CUtensorMap* m, const uint16_t* base, long long rows, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDk), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDk) * 2, static_cast<cuuint64_t>(H) * kDk * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {inner, head, token row} of a (rows, H, inner) bf16 tensor, box
// {64, 1, 64}: one 64-column slice of a chunk's rows, 128-byte swizzled.
inline bool make_rows_map(CUtensorMap* m, const uint16_t* base, long long rows, int H, int inner) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, static_cast<cuuint64_t>(H) * inner * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace gdn

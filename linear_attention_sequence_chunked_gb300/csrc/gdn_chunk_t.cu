// T = (I + A)^-1 of every chunk, chunk-parallel: the operand tiles that the
// chunk-chain kernel and the local-gradient pass read.
//
// Per (chunk, head, sequence), with G the running sum of g inside the chunk,
//   A_ij = beta_i (k_i . k_j) exp(G_i - G_j)  (j < i),   T = (I + A)^-1,
// the triangular inverse of the chunk algebra behind the WY tensors w and u
// (fla issue #1550, "Intermediate rounding diagnosis", lists it among the
// intermediates whose bf16 rounding costs accuracy, so it stays fp32 here
// until the final hi/lo split).  The decay is masked before the exponential,
// so every exponent is <= 0.
//
// One CTA (128 threads) per chunk: the K tile in by TMA (d_k = 128; plain
// loads at d_k = 64), K K^T on the tensor cores (one M = 64 product into
// TMEM), A in fp32 in shared memory, T by a blocked inverse (16x16 diagonal
// blocks by substitution, then the off-diagonal blocks as products, level by
// level), and T written to global memory as bf16 hi/lo operand tiles in the
// 128-byte-swizzled layout, tile row c = column c of T.  The work of all
// chunks runs at once (several CTAs per SM), off the serial chunk chain, so
// the kernel is bound by its shared-memory traffic: the layouts below keep
// every access free of bank conflicts and the block products register-blocked
// 4 x 4.  Every element of T is formed by the same sequence of operations as
// in the chunk chain's own inverse (used when no T tiles are given), so both
// routes give the same bits.
#include <cuda.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

using namespace sm100;
using namespace tc;

constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 64;
constexpr int kKRegion = 64 * 128;   // 64 key rows x 128 bytes (64 key columns)
constexpr int kTS = 36;              // row stride of the fp32 32x32 T blocks (rows on distinct banks)
constexpr int kTB = 32 * kTS;
constexpr int kLdA = 68;             // row stride of A^T: 16-byte rows, rows 8 apart on distinct banks

constexpr int oK = 0;                        // K tile, two 64-column regions
constexpr int oA = oK + 2 * kKRegion;        // A^T fp32 [64][kLdA]
constexpr int oTf = oK;                      // T_00, T_11, T_10 fp32 32x32 blocks (K is dead once K K^T is done)
constexpr int oVec = oA + 64 * kLdA * 4;     // g, beta, G x 64 fp32
constexpr int oBar = oVec + 3 * 64 * 4;      // K K^T done, K tile in
constexpr int oMisc = oBar + 16;
constexpr int kBytes = oMisc + 16;
constexpr int kAlloc = kBytes + 1024;
static_assert(3 * kTB * 4 <= 2 * kKRegion, "T blocks fit in the K tile");
static_assert(kChunkTBytes <= 64 * kLdA * 4, "the T tile stage fits in the A^T scratch");

__global__ void __launch_bounds__(kThreads, 6)
    gdn_chunk_t_kernel(const __grid_constant__ CUtensorMap tmap_k, const ChunkTArgs p) {
    const int ci = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, dk = p.d_k;
    const int q = threadIdx.x;
    const int warp = q >> 5, lane = q & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    if (ci >= nchunks) return;
    const int c0 = t0 + ci * kChunk;
    const int nv = min(kChunk, t1 - c0);
    const long long row_base = static_cast<long long>(b) * p.T;
    const long long slot = chunk_slot_base(p.cu_seqlens, n, p.T) + ci;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    float* At = reinterpret_cast<float*>(sm + oA);  // A^T, row stride kLdA
    float* T00 = reinterpret_cast<float*>(sm + oTf);
    float* T11 = T00 + kTB;
    float* T10 = T00 + 2 * kTB;
    float* gv = reinterpret_cast<float*>(sm + oVec);
    float* bv = gv + 64;
    float* Gv = gv + 128;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMisc);
    const uint32_t bar = smem_u32(sm + oBar);
    const uint32_t kbar = smem_u32(sm + oBar + 8);
    const bool use_tma = dk == kDk;

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (q == 0) {
        mbar_init(bar, 1);
        mbar_init(kbar, 1);
        fence_mbar_init();
        if (use_tma) tma_prefetch_desc(&tmap_k);
    }
    float gq = 0.f, bq = 0.f;
    if (q < nv) {
        const long long idx = (row_base + c0 + q) * H + h;
        gq = p.g[idx];
        bq = bf16_to_f32(p.beta[idx]);
    }
    if (!use_tma) {
        // d_k = 64: the K tile by plain loads (rows beyond the chunk and key
        // columns beyond d_k are zero), every load in flight before the first store
        constexpr int kPer = 2 * 64 * 8 / kThreads;
        uint4 val[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = q + u * kThreads, region = e >> 9, r = (e >> 3) & 63, ch = e & 7;
            val[u] = make_uint4(0, 0, 0, 0);
            if (r < nv && region * 64 < dk)
                val[u] = *reinterpret_cast<const uint4*>(p.k + ((row_base + c0 + r) * H + h) * static_cast<long long>(dk) +
                                                         region * 64 + ch * 8);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = q + u * kThreads, region = e >> 9, r = (e >> 3) & 63, ch = e & 7;
            *reinterpret_cast<uint4*>(sm + oK + region * kKRegion + sw128_offset(r, ch * 16)) = val[u];
        }
    }
    __syncthreads();  // barriers initialised
    // d_k = 128: two 64-column boxes of the chunk's 64 token rows, issued
    // before the gate loads land
    if (use_tma && q == 0) {
        const int z = static_cast<int>(row_base + c0);
        mbar_arrive_expect_tx(kbar, 2 * kKRegion);
        tma_load_3d(smem_u32(sm + oK), &tmap_k, 0, h, z, kbar);
        tma_load_3d(smem_u32(sm + oK + kKRegion), &tmap_k, 64, h, z, kbar);
    }
    if (q < 64) {
        gv[q] = gq;
        bv[q] = bq;
    }
    bool ok = true;
    if (use_tma) {
        ok = mbar_wait(kbar, 0, kDefaultWaitLimit);
        if (nv < kChunk) {
            // the boxes also read the rows after the chunk: zero them
            for (int e = q; e < 2 * 64 * 8; e += kThreads) {
                const int region = e >> 9, r = (e >> 3) & 63, ch = e & 7;
                if (r >= nv)
                    *reinterpret_cast<uint4*>(sm + oK + region * kKRegion + sw128_offset(r, ch * 16)) =
                        make_uint4(0, 0, 0, 0);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // K K^T (M = 64): rows 16 w .. 16 w + 15 land in lanes 0-15 of subpartition w
    if (warp == 0) {
        if (elect_one()) {
            tc_fence_after();
            constexpr uint32_t id = idesc(kFmtBf16, 0, 0, 64, 64);
            const uint32_t ak = smem_u32(sm + oK);
#pragma unroll
            for (int s = 0; s < kDk / 16; ++s) {
                const uint64_t a = desc_sw128(ak + (s >> 2) * kKRegion + (s & 3) * 32, 0, 1024);
                mma_bf16(tmem, a, a, id, s > 0);
            }
            mma_commit(bar);
        }
        __syncwarp();
    }
    // running sum G of g in the chunk
    if (q < 32) {
        const float a = gv[2 * q];
        const float bb = a + gv[2 * q + 1];
        float s = bb;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, s, off);
            if (q >= off) s += o;
        }
        Gv[2 * q] = s - bb + a;
        Gv[2 * q + 1] = s;
    }
    __syncwarp();
    const bool ok_mma = mbar_wait(bar, 0, kDefaultWaitLimit);
    tc_fence_after();
    __syncthreads();

    // A: thread (warp w, lane l) takes row i = 16 w + l % 16, columns 32 (l / 16) .. + 31
    // (lanes l and l + 16 read the two column halves of TMEM row i)
    {
        const int i = 16 * warp + (lane & 15), hf = lane >> 4, j0 = 32 * hf;
        const float Gi = Gv[i], bi = bv[i];
        float mdec[32];
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
            const float4 g4 = *reinterpret_cast<const float4*>(Gv + j0 + 4 * k4);
            const float gj[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 4 * k4 + e;
                mdec[k] = (j0 + k < i) ? exp_nonpos(Gi - gj[e]) : 0.f;
            }
        }
        float lo[32];
        ld_half32(tmem, warp, 0, lo);
#pragma unroll
        for (int k = 0; k < 32; ++k) lo[k] = bi * lo[k] * mdec[k];
        // stores after the loop: they may alias the decay loads.  At step k
        // lanes 0-15 write row k of A^T and lanes 16-31 row 32 + (k + 4) % 32:
        // rows 36 apart, so the two half-warps fall on disjoint banks
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int kk = hf ? ((k + 4) & 31) : k;
            At[(j0 + kk) * kLdA + i] = hf ? lo[(k + 4) & 31] : lo[k];
        }
    }
    tc_fence_before();
    __syncthreads();

    // T_bb = (I + A_bb)^-1 for the four 16x16 diagonal blocks: column c of
    // block d (q < 64) by right-looking forward substitution, x = e_c;
    // for m: for i > m: x_i -= A_im x_m.  Row m of A^T is read as broadcast
    // 16-byte loads.
    if (q < 64) {
        const int d = q >> 4, c = q & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
        const float* ablk = At + 16 * d * kLdA + 16 * d;
#pragma unroll
        for (int m = 0; m < 15; ++m) {
            const float xm = x[m];
            const float4* arow = reinterpret_cast<const float4*>(ablk + m * kLdA);
#pragma unroll
            for (int i4 = (m + 1) >> 2; i4 < 4; ++i4) {
                const float4 a4 = arow[i4];
                if (4 * i4 + 0 > m) x[4 * i4 + 0] = fmaf(-a4.x, xm, x[4 * i4 + 0]);
                if (4 * i4 + 1 > m) x[4 * i4 + 1] = fmaf(-a4.y, xm, x[4 * i4 + 1]);
                if (4 * i4 + 2 > m) x[4 * i4 + 2] = fmaf(-a4.z, xm, x[4 * i4 + 2]);
                if (4 * i4 + 3 > m) x[4 * i4 + 3] = fmaf(-a4.w, xm, x[4 * i4 + 3]);
            }
        }
        // into the 32x32 block T_bb (b = d / 2) at rows/columns 16 (d % 2) ..;
        // the upper-right 16x16 block of T_bb is zero
        float* tb = (d >> 1 ? T11 : T00) + (16 * (d & 1)) * (kTS + 1) + c;
#pragma unroll
        for (int i = 0; i < 16; ++i) tb[i * kTS] = x[i];
        if (!(d & 1)) {
#pragma unroll
            for (int i = 0; i < 16; ++i) tb[i * kTS + 16] = 0.f;
        }
    }
    __syncthreads();
    {
        // lower-left 16x16 block of T_bb (b = 0, 1): X = A_10 T_00 (16x16
        // blocks of the 32x32 diagonal block); threads q < 32 take a 4x4 block
        // of X (block b = q / 16, rows r4 .. r4 + 3, columns c4 .. c4 + 3):
        // per k one 16-byte load of A_10's column and one of T_00's row
        if (q < 32) {
            const int b4 = q >> 4, r4 = ((q >> 2) & 3) * 4, c4 = (q & 3) * 4;
            const float* tb = b4 ? T11 : T00;
            const int o = 32 * b4;
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float4 a4 = *reinterpret_cast<const float4*>(At + (o + k) * kLdA + o + 16 + r4);
                const float4 t4 = *reinterpret_cast<const float4*>(tb + k * kTS + c4);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][0] = fmaf(av[i], t4.x, acc[i][0]); acc[i][1] = fmaf(av[i], t4.y, acc[i][1]);
                    acc[i][2] = fmaf(av[i], t4.z, acc[i][2]); acc[i][3] = fmaf(av[i], t4.w, acc[i][3]);
                }
            }
            float* xs4 = At + (o + 16) * kLdA + o;  // upper triangle of A^T: free
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(xs4 + (r4 + i) * kLdA + c4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        __syncthreads();
        // T_10 = -T_11 X (T_11 the lower-right 16x16 block, unit lower
        // triangular), block b = q / 64, thread q: row r, columns c4 .. c4 + 3
        const int bb = q >> 6, r = (q >> 2) & 15, c4 = (q & 3) * 4;
        float* tb = bb ? T11 : T00;
        const int o = 32 * bb;  // first row/column of the 32x32 block in A
        float* xs = At + (o + 16) * kLdA + o;
        float4 acc = *reinterpret_cast<const float4*>(xs + r * kLdA + c4);
#pragma unroll 4
        for (int k = 0; k < r; ++k) {
            const float a = tb[(16 + r) * kTS + 16 + k];
            const float4 v4 = *reinterpret_cast<const float4*>(xs + k * kLdA + c4);
            acc.x = fmaf(a, v4.x, acc.x); acc.y = fmaf(a, v4.y, acc.y);
            acc.z = fmaf(a, v4.z, acc.z); acc.w = fmaf(a, v4.w, acc.w);
        }
        *reinterpret_cast<float4*>(tb + (16 + r) * kTS + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
    {
        // T_10 of the 64x64 matrix: X = A_10 T_00 (32x32 blocks), threads
        // q < 64 take a 4x4 block of X (rows r4 .. r4 + 3, columns c4 .. c4 + 3):
        // per k one 16-byte load of A_10's column (contiguous in A^T) and one
        // of T_00's row for 16 FMAs; each element sums over k in order.  Warp 1
        // holds columns 16-31, where T_00 is zero for k < 16: it starts at k = 16
        float* xs = At + 32 * kLdA;  // rows 32-63, columns 0-31 of A^T: free
        if (q < 64) {
            const int w = q >> 5, l = q & 31;
            const int r4 = 4 * (l >> 2), c4 = 16 * w + 4 * (l & 3);
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
#pragma unroll 8
            for (int k = 16 * w; k < 32; ++k) {
                const float4 a4 = *reinterpret_cast<const float4*>(At + k * kLdA + 32 + r4);
                const float4 t4 = *reinterpret_cast<const float4*>(T00 + k * kTS + c4);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][0] = fmaf(av[i], t4.x, acc[i][0]); acc[i][1] = fmaf(av[i], t4.y, acc[i][1]);
                    acc[i][2] = fmaf(av[i], t4.z, acc[i][2]); acc[i][3] = fmaf(av[i], t4.w, acc[i][3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(xs + (r4 + i) * kLdA + c4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
        __syncthreads();
        // T_10 = -T_11 X (T_11 unit lower triangular): threads q < 64 take a
        // 4x4 block (rows r4 .. r4 + 3, columns c4 .. c4 + 3), k in steps of
        // four: per step four 16-byte rows of X and four of T_11 (the latter
        // one address per quarter warp) for 64 FMAs.  Row r sums X[r] and then
        // T_11[r][k] X[k] for k = 0 .. r - 1 in order
        if (q < 64) {
            const int r4 = 4 * (q >> 3), c4 = 4 * (q & 7);
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 u = *reinterpret_cast<const float4*>(xs + (r4 + i) * kLdA + c4);
                acc[i][0] = u.x; acc[i][1] = u.y; acc[i][2] = u.z; acc[i][3] = u.w;
            }
            for (int k4 = 0; k4 <= r4; k4 += 4) {
                float xk[4][4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float4 u = *reinterpret_cast<const float4*>(xs + (k4 + kk) * kLdA + c4);
                    xk[kk][0] = u.x; xk[kk][1] = u.y; xk[kk][2] = u.z; xk[kk][3] = u.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 t = *reinterpret_cast<const float4*>(T11 + (r4 + i) * kTS + k4);
                    const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (k4 + kk < r4 + i) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[i][e] = fmaf(tv[kk], xk[kk][e], acc[i][e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(T10 + (r4 + i) * kTS + c4) = make_float4(-acc[i][0], -acc[i][1], -acc[i][2], -acc[i][3]);
        }
    }
    __syncthreads();
    {
        // column col of T = row col of the tile (read MN-major for T, K-major
        // for T^T); this thread writes entries 32 hf .. 32 hf + 31 of it.  The
        // hi/lo tiles are staged in the A^T scratch (dead now) and leave in
        // one 16 KB bulk copy: per-thread 16-byte stores into 128-byte tile
        // rows would each touch their own sector
        const int col = q & 63, hf = q >> 6;
        const float* src = col < 32 ? (hf ? T10 : T00) : (hf ? T11 : nullptr);
        const int cc = col & 31;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src ? src[i * kTS + cc] : 0.f;
        uint8_t* stage = sm + oA;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) store_split_chunk(stage, stage + kTile64, col, 4 * hf + c4, v + 8 * c4);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (q == 0) {
        // the CTA may leave once the copy has read its source; the write
        // itself completes before the kernel does
        bulk_s2g(p.chunk_T + (slot * H + h) * static_cast<long long>(kChunkTBytes), smem_u32(sm + oA), kChunkTBytes);
        bulk_commit();
        bulk_wait_read_all();
    }
    if (!ok || !ok_mma) {  // a copy or the product never signalled: record it and let both land
        record_error(p.err, kErrTimeout);
        if (q == 0) {
            if (!ok) mbar_wait(kbar, 0, kDefaultWaitLimit);
            mbar_wait(bar, 0, kDefaultWaitLimit);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_t(const ChunkTArgs& a, cudaStream_t stream) {
    if (a.max_chunks == 0) return cudaSuccess;
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    CUtensorMap mk;  // d_k = 128 only (d_k = 64 tiles use plain loads)
    memset(&mk, 0, sizeof(mk));
    if (rows > 0 && a.d_k == kDk && !make_qk_map(&mk, a.k, rows, a.H)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_chunk_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_chunks, a.H, a.N);
    gdn_chunk_t_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, a);
    return cudaGetLastError();
}

}  // namespace gdn

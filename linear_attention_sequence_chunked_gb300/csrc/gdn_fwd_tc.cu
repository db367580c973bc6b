// Chunked gated delta rule forward on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), q/k tiles brought in by TMA.
//
// One CTA (128 threads) per (64-column value slice, head, sequence) walks
// the chunks in order, holding its d_k x 64 fp32 state slice S in registers
// (thread d owns row d).  Per chunk of 64 tokens, with G the running sum of
// g (log decay kept as a cumsum, "Research Sprint Day 2 - Rooflines", GDN
// layer pseudocode step 5) and gam = exp(G), dec_j = exp(G_n - G_j):
//   [K;Q] K^T          -> A = beta_i (k_i.k_j) exp(G_i - G_j) (j < i)
//                         P = (q_i.k_j) exp(G_i - G_j)       (j <= i)
//   T  = (I + A)^-1       fp32 blocked forward substitution on CUDA cores
//   K S, Q S           -> R = beta o (V - gam o (K S))
//   Delta = T R        (= u - w S of the WY form: u = T diag(beta) V,
//                         w = T diag(beta gam) K; it is beta_i times the
//                         error v_i - v_old_i of the page-1 GDN update loop)
//   O  = scale [gam o (Q S) + P Delta]
//   S <- gam_n S + K^T (dec o Delta)
// fla issue #1550 ("Intermediate rounding diagnosis") traces the error of
// earlier chunk kernels to bf16 rounding of the triangular inverse, the
// causal score, the WY tensors and u.  Here every computed MMA operand
// (S, R, T, P, Delta) is split into bf16 hi + lo parts (x = hi + lo with
// |lo| <= 2^-9 |x|) and multiplied as hi*hi + hi*lo + lo*hi (or hi + lo
// against an exact bf16 input), so the products carry ~16 mantissa bits;
// all accumulation is fp32 in TMEM.
//
// Shared-memory operands use the 128-byte swizzle: 8-row atoms of 1024
// bytes, 16-byte chunk index XOR (row % 8).  The K and Q tiles of a chunk
// share one region per 64 key columns ([K rows 0-63 ; Q rows 64-127]) so
// that [K;Q] K^T is a single M = 128 product.
#include <cuda.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kVs = 64;       // value columns per CTA
constexpr int kStages = 2;    // K/Q tile stages (TMA double buffer)
constexpr int kLd = 65;       // fp32 row stride of A / T scratch
constexpr uint32_t kTmemCols = 512;

// TMEM column map (fp32 accumulators)
constexpr uint32_t kColG = 0;     // [K;Q] K^T, M = 128, 64 columns
constexpr uint32_t kColKS = 64;   // K S, M = 64
constexpr uint32_t kColQS = 128;  // Q S, M = 64
constexpr uint32_t kColD = 192;   // Delta = T R, M = 64
constexpr uint32_t kColPD = 256;  // P Delta, M = 64
constexpr uint32_t kColS = 320;   // K^T (dec o Delta), M = d_k

template <int K>
struct TcSmem {  // instantiated for K = 128 only (d_k = 64 zero-fills the upper half)
    static constexpr int kRegions = K / 64;             // 64-column key regions
    static constexpr int kRegionBytes = 128 * 128;      // [K;Q] rows x 128 B
    static constexpr int kStageBytes = kRegions * kRegionBytes;
    static constexpr int kTile64 = 64 * 128;            // 64 rows x 128 B
    static constexpr int kTileS = K * 128;              // K rows x 128 B
    // byte offsets (all 1024-aligned)
    static constexpr int oStage = 0;
    static constexpr int oShi = oStage + kStages * kStageBytes;
    static constexpr int oSlo = oShi + kTileS;
    static constexpr int oRhi = oSlo + kTileS;   // R, later dec o Delta
    static constexpr int oRlo = oRhi + kTile64;
    static constexpr int oDhi = oRlo + kTile64;  // Delta
    static constexpr int oDlo = oDhi + kTile64;
    static constexpr int oPhi = oDlo + kTile64;  // P
    static constexpr int oPlo = oPhi + kTile64;
    static constexpr int oThi = oPlo + kTile64;  // T
    static constexpr int oTlo = oThi + kTile64;
    static constexpr int oA = oTlo + kTile64;    // fp32 A [64][kLd]
    static constexpr int oTf = oA + 64 * kLd * 4;  // fp32 T [64][kLd]
    static constexpr int oX = oTf + 64 * kLd * 4;  // fp32 3 x 16 x 16
    static constexpr int oVec = oX + 3 * 256 * 4;  // g, beta, G, gam, dec (5 x 64 fp32)
    static constexpr int oBar = oVec + 5 * 64 * 4; // mbarriers (8 x 8 B) + TMEM slot + flag
    static constexpr int kBytes = oBar + 128;
    static constexpr int kAlloc = kBytes + 1024;   // slack for 1024 alignment
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo_elem));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi_elem));
    return a | (b << 16);
}

// Split 64 fp32 values into bf16 hi / lo rows of two swizzled 128-byte tiles.
__device__ __forceinline__ void store_split_row(uint8_t* tile_hi, uint8_t* tile_lo, int row, const float* x) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = x[ch * 8 + 2 * e], b = x[ch * 8 + 2 * e + 1];
            const float ah = __bfloat162float(__float2bfloat16_rn(a));
            const float bh = __bfloat162float(__float2bfloat16_rn(b));
            h[e] = pack_bf16x2(ah, bh);
            l[e] = pack_bf16x2(a - ah, b - bh);
        }
        const uint32_t off = sw128_offset(row, ch * 16);
        *reinterpret_cast<uint4*>(tile_hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(tile_lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// TMEM row ownership.  M = 128 accumulators: row r in lane r.  M = 64
// accumulators (cta_group::1): rows 16w..16w+15 in lanes 32w..32w+15.
__device__ __forceinline__ int m64_row(int warp, int lane) { return lane < 16 ? warp * 16 + lane : -1; }

__device__ __forceinline__ void ld_row64(uint32_t tmem, int warp, uint32_t col, float* v) {
    const uint32_t a = tmem + (static_cast<uint32_t>(warp * 32) << 16) + col;
    tmem_ld16(a, v);
    tmem_ld16(a + 16, v + 16);
    tmem_ld16(a + 32, v + 32);
    tmem_ld16(a + 48, v + 48);
    tmem_ld_wait();
}

// fp32 blocked inverse of the unit lower triangular (I + A), A strictly
// lower in smem (row stride kLd); writes Tf (row stride kLd, upper zero).
// X is a 3 x 16 x 16 scratch.  All 128 threads call it.
__device__ __forceinline__ void tri_inverse(const float* A, float* Tf, float* X) {
    for (int e = threadIdx.x; e < 64 * 64; e += kThreads) {
        const int i = e >> 6, j = e & 63;
        if ((i >> 4) != (j >> 4)) Tf[i * kLd + j] = 0.f;
    }
    if (threadIdx.x < 64) {
        const int o = (threadIdx.x >> 4) * 16;
        const int c = threadIdx.x & 15;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < i) acc = fmaf(-A[(o + i) * kLd + o + j], col[j], acc);
            col[i] = (i < c) ? 0.f : acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[(o + i) * kLd + o + c] = col[i];
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
        const int nblk = 4 - dist;
        for (int e = threadIdx.x; e < nblk * 256; e += kThreads) {
            const int bi = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int I = bi + dist, J = bi;
            float acc = 0.f;
            for (int L = J; L < I; ++L)
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(A[(I * 16 + r) * kLd + L * 16 + m], Tf[(L * 16 + m) * kLd + J * 16 + c], acc);
            X[bi * 256 + r * 16 + c] = acc;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < nblk * 256; e += kThreads) {
            const int bi = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int I = bi + dist, J = bi;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                acc = fmaf(Tf[(I * 16 + r) * kLd + I * 16 + m], X[bi * 256 + m * 16 + c], acc);
            Tf[(I * 16 + r) * kLd + J * 16 + c] = -acc;
        }
        __syncthreads();
    }
}

struct TcParams {
    FwdArgs a;
    uint32_t wait_limit;
};

template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                      const TcParams prm) {
    using L = TcSmem<K>;
    constexpr int R = L::kRegions;
    const FwdArgs& p = prm.a;
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* Shi = sm + L::oShi;
    uint8_t* Slo = sm + L::oSlo;
    uint8_t* Rhi = sm + L::oRhi;
    uint8_t* Rlo = sm + L::oRlo;
    uint8_t* Dhi = sm + L::oDhi;
    uint8_t* Dlo = sm + L::oDlo;
    uint8_t* Phi = sm + L::oPhi;
    uint8_t* Plo = sm + L::oPlo;
    uint8_t* Thi = sm + L::oThi;
    uint8_t* Tlo = sm + L::oTlo;
    float* Am = reinterpret_cast<float*>(sm + L::oA);
    float* Tf = reinterpret_cast<float*>(sm + L::oTf);
    float* X = reinterpret_cast<float*>(sm + L::oX);
    float* gv = reinterpret_cast<float*>(sm + L::oVec);
    float* bv = gv + 64;
    float* Gv = bv + 64;
    float* gam = Gv + 64;
    float* dec = gam + 64;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::oBar);  // [0,1] TMA stages, [2] MMA
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::oBar + 64);
    int* abort_flag = reinterpret_cast<int*>(sm + L::oBar + 68);

    const uint32_t bar_tma0 = smem_u32(&bars[0]);
    const uint32_t bar_mma = smem_u32(&bars[2]);

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar_tma0 + 8 * s, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *abort_flag = 0;
        if (p.d_k == 128) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    const int dk = p.d_k;                                       // 64 or 128
    const long long row_base = static_cast<long long>(b) * p.T;  // token-row of t = 0
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);
    const long long KV = static_cast<long long>(dk) * V;
    const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kVs;

    // TMA issue for chunk ci into stage ci % kStages (thread 0 only)
    auto issue_tma = [&](int ci) {
        const int st = ci % kStages;
        const uint32_t bar = bar_tma0 + 8 * st;
        uint8_t* base = sm + L::oStage + st * L::kStageBytes;
        const int z = static_cast<int>(row_base + t0 + ci * kChunk);
        mbar_arrive_expect_tx(bar, (dk / 64) * L::kRegionBytes);
        for (int r = 0; r < dk / 64; ++r) {
            tma_load_3d(smem_u32(base + r * L::kRegionBytes), &tmap_k, r * 64, h, z, bar);
            tma_load_3d(smem_u32(base + r * L::kRegionBytes + 64 * 128), &tmap_q, r * 64, h, z, bar);
        }
    };
    // d_k = 64: the upper 64 key columns of every K/Q tile are zero and never loaded
    if (dk < 64 * R) {
        for (int st = 0; st < kStages; ++st) {
            uint4* z = reinterpret_cast<uint4*>(sm + L::oStage + st * L::kStageBytes + (dk / 64) * L::kRegionBytes);
            const int n16 = (R - dk / 64) * L::kRegionBytes / 16;
            for (int i = threadIdx.x; i < n16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncthreads();
    }
    // d_k = 128 streams K/Q tiles with TMA; d_k = 64 loads them with plain
    // vector loads (only the first key region is populated).
    const bool use_tma = dk == 64 * R;
    if (use_tma && threadIdx.x == 0) {
        for (int ci = 0; ci < kStages && ci < nchunks; ++ci) issue_tma(ci);
    }

    // ---- state slice in registers: M = d_k accumulator row ownership ----
    // d_k = 128: thread r owns row r.  d_k = 64: M = 64 layout.
    // S update accumulator is M = 128: thread r owns state row r; rows >= d_k
    // stay zero (their key columns are zero-filled).
    const int srow = static_cast<int>(threadIdx.x) < dk ? static_cast<int>(threadIdx.x) : -1;
    static_assert(K == 128, "one instantiation");
    float S[kVs];
#pragma unroll
    for (int j = 0; j < kVs; ++j) S[j] = 0.f;
    if (srow >= 0 && p.initial_state) {
        const float* src = p.initial_state + state_off + static_cast<long long>(srow) * V;
#pragma unroll
        for (int j = 0; j < kVs; j += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(src + j);
            S[j] = t4.x; S[j + 1] = t4.y; S[j + 2] = t4.z; S[j + 3] = t4.w;
        }
    }
    store_split_row(Shi, Slo, threadIdx.x, S);  // rows >= d_k are zero
    fence_proxy_async_smem();
    __syncthreads();

    const int mrow = m64_row(warp, lane);  // row of M = 64 accumulators
    const float scale = p.scale;
    uint32_t mma_phase = 0;
    bool aborted = false;

    // MMA completion: the phase only advances on success, so that after a
    // timeout the drain below waits for the same, still pending, commit.
    auto wait_mma = [&]() -> bool {
        const bool ok = mbar_wait(bar_mma, mma_phase, prm.wait_limit);
        if (ok) mma_phase ^= 1u;
        else *abort_flag = 1;
        tc_fence_after();
        return ok;
    };
    const bool want_out = p.out != nullptr;
    int tma_issued = use_tma ? min(kStages, nchunks) : 0;  // chunks whose K/Q load was issued
    int tma_done = 0;                         // chunks whose K/Q load was waited for

    for (int ci = 0; ci < nchunks; ++ci) {
        const int c0 = t0 + ci * kChunk;
        const int nv = min(kChunk, t1 - c0);
        const int st = ci % kStages;
        uint8_t* stage = sm + L::oStage + st * L::kStageBytes;
        const uint32_t stage_a = smem_u32(stage);

        if (p.chunk_states && srow >= 0) {
            float* dst = p.chunk_states + ((slot0 + ci) * H + h) * KV + vs * kVs + static_cast<long long>(srow) * V;
#pragma unroll
            for (int j = 0; j < kVs; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        // per-token gates of this chunk (zero beyond the sequence end)
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            const long long idx = (row_base + c0 + r) * H + h;
            gv[r] = (r < nv) ? p.g[idx] : 0.f;
            bv[r] = (r < nv) ? bf16_to_f32(p.beta[idx]) : 0.f;
        }
        // value row of this slice for R (row mrow), loaded early as packed bf16
        uint4 vraw[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) vraw[ch] = make_uint4(0, 0, 0, 0);
        if (mrow >= 0 && mrow < nv) {
            const uint4* src = reinterpret_cast<const uint4*>(
                p.v + ((row_base + c0 + mrow) * H + h) * static_cast<long long>(V) + vs * kVs);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) vraw[ch] = src[ch];
        }
        // this chunk's K/Q tiles
        if (use_tma) {
            const bool ok = mbar_wait(bar_tma0 + 8 * st, (ci / kStages) & 1, prm.wait_limit);
            if (!ok) *abort_flag = 1;
        } else {
            for (int e = threadIdx.x; e < 2 * 64 * 8; e += kThreads) {
                const int which = e >> 9;          // 0: K, 1: Q
                const int r = (e >> 3) & 63, ch = e & 7;
                uint4 val = make_uint4(0, 0, 0, 0);
                if (r < nv) {
                    const uint16_t* src = which ? p.q : p.k;
                    val = *reinterpret_cast<const uint4*>(src + ((row_base + c0 + r) * H + h) * 64LL + ch * 8);
                }
                *reinterpret_cast<uint4*>(stage + which * 64 * 128 + sw128_offset(r, ch * 16)) = val;
            }
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (*abort_flag) { aborted = true; break; }
        tma_done = ci + 1;
        chunk_cumsum(gv, Gv, gam);

        // ---- MMA 1: [K;Q] K^T, K S, Q S ----
        if (threadIdx.x == 0) {
            tc_fence_after();
            constexpr uint32_t id_g = idesc(kFmtBf16, 0, 0, 128, 64);
            constexpr uint32_t id_s = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
            for (int s = 0; s < K / 16; ++s) {
                const uint32_t koff = (s >> 2) * L::kRegionBytes + (s & 3) * 32;
                const uint64_t a_kq = desc_sw128(stage_a + koff, 0, 1024);
                mma_bf16(tmem + kColG, a_kq, a_kq, id_g, s > 0);  // B = K rows 0-63 (N = 64)
            }
#pragma unroll
            for (int s = 0; s < K / 16; ++s) {
                const uint32_t koff = (s >> 2) * L::kRegionBytes + (s & 3) * 32;
                const uint64_t a_k = desc_sw128(stage_a + koff, 0, 1024);
                const uint64_t a_q = desc_sw128(stage_a + koff + 64 * 128, 0, 1024);
                const uint64_t b_hi = desc_sw128(smem_u32(Shi) + s * 2048, L::kTileS, 1024);
                const uint64_t b_lo = desc_sw128(smem_u32(Slo) + s * 2048, L::kTileS, 1024);
                mma_bf16(tmem + kColKS, a_k, b_hi, id_s, s > 0);
                mma_bf16(tmem + kColKS, a_k, b_lo, id_s, 1);
                if (want_out) {
                    mma_bf16(tmem + kColQS, a_q, b_hi, id_s, s > 0);
                    mma_bf16(tmem + kColQS, a_q, b_lo, id_s, 1);
                }
            }
            mma_commit(bar_mma);
        }
        __syncthreads();  // cumsum results visible
        if (threadIdx.x < 64) dec[threadIdx.x] = expf(Gv[63] - Gv[threadIdx.x]);
        wait_mma();
        __syncthreads();
        if (*abort_flag) { aborted = true; break; }

        // ---- A, P from the gram; R from K S ----
        {
            float row[64];
            ld_row64(tmem, warp, kColG, row);
            const int r = threadIdx.x;
            if (r < 64) {
                const float Gi = Gv[r], bi = bv[r];
#pragma unroll
                for (int j = 0; j < 64; ++j) Am[r * kLd + j] = (j < r) ? bi * row[j] * expf(Gi - Gv[j]) : 0.f;
            } else {
                const int i = r - 64;
                const float Gi = Gv[i];
#pragma unroll
                for (int j = 0; j < 64; ++j) row[j] = (j <= i) ? row[j] * expf(Gi - Gv[j]) : 0.f;
                store_split_row(Phi, Plo, i, row);
            }
            ld_row64(tmem, warp, kColKS, row);
            if (mrow >= 0) {
                const float bj = bv[mrow], gj = gam[mrow];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t w4[4] = {vraw[ch].x, vraw[ch].y, vraw[ch].z, vraw[ch].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int c = ch * 8 + 2 * m;
                        row[c] = bj * (__uint_as_float(w4[m] << 16) - gj * row[c]);
                        row[c + 1] = bj * (__uint_as_float(w4[m] & 0xffff0000u) - gj * row[c + 1]);
                    }
                }
                store_split_row(Rhi, Rlo, mrow, row);
            }
        }
        __syncthreads();
        tri_inverse(Am, Tf, X);
        if (threadIdx.x < 64) {
            float row[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) row[j] = Tf[threadIdx.x * kLd + j];
            store_split_row(Thi, Tlo, threadIdx.x, row);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- MMA 2: Delta = T R (hi*hi + hi*lo + lo*hi) ----
        if (threadIdx.x == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t th = desc_sw128(smem_u32(Thi) + s * 32, 0, 1024);
                const uint64_t tl = desc_sw128(smem_u32(Tlo) + s * 32, 0, 1024);
                const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, L::kTile64, 1024);
                const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, L::kTile64, 1024);
                mma_bf16(tmem + kColD, th, rh, id, s > 0);
                mma_bf16(tmem + kColD, th, rl, id, 1);
                mma_bf16(tmem + kColD, tl, rh, id, 1);
            }
            mma_commit(bar_mma);
        }
        __syncwarp();
        wait_mma();
        __syncthreads();
        if (*abort_flag) { aborted = true; break; }

        // ---- Delta -> Delta tiles (for P Delta) and dec o Delta (for S) ----
        {
            float row[64];
            ld_row64(tmem, warp, kColD, row);
            if (mrow >= 0) {
                store_split_row(Dhi, Dlo, mrow, row);
                const float dj = dec[mrow];
#pragma unroll
                for (int c = 0; c < kVs; ++c) row[c] *= dj;
                store_split_row(Rhi, Rlo, mrow, row);  // R is dead: reuse for dec o Delta
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- MMA 3: S update K^T (dec o Delta); P Delta ----
        if (threadIdx.x == 0) {
            tc_fence_after();
            constexpr uint32_t id_s = idesc(kFmtBf16, 1, 1, K, 64);
            constexpr uint32_t id_p = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ak = desc_sw128(stage_a + s * 2048, L::kRegionBytes, 1024);
                const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, L::kTile64, 1024);
                const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, L::kTile64, 1024);
                mma_bf16(tmem + kColS, ak, rh, id_s, s > 0);
                mma_bf16(tmem + kColS, ak, rl, id_s, 1);
            }
#pragma unroll
            for (int s = 0; s < 4 && want_out; ++s) {
                const uint64_t ph = desc_sw128(smem_u32(Phi) + s * 32, 0, 1024);
                const uint64_t pl = desc_sw128(smem_u32(Plo) + s * 32, 0, 1024);
                const uint64_t dh = desc_sw128(smem_u32(Dhi) + s * 2048, L::kTile64, 1024);
                const uint64_t dl = desc_sw128(smem_u32(Dlo) + s * 2048, L::kTile64, 1024);
                mma_bf16(tmem + kColPD, ph, dh, id_p, s > 0);
                mma_bf16(tmem + kColPD, ph, dl, id_p, 1);
                mma_bf16(tmem + kColPD, pl, dh, id_p, 1);
            }
            mma_commit(bar_mma);
        }
        __syncwarp();
        wait_mma();
        __syncthreads();
        if (*abort_flag) { aborted = true; break; }
        // the K/Q stage of this chunk is free: prefetch chunk ci + kStages
        if (use_tma && ci + kStages < nchunks) {
            if (threadIdx.x == 0) issue_tma(ci + kStages);
            tma_issued = ci + kStages + 1;
        }

        // ---- state update and output ----
        {
            float row[64];
            const float gC = gam[63];
            // M = 128 accumulator: lane = state row
            ld_row64(tmem, warp, kColS, row);
#pragma unroll
            for (int c = 0; c < kVs; ++c) S[c] = fmaf(gC, S[c], row[c]);
            store_split_row(Shi, Slo, threadIdx.x, S);
            if (want_out) {
                const bool mine = mrow >= 0 && mrow < nv;
                const float gi = mine ? gam[mrow] : 0.f;
                uint4* dst = reinterpret_cast<uint4*>(
                    p.out + ((row_base + c0 + (mine ? mrow : 0)) * H + h) * static_cast<long long>(V) + vs * kVs);
                const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
                for (int q16 = 0; q16 < 4; ++q16) {
                    float qs[16], pd[16];
                    tmem_ld16(tmem + lane_base + kColQS + q16 * 16, qs);
                    tmem_ld16(tmem + lane_base + kColPD + q16 * 16, pd);
                    tmem_ld_wait();
                    if (mine) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = half * 8 + 2 * e;
                                w4[e] = pack_bf16x2(scale * fmaf(gi, qs[c], pd[c]),
                                                    scale * fmaf(gi, qs[c + 1], pd[c + 1]));
                            }
                            dst[q16 * 2 + half] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    if (aborted) {
        if (threadIdx.x == 0) {
            record_error(p.err, kErrTimeout);
            // drain: the MMAs and K/Q loads still in flight must land before
            // the TMEM is released and the CTA's shared memory goes away
            mbar_wait(bar_mma, mma_phase, prm.wait_limit);
            for (int ci = tma_done; ci < tma_issued; ++ci)
                mbar_wait(bar_tma0 + 8 * (ci % kStages), (ci / kStages) & 1, prm.wait_limit);
        }
    } else if (p.final_state && srow >= 0) {
        float* dst = p.final_state + state_off + static_cast<long long>(srow) * V;
#pragma unroll
        for (int j = 0; j < kVs; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D view {d (inner), head, token row} of a (rows, H, d) bf16 tensor; box
// {64, 1, 64} lands as 64 token rows x 128 bytes, 128-byte swizzled.
bool make_qk_map(CUtensorMap* m, const uint16_t* base, long long rows, int H, int D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_tc(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    constexpr int K = 128;
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    if (rows == 0) return launch_fwd_simt(a, stream);  // nothing to load: state pass-through only
    CUtensorMap mk, mq;  // used only for d_k = 128 (d_k = 64 tiles use plain loads)
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    if (a.d_k == 128 && (!make_qk_map(&mk, a.k, rows, a.H, a.d_k) || !make_qk_map(&mq, a.q, rows, a.H, a.d_k)))
        return cudaErrorInvalidValue;
    const int smem = TcSmem<K>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(gdn_fwd_tc_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    TcParams prm{a, wait_limit};
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_fwd_tc_kernel<K><<<grid, kThreads, smem, stream>>>(mk, mq, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    return launch_tc(a, wait_limit, stream);
}

}  // namespace gdn

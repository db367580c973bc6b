// Chunked gated delta rule forward, d_k = 128, with the T tiles of every
// chunk given (chunk-parallel inverse): the tensor-core chunk chain with
// stacked M = 128 products.
//
// Per chunk (C = 64 tokens, S0 the chunk's start state, one 64-column value
// slice of it per CTA) the chain needs
//     R     = beta o (V - gam o (K S0))
//     Delta = T R                          (= u - w S0 of the WY form)
//     S1    = gam_n S0 + K^T (dec o Delta)
//     O     = scale [gam o (Q S0) + P Delta],   P = (Q K^T) o M (causal decay)
// and only the first three are on the serial path.  Two stacked products
// carry the output along with them at no extra tensor-pipe time (an M = 128
// product costs what an M = 64 one does):
//     [K; Q] S0      -> rows 0-63: K S0,   rows 64-127: Q S0
//     [T; P T] R     -> rows 0-63: Delta,  rows 64-127: P T R = P Delta
// P T is formed one chunk ahead by the prep warps (as T^T P^T, so that its
// rows land as the MN-major operand tile the stacked product reads).  Rows
// 0-63 of an M = 128 accumulator sit in TMEM lanes 0-63 and rows 64-127 in
// lanes 64-127, so the warps of subpartitions 0-1 ("K warps") run the chain's
// epilogues while those of subpartitions 2-3 ("Q warps") form the output
// beside them; all eight update the state.
//
// Warps:
//   0-7   chain: K warps 0, 1, 4, 5 (R, then dec o Delta), Q warps 2, 3, 6, 7
//         (output); all: S <- gam_n S + acc.  S (fp32) lives in registers,
//         thread (subpartition sp, half hs, lane l) holding row 32 sp + l,
//         columns 32 hs .. 32 hs + 31 of the slice.  Warp 0 issues the three
//         chain products.
//   8-11  prep, one chunk ahead: gates (g cumsum, gam, dec), Q K^T on the
//         tensor cores, P = (Q K^T) o M as bf16 hi/lo tiles, the chunk's T
//         tiles copied in from the workspace, T^T P^T on the tensor cores into
//         the P T operand tiles.
//
// Precision: computed operands (S, R, dec o Delta, T, P, P T) enter the
// MMAs as bf16 hi + lo pairs (hi*hi + hi*lo + lo*hi, or hi + lo against an
// exact bf16 input), accumulation is fp32 in TMEM, the state is fp32 in
// registers: fla issue #1550 ("Intermediate rounding diagnosis") traces the
// error of bf16 chunk kernels to rounding the inverse, the score and u.
//
// Hand-offs are mbarriers with bounded waits; a wait that runs out sets the
// CTA's abort flag, and every group decides to leave at a barrier that
// reduces the flag over the whole group, so no thread is left waiting at a
// named barrier.  Before the CTA frees its TMEM every issued MMA, TMA load
// and bulk copy is waited for with the default (long) bound.
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

constexpr int kChainThreads = 256;  // warps 0-7
constexpr int kPrepThreads = 128;   // warps 8-11
constexpr int kThreads = kChainThreads + kPrepThreads;
constexpr int kVs = 64;
constexpr int kStages = 3;     // K/Q stages: chunk c + 3 loads while chunk c finishes
constexpr uint32_t kTmemCols = 512;

#ifndef GDN_FWD_NSTACK
#define GDN_FWD_NSTACK 1
#endif
#ifndef GDN_FWD_GATE
#define GDN_FWD_GATE 0
#endif
// The chain's products against a split operand x = hi + lo run as one
// N = 128 product A [x_hi | x_lo] (the two parts side by side, 128 TMEM
// columns) instead of two N = 64 ones: half the MMA instructions, and A is
// read from shared memory once.  The epilogue adds the two halves.
constexpr bool kNStack = GDN_FWD_NSTACK != 0;
// The prep issues its products in the chain's epilogue windows: Q K^T of
// chunk c once [K; Q] S0 of chunk c - 1 has completed, T^T P^T of chunk c
// once [T; P T] R of chunk c - 1 has.
constexpr bool kGate = GDN_FWD_GATE != 0;
constexpr uint32_t kAccCols = kNStack ? 128 : 64;
constexpr uint32_t kColKQ = 0;                   // [K; Q] S0            (M = 128)
constexpr uint32_t kColD = kAccCols;             // [T; P T] R           (M = 128)
constexpr uint32_t kColS = 2 * kAccCols;         // K^T (dec o Delta)    (M = 128, rows = key index)
constexpr uint32_t kColQK = 3 * kAccCols;        // prep: Q K^T          (M = 64)
constexpr uint32_t kColPT = 3 * kAccCols + 64;   // prep: T^T P^T        (M = 64)
static_assert(kColPT + 64 <= kTmemCols, "tensor memory");

constexpr int kStageBytes = 2 * kRegionBytes;  // two 64-column key regions of [K rows; Q rows]
constexpr int kTileS = kDk * 128;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int oStage = 0;
constexpr int oShi = oStage + kStages * kStageBytes;
constexpr int oSlo = oShi + kTileS;
constexpr int oRhi = oSlo + kTileS;       // R, then dec o Delta (hi)
constexpr int oRlo = oRhi + kTile64;
constexpr int oT = oRlo + kTile64;        // T^T [slot][hi, lo]
constexpr int oPT = oT + 4 * kTile64;     // (P T)^T [slot][hi, lo]; P itself before T^T P^T has read it
constexpr int kVecSlots = 3;
constexpr int oVec = oPT + 4 * kTile64;   // [chunk % 3][g, beta, G, gam, dec] x 64 fp32
constexpr int kVecFloats = 5 * 64;
constexpr int oBar = oVec + kVecSlots * kVecFloats * 4;
constexpr int kBars = 16;
constexpr int oMisc = oBar + kBars * 8;   // TMEM slot, abort flag, chain progress
constexpr int kBytes = oMisc + 16;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 232448, "shared memory");
// the stacked [T; P T] operand: the P T tile of a slot and part sits this far
// after the T tile of the same slot and part (the descriptor's MN-block stride)
constexpr uint32_t kLboTPT = oPT - oT;

enum {
    B_FULL0 = 0, B_FULL1 = 1, B_FULL2 = 2, B_KQ = 3, B_D = 4, B_S = 5, B_GRAM = 6, B_PT = 7,
    B_READY0 = 8, B_READY1 = 9, B_TFREE0 = 10, B_TFREE1 = 11, B_TCOPY = 12,
    B_DRAIN0 = 13, B_DRAIN1 = 14
};
static_assert(B_DRAIN1 < kBars, "barriers");

// bar.sync with an OR-reduction of `pred` over the `count` participating
// threads: every participant gets the same answer
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// 32 consecutive TMEM columns of this thread's lane (row), no wait
__device__ __forceinline__ void ld32_nowait(uint32_t taddr, float* v) {
    tmem_ld16(taddr, v);
    tmem_ld16(taddr + 16, v + 16);
}

struct ChainFwdParams {
    FwdArgs a;
    uint32_t wait_limit;
};

// Bound of the waits that drain in-flight copies and MMAs before the CTA
// leaves; independent of the hand-off bound so that a short hand-off bound
// never lets a copy outlive the CTA.
constexpr uint32_t kDrainLimit = 4000000u;

__global__ void __launch_bounds__(kThreads, 1)
    gdn_fwd_chain_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                         const ChainFwdParams prm) {
    const FwdArgs& p = prm.a;
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oMisc + 4);
    // chain progress for the prep's product scheduling: 2 ci + 1 once [K; Q]
    // S0 of chunk ci has completed, 2 ci + 2 once [T; P T] R has
    volatile int* progress = reinterpret_cast<volatile int*>(sm + oMisc + 8);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const long long row_base = static_cast<long long>(b) * p.T;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    const bool want_out = p.out != nullptr;
    const uint32_t wl = prm.wait_limit;
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        *abort_flag = 0;
        *progress = 0;
        if (nchunks > 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    auto issue_tma = [&](int ci) {
        const int st = ci % kStages;
        uint8_t* base = sm + oStage + st * kStageBytes;
        const int z = static_cast<int>(row_base + t0 + ci * kChunk);
        mbar_arrive_expect_tx(bar(B_FULL0 + st), kStageBytes);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tma_load_3d(smem_u32(base + r * kRegionBytes), &tmap_k, r * 64, h, z, bar(B_FULL0 + st));
            tma_load_3d(smem_u32(base + r * kRegionBytes + 64 * 128), &tmap_q, r * 64, h, z, bar(B_FULL0 + st));
        }
    };

    if (warp < 8) {
        // ============================ chain warps ============================
        const int t = tid;
        const int sp = warp & 3, hs = warp >> 2;
        const bool kw = sp < 2;                 // K warp (rows 0-63 of the stacked products)
        const int srow = 32 * sp + lane;        // state row (key index)
        const int i = 32 * (sp & 1) + lane;     // token row of the chunk (K and Q warps alike)
        const uint32_t lb = static_cast<uint32_t>(sp * 32) << 16;
        const uint32_t cq = 32 * hs;            // first column of this thread's half
        // this thread's 32 values of an M = 128 accumulator at column block col
        // (with the N-stacked split, the hi and lo products' halves added)
        auto ld_acc = [&](uint32_t col, float* x) {
            ld32_nowait(tmem + lb + col + cq, x);
            if (kNStack) {
                float y[32];
                ld32_nowait(tmem + lb + col + 64 + cq, y);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] += y[c];
            } else {
                tmem_ld_wait();
            }
        };
        const long long KV = static_cast<long long>(kDk) * V;
        const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kVs;
        const float scale = p.scale;
        uint8_t* Shi = sm + oShi;
        uint8_t* Slo = sm + oSlo;
        uint8_t* Rhi = sm + oRhi;
        uint8_t* Rlo = sm + oRlo;
        int tma_issued = 0, tma_done = 0;  // thread 0's count of stage loads issued / consumed
        if (t == 0) {
            for (int c = 0; c < kStages && c < nchunks; ++c) issue_tma(c);
            tma_issued = min(kStages, nchunks);
        }

        float S[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = 0.f;
        if (p.initial_state) {
            const float* src = p.initial_state + state_off + static_cast<long long>(srow) * V + cq;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(src + j);
                S[j] = t4.x; S[j + 1] = t4.y; S[j + 2] = t4.z; S[j + 3] = t4.w;
            }
        }
        store_split_half(Shi, Slo, srow, hs, S);
        fence_proxy_async_smem();
        named_bar(1, kChainThreads);

        auto store_state_tiles = [&](int ci) {
            const long long nsl = V / kVs;
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.chunk_states) +
                           (((slot0 + ci) * H + h) * nsl + vs) * (2LL * kDk * 128);
            bulk_s2g(dst, smem_u32(Shi), kDk * 128);
            bulk_s2g(dst + kDk * 128, smem_u32(Slo), kDk * 128);
            bulk_commit();
        };
        // K warps: this row's 32 values of the slice, packed bf16, one chunk ahead
        uint4 vraw[4];
        auto load_v = [&](int cj) {
#pragma unroll
            for (int e = 0; e < 4; ++e) vraw[e] = make_uint4(0, 0, 0, 0);
            if (!kw || cj >= nchunks) return;
            const int cc0 = t0 + cj * kChunk;
            if (i < min(kChunk, t1 - cc0)) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.v + ((row_base + cc0 + i) * H + h) * static_cast<long long>(V) + vs * kVs + cq);
#pragma unroll
                for (int e = 0; e < 4; ++e) vraw[e] = src[e];
            }
        };
        // warp 0: [K; Q] S0 of chunk cj once its stage is full
        auto issue_kq = [&](int cj) -> bool {
            const bool full =
                __all_sync(0xffffffffu, mbar_wait(bar(B_FULL0 + cj % kStages), (cj / kStages) & 1, wl));
            if (full) {
                if (elect_one()) {
                    tc_fence_after();
                    const uint32_t stage_c = smem_u32(sm + oStage + (cj % kStages) * kStageBytes);
                    constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 128, kAccCols);
#pragma unroll
                    for (int s = 0; s < kDk / 16; ++s) {
                        const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                        const uint64_t a = desc_sw128(stage_c + koff, 0, 1024);
                        // N = 128: [S_hi | S_lo], the lo tile kTileS after the hi tile
                        mma_bf16(tmem + kColKQ, a, desc_sw128(smem_u32(Shi) + s * 2048, kTileS, 1024), id, s > 0);
                        if (!kNStack)
                            mma_bf16(tmem + kColKQ, a, desc_sw128(smem_u32(Slo) + s * 2048, kTileS, 1024), id, 1);
                    }
                    mma_commit(bar(B_KQ));
                }
                __syncwarp();
            }
            return full;
        };

        load_v(0);
        bool aborted = false;
        if (nchunks > 0) {
            bool ok = true;
            if (warp == 0) {
                ok = issue_kq(0);
                if (ok) tma_done = 1;
            }
            if (!ok && lane == 0) *abort_flag = 1;
            if (p.chunk_states && t == 0) store_state_tiles(0);
        }
        for (int ci = 0; ci < nchunks; ++ci) {
            const int c0 = t0 + ci * kChunk;
            const int nv = min(kChunk, t1 - c0);
            const int slot = ci & 1, st = ci % kStages;
            const uint32_t ph = ci & 1, ph2 = (ci >> 1) & 1;
            const uint32_t stage_a = smem_u32(sm + oStage + st * kStageBytes);
            const float* vec = reinterpret_cast<const float*>(sm + oVec) + (ci % kVecSlots) * kVecFloats;
            const float* bv = vec + 64;
            const float* gam = vec + 192;
            const float* dec = vec + 256;

            // gates, T and P T of this chunk (prep), [K; Q] S0 (issued at the end of the previous chunk)
            __syncwarp();
            bool ok = mbar_wait(bar(B_READY0 + slot), ph2, wl);
            ok = mbar_wait(bar(B_KQ), ph, wl) && ok;
            tc_fence_after();
            if (bar_or(1, kChainThreads, !ok || *abort_flag)) { aborted = true; break; }
            if (t == 0) *progress = 2 * ci + 1;
            const float gC = gam[63];
            float qs[32];
            if (kw) {
                // ---- C2: R = beta o (V - gam o (K S0)) -> R tiles ----
                float x[32];
                ld_acc(kColKQ, x);
                const float bj = bv[i], gj = gam[i];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t w4[4] = {vraw[e].x, vraw[e].y, vraw[e].z, vraw[e].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int c = e * 8 + 2 * m;
                        x[c] = bj * (__uint_as_float(w4[m] << 16) - gj * x[c]);
                        x[c + 1] = bj * (__uint_as_float(w4[m] & 0xffff0000u) - gj * x[c + 1]);
                    }
                }
                store_split_half(Rhi, Rlo, i, hs, x);
                load_v(ci + 1);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(3, 128);
                // ---- C3: [T; P T] R (warp 0) ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc(kFmtBf16, 1, 1, 128, 64);
                        constexpr uint32_t idw = idesc(kFmtBf16, 1, 1, 128, kAccCols);
                        const uint32_t thi = smem_u32(sm + oT + (slot * 2 + 0) * kTile64);
                        const uint32_t tlo = smem_u32(sm + oT + (slot * 2 + 1) * kTile64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ah = desc_sw128(thi + s * 2048, kLboTPT, 1024);
                            const uint64_t al = desc_sw128(tlo + s * 2048, kLboTPT, 1024);
                            // N = 128: [R_hi | R_lo], the lo tile kTile64 after the hi tile
                            const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                            const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColD, ah, rh, idw, s > 0);
                            if (!kNStack) mma_bf16(tmem + kColD, ah, rl, id, 1);
                            mma_bf16(tmem + kColD, al, rh, id, 1);
                        }
                        mma_commit(bar(B_D));
                    }
                    __syncwarp();
                }
            } else {
                // ---- Q warps: gam o (Q S0) of this row, kept until P Delta arrives ----
                ld_acc(kColKQ, qs);
                const float gi = gam[i];
#pragma unroll
                for (int c = 0; c < 32; ++c) qs[c] *= gi;
            }
            __syncwarp();
            bool bad = !mbar_wait(bar(B_D), ph, wl);
            tc_fence_after();
            // [T; P T] R has read the slot's T and P T tiles (and the prep's
            // T^T P^T long before): the prep may fill the slot for chunk ci + 2
            if (t == 0 && !bad) {
                mbar_arrive(bar(B_TFREE0 + slot));
                *progress = 2 * ci + 2;
            }
            if (kw) {
                // ---- C4: dec o Delta -> R tiles (T R has read them) ----
                float x[32];
                ld_acc(kColD, x);
                const float dj = dec[i];
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] *= dj;
                store_split_half(Rhi, Rlo, i, hs, x);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(3, 128);
                // ---- C5: S update K^T (dec o Delta) (warp 0) ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc(kFmtBf16, 1, 1, kDk, kAccCols);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ak = desc_sw128(stage_a + s * 2048, kRegionBytes, 1024);
                            mma_bf16(tmem + kColS, ak, desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024), id, s > 0);
                            if (!kNStack)
                                mma_bf16(tmem + kColS, ak, desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024), id, 1);
                        }
                        mma_commit(bar(B_S));
                    }
                    __syncwarp();
                }
            } else {
                // ---- output: O = scale [gam o (Q S0) + P Delta] ----
                float pd[32];
                ld_acc(kColD, pd);
                if (want_out && i < nv) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.out + ((row_base + c0 + i) * H + h) * static_cast<long long>(V) + vs * kVs + cq);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t w4[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int c = e * 8 + 2 * m;
                            w4[m] = cvt_bf16x2(scale * (qs[c] + pd[c]), scale * (qs[c + 1] + pd[c + 1]));
                        }
                        dst[e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            __syncwarp();
            // ---- C6: S <- gam_n S + K^T (dec o Delta) ----
            bad = !mbar_wait(bar(B_S), ph, wl) || bad;
            tc_fence_after();
            {
                float x[32];
                ld_acc(kColS, x);
#pragma unroll
                for (int c = 0; c < 32; ++c) S[c] = fmaf(gC, S[c], x[c]);
            }
            // the stage's readers ([K; Q] S0, the update, the prep's Q K^T) have
            // all completed: it takes chunk ci + 3's tiles
            if (t == 0 && ci + kStages < nchunks) {
                issue_tma(ci + kStages);
                tma_issued = ci + kStages + 1;
            }
            if (p.chunk_states) {
                // the bulk copy of this chunk's start-state tiles has read them
                if (t == 0) bulk_wait_read_all();
                named_bar(1, kChainThreads);
            }
            store_split_half(Shi, Slo, srow, hs, S);
            fence_proxy_async_smem();
            tc_fence_before();
            if (bar_or(1, kChainThreads, bad || *abort_flag)) { aborted = true; break; }
            // ---- next chunk's [K; Q] S0 ----
            if (ci + 1 < nchunks) {
                bool ok2 = true;
                if (warp == 0) {
                    ok2 = issue_kq(ci + 1);
                    if (ok2) tma_done = ci + 2;
                }
                if (!ok2 && lane == 0) *abort_flag = 1;
                if (p.chunk_states && t == 0) store_state_tiles(ci + 1);
            }
        }
        if (p.chunk_states && t == 0) bulk_wait_all();
        if (aborted) {
            // nothing warp 0 issued, no stage load and no bulk copy outlives the CTA
            if (warp == 0) {
                if (elect_one()) mma_commit(bar(B_DRAIN0));
                __syncwarp();
            }
            if (t == 0) {
                record_error(p.err, kErrTimeout);
                mbar_wait(bar(B_DRAIN0), 0, kDrainLimit);
                for (int c = tma_done; c < tma_issued; ++c)
                    mbar_wait(bar(B_FULL0 + c % kStages), (c / kStages) & 1, kDrainLimit);
            }
        } else if (p.final_state) {
            float* dst = p.final_state + state_off + static_cast<long long>(srow) * V + cq;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    } else {
        // ============================ prep warps ============================
        const int q = tid - kChainThreads;  // 0..127
        const int sub = warp - 8;           // TMEM subpartition
        float g_pre = 0.f, b_pre = 0.f;
        auto load_gates = [&](int it) {
            g_pre = 0.f;
            b_pre = 0.f;
            if (q < 64 && it < nchunks) {
                const int cc0 = t0 + it * kChunk;
                if (q < min(kChunk, t1 - cc0)) {
                    const long long idx = (row_base + cc0 + q) * H + h;
                    g_pre = p.g[idx];
                    b_pre = bf16_to_f32(p.beta[idx]);
                }
            }
        };
        // warp 8: wait (bounded) until the chain's progress reaches `target`
        auto wait_progress = [&](int target) -> bool {
            for (uint32_t n = 0; n < wl; ++n) {
                if (*progress >= target) return true;
                if (*abort_flag) return false;
                __nanosleep(64);
            }
            return false;
        };
        load_gates(0);
        bool tcopy_out = false;  // thread q == 0: a T tile copy is in flight (phase tcopy_it & 1)
        int tcopy_it = 0;
        bool aborted = false;
        for (int it = 0; it < nchunks; ++it) {
            const int slot = it & 1, st = it % kStages;
            const uint32_t ph = it & 1;
            uint8_t* stage = sm + oStage + st * kStageBytes;
            // P goes where the slot's P T tiles go: T^T P^T reads it before
            // its result is written there
            uint8_t* p_hi = sm + oPT + (slot * 2 + 0) * kTile64;
            uint8_t* p_lo = sm + oPT + (slot * 2 + 1) * kTile64;
            float* vec = reinterpret_cast<float*>(sm + oVec) + (it % kVecSlots) * kVecFloats;
            float* gv = vec;
            float* bv = vec + 64;
            float* Gv = vec + 128;
            float* gam = vec + 192;
            float* dec = vec + 256;

            // stage of this chunk loaded; its slot free ([T; P T] R of chunk it - 2 done)
            bool ok = mbar_wait(bar(B_FULL0 + st), (it / kStages) & 1, wl);
            if (it >= 2) ok = mbar_wait(bar(B_TFREE0 + slot), ((it - 2) >> 1) & 1, wl) && ok;
            if (bar_or(2, kPrepThreads, !ok || *abort_flag)) { aborted = true; break; }

            // Q K^T (M = 64) while the gates are formed
            if (warp == 8) {
                const bool go = !kGate || it == 0 || wait_progress(2 * (it - 1) + 1);
                if (!go && lane == 0) *abort_flag = 1;
                if (go && elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc(kFmtBf16, 0, 0, 64, 64);
                    const uint32_t sa = smem_u32(stage);
#pragma unroll
                    for (int s = 0; s < kDk / 16; ++s) {
                        const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                        mma_bf16(tmem + kColQK, desc_sw128(sa + koff + 64 * 128, 0, 1024),
                                 desc_sw128(sa + koff, 0, 1024), id, s > 0);
                    }
                    mma_commit(bar(B_GRAM));
                }
                __syncwarp();
            }
            if (q == 0) {
                // this chunk's T tiles (chunk-parallel inverse) into the slot
                mbar_arrive_expect_tx(bar(B_TCOPY), 2 * kTile64);
                bulk_g2s(smem_u32(sm + oT + (slot * 2) * kTile64),
                         p.chunk_T + ((slot0 + it) * H + h) * (2LL * kTile64), 2 * kTile64, bar(B_TCOPY));
                tcopy_out = true;
                tcopy_it = it;
            }
            if (q < 64) {
                gv[q] = g_pre;
                bv[q] = b_pre;
            }
            load_gates(it + 1);
            named_bar(2, kPrepThreads);
            if (q < 32) {
                const float a = gv[2 * q];
                const float bb = a + gv[2 * q + 1];
                float s = bb;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, s, off);
                    if (q >= off) s += o;
                }
                const float base = s - bb;
                Gv[2 * q] = base + a;
                Gv[2 * q + 1] = s;
                gam[2 * q] = exp_nonpos(base + a);
                gam[2 * q + 1] = exp_nonpos(s);
            }
            named_bar(2, kPrepThreads);
            if (q < 64) dec[q] = exp_nonpos(Gv[63] - Gv[q]);

            __syncwarp();
            bool bad = !mbar_wait(bar(B_GRAM), ph, wl);
            tc_fence_after();
            {
                // P = (Q K^T) o M: thread (warp 8 + sub, lane l) takes row
                // ii = 16 sub + l % 16, columns 32 (l / 16) .. + 31; the decay of
                // each pair is masked to j <= ii before the exponential
                const int ii = 16 * sub + (lane & 15), hf = lane >> 4, j0 = 32 * hf;
                const float Gi = Gv[ii];
                float x[32];
                ld_half32_nowait(tmem, sub, kColQK, x);
                float mdec[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) mdec[k] = (j0 + k <= ii) ? exp_nonpos(Gi - Gv[j0 + k]) : 0.f;
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] *= mdec[k];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) store_split_chunk(p_hi, p_lo, ii, 4 * hf + c4, x + 8 * c4);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (q == 0) {
                if (mbar_wait(bar(B_TCOPY), it & 1, wl)) tcopy_out = false;
                else bad = true;
            }
            if (bar_or(2, kPrepThreads, bad || *abort_flag)) { aborted = true; break; }

            // (P T)^T = T^T P^T (M = 64): A = T^T tile (K-major), B = P tile (K-major)
            if (warp == 8) {
                const bool go = !kGate || it == 0 || wait_progress(2 * (it - 1) + 2);
                if (!go && lane == 0) *abort_flag = 1;
                if (go && elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc(kFmtBf16, 0, 0, 64, 64);
                    const uint32_t thi = smem_u32(sm + oT + (slot * 2 + 0) * kTile64);
                    const uint32_t tlo = smem_u32(sm + oT + (slot * 2 + 1) * kTile64);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t ah = desc_sw128(thi + s * 32, 0, 1024);
                        const uint64_t al = desc_sw128(tlo + s * 32, 0, 1024);
                        const uint64_t bh = desc_sw128(smem_u32(p_hi) + s * 32, 0, 1024);
                        const uint64_t bl = desc_sw128(smem_u32(p_lo) + s * 32, 0, 1024);
                        mma_bf16(tmem + kColPT, ah, bh, id, s > 0);
                        mma_bf16(tmem + kColPT, ah, bl, id, 1);
                        mma_bf16(tmem + kColPT, al, bh, id, 1);
                    }
                    mma_commit(bar(B_PT));
                }
                __syncwarp();
            }
            __syncwarp();
            bad = !mbar_wait(bar(B_PT), ph, wl);
            tc_fence_after();
            {
                // row m of (P T)^T (= column m of P T) -> row m of the slot's P T
                // tiles (T^T P^T has completed: P is dead)
                const int m = 16 * sub + (lane & 15), hf = lane >> 4;
                float x[32];
                ld_half32(tmem, sub, kColPT, x);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) store_split_chunk(p_hi, p_lo, m, 4 * hf + c4, x + 8 * c4);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (bar_or(2, kPrepThreads, bad || *abort_flag)) { aborted = true; break; }
            if (q == 0) mbar_arrive(bar(B_READY0 + slot));
        }
        if (q == 0 && tcopy_out) mbar_wait(bar(B_TCOPY), tcopy_it & 1, kDrainLimit);  // no copy outlives the CTA
        if (aborted) {
            *abort_flag = 1;
            if (warp == 8) {
                if (elect_one()) mma_commit(bar(B_DRAIN1));
                __syncwarp();
            }
            if (q == 0) {
                record_error(p.err, kErrTimeout);
                mbar_wait(bar(B_DRAIN1), 0, kDrainLimit);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_fwd_chain(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    if (a.d_k != kDk || a.chunk_T == nullptr || a.d_v % kVs != 0) return cudaErrorInvalidValue;
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    CUtensorMap mk, mq;
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    if (rows <= 0 || !make_qk_map(&mk, a.k, rows, a.H) || !make_qk_map(&mq, a.q, rows, a.H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_fwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    ChainFwdParams prm{a, wait_limit};
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_fwd_chain_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, mq, prm);
    return cudaGetLastError();
}

}  // namespace gdn

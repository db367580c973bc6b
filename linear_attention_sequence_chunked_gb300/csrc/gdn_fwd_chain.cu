// Chunked gated delta rule forward, d_k = 128, with the T tiles of every
// chunk given (chunk-parallel inverse): the tensor-core chunk chain.
//
// Per chunk (C = 64 tokens, S0 the chunk's start state) the chain needs
//     R     = beta o (V - gam o (K S0))
//     Delta = T R                          (= u - w S0 of the WY form)
//     S1    = gam_n S0 + K^T (dec o Delta)
//     O     = scale [gam o (Q S0) + P Delta],   P = (Q K^T) o M (causal decay)
// and only the first three are on the serial path.  Two stacked products
// carry the output along at no extra tensor-pipe time (an M = 128 product
// costs what an M = 64 one does):
//     [K; Q] S0      -> rows 0-63: K S0,   rows 64-127: Q S0
//     [T; P T] R     -> rows 0-63: Delta,  rows 64-127: P T R = P Delta
// P T is formed one chunk ahead by the prep warps (as T^T P^T, so that its
// rows land as the MN-major operand tile the stacked product reads).  Rows
// 0-63 of an M = 128 accumulator sit in TMEM lanes 0-63 and rows 64-127 in
// lanes 64-127, so the warps of subpartitions 0-1 ("K warps") run the chain's
// epilogues while those of subpartitions 2-3 ("Q warps") form the output
// beside them; all eight update the state.
//
// The value columns of the state evolve independently ("Research Sprint
// Day 1", the GDN update: column j of S only ever meets v_j), so each CTA's
// 64-column slice runs as two independent sub-chains of 32 columns, A and B,
// half a chunk apart.  Every product of one sub-chain is issued while the
// other sub-chain's warps run an epilogue, so the tensor pipe's latency is
// hidden behind CUDA-core work instead of stalling the chain.  Per chunk c the
// epilogue warps run, in order,
//     (a) R of A            (b) S update of B (chunk c - 1)
//     (c) dec o Delta of A, output of A
//     (d) R of B            (e) S update of A
//     (f) dec o Delta of B, output of B
// and a dedicated issuer warp issues each phase's product as soon as that
// phase's operand tiles are stored.  Split operands x = hi + lo sit side by
// side in one 64-column tile ([x_hi | x_lo], 32 columns each), so one N = 64
// product A [x_hi | x_lo] gives both halves and the epilogue adds them.
//
// Warps:
//   0-7   epilogues.  K warps 0, 1, 4, 5; Q warps 2, 3, 6, 7.  Thread
//         (subpartition sp, half hs, lane l) takes token row 32 (sp & 1) + l of
//         the chunk, state row 32 sp + l, and columns 16 hs .. 16 hs + 15 of
//         each sub-chain.  The fp32 state lives in their registers.
//   8-11  prep, one chunk ahead: gates (g cumsum, gam, dec), Q K^T, P as bf16
//         hi/lo tiles, the chunk's T tiles copied in, T^T P^T into the P T
//         operand tiles.
//   12    issues the chain's products and the K/Q tile loads.
//
// Precision: computed operands (S, R, dec o Delta, T, P, P T) enter the MMAs
// as bf16 hi + lo pairs, accumulation is fp32 in TMEM, the state is fp32 in
// registers (fla issue #1550, "Intermediate rounding diagnosis", traces the
// error of bf16 chunk kernels to rounding the inverse, the score and u).
//
// Hand-offs are mbarriers with bounded waits and named barriers between the
// epilogue warps and the issuer.  A wait that runs out marks the CTA bad; the
// decision to leave is taken at the two per-chunk barriers every epilogue
// thread and the issuer pass (an OR-reduction over all of them), so no
// thread is left waiting at a named barrier.  Before the CTA frees its TMEM,
// every issued MMA, TMA load and bulk copy is waited for with the default
// (long) bound.
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
constexpr int kIssuerWarp = 12;
constexpr int kThreads = kChainThreads + kPrepThreads + 32;
constexpr int kVs = 64;
constexpr int kStages = 3;          // K/Q stages: chunk c + 3 loads while chunk c finishes
constexpr uint32_t kTmemCols = 512;

// TMEM column blocks (M = 128 unless noted; X = sub-chain A or B)
constexpr uint32_t kColKQ = 0;      // [K; Q] [S_hi | S_lo] of X at 64 X
constexpr uint32_t kColD = 128;     // [T; P T] [R_hi | R_lo] of X at 128 + 64 X
constexpr uint32_t kColS = 256;     // K^T [dX_hi | dX_lo] of X at 256 + 64 X
constexpr uint32_t kColQK = 384;    // prep: Q K^T (M = 64)
constexpr uint32_t kColPT = 448;    // prep: T^T P^T (M = 64)

constexpr int kStageBytes = 2 * kRegionBytes;  // two 64-column key regions of [K rows; Q rows]
constexpr int kTileSX = kDk * 128;             // a sub-chain's state tile: 128 key rows x [hi 32 | lo 32]

// shared-memory map (bytes from a 1024-aligned base)
constexpr int oStage = 0;
constexpr int oS = oStage + kStages * kStageBytes;  // state tiles of A, B
constexpr int oR = oS + 2 * kTileSX;                // R, then dec o Delta, of A, B: 64 token rows x [hi | lo]
constexpr int oT = oR + 2 * kTile64;                // T^T [slot][hi, lo]
constexpr int oPT = oT + 4 * kTile64;               // (P T)^T [slot][hi, lo]; P itself before T^T P^T has read it
constexpr int oO = oPT + 4 * kTile64;               // output staging: 64 token rows x 64 columns bf16
constexpr int kVecSlots = 3;
constexpr int oVec = oO + kTile64;                  // [chunk % 3][g, beta, G, gam, dec] x 64 fp32
constexpr int kVecFloats = 5 * 64;
constexpr int oBar = oVec + kVecSlots * kVecFloats * 4;
constexpr int kBars = 20;
constexpr int oMisc = oBar + kBars * 8;             // TMEM slot
constexpr int kBytes = oMisc + 16;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 232448, "shared memory");
// the stacked [T; P T] operand: the P T tile of a slot and part sits this far
// after the T tile of the same slot and part (the descriptor's MN-block stride)
constexpr uint32_t kLboTPT = oPT - oT;

enum {
    B_FULL0 = 0, B_KQ0 = 3, B_D0 = 5, B_S0 = 7,   // FULL: 3 stages; KQ, D, S: one per sub-chain
    B_GRAM = 9, B_PT = 10, B_READY0 = 11, B_TFREE0 = 13, B_TCOPY = 15,
    B_DRAIN0 = 16, B_DRAIN1 = 17, B_STALL = 18     // B_STALL: never signalled (failure-detection test)
};
static_assert(B_DRAIN1 < kBars, "barriers");

// named barriers
constexpr int NB_CHAIN = 1;                         // epilogue warps (256)
constexpr int NB_PREP = 2;                          // prep warps (128)
constexpr int NB_C2 = 3;                            // + X: R of X stored (K warps + issuer, 160)
constexpr int NB_C4 = 5;                            // + X: dec o Delta of X stored (K warps + issuer, 160)
constexpr int NB_C6 = 7;                            // + X: state tile of X stored (epilogue warps + issuer, 288)
constexpr int NB_OUT = 9;                           // Q warps (128)
constexpr int kKIss = 128 + 32;
constexpr int kAllIss = kChainThreads + 32;

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

// 8 values as bf16 hi and lo parts (x = hi + lo to ~16 bits)
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float a = x[2 * e], b = x[2 * e + 1];
        h[e] = cvt_bf16x2(a, b);
        l[e] = cvt_bf16x2(a - __uint_as_float(h[e] << 16), b - __uint_as_float(h[e] & 0xffff0000u));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
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
                         const __grid_constant__ CUtensorMap tmap_o, const ChainFwdParams prm) {
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp < 8) {
        // ============================ epilogue warps ============================
        const int t = tid;
        const int sp = warp & 3, hs = warp >> 2;
        const bool kw = sp < 2;                 // K warp (rows 0-63 of the stacked products)
        const int srow = 32 * sp + lane;        // state row (key index)
        const int i = 32 * (sp & 1) + lane;     // token row of the chunk
        const uint32_t lb = static_cast<uint32_t>(sp * 32) << 16;
        const int c0 = 16 * hs;                 // this thread's first column within a sub-chain
        const long long KV = static_cast<long long>(kDk) * V;
        const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kVs;
        const float scale = p.scale;
        const long long nsl = V / kVs;

        // this thread's 16 values of sub-chain X's accumulator at `col` (the
        // hi and lo products' halves added)
        auto ld_acc = [&](uint32_t col, float* x) {
            float y[16];
            tmem_ld16(tmem + lb + col + c0, x);
            tmem_ld16(tmem + lb + col + 32 + c0, y);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) x[c] += y[c];
        };
        // 16 values into row `row` of a [hi 32 | lo 32] sub-chain tile
        auto store_sub = [&](uint8_t* tile, int row, const float* x) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                uint4 hi, lo;
                split8(x + 8 * e, hi, lo);
                *reinterpret_cast<uint4*>(tile + sw128_offset(row, (2 * hs + e) * 16)) = hi;
                *reinterpret_cast<uint4*>(tile + sw128_offset(row, (4 + 2 * hs + e) * 16)) = lo;
            }
        };
        // the training route keeps every chunk's start state as bf16 hi/lo
        // operand tiles in the layout the backward reads: [slot][head][value
        // slice][hi, lo] of 128 key rows x 128 bytes (64 columns, 128-byte
        // swizzle); this thread writes its 16 columns of sub-chain X
        auto save_state = [&](int cj, int X, const float* x) {
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.chunk_states) +
                           (((slot0 + cj) * H + h) * nsl + vs) * (2LL * kDk * 128);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                uint4 hi, lo;
                split8(x + 8 * e, hi, lo);
                const uint32_t off = sw128_offset(srow, (4 * X + 2 * hs + e) * 16);
                *reinterpret_cast<uint4*>(dst + off) = hi;
                *reinterpret_cast<uint4*>(dst + kDk * 128 + off) = lo;
            }
        };

        // the state: sub-chain A's 16 columns, then B's
        float S[2][16];
#pragma unroll
        for (int X = 0; X < 2; ++X) {
#pragma unroll
            for (int j = 0; j < 16; ++j) S[X][j] = 0.f;
            if (p.initial_state) {
                const float* src = p.initial_state + state_off + static_cast<long long>(srow) * V + 32 * X + c0;
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(src + j);
                    S[X][j] = t4.x; S[X][j + 1] = t4.y; S[X][j + 2] = t4.z; S[X][j + 3] = t4.w;
                }
            }
            store_sub(sm + oS + X * kTileSX, srow, S[X]);
            if (p.chunk_states && nchunks > 0) save_state(0, X, S[X]);
        }
        fence_proxy_async_smem();
        // the issuer takes the initial state tiles from here
        bool aborted = bar_or(NB_C6, kAllIss, false);

        // K warps: the row's 16 values of each sub-chain, packed bf16, one chunk ahead
        uint4 vraw[2][2];
        auto load_v = [&](int cj) {
#pragma unroll
            for (int X = 0; X < 2; ++X) vraw[X][0] = vraw[X][1] = make_uint4(0, 0, 0, 0);
            if (!kw || cj >= nchunks) return;
            const int cc0 = t0 + cj * kChunk;
            if (i < min(kChunk, t1 - cc0)) {
                const uint16_t* row = p.v + ((row_base + cc0 + i) * H + h) * static_cast<long long>(V) + vs * kVs;
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    const uint4* src = reinterpret_cast<const uint4*>(row + 32 * X + c0);
                    vraw[X][0] = src[0];
                    vraw[X][1] = src[1];
                }
            }
        };
        load_v(0);

        float qs[16];
        // (a), (d): R of sub-chain X (K warps) / gam o (Q S0) of X (Q warps)
        auto phase_r = [&](int X, const float* bv, const float* gam) {
            if (kw) {
                float x[16];
                ld_acc(kColKQ + 64 * X, x);
                const float bj = bv[i], gj = gam[i];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t w4[4] = {vraw[X][e].x, vraw[X][e].y, vraw[X][e].z, vraw[X][e].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int c = 8 * e + 2 * m;
                        x[c] = bj * (__uint_as_float(w4[m] << 16) - gj * x[c]);
                        x[c + 1] = bj * (__uint_as_float(w4[m] & 0xffff0000u) - gj * x[c + 1]);
                    }
                }
                store_sub(sm + oR + X * kTile64, i, x);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_arrive(NB_C2 + X, kKIss);
            } else {
                ld_acc(kColKQ + 64 * X, qs);
                const float gi = gam[i];
#pragma unroll
                for (int c = 0; c < 16; ++c) qs[c] *= gi;
            }
        };
        // (c), (f): dec o Delta of X (K warps) / output of X (Q warps)
        auto phase_d = [&](int X, const float* dec, int c0tok, int nv) {
            if (kw) {
                float x[16];
                ld_acc(kColD + 64 * X, x);
                const float dj = dec[i];
#pragma unroll
                for (int c = 0; c < 16; ++c) x[c] *= dj;
                store_sub(sm + oR + X * kTile64, i, x);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_arrive(NB_C4 + X, kKIss);
            } else {
                float pd[16];
                ld_acc(kColD + 64 * X, pd);
                if (want_out) {
                    uint32_t w[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m)
                        w[m] = cvt_bf16x2(scale * (qs[2 * m] + pd[2 * m]), scale * (qs[2 * m + 1] + pd[2 * m + 1]));
                    if (nv == kChunk) {
                        // full chunk: into the staging tile, stored by TMA after B
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            *reinterpret_cast<uint4*>(sm + oO + sw128_offset(i, (4 * X + 2 * hs + e) * 16)) =
                                make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    } else if (i < nv) {
                        // ragged chunk: the rows past its end belong to the next sequence
                        uint4* dst = reinterpret_cast<uint4*>(
                            p.out + ((row_base + c0tok + i) * H + h) * static_cast<long long>(V) + vs * kVs + 32 * X + c0);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
        };
        // (b), (e): S <- gam_n S + K^T (dec o Delta) for sub-chain X, chunk cj
        auto phase_s = [&](int X, int cj, float gC, bool bad) -> bool {
            bad = !mbar_wait(bar(B_S0 + X), cj & 1, wl) || bad;
            tc_fence_after();
            float x[16];
            ld_acc(kColS + 64 * X, x);
#pragma unroll
            for (int c = 0; c < 16; ++c) S[X][c] = fmaf(gC, S[X][c], x[c]);
            store_sub(sm + oS + X * kTileSX, srow, S[X]);
            if (p.chunk_states && cj + 1 < nchunks) save_state(cj + 1, X, S[X]);
            fence_proxy_async_smem();
            tc_fence_before();
            return bar_or(NB_C6 + X, kAllIss, bad || *abort_flag);
        };

        for (int ci = 0; ci < nchunks && !aborted; ++ci) {
            const int c0tok = t0 + ci * kChunk;
            const int nv = min(kChunk, t1 - c0tok);
            const int slot = ci & 1;
            const uint32_t ph = ci & 1;
            const float* vec = reinterpret_cast<const float*>(sm + oVec) + (ci % kVecSlots) * kVecFloats;
            const float* bv = vec + 64;
            const float* gam = vec + 192;
            const float* dec = vec + 256;

            // (a) R of A: gates and P T of this chunk from the prep, [K; Q] S0 of A
            bool bad = !mbar_wait(bar(B_READY0 + slot), (ci >> 1) & 1, wl);
            bad = !mbar_wait(bar(B_KQ0 + 0), ph, wl) || bad;
            tc_fence_after();
            phase_r(0, bv, gam);
            // (b) S update of B for the previous chunk
            if (ci > 0) {
                const float* pvec = reinterpret_cast<const float*>(sm + oVec) + ((ci - 1) % kVecSlots) * kVecFloats;
                if (phase_s(1, ci - 1, pvec[192 + 63], bad)) { aborted = true; break; }
                bad = false;
            }
            // (c) dec o Delta of A, output of A
            if (!kw && want_out && nv == kChunk) {
                // the staging tile's previous TMA store has read it
                if (t == 64) bulk_wait_read_all();
                named_bar(NB_OUT, 128);
            }
            bad = !mbar_wait(bar(B_D0 + 0), ph, wl) || bad;
            tc_fence_after();
            phase_d(0, dec, c0tok, nv);
            // (d) R of B
            bad = !mbar_wait(bar(B_KQ0 + 1), ph, wl) || bad;
            tc_fence_after();
            phase_r(1, bv, gam);
            load_v(ci + 1);
            // (e) S update of A
            if (phase_s(0, ci, gam[63], bad)) { aborted = true; break; }
            // (f) dec o Delta of B, output of B
            bad = !mbar_wait(bar(B_D0 + 1), ph, wl);
            tc_fence_after();
            // both [T; P T] R of this chunk have read the slot's T and P T tiles
            // (and the prep's T^T P^T long before): the prep may refill it
            if (t == 0 && !bad) mbar_arrive(bar(B_TFREE0 + slot));
            phase_d(1, dec, c0tok, nv);
            if (!kw && want_out && nv == kChunk) {
                fence_proxy_async_smem();
                named_bar(NB_OUT, 128);
                if (t == 64) {
                    tma_store_3d(&tmap_o, vs * kVs, h, static_cast<int>(row_base + c0tok), smem_u32(sm + oO));
                    bulk_commit();
                }
            }
            if (bad) *abort_flag = 1;
        }
        if (!aborted && nchunks > 0) {
            // S update of B for the last chunk
            const float* pvec =
                reinterpret_cast<const float*>(sm + oVec) + ((nchunks - 1) % kVecSlots) * kVecFloats;
            aborted = phase_s(1, nchunks - 1, pvec[192 + 63], false);
        }
        if (t == 64) bulk_wait_all();  // the output tile stores
        if (aborted) {
            if (t == 0) record_error(p.err, kErrTimeout);
        } else if (p.final_state) {
#pragma unroll
            for (int X = 0; X < 2; ++X) {
                float* dst = p.final_state + state_off + static_cast<long long>(srow) * V + 32 * X + c0;
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    *reinterpret_cast<float4*>(dst + j) = make_float4(S[X][j], S[X][j + 1], S[X][j + 2], S[X][j + 3]);
            }
        }
    } else if (warp == kIssuerWarp) {
        // ============================ issuer warp ============================
        int tma_issued = 0, tma_done = 0;   // stage loads issued / waited for (chunk counts)
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
        if (lane == 0) {
            if (nchunks > 0) {
                tma_prefetch_desc(&tmap_k);
                tma_prefetch_desc(&tmap_q);
                if (want_out) tma_prefetch_desc(&tmap_o);
            }
            for (int c = 0; c < kStages && c < nchunks; ++c) issue_tma(c);
        }
        tma_issued = min(kStages, nchunks);
        // stage of chunk cj loaded (once per chunk, before its first product)
        auto wait_full = [&](int cj) -> bool {
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_FULL0 + cj % kStages), (cj / kStages) & 1, wl));
            if (ok) tma_done = cj + 1;
            return ok;
        };
        // [K; Q] [S_hi | S_lo] of sub-chain X, chunk cj
        auto issue_kq = [&](int X, int cj) {
            if (elect_one()) {
                tc_fence_after();
                const uint32_t stage_c = smem_u32(sm + oStage + (cj % kStages) * kStageBytes);
                const uint32_t sx = smem_u32(sm + oS + X * kTileSX);
                constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 128, 64);
#pragma unroll
                for (int s = 0; s < kDk / 16; ++s) {
                    const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                    mma_bf16(tmem + kColKQ + 64 * X, desc_sw128(stage_c + koff, 0, 1024),
                             desc_sw128(sx + s * 2048, kTileSX, 1024), id, s > 0);
                }
                mma_commit(bar(B_KQ0 + X));
            }
            __syncwarp();
        };
        // [T; P T] [R_hi | R_lo] of X (both parts of [T; P T])
        auto issue_tr = [&](int X, int cj) {
            if (elect_one()) {
                tc_fence_after();
                const int slot = cj & 1;
                const uint32_t thi = smem_u32(sm + oT + (slot * 2 + 0) * kTile64);
                const uint32_t tlo = smem_u32(sm + oT + (slot * 2 + 1) * kTile64);
                const uint32_t rx = smem_u32(sm + oR + X * kTile64);
                constexpr uint32_t id = idesc(kFmtBf16, 1, 1, 128, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t r = desc_sw128(rx + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColD + 64 * X, desc_sw128(thi + s * 2048, kLboTPT, 1024), r, id, s > 0);
                    mma_bf16(tmem + kColD + 64 * X, desc_sw128(tlo + s * 2048, kLboTPT, 1024), r, id, 1);
                }
                mma_commit(bar(B_D0 + X));
            }
            __syncwarp();
        };
        // K^T [dX_hi | dX_lo] of X (A = K^T read MN-major from the stage)
        auto issue_upd = [&](int X, int cj) {
            if (elect_one()) {
                tc_fence_after();
                const uint32_t stage_c = smem_u32(sm + oStage + (cj % kStages) * kStageBytes);
                const uint32_t rx = smem_u32(sm + oR + X * kTile64);
                constexpr uint32_t id = idesc(kFmtBf16, 1, 1, kDk, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + kColS + 64 * X, desc_sw128(stage_c + s * 2048, kRegionBytes, 1024),
                             desc_sw128(rx + s * 2048, kTile64, 1024), id, s > 0);
                mma_commit(bar(B_S0 + X));
            }
            __syncwarp();
        };

        // failure-detection test: a wait that nothing ends runs out
        bool bad = p.stall && !__all_sync(0xffffffffu, mbar_wait(bar(B_STALL), 0, wl));
        // initial state tiles stored
        bool aborted = bar_or(NB_C6, kAllIss, bad);
        if (!aborted && nchunks > 0) {
            bad = !wait_full(0);
            if (!bad) {
                issue_kq(0, 0);
                issue_kq(1, 0);
            }
        }
        for (int ci = 0; ci < nchunks && !aborted; ++ci) {
            named_bar(NB_C2 + 0, kKIss);             // (a) R of A stored
            issue_tr(0, ci);
            if (ci > 0) {
                if (bar_or(NB_C6 + 1, kAllIss, bad)) { aborted = true; break; }   // (b)
                // every product that reads chunk ci - 1's stage has completed
                if (lane == 0 && ci + 2 < nchunks) issue_tma(ci + 2);
                if (ci + 2 < nchunks) tma_issued = ci + 3;
                issue_kq(1, ci);
            }
            named_bar(NB_C4 + 0, kKIss);             // (c) dec o Delta of A stored
            issue_upd(0, ci);
            named_bar(NB_C2 + 1, kKIss);             // (d) R of B stored
            issue_tr(1, ci);
            if (bar_or(NB_C6 + 0, kAllIss, bad)) { aborted = true; break; }       // (e)
            if (ci + 1 < nchunks) {
                if (wait_full(ci + 1)) issue_kq(0, ci + 1);
                else bad = true;
            }
            named_bar(NB_C4 + 1, kKIss);             // (f) dec o Delta of B stored
            issue_upd(1, ci);
        }
        if (!aborted && nchunks > 0) aborted = bar_or(NB_C6 + 1, kAllIss, bad);   // last (b)
        if (aborted) {
            // nothing this warp issued (products, stage loads) outlives the CTA
            if (elect_one()) mma_commit(bar(B_DRAIN0));
            __syncwarp();
            if (lane == 0) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeout);
                mbar_wait(bar(B_DRAIN0), 0, kDrainLimit);
                for (int c = tma_done; c < tma_issued; ++c)
                    mbar_wait(bar(B_FULL0 + c % kStages), (c / kStages) & 1, kDrainLimit);
            }
            __syncwarp();
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

            // stage of this chunk loaded; its slot free (both [T; P T] R of chunk it - 2 done)
            bool ok = mbar_wait(bar(B_FULL0 + st), (it / kStages) & 1, wl);
            if (it >= 2) ok = mbar_wait(bar(B_TFREE0 + slot), ((it - 2) >> 1) & 1, wl) && ok;
            if (bar_or(2, kPrepThreads, !ok || *abort_flag)) { aborted = true; break; }

            // Q K^T (M = 64) while the gates are formed
            if (warp == 8) {
                if (elect_one()) {
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
                if (elect_one()) {
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
    CUtensorMap mk, mq, mo;
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    memset(&mo, 0, sizeof(mo));
    if (rows <= 0 || !make_qk_map(&mk, a.k, rows, a.H) || !make_qk_map(&mq, a.q, rows, a.H))
        return cudaErrorInvalidValue;
    if (a.out && !make_rows_map(&mo, a.out, rows, a.H, a.d_v)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_fwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    ChainFwdParams prm{a, wait_limit};
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_fwd_chain_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, mq, mo, prm);
    return cudaGetLastError();
}

}  // namespace gdn

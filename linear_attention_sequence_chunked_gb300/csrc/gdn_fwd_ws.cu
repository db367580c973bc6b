// Chunked gated delta rule, warp-specialised tensor-core chunk chain: the
// forward, and the reverse-chunk chain of state gradients of the backward.
//
// One CTA (384 threads) per (64-column value slice, head, sequence).  Two
// groups of warps run concurrently, one chunk apart:
//
//   prep  (warps 8-11), chunk c+1: g cumsum; Q K^T on the tensor cores and
//         the causal score P = (q_i.k_j) exp(G_i - G_j) (j <= i) as bf16 hi/lo
//         operand tiles; T = (I + A)^-1, A = beta_i (k_i.k_j) exp(G_i - G_j)
//         (j < i), copied in from the chunk-parallel kernel's tiles or, with
//         none given, formed here (K K^T on the tensor cores, fp32 inverse on
//         the CUDA cores).
//   chain (warps 0-7), chunk c:    K S, Q S -> R = beta o (V - gam o (K S));
//         Delta = T R; S <- gam_n S + K^T (dec o Delta); O = scale
//         [gam o (Q S) + P Delta].  S (fp32) lives in the chain's registers,
//         each row split between the two warps that share its TMEM
//         subpartition.
//
// Backward mode walks the chunks from last to first with the same prep; the
// chain carries dS, the gradient w.r.t. a chunk's end state, and steps it to
// the chunk's start state by the reverse mode of the update above:
//         dDelta = scale P^T dO + dec o (K dS);   dBhat = T^T dDelta;
//         dS <- gam_n dS + Q^T (scale gam o dO) - K^T (beta gam o dBhat).
// T and P are the same operand tiles read in the other major order.  Per
// chunk it stores dS (end-state gradient) for the chunk-parallel gradient
// pass; the forward in state mode stores each chunk's start state and its T
// tiles for the same pass.
//
// Delta = T R equals u - w S0 of the WY form (u = T diag(beta) V,
// w = T diag(beta gam) K), i.e. beta_i times the error v_i - v_old_i of the
// "Research Sprint Day 1" GDN update loop; decay is kept as a running sum of
// g ("Research Sprint Day 2 - Rooflines", GDN pseudocode step 5).  Computed
// MMA operands are split into bf16 hi + lo parts (fla issue #1550 traces the
// error of bf16 chunk kernels to rounding these intermediates), all
// accumulation is fp32 in tensor memory.
//
// Hand-offs are mbarriers (bounded waits): stage full (TMA), gram done,
// prep ready (T, P, gates of a chunk), slot free (T, P, gates double-buffered
// by chunk parity), and the MMA completions that the chain and the issuer
// warp (warp 12: the MMAs off the chain's critical path) wait on.  Ordering
// within the chain warps and within the prep warps uses named barriers 1 and 2.
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
constexpr int kIssuerWarp = 12;     // forward output: MMAs off the chain's critical path
constexpr int kThreads = kChainThreads + kPrepThreads + 32;
constexpr int kVs = 64;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kColG = 0;
constexpr uint32_t kColKS = 64;
constexpr uint32_t kColQS = 128;
constexpr uint32_t kColD = 192;
constexpr uint32_t kColPD = 256;
constexpr uint32_t kColS = 320;
constexpr uint32_t kColQK = 384;  // prep: Q K^T (K K^T at kColG)
constexpr uint32_t kColQS2 = 448;  // forward: Q S of odd chunks

constexpr int kRegions = kDk / 64;
constexpr int kStageBytes = kRegions * kRegionBytes;
constexpr int kTileS = kDk * 128;

// shared-memory map (bytes from a 1024-aligned base)
constexpr int oStage = 0;
constexpr int oShi = oStage + kStages * kStageBytes;
constexpr int oSlo = oShi + kTileS;
constexpr int oRhi = oSlo + kTileS;
constexpr int oRlo = oRhi + kTile64;
constexpr int oDhi = oRlo + kTile64;
constexpr int oDlo = oDhi + kTile64;
constexpr int oP = oDlo + kTile64;                  // [slot][hi,lo] P tiles
constexpr int oT = oP + 4 * kTile64;                // [slot][hi,lo] T tiles
constexpr int oA = oT + 4 * kTile64;                // A^T fp32 [64][64] (prep)
constexpr int oTf = oA + 64 * 64 * 4;               // fp32 32x32 blocks T_00, T_11, T_10 (prep)
constexpr int kTS = 36;                             // their row stride (16-byte rows, rows on distinct banks)
constexpr int kTB = 32 * kTS;                       // floats per block
constexpr int oVec = oTf + 3 * kTB * 4;             // [slot][g, beta, G, gam, dec] x 64 fp32
constexpr int kVecFloats = 5 * 64;
constexpr int oBar = oVec + 2 * kVecFloats * 4;
constexpr int kBars = 20;
constexpr int oMisc = oBar + kBars * 8;             // TMEM slot, abort flag
constexpr int kBytes = oMisc + 16;
// backward: the dO tile [i][v] bf16 shares the R tiles' space (dead between
// the previous chunk's K^T X and this chunk's dDelta)
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 232448, "shared memory");

// barrier indices
enum {
    B_FULL0 = 0, B_FULL1 = 1, B_GRAM = 2, B_KS = 3, B_D = 4, B_S = 5, B_PD = 6,
    B_READY0 = 7, B_READY1 = 8, B_TFREE0 = 9, B_TFREE1 = 10, B_TCOPY = 11,
    B_SFREE0 = 12, B_SFREE1 = 13, B_DRAIN0 = 14, B_DRAIN1 = 15, B_DRAIN2 = 16,
    // backward: warp 0 has issued K dS (the issuer warp issues P^T dO with
    // it); forward: Q S done; backward: Q^T G done
    B_KSI = 17, B_QSD = 18,
    // failure-detection test: a hand-off that nothing signals
    B_STALL = 19
};

__device__ __forceinline__ void named_bar(int id) { tc::named_bar(id, id == 1 ? kChainThreads : kPrepThreads); }

// Named barrier 1 (chain warps) or 2 (prep warps) that also ORs `pred` over
// its participants, so that every thread of the group takes the same
// decision (to leave after a wait ran out) whatever moment the shared abort
// flag was raised by another group.
__device__ __forceinline__ bool named_bar_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(id == 1 ? kChainThreads : kPrepThreads)
        : "memory");
    return r != 0;
}

// Bound of the waits that drain in-flight copies and products before a CTA
// leaves, independent of the hand-off bound: a short hand-off bound never
// lets a copy or a product outlive the CTA.
constexpr uint32_t kDrainLimit = kDefaultWaitLimit;

// Arguments of both directions.
struct ChainArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;            // forward
    const uint16_t* d_out;        // backward
    const float* g;
    const uint16_t* beta;
    float scale;
    const float* state_in;        // forward: initial state; backward: final-state gradient (may be null)
    const int32_t* cu_seqlens;
    uint16_t* out;                // forward output (may be null)
    float* out_f32;               // forward output in fp32 instead (the fp32-output instantiation only)
    int out_split;                // ... as bf16 hi and lo planes in out_f32's bytes (the split's identity run)
    float* state_out;             // forward: final state; backward: initial-state gradient (may be null)
    float* chunk_states;          // forward: chunk start states; backward: chunk end-state gradients (may be null)
    const uint8_t* chunk_T;       // T operand tiles of every chunk (may be null: formed in place)
    int N, T, H, d_k, d_v;
    int* err;
    int stall;                    // failure-detection test (forward): first wait on a hand-off nothing signals
};

struct WsParams {
    ChainArgs a;
    uint32_t wait_limit;
};

// kF32Out: the forward writes its output in fp32 to out_f32 (the sequence
// split's carry runs, whose outputs are combined later) instead of bf16.
template <bool kBwd, bool kF32Out = false>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chain_ws_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                        const WsParams prm) {
    const ChainArgs& p = prm.a;
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v, dk = p.d_k;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);  // 1024-aligned, still known to be shared memory
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oMisc + 4);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const bool use_tma = dk == kDk;
    const long long row_base = static_cast<long long>(b) * p.T;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    const bool want_out = !kBwd && (kF32Out ? p.out_f32 != nullptr : p.out != nullptr);
    // the prep forms P only where the chain uses it (output, or P^T dO), and
    // takes the T tiles from the chunk-parallel inverse when they are given
    const bool want_p = kBwd || want_out;
    const bool load_t = p.chunk_T != nullptr;
    const uint32_t wl = prm.wait_limit;
    // iteration it works on chunk chunk_of(it): forward in order, backward reversed
    auto chunk_of = [&](int it) { return kBwd ? nchunks - 1 - it : it; };
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);  // first per-chunk workspace slot

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        *abort_flag = 0;
        if (use_tma && nchunks > 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
        }
    }
    // the upper-right 16x16 blocks of the 32x32 inverse blocks T_00, T_11 stay zero
    for (int i = tid; i < 2 * 16 * 16; i += kThreads) {
        float* tb = reinterpret_cast<float*>(sm + oTf) + (i >> 8) * kTB;
        tb[((i >> 4) & 15) * kTS + 16 + (i & 15)] = 0.f;
    }
    // d_k = 64: the upper key region of every stage stays zero
    if (!use_tma) {
        for (int st = 0; st < kStages; ++st) {
            uint4* z = reinterpret_cast<uint4*>(sm + oStage + st * kStageBytes + kRegionBytes);
            for (int i = tid; i < kRegionBytes / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    auto issue_tma = [&](int it) {
        const int st = it % kStages;
        uint8_t* base = sm + oStage + st * kStageBytes;
        const int z = static_cast<int>(row_base + t0 + chunk_of(it) * kChunk);
        mbar_arrive_expect_tx(bar(B_FULL0 + st), kStageBytes);
#pragma unroll
        for (int r = 0; r < kRegions; ++r) {
            tma_load_3d(smem_u32(base + r * kRegionBytes), &tmap_k, r * 64, h, z, bar(B_FULL0 + st));
            tma_load_3d(smem_u32(base + r * kRegionBytes + 64 * 128), &tmap_q, r * 64, h, z, bar(B_FULL0 + st));
        }
    };

    if (warp < 8) {
        // ======================= chain warps =======================
        // Warps w and w + 4 share TMEM subpartition w % 4.  State rows: lane
        // l of warp w holds row 32 (w % 4) + l, columns 32 (w / 4) .. + 31 of
        // the slice.  M = 64 rows: lanes l and l + 16 of warps w and w + 4
        // hold row 16 (w % 4) + l % 16, one 16-column quarter each.
        const int t = tid;
        const int sw = warp & 3, hs = warp >> 2;
        const int srow_all = 32 * sw + lane;
        const int srow = srow_all < dk ? srow_all : -1;
        const int hrow = 16 * sw + (lane & 15);
        const int cq = 16 * (2 * hs + (lane >> 4));  // first column of this lane's quarter
        const uint32_t lb = static_cast<uint32_t>(sw * 32) << 16;
        // quarter row cq .. cq + 15 of M = 64 accumulator row hrow (no wait)
        auto ld_q16 = [&](uint32_t col, float* v) { tmem_ld_pair16(tmem + lb + col + 32 * hs, v); };
        // the two 16-byte chunks of columns cq .. cq + 15 of a split row
        auto store_q16 = [&](uint8_t* thi, uint8_t* tlo, int row, const float* x) {
            store_split_chunk(thi, tlo, row, cq >> 3, x);
            store_split_chunk(thi, tlo, row, (cq >> 3) + 1, x + 8);
        };
        // columns 32 hs .. + 31 of M = 128 accumulator row srow_all
        auto ld_s32 = [&](uint32_t col, float* v) {
            tmem_ld16(tmem + lb + col + 32 * hs, v);
            tmem_ld16(tmem + lb + col + 32 * hs + 16, v + 16);
            tmem_ld_wait();
        };
        const long long KV = static_cast<long long>(dk) * V;
        const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kVs;
        const float scale = p.scale;
        uint8_t* Shi = sm + oShi;
        uint8_t* Slo = sm + oSlo;
        uint8_t* Rhi = sm + oRhi;
        uint8_t* Rlo = sm + oRlo;
        uint8_t* Dhi = sm + oDhi;
        uint8_t* Dlo = sm + oDlo;
        int tma_issued = 0, tma_done = 0;
        if (use_tma && t == 0) {
            for (int ci = 0; ci < kStages && ci < nchunks; ++ci) issue_tma(ci);
        }
        if (use_tma) tma_issued = min(kStages, nchunks);

        float S[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = 0.f;
        if (srow >= 0 && p.state_in) {
            const float* src = p.state_in + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 t4 = *reinterpret_cast<const float4*>(src + j);
                S[j] = t4.x; S[j + 1] = t4.y; S[j + 2] = t4.z; S[j + 3] = t4.w;
            }
        }
        store_split_half(Shi, Slo, srow_all, hs, S);
        fence_proxy_async_smem();
        named_bar(1);

        // This chunk's state tile (forward: start state; backward: gradient
        // w.r.t. the end state) for the chunk-parallel gradient pass: bulk
        // copies of the bf16 hi/lo operand tiles, [slot][head][value slice][hi, lo].
        auto store_state_tiles = [&](int ci) {
            const long long nsl = V / kVs;
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.chunk_states) +
                           (((slot0 + ci) * H + h) * nsl + vs) * (2LL * dk * 128);
            bulk_s2g(dst, smem_u32(Shi), dk * 128);
            bulk_s2g(dst + dk * 128, smem_u32(Slo), dk * 128);
            bulk_commit();
        };
        bool aborted = false;
        if constexpr (!kBwd) {
            // a quarter value row of this slice (row hrow of the chunk, columns
            // cq .. cq + 15 of the slice), packed bf16; the next chunk's is
            // fetched as soon as the current one is consumed
            uint4 vraw[2];
            auto load_v = [&](int cj) {
                vraw[0] = vraw[1] = make_uint4(0, 0, 0, 0);
                const int cc0 = t0 + cj * kChunk;
                if (cj < nchunks && hrow < min(kChunk, t1 - cc0)) {
                    const uint4* src = reinterpret_cast<const uint4*>(
                        p.v + ((row_base + cc0 + hrow) * H + h) * static_cast<long long>(V) + vs * kVs + cq);
                    vraw[0] = src[0];
                    vraw[1] = src[1];
                }
            };
            // Q S goes to one of two column blocks by chunk parity: the output
            // of chunk c reads its block while chunk c+1's Q S is computed
            auto col_qs = [](int cj) { return (cj & 1) ? kColQS2 : kColQS; };
            // C1 of chunk cj: K S (warp 0, stage cj full); Q S follows from the
            // issuer warp, queued behind it
            auto issue_ks = [&](int cj) {
                const uint32_t stage_c = smem_u32(sm + oStage + (cj & 1) * kStageBytes);
                tc_fence_after();
                constexpr uint32_t id_s = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < kDk / 16; ++s) {
                    const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                    const uint64_t a_k = desc_sw128(stage_c + koff, 0, 1024);
                    const uint64_t b_hi = desc_sw128(smem_u32(Shi) + s * 2048, kTileS, 1024);
                    const uint64_t b_lo = desc_sw128(smem_u32(Slo) + s * 2048, kTileS, 1024);
                    mma_bf16(tmem + kColKS, a_k, b_hi, id_s, s > 0);
                    mma_bf16(tmem + kColKS, a_k, b_lo, id_s, 1);
                }
                mma_commit(bar(B_KS));
            };
            // warp 0 issues K S of chunk cj once its stage is full
            auto issue_c1 = [&](int cj) {
                if (warp == 0) {
                    const bool full = __all_sync(0xffffffffu, mbar_wait(bar(B_FULL0 + (cj & 1)), (cj >> 1) & 1, wl));
                    if (full) {
                        if (elect_one()) issue_ks(cj);
                        __syncwarp();
                        tma_done = cj + 1;
                    } else if (lane == 0) {
                        *abort_flag = 1;
                    }
                }
            };
            load_v(0);
            // the K S MMAs (critical path) go out before the start-state copies,
            // which read the same tiles
            if (nchunks > 0) {
                // failure-detection test: a wait that nothing ends runs out
                if (p.stall && warp == 0 && !__all_sync(0xffffffffu, mbar_wait(bar(B_STALL), 0, wl)) && lane == 0)
                    *abort_flag = 1;
                issue_c1(0);
                if (p.chunk_states && t == 0) store_state_tiles(0);
            }
            for (int ci = 0; ci < nchunks; ++ci) {
                const int c0 = t0 + ci * kChunk;
                const int nv = min(kChunk, t1 - c0);
                const int st = ci & 1, slot = ci & 1;
                const uint32_t ph = ci & 1, ph2 = (ci >> 1) & 1;
                const uint32_t stage_a = smem_u32(sm + oStage + st * kStageBytes);
                const float* vec = reinterpret_cast<const float*>(sm + oVec) + slot * kVecFloats;
                const float* bv = vec + 64;
                const float* gam = vec + 192;
                const float* dec = vec + 256;

                // K S and Q S of this chunk were issued at the end of the previous one
                __syncwarp();
                bool ok = mbar_wait(bar(B_READY0 + slot), ph2, wl);
                ok = mbar_wait(bar(B_KS), ph, wl) && ok;
                if (!ok) *abort_flag = 1;
                tc_fence_after();
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }

                // ---- C2: R = beta o (V - gam o (K S)) ----
                {
                    float row[16];
                    ld_q16(kColKS, row);
                    tmem_ld_wait();
                    const float bj = bv[hrow], gj = gam[hrow];
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const uint32_t w4[4] = {vraw[ch].x, vraw[ch].y, vraw[ch].z, vraw[ch].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int c = ch * 8 + 2 * m;
                            row[c] = bj * (__uint_as_float(w4[m] << 16) - gj * row[c]);
                            row[c + 1] = bj * (__uint_as_float(w4[m] & 0xffff0000u) - gj * row[c + 1]);
                        }
                    }
                    store_q16(Rhi, Rlo, hrow, row);
                }
                load_v(ci + 1);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(1);

                // ---- C3: Delta = T R ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        // A = T read MN-major from the T^T tile (row j holds column j of T)
                        constexpr uint32_t id = idesc(kFmtBf16, 1, 1, 64, 64);
                        const uint32_t thi = smem_u32(sm + oT + (slot * 2 + 0) * kTile64);
                        const uint32_t tlo = smem_u32(sm + oT + (slot * 2 + 1) * kTile64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t th = desc_sw128(thi + s * 2048, kTile64, 1024);
                            const uint64_t tl = desc_sw128(tlo + s * 2048, kTile64, 1024);
                            const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                            const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColD, th, rh, id, s > 0);
                            mma_bf16(tmem + kColD, th, rl, id, 1);
                            mma_bf16(tmem + kColD, tl, rh, id, 1);
                        }
                        mma_commit(bar(B_D));
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (!mbar_wait(bar(B_D), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }

                // ---- C4: Delta tiles and dec o Delta tiles ----
                {
                    float row[16];
                    ld_q16(kColD, row);
                    tmem_ld_wait();
                    store_q16(Dhi, Dlo, hrow, row);
                    const float dj = dec[hrow];
#pragma unroll
                    for (int c = 0; c < 16; ++c) row[c] *= dj;
                    store_q16(Rhi, Rlo, hrow, row);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(1);

                // ---- C5: S update (warp 0); P Delta follows from the issuer warp ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id_s = idesc(kFmtBf16, 1, 1, kDk, 64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ak = desc_sw128(stage_a + s * 2048, kRegionBytes, 1024);
                            const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                            const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColS, ak, rh, id_s, s > 0);
                            mma_bf16(tmem + kColS, ak, rl, id_s, 1);
                        }
                        mma_commit(bar(B_S));
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (!mbar_wait(bar(B_S), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                // ---- C6: state update (its TMEM read and FMAs run while Q S,
                // the last reader of the S tiles it overwrites, completes) ----
                {
                    float row[32];
                    const float gC = gam[63];
                    ld_s32(kColS, row);
#pragma unroll
                    for (int c = 0; c < 32; ++c) S[c] = fmaf(gC, S[c], row[c]);
                }
                // the S tiles get overwritten: Q S (issuer warp) has read them
                if (want_out && !mbar_wait(bar(B_QSD), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                if (p.chunk_states && t == 0) bulk_wait_read_all();  // ... and so have the bulk copies
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }
                // every MMA that reads this chunk's K/Q stage has completed (K S,
                // the state update, Q S; the prep's gram long before): the stage
                // takes chunk ci + 2's tiles now, a whole epilogue window earlier
                // than after the output
                if (t == 0) {
                    if (use_tma) {
                        if (ci + kStages < nchunks) {
                            issue_tma(ci + kStages);
                            tma_issued = ci + kStages + 1;  // thread 0's count drives the drain
                        }
                    } else {
                        mbar_arrive(bar(B_SFREE0 + st));
                    }
                }

                store_split_half(Shi, Slo, srow_all, hs, S);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(1);
                // ---- next chunk's C1, issued ahead of this chunk's output ----
                if (ci + 1 < nchunks) {
                    issue_c1(ci + 1);
                    if (p.chunk_states && t == 0) store_state_tiles(ci + 1);
                }
                __syncwarp();
                if (want_out && !mbar_wait(bar(B_PD), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                // ---- output ----
                if (want_out) {
                    const bool mine = hrow < nv;
                    const float gi = gam[hrow];
                    float qs[16], pd[16];
                    ld_q16(col_qs(ci), qs);
                    ld_q16(kColPD, pd);
                    tmem_ld_wait();
                    if (mine) {
                        const long long oo = ((row_base + c0 + hrow) * H + h) * static_cast<long long>(V) + vs * kVs + cq;
                        if constexpr (kF32Out) {
                            if (p.out_split) {
                                // hi plane, then lo plane (x = hi + lo), each [rows][H][d_v] bf16
                                float x[16];
#pragma unroll
                                for (int c = 0; c < 16; ++c) x[c] = scale * fmaf(gi, qs[c], pd[c]);
                                const long long plane =
                                    static_cast<long long>(p.cu_seqlens ? 1 : p.N) * p.T * H * static_cast<long long>(V);
                                uint4* dhi = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out_f32) + oo);
                                uint4* dlo = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out_f32) + plane + oo);
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    uint32_t wh[4], wl4[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int c = j * 8 + 2 * e;
                                        split_bf16x2(x[c], x[c + 1], wh[e], wl4[e]);
                                    }
                                    dhi[j] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                                    dlo[j] = make_uint4(wl4[0], wl4[1], wl4[2], wl4[3]);
                                }
                            } else {
                                float4* dst = reinterpret_cast<float4*>(p.out_f32 + oo);
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    dst[j] = make_float4(scale * fmaf(gi, qs[4 * j], pd[4 * j]),
                                                         scale * fmaf(gi, qs[4 * j + 1], pd[4 * j + 1]),
                                                         scale * fmaf(gi, qs[4 * j + 2], pd[4 * j + 2]),
                                                         scale * fmaf(gi, qs[4 * j + 3], pd[4 * j + 3]));
                            }
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(p.out + oo);
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                uint32_t w4[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int c = j * 8 + 2 * e;
                                    w4[e] = pack_bf16x2(scale * fmaf(gi, qs[c], pd[c]), scale * fmaf(gi, qs[c + 1], pd[c + 1]));
                                }
                                dst[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                const bool quit = named_bar_or(1, *abort_flag);
                if (t == 0) mbar_arrive(bar(B_TFREE0 + slot));  // T tiles and gates of this slot consumed
                if (quit) { aborted = true; break; }
            }
        } else {
            // a quarter dO row of this slice (row hrow of the chunk, columns
            // cq .. cq + 15 of the slice), packed bf16; the next chunk's is
            // fetched as soon as the current one is consumed
            uint4 oraw[2];
            auto load_do = [&](int it) {
                oraw[0] = oraw[1] = make_uint4(0, 0, 0, 0);
                if (it >= nchunks) return;
                const int cc0 = t0 + chunk_of(it) * kChunk;
                if (hrow < min(kChunk, t1 - cc0)) {
                    const uint4* src = reinterpret_cast<const uint4*>(
                        p.d_out + ((row_base + cc0 + hrow) * H + h) * static_cast<long long>(V) + vs * kVs + cq);
                    oraw[0] = src[0];
                    oraw[1] = src[1];
                }
            };
            load_do(0);
            uint8_t* dOt = sm + oRhi;
            for (int it = 0; it < nchunks; ++it) {
                const int ci = chunk_of(it);
                const int st = it & 1, slot = it & 1;
                const uint32_t ph = it & 1, ph2 = (it >> 1) & 1;
                const uint32_t stage_a = smem_u32(sm + oStage + st * kStageBytes);
                const float* vec = reinterpret_cast<const float*>(sm + oVec) + slot * kVecFloats;
                const float* bv = vec + 64;
                const float* gam = vec + 192;
                const float* dec = vec + 256;

                // gradient w.r.t. this chunk's end state, for the chunk-parallel pass
                if (p.chunk_states && t == 0) store_state_tiles(ci);
                // dO tile (single buffer: the previous chunk's P^T dO has completed)
#pragma unroll
                for (int ch = 0; ch < 2; ++ch)
                    *reinterpret_cast<uint4*>(dOt + sw128_offset(hrow, ((cq >> 3) + ch) * 16)) = oraw[ch];
                fence_proxy_async_smem();
                // K/Q tiles of this chunk
                if (!mbar_wait(bar(B_FULL0 + st), ph2, wl)) *abort_flag = 1;
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }
                tma_done = it + 1;

                // ---- C1: K dS (stage and dS tiles only) ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id_s = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                        for (int s = 0; s < kDk / 16; ++s) {
                            const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                            const uint64_t a_k = desc_sw128(stage_a + koff, 0, 1024);
                            const uint64_t b_hi = desc_sw128(smem_u32(Shi) + s * 2048, kTileS, 1024);
                            const uint64_t b_lo = desc_sw128(smem_u32(Slo) + s * 2048, kTileS, 1024);
                            mma_bf16(tmem + kColKS, a_k, b_hi, id_s, s > 0);
                            mma_bf16(tmem + kColKS, a_k, b_lo, id_s, 1);
                        }
                        mma_commit(bar(B_KS));
                        mbar_arrive(bar(B_KSI));
                    }
                    __syncwarp();
                }
                __syncwarp();
                // gates, T and P of this chunk from the prep warps
                if (!mbar_wait(bar(B_READY0 + slot), ph2, wl)) *abort_flag = 1;
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }

                // P^T dO comes from the issuer warp (behind K dS, once P is in)
                // G = scale gam o dO -> D tiles (B operand of Q^T G), while the MMAs run
                {
                    float row[16];
                    const float gi = scale * gam[hrow];  // dO rows beyond the chunk are zero
                    unpack8(oraw[0], row);
                    unpack8(oraw[1], row + 8);
#pragma unroll
                    for (int c = 0; c < 16; ++c) row[c] *= gi;
                    store_q16(Dhi, Dlo, hrow, row);
                }
                fence_proxy_async_smem();
                load_do(it + 1);
                __syncwarp();
                bool ok = mbar_wait(bar(B_KS), ph, wl);
                ok = mbar_wait(bar(B_PD), ph, wl) && ok;
                if (!ok) *abort_flag = 1;
                tc_fence_after();
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }

                // ---- C2: dDelta = scale P^T dO + dec o (K dS) -> R tiles ----
                {
                    const float dj = dec[hrow];
                    float kds[16], pdo[16];
                    ld_q16(kColKS, kds);
                    ld_q16(kColQS, pdo);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c) kds[c] = fmaf(scale, pdo[c], dj * kds[c]);
                    store_q16(Rhi, Rlo, hrow, kds);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(1);

                // ---- C3: dBhat = T^T dDelta (A = T tile read K-major) ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64);
                        const uint32_t thi = smem_u32(sm + oT + (slot * 2 + 0) * kTile64);
                        const uint32_t tlo = smem_u32(sm + oT + (slot * 2 + 1) * kTile64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t th = desc_sw128(thi + s * 32, 0, 1024);
                            const uint64_t tl = desc_sw128(tlo + s * 32, 0, 1024);
                            const uint64_t rh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                            const uint64_t rl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColD, th, rh, id, s > 0);
                            mma_bf16(tmem + kColD, th, rl, id, 1);
                            mma_bf16(tmem + kColD, tl, rh, id, 1);
                        }
                        mma_commit(bar(B_D));
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (!mbar_wait(bar(B_D), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }

                // ---- C4: X = -beta gam o dBhat -> R tiles (dDelta consumed) ----
                {
                    float row[16];
                    ld_q16(kColD, row);
                    tmem_ld_wait();
                    const float f = -bv[hrow] * gam[hrow];
#pragma unroll
                    for (int c = 0; c < 16; ++c) row[c] *= f;
                    store_q16(Rhi, Rlo, hrow, row);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar(1);

                // ---- C5: K^T X (A = K^T read MN-major from the stage); Q^T G comes from the issuer warp ----
                if (warp == 0) {
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc(kFmtBf16, 1, 1, kDk, 64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ak = desc_sw128(stage_a + s * 2048, kRegionBytes, 1024);
                            const uint64_t xh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                            const uint64_t xl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColS, ak, xh, id, s > 0);
                            mma_bf16(tmem + kColS, ak, xl, id, 1);
                        }
                        mma_commit(bar(B_S));
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (!mbar_wait(bar(B_S), ph, wl)) *abort_flag = 1;
                // Q^T G (issuer warp, its own TMEM block) has completed too
                if (!mbar_wait(bar(B_QSD), ph, wl)) *abort_flag = 1;
                tc_fence_after();
                if (p.chunk_states && t == 0) bulk_wait_read_all();  // C6 overwrites the S tiles
                if (named_bar_or(1, *abort_flag)) { aborted = true; break; }
                // every MMA that reads this chunk's K/Q stage has completed
                if (t == 0) {
                    if (use_tma) {
                        if (it + kStages < nchunks) issue_tma(it + kStages);
                    } else {
                        mbar_arrive(bar(B_SFREE0 + st));
                    }
                }
                if (use_tma && it + kStages < nchunks) tma_issued = it + kStages + 1;

                // ---- C6: dS <- gam_n dS + (K^T X + Q^T G) ----
                {
                    float row[32], qg[32];
                    const float gC = gam[63];
                    ld_s32(kColS, row);
                    ld_s32(kColG, qg);
#pragma unroll
                    for (int c = 0; c < 32; ++c) S[c] = fmaf(gC, S[c], row[c] + qg[c]);
                    store_split_half(Shi, Slo, srow_all, hs, S);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                const bool quit = named_bar_or(1, *abort_flag);
                if (t == 0) mbar_arrive(bar(B_TFREE0 + slot));  // T tiles and gates of this slot consumed
                if (quit) { aborted = true; break; }
            }
        }
        if (p.chunk_states && t == 0) bulk_wait_all();
        if (aborted) {
            if (warp == 0) {
                if (elect_one()) mma_commit(bar(B_DRAIN0));
                __syncwarp();
            }
            if (t == 0) {
                record_error(p.err, kErrTimeout);
                mbar_wait(bar(B_DRAIN0), 0, kDrainLimit);
                for (int ci = tma_done; ci < tma_issued; ++ci)
                    mbar_wait(bar(B_FULL0 + (ci & 1)), (ci >> 1) & 1, kDrainLimit);
            }
        } else if (p.state_out && srow >= 0) {
            float* dst = p.state_out + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    } else if (warp < 8 + kPrepThreads / 32) {
        // ======================= prep warps =======================
        const int q = tid - kChainThreads;  // 0..127
        const int sub = warp - 8;           // TMEM subpartition
        float* At = reinterpret_cast<float*>(sm + oA);  // A^T, row stride 64
        float* T00 = reinterpret_cast<float*>(sm + oTf);  // row-major 32x32 blocks of T
        float* T11 = T00 + kTB;
        float* T10 = T00 + 2 * kTB;
        // gates (g, beta) of row q of a chunk, fetched one chunk ahead
        float g_pre = 0.f, b_pre = 0.f;
        auto load_gates = [&](int it) {
            g_pre = 0.f;
            b_pre = 0.f;
            if (q < 64 && it < nchunks) {
                const int cc0 = t0 + chunk_of(it) * kChunk;
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
            const int ci = chunk_of(it);
            const int c0 = t0 + ci * kChunk;
            const int nv = min(kChunk, t1 - c0);
            const int st = it & 1, slot = it & 1;
            const uint32_t ph = it & 1, ph2 = (it >> 1) & 1;
            uint8_t* stage = sm + oStage + st * kStageBytes;
            float* vec = reinterpret_cast<float*>(sm + oVec) + slot * kVecFloats;
            float* gv = vec;
            float* bv = vec + 64;
            float* Gv = vec + 128;
            float* gam = vec + 192;
            float* dec = vec + 256;

            bool ok = true;
            // K/Q tiles
            if (!use_tma) {
                if (it >= 2) ok = mbar_wait(bar(B_SFREE0 + st), ((it - 2) >> 1) & 1, wl);
                if (!ok) *abort_flag = 1;
                if (named_bar_or(2, *abort_flag)) { aborted = true; break; }
                // every load of this thread is in flight before the first
                // store (the stores could alias the loads for the compiler)
                constexpr int kPer = 2 * 64 * 8 / 128;
                uint4 val[kPer];
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int e = q + u * 128, which = e >> 9, r = (e >> 3) & 63, ch = e & 7;
                    val[u] = make_uint4(0, 0, 0, 0);
                    if (r < nv) {
                        const uint16_t* src = which ? p.q : p.k;
                        val[u] = *reinterpret_cast<const uint4*>(src + ((row_base + c0 + r) * H + h) * 64LL + ch * 8);
                    }
                }
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int e = q + u * 128, which = e >> 9, r = (e >> 3) & 63, ch = e & 7;
                    *reinterpret_cast<uint4*>(stage + which * 64 * 128 + sw128_offset(r, ch * 16)) = val[u];
                }
                fence_proxy_async_smem();
                named_bar(2);
                if (q == 0) mbar_arrive(bar(B_FULL0 + st));
            }
            if (!mbar_wait(bar(B_FULL0 + st), ph2, wl)) *abort_flag = 1;
            if (named_bar_or(2, *abort_flag)) { aborted = true; break; }

            // gram K K^T and Q K^T (two M = 64 products), running while the
            // gates are formed.  Forward with T tiles given (only Q K^T): issued
            // once the chain's T R of the previous chunk has completed, so it
            // runs in that chunk's Delta epilogue window instead of beside the
            // state update that follows it
            if (warp == 8) {
                bool go = true;
                if (!kBwd && load_t && it > 0) {
                    go = __all_sync(0xffffffffu, mbar_wait(bar(B_D), (it - 1) & 1, wl));
                    if (!go && lane == 0) *abort_flag = 1;
                }
                if (go && elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_g = idesc(kFmtBf16, 0, 0, 64, 64);
                    const uint32_t stage_a = smem_u32(stage);
#pragma unroll
                    for (int s = 0; s < kDk / 16; ++s) {
                        const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                        const uint64_t a_k = desc_sw128(stage_a + koff, 0, 1024);
                        const uint64_t a_q = desc_sw128(stage_a + koff + 64 * 128, 0, 1024);
                        if (!load_t) mma_bf16(tmem + kColG, a_k, a_k, id_g, s > 0);
                        if (want_p) mma_bf16(tmem + kColQK, a_q, a_k, id_g, s > 0);
                    }
                    mma_commit(bar(B_GRAM));
                }
                __syncwarp();
            }

            // gates of this chunk into its slot (free once the chain finished iteration it - 2)
            ok = true;
            if (it >= 2) ok = mbar_wait(bar(B_TFREE0 + slot), ((it - 2) >> 1) & 1, wl);
            if (!ok) *abort_flag = 1;
            if (named_bar_or(2, *abort_flag)) { aborted = true; break; }
            if (load_t && q == 0) {
                // T tiles of this chunk (from the chunk-parallel inverse) into the free slot
                mbar_arrive_expect_tx(bar(B_TCOPY), 2 * kTile64);
                bulk_g2s(smem_u32(sm + oT + (slot * 2) * kTile64),
                         p.chunk_T + ((slot0 + ci) * H + h) * (2LL * kTile64), 2 * kTile64, bar(B_TCOPY));
                tcopy_out = true;
                tcopy_it = it;
            }
            if (q < 64) {
                gv[q] = g_pre;
                bv[q] = b_pre;
            }
            load_gates(it + 1);
            named_bar(2);
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
            named_bar(2);
            if (q < 64) dec[q] = exp_nonpos(Gv[63] - Gv[q]);

            __syncwarp();
            if (!mbar_wait(bar(B_GRAM), ph, wl)) *abort_flag = 1;
            tc_fence_after();
            if (named_bar_or(2, *abort_flag)) { aborted = true; break; }

            // All four warps form the chunk's decayed products: thread (warp w,
            // lane l) takes row i = 16 (w - 4) + l % 16 and columns 32 (l / 16) ..
            // + 31.  The decay e^{G_i - G_j} is formed once and used for A
            // (j < i) and P (j <= i).  Then warps 4-5 invert the four 16x16
            // diagonal blocks of I + A, and all four warps join the blocks level
            // by level: with T = (I + A)^-1 split into 2x2 blocks,
            // T_bb = (I + A_bb)^-1 and T_10 = -T_11 A_10 T_00, first inside each
            // 32x32 diagonal block (16x16 blocks), then for the 64x64 matrix
            // (32x32 blocks).  The products' scratch X lives in the unused upper
            // triangle of A^T.
            {
                const int i = 16 * sub + (lane & 15), hf = lane >> 4, j0 = 32 * hf;
                const float Gi = Gv[i], bi = bv[i];
                float mdec[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) mdec[k] = (j0 + k <= i) ? exp_nonpos(Gi - Gv[j0 + k]) : 0.f;
                // the M = 64 products sit in lanes 0-15 of each subpartition:
                // lanes l and l + 16 read the two column halves of row i
                if (!load_t) {
                    float lo[32];
                    ld_half32(tmem, sub, kColG, lo);
#pragma unroll
                    for (int k = 0; k < 32; ++k) lo[k] = (j0 + k < i) ? bi * lo[k] * mdec[k] : 0.f;
#pragma unroll
                    for (int k = 0; k < 32; ++k) At[(j0 + k) * 64 + i] = lo[k];
                }
                if (want_p) {
                    float lo[32];
                    ld_half32(tmem, sub, kColQK, lo);
#pragma unroll
                    for (int k = 0; k < 32; ++k) lo[k] *= mdec[k];
                    // P tiles of this slot are free: the chain finished iteration it - 2
                    uint8_t* p_hi = sm + oP + (2 * slot) * kTile64;
                    uint8_t* p_lo = sm + oP + (2 * slot + 1) * kTile64;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) store_split_chunk(p_hi, p_lo, i, 4 * hf + c4, lo + 8 * c4);
                }
            }
            tc_fence_before();
            named_bar(2);
            if (!load_t) {
                if (q < 64) {
                    // column c of the 16x16 diagonal block d = q / 16 by right-looking
                    // forward substitution: x = e_c; for m: for i > m: x_i -= A_im x_m.
                    // Row m of A^T is read as broadcast 16-byte loads.
                    const int d = q >> 4, c = q & 15;
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
                    const float* ablk = At + 16 * d * 64 + 16 * d;
#pragma unroll
                    for (int m = 0; m < 15; ++m) {
                        const float xm = x[m];
                        const float4* arow = reinterpret_cast<const float4*>(ablk + m * 64);
#pragma unroll
                        for (int i4 = (m + 1) >> 2; i4 < 4; ++i4) {
                            const float4 a4 = arow[i4];
                            if (4 * i4 + 0 > m) x[4 * i4 + 0] = fmaf(-a4.x, xm, x[4 * i4 + 0]);
                            if (4 * i4 + 1 > m) x[4 * i4 + 1] = fmaf(-a4.y, xm, x[4 * i4 + 1]);
                            if (4 * i4 + 2 > m) x[4 * i4 + 2] = fmaf(-a4.z, xm, x[4 * i4 + 2]);
                            if (4 * i4 + 3 > m) x[4 * i4 + 3] = fmaf(-a4.w, xm, x[4 * i4 + 3]);
                        }
                    }
                    // into the 32x32 block T_bb (b = d / 2) at rows/columns 16 (d % 2) ..
                    float* tb = (d >> 1 ? T11 : T00) + (16 * (d & 1)) * (kTS + 1) + c;
#pragma unroll
                    for (int i = 0; i < 16; ++i) tb[i * kTS] = x[i];
                }
                ok = true;
                named_bar(2);
                {
                    // lower-left 16x16 block of T_bb (b = q / 64): X = A_10 T_00 (16x16
                    // blocks of the 32x32 diagonal block), thread q: row r, columns c4 .. c4 + 3
                    const int b = q >> 6, r = (q >> 2) & 15, c4 = (q & 3) * 4;
                    float* tb = b ? T11 : T00;
                    const int o = 32 * b;  // first row/column of the 32x32 block in A
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float a = At[(o + k) * 64 + o + 16 + r];
                        const float4 t4 = *reinterpret_cast<const float4*>(tb + k * kTS + c4);
                        acc.x = fmaf(a, t4.x, acc.x); acc.y = fmaf(a, t4.y, acc.y);
                        acc.z = fmaf(a, t4.z, acc.z); acc.w = fmaf(a, t4.w, acc.w);
                    }
                    float* xs = At + (o + 16) * 64 + o;  // upper triangle of A^T: free
                    *reinterpret_cast<float4*>(xs + r * 64 + c4) = acc;
                    named_bar(2);
                    // T_10 = -T_11 X (T_11 the lower-right 16x16 block, unit lower triangular)
                    acc = *reinterpret_cast<const float4*>(xs + r * 64 + c4);
#pragma unroll 4
                    for (int k = 0; k < r; ++k) {
                        const float a = tb[(16 + r) * kTS + 16 + k];
                        const float4 v4 = *reinterpret_cast<const float4*>(xs + k * 64 + c4);
                        acc.x = fmaf(a, v4.x, acc.x); acc.y = fmaf(a, v4.y, acc.y);
                        acc.z = fmaf(a, v4.z, acc.z); acc.w = fmaf(a, v4.w, acc.w);
                    }
                    *reinterpret_cast<float4*>(tb + (16 + r) * kTS + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                named_bar(2);
                {
                    // T_10 of the 64x64 matrix: X = A_10 T_00 (32x32 blocks), thread q:
                    // row r = q / 4, columns c8 .. c8 + 7
                    const int r = q >> 2, c8 = (q & 3) * 8;
                    float acc[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 8
                    for (int k = 0; k < 32; ++k) {
                        const float a = At[k * 64 + 32 + r];
                        const float4 t0 = *reinterpret_cast<const float4*>(T00 + k * kTS + c8);
                        const float4 t1 = *reinterpret_cast<const float4*>(T00 + k * kTS + c8 + 4);
                        acc[0] = fmaf(a, t0.x, acc[0]); acc[1] = fmaf(a, t0.y, acc[1]);
                        acc[2] = fmaf(a, t0.z, acc[2]); acc[3] = fmaf(a, t0.w, acc[3]);
                        acc[4] = fmaf(a, t1.x, acc[4]); acc[5] = fmaf(a, t1.y, acc[5]);
                        acc[6] = fmaf(a, t1.z, acc[6]); acc[7] = fmaf(a, t1.w, acc[7]);
                    }
                    float* xs = At + 32 * 64;  // rows 32-63, columns 0-31 of A^T: free
                    *reinterpret_cast<float4*>(xs + r * 64 + c8) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    *reinterpret_cast<float4*>(xs + r * 64 + c8 + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    named_bar(2);
                    // T_10 = -T_11 X (T_11 unit lower triangular)
                    float4 u0 = *reinterpret_cast<const float4*>(xs + r * 64 + c8);
                    float4 u1 = *reinterpret_cast<const float4*>(xs + r * 64 + c8 + 4);
                    acc[0] = u0.x; acc[1] = u0.y; acc[2] = u0.z; acc[3] = u0.w;
                    acc[4] = u1.x; acc[5] = u1.y; acc[6] = u1.z; acc[7] = u1.w;
#pragma unroll 4
                    for (int k = 0; k < r; ++k) {
                        const float a = T11[r * kTS + k];
                        const float4 v0 = *reinterpret_cast<const float4*>(xs + k * 64 + c8);
                        const float4 v1 = *reinterpret_cast<const float4*>(xs + k * 64 + c8 + 4);
                        acc[0] = fmaf(a, v0.x, acc[0]); acc[1] = fmaf(a, v0.y, acc[1]);
                        acc[2] = fmaf(a, v0.z, acc[2]); acc[3] = fmaf(a, v0.w, acc[3]);
                        acc[4] = fmaf(a, v1.x, acc[4]); acc[5] = fmaf(a, v1.y, acc[5]);
                        acc[6] = fmaf(a, v1.z, acc[6]); acc[7] = fmaf(a, v1.w, acc[7]);
                    }
                    *reinterpret_cast<float4*>(T10 + r * kTS + c8) = make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
                    *reinterpret_cast<float4*>(T10 + r * kTS + c8 + 4) = make_float4(-acc[4], -acc[5], -acc[6], -acc[7]);
                }
                named_bar(2);
                {
                    // column col of T = row col of the T^T tile (read MN-major for T,
                    // K-major for T^T); this thread writes its entries 32 hf .. 32 hf + 31
                    const int col = q & 63, hf = q >> 6;
                    const float* src = col < 32 ? (hf ? T10 : T00) : (hf ? T11 : nullptr);
                    const int cc = col & 31;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = src ? src[i * kTS + cc] : 0.f;
                    uint8_t* t_hi = sm + oT + (slot * 2 + 0) * kTile64;
                    uint8_t* t_lo = sm + oT + (slot * 2 + 1) * kTile64;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) store_split_chunk(t_hi, t_lo, col, 4 * hf + c4, v + 8 * c4);
                }
            }
            fence_proxy_async_smem();
            if (named_bar_or(2, *abort_flag)) { aborted = true; break; }
            if (q == 0) {
                if (load_t) {
                    if (mbar_wait(bar(B_TCOPY), it & 1, wl)) tcopy_out = false;
                    else *abort_flag = 1;
                }
                if (!tcopy_out) mbar_arrive(bar(B_READY0 + slot));
            }
        }
        if (q == 0 && tcopy_out) mbar_wait(bar(B_TCOPY), tcopy_it & 1, kDrainLimit);  // no copy outlives the CTA
        if (aborted) {
            if (warp == 8) {
                if (elect_one()) mma_commit(bar(B_DRAIN1));
                __syncwarp();
            }
            if (q == 0) {
                record_error(p.err, kErrTimeout);
                mbar_wait(bar(B_DRAIN1), 0, kDrainLimit);
            }
        }
    } else if (warp == kIssuerWarp) {
        // ============ off-path MMAs of the forward output (issuer warp) ============
        // Q S and P Delta are needed only by the output epilogue, and the
        // tensor pipe shares its time between MMAs of different issuing
        // threads, so this warp (no epilogue work of its own) issues them
        // only once warp 0's critical product has completed, into the
        // epilogue that follows it: the first half of Q S (key columns 0-63)
        // after K S, the second half after T R, P Delta after the state
        // update.
        if constexpr (kBwd) {
            // backward: P^T dO (A = P tile read MN-major) with K dS once the
            // prep's P tiles are in (dDelta needs both); Q^T G (A = Q^T read
            // MN-major from the stage) once T^T dDelta has completed
            if (nchunks > 0) {
                const uint32_t dot = smem_u32(sm + oRhi), dhi = smem_u32(sm + oDhi), dlo = smem_u32(sm + oDlo);
                bool ok = true;
                for (int it = 0; it < nchunks && ok; ++it) {
                    const uint32_t ph = it & 1, ph2 = (it >> 1) & 1;
                    const int slot = it & 1;
                    const uint32_t stage_c = smem_u32(sm + oStage + (it & 1) * kStageBytes);
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_KSI), ph, wl) && mbar_wait(bar(B_READY0 + slot), ph2, wl));
                    if (!ok) break;
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id_p = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t p_hi = desc_sw128(smem_u32(sm + oP + (2 * slot) * kTile64) + s * 2048, kTile64, 1024);
                            const uint64_t p_lo = desc_sw128(smem_u32(sm + oP + (2 * slot + 1) * kTile64) + s * 2048, kTile64, 1024);
                            const uint64_t b_o = desc_sw128(dot + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColQS, p_hi, b_o, id_p, s > 0);
                            mma_bf16(tmem + kColQS, p_lo, b_o, id_p, 1);
                        }
                        mma_commit(bar(B_PD));
                    }
                    __syncwarp();
                    // Q^T G into its own TMEM block (the K K^T block, free when T
                    // comes from the chunk-parallel kernel), in the X epilogue's
                    // window: after T^T dDelta has completed
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_D), ph, wl));
                    if (!ok) break;
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id = idesc(kFmtBf16, 1, 1, kDk, 64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t aq = desc_sw128(stage_c + 64 * 128 + s * 2048, kRegionBytes, 1024);
                            mma_bf16(tmem + kColG, aq, desc_sw128(dhi + s * 2048, kTile64, 1024), id, s > 0);
                            mma_bf16(tmem + kColG, aq, desc_sw128(dlo + s * 2048, kTile64, 1024), id, 1);
                        }
                        mma_commit(bar(B_QSD));
                    }
                    __syncwarp();
                }
                if (!ok && lane == 0) *abort_flag = 1;  // the chain records the timeout
                if (elect_one()) mma_commit(bar(B_DRAIN2));
                __syncwarp();
                mbar_wait(bar(B_DRAIN2), 0, kDrainLimit);
            }
        } else {
            if (want_out && nchunks > 0) {
                const uint32_t shi = smem_u32(sm + oShi), slo = smem_u32(sm + oSlo);
                const uint32_t dhi = smem_u32(sm + oDhi), dlo = smem_u32(sm + oDlo);
                bool ok = true;
                for (int ci = 0; ci < nchunks && ok; ++ci) {
                    const uint32_t ph = ci & 1;
                    const int slot = ci & 1;
                    const uint32_t stage_c = smem_u32(sm + oStage + (ci & 1) * kStageBytes);
                    const uint32_t cq = (ci & 1) ? kColQS2 : kColQS;
                    constexpr uint32_t id_s = idesc(kFmtBf16, 0, 1, 64, 64);
                    auto qs_steps = [&](int s0, int s1) {
                        tc_fence_after();
#pragma unroll
                        for (int s = s0; s < s1; ++s) {
                            const uint32_t koff = (s >> 2) * kRegionBytes + (s & 3) * 32;
                            const uint64_t a_q = desc_sw128(stage_c + koff + 64 * 128, 0, 1024);
                            mma_bf16(tmem + cq, a_q, desc_sw128(shi + s * 2048, kTileS, 1024), id_s, s > 0);
                            mma_bf16(tmem + cq, a_q, desc_sw128(slo + s * 2048, kTileS, 1024), id_s, 1);
                        }
                    };
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_KS), ph, wl));
                    if (!ok) break;
                    if (elect_one()) qs_steps(0, kDk / 32);
                    __syncwarp();
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_D), ph, wl));
                    if (!ok) break;
                    if (elect_one()) {
                        qs_steps(kDk / 32, kDk / 16);
                        mma_commit(bar(B_QSD));
                    }
                    __syncwarp();
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B_S), ph, wl));
                    if (!ok) break;
                    if (elect_one()) {
                        tc_fence_after();
                        constexpr uint32_t id_p = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t ph_ = desc_sw128(smem_u32(sm + oP + (2 * slot) * kTile64) + s * 32, 0, 1024);
                            const uint64_t pl_ = desc_sw128(smem_u32(sm + oP + (2 * slot + 1) * kTile64) + s * 32, 0, 1024);
                            const uint64_t dh = desc_sw128(dhi + s * 2048, kTile64, 1024);
                            const uint64_t dl = desc_sw128(dlo + s * 2048, kTile64, 1024);
                            mma_bf16(tmem + kColPD, ph_, dh, id_p, s > 0);
                            mma_bf16(tmem + kColPD, ph_, dl, id_p, 1);
                            mma_bf16(tmem + kColPD, pl_, dh, id_p, 1);
                        }
                        mma_commit(bar(B_PD));
                    }
                    __syncwarp();
                }
                if (!ok && lane == 0) *abort_flag = 1;  // the chain records the timeout
                // nothing this warp issued is in flight when the CTA frees its TMEM
                if (elect_one()) mma_commit(bar(B_DRAIN2));
                __syncwarp();
                mbar_wait(bar(B_DRAIN2), 0, kDrainLimit);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <bool kBwd, bool kF32Out = false>
cudaError_t launch_chain(const ChainArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    CUtensorMap mk, mq;  // used for d_k = 128 only (d_k = 64 tiles use plain loads)
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    if (rows > 0 && a.d_k == kDk && (!make_qk_map(&mk, a.k, rows, a.H) || !make_qk_map(&mq, a.q, rows, a.H)))
        return cudaErrorInvalidValue;
    constexpr int smem = kAlloc;
    cudaError_t e = cudaFuncSetAttribute(gdn_chain_ws_kernel<kBwd, kF32Out>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    WsParams prm{a, wait_limit};
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_chain_ws_kernel<kBwd, kF32Out><<<grid, kThreads, smem, stream>>>(mk, mq, prm);
    return cudaGetLastError();
}

// No tokens at all (T = 0): every sequence is empty, so its final state is
// its initial state (or zero).  One block per (head, sequence); the packed
// offsets are still checked.
__global__ void __launch_bounds__(256) gdn_state_passthrough_kernel(FwdArgs p) {
    const int h = blockIdx.x, n = blockIdx.y;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    if (p.final_state == nullptr) return;
    const long long KV = static_cast<long long>(p.d_k) * p.d_v;
    const long long off = (static_cast<long long>(n) * p.H + h) * KV;
    float4* dst = reinterpret_cast<float4*>(p.final_state + off);
    const float4* src = p.initial_state ? reinterpret_cast<const float4*>(p.initial_state + off) : nullptr;
    for (long long i = threadIdx.x; i < KV / 4; i += blockDim.x)
        dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t launch_fwd_ws(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    if (rows == 0) {
        // nothing to load: state pass-through only
        if (a.N == 0 || a.H == 0) return cudaSuccess;
        gdn_state_passthrough_kernel<<<dim3(a.H, a.N), 256, 0, stream>>>(a);
        return cudaGetLastError();
    }
    ChainArgs c{};
    c.q = a.q; c.k = a.k; c.v = a.v; c.d_out = nullptr; c.g = a.g; c.beta = a.beta; c.scale = a.scale;
    c.state_in = a.initial_state; c.cu_seqlens = a.cu_seqlens; c.out = a.out; c.state_out = a.final_state;
    c.chunk_states = a.chunk_states; c.chunk_T = a.chunk_T;
    c.N = a.N; c.T = a.T; c.H = a.H; c.d_k = a.d_k; c.d_v = a.d_v; c.err = a.err; c.stall = a.stall;
    c.out_f32 = nullptr;
    return launch_chain<false>(c, wait_limit, stream);
}

cudaError_t launch_fwd_ws_f32(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    if (rows == 0 || a.out_f32 == nullptr) return cudaErrorInvalidValue;  // only the split's carry runs use it
    ChainArgs c{};
    c.q = a.q; c.k = a.k; c.v = a.v; c.d_out = nullptr; c.g = a.g; c.beta = a.beta; c.scale = a.scale;
    c.state_in = a.initial_state; c.cu_seqlens = a.cu_seqlens; c.out = nullptr; c.out_f32 = a.out_f32;
    c.out_split = a.out_split;
    c.state_out = a.final_state; c.chunk_states = a.chunk_states; c.chunk_T = a.chunk_T;
    c.N = a.N; c.T = a.T; c.H = a.H; c.d_k = a.d_k; c.d_v = a.d_v; c.err = a.err; c.stall = 0;
    return launch_chain<false, true>(c, wait_limit, stream);
}

cudaError_t launch_bwd_chain(const BwdChainArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    // the backward chain takes T from the chunk-parallel kernel: its Q^T G
    // product uses the TMEM block that the in-place K K^T would occupy
    if (a.T > 0 && a.chunk_T == nullptr) return cudaErrorInvalidValue;
    ChainArgs c{};
    c.q = a.q; c.k = a.k; c.v = nullptr; c.d_out = a.d_out; c.g = a.g; c.beta = a.beta; c.scale = a.scale;
    c.state_in = a.d_final_state; c.cu_seqlens = a.cu_seqlens; c.out = nullptr; c.state_out = a.d_initial_state;
    c.chunk_states = a.chunk_dstates; c.chunk_T = a.chunk_T;
    c.N = a.N; c.T = a.T; c.H = a.H; c.d_k = a.d_k; c.d_v = a.d_v; c.err = a.err;
    return launch_chain<true>(c, wait_limit, stream);
}

}  // namespace gdn

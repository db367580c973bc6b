// Backward, pass 3: every local gradient of one chunk, chunk-parallel, on the
// tensor cores.
//
// Given the chunk's start state S0 and its T operand tiles (pass 1) and the
// gradient dS w.r.t. its end state (pass 2), the reverse mode of the chunk
// forward (gdn_common.cuh) gives, with Bhat = diag(beta) V - diag(beta gam) K S0,
// R = beta o (V - gam o (K S0)), Delta = T R:
//   dDelta = scale P^T dO + dec o (K dS);   dBhat = T^T dDelta
//   dP = scale dO Delta^T  -> dQK = dP o M,  dG from dP o P
//   dA = -(dBhat Delta^T) o strict  -> dKK = dA o beta_i Ms,  dbeta, dG
//   dV = beta o dBhat
//   dQ = scale gam o (dO S0^T) + dQK K
//   dK = dQK^T Q + dKK K + dKK^T K + (dec o Delta) dS^T - (beta gam o dBhat) S0^T
//   dbeta, dgam, dG (decays), dg = reverse running sum of dG in the chunk.
// Sums over value columns (dP, dA, dO S0^T, the S-terms of dK) accumulate in
// tensor memory across 64-column value slices, so each CTA writes complete
// gradients: no partial sums leave the chip.
//
// Persistent CTAs (one per SM) walk the (chunk, head, sequence) items with a
// grid stride.  Warps 0-7 load, run every epilogue and write the gradients;
// warp 8 issues every MMA batch, each after a hand-off barrier that delivers
// its operands (a long batch blocks the thread that issues it until the
// tensor pipe has taken most of it, so an epilogue warp that issued would hold
// up every barrier after it).  Warps 9-11 only complete the issuer's
// warpgroup, whose registers go to the epilogue warpgroups.  While one item's
// chunk-wide products run, the next item's K/Q tiles (TMA), T tiles and first
// state tiles (bulk copies) land in buffers the current item no longer reads:
// the K/Q tiles alternate between two buffers, the other one holding the
// current item's -dBhat-side tiles.  Within an item the next value slice's S0
// tiles load into this slice's dS buffer as soon as the products that read dS
// have completed, and its dS tiles into this slice's S0 buffer after the last
// product that reads S0 (the two state buffers swap roles every slice).
// Warps w and w + 4 share a TMEM subpartition and split the 64 columns of each
// accumulator row between them, and within a warp lanes l and l + 16 take 16
// columns each of row 16 w + l (tcgen05.ld 16x32bx2), so every lane works in
// each epilogue.  Computed MMA operands are split into bf16 hi + lo,
// accumulation is fp32.
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

constexpr int kEpi = 256;                 // warps 0-7: loads, epilogues, outputs
constexpr int kIssuerWarp = 8;            // warp 8: issues every MMA (warps 9-11 idle)
constexpr int kThreads = kEpi + 128;
// registers: 168 a thread at launch (384 threads); the epilogue warps need
// ~184 (more measured no faster), the issuer's rolled MMA loops far fewer, so
// the issuer's warpgroup gives 32 a thread to the two epilogue warpgroups:
// 128 x 136 + 256 x 184 = 384 x 168
constexpr int kRegLaunch = 168, kRegIssuer = 136, kRegEpi = 184;
static_assert(128 * kRegIssuer + 256 * kRegEpi == kThreads * kRegLaunch, "register split");
constexpr int kVs = 64;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileS = kDk * 128;  // 128 rows x 128 B

// TMEM columns
constexpr uint32_t cdA = 0;     // dA (M = 64)
constexpr uint32_t cdP = 64;    // dP (M = 64)
constexpr uint32_t cU = 128;    // dO S0^T (M = 64, N = 128)
constexpr uint32_t cdK = 256;   // dK (M = 64, N = 128)
constexpr uint32_t cX1 = 384;   // scratch (M = 64)
constexpr uint32_t cX2 = 448;   // scratch (M = 64)

// shared memory (1024-aligned tiles)
constexpr int oKQ0 = 0;                         // [K;Q] regions of even items, 2 x 16 KB
constexpr int oT = oKQ0 + 2 * kRegionBytes;     // T^T-layout tiles hi, lo
constexpr int oP = oT + 2 * kTile64;            // P tiles hi, lo [i][j]; later the E scratch
constexpr int oSA = oP + 2 * kTile64;           // S0 tiles hi, lo [d][v]
constexpr int oSB = oSA + 2 * kTileS;           // dS tiles hi, lo [d][v]
constexpr int oDO = oSB + 2 * kTileS;           // dO raw [i][v]
constexpr int oRA = oDO + kTile64;              // R -> Delta (hi, lo) [j][v]; later dKK [i][j]
constexpr int oRB = oRA + 2 * kTile64;          // dDelta -> -dBhat; later dQK [i][j]
constexpr int oKQ1 = oRB + 2 * kTile64;         // [K;Q] of odd items; the other item's RC, RD tiles
constexpr int oVec = oKQ1 + 2 * kRegionBytes;   // g, beta, G, gam, dec, colsum
constexpr int oRed = oVec + 6 * 64 * 4;         // 16 floats reduction scratch
constexpr int oPart = oRed + 64;                // [64 rows][8] per-row partial sums of the upper column half;
                                                // earlier in the item's end the [4][64] partial column sums
constexpr int oBar = oPart + 64 * 8 * 4;        // mbarriers: MMA, item inputs, S0 tiles, dS tiles, off-path MMA, drain, stall
constexpr int oMisc = oBar + 56;                // TMEM slot, abort flag
constexpr int oDV = (oMisc + 16 + 1023) / 1024 * 1024;  // a full chunk's dV rows of one slice, staged for the TMA store
constexpr int kBytes = oDV + kTile64;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 232448, "shared memory");
static_assert(2 * kTile64 * 2 == 2 * kRegionBytes, "RC, RD fill a K/Q buffer");

// Named barrier 1: the epilogue warps among themselves.
__device__ __forceinline__ void epi_sync() { named_bar(1, kEpi); }

// Named barrier 2: the hand-off of a batch's operands from the epilogue warps
// to the issuer warp, which also ORs `pred` (a bounded wait ran out) over the
// nine warps, so that both sides leave the item loop at the same hand-off.
__device__ __forceinline__ bool handoff(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(kEpi + 32)
        : "memory");
    return r != 0;
}

// One (chunk, head, sequence) item.
struct Item {
    int ci, h, n, b, t0, t1;
};

__global__ void __launch_bounds__(kThreads, 1)
    gdn_bwd_local_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_dq, const __grid_constant__ CUtensorMap tmap_dk,
                         const __grid_constant__ CUtensorMap tmap_dv, const BwdLocalArgs p) {
    const int H = p.H, V = p.d_v, dk = p.d_k;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // TMEM subpartition of this warp and the column half it takes of a
    // 64-column accumulator row
    const int sub = warp & 3, hc = warp >> 2, col0 = 32 * hc;
    const float scale = p.scale;
    const bool use_tma = dk == kDk;
    const int nsl = V / kVs;
    const uint32_t nb = dk * 128;  // bytes of one state tile (hi or lo)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);  // 1024-aligned, still known to be shared memory
    float* gv = reinterpret_cast<float*>(sm + oVec);
    float* bv = gv + 64;
    float* Gv = gv + 128;
    float* gam = gv + 192;
    float* dec = gv + 256;
    float* colsum = gv + 320;
    float* red = reinterpret_cast<float*>(sm + oRed);
    uint64_t* barp = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oMisc + 4);
    const uint32_t bar = smem_u32(barp);
    const uint32_t ibar = smem_u32(barp + 1);
    const uint32_t s0bar = smem_u32(barp + 2);
    const uint32_t dsbar = smem_u32(barp + 3);
    // MMAs whose results only the item's outputs read (U += dO S0^T, dP +=
    // dO Delta^T) are committed here, after the products an epilogue waits
    // for, so they run in that epilogue's window
    const uint32_t nbar = smem_u32(barp + 4);
    // the issuer's last commit before the CTA leaves
    const uint32_t dbar = smem_u32(barp + 5);
    // failure-detection test: a barrier that nothing signals
    const uint32_t stallbar = smem_u32(barp + 6);
    // bound of the hand-off waits (the drains before the CTA leaves keep the default)
    const uint32_t wl = p.wait_limit ? p.wait_limit : kDefaultWaitLimit;

    // item f of the flat (chunk, head, sequence) order; false for chunks past
    // a sequence's end (and sequences whose bounds are invalid)
    const int maxc = p.max_chunks;
    const long long total = static_cast<long long>(maxc) * H * p.N;
    // (item counts stay far below 2^32: 32-bit division)
    auto decode = [&](long long f, Item& it) -> bool {
        const uint32_t fu = static_cast<uint32_t>(f), mc = static_cast<uint32_t>(maxc);
        const uint32_t ch = fu / mc;
        it.ci = static_cast<int>(fu - ch * mc);
        it.h = static_cast<int>(ch % static_cast<uint32_t>(H));
        it.n = static_cast<int>(ch / static_cast<uint32_t>(H));
        if (!seq_range(p.cu_seqlens, it.n, p.N, p.T, p.err, it.b, it.t0, it.t1)) return false;
        return it.ci < (it.t1 - it.t0 + kChunk - 1) / kChunk;
    };
    auto next_valid = [&](long long f, Item& it) -> long long {
        while (f < total && !decode(f, it)) f += gridDim.x;
        return f;
    };
    auto first_row = [&](const Item& it) {
        return static_cast<long long>(it.b) * p.T + it.t0 + static_cast<long long>(it.ci) * kChunk;
    };
    auto slot_of = [&](const Item& it) { return chunk_slot_base(p.cu_seqlens, it.n, p.T) + it.ci; };

    // async copies (thread 0: K/Q and T; threads 32 and 64: S0 and dS tiles;
    // thread 0 also at set-up); each thread records what it has in flight for
    // its drain
    bool i_out = false, s0_out = false, ds_out = false;
    // K/Q (TMA, d_k = 128) and T tiles of item `it` into K/Q buffer kqb
    auto issue_inputs = [&](const Item& it, uint32_t kqb) {
        const long long slot = slot_of(it);
        mbar_arrive_expect_tx(ibar, kChunkTBytes + (use_tma ? 2 * kRegionBytes : 0));
        if (use_tma) {
            const int z = static_cast<int>(first_row(it));
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                tma_load_3d(kqb + r * kRegionBytes, &tmap_k, r * 64, it.h, z, ibar);
                tma_load_3d(kqb + r * kRegionBytes + 64 * 128, &tmap_q, r * 64, it.h, z, ibar);
            }
        }
        bulk_g2s(smem_u32(sm + oT), p.chunk_T + (slot * H + it.h) * static_cast<long long>(kChunkTBytes),
                 kChunkTBytes, ibar);
        i_out = true;
    };
    // state tiles of value slice vs (bf16 hi/lo operand tiles written by the
    // state passes, [slot][head][slice][hi, lo])
    auto state_src = [&](const float* base, const Item& it, int vs) {
        return reinterpret_cast<const uint8_t*>(base) + ((slot_of(it) * H + it.h) * nsl + vs) * (2LL * dk * 128);
    };
    // The two state buffers SA and SB swap roles every value slice: slice vs
    // reads S0 from SA and dS from SB when vs is even, the other way round
    // when odd.  So the next slice's S0 can land in this slice's dS buffer
    // as soon as the products that read dS complete, and its dS in this
    // slice's S0 buffer after the last product that reads S0.
    auto issue_s0 = [&](const Item& it, int vs, int dst) {
        const uint8_t* s = state_src(p.chunk_states, it, vs);
        mbar_arrive_expect_tx(s0bar, 2 * nb);
        bulk_g2s(smem_u32(sm + dst), s, nb, s0bar);
        bulk_g2s(smem_u32(sm + dst + kTileS), s + nb, nb, s0bar);
        s0_out = true;
    };
    auto issue_ds = [&](const Item& it, int vs, int dst) {
        const uint8_t* s = state_src(p.chunk_dstates, it, vs);
        mbar_arrive_expect_tx(dsbar, 2 * nb);
        bulk_g2s(smem_u32(sm + dst), s, nb, dsbar);
        bulk_g2s(smem_u32(sm + dst + kTileS), s + nb, nb, dsbar);
        ds_out = true;
    };

    Item cur{};
    long long f = next_valid(blockIdx.x, cur);

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 7; ++i) mbar_init(smem_u32(barp + i), 1);
        fence_mbar_init();
        *abort_flag = 0;
        if (use_tma) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
        }
        if (f < total) {
            issue_inputs(cur, smem_u32(sm + oKQ0));
            issue_s0(cur, 0, oSA);
            issue_ds(cur, 0, oSB);
        }
    }
    // d_k = 64: key rows 64-127 of the state tiles stay zero (the copies
    // write rows 0-63 only)
    if (dk < kDk) {
        for (int e = tid; e < 4 * 64 * 8; e += kThreads) {
            const int tile = e >> 9, r = 64 + ((e >> 3) & 63), ch = e & 7;
            *reinterpret_cast<uint4*>(sm + (tile < 2 ? oSA : oSB) + (tile & 1) * kTileS + r * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    uint32_t phase = 0;
    bool failed = false;  // a bounded wait ran out (reported through the error word)
    // wait for the last commit on `bar` (issued inside an MMA batch)
    auto mma_wait = [&]() {
        if (!mbar_wait(bar, phase, wl)) {
            failed = true;
            *abort_flag = 1;
        }
        phase ^= 1u;
        tc_fence_after();
    };
    uint32_t nphase = 0;
    auto off_path_wait = [&]() {
        if (!mbar_wait(nbar, nphase, wl)) {
            failed = true;
            *abort_flag = 1;
        }
        nphase ^= 1u;
        tc_fence_after();
    };
    uint32_t iphase = 0, s0phase = 0, dsphase = 0;
    auto wait_copy = [&](uint32_t b, uint32_t& ph, bool& out) {
        if (mbar_wait(b, ph, wl)) {
            ph ^= 1u;
            out = false;
        } else {
            failed = true;
            *abort_flag = 1;
        }
    };

    // accumulator row of this lane and its 16 columns cb .. cb + 15 of a
    // 64-column block; lanes 0-15 hold the per-row sums after the pair join
    const int mrow = m64_half_row(sub, lane);
    const int cb = col0 + 16 * (lane >> 4);
    const bool lead = lane < 16;
    const uint32_t lb = static_cast<uint32_t>(sub * 32) << 16;
    // columns cb .. cb + 15 of accumulator row mrow (no wait)
    auto ld_cols = [&](uint32_t col, float* v) { tmem_ld_pair16(tmem + lb + col + col0, v); };
    // the two 16-byte chunks of columns cb .. cb + 15 of a split row
    auto store_cols = [&](int off, int row, const float* x) {
        store_split_chunk(sm + off, sm + off + kTile64, row, cb >> 3, x);
        store_split_chunk(sm + off, sm + off + kTile64, row, (cb >> 3) + 1, x + 8);
    };

    // per-item inputs held in registers, fetched one item (or slice) ahead:
    // gates of row tid (tid < 64), two 16-byte pieces of the dO tile, and
    // columns cb .. cb + 15 of value row mrow
    float g_pre = 0.f, b_pre = 0.f;
    uint4 do_raw[2], v_raw[2];
    auto fetch_gates = [&](const Item& it) {
        g_pre = b_pre = 0.f;
        const int nvv = min(kChunk, it.t1 - it.t0 - it.ci * kChunk);
        if (tid < nvv) {
            const long long idx = (first_row(it) + tid) * H + it.h;
            g_pre = p.g[idx];
            b_pre = bf16_to_f32(p.beta[idx]);
        }
    };
    auto fetch_rows = [&](const Item& it, int vs) {
        const int nvv = min(kChunk, it.t1 - it.t0 - it.ci * kChunk);
        const long long r0 = first_row(it);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int e = tid + k * kEpi, r = e >> 3, ch = e & 7;
            do_raw[k] = make_uint4(0, 0, 0, 0);
            if (r < nvv)
                do_raw[k] = *reinterpret_cast<const uint4*>(
                    p.d_out + ((r0 + r) * H + it.h) * static_cast<long long>(V) + vs * kVs + ch * 8);
        }
        v_raw[0] = v_raw[1] = make_uint4(0, 0, 0, 0);
        if (mrow < nvv) {
            const uint4* src = reinterpret_cast<const uint4*>(
                p.v + ((r0 + mrow) * H + it.h) * static_cast<long long>(V) + vs * kVs + cb);
            v_raw[0] = src[0];
            v_raw[1] = src[1];
        }
    };
    if (f < total && warp < kIssuerWarp) {
        fetch_gates(cur);
        fetch_rows(cur, 0);
    }

    if (warp >= kIssuerWarp) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegIssuer));
      // warps 9-11 only complete the issuer's warpgroup
      if (warp == kIssuerWarp) {
        // ---- the issuer warp: every MMA batch, in the epilogue warps' order,
        // each once the hand-off has delivered its operands; the epilogue
        // warps never wait for an issue (a long batch blocks its issuing
        // thread until the tensor pipe has taken most of it) ----
        for (int k = 0; f < total; ++k) {
            const uint32_t oKQ = (k & 1) ? oKQ1 : oKQ0;
            const uint32_t oRC = (k & 1) ? oKQ0 : oKQ1;
            const uint32_t oRD = oRC + 2 * kTile64;
            const uint32_t aKQ = smem_u32(sm + oKQ);
            auto kdesc_K = [&](int s) { return desc_sw128(aKQ + (s >> 2) * kRegionBytes + (s & 3) * 32, 0, 1024); };
            auto kdesc_Q = [&](int s) { return desc_sw128(aKQ + (s >> 2) * kRegionBytes + 64 * 128 + (s & 3) * 32, 0, 1024); };
            // K or Q read MN-major as a B operand [K = token][N = key column], N = 128
            auto mn_K = [&](int s) { return desc_sw128(aKQ + s * 2048, kRegionBytes, 1024); };
            auto mn_Q = [&](int s) { return desc_sw128(aKQ + 64 * 128 + s * 2048, kRegionBytes, 1024); };
            auto t64 = [&](int off) { return smem_u32(sm + off); };
            // P: Q K^T -> X1
            if (handoff(false)) break;
            if (elect_one()) {
                tc_fence_after();
                constexpr uint32_t id = idesc(kFmtBf16, 0, 0, 64, 64);
#pragma unroll 1
                for (int s = 0; s < kDk / 16; ++s) mma_bf16(tmem + cX1, kdesc_Q(s), kdesc_K(s), id, s > 0);
                mma_commit(bar);
            }
            __syncwarp();
            bool quit = false;
            for (int vs = 0; vs < nsl; ++vs) {
                const int oS0 = (vs & 1) ? oSB : oSA;
                const int oDS = (vs & 1) ? oSA : oSB;
                // batch 1
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_k = idesc(kFmtBf16, 0, 1, 64, 64);
                    constexpr uint32_t id_p = idesc(kFmtBf16, 1, 1, 64, 64);
                    constexpr uint32_t id_n = idesc(kFmtBf16, 0, 0, 64, 128);
#pragma unroll 1
                    for (int s = 0; s < kDk / 16; ++s) {
                        mma_bf16(tmem + cX1, kdesc_K(s), desc_sw128(t64(oS0) + s * 2048, kTileS, 1024), id_k, s > 0);
                        mma_bf16(tmem + cX1, kdesc_K(s), desc_sw128(t64(oS0 + kTileS) + s * 2048, kTileS, 1024), id_k, 1);
                    }
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t bo = desc_sw128(t64(oDO) + s * 2048, kTile64, 1024);
                        mma_bf16(tmem + cX2, desc_sw128(t64(oP) + s * 2048, kTile64, 1024), bo, id_p, s > 0);
                        mma_bf16(tmem + cX2, desc_sw128(t64(oP + kTile64) + s * 2048, kTile64, 1024), bo, id_p, 1);
                    }
                    mma_commit(bar);  // K S0 and P^T dO: the R epilogue reads them
                    // U += dO S0^T (B = S0 tile read K-major: [N = key row d][K =
                    // value column]), off the path: it runs in the R epilogue
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t ao = desc_sw128(t64(oDO) + s * 32, 0, 1024);
                        mma_bf16(tmem + cU, ao, desc_sw128(t64(oS0) + s * 32, 0, 1024), id_n, (vs > 0 || s > 0) ? 1u : 0u);
                        mma_bf16(tmem + cU, ao, desc_sw128(t64(oS0 + kTileS) + s * 32, 0, 1024), id_n, 1);
                    }
                    mma_commit(nbar);
                }
                __syncwarp();
                // batch 2: K dS (runs in the R epilogue), then T R
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_k = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll 1
                    for (int s = 0; s < kDk / 16; ++s) {
                        mma_bf16(tmem + cX1, kdesc_K(s), desc_sw128(t64(oDS) + s * 2048, kTileS, 1024), id_k, s > 0);
                        mma_bf16(tmem + cX1, kdesc_K(s), desc_sw128(t64(oDS + kTileS) + s * 2048, kTileS, 1024), id_k, 1);
                    }
                }
                __syncwarp();
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t th = desc_sw128(t64(oT) + s * 2048, kTile64, 1024);
                        const uint64_t tl = desc_sw128(t64(oT + kTile64) + s * 2048, kTile64, 1024);
                        const uint64_t rh = desc_sw128(t64(oRA) + s * 2048, kTile64, 1024);
                        const uint64_t rl = desc_sw128(t64(oRA + kTile64) + s * 2048, kTile64, 1024);
                        mma_bf16(tmem + cX2, th, rh, id_t, s > 0);
                        mma_bf16(tmem + cX2, th, rl, id_t, 1);
                        mma_bf16(tmem + cX2, tl, rh, id_t, 1);
                    }
                    mma_commit(bar);
                }
                __syncwarp();
                // batch 3
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_b = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t th = desc_sw128(t64(oT) + s * 32, 0, 1024);
                        const uint64_t tl = desc_sw128(t64(oT + kTile64) + s * 32, 0, 1024);
                        const uint64_t dh = desc_sw128(t64(oRB) + s * 2048, kTile64, 1024);
                        const uint64_t dl = desc_sw128(t64(oRB + kTile64) + s * 2048, kTile64, 1024);
                        mma_bf16(tmem + cX1, th, dh, id_b, s > 0);
                        mma_bf16(tmem + cX1, th, dl, id_b, 1);
                        mma_bf16(tmem + cX1, tl, dh, id_b, 1);
                    }
                    mma_commit(bar);  // dBhat: the dV epilogue reads it
                }
                __syncwarp();
                // batch 3, second part (once Delta and dec o Delta are stored):
                // read only at the item's end, it runs in the dV epilogue
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_p = idesc(kFmtBf16, 0, 0, 64, 64);
                    constexpr uint32_t id_n = idesc(kFmtBf16, 0, 0, 64, 128);
                    // dK += (dec o Delta) dS^T, the last reader of the dS tiles
                    // (B = dS tile read K-major: [N = key row d][K = value column])
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t eh = desc_sw128(t64(oRC) + s * 32, 0, 1024);
                        const uint64_t el = desc_sw128(t64(oRC + kTile64) + s * 32, 0, 1024);
                        const uint64_t sbh = desc_sw128(t64(oDS) + s * 32, 0, 1024);
                        const uint64_t sbl = desc_sw128(t64(oDS + kTileS) + s * 32, 0, 1024);
                        mma_bf16(tmem + cdK, eh, sbh, id_n, (vs > 0 || s > 0) ? 1u : 0u);
                        mma_bf16(tmem + cdK, eh, sbl, id_n, 1);
                        mma_bf16(tmem + cdK, el, sbh, id_n, 1);
                    }
                    // dP += dO Delta^T
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t ao = desc_sw128(t64(oDO) + s * 32, 0, 1024);
                        const uint64_t dh = desc_sw128(t64(oRA) + s * 32, 0, 1024);
                        const uint64_t dl = desc_sw128(t64(oRA + kTile64) + s * 32, 0, 1024);
                        mma_bf16(tmem + cdP, ao, dh, id_p, (vs > 0 || s > 0) ? 1u : 0u);
                        mma_bf16(tmem + cdP, ao, dl, id_p, 1);
                    }
                    mma_commit(nbar);
                }
                __syncwarp();
                // batch 4
                if (handoff(false)) {
                    quit = true;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after();
                    constexpr uint32_t id_c = idesc(kFmtBf16, 0, 0, 64, 64);
                    constexpr uint32_t id_n = idesc(kFmtBf16, 0, 0, 64, 128);
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t sah = desc_sw128(t64(oS0) + s * 32, 0, 1024);
                        const uint64_t sal = desc_sw128(t64(oS0 + kTileS) + s * 32, 0, 1024);
                        const uint64_t yh = desc_sw128(t64(oRD) + s * 32, 0, 1024);
                        const uint64_t yl = desc_sw128(t64(oRD + kTile64) + s * 32, 0, 1024);
                        mma_bf16(tmem + cdK, yh, sah, id_n, 1);
                        mma_bf16(tmem + cdK, yh, sal, id_n, 1);
                        mma_bf16(tmem + cdK, yl, sah, id_n, 1);
                    }
                    // before the last slice, the epilogue warps wait only for
                    // this last reader of the S0 tiles (the next slice's dS goes
                    // there); dA runs into the next slice's start, and the next
                    // slice's first commit covers it before Delta and -dBhat
                    // are rewritten
                    if (vs + 1 < nsl) mma_commit(bar);
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t ch_ = desc_sw128(t64(oRB) + s * 32, 0, 1024);
                        const uint64_t cl_ = desc_sw128(t64(oRB + kTile64) + s * 32, 0, 1024);
                        const uint64_t dh = desc_sw128(t64(oRA) + s * 32, 0, 1024);
                        const uint64_t dl = desc_sw128(t64(oRA + kTile64) + s * 32, 0, 1024);
                        mma_bf16(tmem + cdA, ch_, dh, id_c, (vs > 0 || s > 0) ? 1u : 0u);
                        mma_bf16(tmem + cdA, ch_, dl, id_c, 1);
                        mma_bf16(tmem + cdA, cl_, dh, id_c, 1);
                    }
                    if (vs + 1 == nsl) {
                        // chunk-wide part: K K^T and Q K^T (M = 64 each) into the
                        // scratch columns, queued behind the last slice's products
                        constexpr uint32_t id = idesc(kFmtBf16, 0, 0, 64, 64);
#pragma unroll 1
                        for (int s = 0; s < kDk / 16; ++s) {
                            mma_bf16(tmem + cX1, kdesc_K(s), kdesc_K(s), id, s > 0);
                            mma_bf16(tmem + cX2, kdesc_Q(s), kdesc_K(s), id, s > 0);
                        }
                        mma_commit(bar);  // the item's end reads dA, K K^T and Q K^T
                    }
                }
                __syncwarp();
            }
            if (quit) break;
            Item nxt{};
            const long long fn = next_valid(f + gridDim.x, nxt);
            // final products
            if (handoff(false)) break;
            if (elect_one()) {
                tc_fence_after();
                constexpr uint32_t id_n = idesc(kFmtBf16, 0, 1, 64, 128);   // A K-major, B MN-major
                constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 128);   // A MN-major (transposed)
#pragma unroll 1
                for (int s = 0; s < 4; ++s) {
                    const uint64_t qh = desc_sw128(t64(oRB) + s * 32, 0, 1024);
                    const uint64_t ql = desc_sw128(t64(oRB + kTile64) + s * 32, 0, 1024);
                    mma_bf16(tmem + cX1, qh, mn_K(s), id_n, s > 0);
                    mma_bf16(tmem + cX1, ql, mn_K(s), id_n, 1);
                }
                mma_commit(bar);  // dQ2: the dq outputs read it
                // the dK products complete while the dq outputs are formed
#pragma unroll 1
                for (int s = 0; s < 4; ++s) {
                    const uint64_t kh = desc_sw128(t64(oRA) + s * 32, 0, 1024);
                    const uint64_t kl = desc_sw128(t64(oRA + kTile64) + s * 32, 0, 1024);
                    mma_bf16(tmem + cdK, kh, mn_K(s), id_n, 1);
                    mma_bf16(tmem + cdK, kl, mn_K(s), id_n, 1);
                    const uint64_t qth = desc_sw128(t64(oRB) + s * 2048, kTile64, 1024);
                    const uint64_t qtl = desc_sw128(t64(oRB + kTile64) + s * 2048, kTile64, 1024);
                    const uint64_t kth = desc_sw128(t64(oRA) + s * 2048, kTile64, 1024);
                    const uint64_t ktl = desc_sw128(t64(oRA + kTile64) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + cdK, qth, mn_Q(s), id_t, 1);
                    mma_bf16(tmem + cdK, qtl, mn_Q(s), id_t, 1);
                    mma_bf16(tmem + cdK, kth, mn_K(s), id_t, 1);
                    mma_bf16(tmem + cdK, ktl, mn_K(s), id_t, 1);
                }
                mma_commit(nbar);
            }
            __syncwarp();
            cur = nxt;
            f = fn;
        }
        // the CTA leaves once every product it issued has completed
        if (elect_one()) mma_commit(dbar);
        __syncwarp();
        if (!mbar_wait(dbar, 0, kDefaultWaitLimit)) record_error(p.err, kErrTimeout);
      }
    } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegEpi));
    for (int k = 0; f < total; ++k) {
        const int h = cur.h;
        const int c0 = cur.t0 + cur.ci * kChunk;
        const int nv = min(kChunk, cur.t1 - c0);
        const long long row_base = static_cast<long long>(cur.b) * p.T;
        const uint32_t oKQ = (k & 1) ? oKQ1 : oKQ0;   // this item's K/Q buffer
        const uint32_t oRC = (k & 1) ? oKQ0 : oKQ1;   // -> dec o Delta, then free
        const uint32_t oRD = oRC + 2 * kTile64;       // Y = -beta gam dBhat

        // ---- item inputs: gates; K/Q (d_k = 64: plain loads), T tiles ----
        if (tid < 64) {
            gv[tid] = g_pre;
            bv[tid] = b_pre;
        }
        if (!use_tma) {
            // rows beyond the chunk and key columns beyond d_k are zero; every
            // load of this thread is in flight before the first store
            constexpr int kPer = 2 * 2 * 64 * 8 / kEpi;
            uint4 val[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int e = tid + u * kEpi;
                const int which = e >> 10;                // 0: K, 1: Q
                const int region = (e >> 9) & 1;          // key columns 0-63 / 64-127
                const int r = (e >> 3) & 63, ch = e & 7;
                val[u] = make_uint4(0, 0, 0, 0);
                if (r < nv && region * 64 < dk) {
                    const uint16_t* src = which ? p.q : p.k;
                    val[u] = *reinterpret_cast<const uint4*>(src + ((row_base + c0 + r) * H + h) * static_cast<long long>(dk) +
                                                             region * 64 + ch * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int e = tid + u * kEpi, which = e >> 10, region = (e >> 9) & 1, r = (e >> 3) & 63, ch = e & 7;
                *reinterpret_cast<uint4*>(sm + oKQ + region * kRegionBytes + which * 64 * 128 + sw128_offset(r, ch * 16)) = val[u];
            }
        }
        wait_copy(ibar, iphase, i_out);
        if (use_tma && nv < kChunk) {
            // the box also read the rows after the chunk: zero them
            for (int e = tid; e < 2 * 2 * 64 * 8; e += kEpi) {
                const int which = e >> 10, region = (e >> 9) & 1, r = (e >> 3) & 63, ch = e & 7;
                if (r >= nv)
                    *reinterpret_cast<uint4*>(sm + oKQ + region * kRegionBytes + which * 64 * 128 + sw128_offset(r, ch * 16)) =
                        make_uint4(0, 0, 0, 0);
            }
        }
        // failure-detection test: a first wait that nothing ends runs out
        if (p.stall && k == 0 && !mbar_wait(stallbar, 0, wl)) {
            failed = true;
            *abort_flag = 1;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        // hand-off: the issuer warp starts Q K^T (both sides leave here, and
        // at every later hand-off, if a bounded wait ran out)
        if (handoff(*abort_flag != 0)) break;
        if (tid < 32) {
            const float a = gv[2 * tid];
            const float bb = a + gv[2 * tid + 1];
            float s = bb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (tid >= off) s += o;
            }
            const float base = s - bb;
            Gv[2 * tid] = base + a;
            Gv[2 * tid + 1] = s;
            gam[2 * tid] = exp_nonpos(base + a);
            gam[2 * tid + 1] = exp_nonpos(s);
        }
        // the previous item's dq tile store has read the P tiles' space
        if (tid == 0) bulk_wait_read_all();
        epi_sync();
        if (tid < 64) dec[tid] = exp_nonpos(Gv[63] - Gv[tid]);

        // ---- P = (Q K^T) o M (j <= i) as operand tiles ----
        mma_wait();
        // decay factors exp(G_i - G_j) (j <= i) of row mrow, columns cb .. cb + 15:
        // the P epilogue and the item's end both read them
        float mdec[16];
        {
            float row[16];
            ld_cols(cX1, row);
            tmem_ld_wait();
            const float Gi = Gv[mrow];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                mdec[kk] = (cb + kk <= mrow) ? exp_nonpos(Gi - Gv[cb + kk]) : 0.f;
                row[kk] = (cb + kk <= mrow) ? row[kk] * mdec[kk] : 0.f;
            }
            store_cols(oP, mrow, row);
        }
        fence_proxy_async_smem();
        tc_fence_before();

        // per-row accumulators (thread mrow) across value slices
        float acc_dbeta = 0.f, acc_dgam = 0.f, acc_dd = 0.f, acc_SdS = 0.f;
        bool quit = false;
        for (int vs = 0; vs < nsl; ++vs) {
            const int oS0 = (vs & 1) ? oSB : oSA;  // this slice's S0 tiles
            const int oDS = (vs & 1) ? oSA : oSB;  // this slice's dS tiles
            // ---- slice loads: S0 tiles, dO tile, V row ----
            wait_copy(s0bar, s0phase, s0_out);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int e = tid + kk * kEpi, r = e >> 3, ch = e & 7;
                *reinterpret_cast<uint4*>(sm + oDO + sw128_offset(r, ch * 16)) = do_raw[kk];
            }
            // columns cb .. cb + 15 of value row mrow
            float vrow[16];
            unpack8(v_raw[0], vrow);
            unpack8(v_raw[1], vrow + 8);
            // the next slice's rows load while this slice runs
            if (vs + 1 < nsl) fetch_rows(cur, vs + 1);
            fence_proxy_async_smem();
            tc_fence_before();
            // the previous item's dq / dk and the previous slice's dV tile
            // stores have read their source tiles (rewritten in this slice)
            if (tid == 0) bulk_wait_read_all();
            // ---- batch 1 (issuer): K S0 -> X1, P^T dO -> X2, U += dO S0^T ----
            if (handoff(*abort_flag != 0)) {
                quit = true;
                break;
            }
            mma_wait();
            float ks0[16], pdo[16];
            ld_cols(cX1, ks0);
            ld_cols(cX2, pdo);
            tmem_ld_wait();
            tc_fence_before();
            // the dS tiles of this slice
            wait_copy(dsbar, dsphase, ds_out);
            // ---- batch 2 (issuer), first part: K dS -> X1 (X1 and X2 are
            // read), while R is formed ----
            if (handoff(*abort_flag != 0)) {
                quit = true;
                break;
            }
            {
                float row[16];
                const float bj = bv[mrow], gj = gam[mrow];
#pragma unroll
                for (int c = 0; c < 16; ++c) row[c] = bj * (vrow[c] - gj * ks0[c]);
                store_cols(oRA, mrow, row);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            // ---- batch 2 (issuer), second part: Delta = T R -> X2 ----
            if (handoff(*abort_flag != 0)) {
                quit = true;
                break;
            }
            {
                // <dS, S0> over 32 values of state row d (hi + lo is the fp32
                // value to ~16 bits), while the batch runs
                const int d = tid & 127, hs = tid >> 7;
                if (d < dk) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint32_t off = sw128_offset(d, (4 * hs + c4) * 16);
                        float ah[8], al[8], bh[8], bl[8];
                        unpack8(*reinterpret_cast<const uint4*>(sm + oS0 + off), ah);
                        unpack8(*reinterpret_cast<const uint4*>(sm + oS0 + kTileS + off), al);
                        unpack8(*reinterpret_cast<const uint4*>(sm + oDS + off), bh);
                        unpack8(*reinterpret_cast<const uint4*>(sm + oDS + kTileS + off), bl);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc_SdS = fmaf(ah[e] + al[e], bh[e] + bl[e], acc_SdS);
                    }
                }
            }
            mma_wait();
            off_path_wait();  // U of this slice (long done: it ran in the R epilogue)
            {
                // dDelta = scale P^T dO + dec o (K dS) -> RB;  Delta -> RA (replaces R);
                // dec o Delta -> RC;  dd = dec * sum_v (K dS) Delta for the decay term of dG
                const float dj = dec[mrow];
                float dd = 0.f;
                float kds[16], dl[16];
                ld_cols(cX1, kds);
                ld_cols(cX2, dl);
                tmem_ld_wait();
                tc_fence_before();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    dd = fmaf(kds[c], dl[c], dd);
                    kds[c] = fmaf(scale, pdo[c], dj * kds[c]);
                }
                store_cols(oRB, mrow, kds);
                fence_proxy_async_smem();
                // ---- batch 3 (issuer): dBhat = T^T dDelta -> X1 ----
                if (handoff(*abort_flag != 0)) {
                    quit = true;
                    break;
                }
                store_cols(oRA, mrow, dl);
#pragma unroll
                for (int c = 0; c < 16; ++c) dl[c] *= dj;
                store_cols(oRC, mrow, dl);
                acc_dd = fmaf(dj, dd, acc_dd);
            }
            fence_proxy_async_smem();
            // ---- batch 3, second part (issuer): dK += (dec o Delta) dS^T;  dP +=
            // dO Delta^T (off the path) ----
            if (handoff(*abort_flag != 0)) {
                quit = true;
                break;
            }
            mma_wait();
            {
                // dV = beta o dBhat; dbeta / dgam row terms; -dBhat -> RB, Y -> RD
                const float bi = bv[mrow], gi = gam[mrow];
                float sv = 0.f, sk = 0.f;
                float db[16], t16[16];
                ld_cols(cX1, db);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    sv = fmaf(vrow[c], db[c], sv);
                    sk = fmaf(ks0[c], db[c], sk);
                }
                uint4 dv4[2];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w4[e] = pack_bf16x2(bi * db[half * 8 + 2 * e], bi * db[half * 8 + 2 * e + 1]);
                    dv4[half] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                if (nv == kChunk) {
                    // a full chunk stages this slice's dV rows, 128-byte
                    // swizzled, for one TMA store
#pragma unroll
                    for (int half = 0; half < 2; ++half)
                        *reinterpret_cast<uint4*>(sm + oDV + sw128_offset(mrow, cb * 2 + 16 * half)) = dv4[half];
                } else if (mrow < nv) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        p.dv + ((row_base + c0 + mrow) * H + h) * static_cast<long long>(V) + vs * kVs + cb);
#pragma unroll
                    for (int half = 0; half < 2; ++half) dst[half] = dv4[half];
                }
#pragma unroll
                for (int c = 0; c < 16; ++c) t16[c] = -db[c];
                store_cols(oRB, mrow, t16);
#pragma unroll
                for (int c = 0; c < 16; ++c) t16[c] = -bi * gi * db[c];
                store_cols(oRD, mrow, t16);
                acc_dbeta += sv - gi * sk;
                acc_dgam -= bi * sk;
            }
            // once dK += (dec o Delta) dS^T has completed, the next slice's S0
            // goes into this slice's dS buffer (the wait leaves the phase to
            // the off-path wait at the slice's end).  The copies are spread
            // over warps 0-2 (thread 0: K/Q and T, 32: S0 tiles, 64: dS tiles),
            // so that no one warp is held by all the issues
            if (tid == 32 && vs + 1 < nsl && !failed) {
                if (mbar_wait(nbar, nphase, wl)) {
                    issue_s0(cur, vs + 1, oDS);
                } else {
                    failed = true;
                    *abort_flag = 1;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            // ---- batch 4 (issuer): dA += (-dBhat) Delta^T;  dK += Y S0^T ----
            if (handoff(*abort_flag != 0)) {
                quit = true;
                break;
            }
            // the hand-off also completed this slice's dV tile
            if (nv == kChunk && tid == 0) {
                tma_store_3d(&tmap_dv, vs * kVs, h, static_cast<int>(row_base + c0), smem_u32(sm + oDV));
                bulk_commit();
            }
            mma_wait();
            off_path_wait();  // dP: the next slice rewrites the dO and Delta tiles it reads
            epi_sync();
            // the S0 tiles are free: the next slice's dS goes there
            if (tid == 64 && vs + 1 < nsl && !failed) issue_ds(cur, vs + 1, oS0);
        }
        if (quit) break;

        Item nxt{};
        const long long fn = next_valid(f + gridDim.x, nxt);

        // ---- chunk-wide part (K K^T and Q K^T came with the last slice's batch) ----
        // column-sum terms E [64][64] fp32 in the (dead) P tiles, column index
        // XOR-swizzled by the row so that row-parallel writes and
        // column-parallel reads both spread over the banks
        float* E = reinterpret_cast<float*>(sm + oP);
        float rowsum = 0.f, dbeta_a = 0.f;
        {
            const int i = mrow;
            const float bi = bv[i];
            float kk[16], da[16], qk[16], dp[16];
            const int col = cb;
            ld_cols(cX1, kk);
            ld_cols(cdA, da);
            ld_cols(cX2, qk);
            ld_cols(cdP, dp);
            tmem_ld_wait();
            float dkk[16], dqk[16], e16[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int j = col + c;
                const float m = mdec[c];
                // A side (strictly lower): dA o (K K^T o Ms)
                const float kkm = (j < i) ? kk[c] * m : 0.f;
                const float a = (j < i) ? da[c] : 0.f;
                dbeta_a = fmaf(a, kkm, dbeta_a);
                const float dms = a * bi * kkm;
                dkk[c] = a * bi * m;
                // P side (diagonal included): dQK = dP o M and dP o P
                const float dpm = scale * dp[c] * m;
                dqk[c] = dpm;
                e16[c] = dms + dpm * qk[c];
                rowsum += e16[c];
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) E[i * 64 + ((col + c) ^ (i & 31))] = e16[c];
            store_cols(oRA, i, dkk);
            store_cols(oRB, i, dqk);
        }
        // <dS, S0> over the whole slice set (gam_n term of dgam)
        {
            float v = acc_SdS;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) red[warp] = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        // ---- final products (issuer): dQ2 = dQK K -> X1..X2;  dK += dQK^T Q + dKK K + dKK^T K ----
        if (handoff(*abort_flag != 0)) break;
        // the next item's inputs land while this item's end runs: K/Q into the
        // other buffer (RC, RD are dead), T, slice 0 states (issued after the
        // hand-off, so that no epilogue warp waits for the issuing thread)
        if (fn < total && !failed) {
            if (tid == 0) issue_inputs(nxt, smem_u32(sm + oRC));
            if (tid == 32) issue_s0(nxt, 0, oSA);
            if (tid == 64) issue_ds(nxt, 0, oSB);
        }
        // column sums of E while the products run: four partial sums of 16
        // rows per column, then their sum
        {
            float* cpart = reinterpret_cast<float*>(sm + oPart);
            const int col = tid & 63, r0 = 16 * (tid >> 6);
            float c = 0.f;
#pragma unroll
            for (int i = r0; i < r0 + 16; ++i) c += E[i * 64 + (col ^ (i & 31))];
            cpart[tid] = c;
        }
        // gates and the first slice's rows of the next item, while the products run
        if (fn < total) {
            fetch_gates(nxt);
            fetch_rows(nxt, 0);
        }
        epi_sync();
        if (tid < 64) {
            const float* cpart = reinterpret_cast<const float*>(sm + oPart);
            colsum[tid] = (cpart[tid] + cpart[64 + tid]) + (cpart[128 + tid] + cpart[192 + tid]);
        }
        mma_wait();  // dQ2
        epi_sync();
        // ---- outputs of row mrow (key columns 64 hc .. 64 hc + 63: 16-column
        // groups 4 hc + 2 r + lane / 16 of this lane) ----
        float dG = 0.f, dbeta = 0.f;
        {
            const int i = mrow;
            const float gi = gam[i];
            // U = dO S0^T: dQ term scale gam U and dgam term scale q . U
            float dgq = 0.f;
            // a full chunk at d_k = 128 stages its dq / dk rows, 128-byte
            // swizzled like the q / k tiles, for one TMA store per 64-column
            // region (dq in the dead E scratch, dk in the dQK tiles once the dK
            // products have read them): consecutive tokens are H d_k apart in
            // global memory, so per-thread 16-byte stores would touch a sector
            // each; a ragged chunk stores per thread (a box would cross into
            // the next rows)
            const bool tma_out = use_tma && nv == kChunk;
            {
                float u[2][16], q2[2][16];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t cpair = 64 * hc + 32 * r;  // lanes 16-31 read 16 columns further
                    tmem_ld_pair16(tmem + lb + cU + cpair, u[r]);
                    tmem_ld_pair16(tmem + lb + cX1 + cpair, q2[r]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int c16 = 4 * hc + 2 * r + (lane >> 4);
                    const int region = c16 >> 2, cc = (c16 & 3) * 16;
                    float qrow[16];
                    {
                        const uint8_t* base = sm + oKQ + region * kRegionBytes + 64 * 128;
                        unpack8(*reinterpret_cast<const uint4*>(base + sw128_offset(i, cc * 2)), qrow);
                        unpack8(*reinterpret_cast<const uint4*>(base + sw128_offset(i, cc * 2 + 16)), qrow + 8);
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) dgq = fmaf(scale * qrow[e], u[r][e], dgq);
                    uint4 wq4[2];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t wq[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = half * 8 + 2 * e;
                            wq[e] = pack_bf16x2(fmaf(scale * gi, u[r][c], q2[r][c]), fmaf(scale * gi, u[r][c + 1], q2[r][c + 1]));
                        }
                        wq4[half] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                    }
                    if (tma_out) {
#pragma unroll
                        for (int half = 0; half < 2; ++half)
                            *reinterpret_cast<uint4*>(sm + oP + region * kTile64 + sw128_offset(i, cc * 2 + 16 * half)) = wq4[half];
                    } else if (i < nv && c16 * 16 < dk) {
                        uint4* dq = reinterpret_cast<uint4*>(p.dq + ((row_base + c0 + i) * H + h) * static_cast<long long>(dk) + c16 * 16);
#pragma unroll
                        for (int half = 0; half < 2; ++half) dq[half] = wq4[half];
                    }
                }
            }
            off_path_wait();  // the dK products
            {
                float kk2[2][16];
#pragma unroll
                for (int r = 0; r < 2; ++r) tmem_ld_pair16(tmem + lb + cdK + 64 * hc + 32 * r, kk2[r]);
                tmem_ld_wait();
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int c16 = 4 * hc + 2 * r + (lane >> 4);
                    const int region = c16 >> 2, cc = (c16 & 3) * 16;
                    uint4 wk4[2];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t wk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = half * 8 + 2 * e;
                            wk[e] = pack_bf16x2(kk2[r][c], kk2[r][c + 1]);
                        }
                        wk4[half] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                    }
                    if (tma_out) {
#pragma unroll
                        for (int half = 0; half < 2; ++half)
                            *reinterpret_cast<uint4*>(sm + oRB + region * kTile64 + sw128_offset(i, cc * 2 + 16 * half)) = wk4[half];
                    } else if (i < nv && c16 * 16 < dk) {
                        uint4* dkp = reinterpret_cast<uint4*>(p.dk + ((row_base + c0 + i) * H + h) * static_cast<long long>(dk) + c16 * 16);
#pragma unroll
                        for (int half = 0; half < 2; ++half) dkp[half] = wk4[half];
                    }
                }
            }
            if (tma_out) fence_proxy_async_smem();
            // dG_63 also collects the decay terms sum_j dd_j (all rows, both halves)
            {
                float v = acc_dd;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) red[8 + warp] = v;
            }
            // lanes l and l + 16 hold the two column quarters of row i
            acc_dbeta += __shfl_xor_sync(0xffffffffu, acc_dbeta, 16);
            acc_dgam += __shfl_xor_sync(0xffffffffu, acc_dgam, 16);
            dgq += __shfl_xor_sync(0xffffffffu, dgq, 16);
            acc_dd += __shfl_xor_sync(0xffffffffu, acc_dd, 16);
            rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 16);
            dbeta_a += __shfl_xor_sync(0xffffffffu, dbeta_a, 16);
            // the row terms of the upper column half join those of the lower half
            float* part = reinterpret_cast<float*>(sm + oPart) + i * 8;
            if (lead && hc == 1) {
                part[0] = acc_dbeta;
                part[1] = acc_dgam + dgq;
                part[2] = acc_dd;
                part[3] = rowsum;
                part[4] = dbeta_a;
            }
            epi_sync();
            if (tma_out && tid == 0) {
                const int z = static_cast<int>(row_base + c0);
#pragma unroll
                for (int region = 0; region < 2; ++region) {
                    tma_store_3d(&tmap_dq, region * 64, h, z, smem_u32(sm + oP + region * kTile64));
                    tma_store_3d(&tmap_dk, region * 64, h, z, smem_u32(sm + oRB + region * kTile64));
                }
                bulk_commit();
            }
            if (lead && hc == 0) {
                float dgam = acc_dgam + dgq + part[1];
                float sdd = 0.f;
                if (i == 63) {
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        dgam += red[w];
                        sdd += red[8 + w];
                    }
                }
                dG = (rowsum + part[3]) - colsum[i] - (acc_dd + part[2]) + dgam * gi + sdd;
                dbeta = acc_dbeta + part[0] + dbeta_a + part[4];
            }
        }
        epi_sync();
        if (lead && hc == 0) {
            colsum[mrow] = dG;  // reuse as dG vector
            bv[mrow] = dbeta;   // reuse as dbeta vector
        }
        epi_sync();
        // dg = reverse running sum of dG over the chunk (warp 0)
        if (tid < 32) {
            const int i0 = 63 - 2 * tid, i1 = 62 - 2 * tid;
            const float a = colsum[i0], bb = colsum[i1];
            float s = a + bb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (tid >= off) s += o;
            }
            const float base = s - (a + bb);
            if (i0 < nv) {
                const long long row = (row_base + c0 + i0) * H + h;
                p.dg[row] = base + a;
                p.dbeta[row] = f32_to_bf16(bv[i0]);
            }
            if (i1 < nv) {
                const long long row = (row_base + c0 + i1) * H + h;
                p.dg[row] = s;
                p.dbeta[row] = f32_to_bf16(bv[i1]);
            }
        }
        epi_sync();
        cur = nxt;
        f = fn;
    }
    if (failed) {
        record_error(p.err, kErrTimeout);
    }
    // let every copy this thread issued land before the CTA leaves
    if (i_out) mbar_wait(ibar, iphase, kDefaultWaitLimit);
    if (s0_out) mbar_wait(s0bar, s0phase, kDefaultWaitLimit);
    if (ds_out) mbar_wait(dsbar, dsphase, kDefaultWaitLimit);
    if (tid == 0) bulk_wait_all();  // the dV / dq / dk tile stores
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_bwd_local(const BwdLocalArgs& a, cudaStream_t stream) {
    if (a.max_chunks == 0) return cudaSuccess;
    const long long rows = static_cast<long long>(a.cu_seqlens ? 1 : a.N) * a.T;
    CUtensorMap mk, mq, mdq, mdk;  // used for d_k = 128 only (d_k = 64 tiles use plain loads and stores)
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    memset(&mdq, 0, sizeof(mdq));
    memset(&mdk, 0, sizeof(mdk));
    if (rows > 0 && a.d_k == kDk &&
        (!make_qk_map(&mk, a.k, rows, a.H) || !make_qk_map(&mq, a.q, rows, a.H) ||
         !make_qk_map(&mdq, a.dq, rows, a.H) || !make_qk_map(&mdk, a.dk, rows, a.H)))
        return cudaErrorInvalidValue;
    CUtensorMap mdv;  // dV tile stores (full chunks, any d_k)
    memset(&mdv, 0, sizeof(mdv));
    if (rows > 0 && !make_rows_map(&mdv, a.dv, rows, a.H, a.d_v)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_bwd_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(a.max_chunks) * a.H * a.N;
    const int grid = static_cast<int>(items < sms ? items : sms);
    gdn_bwd_local_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, mq, mdq, mdk, mdv, a);
    return cudaGetLastError();
}

}  // namespace gdn

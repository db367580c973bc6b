// Tensor-core walk of the chunked per-channel-gate (KDA) forward, d_k = 128.
//
// Per chunk of 64 tokens with start state S0 (d_k x 64 value columns of one
// head) the walk evaluates
//   R     = beta o (V - KG S0)          KG = exp(G) o K
//   Delta = T R
//   O     = scale [QG S0 + P Delta]     QG = exp(G) o Q
//   S1    = diag(exp(G_n)) S0 + Kt^T Delta,  Kt = exp(G_n - G) o K
// With a per-channel gate the decay sits inside the key dot products, so it
// cannot move to the epilogues the way a scalar gate does; instead the
// chunk-parallel kernel (gdn_kda_tp_kernel) forms the decayed operands KG,
// QG, Kt with T and P for every chunk as bf16 hi/lo operand tiles, and the walk
// copies each chunk's block in with two bulk copies: KG/QG, refilled for the
// next chunk as soon as K S and Q S have read them, and Kt/T/P/vectors,
// refilled once the chunk's last products have read them.  Every product is a
// tcgen05.mma with fp32 accumulation in tensor memory; operands computed in
// the walk (S, R, Delta) are split into bf16 hi + lo parts like the ones the
// chunk-parallel kernel writes, and each product takes the hi*hi, hi*lo and
// lo*hi terms.  The state S lives in fp32 registers: thread (warp w, lane l)
// holds key row 32 (w % 4) + l, value columns 32 (w / 4) .. + 31.
//
// One CTA (256 threads, 8 warps) per (64 value columns, head, sequence);
// thread 0 issues the MMAs and the bulk copies.  Every wait is bounded; a CTA
// whose wait runs out records GDN_ERR_TIMEOUT, drains its copies and products
// (with their own bound) and frees its tensor memory.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

using namespace sm100;
using namespace tc;

constexpr int kWalkThreads = 256;
constexpr int kWalkK = 128;
constexpr int kWalkVs = 64;
constexpr uint32_t kWalkTmemCols = 256;

// tensor-memory columns
constexpr uint32_t kColKS = 0;    // K S (M = 64)
constexpr uint32_t kColO = 64;    // Q S, then + P Delta (M = 64)
constexpr uint32_t kColD = 128;   // Delta (M = 64)
constexpr uint32_t kColS = 192;   // Kt^T Delta (M = 128)

// shared-memory map (bytes from a 1024-aligned base)
constexpr int oBlk = 0;                         // the chunk's operand block
constexpr int oShi = oBlk + kKdaBlkBytes;       // S hi, lo: 128 key rows x 128 bytes
constexpr int oSlo = oShi + kWalkK * 128;
constexpr int oRhi = oSlo + kWalkK * 128;       // R hi, lo: 64 token rows x 128 bytes
constexpr int oRlo = oRhi + kTile64;
constexpr int oDhi = oRlo + kTile64;            // Delta hi, lo
constexpr int oDlo = oDhi + kTile64;
constexpr int oBar = oDlo + kTile64;
enum { W_FULLA = 0, W_FULLB, W_KS, W_QS, W_D, W_OS, W_DRAIN, kWalkBars };
constexpr int oMisc = oBar + kWalkBars * 8;     // TMEM slot
constexpr int kWalkBytes = oMisc + 16;
constexpr int kWalkAlloc = kWalkBytes + 1024;
static_assert(kKdaBlkBytes % 1024 == 0, "tiles after the block stay 1024-aligned");
static_assert(kWalkAlloc <= 232448, "shared memory");

__global__ void __launch_bounds__(kWalkThreads, 1) gdn_kda_walk_kernel(const KdaWalkArgs p, uint32_t wl) {
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + oMisc);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const long long row_base = static_cast<long long>(b) * p.T;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);
    const bool want_out = p.out != nullptr;
    auto blk = [&](int ci) { return p.tiles + ((slot0 + ci) * H + h) * static_cast<long long>(kKdaBlkBytes); };
    const uint32_t sblk = smem_u32(sm + oBlk);
    // the two refills of the operand block
    auto copy_a = [&](int ci) {
        mbar_arrive_expect_tx(bar(W_FULLA), kKdaBlkSplit);
        bulk_g2s(sblk, blk(ci), kKdaBlkSplit, bar(W_FULLA));
    };
    auto copy_b = [&](int ci) {
        mbar_arrive_expect_tx(bar(W_FULLB), kKdaBlkBytes - kKdaBlkSplit);
        bulk_g2s(sblk + kKdaBlkSplit, blk(ci) + kKdaBlkSplit, kKdaBlkBytes - kKdaBlkSplit, bar(W_FULLB));
    };

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kWalkTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kWalkBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // copies issued (thread 0's count), for the drain
    int issued_a = 0, issued_b = 0;
    if (tid == 0 && nchunks > 0) {
        copy_a(0);
        copy_b(0);
        issued_a = issued_b = 1;
    }

    // thread layouts: state rows (M = 128) and chunk rows (M = 64, a quarter
    // row of 16 columns each)
    const int sw = warp & 3, hs = warp >> 2;
    const int srow = 32 * sw + lane;
    const int hrow = 16 * sw + (lane & 15);
    const int cq = 16 * (2 * hs + (lane >> 4));
    const uint32_t lb = static_cast<uint32_t>(sw * 32) << 16;
    auto ld_q16 = [&](uint32_t col, float* v) { tmem_ld_pair16(tmem + lb + col + 32 * hs, v); };
    auto store_q16 = [&](uint8_t* thi, uint8_t* tlo, const float* x) {
        store_split_chunk(thi, tlo, hrow, cq >> 3, x);
        store_split_chunk(thi, tlo, hrow, (cq >> 3) + 1, x + 8);
    };
    auto ld_s32 = [&](uint32_t col, float* v) {
        tmem_ld16(tmem + lb + col + 32 * hs, v);
        tmem_ld16(tmem + lb + col + 32 * hs + 16, v + 16);
        tmem_ld_wait();
    };
    uint8_t* Shi = sm + oShi;
    uint8_t* Slo = sm + oSlo;
    uint8_t* Rhi = sm + oRhi;
    uint8_t* Rlo = sm + oRlo;
    uint8_t* Dhi = sm + oDhi;
    uint8_t* Dlo = sm + oDlo;
    const float* vec = reinterpret_cast<const float*>(sm + oBlk + kKdaBlkVec);

    const long long KV = static_cast<long long>(kWalkK) * V;
    const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kWalkVs;
    float S[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = 0.f;
    if (p.initial_state) {
        const float* src = p.initial_state + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(src + j);
            S[j] = t4.x; S[j + 1] = t4.y; S[j + 2] = t4.z; S[j + 3] = t4.w;
        }
    }
    store_split_half(Shi, Slo, srow, hs, S);
    fence_proxy_async_smem();

    // a quarter value row (row hrow, columns cq .. cq + 15 of the slice), bf16
    uint4 vraw[2];
    auto load_v = [&](int cj) {
        vraw[0] = vraw[1] = make_uint4(0, 0, 0, 0);
        const int cc0 = t0 + cj * kChunk;
        if (cj < nchunks && hrow < min(kChunk, t1 - cc0)) {
            const uint4* src = reinterpret_cast<const uint4*>(p.v + ((row_base + cc0 + hrow) * H + h) *
                                                                        static_cast<long long>(V) +
                                                              vs * kWalkVs + cq);
            vraw[0] = src[0];
            vraw[1] = src[1];
        }
    };
    load_v(0);
    tc_fence_before();
    __syncthreads();

    const float scale = p.scale;
    bool ok = true;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int c0 = t0 + ci * kChunk;
        const int nv = min(kChunk, t1 - c0);
        const uint32_t ph = ci & 1;
        if (p.chunk_states) {
            float* dst = p.chunk_states + ((slot0 + ci) * H + h) * KV + static_cast<long long>(srow) * V +
                         vs * kWalkVs + 32 * hs;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
        // ---- K S and Q S, once KG / QG are in ----
        if (warp == 0) {
            const bool full = __all_sync(0xffffffffu, mbar_wait(bar(W_FULLA), ph, wl));
            if (full) {
                if (lane == 0) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                    for (int s = 0; s < kWalkK / 16; ++s) {
                        const uint32_t koff = (s >> 2) * 8192 + (s & 3) * 32;
                        const uint64_t ah = desc_sw128(sblk + kKdaBlkKG + koff, 0, 1024);
                        const uint64_t al = desc_sw128(sblk + kKdaBlkKG + 16384 + koff, 0, 1024);
                        const uint64_t bh = desc_sw128(smem_u32(Shi) + s * 2048, kWalkK * 128, 1024);
                        const uint64_t bl = desc_sw128(smem_u32(Slo) + s * 2048, kWalkK * 128, 1024);
                        mma_bf16(tmem + kColKS, ah, bh, id, s > 0);
                        mma_bf16(tmem + kColKS, ah, bl, id, 1);
                        mma_bf16(tmem + kColKS, al, bh, id, 1);
                    }
                    mma_commit(bar(W_KS));
                    if (want_out) {
#pragma unroll
                        for (int s = 0; s < kWalkK / 16; ++s) {
                            const uint32_t koff = (s >> 2) * 8192 + (s & 3) * 32;
                            const uint64_t ah = desc_sw128(sblk + kKdaBlkQG + koff, 0, 1024);
                            const uint64_t al = desc_sw128(sblk + kKdaBlkQG + 16384 + koff, 0, 1024);
                            const uint64_t bh = desc_sw128(smem_u32(Shi) + s * 2048, kWalkK * 128, 1024);
                            const uint64_t bl = desc_sw128(smem_u32(Slo) + s * 2048, kWalkK * 128, 1024);
                            mma_bf16(tmem + kColO, ah, bh, id, s > 0);
                            mma_bf16(tmem + kColO, ah, bl, id, 1);
                            mma_bf16(tmem + kColO, al, bh, id, 1);
                        }
                    }
                    // Q S (or nothing more) done: KG / QG and the S tiles are free
                    mma_commit(bar(W_QS));
                }
                __syncwarp();
            } else {
                ok = false;
            }
        }
        // ---- R = beta o (V - K S) ----
        bool w_ok = mbar_wait(bar(W_KS), ph, wl) && mbar_wait(bar(W_FULLB), ph, wl);
        tc_fence_after();
        float gnr = 0.f;
        if (w_ok) {
            float row[16];
            ld_q16(kColKS, row);
            tmem_ld_wait();
            const float bj = vec[kWalkK + hrow];
            gnr = vec[srow];
            float vv[16];
            unpack8(vraw[0], vv);
            unpack8(vraw[1], vv + 8);
#pragma unroll
            for (int c = 0; c < 16; ++c) row[c] = bj * (vv[c] - row[c]);
            store_q16(Rhi, Rlo, row);
        }
        load_v(ci + 1);
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // ---- Delta = T R ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkT + s * 32, 0, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkT + 8192 + s * 32, 0, 1024);
                    const uint64_t bh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColD, ah, bh, id, s > 0);
                    mma_bf16(tmem + kColD, ah, bl, id, 1);
                    mma_bf16(tmem + kColD, al, bh, id, 1);
                }
                mma_commit(bar(W_D));
            }
            __syncwarp();
        }
        // KG / QG read by K S and Q S: the next chunk's come in now (after
        // the Delta products went out, so the wait costs the walk nothing)
        if (tid == 0 && ci + 1 < nchunks) {
            if (mbar_wait(bar(W_QS), ph, wl)) {
                copy_a(ci + 1);
                issued_a = ci + 2;
            } else {
                ok = false;
            }
        }
        w_ok = mbar_wait(bar(W_D), ph, wl);
        tc_fence_after();
        if (w_ok) {
            float row[16];
            ld_q16(kColD, row);
            tmem_ld_wait();
            store_q16(Dhi, Dlo, row);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // ---- S update Kt^T Delta, then O += P Delta ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id_s = idesc(kFmtBf16, 1, 1, kWalkK, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkKt + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkKt + 16384 + s * 2048, 8192, 1024);
                    const uint64_t bh = desc_sw128(smem_u32(Dhi) + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(smem_u32(Dlo) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColS, ah, bh, id_s, s > 0);
                    mma_bf16(tmem + kColS, ah, bl, id_s, 1);
                    mma_bf16(tmem + kColS, al, bh, id_s, 1);
                }
                if (want_out) {
                    constexpr uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint64_t ah = desc_sw128(sblk + kKdaBlkP + s * 32, 0, 1024);
                        const uint64_t al = desc_sw128(sblk + kKdaBlkP + 8192 + s * 32, 0, 1024);
                        const uint64_t bh = desc_sw128(smem_u32(Dhi) + s * 2048, kTile64, 1024);
                        const uint64_t bl = desc_sw128(smem_u32(Dlo) + s * 2048, kTile64, 1024);
                        mma_bf16(tmem + kColO, ah, bh, id, 1);
                        mma_bf16(tmem + kColO, ah, bl, id, 1);
                        mma_bf16(tmem + kColO, al, bh, id, 1);
                    }
                }
                mma_commit(bar(W_OS));
            }
            __syncwarp();
        }
        w_ok = mbar_wait(bar(W_OS), ph, wl);
        tc_fence_after();
        // Kt, T, P and the vectors have been read: the next chunk's come in
        if (tid == 0 && w_ok && ci + 1 < nchunks) {
            copy_b(ci + 1);
            issued_b = ci + 2;
        }
        if (w_ok) {
            if (want_out) {
                float row[16];
                ld_q16(kColO, row);
                tmem_ld_wait();
                if (hrow < nv) {
                    uint4 o[2];
                    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
                    for (int m = 0; m < 8; ++m) ow[m] = cvt_bf16x2(scale * row[2 * m], scale * row[2 * m + 1]);
                    uint4* dst = reinterpret_cast<uint4*>(p.out + ((row_base + c0 + hrow) * H + h) *
                                                                      static_cast<long long>(V) +
                                                          vs * kWalkVs + cq);
                    dst[0] = o[0];
                    dst[1] = o[1];
                }
            }
            float row[32];
            ld_s32(kColS, row);
#pragma unroll
            for (int c = 0; c < 32; ++c) S[c] = fmaf(gnr, S[c], row[c]);
            store_split_half(Shi, Slo, srow, hs, S);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
    }

    if (ok && p.final_state) {
        float* dst = p.final_state + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    // drain: copies issued and not yet waited for, and every product issued
    if (tid == 0) {
        if (!ok) record_error(p.err, kErrTimeout);
        // the last copy of each kind has phase (issued - 1) & 1; waiting on it
        // also covers the earlier ones (each was waited for before the next
        // was issued, except after an abort)
        if (issued_a > 0) mbar_wait(bar(W_FULLA), (issued_a - 1) & 1, kDefaultWaitLimit);
        if (issued_b > 0) mbar_wait(bar(W_FULLB), (issued_b - 1) & 1, kDefaultWaitLimit);
    }
    if (warp == 0) {
        if (lane == 0) mma_commit(bar(W_DRAIN));
        __syncwarp();
        mbar_wait(bar(W_DRAIN), 0, kDefaultWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kWalkTmemCols);
}

// ---------------------------------------------------------------------------
// The reverse walk of the backward (state gradients), d_k = 128.  Per chunk,
// from the last, with dS the gradient w.r.t. the chunk's end state:
//   dDelta = scale P^T dO + Kt dS          dR = T^T dDelta
//   dS0    = scale QG^T dO + diag(exp(G_n)) dS - KG^T (beta o dR)
// over the same operand blocks as the forward walk (P^T, T^T, QG^T and KG^T
// are the block's tiles read in the other major order).  dO is exact in bf16;
// dS, dDelta and beta o dR are split into hi + lo parts.  dS lives in fp32
// registers like the forward walk's S.  Per chunk it records dS for the
// chunk-parallel gradient pass; the refills of the operand block follow the
// order the products read it: Kt, T, P and the vectors once T^T dDelta is
// done, KG and QG once the dS0 products are.
// ---------------------------------------------------------------------------

constexpr uint32_t kChainTmemCols = 512;
constexpr uint32_t kColPO = 0;     // P^T dO (M = 64)
constexpr uint32_t kColKD = 64;    // Kt dS (M = 64)
constexpr uint32_t kColR = 128;    // T^T dDelta (M = 64)
constexpr uint32_t kColQO = 192;   // QG^T dO (M = 128)
constexpr uint32_t kColKR = 256;   // KG^T (beta o dR) (M = 128)

constexpr int cBlk = 0;
constexpr int cShi = cBlk + kKdaBlkBytes;     // dS hi, lo
constexpr int cSlo = cShi + kWalkK * 128;
constexpr int cO = cSlo + kWalkK * 128;       // dO (bf16, exact)
constexpr int cEhi = cO + kTile64;            // dDelta hi, lo
constexpr int cElo = cEhi + kTile64;
constexpr int cRhi = cElo + kTile64;          // beta o dR hi, lo
constexpr int cRlo = cRhi + kTile64;
constexpr int cBar = cRlo + kTile64;
enum { C_FULLA = 0, C_FULLB, C_KD, C_PO, C_QO, C_R, C_KR, C_DRAIN, kChainBars };
constexpr int cMisc = cBar + kChainBars * 8;
constexpr int kChainAlloc = cMisc + 16 + 1024;
static_assert(kChainAlloc <= 232448, "shared memory");

__global__ void __launch_bounds__(kWalkThreads, 1) gdn_kda_bwd_chain_tc_kernel(const KdaBwdArgs p, uint32_t wl) {
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + cBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + cMisc);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const long long row_base = static_cast<long long>(b) * p.T;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);
    auto blk = [&](int ci) { return p.tiles + ((slot0 + ci) * H + h) * static_cast<long long>(kKdaBlkBytes); };
    const uint32_t sblk = smem_u32(sm + cBlk);
    auto copy_a = [&](int ci) {
        mbar_arrive_expect_tx(bar(C_FULLA), kKdaBlkSplit);
        bulk_g2s(sblk, blk(ci), kKdaBlkSplit, bar(C_FULLA));
    };
    auto copy_b = [&](int ci) {
        mbar_arrive_expect_tx(bar(C_FULLB), kKdaBlkBytes - kKdaBlkSplit);
        bulk_g2s(sblk + kKdaBlkSplit, blk(ci) + kKdaBlkSplit, kKdaBlkBytes - kKdaBlkSplit, bar(C_FULLB));
    };

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kChainTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kChainBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    int issued_a = 0, issued_b = 0;
    if (tid == 0 && nchunks > 0) {
        copy_a(nchunks - 1);
        copy_b(nchunks - 1);
        issued_a = issued_b = 1;
    }

    const int sw = warp & 3, hs = warp >> 2;
    const int srow = 32 * sw + lane;
    const int hrow = 16 * sw + (lane & 15);
    const int cq = 16 * (2 * hs + (lane >> 4));
    const uint32_t lb = static_cast<uint32_t>(sw * 32) << 16;
    auto ld_q16 = [&](uint32_t col, float* v) { tmem_ld_pair16(tmem + lb + col + 32 * hs, v); };
    auto store_q16 = [&](uint8_t* thi, uint8_t* tlo, const float* x) {
        store_split_chunk(thi, tlo, hrow, cq >> 3, x);
        store_split_chunk(thi, tlo, hrow, (cq >> 3) + 1, x + 8);
    };
    auto ld_s32 = [&](uint32_t col, float* v) {
        tmem_ld16(tmem + lb + col + 32 * hs, v);
        tmem_ld16(tmem + lb + col + 32 * hs + 16, v + 16);
        tmem_ld_wait();
    };
    uint8_t* Shi = sm + cShi;
    uint8_t* Slo = sm + cSlo;
    uint8_t* Ot = sm + cO;
    uint8_t* Ehi = sm + cEhi;
    uint8_t* Elo = sm + cElo;
    uint8_t* Rhi = sm + cRhi;
    uint8_t* Rlo = sm + cRlo;
    const float* vec = reinterpret_cast<const float*>(sm + cBlk + kKdaBlkVec);

    const long long KV = static_cast<long long>(kWalkK) * V;
    const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kWalkVs;
    float dS[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) dS[j] = 0.f;
    if (p.d_final_state) {
        const float* src = p.d_final_state + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(src + j);
            dS[j] = t4.x; dS[j + 1] = t4.y; dS[j + 2] = t4.z; dS[j + 3] = t4.w;
        }
    }
    store_split_half(Shi, Slo, srow, hs, dS);

    // dO of a chunk: two 16-byte pieces a thread (rows t / 8 and t / 8 + 32,
    // the (t % 8)-th 8 columns of the slice), held in registers until stored
    uint4 oraw[2];
    auto load_o = [&](int cj) {
        oraw[0] = oraw[1] = make_uint4(0, 0, 0, 0);
        if (cj < 0) return;
        const int cc0 = t0 + cj * kChunk;
        const int nvj = min(kChunk, t1 - cc0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = (tid >> 3) + 32 * u;
            if (r < nvj)
                oraw[u] = *reinterpret_cast<const uint4*>(p.d_out + ((row_base + cc0 + r) * H + h) *
                                                                        static_cast<long long>(V) +
                                                          vs * kWalkVs + 8 * (tid & 7));
        }
    };
    load_o(nchunks - 1);

    const float scale = p.scale;
    bool ok = true;
    for (int it = 0; it < nchunks; ++it) {
        const int ci = nchunks - 1 - it;
        const uint32_t ph = it & 1;
        {
            // the gradient w.r.t. this chunk's end state
            float* dst = p.chunk_dstates + ((slot0 + ci) * H + h) * KV + static_cast<long long>(srow) * V +
                         vs * kWalkVs + 32 * hs;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
            *reinterpret_cast<uint4*>(Ot + sw128_offset((tid >> 3) + 32 * u, 16 * (tid & 7))) = oraw[u];
        load_o(ci - 1);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- Kt dS (critical), P^T dO, then QG^T dO once KG / QG are in ----
        if (warp == 0) {
            const bool fb = __all_sync(0xffffffffu, mbar_wait(bar(C_FULLB), ph, wl));
            if (fb && lane == 0) {
                tc_fence_after();
                constexpr uint32_t id_k = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < kWalkK / 16; ++s) {
                    const uint32_t koff = (s >> 2) * 8192 + (s & 3) * 32;
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkKt + koff, 0, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkKt + 16384 + koff, 0, 1024);
                    const uint64_t bh = desc_sw128(smem_u32(Shi) + s * 2048, kWalkK * 128, 1024);
                    const uint64_t bl = desc_sw128(smem_u32(Slo) + s * 2048, kWalkK * 128, 1024);
                    mma_bf16(tmem + kColKD, ah, bh, id_k, s > 0);
                    mma_bf16(tmem + kColKD, ah, bl, id_k, 1);
                    mma_bf16(tmem + kColKD, al, bh, id_k, 1);
                }
                mma_commit(bar(C_KD));
                constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkP + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkP + 8192 + s * 2048, 8192, 1024);
                    const uint64_t bo = desc_sw128(smem_u32(Ot) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColPO, ah, bo, id_t, s > 0);
                    mma_bf16(tmem + kColPO, al, bo, id_t, 1);
                }
                mma_commit(bar(C_PO));
            }
            __syncwarp();
            const bool fa = fb && __all_sync(0xffffffffu, mbar_wait(bar(C_FULLA), ph, wl));
            if (fa && lane == 0) {
                tc_fence_after();
                constexpr uint32_t id_q = idesc(kFmtBf16, 1, 1, kWalkK, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkQG + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkQG + 16384 + s * 2048, 8192, 1024);
                    const uint64_t bo = desc_sw128(smem_u32(Ot) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColQO, ah, bo, id_q, s > 0);
                    mma_bf16(tmem + kColQO, al, bo, id_q, 1);
                }
                mma_commit(bar(C_QO));
            }
            __syncwarp();
            if (!fa) ok = false;
        }
        // ---- dDelta = scale P^T dO + Kt dS ----
        bool w_ok = mbar_wait(bar(C_KD), ph, wl) && mbar_wait(bar(C_PO), ph, wl) && mbar_wait(bar(C_FULLB), ph, wl);
        tc_fence_after();
        float be = 0.f, gnr = 0.f;
        if (w_ok) {
            float a[16], k[16];
            ld_q16(kColPO, a);
            ld_q16(kColKD, k);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) a[c] = fmaf(scale, a[c], k[c]);
            store_q16(Ehi, Elo, a);
            be = vec[kWalkK + hrow];
            gnr = vec[srow];
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // ---- dR = T^T dDelta ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkT + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkT + 8192 + s * 2048, 8192, 1024);
                    const uint64_t bh = desc_sw128(smem_u32(Ehi) + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(smem_u32(Elo) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColR, ah, bh, id_t, s > 0);
                    mma_bf16(tmem + kColR, ah, bl, id_t, 1);
                    mma_bf16(tmem + kColR, al, bh, id_t, 1);
                }
                mma_commit(bar(C_R));
            }
            __syncwarp();
        }
        w_ok = mbar_wait(bar(C_R), ph, wl);
        tc_fence_after();
        if (w_ok) {
            float r[16];
            ld_q16(kColR, r);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) r[c] *= be;
            store_q16(Rhi, Rlo, r);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // Kt, T, P read by finished products, the vectors by every thread:
        // the previous chunk's come in now
        if (tid == 0 && ci > 0) {
            copy_b(ci - 1);
            issued_b = it + 2;
        }
        // ---- KG^T (beta o dR) ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id_q = idesc(kFmtBf16, 1, 1, kWalkK, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sblk + kKdaBlkKG + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sblk + kKdaBlkKG + 16384 + s * 2048, 8192, 1024);
                    const uint64_t bh = desc_sw128(smem_u32(Rhi) + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(smem_u32(Rlo) + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + kColKR, ah, bh, id_q, s > 0);
                    mma_bf16(tmem + kColKR, ah, bl, id_q, 1);
                    mma_bf16(tmem + kColKR, al, bh, id_q, 1);
                }
                mma_commit(bar(C_KR));
            }
            __syncwarp();
        }
        // ---- dS0 = scale QG^T dO + diag(exp(G_n)) dS - KG^T (beta o dR) ----
        w_ok = mbar_wait(bar(C_KR), ph, wl) && mbar_wait(bar(C_QO), ph, wl);
        tc_fence_after();
        if (w_ok) {
            float qo[32], kr[32];
            ld_s32(kColQO, qo);
            ld_s32(kColKR, kr);
#pragma unroll
            for (int c = 0; c < 32; ++c) dS[c] = fmaf(scale, qo[c], fmaf(gnr, dS[c], -kr[c]));
            store_split_half(Shi, Slo, srow, hs, dS);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // KG / QG and dO read by finished products: the previous chunk's KG / QG come in
        if (tid == 0 && ci > 0) {
            copy_a(ci - 1);
            issued_a = it + 2;
        }
    }

    if (ok && p.d_initial_state) {
        float* dst = p.d_initial_state + state_off + static_cast<long long>(srow) * V + 32 * hs;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) = make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
    }
    if (tid == 0) {
        if (!ok) record_error(p.err, kErrTimeout);
        if (issued_a > 0) mbar_wait(bar(C_FULLA), (issued_a - 1) & 1, kDefaultWaitLimit);
        if (issued_b > 0) mbar_wait(bar(C_FULLB), (issued_b - 1) & 1, kDefaultWaitLimit);
    }
    if (warp == 0) {
        if (lane == 0) mma_commit(bar(C_DRAIN));
        __syncwarp();
        mbar_wait(bar(C_DRAIN), 0, kDefaultWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kChainTmemCols);
}

}  // namespace

cudaError_t launch_kda_bwd_chain_tc(const KdaBwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_bwd_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kChainAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kWalkVs, a.H, a.N);
    gdn_kda_bwd_chain_tc_kernel<<<grid, kWalkThreads, kChainAlloc, stream>>>(a, wait_limit);
    return cudaGetLastError();
}

cudaError_t launch_kda_walk(const KdaWalkArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kWalkAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kWalkVs, a.H, a.N);
    gdn_kda_walk_kernel<<<grid, kWalkThreads, kWalkAlloc, stream>>>(a, wait_limit);
    return cudaGetLastError();
}

}  // namespace gdn

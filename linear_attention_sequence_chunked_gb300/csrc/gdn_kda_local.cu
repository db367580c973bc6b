// Local gradients of the per-channel-gate (KDA) backward on the tensor cores,
// d_k = 128: one CTA per (chunk, head, sequence).
//
// Given the chunk's start state S0 (forward walk), the gradient dS w.r.t. its
// end state (reverse walk) and its operand block (gdn_kda_tp_kernel: KG, Kt,
// T, P as bf16 hi/lo tiles), every value slice of 64 columns runs
//   K S0, P^T dO, Kt dS      -> R = beta o (V - K S0),  dDelta = scale P^T dO + Kt dS
//   Delta = T R,  dR = T^T dDelta                         dv = beta o dR
// and adds its share of the sums over value columns into tensor memory:
//   [dR; dO] Delta^T  (M = 128: -dA above, dP / scale below)
//   [dR; dO] S0^T     (M = 128: dR S0^T above, dO S0^T below)
//   Delta dS^T        (M = 64)
// (the rows of dR and dO are stacked in one operand tile, so each sum over
// the slices is a single product).  dO is exact in bf16; every computed
// operand is split into bf16 hi + lo parts, every accumulation is fp32.
// After the last slice the sums leave tensor memory into fp32 tiles of
// shared memory, and the CUDA cores finish as in the fp32 kernel: the
// per-channel decay factors of dq, dk and dG, the decayed pair sums (one
// exponential per pair and channel on each side), dbeta, and dg as the
// reverse running sum of dG.
//
// Every wait is bounded; a CTA whose wait runs out records GDN_ERR_TIMEOUT,
// drains its copies and products (default bound) and frees its tensor memory.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_kda_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

using namespace sm100;
using namespace tc;

constexpr int kLThreads = 256;
constexpr int kLK = 128;
constexpr int kLVs = 64;
constexpr uint32_t kLTmemCols = 512;

// tensor-memory columns
constexpr uint32_t tAcc1 = 0;     // [dR; dO] Delta^T, M = 128, N = 64
constexpr uint32_t tAcc2 = 64;    // [dR; dO] S0^T, M = 128, N = 128
constexpr uint32_t tAcc3 = 192;   // Delta dS^T, M = 64, N = 128
constexpr uint32_t tT0 = 320;     // K S0, then Delta (M = 64)
constexpr uint32_t tT1 = 384;     // P^T dO, then dR (M = 64)
constexpr uint32_t tT2 = 448;     // Kt dS (M = 64)

// shared memory, value-slice phase (bytes from a 1024-aligned base)
constexpr int sKG = 0;            // KG hi, lo (2 x 16 KB), from the operand block
constexpr int sKt = 32768;        // Kt hi, lo; T hi, lo; P hi, lo: one copy of the block's [Kt, T, P]
constexpr int sT = sKt + 32768;
constexpr int sP = sT + 16384;
constexpr int sS0 = sP + 16384;   // S0 hi, lo: 128 key rows x 128 bytes each
constexpr int sdS = sS0 + 32768;  // dS hi, lo
constexpr int sA = sdS + 32768;   // stacked hi: rows 0-63 R, then dR; rows 64-127 dO
constexpr int sAl = sA + 16384;   // stacked lo: rows 0-63 R / dR lo; rows 64-127 zero
constexpr int sD = sAl + 16384;   // Delta hi, lo
constexpr int sE = sD + 16384;    // dDelta hi, lo
constexpr int sBar = sE + 16384;
enum { L_BLK = 0, L_KS, L_D1, L_DL, L_R, L_ACC, L_DRAIN, kLBars };
constexpr int sMisc = sBar + kLBars * 8;
constexpr int kLBytes = sMisc + 16;
constexpr int kLAlloc = kLBytes + 1024;
static_assert(sKt - sKG == kKdaBlkQG - kKdaBlkKG && sP + 16384 - sKt == kKdaBlkVec - kKdaBlkKt,
              "the block's KG and [Kt, T, P] come in as two copies");
static_assert(kLAlloc <= 232448, "shared memory");

// end phase (the same space, reused once every product has completed)
constexpr int LDB = kLK + 8;      // bf16 rows of k and q
constexpr int LDF = kLK + 4;      // fp32 rows of d_k values
constexpr int LDP = 64 + 4;       // fp32 rows of pair values
constexpr int eK = 0;
constexpr int eQ = eK + 64 * LDB * 2;
constexpr int eG = eQ + 64 * LDB * 2;
constexpr int edA = eG + 64 * LDF * 4;
constexpr int edP = edA + 64 * LDP * 4;
constexpr int edQ = edP + 64 * LDP * 4;
constexpr int edK = edQ + 64 * LDF * 4;
constexpr int edG = edK + 64 * LDF * 4;
constexpr int eVec = edG + 64 * LDF * 4;  // beta, G_n, exp(G_n), gsum, dbeta parts [4][64], X column parts [4][128], [4][64]
constexpr int kEVecFloats = 64 + 3 * kLK + 4 * 64 + 4 * kLK + 4 * 64 + 16 * kLK;
static_assert(eVec + kEVecFloats * 4 <= sBar, "end-phase tiles fit below the barriers");

__device__ __forceinline__ float bf(const uint16_t* p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }

// Eight rows of one 16 x 16 tile of pairs (rows i = 16 I + 8 half + r of
// sub-block I, the 16 columns j of sub-block J <= I) of the decayed pair sums
// for key channel c, each pair's factor E = exp(G_ic - G_jc) formed once (a
// masked difference, <= 0):
//   u1_i = sum_j dA_ij k_jc E   (j < i),      u2_i = sum_j dP_ij k_jc E   (j <= i),
//   w_j += (beta_i dA_ij k_ic + dP_ij q_ic) E   (i > j for dA, i >= j for dP).
// Each row's u1, u2 go straight into dq, dk, dG of row i (this thread owns
// channel c of these rows), with sum_c k_ic u1_ic (dbeta) summed over the warp's
// channels into dbc; the row loop is kept rolled so the code stays small.
// dA and dP hold every entry of the tile; on the diagonal tile the pairs above
// the diagonal are skipped and dA's diagonal counts as 0.
__device__ __forceinline__ void pair_rows(int I, int J, int half, int c, int lane, int wq, const float* Gs,
                                          const uint16_t* Ks, const uint16_t* Qs, const float* dA, const float* dP,
                                          const float* bs, float* dQ, float* dK, float* dG, float* dbc,
                                          float (&w)[16]) {
    const bool diag = I == J;
    float gj[16], kj[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
        const int j = 16 * J + jj;
        gj[jj] = Gs[j * LDF + c];
        kj[jj] = bf(Ks + j * LDB + c);
    }
#pragma unroll 1
    for (int r = 0; r < 8; ++r) {
        const int ii = 8 * half + r;
        const int i = 16 * I + ii;
        const float gi = Gs[i * LDF + c];
        const float ki = bf(Ks + i * LDB + c);
        const float qi = bf(Qs + i * LDB + c);
        const float be = bs[i];
        const float bki = be * ki;
        float u1 = 0.f, u2 = 0.f, u1b = 0.f, u2b = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
            const float4 av = *reinterpret_cast<const float4*>(dA + i * LDP + 16 * J + 4 * j4);
            const float4 qv = *reinterpret_cast<const float4*>(dP + i * LDP + 16 * J + 4 * j4);
            const float a4[4] = {av.x, av.y, av.z, av.w};
            const float q4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int jj = 4 * j4 + m;
                const bool on = !diag || jj <= ii;
                const float e = on ? __expf(gi - gj[jj]) : 0.f;
                const float ad = (diag && jj == ii) ? 0.f : a4[m];
                const float ke = kj[jj] * e;
                // two accumulators a row keep the dependent FMA chains short
                if (m & 1) {
                    u1b = fmaf(ad, ke, u1b);
                    u2b = fmaf(q4[m], ke, u2b);
                } else {
                    u1 = fmaf(ad, ke, u1);
                    u2 = fmaf(q4[m], ke, u2);
                }
                w[jj] = fmaf(fmaf(ad, bki, q4[m] * qi), e, w[jj]);
            }
        }
        u1 += u1b;
        u2 += u2b;
        dQ[i * LDF + c] += u2;
        dK[i * LDF + c] = fmaf(be, u1, dK[i * LDF + c]);
        dG[i * LDF + c] = fmaf(bki, u1, fmaf(qi, u2, dG[i * LDF + c]));
        float part = ki * u1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) dbc[wq * 64 + i] += part;
    }
}

__global__ void __launch_bounds__(kLThreads, 1) gdn_kda_local_tc_kernel(const KdaBwdArgs p, uint32_t wl) {
    const int ci = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int H = p.H, V = p.d_v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    const int c0 = t0 + ci * kChunk;
    if (c0 >= t1) return;
    const int nv = min(kChunk, t1 - c0);
    const long long slot = (chunk_slot_base(p.cu_seqlens, n, p.T) + ci) * H + h;
    const long long row0 = static_cast<long long>(b) * p.T + c0;
    const float scale = p.scale;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + sBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + sMisc);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const uint32_t sb = smem_u32(sm);
    const uint8_t* blk = p.tiles + slot * static_cast<long long>(kKdaBlkBytes);
    const float* gvec = reinterpret_cast<const float*>(blk + kKdaBlkVec);  // exp(G_n), beta

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kLTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kLBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
    }
    // rows 64-127 of the stacked lo tile stay zero (dO is exact in bf16)
    for (int i = tid; i < 8192 / 16; i += kLThreads)
        reinterpret_cast<uint4*>(sm + sAl + 8192)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {
        mbar_arrive_expect_tx(bar(L_BLK), 32768 + 65536);
        bulk_g2s(sb + sKG, blk + kKdaBlkKG, 32768, bar(L_BLK));
        bulk_g2s(sb + sKt, blk + kKdaBlkKt, 65536, bar(L_BLK));
    }

    // thread layouts: chunk rows (M = 64, a quarter row of 16 columns) and
    // M = 128 rows (lane = row within the warp's subpartition)
    const int sw = warp & 3, hs = warp >> 2;
    const int hrow = 16 * sw + (lane & 15);
    const int cq = 16 * (2 * hs + (lane >> 4));
    const int mrow = 32 * sw + lane;
    const uint32_t lb = static_cast<uint32_t>(sw * 32) << 16;
    auto ld_q16 = [&](uint32_t col, float* v) { tmem_ld_pair16(tmem + lb + col + 32 * hs, v); };
    auto store_q16 = [&](uint8_t* thi, uint8_t* tlo, const float* x) {
        store_split_chunk(thi, tlo, hrow, cq >> 3, x);
        store_split_chunk(thi, tlo, hrow, (cq >> 3) + 1, x + 8);
    };
    const float bj = gvec[kLK + hrow];  // beta of this thread's chunk row

    const float* st0 = p.chunk_states + slot * kLK * V;
    const float* dst1 = p.chunk_dstates + slot * kLK * V;
    float gs = 0.f;    // sum over value columns of dS o S0 for key row tid / 2 (half the columns)
    float dbp = 0.f;   // this quarter row's sum of dR o U over the slices
    bool ok = true;
    const int nsl = V / kLVs;
    for (int sl = 0; sl < nsl; ++sl) {
        const int col0 = sl * kLVs;
        // ---- the slice's operands: S0, dS (split), dO (exact), a quarter row of V
        {
            const int c = tid >> 1, hf = tid & 1;
            float x[32], y[32];
            const float* s0r = st0 + static_cast<long long>(c) * V + col0 + 32 * hf;
            const float* dsr = dst1 + static_cast<long long>(c) * V + col0 + 32 * hf;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 a = *reinterpret_cast<const float4*>(s0r + j);
                const float4 d = *reinterpret_cast<const float4*>(dsr + j);
                x[j] = a.x; x[j + 1] = a.y; x[j + 2] = a.z; x[j + 3] = a.w;
                y[j] = d.x; y[j + 1] = d.y; y[j + 2] = d.z; y[j + 3] = d.w;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) gs = fmaf(x[j], y[j], gs);
            store_split_half(sm + sS0, sm + sS0 + 16384, c, hf, x);
            store_split_half(sm + sdS, sm + sdS + 16384, c, hf, y);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = (tid >> 3) + 32 * u;
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (r < nv)
                o = *reinterpret_cast<const uint4*>(p.d_out + ((row0 + r) * H + h) * static_cast<long long>(V) +
                                                    col0 + 8 * (tid & 7));
            *reinterpret_cast<uint4*>(sm + sA + 8192 + sw128_offset(r, 16 * (tid & 7))) = o;
        }
        float vv[16];
        {
            uint4 raw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (hrow < nv) {
                const uint4* src = reinterpret_cast<const uint4*>(p.v + ((row0 + hrow) * H + h) *
                                                                            static_cast<long long>(V) +
                                                                  col0 + cq);
                raw[0] = src[0];
                raw[1] = src[1];
            }
            unpack8(raw[0], vv);
            unpack8(raw[1], vv + 8);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- K S0, then P^T dO and Kt dS ----
        if (warp == 0) {
            const bool in = sl > 0 || __all_sync(0xffffffffu, mbar_wait(bar(L_BLK), 0, wl));
            if (in && lane == 0) {
                tc_fence_after();
                constexpr uint32_t id_k = idesc(kFmtBf16, 0, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < kLK / 16; ++s) {
                    const uint32_t koff = (s >> 2) * 8192 + (s & 3) * 32;
                    const uint64_t ah = desc_sw128(sb + sKG + koff, 0, 1024);
                    const uint64_t al = desc_sw128(sb + sKG + 16384 + koff, 0, 1024);
                    const uint64_t bh = desc_sw128(sb + sS0 + s * 2048, 16384, 1024);
                    const uint64_t bl = desc_sw128(sb + sS0 + 16384 + s * 2048, 16384, 1024);
                    mma_bf16(tmem + tT0, ah, bh, id_k, s > 0);
                    mma_bf16(tmem + tT0, ah, bl, id_k, 1);
                    mma_bf16(tmem + tT0, al, bh, id_k, 1);
                }
                mma_commit(bar(L_KS));
                constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sb + sP + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sb + sP + 8192 + s * 2048, 8192, 1024);
                    const uint64_t bo = desc_sw128(sb + sA + 8192 + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + tT1, ah, bo, id_t, s > 0);
                    mma_bf16(tmem + tT1, al, bo, id_t, 1);
                }
#pragma unroll
                for (int s = 0; s < kLK / 16; ++s) {
                    const uint32_t koff = (s >> 2) * 8192 + (s & 3) * 32;
                    const uint64_t ah = desc_sw128(sb + sKt + koff, 0, 1024);
                    const uint64_t al = desc_sw128(sb + sKt + 16384 + koff, 0, 1024);
                    const uint64_t bh = desc_sw128(sb + sdS + s * 2048, 16384, 1024);
                    const uint64_t bl = desc_sw128(sb + sdS + 16384 + s * 2048, 16384, 1024);
                    mma_bf16(tmem + tT2, ah, bh, id_k, s > 0);
                    mma_bf16(tmem + tT2, ah, bl, id_k, 1);
                    mma_bf16(tmem + tT2, al, bh, id_k, 1);
                }
                mma_commit(bar(L_D1));
            }
            __syncwarp();
            if (!in) ok = false;
        }
        const uint32_t ph = sl & 1;
        // ---- R = beta o (V - K S0) into the upper rows of the stacked tiles ----
        bool w_ok = mbar_wait(bar(L_KS), ph, wl);
        tc_fence_after();
        float U[16];
        if (w_ok) {
            ld_q16(tT0, U);
            tmem_ld_wait();
            float r[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                U[c] = vv[c] - U[c];
                r[c] = bj * U[c];
            }
            store_q16(sm + sA, sm + sAl, r);
        }
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
                    const uint64_t ah = desc_sw128(sb + sT + s * 32, 0, 1024);
                    const uint64_t al = desc_sw128(sb + sT + 8192 + s * 32, 0, 1024);
                    const uint64_t bh = desc_sw128(sb + sA + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(sb + sAl + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + tT0, ah, bh, id, s > 0);
                    mma_bf16(tmem + tT0, ah, bl, id, 1);
                    mma_bf16(tmem + tT0, al, bh, id, 1);
                }
                mma_commit(bar(L_DL));
            }
            __syncwarp();
        }
        w_ok = mbar_wait(bar(L_DL), ph, wl) && mbar_wait(bar(L_D1), ph, wl);
        tc_fence_after();
        if (w_ok) {
            float d[16], a[16], k[16];
            ld_q16(tT0, d);
            ld_q16(tT1, a);
            ld_q16(tT2, k);
            tmem_ld_wait();
            store_q16(sm + sD, sm + sD + 8192, d);
#pragma unroll
            for (int c = 0; c < 16; ++c) a[c] = fmaf(scale, a[c], k[c]);
            store_q16(sm + sE, sm + sE + 8192, a);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // ---- dR = T^T dDelta; Delta dS^T into its sum ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id_t = idesc(kFmtBf16, 1, 1, 64, 64);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sb + sT + s * 2048, 8192, 1024);
                    const uint64_t al = desc_sw128(sb + sT + 8192 + s * 2048, 8192, 1024);
                    const uint64_t bh = desc_sw128(sb + sE + s * 2048, kTile64, 1024);
                    const uint64_t bl = desc_sw128(sb + sE + 8192 + s * 2048, kTile64, 1024);
                    mma_bf16(tmem + tT1, ah, bh, id_t, s > 0);
                    mma_bf16(tmem + tT1, ah, bl, id_t, 1);
                    mma_bf16(tmem + tT1, al, bh, id_t, 1);
                }
                mma_commit(bar(L_R));
                constexpr uint32_t id_3 = idesc(kFmtBf16, 0, 0, 64, 128);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sb + sD + s * 32, 0, 1024);
                    const uint64_t al = desc_sw128(sb + sD + 8192 + s * 32, 0, 1024);
                    const uint64_t bh = desc_sw128(sb + sdS + s * 32, 0, 1024);
                    const uint64_t bl = desc_sw128(sb + sdS + 16384 + s * 32, 0, 1024);
                    mma_bf16(tmem + tAcc3, ah, bh, id_3, sl > 0 || s > 0);
                    mma_bf16(tmem + tAcc3, ah, bl, id_3, 1);
                    mma_bf16(tmem + tAcc3, al, bh, id_3, 1);
                }
            }
            __syncwarp();
        }
        w_ok = mbar_wait(bar(L_R), ph, wl);
        tc_fence_after();
        if (w_ok) {
            float r[16];
            ld_q16(tT1, r);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) dbp = fmaf(r[c], U[c], dbp);
            if (hrow < nv) {
                uint4 o[2];
                uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
                for (int m = 0; m < 8; ++m) ow[m] = cvt_bf16x2(bj * r[2 * m], bj * r[2 * m + 1]);
                uint4* dst = reinterpret_cast<uint4*>(p.dv + ((row0 + hrow) * H + h) * static_cast<long long>(V) +
                                                      col0 + cq);
                dst[0] = o[0];
                dst[1] = o[1];
            }
            // dR over R (Delta = T R has completed)
            store_q16(sm + sA, sm + sAl, r);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
        tc_fence_after();
        // ---- the slice's shares of [dR; dO] Delta^T and [dR; dO] S0^T ----
        if (warp == 0) {
            if (lane == 0) {
                constexpr uint32_t id_1 = idesc(kFmtBf16, 0, 0, 128, 64);
                constexpr uint32_t id_2 = idesc(kFmtBf16, 0, 0, 128, 128);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_sw128(sb + sA + s * 32, 0, 1024);
                    const uint64_t al = desc_sw128(sb + sAl + s * 32, 0, 1024);
                    const uint64_t dh = desc_sw128(sb + sD + s * 32, 0, 1024);
                    const uint64_t dl = desc_sw128(sb + sD + 8192 + s * 32, 0, 1024);
                    const uint64_t sh = desc_sw128(sb + sS0 + s * 32, 0, 1024);
                    const uint64_t sl_ = desc_sw128(sb + sS0 + 16384 + s * 32, 0, 1024);
                    mma_bf16(tmem + tAcc1, ah, dh, id_1, sl > 0 || s > 0);
                    mma_bf16(tmem + tAcc1, ah, dl, id_1, 1);
                    mma_bf16(tmem + tAcc1, al, dh, id_1, 1);
                    mma_bf16(tmem + tAcc2, ah, sh, id_2, sl > 0 || s > 0);
                    mma_bf16(tmem + tAcc2, ah, sl_, id_2, 1);
                    mma_bf16(tmem + tAcc2, al, sh, id_2, 1);
                }
                mma_commit(bar(L_ACC));
            }
            __syncwarp();
        }
        // the next slice overwrites every tile these products read
        w_ok = mbar_wait(bar(L_ACC), ph, wl);
        tc_fence_after();
        if (__syncthreads_or(!(ok && w_ok))) { ok = false; break; }
    }

    if (ok) {
        // ================= end phase: CUDA cores =================
        uint16_t* Ks = reinterpret_cast<uint16_t*>(sm + eK);
        uint16_t* Qs = reinterpret_cast<uint16_t*>(sm + eQ);
        float* Gs = reinterpret_cast<float*>(sm + eG);
        float* dA = reinterpret_cast<float*>(sm + edA);
        float* dP = reinterpret_cast<float*>(sm + edP);
        float* dQ = reinterpret_cast<float*>(sm + edQ);
        float* dK = reinterpret_cast<float*>(sm + edK);
        float* dG = reinterpret_cast<float*>(sm + edG);
        float* bs = reinterpret_cast<float*>(sm + eVec);
        float* Gn = bs + 64;
        float* gn = Gn + kLK;
        float* gsum = gn + kLK;
        float* dbq = gsum + kLK;      // [4][64]
        float* xs = dbq + 4 * 64;     // [4][128]
        float* dbc = xs + 4 * kLK;    // [4][64]: per warp of the pair sums, sum_c k o u1' of each row
        float* wsc = dbc + 4 * 64;    // [16][128]: column sums of the upper row halves
        for (int e = tid; e < 64 * (kLK / 8); e += kLThreads) {
            const int r = e / (kLK / 8), c = (e % (kLK / 8)) * 8;
            uint4 kk = make_uint4(0u, 0u, 0u, 0u), qq = kk;
            float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
            if (r < nv) {
                const long long off = ((row0 + r) * H + h) * static_cast<long long>(kLK) + c;
                kk = *reinterpret_cast<const uint4*>(p.k + off);
                qq = *reinterpret_cast<const uint4*>(p.q + off);
                g0 = *reinterpret_cast<const float4*>(p.g + off);
                g1 = *reinterpret_cast<const float4*>(p.g + off + 4);
            }
            *reinterpret_cast<uint4*>(Ks + r * LDB + c) = kk;
            *reinterpret_cast<uint4*>(Qs + r * LDB + c) = qq;
            *reinterpret_cast<float4*>(Gs + r * LDF + c) = g0;
            *reinterpret_cast<float4*>(Gs + r * LDF + c + 4) = g1;
        }
        if (tid < 64) bs[tid] = gvec[kLK + tid];
        {
            const float g2 = gs + __shfl_xor_sync(0xffffffffu, gs, 1);
            if ((tid & 1) == 0) gsum[tid >> 1] = g2;
        }
        {
            float d = dbp + __shfl_xor_sync(0xffffffffu, dbp, 16);
            if (lane < 16) dbq[hs * 64 + hrow] = d;   // two quarter rows per warp half: index by hs
        }
        __syncthreads();
        kda::chunk_gate_cumsum<kLK, LDF>(Gs, Gn, gn);
        // [dR; dO] Delta^T -> -dA (upper rows), dP / scale (lower rows);
        // [dR; dO] S0^T -> dR S0^T (upper), dO S0^T (lower)
        {
            float v[32];
            tmem_ld16(tmem + lb + tAcc1 + 32 * hs, v);
            tmem_ld16(tmem + lb + tAcc1 + 32 * hs + 16, v + 16);
            tmem_ld_wait();
            if (mrow < 64) {
#pragma unroll
                for (int j = 0; j < 32; ++j) dA[mrow * LDP + 32 * hs + j] = -v[j];
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) dP[(mrow - 64) * LDP + 32 * hs + j] = scale * v[j];
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                tmem_ld16(tmem + lb + tAcc2 + 64 * hs + 16 * q4, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = 64 * hs + 16 * q4 + j;
                    if (mrow < 64) {
                        const int i = mrow;
                        const float eg = expf(Gs[i * LDF + c]);
                        const float dkg = -bs[i] * v[j];
                        dK[i * LDF + c] = dkg * eg;
                        dG[i * LDF + c] = dkg * eg * bf(Ks + i * LDB + c);
                    } else {
                        const int i = mrow - 64;
                        dQ[i * LDF + c] = scale * v[j] * expf(Gs[i * LDF + c]);
                    }
                }
            }
        }
        __syncthreads();
        if (mrow >= 64) {
            // dG += dQG o QG on the rows the upper warps started (warp-uniform branch)
            const int i = mrow - 64;
            float v[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                tmem_ld16(tmem + lb + tAcc2 + 64 * hs + 16 * q4, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = 64 * hs + 16 * q4 + j;
                    dG[i * LDF + c] = fmaf(scale * v[j] * expf(Gs[i * LDF + c]), bf(Qs + i * LDB + c), dG[i * LDF + c]);
                }
            }
        }
        __syncthreads();
        // Delta dS^T = dKt: dK += dKt o exp(G_n - G), dG -= X, X = dKt o Kt
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            float v[16];
            ld_q16(tAcc3 + 64 * m, v);
            tmem_ld_wait();
            const int i = hrow;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = 64 * m + cq + j;
                const float dn = expf(Gn[c] - Gs[i * LDF + c]);
                const float x = v[j] * bf(Ks + i * LDB + c) * dn;
                dK[i * LDF + c] = fmaf(v[j], dn, dK[i * LDF + c]);
                dG[i * LDF + c] -= x;
                // column sum of X over the 16 rows this warp half holds
                float s = x;
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                if ((lane & 15) == 0) xs[sw * kLK + c] = s;
            }
        }
        __syncthreads();

        // ---- the decayed pair sums, 16 x 16 tiles of pairs: thread t takes
        // key channel t % 128 and half the rows of each tile (t / 128), so each
        // pair's decay factor serves both sides (row i: u1, u2; column j: w);
        // the column sums of the two halves meet in shared memory ----
        {
            const int c = tid & (kLK - 1), half = tid >> 7;
            for (int e = tid; e < 4 * 64; e += kLThreads) dbc[e] = 0.f;
            __syncthreads();
            for (int J = 0; J < 4; ++J) {
                float w[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) w[jj] = 0.f;
                for (int I = J; I < 4; ++I)
                    pair_rows(I, J, half, c, lane, warp & 3, Gs, Ks, Qs, dA, dP, bs, dQ, dK, dG, dbc, w);
                // column side of sub-block J: the upper half's sums, then the rows
                if (half == 1) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) wsc[jj * kLK + c] = w[jj];
                }
                __syncthreads();
                if (half == 0) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = 16 * J + jj;
                        const float wj = w[jj] + wsc[jj * kLK + c];
                        dK[j * LDF + c] += wj;
                        dG[j * LDF + c] = fmaf(-bf(Ks + j * LDB + c), wj, dG[j * LDF + c]);
                    }
                }
                __syncthreads();
            }
        }
        __syncthreads();
        // dbeta = sum_c dR o U (the slices) + sum_c k o u1'
        if (tid < nv)
            p.dbeta[(row0 + tid) * H + h] = f32_to_bf16((dbq[tid] + dbq[64 + tid]) +
                                                        ((dbc[tid] + dbc[64 + tid]) + (dbc[128 + tid] + dbc[192 + tid])));
        __syncthreads();
        // dq, dk (bf16), eight channels a thread
        for (int e = tid; e < 64 * (kLK / 8); e += kLThreads) {
            const int r = e / (kLK / 8), c = (e % (kLK / 8)) * 8;
            if (r < nv) {
                uint4 oq, ok4;
                uint32_t* wq = reinterpret_cast<uint32_t*>(&oq);
                uint32_t* wk = reinterpret_cast<uint32_t*>(&ok4);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    wq[m] = cvt_bf16x2(dQ[r * LDF + c + 2 * m], dQ[r * LDF + c + 2 * m + 1]);
                    wk[m] = cvt_bf16x2(dK[r * LDF + c + 2 * m], dK[r * LDF + c + 2 * m + 1]);
                }
                const long long off = ((row0 + r) * H + h) * static_cast<long long>(kLK) + c;
                *reinterpret_cast<uint4*>(p.dq + off) = oq;
                *reinterpret_cast<uint4*>(p.dk + off) = ok4;
            }
        }
        // dg = reverse running sum of dG; the last row also carries
        // exp(G_n) o rowsum(dS o S0) and the column sum of X
        for (int c = tid; c < kLK; c += kLThreads) {
            float run = gn[c] * gsum[c];
            run += (xs[c] + xs[kLK + c]) + (xs[2 * kLK + c] + xs[3 * kLK + c]);
            for (int i = nv - 1; i >= 0; --i) {
                run += dG[i * LDF + c];
                p.dg[((row0 + i) * H + h) * static_cast<long long>(kLK) + c] = run;
            }
        }
    }

    // drain: the block copy and every product issued
    if (tid == 0) {
        if (!ok) record_error(p.err, kErrTimeout);
        mbar_wait(bar(L_BLK), 0, kDefaultWaitLimit);
    }
    if (warp == 0) {
        if (lane == 0) mma_commit(bar(L_DRAIN));
        __syncwarp();
        mbar_wait(bar(L_DRAIN), 0, kDefaultWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kLTmemCols);
}

}  // namespace

cudaError_t launch_kda_bwd_local_tc(const KdaBwdArgs& a, uint32_t wait_limit, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kLAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_chunks, a.H, a.N);
    gdn_kda_local_tc_kernel<<<grid, kLThreads, kLAlloc, stream>>>(a, wait_limit);
    return cudaGetLastError();
}

}  // namespace gdn

// Sequence split: one sequence run as segments whose affine carries compose.
//
// cuLA issue #126 ("Hypothesis") describes intracard context parallelism:
// each segment maps its start state to its end state by an affine transform,
// S_end = M S_start + b (M: K x K, b: K x V), the carries are composed in
// order, and each segment then runs from its true start.  Here the carries
// come from the chunk chain itself: b is the segment's end state from a zero
// start, M its end state from the identity with zero values (the value
// columns of the recurrence are independent, so a run whose state starts at I
// and whose values are 0 leaves exactly the transition in the state).  This
// file holds the two small kernels around those runs: the setup (segment
// bounds as packed sequences, identity start states) and the composition
// (fp32, sequential over a sequence's segments).
#include <cuda.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

// First packed row of segment j of sequence b: b T + 64 floor(j nch / nseg)
// (whole chunks); segment nseg - 1 ends at b T + T.
__device__ __forceinline__ long long seg_start(long long b, int j, int T, int nseg) {
    const long long nch = (T + kChunk - 1) / kChunk;
    return b * T + (j == 0 ? 0 : kChunk * ((j * nch) / nseg));
}

// cu[s] for s = 0 .. B nseg (the segment bounds above); the identity start
// state of every (segment, head); and the zero-start run's start states:
// a sequence's initial state for its first segment (so that segment's run
// is already its true one), zero for the others.
__global__ void gdn_split_setup_kernel(const SplitArgs a) {
    const long long nseq = static_cast<long long>(a.B) * a.nseg;
    const long long kk = static_cast<long long>(a.d_k) * a.d_k;
    const long long kv = static_cast<long long>(a.d_k) * a.d_v;
    const long long total = nseq * a.H * kk, total_s = nseq * a.H * kv;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total + total_s + nseq + 1;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (i <= nseq) {
            const long long pos = i == nseq ? static_cast<long long>(a.B) * a.T
                                            : seg_start(i / a.nseg, static_cast<int>(i % a.nseg), a.T, a.nseg);
            a.cu[i] = static_cast<int32_t>(pos);
        } else if (i <= nseq + total) {
            const long long e = i - nseq - 1;
            const long long r = (e % kk) / a.d_k, c = e % a.d_k;
            a.ident[e] = r == c ? 1.f : 0.f;
        } else {
            const long long e = i - nseq - 1 - total;   // [n][h][k][v]
            const long long n = e / (a.H * kv), rest = e % (a.H * kv);
            a.starts[e] = (n % a.nseg == 0 && a.initial_state) ? a.initial_state[(n / a.nseg) * a.H * kv + rest] : 0.f;
        }
    }
}

// Per (column block of 32, head, sequence): S = the sequence's initial state;
// for each segment j in order, starts[j] = S and S <- M_j S + b_j (j = 0: S <-
// b_0, the first segment's run having started from the initial state); the
// last S is the sequence's final state.  256 threads: thread t owns row t / 2 and
// columns 16 (t % 2) .. + 15 of the block; S sits in shared memory in rows of
// 16-byte chunks, and each thread's row of M_j comes in 32 values at a time
// (eight 16-byte loads in flight); every sum runs over m in order.
constexpr int kComposeThreads = 256;
constexpr int kCols = 32;
constexpr int kSRow = kCols + 4;  // row stride of S (16-byte rows)
__global__ void __launch_bounds__(kComposeThreads) gdn_split_compose_kernel(const SplitArgs a) {
    const int cb = blockIdx.x * kCols, h = blockIdx.y, b = blockIdx.z;
    const int K = a.d_k, V = a.d_v;
    const int t = threadIdx.x, r = t >> 1, c0 = 16 * (t & 1);
    __shared__ __align__(16) float S[128][kSRow];
    const bool live = r < K;
    if (live) {
        float4* srow = reinterpret_cast<float4*>(&S[r][c0]);
        const float4* src = a.initial_state ? reinterpret_cast<const float4*>(
                                                  a.initial_state + ((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0)
                                            : nullptr;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) srow[c4] = src ? src[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    for (int j = 0; j < a.nseg; ++j) {
        const long long n = static_cast<long long>(b) * a.nseg + j;
        float acc[16];
        if (live) {
            float4* st = reinterpret_cast<float4*>(a.starts + ((n * a.H + h) * K + r) * V + cb + c0);
            const float4* bj = reinterpret_cast<const float4*>(a.b_fin + ((n * a.H + h) * K + r) * V + cb + c0);
            const float4* srow = reinterpret_cast<const float4*>(&S[r][c0]);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                st[c4] = srow[c4];
                const float4 b4 = bj[c4];
                acc[4 * c4] = b4.x; acc[4 * c4 + 1] = b4.y; acc[4 * c4 + 2] = b4.z; acc[4 * c4 + 3] = b4.w;
            }
            const float4* mrow = reinterpret_cast<const float4*>(a.m_fin + ((n * a.H + h) * K + r) * static_cast<long long>(K));
            for (int m32 = 0; j > 0 && m32 < K; m32 += 32) {
                float4 mv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mv[u] = mrow[m32 / 4 + u];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float mvals[4] = {mv[u].x, mv[u].y, mv[u].z, mv[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4* sm4 = reinterpret_cast<const float4*>(&S[m32 + 4 * u + e][c0]);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const float4 s4 = sm4[c4];
                            acc[4 * c4] = fmaf(mvals[e], s4.x, acc[4 * c4]);
                            acc[4 * c4 + 1] = fmaf(mvals[e], s4.y, acc[4 * c4 + 1]);
                            acc[4 * c4 + 2] = fmaf(mvals[e], s4.z, acc[4 * c4 + 2]);
                            acc[4 * c4 + 3] = fmaf(mvals[e], s4.w, acc[4 * c4 + 3]);
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (live) {
            float4* srow = reinterpret_cast<float4*>(&S[r][c0]);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                srow[c4] = make_float4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]);
        }
        __syncthreads();
    }
    if (a.final_state && live) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            a.final_state[((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0 + c] = S[r][c0 + c];
    }
}

// out = bf16(O_b + O_M S_start) for every row of every segment, on the tensor
// cores: per chunk of 64 rows, D[64 x N] = O_M[64 x d_k] S_start[d_k x N]
// with both operands split into bf16 hi + lo (hi hi + hi lo + lo hi, fp32
// accumulation in TMEM), N = 64 or 128 value columns.  The kernel mostly
// moves bytes (O_M and O_b in fp32 in, out in bf16), so it is laid out for
// bandwidth: one persistent CTA per SM walks a contiguous range of (segment,
// head, value block, chunk) units, and each unit's 64 rows of O_M and O_b
// come in as TMA boxes ahead of it: O_M into one fp32 staging tile,
// converted into one of two pairs of hi/lo operand tiles at the top of its
// unit and refilled for the next unit at once; O_b (32-column boxes,
// 128-byte swizzled, so that the epilogue's reads of 16 rows at once fall on
// distinct banks) into one of two staging tiles.  A unit's product runs into
// one of two TMEM accumulators while the epilogue of the unit before it
// (O_b + the product, to bf16) runs.  A unit past the end of its
// segment copies and stores nothing.  A sequence's first segment started its
// zero-start run from the true initial state, so its units only convert
// O_b (no O_M rows, no product).  The start-state block is converted when a
// CTA's range enters a new (segment, head, value block).
constexpr int kCorrThreads = 256;  // warps w and w + 4 share TMEM subpartition w % 4
constexpr int kCorrTile = 64 * 128;  // 64 rows x 128 B

// A unit and where its rows are.  Units run value block fastest, then
// head, then segment (chunk index c innermost of all); a CTA steps through
// its range with corr_next, which does the divisions only when the segment
// changes.
struct CorrUnit {
    int c, vb, h, n;     // chunk, value block, head, segment
    bool first;          // a sequence's first segment: out = O_b
    long long t0, t1;    // the segment's packed rows [t0, t1)
    long long r0;        // first row of the chunk
    int nv;              // its rows inside the segment (0: past the segment's end)
};

__device__ __forceinline__ void corr_rows(const SplitCorrectArgs& a, CorrUnit& x) {
    x.r0 = x.t0 + static_cast<long long>(x.c) * kChunk;
    const long long left = x.t1 - x.r0;
    x.nv = static_cast<int>(left < 0 ? 0 : (left < kChunk ? left : kChunk));
}

__device__ __forceinline__ void corr_segment(const SplitCorrectArgs& a, CorrUnit& x) {
    // the segment's bounds by the setup's rule (no dependent loads of cu)
    const long long b = x.n / a.nseg;
    const int j = x.n % a.nseg;
    x.first = j == 0;
    x.t0 = seg_start(b, j, a.T, a.nseg);
    x.t1 = j + 1 < a.nseg ? seg_start(b, j + 1, a.T, a.nseg) : (b + 1) * a.T;
}

__device__ __forceinline__ CorrUnit corr_unit(const SplitCorrectArgs& a, int nvb, long long u) {
    CorrUnit x;
    const long long combo = u / a.max_chunks;
    x.c = static_cast<int>(u % a.max_chunks);
    x.vb = static_cast<int>(combo % nvb);
    x.h = static_cast<int>((combo / nvb) % a.H);
    x.n = static_cast<int>(combo / (static_cast<long long>(nvb) * a.H));
    corr_segment(a, x);
    corr_rows(a, x);
    return x;
}

__device__ __forceinline__ CorrUnit corr_next(const SplitCorrectArgs& a, int nvb, CorrUnit x) {
    if (++x.c == a.max_chunks) {
        x.c = 0;
        if (++x.vb == nvb) {
            x.vb = 0;
            if (++x.h == a.H) {
                x.h = 0;
                ++x.n;
                if (x.n < a.nseq) corr_segment(a, x);
            }
        }
    }
    corr_rows(a, x);
    return x;
}

__global__ void __launch_bounds__(kCorrThreads, 1)
    gdn_split_correct_kernel(const __grid_constant__ CUtensorMap tmap_omh, const __grid_constant__ CUtensorMap tmap_oml,
                             const __grid_constant__ CUtensorMap tmap_ob,
                             const SplitCorrectArgs a) {
    using namespace sm100;
    using namespace tc;
    const int K = a.d_k, V = a.d_v, H = a.H;
    const int nb = V >= 128 ? 2 : 1;             // 64-column blocks of a unit
    const int nvb = V / (64 * nb);               // value blocks per head
    const int kreg = K / 64;                     // 64-column regions of d_k
    const long long units = static_cast<long long>(a.nseq) * H * nvb * a.max_chunks;
    const long long u_begin = units * blockIdx.x / gridDim.x;
    const long long u_end = units * (blockIdx.x + 1) / gridDim.x;
    if (u_begin >= u_end) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t wl = a.wait_limit;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    // B: S_start block, [d_k rows][64 value columns] per MN block, hi then lo;
    // A: [3] O_M rows, [64 rows][64 key columns] per region, hi then lo (the
    // identity run wrote O_M as bf16 hi and lo planes, so its TMA boxes land
    // as operand tiles); O_b staging [2][2 nb boxes][64 rows][32 values]
    const int bBytes = K * 128;                  // one MN block (hi or lo)
    const int obUnit = 64 * 64 * nb * 4;         // one unit's O_b staging
    uint8_t* Bhi = sm;
    uint8_t* Blo = sm + nb * bBytes;
    uint8_t* Aop = sm + 2 * nb * bBytes;         // [3][hi, lo][kreg regions]
    const int aBytes = 2 * kreg * kCorrTile;
    uint8_t* B32 = Aop + 3 * aBytes;
    uint64_t* barp = reinterpret_cast<uint64_t*>(B32 + 2 * obUnit);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(barp + 10);
    auto bar_a = [&](int i) { return smem_u32(barp + i); };          // O_M tiles of buffer i (of 3)
    auto bar_mma = [&](int i) { return smem_u32(barp + 3 + i); };    // product into accumulator i
    auto bar_b = [&](int i) { return smem_u32(barp + 5 + i); };      // O_b copy of buffer i
    auto bar_tf = [&](int i) { return smem_u32(barp + 7 + i); };     // accumulator i read out
    const uint32_t bar_drain = smem_u32(barp + 9);
    constexpr uint32_t kCorrCols = 256;           // two 128-column accumulators

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kCorrCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 10; ++i) mbar_init(smem_u32(barp + i), 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmap_omh);
        tma_prefetch_desc(&tmap_oml);
        tma_prefetch_desc(&tmap_ob);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // one thread: a unit's O_M tiles into operand buffer j (rows past the
    // segment come along; each output row reads only its own row of A, and
    // those rows are not stored), and its O_b boxes into staging buffer buf;
    // a unit past its segment's end, or of a first segment, loads nothing
    // and only arrives
    auto issue_om = [&](const CorrUnit& x, int j) {
        const bool load = x.nv && !x.first;
        mbar_arrive_expect_tx(bar_a(j), load ? static_cast<uint32_t>(aBytes) : 0u);
        if (load) {
            const uint32_t dst = smem_u32(Aop + j * aBytes);
            for (int r = 0; r < kreg; ++r) {
                tma_load_3d(dst + r * kCorrTile, &tmap_omh, 64 * r, x.h, static_cast<int>(x.r0), bar_a(j));
                tma_load_3d(dst + (kreg + r) * kCorrTile, &tmap_oml, 64 * r, x.h, static_cast<int>(x.r0), bar_a(j));
            }
        }
    };
    auto issue_ob = [&](const CorrUnit& x, int buf) {
        mbar_arrive_expect_tx(bar_b(buf), x.nv ? static_cast<uint32_t>(obUnit) : 0u);
        if (x.nv)
            for (int j = 0; j < 2 * nb; ++j)
                tma_load_3d(smem_u32(B32 + buf * obUnit + j * 8192), &tmap_ob, x.vb * 64 * nb + 32 * j, x.h,
                            static_cast<int>(x.r0), bar_b(buf));
    };
    // S_start[n][h][k][v0 .. v0 + 64 nb) as split MN-major tiles: row k, 8
    // values per 16-byte chunk; loads first, then the splits
    auto load_start = [&](const CorrUnit& x, int th, int nth) {
        const float* src = a.starts + (static_cast<long long>(x.n) * H + x.h) * K * V + x.vb * 64 * nb;
        for (int base = 0; base < K * 8 * nb; base += 4 * nth) {
            float4 sv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + th + nth * i, k = e / (8 * nb), c = e % (8 * nb);
                sv[2 * i] = sv[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e < K * 8 * nb) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<long long>(k) * V + 8 * c);
                    sv[2 * i] = s4[0];
                    sv[2 * i + 1] = s4[1];
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + th + nth * i, k = e / (8 * nb), c = e % (8 * nb);
                if (e < K * 8 * nb) {
                    const float x8[8] = {sv[2 * i].x, sv[2 * i].y, sv[2 * i].z, sv[2 * i].w,
                                         sv[2 * i + 1].x, sv[2 * i + 1].y, sv[2 * i + 1].z, sv[2 * i + 1].w};
                    store_split_chunk(Bhi + (c >> 3) * bBytes, Blo + (c >> 3) * bBytes, k, c & 7, x8);
                }
            }
        }
    };

    // Warps 0-3 produce (the O_M conversion into the operand tiles, the
    // products, the O_M copies), warps 4-7 consume (the epilogues, the O_b
    // copies); the two groups meet only at mbarriers, whose phases follow
    // from the unit index k of the CTA's range: unit k is completion k of the
    // O_M barrier and completion k / 2 of the barriers of its buffer k % 2.
    const bool producer = warp < 4;
    const int gtid = tid & 127;                  // thread in its group
    const int gbar = producer ? 1 : 2;           // the group's named barrier
    auto group_or = [&](bool pred) -> bool {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"(static_cast<uint32_t>(pred)), "r"(gbar)
            : "memory");
        return r != 0;
    };
    auto par = [](long long k) { return static_cast<uint32_t>((k >> 1) & 1); };  // phase of unit k on its buffer
    bool failed = false;
    const long long nk = u_end - u_begin;
    CorrUnit cur = corr_unit(a, nvb, u_begin);

    if (producer) {
        // O_M tiles two units ahead in a ring of three operand buffers
        long long om_issued = nk < 2 ? nk : 2, om_seen = 0;
        CorrUnit ahead = corr_next(a, nvb, cur);      // the unit two ahead, once the loop runs
        if (gtid == 0) {
            issue_om(cur, 0);
            if (nk > 1) issue_om(ahead, 1);
        }
        ahead = corr_next(a, nvb, ahead);
        for (long long k = 0; k < nk; ++k) {
            const int tb = static_cast<int>(k & 1), j = static_cast<int>(k % 3);
            if ((k == 0 || cur.c == 0) && !cur.first) {
                // a new (segment, head, value block): its start-state block,
                // once the previous unit's product (the B tiles' last reader)
                // is done; the group takes one decision to leave
                if (k > 0 && !mbar_wait(bar_mma(tb ^ 1), par(k - 1), wl)) failed = true;
                if (!failed) load_start(cur, gtid, 128);
                fence_proxy_async_smem();
                if (group_or(failed)) break;
            }
            // warp 0 issues; after a wait ran out it only keeps step with the
            // group (whose barriers above every warp must reach) and does no work
            if (warp == 0 && !failed) {
                bool ok = __all_sync(0xffffffffu, mbar_wait(bar_a(j), static_cast<uint32_t>((k / 3) & 1), wl));
                if (ok) ++om_seen;
                // accumulator tb: the epilogue of unit k - 2 has read it
                ok = ok && (k < 2 || __all_sync(0xffffffffu, mbar_wait(bar_tf(tb), par(k - 2), wl)));
                if (ok && elect_one()) {
                    tc_fence_after();
                    const uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64 * nb);
                    const uint32_t ah = smem_u32(Aop + j * aBytes), al = ah + kreg * kCorrTile;
                    const uint32_t bh = smem_u32(Bhi), bl = smem_u32(Blo);
                    const uint32_t d = tmem + 128 * tb;
                    // (a first-segment unit commits with no product: the
                    // barrier then only waits for the products before it)
                    for (int s = 0; !cur.first && s < K / 16; ++s) {
                        const uint32_t ao = (s >> 2) * kCorrTile + (s & 3) * 32;
                        const uint64_t da_h = desc_sw128(ah + ao, 0, 1024), da_l = desc_sw128(al + ao, 0, 1024);
                        const uint64_t db_h = desc_sw128(bh + s * 2048, bBytes, 1024);
                        const uint64_t db_l = desc_sw128(bl + s * 2048, bBytes, 1024);
                        mma_bf16(d, da_h, db_h, id, s > 0);
                        mma_bf16(d, da_h, db_l, id, 1);
                        mma_bf16(d, da_l, db_h, id, 1);
                    }
                    mma_commit(bar_mma(tb));
                }
                __syncwarp();
                // unit k + 2's tiles into buffer (k + 2) % 3, whose last reader
                // was the product of unit k - 1
                if (ok && k + 2 < nk) {
                    ok = k < 1 || __all_sync(0xffffffffu, mbar_wait(bar_mma(tb ^ 1), par(k - 1), wl));
                    if (ok) {
                        if (lane == 0) issue_om(ahead, static_cast<int>((k + 2) % 3));
                        ++om_issued;
                    }
                }
                if (!ok) failed = true;  // the consumer group times out on this unit's product too
            }
            cur = corr_next(a, nvb, cur);
            if (k + 3 < nk) ahead = corr_next(a, nvb, ahead);
        }
        // nothing the group issued outlives the CTA: its products, then its copies
        if (warp == 0) {
            if (elect_one()) mma_commit(bar_drain);
            __syncwarp();
            if (!mbar_wait(bar_drain, 0, kDefaultWaitLimit)) failed = true;
            for (; om_seen < om_issued; ++om_seen)
                if (!mbar_wait(bar_a(static_cast<int>(om_seen % 3)), static_cast<uint32_t>((om_seen / 3) & 1),
                               kDefaultWaitLimit))
                    failed = true;
        }
    } else {
        // consumer: O_b copies (two units ahead) and every epilogue
        long long b_issued = nk < 2 ? nk : 2, b_seen = 0;  // O_b copies issued / seen complete
        CorrUnit ahead = corr_next(a, nvb, cur);          // the unit two ahead, once the loop runs
        if (gtid == 0) {
            issue_ob(cur, 0);
            if (nk > 1) issue_ob(ahead, 1);
        }
        ahead = corr_next(a, nvb, ahead);
        const int sub = warp & 3;
        const int row = 16 * sub + (lane & 15);       // accumulator row of this lane
        const int cpart = 32 * (lane >> 4);           // its 32 columns of each 64-column block
        for (long long k = 0; k < nk; ++k) {
            const int buf = static_cast<int>(k & 1);
            if (mbar_wait(bar_b(buf), par(k), wl)) ++b_seen;
            else failed = true;
            if (!mbar_wait(bar_mma(buf), par(k), wl)) failed = true;
            tc_fence_after();
            // out = bf16(O_b + the product) for row `row`, columns 64 blk + cpart .. + 31
            for (int blk = 0; blk < nb; ++blk) {
                float acc[32];
                if (cur.first) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                } else {
                    ld_half32(tmem, sub, 128 * buf + 64 * blk, acc);
                }
                if (row < cur.nv) {
                    // row `row` of box 2 blk + cpart / 32, its 16-byte chunk q at q ^ (row % 8)
                    const uint8_t* box = B32 + buf * obUnit + (2 * blk + (cpart >> 5)) * 8192 + row * 128;
                    float4 ob4[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) ob4[q] = *reinterpret_cast<const float4*>(box + ((q ^ (row & 7)) << 4));
                    uint4* dst = reinterpret_cast<uint4*>(a.out + (cur.r0 + row) * H * static_cast<long long>(V) +
                                                          static_cast<long long>(cur.h) * V + cur.vb * 64 * nb +
                                                          64 * blk + cpart);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x0 = ob4[2 * q], x1 = ob4[2 * q + 1];
                        const float* y = acc + 8 * q;
                        dst[q] = make_uint4(pack_bf16x2(x0.x + y[0], x0.y + y[1]), pack_bf16x2(x0.z + y[2], x0.w + y[3]),
                                            pack_bf16x2(x1.x + y[4], x1.y + y[5]), pack_bf16x2(x1.z + y[6], x1.w + y[7]));
                    }
                }
            }
            tc_fence_before();
            // staging buffer buf and accumulator buf are read out
            if (group_or(failed)) break;
            if (gtid == 0) {
                mbar_arrive(bar_tf(buf));
                if (k + 2 < nk) issue_ob(ahead, buf);
            }
            if (k + 2 < nk) ++b_issued;
            cur = corr_next(a, nvb, cur);
            if (k + 3 < nk) ahead = corr_next(a, nvb, ahead);
        }
        for (; b_seen < b_issued; ++b_seen)
            if (!mbar_wait(bar_b(static_cast<int>(b_seen & 1)), par(b_seen), kDefaultWaitLimit)) failed = true;
    }
    if (failed) record_error(a.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kCorrCols);
}

}  // namespace

cudaError_t launch_split_setup(const SplitArgs& a, cudaStream_t stream) {
    const long long n = static_cast<long long>(a.B) * a.nseg * a.H * a.d_k * (a.d_k + a.d_v) +
                        static_cast<long long>(a.B) * a.nseg + 1;
    const long long blocks = (n + 255) / 256;
    gdn_split_setup_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_compose(const SplitArgs& a, cudaStream_t stream) {
    dim3 grid(a.d_v / kCols, a.H, a.B);
    gdn_split_compose_kernel<<<grid, kComposeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

namespace {

// 3-D view {inner, head, row} of a (rows, H, inner) fp32 tensor, box
// {box_inner, 1, 64}; 128-byte swizzle when the box is 32 values wide.
bool make_f32_rows_map(CUtensorMap* m, const float* base, long long rows, int H, int inner, int box_inner) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 4, static_cast<cuuint64_t>(H) * inner * 4};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, box_inner == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_split_correct(const SplitCorrectArgs& a, cudaStream_t stream) {
    if (a.max_chunks == 0 || a.nseq == 0 || a.rows == 0) return cudaSuccess;
    const int nb = a.d_v >= 128 ? 2 : 1;
    CUtensorMap momh, moml, mob;
    memset(&momh, 0, sizeof(momh));
    memset(&moml, 0, sizeof(moml));
    memset(&mob, 0, sizeof(mob));
    const uint16_t* omh = reinterpret_cast<const uint16_t*>(a.om);
    const uint16_t* oml = omh + a.rows * a.H * a.d_k;
    if (!tc::make_rows_map(&momh, omh, a.rows, a.H, a.d_k) || !tc::make_rows_map(&moml, oml, a.rows, a.H, a.d_k) ||
        !make_f32_rows_map(&mob, a.ob, a.rows, a.H, a.d_v, 32))
        return cudaErrorInvalidValue;
    const int smem = 2 * nb * a.d_k * 128 + 6 * (a.d_k / 64) * kCorrTile + 2 * 64 * 64 * nb * 4 + 96 + 1024;
    cudaError_t e = cudaFuncSetAttribute(gdn_split_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long units = static_cast<long long>(a.nseq) * a.H * (a.d_v / (64 * nb)) * a.max_chunks;
    const int grid = static_cast<int>(units < sms ? units : sms);
    gdn_split_correct_kernel<<<grid, kCorrThreads, smem, stream>>>(momh, moml, mob, a);
    return cudaGetLastError();
}

}  // namespace gdn

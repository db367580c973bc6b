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
#include "gdn_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"
#include "sm100_ptx.cuh"

namespace gdn {

namespace {

// cu[s] for s = 0 .. B nseg: sequence b's segment j starts at token
// b T + 64 floor(j nch / nseg) (whole chunks), the last one ends at b T + T;
// then the identity start state of every (segment, head).
__global__ void gdn_split_setup_kernel(const SplitArgs a) {
    const long long nch = (a.T + kChunk - 1) / kChunk;
    const long long nseq = static_cast<long long>(a.B) * a.nseg;
    const long long kk = static_cast<long long>(a.d_k) * a.d_k;
    const long long total = nseq * a.H * kk;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total + nseq + 1;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (i <= nseq) {
            const long long b = i / a.nseg, j = i % a.nseg;
            long long pos = b * a.T + (j == 0 ? 0 : kChunk * ((j * nch) / a.nseg));
            if (i == nseq) pos = static_cast<long long>(a.B) * a.T;
            a.cu[i] = static_cast<int32_t>(pos);
        } else {
            const long long e = i - nseq - 1;
            const long long r = (e % kk) / a.d_k, c = e % a.d_k;
            a.ident[e] = r == c ? 1.f : 0.f;
        }
    }
}

// Per (column block of 32, head, sequence): S = the sequence's initial state;
// for each segment j in order, starts[j] = S and S <- M_j S + b_j; the last S
// is the sequence's final state.  256 threads: thread t owns row t / 2 and
// columns 16 (t % 2) .. + 15 of the block.
constexpr int kComposeThreads = 256;
constexpr int kCols = 32;
__global__ void __launch_bounds__(kComposeThreads) gdn_split_compose_kernel(const SplitArgs a) {
    const int cb = blockIdx.x * kCols, h = blockIdx.y, b = blockIdx.z;
    const int K = a.d_k, V = a.d_v;
    const int t = threadIdx.x, r = t >> 1, c0 = 16 * (t & 1);
    __shared__ float S[128][kCols + 1];
    const bool live = r < K;
    if (live) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            S[r][c0 + c] = a.initial_state
                               ? a.initial_state[((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0 + c]
                               : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < a.nseg; ++j) {
        const long long n = static_cast<long long>(b) * a.nseg + j;
        float acc[16];
        if (live) {
            float* st = a.starts + ((n * a.H + h) * K + r) * V + cb + c0;
            const float* bj = a.b_fin + ((n * a.H + h) * K + r) * V + cb + c0;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                st[c] = S[r][c0 + c];
                acc[c] = bj[c];
            }
            const float* mrow = a.m_fin + ((n * a.H + h) * K + r) * static_cast<long long>(K);
            for (int m = 0; m < K; ++m) {
                const float mv = mrow[m];
#pragma unroll
                for (int c = 0; c < 16; ++c) acc[c] = fmaf(mv, S[m][c0 + c], acc[c]);
            }
        }
        __syncthreads();
        if (live) {
#pragma unroll
            for (int c = 0; c < 16; ++c) S[r][c0 + c] = acc[c];
        }
        __syncthreads();
    }
    if (a.final_state && live) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            a.final_state[((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0 + c] = S[r][c0 + c];
    }
}

// out = bf16(O_b + O_M S_start) for the rows of one segment, on the tensor
// cores: per chunk of 64 rows, D[64 x N] = O_M[64 x d_k] S_start[d_k x N]
// with both operands split into bf16 hi + lo (hi hi + hi lo + lo hi, fp32
// accumulation in TMEM), N = 64 or 128 value columns.  Block (group of
// kCorrG chunks, value block of N columns and head, segment); the segment's
// start-state block is converted once and serves every chunk of the group.
constexpr int kCorrThreads = 128;
constexpr int kCorrG = 8;
constexpr int kCorrTile = 64 * 128;  // 64 rows x 128 B

__global__ void __launch_bounds__(kCorrThreads) gdn_split_correct_kernel(const SplitCorrectArgs a) {
    using namespace sm100;
    using namespace tc;
    const int K = a.d_k, V = a.d_v, H = a.H;
    const int nb = V >= 128 ? 2 : 1;             // 64-column blocks of this CTA
    const int nvb = V / (64 * nb);               // value blocks per head
    const int vb = blockIdx.y % nvb, h = blockIdx.y / nvb, n = blockIdx.z;
    const int t0 = a.cu[n], t1 = a.cu[n + 1];
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;
    const int c_begin = blockIdx.x * kCorrG, c_end = min(nch, c_begin + kCorrG);
    if (c_begin >= c_end) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = vb * 64 * nb;                 // first value column of this CTA
    const int kreg = K / 64;                     // 64-column regions of d_k

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + smem_align_pad(smem_raw);
    // B: S_start block, [d_k rows][64 value columns] per MN block, hi then lo;
    // A: O_M rows, [64 rows][64 key columns] per region, hi then lo
    const int bBytes = K * 128;                  // one MN block (hi or lo)
    uint8_t* Bhi = sm;
    uint8_t* Blo = sm + nb * bBytes;
    uint8_t* Ahi = sm + 2 * nb * bBytes;
    uint8_t* Alo = Ahi + kreg * kCorrTile;
    uint64_t* barp = reinterpret_cast<uint64_t*>(Alo + kreg * kCorrTile);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(barp + 1);
    const uint32_t bar = smem_u32(barp);
    constexpr uint32_t kCorrCols = 128;

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), kCorrCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // S_start[n][h][k][v0 .. v0 + 64 nb) as split MN-major tiles: row k, 8 values per 16-byte chunk
    {
        const float* src = a.starts + (static_cast<long long>(n) * H + h) * K * V + v0;
        // K 8 nb chunks of 8 values, 4 .. 16 a thread: loads first, then the splits
        for (int base = 0; base < K * 8 * nb; base += 4 * kCorrThreads) {
            float4 sv[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + tid + kCorrThreads * i, k = e / (8 * nb), c = e % (8 * nb);
                sv[2 * i] = sv[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e < K * 8 * nb) {
                    const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<long long>(k) * V + 8 * c);
                    sv[2 * i] = s4[0];
                    sv[2 * i + 1] = s4[1];
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = base + tid + kCorrThreads * i, k = e / (8 * nb), c = e % (8 * nb);
                if (e < K * 8 * nb) {
                    const float x[8] = {sv[2 * i].x, sv[2 * i].y, sv[2 * i].z, sv[2 * i].w,
                                        sv[2 * i + 1].x, sv[2 * i + 1].y, sv[2 * i + 1].z, sv[2 * i + 1].w};
                    store_split_chunk(Bhi + (c >> 3) * bBytes, Blo + (c >> 3) * bBytes, k, c & 7, x);
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    uint32_t phase = 0;
    bool failed = false;
    const int row = 16 * warp + (lane & 15);      // accumulator row of this lane
    const int cpart = 32 * (lane >> 4);           // its 32 columns of each 64-column block
    // this thread's slots of the A tile: e = tid + 128 i -> row e / (d_k / 8),
    // 8-value chunk e % (d_k / 8); the next chunk's values are loaded while
    // the current chunk's product and epilogue run
    const int na = K / 16;                        // slots per thread (8 or 4)
    float4 pre[16];
    auto load_a = [&](int c) {
        const long long r0 = t0 + static_cast<long long>(c) * kChunk;
        const int nv = min(kChunk, t1 - static_cast<int>(r0));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            pre[2 * i] = pre[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int e = tid + kCorrThreads * i, r = e / (K / 8), c8 = e % (K / 8);
            if (i < na && r < nv) {
                const float4* s4 = reinterpret_cast<const float4*>(a.om + ((r0 + r) * H + h) * K + 8 * c8);
                pre[2 * i] = s4[0];
                pre[2 * i + 1] = s4[1];
            }
        }
    };
    load_a(c_begin);
    for (int c = c_begin; c < c_end; ++c) {
        const long long r0 = t0 + static_cast<long long>(c) * kChunk;
        const int nv = min(kChunk, t1 - static_cast<int>(r0));
        // A = O_M rows r0 .. r0 + 63 (rows past the segment are zero)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < na) {
                const int e = tid + kCorrThreads * i, r = e / (K / 8), c8 = e % (K / 8);
                const float x[8] = {pre[2 * i].x, pre[2 * i].y, pre[2 * i].z, pre[2 * i].w,
                                    pre[2 * i + 1].x, pre[2 * i + 1].y, pre[2 * i + 1].z, pre[2 * i + 1].w};
                store_split_chunk(Ahi + (c8 >> 3) * kCorrTile, Alo + (c8 >> 3) * kCorrTile, r, c8 & 7, x);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            if (elect_one()) {
                tc_fence_after();
                const uint32_t id = idesc(kFmtBf16, 0, 1, 64, 64 * nb);
                const uint32_t ah = smem_u32(Ahi), al = smem_u32(Alo), bh = smem_u32(Bhi), bl = smem_u32(Blo);
                for (int s = 0; s < K / 16; ++s) {
                    const uint32_t ao = (s >> 2) * kCorrTile + (s & 3) * 32;
                    const uint64_t da_h = desc_sw128(ah + ao, 0, 1024), da_l = desc_sw128(al + ao, 0, 1024);
                    const uint64_t db_h = desc_sw128(bh + s * 2048, bBytes, 1024);
                    const uint64_t db_l = desc_sw128(bl + s * 2048, bBytes, 1024);
                    mma_bf16(tmem, da_h, db_h, id, s > 0);
                    mma_bf16(tmem, da_h, db_l, id, 1);
                    mma_bf16(tmem, da_l, db_h, id, 1);
                }
                mma_commit(bar);
            }
            __syncwarp();
        }
        // while the product runs: this chunk's O_b values and the next chunk's O_M
        float4 ob[2][8];
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
            for (int q = 0; q < 8; ++q) ob[blk][q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (blk < nb && row < nv) {
                const float4* b4 = reinterpret_cast<const float4*>(
                    a.ob + (r0 + row) * H * static_cast<long long>(V) + static_cast<long long>(h) * V + v0 + 64 * blk + cpart);
#pragma unroll
                for (int q = 0; q < 8; ++q) ob[blk][q] = b4[q];
            }
        }
        if (c + 1 < c_end) load_a(c + 1);
        if (!mbar_wait(bar, phase, a.wait_limit)) failed = true;
        phase ^= 1u;
        tc_fence_after();
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            if (blk < nb) {
                float acc[32];
                ld_half32(tmem, warp, 64 * blk, acc);
                if (row < nv) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        a.out + (r0 + row) * H * static_cast<long long>(V) + static_cast<long long>(h) * V + v0 + 64 * blk + cpart);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x0 = ob[blk][2 * q], x1 = ob[blk][2 * q + 1];
                        const float* y = acc + 8 * q;
                        dst[q] = make_uint4(pack_bf16x2(x0.x + y[0], x0.y + y[1]), pack_bf16x2(x0.z + y[2], x0.w + y[3]),
                                            pack_bf16x2(x1.x + y[4], x1.y + y[5]), pack_bf16x2(x1.z + y[6], x1.w + y[7]));
                    }
                }
            }
        }
        tc_fence_before();
        // the next chunk rewrites A and the accumulator; every thread takes
        // the same decision to leave
        if (__syncthreads_or(failed)) break;
    }
    if (failed) {
        record_error(a.err, kErrTimeout);
        // the product never signalled: let it land before the TMEM is freed
        mbar_wait(bar, phase ^ 1u, kDefaultWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kCorrCols);
}

}  // namespace

cudaError_t launch_split_setup(const SplitArgs& a, cudaStream_t stream) {
    const long long n = static_cast<long long>(a.B) * a.nseg * a.H * a.d_k * a.d_k + static_cast<long long>(a.B) * a.nseg + 1;
    const long long blocks = (n + 255) / 256;
    gdn_split_setup_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_compose(const SplitArgs& a, cudaStream_t stream) {
    dim3 grid(a.d_v / kCols, a.H, a.B);
    gdn_split_compose_kernel<<<grid, kComposeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_correct(const SplitCorrectArgs& a, cudaStream_t stream) {
    if (a.max_chunks == 0 || a.nseq == 0) return cudaSuccess;
    const int nb = a.d_v >= 128 ? 2 : 1;
    const int smem = 2 * nb * a.d_k * 128 + 2 * (a.d_k / 64) * kCorrTile + 16 + 1024;
    cudaError_t e = cudaFuncSetAttribute(gdn_split_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.max_chunks + kCorrG - 1) / kCorrG, a.H * (a.d_v / (64 * nb)), a.nseq);
    gdn_split_correct_kernel<<<grid, kCorrThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

// Chunked forward of the per-channel-gate (KDA) gated delta rule, fp32 on
// the CUDA cores.
//
// The gate of the KDA variant that cuLA issue #126 reproduces
// (`flash_kda_fwd`) has one log decay per key channel, g_t in R^{d_k}; the
// state update decays each key row of S by its own factor,
//   S <- diag(exp(g_t)) S;  S <- S + beta_t k_t (v_t - S^T k_t)^T,
// and the readout is o_t = scale S^T q_t.  In a chunk of n <= 64 tokens with
// start state S0 and the running sums G_i = g_1 + ... + g_i (now vectors),
// unrolling the update the same way as for a scalar gate gives
//   A_ij  = beta_i sum_c k_ic k_jc exp(G_ic - G_jc),  j < i
//   P_ij  =        sum_c q_ic k_jc exp(G_ic - G_jc),  j <= i
//   T     = (I + A)^-1
//   Delta = T [beta o (V - (exp(G) o K) S0)]
//   O     = scale [(exp(G) o Q) S0 + P Delta]
//   S1    = diag(exp(G_n)) S0 + (exp(G_n - G) o K)^T Delta
// where exp(G) o K scales k_ic by exp(G_ic).  With a scalar gate the decay
// factors leave the dot products and this is the scalar chunk algebra.  With a
// per-channel gate they cannot: the gram and the causal score take the decay
// inside the sum over key channels, pair by pair.  Each exponent is formed as a
// difference G_ic - G_jc with j <= i, so it is <= 0 for any g <= 0 and never
// overflows, at any decay strength (the pair's exponent is masked before exp).
//
// One thread block per (value slice of 64 columns, head, sequence) walks the
// sequence chunk by chunk with its d_k x 64 slice of the state in shared
// memory (the value columns of the recurrence are independent).  Shared rows
// are padded to a multiple of four floats (and to 4 banks mod 32), so every
// product reads its operands as 16-byte vectors: a thread owns four adjacent
// output columns and a few rows, and each step of the reduction takes four
// terms at once.
//
// T and P depend on the keys, queries, gates and betas of one chunk only.
// Given a workspace, gdn_kda_tp_kernel forms them for every chunk in parallel
// (one block per chunk and head) and the walk above loads them, so the
// serial chain keeps only the products with the state: the gram's decay
// exponentials, about a third of a million per chunk, leave the critical
// path.  The walk can also record every chunk's start state (the forward state
// pass of the backward).
#include "gdn_common.cuh"
#include "gdn_kda_common.cuh"
#include "gdn_kernels.h"
#include "gdn_tc_common.cuh"

namespace gdn {

namespace {

using namespace kda;

constexpr int kVs = 64;  // value columns per block; 16 x 16 threads: ti = thread / 16 (rows), tj = thread % 16

template <int K>
struct KdaSmem {
    static constexpr int LDK = K + 4;       // rows of d_k floats
    static constexpr int LDC = kChunk + 4;  // rows of 64 floats
    static constexpr int kFloats = 64 * LDK * 3    // Ks, Qs, Gk
                                   + 64 * LDC * 4  // Vt, Tm, Pm, Au
                                   + K * LDC       // Ss
                                   + 64            // beta
                                   + 2 * K;        // G_n, exp(G_n)
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int K>
__global__ void __launch_bounds__(kThreads, 1) gdn_kda_chunk_kernel(const FwdArgs p) {
    using L = KdaSmem<K>;
    constexpr int LDK = L::LDK;
    constexpr int LDC = L::LDC;
    const int vs = blockIdx.x;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int V = p.d_v;
    const int H = p.H;
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ __align__(16) float sm[];
    float* Ks = sm;              // k; then exp(G) o k; then scratch of the inverse
    float* Qs = Ks + 64 * LDK;   // q; then exp(G) o q
    float* Gk = Qs + 64 * LDK;   // g; then G; then exp(G_n - G) o k
    float* Vt = Gk + 64 * LDK;   // v slice; then beta o (v - (exp(G) o K) S0)
    float* Tm = Vt + 64 * LDC;   // T = (I + A)^-1
    float* Pm = Tm + 64 * LDC;   // causal score P
    float* Au = Pm + 64 * LDC;   // A; then Delta
    float* Ss = Au + 64 * LDC;   // state slice, d_k x 64
    float* bs = Ss + K * LDC;
    float* Gn = bs + 64;         // G of the chunk's last row, per channel
    float* gn = Gn + K;          // exp(G_n)

    const bool with_out = p.out != nullptr;
    const long long slot_base = chunk_slot_base(p.cu_seqlens, n, p.T);
    const long long state_off = (static_cast<long long>(n) * H + h) * K * V + vs * kVs;
    for (int e = threadIdx.x; e < K * kVs / 4; e += blockDim.x) {
        const int i = e / (kVs / 4), j = (e % (kVs / 4)) * 4;
        st4(Ss + i * LDC + j, p.initial_state ? ld4(p.initial_state + state_off + static_cast<long long>(i) * V + j)
                                              : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    const long long row_base = static_cast<long long>(b) * p.T;
    const float scale = p.scale;

    for (int c0 = t0; c0 < t1; c0 += kChunk) {
        const int nv = min(kChunk, t1 - c0);
        const long long slot = (slot_base + (c0 - t0) / kChunk) * H + h;
        const float* tp = p.chunk_tp ? p.chunk_tp + slot * kKdaTpFloats : nullptr;
        __syncthreads();
        if (p.chunk_states) {
            // the state this chunk starts from, fp32 [slot][H][d_k][d_v]
            float* dst = p.chunk_states + slot * K * V + vs * kVs;
            for (int e = threadIdx.x; e < K * kVs / 4; e += blockDim.x) {
                const int i = e / (kVs / 4), j = (e % (kVs / 4)) * 4;
                st4(dst + static_cast<long long>(i) * V + j, ld4(Ss + i * LDC + j));
            }
        }
        load_rows_bf16<K, LDK>(p.k, row_base + c0, H, h, K, 0, nv, Ks);
        if (with_out) load_rows_bf16<K, LDK>(p.q, row_base + c0, H, h, K, 0, nv, Qs);
        load_rows_bf16<kVs, LDC>(p.v, row_base + c0, H, h, V, vs * kVs, nv, Vt);
        load_rows_f32<K, LDK>(p.g, row_base + c0, H, h, nv, Gk);
        if (tp) {
            load_tile64<LDC>(tp, Tm);
            if (with_out) load_tile64<LDC>(tp + 64 * 64, Pm);
        }
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            bs[r] = (r < nv) ? bf16_to_f32(p.beta[(row_base + c0 + r) * H + h]) : 0.f;
        }
        __syncthreads();
        // running sum of the gate per channel (rows >= nv add 0, so G_n is
        // the running sum at the chunk's last token)
        chunk_gate_cumsum<K, LDK>(Gk, Gn, gn);
        if (!tp) {
            gram_and_score<K, LDK, LDC>(Ks, Qs, Gk, bs, Au, Pm, with_out);
            __syncthreads();
        }
        // the decayed operands, in place: exp(G) o k, exp(G) o q, exp(G_n - G) o k
        for (int e = threadIdx.x; e < 64 * K; e += blockDim.x) {
            const int i = e / K, c = e % K;
            const float G = Gk[i * LDK + c];
            const float kv = Ks[i * LDK + c];
            const float eg = expf(G);
            Ks[i * LDK + c] = kv * eg;
            if (with_out) Qs[i * LDK + c] *= eg;
            Gk[i * LDK + c] = kv * expf(Gn[c] - G);
        }
        __syncthreads();
        {
            // R = beta o (V - (exp(G) o K) S0), in place over V
            float acc[4][4] = {};
            mm_rows<4, K>(acc, Ks, LDK, Ss, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = ti + 16 * r;
                float* vr = Vt + i * LDC + 4 * tj;
                const float4 v4 = ld4(vr);
                const float be = bs[i];
                st4(vr, make_float4(be * (v4.x - acc[r][0]), be * (v4.y - acc[r][1]), be * (v4.z - acc[r][2]),
                                    be * (v4.w - acc[r][3])));
            }
        }
        __syncthreads();
        if (!tp) chunk_unit_lower_inverse<LDC>(Au, Tm, Ks);
        {
            // Delta = T R
            float acc[4][4] = {};
            mm_rows<4, 64>(acc, Tm, LDC, Vt, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                st4(Au + (ti + 16 * r) * LDC + 4 * tj, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
        }
        __syncthreads();
        if (with_out) {
            // O = scale [(exp(G) o Q) S0 + P Delta]
            float acc[4][4] = {};
            mm_rows<4, K>(acc, Qs, LDK, Ss, LDC, ti, tj);
            mm_rows<4, 64>(acc, Pm, LDC, Au, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = ti + 16 * r;
                if (i < nv) {
                    const uint32_t lo = static_cast<uint32_t>(f32_to_bf16(scale * acc[r][0])) |
                                        (static_cast<uint32_t>(f32_to_bf16(scale * acc[r][1])) << 16);
                    const uint32_t hi = static_cast<uint32_t>(f32_to_bf16(scale * acc[r][2])) |
                                        (static_cast<uint32_t>(f32_to_bf16(scale * acc[r][3])) << 16);
                    *reinterpret_cast<uint2*>(p.out + ((row_base + c0 + i) * H + h) * static_cast<long long>(V) +
                                              vs * kVs + 4 * tj) = make_uint2(lo, hi);
                }
            }
            __syncthreads();
        }
        {
            // S1 = diag(exp(G_n)) S0 + (exp(G_n - G) o K)^T Delta
            float acc[K / 16][4] = {};
            mm_trans<K>(acc, Gk, LDK, Au, LDC, ti, tj);
#pragma unroll
            for (int m = 0; m < K / 64; ++m)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int a = 64 * m + 4 * ti + e;
                    float* sr = Ss + a * LDC + 4 * tj;
                    const float4 s4 = ld4(sr);
                    const float ga = gn[a];
                    st4(sr, make_float4(fmaf(ga, s4.x, acc[4 * m + e][0]), fmaf(ga, s4.y, acc[4 * m + e][1]),
                                        fmaf(ga, s4.z, acc[4 * m + e][2]), fmaf(ga, s4.w, acc[4 * m + e][3])));
                }
        }
    }
    __syncthreads();
    if (p.final_state) {
        for (int e = threadIdx.x; e < K * kVs / 4; e += blockDim.x) {
            const int i = e / (kVs / 4), j = (e % (kVs / 4)) * 4;
            st4(p.final_state + state_off + static_cast<long long>(i) * V + j, ld4(Ss + i * LDC + j));
        }
    }
}

// One 64-channel region of the decayed operands exp(G) o k, exp(G) o q,
// exp(G_n - G) o k of a chunk (rows of stride LDH, row 63 holding G_n) as
// bf16 hi/lo tiles of the tensor-core walk's operand block, and the region's
// exp(G_n).
template <int LDH>
__device__ __forceinline__ void write_decayed_region(uint8_t* blk, int region, const float* Ks, const float* Qs,
                                                     const float* Gk) {
    uint8_t* r = blk + region * 8192;
    for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
        const int i = e >> 3, ch = e & 7;
        float kg[8], qg[8], kt[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = 8 * ch + j;
            const float G = Gk[i * LDH + c];
            const float kv = Ks[i * LDH + c];
            const float eg = expf(G);
            kg[j] = kv * eg;
            qg[j] = Qs[i * LDH + c] * eg;
            kt[j] = kv * expf(Gk[63 * LDH + c] - G);
        }
        tc::store_split_chunk(r + kKdaBlkKG, r + kKdaBlkKG + 16384, i, ch, kg);
        tc::store_split_chunk(r + kKdaBlkQG, r + kKdaBlkQG + 16384, i, ch, qg);
        tc::store_split_chunk(r + kKdaBlkKt, r + kKdaBlkKt + 16384, i, ch, kt);
    }
    float* vec = reinterpret_cast<float*>(blk + kKdaBlkVec);
    if (threadIdx.x < 64) vec[64 * region + threadIdx.x] = expf(Gk[63 * LDH + threadIdx.x]);
}

// A 64 x 64 shared tile (row stride LD) as a bf16 hi/lo operand tile pair.
template <int LD>
__device__ __forceinline__ void write_split_tile64(uint8_t* hi, uint8_t* lo, const float* src) {
    for (int e = threadIdx.x; e < 64 * 8; e += blockDim.x) {
        const int i = e >> 3, ch = e & 7;
        tc::store_split_chunk(hi, lo, i, ch, src + i * LD + 8 * ch);
    }
}

// T = (I + A)^-1 and the causal score P of one chunk (one block per chunk,
// head and sequence), written to the per-chunk workspace as two row-major
// 64 x 64 fp32 tiles and / or (d_k = 128) with the decayed operands as the
// tensor-core walk's operand block.  The key channels are taken 64 at a time
// (the gram's register sums carry over, in the walk's own order, so both
// routes form the same T and P), which keeps the block at 105 KB of shared
// memory: two blocks share an SM.
struct KdaTpSmem {
    static constexpr int LDH = 64 + 4;      // rows of 64 channels
    static constexpr int LDC = kChunk + 4;
    static constexpr size_t kBytes = sizeof(float) * (64 * LDH * 3 + 64 * LDC * 3 + 64);
};

template <int K>
__global__ void __launch_bounds__(kThreads, 2) gdn_kda_tp_kernel(const KdaTpArgs p) {
    using L = KdaTpSmem;
    constexpr int LDH = L::LDH;
    constexpr int LDC = L::LDC;
    const int ci = blockIdx.x;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int H = p.H;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    const int c0 = t0 + ci * kChunk;
    if (c0 >= t1) return;
    const int nv = min(kChunk, t1 - c0);

    extern __shared__ __align__(16) float sm[];
    float* Ks = sm;             // k (64 channels); then scratch of the inverse
    float* Qs = Ks + 64 * LDH;  // q
    float* Gk = Qs + 64 * LDH;  // g; then G
    float* Au = Gk + 64 * LDH;  // A
    float* Pm = Au + 64 * LDC;  // P
    float* Tm = Pm + 64 * LDC;  // T
    float* bs = Tm + 64 * LDC;

    const long long row0 = static_cast<long long>(b) * p.T + c0;
    const long long slot = (chunk_slot_base(p.cu_seqlens, n, p.T) + ci) * H + h;
    uint8_t* blk = nullptr;
    if constexpr (K == 128) blk = p.tiles ? p.tiles + slot * kKdaBlkBytes : nullptr;
    if (threadIdx.x < 64) {
        const int r = threadIdx.x;
        bs[r] = (r < nv) ? bf16_to_f32(p.beta[(row0 + r) * H + h]) : 0.f;
    }
    float a[4][4] = {}, pp[4][4] = {};
    for (int hf = 0; hf < K / 64; ++hf) {
        if (hf) __syncthreads();
        load_rows_bf16<64, LDH>(p.k, row0, H, h, K, 64 * hf, nv, Ks);
        load_rows_bf16<64, LDH>(p.q, row0, H, h, K, 64 * hf, nv, Qs);
        load_rows_f32_cols<64, LDH>(p.g, row0, H, h, K, 64 * hf, nv, Gk);
        __syncthreads();
        chunk_gate_cumsum<64, LDH>(Gk, nullptr, nullptr);
        gram_accumulate<64, LDH>(Ks, Qs, Gk, a, pp);
        if (blk) write_decayed_region<LDH>(blk, hf, Ks, Qs, Gk);
    }
    gram_store<LDC>(a, pp, bs, Au, Pm, true);
    if (blk && threadIdx.x < 64) reinterpret_cast<float*>(blk + kKdaBlkVec)[K + threadIdx.x] = bs[threadIdx.x];
    __syncthreads();
    chunk_unit_lower_inverse<LDC>(Au, Tm, Ks);
    if (p.chunk_tp) {
        float* dst = p.chunk_tp + slot * kKdaTpFloats;
        store_tile64<LDC>(Tm, dst);
        store_tile64<LDC>(Pm, dst + 64 * 64);
    }
    if (blk) {
        write_split_tile64<LDC>(blk + kKdaBlkT, blk + kKdaBlkT + 8192, Tm);
        write_split_tile64<LDC>(blk + kKdaBlkP, blk + kKdaBlkP + 8192, Pm);
    }
}

template <int K>
cudaError_t launch_kda_tp_k(const KdaTpArgs& a, cudaStream_t stream) {
    const size_t smem = KdaTpSmem::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_tp_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_chunks, a.H, a.N);
    gdn_kda_tp_kernel<K><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_kda_chunk_k(const FwdArgs& a, cudaStream_t stream) {
    const size_t smem = KdaSmem<K>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_chunk_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_kda_chunk_kernel<K><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kda_chunk(const FwdArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_kda_chunk_k<64>(a, stream);
    return launch_kda_chunk_k<128>(a, stream);
}

cudaError_t launch_kda_tp(const KdaTpArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_kda_tp_k<64>(a, stream);
    return launch_kda_tp_k<128>(a, stream);
}

}  // namespace gdn

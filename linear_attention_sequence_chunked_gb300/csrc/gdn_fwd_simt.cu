// Chunked gated delta rule forward, fp32 CUDA-core version.
//
// One thread block per (value slice of 64 columns, head, sequence); it walks
// the sequence chunk by chunk (64 tokens) carrying its d_k x 64 slice of the
// state in shared memory.  The columns of the state evolve independently
// (column j only ever sees v_j in the "Research Sprint Day 1" GDN update
// loop), so slicing the value dimension is exact.
//
// Per chunk (see gdn_common.cuh for the algebra): running sum G of g, the
// decay-masked gram A and causal score P, T = (I + A)^-1 by blocked forward
// substitution, u = T diag(beta) V, w = T diag(beta exp G) K,
// Delta = u - w S0, O = scale [exp(G) o (Q S0) + P Delta],
// S1 = exp(G_n) S0 + K^T diag(exp(G_n - G_j)) Delta.
// Everything is fp32 in shared memory; inputs are widened from bf16 exactly.
//
// With `chunk_states` set the kernel also stores every chunk-start state
// (the backward pass recomputes them this way), and with `out == nullptr`
// it skips the output.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kVs = 64;  // value columns per block

template <int K>
struct FwdSmem {
    static constexpr int LDK = K + 1;
    static constexpr int LDC = kChunk + 1;
    static constexpr int kFloats = 64 * LDK * 3      // Ks, Qs, Ws
                                   + 64 * LDC * 4    // Vt, Tm, Pm, Au
                                   + K * LDC         // Ss
                                   + 6 * 64;         // gs, Gs, gam, bs, dec, spare
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// Load rows [c0, c0 + nv) of a (.., T, H, D) bf16 tensor for head h into a
// 64 x LD fp32 tile (columns [col0, col0 + W)), zero-filling rows >= nv.
template <int W, int LD>
__device__ __forceinline__ void load_tile_bf16(const uint16_t* __restrict__ src, long long row0,
                                               int H, int h, int D, int col0, int nv,
                                               float* dst) {
    constexpr int kVec = 8;
    constexpr int kPerRow = W / kVec;
    for (int e = threadIdx.x; e < 64 * kPerRow; e += blockDim.x) {
        const int r = e / kPerRow;
        const int c = (e % kPerRow) * kVec;
        float vals[kVec];
        if (r < nv) {
            const uint4 raw = *reinterpret_cast<const uint4*>(
                src + ((row0 + r) * H + h) * static_cast<long long>(D) + col0 + c);
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                vals[2 * m] = __uint_as_float(w4[m] << 16);
                vals[2 * m + 1] = __uint_as_float(w4[m] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int m = 0; m < kVec; ++m) vals[m] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < kVec; ++m) dst[r * LD + c + m] = vals[m];
    }
}

template <int K>
__global__ void __launch_bounds__(256) gdn_fwd_simt_kernel(FwdArgs p) {
    using L = FwdSmem<K>;
    constexpr int LDK = L::LDK;
    constexpr int LDC = L::LDC;
    const int vs = blockIdx.x;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int V = p.d_v;
    const int H = p.H;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ float sm[];
    float* Ks = sm;
    float* Qs = Ks + 64 * LDK;
    float* Ws = Qs + 64 * LDK;
    float* Vt = Ws + 64 * LDK;
    float* Tm = Vt + 64 * LDC;
    float* Pm = Tm + 64 * LDC;
    float* Au = Pm + 64 * LDC;
    float* Ss = Au + 64 * LDC;
    float* gs = Ss + K * LDC;
    float* Gs = gs + 64;
    float* gam = Gs + 64;
    float* bs = gam + 64;
    float* dec = bs + 64;

    const long long state_off = (static_cast<long long>(n) * H + h) * K * V + vs * kVs;
    for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
        const int i = e / kVs, j = e % kVs;
        Ss[i * LDC + j] = p.initial_state ? p.initial_state[state_off + static_cast<long long>(i) * V + j] : 0.f;
    }
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);
    const long long row_base = static_cast<long long>(b) * p.T;  // row of token 0 of batch b
    const float scale = p.scale;

    int ci = 0;
    for (int c0 = t0; c0 < t1; c0 += kChunk, ++ci) {
        const int nv = min(kChunk, t1 - c0);
        __syncthreads();
        if (p.chunk_states) {
            float* dst = p.chunk_states + ((slot0 + ci) * H + h) * static_cast<long long>(K) * V + vs * kVs;
            for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
                const int i = e / kVs, j = e % kVs;
                dst[static_cast<long long>(i) * V + j] = Ss[i * LDC + j];
            }
        }
        load_tile_bf16<K, LDK>(p.k, row_base + c0, H, h, K, 0, nv, Ks);
        if (p.out) load_tile_bf16<K, LDK>(p.q, row_base + c0, H, h, K, 0, nv, Qs);
        load_tile_bf16<kVs, LDC>(p.v, row_base + c0, H, h, V, vs * kVs, nv, Vt);
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            const long long idx = (row_base + c0 + r) * H + h;
            gs[r] = (r < nv) ? p.g[idx] : 0.f;
            bs[r] = (r < nv) ? bf16_to_f32(p.beta[idx]) : 0.f;
        }
        __syncthreads();
        chunk_cumsum(gs, Gs, gam);
        __syncthreads();
        if (threadIdx.x < 64) dec[threadIdx.x] = expf(Gs[63] - Gs[threadIdx.x]);
        // A = strict lower beta_i (k_i.k_j) exp(G_i - G_j)
        block_mm<64, 64, K, 4, 4>(
            [&](int i, int kk) { return Ks[i * LDK + kk]; },
            [&](int kk, int j) { return Ks[j * LDK + kk]; },
            [&](int i, int j, float acc) {
                Au[i * LDC + j] = (j < i) ? bs[i] * acc * expf(Gs[i] - Gs[j]) : 0.f;
            });
        if (p.out) {
            // P = (Q K^T) o M, diagonal included
            block_mm<64, 64, K, 4, 4>(
                [&](int i, int kk) { return Qs[i * LDK + kk]; },
                [&](int kk, int j) { return Ks[j * LDK + kk]; },
                [&](int i, int j, float acc) {
                    Pm[i * LDC + j] = (j <= i) ? acc * expf(Gs[i] - Gs[j]) : 0.f;
                });
        }
        __syncthreads();
        chunk_unit_lower_inverse<LDC>(Au, Tm, Ws);
        // u = T diag(beta) V  (into Au); w = T diag(beta gam) K (into Ws)
        block_mm<64, kVs, 64, 4, 4>(
            [&](int i, int jj) { return Tm[i * LDC + jj]; },
            [&](int jj, int c) { return bs[jj] * Vt[jj * LDC + c]; },
            [&](int i, int c, float acc) { Au[i * LDC + c] = acc; });
        block_mm<64, K, 64, 4, (K >= 128 ? 8 : 4)>(
            [&](int i, int jj) { return Tm[i * LDC + jj]; },
            [&](int jj, int d) { return bs[jj] * gam[jj] * Ks[jj * LDK + d]; },
            [&](int i, int d, float acc) { Ws[i * LDK + d] = acc; });
        __syncthreads();
        // Delta = u - w S0
        block_mm<64, kVs, K, 4, 4>(
            [&](int i, int d) { return Ws[i * LDK + d]; },
            [&](int d, int c) { return Ss[d * LDC + c]; },
            [&](int i, int c, float acc) { Au[i * LDC + c] -= acc; });
        __syncthreads();
        if (p.out) {
            // O = scale [gam o (Q S0) + P Delta]
            block_mm<64, kVs, K + 64, 4, 4>(
                [&](int i, int kk) { return kk < K ? gam[i] * Qs[i * LDK + kk] : Pm[i * LDC + kk - K]; },
                [&](int kk, int c) { return kk < K ? Ss[kk * LDC + c] : Au[(kk - K) * LDC + c]; },
                [&](int i, int c, float acc) {
                    if (i < nv)
                        p.out[((row_base + c0 + i) * H + h) * static_cast<long long>(V) + vs * kVs + c] =
                            f32_to_bf16(scale * acc);
                });
            __syncthreads();
        }
        // S1 = gam_n S0 + K^T diag(dec) Delta
        const float gC = gam[63];
        block_mm<K, kVs, 64, 4, 4>(
            [&](int a, int jj) { return Ks[jj * LDK + a]; },
            [&](int jj, int c) { return dec[jj] * Au[jj * LDC + c]; },
            [&](int a, int c, float acc) { Ss[a * LDC + c] = fmaf(gC, Ss[a * LDC + c], acc); });
    }
    __syncthreads();
    if (p.final_state) {
        for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
            const int i = e / kVs, j = e % kVs;
            p.final_state[state_off + static_cast<long long>(i) * V + j] = Ss[i * LDC + j];
        }
    }
}

template <int K>
cudaError_t launch_fwd_simt_k(const FwdArgs& a, cudaStream_t stream) {
    const size_t smem = FwdSmem<K>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_fwd_simt_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_fwd_simt_kernel<K><<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_fwd_simt_k<64>(a, stream);
    return launch_fwd_simt_k<128>(a, stream);
}

}  // namespace gdn

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
// memory (the value columns of the recurrence are independent).
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kVs = 64;        // value columns per block
constexpr int kThreads = 256;

template <int K>
struct KdaSmem {
    static constexpr int LDK = K + 1;
    static constexpr int LDC = kChunk + 1;
    static constexpr int kFloats = 64 * LDK * 3    // Ks, Qs, Gk
                                   + 64 * LDC * 4  // Vt, Tm, Pm, Au
                                   + K * LDC       // Ss
                                   + 64            // beta
                                   + 2 * K;        // G_n, exp(G_n)
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// Rows [row0, row0 + nv) of a (.., T, H, D) tensor for head h, columns
// [col0, col0 + W), into a 64 x LD fp32 tile; rows >= nv are zero.  Eight
// bf16 or four fp32 values per 16-byte load.
template <int W, int LD>
__device__ __forceinline__ void load_rows_bf16(const uint16_t* __restrict__ src, long long row0, int H,
                                               int h, int D, int col0, int nv, float* dst) {
    constexpr int kPerRow = W / 8;
    for (int e = threadIdx.x; e < 64 * kPerRow; e += blockDim.x) {
        const int r = e / kPerRow;
        const int c = (e % kPerRow) * 8;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (r < nv)
            raw = *reinterpret_cast<const uint4*>(src + ((row0 + r) * H + h) * static_cast<long long>(D) +
                                                  col0 + c);
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            dst[r * LD + c + 2 * m] = __uint_as_float(w4[m] << 16);
            dst[r * LD + c + 2 * m + 1] = __uint_as_float(w4[m] & 0xffff0000u);
        }
    }
}

template <int W, int LD>
__device__ __forceinline__ void load_rows_f32(const float* __restrict__ src, long long row0, int H, int h,
                                              int nv, float* dst) {
    constexpr int kPerRow = W / 4;
    for (int e = threadIdx.x; e < 64 * kPerRow; e += blockDim.x) {
        const int r = e / kPerRow;
        const int c = (e % kPerRow) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nv) x = *reinterpret_cast<const float4*>(src + ((row0 + r) * H + h) * static_cast<long long>(W) + c);
        dst[r * LD + c] = x.x;
        dst[r * LD + c + 1] = x.y;
        dst[r * LD + c + 2] = x.z;
        dst[r * LD + c + 3] = x.w;
    }
}

// A (strict lower, times beta_i) and, when `score`, P (lower with the
// diagonal) in one pass over the key channels, sharing each pair's decay
// factor.  Thread t owns rows i = t/16 + 16 r and columns j = t%16 + 16 s
// (r, s < 4); pairs with s > r lie above the diagonal for every thread and are
// skipped at compile time; pairs with s == r that lie above the diagonal take
// a zero exponent (their value is masked on store).
template <int K, int LDK, int LDC>
__device__ __forceinline__ void gram_and_score(const float* Ks, const float* Qs, const float* Gk,
                                               const float* bs, float* Au, float* Pm, bool score) {
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    float a[4][4], p[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) a[r][s] = p[r][s] = 0.f;
#pragma unroll 2
    for (int c = 0; c < K; ++c) {
        float gi[4], ki[4], qi[4], gj[4], kj[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            gi[r] = Gk[(ti + 16 * r) * LDK + c];
            ki[r] = Ks[(ti + 16 * r) * LDK + c];
            qi[r] = Qs[(ti + 16 * r) * LDK + c];
            gj[r] = Gk[(tj + 16 * r) * LDK + c];
            kj[r] = Ks[(tj + 16 * r) * LDK + c];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s <= r; ++s) {
                // s < r: j < i for every thread; s == r: j <= i only when tj <= ti
                const bool below = s < r || tj <= ti;
                const float ke = kj[s] * __expf(below ? gi[r] - gj[s] : 0.f);
                a[r][s] = fmaf(ki[r], ke, a[r][s]);
                p[r][s] = fmaf(qi[r], ke, p[r][s]);
            }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int i = ti + 16 * r, j = tj + 16 * s;
            Au[i * LDC + j] = (j < i) ? bs[i] * a[r][s] : 0.f;
            if (score) Pm[i * LDC + j] = (j <= i) ? p[r][s] : 0.f;
        }
}

template <int K>
__global__ void __launch_bounds__(kThreads) gdn_kda_chunk_kernel(const FwdArgs p) {
    using L = KdaSmem<K>;
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
    const long long state_off = (static_cast<long long>(n) * H + h) * K * V + vs * kVs;
    for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
        const int i = e / kVs, j = e % kVs;
        Ss[i * LDC + j] = p.initial_state ? p.initial_state[state_off + static_cast<long long>(i) * V + j] : 0.f;
    }
    const long long row_base = static_cast<long long>(b) * p.T;
    const float scale = p.scale;

    for (int c0 = t0; c0 < t1; c0 += kChunk) {
        const int nv = min(kChunk, t1 - c0);
        __syncthreads();
        load_rows_bf16<K, LDK>(p.k, row_base + c0, H, h, K, 0, nv, Ks);
        if (with_out) load_rows_bf16<K, LDK>(p.q, row_base + c0, H, h, K, 0, nv, Qs);
        load_rows_bf16<kVs, LDC>(p.v, row_base + c0, H, h, V, vs * kVs, nv, Vt);
        load_rows_f32<K, LDK>(p.g, row_base + c0, H, h, nv, Gk);
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            bs[r] = (r < nv) ? bf16_to_f32(p.beta[(row_base + c0 + r) * H + h]) : 0.f;
        }
        __syncthreads();
        // running sum of the gate per channel (rows >= nv add 0, so G_n is
        // the running sum at the chunk's last token)
        for (int c = threadIdx.x; c < K; c += blockDim.x) {
            float s = 0.f;
            for (int i = 0; i < 64; ++i) {
                s += Gk[i * LDK + c];
                Gk[i * LDK + c] = s;
            }
            Gn[c] = s;
            gn[c] = expf(s);
        }
        __syncthreads();
        gram_and_score<K, LDK, LDC>(Ks, Qs, Gk, bs, Au, Pm, with_out);
        __syncthreads();
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
        // R = beta o (V - (exp(G) o K) S0), in place over V
        block_mm<64, kVs, K, 4, 4>(
            [&](int i, int d) { return Ks[i * LDK + d]; },
            [&](int d, int c) { return Ss[d * LDC + c]; },
            [&](int i, int c, float acc) { Vt[i * LDC + c] = bs[i] * (Vt[i * LDC + c] - acc); });
        __syncthreads();
        chunk_unit_lower_inverse<LDC>(Au, Tm, Ks);
        // Delta = T R
        block_mm<64, kVs, 64, 4, 4>(
            [&](int i, int j) { return Tm[i * LDC + j]; },
            [&](int j, int c) { return Vt[j * LDC + c]; },
            [&](int i, int c, float acc) { Au[i * LDC + c] = acc; });
        __syncthreads();
        if (with_out) {
            // O = scale [(exp(G) o Q) S0 + P Delta]
            block_mm<64, kVs, K + 64, 4, 4>(
                [&](int i, int kk) { return kk < K ? Qs[i * LDK + kk] : Pm[i * LDC + kk - K]; },
                [&](int kk, int c) { return kk < K ? Ss[kk * LDC + c] : Au[(kk - K) * LDC + c]; },
                [&](int i, int c, float acc) {
                    if (i < nv)
                        p.out[((row_base + c0 + i) * H + h) * static_cast<long long>(V) + vs * kVs + c] =
                            f32_to_bf16(scale * acc);
                });
            __syncthreads();
        }
        // S1 = diag(exp(G_n)) S0 + (exp(G_n - G) o K)^T Delta
        block_mm<K, kVs, 64, 4, 4>(
            [&](int a, int j) { return Gk[j * LDK + a]; },
            [&](int j, int c) { return Au[j * LDC + c]; },
            [&](int a, int c, float acc) { Ss[a * LDC + c] = fmaf(gn[a], Ss[a * LDC + c], acc); });
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

}  // namespace gdn

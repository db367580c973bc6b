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
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kVs = 64;        // value columns per block
constexpr int kThreads = 256;  // 16 x 16: ti = thread / 16 (rows), tj = thread % 16 (4-column group)

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

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

__device__ __forceinline__ void fma4(float (&acc)[4], float a, float4 b) {
    acc[0] = fmaf(a, b.x, acc[0]);
    acc[1] = fmaf(a, b.y, acc[1]);
    acc[2] = fmaf(a, b.z, acc[2]);
    acc[3] = fmaf(a, b.w, acc[3]);
}

// Rows [row0, row0 + nv) of a (.., T, H, D) bf16 tensor for head h, columns
// [col0, col0 + W), widened into a 64 x LD fp32 tile; rows >= nv are zero.
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
        st4(dst + r * LD + c, make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                                          __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)));
        st4(dst + r * LD + c + 4, make_float4(__uint_as_float(raw.z << 16), __uint_as_float(raw.z & 0xffff0000u),
                                              __uint_as_float(raw.w << 16), __uint_as_float(raw.w & 0xffff0000u)));
    }
}

// The same for a (.., T, H, W) fp32 tensor (all W columns).
template <int W, int LD>
__device__ __forceinline__ void load_rows_f32(const float* __restrict__ src, long long row0, int H, int h,
                                              int nv, float* dst) {
    constexpr int kPerRow = W / 4;
    for (int e = threadIdx.x; e < 64 * kPerRow; e += blockDim.x) {
        const int r = e / kPerRow;
        const int c = (e % kPerRow) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nv) x = ld4(src + ((row0 + r) * H + h) * static_cast<long long>(W) + c);
        st4(dst + r * LD + c, x);
    }
}

// acc[r][.] += sum_{kk < KD} A[i_r][kk] B[kk][4 tj .. 4 tj + 3] for the rows
// i_r = ti + 16 r: A and B row-major, four reduction terms per step (one
// 16-byte read of each of the TM rows of A and of four rows of B).
template <int TM, int KD>
__device__ __forceinline__ void mm_rows(float (&acc)[TM][4], const float* A, int lda, const float* B, int ldb,
                                        int ti, int tj) {
#pragma unroll 2
    for (int k0 = 0; k0 < KD; k0 += 4) {
        float4 b[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) b[q] = ld4(B + (k0 + q) * ldb + 4 * tj);
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            const float4 a = ld4(A + (ti + 16 * r) * lda + k0);
            fma4(acc[r], a.x, b[0]);
            fma4(acc[r], a.y, b[1]);
            fma4(acc[r], a.z, b[2]);
            fma4(acc[r], a.w, b[3]);
        }
    }
}

// acc[4 m + e][.] += sum_{j < 64} At[j][64 m + 4 ti + e] B[j][4 tj .. 4 tj + 3]
// (m < K / 64, e < 4): the product with a transposed left operand, whose rows
// are read as 16-byte vectors along the output rows.
template <int K>
__device__ __forceinline__ void mm_trans(float (&acc)[K / 16][4], const float* At, int lda, const float* B,
                                         int ldb, int ti, int tj) {
#pragma unroll 4
    for (int j = 0; j < 64; ++j) {
        const float4 b = ld4(B + j * ldb + 4 * tj);
#pragma unroll
        for (int m = 0; m < K / 64; ++m) {
            const float4 a = ld4(At + j * lda + 64 * m + 4 * ti);
            fma4(acc[4 * m + 0], a.x, b);
            fma4(acc[4 * m + 1], a.y, b);
            fma4(acc[4 * m + 2], a.z, b);
            fma4(acc[4 * m + 3], a.w, b);
        }
    }
}

// A (strict lower, times beta_i) and, when `score`, P (lower with the
// diagonal) in one pass over the key channels, four channels per step,
// sharing each pair's decay factor.  Thread t owns rows i = ti + 16 r and
// columns j = tj + 16 s (r, s < 4): pairs with s > r lie above the diagonal
// for every thread and are skipped at compile time; pairs with s == r that lie
// above the diagonal take a zero exponent (their value is masked on store).
template <int K, int LDK, int LDC>
__device__ __forceinline__ void gram_and_score(const float* Ks, const float* Qs, const float* Gk,
                                               const float* bs, float* Au, float* Pm, bool score) {
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    float a[4][4], p[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) a[r][s] = p[r][s] = 0.f;
    for (int c = 0; c < K; c += 4) {
        float gi[4][4], ki[4][4], qi[4][4], gj[4][4], kj[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 g4 = ld4(Gk + (ti + 16 * r) * LDK + c);
            const float4 k4 = ld4(Ks + (ti + 16 * r) * LDK + c);
            const float4 q4 = ld4(Qs + (ti + 16 * r) * LDK + c);
            const float4 h4 = ld4(Gk + (tj + 16 * r) * LDK + c);
            const float4 l4 = ld4(Ks + (tj + 16 * r) * LDK + c);
            gi[r][0] = g4.x; gi[r][1] = g4.y; gi[r][2] = g4.z; gi[r][3] = g4.w;
            ki[r][0] = k4.x; ki[r][1] = k4.y; ki[r][2] = k4.z; ki[r][3] = k4.w;
            qi[r][0] = q4.x; qi[r][1] = q4.y; qi[r][2] = q4.z; qi[r][3] = q4.w;
            gj[r][0] = h4.x; gj[r][1] = h4.y; gj[r][2] = h4.z; gj[r][3] = h4.w;
            kj[r][0] = l4.x; kj[r][1] = l4.y; kj[r][2] = l4.z; kj[r][3] = l4.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s = 0; s <= r; ++s) {
                    // s < r: j < i for every thread; s == r: j <= i only when tj <= ti
                    const bool below = s < r || tj <= ti;
                    const float ke = kj[s][e] * __expf(below ? gi[r][e] - gj[s][e] : 0.f);
                    a[r][s] = fmaf(ki[r][e], ke, a[r][s]);
                    p[r][s] = fmaf(qi[r][e], ke, p[r][s]);
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
        chunk_unit_lower_inverse<LDC>(Au, Tm, Ks);
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

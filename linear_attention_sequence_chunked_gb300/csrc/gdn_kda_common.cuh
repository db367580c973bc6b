// Shared-memory tile helpers of the per-channel-gate (KDA) kernels: fp32 on
// the CUDA cores, 256 threads per block.  Tiles are row-major with rows
// padded to a multiple of four floats (4 banks mod 32), so operands are read
// as 16-byte vectors.
#pragma once

#include "gdn_common.cuh"

namespace gdn {
namespace kda {

constexpr int kThreads = 256;

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
// gram_accumulate adds KC channels (rows of stride LDK) to the register sums;
// channel blocks taken one after another give the same sums, in the same
// order, as one pass over all of them.
template <int KC, int LDK>
__device__ __forceinline__ void gram_accumulate(const float* Ks, const float* Qs, const float* Gk, float (&a)[4][4],
                                                float (&p)[4][4]) {
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    for (int c = 0; c < KC; c += 4) {
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
}

template <int LDC>
__device__ __forceinline__ void gram_store(const float (&a)[4][4], const float (&p)[4][4], const float* bs, float* Au,
                                           float* Pm, bool score) {
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int i = ti + 16 * r, j = tj + 16 * s;
            Au[i * LDC + j] = (j < i) ? bs[i] * a[r][s] : 0.f;
            if (score) Pm[i * LDC + j] = (j <= i) ? p[r][s] : 0.f;
        }
}

template <int K, int LDK, int LDC>
__device__ __forceinline__ void gram_and_score(const float* Ks, const float* Qs, const float* Gk,
                                               const float* bs, float* Au, float* Pm, bool score) {
    float a[4][4] = {}, p[4][4] = {};
    gram_accumulate<K, LDK>(Ks, Qs, Gk, a, p);
    gram_store<LDC>(a, p, bs, Au, Pm, score);
}

// Rows [row0, row0 + nv) of a (.., T, H, D) fp32 tensor for head h, columns
// [col0, col0 + W), into a 64 x LD tile; rows >= nv are zero.
template <int W, int LD>
__device__ __forceinline__ void load_rows_f32_cols(const float* __restrict__ src, long long row0, int H, int h,
                                                   int D, int col0, int nv, float* dst) {
    constexpr int kPerRow = W / 4;
    for (int e = threadIdx.x; e < 64 * kPerRow; e += blockDim.x) {
        const int r = e / kPerRow;
        const int c = (e % kPerRow) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nv) x = ld4(src + ((row0 + r) * H + h) * static_cast<long long>(D) + col0 + c);
        st4(dst + r * LD + c, x);
    }
}

// Generic register-blocked products.  The output has NCG groups of four
// columns; thread t owns column group tj = t % NCG and rows ti + RS r
// (r < TM) with ti = t / NCG and RS = 256 / NCG.

// acc[r][e] += sum_{kk < KD} A[ti + RS r][kk] B[kk][4 tj + e]
template <int TM, int KD, int RS>
__device__ __forceinline__ void mm_nn(float (&acc)[TM][4], const float* A, int lda, const float* B, int ldb, int ti,
                                      int tj) {
#pragma unroll 2
    for (int k0 = 0; k0 < KD; k0 += 4) {
        float4 b[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) b[q] = ld4(B + (k0 + q) * ldb + 4 * tj);
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            const float4 a = ld4(A + (ti + RS * r) * lda + k0);
            fma4(acc[r], a.x, b[0]);
            fma4(acc[r], a.y, b[1]);
            fma4(acc[r], a.z, b[2]);
            fma4(acc[r], a.w, b[3]);
        }
    }
}

// acc[r][e] += sum_{kk < KD} A[kk][ti + RS r] B[kk][4 tj + e]   (A^T B)
template <int TM, int KD, int RS>
__device__ __forceinline__ void mm_tn(float (&acc)[TM][4], const float* A, int lda, const float* B, int ldb, int ti,
                                      int tj) {
#pragma unroll 4
    for (int kk = 0; kk < KD; ++kk) {
        const float4 b = ld4(B + kk * ldb + 4 * tj);
#pragma unroll
        for (int r = 0; r < TM; ++r) fma4(acc[r], A[kk * lda + ti + RS * r], b);
    }
}

// acc[r][e] += sum_{kk < KD} A[ti + RS r][kk] B[tj + NCG e][kk]   (A B^T; the
// thread's output columns are tj + NCG e, so the four B rows a warp reads at
// once fall in different banks)
template <int TM, int KD, int RS, int NCG>
__device__ __forceinline__ void mm_nt(float (&acc)[TM][4], const float* A, int lda, const float* B, int ldb, int ti,
                                      int tj) {
#pragma unroll 2
    for (int k0 = 0; k0 < KD; k0 += 4) {
        float4 b[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) b[e] = ld4(B + (tj + NCG * e) * ldb + k0);
#pragma unroll
        for (int r = 0; r < TM; ++r) {
            const float4 a = ld4(A + (ti + RS * r) * lda + k0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[r][e] = fmaf(a.x, b[e].x, acc[r][e]);
                acc[r][e] = fmaf(a.y, b[e].y, acc[r][e]);
                acc[r][e] = fmaf(a.z, b[e].z, acc[r][e]);
                acc[r][e] = fmaf(a.w, b[e].w, acc[r][e]);
            }
        }
    }
}

// Running sum of the gate down the 64 rows of a chunk, per key channel, in
// place (rows past the chunk's end hold 0, so the last row is G_n); Gn and gn
// receive G_n and exp(G_n) when non-null.  Ends with a barrier.
template <int K, int LDK>
__device__ __forceinline__ void chunk_gate_cumsum(float* Gk, float* Gn, float* gn) {
    for (int c = threadIdx.x; c < K; c += blockDim.x) {
        float s = 0.f;
        for (int i = 0; i < 64; ++i) {
            s += Gk[i * LDK + c];
            Gk[i * LDK + c] = s;
        }
        if (Gn) Gn[c] = s;
        if (gn) gn[c] = expf(s);
    }
    __syncthreads();
}

// A 64 x 64 fp32 tile from global memory (row-major, 64 floats a row) into a
// shared tile of row stride LD.
template <int LD>
__device__ __forceinline__ void load_tile64(const float* __restrict__ src, float* dst) {
    for (int e = threadIdx.x; e < 64 * 16; e += blockDim.x) {
        const int r = e >> 4, c = (e & 15) * 4;
        st4(dst + r * LD + c, ld4(src + r * 64 + c));
    }
}

// The reverse: a shared 64 x 64 tile (row stride LD) to global memory.
template <int LD>
__device__ __forceinline__ void store_tile64(const float* src, float* __restrict__ dst) {
    for (int e = threadIdx.x; e < 64 * 16; e += blockDim.x) {
        const int r = e >> 4, c = (e & 15) * 4;
        st4(dst + r * 64 + c, ld4(src + r * LD + c));
    }
}

}  // namespace kda
}  // namespace gdn

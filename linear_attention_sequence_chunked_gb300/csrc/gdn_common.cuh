// Shared device helpers of the chunked gated delta rule kernels.
//
// Chunk algebra used throughout (one sequence, one head, chunk of n <= 64
// tokens, chunk-start state S0 of shape d_k x d_v):
//   G_i   = g_1 + ... + g_i           (log decay as a running sum; the
//                                      "Research Sprint Day 2 - Rooflines"
//                                      GDN pseudocode keeps g in log space)
//   A_ij  = beta_i (k_i . k_j) exp(G_i - G_j), j < i      (strictly lower)
//   T     = (I + A)^-1                (unit lower triangular)
//   w     = T diag(beta exp(G)) K,  u = T diag(beta) V
//   Delta = u - w S0                  (beta_i times the error v_i - v_old_i
//                                      of the page-1 "GDN update" loop)
//   O     = scale [diag(exp(G)) Q S0 + (Q K^T o M) Delta],
//           M_ij = exp(G_i - G_j) for j <= i (diagonal included)
//   S1    = exp(G_n) S0 + K^T diag(exp(G_n - G_j)) Delta
// The fla issue #1550 "Intermediate rounding diagnosis" names the
// intermediates (triangular inverse, causal QK score, write product w, WY
// value tensor u) whose bf16 rounding causes most of the error of earlier
// chunk kernels.  Here no computed intermediate is rounded to bf16 alone:
// the inverse, the decays and the state are fp32, and where the tensor-core
// kernels feed a computed quantity to an MMA it goes in as two bf16 parts
// (hi + lo, about 16 mantissa bits) with fp32 accumulation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kChunk = 64;

// Codes written to the per-device error word (match gdn_status values).
constexpr int kErrBadSeqlens = 4;
constexpr int kErrTimeout = 5;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Record a device-side error (first writer wins; later codes are dropped).
__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Token range [t0, t1) and batch row of sequence n.  Dense: b = n, [0, T).
// Packed: b = 0, [cu[n], cu[n+1]).  Returns false (after recording
// kErrBadSeqlens) when the offsets are malformed; the caller then exits.
__device__ __forceinline__ bool seq_range(const int32_t* cu, int n, int N, int T, int* err,
                                          int& b, int& t0, int& t1) {
    if (cu == nullptr) {
        b = n;
        t0 = 0;
        t1 = T;
        return true;
    }
    b = 0;
    t0 = cu[n];
    t1 = cu[n + 1];
    bool ok = (t0 >= 0) && (t1 >= t0) && (t1 <= T);
    if (n == 0) ok = ok && (t0 == 0);
    if (n == N - 1) ok = ok && (t1 == T);
    if (!ok) {
        if (threadIdx.x == 0) record_error(err, kErrBadSeqlens);
        return false;
    }
    return true;
}

// First chunk slot of sequence n in a per-chunk workspace array.  Dense:
// n * ceil(T/64).  Packed: floor(cu[n]/64) + n, which never overlaps the
// next sequence's slots and stays below floor(T/64) + N.
__device__ __forceinline__ long long chunk_slot_base(const int32_t* cu, int n, int T) {
    if (cu == nullptr) return static_cast<long long>(n) * ((T + kChunk - 1) / kChunk);
    return static_cast<long long>(cu[n] / kChunk) + n;
}

// T = (I + A)^-1 for a 64 x 64 strictly lower A (row stride LD), written to
// Tm (row stride LD, upper triangle zero).  Blocked forward substitution in
// fp32: the four 16 x 16 diagonal blocks are inverted column by column, then
// the off-diagonal blocks follow by distance from the diagonal:
//   T_IJ = -T_II * sum_{J <= L < I} A_IL T_LJ.
// X is a 64 x LD scratch.  Must be called by all threads of the block.
template <int LD>
__device__ __forceinline__ void chunk_unit_lower_inverse(const float* A, float* Tm, float* X) {
    // zero the strict upper triangle and set the diagonal blocks
    for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
        const int i = e / 64, j = e % 64;
        if ((i >> 4) != (j >> 4)) Tm[i * LD + j] = 0.f;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int blk = threadIdx.x >> 4;
        const int c = threadIdx.x & 15;  // column within the block
        const int o = blk * 16;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < i) acc = fmaf(-A[(o + i) * LD + o + j], col[j], acc);
            col[i] = (i < c) ? 0.f : acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(o + i) * LD + o + c] = col[i];
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
        const int nblk = 4 - dist;  // blocks (I, J) with I - J = dist
        // X_IJ = sum_{J <= L < I} A_IL T_LJ
        for (int e = threadIdx.x; e < nblk * 256; e += blockDim.x) {
            const int bi = e >> 8;
            const int r = (e >> 4) & 15, c = e & 15;
            const int I = bi + dist, J = bi;
            float acc = 0.f;
            for (int L = J; L < I; ++L)
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(A[(I * 16 + r) * LD + L * 16 + m], Tm[(L * 16 + m) * LD + J * 16 + c], acc);
            X[(I * 16 + r) * LD + J * 16 + c] = acc;
        }
        __syncthreads();
        // T_IJ = -T_II X_IJ
        for (int e = threadIdx.x; e < nblk * 256; e += blockDim.x) {
            const int bi = e >> 8;
            const int r = (e >> 4) & 15, c = e & 15;
            const int I = bi + dist, J = bi;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                acc = fmaf(Tm[(I * 16 + r) * LD + I * 16 + m], X[(I * 16 + m) * LD + J * 16 + c], acc);
            Tm[(I * 16 + r) * LD + J * 16 + c] = -acc;
        }
        __syncthreads();
    }
}

}  // namespace gdn

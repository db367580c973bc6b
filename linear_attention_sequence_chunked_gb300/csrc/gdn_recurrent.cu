// Gated delta rule, token-serial ("fused recurrent") forward: the decode path.
//
// Per (sequence, head), with the state S (d_k x d_v, fp32) carried across
// tokens, token t applies the update of the "Research Sprint Day 1" GDN loop
// (section "The GDN update"):
//   S <- exp(g_t) S;  v_old = S^T k_t;  S <- S + beta_t k_t (v_t - v_old)^T;
//   o_t = scale S^T q_t.
// The columns of S evolve independently (column j only sees v_t[j]), so the
// value dimension is split across CTAs.
//
// The per-channel-gate (KDA) variant of cuLA issue #126 takes g of shape
// (B, T, H, d_k): S <- diag(exp(g_t)) S decays each key row by its own factor;
// the rest of the update is unchanged.
//
// One CTA (128 threads) per (32-column value slice, head, sequence).  Thread
// (column jc = tid / 4, key block kb = tid % 4) holds rows kb*d_k/4 ..
// (kb+1)*d_k/4 - 1 of column jc in registers; the two sums over the key
// dimension per token are register FMAs over the thread's rows plus a sum
// over the 4 lanes of the column (shuffles).  Token t + 1's inputs are loaded
// while token t is processed.  The chunked kernels are the fast path for long
// sequences; this one serves decode (a few tokens per call) and is a second,
// independent GPU path that tests compare the chunked kernels with.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 128;
constexpr int kCols = 32;  // value columns per CTA

// One token's inputs as this thread needs them (gk: the per-channel gates of
// this thread's key rows, kPerChannel only).
template <int KB, bool kPerChannel>
struct TokenIn {
    uint4 k[KB / 8];
    uint4 q[KB / 8];
    float4 gk[kPerChannel ? KB / 4 : 1];
    float v, g, beta;
};

template <int KB, bool kPerChannel>
__device__ __forceinline__ void load_token(const RecurrentArgs& p, long long row, int h, int kb, int col,
                                           TokenIn<KB, kPerChannel>& in) {
    const long long kq = (row * p.H + h) * static_cast<long long>(p.d_k) + kb * KB;
    const uint4* ks = reinterpret_cast<const uint4*>(p.k + kq);
    const uint4* qs = reinterpret_cast<const uint4*>(p.q + kq);
#pragma unroll
    for (int c = 0; c < KB / 8; ++c) {
        in.k[c] = ks[c];
        in.q[c] = qs[c];
    }
    const long long gi = row * p.H + h;
    in.v = bf16_to_f32(p.v[gi * p.d_v + col]);
    if constexpr (kPerChannel) {
        const float4* gs = reinterpret_cast<const float4*>(p.g + kq);
#pragma unroll
        for (int c = 0; c < KB / 4; ++c) in.gk[c] = gs[c];
    } else {
        in.g = p.g[gi];
    }
    in.beta = bf16_to_f32(p.beta[gi]);
}

template <int KB>
__device__ __forceinline__ void unpack_rows(const uint4* raw, float* x) {
#pragma unroll
    for (int c = 0; c < KB / 8; ++c) {
        const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            x[8 * c + 2 * m] = __uint_as_float(w4[m] << 16);
            x[8 * c + 2 * m + 1] = __uint_as_float(w4[m] & 0xffff0000u);
        }
    }
}

// sum over the 4 lanes that hold one column
__device__ __forceinline__ float column_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

// x . y over KB values with four independent accumulators
template <int KB>
__device__ __forceinline__ float dot_rows(const float* x, const float* y) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < KB; ++i) a[i & 3] = fmaf(x[i], y[i], a[i & 3]);
    return (a[0] + a[1]) + (a[2] + a[3]);
}

template <int K, bool kPerChannel>
__global__ void __launch_bounds__(kThreads) gdn_recurrent_kernel(const RecurrentArgs p) {
    constexpr int KB = K / 4;  // key rows per thread
    const int vs = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x;
    const int jc = tid >> 2, kb = tid & 3;
    const int col = vs * kCols + jc;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    const long long row_base = static_cast<long long>(b) * p.T;
    const long long state_off = (static_cast<long long>(n) * p.H + h) * K * static_cast<long long>(p.d_v);

    float S[KB];
#pragma unroll
    for (int i = 0; i < KB; ++i)
        S[i] = p.initial_state ? p.initial_state[state_off + static_cast<long long>(kb * KB + i) * p.d_v + col] : 0.f;

    TokenIn<KB, kPerChannel> cur, nxt;
    if (t0 < t1) load_token<KB, kPerChannel>(p, row_base + t0, h, kb, col, cur);
    for (int t = t0; t < t1; ++t) {
        if (t + 1 < t1) load_token<KB, kPerChannel>(p, row_base + t + 1, h, kb, col, nxt);
        float kk[KB], qq[KB];
        unpack_rows<KB>(cur.k, kk);
        unpack_rows<KB>(cur.q, qq);
        // decay, read, write (the error, not the value), readout
        if constexpr (kPerChannel) {
#pragma unroll
            for (int c = 0; c < KB / 4; ++c) {
                S[4 * c] *= expf(cur.gk[c].x);
                S[4 * c + 1] *= expf(cur.gk[c].y);
                S[4 * c + 2] *= expf(cur.gk[c].z);
                S[4 * c + 3] *= expf(cur.gk[c].w);
            }
        } else {
            const float alpha = expf(cur.g);
#pragma unroll
            for (int i = 0; i < KB; ++i) S[i] *= alpha;
        }
        const float v_old = column_sum(dot_rows<KB>(S, kk));
        const float e = cur.beta * (cur.v - v_old);
#pragma unroll
        for (int i = 0; i < KB; ++i) S[i] = fmaf(kk[i], e, S[i]);
        const float o = p.scale * column_sum(dot_rows<KB>(S, qq));
        if (kb == 0) p.out[((row_base + t) * p.H + h) * static_cast<long long>(p.d_v) + col] = f32_to_bf16(o);
        cur = nxt;
    }
    if (p.final_state) {
#pragma unroll
        for (int i = 0; i < KB; ++i) p.final_state[state_off + static_cast<long long>(kb * KB + i) * p.d_v + col] = S[i];
    }
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t stream) {
    dim3 grid(a.d_v / kCols, a.H, a.N);
    if (a.per_channel_gate) {
        if (a.d_k == 64)
            gdn_recurrent_kernel<64, true><<<grid, kThreads, 0, stream>>>(a);
        else
            gdn_recurrent_kernel<128, true><<<grid, kThreads, 0, stream>>>(a);
    } else {
        if (a.d_k == 64)
            gdn_recurrent_kernel<64, false><<<grid, kThreads, 0, stream>>>(a);
        else
            gdn_recurrent_kernel<128, false><<<grid, kThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace gdn

// Prologue of the gated delta rule and its reverse mode: q/k L2
// normalisation and the two gates, from the raw per-token inputs.
//
// "Research Sprint Day 2 - Rooflines", GDN layer pseudocode, steps 4 and 5:
//   q_hat = q / |q|,  k_hat = k / |k|            (per (token, head) row, fp32)
//   beta  = c sigmoid(b),  c = 1, or 2 when negative eigenvalues are allowed
//   g     = -exp(A_log[h]) softplus(a + dt_bias[h])            (decay gate)
// and the bounded gate of fla issue #1550's CP2 test (lower bound -5):
//   g     = lower sigmoid(a + dt_bias[h]).
// The norm is taken as sqrt(|x|^2 + 1e-6) so that a zero row maps to zero.
//
// Reverse mode, with r = (|x|^2 + eps)^-1/2 and y = r x:
//   dx = r (dy - y (y . dy));   db = dbeta c s (1 - s), s = sigmoid(b);
//   decay:   da = -dg exp(A_log) sigmoid(u), u = a + dt_bias;
//            dA_log[h] = sum_rows dg g,  ddt_bias[h] = sum_rows da;
//   bounded: da = dg lower sigmoid(u) (1 - sigmoid(u)),  ddt_bias[h] = sum_rows da.
// One warp per (token, head) row: each lane holds d_k / 32 elements of q and
// of k, the row sums are warp shuffles.  The per-head sums run in a second
// kernel, one CTA per head in a fixed order, so they are deterministic.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// E bf16 values of a row segment <-> fp32
template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float* x) {
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = bf16_to_f32(p[e]);
}
template <int E>
__device__ __forceinline__ void store_bf16(uint16_t* p, const float* x) {
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = f32_to_bf16(x[e]);
}

template <int K>
__global__ void __launch_bounds__(32 * kRowsPerBlock) gdn_prologue_fwd_kernel(const PrologueArgs p) {
    constexpr int E = K / 32;
    const long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= static_cast<long long>(p.rows) * p.H) return;
    const int h = static_cast<int>(row % p.H);
    const long long off = row * K + lane * E;
    // q and k rows (a zero pointer skips the normalisation)
    for (int which = 0; which < 2; ++which) {
        const uint16_t* src = which ? p.k_raw : p.q_raw;
        uint16_t* dst = which ? p.k : p.q;
        if (!src) continue;
        float x[E];
        load_bf16<E>(src + off, x);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
        const float r = 1.0f / sqrtf(warp_sum(ss) + kNormEps);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] *= r;
        store_bf16<E>(dst + off, x);
    }
    if (lane == 0) {
        const float u = p.a[row] + (p.dt_bias ? p.dt_bias[h] : 0.f);
        const float g = p.gate_mode == 1 ? -expf(p.A_log[h]) * softplusf_(u) : p.lower * sigmoidf_(u);
        p.g[row] = g;
        p.beta[row] = f32_to_bf16(p.beta_scale * sigmoidf_(p.b[row]));
    }
}

template <int K>
__global__ void __launch_bounds__(32 * kRowsPerBlock) gdn_prologue_bwd_kernel(const PrologueArgs p) {
    constexpr int E = K / 32;
    const long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= static_cast<long long>(p.rows) * p.H) return;
    const int h = static_cast<int>(row % p.H);
    const long long off = row * K + lane * E;
    for (int which = 0; which < 2; ++which) {
        const uint16_t* src = which ? p.k_raw : p.q_raw;
        const uint16_t* dy_p = which ? p.dk : p.dq;
        uint16_t* dx_p = which ? p.dk_raw : p.dq_raw;
        if (!src) continue;
        float x[E], dy[E];
        load_bf16<E>(src + off, x);
        load_bf16<E>(dy_p + off, dy);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
        const float r = 1.0f / sqrtf(warp_sum(ss) + kNormEps);
        float yd = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) yd = fmaf(x[e] * r, dy[e], yd);
        yd = warp_sum(yd);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = r * (dy[e] - (x[e] * r) * yd);
        store_bf16<E>(dx_p + off, x);
    }
    if (lane == 0) {
        const float u = p.a[row] + (p.dt_bias ? p.dt_bias[h] : 0.f);
        const float su = sigmoidf_(u);
        const float dg = p.dg[row];
        p.da[row] = p.gate_mode == 1 ? -dg * expf(p.A_log[h]) * su : dg * p.lower * su * (1.f - su);
        const float sb = sigmoidf_(p.b[row]);
        p.db[row] = bf16_to_f32(p.dbeta[row]) * p.beta_scale * sb * (1.f - sb);
    }
}

// Per-head sums over every (token) row: ddt_bias[h] = sum da, dA_log[h] =
// sum dg g (decay gate).  One CTA per head, fixed order.
__global__ void __launch_bounds__(256) gdn_prologue_head_sums_kernel(const PrologueArgs p) {
    const int h = blockIdx.x;
    float s_da = 0.f, s_dA = 0.f;
    const float eA = p.gate_mode == 1 ? expf(p.A_log[h]) : 0.f;
    const float dtb = p.dt_bias ? p.dt_bias[h] : 0.f;
    for (long long t = threadIdx.x; t < p.rows; t += blockDim.x) {
        const long long row = t * p.H + h;
        s_da += p.da[row];
        if (p.gate_mode == 1) s_dA = fmaf(p.dg[row], -eA * softplusf_(p.a[row] + dtb), s_dA);
    }
    __shared__ float red[2][256];
    red[0][threadIdx.x] = s_da;
    red[1][threadIdx.x] = s_dA;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            red[0][threadIdx.x] += red[0][threadIdx.x + w];
            red[1][threadIdx.x] += red[1][threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (p.ddt_bias) p.ddt_bias[h] = red[0][0];
        if (p.dA_log && p.gate_mode == 1) p.dA_log[h] = red[1][0];
    }
}

}  // namespace

cudaError_t launch_prologue_fwd(const PrologueArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.rows) * a.H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    if (a.d_k == 64)
        gdn_prologue_fwd_kernel<64><<<grid, 32 * kRowsPerBlock, 0, stream>>>(a);
    else
        gdn_prologue_fwd_kernel<128><<<grid, 32 * kRowsPerBlock, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prologue_bwd(const PrologueArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.rows) * a.H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    if (a.d_k == 64)
        gdn_prologue_bwd_kernel<64><<<grid, 32 * kRowsPerBlock, 0, stream>>>(a);
    else
        gdn_prologue_bwd_kernel<128><<<grid, 32 * kRowsPerBlock, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ddt_bias || a.dA_log) gdn_prologue_head_sums_kernel<<<a.H, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

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
// Each warp takes kRowsPerWarp (token, head) rows, all their loads in flight
// before the row sums (warp shuffles); lane r computes row r's gates.  The
// per-head sums run in a second kernel, one CTA per head, in a fixed order,
// so they are deterministic.
#include <cooperative_groups.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerBlock = kWarps * kRowsPerWarp;
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// E (2 or 4) consecutive bf16 values of a row <-> fp32, one 4- or 8-byte access
template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float* x) {
    static_assert(E == 2 || E == 4, "segment");
    if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        x[0] = __uint_as_float(w.x << 16); x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16); x[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(w << 16); x[1] = __uint_as_float(w & 0xffff0000u);
    }
}
template <int E>
__device__ __forceinline__ void store_bf16(uint16_t* p, const float* x) {
    const uint32_t w0 = static_cast<uint32_t>(f32_to_bf16(x[0])) | (static_cast<uint32_t>(f32_to_bf16(x[1])) << 16);
    if constexpr (E == 4) {
        const uint32_t w1 = static_cast<uint32_t>(f32_to_bf16(x[2])) | (static_cast<uint32_t>(f32_to_bf16(x[3])) << 16);
        *reinterpret_cast<uint2*>(p) = make_uint2(w0, w1);
    } else {
        *reinterpret_cast<uint32_t*>(p) = w0;
    }
}

template <int K>
__global__ void __launch_bounds__(32 * kWarps) gdn_prologue_fwd_kernel(const PrologueArgs p) {
    constexpr int E = K / 32;
    constexpr int R = kRowsPerWarp;
    const long long nrows = static_cast<long long>(p.rows) * p.H;
    const long long row0 = (static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * R;
    const int lane = threadIdx.x & 31;
    if (row0 >= nrows) return;
    // q and k rows (a zero pointer skips the normalisation)
    for (int which = 0; which < 2; ++which) {
        const uint16_t* src = which ? p.k_raw : p.q_raw;
        uint16_t* dst = which ? p.k : p.q;
        if (!src) continue;
        float x[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (row0 + r < nrows) load_bf16<E>(src + (row0 + r) * K + lane * E, x[r]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= nrows) break;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(x[r][e], x[r][e], ss);
            const float inv = 1.0f / sqrtf(warp_sum(ss) + kNormEps);
#pragma unroll
            for (int e = 0; e < E; ++e) x[r][e] *= inv;
            store_bf16<E>(dst + (row0 + r) * K + lane * E, x[r]);
        }
    }
    if (lane < R && row0 + lane < nrows) {
        const long long row = row0 + lane;
        const int h = static_cast<int>(row % p.H);
        const float u = p.a[row] + (p.dt_bias ? p.dt_bias[h] : 0.f);
        const float g = p.gate_mode == 1 ? -expf(p.A_log[h]) * softplusf_(u) : p.lower * sigmoidf_(u);
        p.g[row] = g;
        p.beta[row] = f32_to_bf16(p.beta_scale * sigmoidf_(p.b[row]));
    }
}

template <int K>
__global__ void __launch_bounds__(32 * kWarps) gdn_prologue_bwd_kernel(const PrologueArgs p) {
    constexpr int E = K / 32;
    constexpr int R = kRowsPerWarp;
    const long long nrows = static_cast<long long>(p.rows) * p.H;
    const long long row0 = (static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * R;
    const int lane = threadIdx.x & 31;
    if (row0 >= nrows) return;
    for (int which = 0; which < 2; ++which) {
        const uint16_t* src = which ? p.k_raw : p.q_raw;
        const uint16_t* dy_p = which ? p.dk : p.dq;
        uint16_t* dx_p = which ? p.dk_raw : p.dq_raw;
        if (!src) continue;
        float x[R][E], dy[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r < nrows) {
                load_bf16<E>(src + (row0 + r) * K + lane * E, x[r]);
                load_bf16<E>(dy_p + (row0 + r) * K + lane * E, dy[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= nrows) break;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(x[r][e], x[r][e], ss);
            const float inv = 1.0f / sqrtf(warp_sum(ss) + kNormEps);
            float yd = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) yd = fmaf(x[r][e] * inv, dy[r][e], yd);
            yd = warp_sum(yd);
#pragma unroll
            for (int e = 0; e < E; ++e) x[r][e] = inv * (dy[r][e] - (x[r][e] * inv) * yd);
            store_bf16<E>(dx_p + (row0 + r) * K + lane * E, x[r]);
        }
    }
    if (lane < R && row0 + lane < nrows) {
        const long long row = row0 + lane;
        const int h = static_cast<int>(row % p.H);
        const float u = p.a[row] + (p.dt_bias ? p.dt_bias[h] : 0.f);
        const float su = sigmoidf_(u);
        const float dg = p.dg[row];
        p.da[row] = p.gate_mode == 1 ? -dg * expf(p.A_log[h]) * su : dg * p.lower * su * (1.f - su);
        const float sb = sigmoidf_(p.b[row]);
        p.db[row] = bf16_to_f32(p.dbeta[row]) * p.beta_scale * sb * (1.f - sb);
    }
}

// Per-head sums over every (token) row: ddt_bias[h] = sum da, dA_log[h] =
// sum dg g (decay gate).  One cluster of kSumSplit CTAs per head: CTA r sums
// the r-th contiguous part of the rows (each thread a fixed set of rows, four
// accumulators, four loads in flight, then a fixed-order tree), and CTA 0 adds
// the parts in rank order through distributed shared memory, so the result
// is deterministic.  (A head's rows are H floats apart: one CTA per head left
// most of the GPU idle on a strided read.)
constexpr int kSumThreads = 1024;
constexpr int kSumSplit = 8;
__global__ void __cluster_dims__(kSumSplit, 1, 1) __launch_bounds__(kSumThreads)
    gdn_prologue_head_sums_kernel(const PrologueArgs p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int h = blockIdx.x / kSumSplit;
    const int part = static_cast<int>(cluster.block_rank());
    const long long rows = p.rows;
    const long long r0 = rows * part / kSumSplit, r1 = rows * (part + 1) / kSumSplit;
    const bool decay = p.gate_mode == 1;
    const float eA = decay ? expf(p.A_log[h]) : 0.f;
    const float dtb = p.dt_bias ? p.dt_bias[h] : 0.f;
    float s_da[4] = {0.f, 0.f, 0.f, 0.f}, s_dA[4] = {0.f, 0.f, 0.f, 0.f};
    for (long long t0 = r0 + threadIdx.x; t0 < r1; t0 += 4LL * kSumThreads) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long t = t0 + static_cast<long long>(u) * kSumThreads;
            if (t < r1) {
                const long long row = t * p.H + h;
                s_da[u] += p.da[row];
                if (decay) s_dA[u] = fmaf(p.dg[row], -eA * softplusf_(p.a[row] + dtb), s_dA[u]);
            }
        }
    }
    __shared__ float red[2][kSumThreads];
    red[0][threadIdx.x] = (s_da[0] + s_da[1]) + (s_da[2] + s_da[3]);
    red[1][threadIdx.x] = (s_dA[0] + s_dA[1]) + (s_dA[2] + s_dA[3]);
    __syncthreads();
    for (int w = kSumThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            red[0][threadIdx.x] += red[0][threadIdx.x + w];
            red[1][threadIdx.x] += red[1][threadIdx.x + w];
        }
        __syncthreads();
    }
    cluster.sync();  // every part's sums are in its shared memory
    if (part == 0 && threadIdx.x == 0) {
        float da = 0.f, dA = 0.f;
        for (int r = 0; r < kSumSplit; ++r) {
            const float* rr = cluster.map_shared_rank(&red[0][0], r);
            da += rr[0];
            dA += rr[kSumThreads];
        }
        if (p.ddt_bias) p.ddt_bias[h] = da;
        if (p.dA_log && decay) p.dA_log[h] = dA;
    }
    cluster.sync();  // the parts' shared memory stays until CTA 0 has read it
}

}  // namespace

cudaError_t launch_prologue_fwd(const PrologueArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.rows) * a.H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    if (a.d_k == 64)
        gdn_prologue_fwd_kernel<64><<<grid, 32 * kWarps, 0, stream>>>(a);
    else
        gdn_prologue_fwd_kernel<128><<<grid, 32 * kWarps, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prologue_bwd(const PrologueArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.rows) * a.H;
    if (rows == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    if (a.d_k == 64)
        gdn_prologue_bwd_kernel<64><<<grid, 32 * kWarps, 0, stream>>>(a);
    else
        gdn_prologue_bwd_kernel<128><<<grid, 32 * kWarps, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.ddt_bias || a.dA_log) gdn_prologue_head_sums_kernel<<<a.H * kSumSplit, kSumThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

// Backward of the chunked per-channel-gate (KDA) gated delta rule, fp32 on the
// CUDA cores.
//
// Reverse mode of the chunk algebra of the forward (gdn_kda_chunk.cu), chunk
// by chunk from the last, with dS the gradient w.r.t. a chunk's end state.
// Per chunk (E_ijc = exp(G_ic - G_jc), KG = exp(G) o K, QG = exp(G) o Q,
// Kt = exp(G_n - G) o K, U = V - KG S0, R = beta o U, Delta = T R):
//   dDelta = scale P^T dO + Kt dS          dR = T^T dDelta        dv = beta o dR
//   dS0    = scale QG^T dO + diag(exp(G_n)) dS - KG^T (beta o dR)
//   dP     = scale dO Delta^T (j <= i)     dA = -dR Delta^T (j < i)
//   dQG    = scale dO S0^T                 dKG = -(beta o dR) S0^T
//   dKt    = Delta dS^T                    X = dKt o Kt
//   dq_i   = dQG_i o exp(G_i) + sum_{j<=i} dP_ij k_j o E_ij
//   dk_i   = dKt_i o exp(G_n - G_i) + dKG_i o exp(G_i)
//            + beta_i sum_{j<i} dA_ij k_j o E_ij
//            + sum_{j>i} beta_j dA_ji k_j o E_ji + sum_{j>=i} dP_ji q_j o E_ji
//   dbeta_i = sum_c dR_ic U_ic + sum_c k_ic sum_{j<i} dA_ij k_jc E_ijc
//   dG     = dKG o KG + dQG o QG - X + (the pair terms of the decayed sums)
//            + [last row] exp(G_n) o rowsum(dS o S0) + colsum X
//   dg     = reverse running sum of dG down the chunk, per key channel.
//
// The gradient of the state chain is linear in dO and dS and needs neither
// V nor S, so it runs as its own walk:
//   gdn_kda_bwd_chain_kernel: one block per (64 value columns, head,
//     sequence), chunks in reverse, records each chunk's dS and ends with the
//     gradient w.r.t. the initial state;
//   gdn_kda_bwd_local_kernel: one block per (chunk, head, sequence), with the
//     chunk's start state (from the forward walk) and dS, loops over the value
//     columns in slices of 32, summing dA, dP and the three d_k-wide products
//     over the slices, then evaluates the decayed pair sums once per chunk.
// Both read T and P from the per-chunk workspace (gdn_kda_tp_kernel).  Every
// sum is taken in a fixed order, so results are bitwise reproducible.
#include "gdn_common.cuh"
#include "gdn_kda_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

using namespace kda;

// ---- the reverse state-gradient walk ----

constexpr int kChainVs = 64;  // value columns per block

template <int K>
struct KdaChainSmem {
    static constexpr int LDK = K + 4;
    static constexpr int LDC = kChunk + 4;
    static constexpr size_t kBytes = sizeof(float) * (64 * LDK * 3      // Ks, Qs, Gk
                                                      + 64 * LDC * 5    // Tm, Pm, Ot, Et, Rt
                                                      + K * LDC         // dS
                                                      + 64 + 2 * K);    // beta, G_n, exp(G_n)
};

template <int K>
__global__ void __launch_bounds__(kThreads, 1) gdn_kda_bwd_chain_kernel(const KdaBwdArgs p) {
    using L = KdaChainSmem<K>;
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
    float* Ks = sm;              // k; then exp(G) o k
    float* Qs = Ks + 64 * LDK;   // q; then exp(G) o q
    float* Gk = Qs + 64 * LDK;   // g; then G; then exp(G_n - G) o k
    float* Tm = Gk + 64 * LDK;   // T
    float* Pm = Tm + 64 * LDC;   // P
    float* Ot = Pm + 64 * LDC;   // dO slice
    float* Et = Ot + 64 * LDC;   // dDelta
    float* Rt = Et + 64 * LDC;   // beta o dR
    float* Ss = Rt + 64 * LDC;   // dS slice, d_k x 64
    float* bs = Ss + K * LDC;
    float* Gn = bs + 64;
    float* gn = Gn + K;

    const long long state_off = (static_cast<long long>(n) * H + h) * K * V + vs * kChainVs;
    for (int e = threadIdx.x; e < K * kChainVs / 4; e += blockDim.x) {
        const int i = e / (kChainVs / 4), j = (e % (kChainVs / 4)) * 4;
        st4(Ss + i * LDC + j, p.d_final_state ? ld4(p.d_final_state + state_off + static_cast<long long>(i) * V + j)
                                              : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    const long long row_base = static_cast<long long>(b) * p.T;
    const long long slot_base = chunk_slot_base(p.cu_seqlens, n, p.T);
    const float scale = p.scale;
    const int nch = (t1 - t0 + kChunk - 1) / kChunk;

    for (int ci = nch - 1; ci >= 0; --ci) {
        const int c0 = t0 + ci * kChunk;
        const int nv = min(kChunk, t1 - c0);
        const long long slot = (slot_base + ci) * H + h;
        __syncthreads();
        {
            // the gradient w.r.t. this chunk's end state
            float* dst = p.chunk_dstates + slot * K * V + vs * kChainVs;
            for (int e = threadIdx.x; e < K * kChainVs / 4; e += blockDim.x) {
                const int i = e / (kChainVs / 4), j = (e % (kChainVs / 4)) * 4;
                st4(dst + static_cast<long long>(i) * V + j, ld4(Ss + i * LDC + j));
            }
        }
        load_rows_bf16<K, LDK>(p.k, row_base + c0, H, h, K, 0, nv, Ks);
        load_rows_bf16<K, LDK>(p.q, row_base + c0, H, h, K, 0, nv, Qs);
        load_rows_f32<K, LDK>(p.g, row_base + c0, H, h, nv, Gk);
        load_rows_bf16<kChainVs, LDC>(p.d_out, row_base + c0, H, h, V, vs * kChainVs, nv, Ot);
        load_tile64<LDC>(p.chunk_tp + slot * kKdaTpFloats, Tm);
        load_tile64<LDC>(p.chunk_tp + slot * kKdaTpFloats + 64 * 64, Pm);
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            bs[r] = (r < nv) ? bf16_to_f32(p.beta[(row_base + c0 + r) * H + h]) : 0.f;
        }
        __syncthreads();
        chunk_gate_cumsum<K, LDK>(Gk, Gn, gn);
        for (int e = threadIdx.x; e < 64 * K; e += blockDim.x) {
            const int i = e / K, c = e % K;
            const float G = Gk[i * LDK + c];
            const float kv = Ks[i * LDK + c];
            const float eg = expf(G);
            Ks[i * LDK + c] = kv * eg;
            Qs[i * LDK + c] *= eg;
            Gk[i * LDK + c] = kv * expf(Gn[c] - G);
        }
        __syncthreads();
        {
            // dDelta = scale P^T dO + Kt dS
            float a[4][4] = {}, s[4][4] = {};
            mm_tn<4, 64, 16>(a, Pm, LDC, Ot, LDC, ti, tj);
            mm_nn<4, K, 16>(s, Gk, LDK, Ss, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r)
                st4(Et + (ti + 16 * r) * LDC + 4 * tj,
                    make_float4(fmaf(scale, a[r][0], s[r][0]), fmaf(scale, a[r][1], s[r][1]),
                                fmaf(scale, a[r][2], s[r][2]), fmaf(scale, a[r][3], s[r][3])));
        }
        __syncthreads();
        {
            // beta o dR, dR = T^T dDelta
            float a[4][4] = {};
            mm_tn<4, 64, 16>(a, Tm, LDC, Et, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float be = bs[ti + 16 * r];
                st4(Rt + (ti + 16 * r) * LDC + 4 * tj,
                    make_float4(be * a[r][0], be * a[r][1], be * a[r][2], be * a[r][3]));
            }
        }
        __syncthreads();
        {
            // dS0 = scale QG^T dO + diag(exp(G_n)) dS - KG^T (beta o dR), in place
            float a[K / 16][4] = {}, s[K / 16][4] = {};
            mm_tn<K / 16, 64, 16>(a, Qs, LDK, Ot, LDC, ti, tj);
            mm_tn<K / 16, 64, 16>(s, Ks, LDK, Rt, LDC, ti, tj);
#pragma unroll
            for (int r = 0; r < K / 16; ++r) {
                const int row = ti + 16 * r;
                float* sr = Ss + row * LDC + 4 * tj;
                const float4 d4 = ld4(sr);
                const float ga = gn[row];
                st4(sr, make_float4(fmaf(scale, a[r][0], fmaf(ga, d4.x, -s[r][0])),
                                    fmaf(scale, a[r][1], fmaf(ga, d4.y, -s[r][1])),
                                    fmaf(scale, a[r][2], fmaf(ga, d4.z, -s[r][2])),
                                    fmaf(scale, a[r][3], fmaf(ga, d4.w, -s[r][3]))));
            }
        }
    }
    __syncthreads();
    if (p.d_initial_state) {
        for (int e = threadIdx.x; e < K * kChainVs / 4; e += blockDim.x) {
            const int i = e / (kChainVs / 4), j = (e % (kChainVs / 4)) * 4;
            st4(p.d_initial_state + state_off + static_cast<long long>(i) * V + j, ld4(Ss + i * LDC + j));
        }
    }
}

// ---- the chunk-parallel local gradients ----

constexpr int kLocalVs = 32;  // value columns per slice

template <int K>
struct KdaLocalSmem {
    static constexpr int LDK = K + 4;
    static constexpr int LDC = kChunk + 4;
    static constexpr int LDV = kLocalVs + 4;
    static constexpr int NCGK = K / 4;          // column groups of the d_k-wide products
    static constexpr int RSK = kThreads / NCGK; // their row stride
    static constexpr int kSlice = 64 * LDV * 5 + K * LDV * 2;
    static_assert(kSlice >= 64 * LDK, "the slice region holds G at the start and the end");
    static_assert(2 * 64 * LDC >= 64 * LDK, "T and P make room for the dG tile");
    static constexpr size_t kBytes = sizeof(float) * (64 * LDK * 2        // Ks, Qs
                                                      + 64 * LDC * 4      // Tm, Pm, dA, dP
                                                      + kSlice            // slice tiles / G
                                                      + 64 * 2 + K * 3    // beta, dbeta part, G_n, exp(G_n), gsum
                                                      + RSK * K);         // column-sum parts of X
};

template <int K>
__global__ void __launch_bounds__(kThreads, 1) gdn_kda_bwd_local_kernel(const KdaBwdArgs p) {
    using L = KdaLocalSmem<K>;
    constexpr int LDK = L::LDK;
    constexpr int LDC = L::LDC;
    constexpr int LDV = L::LDV;
    constexpr int NCGK = L::NCGK;
    constexpr int RSK = L::RSK;
    constexpr int TMK = 64 / RSK;
    const int ci = blockIdx.x;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int V = p.d_v;
    const int H = p.H;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;
    const int c0 = t0 + ci * kChunk;
    if (c0 >= t1) return;
    const int nv = min(kChunk, t1 - c0);
    const long long slot = (chunk_slot_base(p.cu_seqlens, n, p.T) + ci) * H + h;
    const long long row0 = static_cast<long long>(b) * p.T + c0;
    const float scale = p.scale;

    // thread layouts: 64 x 32 slice tiles, 64 x 64 pair tiles, 64 x d_k tiles
    const int vi = threadIdx.x >> 3, vj = threadIdx.x & 7;
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    const int ki = threadIdx.x / NCGK, kj = threadIdx.x % NCGK;

    extern __shared__ __align__(16) float sm[];
    float* Ks = sm;                // k; exp(G) o k in the slices; k again at the end
    float* Qs = Ks + 64 * LDK;     // exp(G_n - G) o k in the slices; q at the end
    float* Tm = Qs + 64 * LDK;     // T
    float* Pm = Tm + 64 * LDC;     // P
    float* dA = Pm + 64 * LDC;     // dA, summed over the slices (strict lower part used)
    float* dP = dA + 64 * LDC;     // dP, summed over the slices (lower part used)
    float* Sl = dP + 64 * LDC;     // slice region
    float* Vt = Sl;                // v slice; then U
    float* Rt = Vt + 64 * LDV;     // R; then dR
    float* Dt = Rt + 64 * LDV;     // Delta
    float* Ot = Dt + 64 * LDV;     // dO slice
    float* Et = Ot + 64 * LDV;     // dDelta
    float* S0 = Et + 64 * LDV;     // start state slice, d_k x 32
    float* dS = S0 + K * LDV;      // end-state gradient slice, d_k x 32
    float* Gs = Sl;                // G, outside the slice loop
    float* dGt = Tm;               // dG before the running sum, at the end
    float* bs = Sl + L::kSlice;
    float* dbs = bs + 64;          // sum_c dR_ic U_ic over the slices
    float* Gn = dbs + 64;
    float* gn = Gn + K;
    float* gsum = gn + K;          // sum_j dS_cj S0_cj over the slices
    float* xs = gsum + K;          // [RSK][K] column-sum parts of X

    // ---- chunk set-up: G and the decayed key operands of the slice products
    load_rows_bf16<K, LDK>(p.k, row0, H, h, K, 0, nv, Ks);
    load_rows_f32<K, LDK>(p.g, row0, H, h, nv, Gs);
    load_tile64<LDC>(p.chunk_tp + slot * kKdaTpFloats, Tm);
    load_tile64<LDC>(p.chunk_tp + slot * kKdaTpFloats + 64 * 64, Pm);
    for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
        dA[(e >> 6) * LDC + (e & 63)] = 0.f;
        dP[(e >> 6) * LDC + (e & 63)] = 0.f;
    }
    if (threadIdx.x < 64) {
        const int r = threadIdx.x;
        bs[r] = (r < nv) ? bf16_to_f32(p.beta[(row0 + r) * H + h]) : 0.f;
        dbs[r] = 0.f;
    }
    for (int c = threadIdx.x; c < K; c += blockDim.x) gsum[c] = 0.f;
    __syncthreads();
    chunk_gate_cumsum<K, LDK>(Gs, Gn, gn);
    for (int e = threadIdx.x; e < 64 * K; e += blockDim.x) {
        const int i = e / K, c = e % K;
        const float G = Gs[i * LDK + c];
        const float kv = Ks[i * LDK + c];
        Qs[i * LDK + c] = kv * expf(Gn[c] - G);
        Ks[i * LDK + c] = kv * expf(G);
    }
    __syncthreads();

    // sums over the value slices of dO S0^T, Delta dS^T and dR S0^T (64 x d_k)
    float aq[TMK][4] = {}, akt[TMK][4] = {}, ar[TMK][4] = {};
    const float* st0 = p.chunk_states + slot * K * V;
    const float* dst1 = p.chunk_dstates + slot * K * V;
    for (int col0 = 0; col0 < V; col0 += kLocalVs) {
        load_rows_bf16<kLocalVs, LDV>(p.v, row0, H, h, V, col0, nv, Vt);
        load_rows_bf16<kLocalVs, LDV>(p.d_out, row0, H, h, V, col0, nv, Ot);
        for (int e = threadIdx.x; e < K * kLocalVs / 4; e += blockDim.x) {
            const int a = e / (kLocalVs / 4), j = (e % (kLocalVs / 4)) * 4;
            st4(S0 + a * LDV + j, ld4(st0 + static_cast<long long>(a) * V + col0 + j));
            st4(dS + a * LDV + j, ld4(dst1 + static_cast<long long>(a) * V + col0 + j));
        }
        __syncthreads();
        {
            // U = V - KG S0, R = beta o U
            float acc[2][4] = {};
            mm_nn<2, K, 32>(acc, Ks, LDK, S0, LDV, vi, vj);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = vi + 32 * r;
                float* vr = Vt + i * LDV + 4 * vj;
                const float4 v4 = ld4(vr);
                const float4 u = make_float4(v4.x - acc[r][0], v4.y - acc[r][1], v4.z - acc[r][2], v4.w - acc[r][3]);
                const float be = bs[i];
                st4(vr, u);
                st4(Rt + i * LDV + 4 * vj, make_float4(be * u.x, be * u.y, be * u.z, be * u.w));
            }
        }
        __syncthreads();
        {
            // Delta = T R
            float acc[2][4] = {};
            mm_nn<2, 64, 32>(acc, Tm, LDC, Rt, LDV, vi, vj);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                st4(Dt + (vi + 32 * r) * LDV + 4 * vj, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
        }
        __syncthreads();
        {
            // dDelta = scale P^T dO + Kt dS
            float a[2][4] = {}, s[2][4] = {};
            mm_tn<2, 64, 32>(a, Pm, LDC, Ot, LDV, vi, vj);
            mm_nn<2, K, 32>(s, Qs, LDK, dS, LDV, vi, vj);
#pragma unroll
            for (int r = 0; r < 2; ++r)
                st4(Et + (vi + 32 * r) * LDV + 4 * vj,
                    make_float4(fmaf(scale, a[r][0], s[r][0]), fmaf(scale, a[r][1], s[r][1]),
                                fmaf(scale, a[r][2], s[r][2]), fmaf(scale, a[r][3], s[r][3])));
        }
        __syncthreads();
        {
            // dR = T^T dDelta; dv = beta o dR; dbeta += rowsum(dR o U)
            float acc[2][4] = {};
            mm_tn<2, 64, 32>(acc, Tm, LDC, Et, LDV, vi, vj);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = vi + 32 * r;
                st4(Rt + i * LDV + 4 * vj, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
                const float4 u = ld4(Vt + i * LDV + 4 * vj);
                float part = acc[r][0] * u.x + acc[r][1] * u.y + acc[r][2] * u.z + acc[r][3] * u.w;
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (vj == 0) dbs[i] += part;
                if (i < nv) {
                    const float be = bs[i];
                    const uint32_t lo = static_cast<uint32_t>(f32_to_bf16(be * acc[r][0])) |
                                        (static_cast<uint32_t>(f32_to_bf16(be * acc[r][1])) << 16);
                    const uint32_t hi = static_cast<uint32_t>(f32_to_bf16(be * acc[r][2])) |
                                        (static_cast<uint32_t>(f32_to_bf16(be * acc[r][3])) << 16);
                    *reinterpret_cast<uint2*>(p.dv + ((row0 + i) * H + h) * static_cast<long long>(V) + col0 +
                                              4 * vj) = make_uint2(lo, hi);
                }
            }
        }
        __syncthreads();
        {
            // dA -= dR Delta^T, dP += scale dO Delta^T (each thread its own entries)
            float a[4][4] = {}, q[4][4] = {};
            mm_nt<4, kLocalVs, 16, 16>(a, Rt, LDV, Dt, LDV, ti, tj);
            mm_nt<4, kLocalVs, 16, 16>(q, Ot, LDV, Dt, LDV, ti, tj);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = ti + 16 * r, j = tj + 16 * e;
                    dA[i * LDC + j] -= a[r][e];
                    dP[i * LDC + j] = fmaf(scale, q[r][e], dP[i * LDC + j]);
                }
        }
        mm_nt<TMK, kLocalVs, RSK, NCGK>(aq, Ot, LDV, S0, LDV, ki, kj);
        mm_nt<TMK, kLocalVs, RSK, NCGK>(ar, Rt, LDV, S0, LDV, ki, kj);
        mm_nt<TMK, kLocalVs, RSK, NCGK>(akt, Dt, LDV, dS, LDV, ki, kj);
        for (int c = threadIdx.x; c < K; c += blockDim.x) {
            float s = 0.f;
#pragma unroll 8
            for (int j = 0; j < kLocalVs; ++j) s = fmaf(dS[c * LDV + j], S0[c * LDV + j], s);
            gsum[c] += s;
        }
        __syncthreads();
    }

    // ---- end of chunk: raw k, q and G again
    load_rows_bf16<K, LDK>(p.k, row0, H, h, K, 0, nv, Ks);
    load_rows_bf16<K, LDK>(p.q, row0, H, h, K, 0, nv, Qs);
    load_rows_f32<K, LDK>(p.g, row0, H, h, nv, Gs);
    __syncthreads();
    chunk_gate_cumsum<K, LDK>(Gs, Gn, gn);

    // the slice products in their final form: dq, dk, dG (registers) and X
    float dq[TMK][4], dk[TMK][4], dg[TMK][4];
    {
        float xp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < TMK; ++r) {
            const int i = ki + RSK * r;
            const float be = bs[i];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = kj + NCGK * e;
                const float G = Gs[i * LDK + c];
                const float kv = Ks[i * LDK + c];
                const float qv = Qs[i * LDK + c];
                const float eg = expf(G);
                const float dn = expf(Gn[c] - G);
                const float dqg = scale * aq[r][e];
                const float dkg = -be * ar[r][e];
                const float x = akt[r][e] * kv * dn;
                xp[e] += x;
                dq[r][e] = dqg * eg;
                dk[r][e] = fmaf(akt[r][e], dn, dkg * eg);
                dg[r][e] = fmaf(dkg * kv, eg, fmaf(dqg * qv, eg, -x));
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) xs[ki * K + kj + NCGK * e] = xp[e];
    }

    // the decayed pair sums, row side: for i, over j <= i,
    //   u1_ic = sum_{j<i} dA_ij k_jc E_ijc,  u2_ic = sum_{j<=i} dP_ij k_jc E_ijc
    float dbp[TMK];
#pragma unroll
    for (int r0 = 0; r0 < TMK; r0 += 4) {
        float u1[4][4] = {}, u2[4][4] = {}, gi[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) gi[r][e] = Gs[(ki + RSK * (r0 + r)) * LDK + kj + NCGK * e];
        const int imax = ki + RSK * (r0 + 3);
        for (int j = 0; j <= imax; ++j) {
            float kj4[4], gj4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kj4[e] = Ks[j * LDK + kj + NCGK * e];
                gj4[e] = Gs[j * LDK + kj + NCGK * e];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = ki + RSK * (r0 + r);
                if (j <= i) {
                    const float a = (j < i) ? dA[i * LDC + j] : 0.f;
                    const float q = dP[i * LDC + j];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float ke = kj4[e] * __expf(gi[r][e] - gj4[e]);
                        u1[r][e] = fmaf(a, ke, u1[r][e]);
                        u2[r][e] = fmaf(q, ke, u2[r][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = ki + RSK * (r0 + r);
            const float be = bs[i];
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = kj + NCGK * e;
                const float kv = Ks[i * LDK + c];
                const float qv = Qs[i * LDK + c];
                dq[r0 + r][e] += u2[r][e];
                dk[r0 + r][e] = fmaf(be, u1[r][e], dk[r0 + r][e]);
                dg[r0 + r][e] = fmaf(be * kv, u1[r][e], fmaf(qv, u2[r][e], dg[r0 + r][e]));
                part = fmaf(kv, u1[r][e], part);
            }
            dbp[r0 + r] = part;
        }
    }

    // column side: for j, over i >= j,
    //   w_jc = sum_{i>j} beta_i dA_ij k_ic E_ijc + sum_{i>=j} dP_ij q_ic E_ijc
#pragma unroll
    for (int r0 = 0; r0 < TMK; r0 += 4) {
        float w[4][4] = {}, gj[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) gj[r][e] = Gs[(ki + RSK * (r0 + r)) * LDK + kj + NCGK * e];
        const int jmin = ki + RSK * r0;
        for (int i = jmin; i < 64; ++i) {
            float ki4[4], qi4[4], gi4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ki4[e] = Ks[i * LDK + kj + NCGK * e];
                qi4[e] = Qs[i * LDK + kj + NCGK * e];
                gi4[e] = Gs[i * LDK + kj + NCGK * e];
            }
            const float be = bs[i];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int j = ki + RSK * (r0 + r);
                if (i >= j) {
                    const float a = (i > j) ? be * dA[i * LDC + j] : 0.f;
                    const float q = dP[i * LDC + j];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float t = fmaf(a, ki4[e], q * qi4[e]);
                        w[r][e] = fmaf(t, __expf(gi4[e] - gj[r][e]), w[r][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = ki + RSK * (r0 + r);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float kv = Ks[j * LDK + kj + NCGK * e];
                dk[r0 + r][e] += w[r][e];
                dg[r0 + r][e] = fmaf(-kv, w[r][e], dg[r0 + r][e]);
            }
        }
    }

    // dq, dk (bf16) and dbeta; dG into the tile for the running sum
#pragma unroll
    for (int r = 0; r < TMK; ++r) {
        const int i = ki + RSK * r;
        float part = dbp[r];
#pragma unroll
        for (int o = NCGK / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
#pragma unroll
        for (int e = 0; e < 4; ++e) dGt[i * LDK + kj + NCGK * e] = dg[r][e];
        if (i < nv) {
            const long long off = ((row0 + i) * H + h) * static_cast<long long>(K);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p.dq[off + kj + NCGK * e] = f32_to_bf16(dq[r][e]);
                p.dk[off + kj + NCGK * e] = f32_to_bf16(dk[r][e]);
            }
            if (kj == 0) p.dbeta[(row0 + i) * H + h] = f32_to_bf16(dbs[i] + part);
        }
    }
    __syncthreads();
    // dg = reverse running sum of dG; the last row also carries
    // exp(G_n) o rowsum(dS o S0) and the column sum of X
    for (int c = threadIdx.x; c < K; c += blockDim.x) {
        float run = gn[c] * gsum[c];
        float xsum = 0.f;
        for (int q = 0; q < RSK; ++q) xsum += xs[q * K + c];
        run += xsum;
        for (int i = nv - 1; i >= 0; --i) {
            run += dGt[i * LDK + c];
            p.dg[((row0 + i) * H + h) * static_cast<long long>(K) + c] = run;
        }
    }
}

template <int K>
cudaError_t launch_chain_k(const KdaBwdArgs& a, cudaStream_t stream) {
    const size_t smem = KdaChainSmem<K>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_bwd_chain_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kChainVs, a.H, a.N);
    gdn_kda_bwd_chain_kernel<K><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_local_k(const KdaBwdArgs& a, cudaStream_t stream) {
    const size_t smem = KdaLocalSmem<K>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_kda_bwd_local_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_chunks, a.H, a.N);
    gdn_kda_bwd_local_kernel<K><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kda_bwd_chain(const KdaBwdArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_chain_k<64>(a, stream);
    return launch_chain_k<128>(a, stream);
}

cudaError_t launch_kda_bwd_local(const KdaBwdArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_local_k<64>(a, stream);
    return launch_local_k<128>(a, stream);
}

}  // namespace gdn

// Chunked gated delta rule backward, fp32 CUDA-core version.
//
// The pages list the gradients a chunked GDN kernel returns (dq, dk, dv,
// dg, dbeta: "Research Sprint Day 1", tables of max-relative error per
// tensor) and that backward kernels share the chunk intermediates (fla issue
// #1550, "Proposed scope"); the algebra below is the reverse mode of the
// chunk forward in gdn_common.cuh, derived here.
//
// One block per (32-column value slice, head, sequence) walks the chunks
// from last to first, carrying dS (gradient w.r.t. the chunk-end state
// slice).  The chunk-start states S0 come from a forward pass that stored
// them (launch_fwd_simt with chunk_states).  Per chunk, with
// Bhat = diag(beta) V - diag(beta gam) K S0 and Delta = T Bhat:
//   dP    = scale dO Delta^T;                dQK = dP o M
//   dDelta= scale P^T dO + dec o (K dS)
//   dBhat = T^T dDelta;                       dA = -(dBhat Delta^T) o strict
//   dV    = beta o dBhat
//   dQ    = scale gam o (dO S0^T) + dQK K
//   dK    = dQK^T Q + (dec o Delta) dS^T - (beta gam o dBhat) S0^T
//           + dKK K + dKK^T K,            dKK = dA o beta_i exp(G_i - G_j)
//   dS0   = scale Q^T (gam o dO) + gam_n dS - K^T (beta gam o dBhat)
//   dbeta, dG from every use of beta, exp(G), exp(G_i - G_j); dg is the
//   reverse running sum of dG inside the chunk.
// dq, dk, dg, dbeta sum over value columns, so each block writes fp32
// partials for its slice and launch_bwd_reduce adds the slices in a fixed
// order (deterministic, no atomics).  dv and d_initial_state are complete
// per slice.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kVs = kBwdVs;

template <int K>
struct BwdSmem {
    static constexpr int LDH = K + 2;       // bf16 row stride (odd word count)
    static constexpr int LDV = kVs + 1;     // fp32 C x Vs and K x Vs tiles
    static constexpr int LDC = kChunk + 1;  // fp32 C x C tiles
    static constexpr int kHalfs = 2 * 64 * LDH;
    static constexpr int kFloats = 6 * 64 * LDV + 2 * K * LDV + 5 * 64 * LDC + 12 * 64;
    static constexpr size_t kBytes = sizeof(float) * kFloats + sizeof(uint16_t) * kHalfs;
};

template <int K>
__global__ void __launch_bounds__(256) gdn_bwd_simt_kernel(BwdArgs p) {
    using L = BwdSmem<K>;
    constexpr int LDH = L::LDH;
    constexpr int LDV = L::LDV;
    constexpr int LDC = L::LDC;
    const int vs = blockIdx.x;
    const int h = blockIdx.y;
    const int n = blockIdx.z;
    const int V = p.d_v;
    const int H = p.H;
    int b, t0, t1;
    if (!seq_range(p.cu_seqlens, n, p.N, p.T, p.err, b, t0, t1)) return;

    extern __shared__ float sm[];
    float* Vt = sm;                 // V slice, later Q S0
    float* dOt = Vt + 64 * LDV;
    float* KSt = dOt + 64 * LDV;    // K S0
    float* Dl = KSt + 64 * LDV;     // Delta
    float* dD = Dl + 64 * LDV;      // Bhat (temp), then dDelta
    float* dB = dD + 64 * LDV;      // K dS, then dBhat
    float* S0s = dB + 64 * LDV;     // K x Vs
    float* dSs = S0s + K * LDV;     // K x Vs
    float* KKM = dSs + K * LDV;     // (K K^T) o strict decay
    float* Pm = KKM + 64 * LDC;     // (Q K^T) o M
    float* Tm = Pm + 64 * LDC;      // (I + A)^-1
    float* Bx = Tm + 64 * LDC;      // A, then dA, then dKK
    float* Dx = Bx + 64 * LDC;      // inverse scratch, then dP, then dQK
    float* gs = Dx + 64 * LDC;
    float* Gs = gs + 64;
    float* gam = Gs + 64;
    float* bs = gam + 64;
    float* dec = bs + 64;
    float* dG = dec + 64;
    float* dgam = dG + 64;
    float* dbet = dgam + 64;
    float* rs = dbet + 64;          // row sums
    float* cs = rs + 64;            // column sums
    float* red = cs + 64;           // block reduction scratch (64)
    float* spare = red + 64;
    uint16_t* Qh = reinterpret_cast<uint16_t*>(spare + 64);
    uint16_t* Kh = Qh + 64 * LDH;
    (void)spare;

    auto Qf = [&](int r, int c) { return bf16_to_f32(Qh[r * LDH + c]); };
    auto Kf = [&](int r, int c) { return bf16_to_f32(Kh[r * LDH + c]); };

    const long long KV = static_cast<long long>(K) * V;
    const long long state_off = (static_cast<long long>(n) * H + h) * KV + vs * kVs;
    for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
        const int i = e / kVs, j = e % kVs;
        dSs[i * LDV + j] = p.d_final_state ? p.d_final_state[state_off + static_cast<long long>(i) * V + j] : 0.f;
    }
    const long long slot0 = chunk_slot_base(p.cu_seqlens, n, p.T);
    const long long row_base = static_cast<long long>(b) * p.T;
    const long long rows = static_cast<long long>(p.cu_seqlens ? 1 : p.N) * p.T * H;
    const float scale = p.scale;
    const int nchunks = (t1 - t0 + kChunk - 1) / kChunk;

    for (int ci = nchunks - 1; ci >= 0; --ci) {
        const int c0 = t0 + ci * kChunk;
        const int nv = min(kChunk, t1 - c0);
        __syncthreads();
        // ---- loads ----
        for (int e = threadIdx.x; e < 64 * (K / 8); e += blockDim.x) {
            const int r = e / (K / 8);
            const int c = (e % (K / 8)) * 8;
            uint4 kq = make_uint4(0, 0, 0, 0), qq = make_uint4(0, 0, 0, 0);
            if (r < nv) {
                const long long off = ((row_base + c0 + r) * H + h) * static_cast<long long>(K) + c;
                kq = *reinterpret_cast<const uint4*>(p.k + off);
                qq = *reinterpret_cast<const uint4*>(p.q + off);
            }
            const uint16_t* kp = reinterpret_cast<const uint16_t*>(&kq);
            const uint16_t* qp = reinterpret_cast<const uint16_t*>(&qq);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                Kh[r * LDH + c + m] = kp[m];
                Qh[r * LDH + c + m] = qp[m];
            }
        }
        for (int e = threadIdx.x; e < 64 * kVs; e += blockDim.x) {
            const int r = e / kVs, c = e % kVs;
            float vv = 0.f, dd = 0.f;
            if (r < nv) {
                const long long off = ((row_base + c0 + r) * H + h) * static_cast<long long>(V) + vs * kVs + c;
                vv = bf16_to_f32(p.v[off]);
                dd = bf16_to_f32(p.d_out[off]);
            }
            Vt[r * LDV + c] = vv;
            dOt[r * LDV + c] = dd;
        }
        {
            const float* src = p.chunk_states + ((slot0 + ci) * H + h) * KV + vs * kVs;
            for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
                const int i = e / kVs, j = e % kVs;
                S0s[i * LDV + j] = src[static_cast<long long>(i) * V + j];
            }
        }
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            const long long idx = (row_base + c0 + r) * H + h;
            gs[r] = (r < nv) ? p.g[idx] : 0.f;
            bs[r] = (r < nv) ? bf16_to_f32(p.beta[idx]) : 0.f;
            dG[r] = 0.f;
            dgam[r] = 0.f;
            dbet[r] = 0.f;
        }
        __syncthreads();
        chunk_cumsum(gs, Gs, gam);
        __syncthreads();
        if (threadIdx.x < 64) dec[threadIdx.x] = expf(Gs[63] - Gs[threadIdx.x]);
        // ---- chunk-local forward quantities ----
        block_mm<64, 64, K, 4, 4>(
            Kf, [&](int kk, int j) { return Kf(j, kk); },
            [&](int i, int j, float acc) {
                const float v = (j < i) ? acc * expf(Gs[i] - Gs[j]) : 0.f;
                KKM[i * LDC + j] = v;
                Bx[i * LDC + j] = bs[i] * v;
            });
        block_mm<64, 64, K, 4, 4>(
            Qf, [&](int kk, int j) { return Kf(j, kk); },
            [&](int i, int j, float acc) {
                Pm[i * LDC + j] = (j <= i) ? acc * expf(Gs[i] - Gs[j]) : 0.f;
            });
        block_mm<64, kVs, K, 4, 2>(
            Kf, [&](int d, int c) { return S0s[d * LDV + c]; },
            [&](int i, int c, float acc) { KSt[i * LDV + c] = acc; });
        __syncthreads();
        chunk_unit_lower_inverse<LDC>(Bx, Tm, Dx);
        for (int e = threadIdx.x; e < 64 * kVs; e += blockDim.x) {
            const int i = e / kVs, c = e % kVs;
            dD[i * LDV + c] = bs[i] * (Vt[i * LDV + c] - gam[i] * KSt[i * LDV + c]);
        }
        __syncthreads();
        // Delta = T Bhat
        block_mm<64, kVs, 64, 4, 2>(
            [&](int i, int jj) { return Tm[i * LDC + jj]; },
            [&](int jj, int c) { return dD[jj * LDV + c]; },
            [&](int i, int c, float acc) { Dl[i * LDV + c] = acc; });
        // K dS (dS is the gradient at this chunk's end)
        block_mm<64, kVs, K, 4, 2>(
            Kf, [&](int d, int c) { return dSs[d * LDV + c]; },
            [&](int i, int c, float acc) { dB[i * LDV + c] = acc; });
        __syncthreads();
        // dP = scale dO Delta^T
        block_mm<64, 64, kVs, 4, 4>(
            [&](int i, int c) { return dOt[i * LDV + c]; },
            [&](int c, int j) { return Dl[j * LDV + c]; },
            [&](int i, int j, float acc) { Dx[i * LDC + j] = scale * acc; });
        // gam_n term of dgam: <dS, S0>
        {
            float part = 0.f;
            for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
                const int i = e / kVs, j = e % kVs;
                part = fmaf(dSs[i * LDV + j], S0s[i * LDV + j], part);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
        }
        __syncthreads();
        // dG from M (dP o P), dd from dec, <dS,S0>
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            float r = 0.f;
            for (int j = 0; j <= i; ++j) r = fmaf(Dx[i * LDC + j], Pm[i * LDC + j], r);
            rs[i] = r;
        } else if (threadIdx.x < 128) {
            const int j = threadIdx.x - 64;
            float c = 0.f;
            for (int i = j; i < 64; ++i) c = fmaf(Dx[i * LDC + j], Pm[i * LDC + j], c);
            cs[j] = c;
        } else if (threadIdx.x < 192) {
            const int j = threadIdx.x - 128;
            float s = 0.f;
            for (int c = 0; c < kVs; ++c) s = fmaf(dB[j * LDV + c], Dl[j * LDV + c], s);
            red[8 + j] = s * dec[j];  // dd_j
        }
        __syncthreads();
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            dG[i] += rs[i] - cs[i] - red[8 + i];
        }
        if (threadIdx.x == 64) {
            float s = 0.f;
            for (int j = 0; j < 64; ++j) s += red[8 + j];
            float t = 0.f;
            for (int w = 0; w < 8; ++w) t += red[w];
            red[72] = s;   // sum of dd
            red[73] = t;   // <dS, S0>
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            dG[63] += red[72];
            dgam[63] += red[73];
        }
        // dQK = dP o M (in place)
        for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
            const int i = e / 64, j = e % 64;
            Dx[i * LDC + j] = (j <= i) ? Dx[i * LDC + j] * expf(Gs[i] - Gs[j]) : 0.f;
        }
        // dDelta = scale P^T dO + dec o (K dS)
        block_mm<64, kVs, 64, 4, 2>(
            [&](int i, int jj) { return Pm[jj * LDC + i]; },
            [&](int jj, int c) { return dOt[jj * LDV + c]; },
            [&](int i, int c, float acc) { dD[i * LDV + c] = fmaf(scale, acc, dec[i] * dB[i * LDV + c]); });
        __syncthreads();
        // dBhat = T^T dDelta  (into dB)
        block_mm<64, kVs, 64, 4, 2>(
            [&](int i, int jj) { return Tm[jj * LDC + i]; },
            [&](int jj, int c) { return dD[jj * LDV + c]; },
            [&](int i, int c, float acc) { dB[i * LDV + c] = acc; });
        __syncthreads();
        // dA = -(dBhat Delta^T) o strict lower
        block_mm<64, 64, kVs, 4, 4>(
            [&](int i, int c) { return dB[i * LDV + c]; },
            [&](int c, int j) { return Dl[j * LDV + c]; },
            [&](int i, int j, float acc) { Bx[i * LDC + j] = (j < i) ? -acc : 0.f; });
        // dV = beta o dBhat
        for (int e = threadIdx.x; e < 64 * kVs; e += blockDim.x) {
            const int i = e / kVs, c = e % kVs;
            if (i < nv)
                p.dv[((row_base + c0 + i) * H + h) * static_cast<long long>(V) + vs * kVs + c] =
                    f32_to_bf16(bs[i] * dB[i * LDV + c]);
        }
        // dbeta, dgam from Bhat
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            float sv = 0.f, sk = 0.f;
            for (int c = 0; c < kVs; ++c) {
                sv = fmaf(Vt[i * LDV + c], dB[i * LDV + c], sv);
                sk = fmaf(KSt[i * LDV + c], dB[i * LDV + c], sk);
            }
            dbet[i] += sv - gam[i] * sk;
            dgam[i] -= bs[i] * sk;
        }
        __syncthreads();
        // dbeta and dG from A;  Q S0 for the gam term (into Vt)
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            float r = 0.f;
            for (int j = 0; j < i; ++j) r = fmaf(Bx[i * LDC + j], KKM[i * LDC + j], r);
            dbet[i] += r;
            rs[i] = bs[i] * r;
        } else if (threadIdx.x < 128) {
            const int j = threadIdx.x - 64;
            float c = 0.f;
            for (int i = j + 1; i < 64; ++i) c = fmaf(Bx[i * LDC + j], bs[i] * KKM[i * LDC + j], c);
            cs[j] = c;
        }
        block_mm<64, kVs, K, 4, 2>(
            Qf, [&](int d, int c) { return S0s[d * LDV + c]; },
            [&](int i, int c, float acc) { Vt[i * LDV + c] = acc; });
        __syncthreads();
        if (threadIdx.x < 64) {
            const int i = threadIdx.x;
            dG[i] += rs[i] - cs[i];
            float s = 0.f;
            for (int c = 0; c < kVs; ++c) s = fmaf(Vt[i * LDV + c], dOt[i * LDV + c], s);
            dgam[i] += scale * s;
        }
        // dKK = dA o beta_i exp(G_i - G_j) (in place)
        for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
            const int i = e / 64, j = e % 64;
            Bx[i * LDC + j] = (j < i) ? Bx[i * LDC + j] * bs[i] * expf(Gs[i] - Gs[j]) : 0.f;
        }
        __syncthreads();
        // dQ partial = scale gam o (dO S0^T) + dQK K
        block_mm<64, K, kVs + 64, 4, (K >= 128 ? 8 : 4)>(
            [&](int i, int kk) { return kk < kVs ? scale * gam[i] * dOt[i * LDV + kk] : Dx[i * LDC + kk - kVs]; },
            [&](int kk, int d) { return kk < kVs ? S0s[d * LDV + kk] : Kf(kk - kVs, d); },
            [&](int i, int d, float acc) {
                if (i < nv)
                    p.dq_part[(vs * rows + (row_base + c0 + i) * H + h) * K + d] = acc;
            });
        // dK partial
        block_mm<64, K, 64 + kVs + kVs + 128, 4, (K >= 128 ? 8 : 4)>(
            [&](int i, int kk) {
                if (kk < 64) return Dx[kk * LDC + i];
                if (kk < 64 + kVs) return dec[i] * Dl[i * LDV + kk - 64];
                if (kk < 64 + 2 * kVs) return -bs[i] * gam[i] * dB[i * LDV + kk - 64 - kVs];
                if (kk < 128 + 2 * kVs) return Bx[i * LDC + kk - 64 - 2 * kVs];
                return Bx[(kk - 128 - 2 * kVs) * LDC + i];
            },
            [&](int kk, int d) {
                if (kk < 64) return Qf(kk, d);
                if (kk < 64 + kVs) return dSs[d * LDV + kk - 64];
                if (kk < 64 + 2 * kVs) return S0s[d * LDV + kk - 64 - kVs];
                if (kk < 128 + 2 * kVs) return Kf(kk - 64 - 2 * kVs, d);
                return Kf(kk - 128 - 2 * kVs, d);
            },
            [&](int i, int d, float acc) {
                if (i < nv)
                    p.dk_part[(vs * rows + (row_base + c0 + i) * H + h) * K + d] = acc;
            });
        __syncthreads();
        // dS0 = scale Q^T (gam o dO) + gam_n dS - K^T (beta gam o dBhat)
        const float gC = gam[63];
        block_mm<K, kVs, 128, 4, 2>(
            [&](int d, int kk) { return kk < 64 ? Qf(kk, d) : Kf(kk - 64, d); },
            [&](int kk, int c) {
                return kk < 64 ? scale * gam[kk] * dOt[kk * LDV + c]
                               : -bs[kk - 64] * gam[kk - 64] * dB[(kk - 64) * LDV + c];
            },
            [&](int d, int c, float acc) { dSs[d * LDV + c] = fmaf(gC, dSs[d * LDV + c], acc); });
        // dG += dgam o gam; dg = reverse running sum of dG (warp 0)
        if (threadIdx.x < 32) {
            const int l = threadIdx.x;
            // positions 63 - 2l and 62 - 2l, scanned from the end
            const int i0 = 63 - 2 * l, i1 = 62 - 2 * l;
            const float a = dG[i0] + dgam[i0] * gam[i0];
            const float bb = dG[i1] + dgam[i1] * gam[i1];
            float s = a + bb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (l >= off) s += o;
            }
            const float base = s - (a + bb);
            const float r0 = base + a;   // dg at i0
            const float r1 = s;          // dg at i1
            if (i0 < nv) {
                const long long row = (row_base + c0 + i0) * H + h;
                p.dg_part[vs * rows + row] = r0;
                p.dbeta_part[vs * rows + row] = dbet[i0];
            }
            if (i1 < nv) {
                const long long row = (row_base + c0 + i1) * H + h;
                p.dg_part[vs * rows + row] = r1;
                p.dbeta_part[vs * rows + row] = dbet[i1];
            }
        }
    }
    __syncthreads();
    if (p.d_initial_state) {
        for (int e = threadIdx.x; e < K * kVs; e += blockDim.x) {
            const int i = e / kVs, j = e % kVs;
            p.d_initial_state[state_off + static_cast<long long>(i) * V + j] = dSs[i * LDV + j];
        }
    }
}

__global__ void gdn_bwd_reduce_kernel(const float* __restrict__ dq_part, const float* __restrict__ dk_part,
                                      const float* __restrict__ dg_part, const float* __restrict__ dbeta_part,
                                      int slices, long long rows, int d_k, uint16_t* __restrict__ dq,
                                      uint16_t* __restrict__ dk, float* __restrict__ dg,
                                      uint16_t* __restrict__ dbeta) {
    const long long total = rows * d_k;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total; e += stride) {
        float a = 0.f, c = 0.f;
        for (int s = 0; s < slices; ++s) {
            a += dq_part[s * total + e];
            c += dk_part[s * total + e];
        }
        dq[e] = f32_to_bf16(a);
        dk[e] = f32_to_bf16(c);
        if (e < rows) {
            float x = 0.f, y = 0.f;
            for (int s = 0; s < slices; ++s) {
                x += dg_part[s * rows + e];
                y += dbeta_part[s * rows + e];
            }
            dg[e] = x;
            dbeta[e] = f32_to_bf16(y);
        }
    }
}

template <int K>
cudaError_t launch_bwd_simt_k(const BwdArgs& a, cudaStream_t stream) {
    const size_t smem = BwdSmem<K>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(gdn_bwd_simt_kernel<K>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(a.d_v / kVs, a.H, a.N);
    gdn_bwd_simt_kernel<K><<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t stream) {
    if (a.d_k == 64) return launch_bwd_simt_k<64>(a, stream);
    return launch_bwd_simt_k<128>(a, stream);
}

cudaError_t launch_bwd_reduce(const float* dq_part, const float* dk_part, const float* dg_part,
                              const float* dbeta_part, int slices, long long rows, int d_k,
                              uint16_t* dq, uint16_t* dk, float* dg, uint16_t* dbeta,
                              cudaStream_t stream) {
    const long long total = rows * d_k;
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    gdn_bwd_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        dq_part, dk_part, dg_part, dbeta_part, slices, rows, d_k, dq, dk, dg, dbeta);
    return cudaGetLastError();
}

}  // namespace gdn

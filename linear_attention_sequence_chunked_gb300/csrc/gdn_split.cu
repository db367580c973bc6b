// Sequence split: one sequence run as segments whose affine carries compose.
//
// cuLA issue #126 ("Hypothesis") describes intracard context parallelism:
// each segment maps its start state to its end state by an affine transform,
// S_end = M S_start + b (M: K x K, b: K x V), the carries are composed in
// order, and each segment then runs from its true start.  Here the carries
// come from the chunk chain itself: b is the segment's end state from a zero
// start, M its end state from the identity with zero values (the value
// columns of the recurrence are independent, so a run whose state starts at I
// and whose values are 0 leaves exactly the transition in the state).  This
// file holds the two small kernels around those runs: the setup (segment
// bounds as packed sequences, identity start states) and the composition
// (fp32, sequential over a sequence's segments).
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// cu[s] for s = 0 .. B nseg: sequence b's segment j starts at token
// b T + 64 floor(j nch / nseg) (whole chunks), the last one ends at b T + T;
// then the identity start state of every (segment, head).
__global__ void gdn_split_setup_kernel(const SplitArgs a) {
    const long long nch = (a.T + kChunk - 1) / kChunk;
    const long long nseq = static_cast<long long>(a.B) * a.nseg;
    const long long kk = static_cast<long long>(a.d_k) * a.d_k;
    const long long total = nseq * a.H * kk;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total + nseq + 1;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        if (i <= nseq) {
            const long long b = i / a.nseg, j = i % a.nseg;
            long long pos = b * a.T + (j == 0 ? 0 : kChunk * ((j * nch) / a.nseg));
            if (i == nseq) pos = static_cast<long long>(a.B) * a.T;
            a.cu[i] = static_cast<int32_t>(pos);
        } else {
            const long long e = i - nseq - 1;
            const long long r = (e % kk) / a.d_k, c = e % a.d_k;
            a.ident[e] = r == c ? 1.f : 0.f;
        }
    }
}

// Per (column block of 32, head, sequence): S = the sequence's initial state;
// for each segment j in order, starts[j] = S and S <- M_j S + b_j; the last S
// is the sequence's final state.  256 threads: thread t owns row t / 2 and
// columns 16 (t % 2) .. + 15 of the block.
constexpr int kComposeThreads = 256;
constexpr int kCols = 32;
__global__ void __launch_bounds__(kComposeThreads) gdn_split_compose_kernel(const SplitArgs a) {
    const int cb = blockIdx.x * kCols, h = blockIdx.y, b = blockIdx.z;
    const int K = a.d_k, V = a.d_v;
    const int t = threadIdx.x, r = t >> 1, c0 = 16 * (t & 1);
    __shared__ float S[128][kCols + 1];
    const bool live = r < K;
    if (live) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            S[r][c0 + c] = a.initial_state
                               ? a.initial_state[((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0 + c]
                               : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < a.nseg; ++j) {
        const long long n = static_cast<long long>(b) * a.nseg + j;
        float acc[16];
        if (live) {
            float* st = a.starts + ((n * a.H + h) * K + r) * V + cb + c0;
            const float* bj = a.b_fin + ((n * a.H + h) * K + r) * V + cb + c0;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                st[c] = S[r][c0 + c];
                acc[c] = bj[c];
            }
            const float* mrow = a.m_fin + ((n * a.H + h) * K + r) * static_cast<long long>(K);
            for (int m = 0; m < K; ++m) {
                const float mv = mrow[m];
#pragma unroll
                for (int c = 0; c < 16; ++c) acc[c] = fmaf(mv, S[m][c0 + c], acc[c]);
            }
        }
        __syncthreads();
        if (live) {
#pragma unroll
            for (int c = 0; c < 16; ++c) S[r][c0 + c] = acc[c];
        }
        __syncthreads();
    }
    if (a.final_state && live) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            a.final_state[((static_cast<long long>(b) * a.H + h) * K + r) * V + cb + c0 + c] = S[r][c0 + c];
    }
}

}  // namespace

cudaError_t launch_split_setup(const SplitArgs& a, cudaStream_t stream) {
    const long long n = static_cast<long long>(a.B) * a.nseg * a.H * a.d_k * a.d_k + static_cast<long long>(a.B) * a.nseg + 1;
    const long long blocks = (n + 255) / 256;
    gdn_split_setup_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_split_compose(const SplitArgs& a, cudaStream_t stream) {
    dim3 grid(a.d_v / kCols, a.H, a.B);
    gdn_split_compose_kernel<<<grid, kComposeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

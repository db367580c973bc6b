// Internal kernel-launch interface of the library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct FwdArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;
    const uint16_t* beta;
    float scale;
    const float* initial_state;
    const int32_t* cu_seqlens;
    uint16_t* out;          // may be null: skip the output
    float* out_f32;         // launch_fwd_ws_f32 only: the output in fp32 [rows][H][d_v], or with
                            // out_split its bf16 hi and lo parts as two planes [2][rows][H][d_v]
    int out_split;          // launch_fwd_ws_f32 only (see out_f32)
    float* final_state;     // may be null
    float* chunk_states;    // may be null: per-chunk start states, bf16 hi/lo operand tiles
                            // [slot][H][d_v/64][hi, lo][d_k rows x 128 B] (the bytes of fp32 [d_k][d_v]);
                            // plain fp32 [slot][H][d_k][d_v] for the per-channel-gate walk
    const uint8_t* chunk_T; // may be null: per-chunk T operand tiles [slot][H][2 x 8 KB], read
    const float* chunk_tp;  // may be null (per-channel-gate walk): per-chunk T and P, fp32
                            // [slot][H][2][64][64], read
    int N;                  // sequences (B dense, or cu_seqlens length - 1)
    int T;                  // tokens per batch row (dense) / total tokens (packed)
    int H;
    int d_k;
    int d_v;
    int* err;               // device error word
    int stall;              // failure-detection test only: the chain first waits on a hand-off that
                            // nothing signals (bounded), so the CTA times out
};

// Backward pass 2 (reverse state-gradient chain; the chunk chain kernel in
// backward mode).
struct BwdChainArgs {
    const uint16_t* q;
    const uint16_t* k;
    const float* g;
    const uint16_t* beta;
    const uint16_t* d_out;
    float scale;
    const int32_t* cu_seqlens;
    const float* d_final_state;   // may be null
    float* chunk_dstates;         // gradient w.r.t. each chunk's end state, tiles as FwdArgs::chunk_states
    const uint8_t* chunk_T;       // T operand tiles of every chunk (from the forward state pass), or null
    float* d_initial_state;       // may be null
    int N;
    int T;
    int H;
    int d_k;
    int d_v;
    int* err;
};

// Backward pass 3 (chunk-parallel local gradients).
struct BwdLocalArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;
    const uint16_t* beta;
    const uint16_t* d_out;
    float scale;
    const int32_t* cu_seqlens;
    const float* chunk_states;    // start state of each chunk, tiles as FwdArgs::chunk_states
    const float* chunk_dstates;   // gradient w.r.t. each chunk's end state, same tiles
    const uint8_t* chunk_T;       // [slot][H][2 x 8 KB]
    uint16_t* dq;
    uint16_t* dk;
    uint16_t* dv;
    float* dg;
    uint16_t* dbeta;
    int N;
    int T;
    int H;
    int d_k;
    int d_v;
    int max_chunks;               // chunks of the longest sequence (grid.x)
    int* err;
    uint32_t wait_limit;          // polls of each hand-off wait (0: kDefaultWaitLimit); drains keep the default
    int stall;                    // failure-detection test: the first item first waits on a barrier nothing signals
};

// T = (I + A)^-1 of every chunk as bf16 hi/lo operand tiles (chunk-parallel).
struct ChunkTArgs {
    const uint16_t* k;
    const float* g;
    const uint16_t* beta;
    const int32_t* cu_seqlens;
    uint8_t* chunk_T;             // [slot][H][2 x 8 KB]
    int N;
    int T;
    int H;
    int d_k;
    int max_chunks;               // chunks of the longest sequence (grid.x)
    int* err;
};

cudaError_t launch_chunk_t(const ChunkTArgs& a, cudaStream_t stream);

// Bytes of one chunk's T operand tiles in the backward workspace.
constexpr int kChunkTBytes = 2 * 64 * 128;

// Backward pass 2: the chunk chain kernel of the forward in backward mode.
cudaError_t launch_bwd_chain(const BwdChainArgs& a, uint32_t wait_limit, cudaStream_t stream);
// Backward pass 3: one CTA per (chunk, head, sequence).
cudaError_t launch_bwd_local(const BwdLocalArgs& a, cudaStream_t stream);

// Chunked forward of the per-channel-gate variant (g is (.., H, d_k)), fp32 on
// the CUDA cores; uses q, k, v, g, beta, scale, initial_state, cu_seqlens,
// out (may be null), final_state, chunk_states, chunk_tp and the sizes of
// FwdArgs (not chunk_T).  Without chunk_tp each chunk's T and P are formed in
// the walk.
cudaError_t launch_kda_chunk(const FwdArgs& a, cudaStream_t stream);

// T and P of every chunk of the per-channel-gate variant (chunk-parallel).
struct KdaTpArgs {
    const uint16_t* q;
    const uint16_t* k;
    const float* g;               // (.., H, d_k)
    const uint16_t* beta;
    const int32_t* cu_seqlens;
    float* chunk_tp;              // may be null: [slot][H][2][64][64] fp32 T, P
    uint8_t* tiles;               // may be null (d_k = 128 only): [slot][H] operand blocks of the
                                  // tensor-core walk (layout below)
    int N;
    int T;
    int H;
    int d_k;
    int max_chunks;               // chunks of the longest sequence (grid.x)
    int* err;
};

cudaError_t launch_kda_tp(const KdaTpArgs& a, cudaStream_t stream);

// Per-chunk operand block of the tensor-core per-channel-gate walk (d_k = 128),
// in the byte layout of its shared memory: bf16 hi/lo tiles, rows of 128 bytes
// swizzled in 1024-byte atoms; a d_k-wide tile is two 64-channel regions of 8 KB.
constexpr int kKdaBlkKG = 0;          // exp(G) o k          hi (16 KB), lo (16 KB); rows = tokens
constexpr int kKdaBlkQG = 32768;      // exp(G) o q
constexpr int kKdaBlkKt = 65536;      // exp(G_n - G) o k
constexpr int kKdaBlkT = 98304;       // T                   hi (8 KB), lo (8 KB)
constexpr int kKdaBlkP = 114688;      // P
constexpr int kKdaBlkVec = 131072;    // exp(G_n) (128 fp32), beta (64 fp32)
constexpr int kKdaBlkBytes = 132096;
constexpr int kKdaBlkSplit = kKdaBlkKt;  // the walk refills [0, split) and [split, end) separately

// The tensor-core walk of the per-channel-gate forward (d_k = 128): one CTA
// per (64 value columns, head, sequence) over the operand blocks above.
struct KdaWalkArgs {
    const uint16_t* v;
    const uint8_t* tiles;
    float scale;
    const float* initial_state;   // may be null
    const int32_t* cu_seqlens;
    uint16_t* out;                // may be null
    float* final_state;           // may be null
    float* chunk_states;          // may be null: fp32 [slot][H][d_k][d_v] start state of each chunk
    int N;
    int T;
    int H;
    int d_v;
    int* err;
};

cudaError_t launch_kda_walk(const KdaWalkArgs& a, uint32_t wait_limit, cudaStream_t stream);

// Floats of one chunk's T and P in the per-chunk workspace (T, then P).
constexpr int kKdaTpFloats = 2 * 64 * 64;

// Backward of the per-channel-gate variant: the reverse state-gradient walk
// (one block per 64 value columns, head and sequence) and the chunk-parallel
// local gradients (one block per chunk, head and sequence).
struct KdaBwdArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;               // (.., H, d_k)
    const uint16_t* beta;
    const uint16_t* d_out;
    float scale;
    const int32_t* cu_seqlens;
    const float* d_final_state;   // may be null (zeros)
    const float* chunk_tp;        // [slot][H][2][64][64]: T, P
    const uint8_t* tiles;         // d_k = 128: [slot][H] operand blocks of the tensor-core walk
    const float* chunk_states;    // [slot][H][d_k][d_v]: start state of each chunk
    float* chunk_dstates;         // [slot][H][d_k][d_v]: gradient w.r.t. each chunk's end state
    float* d_initial_state;       // may be null
    uint16_t* dq;
    uint16_t* dk;
    uint16_t* dv;
    float* dg;                    // (.., H, d_k)
    uint16_t* dbeta;
    int N;
    int T;
    int H;
    int d_k;
    int d_v;
    int max_chunks;
    int* err;
};

cudaError_t launch_kda_bwd_chain(const KdaBwdArgs& a, cudaStream_t stream);
cudaError_t launch_kda_bwd_local(const KdaBwdArgs& a, cudaStream_t stream);

// The reverse walk of the per-channel-gate backward on the tensor cores
// (d_k = 128): as launch_kda_bwd_chain, over the operand blocks in a.tiles.
cudaError_t launch_kda_bwd_chain_tc(const KdaBwdArgs& a, uint32_t wait_limit, cudaStream_t stream);
// The local gradients on the tensor cores (d_k = 128): as launch_kda_bwd_local,
// over the operand blocks in a.tiles.
cudaError_t launch_kda_bwd_local_tc(const KdaBwdArgs& a, uint32_t wait_limit, cudaStream_t stream);

// Token-serial forward (decode path; the same recurrence token by token).
struct RecurrentArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;               // (B,T,H) fp32, or (B,T,H,d_k) with per_channel_gate
    const uint16_t* beta;
    float scale;
    const float* initial_state;   // may be null (zeros)
    const int32_t* cu_seqlens;
    uint16_t* out;
    float* final_state;           // may be null
    int per_channel_gate;         // one log decay per key channel (KDA)
    int N, T, H, d_k, d_v;
    int* err;
};

cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t stream);

// Prologue (q/k L2 normalisation, gates) and its reverse mode.
struct PrologueArgs {
    const uint16_t* q_raw;        // (rows, H, d_k) bf16; null: q not normalised here
    const uint16_t* k_raw;        // likewise
    const float* a;               // (rows, H) raw decay-gate input
    const float* b;               // (rows, H) raw beta input
    const float* A_log;           // (H), decay gate only
    const float* dt_bias;         // (H) or null (zeros)
    int gate_mode;                // 1: -exp(A_log) softplus(a + dt_bias); 2: lower sigmoid(a + dt_bias)
    float lower;                  // gate_mode 2
    float beta_scale;             // beta = beta_scale sigmoid(b)
    uint16_t* q;                  // forward outputs: q_hat, k_hat (bf16), g (fp32), beta (bf16)
    uint16_t* k;
    float* g;
    uint16_t* beta;
    const uint16_t* dq;           // backward inputs: gradients w.r.t. q_hat, k_hat, g, beta
    const uint16_t* dk;
    const float* dg;
    const uint16_t* dbeta;
    uint16_t* dq_raw;             // backward outputs
    uint16_t* dk_raw;
    float* da;
    float* db;
    float* dA_log;                // (H) or null
    float* ddt_bias;              // (H) or null
    int rows;                     // tokens (B * T)
    int H;
    int d_k;
};

cudaError_t launch_prologue_fwd(const PrologueArgs& a, cudaStream_t stream);
cudaError_t launch_prologue_bwd(const PrologueArgs& a, cudaStream_t stream);

// Sequence split (segments with composed affine carries): setup of the
// segment bounds and identity start states, and the fp32 composition.
struct SplitArgs {
    int32_t* cu;                  // [B nseg + 1] segment bounds as packed sequences
    float* ident;                 // [B nseg][H][d_k][d_k] identity start states
    const float* initial_state;   // [B][H][d_k][d_v] or null (zeros)
    const float* m_fin;           // [B nseg][H][d_k][d_k] segment transitions M
    const float* b_fin;           // [B nseg][H][d_k][d_v] segment offsets b
    float* starts;                // [B nseg][H][d_k][d_v] true segment start states
    float* final_state;           // [B][H][d_k][d_v] or null
    int B, T, H, d_k, d_v, nseg;
};
cudaError_t launch_split_setup(const SplitArgs& a, cudaStream_t stream);
cudaError_t launch_split_compose(const SplitArgs& a, cudaStream_t stream);
// The split's outputs from its two carry runs: every segment's chain is linear
// in its start state, so out = O_b + O_M S_start (O_b: the run from a zero
// start, fp32 [rows][H][d_v]; O_M: the run from the identity with zero values,
// fp32 [rows][H][d_k]; S_start: the composed start states), rounded to bf16.
struct SplitCorrectArgs {
    const float* ob;
    const float* om;
    const float* starts;          // [nseq][H][d_k][d_v]
    const int32_t* cu;            // [nseq + 1] segment bounds (packed rows)
    uint16_t* out;                // [rows][H][d_v]
    int nseq, H, d_k, d_v;
    long long rows;               // packed rows of all segments
    int T, nseg;                  // tokens per sequence and segments per sequence (nseq = B nseg)
    int max_chunks;               // chunks of the longest segment
    int* err;
    uint32_t wait_limit;
};
cudaError_t launch_split_correct(const SplitCorrectArgs& a, cudaStream_t stream);

// Peak probes (measurement only): a 16-byte-vector copy of `bytes` (a
// multiple of 16), and the bf16 GEMM C[M][N] = A[M][K] B[N][K]^T with
// M % 128 == 0, N % 256 == 0, K % 64 == 0.
cudaError_t launch_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream);
cudaError_t launch_probe_gemm(const uint16_t* A, const uint16_t* B, uint16_t* C, int M, int N, int K, int* err,
                              cudaStream_t stream);
// Warp-specialised tensor-core forward (prep and chain warpgroups);
// wait_limit bounds every hand-off mbarrier wait (polls); the waits that
// drain in-flight copies and products before a CTA leaves keep the default.
cudaError_t launch_fwd_ws(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream);
// The same chain with the output written in fp32 to a.out_f32 (the sequence
// split's carry runs); a.out is ignored.
cudaError_t launch_fwd_ws_f32(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream);
constexpr uint32_t kDefaultWaitLimit = 4000000u;

}  // namespace gdn

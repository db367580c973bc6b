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
    float* final_state;     // may be null
    float* chunk_states;    // may be null: per-chunk start states [slot][H][d_k][d_v]
    int N;                  // sequences (B dense, or cu_seqlens length - 1)
    int T;                  // tokens per batch row (dense) / total tokens (packed)
    int H;
    int d_k;
    int d_v;
    int* err;               // device error word
};

struct BwdArgs {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const float* g;
    const uint16_t* beta;
    float scale;
    const int32_t* cu_seqlens;
    const uint16_t* d_out;
    const float* d_final_state;   // may be null
    const float* chunk_states;    // [slot][H][d_k][d_v]
    float* dq_part;               // [slices][rows][d_k]
    float* dk_part;               // [slices][rows][d_k]
    float* dg_part;               // [slices][rows]
    float* dbeta_part;            // [slices][rows]
    uint16_t* dv;
    float* d_initial_state;       // may be null
    int N;
    int T;
    int H;
    int d_k;
    int d_v;
    int* err;
};

// Value columns handled by one backward block.
constexpr int kBwdVs = 32;

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream);
// Tensor-core forward; wait_limit bounds every mbarrier wait (polls).
cudaError_t launch_fwd_tc(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream);
// Warp-specialised tensor-core forward (prep and chain warpgroups).
cudaError_t launch_fwd_ws(const FwdArgs& a, uint32_t wait_limit, cudaStream_t stream);
constexpr uint32_t kDefaultWaitLimit = 4000000u;
cudaError_t launch_bwd_simt(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_reduce(const float* dq_part, const float* dk_part, const float* dg_part,
                              const float* dbeta_part, int slices, long long rows, int d_k,
                              uint16_t* dq, uint16_t* dk, float* dg, uint16_t* dbeta,
                              cudaStream_t stream);

}  // namespace gdn

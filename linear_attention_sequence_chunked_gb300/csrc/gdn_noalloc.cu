// Backward entry point that allocates nothing: its scratch lives in a
// fixed-size device array that is part of the library image.
//
// Who needs it: callers that are not allowed to allocate device memory on
// their own -- for example an inference or training runtime that fixes its
// whole memory plan at start-up and refuses any allocation afterwards, or a
// plugin whose host framework owns every device allocation.  Such callers
// cannot hand gdn_chunk_bwd the workspace it needs, so this variant brings
// its own.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"

namespace {

// Scratch shared by every call in this process on a given device.  Each
// device that loads the library keeps this much memory until the process
// exits.
constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the real address is looked
// up once per device (with that device current) and cached.
gdn_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_bwd_noalloc(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                 const float* g, const gdn_bf16* beta, float scale,
                                 const float* initial_state, const int32_t* cu_seqlens,
                                 const gdn_bf16* d_out, const float* d_final_state,
                                 gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                                 gdn_bf16* dbeta, float* d_initial_state,
                                 int B, int T, int H, int d_k, int d_v, cudaStream_t stream) {
    const size_t need = gdn_chunk_bwd_workspace_size(B, T, H, d_k, d_v, cu_seqlens != nullptr);
    if (need > kScratchBytes) return GDN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const gdn_status st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
    // The backward writes every scratch byte it later reads (chunk-start
    // states and per-slice partial gradients), so no clearing is needed.
    return gdn_chunk_bwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, d_out, d_final_state, dq, dk, dv,
                         dg, dbeta, d_initial_state, B, T, H, d_k, d_v, scratch, kScratchBytes, stream);
}

}  // extern "C"

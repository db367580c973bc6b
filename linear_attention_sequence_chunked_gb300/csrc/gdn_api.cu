// Host side of the C ABI declared in include/gdn.h: argument validation,
// workspace layout, kernel launches and the per-device error word.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace {

// Device error word (one per device that loads the library).  Kernels get
// its address as an argument; gdn_get_last_device_error reads and clears it.
__device__ int g_gdn_error_word;

constexpr size_t kAlign = 256;

// Kernels launched by this process through the library.
std::atomic<uint64_t> g_launches{0};

// Each launch_* helper enqueues exactly one kernel; count it on success.
bool launched(cudaError_t e) {
    if (e != cudaSuccess) return false;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return true;
}

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int* error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gdn_error_word) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

bool supported_dims(int d_k, int d_v) {
    return (d_k == 64 || d_k == 128) && (d_v == 64 || d_v == 128 || d_v == 256);
}

// Common shape checks.  `rows_b` is the batch extent of the (.,T,H,.) tensors.
gdn_status check_shapes(int B, int T, int H, int d_k, int d_v) {
    if (B < 1 || H < 1 || T < 0) return GDN_ERR_INVALID_ARG;
    if (!supported_dims(d_k, d_v)) return GDN_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return GDN_ERR_UNSUPPORTED;
    const long long elems = static_cast<long long>(B) * T * H * (d_k > d_v ? d_k : d_v);
    if (elems >= (1LL << 40)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Chunk slots of a per-chunk workspace array (see chunk_slot_base).
long long chunk_slots(int B, int T, int varlen) {
    if (varlen) return static_cast<long long>(T / gdn::kChunk) + B;
    return static_cast<long long>(B) * ((T + gdn::kChunk - 1) / gdn::kChunk);
}

struct BwdLayout {
    size_t states, dq, dk, dg, dbeta, total;
};

BwdLayout bwd_layout(int B, int T, int H, int d_k, int d_v, int varlen) {
    BwdLayout L{};
    const long long rows = static_cast<long long>(varlen ? 1 : B) * T * H;
    const int slices = d_v / gdn::kBwdVs;
    const size_t states = round_up(sizeof(float) * chunk_slots(B, T, varlen) * H * d_k * d_v);
    const size_t part_k = round_up(sizeof(float) * slices * rows * d_k);
    const size_t part_r = round_up(sizeof(float) * slices * rows);
    L.states = 0;
    L.dq = states;
    L.dk = L.dq + part_k;
    L.dg = L.dk + part_k;
    L.dbeta = L.dg + part_r;
    L.total = L.dbeta + part_r;
    return L;
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: unsupported size";
        case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED: tensor not 16-byte aligned";
        case GDN_ERR_BAD_SEQLENS: return "GDN_ERR_BAD_SEQLENS: malformed cu_seqlens";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime error";
    }
    return "GDN_ERR_UNKNOWN";
}

size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    (void)B; (void)T; (void)H; (void)d_k; (void)d_v; (void)varlen;
    return 0;
}

size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return bwd_layout(B, T, H, d_k, d_v, varlen).total;
}

gdn_status gdn_chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         gdn_bf16* out, float* final_state,
                         int B, int T, int H, int d_k, int d_v,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    gdn_status st = check_shapes(B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, out, initial_state, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_MISALIGNED;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    gdn::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens;
    a.out = out; a.final_state = final_state; a.chunk_states = nullptr;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err;
    if (!launched(gdn::launch_fwd_ws(a, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_chunk_bwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         const gdn_bf16* d_out, const float* d_final_state,
                         gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                         gdn_bf16* dbeta, float* d_initial_state,
                         int B, int T, int H, int d_k, int d_v,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    gdn_status st = check_shapes(B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (T > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta))
        return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, d_out, dq, dk, dv, dg, dbeta,
                          initial_state, d_final_state, d_initial_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_MISALIGNED;
    const int varlen = cu_seqlens != nullptr;
    const BwdLayout L = bwd_layout(B, T, H, d_k, d_v, varlen);
    if (L.total > 0) {
        if (!workspace || workspace_bytes < L.total) return GDN_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return GDN_ERR_MISALIGNED;
    }
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* states = reinterpret_cast<float*>(ws + L.states);

    gdn::FwdArgs f{};
    f.q = q; f.k = k; f.v = v; f.g = g; f.beta = beta; f.scale = scale;
    f.initial_state = initial_state; f.cu_seqlens = cu_seqlens;
    f.out = nullptr; f.final_state = nullptr; f.chunk_states = states;
    f.N = B; f.T = T; f.H = H; f.d_k = d_k; f.d_v = d_v; f.err = err;
    if (!launched(gdn::launch_fwd_simt(f, stream))) return GDN_ERR_CUDA;

    gdn::BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.cu_seqlens = cu_seqlens; a.d_out = d_out; a.d_final_state = d_final_state;
    a.chunk_states = states;
    a.dq_part = reinterpret_cast<float*>(ws + L.dq);
    a.dk_part = reinterpret_cast<float*>(ws + L.dk);
    a.dg_part = reinterpret_cast<float*>(ws + L.dg);
    a.dbeta_part = reinterpret_cast<float*>(ws + L.dbeta);
    a.dv = dv; a.d_initial_state = d_initial_state;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err;
    if (!launched(gdn::launch_bwd_simt(a, stream))) return GDN_ERR_CUDA;
    const long long rows = static_cast<long long>(varlen ? 1 : B) * T * H;
    if (rows > 0 && !launched(gdn::launch_bwd_reduce(a.dq_part, a.dk_part, a.dg_part, a.dbeta_part,
                                         d_v / gdn::kBwdVs, rows, d_k, dq, dk, dg, dbeta, stream)))
        return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_get_last_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_gdn_error_word, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_gdn_error_word, &zero, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    return static_cast<gdn_status>(value);
}

uint64_t gdn_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

// Host side of the C ABI declared in include/gdn.h: argument validation,
// workspace layout, kernel launches and the per-device error word.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

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

// Count the `kernels` kernels that a launch_* helper enqueued, on success.
// Most helpers enqueue exactly one; the callers of the others pass their count.
bool launched(cudaError_t e, int kernels = 1) {
    if (e != cudaSuccess) return false;
    g_launches.fetch_add(static_cast<uint64_t>(kernels), std::memory_order_relaxed);
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

gdn_status check_prologue(int rows, int H, int d_k, int gate_mode, const float* A_log) {
    if (rows < 0 || H < 1) return GDN_ERR_INVALID_ARG;
    if (d_k != 64 && d_k != 128) return GDN_ERR_UNSUPPORTED;
    if (gate_mode != 1 && gate_mode != 2) return GDN_ERR_INVALID_ARG;
    if (gate_mode == 1 && !A_log) return GDN_ERR_INVALID_ARG;
    if (static_cast<long long>(rows) * H * d_k >= (1LL << 40)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Chunk slots of a per-chunk workspace array (see chunk_slot_base).
long long chunk_slots(int B, int T, int varlen) {
    if (varlen) return static_cast<long long>(T / gdn::kChunk) + B;
    return static_cast<long long>(B) * ((T + gdn::kChunk - 1) / gdn::kChunk);
}

// Per-chunk T operand tiles (both calls' workspace holds them).
size_t tiles_bytes(int B, int T, int H, int varlen) {
    return round_up(static_cast<size_t>(gdn::kChunkTBytes) * chunk_slots(B, T, varlen) * H);
}

// T = (I + A)^-1 of every chunk into `tiles` (chunk-parallel kernel).
bool launch_tiles(const gdn_bf16* k, const float* g, const gdn_bf16* beta, const int32_t* cu_seqlens,
                  uint8_t* tiles, int B, int T, int H, int d_k, int* err, cudaStream_t stream) {
    gdn::ChunkTArgs t{};
    t.k = k; t.g = g; t.beta = beta; t.cu_seqlens = cu_seqlens; t.chunk_T = tiles;
    t.N = B; t.T = T; t.H = H; t.d_k = d_k; t.err = err;
    t.max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk;
    if (t.max_chunks == 0) return true;
    return launched(gdn::launch_chunk_t(t, stream));
}

// Backward workspace: per-chunk start states (pass 1), per-chunk end-state
// gradients (pass 2), per-chunk T tiles (the chunk-parallel inverse).
struct BwdLayout {
    size_t states, dstates, tiles, total;
};

BwdLayout bwd_layout(int B, int T, int H, int d_k, int d_v, int varlen) {
    BwdLayout L{};
    const long long slots = chunk_slots(B, T, varlen);
    const size_t per_state = sizeof(float) * static_cast<size_t>(d_k) * d_v;
    L.states = 0;
    L.dstates = round_up(per_state * slots * H);
    L.tiles = L.dstates + round_up(per_state * slots * H);
    L.total = L.tiles + tiles_bytes(B, T, H, varlen);
    return L;
}

// Saved-for-backward buffer of the training route (gdn_chunk_fwd_save ->
// gdn_chunk_bwd_saved): every chunk's start state in the same per-chunk
// layout as the backward workspace, then the T tiles.
struct SavedLayout {
    size_t states, tiles, total;
};

SavedLayout saved_layout(int B, int T, int H, int d_k, int d_v, int varlen) {
    SavedLayout L{};
    const size_t per_state = sizeof(float) * static_cast<size_t>(d_k) * d_v;
    L.states = 0;
    L.tiles = round_up(per_state * chunk_slots(B, T, varlen) * H);
    L.total = L.tiles + tiles_bytes(B, T, H, varlen);
    return L;
}

// Per-chunk end-state gradients: the only workspace of gdn_chunk_bwd_saved.
size_t dstates_bytes(int B, int T, int H, int d_k, int d_v, int varlen) {
    return round_up(sizeof(float) * static_cast<size_t>(d_k) * d_v * chunk_slots(B, T, varlen) * H);
}

// Host checks shared by the forward entry points.
gdn_status check_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                     const gdn_bf16* beta, const float* initial_state, const int32_t* cu_seqlens,
                     const gdn_bf16* out, const float* final_state, int B, int T, int H, int d_k,
                     int d_v) {
    gdn_status st = check_shapes(B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, out, initial_state, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

// Host checks shared by the backward entry points.
gdn_status check_bwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                     const gdn_bf16* beta, const float* initial_state, const int32_t* cu_seqlens,
                     const gdn_bf16* d_out, const float* d_final_state, const gdn_bf16* dq,
                     const gdn_bf16* dk, const gdn_bf16* dv, const float* dg, const gdn_bf16* dbeta,
                     const float* d_initial_state, int B, int T, int H, int d_k, int d_v) {
    gdn_status st = check_shapes(B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (T > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta))
        return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, d_out, dq, dk, dv, dg, dbeta,
                          initial_state, d_final_state, d_initial_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

// A caller buffer of `need` bytes: present, large enough, 256-byte aligned.
gdn_status check_buffer(const void* p, size_t bytes, size_t need) {
    if (need == 0) return GDN_OK;
    if (!p || bytes < need) return GDN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) & (kAlign - 1)) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

// Backward passes 2 (reverse chain of end-state gradients into `dstates`)
// and 3 (chunk-parallel local gradients), from the chunk start states and T
// tiles that pass 1 or the saving forward left.
gdn_status launch_bwd_passes(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                             const float* g, const gdn_bf16* beta, float scale,
                             const int32_t* cu_seqlens, const gdn_bf16* d_out,
                             const float* d_final_state, gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv,
                             float* dg, gdn_bf16* dbeta, float* d_initial_state, int B, int T,
                             int H, int d_k, int d_v, const float* states, float* dstates,
                             const uint8_t* tiles, int* err, cudaStream_t stream,
                             uint32_t local_wait_limit = gdn::kDefaultWaitLimit, int local_stall = 0) {
    gdn::BwdChainArgs c{};
    c.q = q; c.k = k; c.g = g; c.beta = beta; c.d_out = d_out; c.scale = scale;
    c.cu_seqlens = cu_seqlens; c.d_final_state = d_final_state;
    c.chunk_dstates = dstates; c.chunk_T = tiles; c.d_initial_state = d_initial_state;
    c.N = B; c.T = T; c.H = H; c.d_k = d_k; c.d_v = d_v; c.err = err;
    if (!launched(gdn::launch_bwd_chain(c, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;

    gdn::BwdLocalArgs l{};
    l.q = q; l.k = k; l.v = v; l.g = g; l.beta = beta; l.d_out = d_out; l.scale = scale;
    l.cu_seqlens = cu_seqlens; l.chunk_states = states; l.chunk_dstates = dstates; l.chunk_T = tiles;
    l.dq = dq; l.dk = dk; l.dv = dv; l.dg = dg; l.dbeta = dbeta;
    l.N = B; l.T = T; l.H = H; l.d_k = d_k; l.d_v = d_v; l.err = err;
    l.wait_limit = local_wait_limit; l.stall = local_stall;
    l.max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk;
    if (l.max_chunks > 0 && !launched(gdn::launch_bwd_local(l, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

// Per-chunk T and P of the per-channel-gate variant (fp32, 32 KB per chunk
// and head): the forward's optional workspace and the backward's first part.
size_t kda_tp_bytes(int B, int T, int H, int varlen) {
    return round_up(sizeof(float) * gdn::kKdaTpFloats * chunk_slots(B, T, varlen) * H);
}

// Operand blocks of the tensor-core walk (d_k = 128), 129 KB per chunk and head.
size_t kda_blocks_bytes(int B, int T, int H, int varlen) {
    return round_up(static_cast<size_t>(gdn::kKdaBlkBytes) * chunk_slots(B, T, varlen) * H);
}

// The per-channel-gate forward's workspace: the walk's operand blocks
// (d_k = 128) or fp32 T and P (d_k = 64).
size_t kda_fwd_ws_bytes(int B, int T, int H, int d_k, int varlen) {
    return d_k == 128 ? kda_blocks_bytes(B, T, H, varlen) : kda_tp_bytes(B, T, H, varlen);
}

// T and P of every chunk into `tp` (fp32) and / or the walk's operand blocks
// into `tiles` (chunk-parallel kernel).
bool launch_kda_tp_pass(const gdn_bf16* q, const gdn_bf16* k, const float* g, const gdn_bf16* beta,
                        const int32_t* cu_seqlens, float* tp, uint8_t* tiles, int B, int T, int H, int d_k,
                        int* err, cudaStream_t stream) {
    gdn::KdaTpArgs t{};
    t.q = q; t.k = k; t.g = g; t.beta = beta; t.cu_seqlens = cu_seqlens; t.chunk_tp = tp; t.tiles = tiles;
    t.N = B; t.T = T; t.H = H; t.d_k = d_k; t.err = err;
    t.max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk;
    if (t.max_chunks == 0) return true;
    return launched(gdn::launch_kda_tp(t, stream));
}

// Backward workspace of the per-channel-gate variant: T and P (fp32, d_k = 64
// only), the chunk start states (forward walk), the end-state gradients
// (reverse walk), and at d_k = 128 the tensor-core passes' operand blocks.
struct KdaBwdLayout {
    size_t tp, states, dstates, blocks, total;
};

KdaBwdLayout kda_bwd_layout(int B, int T, int H, int d_k, int d_v, int varlen) {
    KdaBwdLayout L{};
    const size_t per = round_up(sizeof(float) * static_cast<size_t>(d_k) * d_v * chunk_slots(B, T, varlen) * H);
    L.tp = 0;
    L.states = d_k == 128 ? 0 : kda_tp_bytes(B, T, H, varlen);  // fp32 T, P: the CUDA-core passes only
    L.dstates = L.states + per;
    L.blocks = L.dstates + per;
    L.total = L.blocks + (d_k == 128 ? kda_blocks_bytes(B, T, H, varlen) : 0);
    return L;
}

// Workspace of the sequence split: segment bounds, T tiles of the packed
// segments, zero values and a scratch output for the transition run, the
// identity start states, the segments' M and b, and their true start states.
struct SplitLayout {
    size_t cu, tiles, zeros, om, ob, ident, mfin, bfin, starts, total;
};

SplitLayout split_layout(int B, int T, int H, int d_k, int d_v, int nseg) {
    SplitLayout L{};
    const long long nseq = static_cast<long long>(B) * nseg;
    const long long rows = static_cast<long long>(B) * T;
    L.cu = 0;
    L.tiles = round_up(sizeof(int32_t) * (nseq + 1));
    L.zeros = L.tiles + tiles_bytes(static_cast<int>(nseq), static_cast<int>(rows), H, 1);
    L.om = L.zeros + round_up(2ull * rows * H * d_k);
    L.ob = L.om + round_up(4ull * rows * H * d_k);
    L.ident = L.ob + round_up(4ull * rows * H * d_v);
    L.mfin = L.ident + round_up(4ull * nseq * H * d_k * d_k);
    L.bfin = L.mfin + round_up(4ull * nseq * H * d_k * d_k);
    L.starts = L.bfin + round_up(4ull * nseq * H * d_k * d_v);
    L.total = L.starts + round_up(4ull * nseq * H * d_k * d_v);
    return L;
}

// A second stream per device for the split's two carry runs, which run side
// by side (one wave each when the segments' chains leave SMs idle); created
// on first use and kept for the life of the process.
constexpr int kMaxAuxDevices = 64;
cudaStream_t g_aux_stream[kMaxAuxDevices] = {};
std::mutex g_aux_mu;

cudaStream_t aux_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxAuxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_aux_mu);
    if (!g_aux_stream[dev] && cudaStreamCreateWithFlags(&g_aux_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
        g_aux_stream[dev] = nullptr;
    return g_aux_stream[dev];
}

// Segments actually used: at least one chunk each.
int split_segments(int T, int nseg) {
    const int nch = (T + gdn::kChunk - 1) / gdn::kChunk;
    return nseg < nch ? nseg : (nch > 0 ? nch : 1);
}

gdn_status recurrent(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                     const gdn_bf16* beta, float scale, const float* initial_state,
                     const int32_t* cu_seqlens, gdn_bf16* out, float* final_state, int B, int T,
                     int H, int d_k, int d_v, int per_channel, cudaStream_t stream) {
    gdn_status st = check_shapes(B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, out, initial_state, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_MISALIGNED;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    gdn::RecurrentArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.out = out; a.final_state = final_state;
    a.per_channel_gate = per_channel;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err;
    if (!launched(gdn::launch_recurrent(a, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
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
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return tiles_bytes(B, T, H, varlen);
}

size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return bwd_layout(B, T, H, d_k, d_v, varlen).total;
}

}  // extern "C"

namespace {

gdn_status chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                     const gdn_bf16* beta, float scale, const float* initial_state, const int32_t* cu_seqlens,
                     gdn_bf16* out, float* final_state, int B, int T, int H, int d_k, int d_v, void* workspace,
                     size_t workspace_bytes, uint32_t wait_limit, int stall, cudaStream_t stream) {
    gdn_status st = check_fwd(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return GDN_ERR_MISALIGNED;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    // With a workspace, every chunk's T tiles come first from the
    // chunk-parallel kernel and the chunk chain only copies them in; without
    // one, the chain's prep warpgroup forms T itself, one chunk ahead.
    const size_t tb = tiles_bytes(B, T, H, cu_seqlens != nullptr);
    uint8_t* tiles = (workspace && workspace_bytes >= tb && tb > 0) ? static_cast<uint8_t*>(workspace) : nullptr;
    if (tiles && !launch_tiles(k, g, beta, cu_seqlens, tiles, B, T, H, d_k, err, stream)) return GDN_ERR_CUDA;
    gdn::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens;
    a.out = out; a.final_state = final_state; a.chunk_states = nullptr; a.chunk_T = tiles;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err; a.stall = stall;
    if (!launched(gdn::launch_fwd_ws(a, wait_limit, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                         const float* g, const gdn_bf16* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens,
                         gdn_bf16* out, float* final_state,
                         int B, int T, int H, int d_k, int d_v,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, B, T, H, d_k, d_v,
                     workspace, workspace_bytes, gdn::kDefaultWaitLimit, 0, stream);
}

gdn_status gdn_chunk_fwd_wait_limit(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                    const float* g, const gdn_bf16* beta, float scale,
                                    const float* initial_state, const int32_t* cu_seqlens,
                                    gdn_bf16* out, float* final_state,
                                    int B, int T, int H, int d_k, int d_v,
                                    void* workspace, size_t workspace_bytes, uint32_t wait_limit,
                                    int stall_first_wait, cudaStream_t stream) {
    // the route this failure-detection entry covers: d_k = 128 with the T tiles given
    if (d_k != 128) return GDN_ERR_UNSUPPORTED;
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return check_shapes(B, T, H, d_k, d_v);
    const size_t tb = tiles_bytes(B, T, H, cu_seqlens != nullptr);
    if (tb > 0 && (!workspace || workspace_bytes < tb)) return GDN_ERR_UNSUPPORTED;
    return chunk_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, B, T, H, d_k, d_v,
                     workspace, workspace_bytes, wait_limit ? wait_limit : gdn::kDefaultWaitLimit,
                     stall_first_wait != 0, stream);
}

gdn_status gdn_recurrent_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                             const float* g, const gdn_bf16* beta, float scale,
                             const float* initial_state, const int32_t* cu_seqlens,
                             gdn_bf16* out, float* final_state,
                             int B, int T, int H, int d_k, int d_v, cudaStream_t stream) {
    return recurrent(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, B, T, H,
                     d_k, d_v, 0, stream);
}

gdn_status gdn_kda_recurrent_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                 const float* g, const gdn_bf16* beta, float scale,
                                 const float* initial_state, const int32_t* cu_seqlens,
                                 gdn_bf16* out, float* final_state,
                                 int B, int T, int H, int d_k, int d_v, cudaStream_t stream) {
    return recurrent(q, k, v, g, beta, scale, initial_state, cu_seqlens, out, final_state, B, T, H,
                     d_k, d_v, 1, stream);
}

size_t gdn_kda_chunk_fwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return kda_fwd_ws_bytes(B, T, H, d_k, varlen);
}

gdn_status gdn_kda_chunk_fwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                             const gdn_bf16* beta, float scale, const float* initial_state,
                             const int32_t* cu_seqlens, gdn_bf16* out, float* final_state, int B, int T,
                             int H, int d_k, int d_v, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    gdn_status st = check_fwd(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return GDN_ERR_MISALIGNED;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    // With a workspace, every chunk's T and P (and at d_k = 128 the decayed
    // operands) come first from the chunk-parallel kernel: d_k = 128 then runs
    // the tensor-core walk over the operand blocks, d_k = 64 the CUDA-core walk
    // reading T and P.  Without one, the CUDA-core walk forms them itself.
    const size_t need = kda_fwd_ws_bytes(B, T, H, d_k, cu_seqlens != nullptr);
    const bool fast = workspace && workspace_bytes >= need && need > 0;
    if (fast && d_k == 128) {
        uint8_t* tiles = static_cast<uint8_t*>(workspace);
        if (!launch_kda_tp_pass(q, k, g, beta, cu_seqlens, nullptr, tiles, B, T, H, d_k, err, stream))
            return GDN_ERR_CUDA;
        gdn::KdaWalkArgs w{};
        w.v = v; w.tiles = tiles; w.scale = scale; w.initial_state = initial_state; w.cu_seqlens = cu_seqlens;
        w.out = out; w.final_state = final_state; w.chunk_states = nullptr;
        w.N = B; w.T = T; w.H = H; w.d_v = d_v; w.err = err;
        if (!launched(gdn::launch_kda_walk(w, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
        return GDN_OK;
    }
    float* tp = fast ? static_cast<float*>(workspace) : nullptr;
    if (tp && !launch_kda_tp_pass(q, k, g, beta, cu_seqlens, tp, nullptr, B, T, H, d_k, err, stream))
        return GDN_ERR_CUDA;
    gdn::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.out = out; a.final_state = final_state;
    a.chunk_tp = tp;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err;
    if (!launched(gdn::launch_kda_chunk(a, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

size_t gdn_kda_chunk_bwd_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return kda_bwd_layout(B, T, H, d_k, d_v, varlen).total;
}

gdn_status gdn_kda_chunk_bwd(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                             const gdn_bf16* beta, float scale, const float* initial_state,
                             const int32_t* cu_seqlens, const gdn_bf16* d_out, const float* d_final_state,
                             gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg, gdn_bf16* dbeta,
                             float* d_initial_state, int B, int T, int H, int d_k, int d_v, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    gdn_status st = check_bwd(q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state, dq, dk, dv,
                              dg, dbeta, d_initial_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    const KdaBwdLayout L = kda_bwd_layout(B, T, H, d_k, d_v, cu_seqlens != nullptr);
    st = check_buffer(workspace, workspace_bytes, L.total);
    if (st != GDN_OK) return st;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* tp = (L.total && d_k != 128) ? reinterpret_cast<float*>(ws + L.tp) : nullptr;
    float* states = L.total ? reinterpret_cast<float*>(ws + L.states) : nullptr;
    float* dstates = L.total ? reinterpret_cast<float*>(ws + L.dstates) : nullptr;
    uint8_t* blocks = (L.total && d_k == 128) ? reinterpret_cast<uint8_t*>(ws + L.blocks) : nullptr;
    const int max_chunks = (T + gdn::kChunk - 1) / gdn::kChunk;
    if (max_chunks > 0) {
        // T and P of every chunk, then the forward walk recording each chunk's
        // start state (at d_k = 128 the tensor-core walk over the operand blocks)
        if (!launch_kda_tp_pass(q, k, g, beta, cu_seqlens, tp, blocks, B, T, H, d_k, err, stream))
            return GDN_ERR_CUDA;
        if (blocks) {
            gdn::KdaWalkArgs w{};
            w.v = v; w.tiles = blocks; w.scale = scale; w.initial_state = initial_state;
            w.cu_seqlens = cu_seqlens; w.out = nullptr; w.final_state = nullptr; w.chunk_states = states;
            w.N = B; w.T = T; w.H = H; w.d_v = d_v; w.err = err;
            if (!launched(gdn::launch_kda_walk(w, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
        }
    }
    if (max_chunks > 0 && !blocks) {
        gdn::FwdArgs f{};
        f.q = q; f.k = k; f.v = v; f.g = g; f.beta = beta; f.scale = scale;
        f.initial_state = initial_state; f.cu_seqlens = cu_seqlens;
        f.out = nullptr; f.final_state = nullptr; f.chunk_states = states; f.chunk_tp = tp;
        f.N = B; f.T = T; f.H = H; f.d_k = d_k; f.d_v = d_v; f.err = err;
        if (!launched(gdn::launch_kda_chunk(f, stream))) return GDN_ERR_CUDA;
    }
    gdn::KdaBwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.d_out = d_out; a.scale = scale;
    a.cu_seqlens = cu_seqlens; a.d_final_state = d_final_state;
    a.chunk_tp = tp; a.tiles = blocks; a.chunk_states = states; a.chunk_dstates = dstates;
    a.d_initial_state = d_initial_state;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.max_chunks = max_chunks; a.err = err;
    // the reverse walk (also when T = 0: it passes d_final_state to d_initial_state);
    // at d_k = 128 on the tensor cores over the operand blocks
    if (!launched(blocks ? gdn::launch_kda_bwd_chain_tc(a, gdn::kDefaultWaitLimit, stream)
                         : gdn::launch_kda_bwd_chain(a, stream)))
        return GDN_ERR_CUDA;
    if (max_chunks > 0 && !launched(blocks ? gdn::launch_kda_bwd_local_tc(a, gdn::kDefaultWaitLimit, stream)
                                           : gdn::launch_kda_bwd_local(a, stream)))
        return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_prologue_fwd(const gdn_bf16* q_raw, const gdn_bf16* k_raw, const float* a, const float* b,
                            const float* A_log, const float* dt_bias, int gate_mode, float lower,
                            float beta_scale, gdn_bf16* q, gdn_bf16* k, float* g, gdn_bf16* beta,
                            int rows, int H, int d_k, cudaStream_t stream) {
    gdn_status st = check_prologue(rows, H, d_k, gate_mode, A_log);
    if (st != GDN_OK) return st;
    if (rows > 0 && (!a || !b || !g || !beta)) return GDN_ERR_INVALID_ARG;
    if ((q_raw == nullptr) != (q == nullptr) || (k_raw == nullptr) != (k == nullptr)) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q_raw, k_raw, a, b, A_log, dt_bias, q, k, g, beta};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::PrologueArgs pa{};
    pa.q_raw = q_raw; pa.k_raw = k_raw; pa.a = a; pa.b = b; pa.A_log = A_log; pa.dt_bias = dt_bias;
    pa.gate_mode = gate_mode; pa.lower = lower; pa.beta_scale = beta_scale;
    pa.q = q; pa.k = k; pa.g = g; pa.beta = beta; pa.rows = rows; pa.H = H; pa.d_k = d_k;
    if (!launched(gdn::launch_prologue_fwd(pa, stream), static_cast<long long>(rows) * H == 0 ? 0 : 1))
        return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_prologue_bwd(const gdn_bf16* q_raw, const gdn_bf16* k_raw, const float* a, const float* b,
                            const float* A_log, const float* dt_bias, int gate_mode, float lower,
                            float beta_scale, const gdn_bf16* dq, const gdn_bf16* dk, const float* dg,
                            const gdn_bf16* dbeta, gdn_bf16* dq_raw, gdn_bf16* dk_raw, float* da,
                            float* db, float* dA_log, float* ddt_bias, int rows, int H, int d_k,
                            cudaStream_t stream) {
    gdn_status st = check_prologue(rows, H, d_k, gate_mode, A_log);
    if (st != GDN_OK) return st;
    if (rows > 0 && (!a || !b || !dg || !dbeta || !da || !db)) return GDN_ERR_INVALID_ARG;
    if (q_raw && (!dq || !dq_raw)) return GDN_ERR_INVALID_ARG;
    if (k_raw && (!dk || !dk_raw)) return GDN_ERR_INVALID_ARG;
    const void* ptrs[] = {q_raw, k_raw, a, b, A_log, dt_bias, dq, dk, dg, dbeta, dq_raw, dk_raw,
                          da, db, dA_log, ddt_bias};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_MISALIGNED;
    gdn::PrologueArgs pa{};
    pa.q_raw = q_raw; pa.k_raw = k_raw; pa.a = a; pa.b = b; pa.A_log = A_log; pa.dt_bias = dt_bias;
    pa.gate_mode = gate_mode; pa.lower = lower; pa.beta_scale = beta_scale;
    pa.dq = dq; pa.dk = dk; pa.dg = dg; pa.dbeta = dbeta;
    pa.dq_raw = dq_raw; pa.dk_raw = dk_raw; pa.da = da; pa.db = db; pa.dA_log = dA_log; pa.ddt_bias = ddt_bias;
    pa.rows = rows; pa.H = H; pa.d_k = d_k;
    // the row kernel, then the per-head sums when dA_log or ddt_bias is asked for
    const int kernels = static_cast<long long>(rows) * H == 0 ? 0 : 1 + ((dA_log || ddt_bias) ? 1 : 0);
    if (!launched(gdn::launch_prologue_bwd(pa, stream), kernels)) return GDN_ERR_CUDA;
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
    gdn_status st = check_bwd(q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state, dq, dk, dv,
                              dg, dbeta, d_initial_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    const int varlen = cu_seqlens != nullptr;
    const BwdLayout L = bwd_layout(B, T, H, d_k, d_v, varlen);
    st = check_buffer(workspace, workspace_bytes, L.total);
    if (st != GDN_OK) return st;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    float* states = reinterpret_cast<float*>(ws + L.states);
    float* dstates = reinterpret_cast<float*>(ws + L.dstates);
    uint8_t* tiles = reinterpret_cast<uint8_t*>(ws + L.tiles);

    // T tiles of every chunk (chunk-parallel), then pass 1: chunk-start states
    // (forward state pass, no output)
    if (L.total > 0 && !launch_tiles(k, g, beta, cu_seqlens, tiles, B, T, H, d_k, err, stream)) return GDN_ERR_CUDA;
    gdn::FwdArgs f{};
    f.q = q; f.k = k; f.v = v; f.g = g; f.beta = beta; f.scale = scale;
    f.initial_state = initial_state; f.cu_seqlens = cu_seqlens;
    f.out = nullptr; f.final_state = nullptr; f.chunk_states = states; f.chunk_T = tiles;
    f.N = B; f.T = T; f.H = H; f.d_k = d_k; f.d_v = d_v; f.err = err;
    if (!launched(gdn::launch_fwd_ws(f, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
    return launch_bwd_passes(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta,
                             d_initial_state, B, T, H, d_k, d_v, states, dstates, tiles, err, stream);
}

size_t gdn_chunk_saved_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return saved_layout(B, T, H, d_k, d_v, varlen).total;
}

size_t gdn_chunk_bwd_saved_workspace_size(int B, int T, int H, int d_k, int d_v, int varlen) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK) return 0;
    return dstates_bytes(B, T, H, d_k, d_v, varlen);
}

gdn_status gdn_chunk_fwd_save(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                              const float* g, const gdn_bf16* beta, float scale,
                              const float* initial_state, const int32_t* cu_seqlens,
                              gdn_bf16* out, float* final_state,
                              int B, int T, int H, int d_k, int d_v,
                              void* saved, size_t saved_bytes, cudaStream_t stream) {
    gdn_status st = check_fwd(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    const SavedLayout L = saved_layout(B, T, H, d_k, d_v, cu_seqlens != nullptr);
    st = check_buffer(saved, saved_bytes, L.total);
    if (st != GDN_OK) return st;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    char* s = static_cast<char*>(saved);
    float* states = L.total ? reinterpret_cast<float*>(s + L.states) : nullptr;
    uint8_t* tiles = L.total ? reinterpret_cast<uint8_t*>(s + L.tiles) : nullptr;
    if (L.total > 0 && !launch_tiles(k, g, beta, cu_seqlens, tiles, B, T, H, d_k, err, stream)) return GDN_ERR_CUDA;
    // one chain pass writes the output, the final state and every chunk's start state
    gdn::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens;
    a.out = out; a.final_state = final_state; a.chunk_states = states; a.chunk_T = tiles;
    a.N = B; a.T = T; a.H = H; a.d_k = d_k; a.d_v = d_v; a.err = err;
    if (!launched(gdn::launch_fwd_ws(a, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // extern "C"

namespace {

gdn_status chunk_bwd_saved(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                           const gdn_bf16* beta, float scale, const int32_t* cu_seqlens, const gdn_bf16* d_out,
                           const float* d_final_state, gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                           gdn_bf16* dbeta, float* d_initial_state, int B, int T, int H, int d_k, int d_v,
                           const void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                           uint32_t local_wait_limit, int local_stall, cudaStream_t stream) {
    gdn_status st = check_bwd(q, k, v, g, beta, nullptr, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg,
                              dbeta, d_initial_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    const int varlen = cu_seqlens != nullptr;
    const SavedLayout L = saved_layout(B, T, H, d_k, d_v, varlen);
    st = check_buffer(saved, saved_bytes, L.total);
    if (st != GDN_OK) return st;
    st = check_buffer(workspace, workspace_bytes, dstates_bytes(B, T, H, d_k, d_v, varlen));
    if (st != GDN_OK) return st;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    const char* s = static_cast<const char*>(saved);
    const float* states = L.total ? reinterpret_cast<const float*>(s + L.states) : nullptr;
    const uint8_t* tiles = L.total ? reinterpret_cast<const uint8_t*>(s + L.tiles) : nullptr;
    return launch_bwd_passes(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta,
                             d_initial_state, B, T, H, d_k, d_v, states, static_cast<float*>(workspace), tiles,
                             err, stream, local_wait_limit, local_stall);
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_bwd_saved(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                               const float* g, const gdn_bf16* beta, float scale,
                               const int32_t* cu_seqlens,
                               const gdn_bf16* d_out, const float* d_final_state,
                               gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                               gdn_bf16* dbeta, float* d_initial_state,
                               int B, int T, int H, int d_k, int d_v,
                               const void* saved, size_t saved_bytes,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return chunk_bwd_saved(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta,
                           d_initial_state, B, T, H, d_k, d_v, saved, saved_bytes, workspace, workspace_bytes,
                           gdn::kDefaultWaitLimit, 0, stream);
}

gdn_status gdn_chunk_bwd_saved_wait_limit(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v,
                                          const float* g, const gdn_bf16* beta, float scale,
                                          const int32_t* cu_seqlens,
                                          const gdn_bf16* d_out, const float* d_final_state,
                                          gdn_bf16* dq, gdn_bf16* dk, gdn_bf16* dv, float* dg,
                                          gdn_bf16* dbeta, float* d_initial_state,
                                          int B, int T, int H, int d_k, int d_v,
                                          const void* saved, size_t saved_bytes,
                                          void* workspace, size_t workspace_bytes, uint32_t wait_limit,
                                          int stall_first_wait, cudaStream_t stream) {
    return chunk_bwd_saved(q, k, v, g, beta, scale, cu_seqlens, d_out, d_final_state, dq, dk, dv, dg, dbeta,
                           d_initial_state, B, T, H, d_k, d_v, saved, saved_bytes, workspace, workspace_bytes,
                           wait_limit ? wait_limit : gdn::kDefaultWaitLimit, stall_first_wait != 0, stream);
}

size_t gdn_chunk_fwd_split_workspace_size(int B, int T, int H, int d_k, int d_v, int nseg) {
    if (check_shapes(B, T, H, d_k, d_v) != GDN_OK || nseg < 1) return 0;
    if (static_cast<long long>(B) * T >= (1LL << 31)) return 0;
    return split_layout(B, T, H, d_k, d_v, split_segments(T, nseg)).total;
}

gdn_status gdn_chunk_fwd_split(const gdn_bf16* q, const gdn_bf16* k, const gdn_bf16* v, const float* g,
                               const gdn_bf16* beta, float scale, const float* initial_state, gdn_bf16* out,
                               float* final_state, int B, int T, int H, int d_k, int d_v, int nseg,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    gdn_status st = check_fwd(q, k, v, g, beta, initial_state, nullptr, out, final_state, B, T, H, d_k, d_v);
    if (st != GDN_OK) return st;
    if (nseg < 1) return GDN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * T >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if (T == 0)  // nothing to split: the state passes through
        return gdn_chunk_fwd(q, k, v, g, beta, scale, initial_state, nullptr, out, final_state, B, T, H, d_k, d_v,
                             nullptr, 0, stream);
    const int ns = split_segments(T, nseg);
    const SplitLayout L = split_layout(B, T, H, d_k, d_v, ns);
    st = check_buffer(workspace, workspace_bytes, L.total);
    if (st != GDN_OK) return st;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    char* w = static_cast<char*>(workspace);
    gdn::SplitArgs sa{};
    sa.cu = reinterpret_cast<int32_t*>(w + L.cu);
    sa.ident = reinterpret_cast<float*>(w + L.ident);
    sa.initial_state = initial_state;
    sa.m_fin = reinterpret_cast<const float*>(w + L.mfin);
    sa.b_fin = reinterpret_cast<const float*>(w + L.bfin);
    sa.starts = reinterpret_cast<float*>(w + L.starts);
    sa.final_state = final_state;
    sa.B = B; sa.T = T; sa.H = H; sa.d_k = d_k; sa.d_v = d_v; sa.nseg = ns;
    const int nseq = B * ns, rows = B * T;
    uint8_t* tiles = reinterpret_cast<uint8_t*>(w + L.tiles);
    if (!launched(gdn::launch_split_setup(sa, stream))) return GDN_ERR_CUDA;
    if (!launch_tiles(k, g, beta, sa.cu, tiles, nseq, rows, H, d_k, err, stream)) return GDN_ERR_CUDA;
    gdn::FwdArgs f{};
    f.q = q; f.k = k; f.g = g; f.beta = beta; f.scale = scale; f.cu_seqlens = sa.cu; f.chunk_T = tiles;
    f.N = nseq; f.T = rows; f.H = H; f.d_k = d_k; f.err = err; f.chunk_states = nullptr;
    if (ns == 1) {  // one segment per sequence: the plain chain over the packed sequences
        f.v = v; f.d_v = d_v; f.initial_state = initial_state; f.out = out; f.final_state = final_state;
        if (!launched(gdn::launch_fwd_ws(f, gdn::kDefaultWaitLimit, stream))) return GDN_ERR_CUDA;
        return GDN_OK;
    }
    // carries, side by side on two streams, outputs in fp32: b from a zero
    // start (output O_b; a sequence's first segment from its initial state),
    // M from the identity with zero values (output O_M, d_k columns); the
    // chain is linear in its start state, so a later segment's output is
    // O_b + O_M S_start
    cudaStream_t aux = aux_stream();
    if (!aux) return GDN_ERR_CUDA;
    cudaEvent_t forked = nullptr, joined = nullptr;
    if (cudaEventCreateWithFlags(&forked, cudaEventDisableTiming) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaEventCreateWithFlags(&joined, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(forked);
        return GDN_ERR_CUDA;
    }
    gdn_status rs = GDN_OK;
    do {
        if (cudaEventRecord(forked, stream) != cudaSuccess || cudaStreamWaitEvent(aux, forked, 0) != cudaSuccess) {
            rs = GDN_ERR_CUDA;
            break;
        }
        gdn::FwdArgs fb = f;
        // the zero-start run starts each sequence's first segment from its
        // initial state (the setup put it there), so that segment needs no
        // correction
        fb.v = v; fb.d_v = d_v; fb.initial_state = sa.starts; fb.out = nullptr;
        fb.out_f32 = reinterpret_cast<float*>(w + L.ob); fb.final_state = reinterpret_cast<float*>(w + L.bfin);
        if (!launched(gdn::launch_fwd_ws_f32(fb, gdn::kDefaultWaitLimit, stream))) rs = GDN_ERR_CUDA;
        gdn::FwdArgs fm = f;
        fm.v = reinterpret_cast<const gdn_bf16*>(w + L.zeros); fm.d_v = d_k; fm.initial_state = sa.ident;
        fm.out = nullptr; fm.out_f32 = reinterpret_cast<float*>(w + L.om);
        fm.out_split = 1;  // O_M as bf16 hi and lo planes: the correction's operand tiles
        fm.final_state = reinterpret_cast<float*>(w + L.mfin);
        if (cudaMemsetAsync(w + L.zeros, 0, 2ull * rows * H * d_k, aux) != cudaSuccess) rs = GDN_ERR_CUDA;
        else if (!launched(gdn::launch_fwd_ws_f32(fm, gdn::kDefaultWaitLimit, aux))) rs = GDN_ERR_CUDA;
        // the join is recorded whatever happened above, so that the caller's
        // stream never runs ahead of work left on the second stream
        if (cudaEventRecord(joined, aux) != cudaSuccess || cudaStreamWaitEvent(stream, joined, 0) != cudaSuccess)
            rs = GDN_ERR_CUDA;
    } while (false);
    cudaEventDestroy(forked);  // released once the recorded work has passed them
    cudaEventDestroy(joined);
    if (rs != GDN_OK) return rs;
    // true start states (and the final state), then every segment's output
    if (!launched(gdn::launch_split_compose(sa, stream))) return GDN_ERR_CUDA;
    gdn::SplitCorrectArgs ca{};
    ca.ob = reinterpret_cast<const float*>(w + L.ob);
    ca.om = reinterpret_cast<const float*>(w + L.om);
    ca.starts = sa.starts; ca.cu = sa.cu; ca.out = out;
    ca.nseq = nseq; ca.H = H; ca.d_k = d_k; ca.d_v = d_v; ca.rows = rows; ca.T = T; ca.nseg = ns; ca.err = err;
    ca.wait_limit = gdn::kDefaultWaitLimit;
    const int nch = (T + gdn::kChunk - 1) / gdn::kChunk;
    ca.max_chunks = (nch + ns - 1) / ns;
    if (!launched(gdn::launch_split_correct(ca, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_probe_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
    if (bytes % 16) return GDN_ERR_INVALID_ARG;
    if (bytes == 0) return GDN_OK;
    if (!src || !dst) return GDN_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return GDN_ERR_MISALIGNED;
    if (!launched(gdn::launch_probe_copy(src, dst, bytes, stream))) return GDN_ERR_CUDA;
    return GDN_OK;
}

gdn_status gdn_probe_gemm_bf16(const gdn_bf16* A, const gdn_bf16* B, gdn_bf16* C, int M, int N, int K,
                               cudaStream_t stream) {
    if (M <= 0 || N <= 0 || K <= 0) return GDN_ERR_INVALID_ARG;
    if (M % 128 || N % 256 || K % 64) return GDN_ERR_UNSUPPORTED;
    if (M > 65536 || N > 65536 || K > 65536) return GDN_ERR_UNSUPPORTED;
    if (!A || !B || !C) return GDN_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GDN_ERR_MISALIGNED;
    int* err = error_word();
    if (!err) return GDN_ERR_CUDA;
    if (!launched(gdn::launch_probe_gemm(A, B, C, M, N, K, err, stream))) return GDN_ERR_CUDA;
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

// kda_fwd_noalloc: the chunked forward with its workspace in a fixed,
// statically allocated device array instead of memory from cudaMalloc.
//
// Some callers cannot allocate device memory at the point where they run the
// forward: a framework whose allocator owns all device memory and forbids
// out-of-band allocations, real-time serving loops that must not enter the
// driver's allocator, and embedding hosts that own all device memory and hand
// the library only tensors.  For them this entry point uses a
// file-scope __device__ array of KDA_NOALLOC_WS_BYTES (64 MiB), which every GPU
// that loads the library holds until the process exits.
#include <cstdint>
#include <mutex>

#include "kda_common.cuh"

namespace kda {
struct FwdWorkspace;
size_t fwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, FwdWorkspace *ws, char *base);
}  // namespace kda

extern "C" int kda_fwd_ws(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                          const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
                          float *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v,
                          int K, int V, kda_bf16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream);

namespace {

// The shared scratch.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_ws[KDA_NOALLOC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_ws_addr[kMaxDevices] = {nullptr};

// Once per device, with that device current: the array's device address.
int noalloc_ws_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_ws_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
        g_ws_addr[dev] = p;
    }
    *addr = g_ws_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" int kda_fwd_noalloc(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                               const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
                               const float *initial_state, float *final_state, const int32_t *cu_seqlens, int N,
                               int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
                               cudaStream_t stream) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || (cu_seqlens && N < 0)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda::fwd_workspace_bytes(cu_seqlens ? N : 0, B, T, H_v, cu_seqlens != nullptr, nullptr,
                                                 nullptr);
    if (need > (size_t)KDA_NOALLOC_WS_BYTES) return KDA_ERR_WORKSPACE;
    void *ws = nullptr;
    const int rc = noalloc_ws_address(&ws);
    if (rc != KDA_OK) return rc;
    // Nothing in the workspace has to start at zero: every call's plan kernel
    // rewrites the header and tables, and each intermediate is written by the
    // intra-chunk kernel before the scan reads it.
    return kda_fwd_ws(q, k, v, graw, b, A_log, scale, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                      K, V, out, ws, (size_t)KDA_NOALLOC_WS_BYTES, stream);
}

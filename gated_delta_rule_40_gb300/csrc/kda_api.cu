// C-ABI entry points of libkda: argument validation, workspace handling and
// kernel launches.  See include/kda.h for the contract.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "kda_common.cuh"

namespace kda {
__device__ int g_kda_status = 0;

cudaError_t launch_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                          const uint16_t *b, const float *A_log, float scale, float *state, int B, int H_qk,
                          int H_v, uint16_t *out, cudaStream_t stream);
cudaError_t launch_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                       const int32_t *cu, int N, int B, int T, int H_qk, int H_v, uint16_t *out, void *ws_ptr,
                       cudaStream_t stream, int *launches);
cudaError_t launch_fwd_scalar_gate(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                   const uint16_t *b, const float *A_log, float scale, const float *init,
                                   float *fin, const int32_t *cu, int N, int B, int T, int H_qk, int H_v,
                                   uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches);
cudaError_t launch_decode_tokens(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                 const uint16_t *b, const float *A_log, float scale, void *state, bool bf16_state,
                                 int B, int Tq, int H_qk, int H_v, uint16_t *out, cudaStream_t stream);
cudaError_t launch_la_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *slope, float scale,
                          const float *init, float *fin, const int32_t *cu, int N, int B, int T, int H_qk, int H_v,
                          uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches);
size_t la_workspace_bytes(int N, int B, int T, bool varlen);
cudaError_t launch_la_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *slope, float scale,
                             float *state, int B, int H_qk, int H_v, uint16_t *out, cudaStream_t stream);
size_t bwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, int grid);
int bwd_grid(int nseq, int H_v);
cudaError_t launch_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                       const uint16_t *b, const float *A_log, float scale, const float *init, const int32_t *cu, int N,
                       int B, int T, int H_qk, int H_v, const uint16_t *dout, const float *dht, float *dq, float *dk,
                       float *dv, float *dgraw, float *db, float *dA_log, float *dh0, void *ws_ptr, int grid,
                       cudaStream_t stream, int *launches);
cudaError_t launch_fwd_bf16_state(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                  const uint16_t *b, const float *A_log, float scale, const uint16_t *init,
                                  uint16_t *fin, const int32_t *cu, int N, int B, int T, int H_qk, int H_v,
                                  uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches);
struct FwdWorkspace;
size_t fwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, FwdWorkspace *ws, char *base);

// ---- per-kernel event timing (measurement aid, off by default)
namespace {
constexpr int kMaxTimed = 8;
struct TimingState {
    bool enabled = false;
    int n = 0;
    const char *names[kMaxTimed] = {nullptr};
    cudaEvent_t ev[kMaxTimed + 1] = {nullptr};
};
thread_local TimingState t_timing;
}  // namespace

int timing_enable(bool on) {
    TimingState &t = t_timing;
    if (on && !t.ev[0]) {
        for (int i = 0; i <= kMaxTimed; ++i)
            if (cudaEventCreate(&t.ev[i]) != cudaSuccess) return KDA_ERR_CUDA;
    }
    t.enabled = on;
    t.n = 0;
    return KDA_OK;
}
void timing_begin(cudaStream_t s) {
    TimingState &t = t_timing;
    t.n = 0;
    if (t.enabled) cudaEventRecord(t.ev[0], s);
}
void timing_mark(const char *name, cudaStream_t s) {
    TimingState &t = t_timing;
    if (!t.enabled || t.n >= kMaxTimed) return;
    t.names[t.n] = name;
    cudaEventRecord(t.ev[t.n + 1], s);
    ++t.n;
}
int timing_read(float *ms, const char **names, int max_n) {
    TimingState &t = t_timing;
    if (!t.enabled) return 0;
    int n = t.n < max_n ? t.n : max_n;
    for (int i = 0; i < n; ++i) {
        if (cudaEventSynchronize(t.ev[i + 1]) != cudaSuccess) return KDA_ERR_CUDA;
        float v = 0.f;
        cudaEventElapsedTime(&v, t.ev[i], t.ev[i + 1]);
        if (ms) ms[i] = v;
        if (names) names[i] = t.names[i];
    }
    return n;
}
// ---- workspaces of the allocating entry points: one stream-ordered pool per device, created on
// first use, whose release threshold is unbounded.  Memory freed at the end of a call stays
// mapped in the pool when the caller synchronises, so the next call reuses it instead of
// mapping fresh pages (1.8 GB of chunk records for a 2 x 16384-token, 32-head forward took
// about 1.4 ms to map on every call that followed a synchronisation).  kda_release_cached_memory
// returns what no call holds to the driver.
namespace {
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {nullptr};

cudaError_t device_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pool[dev] = pool;
    }
    *out = g_pool[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t stream) {
    cudaMemPool_t pool = nullptr;
    const cudaError_t e = device_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}
cudaError_t ws_free(void *p, cudaStream_t stream) { return cudaFreeAsync(p, stream); }

int release_cached_memory() {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (int d = 0; d < kMaxDevices; ++d)
        if (g_pool[d] && cudaMemPoolTrimTo(g_pool[d], 0) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}
}  // namespace kda

namespace kda {
// One thread waits, with a small bound, on an mbarrier phase that nothing completes; the
// bounded wait gives up and records KDA_ERR_DEVICE_TIMEOUT, exactly as a stalled hand-off
// in the forward kernels would, and the kernel returns normally.
__global__ void selftest_wait_timeout_kernel(uint32_t limit) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t mb = smem_u32(&bar);
    mbar_init(mb, 1);
    mbar_fence_init();
    if (!mbar_spin(mb, 0, limit)) set_status(KDA_ERR_DEVICE_TIMEOUT);
}
}  // namespace kda

namespace {
thread_local int t_last_launches = 0;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Work items carry 32-bit block indices: (sequence, value head) chains times up to four row
// blocks (the scan's two V blocks, the backward's four row quarters) and (b, h) decode pairs
// must stay below 2^31, or a launch would cover only part of the work.
constexpr long long kMaxItems = 0x7fffffffLL;
bool chains_fit(long long nseq, int H_v) { return nseq * H_v * 4 <= kMaxItems; }
bool pairs_fit(int B, int H_v) { return (long long)B * H_v <= kMaxItems; }

int validate_fwd(const void *q, const void *k, const void *v, const void *graw, const void *b,
                 const void *A_log, const void *init, const void *fin, const int32_t *cu, int N, int B, int T,
                 int H_qk, int H_v, int K, int V, const void *out) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0) return KDA_ERR_INVALID_ARG;
    if (H_v % H_qk != 0) return KDA_ERR_INVALID_ARG;
    if (cu) {
        if (B != 1 || N < 0) return KDA_ERR_INVALID_ARG;
    }
    const long long tokens = (long long)B * T;
    if (tokens > 0x7fffffffLL || !chains_fit(cu ? N : B, H_v)) return KDA_ERR_INVALID_ARG;
    if (tokens > 0) {
        if (!q || !k || !v || !graw || !b || !A_log || !out) return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(graw) || !aligned16(out))
            return KDA_ERR_INVALID_ARG;
    }
    if ((init && !aligned16(init)) || (fin && !aligned16(fin))) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}
}  // namespace

extern "C" {

const char *kda_status_string(int code) {
    switch (code) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported head dimension (K and V must be 128)";
        case KDA_ERR_CUDA: return "CUDA runtime or launch error";
        case KDA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
        case KDA_ERR_BAD_SEQLENS: return "malformed cu_seqlens";
        case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        default: return "unknown status";
    }
}

int kda_get_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, kda::g_kda_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(kda::g_kda_status, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

int kda_last_launch_count(void) { return t_last_launches; }

int kda_selftest_wait_timeout(cudaStream_t stream) {
    kda::selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(1u << 12);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_set_kernel_timing(int enable) { return kda::timing_enable(enable != 0); }

int kda_kernel_times(float *ms, const char **names, int max_n) { return kda::timing_read(ms, names, max_n); }

int kda_release_cached_memory(void) { return kda::release_cached_memory(); }

size_t kda_fwd_workspace_size(int N, int B, int T, int H_qk, int H_v, int K, int V) {
    if (K != kda::KD || V != kda::KD || B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || N < 0) return 0;
    // varlen bound: every sequence adds at most one partial chunk
    const size_t a = kda::fwd_workspace_bytes(N, B, T, H_v, true, nullptr, nullptr);
    const size_t b = kda::fwd_workspace_bytes(N, B, T, H_v, false, nullptr, nullptr);
    return a > b ? a : b;
}

int kda_fwd_ws(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
               const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
               float *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K,
               int V, kda_bf16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = validate_fwd(q, k, v, graw, b, A_log, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                          K, V, out);
    if (rc != KDA_OK) return rc;
    const size_t need = kda::fwd_workspace_bytes(cu_seqlens ? N : 0, B, T, H_v, cu_seqlens != nullptr, nullptr,
                                                 nullptr);
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need) return KDA_ERR_WORKSPACE;
    int launches = 0;
    cudaError_t e = kda::launch_fwd(q, k, v, graw, b, A_log, scale, initial_state, final_state, cu_seqlens,
                                    cu_seqlens ? N : 0, B, T, H_qk, H_v, out, ws, stream, &launches);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    t_last_launches = launches;
    return KDA_OK;
}

int kda_fwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
            const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state, float *final_state,
            const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
            cudaStream_t stream) {
    int rc = validate_fwd(q, k, v, graw, b, A_log, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                          K, V, out);
    if (rc != KDA_OK) return rc;
    const size_t need = kda::fwd_workspace_bytes(cu_seqlens ? N : 0, B, T, H_v, cu_seqlens != nullptr, nullptr,
                                                 nullptr);
    void *ws = nullptr;
    if (kda::ws_alloc(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    rc = kda_fwd_ws(q, k, v, graw, b, A_log, scale, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                    K, V, out, ws, need, stream);
    if (kda::ws_free(ws, stream) != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
    return rc;
}

int kda_fwd_bf16_state(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                       const kda_bf16_t *b, const float *A_log, float scale, const kda_bf16_t *initial_state,
                       kda_bf16_t *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v,
                       int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    int rc = validate_fwd(q, k, v, graw, b, A_log, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                          K, V, out);
    if (rc != KDA_OK) return rc;
    const size_t need = kda::fwd_workspace_bytes(cu_seqlens ? N : 0, B, T, H_v, cu_seqlens != nullptr, nullptr,
                                                 nullptr);
    void *ws = nullptr;
    if (kda::ws_alloc(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    int launches = 0;
    const cudaError_t e = kda::launch_fwd_bf16_state(q, k, v, graw, b, A_log, scale, initial_state, final_state,
                                                     cu_seqlens, cu_seqlens ? N : 0, B, T, H_qk, H_v, out, ws, stream,
                                                     &launches);
    rc = e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    if (rc == KDA_OK) t_last_launches = launches;
    if (kda::ws_free(ws, stream) != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
    return rc;
}

int kda_fwd_scalar_gate(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                        const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
                        float *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K,
                        int V, kda_bf16_t *out, cudaStream_t stream) {
    int rc = validate_fwd(q, k, v, graw, b, A_log, initial_state, final_state, cu_seqlens, N, B, T, H_qk, H_v,
                          K, V, out);
    if (rc != KDA_OK) return rc;
    const size_t need = kda::fwd_workspace_bytes(cu_seqlens ? N : 0, B, T, H_v, cu_seqlens != nullptr, nullptr,
                                                 nullptr);
    void *ws = nullptr;
    if (kda::ws_alloc(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    int launches = 0;
    const cudaError_t e = kda::launch_fwd_scalar_gate(q, k, v, graw, b, A_log, scale, initial_state, final_state,
                                                      cu_seqlens, cu_seqlens ? N : 0, B, T, H_qk, H_v, out, ws,
                                                      stream, &launches);
    rc = e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    if (rc == KDA_OK) t_last_launches = launches;
    if (kda::ws_free(ws, stream) != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
    return rc;
}

int kda_decode_tokens(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                      const kda_bf16_t *b, const float *A_log, float scale, void *state, int state_is_bf16, int B,
                      int Tq, int H_qk, int H_v, int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || Tq < 1 || Tq > KDA_DECODE_MAX_TOKENS || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0 ||
        (state_is_bf16 != 0 && state_is_bf16 != 1) || !pairs_fit(B, H_v))
        return KDA_ERR_INVALID_ARG;
    if (B == 0) {
        t_last_launches = 0;
        return KDA_OK;
    }
    if (!q || !k || !v || !graw || !b || !A_log || !state || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(graw) || !aligned16(state) ||
        !aligned16(out))
        return KDA_ERR_INVALID_ARG;
    kda::timing_begin(stream);
    const cudaError_t e = kda::launch_decode_tokens(q, k, v, graw, b, A_log, scale, state, state_is_bf16 != 0, B, Tq,
                                                    H_qk, H_v, out, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    kda::timing_mark("decode_tokens_kernel", stream);
    t_last_launches = 1;
    return KDA_OK;
}

int kda_decode_step(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                    const kda_bf16_t *b, const float *A_log, float scale, float *state, int B, int H_qk, int H_v,
                    int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0 || !pairs_fit(B, H_v)) return KDA_ERR_INVALID_ARG;
    if (B == 0) {
        t_last_launches = 0;
        return KDA_OK;
    }
    if (!q || !k || !v || !graw || !b || !A_log || !state || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(graw) || !aligned16(state) ||
        !aligned16(out))
        return KDA_ERR_INVALID_ARG;
    kda::timing_begin(stream);
    cudaError_t e = kda::launch_decode(q, k, v, graw, b, A_log, scale, state, B, H_qk, H_v, out, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    kda::timing_mark("decode_kernel", stream);
    t_last_launches = 1;
    return KDA_OK;
}

namespace {
int validate_bwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                 const kda_bf16_t *b, const float *A_log, const float *initial_state, const int32_t *cu_seqlens, int N,
                 int B, int T, int H_qk, int H_v, int K, int V, const kda_bf16_t *dout, const float *dht, float *dq,
                 float *dk, float *dv, float *dgraw, float *db, float *dA_log, float *dh0) {
    int rc = validate_fwd(q, k, v, graw, b, A_log, initial_state, nullptr, cu_seqlens, N, B, T, H_qk, H_v, K, V,
                          dout);
    if (rc != KDA_OK) return rc;
    const long long tokens = (long long)B * T;
    if (!A_log || !dA_log || !dh0) return KDA_ERR_INVALID_ARG;
    if (tokens > 0 && (!dq || !dk || !dv || !dgraw || !db)) return KDA_ERR_INVALID_ARG;
    if ((dht && !aligned16(dht)) || !aligned16(dh0) ||
        (tokens > 0 && (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dgraw))))
        return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}
}  // namespace

size_t kda_bwd_workspace_size(int N, int B, int T, int H_qk, int H_v, int K, int V) {
    if (K != kda::KD || V != kda::KD || B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || N < 0) return 0;
    const size_t a = kda::bwd_workspace_bytes(N, B, T, H_v, true, 0);
    const size_t b = kda::bwd_workspace_bytes(N, B, T, H_v, false, 0);
    return a > b ? a : b;
}

int kda_bwd_ws(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
               const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
               const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V,
               const kda_bf16_t *dout, const float *dht, float *dq, float *dk, float *dv, float *dgraw, float *db,
               float *dA_log, float *dh0, void *ws, size_t ws_bytes, cudaStream_t stream) {
    int rc = validate_bwd(q, k, v, graw, b, A_log, initial_state, cu_seqlens, N, B, T, H_qk, H_v, K, V, dout, dht,
                          dq, dk, dv, dgraw, db, dA_log, dh0);
    if (rc != KDA_OK) return rc;
    const bool varlen = cu_seqlens != nullptr;
    const size_t need = kda::bwd_workspace_bytes(varlen ? N : 0, B, T, H_v, varlen, 0);
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need) return KDA_ERR_WORKSPACE;
    int launches = 0;
    kda::timing_begin(stream);
    const cudaError_t e = kda::launch_bwd(q, k, v, graw, b, A_log, scale, initial_state, cu_seqlens, varlen ? N : 0,
                                          B, T, H_qk, H_v, dout, dht, dq, dk, dv, dgraw, db, dA_log, dh0, ws,
                                          kda::bwd_grid(varlen ? N : B, H_v), stream, &launches);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    t_last_launches = launches;
    return KDA_OK;
}

int kda_bwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
            const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
            const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V, const kda_bf16_t *dout,
            const float *dht, float *dq, float *dk, float *dv, float *dgraw, float *db, float *dA_log, float *dh0,
            cudaStream_t stream) {
    int rc = validate_bwd(q, k, v, graw, b, A_log, initial_state, cu_seqlens, N, B, T, H_qk, H_v, K, V, dout, dht,
                          dq, dk, dv, dgraw, db, dA_log, dh0);
    if (rc != KDA_OK) return rc;
    const bool varlen = cu_seqlens != nullptr;
    const size_t need = kda::bwd_workspace_bytes(varlen ? N : 0, B, T, H_v, varlen, 0);
    void *ws = nullptr;
    if (kda::ws_alloc(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    rc = kda_bwd_ws(q, k, v, graw, b, A_log, scale, initial_state, cu_seqlens, N, B, T, H_qk, H_v, K, V, dout, dht,
                    dq, dk, dv, dgraw, db, dA_log, dh0, ws, need, stream);
    if (kda::ws_free(ws, stream) != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
    return rc;
}

int kda_la_fwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const float *slope, float scale,
               const float *initial_state, float *final_state, const int32_t *cu_seqlens, int N, int B, int T,
               int H_qk, int H_v, int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || N < 0)) return KDA_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    const int nseq = cu_seqlens ? N : B;
    if (tokens > 0x7fffffffLL || !chains_fit(nseq, H_v)) return KDA_ERR_INVALID_ARG;
    if (nseq > 0 && !slope) return KDA_ERR_INVALID_ARG;
    if (tokens > 0) {
        if (!q || !k || !v || !out) return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return KDA_ERR_INVALID_ARG;
    }
    if ((initial_state && !aligned16(initial_state)) || (final_state && !aligned16(final_state)))
        return KDA_ERR_INVALID_ARG;
    const size_t need = kda::la_workspace_bytes(cu_seqlens ? N : 0, B, T, cu_seqlens != nullptr);
    void *ws = nullptr;
    if (kda::ws_alloc(&ws, need, stream) != cudaSuccess) return KDA_ERR_CUDA;
    int launches = 0;
    kda::timing_begin(stream);
    const cudaError_t e = kda::launch_la_fwd(q, k, v, slope, scale, initial_state, final_state, cu_seqlens,
                                             cu_seqlens ? N : 0, B, T, H_qk, H_v, out, ws, stream, &launches);
    int rc = e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    if (rc == KDA_OK) {
        kda::timing_mark("la_fwd_kernel", stream);
        t_last_launches = launches;
    }
    if (kda::ws_free(ws, stream) != cudaSuccess && rc == KDA_OK) rc = KDA_ERR_CUDA;
    return rc;
}

int kda_la_decode(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const float *slope, float scale,
                  float *state, int B, int H_qk, int H_v, int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    if (K != kda::KD || V != kda::KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0 || !pairs_fit(B, H_v)) return KDA_ERR_INVALID_ARG;
    if (B == 0) {
        t_last_launches = 0;
        return KDA_OK;
    }
    if (!q || !k || !v || !slope || !state || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(state)) return KDA_ERR_INVALID_ARG;
    kda::timing_begin(stream);
    const cudaError_t e = kda::launch_la_decode(q, k, v, slope, scale, state, B, H_qk, H_v, out, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    kda::timing_mark("la_decode_kernel", stream);
    t_last_launches = 1;
    return KDA_OK;
}

}  // extern "C"

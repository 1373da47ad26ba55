// kda_fwd_host: the chunked forward on host buffers.  The inputs are copied to
// the device and the results back inside the call, split into groups of value
// heads so that the copies of one group overlap the kernels of another: the
// host link is the bottleneck of such a call (its bytes take several times the
// kernels' time), so the kernels and the return copies hide behind the input
// copies.
#include <cstdint>
#include <mutex>

#include "kda_common.cuh"

namespace kda {
struct FwdWorkspace;
size_t fwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, FwdWorkspace *ws, char *base);
cudaError_t launch_fwd_heads(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                             const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                             const int32_t *cu, int N, int B, int T, int H_qk, int H_v, int h0, int Hw, bool plan,
                             uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches);
}  // namespace kda

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGroups = 4;
std::mutex g_stream_mutex;
cudaStream_t g_h2d[kMaxDevices] = {nullptr}, g_d2h[kMaxDevices] = {nullptr};

// Once per device, with that device current: the two copy streams.
int copy_streams(cudaStream_t *h2d, cudaStream_t *d2h) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_stream_mutex);
    if (!g_h2d[dev]) {
        if (cudaStreamCreateWithFlags(&g_h2d[dev], cudaStreamNonBlocking) != cudaSuccess) return KDA_ERR_CUDA;
        if (cudaStreamCreateWithFlags(&g_d2h[dev], cudaStreamNonBlocking) != cudaSuccess) return KDA_ERR_CUDA;
    }
    *h2d = g_h2d[dev];
    *d2h = g_d2h[dev];
    return KDA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Rows of `width` bytes at `pitch` (the same on both sides): one head group of a
// [rows][heads][...] tensor.
cudaError_t copy_rows(void *dst, const void *src, size_t width, size_t pitch, size_t rows, cudaMemcpyKind kind,
                      cudaStream_t s) {
    if (rows == 0 || width == 0) return cudaSuccess;
    if (width == pitch) return cudaMemcpyAsync(dst, src, width * rows, kind, s);
    return cudaMemcpy2DAsync(dst, pitch, src, pitch, width, rows, kind, s);
}

}  // namespace

extern "C" int kda_fwd_host(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                            const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
                            float *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v,
                            int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    using kda::KD;
    if (K != KD || V != KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || N < 0)) return KDA_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    if (tokens > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (tokens > 0 && (!q || !k || !v || !graw || !b || !A_log || !out)) return KDA_ERR_INVALID_ARG;
    const bool varlen = cu_seqlens != nullptr;
    const int nseq = varlen ? N : B;

    // head groups: a divisor of H_qk (so every group holds whole q/k head groups)
    int P = 1;
    for (int c = kMaxGroups; c > 1; --c)
        if (tokens > 0 && H_qk % c == 0) {
            P = c;
            break;
        }
    const int hq_p = H_qk / P, hv_p = H_v / P;

    const size_t qk_row = (size_t)H_qk * KD * 2, v_row = (size_t)H_v * KD * 2;   // bytes per token
    const size_t st_row = (size_t)H_v * KD * KD * 4;                              // bytes per sequence
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const size_t o_q = take(tokens * qk_row), o_k = take(tokens * qk_row);
    const size_t o_v = take(tokens * v_row), o_g = take(tokens * v_row), o_out = take(tokens * v_row);
    const size_t o_b = take((size_t)tokens * H_v * 2), o_a = take((size_t)H_v * 4);
    const size_t o_init = take(initial_state ? nseq * st_row : 0), o_fin = take(final_state ? nseq * st_row : 0);
    const size_t o_cu = take(varlen ? (size_t)(N + 1) * 4 : 0);
    const size_t o_ws = take(kda::fwd_workspace_bytes(varlen ? N : 0, B, T, hv_p, varlen, nullptr, nullptr));

    cudaStream_t h2d = nullptr, d2h = nullptr;
    int rc = copy_streams(&h2d, &d2h);
    if (rc != KDA_OK) return rc;
    char *base = nullptr;
    if (cudaMallocAsync((void **)&base, off, stream) != cudaSuccess) return KDA_ERR_CUDA;
    cudaEvent_t ev_start, ev_end, ev_in[kMaxGroups], ev_out[kMaxGroups];
    cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming);
    cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming);
    for (int p = 0; p < P; ++p) {
        cudaEventCreateWithFlags(&ev_in[p], cudaEventDisableTiming);
        cudaEventCreateWithFlags(&ev_out[p], cudaEventDisableTiming);
    }
    auto dptr = [&](size_t o) { return (void *)(base + o); };
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t x) {
        if (x != cudaSuccess && e == cudaSuccess) e = x;
        return e == cudaSuccess;
    };
    int launches = 0;

    // inputs: the whole-tensor parts, then each head group
    ok(cudaEventRecord(ev_start, stream));
    ok(cudaStreamWaitEvent(h2d, ev_start, 0));
    if (tokens > 0) {
        ok(cudaMemcpyAsync(dptr(o_b), b, (size_t)tokens * H_v * 2, cudaMemcpyHostToDevice, h2d));
        ok(cudaMemcpyAsync(dptr(o_a), A_log, (size_t)H_v * 4, cudaMemcpyHostToDevice, h2d));
    }
    if (varlen) ok(cudaMemcpyAsync(dptr(o_cu), cu_seqlens, (size_t)(N + 1) * 4, cudaMemcpyHostToDevice, h2d));
    for (int p = 0; p < P && e == cudaSuccess; ++p) {
        const size_t qo = (size_t)p * hq_p * KD * 2, vo = (size_t)p * hv_p * KD * 2;
        const size_t qw = (size_t)hq_p * KD * 2, vw = (size_t)hv_p * KD * 2;
        ok(copy_rows((char *)dptr(o_q) + qo, (const char *)q + qo, qw, qk_row, tokens, cudaMemcpyHostToDevice, h2d));
        ok(copy_rows((char *)dptr(o_k) + qo, (const char *)k + qo, qw, qk_row, tokens, cudaMemcpyHostToDevice, h2d));
        ok(copy_rows((char *)dptr(o_v) + vo, (const char *)v + vo, vw, v_row, tokens, cudaMemcpyHostToDevice, h2d));
        ok(copy_rows((char *)dptr(o_g) + vo, (const char *)graw + vo, vw, v_row, tokens, cudaMemcpyHostToDevice,
                     h2d));
        if (initial_state) {
            const size_t so = (size_t)p * hv_p * KD * KD * 4, sw = (size_t)hv_p * KD * KD * 4;
            ok(copy_rows((char *)dptr(o_init) + so, (const char *)initial_state + so, sw, st_row, nseq,
                         cudaMemcpyHostToDevice, h2d));
        }
        ok(cudaEventRecord(ev_in[p], h2d));
    }
    // kernels, group by group on the caller's stream (the chunk tables are built once)
    for (int p = 0; p < P && e == cudaSuccess; ++p) {
        ok(cudaStreamWaitEvent(stream, ev_in[p], 0));
        int n = 0;
        ok(kda::launch_fwd_heads((const uint16_t *)dptr(o_q), (const uint16_t *)dptr(o_k),
                                 (const uint16_t *)dptr(o_v), (const uint16_t *)dptr(o_g),
                                 (const uint16_t *)dptr(o_b), (const float *)dptr(o_a), scale,
                                 initial_state ? (const float *)dptr(o_init) : nullptr,
                                 final_state ? (float *)dptr(o_fin) : nullptr,
                                 varlen ? (const int32_t *)dptr(o_cu) : nullptr, varlen ? N : 0, B, T, H_qk, H_v,
                                 p * hv_p, hv_p, p == 0, (uint16_t *)dptr(o_out), dptr(o_ws), stream, &n));
        launches += n;
        ok(cudaEventRecord(ev_out[p], stream));
    }
    // results, group by group
    for (int p = 0; p < P && e == cudaSuccess; ++p) {
        ok(cudaStreamWaitEvent(d2h, ev_out[p], 0));
        const size_t vo = (size_t)p * hv_p * KD * 2, vw = (size_t)hv_p * KD * 2;
        ok(copy_rows((char *)out + vo, (const char *)dptr(o_out) + vo, vw, v_row, tokens, cudaMemcpyDeviceToHost,
                     d2h));
        if (final_state) {
            const size_t so = (size_t)p * hv_p * KD * KD * 4, sw = (size_t)hv_p * KD * KD * 4;
            ok(copy_rows((char *)final_state + so, (const char *)dptr(o_fin) + so, sw, st_row, nseq,
                         cudaMemcpyDeviceToHost, d2h));
        }
    }
    ok(cudaEventRecord(ev_end, d2h));
    ok(cudaStreamWaitEvent(stream, ev_end, 0));
    const cudaError_t ef = cudaFreeAsync(base, stream);
    cudaEventDestroy(ev_start);
    cudaEventDestroy(ev_end);
    for (int p = 0; p < P; ++p) {
        cudaEventDestroy(ev_in[p]);
        cudaEventDestroy(ev_out[p]);
    }
    (void)launches;
    if (e != cudaSuccess || ef != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

// kda_fwd_host: the chunked forward on host buffers.  The inputs are copied to
// the device and the results back inside the call, in pieces of consecutive
// tokens so that the copies of one piece overlap the kernels of the previous
// one: the host link is the bottleneck of such a call (its bytes take several
// times the kernels' time), so the kernels hide behind the input copies and
// only the last piece's kernels and output copy remain exposed.
//
// A piece is a token range of the packed [sequence][token] layout (dense input
// is B sequences of length T); a sequence that crosses a piece boundary is cut
// at a multiple of the chunk length from its start and its state is carried on
// the device from one piece to the next, which is exactly the chunking and the
// arithmetic of a single call.
#include <cstdint>
#include <mutex>
#include <vector>

#include "kda_common.cuh"

namespace kda {
struct FwdWorkspace;
size_t fwd_workspace_bytes(int N, int B, int T, int H_v, bool varlen, FwdWorkspace *ws, char *base);
cudaError_t launch_fwd_heads(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                             const uint16_t *b, const float *A_log, float scale, const float *init, float *fin,
                             const int32_t *cu, int N, int B, int T, int H_qk, int H_v, int h0, int Hw, bool plan,
                             uint16_t *out, void *ws_ptr, cudaStream_t stream, int *launches);
cudaError_t ws_alloc(void **p, size_t bytes, cudaStream_t stream);
cudaError_t ws_free(void *p, cudaStream_t stream);
}  // namespace kda

namespace {

constexpr int kMaxDevices = 64;
// Up to kMaxPieces equal pieces of at least kMinPieceTokens tokens each (the last one cut into
// a half and two quarters when there are four or more): more pieces shorten the exposed tail
// (the last piece's kernels and output copy) at the price of more launches.
constexpr int kMaxPieces = 16;
constexpr long long kMinPieceTokens = 2048;
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

}  // namespace

extern "C" int kda_fwd_host(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
                            const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
                            float *final_state, const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v,
                            int K, int V, kda_bf16_t *out, cudaStream_t stream) {
    using kda::CH;
    using kda::KD;
    if (K != KD || V != KD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H_qk <= 0 || H_v <= 0 || H_v % H_qk != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || N < 0)) return KDA_ERR_INVALID_ARG;
    const long long tokens = (long long)B * T;
    if (tokens > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (tokens > 0 && (!q || !k || !v || !graw || !b || !A_log || !out)) return KDA_ERR_INVALID_ARG;
    const int nseq = cu_seqlens ? N : B;
    if ((long long)nseq * H_v * 4 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;   // 32-bit work-item indices

    // packed sequence boundaries (host copy; checked here, so a malformed array is an error return)
    std::vector<int32_t> cu((size_t)nseq + 1);
    for (int i = 0; i <= nseq; ++i) cu[i] = cu_seqlens ? cu_seqlens[i] : (int32_t)((long long)i * T);
    if (cu[0] != 0 || cu[nseq] != tokens) return KDA_ERR_BAD_SEQLENS;
    for (int i = 0; i < nseq; ++i)
        if (cu[i + 1] < cu[i]) return KDA_ERR_BAD_SEQLENS;

    // pieces [t0, t1): about tokens / P each, cut at a chunk boundary of the sequence they fall in;
    // with four or more pieces the last one is cut again at 1/2 and 3/4, so that the work left
    // once the last input has arrived (that piece's kernels and output copy) is a quarter piece
    const long long pmax = tokens / kMinPieceTokens;
    const int P = pmax < 1 ? 1 : (pmax > kMaxPieces ? kMaxPieces : (int)pmax);
    std::vector<long long> targets;
    for (int p = 1; p < P; ++p) targets.push_back(tokens * p / P);
    if (P >= 4) {
        targets.push_back((tokens * (2 * P - 1)) / (2 * P));
        targets.push_back((tokens * (4 * P - 1)) / (4 * P));
    }
    std::vector<int> cuts = {0};
    for (const long long target : targets) {
        int s = 0;
        while (s < nseq && cu[s + 1] <= target) ++s;
        long long t = s < nseq ? cu[s] + ((target - cu[s] + CH / 2) / CH) * CH : tokens;
        if (s < nseq && t > cu[s + 1]) t = cu[s + 1];
        if (t > cuts.back() && t < tokens) cuts.push_back((int)t);
    }
    cuts.push_back((int)tokens);
    const int np = (int)cuts.size() - 1;
    struct Piece {
        int t0, t1, n0, n1;
        size_t cu_off;   // offset of its local boundaries in the device cu array (ints)
    };
    std::vector<Piece> pieces(np);
    std::vector<int32_t> cu_all;
    size_t ws_bytes = 0;
    for (int p = 0; p < np; ++p) {
        Piece &pc = pieces[p];
        pc.t0 = cuts[p];
        pc.t1 = cuts[p + 1];
        pc.n0 = 0;
        if (p > 0)
            while (pc.n0 < nseq && cu[pc.n0 + 1] <= pc.t0) ++pc.n0;
        pc.n1 = nseq;
        if (p + 1 < np) {
            pc.n1 = pc.n0;
            while (pc.n1 < nseq && cu[pc.n1] < pc.t1) ++pc.n1;
        }
        pc.cu_off = cu_all.size();
        for (int i = pc.n0; i <= pc.n1; ++i) {
            const int32_t c = cu[i] < pc.t0 ? pc.t0 : (cu[i] > pc.t1 ? pc.t1 : cu[i]);
            cu_all.push_back(c - pc.t0);
        }
        const size_t w = kda::fwd_workspace_bytes(pc.n1 - pc.n0, 1, pc.t1 - pc.t0, H_v, true, nullptr, nullptr);
        if (w > ws_bytes) ws_bytes = w;
    }

    const size_t qk_row = (size_t)H_qk * KD * 2, v_row = (size_t)H_v * KD * 2, b_row = (size_t)H_v * 2;
    const size_t st_row = (size_t)H_v * KD * KD * 4;   // bytes of one sequence's state
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const size_t o_q = take(tokens * qk_row), o_k = take(tokens * qk_row);
    const size_t o_v = take(tokens * v_row), o_g = take(tokens * v_row), o_out = take(tokens * v_row);
    const size_t o_b = take(tokens * b_row), o_a = take((size_t)H_v * 4);
    const size_t o_st = take((size_t)nseq * st_row), o_cu = take(cu_all.size() * 4), o_ws = take(ws_bytes);

    cudaStream_t h2d = nullptr, d2h = nullptr;
    int rc = copy_streams(&h2d, &d2h);
    if (rc != KDA_OK) return rc;
    char *base = nullptr;
    if (kda::ws_alloc((void **)&base, off, stream) != cudaSuccess) return KDA_ERR_CUDA;
    std::vector<cudaEvent_t> ev_in(np), ev_out(np);
    cudaEvent_t ev_start, ev_end, ev_h2d;
    cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming);
    cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming);
    cudaEventCreateWithFlags(&ev_h2d, cudaEventDisableTiming);
    for (int p = 0; p < np; ++p) {
        cudaEventCreateWithFlags(&ev_in[p], cudaEventDisableTiming);
        cudaEventCreateWithFlags(&ev_out[p], cudaEventDisableTiming);
    }
    auto dp = [&](size_t o) { return base + o; };
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t x) {
        if (x != cudaSuccess && e == cudaSuccess) e = x;
    };
    const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;

    // inputs: the per-call parts (boundaries, A_log, the initial states, which the pieces then
    // update in place), then each piece's token rows
    ok(cudaEventRecord(ev_start, stream));
    ok(cudaStreamWaitEvent(h2d, ev_start, 0));
    ok(cudaMemcpyAsync(dp(o_cu), cu_all.data(), cu_all.size() * 4, H2D, h2d));
    if (tokens > 0) ok(cudaMemcpyAsync(dp(o_a), A_log, (size_t)H_v * 4, H2D, h2d));
    if (initial_state) ok(cudaMemcpyAsync(dp(o_st), initial_state, (size_t)nseq * st_row, H2D, h2d));
    else ok(cudaMemsetAsync(dp(o_st), 0, (size_t)nseq * st_row, h2d));
    for (int p = 0; p < np && e == cudaSuccess; ++p) {
        const size_t t0 = pieces[p].t0, nt = (size_t)(pieces[p].t1 - pieces[p].t0);
        if (nt > 0) {
            ok(cudaMemcpyAsync(dp(o_q) + t0 * qk_row, (const char *)q + t0 * qk_row, nt * qk_row, H2D, h2d));
            ok(cudaMemcpyAsync(dp(o_k) + t0 * qk_row, (const char *)k + t0 * qk_row, nt * qk_row, H2D, h2d));
            ok(cudaMemcpyAsync(dp(o_v) + t0 * v_row, (const char *)v + t0 * v_row, nt * v_row, H2D, h2d));
            ok(cudaMemcpyAsync(dp(o_g) + t0 * v_row, (const char *)graw + t0 * v_row, nt * v_row, H2D, h2d));
            ok(cudaMemcpyAsync(dp(o_b) + t0 * b_row, (const char *)b + t0 * b_row, nt * b_row, H2D, h2d));
        }
        ok(cudaEventRecord(ev_in[p], h2d));
    }
    // every input copy queued so far, whether or not all of them could be queued
    const cudaError_t eh = cudaEventRecord(ev_h2d, h2d);
    // kernels, piece by piece on the caller's stream; each piece's sequences start from, and
    // write back, their rows of the device state array
    for (int p = 0; p < np && e == cudaSuccess; ++p) {
        const Piece &pc = pieces[p];
        const size_t t0 = pc.t0;
        ok(cudaStreamWaitEvent(stream, ev_in[p], 0));
        float *st = (float *)(dp(o_st) + (size_t)pc.n0 * st_row);
        int n = 0;
        ok(kda::launch_fwd_heads((const uint16_t *)(dp(o_q) + t0 * qk_row), (const uint16_t *)(dp(o_k) + t0 * qk_row),
                                 (const uint16_t *)(dp(o_v) + t0 * v_row), (const uint16_t *)(dp(o_g) + t0 * v_row),
                                 (const uint16_t *)(dp(o_b) + t0 * b_row), (const float *)dp(o_a), scale, st, st,
                                 (const int32_t *)dp(o_cu) + pc.cu_off, pc.n1 - pc.n0, 1, pc.t1 - pc.t0, H_qk, H_v, 0,
                                 H_v, true, (uint16_t *)(dp(o_out) + t0 * v_row), dp(o_ws), stream, &n));
        ok(cudaEventRecord(ev_out[p], stream));
    }
    // results, piece by piece, then the final states
    for (int p = 0; p < np && e == cudaSuccess; ++p) {
        ok(cudaStreamWaitEvent(d2h, ev_out[p], 0));
        const size_t t0 = pieces[p].t0, nt = (size_t)(pieces[p].t1 - pieces[p].t0);
        if (nt > 0) ok(cudaMemcpyAsync((char *)out + t0 * v_row, dp(o_out) + t0 * v_row, nt * v_row, D2H, d2h));
    }
    if (final_state && e == cudaSuccess)
        ok(cudaMemcpyAsync(final_state, dp(o_st), (size_t)nseq * st_row, D2H, d2h));
    // the device buffer is released on the caller's stream only after every copy queued on
    // either copy stream is done with it, also when a launch or a copy failed midway
    const cudaError_t ee = cudaEventRecord(ev_end, d2h);
    ok(ee);
    ok(eh);
    if (eh == cudaSuccess) ok(cudaStreamWaitEvent(stream, ev_h2d, 0));
    if (ee == cudaSuccess) ok(cudaStreamWaitEvent(stream, ev_end, 0));
    const cudaError_t ef = (eh == cudaSuccess && ee == cudaSuccess) ? kda::ws_free(base, stream) : cudaFree(base);
    cudaEventDestroy(ev_start);
    cudaEventDestroy(ev_end);
    cudaEventDestroy(ev_h2d);
    for (int p = 0; p < np; ++p) {
        cudaEventDestroy(ev_in[p]);
        cudaEventDestroy(ev_out[p]);
    }
    if (e != cudaSuccess || ef != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

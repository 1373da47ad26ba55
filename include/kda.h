/*
 * libkda: Kimi Delta Attention (KDA) forward and single-token decode on
 * NVIDIA GB300 (sm_103a).
 *
 * KDA is a gated delta-rule linear attention with a per-channel decay.  Per
 * sequence and value head h, with state S (V x K, fp32, S[v][k]):
 *
 *   qt   = scale * q / sqrt(|q|^2 + 1e-6)          kh = k / sqrt(|k|^2 + 1e-6)
 *   beta = sigmoid(b)                               g  = -exp(A_log[h]) * softplus(graw)
 *   S_t  = S_{t-1} Diag(exp g_t) (I - beta_t kh_t kh_t^T) + beta_t v_t kh_t^T
 *   o_t  = S_t qt_t
 *
 * The fused gate activation, beta sigmoid and q/k L2 norm follow the FlashKDA
 * library page ("FlashKDA: High-performance KDA CUDA kernels for SM90+ GPUs",
 * section "What exact performance bottlenecks does FlashKDA address",
 * Technical Features); the state layouts [B,H,V,K] and [N,H,V,K] with
 * cu_seqlens and B = 1 follow its section "How does FlashKDA's
 * stateful/streaming (chunked) support work?"; bf16 q/k/v/g/out, fp32 A_log
 * and the K = V = 128 restriction follow its section "How to seamlessly
 * replace flash-linear-attention's chunk_kda" (Technical Analysis).  Grouped
 * value heads (H_v a multiple of H_qk, value head h reading query/key head
 * h / (H_v / H_qk)) follow the h_qk / h_v columns of the FlashQLA H200 table
 * ("benchmark_results_H200.txt", FORWARD BENCHMARKS).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - All tensor pointers are DEVICE pointers (kda_fwd_host's are host
 *    pointers) to contiguous row-major data, owned by the caller; the library
 *    keeps no pointer after a call returns.  bf16 data is passed as its 16-bit
 *    pattern (kda_bf16_t).
 *  - Kernels run on the calling thread's current CUDA device: the device
 *    pointers and `stream` must belong to it.
 *  - q, k, v, graw, out and the states must be 16-byte aligned.
 *  - Calls are asynchronous and ordered on `stream`; no entry point except
 *    kda_get_status and kda_kernel_times synchronises with the host.
 *  - The return value reports host-side validation and launch errors only.
 *    Faults detected on the device (malformed cu_seqlens, a bounded wait that
 *    timed out) are recorded in a per-device status word read by
 *    kda_get_status.
 *  - K and V must both be 128 (KDA_ERR_UNSUPPORTED otherwise).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16_t; /* bit pattern of a bfloat16 value */

enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,    /* NULL required pointer, negative size, H_v % H_qk != 0,
                                    cu_seqlens with B != 1, misaligned pointer, more than
                                    2^31 - 1 tokens (B * T), sequences * H_v above
                                    2^29 - 1 (chunked calls) or B * H_v above 2^31 - 1
                                    (decode calls): work items carry 32-bit indices */
    KDA_ERR_UNSUPPORTED = -2,    /* K != 128 or V != 128 */
    KDA_ERR_CUDA = -3,           /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_DEVICE_TIMEOUT = -4, /* (status word) a bounded device-side wait gave up */
    KDA_ERR_BAD_SEQLENS = -5,    /* (status word) cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T */
    KDA_ERR_WORKSPACE = -6       /* workspace NULL, too small or not 256-byte aligned */
};

/*
 * Chunked KDA forward (prefill).
 *
 *   q, k      [B, T, H_qk, K] bf16
 *   v         [B, T, H_v,  V] bf16
 *   graw      [B, T, H_v,  K] bf16   gate pre-activation (per channel)
 *   b         [B, T, H_v]     bf16   beta pre-activation
 *   A_log     [H_v]           fp32
 *   scale                            multiplies the L2-normalised q (normally 1/sqrt(K))
 *   initial_state [Nseq, H_v, V, K] fp32, or NULL for zeros
 *   final_state   [Nseq, H_v, V, K] fp32 output, or NULL (not written)
 *   cu_seqlens    int32 [N + 1] device array, or NULL.  With cu_seqlens the
 *                 call is packed: B must be 1, sequence n covers tokens
 *                 cu_seqlens[n] .. cu_seqlens[n+1]-1 and Nseq = N; without it
 *                 Nseq = B sequences of length T each and N is ignored.
 *   out       [B, T, H_v, V] bf16 output
 *
 * Each sequence starts from its own initial state; feeding final_state into
 * initial_state of a call on the continuation equals one call on the whole
 * sequence.  A zero-length sequence copies its initial state (or zeros) to
 * final_state.  Takes its workspace from the library's workspace pool on
 * `stream` (see kda_release_cached_memory); use kda_fwd_ws to supply it instead.
 */
int kda_fwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
            const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
            const float *initial_state, float *final_state, const int32_t *cu_seqlens,
            int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
            cudaStream_t stream);

/* Bytes of device workspace kda_fwd_ws needs for these sizes (0 on invalid
 * sizes).  The bound covers any cu_seqlens with N sequences and T tokens. */
size_t kda_fwd_workspace_size(int N, int B, int T, int H_qk, int H_v, int K, int V);

/* kda_fwd with a caller-owned workspace: `ws` is a device pointer, 256-byte
 * aligned, of at least kda_fwd_workspace_size(...) bytes.  The workspace must
 * not be used by anything else until the work queued on `stream` completes. */
int kda_fwd_ws(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
               const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
               const float *initial_state, float *final_state, const int32_t *cu_seqlens,
               int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
               void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kda_fwd for a scalar gate: graw is [B, T, H_v] bf16, one gate pre-activation per
 * token and value head shared by all K channels (the gated delta rule's per-head
 * decay, "broadcast across K").  Every other argument, and the result, as kda_fwd:
 * the output equals kda_fwd's with graw broadcast along K.  A dedicated
 * intra-chunk kernel uses the scalar decay: the gate read shrinks 128-fold and the
 * chunk's products come from one MMA of the raw q and k times a decay mask.
 */
int kda_fwd_scalar_gate(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                        const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
                        const float *initial_state, float *final_state, const int32_t *cu_seqlens,
                        int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
                        cudaStream_t stream);

/*
 * kda_fwd on host buffers: the same problem and the same results, with every
 * tensor (cu_seqlens included) in host memory.  Pinned (page-locked) buffers let
 * the copies run at the host link's bandwidth; pageable ones work, more slowly.
 * The call copies the inputs to the device, runs the forward and copies out and
 * final_state back, in up to eighteen pieces of consecutive tokens (at least
 * 2048 tokens each, the last one split into a half and two quarters) so that
 * one piece's copies overlap the previous piece's kernels (the link, not the
 * kernels, bounds such a call).  A sequence crossing a piece boundary is cut at
 * a chunk boundary and its state carried on the device, which is the chunking
 * and arithmetic of a single call.  cu_seqlens is checked on the host: a
 * malformed array returns KDA_ERR_BAD_SEQLENS before anything is queued.
 * Device buffers come from the library's workspace pool on `stream`; two
 * copy streams per device are created on the first call and kept.
 * Asynchronous like kda_fwd: the results are in host memory once `stream` has
 * passed the call (e.g. after cudaStreamSynchronize), and the host buffers must
 * stay valid and unchanged until then.
 */
int kda_fwd_host(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                 const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
                 const float *initial_state, float *final_state, const int32_t *cu_seqlens,
                 int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
                 cudaStream_t stream);

/*
 * kda_fwd with the initial and final states stored as bf16 ([N, H_v, V, K];
 * FlashKDA's interface admits fp32 or bf16 states, "How does FlashKDA's
 * stateful/streaming (chunked) support work?").  The recurrence runs with an
 * fp32 state exactly as in kda_fwd; the initial state is widened on load and the
 * final state rounded to bf16 (nearest even) once, on store.  Other arguments,
 * asynchrony and errors as kda_fwd.
 */
int kda_fwd_bf16_state(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                       const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
                       const kda_bf16_t *initial_state, kda_bf16_t *final_state,
                       const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V,
                       kda_bf16_t *out, cudaStream_t stream);

/*
 * One decode step for B independent sequences (one token each):
 *
 *   q, k  [B, H_qk, K] bf16     v, graw [B, H_v, V|K] bf16     b [B, H_v] bf16
 *   A_log [H_v] fp32            state [B, H_v, V, K] fp32, updated in place
 *   out   [B, H_v, V] bf16
 *
 * Equivalent to kda_fwd with T = 1, initial_state = final_state = state.
 */
int kda_decode_step(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                    const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log,
                    float scale, float *state, int B, int H_qk, int H_v, int K, int V,
                    kda_bf16_t *out, cudaStream_t stream);

/*
 * Decode of Tq (1..KDA_DECODE_MAX_TOKENS) consecutive tokens per (b, h) in one
 * pass over the state, which is read once and written once (for example the
 * verification step of speculative decoding), with the state stored in fp32
 * (state_is_bf16 = 0) or bf16 (state_is_bf16 = 1; the recurrence runs in fp32
 * and the updated state is rounded to bf16 once, at the end of the pass).
 *
 *   q, k   [B, Tq, H_qk, K] bf16      v, graw [B, Tq, H_v, *] bf16
 *   b      [B, Tq, H_v] bf16          A_log [H_v] fp32
 *   state  [B, H_v, V, K] fp32 or bf16, updated in place
 *   out    [B, Tq, H_v, V] bf16
 *
 * The result equals Tq calls of kda_decode_step (for an fp32 state) up to
 * rounding order.  Returns KDA_ERR_INVALID_ARG for Tq outside 1..8.
 */
#define KDA_DECODE_MAX_TOKENS 8
int kda_decode_tokens(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                      const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log,
                      float scale, void *state, int state_is_bf16, int B, int Tq, int H_qk,
                      int H_v, int K, int V, kda_bf16_t *out, cudaStream_t stream);

/* Human-readable name of a return or status code (static string). */
const char *kda_status_string(int code);

/* Synchronises `stream`, then returns and clears the current device's status
 * word (KDA_OK if no device-side fault was recorded since the last call). */
int kda_get_status(cudaStream_t stream);

/*
 * kda_fwd without any device allocation, for callers that cannot allocate
 * device memory where they run the forward: a framework whose allocator owns
 * all device memory and forbids allocations outside its own pool, a
 * latency-critical serving loop that must not enter the driver's allocator,
 * or an embedding host that hands the library only its own tensors.  The
 * paper has no counterpart; this is a deployment variant of kda_fwd with
 * identical arguments and bit-identical results (it runs the same kernels).
 *
 * The workspace is a file-scope __device__ array of KDA_NOALLOC_WS_BYTES
 * (64 MiB) that every GPU which loads the library holds until the process
 * exits.  Sizes whose workspace (see kda_fwd_workspace_size; about 113 KB per
 * 64-token chunk and value head) exceeds it return KDA_ERR_WORKSPACE without
 * launching anything.  The first call on a device looks up the array's device
 * address with that device current (a one-time set-up); make that first call
 * before any stream capture.  All calls on a device share the array and it
 * keeps the last call's contents (nothing in it needs to start at zero), so
 * calls that overlap on the GPU (different streams without ordering between
 * them) race: order them on one stream or with events.
 */
#define KDA_NOALLOC_WS_BYTES (64u << 20)
int kda_fwd_noalloc(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v,
                    const kda_bf16_t *graw, const kda_bf16_t *b, const float *A_log, float scale,
                    const float *initial_state, float *final_state, const int32_t *cu_seqlens,
                    int N, int B, int T, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
                    cudaStream_t stream);

/*
 * Backward of kda_fwd: gradients of a loss L with respect to every input, given
 * dL/dout and dL/dfinal_state.  The pages report timings of a gated-delta-rule
 * backward (FlashQLA "benchmark_results_H200.txt", BACKWARD BENCHMARKS) without
 * a formula; the gradients are those of the forward recurrence documented above.
 *
 *   inputs   q, k, v, graw, b, A_log, scale, initial_state, cu_seqlens, N, B, T,
 *            H_qk, H_v, K, V exactly as kda_fwd
 *   dout     [B, T, H_v, V] bf16 (dL/dout, required when B*T > 0)
 *   dht      [N, H_v, V, K] fp32 (dL/dfinal_state) or NULL for zero
 *   dq, dk   [B, T, H_qk, K] fp32 (summed over the value heads of each group)
 *   dv       [B, T, H_v, V] fp32      dgraw [B, T, H_v, K] fp32    db [B, T, H_v] fp32
 *   dA_log   [H_v] fp32               dh0 [N, H_v, V, K] fp32 (dL/dinitial_state)
 *
 * All outputs are written (dA_log is zeroed, then accumulated).  Gradient
 * buffers must be 16-byte aligned (db excepted).  Asynchronous on `stream`.  The
 * gradients are computed in the chunk (UT / WY) form of the forward, 64 tokens per
 * chunk, on tensor cores (mma.sync, tf32 operands rounded to nearest, fp32
 * accumulation, fp32 states): per (chunk, value head) the chunk's operands, then
 * the state entering each chunk (a forward chain) and the state gradient leaving
 * it (a reverse chain), then the chunks' gradients in parallel.  The workspace
 * holds, per (chunk, value head), those operands, both states and the value-side
 * gradient sums (about 434 KiB), plus 1 KiB per token and value head (8.4 GB
 * for B=2, T=16384, H_v=32); kda_bwd takes it from the library's workspace
 * pool on `stream` (a failed allocation returns KDA_ERR_CUDA), kda_bwd_ws from the caller.  Errors
 * as kda_fwd.
 */
int kda_bwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
            const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
            const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V,
            const kda_bf16_t *dout, const float *dht, float *dq, float *dk, float *dv, float *dgraw,
            float *db, float *dA_log, float *dh0, cudaStream_t stream);

/* Bytes of device workspace kda_bwd_ws needs for these sizes (0 on invalid
 * sizes).  The bound covers any cu_seqlens with N sequences and T tokens. */
size_t kda_bwd_workspace_size(int N, int B, int T, int H_qk, int H_v, int K, int V);

/* kda_bwd with a caller-owned workspace: `ws` is a device pointer, 256-byte
 * aligned, of at least kda_bwd_workspace_size(...) bytes (KDA_ERR_WORKSPACE
 * otherwise).  The workspace must not be used by anything else until the work
 * queued on `stream` completes. */
int kda_bwd_ws(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const kda_bf16_t *graw,
               const kda_bf16_t *b, const float *A_log, float scale, const float *initial_state,
               const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V,
               const kda_bf16_t *dout, const float *dht, float *dq, float *dk, float *dv, float *dgraw,
               float *db, float *dA_log, float *dh0, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Lightning attention: linear attention with a fixed per-head decay.  The cuLA
 * page ("cuLA benchmark results on GB200") times a lightning-attention forward
 * (fixed-length and varlen tables) and a single-token la_decode with 64 heads of
 * dimension 128, and prints no formula; these calls compute the standard
 * lightning-attention recurrence, per sequence and value head h with
 * lambda = exp(-slope[h]):
 *
 *   S_t = lambda S_{t-1} + v_t k_t^T,      o_t = scale S_t q_t
 *
 * with q and k used as given (no normalisation) and no gate.
 *
 *   q, k   [B, T, H_qk, K] bf16        v, out [B, T, H_v, V] bf16
 *   slope  [H_v] fp32 (decay rate per token; >= 0 for a decaying state)
 *   initial_state / final_state [N, H_v, V, K] fp32, NULL for zeros / not written
 *   cu_seqlens as kda_fwd (B = 1, N packed sequences), else B sequences of T
 *
 * K = V = 128 and H_v a multiple of H_qk (value head h reads q/k head
 * h / (H_v / H_qk)); q, k, v and out 16-byte aligned.  One fused kernel per
 * call (after the sequence plan) streams q, k, v once and writes out once; a
 * few KB of plan tables come from the library's workspace pool on `stream`.  Errors and
 * asynchrony as kda_fwd (a malformed cu_seqlens sets KDA_ERR_BAD_SEQLENS in
 * the status word and writes nothing).
 */
int kda_la_fwd(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const float *slope,
               float scale, const float *initial_state, float *final_state,
               const int32_t *cu_seqlens, int N, int B, int T, int H_qk, int H_v, int K, int V,
               kda_bf16_t *out, cudaStream_t stream);

/*
 * One lightning-attention decode step (the la_decode of the same page) for B
 * independent sequences:
 *
 *   q, k [B, H_qk, K] bf16   v [B, H_v, V] bf16   slope [H_v] fp32
 *   state [B, H_v, V, K] fp32, updated in place   out [B, H_v, V] bf16
 *
 * Equal to kda_la_fwd with T = 1 and initial_state = final_state = state; one
 * pass over the state.  Errors as kda_decode_step.
 */
int kda_la_decode(const kda_bf16_t *q, const kda_bf16_t *k, const kda_bf16_t *v, const float *slope,
                  float scale, float *state, int B, int H_qk, int H_v, int K, int V, kda_bf16_t *out,
                  cudaStream_t stream);

/* Self-test of the device-side failure path: queues one tiny kernel whose bounded
 * wait on a barrier that nothing completes gives up, recording
 * KDA_ERR_DEVICE_TIMEOUT in the status word (read it with kda_get_status); the
 * kernel returns normally and the context stays usable.  No counterpart on the
 * pages; it checks the library's own error reporting. */
int kda_selftest_wait_timeout(cudaStream_t stream);

/* Number of kernel launches the most recent successful kda_fwd / kda_fwd_ws /
 * kda_decode_step call on this host thread queued. */
int kda_last_launch_count(void);

/*
 * Measurement aid (off by default).  While enabled, the forward, decode,
 * backward and lightning-attention entry points record a CUDA event on
 * `stream` before their first and after each kernel launch.  kda_kernel_times waits for the events of the most
 * recent call on this host thread and writes up to max_n per-kernel durations
 * in milliseconds (and static kernel names when `names` is not NULL); it
 * returns the number written, 0 when timing is off, or KDA_ERR_CUDA.
 */
int kda_set_kernel_timing(int enable);
int kda_kernel_times(float *ms, const char **names, int max_n);

/*
 * The allocating entry points (kda_fwd, kda_fwd_bf16_state,
 * kda_fwd_scalar_gate, kda_fwd_host, kda_bwd, kda_la_fwd) take their device
 * workspace from one stream-ordered memory pool per device, created on first
 * use with an unbounded release threshold: what a call frees on its stream
 * stays mapped in the pool after the caller synchronises, and the next call
 * reuses it instead of mapping fresh pages, as a caching allocator does (the
 * device's default pool would hand the pages back at every synchronisation, and
 * mapping the 1.8 GB workspace of a B=2, T=16384, H_v=32 forward again costs
 * about as much as the forward).  The pool therefore keeps the largest
 * workspace used so far.  kda_release_cached_memory returns every byte of
 * every device's pool that no queued call still uses to the driver; it returns
 * KDA_OK, or KDA_ERR_CUDA if the driver refused.
 */
int kda_release_cached_memory(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */

// Single-token KDA decode step: one streaming pass over the [B,H,V,K] fp32
// state (read once, written once), with the per-token pre-processing fused in.
//
// Per (b, h): qt = scale q/|q|, kh = k/|k|, beta = sigmoid(b),
// e_c = exp(-exp(A_log[h]) softplus(graw_c)); then for every state row v
//   s' = S[v,:] * e,  d_k = s'.kh,  d_q = s'.qt,  delta = beta (v_v - d_k)
//   S[v,:] = s' + delta kh,   o_v = d_q + delta (kh.qt)
// which is the recurrence S (Diag e)(I - beta kh kh^T) + beta v kh^T, o = S qt
// evaluated row by row.
#include "kda_common.cuh"

namespace kda {

constexpr int DEC_WARPS = 8;
constexpr int DEC_ROWS = KD / DEC_WARPS;  // state rows per warp

// The state is stored in fp32, or in bf16 (BF16: each row widened to fp32 for the step and
// rounded once on store; with 8-byte rows per lane the kernel fits four CTAs per SM, so more
// of the state is in flight).
template <bool BF16>
__global__ __launch_bounds__(DEC_WARPS * 32, BF16 ? 4 : 2) void decode_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const uint16_t *__restrict__ graw, const uint16_t *__restrict__ b, const float *__restrict__ A_log,
    float scale, void *__restrict__ state, int H_qk, int H_v, uint16_t *__restrict__ out) {
    const int bh = blockIdx.x;
    const int bi = bh / H_v, h = bh - bi * H_v;
    const int hq = h / (H_v / H_qk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // Lane owns channels 4*lane .. 4*lane+3.
    const size_t qk_off = ((size_t)bi * H_qk + hq) * KD + 4 * lane;
    const size_t hv_off = ((size_t)bi * H_v + h) * KD;
    // the warp's 16 state rows are requested first, so that their latency overlaps the token's
    // preparation below
    const int r0 = warp * DEC_ROWS;
    float *S = reinterpret_cast<float *>(state) + (hv_off + r0) * KD;
    uint16_t *Sb = reinterpret_cast<uint16_t *>(state) + (hv_off + r0) * KD;
    float4 s[BF16 ? 1 : DEC_ROWS];
    uint2 sb[BF16 ? DEC_ROWS : 1];
#pragma unroll
    for (int i = 0; i < DEC_ROWS; ++i) {
        if (BF16) sb[i] = __ldcs(reinterpret_cast<const uint2 *>(Sb + (size_t)i * KD) + lane);
        else s[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)i * KD) + lane);
    }
    const float vrow = bf16_to_f(v[hv_off + r0 + (lane & (DEC_ROWS - 1))]);
    const uint2 qw = *reinterpret_cast<const uint2 *>(q + qk_off);
    const uint2 kw = *reinterpret_cast<const uint2 *>(k + qk_off);
    const uint2 gw = *reinterpret_cast<const uint2 *>(graw + hv_off + 4 * lane);
    const float qv[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
    const float kv[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
    const float gv[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        sq = fmaf(qv[i], qv[i], sq);
        sk = fmaf(kv[i], kv[i], sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float rq = scale * rsqrtf(sq + L2_EPS), rk = rsqrtf(sk + L2_EPS);
    const float a = ex2(A_log[h] * LOG2E);
    float qt[4], kh[4], dec[4], kq = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        qt[i] = qv[i] * rq;
        kh[i] = kv[i] * rk;
        dec[i] = ex2(-a * softplus_log2(gv[i]));
        kq = fmaf(kh[i], qt[i], kq);
    }
    kq = warp_sum(kq);
    const float bb = bf16_to_f(b[(size_t)bi * H_v + h]);
    const float beta = 1.0f / (1.0f + ex2(-bb * LOG2E));


    float o_mine = 0.f;
#pragma unroll
    for (int i = 0; i < DEC_ROWS; ++i) {
        float4 x = BF16 ? make_float4(bf16_lo(sb[i].x), bf16_hi(sb[i].x), bf16_lo(sb[i].y), bf16_hi(sb[i].y))
                        : s[BF16 ? 0 : i];
        float dk, dq;
        if constexpr (BF16) {
            x.x *= dec[0];
            x.y *= dec[1];
            x.z *= dec[2];
            x.w *= dec[3];
            dk = x.x * kh[0] + x.y * kh[1] + x.z * kh[2] + x.w * kh[3];
            dq = x.x * qt[0] + x.y * qt[1] + x.z * qt[2] + x.w * qt[3];
        } else {
            // packed fp32 pairs: the decay, then the two dot products on even / odd channel halves
            const float2 xa = __fmul2_rn(make_float2(x.x, x.y), make_float2(dec[0], dec[1]));
            const float2 xb = __fmul2_rn(make_float2(x.z, x.w), make_float2(dec[2], dec[3]));
            x = make_float4(xa.x, xa.y, xb.x, xb.y);
            const float2 dk2 = __ffma2_rn(xb, make_float2(kh[2], kh[3]), __fmul2_rn(xa, make_float2(kh[0], kh[1])));
            const float2 dq2 = __ffma2_rn(xb, make_float2(qt[2], qt[3]), __fmul2_rn(xa, make_float2(qt[0], qt[1])));
            dk = dk2.x + dk2.y;
            dq = dq2.x + dq2.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            dk += __shfl_xor_sync(0xffffffffu, dk, o);
            dq += __shfl_xor_sync(0xffffffffu, dq, o);
        }
        const float vi = __shfl_sync(0xffffffffu, vrow, i);
        const float delta = beta * (vi - dk);
        if constexpr (BF16) {
            x.x = fmaf(delta, kh[0], x.x);
            x.y = fmaf(delta, kh[1], x.y);
            x.z = fmaf(delta, kh[2], x.z);
            x.w = fmaf(delta, kh[3], x.w);
        } else {
            const float2 ua = __ffma2_rn(make_float2(delta, delta), make_float2(kh[0], kh[1]), make_float2(x.x, x.y));
            const float2 ub = __ffma2_rn(make_float2(delta, delta), make_float2(kh[2], kh[3]), make_float2(x.z, x.w));
            x = make_float4(ua.x, ua.y, ub.x, ub.y);
        }
        if (BF16)
            __stcs(reinterpret_cast<uint2 *>(Sb + (size_t)i * KD) + lane,
                   make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w)));
        else
            __stcs(reinterpret_cast<float4 *>(S + (size_t)i * KD) + lane, x);
        if (lane == i) o_mine = fmaf(delta, kq, dq);
    }
    if (lane < DEC_ROWS) out[hv_off + r0 + lane] = f_to_bf16(o_mine);
}

cudaError_t launch_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                          const uint16_t *b, const float *A_log, float scale, float *state, int B, int H_qk,
                          int H_v, uint16_t *out, cudaStream_t stream) {
    const long long nblk = (long long)B * H_v;
    if (nblk == 0) return cudaSuccess;
    decode_kernel<false><<<(unsigned)nblk, DEC_WARPS * 32, 0, stream>>>(q, k, v, graw, b, A_log, scale, state, H_qk,
                                                                      H_v, out);
    return cudaGetLastError();
}

}  // namespace kda

// =====================================================================
// Multi-token decode: Tq <= 8 consecutive tokens per (b, h) applied to the
// state in one pass (read once, Tq updates in registers, written once), the
// state stored in fp32 or bf16.  Warp t < Tq first prepares token t (normalised
// q and k, per-channel decay, beta, k.q, v) in shared memory; then each warp
// streams 16 state rows through all Tq tokens, each lane holding 16 channels of
// four rows so that a row's two dot products reduce over eight lanes.
// =====================================================================
namespace kda {

constexpr int DEC_MAX_T = 8;

template <bool BF16_STATE>
__global__ __launch_bounds__(DEC_WARPS * 32, 2) void decode_tokens_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const uint16_t *__restrict__ graw, const uint16_t *__restrict__ b, const float *__restrict__ A_log, float scale,
    void *__restrict__ state, int Tq, int H_qk, int H_v, uint16_t *__restrict__ out) {
    __shared__ float s_qt[DEC_MAX_T][KD], s_kh[DEC_MAX_T][KD], s_dec[DEC_MAX_T][KD], s_v[DEC_MAX_T][KD];
    __shared__ float s_beta[DEC_MAX_T], s_kq[DEC_MAX_T];
    const int bh = blockIdx.x;
    const int bi = bh / H_v, h = bh - bi * H_v;
    const int hq = h / (H_v / H_qk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // ---- the warp's 16 state rows, requested first so that their latency overlaps the token
    //      preparation below (fp32 in registers; a bf16 state is widened after the loads land).
    //      Lane (g, c) = (lane / 8, lane % 8) keeps channels 32 u + 4 c .. 32 u + 4 c + 3, u = 0..3,
    //      of rows r0 + 4 j + g, j = 0..3 (the eight lanes of a row read 128 contiguous bytes per
    //      load), so that a row's dot products reduce over eight lanes.
    const int r0 = warp * DEC_ROWS, g = lane >> 3, c4 = 4 * (lane & 7);
    const size_t st0 = ((size_t)bh * KD + r0 + g) * KD + c4;   // row r0 + g, channel 4 c
    float4 s[4][4];                                              // [row j][channel quad u]
    uint2 sw[BF16_STATE ? 4 : 1][BF16_STATE ? 4 : 1];
    if (BF16_STATE) {
        const uint16_t *S = reinterpret_cast<const uint16_t *>(state) + st0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) sw[j][u] = __ldcs(reinterpret_cast<const uint2 *>(S + (size_t)4 * j * KD + 32 * u));
    } else {
        const float *S = reinterpret_cast<const float *>(state) + st0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) s[j][u] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)4 * j * KD + 32 * u));
    }

    // ---- token preparation: warp t handles token t; lane owns channels 4 lane .. 4 lane + 3
    if (warp < Tq) {
        const int t = warp;
        const size_t row_qk = (((size_t)bi * Tq + t) * H_qk + hq) * KD + 4 * lane;
        const size_t row_v = (((size_t)bi * Tq + t) * H_v + h) * KD;
        const uint2 qw = *reinterpret_cast<const uint2 *>(q + row_qk);
        const uint2 kw = *reinterpret_cast<const uint2 *>(k + row_qk);
        const uint2 gw = *reinterpret_cast<const uint2 *>(graw + row_v + 4 * lane);
        const uint2 vw = *reinterpret_cast<const uint2 *>(v + row_v + 4 * lane);
        const float qv[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
        const float kv[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
        const float gv[4] = {bf16_lo(gw.x), bf16_hi(gw.x), bf16_lo(gw.y), bf16_hi(gw.y)};
        const float vv[4] = {bf16_lo(vw.x), bf16_hi(vw.x), bf16_lo(vw.y), bf16_hi(vw.y)};
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sq = fmaf(qv[i], qv[i], sq);
            sk = fmaf(kv[i], kv[i], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = scale * rsqrtf(sq + L2_EPS), rk = rsqrtf(sk + L2_EPS);
        const float a = ex2(A_log[h] * LOG2E);
        float kq = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = 4 * lane + i;
            s_qt[t][c] = qv[i] * rq;
            s_kh[t][c] = kv[i] * rk;
            s_dec[t][c] = ex2(-a * softplus_log2(gv[i]));
            s_v[t][c] = vv[i];
            kq = fmaf(kv[i] * rk, qv[i] * rq, kq);
        }
        kq = warp_sum(kq);
        if (lane == 0) {
            s_kq[t] = kq;
            s_beta[t] = 1.0f / (1.0f + ex2(-bf16_to_f(b[((size_t)bi * Tq + t) * H_v + h]) * LOG2E));
        }
    }
    __syncthreads();
    if (BF16_STATE) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint2 w = sw[j][u];
                s[j][u] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
            }
    }
    for (int t = 0; t < Tq; ++t) {
        float4 dec[4], kh[4], qt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            dec[u] = *reinterpret_cast<const float4 *>(&s_dec[t][32 * u + c4]);
            kh[u] = *reinterpret_cast<const float4 *>(&s_kh[t][32 * u + c4]);
            qt[u] = *reinterpret_cast<const float4 *>(&s_qt[t][32 * u + c4]);
        }
        // per row j: dk_j = s'_j . kh (value 2 j) and dq_j = s'_j . qt (value 2 j + 1), lane partials.
        // Packed fp32 pairs (one instruction per two multiplies or fused multiply-adds): the
        // even and odd channels of a quad accumulate separately and are added at the end.
        float red[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 dk = make_float2(0.f, 0.f), dq = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 xa = __fmul2_rn(make_float2(s[j][u].x, s[j][u].y), make_float2(dec[u].x, dec[u].y));
                const float2 xb = __fmul2_rn(make_float2(s[j][u].z, s[j][u].w), make_float2(dec[u].z, dec[u].w));
                s[j][u] = make_float4(xa.x, xa.y, xb.x, xb.y);
                dk = __ffma2_rn(xa, make_float2(kh[u].x, kh[u].y), dk);
                dk = __ffma2_rn(xb, make_float2(kh[u].z, kh[u].w), dk);
                dq = __ffma2_rn(xa, make_float2(qt[u].x, qt[u].y), dq);
                dq = __ffma2_rn(xb, make_float2(qt[u].z, qt[u].w), dq);
            }
            red[2 * j] = dk.x + dk.y;
            red[2 * j + 1] = dq.x + dq.y;
        }
        // reduce-scatter over the eight lanes of a row group: at each level a lane keeps half of
        // its values (the half selected by its lane bit) and adds the partner's copy of that half;
        // after three levels lane (g, c) holds the total of value c (7 shuffles for 8 sums)
#pragma unroll
        for (int o = 4, n = 4; o >= 1; o >>= 1, n >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float send = upper ? red[i] : red[i + n];
                const float keep = upper ? red[i + n] : red[i];
                red[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        // lane (g, 2 j): dk_j -> delta_j; lane (g, 2 j + 1): dq_j -> o = dq_j + delta_j (k.q); row r0 + 4 j + g
        const int jm = (lane & 7) >> 1, row = r0 + 4 * jm + g;
        const float dk_or_dq = red[0];
        const float delta_mine = s_beta[t] * (s_v[t][row] - dk_or_dq);
        const float delta_pair = __shfl_xor_sync(0xffffffffu, delta_mine, 1);
        if (lane & 1)
            out[(((size_t)bi * Tq + t) * H_v + h) * KD + row] = f_to_bf16(fmaf(delta_pair, s_kq[t], dk_or_dq));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float delta = __shfl_sync(0xffffffffu, delta_mine, 8 * g + 2 * j);
            const float2 d2 = make_float2(delta, delta);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 a = __ffma2_rn(d2, make_float2(kh[u].x, kh[u].y), make_float2(s[j][u].x, s[j][u].y));
                const float2 c = __ffma2_rn(d2, make_float2(kh[u].z, kh[u].w), make_float2(s[j][u].z, s[j][u].w));
                s[j][u] = make_float4(a.x, a.y, c.x, c.y);
            }
        }
    }
    if (BF16_STATE) {
        uint16_t *S = reinterpret_cast<uint16_t *>(state) + st0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                __stcs(reinterpret_cast<uint2 *>(S + (size_t)4 * j * KD + 32 * u),
                       make_uint2(pack_bf16x2(s[j][u].x, s[j][u].y), pack_bf16x2(s[j][u].z, s[j][u].w)));
    } else {
        float *S = reinterpret_cast<float *>(state) + st0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) __stcs(reinterpret_cast<float4 *>(S + (size_t)4 * j * KD + 32 * u), s[j][u]);
    }
}

cudaError_t launch_decode_tokens(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *graw,
                                 const uint16_t *b, const float *A_log, float scale, void *state, bool bf16_state,
                                 int B, int Tq, int H_qk, int H_v, uint16_t *out, cudaStream_t stream) {
    const long long nblk = (long long)B * H_v;
    if (nblk == 0) return cudaSuccess;
    if (bf16_state && Tq == 1)   // one token: the single-token kernel on the bf16 state (same layouts)
        decode_kernel<true><<<(unsigned)nblk, DEC_WARPS * 32, 0, stream>>>(q, k, v, graw, b, A_log, scale, state,
                                                                          H_qk, H_v, out);
    else if (bf16_state)
        decode_tokens_kernel<true><<<(unsigned)nblk, DEC_WARPS * 32, 0, stream>>>(q, k, v, graw, b, A_log, scale,
                                                                                   state, Tq, H_qk, H_v, out);
    else
        decode_tokens_kernel<false><<<(unsigned)nblk, DEC_WARPS * 32, 0, stream>>>(q, k, v, graw, b, A_log, scale,
                                                                                    state, Tq, H_qk, H_v, out);
    return cudaGetLastError();
}

}  // namespace kda

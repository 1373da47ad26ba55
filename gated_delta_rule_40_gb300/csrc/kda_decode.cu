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

__global__ __launch_bounds__(DEC_WARPS * 32, 2) void decode_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const uint16_t *__restrict__ graw, const uint16_t *__restrict__ b, const float *__restrict__ A_log,
    float scale, float *__restrict__ state, int H_qk, int H_v, uint16_t *__restrict__ out) {
    const int bh = blockIdx.x;
    const int bi = bh / H_v, h = bh - bi * H_v;
    const int hq = h / (H_v / H_qk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // Lane owns channels 4*lane .. 4*lane+3.
    const size_t qk_off = ((size_t)bi * H_qk + hq) * KD + 4 * lane;
    const size_t hv_off = ((size_t)bi * H_v + h) * KD;
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

    const int r0 = warp * DEC_ROWS;
    float *S = state + (hv_off + r0) * KD;
    float4 s[DEC_ROWS];
#pragma unroll
    for (int i = 0; i < DEC_ROWS; ++i) s[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)i * KD) + lane);
    const float vrow = bf16_to_f(v[hv_off + r0 + (lane & (DEC_ROWS - 1))]);

    float o_mine = 0.f;
#pragma unroll
    for (int i = 0; i < DEC_ROWS; ++i) {
        float4 x = s[i];
        x.x *= dec[0];
        x.y *= dec[1];
        x.z *= dec[2];
        x.w *= dec[3];
        float dk = x.x * kh[0] + x.y * kh[1] + x.z * kh[2] + x.w * kh[3];
        float dq = x.x * qt[0] + x.y * qt[1] + x.z * qt[2] + x.w * qt[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            dk += __shfl_xor_sync(0xffffffffu, dk, o);
            dq += __shfl_xor_sync(0xffffffffu, dq, o);
        }
        const float vi = __shfl_sync(0xffffffffu, vrow, i);
        const float delta = beta * (vi - dk);
        x.x = fmaf(delta, kh[0], x.x);
        x.y = fmaf(delta, kh[1], x.y);
        x.z = fmaf(delta, kh[2], x.z);
        x.w = fmaf(delta, kh[3], x.w);
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
    decode_kernel<<<(unsigned)nblk, DEC_WARPS * 32, 0, stream>>>(q, k, v, graw, b, A_log, scale, state, H_qk,
                                                               H_v, out);
    return cudaGetLastError();
}

}  // namespace kda

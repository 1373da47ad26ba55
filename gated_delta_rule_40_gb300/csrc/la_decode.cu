// Single-token lightning-attention decode: per (b, h), with lambda = exp(-slope[h]),
//   S <- lambda S + v k^T,   o = scale S q
// in one streaming pass over the fp32 [B,H,V,K] state (read once, written once).
// Warp w owns state rows 16 w .. 16 w + 15; lane owns channels 4 lane .. 4 lane + 3.
#include "kda_common.cuh"

namespace kda {

constexpr int LAD_WARPS = 8;
constexpr int LAD_ROWS = KD / LAD_WARPS;   // 16

// Warp sum of 16 per-lane partial sums d[0..15] (one per row).  Halving
// exchanges (xor 16, 8, 4, 2) leave lane l with the partial of row
// 8 b4 + 4 b3 + 2 b2 + b1 (b_i = bit i of l) over its half of the lanes; the
// last exchange (xor 1) completes it.  16 shuffles instead of 80.
__device__ __forceinline__ float la_reduce_scatter16(float (&d)[16], int lane) {
#pragma unroll
    for (int w = 8, m = 16; w >= 1; w >>= 1, m >>= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = up ? d[i] : d[i + w];
            const float keep = up ? d[i + w] : d[i];
            d[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    return d[0] + __shfl_xor_sync(0xffffffffu, d[0], 1);
}

__global__ __launch_bounds__(LAD_WARPS * 32, 2) void la_decode_kernel(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const float *__restrict__ slope, float scale, float *__restrict__ state, int H_qk, int H_v,
    uint16_t *__restrict__ out) {
    const int bh = blockIdx.x;
    const int bi = bh / H_v, h = bh - bi * H_v;
    const int hq = h / (H_v / H_qk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t qk_off = ((size_t)bi * H_qk + hq) * KD + 4 * lane;
    const size_t hv_off = ((size_t)bi * H_v + h) * KD;
    const uint2 qw = *reinterpret_cast<const uint2 *>(q + qk_off);
    const uint2 kw = *reinterpret_cast<const uint2 *>(k + qk_off);
    const float qv[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
    const float kv[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
    const float lambda = ex2(-slope[h] * LOG2E);

    const int r0 = warp * LAD_ROWS;
    float *S = state + (hv_off + r0) * KD;
    float4 s[LAD_ROWS];
#pragma unroll
    for (int i = 0; i < LAD_ROWS; ++i) s[i] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)i * KD) + lane);
    const float vrow = bf16_to_f(v[hv_off + r0 + (lane & (LAD_ROWS - 1))]);
    float d[LAD_ROWS];
#pragma unroll
    for (int i = 0; i < LAD_ROWS; ++i) {
        const float vi = __shfl_sync(0xffffffffu, vrow, i);
        float4 x = s[i];
        x.x = fmaf(lambda, x.x, vi * kv[0]);
        x.y = fmaf(lambda, x.y, vi * kv[1]);
        x.z = fmaf(lambda, x.z, vi * kv[2]);
        x.w = fmaf(lambda, x.w, vi * kv[3]);
        __stcs(reinterpret_cast<float4 *>(S + (size_t)i * KD) + lane, x);
        d[i] = x.x * qv[0] + x.y * qv[1] + x.z * qv[2] + x.w * qv[3];
    }
    const float o = la_reduce_scatter16(d, lane);
    if ((lane & 1) == 0) {
        const int row = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
        out[hv_off + r0 + row] = f_to_bf16(scale * o);
    }
}

cudaError_t launch_la_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *slope, float scale,
                             float *state, int B, int H_qk, int H_v, uint16_t *out, cudaStream_t stream) {
    const long long nblk = (long long)B * H_v;
    if (nblk == 0) return cudaSuccess;
    la_decode_kernel<<<(unsigned)nblk, LAD_WARPS * 32, 0, stream>>>(q, k, v, slope, scale, state, H_qk, H_v, out);
    return cudaGetLastError();
}

}  // namespace kda

// Shared by the chunked forward and backward kernels: the tf32 hi / lo split, a warp's
// three-term split product on mma.sync, and the blocked inverse of I + A for a strictly
// lower-triangular 64 x 64 A.
#pragma once
#include "kda_common.cuh"

namespace kda {

constexpr int AS = CH + 4;              // A / T row stride (floats)
constexpr int XS = 36;                  // inversion scratch row stride (floats)
constexpr int ZS = 20;                  // 16 x 16 inversion scratch row stride (floats)

// tf32 hi / lo split of an fp32 value: x ~ hi + lo with about 21 significant bits
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    const float h = tf32_rn(x);
    hi = __float_as_uint(h);
    lo = tf32_rn_bits(x - h);
}
// One warp: D (16 x 8) += X (16 x 8 KS, row-major, stride xs) . Y (8 KS x 8, row-major, stride ys)
// with mma.sync m16n8k8 tf32 and the three-term split (hi*lo + lo*hi + hi*hi).
// Fragment layout of m16n8k8: a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4);
// b0 (k = t, n = g), b1 (k = t + 4, n = g); d0 (g, 2t), d1 (g, 2t + 1), d2 (g + 8, 2t), d3 (g + 8, 2t + 1).
template <int KS>
__device__ __forceinline__ void split_mma(const float *X, int xs, const float *Y, int ys, int g, int t, float (&d)[4]) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int k = 8 * ks;
        uint32_t ah[4], al[4], bh[2], bl[2];
        split_tf32(X[g * xs + k + t], ah[0], al[0]);
        split_tf32(X[(g + 8) * xs + k + t], ah[1], al[1]);
        split_tf32(X[g * xs + k + t + 4], ah[2], al[2]);
        split_tf32(X[(g + 8) * xs + k + t + 4], ah[3], al[3]);
        split_tf32(Y[(k + t) * ys + g], bh[0], bl[0]);
        split_tf32(Y[(k + t + 4) * ys + g], bh[1], bl[1]);
        mma_tf32(d, ah, bl);
        mma_tf32(d, al, bh);
        mma_tf32(d, ah, bh);
    }
}

// T = (I + A)^{-1} for a strictly lower-triangular 64 x 64 A (fp32, row stride AS): the
// diagonal 16 x 16 blocks by right-looking forward substitution, T10 and T32 as
// -T_ii A_ij T_jj, then the lower-left 32 x 32 block as -T2 (A21 T1), the block products
// on mma.sync with the three-term split.  Reads only the strict lower part of A; all
// threads of the CTA call it (it synchronises them).
template <int NT>
__device__ __forceinline__ void invert_unit_lower64(const float *sA, float *sT, float *sX, int tid, int warp,
                                                    int lane) {
    if (tid < 64) {
        const int bi = tid >> 4, c = tid & 15, o = 16 * bi;
        float t[SUB];
#pragma unroll
        for (int r = 0; r < SUB; ++r) t[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < SUB; ++j)
#pragma unroll
            for (int r = j + 1; r < SUB; ++r) t[r] = fmaf(-sA[(o + r) * AS + o + j], t[j], t[r]);
#pragma unroll
        for (int r = 0; r < SUB; ++r) sT[(o + r) * AS + o + c] = t[r];
    } else {
        for (int idx = tid - 64; idx < 6 * 256; idx += NT - 64) {
            const int blk = idx >> 8, e = idx & 255;
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            sT[(16 * bi + (e >> 4)) * AS + 16 * bj + (e & 15)] = 0.f;
        }
    }
    __syncthreads();
    const int gid = lane >> 2, tig = lane & 3;
    {
        const int b = warp >> 1, n0 = 8 * (warp & 1), bi = 2 * b + 1, bj = 2 * b;
        float *z = sX + b * 16 * ZS;
        if (warp < 4) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            split_mma<2>(sA + (16 * bi) * AS + 16 * bj, AS, sT + (16 * bj) * AS + 16 * bj + n0, AS, gid, tig, d);
            z[gid * ZS + n0 + 2 * tig] = d[0];
            z[gid * ZS + n0 + 2 * tig + 1] = d[1];
            z[(gid + 8) * ZS + n0 + 2 * tig] = d[2];
            z[(gid + 8) * ZS + n0 + 2 * tig + 1] = d[3];
        }
        __syncthreads();
        if (warp < 4) {
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            split_mma<2>(sT + (16 * bi) * AS + 16 * bi, AS, z + n0, ZS, gid, tig, t);
            float *dst = sT + (16 * bi) * AS + 16 * bj + n0;
            dst[gid * AS + 2 * tig] = -t[0];
            dst[gid * AS + 2 * tig + 1] = -t[1];
            dst[(gid + 8) * AS + 2 * tig] = -t[2];
            dst[(gid + 8) * AS + 2 * tig + 1] = -t[3];
        }
    }
    __syncthreads();
    {
        // the 32 x 32 lower-left block: eight 16 x 8 tiles, one per warp (warps past the
        // eighth only take part in the barriers)
        static_assert(NT >= 256, "eight warps compute the lower-left block");
        const bool act = warp < 8;
        const int m0 = 16 * ((warp & 7) >> 2), n0 = 8 * (warp & 3);
        if (act) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            split_mma<4>(sA + (32 + m0) * AS, AS, sT + n0, AS, gid, tig, d);
            sX[(m0 + gid) * XS + n0 + 2 * tig] = d[0];
            sX[(m0 + gid) * XS + n0 + 2 * tig + 1] = d[1];
            sX[(m0 + gid + 8) * XS + n0 + 2 * tig] = d[2];
            sX[(m0 + gid + 8) * XS + n0 + 2 * tig + 1] = d[3];
        }
        __syncthreads();
        if (act) {
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            split_mma<4>(sT + (32 + m0) * AS + 32, AS, sX + n0, XS, gid, tig, t);
            sT[(32 + m0 + gid) * AS + n0 + 2 * tig] = -t[0];
            sT[(32 + m0 + gid) * AS + n0 + 2 * tig + 1] = -t[1];
            sT[(32 + m0 + gid + 8) * AS + n0 + 2 * tig] = -t[2];
            sT[(32 + m0 + gid + 8) * AS + n0 + 2 * tig + 1] = -t[3];
        }
    }
    __syncthreads();
}

}  // namespace kda

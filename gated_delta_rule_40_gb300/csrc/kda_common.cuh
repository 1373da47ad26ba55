// Device helpers shared by the libkda kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda.h"

namespace kda {

constexpr int KD = 128;     // key / value head dimension (K = V = 128)
constexpr int CH = 64;      // chunk length
constexpr int SUB = 16;     // sub-block length inside a chunk
constexpr float LOG2E = 1.4426950408889634f;
constexpr float L2_EPS = 1e-6f;
// Clamp (in log2 units) for the exponents of the diagonal sub-block decay
// factors: 85 nats keeps every factor and its bf16/tf32 image finite.
constexpr float DIAG_CLAMP2 = 85.0f * LOG2E;

// Per-device status word; the first device-side fault of a call wins.
extern __device__ int g_kda_status;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_kda_status, 0, code); }

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Round an fp32 value to the nearest tf32 (ties away), low 13 bits cleared.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
__device__ __forceinline__ uint16_t f_to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
}

// softplus(x) * log2(e) = max(x,0)*log2e + log2(1 + 2^(-|x| log2e))
__device__ __forceinline__ float softplus_log2(float x) {
    float a = fabsf(x) * LOG2E;
    return fmaxf(x, 0.0f) * LOG2E + lg2(1.0f + ex2(-a));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- mma.sync
// D = A * B + D, tf32 inputs (bit patterns), fp32 accumulate, m16n8k8.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// D = A * B + D, bf16 inputs (packed pairs), fp32 accumulate, m16n8k16.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---------------------------------------------------------------- plan
// One entry per chunk of 64 tokens (the last chunk of a sequence may be shorter).
struct ChunkDesc {
    int seq;   // sequence index
    int tok;   // global token row (batch-major: b*T + t)
    int len;   // valid rows (1..64)
    int idx;   // chunk index within its sequence
};
// One entry per sequence.
struct SeqDesc {
    int tok;     // first global token row
    int len;     // tokens
    int chunk0;  // first global chunk index
    int nchunk;  // chunks
};

}  // namespace kda

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
// A tf32 MMA operand rounded to nearest (ties away from zero), as an fp32 bit pattern.  The tensor
// core reads only the upper 19 bits of a tf32 operand, so adding half a tf32 unit in the last place
// (2^12 in the fp32 encoding) before that truncation rounds the magnitude to nearest, ties away from
// zero, in one integer add.  Finite inputs (an infinity would become a NaN pattern).
__device__ __forceinline__ uint32_t tf32_rn_bits(float x) { return __float_as_uint(x) + 0x1000u; }
// The nearest tf32 number itself (the ignored bits cleared), for splitting x into tf32 hi + lo terms.
__device__ __forceinline__ float tf32_rn(float x) { return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u); }
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

// =====================================================================
// tcgen05 / TMEM / mbarrier / bulk-copy helpers (inline PTX, sm_100 family)
// =====================================================================
namespace kda {

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Base of the dynamic shared memory rounded up to ALIGN bytes.  The offset is added to the array
// itself rather than through an integer cast of its address, so the compiler keeps every pointer
// derived from it in the shared state space and emits shared-memory loads and stores (a generic
// pointer would cost 64-bit address arithmetic and a state-space check per access).
template <uint32_t ALIGN>
__device__ __forceinline__ unsigned char *aligned_smem(unsigned char *raw) {
    const uint32_t a = smem_u32(raw);
    return raw + ((ALIGN - (a & (ALIGN - 1u))) & (ALIGN - 1u));
}

// Byte offset of element (row, kbyte) in a K-major, 128-byte-swizzled UMMA
// operand image with `rows` rows: 8-row x 128-byte atoms (1024 B) stacked
// along the rows, then one such column of atoms per 128 bytes of K.  The
// 16-byte chunk index inside a row is XORed with (row % 8).
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int kbyte, int rows) {
    const int atom = kbyte >> 7, kb = kbyte & 127;
    return (uint32_t)(atom * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((kb >> 4) ^ (row & 7))) << 4) +
                      (kb & 15));
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, descriptor version 1, swizzle mode (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptors: fp32 accumulate, K-major A and B, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_smem), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes));
}
// Bounded wait for the phase with the given parity; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, uint32_t limit = (1u << 22)) {
    uint32_t done = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity));
        if (done) return true;
    }
    return false;
}
// Bounded wait that lets the thread sleep up to `hint_ns` per probe (mbarrier.try_wait's
// suspend-time hint): a warp that waits long re-polls rarely and leaves issue slots to the
// others.  The bound is about limit x hint_ns in total; false if it gave up.
__device__ __forceinline__ bool mbar_wait_hint(uint32_t mbar, uint32_t parity, uint32_t hint_ns = 10000u,
                                               uint32_t limit = 200000u) {
    uint32_t done = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity), "r"(hint_ns));
        if (done) return true;
    }
    return false;
}
// Bounded spin on the phase with the given parity with the non-suspending probe
// (test_wait): a thread on a latency-critical hand-off resumes within a probe's
// latency of the phase completing, where a suspended try_wait can take several
// hundred cycles to wake.  False if it gave up.
__device__ __forceinline__ bool mbar_spin(uint32_t mbar, uint32_t parity, uint32_t limit = (1u << 24)) {
    uint32_t done = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}
// Bulk (non-tensor) async copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
                 ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}

}  // namespace kda

namespace kda {
// Bulk shared -> global copies are tracked in bulk groups: commit the issued copies, then
// wait until their shared-memory reads are done (the source may be reused) or they complete.
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
}  // namespace kda

namespace kda {
// Programmatic dependent launch: a kernel launched with programmatic stream serialisation may
// start while the previous kernel on the stream is still running; grid_dep_wait() blocks until
// that kernel has completed and its memory is visible (it returns at once when the kernel was
// launched normally), and grid_dep_launch() lets the next kernel on the stream be scheduled
// early.  Nothing spins on memory: the dependency is resolved by the launch hardware.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
}  // namespace kda

namespace kda {
// Prefetch the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_line_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
// Bulk prefetch of a global range into L2 (no shared memory involved).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
}  // namespace kda

namespace kda {
// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting;
// call tmem_wait_ld() before using the registers.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}
// Named barrier over `nthreads` threads (multiple of 32) with id 1..15.
__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}
}  // namespace kda

namespace kda {
// 16 consecutive fp32 columns of this thread's TMEM lane, without waiting.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
}  // namespace kda

namespace kda {
// L2 policy: lines written by the following accesses are evicted first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// Bulk shared -> global copy with an L2 cache-eviction hint.
__device__ __forceinline__ void bulk_s2g_hint(void *dst, uint32_t src_smem, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;\n" ::"l"(dst),
                 "r"(src_smem), "r"(bytes), "l"(pol)
                 : "memory");
}
}  // namespace kda

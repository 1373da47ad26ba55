// Tensor-memory-accelerator (TMA) helpers shared by the chunked kernels: the device-side
// tiled load and the host-side tensor-map encoding of a [rows][heads][128] bf16 tensor.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace kda {

// Tiled 3-D load of one box into shared memory, completion counted on an mbarrier.
// Coordinates are (channel, head, row); rows past the tensor are filled with zeros.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

// Prefetch of one box of a tiled 3-D tensor into L2 (no shared memory, no completion tracking)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Tiled 3-D store of one box from shared memory (completion tracked by the issuing thread's bulk
// groups: cp.async.bulk.commit_group / wait_group).  The shared-memory writes it reads must be
// made visible to the async proxy (fence.proxy.async) and ordered before it by a barrier.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int x, int y, int z, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (looked up once).
inline cudaError_t tma_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn_out) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *fn_out = enc;
    return cudaSuccess;
}

// [rows][heads][128] bf16 as a 3-D tensor (channel, head, row); boxes of box_ch channels x 1 head
// x 64 rows, with the given shared-memory swizzle, zero fill past the last row.  With a swizzle,
// box_ch x 2 bytes must equal its span (32 channels with 64-byte swizzle, 64 with 128-byte
// swizzle); without one, box_ch = 128 (whole 256-byte rows).
inline cudaError_t tma_map_rows_heads(CUtensorMap *m, const void *base, long long rows, int heads, int box_ch,
                                      CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    const cudaError_t e = tma_encoder(&enc);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {(cuuint64_t)128, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * 2, (cuuint64_t)heads * 128 * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_ch, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace kda

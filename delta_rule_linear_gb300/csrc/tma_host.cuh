// tma_host.cuh -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled),
// reached through the runtime's driver entry point so that the library needs no
// link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace kda {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tiled map over a tensor of `rank` dims (dims[0] innermost, element counts),
// strides in bytes for dims 1..rank-1, box sizes per dim, 128-byte swizzle for
// 16-bit data whose inner box is 64 elements (or no swizzle when swizzle128 = false).
inline bool make_tensor_map(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                            const uint64_t *dims, const uint64_t *strides_bytes,
                            const uint32_t *box, CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    uint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, dt, (cuuint32_t)rank, const_cast<void *>(base),
                     reinterpret_cast<const cuuint64_t *>(dims),
                     reinterpret_cast<const cuuint64_t *>(strides_bytes),
                     reinterpret_cast<const cuuint32_t *>(box), estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
inline bool make_tensor_map(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                            const uint64_t *dims, const uint64_t *strides_bytes,
                            const uint32_t *box, bool swizzle128) {
    return make_tensor_map(map, dt, rank, base, dims, strides_bytes, box,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace kda

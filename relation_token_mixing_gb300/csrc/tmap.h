// Host helper: TMA tensor maps for contiguous [BH, T, d] tensors, obtained
// through the runtime's driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace relation {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a contiguous [BH, T, d] tensor of 2- or 4-byte elements with box
// {box_x (along d), box_y (along T), 1}, 128-byte swizzle, zero fill outside.
inline cudaError_t make_tensor_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                                      uint32_t elem_bytes, uint64_t d, uint64_t T, uint64_t BH, uint32_t box_x,
                                      uint32_t box_y, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {d, T, BH};
    const cuuint64_t strides[2] = {d * elem_bytes, T * d * elem_bytes};
    const cuuint32_t box[3] = {box_x, box_y, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace relation

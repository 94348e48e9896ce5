// Host helpers: TMA tensor maps, obtained through the runtime's driver entry
// point (no link-time dependency on libcuda).
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

// Map over an operand tensor, 2-byte elements, box {box_x (along d), box_y
// (along T)}, 128-byte swizzle: a 4-D map (d, T, H, B) for either layout, or,
// when allow_3d is set, a 3-D map (d, T, B*H) for [B, H, T, d] (layout 0).
// (Measured: the backward runs faster from the 3-D form, the forward from the
// 4-D form.)  Columns past d
// and rows past T read as zero, so a tile of a narrower head is the wider tile
// with zero columns.  Every stride must be a multiple of 16 bytes
// (d * 2 % 16 == 0); the caller checks.
inline cudaError_t make_operand_map(CUtensorMap* map, const void* base, int64_t B, int64_t H, int64_t T, int64_t d,
                                    int layout, uint32_t box_x, uint32_t box_y, bool allow_3d) {
    if (allow_3d && layout == 0)
        return make_tensor_map_3d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)T,
                                  (uint64_t)(B * H), box_x, box_y, CU_TENSOR_MAP_SWIZZLE_128B);
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    const uint64_t e = 2;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {layout == 0 ? (cuuint64_t)(d * e) : (cuuint64_t)(H * d * e),
                                   layout == 0 ? (cuuint64_t)(T * d * e) : (cuuint64_t)(d * e),
                                   (cuuint64_t)(H * T * d * e)};
    const cuuint32_t box[4] = {box_x, box_y, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace relation

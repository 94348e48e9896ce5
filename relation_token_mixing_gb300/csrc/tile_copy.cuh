// Operand tiles for head widths whose rows the tensor memory accelerator cannot
// address (d_h * 2 bytes not a multiple of 16, e.g. d_h = 60): a full warp
// copies the tile with 8-byte cp.async (LDGSTS) into exactly the layout a TMA
// load with 128-byte swizzle would produce, so the MMA descriptors are the same.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace relation {

// 8-byte global -> shared copy.  (Measured: 9 % faster in the forward than the
// zero-filling form with a source-size operand, so padding is stored directly.)
__device__ __forceinline__ void cp_async_8(uint32_t smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void st_shared_zero8(uint32_t smem_dst) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(smem_dst), "r"(0u) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Rows row0 .. row0+127, columns 0..63 of head bh of a bf16 operand tensor of
// width kp.d <= 64 (a multiple of 4) into a 128 x 64 tile: row r at r*128
// bytes, 16-byte chunk c at ((c ^ (r & 7)) * 16).  Columns >= d and rows >= T
// are zero.  Called by all 32 lanes of a warp (64 copies each; lanes 0-15 and
// 16-31 cover two consecutive rows per instruction).
__device__ __forceinline__ void cp_async_tile64(uint8_t* tile, const __nv_bfloat16* src, const KernelProblem& kp,
                                                int64_t bh, int row0, int lane) {
    const uint32_t base = ptx::smem_u32(tile);
#pragma unroll 8
    for (int k = 0; k < 64; ++k) {
        const int idx = lane + 32 * k;
        const int r = idx >> 4, q = idx & 15;  // row, 8-byte unit (columns 4q .. 4q+3)
        const int row = row0 + r, col = 4 * q;
        const bool valid = row < kp.T && col < kp.d;
        const uint32_t dst = base + r * 128 + (((q >> 1) ^ (r & 7)) << 4) + ((q & 1) << 3);
        if (valid)
            cp_async_8(dst, src + row_offset(kp, bh, row) + col);
        else
            st_shared_zero8(dst);
    }
}

// Makes this warp's completed cp.async writes (and zero stores) visible to the
// tensor cores (async proxy): every lane waits for its copies and fences, then
// the warp converges; the caller arrives on the consumers' mbarrier afterwards.
template <int kPendingGroups>
__device__ __forceinline__ void cp_async_publish() {
    cp_async_wait<kPendingGroups>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
}

}  // namespace relation

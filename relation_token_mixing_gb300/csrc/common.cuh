// Shared device-side definitions of the Relation library: problem description
// passed to kernels, the device status word, and small numeric helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace relation {

// Codes written into the device status word (first nonzero code wins).
enum DeviceStatus : unsigned int {
    kDevOk = 0,
    kDevTimeoutFull = 1,    // a consumer gave up waiting for data
    kDevTimeoutEmpty = 2,   // a producer gave up waiting for a free buffer
    kDevTimeoutMma = 3,     // a wait on tensor-core completion expired
    kDevBadLaunch = 4,      // a kernel saw a launch shape it was not built for
    kDevBadPosition = 5,    // a decode position outside the cache (the head was skipped)
};
// Flag OR-ed into the status word (beside the first code) when a CTA that gave up
// waiting also gave up draining its own asynchronous copies or tensor-core work
// and returned with some of it possibly still in flight.
constexpr unsigned int kDevDrainIncomplete = 0x100u;

// Kernel-side view of one problem.  Operand tensors (P1, P2, V, Y, dY, dP1,
// dP2, dV) are contiguous [B, H, T, d] (layout 0) or [B, T, H, d] (layout 1);
// L, D and the dP1 accumulator are always [B*H, T(, d_pad)].
struct KernelProblem {
    int64_t BH;
    int T;
    int d;
    float tau_S;
    float lambda;
    int causal;
    float inv_sqrt_d;
    int H;
    int layout;
};

// RoPE angle: sin and cos of 2 pi pos f_c, with f_c = base^(-2c/d) / (2 pi) given
// as the float pair (hi, lo): pos * f_c is split into its integer and fractional
// turns in float-float arithmetic, so large positions keep the angle accurate.
__device__ __forceinline__ void rope_sincos(float pos, float hi, float lo, float* s, float* c) {
    const float p_hi = pos * hi;
    const float p_err = fmaf(pos, hi, -p_hi);  // exact rounding error of the product
    const float p_lo = fmaf(pos, lo, p_err);
    const float frac = (p_hi - rintf(p_hi)) + p_lo;
    sincospif(2.f * frac, s, c);
}

// Givens mixing of head h's information states with its pair partner (pairing
// 0: (0,1), (2,3), ...; pairing 1: (1,2), ..., (H-1,0), zero-based heads):
// I~_h = cs I_h + sn I_partner.  Returns the partner and the pair index k.
__device__ __forceinline__ int givens_partner(int h, int H, int pairing, int* k, bool* is_first) {
    if (pairing == 0) {
        *k = h >> 1;
        *is_first = (h & 1) == 0;
        return h ^ 1;
    }
    if (h & 1) {  // first of pair (h, h+1 mod H)
        *k = (h - 1) >> 1;
        *is_first = true;
        return (h + 1) % H;
    }
    *k = (h == 0 ? H : h) / 2 - 1;  // second of pair (h-1 mod H, h)
    *is_first = false;
    return (h == 0 ? H : h) - 1;
}

// Element offset of row t of head bh (= b*H + h) in an operand tensor.
__host__ __device__ __forceinline__ size_t row_offset(const KernelProblem& kp, int64_t bh, int64_t t) {
    if (kp.layout == 0) return ((size_t)bh * (size_t)kp.T + (size_t)t) * (size_t)kp.d;
    const int64_t b = bh / kp.H, h = bh - b * kp.H;
    return (((size_t)b * (size_t)kp.T + (size_t)t) * (size_t)kp.H + (size_t)h) * (size_t)kp.d;
}

// Stores columns c..c+7 (four packed bf16 pairs) of one row of width d (d a
// multiple of 4, c a multiple of 8): one 16-byte store when the whole group is
// inside the row and rows are 16-byte aligned (d % 8 == 0), else 8-byte halves;
// columns >= d are not written.
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* row, int c, int d, uint32_t w0, uint32_t w1, uint32_t w2,
                                             uint32_t w3) {
    if (c + 8 <= d && (d & 7) == 0) {
        *reinterpret_cast<uint4*>(row + c) = make_uint4(w0, w1, w2, w3);
        return;
    }
    if (c + 4 <= d) *reinterpret_cast<uint2*>(row + c) = make_uint2(w0, w1);
    if (c + 8 <= d) *reinterpret_cast<uint2*>(row + c + 4) = make_uint2(w2, w3);
}

// CTA launch order of the key-stationary backward: the linear block index
// walks groups of `group` heads; inside a group it walks tile index 0 of all
// those heads, then tile 1, and so on (heaviest first for causal masks), so the
// causal tail stays short while the heads in flight at any time stay few enough
// for their inputs and fp32 accumulators to remain in L2.
__host__ __device__ __forceinline__ void grouped_tile_order(unsigned idx, int64_t BH, int n_tiles, int group,
                                                            int& bh, int& tile) {
    const unsigned per_group = (unsigned)group * (unsigned)n_tiles;
    const int64_t g = idx / per_group;
    const int r = (int)(idx - g * per_group);
    const int heads = (int)((BH - g * group) < group ? (BH - g * group) : group);
    tile = r / heads;
    bh = (int)(g * group) + (r - tile * heads);
}

// Heads per group for grouped_tile_order: at most `most` (what fits in L2), with
// the groups as equal in size as possible.  A small last group would start its
// longest key tiles only when the other groups' CTAs are nearly done, leaving the
// rest of the GPU idle while they finish.
inline int64_t balanced_head_group(int64_t BH, int64_t most) {
    most = most < 1 ? 1 : (most > BH ? BH : most);
    const int64_t groups = (BH + most - 1) / most;
    return (BH + groups - 1) / groups;
}

// Records the first failure in the status word; never traps.
__device__ __forceinline__ void record_status(unsigned int* status, unsigned int code) {
    if (status != nullptr) atomicCAS(status, 0u, code);
}

// Nanoseconds since an arbitrary epoch (used only to bound waits).
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// How long any single device-side wait may last before it is abandoned.
#ifndef RELATION_WAIT_LIMIT_NS
#define RELATION_WAIT_LIMIT_NS 4000000000ull
#endif

__device__ __forceinline__ float bf16_to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_from_float(T* p, float v);
template <>
__device__ __forceinline__ void store_from_float<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_from_float<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

}  // namespace relation

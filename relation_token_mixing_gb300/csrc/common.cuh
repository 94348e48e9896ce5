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
};

// Kernel-side view of one problem.  Strides are in elements of the tensors;
// all tensors are contiguous [B*H, T, d].
struct KernelProblem {
    int64_t BH;
    int T;
    int d;
    float tau_S;
    float lambda;
    int causal;
    float inv_sqrt_d;
};

// CTA launch order of the key-stationary backward: the linear block index
// walks groups of `group` heads; inside a group it walks tile index 0 of all
// those heads, then tile 1, and so on (heaviest first for causal masks), so the
// causal tail stays short while the heads in flight at any time stay few enough
// for their inputs and fp32 accumulators to remain in L2.
__device__ __forceinline__ void grouped_tile_order(unsigned idx, int64_t BH, int n_tiles, int group, int& bh,
                                                   int& tile) {
    const unsigned per_group = (unsigned)group * (unsigned)n_tiles;
    const int64_t g = idx / per_group;
    const int r = (int)(idx - g * per_group);
    const int heads = (int)((BH - g * group) < group ? (BH - g * group) : group);
    tile = r / heads;
    bh = (int)(g * group) + (r - tile * heads);
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

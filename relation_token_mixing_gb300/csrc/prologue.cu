// Input prologue of the operator and its backward ("Ask Self, Ask Others:
// Relation Is All You Need"):
//  - RoPE on the relation coordinates P1, P2 (Sec. 3.1 below eq.(1); Appendix
//    B.3: full head width, base 10^4; the information states stay unrotated).
//    Coordinate c in [0, d/2) turns together with c + d/2 by the angle
//    pos * base^(-2c/d), pos = pos0[b] + t the zero-based token position.
//  - Givens mixing of the information states of adjacent head pairs (Sec. 3.2
//    eq.(4); Appendix A.2.2-A.2.3): I~a = cos(th) Ia - sin(th) Ib,
//    I~b = sin(th) Ia + cos(th) Ib, pairing A = (0,1),(2,3),..., pairing B =
//    (1,2),...,(H-1,0) (zero-based), one angle per pair.
// Backward: the transposed rotations, and d theta_k = sum (dI~b . I~a - dI~a . I~b).
// All passes are HBM-bound elementwise kernels (two columns per thread).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace relation {
namespace {

constexpr int kThreads = 256;

// sin and cos of 2 pi pos f_c, with f_c = base^(-2c/d) / (2 pi) given as the
// float pair (hi, lo): pos * f_c is split into its integer and fractional
// turns in float-float arithmetic, so large positions keep the angle accurate.
__device__ __forceinline__ void rope_sincos(float pos, float hi, float lo, float* s, float* c) {
    const float p_hi = pos * hi;
    const float p_err = fmaf(pos, hi, -p_hi);  // exact rounding error of the product
    const float p_lo = fmaf(pos, lo, p_err);
    const float frac = (p_hi - rintf(p_hi)) + p_lo;
    sincospif(2.f * frac, s, c);
}

template <typename T>
__device__ __forceinline__ void load2(const T* p, float& a, float& b) {
    a = load_as_float(p);
    b = load_as_float(p + 1);
}
template <typename T>
__device__ __forceinline__ void store2(T* p, float a, float b) {
    store_from_float(p, a);
    store_from_float(p + 1, b);
}

// RoPE of operand blockIdx.y (0: P1, 1: P2), forward (sign = +1) or transposed
// (sign = -1, the backward).  One thread per (row, column pair c, c+1) of the
// first half; base <= 0 copies.
template <typename T>
__global__ void __launch_bounds__(kThreads) rope_kernel(KernelProblem kp, const T* __restrict__ x0,
                                                        const T* __restrict__ x1, T* __restrict__ y0,
                                                        T* __restrict__ y1, const int* __restrict__ pos0,
                                                        RopeTable tab, float sign, int64_t units) {
    const T* __restrict__ x = blockIdx.y == 0 ? x0 : x1;
    T* __restrict__ y = blockIdx.y == 0 ? y0 : y1;
    const int half = kp.d / 2, per_row = half / 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < units; k += stride) {
        const int64_t row = k / per_row;
        const int c = (int)(k - row * per_row) * 2;
        const int64_t bh = row / kp.T;
        const int t = (int)(row - bh * kp.T);
        const size_t off = row_offset(kp, bh, t);
        float a0, a1, b0, b1;  // columns c, c+1 and their partners c+d/2, c+1+d/2
        load2(x + off + c, a0, a1);
        load2(x + off + c + half, b0, b1);
        if (tab.enabled) {
            const float pos = (float)((pos0 != nullptr ? pos0[bh / kp.H] : 0) + t);
            float s0, c0, s1, c1;
            rope_sincos(pos, tab.hi[c], tab.lo[c], &s0, &c0);
            rope_sincos(pos, tab.hi[c + 1], tab.lo[c + 1], &s1, &c1);
            s0 *= sign;
            s1 *= sign;
            const float r0 = c0 * a0 - s0 * b0, q0 = s0 * a0 + c0 * b0;
            const float r1 = c1 * a1 - s1 * b1, q1 = s1 * a1 + c1 * b1;
            a0 = r0, b0 = q0, a1 = r1, b1 = q1;
        }
        store2(y + off + c, a0, a1);
        store2(y + off + c + half, b0, b1);
    }
}

// Givens mixing of the information states, forward (I -> I~) or backward
// (dI~ -> dI, plus d theta from the mixed states Im = I~ when dtheta != NULL).
// One warp per (batch, token, head pair); lanes cover column pairs.
template <typename T>
__global__ void __launch_bounds__(kThreads) givens_kernel(KernelProblem kp, const T* __restrict__ x,
                                                          const T* __restrict__ Im, T* __restrict__ y,
                                                          const float* __restrict__ theta, int pairing, float sign,
                                                          float* __restrict__ dtheta, int64_t rows) {
    extern __shared__ float acc[];  // per-block partial d theta, H/2 entries
    const int P = kp.H / 2;
    const int lane = threadIdx.x & 31;
    if (dtheta != nullptr)
        for (int k = threadIdx.x; k < P; k += blockDim.x) acc[k] = 0.f;
    __syncthreads();
    const int64_t wstride = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows; r += wstride) {
        const int pr = (int)(r % P);
        const int64_t bt = r / P;
        const int t = (int)(bt % kp.T);
        const int64_t b = bt / kp.T;
        const int ha = pairing == 0 ? 2 * pr : 2 * pr + 1;
        const int hb = pairing == 0 ? 2 * pr + 1 : (2 * pr + 2) % kp.H;
        const size_t oa = row_offset(kp, b * kp.H + ha, t), ob = row_offset(kp, b * kp.H + hb, t);
        float sn, cs;
        sincosf(theta[pr], &sn, &cs);
        sn *= sign;  // -1: the transposed rotation
        float part = 0.f;
        for (int c = 2 * lane; c < kp.d; c += 64) {
            float a0, a1, b0, b1;
            load2(x + oa + c, a0, a1);
            load2(x + ob + c, b0, b1);
            store2(y + oa + c, cs * a0 - sn * b0, cs * a1 - sn * b1);
            store2(y + ob + c, sn * a0 + cs * b0, sn * a1 + cs * b1);
            if (dtheta != nullptr) {  // x = dI~: dI~b . I~a - dI~a . I~b
                float ma0, ma1, mb0, mb1;
                load2(Im + oa + c, ma0, ma1);
                load2(Im + ob + c, mb0, mb1);
                part += b0 * ma0 + b1 * ma1 - a0 * mb0 - a1 * mb1;
            }
        }
        if (dtheta != nullptr) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) atomicAdd(&acc[pr], part);
        }
    }
    if (dtheta == nullptr) return;
    __syncthreads();
    for (int k = threadIdx.x; k < P; k += blockDim.x)
        if (acc[k] != 0.f) atomicAdd(&dtheta[k], acc[k]);
}

int64_t blocks_for(int64_t units, int num_sms) {
    int64_t b = (units + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms * 8;
    return b < 1 ? 1 : (b > cap ? cap : b);
}

template <typename T>
cudaError_t launch_rope_t(const KernelProblem& kp, const void* x0, const void* x1, void* y0, void* y1,
                          const int* pos0, const RopeTable& tab, float sign, int num_sms, cudaStream_t s) {
    const int64_t units = kp.BH * (int64_t)kp.T * (kp.d / 4);
    rope_kernel<T><<<dim3((unsigned)blocks_for(units, num_sms), 2), kThreads, 0, s>>>(
        kp, (const T*)x0, (const T*)x1, (T*)y0, (T*)y1, pos0, tab, sign, units);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_givens_t(const KernelProblem& kp, const void* x, const void* Im, void* y, const float* theta,
                            int pairing, float sign, float* dtheta, int num_sms, cudaStream_t s) {
    const int64_t rows = (kp.BH / 2) * (int64_t)kp.T;  // (batch, token, head pair)
    const size_t smem = dtheta != nullptr ? sizeof(float) * (size_t)(kp.H / 2) : 0;
    givens_kernel<T><<<(unsigned)blocks_for(rows * 32, num_sms), kThreads, smem, s>>>(
        kp, (const T*)x, (const T*)Im, (T*)y, theta, pairing, sign, dtheta, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const KernelProblem& kp, bool bf16, const void* x0, const void* x1, void* y0, void* y1,
                        const int* pos0, const RopeTable& tab, bool transpose, int num_sms, cudaStream_t s) {
    const float sign = transpose ? -1.f : 1.f;
    return bf16 ? launch_rope_t<__nv_bfloat16>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s)
                : launch_rope_t<float>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s);
}

cudaError_t launch_givens(const KernelProblem& kp, bool bf16, const void* x, const void* Im, void* y,
                          const float* theta, int pairing, bool transpose, float* dtheta, int num_sms,
                          cudaStream_t s) {
    const float sign = transpose ? -1.f : 1.f;
    return bf16 ? launch_givens_t<__nv_bfloat16>(kp, x, Im, y, theta, pairing, sign, dtheta, num_sms, s)
                : launch_givens_t<float>(kp, x, Im, y, theta, pairing, sign, dtheta, num_sms, s);
}

}  // namespace relation

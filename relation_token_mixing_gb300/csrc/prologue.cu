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

// VC consecutive elements as fp32 (16-, 8- or 4-byte loads for bf16 VC = 8, 4, 2;
// 16- / 8-byte for fp32).
template <typename T, int VC>
__device__ __forceinline__ void loadv(const T* p, float (&v)[VC]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t w[VC / 2];
        if constexpr (VC == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p);
            w[0] = u.x;
            w[1] = u.y;
            w[2] = u.z;
            w[3] = u.w;
        } else if constexpr (VC == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            w[0] = u.x;
            w[1] = u.y;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        }
#pragma unroll
        for (int k = 0; k < VC / 2; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else if constexpr (VC == 4) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        v[0] = u.x, v[1] = u.y, v[2] = u.z, v[3] = u.w;
    } else {
        const float2 u = *reinterpret_cast<const float2*>(p);
        v[0] = u.x, v[1] = u.y;
    }
}
template <typename T, int VC>
__device__ __forceinline__ void storev(T* p, const float (&v)[VC]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t w[VC / 2];
#pragma unroll
        for (int k = 0; k < VC / 2; ++k) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&b);
        }
        if constexpr (VC == 8)
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        else if constexpr (VC == 4)
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t*>(p) = w[0];
    } else if constexpr (VC == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    }
}

// RoPE of P1 and P2 (x0 -> y0, x1 -> y1), forward (sign = +1) or transposed
// (sign = -1, the backward).  The angle depends on (batch, token, column) only,
// so one thread takes VC columns c.. of the first half (and their partners
// c + d/2) of one (batch, token) and applies them to every kRopeHeadSplit-th
// head of both tensors (the split gives the loads enough threads in flight).
constexpr int kRopeHeadSplit = 4;
// Idx: the flat index type (32-bit whenever the index space fits: its divisions
// are several times cheaper than 64-bit ones).
template <typename T, int VC, typename Idx>
__global__ void __launch_bounds__(kThreads) rope_kernel(KernelProblem kp, const T* __restrict__ x0,
                                                        const T* __restrict__ x1, T* __restrict__ y0,
                                                        T* __restrict__ y1, const int* __restrict__ pos0,
                                                        RopeTable tab, float sign, Idx units) {
    const int half = kp.d / 2;
    const int hsplit = kp.H < kRopeHeadSplit ? kp.H : kRopeHeadSplit;
    const Idx per_row = (Idx)(half / VC) * hsplit, Tn = (Idx)kp.T;
    const Idx stride = (Idx)gridDim.x * blockDim.x;
    for (Idx k = (Idx)blockIdx.x * blockDim.x + threadIdx.x; k < units; k += stride) {
        const Idx bt = k / per_row;
        const int w = (int)(k - bt * per_row);
        const int hg = w % hsplit;  // this thread's heads: hg, hg + hsplit, ...
        const int c = (w / hsplit) * VC;
        const Idx b = bt / Tn;
        const int t = (int)(bt - b * Tn);
        float sn[VC], cs[VC];
        if (tab.enabled) {
            const float pos = (float)((pos0 != nullptr ? pos0[b] : 0) + t);
#pragma unroll
            for (int v = 0; v < VC; ++v) {
                rope_sincos(pos, tab.hi[c + v], tab.lo[c + v], &sn[v], &cs[v]);
                sn[v] *= sign;
            }
        } else {
#pragma unroll
            for (int v = 0; v < VC; ++v) sn[v] = 0.f, cs[v] = 1.f;
        }
        for (int h = hg; h < kp.H; h += hsplit) {
            const size_t off = row_offset(kp, (int64_t)b * kp.H + h, t) + c;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const T* x = which ? x1 : x0;
                T* y = which ? y1 : y0;
                float a[VC], q[VC], ra[VC], rq[VC];
                loadv<T, VC>(x + off, a);
                loadv<T, VC>(x + off + half, q);
#pragma unroll
                for (int v = 0; v < VC; ++v) {
                    ra[v] = cs[v] * a[v] - sn[v] * q[v];
                    rq[v] = sn[v] * a[v] + cs[v] * q[v];
                }
                storev<T, VC>(y + off, ra);
                storev<T, VC>(y + off + half, rq);
            }
        }
    }
}

// Givens mixing of the information states, forward (I -> I~) or backward
// (dI~ -> dI, plus d theta from the mixed states Im = I~ when dtheta != NULL;
// im_unmixed: Im holds the unmixed states I, mixed here for the d theta products).
// A group of LPR lanes takes one (batch, token, head pair), VC columns per lane
// (LPR * VC >= d), so a warp covers 32 / LPR pairs per step with 16-byte
// accesses where the rows allow them.
template <typename T, int VC, int LPR, typename Idx>
__global__ void __launch_bounds__(kThreads) givens_kernel(KernelProblem kp, const T* __restrict__ x,
                                                          const T* __restrict__ Im, T* __restrict__ y,
                                                          const float* __restrict__ theta, int pairing, float sign,
                                                          float* __restrict__ dtheta, Idx rows, bool im_unmixed) {
    constexpr int kRowsPerWarp = 32 / LPR;
    extern __shared__ float sh[];  // cos, sin, partial d theta: 3 x H/2
    const int P = kp.H / 2;
    float* scos = sh;
    float* ssin = sh + P;
    float* acc = sh + 2 * P;
    for (int k = threadIdx.x; k < P; k += blockDim.x) {
        float sn, cs;
        sincosf(theta[k], &sn, &cs);
        scos[k] = cs;
        ssin[k] = sign * sn;  // -1: the transposed rotation
        acc[k] = 0.f;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, li = lane % LPR;
    const int c = VC * li;
    const bool on = c < kp.d;
    const Idx Pn = (Idx)P, Tn = (Idx)kp.T;
    const Idx first = ((Idx)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * kRowsPerWarp + sub;
    const Idx step = (Idx)gridDim.x * (blockDim.x / 32) * kRowsPerWarp;
    const Idx rows_rounded = (rows + kRowsPerWarp - 1) / kRowsPerWarp * kRowsPerWarp;
    for (Idx r0 = first; r0 < rows_rounded + sub; r0 += step) {  // same trip count for every lane of the warp
        const Idx r = r0;
        const bool valid = r < rows;
        float part = 0.f;
        int pr = 0;
        if (valid) {
            const Idx bt = r / Pn;
            pr = (int)(r - bt * Pn);
            const Idx b = bt / Tn;
            const int t = (int)(bt - b * Tn);
            const int ha = pairing == 0 ? 2 * pr : 2 * pr + 1;
            const int hb = pairing == 0 ? 2 * pr + 1 : (2 * pr + 2) % kp.H;
            const size_t oa = row_offset(kp, (int64_t)b * kp.H + ha, t) + c;
            const size_t ob = row_offset(kp, (int64_t)b * kp.H + hb, t) + c;
            const float cs = scos[pr], sn = ssin[pr];
            if (on) {
                float a[VC], q[VC], ya[VC], yb[VC];
                loadv<T, VC>(x + oa, a);
                loadv<T, VC>(x + ob, q);
#pragma unroll
                for (int v = 0; v < VC; ++v) {
                    ya[v] = cs * a[v] - sn * q[v];
                    yb[v] = sn * a[v] + cs * q[v];
                }
                storev<T, VC>(y + oa, ya);
                storev<T, VC>(y + ob, yb);
                if (dtheta != nullptr) {  // x = dI~: dI~b . I~a - dI~a . I~b
                    float ma[VC], mb[VC];
                    loadv<T, VC>(Im + oa, ma);
                    loadv<T, VC>(Im + ob, mb);
                    if (im_unmixed) {  // sn = -sin here: I~a = cos Ia - sin Ib, I~b = sin Ia + cos Ib
#pragma unroll
                        for (int v = 0; v < VC; ++v) {
                            const float ta = fmaf(cs, ma[v], sn * mb[v]), tb = fmaf(cs, mb[v], -sn * ma[v]);
                            ma[v] = ta;
                            mb[v] = tb;
                        }
                    }
#pragma unroll
                    for (int v = 0; v < VC; ++v) part += q[v] * ma[v] - a[v] * mb[v];
                }
            }
        }
        if (dtheta != nullptr) {
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (valid && li == 0) atomicAdd(&acc[pr], part);
        }
    }
    if (dtheta == nullptr) return;
    __syncthreads();
    for (int k = threadIdx.x; k < P; k += blockDim.x)
        if (acc[k] != 0.f) atomicAdd(&dtheta[k], acc[k]);
}

// dX1 = R^T dP1 from the fp32 dP1 accumulator [BH, T, 64] (rotated coordinates)
// to bf16 in the problem's layout (d_h = 64): one thread per (row, four
// coordinate pairs c, c + 32).
__global__ void __launch_bounds__(kThreads) rope_convert_kernel(KernelProblem kp, const float* __restrict__ dq,
                                                                __nv_bfloat16* __restrict__ dst,
                                                                const int* __restrict__ pos0, RopeTable tab,
                                                                int64_t units) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < units; k += stride) {
        const int64_t row = k >> 3;
        const int c = 4 * (int)(k & 7);
        const int64_t bh = row / kp.T;
        const int t = (int)(row - bh * kp.T);
        const float4 g1 = *reinterpret_cast<const float4*>(dq + (size_t)row * 64 + c);
        const float4 g2 = *reinterpret_cast<const float4*>(dq + (size_t)row * 64 + 32 + c);
        const float a[4] = {g1.x, g1.y, g1.z, g1.w}, b[4] = {g2.x, g2.y, g2.z, g2.w};
        float o1[4], o2[4];
        const float pos = (float)((pos0 != nullptr ? pos0[bh / kp.H] : 0) + t);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            float sn = 0.f, cs = 1.f;
            if (tab.enabled) rope_sincos(pos, tab.hi[c + v], tab.lo[c + v], &sn, &cs);
            o1[v] = fmaf(cs, a[v], sn * b[v]);
            o2[v] = fmaf(cs, b[v], -sn * a[v]);
        }
        __nv_bfloat16* o = dst + row_offset(kp, bh, t);
        storev<__nv_bfloat16, 4>(o + c, o1);
        storev<__nv_bfloat16, 4>(o + 32 + c, o2);
    }
}

int64_t blocks_for(int64_t units, int num_sms) {
    int64_t b = (units + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms * 8;
    return b < 1 ? 1 : (b > cap ? cap : b);
}

template <typename T, int VC>
cudaError_t launch_rope_t(const KernelProblem& kp, const void* x0, const void* x1, void* y0, void* y1,
                          const int* pos0, const RopeTable& tab, float sign, int num_sms, cudaStream_t s) {
    const int hsplit = kp.H < kRopeHeadSplit ? kp.H : kRopeHeadSplit;
    const int64_t units = (kp.BH / kp.H) * (int64_t)kp.T * (kp.d / 2 / VC) * hsplit;  // (batch, token, cols, heads)
    const unsigned blocks = (unsigned)blocks_for(units, num_sms);
    if (units + (int64_t)blocks * kThreads < (int64_t)UINT32_MAX)
        rope_kernel<T, VC, uint32_t><<<blocks, kThreads, 0, s>>>(kp, (const T*)x0, (const T*)x1, (T*)y0, (T*)y1,
                                                                 pos0, tab, sign, (uint32_t)units);
    else
        rope_kernel<T, VC, uint64_t><<<blocks, kThreads, 0, s>>>(kp, (const T*)x0, (const T*)x1, (T*)y0, (T*)y1,
                                                                 pos0, tab, sign, (uint64_t)units);
    return cudaGetLastError();
}

template <typename T, int VC, int LPR>
cudaError_t launch_givens_t(const KernelProblem& kp, const void* x, const void* Im, void* y, const float* theta,
                            int pairing, float sign, float* dtheta, int num_sms, cudaStream_t s, bool im_unmixed) {
    const int64_t rows = (kp.BH / 2) * (int64_t)kp.T;  // (batch, token, head pair)
    const size_t smem = sizeof(float) * 3 * (size_t)(kp.H / 2);
    const unsigned blocks = (unsigned)blocks_for(rows * LPR, num_sms);
    if (rows + (int64_t)blocks * kThreads < (int64_t)UINT32_MAX)
        givens_kernel<T, VC, LPR, uint32_t><<<blocks, kThreads, smem, s>>>(
            kp, (const T*)x, (const T*)Im, (T*)y, theta, pairing, sign, dtheta, (uint32_t)rows, im_unmixed);
    else
        givens_kernel<T, VC, LPR, uint64_t><<<blocks, kThreads, smem, s>>>(
            kp, (const T*)x, (const T*)Im, (T*)y, theta, pairing, sign, dtheta, (uint64_t)rows, im_unmixed);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(const KernelProblem& kp, bool bf16, const void* x0, const void* x1, void* y0, void* y1,
                        const int* pos0, const RopeTable& tab, bool transpose, int num_sms, cudaStream_t s) {
    const float sign = transpose ? -1.f : 1.f;
    // Eight bf16 / four fp32 columns per thread (16-byte accesses) where d/2 allows it,
    // else four or two.
    const bool four = (kp.d / 2) % 4 == 0;
    if (bf16) {
        if ((kp.d / 2) % 8 == 0) return launch_rope_t<__nv_bfloat16, 8>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s);
        return four ? launch_rope_t<__nv_bfloat16, 4>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s)
                    : launch_rope_t<__nv_bfloat16, 2>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s);
    }
    return four ? launch_rope_t<float, 4>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s)
                : launch_rope_t<float, 2>(kp, x0, x1, y0, y1, pos0, tab, sign, num_sms, s);
}

cudaError_t launch_givens(const KernelProblem& kp, bool bf16, const void* x, const void* Im, void* y,
                          const float* theta, int pairing, bool transpose, float* dtheta, int num_sms,
                          cudaStream_t s, bool im_unmixed) {
    const float sign = transpose ? -1.f : 1.f;
    // Widest access the row pitch allows (16 bytes when d * elem is a multiple of 16),
    // and the fewest lanes (a power of two) that cover a row with it.
    const int eb = bf16 ? 2 : 4;
    const int vc = ((kp.d * eb) % 16 == 0) ? 16 / eb : (((kp.d * eb) % 8 == 0) ? 8 / eb : 4 / eb);
    int lpr = 1;
    while (lpr * vc < kp.d) lpr <<= 1;
#define RELATION_GIVENS(T_, VC_, LPR_) \
    return launch_givens_t<T_, VC_, LPR_>(kp, x, Im, y, theta, pairing, sign, dtheta, num_sms, s, im_unmixed)
    if (bf16) {
        if (vc == 8) {
            if (lpr <= 8) RELATION_GIVENS(__nv_bfloat16, 8, 8);
            RELATION_GIVENS(__nv_bfloat16, 8, 16);
        }
        if (vc == 4) {
            if (lpr <= 16) RELATION_GIVENS(__nv_bfloat16, 4, 16);
            RELATION_GIVENS(__nv_bfloat16, 4, 32);
        }
        RELATION_GIVENS(__nv_bfloat16, 2, 32);
    }
    if (vc == 4) {
        if (lpr <= 16) RELATION_GIVENS(float, 4, 16);
        RELATION_GIVENS(float, 4, 32);
    }
    RELATION_GIVENS(float, 2, 32);
#undef RELATION_GIVENS
}

cudaError_t launch_rope_convert(const KernelProblem& kp, const float* dq_acc, void* dX1, const int32_t* pos0,
                                const RopeTable& tab, int num_sms, cudaStream_t s) {
    if (kp.d != 64) return cudaErrorInvalidValue;
    const int64_t units = kp.BH * (int64_t)kp.T * 8;
    rope_convert_kernel<<<(unsigned)blocks_for(units, num_sms), kThreads, 0, s>>>(
        kp, dq_acc, static_cast<__nv_bfloat16*>(dX1), pos0, tab, units);
    return cudaGetLastError();
}

}  // namespace relation

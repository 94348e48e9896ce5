// CUDA-core kernels of the Relation library:
//  - the float32 forward and backward (exact expf/logf arithmetic, fp32
//    accumulation), used for RELATION_F32 problems;
//  - the backward preparation (D_i, dlambda, dP1 accumulator reset) and the
//    dP1 accumulator conversion, shared by both dtypes.
//
// Operator: "Ask Self, Ask Others: Relation Is All You Need", Sec. 3.1
// eq.(1)-(3) (forward, with the -lambda log i count correction of eq.(2)); the
// backward is the chain rule of those equations.  The forward uses the
// online-softmax scan of Sec. 5.1 eq.(12) over every visible entry (Self
// included), so U, R and F are never stored.
//
// Layout: four threads share one row; thread `part` owns columns
// part, part+4, part+8, ... of d, so the four threads of a quad read four
// distinct shared-memory banks when they all read one K/V row.
#include "common.cuh"
#include "kernels.h"

namespace relation {
namespace {

constexpr int kRows = 32;     // rows (queries or keys) per block
constexpr int kTile = 32;     // rows of the streamed operand per shared-memory tile
constexpr int kThreads = 128; // kRows * 4

__device__ __forceinline__ float sigmoid_exact(float x) {
    if (x >= 0.f) return 1.f / (1.f + expf(-x));
    float e = expf(x);
    return e / (1.f + e);
}

__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// Count-correction term lambda * log(c_i) for zero-based row i.
__device__ __forceinline__ float count_correction(const KernelProblem& kp, int i) {
    const int c = kp.causal ? (i + 1) : kp.T;
    return kp.lambda * logf((float)c);
}

// Rows row0 .. row0+kTile-1 of head bh of an operand tensor (any layout) as fp32.
template <typename Tin, int D>
__device__ __forceinline__ void load_tile(float (*dst)[D], const Tin* src, const KernelProblem& kp, int64_t bh,
                                          int row0) {
    for (int e = threadIdx.x; e < kTile * D; e += kThreads) {
        const int rr = e / D, cc = e % D;
        const int row = row0 + rr;
        dst[rr][cc] = (row < kp.T) ? load_as_float(src + row_offset(kp, bh, row) + cc) : 0.f;
    }
}

// ------------------------------------------------------------------ forward
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(KernelProblem kp, const Tin* __restrict__ P1,
                                                            const Tin* __restrict__ P2,
                                                            const Tin* __restrict__ V, Tin* __restrict__ Y,
                                                            float* __restrict__ L) {
    constexpr int S = D / 4;
    __shared__ float sK[kTile][D];
    __shared__ float sV[kTile][D];
    const int64_t bh = blockIdx.y;
    const int T = kp.T;
    const int q0 = blockIdx.x * kRows;
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int i = q0 + r;
    const bool valid = i < T;
    const size_t off_i = row_offset(kp, bh, valid ? i : 0);

    float q[S], acc[S];
#pragma unroll
    for (int k = 0; k < S; ++k) {
        q[k] = valid ? load_as_float(P1 + off_i + part + 4 * k) : 0.f;
        acc[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float corr = count_correction(kp, i);
    const int kv_end = kp.causal ? min(T, q0 + kRows) : T;

    for (int j0 = 0; j0 < kv_end; j0 += kTile) {
        __syncthreads();
        load_tile<Tin, D>(sK, P2, kp, bh, j0);
        load_tile<Tin, D>(sV, V, kp, bh, j0);
        __syncthreads();
        for (int jj = 0; jj < kTile; ++jj) {
            const int j = j0 + jj;
            if (j >= kv_end) break;
            float dot = 0.f;
#pragma unroll
            for (int k = 0; k < S; ++k) dot = fmaf(q[k], sK[jj][part + 4 * k], dot);
            dot = quad_sum(dot);
            const bool visible = valid && (!kp.causal || j <= i);
            if (visible) {
                const float u = dot * kp.inv_sqrt_d;
                const float x = (j == i) ? sigmoid_exact(u / kp.tau_S) : u * sigmoid_exact(u) - corr;
                const float m_new = fmaxf(m, x);
                const float sc = expf(m - m_new);  // 0 on the first visible entry
                const float p = expf(x - m_new);
                l = l * sc + p;
#pragma unroll
                for (int k = 0; k < S; ++k) acc[k] = fmaf(p, sV[jj][part + 4 * k], acc[k] * sc);
                m = m_new;
            }
        }
    }
    if (valid) {
        const float inv_l = 1.f / l;
#pragma unroll
        for (int k = 0; k < S; ++k) store_from_float(Y + off_i + part + 4 * k, acc[k] * inv_l);
        if (L != nullptr && part == 0) L[bh * T + i] = m + logf(l);
    }
}

// Where the preparation stage puts D_t of row (bh, t): D [BH, T] for the
// CUDA-core backward, or the tensor-core kernels' per-query constants (layout
// in kernels.h), including the zero rows that pad each head to a multiple of 128.
struct PrepOut {
    float* D;       // used when qc == nullptr
    float* qc;      // per-query constants
    const float* L; // log-normaliser of the forward [BH, T]
};
__device__ __forceinline__ void put_row_result(const KernelProblem& kp, const PrepOut& po, int64_t row, float D) {
    if (po.qc == nullptr) {
        po.D[row] = D;
        return;
    }
    constexpr float kLog2e = 1.4426950408889634f;
    const int64_t bh = row / kp.T;
    const int t = (int)(row - bh * kp.T);
    const int count = kp.causal ? (t + 1) : kp.T;
    const int64_t tp = qconst_rows(kp.T);
    float* base = po.qc + (size_t)bh * (size_t)tp * 2;
    base[(t >> 1) * 4 + (t & 1)] = -(po.L[row] + kp.lambda * __logf((float)count)) * kLog2e;
    base[(t >> 1) * 4 + 2 + (t & 1)] = -D * (0.5f * kp.inv_sqrt_d);
    for (int64_t u = (int64_t)kp.T + t; u < tp; u += kp.T) {
        base[(u >> 1) * 4 + (u & 1)] = 0.f;
        base[(u >> 1) * 4 + 2 + (u & 1)] = 0.f;
    }
}

// ------------------------------------------------- backward: D_i and dlambda
// One warp per row.  D_i = dY_i . Y_i.  dlambda = sum_i log(c_i) dR_ii, which
// equals -sum_i log(c_i) sum_{j!=i} dR_ij because every row of dR sums to 0.
// Also clears the row of the float32 dP1 accumulator when one is given.
template <typename Tin>
__global__ void __launch_bounds__(256) bwd_prepare_kernel(KernelProblem kp, const Tin* __restrict__ P1,
                                                          const Tin* __restrict__ P2,
                                                          const Tin* __restrict__ V,
                                                          const Tin* __restrict__ Yf,
                                                          const float* __restrict__ L,
                                                          const Tin* __restrict__ dY,
                                                          PrepOut po, float* __restrict__ dq_acc,
                                                          int dq_w, float* __restrict__ dlambda) {
    __shared__ float s_part[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + warp;  // flattened (bh, i)
    const int64_t rows = kp.BH * kp.T;
    const int d = kp.d;
    float contrib = 0.f;
    if (row < rows) {
        const int i = (int)(row % kp.T);
        const size_t off = row_offset(kp, row / kp.T, i);
        float dy_y = 0.f, p1p2 = 0.f, dy_v = 0.f;
        for (int c = lane; c < d; c += 32) {
            const float g = load_as_float(dY + off + c);
            dy_y = fmaf(g, load_as_float(Yf + off + c), dy_y);
            if (dlambda != nullptr) {  // the Self entry's terms, needed only for dlambda
                dy_v = fmaf(g, load_as_float(V + off + c), dy_v);
                p1p2 = fmaf(load_as_float(P1 + off + c), load_as_float(P2 + off + c), p1p2);
            }
        }
        if (dq_acc != nullptr)
            for (int c = lane; c < dq_w; c += 32) dq_acc[(size_t)row * dq_w + c] = 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            dy_y += __shfl_xor_sync(0xffffffffu, dy_y, o);
            dy_v += __shfl_xor_sync(0xffffffffu, dy_v, o);
            p1p2 += __shfl_xor_sync(0xffffffffu, p1p2, o);
        }
        if (lane == 0) {
            put_row_result(kp, po, row, dy_y);
            const float u = p1p2 * kp.inv_sqrt_d;
            const float S = sigmoid_exact(u / kp.tau_S);
            const float Fii = expf(S - L[row]);
            const float dRii = Fii * (dy_v - dy_y);
            const int c = kp.causal ? (i + 1) : kp.T;
            contrib = logf((float)c) * dRii;
        }
    }
    if (dlambda == nullptr) return;
    if (lane == 0) s_part[warp] = contrib;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += s_part[w];
        atomicAdd(dlambda, s);
    }
}

// Vectorised D_i = dY_i . Y_i for bf16 rows of width D plus the reset of the
// row's fp32 dP1 accumulator; used when dlambda is summed elsewhere.  D/8
// threads per row, each owning 16 bytes of dY and Y and D/(D/8)*4 bytes of the
// accumulator.
template <int D>
__global__ void __launch_bounds__(256) bwd_prepare_bf16_kernel(KernelProblem kp, int64_t rows,
                                                               const uint4* __restrict__ Yv,
                                                               const uint4* __restrict__ dYv, PrepOut po,
                                                               float4* __restrict__ dq4) {
    constexpr int kTpr = D / 8;  // threads per row
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = t / kTpr;
    const int part = (int)(t % kTpr);
    float acc = 0.f;
    if (row < rows) {
        const uint4 y = Yv[row * kTpr + part], g = dYv[row * kTpr + part];
        const uint32_t ys[4] = {y.x, y.y, y.z, y.w}, gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[k]));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gs[k]));
            acc = fmaf(yf.x, gf.x, acc);
            acc = fmaf(yf.y, gf.y, acc);
        }
        dq4[row * (D / 4) + 2 * part] = make_float4(0.f, 0.f, 0.f, 0.f);
        dq4[row * (D / 4) + 2 * part + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int o = kTpr / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (row < rows && part == 0) put_row_result(kp, po, row, acc);
}

// bf16 rows of width d <= 64 (d % 4 == 0), either layout, dlambda summed
// elsewhere: D_i = dY_i . Y_i, the row's 64-wide fp32 dP1 accumulator zeroed
// and, when pad.dst[0] is set, the row written zero-padded to 64 columns into
// contiguous [BH, T, 64] copies of P1, P2, V, dY (in that order) in the same
// pass.  16 threads per row, thread u owning columns 4u .. 4u+3 (8 bytes); a
// warp holds two rows, so the reduction stays inside each half-warp.
struct PrepPad {
    const uint2* src[3];  // P1, P2, V
    uint2* dst[4];        // P1, P2, V, dY copies; dst[0] == nullptr: no copies
};
__global__ void __launch_bounds__(256) bwd_prepare_narrow_kernel(KernelProblem kp, int64_t rows,
                                                                 const uint2* __restrict__ Y,
                                                                 const uint2* __restrict__ dY, PrepOut po,
                                                                 float4* __restrict__ dq4, PrepPad pad) {
    const int u = threadIdx.x & 15;
    const unsigned half = 0xffffu << (threadIdx.x & 16);
    const int units = kp.d >> 2;
    const bool copies = pad.dst[0] != nullptr;
    const uint2 zero = make_uint2(0u, 0u);
    const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 4);
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4; row < rows; row += step) {
        // Contiguous rows need no division: row r starts at r * d elements.
        const size_t base = (kp.layout == 0 ? (size_t)row * (size_t)kp.d : row_offset(kp, row / kp.T, row % kp.T)) / 4;
        uint2 g = zero;
        float acc = 0.f;
        if (u < units) {
            g = dY[base + u];
            const uint2 y = Y[base + u];
            const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.x));
            const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.y));
            const float2 y0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.x));
            const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.y));
            acc = fmaf(g0.x, y0.x, fmaf(g0.y, y0.y, fmaf(g1.x, y1.x, g1.y * y1.y)));
        }
        const int64_t out = row * 16 + u;
        dq4[out] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (copies) {
            pad.dst[3][out] = g;
#pragma unroll
            for (int k = 0; k < 3; ++k) pad.dst[k][out] = u < units ? pad.src[k][base + u] : zero;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(half, acc, o);
        if (u == 0) put_row_result(kp, po, row, acc);
    }
}

// Relation entry r_ij and its slope dr/du for zero-based (i, j), j visible.
__device__ __forceinline__ void relation_entry(const KernelProblem& kp, int i, int j, float u, float corr,
                                               float* r, float* slope) {
    if (j == i) {
        const float sg = sigmoid_exact(u / kp.tau_S);
        *r = sg;
        *slope = sg * (1.f - sg) / kp.tau_S;
    } else {
        const float sg = sigmoid_exact(u);
        *r = u * sg - corr;
        *slope = sg * (1.f + u * (1.f - sg));
    }
}

// --------------------------------------- backward: key-stationary dP2 and dV
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) bwd_kv_simt_kernel(KernelProblem kp, const Tin* __restrict__ P1,
                                                               const Tin* __restrict__ P2,
                                                               const Tin* __restrict__ V,
                                                               const float* __restrict__ L,
                                                               const float* __restrict__ Dw,
                                                               const Tin* __restrict__ dY, Tin* __restrict__ dP2,
                                                               Tin* __restrict__ dV) {
    constexpr int S = D / 4;
    __shared__ float sQ[kTile][D];
    __shared__ float sG[kTile][D];
    __shared__ float sL[kTile], sD[kTile], sC[kTile];
    const int64_t bh = blockIdx.y;
    const int T = kp.T;
    const int j0 = blockIdx.x * kRows;
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int j = j0 + r;
    const bool valid = j < T;
    const size_t off_j = row_offset(kp, bh, valid ? j : 0);
    float kreg[S], vreg[S], adv[S], adk[S];
#pragma unroll
    for (int k = 0; k < S; ++k) {
        kreg[k] = valid ? load_as_float(P2 + off_j + part + 4 * k) : 0.f;
        vreg[k] = valid ? load_as_float(V + off_j + part + 4 * k) : 0.f;
        adv[k] = adk[k] = 0.f;
    }
    const int i_begin = kp.causal ? j0 : 0;
    for (int i0 = i_begin; i0 < T; i0 += kTile) {
        __syncthreads();
        load_tile<Tin, D>(sQ, P1, kp, bh, i0);
        load_tile<Tin, D>(sG, dY, kp, bh, i0);
        if (threadIdx.x < kTile) {
            const int i = i0 + threadIdx.x;
            sL[threadIdx.x] = i < T ? L[bh * T + i] : 0.f;
            sD[threadIdx.x] = i < T ? Dw[bh * T + i] : 0.f;
            sC[threadIdx.x] = count_correction(kp, i);
        }
        __syncthreads();
        for (int ii = 0; ii < kTile; ++ii) {
            const int i = i0 + ii;
            if (i >= T) break;
            float du = 0.f, df = 0.f;
#pragma unroll
            for (int k = 0; k < S; ++k) {
                du = fmaf(kreg[k], sQ[ii][part + 4 * k], du);
                df = fmaf(vreg[k], sG[ii][part + 4 * k], df);
            }
            du = quad_sum(du);
            df = quad_sum(df);
            if (valid && (!kp.causal || j <= i)) {
                const float u = du * kp.inv_sqrt_d;
                float rr, slope;
                relation_entry(kp, i, j, u, sC[ii], &rr, &slope);
                const float F = expf(rr - sL[ii]);
                const float dU = F * (df - sD[ii]) * slope * kp.inv_sqrt_d;
#pragma unroll
                for (int k = 0; k < S; ++k) {
                    adv[k] = fmaf(F, sG[ii][part + 4 * k], adv[k]);
                    adk[k] = fmaf(dU, sQ[ii][part + 4 * k], adk[k]);
                }
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int k = 0; k < S; ++k) {
            store_from_float(dP2 + off_j + part + 4 * k, adk[k]);
            store_from_float(dV + off_j + part + 4 * k, adv[k]);
        }
    }
}

// ----------------------------------------------- backward: query-stationary dP1
template <typename Tin, int D>
__global__ void __launch_bounds__(kThreads) bwd_q_simt_kernel(KernelProblem kp, const Tin* __restrict__ P1,
                                                              const Tin* __restrict__ P2,
                                                              const Tin* __restrict__ V,
                                                              const float* __restrict__ L,
                                                              const float* __restrict__ Dw,
                                                              const Tin* __restrict__ dY, Tin* __restrict__ dP1) {
    constexpr int S = D / 4;
    __shared__ float sK[kTile][D];
    __shared__ float sV[kTile][D];
    const int64_t bh = blockIdx.y;
    const int T = kp.T;
    const int q0 = blockIdx.x * kRows;
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    const int i = q0 + r;
    const bool valid = i < T;
    const size_t off_i = row_offset(kp, bh, valid ? i : 0);
    float qreg[S], greg[S], acc[S];
#pragma unroll
    for (int k = 0; k < S; ++k) {
        qreg[k] = valid ? load_as_float(P1 + off_i + part + 4 * k) : 0.f;
        greg[k] = valid ? load_as_float(dY + off_i + part + 4 * k) : 0.f;
        acc[k] = 0.f;
    }
    const float Li = valid ? L[bh * T + i] : 0.f;
    const float Di = valid ? Dw[bh * T + i] : 0.f;
    const float corr = count_correction(kp, i);
    const int kv_end = kp.causal ? min(T, q0 + kRows) : T;
    for (int j0 = 0; j0 < kv_end; j0 += kTile) {
        __syncthreads();
        load_tile<Tin, D>(sK, P2, kp, bh, j0);
        load_tile<Tin, D>(sV, V, kp, bh, j0);
        __syncthreads();
        for (int jj = 0; jj < kTile; ++jj) {
            const int j = j0 + jj;
            if (j >= kv_end) break;
            float du = 0.f, df = 0.f;
#pragma unroll
            for (int k = 0; k < S; ++k) {
                du = fmaf(qreg[k], sK[jj][part + 4 * k], du);
                df = fmaf(greg[k], sV[jj][part + 4 * k], df);
            }
            du = quad_sum(du);
            df = quad_sum(df);
            if (valid && (!kp.causal || j <= i)) {
                const float u = du * kp.inv_sqrt_d;
                float rr, slope;
                relation_entry(kp, i, j, u, corr, &rr, &slope);
                const float F = expf(rr - Li);
                const float dU = F * (df - Di) * slope * kp.inv_sqrt_d;
#pragma unroll
                for (int k = 0; k < S; ++k) acc[k] = fmaf(dU, sK[jj][part + 4 * k], acc[k]);
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int k = 0; k < S; ++k) store_from_float(dP1 + off_i + part + 4 * k, acc[k]);
    }
}

// ------------------------------------------- dP1 accumulator (fp32) -> dtype
template <typename Tout>
__global__ void __launch_bounds__(256) convert_kernel(const float* __restrict__ src, Tout* __restrict__ dst,
                                                      int64_t n4) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n4; k += stride) {
        const float4 v = reinterpret_cast<const float4*>(src)[k];
        store_from_float(dst + 4 * k + 0, v.x);
        store_from_float(dst + 4 * k + 1, v.y);
        store_from_float(dst + 4 * k + 2, v.z);
        store_from_float(dst + 4 * k + 3, v.w);
    }
}

// Two floats as a bf16 pair (round to nearest even; the first in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// The same for bf16 output, 8 values per thread and step (two 16-byte loads, one
// 16-byte store), four steps' loads issued before their stores.
__global__ void __launch_bounds__(256) convert8_bf16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                                            int64_t n8) {
    constexpr int kUnroll = 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k0 < n8; k0 += kUnroll * stride) {
        float4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t k = k0 + u * stride;
            if (k < n8) {
                a[u] = src[2 * k];
                b[u] = src[2 * k + 1];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t k = k0 + u * stride;
            if (k < n8)
                dst[k] = make_uint4(pack_bf16(a[u].x, a[u].y), pack_bf16(a[u].z, a[u].w), pack_bf16(b[u].x, b[u].y),
                                    pack_bf16(b[u].z, b[u].w));
        }
    }
}

// dP1 accumulator [BH, T, dq_w] fp32 -> dP1 in the problem's layout and width;
// one thread per 4 columns of a row.
template <typename Tout>
__global__ void __launch_bounds__(256) convert_rows_kernel(KernelProblem kp, const float* __restrict__ src, int dq_w,
                                                           Tout* __restrict__ dst, int64_t n4) {
    const int q4 = kp.d / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n4; k += stride) {
        const int64_t row = k / q4;
        const int c = (int)(k - row * q4) * 4;
        const float4 v = *reinterpret_cast<const float4*>(src + (size_t)row * dq_w + c);
        Tout* o = dst + row_offset(kp, row / kp.T, row % kp.T) + c;
        store_from_float(o + 0, v.x);
        store_from_float(o + 1, v.y);
        store_from_float(o + 2, v.z);
        store_from_float(o + 3, v.w);
    }
}

// Operand rows of width d (any layout) -> zero-padded contiguous [BH, T, 64]
// bf16 copies (operand blockIdx.y of the n), one thread per 16-byte unit of the
// copy (two 8-byte units of the source row; d is a multiple of 4).
struct PadArgs {
    const uint2* src[4];
    uint4* dst[4];
};
__global__ void __launch_bounds__(256) pad_operands_kernel(KernelProblem kp, PadArgs a, int64_t units) {
    const uint2* __restrict__ src = a.src[blockIdx.y];
    uint4* __restrict__ dst = a.dst[blockIdx.y];
    const int src_units = kp.d / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < units; k += stride) {
        const int64_t row = k >> 3;
        const int u = 2 * (int)(k & 7);
        // Contiguous rows need no division: row r starts at r * d elements.
        const uint2* s = src + (kp.layout == 0 ? (size_t)row * (size_t)src_units
                                               : row_offset(kp, row / kp.T, row % kp.T) / 4);
        uint2 lo = make_uint2(0u, 0u), hi = make_uint2(0u, 0u);
        if (u < src_units) lo = s[u];
        if (u + 1 < src_units) hi = s[u + 1];
        dst[k] = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
}

template <typename Tin>
cudaError_t launch_fwd_simt_t(const KernelProblem& kp, const void* P1, const void* P2, const void* V, void* Y,
                              float* L, cudaStream_t s) {
    dim3 grid((kp.T + kRows - 1) / kRows, (unsigned)kp.BH);
#define RELATION_FWD_SIMT(DD)                                                                               \
    fwd_simt_kernel<Tin, DD><<<grid, kThreads, 0, s>>>(kp, (const Tin*)P1, (const Tin*)P2, (const Tin*)V, \
                                                       (Tin*)Y, L)
    switch (kp.d) {
        case 48: RELATION_FWD_SIMT(48); break;
        case 60: RELATION_FWD_SIMT(60); break;
        case 64: RELATION_FWD_SIMT(64); break;
        case 80: RELATION_FWD_SIMT(80); break;
        case 128: RELATION_FWD_SIMT(128); break;
        default: return cudaErrorInvalidValue;
    }
#undef RELATION_FWD_SIMT
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_bwd_simt_t(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                              const float* L, const float* Dw, const void* dY, void* dP1, void* dP2, void* dV,
                              cudaStream_t s) {
    dim3 grid((kp.T + kRows - 1) / kRows, (unsigned)kp.BH);
#define RELATION_BWD_SIMT(DD)                                                                                     \
    bwd_kv_simt_kernel<Tin, DD><<<grid, kThreads, 0, s>>>(kp, (const Tin*)P1, (const Tin*)P2, (const Tin*)V, L, Dw, \
                                                          (const Tin*)dY, (Tin*)dP2, (Tin*)dV);                    \
    bwd_q_simt_kernel<Tin, DD><<<grid, kThreads, 0, s>>>(kp, (const Tin*)P1, (const Tin*)P2, (const Tin*)V, L, Dw,  \
                                                         (const Tin*)dY, (Tin*)dP1)
    switch (kp.d) {
        case 48: RELATION_BWD_SIMT(48); break;
        case 60: RELATION_BWD_SIMT(60); break;
        case 64: RELATION_BWD_SIMT(64); break;
        case 80: RELATION_BWD_SIMT(80); break;
        case 128: RELATION_BWD_SIMT(128); break;
        default: return cudaErrorInvalidValue;
    }
#undef RELATION_BWD_SIMT
    return cudaGetLastError();
}

}  // namespace

bool simt_grid_fits(const KernelProblem& kp) {
    // Row blocks in gridDim.x, heads in gridDim.y (at most 65535).
    return kp.BH >= 1 && kp.BH <= 65535 && ((int64_t)kp.T + kRows - 1) / kRows <= 2147483647LL;
}

cudaError_t launch_fwd_simt(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                            void* Y, float* L, cudaStream_t s) {
    return bf16 ? launch_fwd_simt_t<__nv_bfloat16>(kp, P1, P2, V, Y, L, s)
                : launch_fwd_simt_t<float>(kp, P1, P2, V, Y, L, s);
}

cudaError_t launch_bwd_simt(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                            const float* L, const float* Dw, const void* dY, void* dP1, void* dP2, void* dV,
                            cudaStream_t s) {
    return bf16 ? launch_bwd_simt_t<__nv_bfloat16>(kp, P1, P2, V, L, Dw, dY, dP1, dP2, dV, s)
                : launch_bwd_simt_t<float>(kp, P1, P2, V, L, Dw, dY, dP1, dP2, dV, s);
}

cudaError_t launch_bwd_prepare(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                               const void* Y, const float* L, const void* dY, float* Dw, float* dq_acc, int dq_w,
                               float* dlambda, cudaStream_t s, void* const* pad_dst, int num_sms, float* qconst) {
    const int64_t rows = kp.BH * kp.T;
    const PrepOut po{Dw, qconst, L};
    // Narrow bf16 rows (and the padded copies, when asked for) in one pass.
    const bool narrow = bf16 && dlambda == nullptr && dq_acc != nullptr && dq_w == 64 && kp.d <= 64 &&
                        (kp.d & 3) == 0 && !(kp.layout == 0 && kp.d == 64);
    if (pad_dst != nullptr && !narrow) return cudaErrorInvalidValue;
    if (narrow) {
        PrepPad pad{};
        if (pad_dst != nullptr) {
            pad.src[0] = static_cast<const uint2*>(P1);
            pad.src[1] = static_cast<const uint2*>(P2);
            pad.src[2] = static_cast<const uint2*>(V);
            for (int k = 0; k < 4; ++k) pad.dst[k] = static_cast<uint2*>(pad_dst[k]);
        }
        int64_t blocks = (rows + 15) / 16;
        const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 1) * 16;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        bwd_prepare_narrow_kernel<<<(unsigned)blocks, 256, 0, s>>>(kp, rows, (const uint2*)Y, (const uint2*)dY, po,
                                                                     (float4*)dq_acc, pad);
        return cudaGetLastError();
    }
    // Vector path: contiguous [B, H, T, d] rows whose width is the accumulator's.
    if (bf16 && dlambda == nullptr && dq_acc != nullptr && kp.layout == 0 && kp.d == dq_w &&
        (kp.d == 64 || kp.d == 128)) {
        const int64_t threads = rows * (kp.d / 8);
        const unsigned blocks = (unsigned)((threads + 255) / 256);
        if (kp.d == 64)
            bwd_prepare_bf16_kernel<64><<<blocks, 256, 0, s>>>(kp, rows, (const uint4*)Y, (const uint4*)dY, po,
                                                               (float4*)dq_acc);
        else
            bwd_prepare_bf16_kernel<128><<<blocks, 256, 0, s>>>(kp, rows, (const uint4*)Y, (const uint4*)dY, po,
                                                                (float4*)dq_acc);
        return cudaGetLastError();
    }
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (bf16)
        bwd_prepare_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            kp, (const __nv_bfloat16*)P1, (const __nv_bfloat16*)P2, (const __nv_bfloat16*)V,
            (const __nv_bfloat16*)Y, L, (const __nv_bfloat16*)dY, po, dq_acc, dq_w, dlambda);
    else
        bwd_prepare_kernel<float><<<blocks, 256, 0, s>>>(kp, (const float*)P1, (const float*)P2, (const float*)V,
                                                         (const float*)Y, L, (const float*)dY, po, dq_acc, dq_w,
                                                         dlambda);
    return cudaGetLastError();
}

cudaError_t launch_pad_operands(const KernelProblem& kp, const void* const* src, void* const* dst, int n,
                                int num_sms, cudaStream_t s) {
    if (n < 1 || n > 4 || kp.d > 64 || (kp.d & 3)) return cudaErrorInvalidValue;
    PadArgs a{};
    for (int k = 0; k < n; ++k) {
        a.src[k] = static_cast<const uint2*>(src[k]);
        a.dst[k] = static_cast<uint4*>(dst[k]);
    }
    const int64_t units = kp.BH * (int64_t)kp.T * 8;
    int64_t blocks = (units + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    pad_operands_kernel<<<dim3((unsigned)blocks, (unsigned)n), 256, 0, s>>>(kp, a, units);
    return cudaGetLastError();
}

// out = x[0] + ... + x[n-1], added in index order by one thread (n is a handful of
// per-slice partial sums).
__global__ void sum_in_order_kernel(const float* __restrict__ x, int n, float* __restrict__ out) {
    float acc = 0.f;
    for (int k = 0; k < n; ++k) acc += x[k];
    *out = acc;
}

cudaError_t launch_sum_in_order(const float* x, int n, float* out, cudaStream_t s) {
    sum_in_order_kernel<<<1, 1, 0, s>>>(x, n, out);
    return cudaGetLastError();
}

cudaError_t launch_convert(const KernelProblem& kp, const float* src, int dq_w, void* dst, bool bf16, int num_sms,
                           cudaStream_t s) {
    const int64_t n4 = kp.BH * (int64_t)kp.T * (kp.d / 4);  // d is a multiple of 4
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (kp.layout == 0 && kp.d == dq_w) {  // same layout on both sides: a flat conversion
        if (bf16) {  // d = dq_w is 64 or 128: whole groups of 8
            const int64_t n8 = n4 / 2;
            int64_t b8 = (n8 + 1023) / 1024;
            const int64_t cap8 = (int64_t)num_sms * 16;
            b8 = b8 > cap8 ? cap8 : (b8 < 1 ? 1 : b8);
            convert8_bf16_kernel<<<(unsigned)b8, 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                                              reinterpret_cast<uint4*>(dst), n8);
        } else
            convert_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(src, (float*)dst, n4);
    } else if (bf16) {
        convert_rows_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(kp, src, dq_w, (__nv_bfloat16*)dst, n4);
    } else {
        convert_rows_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(kp, src, dq_w, (float*)dst, n4);
    }
    return cudaGetLastError();
}

}  // namespace relation

// Elementwise stage shared by the tensor-core backward kernels ("Ask Self, Ask
// Others: Relation Is All You Need", Sec. 3.1 eq.(1)-(3), differentiated): for
// one key row and 16 query columns of S^T (raw dot products P2_j . P1_i) and
// dP^T (dY_i . V_j), rebuild P = F_ij = exp(R_ij - L_i) and form
// dS^T = dU^T / sqrt(d) with dU = dR * R'(U), dR = P (dP - D_i).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace relation {
namespace bwd_elem {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// Per-thread constants of the elementwise stage.
struct ElemConst {
    float2 c_nh, c_hl, k2, one, mone;
    float c_diag, half_inv_tau, diag_off, log_count;
    bool row_valid, causal;
};

// Elementwise arithmetic for 16 columns (8 pairs) of one key row: P (to pp,
// packed bf16) and dS^T / sqrt(d) (to dd, packed bf16).  kMasked selects the
// variant with the diagonal Self entry and masking; the plain variant has no
// branches so that the element pairs interleave.  Returns this block's
// contribution log(c_i) * dR_ii * k_scale to dlambda.
template <bool kMasked>
__device__ __forceinline__ float elementwise16(const uint32_t* sv, const uint32_t* gv, const float4* qc, int col0,
                                               int r, const ElemConst& ec, bool diag_tile, int qlimit,
                                               uint32_t (&pp)[8], uint32_t (&dd)[8]) {
    float dlam = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float2 a = make_float2(as_f(sv[2 * e]), as_f(sv[2 * e + 1]));
        const float2 g = make_float2(as_f(gv[2 * e]), as_f(gv[2 * e + 1]));
        // One 16-byte shared-memory load per column pair, the same address in every
        // lane (a broadcast); the shared state space is explicit so the load does not
        // go through the generic path.
        float4 c4;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(c4.x), "=f"(c4.y), "=f"(c4.z), "=f"(c4.w)
                     : "r"((uint32_t)__cvta_generic_to_shared(qc + e)));
        const float2 nlt2 = make_float2(c4.x, c4.y), ndk2 = make_float2(c4.z, c4.w);
        const float2 nh = ptx::mul2(a, ec.c_nh);
        const float2 nt = make_float2(ptx::tanh_approx(nh.x), ptx::tanh_approx(nh.y));
        const float2 tp1 = ptx::fma2(nt, ec.mone, ec.one);
        const float2 hl = ptx::mul2(a, ec.c_hl);
        const float2 x = ptx::fma2(hl, tp1, nlt2);
        float2 p = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
        const float2 nq = ptx::fma2(nt, nt, ec.mone);
        float2 s2 = ptx::fma2(nh, nq, tp1);
        const float2 gk = ptx::fma2(g, ec.k2, ndk2);
        if (kMasked) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int col = col0 + 2 * e + u;  // column within the query tile
                float& pu = u ? p.y : p.x;
                float& su = u ? s2.y : s2.x;
                if (diag_tile && col == r && ec.row_valid) {
                    const float aa = u ? a.y : a.x;
                    const float td = ptx::tanh_approx(aa * ec.c_diag);
                    pu = ptx::ex2_approx(fmaf(0.5f * kLog2e, td, ec.diag_off + (u ? nlt2.y : nlt2.x)));
                    su = fmaf(-td, td, 1.f) * ec.half_inv_tau;  // 2 S(1-S)/tau_S
                    dlam += ec.log_count * pu * (u ? gk.y : gk.x);
                }
                if (col >= qlimit || !ec.row_valid || (ec.causal && diag_tile && col < r)) pu = 0.f;
            }
        }
        const float2 dr = ptx::mul2(p, gk);
        const float2 ds = ptx::mul2(dr, s2);
        pp[e] = ptx::pack_bf16x2(p.x, p.y);
        dd[e] = ptx::pack_bf16x2(ds.x, ds.y);
    }
    return dlam;
}

}  // namespace bwd_elem
}  // namespace relation

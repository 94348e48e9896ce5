// Input prologue applied to operand tiles in shared memory, for the tensor-core
// kernels that fuse it into their loads ("Ask Self, Ask Others: Relation Is All
// You Need", Sec. 3.1 below eq.(1) and Appendix B.3: RoPE on the relation
// coordinates, coordinate c < d/2 turning with c + d/2; Sec. 3.2 eq.(4) and
// Appendix A.2.2-A.2.3: Givens mixing of a head pair's information states).
// Tiles are 128 rows x 64 bf16 columns with 128-byte rows, the 16-byte chunk k of
// row r stored at chunk k ^ (r % 8) (the TMA 128-byte swizzle of a 1 KB-aligned tile).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace relation {

struct ProArgs {
    RopeTable tab;         // RoPE frequencies (tab.enabled == 0: no rotation)
    const float* theta;    // Givens angles [H/2]
    const int32_t* pos0;   // first position of each batch, or NULL
    int pairing;
};

// RoPE angles of one thread's four coordinates 4 (tr % 8) .. +3 for a stream of
// consecutive tiles: cos / sin at the thread's current row and the turn through
// the angle of kN / 8 rows (one row step), from rope_sincos once.  A tile takes
// 128 / (kN / 8) steps, which bring the angles to the same row of the next tile;
// the turns are exact rotations in fp32 (about 1e-7 relative error each), far
// below the bf16 rounding of the rotated values over any stream of tiles.
template <int kN>
struct RopeAngles {
    float cs[4], sn[4], cd[4], sd[4];
    // Angles of row pos_first + tr / 8; sign = -1: the transposed rotation.
    __device__ __forceinline__ void init(int tr, float pos_first, const RopeTable& tab, float sign) {
        const int q4 = tr & 7, g = tr >> 3;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int c = 4 * q4 + v;
            rope_sincos(pos_first + (float)g, tab.hi[c], tab.lo[c], &sn[v], &cs[v]);
            rope_sincos((float)(kN / 8), tab.hi[c], tab.lo[c], &sd[v], &cd[v]);
            sn[v] *= sign;
            sd[v] *= sign;
        }
    }
};

// Turns (c, s) through the angle with cosine cd and sine sd.
__device__ __forceinline__ void rope_turn(float& c, float& s, float cd, float sd) {
    const float c2 = fmaf(c, cd, -s * sd);
    s = fmaf(s, cd, c * sd);
    c = c2;
}

// RoPE of a tile in place by kN threads (tr = 0 .. kN-1): coordinate c < 32 turns
// with c + 32 by the angle of its row.  Thread tr takes the four coordinates
// 4 (tr % 8) .. +3 of rows tr / 8 + (kN / 8) m, starting from the angles in `a`
// (its row tr / 8 of this tile); on return `a` holds the angles of the same row
// of the next tile.
template <int kN>
__device__ __forceinline__ void rope_tile64(uint8_t* tile, int tr, RopeAngles<kN>& a) {
    static_assert(kN % 8 == 0 && 128 % (kN / 8) == 0, "thread count");
    constexpr int kStep = kN / 8, kRows = 128 / kStep;
    const int q4 = tr & 7, g = tr >> 3;
    const int chunk = q4 >> 1, sub = (q4 & 1) * 8;  // byte offset inside the 16-byte chunk
#pragma unroll 4
    for (int m = 0; m < kRows; ++m) {
        const int r = g + kStep * m;
        uint8_t* row = tile + r * 128;
        uint2* pa = reinterpret_cast<uint2*>(row + ((chunk ^ (r & 7)) << 4) + sub);
        uint2* pb = reinterpret_cast<uint2*>(row + (((chunk + 4) ^ (r & 7)) << 4) + sub);
        const uint2 x = *pa, y = *pb;
        const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
        const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
        const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.x));
        const float2 b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y.y));
        // Packed pairs of coordinates: (v0, v1) and (v2, v3).
        const float2 c01 = make_float2(a.cs[0], a.cs[1]), c23 = make_float2(a.cs[2], a.cs[3]);
        const float2 s01 = make_float2(a.sn[0], a.sn[1]), s23 = make_float2(a.sn[2], a.sn[3]);
        const float2 ra0 = ptx::fma2(c01, a0, ptx::mul2(make_float2(-s01.x, -s01.y), b0));
        const float2 ra1 = ptx::fma2(c23, a1, ptx::mul2(make_float2(-s23.x, -s23.y), b1));
        const float2 rb0 = ptx::fma2(s01, a0, ptx::mul2(c01, b0));
        const float2 rb1 = ptx::fma2(s23, a1, ptx::mul2(c23, b1));
        *pa = make_uint2(ptx::pack_bf16x2(ra0.x, ra0.y), ptx::pack_bf16x2(ra1.x, ra1.y));
        *pb = make_uint2(ptx::pack_bf16x2(rb0.x, rb0.y), ptx::pack_bf16x2(rb1.x, rb1.y));
#pragma unroll
        for (int v = 0; v < 4; ++v) rope_turn(a.cs[v], a.sn[v], a.cd[v], a.sd[v]);
    }
}

// Givens mixing of a tile in place by kN threads: v <- cs v + sn w, w the pair
// partner's tile in the same layout (the map is elementwise, so 16-byte chunks
// are taken in storage order).
template <int kN>
__device__ __forceinline__ void mix_tile64(uint8_t* v, const uint8_t* w, int tr, float cs, float sn) {
    const float2 c2 = make_float2(cs, cs), s2 = make_float2(sn, sn);
#pragma unroll 4
    for (int m = 0; m < 1024 / kN; ++m) {
        uint4* pv = reinterpret_cast<uint4*>(v) + tr + kN * m;
        const uint4 a = *pv, b = *(reinterpret_cast<const uint4*>(w) + tr + kN * m);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[k]));
            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[k]));
            const float2 r = ptx::fma2(c2, fa, ptx::mul2(s2, fb));
            o[k] = ptx::pack_bf16x2(r.x, r.y);
        }
        *pv = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Givens coefficients of head h: I~_h = cs I_h + sn I_partner.
__device__ __forceinline__ int givens_coeffs(int head, int H, const ProArgs& pro, float* cs, float* sn) {
    int k = 0;
    bool first = true;
    const int partner = givens_partner(head, H, pro.pairing, &k, &first);
    sincosf(pro.theta[k], sn, cs);
    if (first) *sn = -*sn;  // first of the pair: cos I_a - sin I_b
    return partner;
}

}  // namespace relation

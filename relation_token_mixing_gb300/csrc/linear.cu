// Linear Relation ("Ask Self, Ask Others: Relation Is All You Need", Sec. 5.2
// eq.(15)-(17), Appendix A.4): per head a d x d relational state C with
// channel-wise retention alpha_t = exp(g_t),
//     C-_t = Diag(alpha_t) C_{t-1},  E_t = S_t (C-_t)^T p^1_t,  Y_t = I~_t + E_t,
//     C_t  = C-_t + S_t p^2_t I~_t^T,  S_t = sigmoid(p1_t . p2_t / (tau_S sqrt d)),
// p^ = p / ||p|| (a zero vector stays zero).
//
// Execution.  One warp owns one (head, segment) pair and walks the segment in
// chunks of 16 tokens, with q = S p^1 and k = S p^2:
//   * the state enters a chunk through two warp-level bf16 tensor-core products
//     (E += (q . F) C and C <- Diag(a) C + (k . B)^T I~, F / B the retention
//     products from the chunk start to t / from t to the chunk end, a = F_15);
//   * pairs inside the chunk use the exact retention product of every pair,
//     prod_{u=j+1..i} alpha_u, formed by running multiplications on the fp32
//     pipes, so no factor ever exceeds 1 and any g <= 0 is exact;
//   * long sequences with few heads are split into segments: a state pass gives
//     each segment's own contribution and retention, a scan over segments gives
//     every segment's entering state, and the output pass runs from it.
// The state lives in registers as mma accumulators holding C^T (rows = value
// channel v, columns = key channel c), so it feeds the next chunk's products
// without passing through shared memory.
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"
#include "tile_copy.cuh"

namespace relation {
namespace lin {

constexpr int kC = 16;          // tokens per chunk
constexpr int kDp = 64;         // head width the kernels work in (narrower heads are zero-padded)
constexpr int kWarpsPerCta = 3;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// (lo, hi) -> packed bf16 pair, lo in the low half.
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed fp32 pairs.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
          "l"(*reinterpret_cast<unsigned long long*>(&c)));
    return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void st_zero16(uint32_t dst) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
}

// Byte offset of (row r, column c) in a 16 x 64 bf16 tile: 128-byte rows whose
// 16-byte chunks are permuted by the row (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * 128 + ((((c >> 3) ^ r) & 7) << 4) + ((c & 7) << 1));
}
constexpr int kArow = 48;  // bytes per row of the 16 x 16 bf16 intra-chunk matrix

// --------------------------------------------------------------- per-warp smem
struct Stage {
    uint8_t p1[kC * 128];  // bf16, swizzled
    uint8_t p2[kC * 128];
    uint8_t v[kC * 128];
    float g[kC * kDp];  // fp32 rows of 64; overwritten in place by alpha = exp(g)
};
struct WarpSmem {
    Stage st[2];
    uint8_t qt[kC * 128];  // q . F        (bf16, swizzled)
    uint8_t kb[kC * 128];  // k . B        (bf16, swizzled)
    float qf[kC * kDp];    // q (fp32)
    float kf[kC * kDp];    // k (fp32)
    uint8_t amat[kC * kArow];
    float2 rs[kC];    // (S / ||p1||, S / ||p2||) per token
    float avec[kDp];  // retention over the whole chunk
};

struct Args {
    const __nv_bfloat16* P1;
    const __nv_bfloat16* P2;
    const __nv_bfloat16* V;
    const float* G;
    __nv_bfloat16* Y;
    float* state_out;  // [BH, d, d] or null
    float* hseg;       // [BH, nseg, 64, 64]: segment contributions, then entering states
    float* aseg;       // [BH, nseg, 64]: retention over each segment
    KernelProblem kp;
    float zscale;  // 1 / (tau_S sqrt d)
    int nseg;
    int seg_len;  // tokens per segment, a multiple of kC
};

// Issues the copies of chunk rows t0 .. t0+15 into a stage (rows >= T and the
// columns >= d of the fp32 tile are zero / unused; the bf16 tiles' columns >= d
// are zeroed once at kernel start and never written).
template <bool kVec16>
__device__ __forceinline__ void load_chunk(Stage& s, const Args& a, int64_t bh, int t0, int lane) {
    const KernelProblem& kp = a.kp;
    const __nv_bfloat16* src[3] = {a.P1, a.P2, a.V};
    uint8_t* dst[3] = {s.p1, s.p2, s.v};
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        const uint32_t base = ptx::smem_u32(dst[m]);
        if (kVec16) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int idx = lane + 32 * k, r = idx >> 3, q = idx & 7, col = 8 * q;
                if (col >= kp.d) continue;
                const uint32_t d = base + r * 128 + (((q ^ r) & 7) << 4);
                if (t0 + r < kp.T)
                    cp_async_16(d, src[m] + row_offset(kp, bh, t0 + r) + col);
                else
                    st_zero16(d);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int idx = lane + 32 * k, r = idx >> 4, q = idx & 15, col = 4 * q;
                if (col >= kp.d) continue;
                const uint32_t d = base + r * 128 + ((((q >> 1) ^ r) & 7) << 4) + ((q & 1) << 3);
                if (t0 + r < kp.T)
                    cp_async_8(d, src[m] + row_offset(kp, bh, t0 + r) + col);
                else
                    st_shared_zero8(d);
            }
        }
    }
    const uint32_t gb = ptx::smem_u32(s.g);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int idx = lane + 32 * k, r = idx >> 4, q = idx & 15, col = 4 * q;
        if (col >= kp.d) continue;
        const uint32_t d = gb + (r * kDp + col) * 4;
        if (t0 + r < kp.T)
            cp_async_16(d, a.G + row_offset(kp, bh, t0 + r) + col);
        else
            st_zero16(d);
    }
    cp_async_commit();
}

// Lanes (token i = lane & 15, channel half lane >> 4): S, then s1 = S/||p1||,
// s2 = S/||p2|| into ws.rs.
__device__ __forceinline__ void row_scalars(WarpSmem& ws, const Stage& s, float zscale, int lane) {
    const int i = lane & 15, h = lane >> 4;
    float n1 = 0.f, n2 = 0.f, dt = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const int col = 32 * h + 8 * c8;
        const uint4 x = *reinterpret_cast<const uint4*>(s.p1 + swz(i, col));
        const uint4 y = *reinterpret_cast<const uint4*>(s.p2 + swz(i, col));
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float a0 = lo_f(xs[w]), a1 = hi_f(xs[w]), b0 = lo_f(ys[w]), b1 = hi_f(ys[w]);
            n1 = fmaf(a0, a0, fmaf(a1, a1, n1));
            n2 = fmaf(b0, b0, fmaf(b1, b1, n2));
            dt = fmaf(a0, b0, fmaf(a1, b1, dt));
        }
    }
    n1 += __shfl_xor_sync(0xffffffffu, n1, 16);
    n2 += __shfl_xor_sync(0xffffffffu, n2, 16);
    dt += __shfl_xor_sync(0xffffffffu, dt, 16);
    const float S = 1.f / (1.f + __expf(-dt * zscale));
    if (h == 0) ws.rs[i] = make_float2(n1 > 0.f ? S * rsqrtf(n1) : 0.f, n2 > 0.f ? S * rsqrtf(n2) : 0.f);
}

// Lane l owns channels c = 2l, 2l+1 of all 16 tokens: alpha (in place of g),
// q, k (fp32), q . F and k . B (bf16 operands) and the chunk retention a = F_15.
// kQ = false skips the query side (state passes).
template <bool kQ>
__device__ __forceinline__ void channel_pass(WarpSmem& ws, Stage& s, int d, int lane) {
    const int c = 2 * lane;
    const bool valid = c < d;
    float2 F = make_float2(1.f, 1.f);
    float2 al[kC], kk[kC];
#pragma unroll
    for (int i = 0; i < kC; ++i) {
        float2* gp = reinterpret_cast<float2*>(s.g + i * kDp + c);
        const float2 g = *gp;
        al[i] = valid ? make_float2(__expf(g.x), __expf(g.y)) : make_float2(1.f, 1.f);
        *gp = al[i];
        F = mul2(F, al[i]);
        const float2 r = ws.rs[i];
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(s.p2 + swz(i, c));
        kk[i] = make_float2(lo_f(w2) * r.y, hi_f(w2) * r.y);
        if (kQ) {
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(s.p1 + swz(i, c));
            const float2 q = make_float2(lo_f(w1) * r.x, hi_f(w1) * r.x);
            *reinterpret_cast<float2*>(ws.qf + i * kDp + c) = q;
            *reinterpret_cast<float2*>(ws.kf + i * kDp + c) = kk[i];
            const float2 qF = mul2(q, F);
            *reinterpret_cast<uint32_t*>(ws.qt + swz(i, c)) = pack2(qF.x, qF.y);
        }
    }
    *reinterpret_cast<float2*>(ws.avec + c) = F;
    float2 Bk = make_float2(1.f, 1.f);
#pragma unroll
    for (int i = kC - 1; i >= 0; --i) {
        const float2 kB = mul2(kk[i], Bk);
        *reinterpret_cast<uint32_t*>(ws.kb + swz(i, c)) = pack2(kB.x, kB.y);
        Bk = mul2(Bk, al[i]);
    }
}

// Intra-chunk matrix A[i][j] = sum_c q_ic k_jc prod_{u=j+1..i} alpha_uc (j < i,
// zero elsewhere) into ws.amat (bf16).  Lane = (key j = lane & 15, channel half
// lane >> 4); W = k_j . prod alpha is carried down the rows.
__device__ __forceinline__ void intra_matrix(WarpSmem& ws, const Stage& s, int lane) {
    const int j = lane & 15, h = lane >> 4, c0 = 32 * h;
    float2 W[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) W[m] = *reinterpret_cast<const float2*>(ws.kf + j * kDp + c0 + 2 * m);
    __nv_bfloat16* A = reinterpret_cast<__nv_bfloat16*>(ws.amat);
    if (h == 0) A[j] = __float2bfloat16_rn(0.f);  // row 0
#pragma unroll 1
    for (int i = 1; i < kC; ++i) {
        const float2* al = reinterpret_cast<const float2*>(s.g + i * kDp + c0);
        const float2* q = reinterpret_cast<const float2*>(ws.qf + i * kDp + c0);
        if (i > j) {
#pragma unroll
            for (int m = 0; m < 16; ++m) W[m] = mul2(W[m], al[m]);
        }
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fma2(W[m], q[m], acc);
        float dot = acc.x + acc.y;
        dot += __shfl_xor_sync(0xffffffffu, dot, 16);
        if (h == 0) A[i * (kArow / 2) + j] = __float2bfloat16_rn(i > j ? dot : 0.f);
    }
}

// ldmatrix lane addresses (see the PTX fragment layouts of m16n8k16).
// A operand 16 x 16 from a row-major [m][k] swizzled tile at column k0.
__device__ __forceinline__ uint32_t addr_a(const uint8_t* tile, int k0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), c = k0 + 8 * (m >> 1);
    return ptx::smem_u32(tile) + swz(r, c);
}
// Operand fragments from a [k][n] (or [k][m]) tile with .trans: two 8-wide
// column blocks n0, n0+8, rows k = 0..15.
__device__ __forceinline__ uint32_t addr_bt(const uint8_t* tile, int n0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), c = n0 + 8 * (m >> 1);
    return ptx::smem_u32(tile) + swz(r, c);
}
// Same for the A operand from a [k][m] tile (.trans): a0..a3 = (m0-7,k0-7),
// (m8-15,k0-7), (m0-7,k8-15), (m8-15,k8-15).
__device__ __forceinline__ uint32_t addr_at(const uint8_t* tile, int m0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m >> 1), c = m0 + 8 * (m & 1);
    return ptx::smem_u32(tile) + swz(r, c);
}

// State C^T as mma accumulators: hT[mt][nt][r] = C^T[v][c], v = 16 mt + g (+8
// for r >= 2), c = 8 nt + 2 t + (r & 1), g = lane / 4, t = lane % 4.
struct State {
    float x[4][8][4];
};

__device__ __forceinline__ void state_zero(State& S) {
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) S.x[mt][nt][r] = 0.f;
}
// C [64][64] (row = key channel c, column = value channel v) <-> registers.
__device__ __forceinline__ void state_load(State& S, const float* C, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int v = 16 * mt + g + 8 * (r >> 1), c = 8 * nt + 2 * t + (r & 1);
                S.x[mt][nt][r] = C[c * kDp + v];
            }
}
__device__ __forceinline__ void state_store(const State& S, float* C, int ld, int d, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int v = 16 * mt + g + 8 * (r >> 1), c = 8 * nt + 2 * t + (r & 1);
                if (v < d && c < d) C[c * ld + v] = S.x[mt][nt][r];
            }
}

// C <- Diag(a) C + (k . B)^T I~ for the chunk in ws / s.
__device__ __forceinline__ void state_update(State& S, const WarpSmem& ws, const Stage& s, int lane) {
    const int t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const float2 a = *reinterpret_cast<const float2*>(ws.avec + 8 * nt + 2 * t);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            S.x[mt][nt][0] *= a.x;
            S.x[mt][nt][1] *= a.y;
            S.x[mt][nt][2] *= a.x;
            S.x[mt][nt][3] *= a.y;
        }
    }
    uint32_t b[8][2];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t r[4];
        ldsm4t(r, addr_bt(ws.kb, 16 * p, lane));
        b[2 * p][0] = r[0];
        b[2 * p][1] = r[1];
        b[2 * p + 1][0] = r[2];
        b[2 * p + 1][1] = r[3];
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
        uint32_t af[4];
        ldsm4t(af, addr_at(s.v, 16 * mt, lane));
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) mma16816(S.x[mt][nt], af, b[nt][0], b[nt][1]);
    }
}

// E = (q . F) C + A I~ as mma accumulators E[nv][r]: token g (+8), v = 8 nv + 2t (+1).
__device__ __forceinline__ void chunk_output(float (&E)[8][4], const State& S, const WarpSmem& ws, const Stage& s,
                                             int lane) {
#pragma unroll
    for (int nv = 0; nv < 8; ++nv)
#pragma unroll
        for (int r = 0; r < 4; ++r) E[nv][r] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t af[4];
        ldsm4(af, addr_a(ws.qt, 16 * ks, lane));
#pragma unroll
        for (int nv = 0; nv < 8; ++nv) {
            const int mt = nv >> 1, rr = (nv & 1) * 2;
            const uint32_t b0 = pack2(S.x[mt][2 * ks][rr], S.x[mt][2 * ks][rr + 1]);
            const uint32_t b1 = pack2(S.x[mt][2 * ks + 1][rr], S.x[mt][2 * ks + 1][rr + 1]);
            mma16816(E[nv], af, b0, b1);
        }
    }
    uint32_t af[4];
    {
        const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), cb = 16 * (m >> 1);
        ldsm4(af, ptx::smem_u32(ws.amat) + r * kArow + cb);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t r[4];
        ldsm4t(r, addr_bt(s.v, 16 * p, lane));
        mma16816(E[2 * p], af, r[0], r[1]);
        mma16816(E[2 * p + 1], af, r[2], r[3]);
    }
}

__device__ __forceinline__ void zero_warp_smem(WarpSmem& ws, int lane) {
    uint4* p = reinterpret_cast<uint4*>(&ws);
    const int n = (int)(sizeof(WarpSmem) / 16);
    for (int k = lane; k < n; k += 32) p[k] = make_uint4(0, 0, 0, 0);
    __syncwarp();
}

// ------------------------------------------------------------------- kernels
// Work item w = bh * nseg + segment; one warp per item.
template <bool kVec16>
__global__ void __launch_bounds__(32 * kWarpsPerCta) linear_state_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem_raw)[warp];
    const int64_t item = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    if (item >= a.kp.BH * a.nseg) return;
    const int64_t bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const int t_begin = seg * a.seg_len, t_end = min(a.kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    zero_warp_smem(ws, lane);

    State S;
    state_zero(S);
    float2 aseg = make_float2(1.f, 1.f);
    load_chunk<kVec16>(ws.st[0], a, bh, t_begin, lane);
    for (int n = 0; n < nchunks; ++n) {
        Stage& s = ws.st[n & 1];
        if (n + 1 < nchunks) {
            load_chunk<kVec16>(ws.st[(n + 1) & 1], a, bh, t_begin + (n + 1) * kC, lane);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        row_scalars(ws, s, a.zscale, lane);
        __syncwarp();
        channel_pass<false>(ws, s, a.kp.d, lane);
        aseg = mul2(aseg, *reinterpret_cast<const float2*>(ws.avec + 2 * lane));
        __syncwarp();
        state_update(S, ws, s, lane);
        __syncwarp();
    }
    float* H = a.hseg + (size_t)item * kDp * kDp;
    state_store(S, H, kDp, kDp, lane);
    *reinterpret_cast<float2*>(a.aseg + (size_t)item * kDp + 2 * lane) = aseg;
}

// One block per head: entering state of every segment (in place of its own
// contribution) and the final state.
__global__ void __launch_bounds__(256) linear_scan_kernel(float* hseg, const float* aseg, int nseg, float* state_out,
                                                          int d) {
    const int64_t bh = blockIdx.x;
    const int c = threadIdx.x >> 2, v0 = (threadIdx.x & 3) * 16;
    float h[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) h[k] = 0.f;
    for (int s = 0; s < nseg; ++s) {
        float4* p = reinterpret_cast<float4*>(hseg + ((size_t)(bh * nseg + s) * kDp + c) * kDp + v0);
        const float al = aseg[(size_t)(bh * nseg + s) * kDp + c];
        float4 dh[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) dh[k] = p[k];
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = make_float4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            h[4 * k] = fmaf(al, h[4 * k], dh[k].x);
            h[4 * k + 1] = fmaf(al, h[4 * k + 1], dh[k].y);
            h[4 * k + 2] = fmaf(al, h[4 * k + 2], dh[k].z);
            h[4 * k + 3] = fmaf(al, h[4 * k + 3], dh[k].w);
        }
    }
    if (state_out != nullptr && c < d) {
        float* o = state_out + ((size_t)bh * d + c) * d;
#pragma unroll
        for (int k = 0; k < 16; ++k)
            if (v0 + k < d) o[v0 + k] = h[k];
    }
}

template <bool kVec16>
__global__ void __launch_bounds__(32 * kWarpsPerCta) linear_fwd_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem_raw)[warp];
    const int64_t item = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    if (item >= a.kp.BH * a.nseg) return;
    const int64_t bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const int t_begin = seg * a.seg_len, t_end = min(a.kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    const KernelProblem& kp = a.kp;
    zero_warp_smem(ws, lane);

    State S;
    if (a.nseg > 1)
        state_load(S, a.hseg + (size_t)item * kDp * kDp, lane);
    else
        state_zero(S);
    const int g = lane >> 2, t = lane & 3;
    load_chunk<kVec16>(ws.st[0], a, bh, t_begin, lane);
    for (int n = 0; n < nchunks; ++n) {
        Stage& s = ws.st[n & 1];
        const int t0 = t_begin + n * kC;
        if (n + 1 < nchunks) {
            load_chunk<kVec16>(ws.st[(n + 1) & 1], a, bh, t0 + kC, lane);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        row_scalars(ws, s, a.zscale, lane);
        __syncwarp();
        channel_pass<true>(ws, s, kp.d, lane);
        __syncwarp();
        intra_matrix(ws, s, lane);
        __syncwarp();
        float E[8][4];
        chunk_output(E, S, ws, s, lane);
        // Y = I~ + E
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = g + 8 * half, tok = t0 + r;
            if (tok < kp.T) {
                __nv_bfloat16* yrow = a.Y + row_offset(kp, bh, tok);
#pragma unroll
                for (int nv = 0; nv < 8; ++nv) {
                    const int v = 8 * nv + 2 * t;
                    if (v < kp.d) {
                        const uint32_t iw = *reinterpret_cast<const uint32_t*>(s.v + swz(r, v));
                        *reinterpret_cast<uint32_t*>(yrow + v) =
                            pack2(lo_f(iw) + E[nv][2 * half], hi_f(iw) + E[nv][2 * half + 1]);
                    }
                }
            }
        }
        state_update(S, ws, s, lane);
        __syncwarp();
    }
    if (a.nseg == 1 && a.state_out != nullptr) state_store(S, a.state_out + (size_t)bh * kp.d * kp.d, kp.d, kp.d, lane);
}

}  // namespace lin

// ------------------------------------------------------------------ launchers
int linear_segments(const KernelProblem& kp, int num_sms, int* seg_len) {
    // Enough warps to fill the GPU about twice over; segments of at least 128 tokens.
    const int64_t want = (int64_t)num_sms * 2 * 2 * lin::kWarpsPerCta;
    int nseg = 1;
    if (kp.BH < want) nseg = (int)((want + kp.BH - 1) / kp.BH);
    const int max_seg = (kp.T + 127) / 128;
    if (nseg > max_seg) nseg = max_seg;
    if (nseg < 1) nseg = 1;
    int len = (kp.T + nseg - 1) / nseg;
    len = (len + lin::kC - 1) / lin::kC * lin::kC;
    nseg = (kp.T + len - 1) / len;
    *seg_len = len;
    return nseg;
}

size_t linear_smem_bytes() { return sizeof(lin::WarpSmem) * lin::kWarpsPerCta; }

cudaError_t launch_linear_fwd(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* G,
                              void* Y, float* state_out, float* ws, int num_sms, cudaStream_t s) {
    lin::Args a;
    a.P1 = static_cast<const __nv_bfloat16*>(P1);
    a.P2 = static_cast<const __nv_bfloat16*>(P2);
    a.V = static_cast<const __nv_bfloat16*>(V);
    a.G = G;
    a.Y = static_cast<__nv_bfloat16*>(Y);
    a.state_out = state_out;
    a.kp = kp;
    a.zscale = kp.inv_sqrt_d / kp.tau_S;
    a.nseg = linear_segments(kp, num_sms, &a.seg_len);
    a.hseg = ws;
    a.aseg = ws + (size_t)kp.BH * a.nseg * lin::kDp * lin::kDp;
    const size_t smem = linear_smem_bytes();
    const bool vec16 = (kp.d % 8) == 0;
    static bool attr_done = false;
    if (!attr_done) {
        cudaFuncSetAttribute(lin::linear_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(lin::linear_fwd_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(lin::linear_state_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(lin::linear_state_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        attr_done = true;
    }
    const int64_t items = kp.BH * a.nseg;
    const unsigned grid = (unsigned)((items + lin::kWarpsPerCta - 1) / lin::kWarpsPerCta);
    const dim3 block(32 * lin::kWarpsPerCta);
    if (a.nseg > 1) {
        if (vec16)
            lin::linear_state_kernel<true><<<grid, block, smem, s>>>(a);
        else
            lin::linear_state_kernel<false><<<grid, block, smem, s>>>(a);
        lin::linear_scan_kernel<<<(unsigned)kp.BH, 256, 0, s>>>(a.hseg, a.aseg, a.nseg, state_out, kp.d);
    }
    if (vec16)
        lin::linear_fwd_kernel<true><<<grid, block, smem, s>>>(a);
    else
        lin::linear_fwd_kernel<false><<<grid, block, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace relation

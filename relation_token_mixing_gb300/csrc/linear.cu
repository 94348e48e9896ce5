// Linear Relation ("Ask Self, Ask Others: Relation Is All You Need", Sec. 5.2
// eq.(15)-(17), Appendix A.4): per head a d x d relational state C with
// channel-wise retention alpha_t = exp(g_t),
//     C-_t = Diag(alpha_t) C_{t-1},  E_t = S_t (C-_t)^T p^1_t,  Y_t = I~_t + E_t,
//     C_t  = C-_t + S_t p^2_t I~_t^T,  S_t = sigmoid(p1_t . p2_t / (tau_S sqrt d)),
// p^ = p / ||p|| (a zero vector stays zero).
//
// Execution.  One CTA of 4 warps owns one (head, segment) pair and walks the
// segment in chunks of 16 tokens, with q = S p^1 and k = S p^2:
//   * the state enters a chunk through warp-level bf16 tensor-core products,
//     E += (q . F) C and C <- Diag(a) C + (k . B)^T I~ (F / B the retention
//     products from the chunk start to t / from t to the chunk end, a = F_15);
//     warp w owns the value channels [16w, 16w+16) of C and of E;
//   * pairs inside the chunk: split at the highest bit in which the two token
//     indices differ, every pair (i, j) has a boundary r with j < r <= i, and
//     prod_{u=j+1..i} alpha_u = prod_{u=r..i} alpha_u * prod_{u=j+1..r-1} alpha_u;
//     the four bit levels are four small tensor-core products whose operands
//     carry these factors, all <= 1, so any g <= 0 is exact;
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

// ldmatrix lane addresses (PTX fragment layouts of m16n8k16).
// A operand 16 x 16 from a row-major [m][k] swizzled tile at column k0.
__device__ __forceinline__ uint32_t addr_a(const uint8_t* tile, int k0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), c = k0 + 8 * (m >> 1);
    return ptx::smem_u32(tile) + swz(r, c);
}
// B fragments of two 8-wide column blocks n0, n0+8 from a [k][n] tile (.trans).
__device__ __forceinline__ uint32_t addr_bt(const uint8_t* tile, int n0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), c = n0 + 8 * (m >> 1);
    return ptx::smem_u32(tile) + swz(r, c);
}
// A operand from a [k][m] tile (.trans): a0..a3 = (m0-7,k0-7), (m8-15,k0-7),
// (m0-7,k8-15), (m8-15,k8-15).
__device__ __forceinline__ uint32_t addr_at(const uint8_t* tile, int m0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m >> 1), c = m0 + 8 * (m & 1);
    return ptx::smem_u32(tile) + swz(r, c);
}


// ------------------------------------------------------------- group smem
// One group of 4 warps (one CTA) owns a (head, segment) pair.  Warp w owns the
// value channels v in [16w, 16w+16) of the state and of the outputs.
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

struct Stage {
    uint8_t p1[kC * 128];  // bf16, swizzled
    uint8_t p2[kC * 128];
    uint8_t v[kC * 128];
    float g[kC * kDp];  // fp32 rows of 64
};
struct GroupSmem {
    static constexpr bool kNorms = false;
    Stage st[2];
    uint8_t qt[kC * 128];     // q . F   (F: retention from the chunk start to t)
    uint8_t kb[kC * 128];     // k . B   (B: retention from t to the chunk end)
    uint8_t ql[4][kC * 128];  // level query operands (rows that are queries at that level)
    uint8_t kl[4][8 * 128];   // level key operands, the 8 key rows of each level compacted
    uint8_t amat[kC * kArow]; // intra-chunk matrix (bf16)
    float2 rs[kC];            // (S / ||p1||, S / ||p2||)
    float avec[kDp];          // retention over the chunk
    float tot[4][kDp];        // retention over each quarter (4 tokens) of the chunk
};

struct Args {
    const __nv_bfloat16* P1;
    const __nv_bfloat16* P2;
    const __nv_bfloat16* V;
    const float* G;         // log-retention g, or the gate's input r (gate_alog != nullptr)
    const float* gate_alog;  // KDA gate [H, d]: A_log, or nullptr (G holds g itself)
    const float* gate_dtb;   // KDA gate [H, d]: dt_bias
    __nv_bfloat16* Y;
    float* state_out;  // [BH, d, d] or null
    float* hseg;       // [BH, nseg, 64, 64]: segment contributions, then entering states
    float* aseg;       // [BH, nseg, 64]: retention over each segment
    KernelProblem kp;
    float zscale;  // 1 / (tau_S sqrt d)
    int nseg;
    int seg_len;  // tokens per segment, a multiple of kC
};

// Element offset of row 0 of head bh and the distance between rows.
struct RowMap {
    size_t base;
    size_t stride;
};
__device__ __forceinline__ RowMap row_map(const KernelProblem& kp, int64_t bh) {
    return RowMap{row_offset(kp, bh, 0), kp.layout == 0 ? (size_t)kp.d : (size_t)kp.H * kp.d};
}

// Warp w issues the copies of tensor w (P1, P2, I~, G) for chunk rows
// t0 .. t0+15 (rows >= T zero; bf16 columns >= d stay zero from the start).
template <bool kVec16>
__device__ __forceinline__ void load_chunk(Stage& s, const Args& a, const RowMap& rm, int t0, int warp, int lane) {
    const KernelProblem& kp = a.kp;
    if (warp < 3) {
        const __nv_bfloat16* src = (warp == 0 ? a.P1 : (warp == 1 ? a.P2 : a.V)) + rm.base + (size_t)t0 * rm.stride;
        const uint32_t base = ptx::smem_u32(warp == 0 ? s.p1 : (warp == 1 ? s.p2 : s.v));
        if (kVec16) {
            const int q = lane & 7, col = 8 * q;
            if (col < kp.d) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (lane >> 3) + 4 * k;
                    const uint32_t dst = base + r * 128 + (((q ^ r) & 7) << 4);
                    if (t0 + r < kp.T)
                        cp_async_16(dst, src + (size_t)r * rm.stride + col);
                    else
                        st_zero16(dst);
                }
            }
        } else {
            const int q = lane & 15, col = 4 * q;
            if (col < kp.d) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = (lane >> 4) + 2 * k;
                    const uint32_t dst = base + r * 128 + ((((q >> 1) ^ r) & 7) << 4) + ((q & 1) << 3);
                    if (t0 + r < kp.T)
                        cp_async_8(dst, src + (size_t)r * rm.stride + col);
                    else
                        st_shared_zero8(dst);
                }
            }
        }
    } else {
        const float* src = a.G + rm.base + (size_t)t0 * rm.stride;
        const int q = lane & 15, col = 4 * q;
        const uint32_t gb = ptx::smem_u32(s.g);
        if (col < kp.d) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = (lane >> 4) + 2 * k;
                const uint32_t dst = gb + (r * kDp + col) * 4;
                if (t0 + r < kp.T)
                    cp_async_16(dst, src + (size_t)r * rm.stride + col);
                else
                    st_zero16(dst);
            }
        }
    }
    cp_async_commit();
}

// Warp w, lanes (token 4w + lane/8, channels 8*(lane%8) .. +7): S, then
// s1 = S/||p1||, s2 = S/||p2|| into gs.rs.
template <class GS, class ST>
__device__ __forceinline__ void row_scalars(GS& gs, const ST& s, float zscale, int warp, int lane) {
    const int i = 4 * warp + (lane >> 3), col = 8 * (lane & 7);
    const uint4 x = *reinterpret_cast<const uint4*>(s.p1 + swz(i, col));
    const uint4 y = *reinterpret_cast<const uint4*>(s.p2 + swz(i, col));
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
    float n1 = 0.f, n2 = 0.f, dt = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float a0 = lo_f(xs[w]), a1 = hi_f(xs[w]), b0 = lo_f(ys[w]), b1 = hi_f(ys[w]);
        n1 = fmaf(a0, a0, fmaf(a1, a1, n1));
        n2 = fmaf(b0, b0, fmaf(b1, b1, n2));
        dt = fmaf(a0, b0, fmaf(a1, b1, dt));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        n1 += __shfl_xor_sync(0xffffffffu, n1, o);
        n2 += __shfl_xor_sync(0xffffffffu, n2, o);
        dt += __shfl_xor_sync(0xffffffffu, dt, o);
    }
    if ((lane & 7) == 0) {
        const float S = 1.f / (1.f + __expf(-dt * zscale));
        const float i1 = n1 > 0.f ? rsqrtf(n1) : 0.f, i2 = n2 > 0.f ? rsqrtf(n2) : 0.f;
        gs.rs[i] = make_float2(S * i1, S * i2);
        if constexpr (GS::kNorms) gs.rn[i] = make_float4(i1, i2, S, 0.f);
    }
}

// Compacted row of key token i among the 8 keys of level bit b.
__device__ __forceinline__ int key_row(int i, int b) { return ((i >> (b + 1)) << b) | (i & ((1 << b) - 1)); }

// Channel pass.  Warp w owns the tokens 4w .. 4w+3 (a quarter of the chunk),
// lane l the channels c = 2l, 2l+1, so every branch below is warp-uniform.
// Phase A: alpha = exp(g) and the products inside the quarter, f (from the
// quarter start to t) and b (from t+1 to the quarter end); the quarter totals go
// to gs.tot.  Phase B (after a barrier) writes q . F, k . B, the level operands
// and the chunk retention.  Every factor is a product of retentions over a run
// of tokens lying between the two tokens of the pairs it serves, so all factors
// are <= 1.  Levels (bit b of the token index): pairs (i, j), j < i, that first
// differ in bit b meet at the boundary r = i with bits < b cleared: query factor
// prod_{u=r..i} alpha_u, key factor prod_{u=j+1..r-1} alpha_u.
struct Quarter {
    float2 al[4], f[4], b[4];
};

// KDA-style retention gate ("Ask Self, Ask Others", Sec. 5.2 eq.(16); Appendix
// A.4.1) of one thread's channels c = 2 lane, 2 lane + 1 of head h:
// g = -exp(A_log[h, c]) softplus(r + dt_bias[h, c]).  on == false: the loaded
// values are g itself.  The kernels take the gate as a template parameter, so
// `on` is a compile-time constant and the ungated kernels carry none of it.
struct GateCh {
    float2 na, db;  // -exp(A_log), dt_bias
    bool on;
};
template <bool kGate, class A>
__device__ __forceinline__ GateCh gate_channels(const A& a, int64_t bh, int lane) {
    GateCh gc{make_float2(0.f, 0.f), make_float2(0.f, 0.f), kGate};
    const int c = 2 * lane, d = a.kp.d;
    if (kGate && c < d) {
        const size_t o = (size_t)(bh % a.kp.H) * d + c;
        gc.na = make_float2(-expf(a.gate_alog[o]), -expf(a.gate_alog[o + 1]));
        gc.db = make_float2(a.gate_dtb[o], a.gate_dtb[o + 1]);
    }
    return gc;
}
// softplus(x) = max(x, 0) + log(1 + e^-|x|), which overflows for no x; the
// logarithm's argument is rounded to fp32, an absolute error below 1e-7 in g,
// i.e. in the retention alpha = exp(g) a relative error below 1e-7 x alpha.
__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x))); }
__device__ __forceinline__ float2 gate_g(float2 r, const GateCh& gc) {
    return make_float2(gc.na.x * softplus_f(r.x + gc.db.x), gc.na.y * softplus_f(r.y + gc.db.y));
}

template <class GS, class ST>
__device__ __forceinline__ void channel_phase_a(Quarter& Q, GS& gs, const ST& s, int d, int warp, int lane,
                                                const GateCh& gc) {
    const int c = 2 * lane;
    const bool valid = c < d;
    float2 prod = make_float2(1.f, 1.f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float2 g = *reinterpret_cast<const float2*>(s.g + (4 * warp + r) * kDp + c);
        if (gc.on) g = gate_g(g, gc);
        Q.al[r] = valid ? make_float2(__expf(g.x), __expf(g.y)) : make_float2(1.f, 1.f);
        prod = mul2(prod, Q.al[r]);
        Q.f[r] = prod;
    }
    float2 back = make_float2(1.f, 1.f);
#pragma unroll
    for (int r = 3; r >= 0; --r) {
        Q.b[r] = back;
        back = mul2(back, Q.al[r]);
    }
    *reinterpret_cast<float2*>(&gs.tot[warp][c]) = prod;
}

// Products shared by every token of the quarter (read after the barrier).
struct QuarterTotals {
    float2 P[4], pre, suf;
};
template <class GS>
__device__ __forceinline__ QuarterTotals quarter_totals(GS& gs, int warp, int lane) {
    const int c = 2 * lane;
    QuarterTotals T;
#pragma unroll
    for (int k = 0; k < 4; ++k) T.P[k] = *reinterpret_cast<const float2*>(&gs.tot[k][c]);
    T.pre = make_float2(1.f, 1.f);
    T.suf = make_float2(1.f, 1.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (k < warp) T.pre = mul2(T.pre, T.P[k]);
        if (k > warp) T.suf = mul2(T.suf, T.P[k]);
    }
    return T;
}
// Factor of token r of quarter `warp` at level bit b (query side / key side).
__device__ __forceinline__ float2 query_factor(const Quarter& Q, const QuarterTotals& T, int warp, int r, int b) {
    if (b == 3) return warp == 3 ? mul2(T.P[2], Q.f[r]) : Q.f[r];
    if (b == 2) return Q.f[r];
    if (b == 1) return r == 2 ? Q.al[2] : mul2(Q.al[2], Q.al[3]);
    return Q.al[r];
}
__device__ __forceinline__ float2 key_factor(const Quarter& Q, const QuarterTotals& T, int warp, int r, int b) {
    if (b == 3) return warp == 0 ? mul2(Q.b[r], T.P[1]) : Q.b[r];
    if (b == 2) return Q.b[r];
    if (b == 1) return r == 0 ? Q.al[1] : make_float2(1.f, 1.f);
    return make_float2(1.f, 1.f);
}
__device__ __forceinline__ bool is_query(int i, int b) { return (i >> b) & 1; }

// Writes the operands of the chunk: q . F (kQT), k . B (kKB), the level query
// (kLQ) and key (kLK) operands; warp 0 writes the chunk retention.
template <bool kQT, bool kKB, bool kLQ, bool kLK, class GS, class ST>
__device__ __forceinline__ void channel_phase_b(const Quarter& Q, const QuarterTotals& T, GS& gs, const ST& s,
                                                int warp, int lane) {
    const int c = 2 * lane;
    if (warp == 0) *reinterpret_cast<float2*>(gs.avec + c) = mul2(mul2(T.P[0], T.P[1]), mul2(T.P[2], T.P[3]));
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = 4 * warp + r;
        const uint32_t sw = swz(i, c);
        const float2 rr = gs.rs[i];
        float2 k = make_float2(0.f, 0.f), q = make_float2(0.f, 0.f);
        if (kKB || kLK) {
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(s.p2 + sw);
            k = make_float2(lo_f(w2) * rr.y, hi_f(w2) * rr.y);
        }
        if (kQT || kLQ) {
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(s.p1 + sw);
            q = make_float2(lo_f(w1) * rr.x, hi_f(w1) * rr.x);
        }
        if (kKB) {
            const float2 x = mul2(k, mul2(Q.b[r], T.suf));
            *reinterpret_cast<uint32_t*>(gs.kb + sw) = pack2(x.x, x.y);
        }
        if (kQT) {
            const float2 x = mul2(q, mul2(T.pre, Q.f[r]));
            *reinterpret_cast<uint32_t*>(gs.qt + sw) = pack2(x.x, x.y);
        }
#pragma unroll
        for (int lvl = 0; lvl < 4; ++lvl) {
            const int b = 3 - lvl;
            if (is_query(i, b)) {
                if (kLQ) {
                    const float2 x = mul2(q, query_factor(Q, T, warp, r, b));
                    *reinterpret_cast<uint32_t*>(gs.ql[lvl] + sw) = pack2(x.x, x.y);
                }
            } else if (kLK) {
                const float2 x = mul2(k, key_factor(Q, T, warp, r, b));
                *reinterpret_cast<uint32_t*>(gs.kl[lvl] + swz(key_row(i, b), c)) = pack2(x.x, x.y);
            }
        }
    }
}

// Warp w computes level bit b = 3 - w of the intra-chunk matrix: the 16 x 8
// product of its query and key operands, and writes the entries (i, j) whose
// first differing bit is b into gs.amat (zeroed beforehand).
template <class GS>
__device__ __forceinline__ void level_matrix(GS& gs, int warp, int lane) {
    const int lvl = warp, b = 3 - warp;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t af[4], bf[4];
        ldsm4(af, addr_a(gs.ql[lvl], 16 * ks, lane));
        // B from the [n][k] key tile (8 rows): matrices (k 0-7), (k 8-15) for n 0-7.
        const int m = lane >> 3;
        ldsm4(bf, ptx::smem_u32(gs.kl[lvl]) + swz(lane & 7, 16 * ks + 8 * (m & 1)));
        mma16816(acc, af, bf[0], bf[1]);
    }
    const int g = lane >> 2, t = lane & 3;
    __nv_bfloat16* A = reinterpret_cast<__nv_bfloat16*>(gs.amat);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int i = g + 8 * (e >> 1), n = 2 * t + (e & 1);
        const int j = ((n >> b) << (b + 1)) | (n & ((1 << b) - 1));
        if (((i >> b) & 1) && (i >> (b + 1)) == (j >> (b + 1))) A[i * (kArow / 2) + j] = __float2bfloat16_rn(acc[e]);
    }
}

// The warp's slice of the state C^T: rows v = 16w + g (+8 for r >= 2), columns
// c = 8 nt + 2t + (r & 1) (mma accumulator layout, g = lane/4, t = lane%4).
struct State {
    float x[8][4];
};

__device__ __forceinline__ void state_zero(State& S) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) S.x[nt][r] = 0.f;
}
// C [64][64] (row = key channel c, column = value channel v) <-> registers.
__device__ __forceinline__ void state_load(State& S, const float* C, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int v = 16 * warp + g + 8 * (r >> 1), c = 8 * nt + 2 * t + (r & 1);
            S.x[nt][r] = C[c * kDp + v];
        }
}
__device__ __forceinline__ void state_store(const State& S, float* C, int ld, int d, int warp, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int v = 16 * warp + g + 8 * (r >> 1), c = 8 * nt + 2 * t + (r & 1);
            if (v < d && c < d) C[c * ld + v] = S.x[nt][r];
        }
}

// C <- Diag(a) C + (k . B)^T I~ on the warp's slice.
template <class GS, class ST>
__device__ __forceinline__ void state_update(State& S, const GS& gs, const ST& s, int warp, int lane) {
    const int t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const float2 a = *reinterpret_cast<const float2*>(gs.avec + 8 * nt + 2 * t);
        S.x[nt][0] *= a.x;
        S.x[nt][1] *= a.y;
        S.x[nt][2] *= a.x;
        S.x[nt][3] *= a.y;
    }
    uint32_t af[4];
    ldsm4t(af, addr_at(s.v, 16 * warp, lane));
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t r[4];
        ldsm4t(r, addr_bt(gs.kb, 16 * p, lane));
        mma16816(S.x[2 * p], af, r[0], r[1]);
        mma16816(S.x[2 * p + 1], af, r[2], r[3]);
    }
}

// E = (q . F) C + A I~ on the warp's value channels: E[s][r], token g (+8 for
// r >= 2), v = 16w + 8s + 2t (+1).
__device__ __forceinline__ void chunk_output(float (&E)[2][4], const State& S, const GroupSmem& gs, const Stage& s,
                                             int warp, int lane) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r) E[h][r] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t af[4];
        ldsm4(af, addr_a(gs.qt, 16 * ks, lane));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t b0 = pack2(S.x[2 * ks][2 * h], S.x[2 * ks][2 * h + 1]);
            const uint32_t b1 = pack2(S.x[2 * ks + 1][2 * h], S.x[2 * ks + 1][2 * h + 1]);
            mma16816(E[h], af, b0, b1);
        }
    }
    uint32_t af[4];
    {
        const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), cb = 16 * (m >> 1);
        ldsm4(af, ptx::smem_u32(gs.amat) + r * kArow + cb);
    }
    uint32_t r[4];
    ldsm4t(r, addr_bt(s.v, 16 * warp, lane));
    mma16816(E[0], af, r[0], r[1]);
    mma16816(E[1], af, r[2], r[3]);
}

__device__ __forceinline__ void zero_group_smem(GroupSmem& gs) {
    uint4* p = reinterpret_cast<uint4*>(&gs);
    const int n = (int)(sizeof(GroupSmem) / 16);
    for (int k = threadIdx.x; k < n; k += kThreads) p[k] = make_uint4(0, 0, 0, 0);
    __syncthreads();
}

// ------------------------------------------------------------------- kernels
// One CTA (4 warps) per work item bh * nseg + segment.
template <bool kVec16, bool kOut, bool kGate>
__device__ __forceinline__ void segment_pass(const Args& a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    GroupSmem& gs = *reinterpret_cast<GroupSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x;
    const int64_t bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const KernelProblem& kp = a.kp;
    const int t_begin = seg * a.seg_len, t_end = min(kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    zero_group_smem(gs);

    State S;
    if (kOut && a.nseg > 1)
        state_load(S, a.hseg + (size_t)item * kDp * kDp, warp, lane);
    else
        state_zero(S);
    float2 aseg = make_float2(1.f, 1.f);
    const int g = lane >> 2, t = lane & 3;
    const RowMap rm = row_map(kp, bh);
    const GateCh gc = gate_channels<kGate>(a, bh, lane);
    load_chunk<kVec16>(gs.st[0], a, rm, t_begin, warp, lane);
    for (int n = 0; n < nchunks; ++n) {
        Stage& s = gs.st[n & 1];
        const int t0 = t_begin + n * kC;
        cp_async_wait<0>();
        __syncthreads();  // chunk n visible; every warp is done with chunk n-1
        if (n + 1 < nchunks) load_chunk<kVec16>(gs.st[(n + 1) & 1], a, rm, t0 + kC, warp, lane);
        row_scalars(gs, s, a.zscale, warp, lane);
        Quarter Q;
        channel_phase_a(Q, gs, s, kp.d, warp, lane, gc);
        if (kOut && warp == 0) {
            uint4* A = reinterpret_cast<uint4*>(gs.amat);
            for (int k = lane; k < (int)(sizeof(gs.amat) / 16); k += 32) A[k] = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
        {
            const QuarterTotals T = quarter_totals(gs, warp, lane);
            channel_phase_b<kOut, true, kOut, kOut>(Q, T, gs, s, warp, lane);
        }
        __syncthreads();
        if (kOut) {
            level_matrix(gs, warp, lane);
            __syncthreads();
            float E[2][4];
            chunk_output(E, S, gs, s, warp, lane);
            const size_t yrow0 = rm.base + (size_t)t0 * rm.stride;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = g + 8 * half;
                if (t0 + r < kp.T) {
                    __nv_bfloat16* yrow = a.Y + yrow0 + (size_t)r * rm.stride;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int v = 16 * warp + 8 * h + 2 * t;
                        if (v < kp.d) {
                            const uint32_t iw = *reinterpret_cast<const uint32_t*>(s.v + swz(r, v));
                            *reinterpret_cast<uint32_t*>(yrow + v) =
                                pack2(lo_f(iw) + E[h][2 * half], hi_f(iw) + E[h][2 * half + 1]);
                        }
                    }
                }
            }
        } else if (warp == 0) {
            aseg = mul2(aseg, *reinterpret_cast<const float2*>(gs.avec + 2 * lane));
        }
        state_update(S, gs, s, warp, lane);
    }
    if (kOut) {
        if (a.nseg == 1 && a.state_out != nullptr)
            state_store(S, a.state_out + (size_t)bh * kp.d * kp.d, kp.d, kp.d, warp, lane);
    } else {
        state_store(S, a.hseg + (size_t)item * kDp * kDp, kDp, kDp, warp, lane);
        if (warp == 0) *reinterpret_cast<float2*>(a.aseg + (size_t)item * kDp + 2 * lane) = aseg;
    }
}

template <bool kVec16, bool kGate>
__global__ void __launch_bounds__(kThreads, 4) linear_state_kernel(Args a) {
    segment_pass<kVec16, false, kGate>(a);
}
template <bool kVec16, bool kGate>
__global__ void __launch_bounds__(kThreads, 4) linear_fwd_kernel(Args a) {
    segment_pass<kVec16, true, kGate>(a);
}

// Entering state of every segment (in place of its own contribution) and the
// final state.  One thread per state entry (c, v); 16 blocks per head.
__global__ void __launch_bounds__(256) linear_scan_kernel(float* hseg, const float* aseg, int nseg, float* state_out,
                                                          int d) {
    const int64_t bh = blockIdx.x >> 4;
    const int e = ((blockIdx.x & 15) << 8) | threadIdx.x, c = e >> 6, v = e & 63;
    float* H = hseg + (size_t)bh * nseg * kDp * kDp + e;
    const float* A = aseg + (size_t)bh * nseg * kDp + c;
    float h = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += 16) {
        float dh[16], al[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const bool ok = s0 + k < nseg;
            dh[k] = ok ? H[(size_t)(s0 + k) * kDp * kDp] : 0.f;
            al[k] = ok ? A[(size_t)(s0 + k) * kDp] : 1.f;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (s0 + k < nseg) H[(size_t)(s0 + k) * kDp * kDp] = h;
            h = fmaf(al[k], h, dh[k]);
        }
    }
    if (state_out != nullptr && c < d && v < d) state_out[((size_t)bh * d + c) * d + v] = h;
}

// ================================================================= backward
// With q = S p^1, k = S p^2, the chunk products give (dE = dY):
//   dq_i = F_i . (C dE_i) + sum_{j<i} dA_ij k_j . P(j, i),   dA_ij = dE_i . I~_j,
//   dk_j = B_j . (dC v_j) + sum_{i>j} dA_ij q_i . P(j, i),   dv_j = dC^T (k_j . B_j)
//          + sum_{i>j} A_ij dE_i + dY_j,
// with C the state entering the chunk (forward in time) and dC the gradient of the
// state leaving it (backward in time: dC <- Diag(a) dC + (q . F)^T dE).  The
// retention gradient uses dg_u = sum_{t >= u} (q_t . dq_t - k_t . dk_t), the sum
// running to the end of the sequence; from a segment end on it equals the row
// sums of C_end . dC_end.  Sweep A (forward) writes q . dq into dG as scratch,
// the normalisation part of dP1 into dP1 and p^1 . dq per token; sweep B
// (backward) finishes dG, dP1, dP2 and dI~.
struct BStage {
    uint8_t p1[kC * 128];
    uint8_t p2[kC * 128];
    uint8_t v[kC * 128];
    uint8_t dy[kC * 128];
    float g[kC * kDp];
};
// Row stride (floats) of the fp32 exchange tiles: 72 rather than 64 so the 8-byte
// stores from the accumulator layout (8 rows x 4 column pairs per instruction) take
// two shared-memory wavefronts instead of eight.
constexpr int kXs = 72;
struct BwdSmem {
    static constexpr bool kNorms = true;
    BStage st[2];
    uint8_t qt[kC * 128];
    uint8_t kb[kC * 128];
    uint8_t ql[4][kC * 128];
    uint8_t kl[4][8 * 128];
    uint8_t amat[kC * kArow];
    uint8_t dal[4][kC * kArow];  // dA on the pairs of each level, keys compacted (columns 8..15 zero)
    float xq[kC * kXs];          // dQ~ (sweep A) or dK~ (sweep B), fp32 [row][channel]
    float xl[4][kC * kXs];       // per level: dQ_L [token][c] (sweep A) or dK_L [key row][c] (sweep B)
    float2 rs[kC];               // (S / ||p1||, S / ||p2||)
    float4 rn[kC];               // (1 / ||p1||, 1 / ||p2||, S, -)
    float avec[kDp];
    float tot[4][kDp];
    float zt[4][kDp];   // quarter sums of q . dq - k . dk
    float bnd[kDp];     // row sums of C_end . dC_end at the segment end
};

struct BArgs {
    const __nv_bfloat16* P1;
    const __nv_bfloat16* P2;
    const __nv_bfloat16* V;
    const float* G;         // log-retention g, or the gate's input r (gate_alog != nullptr)
    const float* gate_alog;  // KDA gate [H, d]: A_log, or nullptr
    const float* gate_dtb;   // KDA gate [H, d]: dt_bias
    float* gate_dalog;       // gate: d A_log [H, d] (+=), or nullptr
    float* gate_ddtb;        // gate: d dt_bias [H, d] (+=)
    const __nv_bfloat16* dY;
    __nv_bfloat16* dP1;
    __nv_bfloat16* dP2;
    __nv_bfloat16* dV;
    float* dG;
    float* hseg;   // entering states of the segments (after the forward scan)
    float* aseg;   // retention over each segment
    float* dcseg;  // gradient of the state at each segment end (after the reverse scan)
    float* pdq;    // [BH, T]: p^1 . dq per token
    KernelProblem kp;
    float zscale;
    int nseg;
    int seg_len;
};

// Copies of chunk rows t0..t0+15: warps 0-2 take P1, P2, I~; warp 3 takes G and dY.
template <bool kVec16>
__device__ __forceinline__ void copy_bf16_rows(uint8_t* tile, const __nv_bfloat16* src, const RowMap& rm, int t0,
                                               int T, int d, int lane) {
    const uint32_t base = ptx::smem_u32(tile);
    if (kVec16) {
        const int q = lane & 7, col = 8 * q;
        if (col < d) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = (lane >> 3) + 4 * k;
                const uint32_t dst = base + r * 128 + (((q ^ r) & 7) << 4);
                if (t0 + r < T)
                    cp_async_16(dst, src + (size_t)r * rm.stride + col);
                else
                    st_zero16(dst);
            }
        }
    } else {
        const int q = lane & 15, col = 4 * q;
        if (col < d) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = (lane >> 4) + 2 * k;
                const uint32_t dst = base + r * 128 + ((((q >> 1) ^ r) & 7) << 4) + ((q & 1) << 3);
                if (t0 + r < T)
                    cp_async_8(dst, src + (size_t)r * rm.stride + col);
                else
                    st_shared_zero8(dst);
            }
        }
    }
}
template <bool kVec16>
__device__ __forceinline__ void load_chunk_b(BStage& s, const BArgs& a, const RowMap& rm, int t0, int warp, int lane,
                                             bool need_v) {
    const KernelProblem& kp = a.kp;
    const size_t off = rm.base + (size_t)t0 * rm.stride;
    if (warp == 0) copy_bf16_rows<kVec16>(s.p1, a.P1 + off, rm, t0, kp.T, kp.d, lane);
    if (warp == 1) copy_bf16_rows<kVec16>(s.p2, a.P2 + off, rm, t0, kp.T, kp.d, lane);
    if (warp == 2) {
        if (need_v) copy_bf16_rows<kVec16>(s.v, a.V + off, rm, t0, kp.T, kp.d, lane);
        copy_bf16_rows<kVec16>(s.dy, a.dY + off, rm, t0, kp.T, kp.d, lane);
    }
    if (warp == 3) {
        const float* src = a.G + off;
        const int q = lane & 15, col = 4 * q;
        const uint32_t gb = ptx::smem_u32(s.g);
        if (col < kp.d) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int r = (lane >> 4) + 2 * k;
                const uint32_t dst = gb + (r * kDp + col) * 4;
                if (t0 + r < kp.T)
                    cp_async_16(dst, src + (size_t)r * rm.stride + col);
                else
                    st_zero16(dst);
            }
        }
    }
    cp_async_commit();
}

// B fragments of two 8-row blocks n0.., n0+8.. from an [n][k] tile (no .trans):
// r0 = b0 (n 0-7), r1 = b1 (n 0-7), r2 = b0 (n 8-15), r3 = b1 (n 8-15).
__device__ __forceinline__ uint32_t addr_b(const uint8_t* tile, int k0, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m >> 1), c = k0 + 8 * (m & 1);
    return ptx::smem_u32(tile) + swz(r, c);
}
// A operand from a [k][m] 16 x 16 tile with 48-byte rows (.trans).
__device__ __forceinline__ uint32_t addr_at48(const uint8_t* tile, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m >> 1), c = 8 * (m & 1);
    return ptx::smem_u32(tile) + r * kArow + 2 * c;
}
// A operand from a row-major [m][k] 16 x 16 tile with 48-byte rows.
__device__ __forceinline__ uint32_t addr_a48(const uint8_t* tile, int lane) {
    const int m = lane >> 3, r = (lane & 7) + 8 * (m & 1), c = 8 * (m >> 1);
    return ptx::smem_u32(tile) + r * kArow + 2 * c;
}
__device__ __forceinline__ void ldsm2t(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// dA = dE I~^T (16 x 16) and the level-w tile of it (keys compacted, zero elsewhere).
__device__ __forceinline__ void level_dA(BwdSmem& gs, const BStage& s, int warp, int lane) {
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t af[4], bf[4];
        ldsm4(af, addr_a(s.dy, 16 * ks, lane));
        ldsm4(bf, addr_b(s.v, 16 * ks, lane));
        mma16816(acc[0], af, bf[0], bf[1]);
        mma16816(acc[1], af, bf[2], bf[3]);
    }
    uint8_t* tile = gs.dal[warp];
    {
        uint4* z = reinterpret_cast<uint4*>(tile);
        for (int k = lane; k < (int)(kC * kArow / 16); k += 32) z[k] = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    const int b = 3 - warp, g = lane >> 2, t = lane & 3;
    __nv_bfloat16* D = reinterpret_cast<__nv_bfloat16*>(tile);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = g + 8 * (e >> 1), j = 8 * h + 2 * t + (e & 1);
            if (is_query(i, b) && !is_query(j, b) && (i >> (b + 1)) == (j >> (b + 1)))
                D[i * (kArow / 2) + key_row(j, b)] = __float2bfloat16_rn(acc[h][e]);
        }
}

// ---- state passes of the backward (segment contributions of the reverse state)
template <bool kVec16, bool kGate>
__global__ void __launch_bounds__(kThreads, 3) linear_bstate_kernel(BArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BwdSmem& gs = *reinterpret_cast<BwdSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x, bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const KernelProblem& kp = a.kp;
    const int t_begin = seg * a.seg_len, t_end = min(kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    {
        uint4* p = reinterpret_cast<uint4*>(&gs);
        for (int k = threadIdx.x; k < (int)(sizeof(BwdSmem) / 16); k += kThreads) p[k] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    State D;  // dC rows c = 16w + g (+8), columns v
    state_zero(D);
    const RowMap rm = row_map(kp, bh);
    const GateCh gc = gate_channels<kGate>(a, bh, lane);
    load_chunk_b<kVec16>(gs.st[(nchunks - 1) & 1], a, rm, t_begin + (nchunks - 1) * kC, warp, lane, false);
    for (int n = nchunks - 1; n >= 0; --n) {
        BStage& s = gs.st[n & 1];
        cp_async_wait<0>();
        __syncthreads();
        if (n > 0) load_chunk_b<kVec16>(gs.st[(n - 1) & 1], a, rm, t_begin + (n - 1) * kC, warp, lane, false);
        row_scalars(gs, s, a.zscale, warp, lane);
        Quarter Q;
        channel_phase_a(Q, gs, s, kp.d, warp, lane, gc);
        __syncthreads();
        {
            const QuarterTotals T = quarter_totals(gs, warp, lane);
            channel_phase_b<true, false, false, false>(Q, T, gs, s, warp, lane);
        }
        __syncthreads();
        // dC <- Diag(a) dC + (q . F)^T dE on rows c of this warp
        const int g = lane >> 2;
        const float a0 = gs.avec[16 * warp + g], a1 = gs.avec[16 * warp + 8 + g];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            D.x[nt][0] *= a0;
            D.x[nt][1] *= a0;
            D.x[nt][2] *= a1;
            D.x[nt][3] *= a1;
        }
        uint32_t af[4];
        ldsm4t(af, addr_at(gs.qt, 16 * warp, lane));
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t r[4];
            ldsm4t(r, addr_bt(s.dy, 16 * p, lane));
            mma16816(D.x[2 * p], af, r[0], r[1]);
            mma16816(D.x[2 * p + 1], af, r[2], r[3]);
        }
    }
    // store rows c of dC as [c][v]
    const int g = lane >> 2, t = lane & 3;
    float* out = a.dcseg + (size_t)item * kDp * kDp;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) out[(16 * warp + g + 8 * (r >> 1)) * kDp + 8 * nt + 2 * t + (r & 1)] = D.x[nt][r];
}

// Gradient of the state at every segment end (in place of the segment's own
// contribution); zero after the last segment.
__global__ void __launch_bounds__(256) linear_bscan_kernel(float* dcseg, const float* aseg, int nseg) {
    const int64_t bh = blockIdx.x >> 4;
    const int e = ((blockIdx.x & 15) << 8) | threadIdx.x, c = e >> 6;
    float* H = dcseg + (size_t)bh * nseg * kDp * kDp + e;
    const float* A = aseg + (size_t)bh * nseg * kDp + c;
    float h = 0.f;
    for (int s1 = nseg - 1; s1 >= 0; s1 -= 16) {
        float dh[16], al[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const bool ok = s1 - k >= 0;
            dh[k] = ok ? H[(size_t)(s1 - k) * kDp * kDp] : 0.f;
            al[k] = ok ? A[(size_t)(s1 - k) * kDp] : 1.f;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (s1 - k >= 0) H[(size_t)(s1 - k) * kDp * kDp] = h;
            h = fmaf(al[k], h, dh[k]);
        }
    }
}

// ---- sweep A: forward in time, dq
template <bool kVec16, bool kGate>
__global__ void __launch_bounds__(kThreads, 3) linear_bwd_a_kernel(BArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BwdSmem& gs = *reinterpret_cast<BwdSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x, bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const KernelProblem& kp = a.kp;
    const int t_begin = seg * a.seg_len, t_end = min(kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    {
        uint4* p = reinterpret_cast<uint4*>(&gs);
        for (int k = threadIdx.x; k < (int)(sizeof(BwdSmem) / 16); k += kThreads) p[k] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    const int g = lane >> 2, t = lane & 3, c = 2 * lane;
    // Entering state C, rows c = 16w + g (+8), columns v.
    State H;
    if (a.nseg > 1) {
        const float* src = a.hseg + (size_t)item * kDp * kDp;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                H.x[nt][r] = src[(16 * warp + g + 8 * (r >> 1)) * kDp + 8 * nt + 2 * t + (r & 1)];
    } else {
        state_zero(H);
    }
    const RowMap rm = row_map(kp, bh);
    const GateCh gc = gate_channels<kGate>(a, bh, lane);
    load_chunk_b<kVec16>(gs.st[0], a, rm, t_begin, warp, lane, true);
    for (int n = 0; n < nchunks; ++n) {
        BStage& s = gs.st[n & 1];
        const int t0 = t_begin + n * kC;
        cp_async_wait<0>();
        __syncthreads();  // B1
        if (n + 1 < nchunks) load_chunk_b<kVec16>(gs.st[(n + 1) & 1], a, rm, t0 + kC, warp, lane, true);
        row_scalars(gs, s, a.zscale, warp, lane);
        Quarter Q;
        channel_phase_a(Q, gs, s, kp.d, warp, lane, gc);
        __syncthreads();  // B2
        const QuarterTotals T = quarter_totals(gs, warp, lane);
        channel_phase_b<false, true, false, true>(Q, T, gs, s, warp, lane);
        level_dA(gs, s, warp, lane);
        __syncthreads();  // B3
        {
            // dQ~ = dE C^T and dQ_L = dA_L K_L on channels [16w, 16w+16)
            float dq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t af[4];
                ldsm4(af, addr_a(s.dy, 16 * ks, lane));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t b0 = pack2(H.x[2 * ks][2 * h], H.x[2 * ks][2 * h + 1]);
                    const uint32_t b1 = pack2(H.x[2 * ks + 1][2 * h], H.x[2 * ks + 1][2 * h + 1]);
                    mma16816(dq[h], af, b0, b1);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = 16 * warp + 8 * h + 2 * t;
                *reinterpret_cast<float2*>(gs.xq + g * kXs + col) = make_float2(dq[h][0], dq[h][1]);
                *reinterpret_cast<float2*>(gs.xq + (g + 8) * kXs + col) = make_float2(dq[h][2], dq[h][3]);
            }
#pragma unroll
            for (int lvl = 0; lvl < 4; ++lvl) {
                uint32_t af[4], b0a, b0b;
                ldsm4(af, addr_a48(gs.dal[lvl], lane));
                ldsm2t(b0a, b0b, ptx::smem_u32(gs.kl[lvl]) + swz(lane & 7, 16 * warp + 8 * ((lane >> 3) & 1)));
                float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                mma16816(o[0], af, b0a, 0u);
                mma16816(o[1], af, b0b, 0u);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col = 16 * warp + 8 * h + 2 * t;
                    *reinterpret_cast<float2*>(gs.xl[lvl] + g * kXs + col) = make_float2(o[h][0], o[h][1]);
                    *reinterpret_cast<float2*>(gs.xl[lvl] + (g + 8) * kXs + col) = make_float2(o[h][2], o[h][3]);
                }
            }
            // C <- Diag(a) C + (k . B)^T I~ on rows c of this warp
            const float a0 = gs.avec[16 * warp + g], a1 = gs.avec[16 * warp + 8 + g];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                H.x[nt][0] *= a0;
                H.x[nt][1] *= a0;
                H.x[nt][2] *= a1;
                H.x[nt][3] *= a1;
            }
            uint32_t af[4];
            ldsm4t(af, addr_at(gs.kb, 16 * warp, lane));
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t r[4];
                ldsm4t(r, addr_bt(s.v, 16 * p, lane));
                mma16816(H.x[2 * p], af, r[0], r[1]);
                mma16816(H.x[2 * p + 1], af, r[2], r[3]);
            }
        }
        __syncthreads();  // B4
        // Channel layout: warp = token quarter, lane = channels c, c+1.
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * warp + r, tok = t0 + i;
            float2 dq = mul2(mul2(T.pre, Q.f[r]), *reinterpret_cast<const float2*>(gs.xq + i * kXs + c));
#pragma unroll
            for (int lvl = 0; lvl < 4; ++lvl) {
                const int b = 3 - lvl;
                if (is_query(i, b))
                    dq = fma2(query_factor(Q, T, warp, r, b), *reinterpret_cast<const float2*>(gs.xl[lvl] + i * kXs + c),
                              dq);
            }
            const float4 rn = gs.rn[i];
            const float s1 = gs.rs[i].x;
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(s.p1 + swz(i, c));
            const float2 p1 = make_float2(lo_f(w1), hi_f(w1));
            const float2 ph = make_float2(p1.x * rn.x, p1.y * rn.x);
            float pd = ph.x * dq.x + ph.y * dq.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, o);
            if (tok < kp.T) {
                const size_t off = rm.base + (size_t)tok * rm.stride;
                if (c < kp.d) {
                    const float2 q = make_float2(p1.x * s1, p1.y * s1);
                    *reinterpret_cast<float2*>(a.dG + off + c) = mul2(q, dq);
                    *reinterpret_cast<uint32_t*>(a.dP1 + off + c) =
                        pack2(s1 * (dq.x - ph.x * pd), s1 * (dq.y - ph.y * pd));
                }
                if (lane == 0) a.pdq[(size_t)bh * kp.T + tok] = pd;
            }
        }
    }
}

// ---- sweep B: backward in time, dk, dv and the outputs
template <bool kVec16, bool kGate>
__global__ void __launch_bounds__(kThreads, 3) linear_bwd_b_kernel(BArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    BwdSmem& gs = *reinterpret_cast<BwdSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t item = blockIdx.x, bh = item / a.nseg;
    const int seg = (int)(item - bh * a.nseg);
    const KernelProblem& kp = a.kp;
    const int t_begin = seg * a.seg_len, t_end = min(kp.T, t_begin + a.seg_len);
    const int nchunks = (t_end - t_begin + kC - 1) / kC;
    {
        uint4* p = reinterpret_cast<uint4*>(&gs);
        for (int k = threadIdx.x; k < (int)(sizeof(BwdSmem) / 16); k += kThreads) p[k] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    const int g = lane >> 2, t = lane & 3, c = 2 * lane;
    // Gradient of the state leaving the segment: DC rows c = 16w + g (+8), columns v;
    // DT the same matrix with rows v = 16w + g (+8), columns c.
    State DC, DT;
    const bool has_end = a.nseg > 1 && seg + 1 < a.nseg;
    if (has_end) {
        const float* src = a.dcseg + (size_t)item * kDp * kDp;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int rr = 16 * warp + g + 8 * (r >> 1), cc = 8 * nt + 2 * t + (r & 1);
                DC.x[nt][r] = src[rr * kDp + cc];
                DT.x[nt][r] = src[cc * kDp + rr];
            }
        // bnd_c = sum_v C_end[c][v] dC_end[c][v], C_end = entering state of the next segment
        const float* hn = a.hseg + (size_t)(item + 1) * kDp * kDp;
        const int cc = threadIdx.x >> 1, v0 = (threadIdx.x & 1) * 32;
        float acc = 0.f;
        for (int v = 0; v < 32; ++v) acc = fmaf(hn[cc * kDp + v0 + v], src[cc * kDp + v0 + v], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if ((threadIdx.x & 1) == 0) gs.bnd[cc] = acc;
    } else {
        state_zero(DC);
        state_zero(DT);
    }
    __syncthreads();
    float2 carry = *reinterpret_cast<const float2*>(gs.bnd + c);  // sum of z over the later tokens (+ boundary)
    const RowMap rm = row_map(kp, bh);
    const GateCh gc = gate_channels<kGate>(a, bh, lane);
    float2 acc_dalog = make_float2(0.f, 0.f), acc_ddtb = make_float2(0.f, 0.f);  // gate: this thread's token sums
    load_chunk_b<kVec16>(gs.st[(nchunks - 1) & 1], a, rm, t_begin + (nchunks - 1) * kC, warp, lane, true);
    for (int n = nchunks - 1; n >= 0; --n) {
        BStage& s = gs.st[n & 1];
        const int t0 = t_begin + n * kC;
        cp_async_wait<0>();
        __syncthreads();  // B1
        if (n > 0) load_chunk_b<kVec16>(gs.st[(n - 1) & 1], a, rm, t0 - kC, warp, lane, true);
        row_scalars(gs, s, a.zscale, warp, lane);
        Quarter Q;
        channel_phase_a(Q, gs, s, kp.d, warp, lane, gc);
        if (warp == 0) {
            uint4* A = reinterpret_cast<uint4*>(gs.amat);
            for (int k = lane; k < (int)(sizeof(gs.amat) / 16); k += 32) A[k] = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();  // B2
        const QuarterTotals T = quarter_totals(gs, warp, lane);
        channel_phase_b<true, true, true, true>(Q, T, gs, s, warp, lane);
        __syncthreads();  // B3
        // Scratch written by sweep A for this warp's tokens (q . dq, the normalisation
        // part of dP1, p^1 . dq), loaded now so the latency hides under the products.
        float2 xs[4];
        uint32_t p1w[4];
        float pq[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int tok = t0 + 4 * warp + r;
            xs[r] = make_float2(0.f, 0.f);
            p1w[r] = 0u;
            pq[r] = 0.f;
            if (tok < kp.T) {
                const size_t off = rm.base + (size_t)tok * rm.stride + c;
                if (c < kp.d) {
                    xs[r] = *reinterpret_cast<const float2*>(a.dG + off);
                    p1w[r] = *reinterpret_cast<const uint32_t*>(a.dP1 + off);
                }
                pq[r] = a.pdq[(size_t)bh * kp.T + tok];
            }
        }
        level_matrix(gs, warp, lane);
        level_dA(gs, s, warp, lane);
        __syncthreads();  // B4
        {
            // dK~ = I~ dC^T on channels [16w, 16w+16)
            float dk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t af[4];
                ldsm4(af, addr_a(s.v, 16 * ks, lane));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t b0 = pack2(DC.x[2 * ks][2 * h], DC.x[2 * ks][2 * h + 1]);
                    const uint32_t b1 = pack2(DC.x[2 * ks + 1][2 * h], DC.x[2 * ks + 1][2 * h + 1]);
                    mma16816(dk[h], af, b0, b1);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = 16 * warp + 8 * h + 2 * t;
                *reinterpret_cast<float2*>(gs.xq + g * kXs + col) = make_float2(dk[h][0], dk[h][1]);
                *reinterpret_cast<float2*>(gs.xq + (g + 8) * kXs + col) = make_float2(dk[h][2], dk[h][3]);
            }
            // dK_L = dA_L^T Q_L (rows: compacted keys 0..7)
#pragma unroll
            for (int lvl = 0; lvl < 4; ++lvl) {
                uint32_t af[4], r4[4];
                ldsm4t(af, addr_at48(gs.dal[lvl], lane));
                ldsm4t(r4, addr_bt(gs.ql[lvl], 16 * warp, lane));
                float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                mma16816(o[0], af, r4[0], r4[1]);
                mma16816(o[1], af, r4[2], r4[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<float2*>(gs.xl[lvl] + g * kXs + 16 * warp + 8 * h + 2 * t) =
                        make_float2(o[h][0], o[h][1]);
            }
            // dI~ = (k . B) dC + A^T dE + dY on value channels [16w, 16w+16)
            float dv[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t af[4];
                ldsm4(af, addr_a(gs.kb, 16 * ks, lane));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t b0 = pack2(DT.x[2 * ks][2 * h], DT.x[2 * ks][2 * h + 1]);
                    const uint32_t b1 = pack2(DT.x[2 * ks + 1][2 * h], DT.x[2 * ks + 1][2 * h + 1]);
                    mma16816(dv[h], af, b0, b1);
                }
            }
            {
                uint32_t af[4], r4[4];
                ldsm4t(af, addr_at48(gs.amat, lane));
                ldsm4t(r4, addr_bt(s.dy, 16 * warp, lane));
                mma16816(dv[0], af, r4[0], r4[1]);
                mma16816(dv[1], af, r4[2], r4[3]);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = g + 8 * half, tok = t0 + r;
                if (tok < kp.T) {
                    __nv_bfloat16* row = a.dV + rm.base + (size_t)tok * rm.stride;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int v = 16 * warp + 8 * h + 2 * t;
                        if (v < kp.d) {
                            const uint32_t yw = *reinterpret_cast<const uint32_t*>(s.dy + swz(r, v));
                            *reinterpret_cast<uint32_t*>(row + v) =
                                pack2(lo_f(yw) + dv[h][2 * half], hi_f(yw) + dv[h][2 * half + 1]);
                        }
                    }
                }
            }
            // dC <- Diag(a) dC + (q . F)^T dE, in both layouts
            const float a0 = gs.avec[16 * warp + g], a1 = gs.avec[16 * warp + 8 + g];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                DC.x[nt][0] *= a0;
                DC.x[nt][1] *= a0;
                DC.x[nt][2] *= a1;
                DC.x[nt][3] *= a1;
                const float2 ac = *reinterpret_cast<const float2*>(gs.avec + 8 * nt + 2 * t);
                DT.x[nt][0] *= ac.x;
                DT.x[nt][1] *= ac.y;
                DT.x[nt][2] *= ac.x;
                DT.x[nt][3] *= ac.y;
            }
            uint32_t aq[4], ad[4];
            ldsm4t(aq, addr_at(gs.qt, 16 * warp, lane));
            ldsm4t(ad, addr_at(s.dy, 16 * warp, lane));
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t r4[4];
                ldsm4t(r4, addr_bt(s.dy, 16 * p, lane));
                mma16816(DC.x[2 * p], aq, r4[0], r4[1]);
                mma16816(DC.x[2 * p + 1], aq, r4[2], r4[3]);
                ldsm4t(r4, addr_bt(gs.qt, 16 * p, lane));
                mma16816(DT.x[2 * p], ad, r4[0], r4[1]);
                mma16816(DT.x[2 * p + 1], ad, r4[2], r4[3]);
            }
        }
        __syncthreads();  // B5
        // Channel layout: dk, then z = q . dq - k . dk and its suffix sums.
        float2 dkv[4], zs[4];
        float2 zq = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * warp + r;
            float2 dk = mul2(mul2(Q.b[r], T.suf), *reinterpret_cast<const float2*>(gs.xq + i * kXs + c));
#pragma unroll
            for (int lvl = 0; lvl < 4; ++lvl) {
                const int b = 3 - lvl;
                if (!is_query(i, b))
                    dk = fma2(key_factor(Q, T, warp, r, b),
                              *reinterpret_cast<const float2*>(gs.xl[lvl] + key_row(i, b) * kXs + c), dk);
            }
            dkv[r] = dk;
            const float s2 = gs.rs[i].y;
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(s.p2 + swz(i, c));
            const float2 k = make_float2(lo_f(w2) * s2, hi_f(w2) * s2);
            zs[r] = make_float2(xs[r].x - k.x * dk.x, xs[r].y - k.y * dk.y);
            zq = make_float2(zq.x + zs[r].x, zq.y + zs[r].y);
        }
        *reinterpret_cast<float2*>(&gs.zt[warp][c]) = zq;
        __syncthreads();  // B6
        float2 later = carry;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 zk = *reinterpret_cast<const float2*>(&gs.zt[k][c]);
            if (k > warp) later = make_float2(later.x + zk.x, later.y + zk.y);
            carry = make_float2(carry.x + zk.x, carry.y + zk.y);
        }
#pragma unroll
        for (int r = 3; r >= 0; --r) {
            const int i = 4 * warp + r, tok = t0 + i;
            later = make_float2(later.x + zs[r].x, later.y + zs[r].y);
            const float4 rn = gs.rn[i];
            const float s2 = gs.rs[i].y;
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(s.p1 + swz(i, c));
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(s.p2 + swz(i, c));
            const float2 p1 = make_float2(lo_f(w1), hi_f(w1)), p2 = make_float2(lo_f(w2), hi_f(w2));
            const float2 ph = make_float2(p2.x * rn.y, p2.y * rn.y);
            const float2 dk = dkv[r];
            float pd = ph.x * dk.x + ph.y * dk.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, o);
            if (tok < kp.T) {
                const size_t off = rm.base + (size_t)tok * rm.stride;
                const float S = rn.z;
                const float dz = (pq[r] + pd) * S * (1.f - S) * a.zscale;
                if (c < kp.d) {
                    float2 dg = later;
                    if (gc.on) {
                        // Chain rule through the gate: dg/dA_log = g, dg/dr = -exp(A_log) sigmoid(r + dt_bias).
                        const float2 rr = *reinterpret_cast<const float2*>(s.g + i * kDp + c);
                        const float2 gg = gate_g(rr, gc);
                        const float2 sg = make_float2(1.f / (1.f + __expf(-(rr.x + gc.db.x))),
                                                      1.f / (1.f + __expf(-(rr.y + gc.db.y))));
                        acc_dalog = make_float2(fmaf(later.x, gg.x, acc_dalog.x), fmaf(later.y, gg.y, acc_dalog.y));
                        dg = make_float2(later.x * gc.na.x * sg.x, later.y * gc.na.y * sg.y);
                        acc_ddtb = make_float2(acc_ddtb.x + dg.x, acc_ddtb.y + dg.y);
                    }
                    *reinterpret_cast<float2*>(a.dG + off + c) = dg;
                    *reinterpret_cast<uint32_t*>(a.dP1 + off + c) =
                        pack2(lo_f(p1w[r]) + dz * p2.x, hi_f(p1w[r]) + dz * p2.y);
                    *reinterpret_cast<uint32_t*>(a.dP2 + off + c) =
                        pack2(s2 * (dk.x - ph.x * pd) + dz * p1.x, s2 * (dk.y - ph.y * pd) + dz * p1.y);
                }
            }
        }
    }
    if (gc.on && c < kp.d) {
        const size_t o = (size_t)(bh % kp.H) * kp.d + c;
        atomicAdd(a.gate_dalog + o, acc_dalog.x);
        atomicAdd(a.gate_dalog + o + 1, acc_dalog.y);
        atomicAdd(a.gate_ddtb + o, acc_ddtb.x);
        atomicAdd(a.gate_ddtb + o + 1, acc_ddtb.y);
    }
}

}  // namespace lin

// ------------------------------------------------------------------ launchers
int linear_segments(const KernelProblem& kp, int num_sms, int* seg_len) {
    // Segments trade parallelism for an extra state pass over every token (about a
    // quarter of the output passes' work).  Pick the count that minimises
    // waves x chunks per segment x (1 + that overhead), with three resident CTAs per
    // SM and segments of at least 128 tokens.
    const int64_t slots = (int64_t)num_sms * 3;
    const int max_seg = (kp.T + 127) / 128;
    int best = 1;
    double best_cost = 0.0;
    for (int n = 1; n <= max_seg; ++n) {
        const int len = ((kp.T + n - 1) / n + lin::kC - 1) / lin::kC * lin::kC;
        const int nn = (kp.T + len - 1) / len;
        const double waves = (double)((kp.BH * nn + slots - 1) / slots);
        const double cost = waves * (double)(len / lin::kC) * (nn > 1 ? 1.25 : 1.0);
        if (n == 1 || cost < best_cost - 1e-9) {
            best = nn;
            best_cost = cost;
        }
    }
    int len = (kp.T + best - 1) / best;
    len = (len + lin::kC - 1) / lin::kC * lin::kC;
    *seg_len = len;
    return (kp.T + len - 1) / len;
}

namespace lin {
// The launches of one direction for one (row width, gate) instantiation; each sets
// its kernels' shared-memory limit once.
template <bool kVec16, bool kGate>
cudaError_t fwd_passes(const Args& a, float* state_out, cudaStream_t s) {
    const size_t smem = sizeof(GroupSmem);
    static bool attr_done = false;
    if (!attr_done) {
        cudaFuncSetAttribute(linear_fwd_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(linear_state_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        attr_done = true;
    }
    const unsigned grid = (unsigned)(a.kp.BH * a.nseg);
    const dim3 block(kThreads);
    if (a.nseg > 1) {
        linear_state_kernel<kVec16, kGate><<<grid, block, smem, s>>>(a);
        linear_scan_kernel<<<(unsigned)a.kp.BH * 16, 256, 0, s>>>(a.hseg, a.aseg, a.nseg, state_out, a.kp.d);
    }
    linear_fwd_kernel<kVec16, kGate><<<grid, block, smem, s>>>(a);
    return cudaGetLastError();
}

template <bool kVec16, bool kGate>
cudaError_t bwd_passes(const Args& fa, const BArgs& b, bool reuse_fwd_states, cudaStream_t s) {
    const size_t fsmem = sizeof(GroupSmem), bsmem = sizeof(BwdSmem);
    static bool attr_done = false;
    if (!attr_done) {
        cudaFuncSetAttribute(linear_state_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)fsmem);
        cudaFuncSetAttribute(linear_bstate_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bsmem);
        cudaFuncSetAttribute(linear_bwd_a_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bsmem);
        cudaFuncSetAttribute(linear_bwd_b_kernel<kVec16, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bsmem);
        attr_done = true;
    }
    const unsigned grid = (unsigned)(b.kp.BH * b.nseg);
    const dim3 block(kThreads);
    if (fa.nseg > 1) {
        if (!reuse_fwd_states) {
            linear_state_kernel<kVec16, kGate><<<grid, block, fsmem, s>>>(fa);
            linear_scan_kernel<<<(unsigned)fa.kp.BH * 16, 256, 0, s>>>(fa.hseg, fa.aseg, fa.nseg, nullptr, fa.kp.d);
        }
        linear_bstate_kernel<kVec16, kGate><<<grid, block, bsmem, s>>>(b);
        linear_bscan_kernel<<<(unsigned)b.kp.BH * 16, 256, 0, s>>>(b.dcseg, b.aseg, b.nseg);
    }
    linear_bwd_a_kernel<kVec16, kGate><<<grid, block, bsmem, s>>>(b);
    linear_bwd_b_kernel<kVec16, kGate><<<grid, block, bsmem, s>>>(b);
    return cudaGetLastError();
}
}  // namespace lin

cudaError_t launch_linear_fwd(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* G,
                              void* Y, float* state_out, float* ws, int num_sms, cudaStream_t s, const float* gate_alog,
                              const float* gate_dtb) {
    lin::Args a;
    a.gate_alog = gate_alog;
    a.gate_dtb = gate_dtb;
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
    const bool vec16 = (kp.d % 8) == 0, gate = gate_alog != nullptr;
    if (vec16)
        return gate ? lin::fwd_passes<true, true>(a, state_out, s) : lin::fwd_passes<true, false>(a, state_out, s);
    return gate ? lin::fwd_passes<false, true>(a, state_out, s) : lin::fwd_passes<false, false>(a, state_out, s);
}

cudaError_t launch_linear_bwd(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* G,
                              const void* dY, void* dP1, void* dP2, void* dV, float* dG, bool reuse_fwd_states,
                              float* ws, int num_sms, cudaStream_t s, const float* gate_alog, const float* gate_dtb,
                              float* gate_dalog, float* gate_ddtb) {
    lin::Args fa;
    fa.gate_alog = gate_alog;
    fa.gate_dtb = gate_dtb;
    fa.P1 = static_cast<const __nv_bfloat16*>(P1);
    fa.P2 = static_cast<const __nv_bfloat16*>(P2);
    fa.V = static_cast<const __nv_bfloat16*>(V);
    fa.G = G;
    fa.Y = nullptr;
    fa.state_out = nullptr;
    fa.kp = kp;
    fa.zscale = kp.inv_sqrt_d / kp.tau_S;
    fa.nseg = linear_segments(kp, num_sms, &fa.seg_len);
    const size_t per_seg = (size_t)kp.BH * fa.nseg;
    fa.hseg = ws;
    fa.aseg = ws + per_seg * lin::kDp * lin::kDp;
    lin::BArgs b;
    b.gate_alog = gate_alog;
    b.gate_dtb = gate_dtb;
    b.gate_dalog = gate_dalog;
    b.gate_ddtb = gate_ddtb;
    b.P1 = fa.P1;
    b.P2 = fa.P2;
    b.V = fa.V;
    b.G = G;
    b.dY = static_cast<const __nv_bfloat16*>(dY);
    b.dP1 = static_cast<__nv_bfloat16*>(dP1);
    b.dP2 = static_cast<__nv_bfloat16*>(dP2);
    b.dV = static_cast<__nv_bfloat16*>(dV);
    b.dG = dG;
    b.hseg = fa.hseg;
    b.aseg = fa.aseg;
    b.dcseg = fa.aseg + per_seg * lin::kDp;
    b.pdq = b.dcseg + per_seg * lin::kDp * lin::kDp;
    b.kp = kp;
    b.zscale = fa.zscale;
    b.nseg = fa.nseg;
    b.seg_len = fa.seg_len;
    const bool vec16 = (kp.d % 8) == 0, gate = gate_alog != nullptr;
    if (vec16)
        return gate ? lin::bwd_passes<true, true>(fa, b, reuse_fwd_states, s)
                    : lin::bwd_passes<true, false>(fa, b, reuse_fwd_states, s);
    return gate ? lin::bwd_passes<false, true>(fa, b, reuse_fwd_states, s)
                : lin::bwd_passes<false, false>(fa, b, reuse_fwd_states, s);
}

}  // namespace relation

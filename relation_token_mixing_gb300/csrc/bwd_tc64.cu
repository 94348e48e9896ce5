// Fused Full Relation backward for head width 64 on the sm_103a tensor cores:
// the pipelined variant of the key-stationary backward (bf16 in, fp32 accumulate).
//
// Mathematics: the chain rule of "Ask Self, Ask Others: Relation Is All You
// Need", Sec. 3.1 eq.(1)-(3) (the paper gives no backward), with
// F_ij = exp(R_ij - L_i) rebuilt from the forward's log-normaliser:
//   dR_ij = F_ij (dY_i . V_j - D_i),  dU_ij = dR_ij * slope_ij,
//   slope_ii = S_i (1 - S_i) / tau_S,   slope_ij = SiLU'(U_ij) = s (1 + U (1 - s)),
//   dP1 = dU P2 / 8, dP2 = dU^T P1 / 8 (1/sqrt(64)), dV = F^T dY.
// With t = tanh(U/2):  s = (1 + t)/2 and SiLU'(U) = (1 + t + (U/2)(1 - t^2)) / 2,
// so one MUFU tanh serves both SiLU (forward value) and its slope.
//
// One CTA = one head x one 128-row key tile; it walks the query tiles i that
// see it.  Each query tile is processed as two 64-column halves so that the
// two elementwise warpgroups and the tensor core ping-pong:
//   tensor core:  S_lo dP_lo | S_hi dP_hi | dV,dP2 += lo | S_lo dP_lo (i+1) | dV,dP2 += hi, dP1(i) | S_hi dP_hi (i+1)
//   WG lo:                   |  lo(i)                     |                  lo(i+1) ...
//   WG hi:                                 |  hi(i)                          |  hi(i+1) ...
// Warps: 0 loader (TMA + per-query constants), 1 MMA issuer / TMEM owner,
// 2-3 idle (complete the first warpgroup), 4-7 elementwise for query columns
// 0-63, 8-11 for columns 64-127, 12-15 dP1 reduction (TMEM -> fp32
// accumulator in global memory, atomics).
// TMEM: S^T [0,128) | dP^T [128,256) | dV [256,320) | dP2 [320,384) | dP1 part [384,448).
// P^T and dS^T (bf16) overwrite the first half of each S^T / dP^T half they came from.
// dS^T also goes to shared memory (double-buffered) as the MN-major A operand
// of dP1 = dS P2.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx_sm100.cuh"
#include "tmap.h"

namespace relation {
namespace {

constexpr int kD = 64;
constexpr int kTile = 128;
constexpr int kThreads = 512;
// Register split after launch at 128 per thread: load/MMA warpgroup 56, the two
// elementwise warpgroups 176, the dP1-reduce warpgroup 88:
// 128*56 + 256*176 + 128*88 = 63488 <= 512*128.
constexpr uint32_t kRegsControl = 56, kRegsElementwise = 176, kRegsReduce = 88;
constexpr int kTileBytes = kTile * kD * 2;  // 16 KB: one 128-row x 128-byte swizzled panel
constexpr int kHalfBytes = kTileBytes / 2;  // 64 rows
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384;

struct Smem {
    uint8_t k[kTileBytes];        // P2_j
    uint8_t v[kTileBytes];        // V_j
    uint8_t q[2][kTileBytes];     // P1_i, two stages
    uint8_t g[2][kTileBytes];     // dY_i, two stages
    uint8_t ds[2][2 * kTileBytes];  // dS^T, two buffers of two 64-query panels
    float neg_lt[2][kTile];       // -(L_q + lambda log c_q) * log2(e)
    float neg_dk[2][kTile];       // -D_q * (1/2) / sqrt(d)
    uint64_t kv_full;
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t ds_free[2];
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
// Alignment slack and a 16 KB guard band after the tiles.
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024 + 16384;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > RELATION_WAIT_LIMIT_NS) return;
    }
}

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {  // K-major, 128-byte swizzle
    return ptx::smem_desc(addr, 16, 1024, ptx::kSwizzle128B);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t addr) {  // MN-major, 128-byte swizzle, 64-wide panels 16 KB apart
    return ptx::smem_desc(addr, kTileBytes, 1024, ptx::kSwizzle128B);
}

// Per-thread constants of the elementwise stage.
struct ElemConst {
    float2 c_nh, c_hl, k2, one, mone;
    float c_diag, half_inv_tau, diag_off, log_count;
    bool row_valid, causal;
};

// Elementwise stage for one 64-column half of a query tile, one key row per
// thread: P^T and dS^T (scaled by 1/sqrt(d)) to TMEM over the consumed
// columns, dS^T to the shared-memory row.  kMasked selects the variant with
// the diagonal Self entry and masking; the plain variant has no branches so
// that the 32 independent element pairs of a chunk interleave.
template <bool kMasked>
__device__ __forceinline__ void elementwise_half(const uint32_t (&sv)[64], const uint32_t (&gv)[64],
                                                 const float* nlt, const float* ndk, uint32_t lane_addr, int h,
                                                 int r, uint8_t* ds_row, const ElemConst& ec, bool diag_tile,
                                                 int qlimit, float* dlam) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int cc0 = 32 * c + 2 * e;  // column within the half
            const float2 a = make_float2(as_f(sv[cc0]), as_f(sv[cc0 + 1]));
            const float2 g = make_float2(as_f(gv[cc0]), as_f(gv[cc0 + 1]));
            const float2 nh = ptx::mul2(a, ec.c_nh);
            const float2 nt = make_float2(ptx::tanh_approx(nh.x), ptx::tanh_approx(nh.y));
            const float2 tp1 = ptx::fma2(nt, ec.mone, ec.one);
            const float2 hl = ptx::mul2(a, ec.c_hl);
            const float2 x = ptx::fma2(hl, tp1, *reinterpret_cast<const float2*>(nlt + cc0));
            float2 p = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
            const float2 nq = ptx::fma2(nt, nt, ec.mone);
            float2 s2 = ptx::fma2(nh, nq, tp1);
            const float2 gk = ptx::fma2(g, ec.k2, *reinterpret_cast<const float2*>(ndk + cc0));
            if (kMasked) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int cc = cc0 + u;
                    const int col = 64 * h + cc;  // column within the query tile
                    float& pu = u ? p.y : p.x;
                    float& su = u ? s2.y : s2.x;
                    if (diag_tile && col == r && ec.row_valid) {
                        const float aa = u ? a.y : a.x;
                        const float td = ptx::tanh_approx(aa * ec.c_diag);
                        pu = ptx::ex2_approx(fmaf(0.5f * kLog2e, td, ec.diag_off + nlt[cc]));
                        su = fmaf(-td, td, 1.f) * ec.half_inv_tau;  // 2 S(1-S)/tau_S
                        *dlam += ec.log_count * pu * (u ? gk.y : gk.x);
                    }
                    if (cc >= qlimit || !ec.row_valid || (ec.causal && diag_tile && col < r)) pu = 0.f;
                }
            }
            const float2 dr = ptx::mul2(p, gk);
            const float2 ds = ptx::mul2(dr, s2);
            pp[e] = ptx::pack_bf16x2(p.x, p.y);
            dd[e] = ptx::pack_bf16x2(ds.x, ds.y);
        }
        // P^T and dS^T over already-read columns of this half.
        ptx::tmem_st16(lane_addr + kColS + 64 * h + 16 * c, pp);
        ptx::tmem_st16(lane_addr + kColDP + 64 * h + 16 * c, dd);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int chunk = 4 * c + k4;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(dd[4 * k4], dd[4 * k4 + 1], dd[4 * k4 + 2], dd[4 * k4 + 3]);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    relation_bwd_tc64_kernel(const __grid_constant__ CUtensorMap tm_p1, const __grid_constant__ CUtensorMap tm_p2,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                             const KernelProblem kp, const float* __restrict__ L, const float* __restrict__ Dw,
                             float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dP2,
                             __nv_bfloat16* __restrict__ dV, float* __restrict__ dlambda, unsigned int* status) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int jt = blockIdx.y;
    const int T = kp.T;
    const int kv0 = jt * kTile;
    const int nq_all = (T + kTile - 1) / kTile;
    const int i_first = kp.causal ? jt : 0;
    const int n_q = nq_all - i_first;
    const float k_scale = 0.5f * kp.inv_sqrt_d;

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sm.q_full[s], 32);
            ptx::mbar_init(&sm.q_empty[s], 1);
            ptx::mbar_init(&sm.s_full[s], 1);
            ptx::mbar_init(&sm.p_full[s], 128);
            ptx::mbar_init(&sm.ds_free[s], 1);
        }
        ptx::mbar_init(&sm.dq_full, 1);
        ptx::mbar_init(&sm.dq_free, 128);
        ptx::mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&sm.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int* abort_flag = &sm.abort_flag;

    if (warp == 0) {
        // -------------------------------------------------------------- loader
        ptx::regs_dec<kRegsControl>();
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_p1);
            ptx::tma_prefetch_desc(&tm_p2);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_dy);
            ptx::mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
            ptx::tma_load_3d(sm.k, &tm_p2, &sm.kv_full, 0, kv0, bh);
            ptx::tma_load_3d(sm.v, &tm_v, &sm.kv_full, 0, kv0, bh);
        }
        int it = 0;
        for (; it < n_q; ++it) {
            const int s = it & 1;
            const int i = i_first + it;
            // Global loads first: they do not depend on the stage being free.
            float nlt[4], ndk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int q = i * kTile + lane + 32 * k;
                nlt[k] = 0.f;
                ndk[k] = 0.f;
                if (q < T) {
                    const int count = kp.causal ? (q + 1) : T;
                    nlt[k] = -(L[(size_t)bh * T + q] + kp.lambda * __logf((float)count)) * kLog2e;
                    ndk[k] = -Dw[(size_t)bh * T + q] * k_scale;
                }
            }
            if (it >= 2 &&
                !ptx::mbar_wait_warp(&sm.q_empty[s], ((it >> 1) - 1) & 1, abort_flag, status, kDevTimeoutEmpty))
                break;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sm.neg_lt[s][lane + 32 * k] = nlt[k];
                sm.neg_dk[s][lane + 32 * k] = ndk[k];
            }
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(&sm.q_full[s], 2 * kTileBytes);
                ptx::tma_load_3d(sm.q[s], &tm_p1, &sm.q_full[s], 0, i * kTile, bh);
                ptx::tma_load_3d(sm.g[s], &tm_dy, &sm.q_full[s], 0, i * kTile, bh);
            } else {
                ptx::mbar_arrive(&sm.q_full[s]);
            }
        }
        if (lane == 0 && *abort_flag) {
            drain_wait(&sm.kv_full, 0);
            for (int jj = max(0, it - 2); jj < it; ++jj) drain_wait(&sm.q_full[jj & 1], (jj >> 1) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        ptx::regs_dec<kRegsControl>();
        if (lane == 0) {
            const uint32_t id_half = ptx::idesc_bf16(kTile, 64, false, false);  // S^T, dP^T halves (N = 64)
            const uint32_t id_acc = ptx::idesc_bf16(kTile, kD, false, true);    // dV, dP2 (B MN-major)
            const uint32_t id_dq = ptx::idesc_bf16(kTile, kD, true, true);      // dP1 (A, B MN-major)
            const uint32_t ka = ptx::smem_u32(sm.k), va = ptx::smem_u32(sm.v);
            auto issue_s_dp = [&](int it, int h) {
                const int s = it & 1;
                const uint32_t qa = ptx::smem_u32(sm.q[s]) + h * kHalfBytes;
                const uint32_t ga = ptx::smem_u32(sm.g[s]) + h * kHalfBytes;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    ptx::mma_ss(tmem + kColS + 64 * h, kdesc(ka + ks * 32), kdesc(qa + ks * 32), id_half,
                                ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    ptx::mma_ss(tmem + kColDP + 64 * h, kdesc(va + ks * 32), kdesc(ga + ks * 32), id_half,
                                ks > 0 ? 1u : 0u);
                ptx::mma_commit(&sm.s_full[h]);
            };
            auto issue_acc = [&](int it, int h) {
                const int s = it & 1;
                const uint32_t qa = ptx::smem_u32(sm.q[s]) + h * kHalfBytes;
                const uint32_t ga = ptx::smem_u32(sm.g[s]) + h * kHalfBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    ptx::mma_ts(tmem + kColDV, tmem + kColS + 64 * h + 8 * ks, mdesc(ga + ks * 2048), id_acc,
                                (it > 0 || h > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    ptx::mma_ts(tmem + kColDK, tmem + kColDP + 64 * h + 8 * ks, mdesc(qa + ks * 2048), id_acc,
                                (it > 0 || h > 0 || ks > 0) ? 1u : 0u);
            };
            bool ok = ptx::mbar_wait(&sm.kv_full, 0, abort_flag, status, kDevTimeoutFull);
            if (ok && n_q > 0) ok = ptx::mbar_wait(&sm.q_full[0], 0, abort_flag, status, kDevTimeoutFull);
            if (ok && n_q > 0) {
                ptx::tc_fence_after();
                issue_s_dp(0, 0);
                issue_s_dp(0, 1);
            }
            for (int it = 0; ok && it < n_q; ++it) {
                const bool more = it + 1 < n_q;
                // low half of query tile it
                if (!ptx::mbar_wait(&sm.p_full[0], it & 1, abort_flag, status, kDevTimeoutFull)) break;
                ptx::tc_fence_after();
                issue_acc(it, 0);
                if (more) {
                    if (!ptx::mbar_wait(&sm.q_full[(it + 1) & 1], ((it + 1) >> 1) & 1, abort_flag, status,
                                        kDevTimeoutFull))
                        break;
                    ptx::tc_fence_after();
                    issue_s_dp(it + 1, 0);
                }
                // high half, then dP1 for the whole tile
                if (!ptx::mbar_wait(&sm.p_full[1], it & 1, abort_flag, status, kDevTimeoutFull)) break;
                ptx::tc_fence_after();
                issue_acc(it, 1);
                if (it > 0 && !ptx::mbar_wait(&sm.dq_free, (it - 1) & 1, abort_flag, status, kDevTimeoutMma)) break;
                const uint32_t dsa = ptx::smem_u32(sm.ds[it & 1]);
#pragma unroll
                for (int ks = 0; ks < kTile / 16; ++ks)
                    ptx::mma_ss(tmem + kColDQ, mdesc(dsa + ks * 2048), mdesc(ka + ks * 2048), id_dq, ks > 0 ? 1u : 0u);
                ptx::mma_commit(&sm.dq_full);
                ptx::mma_commit(&sm.ds_free[it & 1]);
                ptx::mma_commit(&sm.q_empty[it & 1]);
                if (more) issue_s_dp(it + 1, 1);
            }
            ptx::mma_commit(&sm.mma_done);
            drain_wait(&sm.mma_done, 0);
        }
    } else if (warp < 4) {
        ptx::regs_dec<kRegsControl>();
    } else if (warp < 12) {
        // --------------------------------------------------- elementwise halves
        ptx::regs_inc<kRegsElementwise>();
        const int h = (warp - 4) >> 2;  // query columns 64h .. 64h+63
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key row within the tile
        const int kv = kv0 + r;
        const bool row_valid = kv < T;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        // Signs are folded into the constants so that no negation is issued:
        // nh = -U/2, nt = tanh(nh) = -t, tp1 = 1 + t, nq = t^2 - 1, s2 = tp1 + nh*nq.
        ElemConst ec;
        ec.c_nh = make_float2(-0.5f * kp.inv_sqrt_d, -0.5f * kp.inv_sqrt_d);
        ec.c_hl = make_float2(0.5f * kp.inv_sqrt_d * kLog2e, 0.5f * kp.inv_sqrt_d * kLog2e);
        ec.k2 = make_float2(k_scale, k_scale);
        ec.one = make_float2(1.f, 1.f);
        ec.mone = make_float2(-1.f, -1.f);
        ec.c_diag = 0.5f * kp.inv_sqrt_d / kp.tau_S;
        ec.half_inv_tau = 0.5f / kp.tau_S;
        const int count_kv = kp.causal ? (kv + 1) : T;
        ec.log_count = __logf((float)count_kv);
        ec.diag_off = (0.5f + kp.lambda * ec.log_count) * kLog2e;  // (1/2 + lambda log c) log2(e)
        ec.row_valid = row_valid;
        ec.causal = kp.causal != 0;
        float dlam = 0.f;
        bool ok = true;
        for (int it = 0; ok && it < n_q; ++it) {
            const int s = it & 1;
            const int i = i_first + it;
            if (!ptx::mbar_wait_warp(&sm.s_full[h], it & 1, abort_flag, status, kDevTimeoutMma) ||
                !ptx::mbar_wait_warp(&sm.q_full[s], (it >> 1) & 1, abort_flag, status, kDevTimeoutFull) ||
                (it >= 2 &&
                 !ptx::mbar_wait_warp(&sm.ds_free[s], ((it >> 1) - 1) & 1, abort_flag, status, kDevTimeoutMma))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t sv[64], gv[64];
            ptx::tmem_ld32(lane_addr + kColS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(sv));
            ptx::tmem_ld32(lane_addr + kColS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
            ptx::tmem_ld32(lane_addr + kColDP + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(gv));
            ptx::tmem_ld32(lane_addr + kColDP + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(gv + 32));
            ptx::tmem_ld_wait();
            ptx::pin_regs(sv);
            ptx::pin_regs(gv);
            const float* nlt = sm.neg_lt[s] + 64 * h;
            const float* ndk = sm.neg_dk[s] + 64 * h;
            const bool diag_tile = (i == jt);
            const int qlimit = T - i * kTile - 64 * h;  // columns cc < qlimit hold queries < T
            // The two bodies contain warp-collective TMEM stores, so the choice must be
            // warp-uniform: a warp takes the masked body if any of its rows needs it.
            const bool special = __any_sync(0xffffffffu, diag_tile || qlimit < 64 || !row_valid);
            uint8_t* ds_row = sm.ds[s] + h * kTileBytes + r * 128;
            if (!special) {
                elementwise_half<false>(sv, gv, nlt, ndk, lane_addr, h, r, ds_row, ec, false, 0, &dlam);
            } else {
                elementwise_half<true>(sv, gv, nlt, ndk, lane_addr, h, r, ds_row, ec, diag_tile, qlimit, &dlam);
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.p_full[h]);
        }
        if (dlambda != nullptr) {
            // dR_ii = p (g - D) = dr / k_scale; sum log(c_i) dR_ii.
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, o);
            if (lane == 0 && dlam != 0.f) atomicAdd(dlambda, dlam / k_scale);
        }
        // Epilogue: warpgroup 0 writes dV rows, warpgroup 1 writes dP2 rows.
        if (ok && ptx::mbar_wait_warp(&sm.mma_done, 0, abort_flag, status, kDevTimeoutMma)) {
            ptx::tc_fence_after();
            __nv_bfloat16* dst_row = (h == 0 ? dV : dP2) + ((size_t)bh * T + kv) * kD;
            const uint32_t col = h == 0 ? kColDV : kColDK;
#pragma unroll
            for (int c0 = 0; c0 < kD / 32; ++c0) {
                uint32_t ov[32];
                ptx::tmem_ld32(lane_addr + col + 32 * c0, ov);
                ptx::tmem_ld_wait();
                ptx::pin_regs(ov);
                if (row_valid) {
                    uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(ptx::pack_bf16x2(as_f(ov[8 * k + 0]), as_f(ov[8 * k + 1])),
                                            ptx::pack_bf16x2(as_f(ov[8 * k + 2]), as_f(ov[8 * k + 3])),
                                            ptx::pack_bf16x2(as_f(ov[8 * k + 4]), as_f(ov[8 * k + 5])),
                                            ptx::pack_bf16x2(as_f(ov[8 * k + 6]), as_f(ov[8 * k + 7])));
                }
            }
        }
    } else {
        // -------------------------------------------------- dP1 partial reduce
        ptx::regs_dec<kRegsReduce>();
        const int quarter = warp & 3;
        const int rq = quarter * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        for (int it = 0; it < n_q; ++it) {
            const int i = i_first + it;
            if (!ptx::mbar_wait_warp(&sm.dq_full, it & 1, abort_flag, status, kDevTimeoutMma)) break;
            ptx::tc_fence_after();
            const int q = i * kTile + rq;
            uint32_t ov[2][32];
            ptx::tmem_ld32(lane_addr + kColDQ, ov[0]);
            ptx::tmem_ld32(lane_addr + kColDQ + 32, ov[1]);
            ptx::tmem_ld_wait();
            ptx::pin_regs(ov[0]);
            ptx::pin_regs(ov[1]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.dq_free);  // TMEM copy is in registers; the next dP1 MMA may start
            if (q < T) {
                float4* dst = reinterpret_cast<float4*>(dq_acc + ((size_t)bh * T + q) * kD);
#pragma unroll
                for (int c0 = 0; c0 < 2; ++c0)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        atomicAdd(dst + 8 * c0 + k, make_float4(as_f(ov[c0][4 * k]), as_f(ov[c0][4 * k + 1]),
                                                                as_f(ov[c0][4 * k + 2]), as_f(ov[c0][4 * k + 3])));
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_bwd_tc64(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* L,
                            const float* Dw, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                            const TcLaunch& tl, cudaStream_t s) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(relation_bwd_tc64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap m1, m2, mv, mg;
    const void* bases[4] = {P1, P2, V, dY};
    CUtensorMap* maps[4] = {&m1, &m2, &mv, &mg};
    for (int k = 0; k < 4; ++k) {
        cudaError_t e = make_tensor_map_3d(maps[k], bases[k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, kp.T, kp.BH,
                                           64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)kp.BH, (unsigned)((kp.T + kTile - 1) / kTile));
    relation_bwd_tc64_kernel<<<grid, kThreads, kSmemBytes, s>>>(m1, m2, mv, mg, kp, L, Dw, dq_acc,
                                                                (__nv_bfloat16*)dP2, (__nv_bfloat16*)dV, dlambda,
                                                                tl.status);
    return cudaGetLastError();
}

}  // namespace relation

// Fused Full Relation backward for head width 64 on the sm_103a tensor cores
// (bf16 in, fp32 accumulate): key-stationary, with the tensor core and the
// elementwise stage overlapped across query tiles.
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
// Work unit = one head x one 128-row key tile, walking the query tiles i that
// see it; the grid has one CTA per unit, and a CTA goes on with the units of
// CTAs not launched yet (launch control, below), so at most one CTA per SM runs
// the grid.  Per query tile (everything transposed so key rows sit on TMEM lanes):
//   S^T = P2_j P1_i^T, dP^T = V_j dY_i^T        (SS, two N = 64 halves each)
//   elementwise: P^T -> TMEM (bf16), dS^T = dU^T/8 -> shared memory (bf16)
//   dV  += P^T dY_i     (TS)
//   dP2 += dS^T P1_i    (SS, dS^T read K-major from shared memory)
//   dP1_i = dS P2_j     (SS, dS read MN-major from the same bytes), then added
//                       to an fp32 accumulator in global memory by TMA bulk reduce
// S^T and dP^T are produced and consumed in two halves of 64 queries with their
// own full/free barriers.  Every elementwise warp copies its part of a half to
// registers before working on it, so the first MMA warp issues that half of tile
// i+1 right away: the products of tile i+1 run while tile i is still being
// worked on, and the accumulations of tile i (issued by the second MMA warp as
// soon as its P^T and dS^T are stored) run while tile i+1 is.
// Warps: 0 loader (TMA + per-query constants), 1-2 MMA issuers (1: S^T/dP^T,
// also TMEM owner; 2: dV, dP2, dP1), 3 idle (completes the first warpgroup),
// 4-19 elementwise: four warpgroups, one per 16 query columns of each half,
// 20-23 dP1 reduction (TMEM -> swizzled shared staging -> TMA reduce-add).
// TMEM: S^T [0,128) | dP^T [128,256) | P^T [256,320) | dV [320,384) | dP2 [384,448) | dP1 part [448,512).
#include <cuda_bf16.h>

#include "bwd_elementwise.cuh"
#include "kernels.h"
#include "prologue_tiles.cuh"
#include "ptx_sm100.cuh"
#include "tmap.h"

namespace relation {
namespace {

using bwd_elem::ElemConst;
using bwd_elem::elementwise16;

constexpr int kD = 64;
constexpr int kTile = 128;
constexpr int kThreads = 768;
constexpr int kElemWarps = 16;
// Register split after launch at 80 per thread (six warps per SM sub-partition):
// load/MMA warpgroup 56, the four elementwise warpgroups 88, the dP1-reduce
// warpgroup 56:  128*56 + 512*88 + 128*56 = 59392 <= 768*80.
constexpr uint32_t kRegsControl = 56, kRegsElementwise = 88, kRegsReduce = 56;
constexpr int kTileBytes = kTile * kD * 2;  // 16 KB: one 128-row x 128-byte swizzled panel
constexpr uint32_t kQConstBytes = kTile / 2 * 16;  // per-query constants of one query tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDV = 320, kColDK = 384, kColDQ = 448;
// Depth of the P1/dY ring: loads for tile i+2 are in flight while tile i is processed.
constexpr int kQStages = 3;

struct Smem {
    uint8_t k[kTileBytes];            // P2_j
    uint8_t v[kTileBytes];            // V_j
    uint8_t q[kQStages][kTileBytes];  // P1_i ring
    uint8_t g[kQStages][kTileBytes];  // dY_i ring
    uint8_t ds[2][2 * kTileBytes];    // dS^T, two buffers of two 64-query panels
    uint8_t dq_stage[kTileBytes];     // one 32-column panel of the dP1 partial, fp32 [128][32], swizzled
    // Per-query constants, interleaved per column pair (2c, 2c+1):
    // { -(L + lambda log c) log2(e) [2c], [2c+1],  -D (1/2)/sqrt(d) [2c], [2c+1] },
    // brought in with P1_i and dY_i (written by the preparation stage).
    float4 qconst[kQStages][kTile / 2];
    uint4 clc_resp[2];  // launch-control answers (the key tile after the current one)
    uint64_t kv_full;
    uint64_t kv_rot;              // fused prologue: P2_j rotated and V_j mixed
    uint64_t q_rot[kQStages];     // fused prologue: P1_i rotated
    uint64_t q_full[kQStages];
    uint64_t q_empty[kQStages];
    uint64_t s_full[2];  // S^T / dP^T of query half h (columns 64h..64h+63) computed
    uint64_t s_free[2];  // ... and read by every elementwise warp
    uint64_t p_full;
    uint64_t pv_done;
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t mma_done[2];  // per MMA issuer: all of its products complete
    uint64_t acc_done;     // dV and dP2 of the key tile final (its last tile's accumulations complete)
    uint64_t kv_free;      // both MMA issuers have finished reading the key tile's P2_j and V_j
    uint64_t clc_full[2];  // launch-control answer in clc_resp[slot]
    uint64_t clc_empty[2]; // ... read by every reading warp
    uint32_t tmem_base;
    int abort_flag;
};
// Alignment slack.
constexpr int kSmemBytes = (int)sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {  // K-major, 128-byte swizzle
    return ptx::smem_desc(addr, 16, 1024, ptx::kSwizzle128B);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t addr) {  // MN-major, 128-byte swizzle, 64-wide panels 16 KB apart
    return ptx::smem_desc(addr, kTileBytes, 1024, ptx::kSwizzle128B);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Operand loads: TMA through 3-D maps ([B, H, T, d] layout and the zero-padded
// copies of widths whose rows TMA cannot address) or 4-D maps ([B, T, H, d]).
enum LoadMode { kLoadTma3 = 0, kLoadTma4 = 1 };

// One unit of work: key tile jt of head bh and the query tiles i_first.. that see it.
struct KeyTile {
    int bh, jt, batch, head, kv0, i_first, n_q;
};
__device__ __forceinline__ KeyTile key_tile(int idx, const KernelProblem& kp, int nt_all, int head_group) {
    KeyTile w;
    grouped_tile_order((unsigned)idx, kp.BH, nt_all, head_group, w.bh, w.jt);
    w.batch = w.bh / kp.H;
    w.head = w.bh - w.batch * kp.H;
    w.kv0 = w.jt * kTile;
    w.i_first = kp.causal ? w.jt : 0;
    w.n_q = nt_all - w.i_first;
    return w;
}

// Warps that read each launch-control answer: all but warp 3.
constexpr int kClcReaders = kThreads / 32 - 1;

// The grid has one CTA per key tile (heads in L2-sized groups; causal: low key
// tiles, with the most query tiles, first).  A CTA that has issued the loads of
// its key tile's last query tile asks the scheduler for the key tile of a CTA not
// launched yet (launch control) and goes on with it: the next key tile's loads
// and first products overlap the current one's last products, its dP1 drain and
// its dV/dP2 epilogue, and no CTA launch separates them.  Every role walks the
// same sequence of key tiles; ring stages and barrier phases count the query
// tiles of all of them.
// kPro: the operands are the prologue's inputs X1, X2, I (d_h = 64): warp 3 rotates
// the key tile and mixes the V tile with the pair partner's (loaded into the dP1
// staging panel, which is free until the first dP1 drain); the four dP1-reduce
// warps rotate each query tile two tiles ahead.  dP2 leaves the epilogue
// un-rotated (dX2); dV is the gradient of the mixed states, and the dP1
// accumulator stays in rotated coordinates (both finished by later passes).  Such
// a CTA does its own key tile only.
template <int kLoad, bool kPro = false>
__global__ void __launch_bounds__(kThreads, 1)
    relation_bwd_tc64_kernel(const __grid_constant__ CUtensorMap tm_p1, const __grid_constant__ CUtensorMap tm_p2,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                             const __grid_constant__ CUtensorMap tm_dq, const KernelProblem kp,
                             const float4* __restrict__ qconst, __nv_bfloat16* __restrict__ dP2,
                             __nv_bfloat16* __restrict__ dV, float* __restrict__ dlambda, unsigned int* status,
                             int head_group, const __grid_constant__ ProArgs pro) {
    constexpr bool kRank3 = kLoad == kLoadTma3;
    constexpr bool kSteal = !kPro;  // go on with key tiles of CTAs not launched yet
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = kp.T;
    const int nt_all = (T + kTile - 1) / kTile;
    const float k_scale = 0.5f * kp.inv_sqrt_d;
    const KeyTile w0 = key_tile((int)blockIdx.x, kp, nt_all, head_group);
    int partner = w0.head;
    float g_cs = 1.f, g_sn = 0.f;  // Givens coefficients of this head (fused prologue)
    if constexpr (kPro) partner = givens_coeffs(w0.head, kp.H, pro, &g_cs, &g_sn);
    const float pos_base = (kPro && pro.pos0 != nullptr) ? (float)pro.pos0[w0.batch] : 0.f;

    // Loads of key tile w, and of its query tile it (P1_i, dY_i and the per-query
    // constants of the head, 64 float4 = 1 KB per query tile) into ring stage
    // q % kQStages, q counting all query tiles of this CTA.
    auto issue_kv = [&](const KeyTile& w) {
        ptx::mbar_arrive_expect_tx(&sm.kv_full, (kPro ? 3 : 2) * kTileBytes);
        ptx::tma_load_operand(sm.k, &tm_p2, &sm.kv_full, 0, w.kv0, w.bh, w.head, w.batch, kRank3);
        ptx::tma_load_operand(sm.v, &tm_v, &sm.kv_full, 0, w.kv0, w.bh, w.head, w.batch, kRank3);
        if constexpr (kPro)  // the Givens partner's states, into the (still unused) dP1 staging panel
            ptx::tma_load_operand(sm.dq_stage, &tm_v, &sm.kv_full, 0, w.kv0, w.bh - w.head + partner, partner,
                                  w.batch, kRank3);
    };
    auto issue_q = [&](const KeyTile& w, int it, int q) {
        const int s = q % kQStages;
        const int i = w.i_first + it;
        const float4* qsrc = qconst + (size_t)w.bh * (size_t)(qconst_rows(T) / 2);
        ptx::mbar_arrive_expect_tx(&sm.q_full[s], 2 * kTileBytes + kQConstBytes);
        ptx::bulk_load(sm.qconst[s], qsrc + i * (kTile / 2), kQConstBytes, &sm.q_full[s]);
        ptx::tma_load_operand(sm.q[s], &tm_p1, &sm.q_full[s], 0, i * kTile, w.bh, w.head, w.batch, kRank3);
        ptx::tma_load_operand(sm.g[s], &tm_dy, &sm.q_full[s], 0, i * kTile, w.bh, w.head, w.batch, kRank3);
    };
    if (threadIdx.x == 0) {
        ptx::tma_prefetch_desc(&tm_p1);
        ptx::tma_prefetch_desc(&tm_p2);
        ptx::tma_prefetch_desc(&tm_v);
        ptx::tma_prefetch_desc(&tm_dy);
        ptx::tma_prefetch_desc(&tm_dq);
        ptx::mbar_init(&sm.kv_full, 1);
        ptx::mbar_init(&sm.kv_rot, 1);
        ptx::mbar_init(&sm.kv_free, 2);  // released by both MMA issuers
        for (int s = 0; s < kQStages; ++s) ptx::mbar_init(&sm.q_rot[s], 4);
        for (int s = 0; s < kQStages; ++s) {
            ptx::mbar_init(&sm.q_full[s], 1);
            ptx::mbar_init(&sm.q_empty[s], 2);  // released by both MMA issuers
        }
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(&sm.s_full[h], 1);
            ptx::mbar_init(&sm.s_free[h], kElemWarps);
            ptx::mbar_init(&sm.clc_full[h], 1);
            ptx::mbar_init(&sm.clc_empty[h], kClcReaders);
        }
        ptx::mbar_init(&sm.p_full, kElemWarps);
        ptx::mbar_init(&sm.pv_done, 1);
        ptx::mbar_init(&sm.dq_full, 1);
        ptx::mbar_init(&sm.dq_free, 128);
        ptx::mbar_init(&sm.mma_done[0], 1);
        ptx::mbar_init(&sm.mma_done[1], 1);
        ptx::mbar_init(&sm.acc_done, 1);
        sm.abort_flag = 0;
        ptx::fence_barrier_init();
        // The loads that need no free stage leave before the block-wide barrier (and
        // the TMEM allocation behind it): the key tile and its first query tiles.
        issue_kv(w0);
        for (int it = 0; it < w0.n_q && it < kQStages; ++it) issue_q(w0, it, it);
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

    // The key tile after this CTA's k-th (k from 0): the answer to the request
    // the loader made during the k-th, read by every reading warp, which then
    // releases its slot.  -1: none (or the wait gave up).
    auto next_tile = [&](int k) -> int {
        if constexpr (!kSteal) return -1;
        const int slot = k & 1;
        if (!ptx::mbar_wait_warp(&sm.clc_full[slot], (k >> 1) & 1, abort_flag, status, kDevTimeoutFull)) return -1;
        const int x = ptx::clc_cancelled_x(&sm.clc_resp[slot]);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.clc_empty[slot]);
        return x;
    };

    if (warp == 0) {
        // -------------------------------------------------------------- loader
        ptx::regs_dec<kRegsControl>();
        KeyTile w = w0;
        int q = w0.n_q < kQStages ? w0.n_q : kQStages;  // query tiles issued (the first ones at the start)
        int it = q;                                     // ... of the current key tile
        int k = 0;                                      // key tiles begun after the first
        bool ok = true, asked = false;                  // asked: a request whose answer is not read yet
        for (;;) {
            for (; it < w.n_q; ++it, ++q) {
                if (q >= kQStages && !ptx::mbar_wait_warp(&sm.q_empty[q % kQStages], ((q / kQStages) - 1) & 1,
                                                          abort_flag, status, kDevTimeoutEmpty)) {
                    ok = false;
                    break;
                }
                if (lane == 0) issue_q(w, it, q);
            }
            if (!ok || !kSteal) break;
            // Every load of this key tile is out: ask for the next key tile.
            const int slot = k & 1;
            if (k >= 2 && !ptx::mbar_wait_warp(&sm.clc_empty[slot], ((k - 2) >> 1) & 1, abort_flag, status,
                                               kDevTimeoutEmpty)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(&sm.clc_full[slot], 16);
                ptx::clc_try_cancel(&sm.clc_resp[slot], &sm.clc_full[slot]);
            }
            asked = true;
            const int nx = next_tile(k);
            if (*abort_flag) {
                ok = false;
                break;
            }
            asked = false;
            if (nx < 0) break;
            // Its operands replace this one's once both MMA issuers have finished reading them.
            if (!ptx::mbar_wait_warp(&sm.kv_free, k & 1, abort_flag, status, kDevTimeoutMma)) {
                ok = false;
                break;
            }
            w = key_tile(nx, kp, nt_all, head_group);
            ++k;
            it = 0;
            if (lane == 0) issue_kv(w);
        }
        if (lane == 0 && *abort_flag) {
            // Let the copies in flight land before the CTA's shared memory goes.
            ptx::mbar_drain(&sm.kv_full, k & 1, status);
            for (int jj = max(0, q - kQStages); jj < q; ++jj)
                ptx::mbar_drain(&sm.q_full[jj % kQStages], (jj / kQStages) & 1, status);
            if (asked) ptx::mbar_drain(&sm.clc_full[k & 1], (k >> 1) & 1, status);
        }
    } else if (warp == 1 || warp == 2) {
        // --------------------------------------------------------- MMA issuers
        // Two instruction streams, each a converged warp with an elected lane:
        //   warp 1: S^T and dP^T of the next query tile, per half, as soon as the
        //           elementwise warps hold that half of the current tile;
        //   warp 2: dV and dP2 of the current tile once its P^T and dS^T are
        //           stored, then its dP1 partial.
        // They write disjoint TMEM columns; the tensor core runs each stream's
        // products in issue order, and every hand-off between them goes through
        // the elementwise warps' barriers.
        ptx::regs_dec<kRegsControl>();
        const uint32_t hi_k = ptx::desc_hi(kdesc(ptx::smem_u32(sm.k)));
        const uint32_t hi_m = ptx::desc_hi(mdesc(ptx::smem_u32(sm.k)));
        constexpr uint32_t kStageQ = kTileBytes >> 4, kStageS = (2 * kTileBytes) >> 4, kHalfQ = (kTileBytes / 2) >> 4;
        bool ok = true;
        int n_q = w0.n_q;
        if (warp == 1) {
            const uint32_t id_s = ptx::idesc_bf16(kTile, kTile / 2, false, false);  // S^T, dP^T halves (N = 64)
            // Descriptor low words: start address >> 4 (plus the leading byte offset
            // field), advanced by (byte offset >> 4) per K-step.
            const uint32_t k_lo = ptx::desc_lo(kdesc(ptx::smem_u32(sm.k)));
            const uint32_t v_lo = ptx::desc_lo(kdesc(ptx::smem_u32(sm.v)));
            const uint32_t q_lo0 = ptx::desc_lo(kdesc(ptx::smem_u32(sm.q[0])));
            const uint32_t g_lo0 = ptx::desc_lo(kdesc(ptx::smem_u32(sm.g[0])));
            // S^T and dP^T of query half h (64 queries): N = 64 products into columns
            // 64h..64h+63 of their regions; B starts 64 rows (8 KB) into the tile.
            auto issue_s_dp = [&](int qs, int h) {
                const uint32_t q_lo = q_lo0 + qs * kStageQ + h * kHalfQ, g_lo = g_lo0 + qs * kStageQ + h * kHalfQ;
                // K-step ks: 32-byte step inside the 128-byte swizzled rows.
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    ptx::mma_ss_elect(tmem + kColS + 64 * h, k_lo + 2 * ks, hi_k, q_lo + 2 * ks, hi_k, id_s,
                                      ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    ptx::mma_ss_elect(tmem + kColDP + 64 * h, v_lo + 2 * ks, hi_k, g_lo + 2 * ks, hi_k, id_s,
                                      ks > 0 ? 1u : 0u);
                ptx::mma_commit_elect(&sm.s_full[h]);
            };
            for (int k = 0, q = 0; ok; ++k) {
                ok = ptx::mbar_wait_warp(kPro ? &sm.kv_rot : &sm.kv_full, k & 1, abort_flag, status, kDevTimeoutFull);
                for (int it = 0; ok && it < n_q; ++it, ++q) {
                    // Products of tile q: half h once every elementwise warp holds half h
                    // of tile q-1 (the columns are then free).
                    const int qs = q % kQStages;
                    if (!ptx::mbar_wait_warp(kPro ? &sm.q_rot[qs] : &sm.q_full[qs], (q / kQStages) & 1, abort_flag,
                                             status, kDevTimeoutFull)) {
                        ok = false;
                        break;
                    }
                    for (int h = 0; ok && h < 2; ++h) {
                        if (q > 0 && !ptx::mbar_wait_warp(&sm.s_free[h], (q - 1) & 1, abort_flag, status,
                                                          kDevTimeoutFull)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        issue_s_dp(qs, h);
                    }
                    if (ok) ptx::mma_commit_elect(&sm.q_empty[qs]);  // this stream no longer reads P1_i, dY_i
                }
                if (!ok) break;
                ptx::mma_commit_elect(&sm.kv_free);  // nor P2_j and V_j of this key tile
                const int nx = next_tile(k);
                if (nx < 0) break;
                n_q = key_tile(nx, kp, nt_all, head_group).n_q;
            }
            ptx::mma_commit_elect(&sm.mma_done[0]);
            ptx::mbar_drain(&sm.mma_done[0], 0, status);
        } else {
            const uint32_t id_dv = ptx::idesc_bf16(kTile, kD, false, true);  // dV (B MN-major)
            const uint32_t id_dk = ptx::idesc_bf16(kTile, kD, false, true);  // dP2 (A K-major, B MN-major)
            const uint32_t id_dq = ptx::idesc_bf16(kTile, kD, true, true);   // dP1 (A, B MN-major)
            const uint32_t km_lo = ptx::desc_lo(mdesc(ptx::smem_u32(sm.k)));
            const uint32_t qm_lo0 = ptx::desc_lo(mdesc(ptx::smem_u32(sm.q[0])));
            const uint32_t gm_lo0 = ptx::desc_lo(mdesc(ptx::smem_u32(sm.g[0])));
            const uint32_t sk_lo0 = ptx::desc_lo(kdesc(ptx::smem_u32(sm.ds[0])));
            const uint32_t sm_lo0 = ptx::desc_lo(mdesc(ptx::smem_u32(sm.ds[0])));
            bool acc_committed = false;  // acc_done of the current key tile
            for (int k = 0, q = 0; ok; ++k) {
                acc_committed = false;
                for (int it = 0; ok && it < n_q; ++it, ++q) {
                    const int s = q & 1;          // dS buffer
                    const int qs = q % kQStages;  // P1/dY stage
                    if (!ptx::mbar_wait_warp(&sm.p_full, q & 1, abort_flag, status, kDevTimeoutFull)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // dV += P^T dY_i: K-step ks covers queries 16ks..16ks+15 (8 packed TMEM
                    // columns; 16 dY rows = 2048 bytes of the MN-major tile).  The first
                    // query tile of a key tile starts the accumulators afresh.
                    const uint32_t gm_lo = gm_lo0 + qs * kStageQ, qm_lo = qm_lo0 + qs * kStageQ;
                    const uint32_t sk_lo = sk_lo0 + (s ? kStageS : 0u);
                    const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        ptx::mma_ts_elect(tmem + kColDV, tmem + kColP + 8 * ks, gm_lo + 128 * ks, hi_m, id_dv,
                                          ks > 0 ? 1u : acc0);
                    ptx::mma_commit_elect(&sm.pv_done);
                    // dP2 += dS^T P1_i: A K-major over the two 64-query panels of dS^T.
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        ptx::mma_ss_elect(tmem + kColDK, sk_lo + (ks >> 2) * kStageQ + 2 * (ks & 3), hi_k,
                                          qm_lo + 128 * ks, hi_m, id_dk, ks > 0 ? 1u : acc0);
                    ptx::mma_commit_elect(&sm.q_empty[qs]);  // this stream no longer reads P1_i, dY_i
                    if (it == n_q - 1) {
                        ptx::mma_commit_elect(&sm.acc_done);  // dV and dP2 are final: the epilogue may start
                        acc_committed = true;
                    }
                    // dP1_i = dS P2_j: A = dS (MN-major view of dS^T buffer s), K over key
                    // rows, into the partial's columns once the reduce warps drained the
                    // previous tile's.
                    if (q > 0 &&
                        !ptx::mbar_wait_warp(&sm.dq_free, (q - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sm_lo = sm_lo0 + (s ? kStageS : 0u);
#pragma unroll
                    for (int ks = 0; ks < kTile / 16; ++ks)
                        ptx::mma_ss_elect(tmem + kColDQ, sm_lo + 128 * ks, hi_m, km_lo + 128 * ks, hi_m, id_dq,
                                          ks > 0 ? 1u : 0u);
                    ptx::mma_commit_elect(&sm.dq_full);
                }
                if (!ok) break;
                ptx::mma_commit_elect(&sm.kv_free);  // the last dP1 was the last read of P2_j
                const int nx = next_tile(k);
                if (nx < 0) break;
                n_q = key_tile(nx, kp, nt_all, head_group).n_q;
            }
            if (!acc_committed) ptx::mma_commit_elect(&sm.acc_done);  // left early: the epilogue's wait still ends
            ptx::mma_commit_elect(&sm.mma_done[1]);
            ptx::mbar_drain(&sm.mma_done[1], 0, status);
        }
    } else if (warp < 4) {
        ptx::regs_dec<kRegsControl>();
        if constexpr (kPro) {
            // Fused prologue of the key tile: rotate P2_j, mix V_j with the partner's states.
            if (ptx::mbar_wait_warp(&sm.kv_full, 0, abort_flag, status, kDevTimeoutFull)) {
                if (pro.tab.enabled) {
                    RopeAngles<32> ang;
                    ang.init(lane, pos_base + (float)w0.kv0, pro.tab, 1.f);
                    rope_tile64<32>(sm.k, lane, ang);
                }
                mix_tile64<32>(sm.v, sm.dq_stage, lane, g_cs, g_sn);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.kv_rot);
            }
        }
    } else if (warp < 4 + kElemWarps) {
        // ------------------------------------------------- elementwise blocks
        ptx::regs_inc<kRegsElementwise>();
        const int blk = (warp - 4) >> 2;  // query columns 64h + 16*blk .. +15 of each half h
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key row within the tile
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
        ec.causal = kp.causal != 0;
        float dlam = 0.f;
        bool ok = true;
        KeyTile w = w0;
        for (int k = 0, q = 0;; ++k) {
            const int kv = w.kv0 + r;
            const bool row_valid = kv < T;
            const int count_kv = kp.causal ? (kv + 1) : T;
            ec.log_count = __logf((float)count_kv);
            ec.diag_off = (0.5f + kp.lambda * ec.log_count) * kLog2e;  // (1/2 + lambda log c) log2(e)
            ec.row_valid = row_valid;
            for (int it = 0; ok && it < w.n_q; ++it, ++q) {
                const int s = q & 1;
                const int i = w.i_first + it;
                const int qs = q % kQStages;
                const bool diag_tile = (i == w.jt);
                const int qlimit = T - i * kTile;  // columns col < qlimit hold queries < T
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // query half: columns 64h + 16blk .. +15 of this warp
                    const int col0 = 64 * h + 16 * blk;
                    if (!ptx::mbar_wait_warp(&sm.s_full[h], q & 1, abort_flag, status, kDevTimeoutMma) ||
                        // Per-query constants of this tile (loaded with P1_i and dY_i).
                        (h == 0 && !ptx::mbar_wait_warp(&sm.q_full[qs], (q / kQStages) & 1, abort_flag, status,
                                                        kDevTimeoutFull))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    uint32_t sv[16], gv[16];
                    ptx::tmem_ld16(lane_addr + kColS + col0, sv);
                    ptx::tmem_ld16(lane_addr + kColDP + col0, gv);
                    ptx::tmem_ld_wait();
                    ptx::pin_regs(sv);
                    ptx::pin_regs(gv);
                    // This warp's part of half h is in registers: the next tile's products
                    // may overwrite those TMEM columns.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&sm.s_free[h]);
                    const float4* qc = sm.qconst[qs] + col0 / 2;
                    // The masked variant is chosen per warp (uniformly) if any of its rows needs it.
                    const bool special = __any_sync(0xffffffffu, diag_tile || qlimit < col0 + 16 || !row_valid);
                    uint32_t pp[8], dd[8];
                    if (!special)
                        elementwise16<false>(sv, gv, qc, col0, r, ec, false, 0, pp, dd);
                    else
                        dlam += elementwise16<true>(sv, gv, qc, col0, r, ec, diag_tile, qlimit, pp, dd);
                    if (h == 0) {
                        // Before the first store: P^T(q-1) must have been read by dV(q-1), and
                        // dS buffer s by the dP2 and dP1 products of tile q-2.  One wait covers
                        // both: the second MMA warp issues dP2(q-2), dP1(q-2) before dV(q-1), and
                        // a commit completes only when every earlier product of its thread has.
                        if (q > 0 &&
                            !ptx::mbar_wait_warp(&sm.pv_done, (q - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    // P^T packs query pairs: query column c lives in TMEM column c/2.
                    tmem_st8(lane_addr + kColP + col0 / 2, pp);
                    // dS^T: panel h (64 queries), 16-byte chunks 2blk, 2blk+1 of the 128-byte row.
                    uint8_t* ds_row = sm.ds[s] + h * kTileBytes + r * 128;
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int chunk = 2 * blk + k2;
                        *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                            make_uint4(dd[4 * k2], dd[4 * k2 + 1], dd[4 * k2 + 2], dd[4 * k2 + 3]);
                    }
                }
                if (!ok) break;
                ptx::tmem_st_wait();
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.p_full);
            }
            // Epilogue of the key tile: blocks 0-1 write dV, blocks 2-3 write dP2, 32
            // columns each, once the last accumulations are complete; the next key
            // tile's first dV and dP2 (which start the accumulators afresh) follow the
            // p_full of its first query tile, which these warps give after this.
            if (!ok || !ptx::mbar_wait_warp(&sm.acc_done, k & 1, abort_flag, status, kDevTimeoutMma)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            {
                const int c0 = blk & 1;
                __nv_bfloat16* dst_row = (blk < 2 ? dV : dP2) + row_offset(kp, w.bh, row_valid ? kv : 0);
                const uint32_t col = (blk < 2 ? kColDV : kColDK) + 32 * c0;
                uint32_t ov[32];
                ptx::tmem_ld32(lane_addr + col, ov);
                ptx::tmem_ld_wait();
                ptx::pin_regs(ov);
                if constexpr (kPro) {
                    if (blk >= 2 && pro.tab.enabled) {
                        // dX2 = R^T dP2: coordinate c (< 32) of this row pairs with c + 32, the
                        // other block's column; each block writes its half.
                        uint32_t ow[32];
                        ptx::tmem_ld32(lane_addr + kColDK + 32 * (1 - c0), ow);
                        ptx::tmem_ld_wait();
                        ptx::pin_regs(ow);
                        const float pos = pos_base + (float)kv;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            float sn, cs;
                            rope_sincos(pos, pro.tab.hi[c], pro.tab.lo[c], &sn, &cs);
                            const float g1 = as_f(c0 == 0 ? ov[c] : ow[c]), g2 = as_f(c0 == 0 ? ow[c] : ov[c]);
                            ov[c] = __float_as_uint(c0 == 0 ? fmaf(cs, g1, sn * g2) : fmaf(cs, g2, -sn * g1));
                        }
                    }
                }
                ptx::tc_fence_before();
                if (row_valid) {
                    // Columns past the head width (zero padding of the tiles) are not written.
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        store_bf16x8(dst_row, 32 * c0 + 8 * k4, kp.d,
                                     ptx::pack_bf16x2(as_f(ov[8 * k4 + 0]), as_f(ov[8 * k4 + 1])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k4 + 2]), as_f(ov[8 * k4 + 3])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k4 + 4]), as_f(ov[8 * k4 + 5])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k4 + 6]), as_f(ov[8 * k4 + 7])));
                }
            }
            const int nx = next_tile(k);
            if (nx < 0) break;
            w = key_tile(nx, kp, nt_all, head_group);
        }
        if (dlambda != nullptr) {
            // dR_ii = p (g - D) = dr / k_scale; sum log(c_i) dR_ii.
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, o);
            if (lane == 0 && dlam != 0.f) atomicAdd(dlambda, dlam / k_scale);
        }
    } else {
        // -------------------------------------------------- dP1 partial reduce
        // TMEM -> swizzled shared staging -> one TMA bulk reduce-add (fp32) per
        // 32-column panel into the accumulator; rows past T are dropped by TMA.
        ptx::regs_dec<kRegsReduce>();
        const int quarter = warp & 3;
        const int rq = quarter * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool leader = (warp == 4 + kElemWarps) && lane == 0;
        // Fused prologue (one key tile): rotate P1 of query tile it2 once it has
        // landed (a no-op past the last tile); tiles 0 and 1 first, then tile it + 2
        // in iteration it.  Query tiles come in order, so the angles carry from one
        // tile to the next.
        RopeAngles<128> ang;
        if (kPro && pro.tab.enabled) ang.init(rq, pos_base + (float)(w0.i_first * kTile), pro.tab, 1.f);
        auto rotate_q = [&](int it2) -> bool {
            if constexpr (kPro) {
                if (it2 >= w0.n_q) return true;
                const int s2 = it2 % kQStages;
                if (!ptx::mbar_wait_warp(&sm.q_full[s2], (it2 / kQStages) & 1, abort_flag, status, kDevTimeoutFull))
                    return false;
                if (pro.tab.enabled) rope_tile64<128>(sm.q[s2], rq, ang);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sm.q_rot[s2]);
            }
            return true;
        };
        bool rot_ok = rotate_q(0) && rotate_q(1);
        KeyTile w = w0;
        for (int k = 0, q = 0;; ++k) {
            bool left = false;
            for (int it = 0; it < w.n_q; ++it, ++q) {
                const int i = w.i_first + it;
                rot_ok = rot_ok && rotate_q(it + 2);
                // The four warps take one decision per tile (a 128-thread vote on named
                // barrier 1): if any warp's bounded wait gave up, all four leave together,
                // so none is left at the bar.sync below waiting for a warp that left.
                const bool got = rot_ok && ptx::mbar_wait_warp(&sm.dq_full, q & 1, abort_flag, status, kDevTimeoutMma);
                if (!ptx::bar_vote_all<1, 128>(got)) {
                    left = true;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < 2; ++c0) {
                    uint32_t ov[32];
                    ptx::tmem_ld32(lane_addr + kColDQ + 32 * c0, ov);
                    ptx::tmem_ld_wait();
                    ptx::pin_regs(ov);
                    if (c0 == 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&sm.dq_free);  // both halves have left TMEM
                    }
                    // The previous bulk reduce must have finished reading the staging panel.
                    if (leader) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    uint8_t* row = sm.dq_stage + rq * 128;
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8)
                        *reinterpret_cast<uint4*>(row + ((k8 ^ (rq & 7)) << 4)) =
                            make_uint4(ov[4 * k8], ov[4 * k8 + 1], ov[4 * k8 + 2], ov[4 * k8 + 3]);
                    ptx::fence_proxy_async_smem();
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (leader) {
                        asm volatile(
                            "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, "
                            "%3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)),
                            "r"(32 * c0), "r"(i * kTile), "r"(w.bh), "r"(ptx::smem_u32(sm.dq_stage))
                            : "memory");
                        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    }
                }
            }
            if (left) break;
            // The next key tile, by the same vote (a warp whose wait gave up takes
            // the other three with it).
            const int nx = next_tile(k);
            if (!ptx::bar_vote_all<1, 128>(nx >= 0)) break;
            w = key_tile(nx, kp, nt_all, head_group);
        }
        // The staging panel must be read before the CTA's shared memory goes; the
        // reduce-adds complete in global memory before the grid does.
        if (leader) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

namespace {
template <bool kPro>
cudaError_t launch_bwd_tc64_t(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                              const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV,
                              float* dlambda, const TcLaunch& tl, cudaStream_t s, bool padded64, const ProArgs& pro) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        const void* fns[2] = {(const void*)relation_bwd_tc64_kernel<kLoadTma3, kPro>,
                              (const void*)relation_bwd_tc64_kernel<kLoadTma4, kPro>};
        for (const void* f : fns)
            if (attr_err == cudaSuccess)
                attr_err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // Operands in the problem's layout; heads narrower than 64 read as 64-wide
    // tiles whose extra columns are zero (so they add nothing to any product).
    // Rows TMA cannot step through (d * 2 bytes not a multiple of 16) arrive as
    // zero-padded contiguous copies of 64 columns (padded64).
    if (!padded64 && (kp.d * 2) % 16 != 0) return cudaErrorInvalidValue;
    const int mode = padded64 ? kLoadTma3 : (kp.layout == 0 ? kLoadTma3 : kLoadTma4);
    const int map_d = padded64 ? 64 : kp.d, map_layout = padded64 ? 0 : kp.layout;
    CUtensorMap m1{}, m2{}, mv{}, mg{}, mq{};
    const void* bases[4] = {P1, P2, V, dY};
    CUtensorMap* maps[4] = {&m1, &m2, &mv, &mg};
    for (int k = 0; k < 4; ++k) {
        cudaError_t e =
            make_operand_map(maps[k], bases[k], kp.BH / kp.H, kp.H, kp.T, map_d, map_layout, 64, 128, true);
        if (e != cudaSuccess) return e;
    }
    // dP1 accumulator: fp32 [BH, T, 64] (its own padded layout), reduced in
    // 32-column (128-byte) swizzled boxes.
    cudaError_t e = make_tensor_map_3d(&mq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kD, kp.T, kp.BH, 32, 128,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int64_t ctas = kp.BH * ((kp.T + kTile - 1) / kTile);
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    // Heads in flight: as many as fit in three quarters of L2 with P1, P2, V, dY
    // (bf16) and the fp32 dP1 accumulator of each, i.e. 12 T d bytes per head.
    static std::once_flag l2_once;
    static int l2_bytes = 0;
    std::call_once(l2_once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev);
    });
    const int64_t per_head = 12 * (int64_t)kp.T * kD;
    const int64_t group =
        balanced_head_group(kp.BH, (l2_bytes > 0 ? (int64_t)l2_bytes * 3 / 4 : (int64_t)96 << 20) / per_head);
    dim3 grid((unsigned)ctas);
#define RELATION_BWD64(M)                                                                                        \
    relation_bwd_tc64_kernel<M, kPro><<<grid, kThreads, kSmemBytes, s>>>(                                        \
        m1, m2, mv, mg, mq, kp, qconst, (__nv_bfloat16*)dP2, (__nv_bfloat16*)dV, dlambda, tl.status, (int)group, pro)
    if (mode == kLoadTma3)
        RELATION_BWD64(kLoadTma3);
    else
        RELATION_BWD64(kLoadTma4);
#undef RELATION_BWD64
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc64(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                            const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                            const TcLaunch& tl, cudaStream_t s, bool padded64) {
    return launch_bwd_tc64_t<false>(kp, P1, P2, V, qconst, dY, dq_acc, dP2, dV, dlambda, tl, s, padded64, ProArgs{});
}

cudaError_t launch_bwd_tc64_prologue(const KernelProblem& kp, const void* X1, const void* X2, const void* I,
                                     const float4* qconst, const void* dY, float* dq_acc, void* dX2, void* dImix,
                                     float* dlambda, const TcLaunch& tl, cudaStream_t s, const RopeTable& tab,
                                     const float* theta, const int32_t* pos0, int pairing) {
    if (kp.d != 64 || kp.H % 2 != 0) return cudaErrorInvalidValue;
    ProArgs pro{};
    pro.tab = tab;
    pro.theta = theta;
    pro.pos0 = pos0;
    pro.pairing = pairing;
    return launch_bwd_tc64_t<true>(kp, X1, X2, I, qconst, dY, dq_acc, dX2, dImix, dlambda, tl, s, false, pro);
}

}  // namespace relation

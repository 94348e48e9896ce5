// Fused Full Relation forward on the sm_103a tensor cores (bf16 in, fp32 accumulate).
//
// Operator: "Ask Self, Ask Others: Relation Is All You Need", Sec. 3.1
// eq.(1)-(3): U = P1 P2^T / sqrt(d), Self S_i = sigmoid(U_ii / tau_S) on the
// diagonal, Exchange E_ij = SiLU(U_ij) - lambda log c_i off it, -inf above it
// (causal), F = Softmax(R), Y = F V.  U, R and F are never stored: each
// 128 x 128 block of U lives in tensor memory for one step of an online
// softmax (the running max / sum scan of Sec. 5.1 eq.(12), applied to whole
// rows of R rather than to the Exchange part only).
//
// Count correction: every off-diagonal entry of row i carries -lambda log c_i
// and softmax is invariant to a per-row shift (Appendix A.1.5), so the kernel
// adds +lambda log c_i to the diagonal entry instead and leaves off-diagonal
// blocks as plain SiLU.  L is reported in the paper's convention.
//
// One CTA = one head x two 128-row query tiles (rows q_base .. q_base+255).
//   warp 0      TMA producer: both Q tiles once, then K/V tiles through a ring
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 2-3   idle (they complete the first warpgroup for register reallocation)
//   warps 4-7   softmax of query tile 0 (one thread per row)
//   warps 8-11  softmax of query tile 1
// TMEM (512 columns): S0 | S1 (128 fp32 columns each; P overwrites the first
// 64 columns as packed bf16) | O0 | O1 (d columns each).
// Per key tile j, per query tile t:  S_t = Q_t K_j^T (SS MMA) -> softmax ->
// P_t -> O_t += P_t V_j (TS MMA, P read from TMEM).  The two query tiles
// alternate so the tensor core works on one while the other is in softmax.
// At D = 128 their softmax warps also take turns on the special-function unit
// (one mbarrier pair per sub-partition), so that one tile's tanh / ex2 loops
// run while the other tile waits for its next S or stores P.
#include <cuda_bf16.h>

#include "kernels.h"
#include "prologue_tiles.cuh"
#include "tile_copy.cuh"
#include "ptx_sm100.cuh"
#include "tmap.h"

namespace relation {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;
// Register split (per thread) after launch at 168: the load/MMA warpgroup
// gives back, the two softmax warpgroups take: 128*56 + 256*224 = 64512 <= 384*168.
constexpr uint32_t kRegsControl = 56, kRegsSoftmax = 224;
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running max (natural units) is raised only when a block's max exceeds
// it by more than 8 ln 2 (a factor 256); exact, since numerator and
// denominator share whatever max is used.
constexpr float kRescaleThreshold = 8.0f * 0.6931471805599453f;

template <int D, bool kPro = false>
struct FwdCfg {
    // d = 64 leaves 128 TMEM columns free: P gets its own region per tile, so the
    // next S can be issued while the softmax still works on the current one.
    // d = 128 fills TMEM with S and O, and P overwrites S.
    static constexpr bool kSepP = (D == 64);
    static constexpr uint32_t kColP = 384;
    static constexpr int kPanels = D / 64;
    static constexpr int kTileBytes = kBM * D * 2;
    // With the fused prologue each stage also holds the pair partner's information
    // tile (kVb), and the ring is one stage shorter to make room for it.
    static constexpr int kStages = (D == 64) ? (kPro ? 3 : 4) : 2;
    static constexpr int kVb = kPro ? 1 : 0;
    // 1 KB for 1024-byte alignment of the swizzled tiles, the tiles, the
    // barriers, and a 16 KB guard band that keeps any descriptor walk past a
    // tile's end inside the CTA's allocation.
    static constexpr int kSmemBytes = 1024 + (2 + (2 + kVb) * kStages) * kTileBytes + 512 + 16384;
};

struct FwdBarriers {
    uint64_t q_full[2];
    uint64_t k_full[4];
    uint64_t v_full[4];
    uint64_t kv_empty[4];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[2];
    uint64_t o_done[2];
    uint64_t drain;
    // Fused prologue: Q / K tiles rotated and V tiles mixed in shared memory.
    uint64_t q_rot[2];
    uint64_t k_rot[4];
    uint64_t v_mix[4];
    // Turns of the two query tiles' softmax warps on each sub-partition's
    // special-function unit (one barrier per tile and warp quarter).
    uint64_t turn[2][4];
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(FwdBarriers) <= 512, "the barriers' 512-byte region");

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t as_u(float f) { return __float_as_uint(f); }

// Dot product of row r of two staged tiles (D/64 swizzled panels of 128 rows x
// 128 bytes; 16-byte chunk k of row r sits at chunk k ^ (r % 8)).
template <int kPanels>
__device__ __forceinline__ float row_dot(const uint8_t* a_tile, const uint8_t* b_tile, int r) {
    float acc = 0.f;
#pragma unroll
    for (int p = 0; p < kPanels; ++p) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int off = p * kPanelBytes + r * 128 + ((k ^ (r & 7)) << 4);
            const uint4 x = *reinterpret_cast<const uint4*>(a_tile + off);
            const uint4 y = *reinterpret_cast<const uint4*>(b_tile + off);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[w]));
                const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[w]));
                acc = fmaf(xf.x, yf.x, acc);
                acc = fmaf(xf.y, yf.y, acc);
            }
        }
    }
    return acc;
}

// kCp: operand tiles copied by the producer warp with cp.async from the raw
// pointers (head widths whose rows TMA cannot address; D = 64 only), else TMA.
// kPro: the operands are the prologue's inputs X1, X2, I (D = 64, TMA): warps
// 2-3 rotate the Q and K tiles and mix each V tile with the pair partner's
// before the tensor core reads them.
template <int D, bool kCp, bool kPro = false>
__global__ void __launch_bounds__(kThreads, 1)
    relation_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_p1, const __grid_constant__ CUtensorMap tm_p2,
                           const __grid_constant__ CUtensorMap tm_v, const KernelProblem kp,
                           const __nv_bfloat16* __restrict__ P1, const __nv_bfloat16* __restrict__ P2,
                           const __nv_bfloat16* __restrict__ V, __nv_bfloat16* __restrict__ Y,
                           float* __restrict__ L, unsigned int* status, const __grid_constant__ ProArgs pro) {
    static_assert(!kCp || D == 64, "cp.async tiles are 64 columns wide");
    static_assert(!kPro || (D == 64 && !kCp), "the fused prologue works on 64-column TMA tiles");
    using C = FwdCfg<D, kPro>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + 2 * C::kTileBytes;
    uint8_t* sV = sK + C::kStages * C::kTileBytes;
    uint8_t* sVb = sV + C::kStages * C::kTileBytes;  // pair partner's information tiles (kPro)
    FwdBarriers* bars = reinterpret_cast<FwdBarriers*>(sVb + C::kVb * C::kStages * C::kTileBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int batch = bh / kp.H, head = bh - batch * kp.H;
    int partner = head;
    float g_cs = 1.f, g_sn = 0.f;  // Givens coefficients of this head (fused prologue)
    if constexpr (kPro) partner = givens_coeffs(head, kp.H, pro, &g_cs, &g_sn);
    const int pair = (int)gridDim.y - 1 - (int)blockIdx.y;  // heaviest (latest) query rows first
    const int T = kp.T;
    const int q_base = pair * 2 * kBM;
    const int n_kv_all = (T + kBN - 1) / kBN;
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int row0 = q_base + t * kBM;
        n_t[t] = (row0 >= T) ? 0 : (kp.causal ? (row0 / kBN + 1) : n_kv_all);
    }
    const int n_max = max(n_t[0], n_t[1]);

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(&bars->q_full[t], 1);
            ptx::mbar_init(&bars->s_full[t], 1);
            ptx::mbar_init(&bars->s_free[t], 128);
            ptx::mbar_init(&bars->p_full[t], 128);
            ptx::mbar_init(&bars->o_done[t], 1);
        }
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bars->k_full[s], 1);
            ptx::mbar_init(&bars->v_full[s], 1);
            ptx::mbar_init(&bars->kv_empty[s], 1);
        }
        ptx::mbar_init(&bars->drain, 1);
        for (int t = 0; t < 2; ++t) ptx::mbar_init(&bars->q_rot[t], 2);
        if constexpr (!C::kSepP)
            for (int t = 0; t < 2; ++t)
                for (int q = 0; q < 4; ++q) ptx::mbar_init(&bars->turn[t][q], 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bars->k_rot[s], 2);
            ptx::mbar_init(&bars->v_mix[s], 2);
        }
        bars->abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bars->tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    volatile int* abort_flag = &bars->abort_flag;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        ptx::regs_dec<kRegsControl>();
        if constexpr (kCp) {
            // The whole warp copies the two query tiles, then streams the K/V stages.
            for (int t = 0; t < 2; ++t)
                if (n_t[t] > 0) cp_async_tile64(sQ + t * C::kTileBytes, P1, kp, bh, q_base + t * kBM, lane);
            cp_async_commit();
            cp_async_publish<0>();
            if (lane == 0)
                for (int t = 0; t < 2; ++t)
                    if (n_t[t] > 0) ptx::mbar_arrive(&bars->q_full[t]);
            // Stage j is issued, then stage j - kAhead is published (kAhead < kStages, so
            // the wait for a free stage never waits on a stage still unpublished).
            constexpr int kAhead = 2;
            static_assert(kAhead < C::kStages, "lookahead must leave a stage");
            int j = 0;
            for (; j < n_max; ++j) {
                const int s = j % C::kStages;
                if (j >= C::kStages && !ptx::mbar_wait_warp(&bars->kv_empty[s], ((j / C::kStages) - 1) & 1,
                                                            abort_flag, status, kDevTimeoutEmpty))
                    break;
                cp_async_tile64(sK + s * C::kTileBytes, P2, kp, bh, j * kBN, lane);
                cp_async_commit();
                cp_async_tile64(sV + s * C::kTileBytes, V, kp, bh, j * kBN, lane);
                cp_async_commit();
                if (j >= kAhead) {
                    cp_async_publish<2 * kAhead>();  // stage j - kAhead has landed
                    if (lane == 0) {
                        const int sp = (j - kAhead) % C::kStages;
                        ptx::mbar_arrive(&bars->k_full[sp]);
                        ptx::mbar_arrive(&bars->v_full[sp]);
                    }
                }
            }
            cp_async_publish<0>();  // every copy has landed before the warp moves on
            if (j == n_max && lane == 0)
                for (int jj = max(0, n_max - kAhead); jj < n_max; ++jj) {
                    ptx::mbar_arrive(&bars->k_full[jj % C::kStages]);
                    ptx::mbar_arrive(&bars->v_full[jj % C::kStages]);
                }
        } else if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_p1);
            ptx::tma_prefetch_desc(&tm_p2);
            ptx::tma_prefetch_desc(&tm_v);
            for (int t = 0; t < 2; ++t) {
                if (n_t[t] == 0) continue;
                ptx::mbar_arrive_expect_tx(&bars->q_full[t], C::kTileBytes);
                for (int p = 0; p < C::kPanels; ++p)
                    ptx::tma_load_4d(sQ + t * C::kTileBytes + p * kPanelBytes, &tm_p1, &bars->q_full[t], p * 64,
                                     q_base + t * kBM, head, batch);
            }
            int j = 0;
            for (; j < n_max; ++j) {
                const int s = j % C::kStages;
                if (j >= C::kStages &&
                    !ptx::mbar_wait(&bars->kv_empty[s], ((j / C::kStages) - 1) & 1, abort_flag, status,
                                    kDevTimeoutEmpty))
                    break;
                ptx::mbar_arrive_expect_tx(&bars->k_full[s], C::kTileBytes);
                for (int p = 0; p < C::kPanels; ++p)
                    ptx::tma_load_4d(sK + s * C::kTileBytes + p * kPanelBytes, &tm_p2, &bars->k_full[s], p * 64,
                                     j * kBN, head, batch);
                ptx::mbar_arrive_expect_tx(&bars->v_full[s], (1 + C::kVb) * C::kTileBytes);
                for (int p = 0; p < C::kPanels; ++p)
                    ptx::tma_load_4d(sV + s * C::kTileBytes + p * kPanelBytes, &tm_v, &bars->v_full[s], p * 64,
                                     j * kBN, head, batch);
                if constexpr (kPro)
                    ptx::tma_load_4d(sVb + s * C::kTileBytes, &tm_v, &bars->v_full[s], 0, j * kBN, partner, batch);
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                for (int jj = max(0, j - C::kStages); jj < j; ++jj) {
                    const int s = jj % C::kStages;
                    ptx::mbar_drain(&bars->k_full[s], (jj / C::kStages) & 1, status);
                    ptx::mbar_drain(&bars->v_full[s], (jj / C::kStages) & 1, status);
                }
                for (int t = 0; t < 2; ++t)
                    if (n_t[t] > 0) ptx::mbar_drain(&bars->q_full[t], 0, status);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the issue loop; one elected lane issues each MMA.
        ptx::regs_dec<kRegsControl>();
        {
            // With the fused prologue the tensor core waits for the rotated / mixed tiles.
            uint64_t* q_ready = kPro ? bars->q_rot : bars->q_full;
            uint64_t* k_ready = kPro ? bars->k_rot : bars->k_full;
            uint64_t* v_ready_bar = kPro ? bars->v_mix : bars->v_full;
            const uint32_t id_s = ptx::idesc_bf16(kBM, kBN, false, false);
            const uint32_t id_o = ptx::idesc_bf16(kBM, D, false, true);
            // Descriptors are built once; a byte offset is added as offset >> 4.
            const uint64_t dq0 = ptx::smem_desc(ptx::smem_u32(sQ), 16, 1024, ptx::kSwizzle128B);
            const uint64_t dk0 = ptx::smem_desc(ptx::smem_u32(sK), 16, 1024, ptx::kSwizzle128B);
            const uint64_t dv0 = ptx::smem_desc(ptx::smem_u32(sV), kPanelBytes, 1024, ptx::kSwizzle128B);
            constexpr uint64_t kTileStep = C::kTileBytes >> 4, kPanelStep = kPanelBytes >> 4;
            auto issue_s = [&](int t, int s) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t off = (ks / 4) * kPanelStep + (ks % 4) * 2;  // 32 bytes per K-step
                    ptx::mma_ss_elect(tmem + t * 128, dq0 + t * kTileStep + off, dk0 + s * kTileStep + off, id_s,
                                ks > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int s, bool accumulate) {
#pragma unroll
                for (int ks = 0; ks < kBN / 16; ++ks) {
                    // 16 key rows of V per K-step: 2048 bytes of the MN-major tile.
                    const uint32_t p_col = C::kSepP ? C::kColP + 64 * t : 128 * t;
                    ptx::mma_ts_elect(tmem + 256 + t * D, tmem + p_col + ks * 8, dv0 + s * kTileStep + ks * 128, id_o,
                                (accumulate || ks > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            for (int t = 0; t < 2 && ok; ++t)
                if (n_t[t] > 0) ok = ptx::mbar_wait_warp(&q_ready[t], 0, abort_flag, status, kDevTimeoutFull);
            if (ok && n_max > 0) ok = ptx::mbar_wait_warp(&k_ready[0], 0, abort_flag, status, kDevTimeoutFull);
            if (ok) {
                ptx::tc_fence_after();
                for (int t = 0; t < 2; ++t) {
                    if (n_t[t] == 0) continue;
                    issue_s(t, 0);
                    ptx::mma_commit_elect(&bars->s_full[t]);
                }
            }
            for (int j = 0; ok && j < n_max; ++j) {
                const int s = j % C::kStages;
                const int s1 = (j + 1) % C::kStages;
                bool v_ready = false, k_next_ready = false;
                if constexpr (C::kSepP) {
                    // Next S of each tile as soon as its softmax has S(j) in registers.
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j + 1 >= n_t[t]) continue;
                        if (!ptx::mbar_wait_warp(&bars->s_free[t], j & 1, abort_flag, status, kDevTimeoutFull)) {
                            ok = false;
                            break;
                        }
                        if (!k_next_ready) {
                            if (!ptx::mbar_wait_warp(&k_ready[s1], ((j + 1) / C::kStages) & 1, abort_flag, status,
                                                kDevTimeoutFull)) {
                                ok = false;
                                break;
                            }
                            k_next_ready = true;
                        }
                        ptx::tc_fence_after();
                        issue_s(t, s1);
                        ptx::mma_commit_elect(&bars->s_full[t]);
                    }
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= n_t[t]) continue;
                        if (!ptx::mbar_wait_warp(&bars->p_full[t], j & 1, abort_flag, status, kDevTimeoutFull)) {
                            ok = false;
                            break;
                        }
                        if (!v_ready) {
                            if (!ptx::mbar_wait_warp(&v_ready_bar[s], (j / C::kStages) & 1, abort_flag, status,
                                                kDevTimeoutFull)) {
                                ok = false;
                                break;
                            }
                            v_ready = true;
                        }
                        ptx::tc_fence_after();
                        issue_pv(t, s, j > 0);
                        ptx::mma_commit_elect(&bars->o_done[t]);
                    }
                } else {
                    for (int t = 0; t < 2; ++t) {
                        if (j >= n_t[t]) continue;
                        if (!ptx::mbar_wait_warp(&bars->p_full[t], j & 1, abort_flag, status, kDevTimeoutFull)) {
                            ok = false;
                            break;
                        }
                        if (!v_ready) {
                            if (!ptx::mbar_wait_warp(&v_ready_bar[s], (j / C::kStages) & 1, abort_flag, status,
                                                kDevTimeoutFull)) {
                                ok = false;
                                break;
                            }
                            v_ready = true;
                        }
                        ptx::tc_fence_after();
                        issue_pv(t, s, j > 0);
                        ptx::mma_commit_elect(&bars->o_done[t]);
                        if (j + 1 < n_t[t]) {
                            if (!k_next_ready) {
                                if (!ptx::mbar_wait_warp(&k_ready[s1], ((j + 1) / C::kStages) & 1, abort_flag,
                                                    status, kDevTimeoutFull)) {
                                    ok = false;
                                    break;
                                }
                                k_next_ready = true;
                                ptx::tc_fence_after();
                            }
                            issue_s(t, s1);
                            ptx::mma_commit_elect(&bars->s_full[t]);
                        }
                    }
                }
                if (ok) ptx::mma_commit_elect(&bars->kv_empty[s]);
            }
            ptx::mma_commit_elect(&bars->drain);
            ptx::mbar_drain(&bars->drain, 0, status);
        }
    } else if (warp < 4) {
        ptx::regs_dec<kRegsControl>();
        if constexpr (kPro) {
            // ------------------------------------------------- fused prologue
            const int tr = threadIdx.x - 64;
            const float pos_base = pro.pos0 != nullptr ? (float)pro.pos0[batch] : 0.f;
            bool ok = true;
            RopeAngles<64> ang;  // the query tiles (consecutive), then the key tiles from row 0
            if (pro.tab.enabled) ang.init(tr, pos_base + (float)q_base, pro.tab, 1.f);
            for (int t = 0; t < 2 && ok; ++t) {
                if (n_t[t] == 0) continue;
                if (!(ok = ptx::mbar_wait_warp(&bars->q_full[t], 0, abort_flag, status, kDevTimeoutFull))) break;
                if (pro.tab.enabled) rope_tile64<64>(sQ + t * C::kTileBytes, tr, ang);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->q_rot[t]);
            }
            if (pro.tab.enabled) ang.init(tr, pos_base, pro.tab, 1.f);
            for (int j = 0; ok && j < n_max; ++j) {
                const int s = j % C::kStages;
                if (!ptx::mbar_wait_warp(&bars->k_full[s], (j / C::kStages) & 1, abort_flag, status, kDevTimeoutFull))
                    break;
                if (pro.tab.enabled) rope_tile64<64>(sK + s * C::kTileBytes, tr, ang);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->k_rot[s]);
                if (!ptx::mbar_wait_warp(&bars->v_full[s], (j / C::kStages) & 1, abort_flag, status, kDevTimeoutFull))
                    break;
                mix_tile64<64>(sV + s * C::kTileBytes, sVb + s * C::kTileBytes, tr, g_cs, g_sn);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->v_mix[s]);
            }
        }
    } else {
        // ------------------------------------------------------------- softmax
        ptx::regs_inc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int i = q_base + t * kBM + r;
        const int nt = n_t[t];
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t s_col = t * 128, o_col = 256 + t * D;
        const float c_half = 0.5f * kp.inv_sqrt_d;         // U/2 per raw dot product
        const float c_diag = 0.5f * kp.inv_sqrt_d / kp.tau_S;  // U/(2 tau_S)
        const int count = kp.causal ? (i + 1) : T;
        const float corr = kp.lambda * logf((float)count);    // lambda log c_i
        const int diag_tile = (q_base + t * kBM) / kBN;
        const int tail_cols = T - (n_kv_all - 1) * kBN;
        // When P overwrites S (D = 128), a tile's next S is computed only after its
        // transport product, so each step spends long stretches in TMEM traffic and
        // waits.  There the warps of the two tiles that share a sub-partition take
        // turns on its special-function unit for the first min(n_0, n_1) steps: tile
        // 0's step j, then tile 1's step j, each running its tanh / ex2 loops while the
        // other waits for S or stores P.  Tile 1's remaining steps run without turns.
        // At D = 64 the next S is ready early and that stretch is short: one warp alone
        // drives the unit at about three quarters of its rate, so the tiles share it.
        const int n_pair = C::kSepP ? 0 : min(n_t[0], n_t[1]);
        uint64_t* turn_mine = &bars->turn[t][quarter];
        uint64_t* turn_next = &bars->turn[t ^ 1][quarter];
        float m = -INFINITY, l = 0.f;
        bool ok = nt > 0;
        for (int j = 0; ok && j < nt; ++j) {
            if (!ptx::mbar_wait_warp(&bars->s_full[t], j & 1, abort_flag, status, kDevTimeoutMma)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint32_t sv[128];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                ptx::tmem_ld32(lane_addr + s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
            ptx::tmem_ld_wait();
            ptx::pin_regs(sv);
            if constexpr (C::kSepP) {
                // S(j) is in registers: the next S of this tile may overwrite it.
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars->s_free[t]);
            }
            if constexpr (!C::kSepP) {
                if (j < n_pair && j + t > 0 &&
                    !ptx::mbar_wait_warp(turn_mine, (j + t - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                    ok = false;
                    break;
                }
                ptx::pin_regs(sv);  // the loops below start after the turn is taken
            }
            // sv[c] becomes R'_ic (natural units) in place, R' = R + lambda log c_i.
            const bool is_diag = (j == diag_tile);
            const int climit = (j == n_kv_all - 1) ? tail_cols : kBN;
            const float2 ch2 = make_float2(c_half, c_half);
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const float2 h = ptx::mul2(make_float2(as_f(sv[2 * e]), as_f(sv[2 * e + 1])), ch2);
                const float2 th = make_float2(ptx::tanh_approx(h.x), ptx::tanh_approx(h.y));
                const float2 E = ptx::fma2(h, th, h);  // SiLU(U) = (U/2)(1 + tanh(U/2))
                sv[2 * e] = as_u(E.x);
                sv[2 * e + 1] = as_u(E.y);
            }
            if (is_diag || climit < kBN) {
                // Self entry sigmoid(U_ii/tau_S) = (1 + tanh(U_ii/(2 tau_S)))/2 plus the folded
                // count correction; U_ii is recomputed from the staged P1 and P2 rows.
                // Masked entries (future keys, keys past T) become -inf.
                float s_diag = 0.f;
                if (is_diag) {
                    const float a_diag = row_dot<C::kPanels>(sQ + t * C::kTileBytes, sK + (j % C::kStages) * C::kTileBytes, r);
                    s_diag = fmaf(0.5f, ptx::tanh_approx(a_diag * c_diag), 0.5f) + corr;
                }
                const int cmax = (kp.causal && is_diag) ? min(r, climit - 1) : climit - 1;  // last visible column
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    float v = (c > cmax) ? -INFINITY : as_f(sv[c]);
                    sv[c] = as_u((is_diag && c == r) ? s_diag : v);
                }
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 128; c += 8) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mx[k] = ptx::max3(mx[k], as_f(sv[c + 2 * k]), as_f(sv[c + 2 * k + 1]));
            }
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            const float m_new = fmaxf(m, mt);
            const bool rescale = __any_sync(0xffffffffu, m_new > m + kRescaleThreshold);
            float scale = 1.f;
            if (rescale) {
                scale = ptx::ex2_approx((m - m_new) * kLog2e);  // 0 when m = -inf
                l *= scale;
                m = m_new;
            }
            const float2 l2e2 = make_float2(kLog2e, kLog2e);
            const float2 nm2 = make_float2(-m * kLog2e, -m * kLog2e);
            float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[2][32];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float2 y = ptx::fma2(make_float2(as_f(sv[2 * c]), as_f(sv[2 * c + 1])), l2e2, nm2);
                const float2 p = make_float2(ptx::ex2_approx(y.x), ptx::ex2_approx(y.y));
                ls[c & 3] = ptx::add2(ls[c & 3], p);
                pk[c >> 5][c & 31] = ptx::pack_bf16x2(p.x, p.y);
            }
            {
                const float2 s01 = ptx::add2(ls[0], ls[1]), s23 = ptx::add2(ls[2], ls[3]);
                const float2 st = ptx::add2(s01, s23);
                l += st.x + st.y;
            }
            if constexpr (!C::kSepP) {
                ptx::pin_regs(pk[0]);  // and end before it is passed on
                ptx::pin_regs(pk[1]);
                __syncwarp();
                if (j < n_pair && lane == 0) ptx::mbar_arrive(turn_next);
            }
            if constexpr (C::kSepP) {
                // P(j) replaces P(j-1) once the transport of block j-1 has read it (that
                // also makes O final for a rescale).
                if (j > 0) {
                    if (!ptx::mbar_wait_warp(&bars->o_done[t], (j - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
                ptx::tmem_st32(lane_addr + C::kColP + 64 * t, pk[0]);
                ptx::tmem_st32(lane_addr + C::kColP + 64 * t + 32, pk[1]);
            } else {
                ptx::tmem_st32(lane_addr + s_col, pk[0]);
                ptx::tmem_st32(lane_addr + s_col + 32, pk[1]);
            }
            if (rescale && j > 0) {
                // O holds the sums of key blocks 0..j-1; rescale it once the
                // transport MMA of block j-1 has landed (already awaited above when P
                // has its own region).  Block j's MMA waits for p_full, which is
                // signalled only after this.
                if (!C::kSepP) {
                    if (!ptx::mbar_wait_warp(&bars->o_done[t], (j - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
#pragma unroll
                for (int c0 = 0; c0 < D / 32; ++c0) {
                    uint32_t ov[32];
                    ptx::tmem_ld32(lane_addr + o_col + 32 * c0, ov);
                    ptx::tmem_ld_wait();
                    ptx::pin_regs(ov);
#pragma unroll
                    for (int k = 0; k < 32; ++k) ov[k] = as_u(as_f(ov[k]) * scale);
                    ptx::tmem_st32(lane_addr + o_col + 32 * c0, ov);
                }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars->p_full[t]);
        }
        if (ok && nt > 0 && ptx::mbar_wait_warp(&bars->o_done[t], (nt - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
            ptx::tc_fence_after();
            const float inv_l = 1.f / l;
            __nv_bfloat16* yrow = Y + row_offset(kp, bh, i < T ? i : 0);
#pragma unroll
            for (int c0 = 0; c0 < D / 32; ++c0) {
                if (32 * c0 >= kp.d) break;  // columns past the head width are zero padding
                uint32_t ov[32];
                ptx::tmem_ld32(lane_addr + o_col + 32 * c0, ov);
                ptx::tmem_ld_wait();
                ptx::pin_regs(ov);
                if (i < T) {
                    uint32_t pkd[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        pkd[k] = ptx::pack_bf16x2(as_f(ov[2 * k]) * inv_l, as_f(ov[2 * k + 1]) * inv_l);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        store_bf16x8(yrow, 32 * c0 + 8 * k, kp.d, pkd[4 * k], pkd[4 * k + 1], pkd[4 * k + 2],
                                     pkd[4 * k + 3]);
                }
            }
            if (L != nullptr && i < T) L[(size_t)bh * T + i] = m + __log2f(l) * kLn2 - corr;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D, bool kCp, bool kPro = false>
cudaError_t launch_fwd_tc_d(const KernelProblem& kp, const void* P1, const void* P2, const void* V, void* Y,
                            float* L, const TcLaunch& tl, cudaStream_t s, bool padded64 = false,
                            const ProArgs& pro = ProArgs{}) {
    using C = FwdCfg<D, kPro>;
    static_assert(C::kSmemBytes <= 232448, "shared memory budget");
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(relation_fwd_tc_kernel<D, kCp, kPro>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // Heads narrower than D read as D-wide tiles whose extra columns are zero.
    // Padded copies are contiguous [B, H, T, 64] whatever the caller's layout;
    // Y and L are still written in the caller's layout and width.
    CUtensorMap m1{}, m2{}, mv{};  // unused by the cp.async producer
    if (!kCp) {
        cudaError_t e;
        const int64_t B = kp.BH / kp.H;
        const int64_t md = padded64 ? 64 : kp.d;
        const int ml = padded64 ? 0 : kp.layout;
        if ((e = make_operand_map(&m1, P1, B, kp.H, kp.T, md, ml, 64, 128, false)) != cudaSuccess) return e;
        if ((e = make_operand_map(&m2, P2, B, kp.H, kp.T, md, ml, 64, 128, false)) != cudaSuccess) return e;
        if ((e = make_operand_map(&mv, V, B, kp.H, kp.T, md, ml, 64, 128, false)) != cudaSuccess) return e;
    }
    const unsigned pairs = (unsigned)((kp.T + 2 * kBM - 1) / (2 * kBM));
    dim3 grid((unsigned)kp.BH, pairs);
    relation_fwd_tc_kernel<D, kCp, kPro><<<grid, kThreads, C::kSmemBytes, s>>>(
        m1, m2, mv, kp, (const __nv_bfloat16*)P1, (const __nv_bfloat16*)P2, (const __nv_bfloat16*)V, (__nv_bfloat16*)Y,
        L, tl.status, pro);
    return cudaGetLastError();
}

}  // namespace

bool fwd_tc_grid_fits(const KernelProblem& kp) {
    // Heads in gridDim.x, pairs of kBM-row query tiles in gridDim.y (at most 65535).
    return kp.BH >= 1 && kp.BH <= 2147483647LL && ((int64_t)kp.T + 2 * kBM - 1) / (2 * kBM) <= 65535;
}

cudaError_t launch_fwd_tc(const KernelProblem& kp, const void* P1, const void* P2, const void* V, void* Y, float* L,
                          const TcLaunch& tl, cudaStream_t s, bool padded64) {
    if (kp.BH > 2147483647LL) return cudaErrorInvalidValue;
    if (padded64) {
        if (kp.d > 64) return cudaErrorInvalidValue;
        return launch_fwd_tc_d<64, false>(kp, P1, P2, V, Y, L, tl, s, true);
    }
    if (kp.d == 48 || kp.d == 64) return launch_fwd_tc_d<64, false>(kp, P1, P2, V, Y, L, tl, s);
    if (kp.d == 60) return launch_fwd_tc_d<64, true>(kp, P1, P2, V, Y, L, tl, s);  // 120-byte rows: no TMA
    if (kp.d == 80 || kp.d == 128) return launch_fwd_tc_d<128, false>(kp, P1, P2, V, Y, L, tl, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_tc_prologue(const KernelProblem& kp, const void* X1, const void* X2, const void* I, void* Y,
                                   float* L, const TcLaunch& tl, cudaStream_t s, const RopeTable& tab,
                                   const float* theta, const int32_t* pos0, int pairing) {
    if (kp.BH > 2147483647LL || kp.d != 64 || kp.H % 2 != 0) return cudaErrorInvalidValue;
    ProArgs pro{};
    pro.tab = tab;
    pro.theta = theta;
    pro.pos0 = pos0;
    pro.pairing = pairing;
    return launch_fwd_tc_d<64, false, true>(kp, X1, X2, I, Y, L, tl, s, false, pro);
}

}  // namespace relation

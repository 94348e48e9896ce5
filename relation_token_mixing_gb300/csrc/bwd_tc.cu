// Fused Full Relation backward on the sm_103a tensor cores (bf16 in, fp32 accumulate).
//
// The paper ("Ask Self, Ask Others: Relation Is All You Need") gives no
// backward; this is the chain rule of Sec. 3.1 eq.(1)-(3), with the forward's
// row log-normaliser L_i used to rebuild F_ij = exp(R_ij - L_i) block by block:
//   dF_ij = dY_i . V_j,  dR_ij = F_ij (dF_ij - D_i),  D_i = dY_i . Y_i,
//   dU_ii = dR_ii S_i (1 - S_i) / tau_S,  dU_ij = dR_ij SiLU'(U_ij),
//   dP1 = dU P2 / sqrt(d),  dP2 = dU^T P1 / sqrt(d),  dV = F^T dY.
//
// One CTA = one head x one 128-row key tile j (rows of P2 and V); it walks the
// query tiles i that can see it (i >= j when causal).  Head widths 80 and 128
// (128-wide tiles; a narrower head reads as a tile with zero columns).
//   warp 0       loader: P2_j, V_j once (TMA); per query tile P1_i, dY_i (TMA)
//                and the per-query constants (L_i folded with lambda log c_i, D_i)
//   warp 1       MMA issuer and TMEM owner
//   warps 4-19   elementwise stage: warp (quarter q, block b) owns key rows
//                32q..32q+31 (its TMEM lanes) and query columns 32b..32b+31
//   warps 20-23  dP1 reduction: TMEM -> swizzled shared staging -> TMA bulk
//                reduce-add (fp32) into the accumulator in global memory
// Per query tile, with everything transposed so that key rows sit on TMEM lanes:
//   S^T  = P2_j P1_i^T          (SS)      dP^T = V_j dY_i^T    (SS)
//   elementwise: P^T, dS^T = dU^T / sqrt(d) -> TMEM (bf16) and dS^T -> smem
//   dV  += P^T dY_i             (TS)      dP2 += dS^T P1_i     (TS)
//   dP1_i (partial) = dS P2_j   (SS, dS read MN-major from smem)
// TMEM: S^T [0,128) | dP^T [128,256) | dV [256,384) | dP2 [384,512).  Block b of
// a lane quarter reads S^T and dP^T columns 32b..32b+31 of its rows and packs
// its 32 queries' pairs into the dP^T columns it has read: dS^T into 32b..32b+15,
// P^T into 32b+16..32b+31 (after both halves are in registers).  The S^T columns
// are then free, so the dP1 partial goes there first and drains while dV and dP2
// run.
#include <cuda_bf16.h>

#include "bwd_elementwise.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"
#include "tmap.h"

namespace relation {
namespace {

using bwd_elem::ElemConst;
using bwd_elem::elementwise16;

constexpr int kTile = 128;
constexpr uint32_t kQConstBytes = kTile / 2 * 16;  // per-query constants of one query tile
constexpr int kElemWarps = 16;                     // warps 4 .. 19
constexpr int kReduceWarp0 = 4 + kElemWarps;       // warps 20 .. 23
constexpr int kThreads = 32 * (kReduceWarp0 + 4);  // 768
constexpr int kPanelBytes = 128 * 128;
constexpr int kStageBytes = kTile * 128;  // one dP1 staging panel: 128 rows x 32 fp32 columns
constexpr int kStagePanels = 2;           // staging panels in flight
constexpr float kLog2e = 1.4426950408889634f;
// Register split after launch at 80 per thread (six warps per SM sub-partition):
// load/MMA warpgroup 56, the four elementwise warpgroups 88, the dP1-reduce
// warpgroup 56:  128*56 + 512*88 + 128*56 = 59392 <= 768*80.
constexpr uint32_t kRegsControl = 56, kRegsElementwise = 88, kRegsReduce = 56;

template <int D>
struct BwdCfg {
    static_assert(D == 128, "the 128-wide backward");
    static constexpr int kPanels = D / 64;
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kStages = 1;
    static constexpr int kDsBytes = kTile * kTile * 2;
    // TMEM column map.
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D, kColDQ = 0;
    // alignment slack, tiles, dS^T, dP1 staging, per-query constants, barriers, 16 KB guard band
    static constexpr int kSmemBytes = 1024 + 2 * kTileBytes + kStages * 2 * kTileBytes + kDsBytes +
                                      kStagePanels * kStageBytes + kStages * 2 * kTile * 4 + 256 + 16384;
};

// TMEM column (relative to the S^T or dP^T region) of the packed pairs of the
// 16 queries 16ks..16ks+15: block ks/2 keeps its pairs in its own first 16 columns.
__host__ __device__ constexpr uint32_t packed_col(int ks) { return 32u * (ks >> 1) + 8u * (ks & 1); }
// The same queries' P^T pairs: the block's second 16 columns of the dP^T region.
__host__ __device__ constexpr uint32_t packed_p_col(int ks) { return packed_col(ks) + 16u; }

struct BwdBarriers {
    uint64_t kv_full;
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full;
    uint64_t p_full;
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    relation_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_p1, const __grid_constant__ CUtensorMap tm_p2,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_dy,
                           const __grid_constant__ CUtensorMap tm_dq, const KernelProblem kp,
                           const float4* __restrict__ qconst, __nv_bfloat16* __restrict__ dP2,
                           __nv_bfloat16* __restrict__ dV, float* __restrict__ dlambda, unsigned int* status,
                           int head_group) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;                              // P2_j
    uint8_t* sV = sK + C::kTileBytes;                // V_j
    uint8_t* sQ = sV + C::kTileBytes;                // P1_i per stage
    uint8_t* sG = sQ + C::kStages * C::kTileBytes;   // dY_i per stage
    uint8_t* sDS = sG + C::kStages * C::kTileBytes;  // dS^T (bf16), [key row][query], MN-major for dS
    uint8_t* sDQ = sDS + C::kDsBytes;                 // dP1 staging panels (fp32, 128-byte swizzled rows)
    // Per stage and query column pair (2c, 2c+1): -(L + lambda log c) log2(e) of both, then -D k_scale of both.
    float4* sQC = reinterpret_cast<float4*>(sDQ + kStagePanels * kStageBytes);
    BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(sQC + C::kStages * (kTile / 2));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = kp.T;
    const int nt_all = (T + kTile - 1) / kTile;
    int bh, jt;  // head and key tile; low tiles see the most query tiles and go first
    grouped_tile_order(blockIdx.x, kp.BH, nt_all, head_group, bh, jt);
    const int batch = bh / kp.H, head = bh - batch * kp.H;
    const int kv0 = jt * kTile;
    const int nq_all = (T + kTile - 1) / kTile;
    const int i_first = kp.causal ? jt : 0;
    const int n_q = nq_all - i_first;
    const float k_scale = 0.5f * kp.inv_sqrt_d;  // dS^T = dR R'(U) / sqrt(d) with R'(U) carried as 2 R'(U)

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bars->q_full[s], 1);
            ptx::mbar_init(&bars->q_empty[s], 1);
        }
        ptx::mbar_init(&bars->s_full, 1);
        ptx::mbar_init(&bars->p_full, kElemWarps);
        ptx::mbar_init(&bars->dq_full, 1);
        ptx::mbar_init(&bars->dq_free, 128);
        ptx::mbar_init(&bars->mma_done, 1);
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
        // -------------------------------------------------------------- loader
        ptx::regs_dec<kRegsControl>();
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_p1);
            ptx::tma_prefetch_desc(&tm_p2);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::tma_prefetch_desc(&tm_dy);
            ptx::tma_prefetch_desc(&tm_dq);
            ptx::mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTileBytes);
            for (int p = 0; p < C::kPanels; ++p) {
                ptx::tma_load_operand(sK + p * kPanelBytes, &tm_p2, &bars->kv_full, p * 64, kv0, bh, head, batch,
                                      kp.layout == 0);
                ptx::tma_load_operand(sV + p * kPanelBytes, &tm_v, &bars->kv_full, p * 64, kv0, bh, head, batch,
                                      kp.layout == 0);
            }
        }
        // Per-query constants of this head, 64 float4 (1 KB) per query tile.
        const float4* qsrc = qconst + (size_t)bh * (size_t)(qconst_rows(T) / 2);
        int it = 0;
        for (; it < n_q; ++it) {
            const int s = it % C::kStages;
            const int i = i_first + it;
            if (it >= C::kStages &&
                !ptx::mbar_wait_warp(&bars->q_empty[s], ((it / C::kStages) - 1) & 1, abort_flag, status,
                                     kDevTimeoutEmpty))
                break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(&bars->q_full[s], 2 * C::kTileBytes + kQConstBytes);
                ptx::bulk_load(sQC + s * (kTile / 2), qsrc + i * (kTile / 2), kQConstBytes, &bars->q_full[s]);
                for (int p = 0; p < C::kPanels; ++p) {
                    ptx::tma_load_operand(sQ + s * C::kTileBytes + p * kPanelBytes, &tm_p1, &bars->q_full[s], p * 64,
                                     i * kTile, bh, head, batch, kp.layout == 0);
                    ptx::tma_load_operand(sG + s * C::kTileBytes + p * kPanelBytes, &tm_dy, &bars->q_full[s], p * 64,
                                     i * kTile, bh, head, batch, kp.layout == 0);
                }
            }
        }
        if (lane == 0 && *abort_flag) {
            ptx::mbar_drain(&bars->kv_full, 0, status);
            for (int jj = max(0, it - C::kStages); jj < it; ++jj)
                ptx::mbar_drain(&bars->q_full[jj % C::kStages], (jj / C::kStages) & 1, status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the issue loop; one elected lane issues each MMA.
        // Descriptors are built once; a byte offset is added as offset >> 4.
        ptx::regs_dec<kRegsControl>();
        const uint32_t id_nn = ptx::idesc_bf16(kTile, kTile, false, false);  // S^T, dP^T
        const uint32_t id_tb = ptx::idesc_bf16(kTile, D, false, true);       // dV, dP2 (B MN-major)
        const uint32_t id_dq = ptx::idesc_bf16(kTile, D, true, true);        // dP1 (A, B MN-major)
        const uint64_t dk = ptx::smem_desc(ptx::smem_u32(sK), 16, 1024, ptx::kSwizzle128B);    // K-major views
        const uint64_t dv = ptx::smem_desc(ptx::smem_u32(sV), 16, 1024, ptx::kSwizzle128B);
        const uint64_t dq = ptx::smem_desc(ptx::smem_u32(sQ), 16, 1024, ptx::kSwizzle128B);
        const uint64_t dg = ptx::smem_desc(ptx::smem_u32(sG), 16, 1024, ptx::kSwizzle128B);
        const uint64_t mg = ptx::smem_desc(ptx::smem_u32(sG), kPanelBytes, 1024, ptx::kSwizzle128B);  // MN-major
        const uint64_t mq = ptx::smem_desc(ptx::smem_u32(sQ), kPanelBytes, 1024, ptx::kSwizzle128B);
        const uint64_t mds = ptx::smem_desc(ptx::smem_u32(sDS), kPanelBytes, 1024, ptx::kSwizzle128B);
        const uint64_t mk = ptx::smem_desc(ptx::smem_u32(sK), kPanelBytes, 1024, ptx::kSwizzle128B);
        constexpr uint64_t kStageStep = C::kTileBytes >> 4;
        bool ok = ptx::mbar_wait_warp(&bars->kv_full, 0, abort_flag, status, kDevTimeoutFull);
        for (int it = 0; ok && it < n_q; ++it) {
            const int s = it % C::kStages;
            const uint64_t st = s * kStageStep;
            if (!ptx::mbar_wait_warp(&bars->q_full[s], (it / C::kStages) & 1, abort_flag, status, kDevTimeoutFull)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // dP^T first: its columns held the previous tile's dS^T, which dP2 has
            // read (issued earlier), so it runs while the previous dP1 partial drains.
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t off = (uint64_t)(((ks / 4) * kPanelBytes + (ks % 4) * 32) >> 4);
                ptx::mma_ss_elect(tmem + C::kColDP, dv + off, dg + st + off, id_nn, ks > 0 ? 1u : 0u);
            }
            // S^T reuses the columns of the previous tile's dP1 partial.
            if (it > 0 && !ptx::mbar_wait_warp(&bars->dq_free, (it - 1) & 1, abort_flag, status, kDevTimeoutMma)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t off = (uint64_t)(((ks / 4) * kPanelBytes + (ks % 4) * 32) >> 4);
                ptx::mma_ss_elect(tmem + C::kColS, dk + off, dq + st + off, id_nn, ks > 0 ? 1u : 0u);
            }
            ptx::mma_commit_elect(&bars->s_full);
            if (!ptx::mbar_wait_warp(&bars->p_full, it & 1, abort_flag, status, kDevTimeoutFull)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // dP1 first, into the S^T columns (free now), so that it drains while dV and dP2 run.
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
                ptx::mma_ss_elect(tmem + C::kColDQ, mds + ks * 128, mk + ks * 128, id_dq, ks > 0 ? 1u : 0u);
            ptx::mma_commit_elect(&bars->dq_full);
            // K-step ks covers queries 16ks..16ks+15: 16 rows (2048 bytes) of the MN-major tiles.
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
                ptx::mma_ts_elect(tmem + C::kColDV, tmem + C::kColDP + packed_p_col(ks), mg + st + ks * 128, id_tb,
                                  (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
                ptx::mma_ts_elect(tmem + C::kColDK, tmem + C::kColDP + packed_col(ks), mq + st + ks * 128, id_tb,
                                  (it > 0 || ks > 0) ? 1u : 0u);
            ptx::mma_commit_elect(&bars->q_empty[s]);
        }
        ptx::mma_commit_elect(&bars->mma_done);
        if (lane == 0) ptx::mbar_drain(&bars->mma_done, 0, status);
        __syncwarp();
    } else if (warp < 4) {
        // warps 2-3: no role (they complete the first warpgroup)
        ptx::regs_dec<kRegsControl>();
    } else if (warp < kReduceWarp0) {
        // --------------------------------------------------- elementwise stage
        ptx::regs_inc<kRegsElementwise>();
        const int quarter = warp & 3;
        const int blk = (warp - 4) >> 2;    // query columns 32blk .. 32blk+31
        const int r = quarter * 32 + lane;  // key row within the tile
        const int kv = kv0 + r;
        const bool row_valid = kv < T;
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        ElemConst ec;
        ec.c_nh = make_float2(-0.5f * kp.inv_sqrt_d, -0.5f * kp.inv_sqrt_d);
        ec.c_hl = make_float2(0.5f * kp.inv_sqrt_d * kLog2e, 0.5f * kp.inv_sqrt_d * kLog2e);
        ec.k2 = make_float2(k_scale, k_scale);
        ec.one = make_float2(1.f, 1.f);
        ec.mone = make_float2(-1.f, -1.f);
        ec.c_diag = 0.5f * kp.inv_sqrt_d / kp.tau_S;
        ec.half_inv_tau = 0.5f / kp.tau_S;
        ec.log_count = __logf((float)(kp.causal ? (kv + 1) : T));
        ec.diag_off = (0.5f + kp.lambda * ec.log_count) * kLog2e;  // (1/2 + lambda log c) log2(e)
        ec.row_valid = row_valid;
        ec.causal = kp.causal != 0;
        float dlam = 0.f;  // sum of log(c_i) dR_ii * k_scale over this warp's diagonal entries
        bool ok = true;
        for (int it = 0; ok && it < n_q; ++it) {
            const int s = it % C::kStages;
            const int i = i_first + it;
            if (!ptx::mbar_wait_warp(&bars->s_full, it & 1, abort_flag, status, kDevTimeoutMma)) {
                ok = false;
                break;
            }
            // q_full of this stage has completed (the MMA waited on it before S^T).
            ptx::tc_fence_after();
            const bool diag_tile = (i == jt);
            const int qlimit = T - i * kTile;  // query columns c < qlimit exist
            uint8_t* ds_row = sDS + r * 128;
            uint32_t pp[2][8];  // P^T pairs of both halves: stored once both halves' dP^T columns are read
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int ks = 2 * blk + half;  // 16 queries 16ks .. 16ks+15
                const int col0 = 16 * ks;
                uint32_t sv[16], gv[16];
                ptx::tmem_ld16(lane_addr + C::kColS + col0, sv);
                ptx::tmem_ld16(lane_addr + C::kColDP + col0, gv);
                ptx::tmem_ld_wait();
                ptx::pin_regs(sv);
                ptx::pin_regs(gv);
                const float4* qc = sQC + s * (kTile / 2) + col0 / 2;
                // The masked variant is chosen per warp (uniformly) if any of its rows needs it.
                const bool special = __any_sync(0xffffffffu, diag_tile || qlimit < col0 + 16 || !row_valid);
                uint32_t dp[8];
                if (!special)
                    elementwise16<false>(sv, gv, qc, col0, r, ec, false, 0, pp[half], dp);
                else
                    dlam += elementwise16<true>(sv, gv, qc, col0, r, ec, diag_tile, qlimit, pp[half], dp);
                // dS^T pairs -> dP^T columns this warp has already read.
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                        lane_addr + C::kColDP + packed_col(ks)),
                    "r"(dp[0]), "r"(dp[1]), "r"(dp[2]), "r"(dp[3]), "r"(dp[4]), "r"(dp[5]), "r"(dp[6]), "r"(dp[7])
                    : "memory");
                // dS^T row r, queries 16ks..16ks+15: two 16-byte chunks of the
                // 128-byte swizzled row in panel ks/4.
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int chunk = (2 * ks + h) & 7;
                    const int panel = (2 * ks + h) >> 3;
                    uint4* dst = reinterpret_cast<uint4*>(ds_row + panel * kPanelBytes + ((chunk ^ (r & 7)) << 4));
                    *dst = make_uint4(dp[4 * h], dp[4 * h + 1], dp[4 * h + 2], dp[4 * h + 3]);
                }
            }
            // Both halves' dP^T columns are read: P^T pairs -> the block's second 16 dP^T columns.
#pragma unroll
            for (int half = 0; half < 2; ++half)
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                        lane_addr + C::kColDP + packed_p_col(2 * blk + half)),
                    "r"(pp[half][0]), "r"(pp[half][1]), "r"(pp[half][2]), "r"(pp[half][3]), "r"(pp[half][4]),
                    "r"(pp[half][5]), "r"(pp[half][6]), "r"(pp[half][7])
                    : "memory");
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->p_full);
        }
        if (dlambda != nullptr) {
            // dR_ii = p (g - D) = dr / k_scale; sum log(c_i) dR_ii.
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dlam += __shfl_xor_sync(0xffffffffu, dlam, o);
            if (lane == 0 && dlam != 0.f) atomicAdd(dlambda, dlam / k_scale);
        }
        // Epilogue: block b writes columns 32b .. 32b+31 of the dV and dP2 rows of this key tile.
        if (ok && ptx::mbar_wait_warp(&bars->mma_done, 0, abort_flag, status, kDevTimeoutMma) && 32 * blk < kp.d) {
            ptx::tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                __nv_bfloat16* dst_row = (which == 0 ? dV : dP2) + row_offset(kp, bh, row_valid ? kv : 0);
                const uint32_t col = (which == 0 ? C::kColDV : C::kColDK) + 32 * blk;
                uint32_t ov[32];
                ptx::tmem_ld32(lane_addr + col, ov);
                ptx::tmem_ld_wait();
                ptx::pin_regs(ov);
                if (row_valid) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        store_bf16x8(dst_row, 32 * blk + 8 * k, kp.d,
                                     ptx::pack_bf16x2(as_f(ov[8 * k + 0]), as_f(ov[8 * k + 1])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k + 2]), as_f(ov[8 * k + 3])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k + 4]), as_f(ov[8 * k + 5])),
                                     ptx::pack_bf16x2(as_f(ov[8 * k + 6]), as_f(ov[8 * k + 7])));
                }
            }
        }
    } else {
        // -------------------------------------------------- dP1 partial reduce
        // Per query tile, four 32-column panels: TMEM -> swizzled shared staging
        // -> one TMA bulk reduce-add (fp32) into the accumulator; rows past T are
        // dropped by TMA.  TMEM is released once the last panel is in registers.
        ptx::regs_dec<kRegsReduce>();
        const int quarter = warp & 3;
        const int rq = quarter * 32 + lane;  // query row within the tile
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool leader = (warp == kReduceWarp0) && lane == 0;
        for (int it = 0; it < n_q; ++it) {
            const int i = i_first + it;
            // The four warps take one decision per tile (a 128-thread vote on named
            // barrier 1): if any warp's bounded wait gave up, all four leave together,
            // so none is left at the bar.sync below waiting for a warp that left.
            const bool got = ptx::mbar_wait_warp(&bars->dq_full, it & 1, abort_flag, status, kDevTimeoutMma);
            if (!ptx::bar_vote_all<1, 128>(got)) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < D / 32; ++c0) {
                uint32_t ov[32];
                ptx::tmem_ld32(lane_addr + C::kColDQ + 32 * c0, ov);
                ptx::tmem_ld_wait();
                ptx::pin_regs(ov);
                if (c0 == D / 32 - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(&bars->dq_free);  // every panel has left TMEM
                }
                // The bulk reduce issued two panels ago (same staging buffer) must have
                // finished reading it; bulk groups complete in order.
                if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                asm volatile("bar.sync 1, 128;" ::: "memory");
                uint8_t* stage = sDQ + (c0 & 1) * kStageBytes;
                uint8_t* row = stage + rq * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<uint4*>(row + ((k ^ (rq & 7)) << 4)) =
                        make_uint4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
                ptx::fence_proxy_async_smem();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (leader) {
                    asm volatile(
                        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], "
                        "[%4];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)),
                        "r"(32 * c0), "r"(i * kTile), "r"(bh), "r"(ptx::smem_u32(stage))
                        : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            }
        }
        if (leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_bwd_tc_d(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                            const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                            const TcLaunch& tl, cudaStream_t s) {
    using C = BwdCfg<D>;
    static_assert(C::kSmemBytes <= 232448, "shared memory budget");
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(relation_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // Operands in the problem's layout; heads narrower than D read as D-wide tiles
    // with zero columns.
    CUtensorMap m1, m2, mv, mg;
    const void* bases[4] = {P1, P2, V, dY};
    CUtensorMap* maps[4] = {&m1, &m2, &mv, &mg};
    for (int k = 0; k < 4; ++k) {
        cudaError_t e =
            make_operand_map(maps[k], bases[k], kp.BH / kp.H, kp.H, kp.T, kp.d, kp.layout, 64, 128, true);
        if (e != cudaSuccess) return e;
    }
    // dP1 accumulator: fp32 [BH, T, D], reduced in 32-column (128-byte) swizzled boxes.
    CUtensorMap mq;
    cudaError_t e = make_tensor_map_3d(&mq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, kp.T, kp.BH, 32, 128,
                                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int64_t ctas = kp.BH * ((kp.T + kTile - 1) / kTile);
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    // Heads in flight: as many as fit in three quarters of L2 with P1, P2, V, dY
    // (bf16) and the fp32 dP1 accumulator of each, i.e. 12 T D bytes per head.
    static std::once_flag l2_once;
    static int l2_bytes = 0;
    std::call_once(l2_once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, dev);
    });
    const int64_t per_head = 12 * (int64_t)kp.T * D;
    const int64_t group =
        balanced_head_group(kp.BH, (l2_bytes > 0 ? (int64_t)l2_bytes * 3 / 4 : (int64_t)96 << 20) / per_head);
    relation_bwd_tc_kernel<D><<<dim3((unsigned)ctas), kThreads, C::kSmemBytes, s>>>(
        m1, m2, mv, mg, mq, kp, qconst, (__nv_bfloat16*)dP2, (__nv_bfloat16*)dV, dlambda, tl.status, (int)group);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                          const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                          const TcLaunch& tl, cudaStream_t s, bool padded64) {
    if (kp.d == 48 || kp.d == 60 || kp.d == 64)
        return launch_bwd_tc64(kp, P1, P2, V, qconst, dY, dq_acc, dP2, dV, dlambda, tl, s, padded64);
    if (kp.d == 80 || kp.d == 128)
        return launch_bwd_tc_d<128>(kp, P1, P2, V, qconst, dY, dq_acc, dP2, dV, dlambda, tl, s);
    return cudaErrorInvalidValue;
}

}  // namespace relation

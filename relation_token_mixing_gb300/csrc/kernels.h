// Internal launch functions of the Relation library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace relation {

// float32 CUDA-core path (also instantiated for bf16 storage).  Its grids hold
// the heads in gridDim.y: simt_grid_fits() says whether a problem fits.
bool simt_grid_fits(const KernelProblem& kp);
cudaError_t launch_fwd_simt(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                            void* Y, float* L, cudaStream_t s);
cudaError_t launch_bwd_simt(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                            const float* L, const float* Dw, const void* dY, void* dP1, void* dP2, void* dV,
                            cudaStream_t s);

// Per-query constants of the tensor-core backward kernels, written by the
// preparation stage: for query t of head bh, nlt = -(L_t + lambda log c_t) log2(e)
// and ndk = -D_t / (2 sqrt(d)) with D_t = dY_t . Y_t.  They are stored per query
// pair (2p, 2p+1) as one float4 {nlt(2p), nlt(2p+1), ndk(2p), ndk(2p+1)}, each
// head's rows padded with zeros to a multiple of 128 queries, so that the
// constants of one 128-query tile are a single 1 KB bulk copy.
constexpr int kQConstTile = 128;
__host__ __device__ inline int64_t qconst_rows(int64_t T) { return (T + kQConstTile - 1) / kQConstTile * kQConstTile; }

// Shared backward stages.
// dq_acc (optional) is the fp32 dP1 accumulator [BH, T, dq_w]; it is zeroed.
// pad_dst (bf16, d_h <= 64, dlambda summed elsewhere): also write zero-padded
// contiguous [BH, T, 64] copies of P1, P2, V, dY to pad_dst[0..3] in the same pass.
// qconst == nullptr: D_t is written to Dw [BH, T]; otherwise the per-query
// constants [BH, qconst_rows(T), 2] are written to qconst and Dw is unused.
cudaError_t launch_bwd_prepare(const KernelProblem& kp, bool bf16, const void* P1, const void* P2, const void* V,
                               const void* Y, const float* L, const void* dY, float* Dw, float* dq_acc, int dq_w,
                               float* dlambda, cudaStream_t s, void* const* pad_dst = nullptr, int num_sms = 0,
                               float* qconst = nullptr);
// Input prologue.  RoPE frequencies base^(-2c/d) / (2 pi), c < d/2, as float
// pairs hi + lo (enabled = 0: no rotation, a copy).
struct RopeTable {
    int enabled;
    float hi[64];
    float lo[64];
};
// The tensor-core forward with the input prologue fused into its operand
// loads (bf16, d_h = 64): X1, X2 are rotated and I mixed with the pair partner's
// states in shared memory, so P1, P2 and the mixed states are never stored.
struct TcLaunch;
cudaError_t launch_fwd_tc_prologue(const KernelProblem& kp, const void* X1, const void* X2, const void* I, void* Y,
                                   float* L, const TcLaunch& tl, cudaStream_t s, const RopeTable& tab,
                                   const float* theta, const int32_t* pos0, int pairing);
// The d_h = 64 tensor-core backward main pass with the prologue fused into its
// loads: dX2 (un-rotated) and the gradient of the mixed states dImix (bf16, the
// problem's layout); the dP1 accumulator holds dP1 in rotated coordinates.
cudaError_t launch_bwd_tc64_prologue(const KernelProblem& kp, const void* X1, const void* X2, const void* I,
                                     const float4* qconst, const void* dY, float* dq_acc, void* dX2, void* dImix,
                                     float* dlambda, const TcLaunch& tl, cudaStream_t s, const RopeTable& tab,
                                     const float* theta, const int32_t* pos0, int pairing);
// dX1 = R^T dP1 from the fp32 dP1 accumulator [BH, T, 64] (d_h = 64, bf16 out, the
// problem's layout).
cudaError_t launch_rope_convert(const KernelProblem& kp, const float* dq_acc, void* dX1, const int32_t* pos0,
                                const RopeTable& tab, int num_sms, cudaStream_t s);
// RoPE of two operand tensors (x0 -> y0, x1 -> y1); transpose: the backward.
cudaError_t launch_rope(const KernelProblem& kp, bool bf16, const void* x0, const void* x1, void* y0, void* y1,
                        const int* pos0, const RopeTable& tab, bool transpose, int num_sms, cudaStream_t s);
// Givens head-pair mixing x -> y; transpose: the backward, with d theta (+=)
// accumulated from the mixed states Im when dtheta is not NULL (im_unmixed: Im
// holds the unmixed states, mixed in the kernel).
cudaError_t launch_givens(const KernelProblem& kp, bool bf16, const void* x, const void* Im, void* y,
                          const float* theta, int pairing, bool transpose, float* dtheta, int num_sms,
                          cudaStream_t s, bool im_unmixed = false);
// Relation Cache decode: kp.T is the cache capacity (rows per head of the caches,
// stored in kp.layout); part holds decode_chunks(kp, bf16) x (d + 2) floats per head.
int decode_chunks(const KernelProblem& kp, bool bf16);
// The merge keeps one float per chunk of a head in shared memory (32 KB at most).
constexpr int kDecodeMaxChunks = 8192;
bool decode_grid_fits(const KernelProblem& kp, bool bf16);
// Kernel launches of one decoding step: 1 for streamed caches (partial pass and
// merge in one cluster launch), 2 for direct-read caches (partial pass, merge).
int decode_launches(const KernelProblem& kp, bool bf16);
cudaError_t launch_decode(const KernelProblem& kp, bool bf16, const void* P1n, const void* P2n, const void* Vn,
                          void* P2c, void* Vc, const int* pos, int append, void* Y, float* L, float* part,
                          unsigned int* status, int num_sms, cudaStream_t s);
// n (<= 4) bf16 operand tensors of width kp.d <= 64 (any layout) -> zero-padded
// contiguous [BH, T, 64] copies.
cudaError_t launch_pad_operands(const KernelProblem& kp, const void* const* src, void* const* dst, int n,
                                int num_sms, cudaStream_t s);
// dP1 accumulator [BH, T, dq_w] -> dP1 in the problem's layout and width.
// *out = x[0] + ... + x[n-1] (one thread, index order).
cudaError_t launch_sum_in_order(const float* x, int n, float* out, cudaStream_t s);
cudaError_t launch_convert(const KernelProblem& kp, const float* src, int dq_w, void* dst, bool bf16, int num_sms,
                           cudaStream_t s);

// Linear Relation (bf16 operands, fp32 log-retention G, d <= 64).  The forward's
// workspace holds BH * nseg * (64 * 64 + 64) floats for the segment states.
int linear_segments(const KernelProblem& kp, int num_sms, int* seg_len);
// gate_alog != nullptr: G holds the KDA gate's input r, and g = -exp(A_log) softplus(r + dt_bias)
// per head and channel ([H, d] parameters).
cudaError_t launch_linear_fwd(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* G,
                              void* Y, float* state_out, float* ws, int num_sms, cudaStream_t s,
                              const float* gate_alog = nullptr, const float* gate_dtb = nullptr);
// The backward's workspace adds BH * nseg * 64 * 64 floats (reverse segment states)
// and BH * T floats (p^1 . dq per token).
// reuse_fwd_states: the workspace already holds the forward's segment states.
// With the gate, dG receives dR and gate_dalog / gate_ddtb ([H, d], zeroed by the
// caller) accumulate the parameters' gradients.
cudaError_t launch_linear_bwd(const KernelProblem& kp, const void* P1, const void* P2, const void* V, const float* G,
                              const void* dY, void* dP1, void* dP2, void* dV, float* dG, bool reuse_fwd_states,
                              float* ws, int num_sms, cudaStream_t s, const float* gate_alog = nullptr,
                              const float* gate_dtb = nullptr, float* gate_dalog = nullptr,
                              float* gate_ddtb = nullptr);

// One warp waits on an mbarrier nothing arrives on, through the kernels' bounded
// wait with a limit of limit_ns; the timeout is recorded in *status.
cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t s);

// Tensor-core (tcgen05) bf16 path.
struct TcLaunch {
    int num_sms;
    unsigned int* status;
};
// padded64: P1, P2, V point to zero-padded contiguous [BH, T, 64] copies (d <= 64);
// Y and L are written in the problem's layout and width.
cudaError_t launch_fwd_tc(const KernelProblem& kp, const void* P1, const void* P2, const void* V, void* Y, float* L,
                          const TcLaunch& tl, cudaStream_t s, bool padded64 = false);
// Whether the forward's grid (heads x query-tile pairs) fits the launch limits.
bool fwd_tc_grid_fits(const KernelProblem& kp);
// Whether the tensor-core backward kernel for this head width also sums dlambda.
inline bool bwd_tc_sums_dlambda(int) { return true; }  // both tensor-core kernels sum it from the diagonal
// padded64: P1, P2, V, dY point to zero-padded contiguous [BH, T, 64] copies
// (made by launch_pad_operands) instead of the caller's tensors; dP2 and dV are
// still written in the problem's layout and width.
cudaError_t launch_bwd_tc(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                          const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                          const TcLaunch& tl, cudaStream_t s, bool padded64 = false);
cudaError_t launch_bwd_tc64(const KernelProblem& kp, const void* P1, const void* P2, const void* V,
                            const float4* qconst, const void* dY, float* dq_acc, void* dP2, void* dV, float* dlambda,
                            const TcLaunch& tl, cudaStream_t s, bool padded64 = false);

}  // namespace relation

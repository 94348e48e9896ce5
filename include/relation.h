/*
 * relation.h -- C ABI of the Full Relation operator on NVIDIA GB300 (sm_103a).
 *
 * The operator ("Ask Self, Ask Others: Relation Is All You Need",
 * arXiv:2608.20172, Sec. 3.1 eq.(1)-(3), Appendix A.1.1), per head with
 * P1, P2, V in R^{T x d_h} and one-based row index i:
 *
 *   U_ij = p1_i . p2_j / sqrt(d_h)                               eq.(1)
 *   R_ii = sigmoid(U_ii / tau_S)                       (Self)     eq.(2)
 *   R_ij = SiLU(U_ij) - lambda * log(c_i),  j != i     (Exchange) eq.(2)
 *   R_ij = -inf for j > i when causal                  (mask)     eq.(2)
 *   F_i  = Softmax(R_i),   Y_i = sum_j F_ij V_j                   eq.(3)
 *
 * c_i = i when causal (the paper's count correction "-lambda_l log i",
 * Sec. 3.1 and Appendix A.1.5); c_i = T when non-causal (the paper defines
 * only the causal operator; non-causal uses the visible-candidate count).
 * V is the information state after Givens head mixing (I~ of eq.(4)-(5));
 * P1 and P2 arrive already rotated by RoPE (Appendix B.3).
 *
 * Conventions shared by every entry point:
 *  - Operand tensors (P1, P2, V, Y, dY, dP1, dP2, dV) are contiguous in the
 *    problem's dtype and layout: [B, H, T, d_h] (RELATION_LAYOUT_BHTD) or
 *    [B, T, H, d_h] (RELATION_LAYOUT_BTHD, the heads of a [B, T, H*d_h]
 *    projection output used in place); d_h is innermost in both.  L is always
 *    [B, H, T] float32; the workspace is float32.  All tensor pointers are
 *    device pointers owned by the caller; the library keeps no reference after
 *    a call returns and allocates no device memory per call.
 *  - Every tensor pointer must be 16-byte aligned (RELATION_ERR_MISALIGNED).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and nothing synchronises.  Argument errors are reported before any
 *    work is enqueued; launch failures return RELATION_ERR_CUDA.
 *  - Device-side waits are bounded: if one expires the kernel records the
 *    event in a library-owned device word and returns early;
 *    relation_check_device_status() reports it after the caller synchronises.
 *  - Supported: d_h in {48, 60, 64, 80, 128} (the paper's model widths,
 *    Table 2 and Appendix F.1, plus 128); dtype RELATION_BF16 (tensor-core
 *    path with fp32 accumulation; widths below 64 / 128 run as zero-padded
 *    64- / 128-wide tiles) or RELATION_F32 (fp32 CUDA-core path); any T >= 1;
 *    causal or not; either layout.  Other widths return
 *    RELATION_ERR_UNSUPPORTED.
 *  - Sizes: B, H, T >= 1; B, H, T and B*H at most 2^31 - 1; B*H*T at most
 *    2^33 rows and B*H*T*d_h at most 10^12 elements (beyond:
 *    RELATION_ERR_INVALID_ARGUMENT).  Two paths have tighter launch-grid
 *    limits and return RELATION_ERR_UNSUPPORTED before enqueuing anything:
 *    the bf16 forward takes T <= 16,776,960 and the fp32 forward and backward
 *    B*H <= 65535; decoding's limit is stated with relation_decode.  The
 *    workspace queries return 0 for such problems.
 *  - No entry point throws, aborts, or falls back to the CPU.
 */
#ifndef RELATION_GB300_RELATION_H_
#define RELATION_GB300_RELATION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 2: relation_problem_t gained `layout`. */
#define RELATION_ABI_VERSION 2

typedef enum {
    RELATION_OK = 0,
    RELATION_ERR_INVALID_ARGUMENT = 1, /* bad size, NULL pointer, tau_S <= 0, aliasing */
    RELATION_ERR_UNSUPPORTED = 2,      /* d_h, dtype or size the library has no kernel for */
    RELATION_ERR_MISALIGNED = 3,       /* a tensor pointer is not 16-byte aligned */
    RELATION_ERR_WORKSPACE_TOO_SMALL = 4,
    RELATION_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
    RELATION_ERR_DEVICE_TIMEOUT = 6,   /* a bounded device-side wait expired */
    RELATION_ERR_DEVICE_UNSAFE = 7     /* as 6, and a kernel then also gave up draining its own
                                          copies or products: some may have been in flight when
                                          it returned, so the context should be recreated */
} relation_status_t;

typedef enum { RELATION_F32 = 0, RELATION_BF16 = 1 } relation_dtype_t;

/* Memory order of the operand tensors (see the conventions above). */
typedef enum { RELATION_LAYOUT_BHTD = 0, RELATION_LAYOUT_BTHD = 1 } relation_layout_t;

/* One operator invocation: B*H independent heads of length T and width d_h. */
typedef struct {
    int64_t B, H, T, d_h;
    int32_t dtype;  /* relation_dtype_t */
    float tau_S;    /* Self temperature, > 0 (eq.(2); the paper fixes 2) */
    float lambda;   /* count-correction coefficient lambda_l (eq.(2); init 0.5); 0 disables it */
    int32_t causal; /* nonzero: mask j > i as in eq.(2) */
    int32_t layout; /* relation_layout_t of P1, P2, V, Y, dY, dP1, dP2, dV; L stays [B, H, T] */
} relation_problem_t;

/*
 * Forward, eq.(1)-(3).  Reads P1, P2, V; writes Y [B,H,T,d_h] (dtype) and,
 * when L is not NULL, L [B,H,T] float32 with L_i = log sum_j exp(R_ij) in the
 * paper's convention (correction included).  The backward needs L.
 * Y and L must not overlap any input.
 * bf16 d_h = 60 without a workspace takes the slow route: its 120-byte rows
 * cannot be read by the tensor memory accelerator, so the forward's producer
 * warp copies every tile with 8-byte cp.async (about 4x slower at B16 H8
 * T2048).  Callers that can spare a workspace use relation_fwd_ws below,
 * which pads the operands once and runs the fast kernel; results are
 * identical.
 */
relation_status_t relation_fwd(const relation_problem_t* p, const void* P1, const void* P2,
                               const void* V, void* Y, float* L, void* stream);

/*
 * The same forward with a caller-owned device workspace, for head widths whose
 * rows the tensor memory accelerator cannot step through (bf16 d_h = 60: rows
 * of 120 bytes, not a multiple of 16).  For those, one extra launch first
 * writes zero-padded contiguous [B*H, T, 64] copies of P1, P2 and V into the
 * workspace, and the forward reads its tiles from them; Y and L are written
 * exactly as relation_fwd writes them (the problem's layout and width), and
 * the results are identical to relation_fwd's.  Every other problem needs no
 * workspace: then this equals relation_fwd and workspace may be NULL.
 * relation_fwd_workspace_bytes(p) is the size needed (0 = none, or p invalid).
 * workspace: 16-byte aligned, contents ignored on entry, must not overlap any
 * input or output.  Errors as relation_fwd, plus
 * RELATION_ERR_WORKSPACE_TOO_SMALL.
 */
size_t relation_fwd_workspace_bytes(const relation_problem_t* p);
relation_status_t relation_fwd_ws(const relation_problem_t* p, const void* P1, const void* P2,
                                  const void* V, void* Y, float* L, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Bytes of float32 workspace relation_bwd needs for problem p (0 if p is invalid). */
size_t relation_bwd_workspace_bytes(const relation_problem_t* p);

/*
 * Backward of the forward above (the paper gives no backward; it is the chain
 * rule of eq.(1)-(3)):
 *   D_i = dY_i . Y_i,  dR_ij = F_ij (dY_i . V_j - D_i),
 *   dU_ii = dR_ii S_i (1 - S_i) / tau_S,  dU_ij = dR_ij SiLU'(U_ij)  (j != i),
 *   dP1 = dU P2 / sqrt(d_h),  dP2 = dU^T P1 / sqrt(d_h),  dV = F^T dY,
 *   dlambda = -sum_i log(c_i) sum_{j != i} dR_ij.
 * Inputs: P1, P2, V, the forward's Y and L, upstream dY.  Outputs dP1, dP2,
 * dV [B,H,T,d_h] (dtype) are fully overwritten.  dlambda (device float, may
 * be NULL) is overwritten with the gradient summed over all heads.
 * workspace: device memory of at least relation_bwd_workspace_bytes(p) bytes,
 * 16-byte aligned, owned by the caller, contents ignored on entry.  Outputs
 * and workspace must not overlap each other or any input.
 */
relation_status_t relation_bwd(const relation_problem_t* p, const void* P1, const void* P2,
                               const void* V, const void* Y, const float* L, const void* dY,
                               void* dP1, void* dP2, void* dV, float* dlambda, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * The three stages relation_bwd runs in order, with the same arguments, for
 * callers that time or schedule them separately.  prepare: D_i (on the bf16
 * path folded with L_i and the count correction into the per-query constants
 * the main pass reads, -(L_i + lambda log c_i) log2(e) and -D_i / (2 sqrt(d_h))),
 * dlambda set to zero (and, on the fp32 path, summed), the dP1 accumulator
 * reset and, for bf16 d_h = 60, the zero-padded operand copies in the workspace.  main: the
 * tensor-core (or fp32) pass producing dP2, dV, the dP1 partial sums and, for
 * bf16, dlambda.  finish: dP1 accumulator to dtype.
 */
relation_status_t relation_bwd_prepare(const relation_problem_t* p, const void* P1, const void* P2,
                                       const void* V, const void* Y, const float* L,
                                       const void* dY, void* dP1, void* dP2, void* dV,
                                       float* dlambda, void* workspace, size_t workspace_bytes,
                                       void* stream);
relation_status_t relation_bwd_main(const relation_problem_t* p, const void* P1, const void* P2,
                                    const void* V, const void* Y, const float* L, const void* dY,
                                    void* dP1, void* dP2, void* dV, float* dlambda, void* workspace,
                                    size_t workspace_bytes, void* stream);
relation_status_t relation_bwd_finish(const relation_problem_t* p, const void* P1, const void* P2,
                                      const void* V, const void* Y, const float* L,
                                      const void* dY, void* dP1, void* dP2, void* dV,
                                      float* dlambda, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * relation_bwd for callers that cannot allocate device memory (the paper has
 * no counterpart; this is an interface for the library's users).  Such callers
 * include code whose device memory all belongs to a host framework's own
 * allocator that a C caller cannot reach, and serving loops that must not
 * allocate after start-up because cudaMalloc can synchronise the device.
 * Same arguments and results as relation_bwd without workspace and
 * workspace_bytes: the workspace is a fixed device array inside the library of
 * RELATION_NOALLOC_SCRATCH_BYTES (32 MiB), held on every GPU that loads the
 * library until the process exits.  Problems whose
 * relation_bwd_workspace_bytes() exceeds it return
 * RELATION_ERR_WORKSPACE_TOO_SMALL before any work is enqueued.  The function
 * calls no allocator.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current).  CUDA loads
 * a library's device code lazily by default, so that first call can also be
 * when the array is reserved on the device, which may allocate and synchronise
 * inside the driver: make the first call at start-up, before any stream
 * capture or latency-bound loop; later calls reserve nothing.  All calls share
 * the array and overwrite what they need, so calls whose work overlaps on the
 * GPU race and must not run concurrently.
 */
#define RELATION_NOALLOC_SCRATCH_BYTES (32u << 20)
relation_status_t relation_bwd_noalloc(const relation_problem_t* p, const void* P1, const void* P2,
                                       const void* V, const void* Y, const float* L, const void* dY,
                                       void* dP1, void* dP2, void* dV, float* dlambda, void* stream);

/*
 * One training step of the operator from and to HOST memory: relation_fwd
 * then relation_bwd (eq.(1)-(3) and their chain rule) on inputs P1, P2, V and
 * upstream dY held in host memory, with Y, dP1, dP2, dV (and L when not NULL)
 * written to host memory and dlambda (a host float, may be NULL) set to the
 * gradient summed over all heads.  The paper has no counterpart: this is the
 * library's entry point for callers whose tensors live on the host.
 * Heads are independent, so the batch is processed in `chunks` slices of
 * B / chunks whole sequences (chunks must divide B).  Slice c+1 is copied in,
 * and slice c-1 copied out, on two streams of the library's own while slice c
 * is computed on `stream`.  So with page-locked (pinned) host buffers most of
 * the host <-> device traffic overlaps the kernels; pageable buffers give the
 * same results with the copies serialised.  Results equal relation_fwd's and
 * relation_bwd's on the whole batch up to the order of floating-point
 * accumulation (dP1's partial sums; dlambda's slice sums are added in slice
 * order).
 * Host tensors: the problem's layout and dtype, whole [B, ...] tensors, any
 * alignment; inputs must not overlap outputs.  device_buffer: device memory
 * of at least relation_step_host_device_bytes(p, chunks) bytes (0 = p or
 * chunks unsupported), 16-byte aligned, owned by the caller, contents ignored.
 * The call returns once the work is queued; `stream` (NULL: the legacy default
 * stream) completes after all of it, so the host results are ready once that
 * stream has been synchronised.  Calls on one stream may reuse one device buffer
 * back to back; a buffer passed to calls on different streams must be ordered by
 * the caller (the second call's stream waiting for the first's).  Enqueueing holds
 * a per-device lock: calls from several threads are queued one after another.  On an error return, part of
 * the work may already be queued: synchronise the device before reusing the
 * buffers.
 */
size_t relation_step_host_device_bytes(const relation_problem_t* p, int chunks);
relation_status_t relation_step_host(const relation_problem_t* p, const void* P1, const void* P2,
                                     const void* V, const void* dY, void* Y, float* L, void* dP1,
                                     void* dP2, void* dV, float* dlambda, int chunks,
                                     void* device_buffer, size_t device_bytes, void* stream);

/*
 * Relation Cache decoding (Sec. 5.3 eq.(18); Appendix A.5): one autoregressive
 * step for B*H heads.  The cache of a head holds the P2 rows and information
 * states I~ of the tokens already processed; only the new Relation row is
 * formed:
 *   U_j = p1_new . p2_j / sqrt(d_h) for j = 1..t (cached) and j = t+1 (p2_new),
 *   R_{t+1} = sigmoid(U_{t+1} / tau_S) (Self),
 *   R_j = SiLU(U_j) - lambda log(t+1) for j <= t (Exchange, c = t+1),
 *   Y = sum_j Softmax(R)_j I~_j,
 * i.e. exactly row t+1 of the causal relation_fwd over the t+1 tokens.
 *
 * p: B, H, d_h, dtype, tau_S, lambda, layout as for relation_fwd; p->T is the
 *    cache capacity (rows per head); p->causal is ignored (decoding is causal).
 *    The capacity is read in at most 8192 chunks: T <= 2,097,152 for bf16
 *    d_h 48 or 64 in the [B, H, T, d_h] layout; 1,048,576 for bf16 d_h 80 or
 *    128 and fp32 d_h 48, 60 or 64 in that layout; 524,288 for fp32 d_h 80 or
 *    128 in that layout; 4,194,304 for [B, T, H, d_h] caches and bf16 d_h 60.
 *    A larger capacity returns RELATION_ERR_UNSUPPORTED.
 * P1_new, P2_new, V_new: [B, H, d_h] (dtype), the new token's states.
 * P2_cache, V_cache: [B, H, T, d_h] or [B, T, H, d_h] per p->layout (dtype);
 *    rows 0 .. positions[b]-1 of batch b hold the history.
 * positions: device int32 [B], t = number of cached tokens of batch b
 *    (0 <= t < T; t = 0 is the first token, whose output is V_new exactly).
 *    A position outside [0, T) is reported by relation_check_device_status()
 *    as RELATION_ERR_INVALID_ARGUMENT and that batch's outputs are not written.
 * append: nonzero also stores P2_new and V_new at row t of the caches (the
 *    cache update of Appendix A.5.3), after which positions[b] + 1 is the next
 *    step's position; the library does not change `positions`.
 * Y: [B, H, d_h] (dtype).  L: optional [B, H] float32 log-normaliser of the row.
 * workspace: at least relation_decode_workspace_bytes(p) bytes, float32
 *    partial results (used by direct-read caches; streamed caches merge in
 *    shared memory and leave it untouched).  Outputs must not overlap inputs
 *    or caches.
 * Caches in the [B, H, T, d_h] layout whose rows are a multiple of 16 bytes
 * are streamed: one launch, a thread-block cluster of up to 8 CTAs per head
 * whose CTAs each read a share of the history and merge in distributed shared
 * memory.  Other caches take two launches (per-chunk partials, then one merge
 * per head).
 */
size_t relation_decode_workspace_bytes(const relation_problem_t* p);
relation_status_t relation_decode(const relation_problem_t* p, const void* P1_new, const void* P2_new,
                                  const void* V_new, void* P2_cache, void* V_cache, const int32_t* positions,
                                  int append, void* Y, float* L, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * Input prologue of the operator and its backward.
 *  - RoPE on the relation coordinates (Sec. 3.1 below eq.(1); Appendix B.3: full
 *    head width, base 10^4 in the paper; the information states stay
 *    unrotated): coordinate c < d_h/2 turns together with c + d_h/2 by the
 *    angle pos * rope_base^(-2c/d_h), pos = pos0[b] + t the zero-based token
 *    position (the pages do not fix the pairing of coordinates; this is the
 *    half-split form).  rope_base <= 0 disables the rotation (a copy).
 *  - Givens mixing of the information states of adjacent head pairs (Sec. 3.2
 *    eq.(4); Appendix A.2.2-A.2.3): for pair k = (a, b) with angle theta[k],
 *      I~a = cos(theta) Ia - sin(theta) Ib,  I~b = sin(theta) Ia + cos(theta) Ib,
 *    pairing 0: (1,2), (3,4), ..., (H-1,H); pairing 1: (2,3), ..., (H,1)
 *    (one-based heads, alternating between layers).  H must be even.
 * relation_prologue_fwd: X1, X2, I (unrotated / unmixed, [B,H,T,d_h] per
 *   p->layout, dtype) -> P1, P2, I_mixed (the operator's P1, P2, V).
 * relation_prologue_bwd: the operator's dP1, dP2, dV (= dI_mixed) and the
 *   forward's I_mixed -> dX1, dX2, dI and, when dtheta is not NULL, dtheta
 *   [H/2] float32 (overwritten; dtheta_k = sum dI~b . I~a - dI~a . I~b).
 * theta: device float32 [H/2].  pos0: optional device int32 [B] (NULL: 0),
 * e.g. the decode position.  Outputs must not overlap inputs.  Two kernel
 * launches each (HBM-bound elementwise passes).
 */
relation_status_t relation_prologue_fwd(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        void* P1, void* P2, void* I_mixed, void* stream);
relation_status_t relation_prologue_bwd(const relation_problem_t* p, const void* dP1, const void* dP2,
                                        const void* dI_mixed, const void* I_mixed, const float* theta, int pairing,
                                        float rope_base, const int32_t* pos0, void* dX1, void* dX2, void* dI,
                                        float* dtheta, void* stream);

/*
 * The operator with its input prologue fused into the tensor-core forward's
 * operand loads (same passages as above): the results of relation_prologue_fwd
 * followed by relation_fwd, without storing P1, P2 or I_mixed.  The kernel
 * loads tiles of X1, X2 and of I for the head and its Givens partner; two of its
 * warps rotate the X1 / X2 tiles (RoPE, rope_base and pos0 as above) and mix the
 * I tiles in shared memory before the tensor core reads them, each rotated or
 * mixed value rounded once to bf16 as the standalone prologue rounds it.
 * X1, X2, I: [B,H,T,d_h] per p->layout.  Y, L as in relation_fwd.  theta,
 * pairing, rope_base, pos0 as in relation_prologue_fwd.  Supported: dtype
 * RELATION_BF16, d_h = 64, H even (else RELATION_ERR_UNSUPPORTED or
 * RELATION_ERR_INVALID_ARGUMENT); one kernel launch.
 */
relation_status_t relation_fwd_prologue(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        void* Y, float* L, void* stream);
/*
 * The matching backward: the results of relation_bwd followed by
 * relation_prologue_bwd (dX1, dX2, dI, and dtheta when not NULL; dlambda as in
 * relation_bwd), from X1, X2, I and the forward's Y, L.  The main pass loads X1,
 * X2, I like the fused forward and rotates / mixes them in shared memory; dX2
 * leaves it un-rotated, dX1 is un-rotated while the dP1 accumulator is converted,
 * and a last pass takes the gradient of the mixed states to dI and dtheta (the
 * mixed states for dtheta recomputed from I).  dX1, dX2, dI: bf16 [B,H,T,d_h]
 * per p->layout, fully overwritten; dtheta [H/2] float32, overwritten.
 * workspace: at least relation_bwd_prologue_workspace_bytes(p) bytes (relation_bwd's
 * workspace followed by a bf16 tensor for the mixed states' gradient), 16-byte
 * aligned, not overlapping any argument.  Supported as relation_fwd_prologue;
 * four kernel launches.
 */
size_t relation_bwd_prologue_workspace_bytes(const relation_problem_t* p);
relation_status_t relation_bwd_prologue(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        const void* Y, const float* L, const void* dY, void* dX1, void* dX2, void* dI,
                                        float* dtheta, float* dlambda, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * Linear Relation ("Ask Self, Ask Others", Sec. 5.2 eq.(15)-(17); Appendix
 * A.4): per head a d_h x d_h relational state C with C_0 = 0 and channel-wise
 * retention alpha_t = exp(G_t) (Sec. 5.2 eq.(16); the projection producing G
 * from the token is the caller's), read before it is written:
 *
 *   S_t  = sigmoid(p1_t . p2_t / (tau_S sqrt(d_h)))                  eq.(15)
 *   p^_t = p_t / ||p_t||   (a zero vector stays zero)
 *   C-_t = Diag(alpha_t) C_{t-1},  E_t = S_t (C-_t)^T p^1_t,  Y_t = I~_t + E_t,
 *   C_t  = C-_t + S_t p^2_t I~_t^T                                    eq.(17)
 *
 * P1, P2 (after RoPE), I (= I~) and Y: [B,H,T,d_h] or [B,T,H,d_h] per
 * p->layout, bfloat16.  G: log-retention (<= 0 for alpha in (0, 1]; any
 * finite value is accepted), float32, same layout.  p->lambda and p->causal
 * are ignored (the recurrence is causal by construction).  Supported: d_h in
 * {48, 60, 64}, dtype RELATION_BF16 (fp32 state and accumulation); others
 * return RELATION_ERR_UNSUPPORTED.
 *
 * relation_linear_fwd: Y and, when `state` is not NULL, the final state C_T
 *   per head, float32 [B, H, d_h, d_h] (row = key channel, column = value
 *   channel).  1 to 3 kernel launches (segment state pass and scan only when
 *   B*H is too small to fill the GPU).
 * relation_linear_bwd: from dY (bf16, like Y): dP1, dP2, dI (bf16) and dG
 *   (float32), all fully overwritten (gradients of sum(Y * dY) with C_0 = 0).
 *   2 to 6 kernel launches (the forward and reverse segment state passes and
 *   scans only when B*H is too small to fill the GPU).  states_from_forward
 *   nonzero: the workspace still holds what relation_linear_fwd left in it for
 *   the same problem and inputs (as in a training step that keeps the workspace
 *   from the forward to the backward), and the forward segment states are reused
 *   instead of recomputed; any other use gives wrong gradients.  0: recompute.
 * relation_linear_workspace_bytes: the float32 workspace both directions need
 *   (16-byte aligned, caller-owned, contents need not be preserved between
 *   calls); 0 on invalid arguments.
 * Outputs must not overlap inputs or each other.
 */
size_t relation_linear_workspace_bytes(const relation_problem_t* p);
relation_status_t relation_linear_fwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                      const float* G, void* Y, float* state, void* workspace,
                                      size_t workspace_bytes, void* stream);
relation_status_t relation_linear_bwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                      const float* G, const void* dY, void* dP1, void* dP2, void* dI, float* dG,
                                      int states_from_forward, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * Linear Relation with the KDA-style retention gate fused into its kernels
 * ("Ask Self, Ask Others", Sec. 5.2 eq.(16); Appendix A.4.1): instead of G the
 * gate's input R (the per-token projection output r_t; float32, laid out as G)
 * and per-head, per-channel parameters A_log, dt_bias (float32 [H, d_h]):
 *   g = -exp(A_log) * softplus(r + dt_bias),   alpha = exp(g) in (0, 1].
 * relation_linear_fwd_gate: relation_linear_fwd with G = g (computed as each
 *   chunk is read; g is never stored).
 * relation_linear_bwd_gate: relation_linear_bwd with dR (float32, laid out as R,
 *   fully overwritten) in place of dG, plus dA_log and d_dt_bias [H, d_h]
 *   (float32, overwritten: sums over batches and tokens).  states_from_forward
 *   refers to relation_linear_fwd_gate with the same arguments.
 * Same support, workspace, launches and errors as the ungated calls; A_log and
 * dt_bias must not be NULL and must not overlap any tensor argument.
 */
relation_status_t relation_linear_fwd_gate(const relation_problem_t* p, const void* P1, const void* P2,
                                           const void* I, const float* R, const float* A_log, const float* dt_bias,
                                           void* Y, float* state, void* workspace, size_t workspace_bytes,
                                           void* stream);
relation_status_t relation_linear_bwd_gate(const relation_problem_t* p, const void* P1, const void* P2,
                                           const void* I, const float* R, const float* A_log, const float* dt_bias,
                                           const void* dY, void* dP1, void* dP2, void* dI, float* dR, float* dA_log,
                                           float* d_dt_bias, int states_from_forward, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * Reads and clears the device status word of the current device.  Call after
 * synchronising the streams used.  Returns RELATION_OK,
 * RELATION_ERR_DEVICE_TIMEOUT (a bounded wait expired; outputs of the calls
 * since the last check are invalid), RELATION_ERR_DEVICE_UNSAFE (a wait expired
 * and the kernel's second, also bounded, wait for its own copies or products in
 * flight expired too, so it returned while they may still have been writing
 * shared memory: discard the outputs and recreate the context),
 * RELATION_ERR_INVALID_ARGUMENT (a decode position outside its cache) or
 * RELATION_ERR_CUDA.
 */
relation_status_t relation_check_device_status(void);

/*
 * Self-test of the failure-detection path: enqueues one kernel on `stream` in
 * which a warp waits, through the same bounded wait every kernel uses, on a
 * barrier that nothing completes.  After limit_ms milliseconds (1..10000) the
 * wait gives up, records a timeout in the device status word and the kernel
 * returns; nothing faults or hangs and the context stays usable.  After the
 * caller synchronises, relation_check_device_status() returns
 * RELATION_ERR_DEVICE_TIMEOUT (and clears the word).  Returns
 * RELATION_ERR_INVALID_ARGUMENT for a limit outside 1..10000 ms.
 */
relation_status_t relation_selftest_wait_timeout(uint32_t limit_ms, void* stream);

/* Number of kernel launches the last successful call on this thread enqueued. */
int relation_last_launch_count(void);

/* Static description of a status code; never NULL. */
const char* relation_status_string(relation_status_t s);

/* RELATION_ABI_VERSION of the loaded library. */
int relation_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RELATION_GB300_RELATION_H_ */

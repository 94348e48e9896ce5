// Relation Cache decoding ("Ask Self, Ask Others: Relation Is All You Need",
// Sec. 5.3 eq.(18) and Appendix A.5): at autoregressive position t+1 (one
// based) only the new Relation row is formed, from the new p1 against the
// cached P2_{1:t} and the new p2 (the Self entry), and it transports the cached
// information states I~_{1:t} and the new one:
//   U_j = p1 . p2_j / sqrt(d),  R_{t+1} = sigmoid(U_{t+1} / tau_S),
//   R_j = SiLU(U_j) - lambda log(t+1) (j <= t),  Y = sum_j softmax(R)_j I~_j.
// The cache update appends p2_{t+1} and I~_{t+1} (Appendix A.5.3).
//
// The pass is HBM-bound (it reads 2 t d values per head), so it runs on CUDA
// cores in fp32.  Caches whose rows bulk copies can move (contiguous
// [B, H, T, d], rows a multiple of 16 bytes) are streamed: about two CTAs per
// SM, each taking a share of a head's cached rows through a ring of shared-memory
// stages with an online softmax per lane group.  Other caches are split into
// chunks read directly (16- or 8-byte loads).  One CTA per head then merges the
// shares, launched as a programmatic dependent of the partial pass.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace relation {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float sigmoid_exact(float x) {
    if (x >= 0.f) return 1.f / (1.f + expf(-x));
    const float e = expf(x);
    return e / (1.f + e);
}

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[0];
    for (int w = 1; w < kThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
    return v;
}

// Vector of VEC consecutive elements as fp32 (16-byte or 8-byte loads).
template <typename Tin, int VEC>
__device__ __forceinline__ void load_vec(const Tin* p, float (&v)[VEC]) {
    if constexpr (sizeof(Tin) == 2 && VEC == 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else if constexpr (sizeof(Tin) == 2 && VEC == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        const uint32_t w[2] = {u.x, u.y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else {
        static_assert(sizeof(Tin) == 4 && VEC == 4, "fp32 rows are read 16 bytes at a time");
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x;
        v[1] = u.y;
        v[2] = u.z;
        v[3] = u.w;
    }
}

// VEC consecutive elements as fp32 from 16-byte pieces (bf16 VEC = 8 or 16,
// fp32 VEC = 4 or 8); `Shared`: p points into shared memory, else global (read
// through the non-coherent path).
template <typename Tin, int VEC, bool Shared>
__device__ __forceinline__ void load_vec16(const Tin* p, float (&v)[VEC]) {
    constexpr int kPer = 16 / (int)sizeof(Tin);  // elements per 16-byte piece
    static_assert(VEC % kPer == 0, "whole 16-byte pieces");
#pragma unroll
    for (int piece = 0; piece < VEC / kPer; ++piece) {
        const uint4 u = Shared ? *reinterpret_cast<const uint4*>(p + piece * kPer)
                               : __ldg(reinterpret_cast<const uint4*>(p + piece * kPer));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (sizeof(Tin) == 2) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
                v[piece * kPer + 2 * k] = f.x;
                v[piece * kPer + 2 * k + 1] = f.y;
            } else {
                v[piece * kPer + k] = __uint_as_float(w[k]);
            }
        }
    }
}

// sigmoid and exp for the bf16-cache streaming pass on the special-function unit
// (ex2.approx, rcp.approx: relative errors near 2^-22, far below the bf16 inputs'
// 2^-9); the fp32 path keeps expf.
template <bool kFast>
__device__ __forceinline__ float exp_f(float x) {
    if constexpr (kFast) return ptx::ex2_approx(x * 1.4426950408889634f);
    return expf(x);
}
template <bool kFast>
__device__ __forceinline__ float sigmoid_f(float x) {
    if constexpr (kFast) return __frcp_rn(1.f + exp_f<true>(-x));
    return sigmoid_exact(x);
}

// One bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    ptx::bulk_load(dst, src, bytes, bar);
}

// Cluster barrier halves (every thread of every CTA of the cluster takes part).
// The relaxed arrive only marks that the CTA has started (so that its shared
// memory may be written by the cluster once the phase completes); the release /
// acquire pair makes shared-memory writes before it visible to reads after it.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Writes v to the float at the same shared-memory offset as `p` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32(float* p, int rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ptx::smem_u32(p)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Partial pass: CTA (bh, chunk) handles keys [chunk*C, min(chunk*C + C, t+1));
// key t is the new token (read from the new-row tensors).  A group of G lanes
// reads one key row, VEC elements per lane (lane li owns columns li*VEC ..),
// so one warp instruction covers 32/G whole rows.  Writes (m, l, o[d]) of the
// chunk to part[bh][chunk].
template <typename Tin, int VEC, int G>
__global__ void __launch_bounds__(kThreads) decode_partial_kernel(
    KernelProblem kp, const Tin* __restrict__ P1n, const Tin* __restrict__ P2n, const Tin* __restrict__ Vn,
    Tin* __restrict__ P2c, Tin* __restrict__ Vc, const int* __restrict__ pos, int append, int chunk,
    float* __restrict__ part, unsigned int* status) {
    constexpr int kGroups = kThreads / G;  // key rows in flight per CTA step
    extern __shared__ float sm[];
    float* sr = sm;           // chunk scores
    float* red = sr + chunk;  // per-warp reductions (8)
    float* oacc = red + 8;    // kGroups x d partial outputs
    const int64_t bh = blockIdx.x;
    const int b = (int)(bh / kp.H);
    const int d = kp.d;
    const int t = pos[b];
    float* out = part + ((size_t)bh * gridDim.y + blockIdx.y) * (size_t)(d + 2);
    if (t < 0 || t >= kp.T) {  // position outside the cache: reported, head skipped
        if (threadIdx.x == 0) {
            record_status(status, kDevBadPosition);
            out[0] = -INFINITY;
            out[1] = 0.f;
        }
        return;
    }
    const int n = t + 1;  // keys visible to the new row
    const int j0 = blockIdx.y * chunk, j1 = min(n, j0 + chunk);
    const size_t new_off = (size_t)bh * d;  // [B, H, d] new-row tensors
    if (append && blockIdx.y == 0)          // the new row goes to cache row t, which no CTA reads
        for (int c = threadIdx.x; c < d; c += kThreads) {
            P2c[row_offset(kp, bh, t) + c] = P2n[new_off + c];
            Vc[row_offset(kp, bh, t) + c] = Vn[new_off + c];
        }
    if (j0 >= j1) {
        if (threadIdx.x == 0) {
            out[0] = -INFINITY;
            out[1] = 0.f;
        }
        return;
    }
    const int grp = threadIdx.x / G, li = threadIdx.x % G;
    const int col = li * VEC;
    const bool active = col < d;
    float q[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) q[k] = 0.f;
    if (active) load_vec<Tin, VEC>(P1n + new_off + col, q);
    const float corr = kp.lambda * logf((float)n);  // lambda log c, c = t+1
    // Pass 1: scores.  The loop bounds are the same for every thread (the shuffles
    // need the whole warp); a group past the chunk end only idles.
    float mloc = -INFINITY;
    for (int base = j0; base < j1; base += kGroups) {
        const int j = base + grp;
        float dot = 0.f;
        if (j < j1 && active) {
            float kv[VEC];
            load_vec<Tin, VEC>(((j == t) ? P2n + new_off : P2c + row_offset(kp, bh, j)) + col, kv);
#pragma unroll
            for (int k = 0; k < VEC; ++k) dot = fmaf(q[k], kv[k], dot);
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (j < j1) {
            const float u = dot * kp.inv_sqrt_d;
            const float r = (j == t) ? sigmoid_exact(u / kp.tau_S) : u * sigmoid_exact(u) - corr;
            if (li == 0) sr[j - j0] = r;
            mloc = fmaxf(mloc, r);
        }
    }
    const float m = block_reduce(mloc, red, true);  // also orders the score stores
    // Pass 2: weights and the weighted sum of the information states.
    float o[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) o[k] = 0.f;
    float lloc = 0.f;
    for (int j = j0 + grp; j < j1; j += kGroups) {  // no shuffles here
        const float p = expf(sr[j - j0] - m);
        if (li == 0) lloc += p;
        if (active) {
            float vv[VEC];
            load_vec<Tin, VEC>(((j == t) ? Vn + new_off : Vc + row_offset(kp, bh, j)) + col, vv);
#pragma unroll
            for (int k = 0; k < VEC; ++k) o[k] = fmaf(p, vv[k], o[k]);
        }
    }
    const float l = block_reduce(lloc, red, false);
    if (active) {
        float* dst = oacc + (size_t)grp * d + col;
#pragma unroll
        for (int k = 0; k < VEC; ++k) dst[k] = o[k];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < d; c += kThreads) {
        float acc = 0.f;
        for (int g = 0; g < kGroups; ++g) acc += oacc[(size_t)g * d + c];
        out[2 + c] = acc;
    }
    if (threadIdx.x == 0) {
        out[0] = m;
        out[1] = l;
    }
}

// Streaming pass for contiguous [B, H, T, d] caches whose rows are a multiple of
// 16 bytes.  The S CTAs of a head form one thread-block cluster; CTA s takes an
// equal share of whole chunks of the cached rows 0..t-1 (CH rows per chunk) and
// streams them through a ring of kStreamStages shared-memory stages, each filled
// by two bulk copies (P2 rows, I~ rows) completing on the stage's mbarrier, so
// the copies of the next chunks are in flight while the current one is scored
// (a stage left without a chunk gets a plain arrive, which ends the loop).  Every
// group of G lanes keeps an online softmax over its rows (running max m, sum l
// and weighted sum o of the I~ rows: the scan of Sec. 5.1 eq.(12)); the groups
// merge into the CTA's (m, l, o), which every CTA writes into CTA 0's shared
// memory; after one cluster barrier CTA 0 merges the S results and writes Y and
// L.  The new token's rows come by bulk copies issued before anything else: its
// P1 row to every CTA, its P2 and I~ rows to CTA 0, which scores the Self entry
// and appends the row to the cache row t (which no CTA reads).
constexpr int kStreamStages = 3;
constexpr int kEmptyStage = -2;    // a stage filled with a wrongly guessed chunk (scored as nothing)
constexpr int kMaxCluster = 8;    // portable cluster size
constexpr int kStreamMaxD = 128;  // widest head the streaming pass takes

template <typename Tin, int VEC, int G>
__global__ void __launch_bounds__(kThreads, 2) decode_cluster_kernel(
    KernelProblem kp, const Tin* __restrict__ P1n, const Tin* __restrict__ P2n, const Tin* __restrict__ Vn,
    Tin* __restrict__ P2c, Tin* __restrict__ Vc, const int* __restrict__ pos, int append, int ch,
    Tin* __restrict__ Y, float* __restrict__ L, unsigned int* status) {
    constexpr int kGroups = kThreads / G;
    constexpr int kWarps = kThreads / 32;
    constexpr bool kFast = sizeof(Tin) == 2;
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ __align__(8) uint64_t full[kStreamStages];
    __shared__ __align__(8) uint64_t new_full;
    __shared__ int stage_chunk[kStreamStages];  // the chunk in each stage; -1: none (the loop ends)
    __shared__ int abort_flag;
    __shared__ __align__(16) Tin new_rows[3 * kStreamMaxD];  // the new token's P1, P2 and I~ rows
    // CTA 0's copy receives every CTA's (m, l, o); the same offsets in the other
    // CTAs stay unused.
    __shared__ float cl_m[kMaxCluster], cl_l[kMaxCluster];
    __shared__ __align__(16) float cl_o[kMaxCluster * kStreamMaxD];
    const int d = kp.d;
    const size_t row_bytes = (size_t)d * sizeof(Tin);
    const size_t stage_bytes = 2 * (size_t)ch * row_bytes;
    // After the stream the stage area holds the merge of the warps: per warp o
    // (kWarps x d), m and l.
    float* og = reinterpret_cast<float*>(smb);
    float* gm = og + (size_t)kWarps * d;
    float* gl = gm + kWarps;
    const int64_t bh = blockIdx.x;
    const int b = (int)(bh / kp.H);
    const int S = (int)gridDim.y, sidx = (int)blockIdx.y;  // cluster = the S CTAs of head bh
    const size_t new_off = (size_t)bh * d;                 // [B, H, d] new-row tensors
    // The first stage is filled before the position is known, with the first chunk
    // this CTA would take were the cache full (t = T-1, rows of the allocation only);
    // once t is known, a wrong guess is consumed as an empty stage.
    const int spec_n = (kp.T - 1 + ch - 1) / ch;  // chunks of a full cache
    const int spec_c = sidx * ((spec_n + S - 1) / S);
    const bool spec = spec_c < spec_n;
    if (threadIdx.x == 0) {
        for (int k = 0; k < kStreamStages; ++k) ptx::mbar_init(&full[k], 1);
        ptx::mbar_init(&new_full, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
        if (spec) {
            const int j0 = spec_c * ch;
            const uint32_t bytes = (uint32_t)((min(kp.T - 1, j0 + ch) - j0) * row_bytes);
            stage_chunk[0] = spec_c;
            ptx::mbar_arrive_expect_tx(&full[0], 2 * bytes);
            bulk_copy_g2s(smb, P2c + row_offset(kp, bh, j0), bytes, &full[0]);
            bulk_copy_g2s(smb + (size_t)ch * row_bytes, Vc + row_offset(kp, bh, j0), bytes, &full[0]);
        }
        ptx::mbar_arrive_expect_tx(&new_full, (uint32_t)row_bytes * (sidx == 0 ? 3u : 1u));
        bulk_copy_g2s(new_rows, P1n + new_off, (uint32_t)row_bytes, &new_full);
        if (sidx == 0) {
            bulk_copy_g2s(new_rows + kStreamMaxD, P2n + new_off, (uint32_t)row_bytes, &new_full);
            bulk_copy_g2s(new_rows + 2 * kStreamMaxD, Vn + new_off, (uint32_t)row_bytes, &new_full);
        }
    }
    const int t = pos[b];
    const bool t_ok = t >= 0 && t < kp.T;
    const int n_all = t_ok ? (t + ch - 1) / ch : 0;  // chunks of cached rows
    const int per = (n_all + S - 1) / S;
    const int k0 = sidx * per;
    const int nck = max(0, min(n_all, k0 + per) - k0);
    // The guess is right when this CTA's first chunk is the one guessed (then the copy
    // holds at least its rows); otherwise stage 0 is marked empty before anyone reads it.
    const bool spec_ok = spec && nck > 0 && k0 == spec_c;
    if (threadIdx.x == 0 && spec && !spec_ok) stage_chunk[0] = kEmptyStage;
    __syncthreads();  // the barriers are initialised, stage 0's chunk is settled
    if (!t_ok) {  // position outside the cache (the whole cluster returns): reported, not written
        if (threadIdx.x == 0) {
            if (sidx == 0) record_status(status, kDevBadPosition);
            // The copies land before the CTA's memory is released.
            ptx::mbar_drain(&new_full, 0, status);
            if (spec) ptx::mbar_drain(&full[0], 0, status);
        }
        return;
    }
    cluster_arrive_relaxed();  // this CTA has started; waited on before the first remote write
    // Fill f carries chunk k0 + f - lag (lag 1 after an empty stage 0), none past the share.
    const int lag = (spec && !spec_ok) ? 1 : 0;
    // Thread 0 fills stage f % kStreamStages for the f-th time: chunk c, or none (c < 0).
    auto fill = [&](int f, int c) {
        const int st = f % kStreamStages;
        uint64_t* bar = &full[st];
        stage_chunk[st] = c;
        if (c < 0) {
            ptx::mbar_arrive(bar);
            return;
        }
        const int j0 = c * ch;
        const uint32_t bytes = (uint32_t)((min(t, j0 + ch) - j0) * row_bytes);
        uint8_t* dst = smb + (size_t)st * stage_bytes;
        ptx::mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_copy_g2s(dst, P2c + row_offset(kp, bh, j0), bytes, bar);
        bulk_copy_g2s(dst + (size_t)ch * row_bytes, Vc + row_offset(kp, bh, j0), bytes, bar);
    };
    auto chunk_of_fill = [&](int f) { return (f - lag >= 0 && f - lag < nck) ? k0 + f - lag : -1; };
    int fills = spec ? 1 : 0;  // thread 0: stage fills issued (the guessed one included)
    if (threadIdx.x == 0)
        for (; fills < kStreamStages; ++fills) fill(fills, chunk_of_fill(fills));
    const int grp = threadIdx.x / G, li = threadIdx.x % G;
    const int col = li * VEC;
    const bool active = col < d;
    const float corr = kp.lambda * logf((float)(t + 1));  // lambda log c, c = t+1
    float m = -INFINITY, l = 0.f, o[VEC], q[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) o[k] = q[k] = 0.f;
    // One row (its P2 and I~ values kv, vv) into the group's running state.  Every
    // lane of the warp calls this together (the shuffles span the warp); lanes of a
    // group without a row this round pass valid = false and keep their state.
    auto take = [&](const float (&kv)[VEC], const float (&vv)[VEC], bool self, bool valid) {
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < VEC; ++k) dot = fmaf(q[k], kv[k], dot);
#pragma unroll
        for (int w = G / 2; w > 0; w >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, w);
        if (!valid) return;
        const float u = dot * kp.inv_sqrt_d;
        const float r = self ? sigmoid_f<kFast>(u / kp.tau_S) : u * sigmoid_f<kFast>(u) - corr;
        // The running maximum is raised only when a row exceeds it (then the state is
        // rescaled); otherwise the row adds exp(r - m).
        if (r > m) {
            const float s1 = (m == -INFINITY) ? 0.f : exp_f<kFast>(m - r);
            l = fmaf(l, s1, 1.f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) o[k] = fmaf(o[k], s1, vv[k]);
            m = r;
        } else {
            const float p = exp_f<kFast>(r - m);
            l += p;
#pragma unroll
            for (int k = 0; k < VEC; ++k) o[k] = fmaf(p, vv[k], o[k]);
        }
    };
    // Two Exchange rows into the group's running state at once (independent dot
    // products, split accumulators, one rescale at most); as take() otherwise.
    auto take2 = [&](const float (&k1)[VEC], const float (&v1)[VEC], bool ok1, const float (&k2)[VEC],
                     const float (&v2)[VEC], bool ok2) {
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int k = 0; k < VEC; k += 2) {
            a0 = fmaf(q[k], k1[k], a0);
            a1 = fmaf(q[k + 1], k1[k + 1], a1);
            b0 = fmaf(q[k], k2[k], b0);
            b1 = fmaf(q[k + 1], k2[k + 1], b1);
        }
        float d1 = a0 + a1, d2 = b0 + b1;
#pragma unroll
        for (int w = G / 2; w > 0; w >>= 1) {
            d1 += __shfl_xor_sync(0xffffffffu, d1, w);
            d2 += __shfl_xor_sync(0xffffffffu, d2, w);
        }
        const float u1 = d1 * kp.inv_sqrt_d, u2 = d2 * kp.inv_sqrt_d;
        const float r1 = ok1 ? u1 * sigmoid_f<kFast>(u1) - corr : -INFINITY;
        const float r2 = ok2 ? u2 * sigmoid_f<kFast>(u2) - corr : -INFINITY;
        const float mx = fmaxf(r1, r2);
        if (mx > m) {  // raise the running maximum (rescale the state)
            const float s1 = (m == -INFINITY) ? 0.f : exp_f<kFast>(m - mx);
            l *= s1;
#pragma unroll
            for (int k = 0; k < VEC; ++k) o[k] *= s1;
            m = mx;
        }
        const float p1 = ok1 ? exp_f<kFast>(r1 - m) : 0.f, p2 = ok2 ? exp_f<kFast>(r2 - m) : 0.f;
        l += p1 + p2;
#pragma unroll
        for (int k = 0; k < VEC; ++k) o[k] = fmaf(p1, v1[k], fmaf(p2, v2[k], o[k]));
    };
    // The new token's rows: q for every lane; the Self entry (group 0 of warp 0,
    // the warp shuffling together) and the append in CTA 0.
    bool ok = ptx::mbar_wait(&new_full, 0, &abort_flag, status, kDevTimeoutFull);
    if (ok) {
        if (active) load_vec16<Tin, VEC, true>(new_rows + col, q);
        if (append && sidx == 0)
            for (int c = threadIdx.x; c < d; c += kThreads) {
                P2c[row_offset(kp, bh, t) + c] = new_rows[kStreamMaxD + c];
                Vc[row_offset(kp, bh, t) + c] = new_rows[2 * kStreamMaxD + c];
            }
    }
    if (sidx == 0 && threadIdx.x < 32) {
        float kv[VEC], vv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) kv[e] = vv[e] = 0.f;
        const bool mine = ok && active && grp == 0;
        if (mine) {
            load_vec16<Tin, VEC, true>(new_rows + kStreamMaxD + col, kv);
            load_vec16<Tin, VEC, true>(new_rows + 2 * kStreamMaxD + col, vv);
        }
        take(kv, vv, true, grp == 0);
    }
    for (int k = 0;; ++k) {
        const int st = k % kStreamStages;
        if (!ptx::mbar_wait(&full[st], (k / kStreamStages) & 1, &abort_flag, status, kDevTimeoutFull)) ok = false;
        if (!__syncthreads_and(ok)) {  // every thread leaves together
            ok = false;
            break;
        }
        const int c = stage_chunk[st];
        if (c == kEmptyStage) {  // a wrong guess: nothing to score, refill the stage
            __syncthreads();
            if (threadIdx.x == 0) {
                fill(fills, chunk_of_fill(fills));
                ++fills;
            }
            continue;
        }
        if (c < 0) break;  // the same in every thread
        const Tin* sK = reinterpret_cast<const Tin*>(smb + (size_t)st * stage_bytes);
        const Tin* sV = sK + (size_t)ch * d;
        const int rc = min(t, c * ch + ch) - c * ch;
        for (int base = 0; base < rc; base += 2 * kGroups) {  // same trip count in every lane
            const int r1 = base + grp, r2 = r1 + kGroups;
            float kv1[VEC], vv1[VEC], kv2[VEC], vv2[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) kv1[e] = vv1[e] = kv2[e] = vv2[e] = 0.f;
            if (active && r1 < rc) {
                load_vec16<Tin, VEC, true>(sK + (size_t)r1 * d + col, kv1);
                load_vec16<Tin, VEC, true>(sV + (size_t)r1 * d + col, vv1);
            }
            if (active && r2 < rc) {
                load_vec16<Tin, VEC, true>(sK + (size_t)r2 * d + col, kv2);
                load_vec16<Tin, VEC, true>(sV + (size_t)r2 * d + col, vv2);
            }
            take2(kv1, vv1, r1 < rc, kv2, vv2, r2 < rc);
        }
        __syncthreads();  // the stage is consumed: refill it
        if (threadIdx.x == 0) {
            fill(fills, chunk_of_fill(fills));
            ++fills;
        }
    }
    if (!ok && threadIdx.x == 0)
        // Give the copies in flight (the last fill of each stage) a second bounded
        // wait before the stage area is reused.
        for (int f = max(0, fills - kStreamStages); f < fills; ++f)
            ptx::mbar_drain(&full[f % kStreamStages], (f / kStreamStages) & 1, status);
    if (!ok) m = -INFINITY;  // a share whose rows did not arrive is left out (the timeout is reported)
    // Merge of the groups into this CTA's (m, l, o): first the warp's groups by
    // shuffles (lanes li of the groups pair up), then the warps through shared
    // memory (the stages are no longer read).
#pragma unroll
    for (int w = G; w < 32; w <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, w), l2 = __shfl_xor_sync(0xffffffffu, l, w);
        const float M = fmaxf(m, m2);
        const float s1 = (m == -INFINITY) ? 0.f : exp_f<kFast>(m - M);
        const float s2 = (m2 == -INFINITY) ? 0.f : exp_f<kFast>(m2 - M);
        l = l * s1 + l2 * s2;
#pragma unroll
        for (int k = 0; k < VEC; ++k) o[k] = o[k] * s1 + __shfl_xor_sync(0xffffffffu, o[k], w) * s2;
        m = M;
    }
    __syncthreads();  // the stage area is free (copies in flight drained above)
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) < G) {  // the first group of each warp now holds the warp's state
        if (active) {
#pragma unroll
            for (int k = 0; k < VEC; ++k) og[(size_t)wid * d + col + k] = o[k];
        }
        if (li == 0) {
            gm[wid] = m;
            gl[wid] = l;
        }
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started: CTA 0's shared memory may be written
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < kWarps; ++g) M = fmaxf(M, gm[g]);
    for (int c = threadIdx.x; c < d; c += kThreads) {
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < kWarps; ++g)
            if (gm[g] != -INFINITY) acc = fmaf(exp_f<kFast>(gm[g] - M), og[(size_t)g * d + c], acc);
        st_cluster_f32(cl_o + (size_t)sidx * kStreamMaxD + c, 0, acc);
    }
    if (threadIdx.x == 0) {
        float Lc = 0.f;
#pragma unroll
        for (int g = 0; g < kWarps; ++g)
            if (gm[g] != -INFINITY) Lc = fmaf(exp_f<kFast>(gm[g] - M), gl[g], Lc);
        st_cluster_f32(cl_m + sidx, 0, M);
        st_cluster_f32(cl_l + sidx, 0, Lc);
    }
    // After the barrier CTA 0 holds the S results in its own shared memory and
    // merges them (Y = sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s, L = M + log
    // of the denominator, the paper's convention with the correction included);
    // no CTA's shared memory is accessed by another after it.
    cluster_sync();
    if (sidx == 0) {
        float Mc = -INFINITY;
        for (int r = 0; r < S; ++r) Mc = fmaxf(Mc, cl_m[r]);
        float den = 0.f;
        for (int r = 0; r < S; ++r)
            if (cl_m[r] != -INFINITY) den = fmaf(exp_f<kFast>(cl_m[r] - Mc), cl_l[r], den);
        for (int c = threadIdx.x; c < d; c += kThreads) {
            float num = 0.f;
            for (int r = 0; r < S; ++r)
                if (cl_m[r] != -INFINITY)
                    num = fmaf(exp_f<kFast>(cl_m[r] - Mc), cl_o[(size_t)r * kStreamMaxD + c], num);
            store_from_float(Y + new_off + c, num / den);
        }
        if (L != nullptr && threadIdx.x == 0) L[bh] = Mc + logf(den);
    }
}

// Merge of the chunks of one head: Y = sum_c e^{m_c - M} o_c / sum_c e^{m_c - M} l_c,
// L = M + log(sum_c e^{m_c - M} l_c) (the paper's convention, correction included).
template <typename Tin>
__global__ void __launch_bounds__(128) decode_combine_kernel(KernelProblem kp, const float* __restrict__ part,
                                                              int n_chunks, Tin* __restrict__ Y,
                                                              float* __restrict__ L) {
    extern __shared__ float w[];  // per chunk: its maximum m_c, then its weight e^{m_c - M}
    __shared__ float red[4];
    // Launched as a programmatic dependent of the partial pass: wait until that
    // grid has completed and its writes are visible (a no-op for a plain launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t bh = blockIdx.x;
    const int d = kp.d;
    const float* ph = part + (size_t)bh * n_chunks * (d + 2);
    float mloc = -INFINITY;
    for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) {
        const float mc = ph[(size_t)c * (d + 2)];
        w[c] = mc;
        mloc = fmaxf(mloc, mc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mloc;
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    if (M == -INFINITY) return;  // a position outside the cache (reported by the partial pass)
    float dloc = 0.f;
    for (int c = threadIdx.x; c < n_chunks; c += blockDim.x) {
        const float e = (w[c] == -INFINITY) ? 0.f : expf(w[c] - M);
        w[c] = e;
        dloc = fmaf(e, ph[(size_t)c * (d + 2) + 1], dloc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dloc += __shfl_xor_sync(0xffffffffu, dloc, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dloc;
    __syncthreads();
    const float den = red[0] + red[1] + red[2] + red[3];
    for (int col = threadIdx.x; col < d; col += blockDim.x) {
        // Eight chunks' loads in flight at a time.  A chunk past the position wrote
        // only (m, l): its weight is 0 and its (allocated, unwritten) outputs are
        // loaded but not used.
        float num = 0.f;
        for (int c0 = 0; c0 < n_chunks; c0 += 8) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = (c0 + k < n_chunks) ? ph[(size_t)(c0 + k) * (d + 2) + 2 + col] : 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (c0 + k < n_chunks && w[c0 + k] != 0.f) num = fmaf(w[c0 + k], v[k], num);
        }
        store_from_float(Y + (size_t)bh * d + col, num / den);
    }
    if (L != nullptr && threadIdx.x == 0) L[bh] = M + logf(den);
}

// The bulk-copy pass serves contiguous [B, H, T, d] caches whose rows are a
// multiple of 16 bytes; its chunk keeps both tensors' rows within 64 KB.
bool decode_bulk(const KernelProblem& kp, bool bf16) {
    return kp.layout == 0 && ((int64_t)kp.d * (bf16 ? 2 : 4)) % 16 == 0;
}

int decode_chunk_rows(const KernelProblem& kp, bool bf16) {
    if (!decode_bulk(kp, bf16)) return 512;
    const int row_bytes = kp.d * (bf16 ? 2 : 4);
    return (2 * 256 * row_bytes <= 65536) ? 256 : (2 * 128 * row_bytes <= 65536) ? 128 : 64;
}

// Rows per chunk of the streaming pass: at most 16 KB of each tensor per stage.
int stream_chunk_rows(const KernelProblem& kp, bool bf16) {
    const int rows = 16384 / (kp.d * (bf16 ? 2 : 4));
    return rows < 128 ? rows : 128;
}
constexpr int kStreamSmemMax = 120 * 1024;

// The merge, launched as a programmatic dependent of the partial pass (it may be
// scheduled while that pass finishes and waits for its writes in-kernel).
template <typename Tin>
cudaError_t launch_combine(const KernelProblem& kp, const float* part, int n_chunks, Tin* Y, float* L,
                           cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)kp.BH);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = sizeof(float) * (size_t)n_chunks;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<Tin>, kp, part, n_chunks, Y, L);
}

// Streaming pass (bulk-copy caches): one cluster of S CTAs per head, S chosen so
// that the grid fills the GPU once at the occupancy the kernel's shared memory
// allows (at most the portable cluster size of 8).  One launch: the merge
// happens inside each cluster.
template <typename Tin, int VEC, int G>
cudaError_t launch_stream(const KernelProblem& kp, const void* P1n, const void* P2n, const void* Vn, void* P2c,
                          void* Vc, const int* pos, int append, void* Y, float* L, unsigned int* status,
                          int num_sms, cudaStream_t s) {
    auto kern = decode_cluster_kernel<Tin, VEC, G>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemMax);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int ch = stream_chunk_rows(kp, sizeof(Tin) == 2);
    const size_t stages = (size_t)kStreamStages * 2 * ch * kp.d * sizeof(Tin);
    const size_t merge = sizeof(float) * ((size_t)(kThreads / 32) * (kp.d + 2));
    const size_t smem = stages > merge ? stages : merge;
    if (smem > (size_t)kStreamSmemMax) return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int64_t chunks_max = ((int64_t)kp.T + ch - 1) / ch;
    int64_t S = ((int64_t)(per_sm > 0 ? per_sm : 1) * (num_sms > 0 ? num_sms : 148)) / kp.BH;
    S = S < 1 ? 1 : S;
    S = S > kMaxCluster ? kMaxCluster : S;
    S = S > chunks_max ? chunks_max : S;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)kp.BH, (unsigned)S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, kp, (const Tin*)P1n, (const Tin*)P2n, (const Tin*)Vn, (Tin*)P2c, (Tin*)Vc,
                              pos, append, ch, (Tin*)Y, L, status);
}

// Direct pass (other caches): CTA (bh, chunk) over `chunk` keys read from HBM,
// then the merge.
template <typename Tin, int VEC, int G>
cudaError_t launch_direct(const KernelProblem& kp, const void* P1n, const void* P2n, const void* Vn, void* P2c,
                          void* Vc, const int* pos, int append, void* Y, float* L, float* part, int chunk,
                          int n_chunks, unsigned int* status, cudaStream_t s) {
    constexpr int kGroups = kThreads / G;
    dim3 grid((unsigned)kp.BH, (unsigned)n_chunks);
    const size_t smem = sizeof(float) * ((size_t)chunk + 8 + (size_t)kGroups * kp.d);
    decode_partial_kernel<Tin, VEC, G><<<grid, kThreads, smem, s>>>(kp, (const Tin*)P1n, (const Tin*)P2n,
                                                                    (const Tin*)Vn, (Tin*)P2c, (Tin*)Vc, pos, append,
                                                                    chunk, part, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine<Tin>(kp, part, n_chunks, (Tin*)Y, L, s);
}

}  // namespace

int decode_chunks(const KernelProblem& kp, bool bf16) {
    const int c = decode_chunk_rows(kp, bf16);
    return (int)(((int64_t)kp.T + c - 1) / c);
}

int decode_launches(const KernelProblem& kp, bool bf16) { return decode_bulk(kp, bf16) ? 1 : 2; }

bool decode_grid_fits(const KernelProblem& kp, bool bf16) {
    return kp.BH >= 1 && kp.BH <= 2147483647LL && decode_chunks(kp, bf16) <= kDecodeMaxChunks;
}

cudaError_t launch_decode(const KernelProblem& kp, bool bf16, const void* P1n, const void* P2n, const void* Vn,
                          void* P2c, void* Vc, const int* pos, int append, void* Y, float* L, float* part,
                          unsigned int* status, int num_sms, cudaStream_t s) {
    const int n_chunks = decode_chunks(kp, bf16);
    if (!decode_grid_fits(kp, bf16)) return cudaErrorInvalidValue;
    const int chunk = decode_chunk_rows(kp, bf16);
    if (decode_bulk(kp, bf16)) {
        // Streaming pass: 16 bf16 or 8 fp32 elements per lane (two 16-byte pieces),
        // G lanes per key row (a power of two covering d; fp32 d = 60 in 4-element
        // pieces, its rows being 240 bytes).
#define RELATION_STREAM(T_, VEC, G)                                                                              \
    return launch_stream<T_, VEC, G>(kp, P1n, P2n, Vn, P2c, Vc, pos, append, Y, L, status, num_sms, s)
        if (bf16) {
            switch (kp.d) {
                case 48: RELATION_STREAM(__nv_bfloat16, 16, 4);
                case 64: RELATION_STREAM(__nv_bfloat16, 16, 4);
                case 80: RELATION_STREAM(__nv_bfloat16, 16, 8);
                case 128: RELATION_STREAM(__nv_bfloat16, 16, 8);
                default: return cudaErrorInvalidValue;
            }
        }
        switch (kp.d) {
            case 48: RELATION_STREAM(float, 8, 8);
            case 60: RELATION_STREAM(float, 4, 16);
            case 64: RELATION_STREAM(float, 8, 8);
            case 80: RELATION_STREAM(float, 8, 16);
            case 128: RELATION_STREAM(float, 8, 16);
            default: return cudaErrorInvalidValue;
        }
#undef RELATION_STREAM
    }
    // Direct pass: rows read 16 bytes per lane where the row pitch allows it (8
    // bytes for bf16 d = 60).
#define RELATION_DECODE(T_, VEC, G) \
    return launch_direct<T_, VEC, G>(kp, P1n, P2n, Vn, P2c, Vc, pos, append, Y, L, part, chunk, n_chunks, status, s)
    if (bf16) {
        switch (kp.d) {
            case 48: RELATION_DECODE(__nv_bfloat16, 8, 8);
            case 60: RELATION_DECODE(__nv_bfloat16, 4, 16);
            case 64: RELATION_DECODE(__nv_bfloat16, 8, 8);
            case 80: RELATION_DECODE(__nv_bfloat16, 8, 16);
            case 128: RELATION_DECODE(__nv_bfloat16, 8, 16);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (kp.d) {
        case 48: RELATION_DECODE(float, 4, 16);
        case 60: RELATION_DECODE(float, 4, 16);
        case 64: RELATION_DECODE(float, 4, 16);
        case 80: RELATION_DECODE(float, 4, 32);
        case 128: RELATION_DECODE(float, 4, 32);
        default: return cudaErrorInvalidValue;
    }
#undef RELATION_DECODE
}

}  // namespace relation

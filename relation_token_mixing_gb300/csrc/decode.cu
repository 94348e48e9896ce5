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
// cores in fp32, split over key chunks: each CTA reads its chunk's cached rows
// once (by two bulk copies into shared memory where the rows allow it, else by
// direct 16- or 8-byte loads), computes the chunk's scores, maximum, weights and
// weighted sum, and one CTA per head then merges the chunks.
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

// The same from shared memory (rows staged by the bulk-copy pass).
template <typename Tin, int VEC>
__device__ __forceinline__ void load_vec_shared(const Tin* p, float (&v)[VEC]) {
    if constexpr (sizeof(Tin) == 2 && VEC == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else {
        static_assert(sizeof(Tin) == 4 && VEC == 4, "the bulk-copy pass reads 16-byte vectors");
        const float4 u = *reinterpret_cast<const float4*>(p);
        v[0] = u.x;
        v[1] = u.y;
        v[2] = u.z;
        v[3] = u.w;
    }
}

// One bulk copy global -> shared, completion counted on `bar` in bytes (both
// addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     ptx::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(ptx::smem_u32(bar))
                 : "memory");
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

// Partial pass for contiguous [B, H, T, d] caches whose rows are a multiple of 16
// bytes: the chunk's cached P2 and I~ rows arrive in shared memory by two bulk
// copies (one instruction each, completion on one mbarrier); the new token's row
// is stored next to them; the scores and the weighted sum then read shared memory.
// Same outputs as decode_partial_kernel.
template <typename Tin, int VEC, int G>
__global__ void __launch_bounds__(kThreads) decode_partial_bulk_kernel(
    KernelProblem kp, const Tin* __restrict__ P1n, const Tin* __restrict__ P2n, const Tin* __restrict__ Vn,
    Tin* __restrict__ P2c, Tin* __restrict__ Vc, const int* __restrict__ pos, int append, int chunk,
    float* __restrict__ part, unsigned int* status) {
    constexpr int kGroups = kThreads / G;
    extern __shared__ __align__(128) uint8_t smb[];
    __shared__ int abort_flag;
    const int d = kp.d;
    const size_t row_bytes = (size_t)d * sizeof(Tin);
    Tin* sK = reinterpret_cast<Tin*>(smb);
    Tin* sV = reinterpret_cast<Tin*>(smb + (size_t)chunk * row_bytes);
    float* sr = reinterpret_cast<float*>(smb + 2 * (size_t)chunk * row_bytes);  // chunk scores
    float* red = sr + chunk;                                                     // per-warp reductions (8)
    float* oacc = red + 8;                                                       // kGroups x d partial outputs
    uint64_t* bar = reinterpret_cast<uint64_t*>(oacc + (size_t)kGroups * d);
    const int64_t bh = blockIdx.x;
    const int b = (int)(bh / kp.H);
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
    const int rc = max(0, min(j1, t) - j0);  // cached rows of this chunk (row t is the new token)
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (rc > 0) {
            const uint32_t bytes = (uint32_t)(rc * row_bytes);
            ptx::mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_copy_g2s(sK, P2c + row_offset(kp, bh, j0), bytes, bar);
            bulk_copy_g2s(sV, Vc + row_offset(kp, bh, j0), bytes, bar);
        } else {
            ptx::mbar_arrive(bar);
        }
    }
    if (t >= j0 && t < j1)  // the new token's row, next to the copied rows (disjoint from them)
        for (int c = threadIdx.x; c < d; c += kThreads) {
            sK[(size_t)(t - j0) * d + c] = P2n[new_off + c];
            sV[(size_t)(t - j0) * d + c] = Vn[new_off + c];
        }
    (void)ptx::mbar_wait(bar, 0, &abort_flag, status, kDevTimeoutFull);
    __syncthreads();
    if (abort_flag) {  // the copies did not land within the limit (recorded in the status word)
        if (threadIdx.x == 0) {
            ptx::mbar_drain(bar, 0, status);  // give the copies in flight a second bounded wait before leaving
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
    float mloc = -INFINITY;
    for (int base = j0; base < j1; base += kGroups) {
        const int j = base + grp;
        float dot = 0.f;
        if (j < j1 && active) {
            float kv[VEC];
            load_vec_shared<Tin, VEC>(sK + (size_t)(j - j0) * d + col, kv);
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
    float o[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) o[k] = 0.f;
    float lloc = 0.f;
    for (int j = j0 + grp; j < j1; j += kGroups) {
        const float p = expf(sr[j - j0] - m);
        if (li == 0) lloc += p;
        if (active) {
            float vv[VEC];
            load_vec_shared<Tin, VEC>(sV + (size_t)(j - j0) * d + col, vv);
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

// Merge of the chunks of one head: Y = sum_c e^{m_c - M} o_c / sum_c e^{m_c - M} l_c,
// L = M + log(sum_c e^{m_c - M} l_c) (the paper's convention, correction included).
template <typename Tin>
__global__ void __launch_bounds__(128) decode_combine_kernel(KernelProblem kp, const float* __restrict__ part,
                                                              int n_chunks, Tin* __restrict__ Y,
                                                              float* __restrict__ L) {
    extern __shared__ float w[];  // per chunk: its maximum m_c, then its weight e^{m_c - M}
    __shared__ float red[4];
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

// Shared memory the bulk-copy pass may ask for (two tensors' rows, at most 64 KB,
// plus scores, reductions, partial outputs and the barrier).
constexpr int kBulkSmemMax = 96 * 1024;

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

template <typename Tin, int VEC, int G>
cudaError_t launch_decode_t(const KernelProblem& kp, const void* P1n, const void* P2n, const void* Vn, void* P2c,
                            void* Vc, const int* pos, int append, void* Y, float* L, float* part, bool bulk,
                            int chunk, int n_chunks, unsigned int* status, cudaStream_t s) {
    constexpr int kGroups = kThreads / G;
    dim3 grid((unsigned)kp.BH, (unsigned)n_chunks);
    bool launched = false;
    if constexpr (!(sizeof(Tin) == 2 && VEC == 4)) {  // 16-byte rows vectors only
        if (bulk) {
            static std::once_flag attr_once;
            static cudaError_t attr_err = cudaSuccess;
            std::call_once(attr_once, [] {
                attr_err = cudaFuncSetAttribute(decode_partial_bulk_kernel<Tin, VEC, G>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmemMax);
            });
            if (attr_err != cudaSuccess) return attr_err;
            const size_t smem = 2 * (size_t)chunk * kp.d * sizeof(Tin) +
                                sizeof(float) * ((size_t)chunk + 8 + (size_t)kGroups * kp.d) + 16;
            if (smem > (size_t)kBulkSmemMax) return cudaErrorInvalidValue;
            decode_partial_bulk_kernel<Tin, VEC, G><<<grid, kThreads, smem, s>>>(
                kp, (const Tin*)P1n, (const Tin*)P2n, (const Tin*)Vn, (Tin*)P2c, (Tin*)Vc, pos, append, chunk, part,
                status);
            launched = true;
        }
    }
    if (!launched) {
        const size_t smem = sizeof(float) * ((size_t)chunk + 8 + (size_t)kGroups * kp.d);
        decode_partial_kernel<Tin, VEC, G><<<grid, kThreads, smem, s>>>(kp, (const Tin*)P1n, (const Tin*)P2n,
                                                                        (const Tin*)Vn, (Tin*)P2c, (Tin*)Vc, pos,
                                                                        append, chunk, part, status);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<Tin><<<(unsigned)kp.BH, 128, sizeof(float) * n_chunks, s>>>(kp, part, n_chunks, (Tin*)Y, L);
    return cudaGetLastError();
}

}  // namespace

int decode_chunks(const KernelProblem& kp, bool bf16) {
    const int c = decode_chunk_rows(kp, bf16);
    return (int)(((int64_t)kp.T + c - 1) / c);
}

bool decode_grid_fits(const KernelProblem& kp, bool bf16) {
    return kp.BH >= 1 && kp.BH <= 2147483647LL && decode_chunks(kp, bf16) <= kDecodeMaxChunks;
}

cudaError_t launch_decode(const KernelProblem& kp, bool bf16, const void* P1n, const void* P2n, const void* Vn,
                          void* P2c, void* Vc, const int* pos, int append, void* Y, float* L, float* part,
                          unsigned int* status, cudaStream_t s) {
    const int n_chunks = decode_chunks(kp, bf16);
    if (!decode_grid_fits(kp, bf16)) return cudaErrorInvalidValue;
    const bool bulk = decode_bulk(kp, bf16);
    const int chunk = decode_chunk_rows(kp, bf16);
    // Vector width and lanes per key row by (dtype, d): rows are read 16 bytes per
    // lane where the row pitch allows it (8 bytes for bf16 d = 60).
#define RELATION_DECODE(T_, VEC, G)                                                                           \
    return launch_decode_t<T_, VEC, G>(kp, P1n, P2n, Vn, P2c, Vc, pos, append, Y, L, part, bulk, chunk, n_chunks, \
                                       status, s)
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

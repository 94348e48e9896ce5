// Host side of the Relation C ABI (include/relation.h): argument checks,
// kernel selection by dtype, launch bookkeeping and the device status word.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/relation.h"
#include "common.cuh"
#include "kernels.h"

namespace relation {

// One status word per device; kernels write it through a pointer obtained by
// cudaGetSymbolAddress (the host-side symbol is not a device address).
__device__ unsigned int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
thread_local int t_last_launches = 0;

struct DeviceInfo {
    unsigned int* status;
    int num_sms;
};

relation_status_t device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RELATION_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_status_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return RELATION_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return RELATION_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned int*>(ptr);
        g_num_sms[dev] = sms;
    }
    out->status = g_status_ptr[dev];
    out->num_sms = g_num_sms[dev];
    return RELATION_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_bytes(const relation_problem_t* p) { return p->dtype == RELATION_BF16 ? 2 : 4; }

size_t tensor_bytes(const relation_problem_t* p) {
    return (size_t)p->B * (size_t)p->H * (size_t)p->T * (size_t)p->d_h * elem_bytes(p);
}

size_t rows_of(const relation_problem_t* p) { return (size_t)p->B * (size_t)p->H * (size_t)p->T; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Problem checks shared by every entry point.
relation_status_t check_problem(const relation_problem_t* p) {
    if (p == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (p->B < 1 || p->H < 1 || p->T < 1 || p->d_h < 1) return RELATION_ERR_INVALID_ARGUMENT;
    if (p->T > (int64_t)INT32_MAX || p->B > (int64_t)INT32_MAX || p->H > (int64_t)INT32_MAX)
        return RELATION_ERR_INVALID_ARGUMENT;
    // Heads index gridDim.x (at most 2^31 - 1); 2^33 rows keep every one-dimensional
    // grid over rows or row tiles in range.  Both allow tensors far beyond one GPU.
    if (p->B * p->H > (int64_t)INT32_MAX || p->B * p->H * p->T > ((int64_t)1 << 33))
        return RELATION_ERR_INVALID_ARGUMENT;
    const double elems = (double)p->B * (double)p->H * (double)p->T * (double)p->d_h;
    if (elems > 1.0e12) return RELATION_ERR_INVALID_ARGUMENT;
    if (p->dtype != RELATION_F32 && p->dtype != RELATION_BF16) return RELATION_ERR_INVALID_ARGUMENT;
    if (!(p->tau_S > 0.f) || !isfinite(p->tau_S) || !isfinite(p->lambda)) return RELATION_ERR_INVALID_ARGUMENT;
    if (p->layout != RELATION_LAYOUT_BHTD && p->layout != RELATION_LAYOUT_BTHD) return RELATION_ERR_INVALID_ARGUMENT;
    if (p->d_h != 48 && p->d_h != 60 && p->d_h != 64 && p->d_h != 80 && p->d_h != 128) return RELATION_ERR_UNSUPPORTED;
    return RELATION_OK;
}

KernelProblem kernel_problem(const relation_problem_t* p) {
    KernelProblem kp;
    kp.BH = p->B * p->H;
    kp.T = (int)p->T;
    kp.d = (int)p->d_h;
    kp.tau_S = p->tau_S;
    kp.lambda = p->lambda;
    kp.causal = p->causal ? 1 : 0;
    kp.inv_sqrt_d = (float)(1.0 / sqrt((double)p->d_h));
    kp.H = (int)p->H;
    kp.layout = (int)p->layout;
    return kp;
}

// Every bf16 problem runs on the tensor cores.  d_h = 60, whose 120-byte rows TMA
// cannot step through, reads zero-padded copies of its operands (relation_fwd_ws
// and the backward), or copies its tiles with cp.async (relation_fwd without a
// workspace).
bool use_tensor_cores(const relation_problem_t* p) { return p->dtype == RELATION_BF16; }

// Launch-grid limits tighter than the generic ones, per path, checked before any
// work is enqueued: the tensor-core forward holds query-tile pairs in gridDim.y,
// the CUDA-core path the heads, and decoding keeps its chunk count bounded.
// (The backward's tensor-core grid is one-dimensional and within the generic limits.)
bool fwd_fits(const relation_problem_t* p) {
    return use_tensor_cores(p) ? fwd_tc_grid_fits(kernel_problem(p)) : simt_grid_fits(kernel_problem(p));
}
bool bwd_fits(const relation_problem_t* p) { return use_tensor_cores(p) || simt_grid_fits(kernel_problem(p)); }
bool decode_fits(const relation_problem_t* p) {
    return decode_grid_fits(kernel_problem(p), p->dtype == RELATION_BF16);
}

// Width of the fp32 dP1 accumulator rows: the tensor-core tile width that the
// head width is padded to.
int dq_width(const relation_problem_t* p) { return p->d_h <= 64 ? 64 : 128; }

// bf16 operands whose rows TMA cannot step through (d_h = 60) are copied once,
// zero-padded to 64 columns, into the workspace by the preparation stage.
bool pads_operands(const relation_problem_t* p) { return use_tensor_cores(p) && (p->d_h * 2) % 16 != 0; }

// Workspace: D [rows] fp32 (CUDA-core path) or the tensor-core kernels' per-query
// constants [B*H, T rounded up to 128, 2] fp32 | dP1 accumulator [rows, dq_width]
// fp32 | (d_h = 60) padded copies of P1, P2, V, dY [rows, 64] bf16; each part
// 256-byte aligned.
size_t workspace_layout(const relation_problem_t* p, size_t* dq_offset, size_t* pad_offset = nullptr) {
    const size_t d_bytes =
        use_tensor_cores(p)
            ? round_up((size_t)p->B * (size_t)p->H * (size_t)qconst_rows(p->T) * 2 * sizeof(float), 256)
            : round_up(rows_of(p) * sizeof(float), 256);
    const size_t dq_bytes = use_tensor_cores(p) ? round_up(rows_of(p) * (size_t)dq_width(p) * sizeof(float), 256) : 0;
    const size_t pad_bytes = pads_operands(p) ? 4 * round_up(rows_of(p) * 64 * 2, 256) : 0;
    if (dq_offset) *dq_offset = d_bytes;
    if (pad_offset) *pad_offset = d_bytes + dq_bytes;
    return d_bytes + dq_bytes + pad_bytes;
}

// The four padded operand copies inside the workspace (P1, P2, V, dY).
void padded_operands(const relation_problem_t* p, void* workspace, void* out[4]) {
    size_t pad_off = 0;
    workspace_layout(p, nullptr, &pad_off);
    const size_t each = round_up(rows_of(p) * 64 * 2, 256);
    for (int k = 0; k < 4; ++k) out[k] = static_cast<char*>(workspace) + pad_off + k * each;
}


struct BwdArgs {
    const relation_problem_t* p;
    const void *P1, *P2, *V, *Y;
    const float* L;
    const void* dY;
    void *dP1, *dP2, *dV;
    float* dlambda;
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
};

relation_status_t check_bwd(const BwdArgs& a) {
    relation_status_t st = check_problem(a.p);
    if (st != RELATION_OK) return st;
    if (!bwd_fits(a.p)) return RELATION_ERR_UNSUPPORTED;
    const void* ins[] = {a.P1, a.P2, a.V, a.Y, a.L, a.dY};
    void* outs[] = {a.dP1, a.dP2, a.dV};
    for (const void* x : ins)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (void* x : outs)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (a.workspace == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (const void* x : ins)
        if (!aligned16(x)) return RELATION_ERR_MISALIGNED;
    for (void* x : outs)
        if (!aligned16(x)) return RELATION_ERR_MISALIGNED;
    if (!aligned16(a.workspace)) return RELATION_ERR_MISALIGNED;
    if (a.dlambda != nullptr && (reinterpret_cast<uintptr_t>(a.dlambda) & 3u)) return RELATION_ERR_MISALIGNED;
    const size_t need = workspace_layout(a.p, nullptr);
    if (a.workspace_bytes < need) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const size_t tb = tensor_bytes(a.p), lb = rows_of(a.p) * sizeof(float);
    const void* in_ptr[] = {a.P1, a.P2, a.V, a.Y, a.L, a.dY};
    const size_t in_len[] = {tb, tb, tb, tb, lb, tb};
    const void* out_ptr[] = {a.dP1, a.dP2, a.dV, a.workspace, a.dlambda};
    const size_t out_len[] = {tb, tb, tb, need, a.dlambda ? sizeof(float) : 0};
    for (int o = 0; o < 5; ++o) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(out_ptr[o], out_len[o], in_ptr[i], in_len[i])) return RELATION_ERR_INVALID_ARGUMENT;
        for (int o2 = o + 1; o2 < 5; ++o2)
            if (overlaps(out_ptr[o], out_len[o], out_ptr[o2], out_len[o2])) return RELATION_ERR_INVALID_ARGUMENT;
    }
    return RELATION_OK;
}

relation_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? RELATION_OK : RELATION_ERR_CUDA; }

relation_status_t run_prepare(const BwdArgs& a, int* launches) {
    size_t dq_off = 0;
    workspace_layout(a.p, &dq_off);
    float* Dw = static_cast<float*>(a.workspace);
    float* dq = use_tensor_cores(a.p) ? reinterpret_cast<float*>(static_cast<char*>(a.workspace) + dq_off) : nullptr;
    if (a.dlambda != nullptr) {
        if (cudaMemsetAsync(a.dlambda, 0, sizeof(float), a.stream) != cudaSuccess) return RELATION_ERR_CUDA;
    }
    const KernelProblem kp = kernel_problem(a.p);
    // dlambda is summed by the main pass where that kernel does it, else here.
    float* dlam_here = (use_tensor_cores(a.p) && bwd_tc_sums_dlambda(kp.d)) ? nullptr : a.dlambda;
    DeviceInfo di;
    relation_status_t st = device_info(&di);
    if (st != RELATION_OK) return st;
    // Widths whose rows TMA cannot step through also get their padded operand
    // copies here, in the same pass.
    void* pad[4];
    if (pads_operands(a.p)) padded_operands(a.p, a.workspace, pad);
    st = from_cuda(launch_bwd_prepare(kp, a.p->dtype == RELATION_BF16, a.P1, a.P2, a.V, a.Y, a.L, a.dY, Dw, dq,
                                      dq_width(a.p), dlam_here, a.stream, pads_operands(a.p) ? pad : nullptr,
                                      di.num_sms, use_tensor_cores(a.p) ? Dw : nullptr));
    if (st == RELATION_OK) *launches += 1;
    return st;
}

relation_status_t run_main(const BwdArgs& a, int* launches) {
    size_t dq_off = 0;
    workspace_layout(a.p, &dq_off);
    const float* Dw = static_cast<const float*>(a.workspace);
    const float4* qconst = static_cast<const float4*>(a.workspace);  // tensor-core layout of the same region
    const KernelProblem kp = kernel_problem(a.p);
    if (use_tensor_cores(a.p)) {
        DeviceInfo di;
        relation_status_t st = device_info(&di);
        if (st != RELATION_OK) return st;
        float* dq = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + dq_off);
        TcLaunch tl{di.num_sms, di.status};
        float* dlam_main = bwd_tc_sums_dlambda(kp.d) ? a.dlambda : nullptr;
        if (pads_operands(a.p)) {
            void* pad[4];
            padded_operands(a.p, a.workspace, pad);
            st = from_cuda(launch_bwd_tc(kp, pad[0], pad[1], pad[2], qconst, pad[3], dq, a.dP2, a.dV, dlam_main, tl,
                                         a.stream, true));
        } else {
            st = from_cuda(launch_bwd_tc(kp, a.P1, a.P2, a.V, qconst, a.dY, dq, a.dP2, a.dV, dlam_main, tl,
                                         a.stream));
        }
        if (st == RELATION_OK) *launches += 1;
        return st;
    }
    relation_status_t st = from_cuda(launch_bwd_simt(kp, a.p->dtype == RELATION_BF16, a.P1, a.P2, a.V, a.L, Dw,
                                                     a.dY, a.dP1, a.dP2, a.dV, a.stream));
    if (st == RELATION_OK) *launches += 2;
    return st;
}

// Forward workspace (relation_fwd_ws): the padded copies of P1, P2, V [rows, 64]
// bf16, each 256-byte aligned, for widths whose rows TMA cannot step through.
size_t fwd_workspace_bytes(const relation_problem_t* p) {
    return pads_operands(p) ? 3 * round_up(rows_of(p) * 64 * 2, 256) : 0;
}

relation_status_t run_fwd(const relation_problem_t* p, const void* P1, const void* P2, const void* V, void* Y,
                          float* L, void* workspace, size_t workspace_bytes, bool with_ws, cudaStream_t s) {
    relation_status_t st = check_problem(p);
    if (st != RELATION_OK) return st;
    if (!fwd_fits(p)) return RELATION_ERR_UNSUPPORTED;
    if (!P1 || !P2 || !V || !Y) return RELATION_ERR_INVALID_ARGUMENT;
    if (!aligned16(P1) || !aligned16(P2) || !aligned16(V) || !aligned16(Y) || (L && !aligned16(L)))
        return RELATION_ERR_MISALIGNED;
    const size_t need = with_ws ? fwd_workspace_bytes(p) : 0;
    if (need > 0) {
        if (workspace == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
        if (!aligned16(workspace)) return RELATION_ERR_MISALIGNED;
    }
    const size_t tb = tensor_bytes(p), lb = rows_of(p) * sizeof(float);
    const void* ins[] = {P1, P2, V};
    for (const void* x : ins) {
        if (overlaps(Y, tb, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
        if (L && overlaps(L, lb, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
        if (need > 0 && overlaps(workspace, need, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    if (L && overlaps(L, lb, Y, tb)) return RELATION_ERR_INVALID_ARGUMENT;
    if (need > 0 && (overlaps(workspace, need, Y, tb) || (L && overlaps(workspace, need, L, lb))))
        return RELATION_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < need) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const KernelProblem kp = kernel_problem(p);
    int launches = 0;
    if (use_tensor_cores(p)) {
        DeviceInfo di;
        st = device_info(&di);
        if (st != RELATION_OK) return st;
        TcLaunch tl{di.num_sms, di.status};
        if (need > 0) {
            const void* src[3] = {P1, P2, V};
            void* dst[3];
            const size_t each = round_up(rows_of(p) * 64 * 2, 256);
            for (int k = 0; k < 3; ++k) dst[k] = static_cast<char*>(workspace) + k * each;
            st = from_cuda(launch_pad_operands(kp, src, dst, 3, di.num_sms, s));
            if (st == RELATION_OK) {
                launches += 1;
                st = from_cuda(launch_fwd_tc(kp, dst[0], dst[1], dst[2], Y, L, tl, s, true));
            }
        } else {
            st = from_cuda(launch_fwd_tc(kp, P1, P2, V, Y, L, tl, s));
        }
    } else {
        st = from_cuda(launch_fwd_simt(kp, p->dtype == RELATION_BF16, P1, P2, V, Y, L, s));
    }
    if (st == RELATION_OK) t_last_launches = launches + 1;
    return st;
}

relation_status_t run_finish(const BwdArgs& a, int* launches) {
    if (!use_tensor_cores(a.p)) return RELATION_OK;  // the CUDA-core path writes dP1 directly
    size_t dq_off = 0;
    workspace_layout(a.p, &dq_off);
    DeviceInfo di;
    relation_status_t st = device_info(&di);
    if (st != RELATION_OK) return st;
    const float* dq = reinterpret_cast<const float*>(static_cast<const char*>(a.workspace) + dq_off);
    st = from_cuda(launch_convert(kernel_problem(a.p), dq, dq_width(a.p), a.dP1, true, di.num_sms, a.stream));
    if (st == RELATION_OK) *launches += 1;
    return st;
}

// ------------------------------------------------------------------ host step
// relation_step_host: one training step from and to host memory, in slices of
// whole sequences.  Per device it keeps two non-blocking streams (copies in,
// copies out) and the events that order them against the compute stream; the
// enqueueing of one call holds the device's lock.
struct HostStepRes {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev_in[2], ev_dy[2], ev_fwd[2], ev_comp[2], ev_out[2], ev_start, ev_sum, ev_done;
    bool ready = false;
};
constexpr int kHostStepDevices = 64;
HostStepRes g_host_step[kHostStepDevices];
std::mutex g_host_step_mu[kHostStepDevices];

relation_status_t host_step_resources(int dev, HostStepRes** out) {
    HostStepRes& h = g_host_step[dev];
    if (!h.ready) {
        if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess)
            return RELATION_ERR_CUDA;
        cudaEvent_t* evs[] = {&h.ev_in[0],  &h.ev_in[1],   &h.ev_dy[0],   &h.ev_dy[1], &h.ev_fwd[0],
                              &h.ev_fwd[1], &h.ev_comp[0], &h.ev_comp[1], &h.ev_out[0], &h.ev_out[1],
                              &h.ev_start,  &h.ev_sum,     &h.ev_done};
        for (cudaEvent_t* e : evs)
            if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return RELATION_ERR_CUDA;
        h.ready = true;
    }
    *out = &h;
    return RELATION_OK;
}

// Device buffer of relation_step_host: two slots, each [P1 P2 V dY Y dP1 dP2 dV | L | backward
// workspace | forward workspace] for one slice, then the slices' dlambda and their sum.
struct HostStepLayout {
    relation_problem_t ps;  // one slice: B / chunks sequences
    size_t tb, lb, bws, fws, slot, total;
};

bool host_step_layout(const relation_problem_t* p, int chunks, HostStepLayout* l) {
    if (check_problem(p) != RELATION_OK || chunks < 1 || p->B % chunks != 0) return false;
    l->ps = *p;
    l->ps.B = p->B / chunks;
    if (!fwd_fits(&l->ps) || !bwd_fits(&l->ps)) return false;
    l->tb = round_up(tensor_bytes(&l->ps), 256);
    l->lb = round_up(rows_of(&l->ps) * sizeof(float), 256);
    l->bws = round_up(workspace_layout(&l->ps, nullptr), 256);
    l->fws = round_up(fwd_workspace_bytes(&l->ps), 256);
    l->slot = 8 * l->tb + l->lb + l->bws + l->fws;
    l->total = 2 * l->slot + round_up((size_t)(chunks + 1) * sizeof(float), 256);
    return true;
}

}  // namespace
}  // namespace relation

using namespace relation;

extern "C" {

size_t relation_step_host_device_bytes(const relation_problem_t* p, int chunks) {
    HostStepLayout l;
    return host_step_layout(p, chunks, &l) ? l.total : 0;
}

relation_status_t relation_step_host(const relation_problem_t* p, const void* P1, const void* P2, const void* V,
                                     const void* dY, void* Y, float* L, void* dP1, void* dP2, void* dV,
                                     float* dlambda, int chunks, void* device_buffer, size_t device_bytes,
                                     void* stream) {
    relation_status_t st = check_problem(p);
    if (st != RELATION_OK) return st;
    if (chunks < 1 || p->B % chunks != 0) return RELATION_ERR_INVALID_ARGUMENT;
    HostStepLayout l;
    if (!host_step_layout(p, chunks, &l)) return RELATION_ERR_UNSUPPORTED;
    const void* h_in[4] = {P1, P2, V, dY};
    void* h_out[4] = {Y, dP1, dP2, dV};
    for (const void* x : h_in)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (void* x : h_out)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (device_buffer == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (!aligned16(device_buffer)) return RELATION_ERR_MISALIGNED;
    if (device_bytes < l.total) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostStepDevices) return RELATION_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_host_step_mu[dev]);
    HostStepRes* r = nullptr;
    if ((st = host_step_resources(dev, &r)) != RELATION_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t tbc = tensor_bytes(&l.ps), lbc = rows_of(&l.ps) * sizeof(float);  // one slice's bytes
    char* base = static_cast<char*>(device_buffer);
    // Slot k's tensors: 0 P1, 1 P2, 2 V, 3 dY, 4 Y, 5 dP1, 6 dP2, 7 dV; then L and the workspaces.
    auto dt = [&](int slot, int k) -> void* { return base + slot * l.slot + k * l.tb; };
    auto dl = [&](int slot) { return reinterpret_cast<float*>(base + slot * l.slot + 8 * l.tb); };
    auto dbw = [&](int slot) -> void* { return base + slot * l.slot + 8 * l.tb + l.lb; };
    auto dfw = [&](int slot) -> void* { return base + slot * l.slot + 8 * l.tb + l.lb + l.bws; };
    float* dlam = reinterpret_cast<float*>(base + 2 * l.slot);  // per slice, then their sum
#define RELATION_CK(x)                                      do {                                                        if ((x) != cudaSuccess) return RELATION_ERR_CUDA;     } while (0)
    // Nothing starts before the work already queued on the caller's stream.
    RELATION_CK(cudaEventRecord(r->ev_start, s));
    RELATION_CK(cudaStreamWaitEvent(r->in, r->ev_start, 0));
    RELATION_CK(cudaStreamWaitEvent(r->out, r->ev_start, 0));
    int launches = 0;
    for (int c = 0; c < chunks; ++c) {
        const int slot = c & 1;
        // In: slice c into its slot once slice c-2 has left it; the forward's operands
        // first, dY (needed by the backward only) after them.
        if (c >= 2) RELATION_CK(cudaStreamWaitEvent(r->in, r->ev_out[slot], 0));
        for (int k = 0; k < 4; ++k) {
            RELATION_CK(cudaMemcpyAsync(dt(slot, k), static_cast<const char*>(h_in[k]) + (size_t)c * tbc, tbc,
                                        cudaMemcpyHostToDevice, r->in));
            if (k == 2) RELATION_CK(cudaEventRecord(r->ev_in[slot], r->in));
        }
        RELATION_CK(cudaEventRecord(r->ev_dy[slot], r->in));
        // Compute on the caller's stream.
        RELATION_CK(cudaStreamWaitEvent(s, r->ev_in[slot], 0));
        if (c >= 2) RELATION_CK(cudaStreamWaitEvent(s, r->ev_out[slot], 0));
        st = run_fwd(&l.ps, dt(slot, 0), dt(slot, 1), dt(slot, 2), dt(slot, 4), dl(slot), dfw(slot), l.fws, true, s);
        if (st != RELATION_OK) return st;
        launches += t_last_launches;
        RELATION_CK(cudaEventRecord(r->ev_fwd[slot], s));
        RELATION_CK(cudaStreamWaitEvent(s, r->ev_dy[slot], 0));
        const BwdArgs a{&l.ps,       dt(slot, 0), dt(slot, 1), dt(slot, 2), dt(slot, 4), dl(slot),
                        dt(slot, 3), dt(slot, 5), dt(slot, 6), dt(slot, 7), dlambda ? dlam + c : nullptr,
                        dbw(slot),   l.bws,       s};
        if ((st = check_bwd(a)) != RELATION_OK) return st;
        if ((st = run_prepare(a, &launches)) != RELATION_OK) return st;
        if ((st = run_main(a, &launches)) != RELATION_OK) return st;
        if ((st = run_finish(a, &launches)) != RELATION_OK) return st;
        RELATION_CK(cudaEventRecord(r->ev_comp[slot], s));
        // Out: slice c's Y (and L) once its forward is done, its gradients once its
        // backward is, while the next slice is computed.
        RELATION_CK(cudaStreamWaitEvent(r->out, r->ev_fwd[slot], 0));
        RELATION_CK(cudaMemcpyAsync(static_cast<char*>(h_out[0]) + (size_t)c * tbc, dt(slot, 4), tbc,
                                    cudaMemcpyDeviceToHost, r->out));
        if (L != nullptr)
            RELATION_CK(cudaMemcpyAsync(reinterpret_cast<char*>(L) + (size_t)c * lbc, dl(slot), lbc,
                                        cudaMemcpyDeviceToHost, r->out));
        RELATION_CK(cudaStreamWaitEvent(r->out, r->ev_comp[slot], 0));
        for (int k = 1; k < 4; ++k)
            RELATION_CK(cudaMemcpyAsync(static_cast<char*>(h_out[k]) + (size_t)c * tbc, dt(slot, 4 + k), tbc,
                                        cudaMemcpyDeviceToHost, r->out));
        RELATION_CK(cudaEventRecord(r->ev_out[slot], r->out));
    }
    if (dlambda != nullptr) {
        RELATION_CK(launch_sum_in_order(dlam, chunks, dlam + chunks, s));
        ++launches;
        RELATION_CK(cudaEventRecord(r->ev_sum, s));
        RELATION_CK(cudaStreamWaitEvent(r->out, r->ev_sum, 0));
        RELATION_CK(cudaMemcpyAsync(dlambda, dlam + chunks, sizeof(float), cudaMemcpyDeviceToHost, r->out));
    }
    // The caller's stream completes after every copy out.
    RELATION_CK(cudaEventRecord(r->ev_done, r->out));
    RELATION_CK(cudaStreamWaitEvent(s, r->ev_done, 0));
#undef RELATION_CK
    t_last_launches = launches;
    return RELATION_OK;
}

relation_status_t relation_fwd(const relation_problem_t* p, const void* P1, const void* P2, const void* V, void* Y,
                               float* L, void* stream) {
    return run_fwd(p, P1, P2, V, Y, L, nullptr, 0, false, static_cast<cudaStream_t>(stream));
}

size_t relation_fwd_workspace_bytes(const relation_problem_t* p) {
    if (check_problem(p) != RELATION_OK || !fwd_fits(p)) return 0;
    return fwd_workspace_bytes(p);
}

relation_status_t relation_fwd_ws(const relation_problem_t* p, const void* P1, const void* P2, const void* V, void* Y,
                                  float* L, void* workspace, size_t workspace_bytes, void* stream) {
    return run_fwd(p, P1, P2, V, Y, L, workspace, workspace_bytes, true, static_cast<cudaStream_t>(stream));
}

size_t relation_bwd_workspace_bytes(const relation_problem_t* p) {
    if (check_problem(p) != RELATION_OK || !bwd_fits(p)) return 0;
    return workspace_layout(p, nullptr);
}

#define RELATION_BWD_ARGS                                                                                     \
    const relation_problem_t *p, const void *P1, const void *P2, const void *V, const void *Y, const float *L, \
        const void *dY, void *dP1, void *dP2, void *dV, float *dlambda, void *workspace, size_t workspace_bytes, \
        void *stream
#define RELATION_BWD_PACK \
    BwdArgs a{p, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)}

relation_status_t relation_bwd(RELATION_BWD_ARGS) {
    RELATION_BWD_PACK;
    relation_status_t st = check_bwd(a);
    if (st != RELATION_OK) return st;
    int launches = 0;
    if ((st = run_prepare(a, &launches)) != RELATION_OK) return st;
    if ((st = run_main(a, &launches)) != RELATION_OK) return st;
    if ((st = run_finish(a, &launches)) != RELATION_OK) return st;
    t_last_launches = launches;
    return RELATION_OK;
}

relation_status_t relation_bwd_prepare(RELATION_BWD_ARGS) {
    RELATION_BWD_PACK;
    relation_status_t st = check_bwd(a);
    if (st != RELATION_OK) return st;
    int launches = 0;
    st = run_prepare(a, &launches);
    if (st == RELATION_OK) t_last_launches = launches;
    return st;
}

relation_status_t relation_bwd_main(RELATION_BWD_ARGS) {
    RELATION_BWD_PACK;
    relation_status_t st = check_bwd(a);
    if (st != RELATION_OK) return st;
    int launches = 0;
    st = run_main(a, &launches);
    if (st == RELATION_OK) t_last_launches = launches;
    return st;
}

relation_status_t relation_bwd_finish(RELATION_BWD_ARGS) {
    RELATION_BWD_PACK;
    relation_status_t st = check_bwd(a);
    if (st != RELATION_OK) return st;
    int launches = 0;
    st = run_finish(a, &launches);
    if (st == RELATION_OK) t_last_launches = launches;
    return st;
}

relation_status_t relation_selftest_wait_timeout(uint32_t limit_ms, void* stream) {
    if (limit_ms < 1 || limit_ms > 10000) return RELATION_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    relation_status_t st = device_info(&di);
    if (st != RELATION_OK) return st;
    st = from_cuda(launch_wait_selftest((uint64_t)limit_ms * 1000000ull, di.status, static_cast<cudaStream_t>(stream)));
    if (st == RELATION_OK) t_last_launches = 1;
    return st;
}

relation_status_t relation_check_device_status(void) {
    DeviceInfo di;
    relation_status_t st = device_info(&di);
    if (st != RELATION_OK) return st;
    unsigned int word = 0;
    if (cudaMemcpy(&word, di.status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return RELATION_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(di.status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return RELATION_ERR_CUDA;
        if (word & kDevDrainIncomplete) return RELATION_ERR_DEVICE_UNSAFE;
        return word == kDevBadPosition ? RELATION_ERR_INVALID_ARGUMENT : RELATION_ERR_DEVICE_TIMEOUT;
    }
    return RELATION_OK;
}

namespace relation {
namespace {
// RoPE frequencies base^(-2c/d) / (2 pi) for c < d/2 as float pairs (computed in double).
RopeTable rope_table(int d, float base) {
    RopeTable tab{};
    tab.enabled = base > 0.f ? 1 : 0;
    for (int c = 0; c < d / 2 && tab.enabled; ++c) {
        const double f = pow((double)base, -2.0 * c / d) / (2.0 * 3.14159265358979323846);
        tab.hi[c] = (float)f;
        tab.lo[c] = (float)(f - (double)tab.hi[c]);
    }
    return tab;
}

relation_status_t check_prologue(const relation_problem_t* p, const void* const* in, int n_in, const void* const* out,
                                 int n_out, const float* theta, int pairing, float rope_base) {
    relation_status_t st = check_problem(p);
    if (st != RELATION_OK) return st;
    if (p->H % 2 != 0 || (pairing != 0 && pairing != 1) || !isfinite(rope_base) || theta == nullptr)
        return RELATION_ERR_INVALID_ARGUMENT;
    for (int k = 0; k < n_in; ++k)
        if (in[k] == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (int k = 0; k < n_out; ++k)
        if (out[k] == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (int k = 0; k < n_in; ++k)
        if (!aligned16(in[k])) return RELATION_ERR_MISALIGNED;
    for (int k = 0; k < n_out; ++k)
        if (!aligned16(out[k])) return RELATION_ERR_MISALIGNED;
    const size_t tb = tensor_bytes(p);
    for (int o = 0; o < n_out; ++o) {
        for (int i = 0; i < n_in; ++i)
            if (overlaps(out[o], tb, in[i], tb)) return RELATION_ERR_INVALID_ARGUMENT;
        for (int o2 = o + 1; o2 < n_out; ++o2)
            if (overlaps(out[o], tb, out[o2], tb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    return RELATION_OK;
}
}  // namespace
}  // namespace relation

relation_status_t relation_prologue_fwd(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        void* P1, void* P2, void* I_mixed, void* stream) {
    const void* in[] = {X1, X2, I};
    const void* out[] = {P1, P2, I_mixed};
    relation_status_t st = check_prologue(p, in, 3, out, 3, theta, pairing, rope_base);
    if (st != RELATION_OK) return st;
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    const KernelProblem kp = kernel_problem(p);
    const bool bf16 = p->dtype == RELATION_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = from_cuda(launch_rope(kp, bf16, X1, X2, P1, P2, pos0, rope_table((int)p->d_h, rope_base), false,
                               di.num_sms, s));
    if (st != RELATION_OK) return st;
    st = from_cuda(launch_givens(kp, bf16, I, nullptr, I_mixed, theta, pairing, false, nullptr, di.num_sms, s));
    if (st == RELATION_OK) t_last_launches = 2;
    return st;
}

relation_status_t relation_prologue_bwd(const relation_problem_t* p, const void* dP1, const void* dP2,
                                        const void* dI_mixed, const void* I_mixed, const float* theta, int pairing,
                                        float rope_base, const int32_t* pos0, void* dX1, void* dX2, void* dI,
                                        float* dtheta, void* stream) {
    const void* in[] = {dP1, dP2, dI_mixed, I_mixed};
    const void* out[] = {dX1, dX2, dI};
    relation_status_t st = check_prologue(p, in, 4, out, 3, theta, pairing, rope_base);
    if (st != RELATION_OK) return st;
    if (dtheta != nullptr && (reinterpret_cast<uintptr_t>(dtheta) & 3u)) return RELATION_ERR_MISALIGNED;
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    const KernelProblem kp = kernel_problem(p);
    const bool bf16 = p->dtype == RELATION_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtheta != nullptr && cudaMemsetAsync(dtheta, 0, sizeof(float) * (size_t)(p->H / 2), s) != cudaSuccess)
        return RELATION_ERR_CUDA;
    st = from_cuda(launch_rope(kp, bf16, dP1, dP2, dX1, dX2, pos0, rope_table((int)p->d_h, rope_base), true,
                               di.num_sms, s));
    if (st != RELATION_OK) return st;
    st = from_cuda(launch_givens(kp, bf16, dI_mixed, I_mixed, dI, theta, pairing, true, dtheta, di.num_sms, s));
    if (st == RELATION_OK) t_last_launches = 2;
    return st;
}

relation_status_t relation_fwd_prologue(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        void* Y, float* L, void* stream) {
    const void* in[] = {X1, X2, I};
    const void* out[] = {Y};
    relation_status_t st = check_prologue(p, in, 3, out, 1, theta, pairing, rope_base);
    if (st != RELATION_OK) return st;
    if (p->dtype != RELATION_BF16 || p->d_h != 64 || !fwd_fits(p)) return RELATION_ERR_UNSUPPORTED;
    if (L != nullptr) {
        if (!aligned16(L)) return RELATION_ERR_MISALIGNED;
        const size_t tb = tensor_bytes(p), lb = rows_of(p) * sizeof(float);
        for (const void* x : {X1, X2, I, (const void*)Y})
            if (overlaps(L, lb, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    TcLaunch tl{di.num_sms, di.status};
    st = from_cuda(launch_fwd_tc_prologue(kernel_problem(p), X1, X2, I, Y, L, tl, static_cast<cudaStream_t>(stream),
                                          rope_table((int)p->d_h, rope_base), theta, pos0, pairing));
    if (st == RELATION_OK) t_last_launches = 1;
    return st;
}

size_t relation_bwd_prologue_workspace_bytes(const relation_problem_t* p) {
    if (check_problem(p) != RELATION_OK || p->dtype != RELATION_BF16 || p->d_h != 64 || p->H % 2 != 0) return 0;
    // relation_bwd's workspace, then the gradient of the mixed states (bf16, the problem's layout).
    return round_up(workspace_layout(p, nullptr), 256) + round_up(tensor_bytes(p), 256);
}

relation_status_t relation_bwd_prologue(const relation_problem_t* p, const void* X1, const void* X2, const void* I,
                                        const float* theta, int pairing, float rope_base, const int32_t* pos0,
                                        const void* Y, const float* L, const void* dY, void* dX1, void* dX2, void* dI,
                                        float* dtheta, float* dlambda, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    const void* in[] = {X1, X2, I, Y, dY};
    const void* out[] = {dX1, dX2, dI};
    relation_status_t st = check_prologue(p, in, 5, out, 3, theta, pairing, rope_base);
    if (st != RELATION_OK) return st;
    if (p->dtype != RELATION_BF16 || p->d_h != 64) return RELATION_ERR_UNSUPPORTED;
    if (L == nullptr || workspace == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (!aligned16(L) || !aligned16(workspace) || (dtheta && (reinterpret_cast<uintptr_t>(dtheta) & 3u)) ||
        (dlambda && (reinterpret_cast<uintptr_t>(dlambda) & 3u)))
        return RELATION_ERR_MISALIGNED;
    const size_t need = relation_bwd_prologue_workspace_bytes(p);
    if (workspace_bytes < need) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const size_t tb = tensor_bytes(p), lb = rows_of(p) * sizeof(float);
    for (const void* x : {X1, X2, I, Y, dY, (const void*)L, (const void*)dX1, (const void*)dX2, (const void*)dI})
        if (overlaps(workspace, need, x, x == (const void*)L ? lb : tb)) return RELATION_ERR_INVALID_ARGUMENT;
    for (const void* o : {(const void*)dX1, (const void*)dX2, (const void*)dI})
        if (overlaps(L, lb, o, tb)) return RELATION_ERR_INVALID_ARGUMENT;
    const size_t small = sizeof(float) * (size_t)(p->H / 2);
    for (const void* o : {(const void*)dtheta, (const void*)dlambda}) {
        if (o == nullptr) continue;
        for (const void* x : {X1, X2, I, Y, dY, (const void*)dX1, (const void*)dX2, (const void*)dI})
            if (overlaps(o, small, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
        if (overlaps(o, small, workspace, need) || overlaps(o, small, L, lb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    if (dtheta != nullptr && dlambda != nullptr && overlaps(dtheta, small, dlambda, sizeof(float)))
        return RELATION_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const KernelProblem kp = kernel_problem(p);
    const RopeTable tab = rope_table((int)p->d_h, rope_base);
    void* dImix = static_cast<char*>(workspace) + round_up(workspace_layout(p, nullptr), 256);
    size_t dq_off = 0;
    workspace_layout(p, &dq_off);
    float* dq = reinterpret_cast<float*>(static_cast<char*>(workspace) + dq_off);
    // Preparation as in relation_bwd (per-query constants from Y, dY, L; the dP1
    // accumulator reset; dlambda zeroed): it reads none of X1, X2, I.
    BwdArgs a{p, X1, X2, I, Y, L, dY, dX1, dX2, dImix, dlambda, workspace, workspace_bytes, s};
    int launches = 0;
    if ((st = run_prepare(a, &launches)) != RELATION_OK) return st;
    TcLaunch tl{di.num_sms, di.status};
    st = from_cuda(launch_bwd_tc64_prologue(kp, X1, X2, I, static_cast<const float4*>(workspace), dY, dq, dX2, dImix,
                                            dlambda, tl, s, tab, theta, pos0, pairing));
    if (st != RELATION_OK) return st;
    st = from_cuda(launch_rope_convert(kp, dq, dX1, pos0, tab, di.num_sms, s));
    if (st != RELATION_OK) return st;
    if (dtheta != nullptr && cudaMemsetAsync(dtheta, 0, small, s) != cudaSuccess) return RELATION_ERR_CUDA;
    st = from_cuda(launch_givens(kp, true, dImix, I, dI, theta, pairing, true, dtheta, di.num_sms, s, true));
    if (st == RELATION_OK) t_last_launches = launches + 3;
    return st;
}

namespace relation {
namespace {
relation_status_t check_linear(const relation_problem_t* p) {
    relation_status_t st = check_problem(p);
    if (st != RELATION_OK) return st;
    if (p->dtype != RELATION_BF16) return RELATION_ERR_UNSUPPORTED;
    if (p->d_h != 48 && p->d_h != 60 && p->d_h != 64) return RELATION_ERR_UNSUPPORTED;
    return RELATION_OK;
}
// Floats of the workspace: segment states and retentions (forward), plus the
// reverse segment states and one float per token (backward).
size_t linear_ws_floats(const relation_problem_t* p, int num_sms, bool backward) {
    int len = 0;
    const int nseg = linear_segments(kernel_problem(p), num_sms, &len);
    const size_t bh = (size_t)p->B * (size_t)p->H;
    size_t n = bh * (size_t)nseg * (64 * 64 + 64);
    if (backward) n += bh * (size_t)nseg * 64 * 64 + bh * (size_t)p->T;
    return n;
}
}  // namespace
}  // namespace relation

size_t relation_linear_workspace_bytes(const relation_problem_t* p) {
    if (check_linear(p) != RELATION_OK) return 0;
    DeviceInfo di;
    if (device_info(&di) != RELATION_OK) return 0;
    return linear_ws_floats(p, di.num_sms, true) * sizeof(float);
}

namespace relation {
namespace {
// Gate parameters [H, d_h] float32: both given or both absent; 4-byte aligned.
// tensors[k] spans bytes[k] (bf16 operands, fp32 gate inputs / outputs).
relation_status_t check_gate(const relation_problem_t* p, const float* a, const float* b, const void* const* tensors,
                             const size_t* bytes, int n) {
    if (a == nullptr || b == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(a) & 3u) || (reinterpret_cast<uintptr_t>(b) & 3u)) return RELATION_ERR_MISALIGNED;
    const size_t pb = (size_t)p->H * (size_t)p->d_h * sizeof(float);
    for (int k = 0; k < n; ++k)
        if (overlaps(a, pb, tensors[k], bytes[k]) || overlaps(b, pb, tensors[k], bytes[k]))
            return RELATION_ERR_INVALID_ARGUMENT;
    return RELATION_OK;
}

relation_status_t run_linear_fwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                 const float* G, const float* gate_alog, const float* gate_dtb, void* Y, float* state,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    relation_status_t st = check_linear(p);
    if (st != RELATION_OK) return st;
    if (!P1 || !P2 || !I || !G || !Y || !workspace) return RELATION_ERR_INVALID_ARGUMENT;
    if (!aligned16(P1) || !aligned16(P2) || !aligned16(I) || !aligned16(G) || !aligned16(Y) ||
        !aligned16(workspace) || (state && !aligned16(state)))
        return RELATION_ERR_MISALIGNED;
    const size_t tb = tensor_bytes(p), gb = rows_of(p) * (size_t)p->d_h * sizeof(float);
    const size_t sb = (size_t)p->B * p->H * p->d_h * p->d_h * sizeof(float);
    const void* ins[] = {P1, P2, I};
    for (const void* x : ins) {
        if (overlaps(Y, tb, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
        if (state && overlaps(state, sb, x, tb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    if (overlaps(Y, tb, G, gb) || (state && (overlaps(state, sb, G, gb) || overlaps(state, sb, Y, tb))))
        return RELATION_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    if (workspace_bytes < linear_ws_floats(p, di.num_sms, false) * sizeof(float))
        return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const KernelProblem kp = kernel_problem(p);
    int len = 0;
    const int nseg = linear_segments(kp, di.num_sms, &len);
    st = from_cuda(launch_linear_fwd(kp, P1, P2, I, G, Y, state, static_cast<float*>(workspace), di.num_sms,
                                     static_cast<cudaStream_t>(stream), gate_alog, gate_dtb));
    if (st == RELATION_OK) t_last_launches = nseg > 1 ? 3 : 1;
    return st;
}

relation_status_t run_linear_bwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                 const float* G, const float* gate_alog, const float* gate_dtb, const void* dY,
                                 void* dP1, void* dP2, void* dI, float* dG, float* gate_dalog, float* gate_ddtb,
                                 int states_from_forward, void* workspace, size_t workspace_bytes, void* stream) {
    relation_status_t st = check_linear(p);
    if (st != RELATION_OK) return st;
    const void* ins[] = {P1, P2, I, G, dY};
    void* outs[] = {dP1, dP2, dI, dG};
    for (const void* x : ins)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (const void* x : outs)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (const void* x : ins)
        if (!aligned16(x)) return RELATION_ERR_MISALIGNED;
    for (const void* x : outs)
        if (!aligned16(x)) return RELATION_ERR_MISALIGNED;
    if (!aligned16(workspace)) return RELATION_ERR_MISALIGNED;
    const size_t tb = tensor_bytes(p), gb = rows_of(p) * (size_t)p->d_h * sizeof(float);
    const size_t in_len[] = {tb, tb, tb, gb, tb}, out_len[] = {tb, tb, tb, gb};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 5; ++i)
            if (overlaps(outs[o], out_len[o], ins[i], in_len[i])) return RELATION_ERR_INVALID_ARGUMENT;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlaps(outs[o], out_len[o], outs[o2], out_len[o2])) return RELATION_ERR_INVALID_ARGUMENT;
    }
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    if (workspace_bytes < linear_ws_floats(p, di.num_sms, true) * sizeof(float))
        return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const KernelProblem kp = kernel_problem(p);
    int len = 0;
    const int nseg = linear_segments(kp, di.num_sms, &len);
    const bool reuse = states_from_forward != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (gate_dalog != nullptr) {
        const size_t pb = (size_t)p->H * (size_t)p->d_h * sizeof(float);
        if (cudaMemsetAsync(gate_dalog, 0, pb, s) != cudaSuccess || cudaMemsetAsync(gate_ddtb, 0, pb, s) != cudaSuccess)
            return RELATION_ERR_CUDA;
    }
    st = from_cuda(launch_linear_bwd(kp, P1, P2, I, G, dY, dP1, dP2, dI, dG, reuse, static_cast<float*>(workspace),
                                     di.num_sms, s, gate_alog, gate_dtb, gate_dalog, gate_ddtb));
    if (st == RELATION_OK) t_last_launches = nseg > 1 ? (reuse ? 4 : 6) : 2;
    return st;
}
}  // namespace
}  // namespace relation

relation_status_t relation_linear_fwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                      const float* G, void* Y, float* state, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    return run_linear_fwd(p, P1, P2, I, G, nullptr, nullptr, Y, state, workspace, workspace_bytes, stream);
}

relation_status_t relation_linear_bwd(const relation_problem_t* p, const void* P1, const void* P2, const void* I,
                                      const float* G, const void* dY, void* dP1, void* dP2, void* dI, float* dG,
                                      int states_from_forward, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    return run_linear_bwd(p, P1, P2, I, G, nullptr, nullptr, dY, dP1, dP2, dI, dG, nullptr, nullptr,
                          states_from_forward, workspace, workspace_bytes, stream);
}

relation_status_t relation_linear_fwd_gate(const relation_problem_t* p, const void* P1, const void* P2,
                                           const void* I, const float* R, const float* A_log, const float* dt_bias,
                                           void* Y, float* state, void* workspace, size_t workspace_bytes,
                                           void* stream) {
    relation_status_t st = check_linear(p);
    if (st != RELATION_OK) return st;
    const size_t tb = tensor_bytes(p), sb = (size_t)p->B * p->H * p->d_h * p->d_h * sizeof(float);
    const void* ts[] = {P1, P2, I, R, Y, state};
    const size_t bs[] = {tb, tb, tb, 2 * tb, tb, sb};
    if ((st = check_gate(p, A_log, dt_bias, ts, bs, state ? 6 : 5)) != RELATION_OK) return st;
    return run_linear_fwd(p, P1, P2, I, R, A_log, dt_bias, Y, state, workspace, workspace_bytes, stream);
}

relation_status_t relation_linear_bwd_gate(const relation_problem_t* p, const void* P1, const void* P2,
                                           const void* I, const float* R, const float* A_log, const float* dt_bias,
                                           const void* dY, void* dP1, void* dP2, void* dI, float* dR, float* dA_log,
                                           float* d_dt_bias, int states_from_forward, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    relation_status_t st = check_linear(p);
    if (st != RELATION_OK) return st;
    const size_t tb = tensor_bytes(p);
    const void* ts[] = {P1, P2, I, R, dY, dP1, dP2, dI, dR};
    const size_t bs[] = {tb, tb, tb, 2 * tb, tb, tb, tb, tb, 2 * tb};
    if ((st = check_gate(p, A_log, dt_bias, ts, bs, 9)) != RELATION_OK) return st;
    float* outs[] = {dA_log, d_dt_bias};
    const size_t pb = (size_t)p->H * (size_t)p->d_h * sizeof(float);
    for (float* o : outs) {
        if (o == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
        if (reinterpret_cast<uintptr_t>(o) & 3u) return RELATION_ERR_MISALIGNED;
        for (int k = 0; k < 9; ++k)
            if (overlaps(o, pb, ts[k], bs[k])) return RELATION_ERR_INVALID_ARGUMENT;
        if (overlaps(o, pb, A_log, pb) || overlaps(o, pb, dt_bias, pb)) return RELATION_ERR_INVALID_ARGUMENT;
    }
    if (overlaps(dA_log, pb, d_dt_bias, pb)) return RELATION_ERR_INVALID_ARGUMENT;
    return run_linear_bwd(p, P1, P2, I, R, A_log, dt_bias, dY, dP1, dP2, dI, dR, dA_log, d_dt_bias,
                          states_from_forward, workspace, workspace_bytes, stream);
}

size_t relation_decode_workspace_bytes(const relation_problem_t* p) {
    if (check_problem(p) != RELATION_OK || !decode_fits(p)) return 0;
    const KernelProblem kp = kernel_problem(p);
    return (size_t)kp.BH * (size_t)decode_chunks(kp, p->dtype == RELATION_BF16) * (size_t)(p->d_h + 2) * sizeof(float);
}

relation_status_t relation_decode(const relation_problem_t* p, const void* P1_new, const void* P2_new,
                                  const void* V_new, void* P2_cache, void* V_cache, const int32_t* positions,
                                  int append, void* Y, float* L, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    relation_status_t st = check_problem(p);
    if (st != RELATION_OK) return st;
    if (!decode_fits(p)) return RELATION_ERR_UNSUPPORTED;
    const void* ptrs[] = {P1_new, P2_new, V_new, P2_cache, V_cache, positions, Y, workspace};
    for (const void* x : ptrs)
        if (x == nullptr) return RELATION_ERR_INVALID_ARGUMENT;
    for (const void* x : ptrs)
        if (!aligned16(x)) return RELATION_ERR_MISALIGNED;
    if (L != nullptr && !aligned16(L)) return RELATION_ERR_MISALIGNED;
    const size_t need = relation_decode_workspace_bytes(p);
    if (workspace_bytes < need) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    const size_t rows = (size_t)p->B * (size_t)p->H, eb = elem_bytes(p);
    const size_t nb = rows * (size_t)p->d_h * eb, cb = tensor_bytes(p);
    const void* in_ptr[] = {P1_new, P2_new, V_new, P2_cache, V_cache, positions};
    const size_t in_len[] = {nb, nb, nb, cb, cb, (size_t)p->B * sizeof(int32_t)};
    const void* out_ptr[] = {Y, L, workspace};
    const size_t out_len[] = {nb, L ? rows * sizeof(float) : 0, need};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(out_ptr[o], out_len[o], in_ptr[i], in_len[i])) return RELATION_ERR_INVALID_ARGUMENT;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(out_ptr[o], out_len[o], out_ptr[o2], out_len[o2])) return RELATION_ERR_INVALID_ARGUMENT;
    }
    if (overlaps(P2_cache, cb, V_cache, cb)) return RELATION_ERR_INVALID_ARGUMENT;
    DeviceInfo di;
    if ((st = device_info(&di)) != RELATION_OK) return st;
    st = from_cuda(launch_decode(kernel_problem(p), p->dtype == RELATION_BF16, P1_new, P2_new, V_new, P2_cache,
                                 V_cache, positions, append, Y, L, static_cast<float*>(workspace), di.status,
                                 di.num_sms, static_cast<cudaStream_t>(stream)));
    if (st == RELATION_OK) t_last_launches = decode_launches(kernel_problem(p), p->dtype == RELATION_BF16);
    return st;
}

int relation_last_launch_count(void) { return t_last_launches; }

const char* relation_status_string(relation_status_t s) {
    switch (s) {
        case RELATION_OK: return "ok";
        case RELATION_ERR_INVALID_ARGUMENT: return "invalid argument";
        case RELATION_ERR_UNSUPPORTED: return "unsupported problem (no kernel for this head width, dtype or size)";
        case RELATION_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case RELATION_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than relation_bwd_workspace_bytes()";
        case RELATION_ERR_CUDA: return "CUDA runtime error";
        case RELATION_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
        case RELATION_ERR_DEVICE_UNSAFE:
            return "a bounded device-side wait expired and a kernel returned with its own copies or products "
                   "possibly still in flight; the CUDA context should not be trusted";
    }
    return "unknown status";
}

int relation_abi_version(void) { return RELATION_ABI_VERSION; }

}  // extern "C"

// relation_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host framework
// whose device memory all belongs to that framework's own allocator (which a
// plain C caller cannot reach), and latency-bound serving loops that must not
// allocate after start-up because cudaMalloc can synchronise the device.  For
// them this entry point runs relation_bwd with its workspace placed in a
// fixed-size device array owned by this library instead of a caller buffer.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds RELATION_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Its host-side name is only a stand-in, so the first call on each device
// looks up its device address with cudaGetSymbolAddress (with that device
// current) and caches it.  With CUDA's default lazy loading of device code,
// that lookup can also be the moment the array is reserved on the device (an
// allocation and possibly a synchronisation inside the driver), so callers
// make the first call at start-up, before any stream capture; later calls
// reserve nothing.
// All calls share the array: relation_bwd's prepare stage rewrites the parts
// that must start at zero on every call, and calls whose work overlaps on the
// GPU (different streams, or different host threads) race on it.
#include <mutex>

#include "../../include/relation.h"

namespace relation {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RELATION_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
relation_status_t scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RELATION_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return RELATION_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return RELATION_OK;
}

}  // namespace
}  // namespace relation

extern "C" relation_status_t relation_bwd_noalloc(const relation_problem_t* p, const void* P1, const void* P2,
                                                  const void* V, const void* Y, const float* L, const void* dY,
                                                  void* dP1, void* dP2, void* dV, float* dlambda, void* stream) {
    const size_t need = relation_bwd_workspace_bytes(p);
    if (need > (size_t)RELATION_NOALLOC_SCRATCH_BYTES) return RELATION_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    if (need > 0) {
        relation_status_t st = relation::scratch_for_current_device(&scratch);
        if (st != RELATION_OK) return st;
    }
    // need == 0 means p is invalid; relation_bwd reports which rule it breaks.
    return relation_bwd(p, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, scratch, (size_t)RELATION_NOALLOC_SCRATCH_BYTES,
                        stream);
}

// sift_noalloc.cu -- sift_dense_prefill without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call us: a serving
// runtime that plans every buffer at start-up and forbids allocation on the
// request path, code that must not risk the implicit device synchronisation
// cudaMalloc/cudaFree can cause, or a host thread that holds no allocator at
// all.  For them this file keeps the dense prefill's scratch (the persistent
// scheduler's work counter, the per-row tile counts and the longest-first
// schedule) in one fixed array in device memory that the library owns.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  Host code
// cannot use the symbol as a device address, so a call asks the runtime for
// the array's address (cudaGetSymbolAddress, with the device current) and
// caches it together with the unique id of the context it was taken in.  A
// later call from another context of that device -- after cudaDeviceReset
// destroyed the primary context and a new one took its place, for instance --
// sees a different id and looks the address up again.
#include <cuda.h>

#include <mutex>

#include "sift_internal.h"

namespace sift {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchSlot {
    unsigned long long ctx_id;  // context the address was taken in (0: none yet)
    void *ptr;
};

std::mutex g_setup_mutex;
ScratchSlot g_slot[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// unique id (for the life of the process) of the calling thread's current context;
// false when there is none or it cannot be read
bool current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(a);
            get_id = reinterpret_cast<CtxGetIdFn>(b);
        }
    });
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// address of this device's copy of the array in the current context; nullptr on failure
void *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    if (current_context_id(&id) && g_slot[dev].ctx_id == id && g_slot[dev].ptr != nullptr)
        return g_slot[dev].ptr;
    // first call in this context (the lookup also makes the device's context current)
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return nullptr;
    if (!current_context_id(&id)) id = 0;  // unknown context: look it up again next time
    g_slot[dev] = ScratchSlot{id, ptr};
    return ptr;
}

}  // namespace
}  // namespace sift

extern "C" sift_status sift_dense_prefill_noalloc(const sift_problem *prob, const void *q,
                                                  const void *k, const void *v,
                                                  float softmax_scale, void *o, float *lse,
                                                  int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_dense_prefill_noalloc");
    sift_status st = validate_problem(prob, true);
    if (st != SIFT_OK) return st;
    const size_t need = sift_workspace_bytes(prob);
    if (need == 0) return SIFT_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return SIFT_ERR_UNSUPPORTED;  // problem too large for the array
    void *scratch = scratch_for_current_device();
    if (scratch == nullptr) return SIFT_ERR_CUDA;
    // the dense path zeroes the work counter itself (an async memset, no allocation)
    // and overwrites the counts and schedule it keeps in the scratch
    return sift_dense_prefill(prob, q, k, v, softmax_scale, o, lse, scratch,
                              kNoAllocScratchBytes, dev_status, stream);
}

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
// cannot use the symbol as a device address, so the first call on each device
// asks the runtime for the array's address (cudaGetSymbolAddress, with that
// device current) and caches it.
#include <mutex>

#include "sift_internal.h"

namespace sift {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// address of this device's copy of the array; nullptr on failure
void *scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace sift

extern "C" sift_status sift_dense_prefill_noalloc(const sift_problem *prob, const void *q,
                                                  const void *k, const void *v,
                                                  float softmax_scale, void *o, float *lse,
                                                  int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
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

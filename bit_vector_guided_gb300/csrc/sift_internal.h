// sift_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/sift.h"

namespace sift {

// An NVTX range named after the entry point, open for the duration of the call (host
// side: validation and enqueueing).  Without a profiler attached it costs a load and a
// branch.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// default limit of every device-side wait; the kernels never spin unbounded
constexpr uint64_t kDefaultWaitTimeoutNs = 2000000000ull;

struct DebugWaits {
    uint64_t timeout_ns;
    int32_t stall;
};
DebugWaits debug_waits();

// scalar / pointer validation shared by every entry point of the aligned layout
sift_status validate_problem(const sift_problem *p, bool attention);

// the same for the general (ragged) layout of sift_decode_ragged and friends
sift_status validate_ragged(const sift_problem *p, bool attention);

// upper bound on the per-segment query tiles: ceil(tokens/tile) + documents + prompts
int64_t max_query_tiles(const sift_problem *p);

// sift_decode_ragged with `exact` = false: num_query_tiles is an upper bound, the rows past
// the real count get an empty query tile (computed, never stored)
sift_status decode_ragged_impl(const sift_problem *prob, int32_t num_query_tiles,
                               const uint64_t *la_words, const uint64_t *ca_words,
                               int32_t *qtiles, int32_t *kv, int32_t *counts, int32_t *sched,
                               int32_t *pages, int32_t page_cap, int32_t *dev_status,
                               cudaStream_t stream, bool exact);

// general layout: CA pages below the tile (and a multiple of 8 tokens) are gathered
// into dense tiles rather than masked inside contiguous ones
inline bool gathers_pages(const sift_problem *p) {
    const int page = p->page ? p->page : p->tile;
    return page < p->tile && page % 8 == 0;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// number of SMs of the current device (cached per device)
int device_sm_count();

// Longest-first ordering of `layers` groups of `units` counts each:
// sched[l*units + r] = unit with the r-th largest count of group l.
cudaError_t launch_schedule(const int32_t *counts, int32_t *sched, int layers, int units,
                            int rowcap, int32_t *dev_status, cudaStream_t stream);

// counts[h*N + i] = number of tiles of prompt(i) up to and including i (dense rows)
cudaError_t launch_dense_counts(const sift_problem *p, int32_t *counts, int32_t *dev_status,
                                cudaStream_t stream);

// workspace layout: [0,256) work counter and padding; then dense counts and schedule
constexpr size_t kWsHeader = 256;

}  // namespace sift

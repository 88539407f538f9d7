// sift_abi.cu -- status strings, argument validation, workspace sizing and the
// wait-limit test hook of the C ABI declared in include/sift.h.
#include <atomic>
#include <climits>

#include "sift_internal.h"

namespace sift {

static std::atomic<uint64_t> g_timeout_ns{kDefaultWaitTimeoutNs};
static std::atomic<int32_t> g_stall{0};

DebugWaits debug_waits() { return DebugWaits{g_timeout_ns.load(), g_stall.load()}; }

sift_status validate_problem(const sift_problem *p, bool attention) {
    if (p == nullptr) return SIFT_ERR_INVALID_ARG;
    if (p->num_prompts < 1 || p->num_docs < 0 || p->num_layers < 1 || p->num_q_heads < 1 ||
        p->num_kv_heads < 1 || p->tile < 1 || p->total_tokens < 1 ||
        p->max_tiles_per_prompt < 1 || p->la_words_len < 0 || p->ca_words_len < 0)
        return SIFT_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return SIFT_ERR_INVALID_ARG;
    if (p->total_tokens % p->tile != 0) return SIFT_ERR_UNSUPPORTED;
    if (p->page != 0 && p->page != p->tile) return SIFT_ERR_UNSUPPORTED;
    if (p->cu_seqlens == nullptr || p->doc_cu == nullptr) return SIFT_ERR_INVALID_ARG;
    if (p->num_docs > 0 && (p->doc_end == nullptr || p->la_off == nullptr || p->ca_off == nullptr))
        return SIFT_ERR_INVALID_ARG;
    const int64_t N = p->total_tokens / p->tile;
    if (N * p->num_kv_heads > INT32_MAX / 2) return SIFT_ERR_UNSUPPORTED;
    if (p->max_tiles_per_prompt > N || p->max_tiles_per_prompt > 49152)
        return SIFT_ERR_INVALID_ARG;
    if (attention) {
        if (p->head_dim != 64 && p->head_dim != 128) return SIFT_ERR_UNSUPPORTED;
        if (p->tile != 64 && p->tile != 128) return SIFT_ERR_UNSUPPORTED;
        if ((p->num_q_heads / p->num_kv_heads) % 2 != 0) return SIFT_ERR_UNSUPPORTED;
        if (static_cast<int64_t>(p->total_tokens) * p->num_q_heads * p->head_dim > INT32_MAX * 8ll)
            return SIFT_ERR_UNSUPPORTED;
    }
    return SIFT_OK;
}

static bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

sift_status validate_ragged(const sift_problem *p, bool attention) {
    if (p == nullptr) return SIFT_ERR_INVALID_ARG;
    if (p->num_prompts < 1 || p->num_docs < 0 || p->num_layers < 1 || p->num_q_heads < 1 ||
        p->num_kv_heads < 1 || p->tile < 1 || p->total_tokens < 1 ||
        p->max_tiles_per_prompt < 1 || p->la_words_len < 0 || p->ca_words_len < 0 ||
        p->page < 0)
        return SIFT_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return SIFT_ERR_INVALID_ARG;
    if (p->cu_seqlens == nullptr || p->doc_cu == nullptr) return SIFT_ERR_INVALID_ARG;
    if (p->num_docs > 0 && (p->doc_end == nullptr || p->la_off == nullptr || p->ca_off == nullptr))
        return SIFT_ERR_INVALID_ARG;
    // the list format holds a tile's length in 8 bits and at most 16 page bits
    if (!pow2(p->tile) || p->tile < 8 || p->tile > 128) return SIFT_ERR_UNSUPPORTED;
    const int page = p->page ? p->page : p->tile;
    if (!pow2(page) || page < p->tile / 16 || page > (1 << 24)) return SIFT_ERR_UNSUPPORTED;
    if (p->max_tiles_per_prompt > 49152) return SIFT_ERR_INVALID_ARG;
    const int64_t cap = max_query_tiles(p);
    if (cap * p->num_kv_heads > INT32_MAX / 2) return SIFT_ERR_UNSUPPORTED;
    if (attention) {
        if (p->head_dim != 64 && p->head_dim != 128) return SIFT_ERR_UNSUPPORTED;
        if (p->tile != 64 && p->tile != 128) return SIFT_ERR_UNSUPPORTED;
        if ((p->num_q_heads / p->num_kv_heads) % 2 != 0) return SIFT_ERR_UNSUPPORTED;
        if (static_cast<int64_t>(p->total_tokens) * p->num_q_heads * p->head_dim > INT32_MAX * 8ll)
            return SIFT_ERR_UNSUPPORTED;
    }
    return SIFT_OK;
}

int64_t max_query_tiles(const sift_problem *p) {
    // each segment (documents and suffixes) adds at most one partial tile
    return (static_cast<int64_t>(p->total_tokens) + p->tile - 1) / p->tile + p->num_docs +
           p->num_prompts;
}

int device_sm_count() {
    // several host threads may launch at once: each slot is read and written atomically
    // (a race only repeats the attribute query, which returns the same value)
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace sift

extern "C" {

const char *sift_status_string(sift_status s) {
    switch (s) {
        case SIFT_OK: return "SIFT_OK";
        case SIFT_ERR_INVALID_ARG: return "SIFT_ERR_INVALID_ARG";
        case SIFT_ERR_UNSUPPORTED: return "SIFT_ERR_UNSUPPORTED";
        case SIFT_ERR_CUDA: return "SIFT_ERR_CUDA";
        case SIFT_ERR_TIMEOUT: return "SIFT_ERR_TIMEOUT";
        case SIFT_ERR_DEVICE_CHECK: return "SIFT_ERR_DEVICE_CHECK";
    }
    return "SIFT_ERR_UNKNOWN";
}

size_t sift_workspace_bytes(const sift_problem *p) {
    size_t units = 0;
    if (sift::validate_problem(p, false) == SIFT_OK)
        units = static_cast<size_t>(p->total_tokens / p->tile) * p->num_kv_heads;
    else if (sift::validate_ragged(p, false) == SIFT_OK)
        units = static_cast<size_t>(sift::max_query_tiles(p)) * p->num_kv_heads;
    else
        return 0;
    return sift::kWsHeader + 2 * units * sizeof(int32_t);
}

void sift_debug_set_waits(uint64_t wait_timeout_ns, int32_t stall_flag) {
    sift::g_timeout_ns.store(wait_timeout_ns ? wait_timeout_ns : sift::kDefaultWaitTimeoutNs);
    sift::g_stall.store(stall_flag);
}

int32_t sift_abi_version(void) { return 101; }

}  // extern "C"

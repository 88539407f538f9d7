// sift_decode.cu -- bit-vector decode (SIFT pages, "Dettagli di Implementazione":
// a custom kernel turns the LA/CA bit vectors into explicit tile indices) and
// the longest-first schedule consumed by the persistent attention kernel.
//
// One warp decodes one (layer, kv head, query tile) row.  The candidate tiles
// of a row arrive as 64-bit words (CA words of every earlier document of the
// prompt, then the row's own LA word(s)); every lane sees the same word, tests
// its own bit, and takes its output slot from the popcount of the lower lanes'
// bits, so each 32-bit half-word is compacted with one popc and written with
// one coalesced store.  Document metadata for up to 32 earlier documents is
// fetched by the 32 lanes at once and broadcast with shuffles.
#include "ptx.cuh"
#include "sift_internal.h"

namespace sift {
namespace {

constexpr int kDecodeWarps = 8;

struct DecodeArgs {
    const int32_t *cu;
    const int32_t *doc_cu;
    const int32_t *doc_end;
    const int64_t *la_off;
    const int64_t *ca_off;
    const uint64_t *la;
    const uint64_t *ca;
    int64_t la_len, ca_len;
    int32_t *kv_idx;
    int32_t *counts;
    int32_t *status;
    int P, D, Hkv, B, N, rowcap;
    int64_t rows;
};

__device__ __forceinline__ void set_status(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ int find_prompt(const int32_t *cu, int P, int64_t tok) {
    int lo = 0, hi = P - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= tok) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct RowWriter {
    int32_t *out;
    int n;
    int rowcap;
    uint32_t lane;
    // compact the first nb (<= 64) bits of `word`; bit b stands for tile tile0 + b
    __device__ __forceinline__ void emit(uint64_t word, int nb, int tile0) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int rem = nb - 32 * half;
            if (rem <= 0) break;
            uint32_t bits = static_cast<uint32_t>(word >> (32 * half));
            if (rem < 32) bits &= (1u << rem) - 1u;
            if (bits == 0) continue;
            if ((bits >> lane) & 1u) {
                const int pos = n + __popc(bits & ((1u << lane) - 1u));
                if (pos < rowcap) out[pos] = tile0 + 32 * half + static_cast<int>(lane);
            }
            n += __popc(bits);
        }
    }
};

__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_rows_kernel(const DecodeArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kDecodeWarps + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const int i = static_cast<int>(row % a.N);
    const int h = static_cast<int>((row / a.N) % a.Hkv);
    const int l = static_cast<int>(row / (static_cast<int64_t>(a.N) * a.Hkv));
    const int B = a.B;
    const int64_t tok = static_cast<int64_t>(i) * B;

    const int p = find_prompt(a.cu, a.P, tok);
    const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
    const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
    bool ok = (p0 % B == 0) && (p1 % B == 0) && tok >= p0 && tok < p1 && g0 >= 0 &&
              g0 <= g1 && g1 <= a.D;
    RowWriter w{a.kv_idx + row * a.rowcap, 0, a.rowcap, lane};
    if (!ok) {
        if (lane == 0) {
            set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            w.out[0] = i;
            a.counts[row] = 1;
        }
        return;
    }
    // own document: the first one ending after tok (none -> query suffix)
    int lo = g0, hi = g1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.doc_end + mid) > tok) hi = mid; else lo = mid + 1;
    }
    const int g = lo;
    if (g == g1) {
        // suffix row: every tile of the prompt up to the diagonal
        const int pt = p0 / B;
        int n = i - pt + 1;
        if (n > a.rowcap) { if (lane == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK); n = a.rowcap; }
        for (int k = static_cast<int>(lane); k < n; k += 32) w.out[k] = pt + k;
        if (lane == 0) a.counts[row] = n;
        return;
    }
    bool bad = false;
    // CA pages of the earlier documents, 32 documents per round trip
    for (int base = g0; base < g; base += 32) {
        const int gk = base + static_cast<int>(lane);
        int ds = 0, T = 0;
        int64_t off = 0;
        uint64_t w0 = 0;
        if (gk < g) {
            ds = (gk == g0) ? p0 : __ldg(a.doc_end + gk - 1);
            const int de = __ldg(a.doc_end + gk);
            T = (de - ds) / B;
            const int W = (T + 63) / 64;
            off = __ldg(a.ca_off + gk) + (static_cast<int64_t>(l) * a.Hkv + h) * W;
            if (de <= ds || (de - ds) % B != 0 || ds % B != 0 || off < 0 || off + W > a.ca_len) {
                bad = true;
                T = 0;
            } else {
                w0 = __ldg(a.ca + off);
            }
        }
        const int nd = min(32, g - base);
        for (int k = 0; k < nd; ++k) {
            const int Tk = __shfl_sync(0xffffffffu, T, k);
            const int dsk = __shfl_sync(0xffffffffu, ds, k);
            const int64_t offk = __shfl_sync(0xffffffffu, off, k);
            const uint64_t wk = __shfl_sync(0xffffffffu, w0, k);
            const int W = (Tk + 63) / 64;
            for (int wi = 0; wi < W; ++wi) {
                const uint64_t word = wi == 0 ? wk : __ldg(a.ca + offk + wi);
                w.emit(word, min(64, Tk - 64 * wi), dsk / B + 64 * wi);
            }
        }
    }
    // LA tiles j < i of the own document
    {
        const int ds = (g == g0) ? p0 : __ldg(a.doc_end + g - 1);
        const int de = __ldg(a.doc_end + g);
        const int T = (de - ds) / B;
        const int W = (T + 63) / 64;
        const int il = i - ds / B;
        const int64_t off = __ldg(a.la_off + g) + ((static_cast<int64_t>(l) * a.Hkv + h) * T + il) * W;
        if (de <= ds || (de - ds) % B != 0 || ds % B != 0 || off < 0 || off + W > a.la_len) {
            bad = true;
        } else {
            for (int wi = 0; 64 * wi < il; ++wi)
                w.emit(__ldg(a.la + off + wi), min(64, il - 64 * wi), ds / B + 64 * wi);
        }
    }
    if (lane == 0 && w.n < a.rowcap) w.out[w.n] = i;
    w.n += 1;
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        if (bad || w.n > a.rowcap) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
        a.counts[row] = min(w.n, a.rowcap);
    }
}

// one block per group: counting sort by count, descending
__global__ void __launch_bounds__(1024)
schedule_kernel(const int32_t *counts, int32_t *sched, int units, int rowcap) {
    extern __shared__ int hist[];  // rowcap + 1 bins
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    const int nb = rowcap + 1;
    const int32_t *c = counts + static_cast<int64_t>(blockIdx.x) * units;
    int32_t *s = sched + static_cast<int64_t>(blockIdx.x) * units;
    for (int b = tid; b < nb; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int u = tid; u < units; u += blockDim.x) atomicAdd(&hist[min(max(c[u], 0), rowcap)], 1);
    __syncthreads();
    // exclusive scan over bins in descending count order (bin rowcap first)
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int r0 = tid * per, r1 = min(r0 + per, nb);
    int local = 0;
    for (int r = r0; r < r1; ++r) local += hist[rowcap - r];
    const int lane = tid & 31, wid = tid >> 5;
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        warp_sums[lane] = v;  // inclusive prefix of warp totals
    }
    __syncthreads();
    int run = incl - local + (wid > 0 ? warp_sums[wid - 1] : 0);
    for (int r = r0; r < r1; ++r) {
        const int b = rowcap - r;
        const int v = hist[b];
        hist[b] = run;
        run += v;
    }
    __syncthreads();
    for (int u = tid; u < units; u += blockDim.x) {
        const int pos = atomicAdd(&hist[min(max(c[u], 0), rowcap)], 1);
        s[pos] = u;
    }
}

__global__ void dense_counts_kernel(const int32_t *cu, int P, int B, int N, int Hkv,
                                    int32_t *counts) {
    const int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= static_cast<int64_t>(N) * Hkv) return;
    const int i = static_cast<int>(u % N);
    const int p = find_prompt(cu, P, static_cast<int64_t>(i) * B);
    counts[u] = i - __ldg(cu + p) / B + 1;
}

}  // namespace

cudaError_t launch_schedule(const int32_t *counts, int32_t *sched, int layers, int units,
                            int rowcap, int32_t * /*dev_status*/, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(rowcap + 1) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(schedule_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    schedule_kernel<<<layers, 1024, smem, stream>>>(counts, sched, units, rowcap);
    return cudaGetLastError();
}

cudaError_t launch_dense_counts(const sift_problem *p, int32_t *counts, int32_t * /*dev_status*/,
                                cudaStream_t stream) {
    const int N = p->total_tokens / p->tile;
    const int64_t units = static_cast<int64_t>(N) * p->num_kv_heads;
    const int threads = 256;
    dense_counts_kernel<<<static_cast<unsigned>((units + threads - 1) / threads), threads, 0,
                          stream>>>(p->cu_seqlens, p->num_prompts, p->tile, N, p->num_kv_heads,
                                    counts);
    return cudaGetLastError();
}

}  // namespace sift

extern "C" sift_status sift_decode(const sift_problem *prob, const uint64_t *la_words,
                                   const uint64_t *ca_words, int32_t *kv_idx, int32_t *counts,
                                   int32_t *sched, int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
    sift_status st = validate_problem(prob, false);
    if (st != SIFT_OK) return st;
    if (kv_idx == nullptr || counts == nullptr || sched == nullptr || dev_status == nullptr)
        return SIFT_ERR_INVALID_ARG;
    if ((prob->la_words_len > 0 && la_words == nullptr) ||
        (prob->ca_words_len > 0 && ca_words == nullptr))
        return SIFT_ERR_INVALID_ARG;
    DecodeArgs a;
    a.cu = prob->cu_seqlens;
    a.doc_cu = prob->doc_cu;
    a.doc_end = prob->doc_end;
    a.la_off = prob->la_off;
    a.ca_off = prob->ca_off;
    a.la = la_words;
    a.ca = ca_words;
    a.la_len = prob->la_words_len;
    a.ca_len = prob->ca_words_len;
    a.kv_idx = kv_idx;
    a.counts = counts;
    a.status = dev_status;
    a.P = prob->num_prompts;
    a.D = prob->num_docs;
    a.Hkv = prob->num_kv_heads;
    a.B = prob->tile;
    a.N = prob->total_tokens / prob->tile;
    a.rowcap = prob->max_tiles_per_prompt;
    a.rows = static_cast<int64_t>(prob->num_layers) * a.Hkv * a.N;
    const int64_t blocks = (a.rows + kDecodeWarps - 1) / kDecodeWarps;
    if (blocks > INT32_MAX) return SIFT_ERR_UNSUPPORTED;
    decode_rows_kernel<<<static_cast<unsigned>(blocks), kDecodeWarps * 32, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    if (launch_schedule(counts, sched, prob->num_layers, a.N * a.Hkv, a.rowcap, dev_status,
                        stream) != cudaSuccess)
        return SIFT_ERR_CUDA;
    return SIFT_OK;
}

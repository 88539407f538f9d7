// sift_decode.cu -- bit-vector decode (SIFT pages, "Dettagli di Implementazione":
// a custom kernel turns the LA/CA bit vectors into explicit tile indices) and
// the longest-first schedule consumed by the persistent attention kernel.
//
// One warp decodes all rows of one (layer, kv head, document) -- or of one prompt's
// query suffix.  Candidate tiles arrive as 64-bit words (the CA words of every earlier
// document of the prompt, then each row's own LA word(s)); every lane sees the same
// word, tests its own bit, and takes its output slot from the popcount of the lower
// lanes' bits, so each 32-bit half-word is compacted with one popc and written with
// one coalesced store.  The CA prefix is the same for every row of a document, so it
// is compacted once per document and copied; document metadata for up to 32 earlier
// documents, and the first LA word of up to 32 rows, are fetched by the 32 lanes at
// once and broadcast with shuffles.
#include "ptx.cuh"
#include "sift_internal.h"

namespace sift {
namespace {


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

// One warp per segment of a (layer, kv head): a document of a prompt, or a prompt's
// query suffix.  Every row of a document shares the same CA prefix (the flagged pages
// of the earlier documents), so the warp compacts that prefix once -- into shared
// memory and into the document's first row -- and then writes each row as prefix +
// its own LA tiles + the diagonal.  Suffix rows list every tile of the prompt up to
// the diagonal.
constexpr int kSegWarps = 4;
constexpr int kPrefixCap = 1024;  // CA prefix entries staged in shared memory per warp

__global__ void __launch_bounds__(kSegWarps * 32)
decode_segments_kernel(const DecodeArgs a) {
    __shared__ int32_t prefix_smem[kSegWarps][kPrefixCap];
    const uint32_t lane = threadIdx.x & 31u;
    const int wib = static_cast<int>(threadIdx.x >> 5);
    const int64_t w = static_cast<int64_t>(blockIdx.x) * kSegWarps + wib;
    const int S = a.D + a.P;
    if (w >= a.rows) return;  // rows = layers * Hkv * segments here
    const int seg = static_cast<int>(w % S);
    const int64_t lh = w / S;  // layer * Hkv + kv head
    const int h = static_cast<int>(lh % a.Hkv);
    const int l = static_cast<int>(lh / a.Hkv);
    const int B = a.B;
    const int64_t rowbase = lh * a.N;  // row of global tile 0 for this (layer, kv head)
    int32_t *pre = prefix_smem[wib];

    if (seg >= a.D) {
        // ---- the query suffix of prompt p: dense over the prompt
        const int p = seg - a.D;
        const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
        const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
        if (p0 % B || p1 % B || p0 > p1 || g0 < 0 || g0 > g1 || g1 > a.D) {
            if (lane == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int sstart = g1 > g0 ? __ldg(a.doc_end + g1 - 1) : p0;
        if (sstart % B || sstart < p0 || sstart > p1) {
            if (lane == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int pt = p0 / B;
        for (int i = sstart / B; i < p1 / B; ++i) {
            int32_t *out = a.kv_idx + (rowbase + i) * a.rowcap;
            int n = i - pt + 1;
            if (n > a.rowcap) {
                if (lane == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                n = a.rowcap;
            }
            for (int k = static_cast<int>(lane); k < n; k += 32) out[k] = pt + k;
            if (lane == 0) a.counts[rowbase + i] = n;
        }
        return;
    }

    // ---- document g
    const int g = seg;
    int lo = 0, hi = a.P - 1;  // prompt owning g: the last p with doc_cu[p] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.doc_cu + mid) <= g) lo = mid; else hi = mid - 1;
    }
    const int p = lo;
    const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
    const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
    const int ds = (g == g0) ? p0 : __ldg(a.doc_end + g - 1);
    const int de = __ldg(a.doc_end + g);
    if (g < g0 || g >= g1 || p0 % B || ds % B || de % B || de <= ds || ds < p0 || de > p1) {
        if (lane == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
        return;
    }
    const int T = (de - ds) / B;
    const int W = (T + 63) / 64;
    const int t0 = ds / B;
    int32_t *row0 = a.kv_idx + (rowbase + t0) * a.rowcap;
    bool bad = false;

    // CA prefix of the earlier documents, 32 documents per round trip
    int c = 0;  // warp-uniform
    for (int base = g0; base < g; base += 32) {
        const int gk = base + static_cast<int>(lane);
        int dsk = 0, Tk = 0;
        int64_t offk = 0;
        uint64_t w0 = 0;
        if (gk < g) {
            dsk = (gk == g0) ? p0 : __ldg(a.doc_end + gk - 1);
            const int dek = __ldg(a.doc_end + gk);
            Tk = (dek - dsk) / B;
            const int Wk = (Tk + 63) / 64;
            offk = __ldg(a.ca_off + gk) + (static_cast<int64_t>(l) * a.Hkv + h) * Wk;
            if (dek <= dsk || (dek - dsk) % B != 0 || dsk % B != 0 || offk < 0 ||
                offk + Wk > a.ca_len) {
                bad = true;
                Tk = 0;
            } else {
                w0 = __ldg(a.ca + offk);
            }
        }
        const int nd = min(32, g - base);
        for (int k = 0; k < nd; ++k) {
            const int Tq = __shfl_sync(0xffffffffu, Tk, k);
            const int dsq = __shfl_sync(0xffffffffu, dsk, k);
            const int64_t offq = __shfl_sync(0xffffffffu, offk, k);
            const uint64_t wq = __shfl_sync(0xffffffffu, w0, k);
            const int Wq = (Tq + 63) / 64;
            for (int wi = 0; wi < Wq; ++wi) {
                const uint64_t word = wi == 0 ? wq : __ldg(a.ca + offq + wi);
                const int nb = min(64, Tq - 64 * wi);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int rem = nb - 32 * half;
                    if (rem <= 0) break;
                    uint32_t bits = static_cast<uint32_t>(word >> (32 * half));
                    if (rem < 32) bits &= (1u << rem) - 1u;
                    if (bits == 0) continue;
                    if ((bits >> lane) & 1u) {
                        const int pos = c + __popc(bits & ((1u << lane) - 1u));
                        const int tile = dsq / B + 64 * wi + 32 * half + static_cast<int>(lane);
                        if (pos < kPrefixCap) pre[pos] = tile;
                        if (pos < a.rowcap) row0[pos] = tile;
                    }
                    c += __popc(bits);
                }
            }
        }
    }
    __syncwarp();

    // rows of the document: prefix, LA tiles j < il, diagonal
    const int64_t la_base = __ldg(a.la_off + g) + (static_cast<int64_t>(l) * a.Hkv + h) * T * W;
    if (la_base < 0 || la_base + static_cast<int64_t>(T) * W > a.la_len) bad = true;
    bad = __any_sync(0xffffffffu, bad);  // warp-uniform from here on
    const int cc = min(c, a.rowcap);
    for (int rb = 0; rb < T; rb += 32) {
        // first LA word of 32 rows in one round trip
        const int rl = rb + static_cast<int>(lane);
        uint64_t lw = 0;
        if (!bad && rl < T) lw = __ldg(a.la + la_base + static_cast<int64_t>(rl) * W);
        const int nr = min(32, T - rb);
        for (int r = 0; r < nr; ++r) {
            const int il = rb + r;
            const uint64_t word0 = __shfl_sync(0xffffffffu, lw, r);
            RowWriter wr{a.kv_idx + (rowbase + t0 + il) * a.rowcap, cc, a.rowcap, lane};
            if (il > 0)
                for (int k = static_cast<int>(lane); k < cc; k += 32)
                    wr.out[k] = k < kPrefixCap ? pre[k] : row0[k];
            wr.n = c;
            if (!bad) {
                for (int wi = 0; 64 * wi < il; ++wi) {
                    const uint64_t word =
                        wi == 0 ? word0 : __ldg(a.la + la_base + static_cast<int64_t>(il) * W + wi);
                    wr.emit(word, min(64, il - 64 * wi), t0 + 64 * wi);
                }
            }
            if (lane == 0 && wr.n < a.rowcap) wr.out[wr.n] = t0 + il;
            wr.n += 1;
            if (lane == 0) {
                if (wr.n > a.rowcap) bad = true;
                a.counts[rowbase + t0 + il] = min(wr.n, a.rowcap);
            }
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0 && bad) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
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
    // one warp per (layer, kv head, segment), a segment being a document or a suffix
    a.rows = static_cast<int64_t>(prob->num_layers) * a.Hkv * (a.D + a.P);
    const int64_t blocks = (a.rows + kSegWarps - 1) / kSegWarps;
    if (blocks > INT32_MAX) return SIFT_ERR_UNSUPPORTED;
    decode_segments_kernel<<<static_cast<unsigned>(blocks), kSegWarps * 32, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    if (launch_schedule(counts, sched, prob->num_layers, a.N * a.Hkv, a.rowcap, dev_status,
                        stream) != cudaSuccess)
        return SIFT_ERR_CUDA;
    return SIFT_OK;
}

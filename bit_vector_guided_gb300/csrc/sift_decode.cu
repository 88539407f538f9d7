// sift_decode.cu -- bit-vector decode (SIFT pages, "Dettagli di Implementazione":
// a custom kernel turns the LA/CA bit vectors into explicit tile indices) and
// the longest-first schedule consumed by the persistent attention kernel.
//
// One launch does both.  Its first L blocks are the schedule of the L layers:
// block l counts every row of layer l straight from the bits (the CA pages of the
// earlier documents, popcounts over each document once; the row's LA tiles; the
// diagonal; dense rows in the suffix), then sorts the rows longest-first with a
// counting sort in shared memory.  The other blocks write the lists, one block of
// eight warps per (layer, kv head, document or suffix): the CA prefix -- the same
// for every row of a document -- is compacted once, by a scan over the earlier
// documents' popcounts (one warp's shuffles up to 32 documents, the block beyond),
// then each warp takes every eighth row: the prefix, its own LA tiles (each lane
// tests one bit; the slot is the popcount of the lower lanes' bits) and the
// diagonal.  Both kinds of block read only the bits, so they run side by side.
#include <climits>

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
    int32_t *sched;
    int32_t *status;
    int P, D, L, Hkv, B, N, rowcap;
    int sched_blocks;    // blocks [0, sched_blocks) count and schedule one layer each
    int64_t seg_blocks;  // then one block per (layer, kv head, segment)
    int cnt_smem;        // the schedule blocks keep the layer's counts in shared memory
};

constexpr int kDecThreads = 256;
constexpr int kPrefixCap = 2048;  // CA prefix entries staged in shared memory

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

// the prompt owning document g: the last p with doc_cu[p] <= g
__device__ __forceinline__ int doc_prompt(const int32_t *doc_cu, int P, int g) {
    int lo = 0, hi = P - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(doc_cu + mid) <= g) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint64_t low_bits(uint64_t word, int nb) {
    return nb >= 64 ? word : (nb <= 0 ? 0ull : (word & ((1ull << nb) - 1ull)));
}

// Document g of prompt p: first token ds and tile count T; false when its bounds are
// inconsistent (not multiples of B, empty, outside the prompt or the batch)
__device__ __forceinline__ bool doc_span(const DecodeArgs &a, int p, int g, int &ds, int &T) {
    const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
    const int g0 = __ldg(a.doc_cu + p);
    T = 0;
    ds = p0;
    if (g0 < 0 || g < g0 || g >= a.D || p0 < 0) return false;
    if (g > g0) ds = __ldg(a.doc_end + g - 1);
    const int de = __ldg(a.doc_end + g);
    if (p0 % a.B || ds % a.B || de % a.B || de <= ds || ds < p0 || de > p1 ||
        static_cast<int64_t>(de) > static_cast<int64_t>(a.N) * a.B)
        return false;
    T = (de - ds) / a.B;
    return true;
}

// number of set bits among the T CA bits of document g for (layer, kv head); -1 when the
// words lie outside the array
__device__ __forceinline__ int ca_popcount(const DecodeArgs &a, int g, int T, int64_t lh) {
    const int W = (T + 63) / 64;
    const int64_t off = __ldg(a.ca_off + g) + lh * W;
    if (off < 0 || off + W > a.ca_len) return -1;
    int n = 0;
    for (int wi = 0; wi < W; ++wi) n += __popcll(low_bits(__ldg(a.ca + off + wi), T - 64 * wi));
    return n;
}

// exclusive prefix sum over the block; *total receives the sum
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    int before = 0, all = 0;
    const int nw = static_cast<int>(blockDim.x >> 5);
    for (int w = 0; w < nw; ++w) {
        const int ws = warp_sums[w];
        if (w < wid) before += ws;
        all += ws;
    }
    __syncthreads();  // warp_sums may be reused by the next scan
    *total = all;
    return before + incl - v;
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

// Longest-first order of `units` counts: sched[r] = the unit with the r-th largest count
// (ties in any order), by a counting sort in shared memory.  Counts are read from cnt and
// clamped to [1, rowcap]; hist holds rowcap + 1 ints of shared memory.  The whole block
// calls it.
__device__ void sort_longest_first(const int32_t *cnt, int32_t *sched, int units, int rowcap,
                                   int *hist, int *warp_sums) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int nb = rowcap + 1;
    auto bin = [&](int c) { return min(max(c, 1), rowcap); };
    for (int b = tid; b < nb; b += nt) hist[b] = 0;
    __syncthreads();
    for (int u = tid; u < units; u += nt) atomicAdd(&hist[bin(cnt[u])], 1);
    __syncthreads();
    // exclusive scan over the bins in descending count order (bin rowcap first)
    const int per = (nb + nt - 1) / nt;
    const int r0 = tid * per, r1 = min(r0 + per, nb);
    int local = 0;
    for (int r = r0; r < r1; ++r) local += hist[rowcap - r];
    int total = 0;
    int run = block_exclusive_scan(local, warp_sums, &total);
    for (int r = r0; r < r1; ++r) {
        const int b = rowcap - r;
        const int v = hist[b];
        hist[b] = run;
        run += v;
    }
    __syncthreads();
    for (int u = tid; u < units; u += nt) {
        const int pos = atomicAdd(&hist[bin(cnt[u])], 1);
        if (pos < units) sched[pos] = u;
    }
}

// ---- schedule blocks: every row count of layer l from the bits, then the counting sort
// Shared memory: hist[rowcap + 1] | cap[Hkv * D] (CA prefix count of (kv head, document))
// | dstart[D], dT[D] (first tile and tile count of each document, dT = -1 when bad)
// | tinfo[N] (tile i: its document g >= 0, or -1 - p for the suffix of prompt p)
// | cnts[Hkv * N] (the counts again, when a.cnt_smem; else they are read back)
constexpr int kTileUnset = INT_MIN;

__device__ void schedule_layer(const DecodeArgs &a, int l, int32_t *smem) {
    __shared__ int warp_sums[kDecThreads / 32];
    const int tid = threadIdx.x;
    const int nb = a.rowcap + 1;
    const int U = a.Hkv * a.N;
    int *hist = smem;
    int *cap = hist + nb;
    int *dstart = cap + a.Hkv * a.D;
    int *dT = dstart + a.D;
    int *tinfo = dT + a.D;
    int *cnts = tinfo + a.N;
    for (int i = tid; i < a.N; i += kDecThreads) tinfo[i] = kTileUnset;
    __syncthreads();
    for (int g = tid; g < a.D; g += kDecThreads) {
        const int p = doc_prompt(a.doc_cu, a.P, g);
        int ds = 0, T = 0;
        const bool ok = doc_span(a, p, g, ds, T);
        if (!ok) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
        dstart[g] = ds / a.B;
        dT[g] = ok ? T : -1;
        for (int r = 0; r < T; ++r) tinfo[ds / a.B + r] = g;  // T > 0 only inside [0, N)
    }
    for (int p = tid; p < a.P; p += kDecThreads) {
        const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
        const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
        int sstart = p0;
        if (g0 >= 0 && g0 < g1 && g1 <= a.D) sstart = __ldg(a.doc_end + g1 - 1);
        if (p0 % a.B || p1 % a.B || p0 < 0 || sstart % a.B || sstart < p0 || sstart > p1 ||
            static_cast<int64_t>(p1) > static_cast<int64_t>(a.N) * a.B) {
            set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            continue;
        }
        for (int i = sstart / a.B; i < p1 / a.B; ++i) tinfo[i] = -1 - p;
    }
    __syncthreads();
    for (int idx = tid; idx < a.Hkv * a.D; idx += kDecThreads) {
        const int h = idx / a.D, g = idx - (idx / a.D) * a.D;
        int n = 0;
        if (dT[g] > 0) {
            n = ca_popcount(a, g, dT[g], static_cast<int64_t>(l) * a.Hkv + h);
            if (n < 0) {
                set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                n = 0;
            }
        }
        cap[idx] = n;
    }
    __syncthreads();
    // CA prefix of each document: the flagged pages of the earlier documents of its prompt
    for (int idx = tid; idx < a.Hkv * a.P; idx += kDecThreads) {
        const int h = idx / a.P, p = idx - (idx / a.P) * a.P;
        const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
        int run = 0;
        for (int g = max(g0, 0); g < min(g1, a.D); ++g) {
            const int c = cap[h * a.D + g];
            cap[h * a.D + g] = run;
            run += c;
        }
    }
    __syncthreads();
    // every row: prefix + LA tiles below the diagonal + the diagonal; suffix rows dense.
    // Four rows per thread and round, their first LA words loaded before any is used.
    int32_t *cnt = a.counts + static_cast<int64_t>(l) * U;
    constexpr int kR = 4;
    for (int u0 = tid; u0 < U; u0 += kR * kDecThreads) {
        int n[kR];
        uint64_t w0[kR];
        int64_t row[kR];
        int il[kR], W[kR];
#pragma unroll
        for (int k = 0; k < kR; ++k) {
            const int u = u0 + k * kDecThreads;
            n[k] = 0;
            w0[k] = 0;
            row[k] = -1;
            il[k] = 0;
            W[k] = 1;
            if (u >= U) continue;
            const int h = u / a.N, i = u - (u / a.N) * a.N;
            const int info = tinfo[i];
            if (info >= 0 && dT[info] > 0) {
                const int g = info, T = dT[g];
                W[k] = (T + 63) / 64;
                il[k] = i - dstart[g];
                const int64_t r = __ldg(a.la_off + g) +
                                  ((static_cast<int64_t>(l) * a.Hkv + h) * T + il[k]) * W[k];
                n[k] = cap[h * a.D + g] + 1;
                if (r < 0 || r + W[k] > a.la_len) {
                    set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                } else {
                    row[k] = r;
                    if (il[k] > 0) w0[k] = __ldg(a.la + r);
                }
            } else if (info != kTileUnset && info < 0) {
                n[k] = i - __ldg(a.cu + (-1 - info)) / a.B + 1;  // the query suffix: dense
            } else {
                set_status(a.status, SIFT_ERR_DEVICE_CHECK);  // a tile of no segment
                n[k] = 1;
            }
        }
#pragma unroll
        for (int k = 0; k < kR; ++k) {
            const int u = u0 + k * kDecThreads;
            if (u >= U) continue;
            if (row[k] >= 0 && il[k] > 0) {
                n[k] += __popcll(low_bits(w0[k], il[k]));
                for (int wi = 1; 64 * wi < il[k]; ++wi)
                    n[k] += __popcll(low_bits(__ldg(a.la + row[k] + wi), il[k] - 64 * wi));
            }
            int v = n[k];
            if (v > a.rowcap || v < 1) {
                set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                v = v < 1 ? 1 : a.rowcap;
            }
            cnt[u] = v;
            if (a.cnt_smem) cnts[u] = v;
        }
    }
    __syncthreads();
    sort_longest_first(a.cnt_smem ? cnts : cnt, a.sched + static_cast<int64_t>(l) * U, U,
                       a.rowcap, hist, warp_sums);
}

// ---- list blocks: all rows of one (layer, kv head, document) or one prompt's suffix
__device__ void decode_segment(const DecodeArgs &a, int64_t w, int32_t *pre) {
    __shared__ int warp_sums[kDecThreads / 32];
    const int tid = threadIdx.x;
    const uint32_t lane = threadIdx.x & 31u;
    const int wid = threadIdx.x >> 5;
    const int S = a.D + a.P;
    const int seg = static_cast<int>(w % S);
    const int64_t lh = w / S;  // layer * Hkv + kv head
    const int B = a.B;
    const int64_t rowbase = lh * a.N;  // row of global tile 0 for this (layer, kv head)

    if (seg >= a.D) {
        // ---- the query suffix of prompt p: dense over the prompt
        const int p = seg - a.D;
        const int p0 = __ldg(a.cu + p), p1 = __ldg(a.cu + p + 1);
        const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
        if (p0 % B || p1 % B || p0 < 0 || p0 > p1 || g0 < 0 || g0 > g1 || g1 > a.D ||
            static_cast<int64_t>(p1) > static_cast<int64_t>(a.N) * B) {
            if (tid == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int sstart = g1 > g0 ? __ldg(a.doc_end + g1 - 1) : p0;
        if (sstart % B || sstart < p0 || sstart > p1) {
            if (tid == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int pt = p0 / B;
        for (int i = sstart / B + wid; i < p1 / B; i += kDecThreads / 32) {
            int32_t *out = a.kv_idx + (rowbase + i) * a.rowcap;
            const int n = min(i - pt + 1, a.rowcap);  // a longer row is reported by the counts
            for (int k = static_cast<int>(lane); k < n; k += 32) out[k] = pt + k;
        }
        return;
    }

    // ---- document g
    const int g = seg;
    const int p = doc_prompt(a.doc_cu, a.P, g);
    const int p0 = __ldg(a.cu + p);
    const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
    int ds = 0, T = 0;
    if (g < g0 || g >= g1 || !doc_span(a, p, g, ds, T)) {
        if (tid == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
        return;
    }
    const int W = (T + 63) / 64;
    const int t0 = ds / B;
    int32_t *rows = a.kv_idx + (rowbase + t0) * a.rowcap;  // row il at rows + il*rowcap

    // CA prefix of the earlier documents: each thread counts one earlier document's flagged
    // pages, a scan places them, each thread writes its pages.  Up to 32 earlier documents
    // (the usual case) warp 0 does it alone with a shuffle scan; beyond, the whole block
    // takes kDecThreads documents per round.
    auto count_doc = [&](int gk, int &dsk, int &Tk, int64_t &offk) {
        int cnt = 0;
        Tk = 0;
        if (gk < g) {
            if (!doc_span(a, p, gk, dsk, Tk)) {
                set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                Tk = 0;
            } else {
                const int Wk = (Tk + 63) / 64;
                offk = __ldg(a.ca_off + gk) + lh * Wk;
                if (offk < 0 || offk + Wk > a.ca_len) {
                    set_status(a.status, SIFT_ERR_DEVICE_CHECK);
                    Tk = 0;
                } else {
                    for (int wi = 0; wi < Wk; ++wi)
                        cnt += __popcll(low_bits(__ldg(a.ca + offk + wi), Tk - 64 * wi));
                }
            }
        }
        return cnt;
    };
    auto write_doc = [&](int pos, int dsk, int Tk, int64_t offk) {
        for (int wi = 0; 64 * wi < Tk; ++wi) {
            uint64_t word = low_bits(__ldg(a.ca + offk + wi), Tk - 64 * wi);
            while (word) {
                const int b = __ffsll(static_cast<long long>(word)) - 1;
                word &= word - 1;
                const int tile = dsk / B + 64 * wi + b;
                if (pos < kPrefixCap) {
                    pre[pos] = tile;
                } else if (pos < a.rowcap) {  // rare: beyond the staged prefix, straight to every row
                    for (int r = 0; r < T; ++r) rows[static_cast<int64_t>(r) * a.rowcap + pos] = tile;
                }
                ++pos;
            }
        }
    };
    __shared__ int prefix_total;
    int c = 0;  // block-uniform
    if (g - g0 <= 32) {
        if (wid == 0) {
            int dsk = 0, Tk = 0;
            int64_t offk = 0;
            const int cnt = count_doc(g0 + static_cast<int>(lane), dsk, Tk, offk);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (static_cast<int>(lane) >= o) incl += t;
            }
            write_doc(incl - cnt, dsk, Tk, offk);
            if (lane == 31) prefix_total = incl;
        }
        __syncthreads();
        c = prefix_total;
    } else {
        for (int base = g0; base < g; base += kDecThreads) {
            int dsk = 0, Tk = 0;
            int64_t offk = 0;
            const int cnt = count_doc(base + tid, dsk, Tk, offk);
            int total = 0;
            const int pos = c + block_exclusive_scan(cnt, warp_sums, &total);
            write_doc(pos, dsk, Tk, offk);
            c += total;
        }
        __syncthreads();
    }

    // rows of the document, warp w taking every eighth row from w: prefix, LA tiles j < il,
    // diagonal
    const int64_t la_base = __ldg(a.la_off + g) + (lh * T) * W;
    const bool la_ok = la_base >= 0 && la_base + static_cast<int64_t>(T) * W <= a.la_len;
    if (!la_ok && tid == 0) set_status(a.status, SIFT_ERR_DEVICE_CHECK);
    const int cc = min(min(c, kPrefixCap), a.rowcap);
    for (int il = wid; il < T; il += kDecThreads / 32) {
        RowWriter wr{rows + static_cast<int64_t>(il) * a.rowcap, c, a.rowcap, lane};
        for (int k = static_cast<int>(lane); k < cc; k += 32) wr.out[k] = pre[k];
        if (la_ok) {
            for (int wi = 0; 64 * wi < il; ++wi)
                wr.emit(__ldg(a.la + la_base + static_cast<int64_t>(il) * W + wi),
                        min(64, il - 64 * wi), t0 + 64 * wi);
        }
        if (lane == 0 && wr.n < a.rowcap) wr.out[wr.n] = t0 + il;
    }
}

__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeArgs a) {
    extern __shared__ int32_t dec_smem[];
    if (static_cast<int>(blockIdx.x) < a.sched_blocks)
        schedule_layer(a, blockIdx.x, dec_smem);
    else
        decode_segment(a, static_cast<int64_t>(blockIdx.x) - a.sched_blocks, dec_smem);
}

// one block per layer: longest-first over the layer's units
__global__ void __launch_bounds__(1024)
schedule_kernel(const int32_t *counts, int32_t *sched, int units, int rowcap) {
    extern __shared__ int hist[];  // rowcap + 1 bins
    __shared__ int warp_sums[32];
    const int64_t off = static_cast<int64_t>(blockIdx.x) * units;
    sort_longest_first(counts + off, sched + off, units, rowcap, hist, warp_sums);
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
    NvtxRange nvtx_range("sift_decode");
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
    a.sched = sched;
    a.status = dev_status;
    a.P = prob->num_prompts;
    a.D = prob->num_docs;
    a.L = prob->num_layers;
    a.Hkv = prob->num_kv_heads;
    a.B = prob->tile;
    a.N = prob->total_tokens / prob->tile;
    a.rowcap = prob->max_tiles_per_prompt;
    // one list block per (layer, kv head, segment), a segment being a document or a suffix
    const int64_t seg_blocks = static_cast<int64_t>(a.L) * a.Hkv * (a.D + a.P);
    // schedule blocks: hist, cap, dstart, dT, tinfo (+ the counts when they fit)
    const size_t sched_base = (static_cast<size_t>(a.rowcap) + 1 +
                               static_cast<size_t>(a.Hkv) * a.D + 2 * static_cast<size_t>(a.D) +
                               static_cast<size_t>(a.N)) *
                              sizeof(int32_t);
    const size_t cnt_bytes = static_cast<size_t>(a.Hkv) * a.N * sizeof(int32_t);
    const size_t list_smem = kPrefixCap * sizeof(int32_t);
    // 227 KB per block, less the kernel's own static shared memory
    constexpr size_t kSmemMax = 226 * 1024;
    if (sched_base > kSmemMax) return SIFT_ERR_UNSUPPORTED;
    a.cnt_smem = sched_base + cnt_bytes <= kSmemMax;
    const size_t sched_smem = sched_base + (a.cnt_smem ? cnt_bytes : 0);
    if (seg_blocks + a.L > INT32_MAX) return SIFT_ERR_UNSUPPORTED;
    // opt in to more than the default 48 KB of dynamic shared memory only when needed
    auto allow_smem = [](size_t bytes) {
        return bytes <= 48 * 1024 ||
               cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(bytes)) == cudaSuccess;
    };
    // one launch (the schedule blocks beside the list blocks) while the schedule's shared
    // memory is small; otherwise the list blocks keep theirs small in a launch of their own
    constexpr size_t kOneLaunchSmem = 32 * 1024;
    if (sched_smem <= kOneLaunchSmem) {
        a.sched_blocks = a.L;
        a.seg_blocks = seg_blocks;
        const size_t smem = sched_smem > list_smem ? sched_smem : list_smem;
        decode_kernel<<<static_cast<unsigned>(a.L + seg_blocks), kDecThreads, smem, stream>>>(a);
        return cudaGetLastError() == cudaSuccess ? SIFT_OK : SIFT_ERR_CUDA;
    }
    if (!allow_smem(sched_smem)) return SIFT_ERR_CUDA;
    a.sched_blocks = a.L;
    a.seg_blocks = 0;
    decode_kernel<<<static_cast<unsigned>(a.L), kDecThreads, sched_smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    a.sched_blocks = 0;
    a.seg_blocks = seg_blocks;
    decode_kernel<<<static_cast<unsigned>(seg_blocks), kDecThreads, list_smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SIFT_OK : SIFT_ERR_CUDA;
}

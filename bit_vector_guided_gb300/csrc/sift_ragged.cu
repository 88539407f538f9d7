// sift_ragged.cu -- bit decode on a general layout: documents and query suffixes of any
// length, each tiled from its own first token, and CA pages of a size of their own (SIFT
// pages, "Dettagli di Implementazione": a decoding kernel turns the LA/CA bits into the
// tile indices the sparse kernel iterates over; the pages fix no tile or page size).
//
// Three launches:
//   ragged_tiles_kernel   one block: cuts every segment into query tiles (a block-wide
//                         scan of the per-segment tile counts) and writes (first, rows);
//   ragged_decode_kernel  one warp per (layer, kv head, segment): the CA prefix (tiles of
//                         the earlier documents holding a flagged page, or -- for pages
//                         below the tile -- the flagged whole pages gathered tile/page at
//                         a time, then the flagged partial last pages) is compacted once
//                         with ballots into the segment's first row and copied to the
//                         others; each row then appends its LA tiles and its own tile;
//   schedule_kernel       the longest-first order shared with the aligned decode.
// List entries are (first token, info) pairs, info = len | causal << 8 | gather << 9 |
// mask << 16; a gathered entry's first field indexes the page array instead (the format
// and its reading are stated in include/sift.h).
#include "sift_internal.h"

namespace sift {
namespace {

constexpr int kRaggedWarps = 8;
constexpr uint32_t kAll = 0xffffffffu;

struct RaggedArgs {
    const int32_t *cu, *doc_cu, *doc_end;
    const int64_t *la_off, *ca_off;
    const uint64_t *la, *ca;
    int64_t la_len, ca_len;
    int32_t *qt, *kv, *counts, *status;
    int32_t *pages;  // gathered pages [L][Hkv][D][page_cap] (gather only)
    int P, D, Hkv, L, B, page, NQ, rowcap, page_cap, T;
    uint32_t full;   // mask bits of a tile with every page kept
    bool gather;     // page < tile and a multiple of 8: CA pages are gathered into tiles
    bool exact;      // NQ is the exact tile count (else an upper bound; spare rows stay empty)
};

__device__ __forceinline__ void rstatus(int32_t *st, int code) { atomicCAS(st, 0, code); }

struct Seg {
    int start, end;  // tokens [start, end)
    int g;           // document, or -1 for the prompt's query suffix
    int p;           // prompt
    int g0;          // first document of the prompt
    bool ok;
};

// segment idx in token order: the documents of prompt 0, its suffix, the documents of
// prompt 1, ...  Segment idx belongs to the last prompt p with doc_cu[p] + p <= idx.
__device__ Seg seg_geom(const RaggedArgs &a, int idx) {
    Seg s{0, 0, -1, 0, 0, false};
    int lo = 0, hi = a.P - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.doc_cu + mid) + mid <= idx) lo = mid; else hi = mid - 1;
    }
    const int p = lo;
    const int g0 = __ldg(a.doc_cu + p), g1 = __ldg(a.doc_cu + p + 1);
    const int c0 = __ldg(a.cu + p), c1 = __ldg(a.cu + p + 1);
    if (g0 < 0 || g1 < g0 || g1 > a.D || c0 < 0 || c1 < c0) return s;
    const int j = idx - p;
    s.p = p;
    s.g0 = g0;
    if (j < g1) {
        if (j < g0) return s;
        s.g = j;
        s.start = (j == g0) ? c0 : __ldg(a.doc_end + j - 1);
        s.end = __ldg(a.doc_end + j);
    } else if (j == g1) {
        s.g = -1;
        s.start = g1 > g0 ? __ldg(a.doc_end + g1 - 1) : c0;
        s.end = c1;
    } else {
        return s;
    }
    s.ok = c0 <= s.start && s.start <= s.end && s.end <= c1;
    return s;
}

// query tiles of every segment, numbered in token order
__global__ void __launch_bounds__(1024) ragged_tiles_kernel(RaggedArgs a) {
    __shared__ int32_t scan[1024];
    __shared__ int32_t carry;
    const int tid = threadIdx.x;
    const int S = a.D + a.P;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < S; base += 1024) {
        const int idx = base + tid;
        Seg sg{};
        int nt = 0;
        if (idx < S) {
            sg = seg_geom(a, idx);
            if (!sg.ok) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
            else nt = (sg.end - sg.start + a.B - 1) / a.B;
        }
        scan[tid] = nt;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan (Hillis-Steele)
            const int v = tid >= off ? scan[tid - off] : 0;
            __syncthreads();
            scan[tid] += v;
            __syncthreads();
        }
        const int first = carry + scan[tid] - nt;
        for (int t = 0; t < nt; ++t) {
            const int q = first + t;
            if (q < a.NQ) {
                const int x = sg.start + t * a.B;
                a.qt[2 * q] = x;
                a.qt[2 * q + 1] = min(a.B, sg.end - x);
            }
        }
        __syncthreads();
        if (tid == 1023) carry += scan[1023];
        __syncthreads();
    }
    const int total = carry;
    if (tid == 0 && (a.exact ? total != a.NQ : total > a.NQ))
        rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
    // rows the segments did not fill (a row count given as an upper bound, or an
    // inconsistency): an empty query tile at the end of the batch -- which keeps the table
    // ascending -- with a one-entry list, so that every row the attention kernel reads is
    // defined (its loads fall past the tensors and read zeros; nothing is stored)
    for (int q = total + tid; q < a.NQ; q += 1024) {
        a.qt[2 * q] = a.T;
        a.qt[2 * q + 1] = 0;
        for (int lh = 0; lh < a.L * a.Hkv; ++lh) {
            const int64_t row = static_cast<int64_t>(lh) * a.NQ + q;
            a.counts[row] = 1;
            a.kv[2 * row * a.rowcap] = a.T;
            a.kv[2 * row * a.rowcap + 1] = static_cast<int32_t>(1u | 1u << 8 | a.full << 16);
        }
    }
}

// mask bits of CA tile t (first key y, len keys) of a document whose CA words start at off
__device__ __forceinline__ uint32_t ca_tile_mask(const RaggedArgs &a, int64_t off, int t,
                                                 int len) {
    if (a.page >= a.B) {  // the tile lies inside page t*B/page
        const int pg = static_cast<int>(static_cast<int64_t>(t) * a.B / a.page);
        return static_cast<uint32_t>((__ldg(a.ca + off + pg / 64) >> (pg % 64)) & 1ull);
    }
    const int ppt = a.B / a.page;  // pages per tile, a divisor of 64
    const int pg0 = t * ppt;
    uint32_t m = static_cast<uint32_t>((__ldg(a.ca + off + pg0 / 64) >> (pg0 % 64)) & a.full);
    const int pages = (len + a.page - 1) / a.page;  // pages that start inside the tile
    return pages >= 32 ? m : (m & ((1u << pages) - 1u));
}

__global__ void __launch_bounds__(kRaggedWarps * 32) ragged_decode_kernel(RaggedArgs a) {
    const int S = a.D + a.P;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * kRaggedWarps + (threadIdx.x >> 5);
    const uint32_t lane = threadIdx.x & 31u;
    if (wid >= static_cast<int64_t>(a.L) * a.Hkv * S) return;
    const int idx = static_cast<int>(wid % S);
    const int lh = static_cast<int>(wid / S);
    const int h = lh % a.Hkv, l = lh / a.Hkv;
    const Seg sg = seg_geom(a, idx);
    if (!sg.ok || sg.end == sg.start) return;  // reported by the tiles kernel
    // the segment's first query tile (the table ascends by first token)
    int lo = 0, hi = a.NQ;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.qt + 2 * mid) < sg.start) lo = mid + 1; else hi = mid;
    }
    if (lo >= a.NQ || __ldg(a.qt + 2 * lo) != sg.start) {
        if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
        return;
    }
    const int qfirst = lo;
    const int B = a.B;
    const int nt = (sg.end - sg.start + B - 1) / B;
    const bool suffix = sg.g < 0;
    const int g_end = suffix ? __ldg(a.doc_cu + sg.p + 1) : sg.g;
    const uint32_t lt = (1u << lane) - 1u;
    auto row_of = [&](int q) { return (static_cast<int64_t>(lh) * a.NQ + q) * a.rowcap; };

    // ---- prefix: tiles of the earlier documents, into the first row's list
    const int64_t r0 = row_of(qfirst);
    int npre = 0;
    if (!suffix && a.gather) {
        // whole flagged pages of the earlier documents, ascending, into the page array
        const int64_t pbase = (static_cast<int64_t>(lh) * a.D + sg.g) * a.page_cap;
        const int64_t rel = (static_cast<int64_t>(h) * a.D + sg.g) * a.page_cap;
        int npg = 0;
        for (int gp = sg.g0; gp < g_end; ++gp) {
            const int ds = (gp == sg.g0) ? __ldg(a.cu + sg.p) : __ldg(a.doc_end + gp - 1);
            const int de = __ldg(a.doc_end + gp);
            if (de < ds) {
                if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
                continue;
            }
            const int C = (de - ds + a.page - 1) / a.page;
            const int V = (C + 63) / 64;
            const int64_t off = __ldg(a.ca_off + gp) + static_cast<int64_t>(lh) * V;
            if (off < 0 || off + V > a.ca_len) {
                if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
                continue;
            }
            const int whole = (de - ds) / a.page;
            for (int j0 = 0; j0 < whole; j0 += 32) {
                const int j = j0 + static_cast<int>(lane);
                const bool inc = j < whole && ((__ldg(a.ca + off + j / 64) >> (j % 64)) & 1ull);
                const uint32_t bal = __ballot_sync(kAll, inc);
                const int pos = npg + __popc(bal & lt);
                if (inc && pos < a.page_cap) a.pages[pbase + pos] = ds + j * a.page;
                npg += __popc(bal);
            }
        }
        if (npg > a.page_cap) {
            if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
            npg = a.page_cap;
        }
        const int per = a.B / a.page;
        const int ngroups = (npg + per - 1) / per;
        for (int k = static_cast<int>(lane); k < ngroups; k += 32) {
            const int pos = npre + k;
            if (pos < a.rowcap) {
                const int in_group = min(per, npg - k * per);
                a.kv[2 * (r0 + pos)] = static_cast<int32_t>(rel + k * per);
                a.kv[2 * (r0 + pos) + 1] = static_cast<int32_t>(
                    static_cast<uint32_t>(in_group * a.page) | 1u << 9 | a.full << 16);
            }
        }
        npre += ngroups;
        // then each earlier document's last page when it is partial and flagged
        for (int gb = sg.g0; gb < g_end; gb += 32) {
            const int gp = gb + static_cast<int>(lane);
            bool inc = false;
            int first = 0, rem = 0;
            if (gp < g_end) {
                const int ds = (gp == sg.g0) ? __ldg(a.cu + sg.p) : __ldg(a.doc_end + gp - 1);
                const int de = __ldg(a.doc_end + gp);
                rem = de >= ds ? (de - ds) % a.page : 0;
                if (rem) {
                    const int C = (de - ds + a.page - 1) / a.page;
                    const int V = (C + 63) / 64;
                    const int64_t off = __ldg(a.ca_off + gp) + static_cast<int64_t>(lh) * V;
                    const int j = C - 1;
                    inc = off >= 0 && off + V <= a.ca_len &&
                          ((__ldg(a.ca + off + j / 64) >> (j % 64)) & 1ull);
                    first = de - rem;
                }
            }
            const uint32_t bal = __ballot_sync(kAll, inc);
            const int pos = npre + __popc(bal & lt);
            if (inc && pos < a.rowcap) {
                a.kv[2 * (r0 + pos)] = first;
                a.kv[2 * (r0 + pos) + 1] = static_cast<int32_t>(static_cast<uint32_t>(rem) | 1u << 16);
            }
            npre += __popc(bal);
        }
    }
    for (int gp = sg.g0; gp < g_end && !(!suffix && a.gather); ++gp) {
        const int ds = (gp == sg.g0) ? __ldg(a.cu + sg.p) : __ldg(a.doc_end + gp - 1);
        const int de = __ldg(a.doc_end + gp);
        if (de < ds) {
            if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
            continue;
        }
        const int ntp = (de - ds + B - 1) / B;
        int64_t off = 0;
        if (!suffix) {
            const int C = (de - ds + a.page - 1) / a.page;
            const int V = (C + 63) / 64;
            off = __ldg(a.ca_off + gp) + static_cast<int64_t>(lh) * V;
            if (off < 0 || off + V > a.ca_len) {
                if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
                continue;
            }
        }
        for (int t0 = 0; t0 < ntp; t0 += 32) {
            const int t = t0 + static_cast<int>(lane);
            uint32_t info = 0;
            bool inc = false;
            int y = 0;
            if (t < ntp) {
                y = ds + t * B;
                const int len = min(B, de - y);
                const uint32_t mask = suffix ? a.full : ca_tile_mask(a, off, t, len);
                inc = mask != 0;
                info = static_cast<uint32_t>(len) | mask << 16;
            }
            const uint32_t bal = __ballot_sync(kAll, inc);
            const int pos = npre + __popc(bal & lt);
            if (inc && pos < a.rowcap) {
                a.kv[2 * (r0 + pos)] = y;
                a.kv[2 * (r0 + pos) + 1] = static_cast<int32_t>(info);
            }
            npre += __popc(bal);
        }
    }
    __syncwarp();  // the prefix in row qfirst is read back by every lane below

    // ---- each row: prefix, then its own document's (suffix's) earlier tiles, then itself
    const int T = nt;
    const int Wla = (T + 63) / 64;
    int64_t la_base = 0;
    bool la_ok = true;
    if (!suffix) {
        la_base = __ldg(a.la_off + sg.g) + static_cast<int64_t>(lh) * T * Wla;
        la_ok = la_base >= 0 && la_base + static_cast<int64_t>(T) * Wla <= a.la_len;
        if (!la_ok && lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
    }
    const uint32_t full_info = static_cast<uint32_t>(B) | a.full << 16;
    for (int i = 0; i < nt; ++i) {
        const int q = qfirst + i;
        if (q >= a.NQ) {
            if (lane == 0) rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
            break;
        }
        const int64_t rb = row_of(q);
        const int ncopy = min(npre, a.rowcap);
        if (i > 0)
            for (int e = static_cast<int>(lane); e < ncopy; e += 32) {
                a.kv[2 * (rb + e)] = a.kv[2 * (r0 + e)];
                a.kv[2 * (rb + e) + 1] = a.kv[2 * (r0 + e) + 1];
            }
        int n = npre;
        for (int b0 = 0; b0 < i; b0 += 32) {
            const int b = b0 + static_cast<int>(lane);
            bool inc = b < i;
            if (inc && !suffix)
                inc = la_ok &&
                      ((__ldg(a.la + la_base + static_cast<int64_t>(i) * Wla + b / 64) >> (b % 64)) &
                       1ull);
            const uint32_t bal = __ballot_sync(kAll, inc);
            const int pos = n + __popc(bal & lt);
            if (inc && pos < a.rowcap) {
                a.kv[2 * (rb + pos)] = sg.start + b * B;
                a.kv[2 * (rb + pos) + 1] = static_cast<int32_t>(full_info);
            }
            n += __popc(bal);
        }
        const int x = sg.start + i * B;
        if (lane == 0) {
            if (n < a.rowcap) {
                a.kv[2 * (rb + n)] = x;
                a.kv[2 * (rb + n) + 1] =
                    static_cast<int32_t>(static_cast<uint32_t>(min(B, sg.end - x)) | 1u << 8 |
                                         a.full << 16);
            } else {
                rstatus(a.status, SIFT_ERR_DEVICE_CHECK);
            }
            a.counts[static_cast<int64_t>(lh) * a.NQ + q] = min(n + 1, a.rowcap);
        }
    }
}

}  // namespace
}  // namespace sift

namespace sift {

sift_status decode_ragged_impl(const sift_problem *prob, int32_t num_query_tiles,
                               const uint64_t *la_words, const uint64_t *ca_words,
                               int32_t *qtiles, int32_t *kv, int32_t *counts, int32_t *sched,
                               int32_t *pages, int32_t page_cap, int32_t *dev_status,
                               cudaStream_t stream, bool exact) {
    sift_status st = validate_ragged(prob, false);
    if (st != SIFT_OK) return st;
    if (num_query_tiles < 1 || num_query_tiles > max_query_tiles(prob)) return SIFT_ERR_INVALID_ARG;
    if (qtiles == nullptr || kv == nullptr || counts == nullptr || sched == nullptr ||
        dev_status == nullptr)
        return SIFT_ERR_INVALID_ARG;
    if ((prob->la_words_len > 0 && la_words == nullptr) ||
        (prob->ca_words_len > 0 && ca_words == nullptr))
        return SIFT_ERR_INVALID_ARG;
    const bool gather = gathers_pages(prob);
    if (gather && prob->num_docs > 0 &&
        (pages == nullptr || page_cap < 1 ||
         static_cast<int64_t>(prob->num_kv_heads) * prob->num_docs * page_cap > INT32_MAX))
        return SIFT_ERR_INVALID_ARG;
    RaggedArgs a{};
    a.pages = pages;
    a.page_cap = gather ? page_cap : 0;
    a.gather = gather;
    a.cu = prob->cu_seqlens;
    a.doc_cu = prob->doc_cu;
    a.doc_end = prob->doc_end;
    a.la_off = prob->la_off;
    a.ca_off = prob->ca_off;
    a.la = la_words;
    a.ca = ca_words;
    a.la_len = prob->la_words_len;
    a.ca_len = prob->ca_words_len;
    a.qt = qtiles;
    a.kv = kv;
    a.counts = counts;
    a.status = dev_status;
    a.P = prob->num_prompts;
    a.D = prob->num_docs;
    a.Hkv = prob->num_kv_heads;
    a.L = prob->num_layers;
    a.B = prob->tile;
    a.page = prob->page ? prob->page : prob->tile;
    a.NQ = num_query_tiles;
    a.T = prob->total_tokens;
    a.rowcap = prob->max_tiles_per_prompt;
    const int pin = a.page < a.B ? a.page : a.B;
    a.full = (1u << (a.B / pin)) - 1u;
    a.exact = exact;
    ragged_tiles_kernel<<<1, 1024, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    const int64_t warps = static_cast<int64_t>(a.L) * a.Hkv * (a.D + a.P);
    const int64_t blocks = (warps + kRaggedWarps - 1) / kRaggedWarps;
    if (blocks > INT32_MAX) return SIFT_ERR_UNSUPPORTED;
    ragged_decode_kernel<<<static_cast<unsigned>(blocks), kRaggedWarps * 32, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    if (launch_schedule(counts, sched, a.L, a.NQ * a.Hkv, a.rowcap, dev_status, stream) !=
        cudaSuccess)
        return SIFT_ERR_CUDA;
    return SIFT_OK;
}

}  // namespace sift

extern "C" sift_status sift_decode_ragged(const sift_problem *prob, int32_t num_query_tiles,
                                          const uint64_t *la_words, const uint64_t *ca_words,
                                          int32_t *qtiles, int32_t *kv, int32_t *counts,
                                          int32_t *sched, int32_t *pages, int32_t page_cap,
                                          int32_t *dev_status, cudaStream_t stream) {
    sift::NvtxRange nvtx_range("sift_decode_ragged");
    return sift::decode_ragged_impl(prob, num_query_tiles, la_words, ca_words, qtiles, kv,
                                    counts, sched, pages, page_cap, dev_status, stream, true);
}

// sift_build.cu -- offline construction of the LA / CA bit vectors of one layer (SIFT
// pages, "Design del Sistema": offline, each retrieved document is prefilled densely
// on its own, the positions that draw high attention are found, and they are stored
// as LA bits -- tiles of the document's own attention matrix -- and CA bits -- KV
// pages that attract attention).  The pages do not give the selection rule; the one
// used here is stated beside sift_build_bits in include/sift.h.
//
// The attention mass comes from the tensor-core attention kernel itself: every document
// (and every query suffix) becomes a prompt of its own, listed densely by the
// general-layout decode, and V is replaced by one-hot indicators of the key's unit
// (min(page, tile) tokens from the document start), so output row t of query head qh
// is the probability mass that row puts on each unit of its document.  Small kernels
// then sum rows into per-(query tile, unit) masses, reduce units into tile masses and
// page scores in a fixed order, and pick the top-k tiles / pages into packed words.
#include <cuda_bf16.h>

#include "sift_internal.h"

namespace sift {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMassWarps = 8;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Geometry {  // sizes shared by the host plan and the kernels
    int B, page, unit;     // tile, CA page, mass unit = min(page, tile)
    int maxT, maxU, maxC;  // per document: tiles, units, pages (upper bounds)
};

Geometry geometry(const sift_problem *p, int max_doc_tiles) {
    Geometry g{};
    g.B = p->tile;
    g.page = p->page ? p->page : p->tile;
    g.unit = g.page < g.B ? g.page : g.B;
    g.maxT = max_doc_tiles;
    g.maxU = max_doc_tiles * (g.B / g.unit);
    g.maxC = static_cast<int>((static_cast<int64_t>(max_doc_tiles) * g.B + g.page - 1) / g.page);
    return g;
}

struct BuildLayout {  // byte offsets inside the workspace
    size_t seg_cu, seg_doc_cu, v1, o, lse, mu, mt, cs, qt, kv, counts, sched, attn_ws, total;
    int segments, nq_cap, rowcap;
};

BuildLayout build_layout(const sift_problem *p, const Geometry &g) {
    BuildLayout L{};
    const int S = p->num_docs + p->num_prompts;
    const size_t T = static_cast<size_t>(p->total_tokens);
    const size_t D = static_cast<size_t>(p->num_docs > 0 ? p->num_docs : 1);
    const size_t Hkv = static_cast<size_t>(p->num_kv_heads);
    L.segments = S;
    L.nq_cap = static_cast<int>((T + g.B - 1) / g.B) + S;
    L.rowcap = p->max_tiles_per_prompt;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    L.seg_cu = take(sizeof(int32_t) * (S + 1));
    L.seg_doc_cu = take(sizeof(int32_t) * (S + 1));
    L.v1 = take(2 * T * Hkv * p->head_dim);
    L.o = take(2 * T * p->num_q_heads * p->head_dim);
    L.lse = take(4 * T * p->num_q_heads);
    L.mu = take(4 * D * Hkv * g.maxT * g.maxU);
    L.mt = take(4 * D * Hkv * g.maxT * g.maxT);
    L.cs = take(4 * D * Hkv * g.maxC);
    L.qt = take(2 * sizeof(int32_t) * L.nq_cap);
    L.kv = take(2 * sizeof(int32_t) * Hkv * L.nq_cap * L.rowcap);
    L.counts = take(sizeof(int32_t) * Hkv * L.nq_cap);
    L.sched = take(sizeof(int32_t) * Hkv * L.nq_cap);
    L.attn_ws = take(kWsHeader + 2 * sizeof(int32_t) * Hkv * L.nq_cap);
    L.total = off;
    return L;
}

__device__ __forceinline__ void bstatus(int32_t *st, int code) { atomicCAS(st, 0, code); }

// segment boundaries: the documents of every prompt, then the prompt's suffix (maybe empty)
__global__ void segments_kernel(const int32_t *cu, const int32_t *doc_cu, const int32_t *doc_end,
                                int P, int D, int B, int max_doc_tiles, int32_t *seg_cu,
                                int32_t *seg_doc_cu, int32_t *status) {
    if (threadIdx.x != 0) return;
    int s = 0;
    seg_cu[0] = 0;
    for (int p = 0; p < P; ++p) {
        int pos = cu[p];
        const int g0 = doc_cu[p], g1 = doc_cu[p + 1];
        if (g0 < 0 || g1 < g0 || g1 > D) {
            bstatus(status, SIFT_ERR_DEVICE_CHECK);
            break;
        }
        for (int g = g0; g < g1; ++g) {
            const int e = doc_end[g];
            if (e < pos || e > cu[p + 1] || (e - pos + B - 1) / B > max_doc_tiles)
                bstatus(status, SIFT_ERR_DEVICE_CHECK);
            seg_cu[++s] = e;
            pos = e;
        }
        seg_cu[++s] = cu[p + 1];
    }
    for (int k = s + 1; k <= P + D; ++k) seg_cu[k] = seg_cu[s];  // only after a malformed prompt
    for (int k = 0; k <= P + D; ++k) seg_doc_cu[k] = 0;
}

// V[u][h][c] = 1 where c is the unit of token u inside its segment minus the window
// start; one thread per 8 columns (one 16-byte store), consecutive threads on
// consecutive bytes
__global__ void onehot_kernel(const int32_t *seg_cu, int S, int T, int Hkv, int d, int unit,
                              int window, uint4 *v) {
    const int chunks = d / 8;
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= static_cast<int64_t>(T) * Hkv * chunks) return;
    const int u = static_cast<int>(e / (static_cast<int64_t>(Hkv) * chunks));
    const int c0 = static_cast<int>(e % chunks) * 8;
    int lo = 0, hi = S - 1;  // segment of u: last s with seg_cu[s] <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(seg_cu + mid) <= u) lo = mid; else hi = mid - 1;
    }
    const int k = (u - __ldg(seg_cu + lo)) / unit - window * d - c0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (k >= 0 && k < 8) w[k >> 1] = (k & 1) ? 0x3f800000u : 0x00003f80u;  // bf16 1.0
    v[e] = make_uint4(w[0], w[1], w[2], w[3]);
}

struct DocGeom {
    int start, n;  // first token, tokens
};

// first token and length of document g (documents of a prompt are back to back)
__device__ __forceinline__ DocGeom doc_geom(const int32_t *cu, const int32_t *doc_cu,
                                            const int32_t *doc_end, int P, int g) {
    int lo = 0, hi = P - 1;  // prompt of g: last p with doc_cu[p] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(doc_cu + mid) <= g) lo = mid; else hi = mid - 1;
    }
    const int start = (g == __ldg(doc_cu + lo)) ? __ldg(cu + lo) : __ldg(doc_end + g - 1);
    return DocGeom{start, __ldg(doc_end + g) - start};
}

__device__ __forceinline__ bool doc_ok(const DocGeom &dg, const Geometry &G, int total_tokens) {
    return dg.start >= 0 && dg.n >= 0 && (dg.n + G.B - 1) / G.B <= G.maxT &&
           static_cast<int64_t>(dg.start) + dg.n <= total_tokens;
}

// Mu[g][h][i][u] for the units u of this window: sum over the group's query heads and the
// rows of query tile i (inside the document) of O[t][qh][u - window*d].  One 256-thread
// block per (document, kv head, query tile): warp w sums rows w, w+8, ... (lane = 4
// columns, one 8-byte load per row), then the 8 partial sums are added in warp order.
__global__ void __launch_bounds__(32 * kMassWarps)
mass_kernel(const __nv_bfloat16 *o, const int32_t *cu, const int32_t *doc_cu,
            const int32_t *doc_end, int P, Geometry G, int Hq, int Hkv, int d, int window,
            int total_tokens, float *mu) {
    __shared__ float part[kMassWarps][128];
    const int g = blockIdx.y;
    const int h = blockIdx.x / G.maxT, i = blockIdx.x % G.maxT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DocGeom dg = doc_geom(cu, doc_cu, doc_end, P, g);
    const int T = (dg.n + G.B - 1) / G.B;
    if (h >= Hkv || !doc_ok(dg, G, total_tokens) || i >= T)
        return;  // block-uniform; malformed documents are reported by the segments kernel
    const int rows = min(G.B, dg.n - i * G.B);
    const int GQ = Hq / Hkv;
    const int c = 4 * lane;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < d) {
        const int64_t t0 = static_cast<int64_t>(dg.start) + static_cast<int64_t>(i) * G.B;
#pragma unroll 4
        for (int rr = warp; rr < GQ * rows; rr += kMassWarps) {
            const int qh = h * GQ + rr / rows;
            const int64_t t = t0 + rr % rows;
            const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(o + (t * Hq + qh) * d + c));
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
            acc[0] += a.x;
            acc[1] += a.y;
            acc[2] += b.x;
            acc[3] += b.y;
        }
        for (int q = 0; q < 4; ++q) part[warp][c + q] = acc[q];
    }
    __syncthreads();
    const int nu = (dg.n + G.unit - 1) / G.unit;
    if (static_cast<int>(threadIdx.x) < d) {
        float sum = 0.f;
        for (int w = 0; w < kMassWarps; ++w) sum += part[w][threadIdx.x];
        const int u = window * d + static_cast<int>(threadIdx.x);
        if (u < nu)
            mu[((static_cast<int64_t>(g) * Hkv + h) * G.maxT + i) * G.maxU + u] = sum;
    }
}

// per (document, kv head): tile masses Mt[i][j] = sum of the units of tile j, and page
// scores Cs[c] = sum over query tiles i >= t(c) of the mass on page c's units, over
// (T - t(c)), t(c) being the tile of page c's first token -- both in a fixed order
__global__ void __launch_bounds__(256)
reduce_kernel(const float *mu, const int32_t *cu, const int32_t *doc_cu, const int32_t *doc_end,
              int P, Geometry G, int Hkv, int total_tokens, float *mt, float *cs) {
    const int g = blockIdx.y, h = blockIdx.x;
    const DocGeom dg = doc_geom(cu, doc_cu, doc_end, P, g);
    if (!doc_ok(dg, G, total_tokens)) return;
    const int T = (dg.n + G.B - 1) / G.B;
    const int nu = (dg.n + G.unit - 1) / G.unit;
    const int C = (dg.n + G.page - 1) / G.page;
    const int per_tile = G.B / G.unit;                        // units in a tile
    const int per_page = G.page >= G.B ? G.page / G.B : 1;    // units in a page
    const float *M = mu + (static_cast<int64_t>(g) * Hkv + h) * G.maxT * G.maxU;
    float *Mt = mt + (static_cast<int64_t>(g) * Hkv + h) * G.maxT * G.maxT;
    float *Cs = cs + (static_cast<int64_t>(g) * Hkv + h) * G.maxC;
    for (int e = threadIdx.x; e < T * T; e += blockDim.x) {
        const int i = e / T, j = e % T;
        float s = 0.f;
        for (int u = j * per_tile; u < min((j + 1) * per_tile, nu); ++u)
            s += M[static_cast<int64_t>(i) * G.maxU + u];
        Mt[static_cast<int64_t>(i) * G.maxT + j] = s;
    }
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        const int t = static_cast<int>(static_cast<int64_t>(c) * G.page / G.B);
        const int u0 = G.page >= G.B ? c * per_page : c;
        const int u1 = min(u0 + per_page, nu);
        float s = 0.f;
        for (int i = t; i < T; ++i)
            for (int u = u0; u < u1; ++u) s += M[static_cast<int64_t>(i) * G.maxU + u];
        Cs[c] = s / static_cast<float>(T - t);
    }
}

// ceil(fraction * candidates - 1e-4) in float32, each operation rounded on its own (no
// fused multiply-add), so that every host computing the same rule gets the same count
__device__ __forceinline__ int top_count(float fraction, int candidates) {
    return static_cast<int>(
        ceilf(__fsub_rn(__fmul_rn(fraction, static_cast<float>(candidates)), 1e-4f)));
}

// warp-collective: 64-bit word w of the top-k selection over vals[0 .. n) (rank =
// heavier candidates + equal ones at a lower index; kept iff rank < k)
__device__ __forceinline__ uint64_t top_word(const float *vals, int n, int k, int w,
                                             uint32_t lane) {
    uint64_t word = 0;
    for (int half = 0; half < 2; ++half) {
        const int j = 64 * w + 32 * half + static_cast<int>(lane);
        bool sel = false;
        if (j < n) {
            const float mj = vals[j];
            int rank = 0;
            for (int jp = 0; jp < n; ++jp) {
                const float m2 = vals[jp];
                rank += (m2 > mj) || (m2 == mj && jp < j);
            }
            sel = rank < k;
        }
        word |= static_cast<uint64_t>(__ballot_sync(0xffffffffu, sel)) << (32 * half);
    }
    return word;
}

// one warp per (document, kv head, row): LA row words; the warp of row maxT does the CA words
__global__ void select_kernel(const float *mt, const float *cs, const int32_t *cu,
                              const int32_t *doc_cu, const int32_t *doc_end,
                              const int64_t *la_off, const int64_t *ca_off, int P, Geometry G,
                              int Hkv, int layer, int total_tokens, float la_frac, float ca_frac,
                              int64_t la_len, int64_t ca_len, uint64_t *la, uint64_t *ca,
                              int32_t *status) {
    const int g = blockIdx.y;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const int h = wid / (G.maxT + 1), r = wid % (G.maxT + 1);
    if (h >= Hkv) return;
    const DocGeom dg = doc_geom(cu, doc_cu, doc_end, P, g);
    if (!doc_ok(dg, G, total_tokens) || dg.n < 1) return;  // reported by the segments kernel
    const int T = (dg.n + G.B - 1) / G.B;
    const int C = (dg.n + G.page - 1) / G.page;
    const int W = (T + 63) / 64, V = (C + 63) / 64;
    if (r < T) {
        // LA row r: the top_count(la_frac, r) tiles j < r of largest Mt[r][j]
        const float *row = mt + ((static_cast<int64_t>(g) * Hkv + h) * G.maxT + r) * G.maxT;
        const int64_t base =
            __ldg(la_off + g) + ((static_cast<int64_t>(layer) * Hkv + h) * T + r) * W;
        if (base < 0 || base + W > la_len) {
            if (lane == 0) bstatus(status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int k = top_count(la_frac, r);
        for (int w = 0; w < W; ++w) {
            const uint64_t word = top_word(row, r, k, w, lane);
            if (lane == 0) la[base + w] = word;
        }
    } else if (r == G.maxT) {
        // CA: the top_count(ca_frac, C) pages of largest score
        const float *score = cs + (static_cast<int64_t>(g) * Hkv + h) * G.maxC;
        const int64_t base = __ldg(ca_off + g) + (static_cast<int64_t>(layer) * Hkv + h) * V;
        if (base < 0 || base + V > ca_len) {
            if (lane == 0) bstatus(status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        const int k = top_count(ca_frac, C);
        for (int w = 0; w < V; ++w) {
            const uint64_t word = top_word(score, C, k, w, lane);
            if (lane == 0) ca[base + w] = word;
        }
    }
}

sift_status validate_any(const sift_problem *prob) {
    if (validate_problem(prob, true) == SIFT_OK) return SIFT_OK;
    return validate_ragged(prob, true);
}

}  // namespace
}  // namespace sift

extern "C" size_t sift_build_bits_workspace_bytes(const sift_problem *prob, int32_t max_doc_tiles) {
    if (sift::validate_any(prob) != SIFT_OK || max_doc_tiles < 1) return 0;
    return sift::build_layout(prob, sift::geometry(prob, max_doc_tiles)).total;
}

extern "C" sift_status sift_build_bits(const sift_problem *prob, int32_t layer, const void *q,
                                       const void *k, int32_t max_doc_tiles, float la_fraction,
                                       float ca_fraction, float softmax_scale,
                                       uint64_t *la_words, uint64_t *ca_words, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_build_bits");
    sift_status st = validate_any(prob);
    if (st != SIFT_OK) return st;
    if (layer < 0 || layer >= prob->num_layers || q == nullptr || k == nullptr ||
        workspace == nullptr || dev_status == nullptr || max_doc_tiles < 1 ||
        max_doc_tiles > prob->max_tiles_per_prompt || !(la_fraction >= 0.f) ||
        !(la_fraction <= 1.f) || !(ca_fraction >= 0.f) || !(ca_fraction <= 1.f))
        return SIFT_ERR_INVALID_ARG;
    if (prob->num_docs == 0) return SIFT_OK;
    if (la_words == nullptr || ca_words == nullptr || !aligned16(workspace))
        return SIFT_ERR_INVALID_ARG;
    const Geometry G = geometry(prob, max_doc_tiles);
    const BuildLayout bl = build_layout(prob, G);
    if (workspace_bytes < bl.total) return SIFT_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    auto at = [&](size_t off) { return ws + off; };
    int32_t *seg_cu = reinterpret_cast<int32_t *>(at(bl.seg_cu));
    int32_t *seg_doc_cu = reinterpret_cast<int32_t *>(at(bl.seg_doc_cu));
    __nv_bfloat16 *v1 = reinterpret_cast<__nv_bfloat16 *>(at(bl.v1));
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(at(bl.o));
    float *lse = reinterpret_cast<float *>(at(bl.lse));
    float *mu = reinterpret_cast<float *>(at(bl.mu));
    float *mt = reinterpret_cast<float *>(at(bl.mt));
    float *cs = reinterpret_cast<float *>(at(bl.cs));
    int32_t *qt = reinterpret_cast<int32_t *>(at(bl.qt));
    int32_t *kv = reinterpret_cast<int32_t *>(at(bl.kv));
    int32_t *counts = reinterpret_cast<int32_t *>(at(bl.counts));
    int32_t *sched = reinterpret_cast<int32_t *>(at(bl.sched));
    void *aws = at(bl.attn_ws);
    const size_t aws_bytes = bl.total - bl.attn_ws;
    const int T = prob->total_tokens, d = prob->head_dim;
    const int Hkv = prob->num_kv_heads, Hq = prob->num_q_heads, D = prob->num_docs;

    segments_kernel<<<1, 32, 0, stream>>>(prob->cu_seqlens, prob->doc_cu, prob->doc_end,
                                          prob->num_prompts, D, G.B, max_doc_tiles, seg_cu,
                                          seg_doc_cu, dev_status);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    // every document and suffix as a prompt of its own, no documents or bits, listed densely
    sift_problem seg = *prob;
    seg.num_prompts = bl.segments;
    seg.num_docs = 0;
    seg.num_layers = 1;
    seg.page = 0;
    seg.cu_seqlens = seg_cu;
    seg.doc_cu = seg_doc_cu;
    seg.doc_end = nullptr;
    seg.la_off = nullptr;
    seg.ca_off = nullptr;
    seg.la_words_len = 0;
    seg.ca_words_len = 0;
    st = decode_ragged_impl(&seg, bl.nq_cap, nullptr, nullptr, qt, kv, counts, sched, nullptr, 0,
                            dev_status, stream, false);
    if (st != SIFT_OK) return st;
    const int windows = (G.maxU + d - 1) / d;
    for (int w = 0; w < windows; ++w) {
        const int64_t n = static_cast<int64_t>(T) * Hkv * (d / 8);
        onehot_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
            seg_cu, bl.segments, T, Hkv, d, G.unit, w, reinterpret_cast<uint4 *>(v1));
        if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
        st = sift_sparse_prefill_ragged(&seg, bl.nq_cap, 0, q, k, v1, qt, kv, counts, sched,
                                        nullptr, 0, softmax_scale, o, lse, aws, aws_bytes,
                                        dev_status, stream);
        if (st != SIFT_OK) return st;
        dim3 grid(static_cast<unsigned>(Hkv * G.maxT), static_cast<unsigned>(D));
        mass_kernel<<<grid, 32 * kMassWarps, 0, stream>>>(o, prob->cu_seqlens, prob->doc_cu,
                                                          prob->doc_end, prob->num_prompts, G, Hq,
                                                          Hkv, d, w, T, mu);
        if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    }
    reduce_kernel<<<dim3(static_cast<unsigned>(Hkv), static_cast<unsigned>(D)), 256, 0, stream>>>(
        mu, prob->cu_seqlens, prob->doc_cu, prob->doc_end, prob->num_prompts, G, Hkv, T, mt, cs);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    const int warps = Hkv * (G.maxT + 1);
    dim3 grid(static_cast<unsigned>((warps + 7) / 8), static_cast<unsigned>(D));
    select_kernel<<<grid, 256, 0, stream>>>(mt, cs, prob->cu_seqlens, prob->doc_cu, prob->doc_end,
                                            prob->la_off, prob->ca_off, prob->num_prompts, G, Hkv,
                                            layer, T, la_fraction, ca_fraction,
                                            prob->la_words_len, prob->ca_words_len, la_words,
                                            ca_words, dev_status);
    return cudaGetLastError() == cudaSuccess ? SIFT_OK : SIFT_ERR_CUDA;
}

// sift_build.cu -- offline construction of the LA / CA bit vectors of one layer (SIFT
// pages, "Design del Sistema": offline, each retrieved document is prefilled densely
// on its own, the positions that draw high attention are found, and they are stored
// as LA bits -- tiles of the document's own attention matrix -- and CA bits -- KV
// pages that attract attention).  The pages do not give the selection rule; the one
// used here is stated beside sift_build_bits in include/sift.h.
//
// The per-tile attention mass comes from the dense tensor-core kernel itself: every
// document (and every query suffix) becomes a prompt of its own, and V is replaced by
// one-hot tile indicators, so output row t of query head qh is the probability mass
// that row puts on each key tile of its document.  Small kernels then sum rows into
// tile masses in a fixed order and pick the top-k tiles / pages into packed words.
#include <cuda_bf16.h>

#include "sift_internal.h"

namespace sift {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct BuildLayout {  // byte offsets inside the workspace
    size_t seg_cu, seg_doc_cu, v1, o, lse, mass, dense_ws, total;
    int segments;
};

BuildLayout build_layout(const sift_problem *p, int max_doc_tiles) {
    BuildLayout L{};
    const int S = p->num_docs + p->num_prompts;
    const size_t T = static_cast<size_t>(p->total_tokens);
    size_t off = 0;
    L.segments = S;
    L.seg_cu = off;
    off = align_up(off + sizeof(int32_t) * (S + 1));
    L.seg_doc_cu = off;
    off = align_up(off + sizeof(int32_t) * (S + 1));
    L.v1 = off;
    off = align_up(off + 2 * T * p->num_kv_heads * p->head_dim);
    L.o = off;
    off = align_up(off + 2 * T * p->num_q_heads * p->head_dim);
    L.lse = off;
    off = align_up(off + 4 * T * p->num_q_heads);
    L.mass = off;
    off = align_up(off + 4 * static_cast<size_t>(p->num_docs > 0 ? p->num_docs : 1) *
                             p->num_kv_heads * max_doc_tiles * max_doc_tiles);
    L.dense_ws = off;
    const size_t units = static_cast<size_t>(p->total_tokens / p->tile) * p->num_kv_heads;
    off = align_up(off + kWsHeader + 2 * units * sizeof(int32_t));
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
            if (e < pos || e > cu[p + 1] || (e - pos) % B || (e - pos) / B > max_doc_tiles)
                bstatus(status, SIFT_ERR_DEVICE_CHECK);
            seg_cu[++s] = e;
            pos = e;
        }
        seg_cu[++s] = cu[p + 1];
    }
    for (int k = s + 1; k <= P + D; ++k) seg_cu[k] = seg_cu[s];  // only after a malformed prompt
    for (int k = 0; k <= P + D; ++k) seg_doc_cu[k] = 0;
}

// V[u][h][c] = 1 where c is the tile of u inside its segment minus the window start; one
// thread per 8 columns (one 16-byte store), consecutive threads on consecutive bytes
__global__ void onehot_kernel(const int32_t *seg_cu, int S, int T, int Hkv, int d, int B,
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
    const int k = (u - __ldg(seg_cu + lo)) / B - window * d - c0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (k >= 0 && k < 8) w[k >> 1] = (k & 1) ? 0x3f800000u : 0x00003f80u;  // bf16 1.0
    v[e] = make_uint4(w[0], w[1], w[2], w[3]);
}

struct DocGeom {
    int start, tiles;
};

// start token and tile count of document g (documents of a prompt are back to back)
__device__ __forceinline__ DocGeom doc_geom(const int32_t *cu, const int32_t *doc_cu,
                                            const int32_t *doc_end, int P, int g, int B) {
    int lo = 0, hi = P - 1;  // prompt of g: last p with doc_cu[p] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(doc_cu + mid) <= g) lo = mid; else hi = mid - 1;
    }
    const int start = (g == __ldg(doc_cu + lo)) ? __ldg(cu + lo) : __ldg(doc_end + g - 1);
    return DocGeom{start, (__ldg(doc_end + g) - start) / B};
}

// M[g][h][i][j] for the key tiles j of this window: sum over the group's query heads and
// the rows of query tile i of O[t][qh][j - window*d].  One 256-thread block per (document,
// kv head, query tile): warp w sums rows w, w+8, ... (lane = 4 columns, one 8-byte load
// per row), then the 8 partial sums are added in warp order -- a fixed order.
constexpr int kMassWarps = 8;

__global__ void __launch_bounds__(32 * kMassWarps)
mass_kernel(const __nv_bfloat16 *o, const int32_t *cu, const int32_t *doc_cu,
            const int32_t *doc_end, int P, int B, int Hq, int Hkv, int d, int maxT, int window,
            int total_tokens, float *mass) {
    __shared__ float part[kMassWarps][128];
    const int g = blockIdx.y;
    const int h = blockIdx.x / maxT, i = blockIdx.x % maxT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DocGeom dg = doc_geom(cu, doc_cu, doc_end, P, g, B);
    if (h >= Hkv || i >= dg.tiles || dg.tiles > maxT || dg.start < 0 ||
        static_cast<int64_t>(dg.start) + static_cast<int64_t>(dg.tiles) * B > total_tokens)
        return;  // block-uniform; malformed documents are reported by the segments kernel
    const int G = Hq / Hkv;
    const int c = 4 * lane;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < d) {
        const int64_t t0 = static_cast<int64_t>(dg.start) + static_cast<int64_t>(i) * B;
#pragma unroll 4
        for (int rr = warp; rr < G * B; rr += kMassWarps) {
            const int qh = h * G + rr / B;
            const int64_t t = t0 + rr % B;
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
    if (threadIdx.x < d) {
        float sum = 0.f;
        for (int w = 0; w < kMassWarps; ++w) sum += part[w][threadIdx.x];
        const int j = window * d + static_cast<int>(threadIdx.x);
        if (j <= i && j < dg.tiles)
            mass[((static_cast<int64_t>(g) * Hkv + h) * maxT + i) * maxT + j] = sum;
    }
}

// ceil(fraction * candidates - 1e-4) in float32, each operation rounded on its own (no
// fused multiply-add), so that every host computing the same rule gets the same count
__device__ __forceinline__ int top_count(float fraction, int candidates) {
    return static_cast<int>(
        ceilf(__fsub_rn(__fmul_rn(fraction, static_cast<float>(candidates)), 1e-4f)));
}

// one warp per (document, kv head, row): LA row words; the warp of row maxT does the CA words
__global__ void select_kernel(const float *mass, const int32_t *cu, const int32_t *doc_cu,
                              const int32_t *doc_end, const int64_t *la_off, const int64_t *ca_off,
                              int P, int B, int Hkv, int layer, int maxT, float la_frac,
                              float ca_frac, int64_t la_len, int64_t ca_len, uint64_t *la,
                              uint64_t *ca, int32_t *status) {
    const int g = blockIdx.y;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t lane = threadIdx.x & 31u;
    const int h = wid / (maxT + 1), r = wid % (maxT + 1);
    if (h >= Hkv) return;
    const DocGeom dg = doc_geom(cu, doc_cu, doc_end, P, g, B);
    const int T = dg.tiles;
    if (T > maxT || T < 1) return;  // reported by the segments kernel
    const int W = (T + 63) / 64;
    const float *M = mass + (static_cast<int64_t>(g) * Hkv + h) * maxT * maxT;
    if (r < T) {
        // LA row r: the top_count(la_frac, r) tiles j < r of largest M[r][j]
        const int i = r;
        const int kk = top_count(la_frac, i);
        const int64_t base = __ldg(la_off + g) + ((static_cast<int64_t>(layer) * Hkv + h) * T + i) * W;
        if (base < 0 || base + W > la_len) {
            if (lane == 0) bstatus(status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        for (int w = 0; w < W; ++w) {
            uint64_t word = 0;
            for (int half = 0; half < 2; ++half) {
                const int j = 64 * w + 32 * half + static_cast<int>(lane);
                bool sel = false;
                if (j < i) {
                    const float mj = M[static_cast<int64_t>(i) * maxT + j];
                    int rank = 0;
                    for (int jp = 0; jp < i; ++jp) {
                        const float m2 = M[static_cast<int64_t>(i) * maxT + jp];
                        rank += (m2 > mj) || (m2 == mj && jp < j);
                    }
                    sel = rank < kk;
                }
                word |= static_cast<uint64_t>(__ballot_sync(0xffffffffu, sel)) << (32 * half);
            }
            if (lane == 0) la[base + w] = word;
        }
    } else if (r == maxT) {
        // CA: the top_count(ca_frac, T) pages of largest mean mass over the rows i >= j
        const int kk = top_count(ca_frac, T);
        const int64_t base = __ldg(ca_off + g) + (static_cast<int64_t>(layer) * Hkv + h) * W;
        if (base < 0 || base + W > ca_len) {
            if (lane == 0) bstatus(status, SIFT_ERR_DEVICE_CHECK);
            return;
        }
        auto col = [&](int j) {
            float s = 0.f;
            for (int i = j; i < T; ++i) s += M[static_cast<int64_t>(i) * maxT + j];
            return s / static_cast<float>(T - j);
        };
        for (int w = 0; w < W; ++w) {
            uint64_t word = 0;
            for (int half = 0; half < 2; ++half) {
                const int j = 64 * w + 32 * half + static_cast<int>(lane);
                bool sel = false;
                if (j < T) {
                    const float mj = col(j);
                    int rank = 0;
                    for (int jp = 0; jp < T; ++jp) {
                        const float m2 = col(jp);
                        rank += (m2 > mj) || (m2 == mj && jp < j);
                    }
                    sel = rank < kk;
                }
                word |= static_cast<uint64_t>(__ballot_sync(0xffffffffu, sel)) << (32 * half);
            }
            if (lane == 0) ca[base + w] = word;
        }
    }
}

}  // namespace
}  // namespace sift

extern "C" size_t sift_build_bits_workspace_bytes(const sift_problem *prob, int32_t max_doc_tiles) {
    if (sift::validate_problem(prob, true) != SIFT_OK || max_doc_tiles < 1) return 0;
    return sift::build_layout(prob, max_doc_tiles).total;
}

extern "C" sift_status sift_build_bits(const sift_problem *prob, int32_t layer, const void *q,
                                       const void *k, int32_t max_doc_tiles, float la_fraction,
                                       float ca_fraction, float softmax_scale,
                                       uint64_t *la_words, uint64_t *ca_words, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       cudaStream_t stream) {
    using namespace sift;
    sift_status st = validate_problem(prob, true);
    if (st != SIFT_OK) return st;
    if (layer < 0 || layer >= prob->num_layers || q == nullptr || k == nullptr ||
        workspace == nullptr || dev_status == nullptr || max_doc_tiles < 1 ||
        max_doc_tiles > prob->max_tiles_per_prompt || !(la_fraction >= 0.f) ||
        !(la_fraction <= 1.f) || !(ca_fraction >= 0.f) || !(ca_fraction <= 1.f))
        return SIFT_ERR_INVALID_ARG;
    if (prob->num_docs == 0) return SIFT_OK;
    if (la_words == nullptr || ca_words == nullptr || !aligned16(workspace))
        return SIFT_ERR_INVALID_ARG;
    const BuildLayout bl = build_layout(prob, max_doc_tiles);
    if (workspace_bytes < bl.total) return SIFT_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    int32_t *seg_cu = reinterpret_cast<int32_t *>(ws + bl.seg_cu);
    int32_t *seg_doc_cu = reinterpret_cast<int32_t *>(ws + bl.seg_doc_cu);
    __nv_bfloat16 *v1 = reinterpret_cast<__nv_bfloat16 *>(ws + bl.v1);
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(ws + bl.o);
    float *lse = reinterpret_cast<float *>(ws + bl.lse);
    float *mass = reinterpret_cast<float *>(ws + bl.mass);
    void *dws = ws + bl.dense_ws;
    const size_t dws_bytes = bl.total - bl.dense_ws;
    const int T = prob->total_tokens, d = prob->head_dim, B = prob->tile;
    const int Hkv = prob->num_kv_heads, Hq = prob->num_q_heads, D = prob->num_docs;

    segments_kernel<<<1, 32, 0, stream>>>(prob->cu_seqlens, prob->doc_cu, prob->doc_end,
                                          prob->num_prompts, D, B, max_doc_tiles, seg_cu,
                                          seg_doc_cu, dev_status);
    if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    // every document and suffix as a prompt of its own, no bits
    sift_problem seg = *prob;
    seg.num_prompts = bl.segments;
    seg.num_docs = 0;
    seg.cu_seqlens = seg_cu;
    seg.doc_cu = seg_doc_cu;
    seg.doc_end = nullptr;
    seg.la_off = nullptr;
    seg.ca_off = nullptr;
    seg.la_words_len = 0;
    seg.ca_words_len = 0;
    const int windows = (max_doc_tiles + d - 1) / d;
    for (int w = 0; w < windows; ++w) {
        const int64_t n = static_cast<int64_t>(T) * Hkv * (d / 8);
        onehot_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
            seg_cu, bl.segments, T, Hkv, d, B, w, reinterpret_cast<uint4 *>(v1));
        if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
        st = sift_dense_prefill(&seg, q, k, v1, softmax_scale, o, lse, dws, dws_bytes, dev_status,
                                stream);
        if (st != SIFT_OK) return st;
        dim3 grid(static_cast<unsigned>(Hkv * max_doc_tiles), static_cast<unsigned>(D));
        mass_kernel<<<grid, 32 * kMassWarps, 0, stream>>>(o, prob->cu_seqlens, prob->doc_cu, prob->doc_end,
                                              prob->num_prompts, B, Hq, Hkv, d, max_doc_tiles, w,
                                              T, mass);
        if (cudaGetLastError() != cudaSuccess) return SIFT_ERR_CUDA;
    }
    const int warps = Hkv * (max_doc_tiles + 1);
    dim3 grid(static_cast<unsigned>((warps + 7) / 8), static_cast<unsigned>(D));
    select_kernel<<<grid, 256, 0, stream>>>(mass, prob->cu_seqlens, prob->doc_cu, prob->doc_end,
                                            prob->la_off, prob->ca_off, prob->num_prompts, B, Hkv,
                                            layer, max_doc_tiles, la_fraction, ca_fraction,
                                            prob->la_words_len, prob->ca_words_len, la_words,
                                            ca_words, dev_status);
    return cudaGetLastError() == cudaSuccess ? SIFT_OK : SIFT_ERR_CUDA;
}

/*
 * sift.h -- C ABI of the SIFT online-prefill hot path on GB300 (sm_103a).
 *
 * SIFT (gist.science/it/paper/2606.09441, "Design del Sistema") keeps, for
 * every retrieved document, layer and head, two bit vectors: Local-Attention
 * (LA) bits flag tiles of the document's own causal self-attention matrix,
 * Cross-Attention (CA) bits flag KV pages (tile columns) of the document that
 * later documents of the same prompt attend to.  At prefill time a decoding
 * kernel turns the bits into explicit tile index lists ("Dettagli di
 * Implementazione", decoding kernel) and a sparse flash-attention kernel
 * computes only the flagged tiles and skips the rest ("Esecuzione Online";
 * "Dettagli di Implementazione", sparse attention kernel).  The full
 * recompute it is measured against ("Risultati") is dense causal attention.
 *
 * Readings where the pages are silent (all stated here, applied everywhere):
 *   - bits are kept per KV head (grouped-query attention shares one list per
 *     KV head among its query heads);
 *   - sift_decode / sift_sparse_prefill / sift_fused_prefill / sift_dense_prefill:
 *     tile size == KV page size == `tile` tokens and every prompt, document and
 *     suffix boundary is a multiple of `tile`;
 *   - sift_decode_ragged / sift_sparse_prefill_ragged: documents and suffixes
 *     of any length, each tiled from its own first token (the last tile
 *     partial), and CA pages of `page` tokens counted the same way;
 *   - diagonal tiles are always computed, causally inside the tile;
 *   - the user-query suffix after the last document attends densely to the
 *     whole prompt;
 *   - a CA bit of document g' page j admits that page to every row of every
 *     later document of the same prompt; LA bits at j >= i are ignored;
 *   - skipped tiles are excluded from the softmax (exactly -inf);
 *   - softmax_scale <= 0 means 1/sqrt(head_dim); LSE is a natural log.
 *
 * Conventions for every entry point:
 *   - all array pointers are DEVICE pointers owned by the caller; the library
 *     allocates no memory and keeps no state between calls (except the fixed
 *     scratch array of sift_dense_prefill_noalloc, described there);
 *   - work is enqueued on `stream` and returns without synchronising;
 *   - arguments are validated on the host before anything is launched
 *     (SIFT_ERR_INVALID_ARG / SIFT_ERR_UNSUPPORTED, nothing enqueued);
 *   - a failed launch returns SIFT_ERR_CUDA;
 *   - problems only visible on the device (inconsistent offsets, an index
 *     outside its row, a bounded wait that ran out) are written to
 *     `*dev_status` (device int32, first error wins, never cleared by the
 *     library: the caller zeroes it and reads it after synchronising).
 *     Kernels never trap: on such an error they finish or return early, and
 *     the affected outputs are unspecified.
 */
#ifndef SIFT_H
#define SIFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;

typedef enum {
    SIFT_OK = 0,
    SIFT_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, inconsistent sizes          */
    SIFT_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim, tile, odd GQA)  */
    SIFT_ERR_CUDA = 3,          /* a CUDA call or launch failed                          */
    SIFT_ERR_TIMEOUT = 4,       /* device: a bounded wait ran out (written to dev_status) */
    SIFT_ERR_DEVICE_CHECK = 5   /* device: inconsistent offsets or indices (dev_status)  */
} sift_status;

/*
 * One packed varlen batch of prompts.  Prompt p covers tokens
 * [cu_seqlens[p], cu_seqlens[p+1]); it holds documents doc_cu[p] ..
 * doc_cu[p+1]-1, laid out back to back from the prompt start (document g ends
 * at token doc_end[g], exclusive), followed by the user-query suffix up to
 * the prompt end (possibly empty).  In the aligned entry points tiles are
 * numbered globally: tile i covers tokens [i*tile, (i+1)*tile);
 * N = total_tokens / tile.
 *
 * Bit words (uint64, bit j of a row is bit j%64 of word j/64, LSB first), for
 * a document of n_g tokens with T_g = ceil(n_g/tile) tiles and
 * C_g = ceil(n_g/page) pages, both counted from its first token:
 *   LA of document g (W_g = ceil(T_g/64)) for (layer l, kv head h):
 *     T_g rows of W_g words at la_words[la_off[g] + (l*Hkv + h)*T_g*W_g + row*W_g];
 *   CA of document g for (l, h) (V_g = ceil(C_g/64)): V_g words at
 *     ca_words[ca_off[g] + (l*Hkv + h)*V_g].
 * On an aligned layout with page == tile, T_g = C_g = n_g/tile and V_g = W_g.
 */
typedef struct {
    int32_t num_prompts;           /* P >= 1                                            */
    int32_t num_docs;              /* D >= 0, all prompts together                      */
    int32_t num_layers;            /* layers covered by the bit words and by sift_decode */
    int32_t num_q_heads;           /* Hq                                                */
    int32_t num_kv_heads;          /* Hkv; Hq/Hkv must be even (query heads go in pairs) */
    int32_t head_dim;              /* d: 64 or 128                                      */
    int32_t tile;                  /* LA tile / attention tile in tokens: 64 or 128     */
    int32_t total_tokens;          /* cu_seqlens[P]                                     */
    int32_t max_tiles_per_prompt;  /* rowcap: capacity of one list row, >= the key tiles of
                                      the longest prompt (ragged: the sum over its segments
                                      of ceil(length/tile), plus its number of documents
                                      when CA pages are gathered)                       */
    int32_t page;                  /* CA page size in tokens; 0 = tile.  The aligned entry
                                      points need 0 or tile; the ragged ones a power of two
                                      that nests with tile, at most 16 pages per tile   */
    const int32_t *cu_seqlens;     /* device [P+1]                                      */
    const int32_t *doc_cu;         /* device [P+1]                                      */
    const int32_t *doc_end;        /* device [D] (may be NULL when D == 0)              */
    const int64_t *la_off;         /* device [D]                                        */
    const int64_t *ca_off;         /* device [D]                                        */
    int64_t la_words_len;          /* number of uint64 words behind la_words            */
    int64_t ca_words_len;          /* number of uint64 words behind ca_words            */
} sift_problem;

/*
 * Bytes of caller-provided scratch that sift_sparse_prefill and
 * sift_dense_prefill need for `prob` (a work counter for the persistent
 * scheduler, plus the dense schedule).  Returns 0 if prob is invalid.
 */
size_t sift_workspace_bytes(const sift_problem *prob);

/*
 * Decode the LA/CA bits of every (layer, kv head, query tile) row into its
 * list of key tiles to compute, and order each layer's rows longest first
 * for the persistent attention scheduler.
 * (SIFT pages, "Dettagli di Implementazione": decoding kernel.)
 *
 *   kv_idx  int32 [num_layers][Hkv][N][max_tiles_per_prompt]: row (l,h,i)
 *           lists counts[l][h][i] global tile indices, strictly ascending:
 *           CA-flagged pages of the earlier documents of i's prompt, then
 *           the LA-flagged tiles of i's own document, then i itself; a
 *           suffix row lists every tile of its prompt up to i.  Entries past
 *           the count are not written.
 *   counts  int32 [num_layers][Hkv][N]
 *   sched   int32 [num_layers][Hkv*N]: a permutation of the units
 *           u = h*N + i of each layer with non-increasing counts.
 * Bit-exact for kv_idx and counts.  One kernel launch, in which one block per
 * layer counts that layer's rows from the bits and sorts them while the other
 * blocks write the lists; two launches (the same kernel, schedule blocks
 * first) when the schedule blocks' shared memory exceeds 32 KB: (rowcap + 1 +
 * Hkv*D + 2*D + N) x 4 bytes, plus Hkv*N x 4 for the counts when the total
 * stays within 226 KB (rowcap = max_tiles_per_prompt, D documents).
 * SIFT_ERR_UNSUPPORTED when the first part alone exceeds 226 KB.
 */
sift_status sift_decode(const sift_problem *prob, const uint64_t *la_words,
                        const uint64_t *ca_words, int32_t *kv_idx, int32_t *counts,
                        int32_t *sched, int32_t *dev_status, cudaStream_t stream);

/*
 * Block-sparse causal grouped-query flash attention of one layer over the
 * decoded lists: each query tile of query head qh attends to the key tiles of
 * row (layer, qh / (Hq/Hkv), i) only, the diagonal tile causally.
 * (SIFT pages, "Dettagli di Implementazione": sparse attention kernel.)
 *
 *   q       bf16 [total_tokens][Hq][d]   (16-byte aligned, contiguous)
 *   k, v    bf16 [total_tokens][Hkv][d]
 *   kv_idx, counts, sched: sift_decode's outputs (all layers; `layer` picks the slice)
 *   o       bf16 [total_tokens][Hq][d]   output, O = softmax(scale*QK^T) V over the list
 *   lse     fp32 [Hq][total_tokens]      output, natural-log sum of exp(scale*qk)
 *   workspace  >= sift_workspace_bytes(prob) bytes of device scratch; clobbered;
 *              calls that share a workspace must not overlap on the GPU.
 * One memset and one kernel launch.
 */
sift_status sift_sparse_prefill(const sift_problem *prob, int32_t layer, const void *q,
                                const void *k, const void *v, const int32_t *kv_idx,
                                const int32_t *counts, const int32_t *sched, float softmax_scale,
                                void *o, float *lse, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, cudaStream_t stream);

/*
 * Decode fused into the prefill (SIFT pages, "Dettagli di Implementazione": the
 * bits become tile indices, the sparse kernel iterates over them): one launch
 * that walks the LA/CA words of each row on the fly and turns every set bit into
 * a tile load, with no kv_idx list in memory and no separate decode.  Same
 * result as sift_decode followed by sift_sparse_prefill (the same MMAs on the
 * same tiles in the same order); rows are taken longest-first by their position
 * in the prompt instead of by a decoded count.
 *   la_words, ca_words: the bit words of sift_decode (all layers); `layer` picks one
 *   q, k, v, o, lse, workspace, dev_status: as for sift_sparse_prefill
 * At most 64 prompts per batch (SIFT_ERR_UNSUPPORTED beyond).  One memset and one
 * kernel launch.
 */
sift_status sift_fused_prefill(const sift_problem *prob, int32_t layer, const uint64_t *la_words,
                               const uint64_t *ca_words, const void *q, const void *k,
                               const void *v, float softmax_scale, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               cudaStream_t stream);

/*
 * Dense causal grouped-query flash attention over each whole prompt: the full
 * recompute baseline of the SIFT pages ("Risultati").  Same kernel as
 * sift_sparse_prefill with the implicit list {prompt start .. i}; the bit
 * words, kv_idx and layer are not used.  Same layouts as above.
 * One memset and three kernel launches (row lengths, schedule, attention).
 */
sift_status sift_dense_prefill(const sift_problem *prob, const void *q, const void *k,
                               const void *v, float softmax_scale, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               cudaStream_t stream);

/*
 * sift_dense_prefill for callers that cannot allocate device memory at call
 * time (the SIFT pages have no counterpart; this is a deployment aid).  A
 * serving runtime that plans all of its buffers at start-up, code that must
 * not risk the implicit device synchronisation of cudaMalloc/cudaFree, or a
 * host thread without an allocator can call this instead: it takes no
 * workspace and uses a scratch array that the library keeps in device memory.
 *   - Same arguments, layouts and results as sift_dense_prefill, minus the
 *     workspace.
 *   - The scratch is a fixed 1 MiB array per GPU, held from the moment the
 *     library is loaded on that GPU until the process exits.  A problem whose
 *     sift_workspace_bytes() exceeds 1 MiB (about 131,000 kv-head x query-tile
 *     units) is rejected with SIFT_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the array's device address, with
 *     that device current; make that first call outside any stream capture.
 *     The address is kept with the id of the context it was taken in.  A
 *     call from another context of the device (after cudaDeviceReset
 *     replaced the primary context, for instance) looks it up again, so the
 *     first call after such a reset must also be made outside stream capture.
 *   - Every call shares the one array and it keeps the last call's contents:
 *     calls whose work may overlap on the GPU (different streams, or several
 *     host threads) race on it and must be serialised by the caller.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
sift_status sift_dense_prefill_noalloc(const sift_problem *prob, const void *q, const void *k,
                                       const void *v, float softmax_scale, void *o, float *lse,
                                       int32_t *dev_status, cudaStream_t stream);

/*
 * Offline construction of one layer's LA and CA bit vectors (SIFT pages,
 * "Design del Sistema": each document is prefilled densely on its own once,
 * the tiles and pages that draw high attention are found and stored as bits).
 * Works on both layouts: aligned, and documents of any length with CA pages
 * of their own size (tiles and pages counted from each document's first
 * token, the last ones partial).  The pages name no selection rule; this
 * library's rule, per document, kv head h, T tiles and C pages:
 *   - masses are gathered per unit of min(page, tile) tokens from a causal
 *     prefill of the document alone: the attention probability that the rows
 *     of query tile i, over the query heads of h's group, put on each unit;
 *   - tile mass M[i][j] = the mass of tile j's units;
 *   - LA row i: the top ceil(la_fraction * i - 1e-4) tiles j < i by M[i][j]
 *     (the diagonal is implicit and never written; bits at j >= i are zero);
 *   - CA: the top ceil(ca_fraction * C - 1e-4) pages by score(c) = sum over
 *     query tiles i >= t(c) of the mass on page c, over (T - t(c)), where t(c)
 *     is the tile of page c's first token (page == tile: the mean mass that
 *     tile j receives from the rows i >= j);
 *   - counts in float32 with each operation rounded on its own; ties go to
 *     the lower index; masses come from the bf16 attention kernel, so tiles of
 *     nearly equal mass may swap against an exact computation.
 *   prob:           the attention problem (device arrays as for sift_decode);
 *                   its la_off, ca_off, la_words_len, ca_words_len say where
 *                   the words go; the documents' queries and keys are the
 *                   prompt's own rows in q and k
 *   layer:          which layer's words to write (q and k are that layer's)
 *   q, k:           bf16 [total_tokens][heads][head_dim], as for the prefill
 *   max_doc_tiles:  upper bound on any document's tiles, ceil(length/tile)
 *                   (1 .. max_tiles_per_prompt); sizes the workspace
 *   la_fraction, ca_fraction: in [0, 1]
 *   softmax_scale:  0 selects 1/sqrt(head_dim)
 *   la_words, ca_words: device, written only at this layer's blocks
 *   workspace:      device, >= sift_build_bits_workspace_bytes(), 16-byte aligned
 * A document longer than max_doc_tiles, or offsets outside the word arrays,
 * set SIFT_ERR_DEVICE_CHECK in dev_status; those words are not written.  A
 * batch without documents returns SIFT_OK and enqueues nothing.
 * Launches: 4 + ceil(units of the longest document / head_dim) x 3 + 2.
 */
size_t sift_build_bits_workspace_bytes(const sift_problem *prob, int32_t max_doc_tiles);
sift_status sift_build_bits(const sift_problem *prob, int32_t layer, const void *q, const void *k,
                            int32_t max_doc_tiles, float la_fraction, float ca_fraction,
                            float softmax_scale, uint64_t *la_words, uint64_t *ca_words,
                            void *workspace, size_t workspace_bytes, int32_t *dev_status,
                            cudaStream_t stream);

/*
 * Decode on a general layout: documents and suffixes of any length, CA pages
 * of their own size.  (SIFT pages, "Dettagli di Implementazione": decoding
 * kernel; the pages give no tile or page size.)
 *
 * Segments are the documents and the query suffixes; each is cut into query
 * tiles of `tile` tokens from its own first token, the last one partial, and
 * the tiles of all segments are numbered q = 0 .. num_query_tiles-1 in token
 * order.  num_query_tiles must equal the sum over segments of
 * ceil(length/tile) (the host knows the lengths; a mismatch found on the
 * device is SIFT_ERR_DEVICE_CHECK).
 *   qtiles  int32 [num_query_tiles][2]: (first token, rows) of each query tile
 *   kv      int32 [num_layers][Hkv][num_query_tiles][max_tiles_per_prompt][2]:
 *           row (l, h, q) holds counts[l][h][q] pairs (first token, info) of
 *           key tiles, by ascending first token: every tile of each earlier
 *           document of the prompt holding a CA-flagged page, then the
 *           LA-flagged tiles below the row inside its own document, then the
 *           row's own tile; a suffix row lists every tile of its prompt's
 *           documents, its earlier suffix tiles, then its own tile.
 *           info = len | causal << 8 | gather << 9 | mask << 16, with
 *           Pin = min(page, tile):
 *             len    keys of the tile inside its segment (1 .. tile);
 *             causal 1 on the row's own tile only;
 *             mask   bit k covers keys [k*Pin, (k+1)*Pin) of the tile: the
 *                    flagged pages of a CA tile, every bit otherwise.
 *           Key (first + c) is visible to query row r iff c < len, mask bit
 *           c/Pin is set and, when causal, c <= r.  Entries past the count
 *           are not written.
 *           Gathered pages (page < tile and page a multiple of 8): a document
 *           row's CA part lists instead the whole flagged pages of the
 *           earlier documents, tile/page at a time (gather = 1, len = pages x
 *           page, first = index of the group's first page in the layer's
 *           slice of `pages`; key c is token pages[first + c/page] + c%page),
 *           then each earlier document's partial last page when flagged.
 *   counts  int32 [num_layers][Hkv][num_query_tiles]
 *   sched   int32 [num_layers][Hkv*num_query_tiles]: per layer, a permutation
 *           of the units u = h*num_query_tiles + q with non-increasing counts.
 *   pages   int32 [num_layers][Hkv][num_docs][page_cap]: for the rows of
 *           document g, the first tokens of the gathered pages, ascending.
 *           Needed (non-NULL, page_cap >= the flagged whole pages before any
 *           document; tile/page x max_tiles_per_prompt always suffices) only
 *           when pages are gathered; NULL and 0 otherwise.
 * Bit-exact for qtiles, kv, counts and the pages used.  Three kernel launches.
 */
sift_status sift_decode_ragged(const sift_problem *prob, int32_t num_query_tiles,
                               const uint64_t *la_words, const uint64_t *ca_words,
                               int32_t *qtiles, int32_t *kv, int32_t *counts, int32_t *sched,
                               int32_t *pages, int32_t page_cap, int32_t *dev_status,
                               cudaStream_t stream);

/*
 * Block-sparse causal grouped-query flash attention of one layer on a general
 * layout, over sift_decode_ragged's lists: query tile q of query head qh
 * attends to the visible keys of the entries of row
 * (layer, qh / (Hq/Hkv), q).  Same q, k, v, o, lse layouts and workspace as
 * sift_sparse_prefill (total_tokens need not be a multiple of tile); only the
 * rows of each query tile inside its segment are written.  Gathered pages
 * are loaded by TMA page rows at a time side by side into one key tile.
 * qtiles, kv, counts, sched, pages, page_cap: as from sift_decode_ragged.
 * With 128-token tiles every entry sift_decode_ragged writes leaves its visible
 * keys a prefix of each row (kept pages with holes between them arise only from
 * 4-token pages under 64-token tiles); an entry whose mask leaves holes is read
 * there as its first len keys and reported as SIFT_ERR_DEVICE_CHECK.
 * One memset and one kernel launch.
 */
sift_status sift_sparse_prefill_ragged(const sift_problem *prob, int32_t num_query_tiles,
                                       int32_t layer, const void *q, const void *k,
                                       const void *v, const int32_t *qtiles, const int32_t *kv,
                                       const int32_t *counts, const int32_t *sched,
                                       const int32_t *pages, int32_t page_cap,
                                       float softmax_scale, void *o, float *lse,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char *sift_status_string(sift_status status);

/*
 * Test hook for the bounded waits (no counterpart on the pages).  Applies to
 * launches made after the call, process-wide:
 *   wait_timeout_ns  limit of every device-side wait (0 restores the default,
 *                    2 s);
 *   stall_flag       nonzero: the attention kernel's MMA issuer first waits
 *                    on a barrier that nothing ever signals, so the wait runs
 *                    out, the kernel unwinds and reports SIFT_ERR_TIMEOUT.
 */
void sift_debug_set_waits(uint64_t wait_timeout_ns, int32_t stall_flag);

/* ABI version of this header (major*100 + minor). */
int32_t sift_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SIFT_H */

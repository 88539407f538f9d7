/*
 * sift_oracle.c -- plain CPU oracle for SIFT's online prefill hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it is built and used by tests/, by the smoke check and by
 * bench.py's CPU-baseline leg, and it shares no code, header or table with
 * the CUDA library.
 *
 * What it restates (SIFT pages, gist.science/it/paper/2606.09441 and
 * gist.science/zh/paper/2606.09441):
 *   - "Design del Sistema" / "Esecuzione Online": at prefill time a sparse
 *     attention kernel reads the per-(document, layer, head) LA and CA bit
 *     vectors, computes attention scores only for the flagged tiles/pages and
 *     skips the rest.  A skipped key is simply absent from the softmax.
 *   - "Vettore di Bit Local-Attention (LA)": flags high-score tiles of a
 *     document's own self-attention matrix.
 *   - "Vettore di Bit Cross-Attention (CA)": flags KV pages (tile columns) of
 *     a document that attract attention from the other documents placed
 *     after it in the prompt.
 *   - "Dettagli di Implementazione", decoding kernel: the bit vectors become
 *     explicit tile index lists.
 * Readings where the pages are silent (bit order, diagonal tiles, the query
 * suffix, softmax scale) are the ones stated beside each function.
 *
 * Precision: bf16 inputs are widened exactly to double and every sum,
 * exponential and division is done in double, one row at a time, keys in
 * ascending order.  Rows are independent, so OpenMP over rows changes no
 * result.
 *
 * Documents of any length and a CA page size that differs from the tile
 * (the pages fix neither) follow one reading: tiles and pages are counted
 * from each document's first token, the last ones partial (key_visible and
 * sift_oracle_decode_ragged below).
 *
 * Parity pins (checked by the "not gpu" tests): hand-derived decode fixtures
 * (aligned and ragged), popcount identities, all-ones bits == dense causal
 * attention (library SDPA), per-document / block-diagonal / cross-document
 * special cases against SDPA with a mask built from their plain description,
 * closed forms (first token, constant V), single planted CA bits against their
 * page's token range, and dense-mask numpy brute forces on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int num_prompts, num_docs, num_kv_heads, tile;
    int page;                  /* CA page size in tokens (equal to tile unless stated) */
    const int32_t *cu_seqlens; /* [P+1] token offsets of each prompt          */
    const int32_t *doc_cu;     /* [P+1] prompt p owns docs doc_cu[p]..[p+1]-1 */
    const int32_t *doc_end;    /* [D] absolute end token (exclusive)          */
    const int64_t *la_off;     /* [D] word offset of doc g's LA blocks        */
    const int64_t *ca_off;     /* [D] word offset of doc g's CA blocks        */
    const uint64_t *la_words, *ca_words;
} sift_bits_view;

/* prompt holding token t (linear scan; plain on purpose) */
static int prompt_of(const sift_bits_view *s, int64_t t) {
    for (int p = 0; p < s->num_prompts; ++p)
        if (t >= s->cu_seqlens[p] && t < s->cu_seqlens[p + 1]) return p;
    return -1;
}

/* first token of document g (documents of a prompt are contiguous from its start) */
static int64_t doc_begin(const sift_bits_view *s, int p, int g) {
    return g == s->doc_cu[p] ? s->cu_seqlens[p] : s->doc_end[g - 1];
}

/* document of prompt p holding token t, or -1 when t lies in the query suffix */
static int doc_of(const sift_bits_view *s, int p, int64_t t) {
    for (int g = s->doc_cu[p]; g < s->doc_cu[p + 1]; ++g)
        if (t >= doc_begin(s, p, g) && t < s->doc_end[g]) return g;
    return -1;
}

/* LA tiles of document g, counted from its first token; the last may be partial */
static int doc_tiles(const sift_bits_view *s, int p, int g) {
    int64_t n = s->doc_end[g] - doc_begin(s, p, g);
    return (int)((n + s->tile - 1) / s->tile);
}

/* CA pages of document g, counted from its first token; the last may be partial */
static int doc_pages(const sift_bits_view *s, int p, int g) {
    int64_t n = s->doc_end[g] - doc_begin(s, p, g);
    return (int)((n + s->page - 1) / s->page);
}

/* LA bit (row i, column j) of document g for (layer, kv head h).
 * Reading of the (unstated) layout: square row-major, ceil(T/64) words per row,
 * bit j at word j/64, bit position j%64 counted from the least significant bit. */
static int la_bit(const sift_bits_view *s, int p, int g, int layer, int h, int i, int j) {
    int T = doc_tiles(s, p, g);
    int W = (T + 63) / 64;
    int64_t base = s->la_off[g] + ((int64_t)layer * s->num_kv_heads + h) * T * W;
    uint64_t word = s->la_words[base + (int64_t)i * W + j / 64];
    return (int)((word >> (j % 64)) & 1u);
}

/* CA bit of page j of document g for (layer, kv head h); same bit order as LA,
 * ceil(C/64) words for the document's C pages. */
static int ca_bit(const sift_bits_view *s, int p, int g, int layer, int h, int j) {
    int C = doc_pages(s, p, g);
    int W = (C + 63) / 64;
    int64_t base = s->ca_off[g] + ((int64_t)layer * s->num_kv_heads + h) * W;
    uint64_t word = s->ca_words[base + j / 64];
    return (int)((word >> (j % 64)) & 1u);
}

/*
 * Is key token u part of query token t's softmax at (layer, kv head h)?
 *   - keys come from t's own prompt and are causal (u <= t);
 *   - a query in the user suffix attends to every earlier key of the prompt
 *     (no metadata exists for the fresh query);
 *   - tiles and pages are counted from the first token of their document:
 *     token x of document g lies in tile (x - start_g) / tile and in page
 *     (x - start_g) / page;
 *   - the diagonal tile (key tile == query tile of the same document) is
 *     always computed;
 *   - a key in t's own document g: its tile column j is kept iff LA[g][i][j];
 *   - a key in an earlier document g' of the prompt: its page is kept iff
 *     CA[g'][page];
 *   - everything else is skipped.
 * With every boundary a multiple of the tile and page == tile, document tiles
 * coincide with the global tiles token / tile.
 */
static int key_visible(const sift_bits_view *s, int layer, int h, int64_t t, int64_t u) {
    int p = prompt_of(s, t);
    if (p < 0 || u < s->cu_seqlens[p] || u > t) return 0;
    int g = doc_of(s, p, t);
    if (g < 0) return 1;
    int64_t B = s->tile;
    int gu = doc_of(s, p, u);
    if (gu == g) {
        int64_t d0 = doc_begin(s, p, g);
        if ((t - d0) / B == (u - d0) / B) return 1;
        return la_bit(s, p, g, layer, h, (int)((t - d0) / B), (int)((u - d0) / B));
    }
    int64_t d0u = doc_begin(s, p, gu);
    return ca_bit(s, p, gu, layer, h, (int)((u - d0u) / s->page));
}

/*
 * Decode every (layer, kv head, query tile) row into its tile index list.
 * Query tiles and key tiles are numbered globally (tile index = token / B).
 * List order (the pages give none): ascending tile index -- CA-flagged pages
 * of the earlier documents in document order, then the LA-flagged tiles of
 * the row's own document, then the diagonal tile.  Suffix rows list every
 * tile of the prompt up to and including the diagonal.
 * Output: kv_idx[((l*Hkv + h)*N + i)*rowcap + k] for k < counts[(l*Hkv+h)*N + i].
 * Returns 0, or -1 if a row would exceed rowcap.
 */
int sift_oracle_decode(int num_prompts, int num_docs, int num_layers, int num_kv_heads, int tile,
                       const int32_t *cu_seqlens, const int32_t *doc_cu, const int32_t *doc_end,
                       const int64_t *la_off, const int64_t *ca_off,
                       const uint64_t *la_words, const uint64_t *ca_words,
                       int rowcap, int32_t *kv_idx, int32_t *counts) {
    sift_bits_view s = {num_prompts, num_docs, num_kv_heads, tile, tile, cu_seqlens, doc_cu,
                        doc_end, la_off, ca_off, la_words, ca_words};
    int64_t N = cu_seqlens[num_prompts] / tile;
    int bad = 0;
    for (int l = 0; l < num_layers; ++l)
        for (int h = 0; h < num_kv_heads; ++h)
            for (int64_t i = 0; i < N; ++i) {
                int64_t row = ((int64_t)l * num_kv_heads + h) * N + i;
                int32_t *out = kv_idx + row * rowcap;
                int n = 0;
                int p = prompt_of(&s, i * tile);
                int g = doc_of(&s, p, i * tile);
#define EMIT(x) do { if (n < rowcap) out[n] = (int32_t)(x); else bad = 1; ++n; } while (0)
                if (g < 0) {
                    for (int64_t j = cu_seqlens[p] / tile; j <= i; ++j) EMIT(j);
                } else {
                    for (int gp = doc_cu[p]; gp < g; ++gp) {
                        int64_t t0 = doc_begin(&s, p, gp) / tile;
                        int T = doc_tiles(&s, p, gp);
                        for (int j = 0; j < T; ++j)
                            if (ca_bit(&s, p, gp, l, h, j)) EMIT(t0 + j);
                    }
                    int64_t t0 = doc_begin(&s, p, g) / tile;
                    int il = (int)(i - t0);
                    for (int j = 0; j < il; ++j)
                        if (la_bit(&s, p, g, l, h, il, j)) EMIT(t0 + j);
                    EMIT(i);
                }
#undef EMIT
                counts[row] = n;
            }
    return bad ? -1 : 0;
}

/*
 * Decode for documents of any length and a CA page size of its own.
 *
 * Query tiles: every segment -- a document, or a prompt's query suffix -- is
 * cut into tiles of `tile` tokens from its own first token, the last one
 * possibly partial.  Tiles are numbered q = 0, 1, ... in token order and
 * qtiles[2q], qtiles[2q+1] = (first token, rows).  Key tiles are cut the
 * same way.
 *
 * Row (l, h, q) lists key tiles as pairs (first token, info), by ascending
 * first token:
 *   - a document row: every tile of each earlier document of the prompt
 *     that holds a CA-flagged page, then the LA-flagged tiles j < i of the
 *     row's own document, then the diagonal tile;
 *   - a suffix row: every tile of every document of the prompt, the suffix's
 *     own tiles before the diagonal, then the diagonal.
 * info = len | causal << 8 | gather << 9 | mask << 16, with Pin = min(page, tile):
 *   len     keys of the tile inside its segment (1 .. tile);
 *   causal  1 on the diagonal only;
 *   mask    bit k covers keys [k*Pin, (k+1)*Pin) of the tile; all tile/Pin
 *           bits for every tile but a CA one, whose bit k is the CA bit of
 *           the page holding key k*Pin (0 when k*Pin >= len).
 * Key (first + c) of an entry is visible to row r of the query tile iff
 * c < len, mask bit c / Pin is set, and c <= r when causal -- the same key
 * set as key_visible().
 *
 * Gathered pages (page < tile and page a multiple of 8): a document row's
 * CA part is instead made of pages, not tiles.  The whole flagged pages of
 * the earlier documents (page j of a document with (j+1)*page <= its length),
 * in ascending order, are written to pages[((l*Hkv + h)*D + g)*page_cap + k]
 * (first token of the k-th) for the row's document g, and listed tile/page at
 * a time: entry (first = (h*D + g)*page_cap + k0, info = n*page | 1 << 9 |
 * all mask bits) stands for the n <= tile/page pages k0 .. k0+n-1, laid side
 * by side (key c is token pages[.. + k0 + c/page] + c%page).  After these
 * groups comes each earlier document's last page when it is partial and
 * flagged, as an ordinary entry (its first token, len = length % page, mask
 * bit 0).  The rest of the row is as above.
 *
 * kv holds rowcap pairs per row, row (l*Hkv + h)*nq + q.  Returns 0, or -1
 * if the segments do not make nq tiles, a row exceeds rowcap or a document's
 * pages exceed page_cap.
 */
int sift_oracle_decode_ragged(int num_prompts, int num_docs, int num_layers, int num_kv_heads,
                              int tile, int page, const int32_t *cu_seqlens,
                              const int32_t *doc_cu, const int32_t *doc_end,
                              const int64_t *la_off, const int64_t *ca_off,
                              const uint64_t *la_words, const uint64_t *ca_words, int nq,
                              int rowcap, int page_cap, int32_t *qtiles, int32_t *kv,
                              int32_t *counts, int32_t *pages) {
    sift_bits_view s = {num_prompts, num_docs, num_kv_heads, tile, page, cu_seqlens, doc_cu,
                        doc_end, la_off, ca_off, la_words, ca_words};
    if (tile < 1 || page < 1 || (page < tile ? tile % page : page % tile) != 0 ||
        tile / (page < tile ? page : tile) > 16)
        return -1;  /* pages must nest with tiles, at most 16 pages per tile */
    const int pin = page < tile ? page : tile;
    const int nbits = tile / pin;
    const uint32_t full = (1u << nbits) - 1u;
    const int gather = page < tile && page % 8 == 0;
    int bad = 0;
    int q = 0;
    for (int p = 0; p < num_prompts; ++p)
        for (int g = doc_cu[p]; g <= doc_cu[p + 1]; ++g) {  /* g == doc_cu[p+1]: the suffix */
            int64_t start = g < doc_cu[p + 1] ? doc_begin(&s, p, g)
                            : (doc_cu[p + 1] > doc_cu[p] ? doc_end[doc_cu[p + 1] - 1]
                                                         : cu_seqlens[p]);
            int64_t end = g < doc_cu[p + 1] ? doc_end[g] : cu_seqlens[p + 1];
            for (int64_t x = start; x < end; x += tile, ++q)
                if (q < nq) {
                    qtiles[2 * q] = (int32_t)x;
                    qtiles[2 * q + 1] = (int32_t)(end - x < tile ? end - x : tile);
                }
        }
    if (q != nq) return -1;
    for (int l = 0; l < num_layers; ++l)
        for (int h = 0; h < num_kv_heads; ++h) {
            q = 0;
            for (int p = 0; p < num_prompts; ++p)
                for (int g = doc_cu[p]; g <= doc_cu[p + 1]; ++g) {
                    int suffix = g == doc_cu[p + 1];
                    int64_t start = !suffix ? doc_begin(&s, p, g)
                                    : (doc_cu[p + 1] > doc_cu[p] ? doc_end[doc_cu[p + 1] - 1]
                                                                 : cu_seqlens[p]);
                    int64_t end = !suffix ? doc_end[g] : cu_seqlens[p + 1];
                    for (int64_t x = start; x < end; x += tile, ++q) {
                        int64_t row = ((int64_t)l * num_kv_heads + h) * nq + q;
                        int32_t *out = kv + row * rowcap * 2;
                        int n = 0;
#define EMIT(first, info) do { if (n < rowcap) { out[2 * n] = (int32_t)(first); \
                               out[2 * n + 1] = (int32_t)(info); } else bad = 1; ++n; } while (0)
                        if (!suffix && gather) {
                            int64_t pbase = (((int64_t)l * num_kv_heads + h) * num_docs + g) * page_cap;
                            int64_t rel = ((int64_t)h * num_docs + g) * page_cap;
                            int npg = 0;
                            for (int gp = doc_cu[p]; gp < g; ++gp) {
                                int64_t ds = doc_begin(&s, p, gp), de = doc_end[gp];
                                for (int j = 0; (int64_t)(j + 1) * page <= de - ds; ++j)
                                    if (ca_bit(&s, p, gp, l, h, j)) {
                                        if (npg < page_cap) pages[pbase + npg] = (int32_t)(ds + (int64_t)j * page);
                                        else bad = 1;
                                        ++npg;
                                    }
                            }
                            for (int k0 = 0; k0 < npg; k0 += nbits) {
                                int in_group = npg - k0 < nbits ? npg - k0 : nbits;
                                EMIT(rel + k0, (uint32_t)(in_group * page) | 1u << 9 | full << 16);
                            }
                            for (int gp = doc_cu[p]; gp < g; ++gp) {
                                int64_t ds = doc_begin(&s, p, gp), de = doc_end[gp];
                                int64_t rem = (de - ds) % page;
                                if (rem && ca_bit(&s, p, gp, l, h, (int)((de - ds) / page)))
                                    EMIT(de - rem, (uint32_t)rem | 1u << 16);
                            }
                        }
                        for (int gp = doc_cu[p]; gp < g && !(!suffix && gather); ++gp) {
                            int64_t ds = doc_begin(&s, p, gp), de = doc_end[gp];
                            for (int64_t y = ds; y < de; y += tile) {
                                int64_t len = de - y < tile ? de - y : tile;
                                uint32_t mask = 0;
                                if (suffix) {
                                    mask = full;
                                } else {
                                    for (int k = 0; k < nbits && (int64_t)k * pin < len; ++k)
                                        if (ca_bit(&s, p, gp, l, h, (int)((y - ds + (int64_t)k * pin) / page)))
                                            mask |= 1u << k;
                                }
                                if (mask) EMIT(y, (uint32_t)len | mask << 16);
                            }
                        }
                        int64_t i = (x - start) / tile;
                        for (int64_t j = 0; j < i; ++j)
                            if (suffix || la_bit(&s, p, g, l, h, (int)i, (int)j))
                                EMIT(start + j * tile, (uint32_t)tile | full << 16);
                        EMIT(x, (uint32_t)(end - x < tile ? end - x : tile) | 1u << 8 | full << 16);
#undef EMIT
                        counts[row] = n;
                    }
                }
        }
    return bad ? -1 : 0;
}

static double bf16_to_double(uint16_t x) {
    uint32_t b = (uint32_t)x << 16;
    float f;
    memcpy(&f, &b, sizeof f);
    return (double)f;
}

/*
 * Masked softmax attention for selected (query token, query head) rows of one
 * layer.  The key set of each row comes straight from the bits via
 * key_visible(), never from the decoded lists, so the two routes check each
 * other.  Query head qh uses kv head qh / (Hq / Hkv) (grouped-query attention;
 * bits are read per kv head).
 *   o   = sum_u exp(s_u - m) v_u / sum_u exp(s_u - m),  s_u = scale * <q_t, k_u>
 *   lse = m + ln(sum_u exp(s_u - m))   (natural log)
 * q: bf16 [tokens][Hq][d]; k, v: bf16 [tokens][Hkv][d]; out_o: [nrows][d].
 * Returns 0, or -1 on a row outside the batch.
 */
int sift_oracle_attention_rows(int num_prompts, int num_docs, int num_kv_heads, int tile,
                               int page, const int32_t *cu_seqlens, const int32_t *doc_cu,
                               const int32_t *doc_end, const int64_t *la_off,
                               const int64_t *ca_off, const uint64_t *la_words,
                               const uint64_t *ca_words, int layer, int num_q_heads,
                               int head_dim, double scale, const uint16_t *q,
                               const uint16_t *k, const uint16_t *v, int64_t nrows,
                               const int32_t *row_tok, const int32_t *row_head,
                               double *out_o, double *out_lse) {
    sift_bits_view s = {num_prompts, num_docs, num_kv_heads, tile, page, cu_seqlens, doc_cu,
                        doc_end, la_off, ca_off, la_words, ca_words};
    const int G = num_q_heads / num_kv_heads;
    const int d = head_dim;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 8) reduction(| : bad)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = row_tok[r];
        int qh = row_head[r];
        int p = prompt_of(&s, t);
        if (p < 0 || qh < 0 || qh >= num_q_heads) { bad = 1; continue; }
        int h = qh / G;
        int64_t u0 = cu_seqlens[p];
        int64_t nk = t - u0 + 1;
        double *sc = (double *)malloc(sizeof(double) * (size_t)nk);
        char *vis = (char *)malloc((size_t)nk);
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        for (int c = 0; c < d; ++c) qd[c] = bf16_to_double(q[(t * num_q_heads + qh) * d + c]);
        double m = -INFINITY;
        for (int64_t u = u0; u <= t; ++u) {
            vis[u - u0] = (char)key_visible(&s, layer, h, t, u);
            if (!vis[u - u0]) continue;
            const uint16_t *kr = k + (u * num_kv_heads + h) * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qd[c] * bf16_to_double(kr[c]);
            sc[u - u0] = scale * acc;
            if (sc[u - u0] > m) m = sc[u - u0];
        }
        double l = 0.0;
        double *o = out_o + r * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int64_t u = u0; u <= t; ++u) {
            if (!vis[u - u0]) continue;
            double w = exp(sc[u - u0] - m);
            l += w;
            const uint16_t *vr = v + (u * num_kv_heads + h) * d;
            for (int c = 0; c < d; ++c) o[c] += w * bf16_to_double(vr[c]);
        }
        for (int c = 0; c < d; ++c) o[c] /= l;
        out_lse[r] = m + log(l);
        free(sc);
        free(vis);
        free(qd);
    }
    return bad ? -1 : 0;
}

/* Same key-set definition, exposed for the cross-check against the decoded lists:
 * writes a [nq][nk] 0/1 matrix for query tokens q_tok and key tokens k_tok. */
int sift_oracle_key_mask(int num_prompts, int num_docs, int num_kv_heads, int tile, int page,
                         const int32_t *cu_seqlens, const int32_t *doc_cu, const int32_t *doc_end,
                         const int64_t *la_off, const int64_t *ca_off, const uint64_t *la_words,
                         const uint64_t *ca_words, int layer, int kv_head, int64_t nq,
                         const int32_t *q_tok, int64_t nk, const int32_t *k_tok, uint8_t *out) {
    sift_bits_view s = {num_prompts, num_docs, num_kv_heads, tile, page, cu_seqlens, doc_cu,
                        doc_end, la_off, ca_off, la_words, ca_words};
    for (int64_t a = 0; a < nq; ++a)
        for (int64_t b = 0; b < nk; ++b)
            out[a * nk + b] = (uint8_t)key_visible(&s, layer, kv_head, q_tok[a], k_tok[b]);
    return 0;
}

int sift_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

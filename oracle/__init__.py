"""CPU oracle for SIFT's online prefill hot path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) import this package.  The product path
(``bit_vector_guided_gb300``) never does, and the two share no code: the only
common dependency is the seeded input generator in ``workloads``.

Two independent restatements of the same definition live here:
  * ``sift_oracle.c`` (built by :func:`build`): row-by-row masked softmax
    attention whose key set is read straight from the LA/CA bits, plus a
    plain nested-loop bit decode;
  * :func:`brute_force_attention` (numpy, fp64): a tile-level mask is expanded
    to an explicit token mask and dense softmax attention is taken with
    ``-inf`` outside it -- only for tiny inputs.

:func:`build_bits` restates the offline step (each document prefilled alone, its
tile masses ranked into LA/CA bits) in fp64 numpy; the pages give no selection
rule, so the rule there is this library's reading.

See ``sift_oracle.c`` for the readings of the pages (gist.science/it/paper/
2606.09441, "Design del Sistema", "Dettagli di Implementazione") and the pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sift_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libsift_oracle.so")
_lib = None

__all__ = ["build", "load", "decode", "schedule", "attention_rows", "attention_all",
           "key_mask", "brute_force_attention", "tile_mask", "set_threads", "decode_ragged",
           "token_mask", "page_capacity",
           "doc_tile_masses", "doc_unit_masses", "top_count", "select_top", "build_bits"]


def build(force: bool = False) -> str:
    """Compile sift_oracle.c with gcc (-O2 -fopenmp) into oracle/_build/."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def load():
    """The compiled oracle.  SIFT_ORACLE_LIB, when set, names another build of the same
    source to load instead (the mutation tests point it at copies with planted
    mistakes to show that the pins catch them)."""
    global _lib
    if _lib is None:
        override = os.environ.get("SIFT_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.sift_oracle_decode.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32, P, P]
        lib.sift_oracle_decode.restype = i32
        lib.sift_oracle_decode_ragged.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P,
                                                  P, P, i32, i32, i32, P, P, P, P]
        lib.sift_oracle_decode_ragged.restype = i32
        lib.sift_oracle_attention_rows.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P,
                                                   i32, i32, i32, f64, P, P, P, i64, P, P, P, P]
        lib.sift_oracle_attention_rows.restype = i32
        lib.sift_oracle_key_mask.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, i32,
                                             i32, i64, P, i64, P, P]
        lib.sift_oracle_key_mask.restype = i32
        lib.sift_oracle_set_threads.argtypes = [i32]
        lib.sift_oracle_set_threads.restype = i32
        _lib = lib
    return _lib


def set_threads(n: int = 0) -> int:
    """Set (n > 0) and return the number of OpenMP threads the oracle uses."""
    return int(load().sift_oracle_set_threads(int(n)))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _layout_args(layout, la_words, ca_words):
    arrs = [np.ascontiguousarray(layout.cu_seqlens, np.int32),
            np.ascontiguousarray(layout.doc_cu, np.int32),
            np.ascontiguousarray(layout.doc_end, np.int32),
            np.ascontiguousarray(layout.la_off, np.int64),
            np.ascontiguousarray(layout.ca_off, np.int64),
            np.ascontiguousarray(la_words, np.uint64) if len(la_words) else np.zeros(1, np.uint64),
            np.ascontiguousarray(ca_words, np.uint64) if len(ca_words) else np.zeros(1, np.uint64)]
    if len(arrs[2]) == 0:
        arrs[2] = np.zeros(1, np.int32)
        arrs[3] = np.zeros(1, np.int64)
        arrs[4] = np.zeros(1, np.int64)
    return arrs


def _page(layout) -> int:
    page = int(getattr(layout, "page", 0) or 0)
    return page if page > 0 else int(layout.tile)


def decode(layout, la_words, ca_words, rowcap: Optional[int] = None):
    """Tile index lists of every (layer, kv head, query tile) row (aligned layouts:
    page == tile and every boundary a multiple of the tile).

    Returns (kv_idx int32 [L, Hkv, N, rowcap] with -1 padding, counts int32 [L, Hkv, N]).
    """
    lib = load()
    rowcap = rowcap or layout.max_tiles_per_prompt
    L, Hkv, N = layout.num_layers, layout.num_kv_heads, layout.num_tiles
    kv_idx = np.full((L, Hkv, N, rowcap), -1, np.int32)
    counts = np.zeros((L, Hkv, N), np.int32)
    arrs = _layout_args(layout, la_words, ca_words)
    rc = lib.sift_oracle_decode(layout.num_prompts, layout.num_docs, L, Hkv, layout.tile,
                                *[_ptr(a) for a in arrs], rowcap, _ptr(kv_idx), _ptr(counts))
    if rc != 0:
        raise ValueError("oracle decode: a row exceeds rowcap")
    return kv_idx, counts


def page_capacity(layout) -> int:
    """Gathered pages per (layer, kv head, document): rowcap x pages per tile when pages
    are gathered (page < tile, a multiple of 8), else 0."""
    P, B = _page(layout), int(layout.tile)
    return int(layout.max_tiles_per_prompt) * (B // P) if (P < B and P % 8 == 0) else 0


def decode_ragged(layout, la_words, ca_words, rowcap: Optional[int] = None,
                  page_cap: Optional[int] = None):
    """Per-segment query tiles and their (first token, info) key-tile lists, for documents
    of any length and a CA page size of its own (rule in sift_oracle.c).

    Returns (qtiles int32 [NQ, 2], kv int32 [L, Hkv, NQ, rowcap, 2] with -1 padding,
    counts int32 [L, Hkv, NQ], pages int32 [L, Hkv, D, page_cap] with -1 padding).
    """
    lib = load()
    rowcap = rowcap or layout.max_tiles_per_prompt
    page_cap = page_capacity(layout) if page_cap is None else int(page_cap)
    L, Hkv, NQ, D = layout.num_layers, layout.num_kv_heads, layout.num_query_tiles, layout.num_docs
    qtiles = np.zeros((max(NQ, 1), 2), np.int32)
    kv = np.full((L, Hkv, max(NQ, 1), rowcap, 2), -1, np.int32)
    counts = np.zeros((L, Hkv, max(NQ, 1)), np.int32)
    pages = np.full((L, Hkv, max(D, 1), max(page_cap, 1)), -1, np.int32)
    arrs = _layout_args(layout, la_words, ca_words)
    rc = lib.sift_oracle_decode_ragged(layout.num_prompts, layout.num_docs, L, Hkv, layout.tile,
                                       _page(layout), *[_ptr(a) for a in arrs], NQ, rowcap,
                                       page_cap, _ptr(qtiles), _ptr(kv), _ptr(counts),
                                       _ptr(pages))
    if rc != 0:
        raise ValueError("oracle ragged decode: bad page size, tile count or capacity")
    return qtiles[:NQ], kv[:, :, :NQ], counts[:, :, :NQ], pages[:, :, :D, :page_cap]


def schedule(counts: np.ndarray) -> np.ndarray:
    """Longest-first order of the (kv head, query tile) units of each layer.

    counts [L, Hkv, N] -> sched [L, Hkv*N] with unit index u = h*N + i, sorted by
    count descending, ties by u ascending.  Any order with non-increasing counts is
    an equally valid schedule; this one is the unique stable representative.
    """
    L = counts.shape[0]
    flat = counts.reshape(L, -1)
    return np.stack([np.argsort(-flat[l], kind="stable") for l in range(L)]).astype(np.int32)


def _bf16_bits(x) -> np.ndarray:
    """torch bf16 tensor (any device) or uint16 array -> contiguous uint16 numpy."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, np.uint16)
    import torch
    return np.ascontiguousarray(x.detach().to("cpu").contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def attention_rows(layout, la_words, ca_words, layer, q, k, v, row_tok, row_head,
                   scale: Optional[float] = None):
    """O (fp64 [n, d]) and LSE (fp64 [n]) for the requested (token, query head) rows."""
    lib = load()
    d = layout.head_dim
    scale = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    row_tok = np.ascontiguousarray(row_tok, np.int32)
    row_head = np.ascontiguousarray(row_head, np.int32)
    n = len(row_tok)
    out_o = np.zeros((max(n, 1), d), np.float64)
    out_lse = np.zeros(max(n, 1), np.float64)
    arrs = _layout_args(layout, la_words, ca_words)
    rc = lib.sift_oracle_attention_rows(
        layout.num_prompts, layout.num_docs, layout.num_kv_heads, layout.tile, _page(layout),
        *[_ptr(a) for a in arrs], int(layer), layout.num_q_heads, d, scale,
        _ptr(qb), _ptr(kb), _ptr(vb), n, _ptr(row_tok), _ptr(row_head),
        _ptr(out_o), _ptr(out_lse))
    if rc != 0:
        raise ValueError("oracle attention: row outside the batch")
    return out_o[:n], out_lse[:n]


def attention_all(layout, la_words, ca_words, layer, q, k, v, scale=None):
    """Every row of one layer: O fp64 [tokens, Hq, d], LSE fp64 [Hq, tokens]."""
    T, Hq, d = layout.total_tokens, layout.num_q_heads, layout.head_dim
    tok = np.repeat(np.arange(T, dtype=np.int32), Hq)
    head = np.tile(np.arange(Hq, dtype=np.int32), T)
    o, lse = attention_rows(layout, la_words, ca_words, layer, q, k, v, tok, head, scale)
    return o.reshape(T, Hq, d), lse.reshape(T, Hq).T.copy()


def key_mask(layout, la_words, ca_words, layer, kv_head, q_tok, k_tok) -> np.ndarray:
    """0/1 [len(q_tok), len(k_tok)] visibility matrix from the bits (same rule as attention_rows)."""
    lib = load()
    q_tok = np.ascontiguousarray(q_tok, np.int32)
    k_tok = np.ascontiguousarray(k_tok, np.int32)
    out = np.zeros((len(q_tok), len(k_tok)), np.uint8)
    arrs = _layout_args(layout, la_words, ca_words)
    lib.sift_oracle_key_mask(layout.num_prompts, layout.num_docs, layout.num_kv_heads,
                             layout.tile, _page(layout), *[_ptr(a) for a in arrs], int(layer),
                             int(kv_head),
                             len(q_tok), _ptr(q_tok), len(k_tok), _ptr(k_tok), _ptr(out))
    return out.astype(bool)


# --------------------------------------------------------------------------------------
# Second, independent restatement for tiny inputs: explicit dense masks in numpy.
# --------------------------------------------------------------------------------------

def _unpack(words: np.ndarray, nbits: int) -> np.ndarray:
    """uint64 words [..., W] -> bool [..., nbits], bit j = bit (j%64) of word j//64."""
    by = np.ascontiguousarray(words, "<u8").view(np.uint8)
    bits = np.unpackbits(by.reshape(words.shape[:-1] + (-1,)), axis=-1, bitorder="little")
    return bits[..., :nbits].astype(bool)


def tile_mask(layout, la_words, ca_words, layer, kv_head) -> np.ndarray:
    """Global tile-level mask M[i, j] (query tile i may use key tile j).

    Built block by block from the plain description: a prompt's tiles see only
    tiles of the same prompt; suffix rows see every tile up to the diagonal;
    document rows see the diagonal, the LA-flagged tiles below it inside the
    document, and the CA-flagged pages of every earlier document.
    """
    B, Hkv = layout.tile, layout.num_kv_heads
    N = layout.num_tiles
    M = np.zeros((N, N), bool)
    for p in range(layout.num_prompts):
        t0, t1 = layout.cu_seqlens[p] // B, layout.cu_seqlens[p + 1] // B
        docs = range(layout.doc_cu[p], layout.doc_cu[p + 1])
        spans = []
        for g in docs:
            s = layout.doc_start(g) // B
            T = layout.doc_tiles(g)
            W = (T + 63) // 64
            base = layout.la_off[g] + (layer * Hkv + kv_head) * T * W
            la = _unpack(la_words[base: base + T * W].reshape(T, W), T)
            cbase = layout.ca_off[g] + (layer * Hkv + kv_head) * W
            ca = _unpack(ca_words[cbase: cbase + W].reshape(1, W), T)[0]
            spans.append((s, T, la, ca))
        for k, (s, T, la, ca) in enumerate(spans):
            M[s:s + T, s:s + T] |= np.tril(la, -1)
            for (s2, T2, _, ca2) in spans[:k]:
                M[s:s + T, s2:s2 + T2] |= ca2[None, :]
        last = spans[-1][0] + spans[-1][1] if spans else t0
        for i in range(last, t1):
            M[i, t0:i + 1] = True
        for i in range(t0, t1):
            M[i, i] = True
    return M


def token_mask(layout, la_words, ca_words, layer, kv_head) -> np.ndarray:
    """Token-level mask M[t, u] (query token t may use key token u), any layout.

    Built block by block from the plain description, with tiles and pages counted
    from each document's first token: a document's block holds its own LA tiles
    (plus every token's own tile), a later document's block against an earlier one
    holds the earlier one's CA-flagged pages, the query suffix sees its whole prompt,
    and everything is causal.
    """
    B, Pg, Hkv = layout.tile, _page(layout), layout.num_kv_heads
    T = layout.total_tokens
    M = np.zeros((T, T), bool)
    for p in range(layout.num_prompts):
        c0, c1 = int(layout.cu_seqlens[p]), int(layout.cu_seqlens[p + 1])
        earlier = []
        last = c0
        for g in range(int(layout.doc_cu[p]), int(layout.doc_cu[p + 1])):
            s0, e0 = layout.doc_start(g), int(layout.doc_end[g])
            n = e0 - s0
            Tg, Cg = -(-n // B), -(-n // Pg)
            W, V = -(-Tg // 64), -(-Cg // 64)
            base = int(layout.la_off[g]) + (layer * Hkv + kv_head) * Tg * W
            la = _unpack(np.asarray(la_words[base: base + Tg * W]).reshape(Tg, W), Tg)
            cbase = int(layout.ca_off[g]) + (layer * Hkv + kv_head) * V
            ca = _unpack(np.asarray(ca_words[cbase: cbase + V]).reshape(1, V), Cg)[0]
            tl = np.arange(n) // B
            same = tl[:, None] == tl[None, :]
            below = la[tl[:, None], tl[None, :]] & (tl[None, :] < tl[:, None])
            M[s0:e0, s0:e0] = same | below
            for (s2, e2, keep2) in earlier:
                M[s0:e0, s2:e2] = keep2[None, :]
            earlier.append((s0, e0, ca[np.arange(n) // Pg]))
            last = e0
        M[last:c1, c0:c1] = True
    return M & np.tril(np.ones((T, T), bool))


def brute_force_attention(layout, la_words, ca_words, layer, q, k, v, scale=None):
    """Dense fp64 attention with -inf outside the token mask (tiny inputs only): the tile
    mask expanded to tokens for aligned layouts, token_mask otherwise."""
    qb = _bf16_bits(q).astype(np.uint32) << 16
    kb = _bf16_bits(k).astype(np.uint32) << 16
    vb = _bf16_bits(v).astype(np.uint32) << 16
    qf = qb.view(np.float32).astype(np.float64)
    kf = kb.view(np.float32).astype(np.float64)
    vf = vb.view(np.float32).astype(np.float64)
    T, Hq, d = qf.shape
    Hkv = kf.shape[1]
    G = Hq // Hkv
    B = layout.tile
    scale = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    causal = np.tril(np.ones((T, T), bool))
    O = np.zeros((T, Hq, d))
    LSE = np.zeros((Hq, T))
    aligned = getattr(layout, "aligned", True)
    for h in range(Hkv):
        if aligned:
            M = np.kron(tile_mask(layout, la_words, ca_words, layer, h),
                        np.ones((B, B), bool)) & causal
        else:
            M = token_mask(layout, la_words, ca_words, layer, h)
        for qh in range(h * G, (h + 1) * G):
            S = scale * qf[:, qh, :] @ kf[:, h, :].T
            S = np.where(M, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            P = np.exp(S - m)
            l = P.sum(axis=1, keepdims=True)
            O[:, qh, :] = (P / l) @ vf[:, h, :]
            LSE[qh] = (m + np.log(l))[:, 0]
    return O, LSE


# --------------------------------------------------------------------------------------
# Offline bit building (the step before the online path), restated in fp64 numpy.
# --------------------------------------------------------------------------------------

def doc_tile_masses(q, k, start, end, h, G, tile, scale):
    """M[i][j]: attention probability mass that the query rows of tile i (all query heads
    of kv head h's group) put on key tile j, in causal attention inside the document
    [start, end) alone.  Rows of M sum to G*tile."""
    qf = np.asarray(_bf16_bits(q[start:end, h * G:(h + 1) * G]).astype(np.uint32) << 16
                    ).view(np.float32).astype(np.float64)
    kf = np.asarray(_bf16_bits(k[start:end, h:h + 1]).astype(np.uint32) << 16
                    ).view(np.float32).astype(np.float64)[:, 0]
    n = end - start
    T = n // tile
    causal = np.tril(np.ones((n, n), bool))
    M = np.zeros((T, T))
    for g in range(G):
        S = scale * qf[:, g, :] @ kf.T
        S = np.where(causal, S, -np.inf)
        S -= S.max(axis=1, keepdims=True)
        Pm = np.exp(S)
        Pm /= Pm.sum(axis=1, keepdims=True)
        M += Pm.reshape(T, tile, T, tile).sum(axis=(1, 3))
    return M


def top_count(fraction: float, candidates: int) -> int:
    """Number of candidates kept: ceil(fraction * candidates - 1e-4), each operation rounded
    to float32 (the slack keeps exact products such as 0.25 * 8 from rounding up)."""
    prod = np.float32(np.float32(fraction) * np.float32(candidates))
    return int(np.ceil(np.float32(prod - np.float32(1e-4))))


def select_top(mass: np.ndarray, kcount: int) -> np.ndarray:
    """Indices of the kcount largest entries (ties: lower index first)."""
    order = sorted(range(len(mass)), key=lambda j: (-mass[j], j))
    return np.array(sorted(order[:kcount]), dtype=np.int64)


def doc_unit_masses(q, k, start, end, h, G, tile, unit, scale):
    """Mu[i][u]: attention probability mass that the query rows of tile i (all query heads of
    kv head h's group; tiles of `tile` tokens from the document start, the last partial) put
    on key unit u (units of `unit` tokens, counted the same way), in causal attention inside
    the document [start, end) alone.  Row i sums to G x (rows of tile i)."""
    qf = np.asarray(_bf16_bits(q[start:end, h * G:(h + 1) * G]).astype(np.uint32) << 16
                    ).view(np.float32).astype(np.float64)
    kf = np.asarray(_bf16_bits(k[start:end, h:h + 1]).astype(np.uint32) << 16
                    ).view(np.float32).astype(np.float64)[:, 0]
    n = end - start
    causal = np.tril(np.ones((n, n), bool))
    P = np.zeros((n, n))
    for g in range(G):
        S = scale * qf[:, g, :] @ kf.T
        S = np.where(causal, S, -np.inf)
        S -= S.max(axis=1, keepdims=True)
        Pm = np.exp(S)
        P += Pm / Pm.sum(axis=1, keepdims=True)
    rows = np.add.reduceat(P, np.arange(0, n, tile), axis=0)
    return np.add.reduceat(rows, np.arange(0, n, unit), axis=1)


def build_bits(layout, layer, q, k, la_fraction, ca_fraction, scale=None):
    """LA/CA words of one layer from document-alone attention (the offline profiler).
    Tiles and pages are counted from each document's first token (the last ones partial);
    masses are gathered per unit of min(page, tile) tokens:
      M[i][j]  = mass that query tile i puts on key tile j (its units summed);
      LA row i keeps the top_count(la_fraction, i) tiles j < i of largest M[i][j];
      page c, whose first token lies in tile t(c), scores the mean mass it receives from
      the query tiles i >= t(c), sum_{i >= t(c)} mass_i(c) / (T - t(c));
      CA keeps the top_count(ca_fraction, C) pages of largest score.
    With page == tile this is the tile rule: score(j) = sum_{i>=j} M[i][j] / (T - j).
    Returns (la_words, ca_words, masses, scores) with the layer's blocks filled (other
    layers 0), masses[(g, h)] = M and scores[(g, h)] = the page scores, for validation."""
    B, Hkv = layout.tile, layout.num_kv_heads
    Pg = _page(layout)
    U = min(Pg, B)
    G = layout.num_q_heads // Hkv
    scale = (1.0 / np.sqrt(layout.head_dim)) if scale is None else float(scale)
    la = np.zeros(layout.la_words_len, np.uint64)
    ca = np.zeros(layout.ca_words_len, np.uint64)
    masses, scores = {}, {}
    for g in range(layout.num_docs):
        s0, e0 = layout.doc_start(g), int(layout.doc_end[g])
        n = e0 - s0
        T, C = -(-n // B), -(-n // Pg)
        W, V = -(-T // 64), -(-C // 64)
        unit_tile = (np.arange(-(-n // U)) * U) // B     # tile of each unit
        unit_page = (np.arange(-(-n // U)) * U) // Pg    # page of each unit
        for h in range(Hkv):
            Mu = doc_unit_masses(q, k, s0, e0, h, G, B, U, scale)
            M = np.zeros((T, T))
            Mp = np.zeros((T, C))
            for u in range(Mu.shape[1]):
                M[:, unit_tile[u]] += Mu[:, u]
                Mp[:, unit_page[u]] += Mu[:, u]
            t_of = (np.arange(C) * Pg) // B
            score = np.array([Mp[t_of[c]:, c].sum() / (T - t_of[c]) for c in range(C)])
            masses[(g, h)], scores[(g, h)] = M, score
            lab = np.zeros((T, W * 64), bool)
            for i in range(1, T):
                lab[i, select_top(M[i, :i], top_count(la_fraction, i))] = True
            cab = np.zeros(V * 64, bool)
            cab[select_top(score, top_count(ca_fraction, C))] = True
            base = layout.la_off[g] + (layer * Hkv + h) * T * W
            la[base: base + T * W] = np.packbits(lab, axis=1, bitorder="little").view("<u8").reshape(-1)
            cbase = layout.ca_off[g] + (layer * Hkv + h) * V
            ca[cbase: cbase + V] = np.packbits(cab, bitorder="little").view("<u8")
    return la, ca, masses, scores

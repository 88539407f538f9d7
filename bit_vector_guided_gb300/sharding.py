"""KV-head sharding of one SIFT prefill across GPUs (host-side layout only).

The hot path has no exchange step: bits are kept per KV head and every query head
of a GQA group reads only its own KV head, so a contiguous range of KV heads (with
their query heads) is an independent problem.  A rank takes its range, slices Q/K/V
along the head axis and runs the unchanged C ABI on the shard; the outputs of the
ranks are the head slices of the unsharded output.  No collective runs inside the
op (a tensor-parallel O-projection would all-reduce downstream of it).

This module only re-packs the LA/CA words and offsets of a head range -- a copy of
contiguous word blocks -- and computes which heads a rank owns.
"""
from __future__ import annotations

import numpy as np

__all__ = ["kv_head_range", "shard_bits"]


def kv_head_range(rank: int, world: int, num_kv_heads: int):
    """[h0, h1) of the KV heads owned by `rank`: contiguous, sizes differing by at most one."""
    if not (0 <= rank < world) or world < 1:
        raise ValueError("rank outside the world")
    base, extra = divmod(num_kv_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def _doc_sizes(cu_seqlens, doc_cu, doc_end, tile, page):
    """LA tiles and CA words (per layer and head) of every document: ceil(n/tile) rows and
    ceil(ceil(n/page)/64) words, counted from the document's first token."""
    cu = np.asarray(cu_seqlens, np.int64)
    dcu = np.asarray(doc_cu, np.int64)
    de = np.asarray(doc_end, np.int64)
    tiles = np.zeros(len(de), np.int64)
    ca_words = np.zeros(len(de), np.int64)
    for p in range(len(cu) - 1):
        start = cu[p]
        for g in range(dcu[p], dcu[p + 1]):
            n = de[g] - start
            tiles[g] = (n + tile - 1) // tile
            ca_words[g] = ((n + page - 1) // page + 63) // 64
            start = de[g]
    return tiles, ca_words


def shard_bits(cu_seqlens, doc_cu, doc_end, la_off, ca_off, la_words, ca_words, num_layers,
               num_kv_heads, tile, h0, h1, page=0):
    """LA/CA words and offsets of KV heads [h0, h1) in the layout the C ABI expects for a
    problem with h1 - h0 KV heads, on either layout (page 0 means the tile).  Returns
    (la_off, ca_off, la_words, ca_words) as numpy arrays; the prompt/document arrays are
    unchanged."""
    if not (0 <= h0 < h1 <= num_kv_heads):
        raise ValueError("bad head range")
    tiles, ca_w = _doc_sizes(cu_seqlens, doc_cu, doc_end, tile, page if page > 0 else tile)
    la_words = np.asarray(la_words, np.uint64)
    ca_words = np.asarray(ca_words, np.uint64)
    la_parts, ca_parts = [], []
    la_off_s = np.zeros(len(tiles), np.int64)
    ca_off_s = np.zeros(len(tiles), np.int64)
    la_pos = ca_pos = 0
    H = h1 - h0
    for g, T in enumerate(tiles):
        W = (int(T) + 63) // 64
        V = int(ca_w[g])
        la_off_s[g] = la_pos
        ca_off_s[g] = ca_pos
        for l in range(num_layers):
            a = int(la_off[g]) + (l * num_kv_heads + h0) * int(T) * W
            la_parts.append(la_words[a: a + H * int(T) * W])
            b = int(ca_off[g]) + (l * num_kv_heads + h0) * V
            ca_parts.append(ca_words[b: b + H * V])
        la_pos += num_layers * H * int(T) * W
        ca_pos += num_layers * H * V
    la_s = np.concatenate(la_parts) if la_parts else np.zeros(0, np.uint64)
    ca_s = np.concatenate(ca_parts) if ca_parts else np.zeros(0, np.uint64)
    return la_off_s, ca_off_s, la_s, ca_s

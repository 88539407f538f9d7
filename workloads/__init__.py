"""Seeded synthetic inputs for the SIFT online-prefill hot path.

This module only *generates* inputs: prompt layouts (documents + query
suffix, packed varlen), packed LA/CA bit vectors and bf16 Q/K/V.  It holds
none of the method's arithmetic (no decoding of bits into tile lists, no
attention), so that both the CUDA path and the CPU oracle can consume the
same inputs without sharing any computation.

Workload shapes follow the SIFT pages (gist.science/it/paper/2606.09441,
"Design del Sistema": one LA and one CA bit vector per document, layer and
head; "Risultati": Llama-3.1-8B and Qwen3-235B-A22B head layouts, 32K-64K
contexts).  The pages print no bit statistics; the densities below are the
synthetic stand-ins for the LongBench workloads that the pages evaluate on.

Bit layout (the pages give none; this is the reading used everywhere):
  * LA block of document g (T_g tiles, W_g = ceil(T_g/64) words per row) for
    (layer l, kv head h) is a T_g x W_g row-major array of uint64 words at
    word offset ``la_off[g] + (l*Hkv + h) * T_g * W_g``.  Bit j of row i is
    bit (j & 63) (LSB first) of word (j >> 6); only j < i is meaningful.
  * CA block of document g for (l, h) is V_g = ceil(C_g/64) words at
    ``ca_off[g] + (l*Hkv + h) * V_g``; bit j marks KV page j of document g.
  * Tiles and pages are counted from the document's own first token:
    T_g = ceil(n_g / tile) LA tiles and C_g = ceil(n_g / page) CA pages for a
    document of n_g tokens, the last ones possibly partial.  With page == tile
    and every length a multiple of the tile (the default workloads) both
    counts are n_g / tile and V_g = W_g.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Callable, Optional, Sequence

import numpy as np

__all__ = [
    "BitSpec", "Config", "Layout", "CONFIGS", "get_config", "custom_config",
    "make_layout", "make_bits", "make_qkv", "seed_for",
]


def seed_for(*parts) -> int:
    """Stable 32-bit seed from a tuple of names/ints (crc32 of their repr)."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0xFFFFFFFF


@dataclasses.dataclass(frozen=True)
class BitSpec:
    """How the synthetic LA / CA bits of one configuration are drawn.

    la_p / ca_p      Bernoulli probability of a set bit (LA: tiles j < i-window,
                     CA: every page).  Ignored when ``head_density`` is set.
    la_window        number of tiles directly below the diagonal that are always on.
    ca_first_page    page 0 of every document always on.
    head_density     (lo, hi): per (layer, kv head) draw s ~ U[lo, hi]; then
                     LA p = s and CA p = s * head_ca_ratio.
    pattern          'random' | 'ones' | 'zeros' | 'la_only' | 'ca_only':
                     deterministic special cases used by the pins.
    """
    la_p: float = 0.0
    ca_p: float = 0.0
    la_window: int = 0
    ca_first_page: bool = False
    head_density: Optional[tuple] = None
    head_ca_ratio: float = 0.5
    pattern: str = "random"


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    tile: int
    # one entry per prompt: (list of document lengths in tokens, suffix length)
    prompts: tuple
    bits: BitSpec
    description: str = ""
    page: int = 0  # CA page size in tokens; 0 = the tile size

    @property
    def total_tokens(self) -> int:
        return sum(sum(d) + s for d, s in self.prompts)

    @property
    def page_size(self) -> int:
        return self.page if self.page > 0 else self.tile


@dataclasses.dataclass
class Layout:
    """Host-side (numpy) description of one packed varlen batch."""
    num_prompts: int
    num_docs: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    tile: int
    total_tokens: int
    max_tiles_per_prompt: int
    cu_seqlens: np.ndarray   # int32 [P+1] token offsets
    doc_cu: np.ndarray       # int32 [P+1] document offsets
    doc_end: np.ndarray      # int32 [D]   absolute end token (exclusive) of each doc
    la_off: np.ndarray       # int64 [D]   word offset of each doc's LA blocks
    ca_off: np.ndarray       # int64 [D]   word offset of each doc's CA blocks
    la_words_len: int
    ca_words_len: int
    page: int = 0  # CA page size in tokens; 0 = the tile size

    @property
    def page_size(self) -> int:
        return self.page if self.page > 0 else self.tile

    @property
    def num_tiles(self) -> int:
        return self.total_tokens // self.tile

    @property
    def aligned(self) -> bool:
        """page == tile and every prompt and document boundary a multiple of the tile."""
        B = self.tile
        return (self.page_size == B and all(int(x) % B == 0 for x in self.cu_seqlens)
                and all(int(x) % B == 0 for x in self.doc_end))

    def segments(self):
        """(start, end, document or -1 for the query suffix) of every segment, in token order."""
        out = []
        for p in range(self.num_prompts):
            pos = int(self.cu_seqlens[p])
            for g in range(int(self.doc_cu[p]), int(self.doc_cu[p + 1])):
                out.append((pos, int(self.doc_end[g]), g))
                pos = int(self.doc_end[g])
            out.append((pos, int(self.cu_seqlens[p + 1]), -1))
        return out

    @property
    def num_query_tiles(self) -> int:
        """Query tiles counted per segment (documents and suffixes tile from their own start)."""
        B = self.tile
        return sum((e - s + B - 1) // B for s, e, _ in self.segments())

    def doc_tiles(self, g: int) -> int:
        start = self.doc_start(g)
        return (int(self.doc_end[g]) - start + self.tile - 1) // self.tile

    def doc_pages(self, g: int) -> int:
        start = self.doc_start(g)
        P = self.page_size
        return (int(self.doc_end[g]) - start + P - 1) // P

    def doc_start(self, g: int) -> int:
        p = int(np.searchsorted(self.doc_cu, g, side="right")) - 1
        return int(self.cu_seqlens[p]) if g == int(self.doc_cu[p]) else int(self.doc_end[g - 1])


def custom_config(name, prompts, bits, num_layers=1, num_q_heads=4, num_kv_heads=2,
                  head_dim=128, tile=128, description="", page=0) -> Config:
    prompts = tuple((tuple(int(x) for x in docs), int(suf)) for docs, suf in prompts)
    return Config(name, num_layers, num_q_heads, num_kv_heads, head_dim, tile, prompts,
                  bits, description, int(page))


def _ragged_lengths(name: str, n: int, lo: int, hi: int, total: int) -> list:
    """n seeded document lengths drawn from U[lo, hi], rescaled to sum to `total`."""
    rng = np.random.Generator(np.random.PCG64(seed_for(name, "lengths")))
    raw = rng.integers(lo, hi + 1, size=n).astype(np.float64)
    out = [int(x) for x in np.floor(raw * total / raw.sum())]
    out[-1] += total - sum(out)
    return out


def _batch4(p: float) -> Config:
    tag = f"batch4_p{int(round(p * 100)):03d}"
    return custom_config(
        tag, [([2048] * n, 256) for n in (8, 16, 24, 32)],
        BitSpec(la_p=p, ca_p=p, pattern="ones" if p >= 1.0 else "random"),
        num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128, tile=128,
        description=f"Llama-8B head layout, batch of 4 prompts (8/16/24/32 docs x 2048 + 256), "
                    f"LA = CA density {p:.2f}")


CONFIGS = {
    "tiny": custom_config(
        "tiny", [([256, 256], 64)], BitSpec(la_p=0.4, ca_p=0.3),
        num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=64, tile=64,
        description="2 docs x 256 + 64-token query, GQA 2:1, d=64, tile 64, LA 0.4, CA 0.3"),
    "llama_10doc": custom_config(
        "llama_10doc", [([1024] * 10, 128)],
        BitSpec(la_p=0.15, ca_p=0.15, la_window=2, ca_first_page=True),
        num_layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128, tile=128,
        description="Llama-3.1-8B layer, 10 docs x 1024 + 128 (10368 tokens), "
                    "LA window 2 + Bernoulli 0.15, CA 0.15 + first page"),
    "llama_32k": custom_config(
        "llama_32k", [([2048] * 16, 256)],
        BitSpec(head_density=(0.05, 0.35), head_ca_ratio=0.5),
        num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, tile=128,
        description="Llama-3.1-8B, 16 docs x 2048 + 256 (33024 tokens) x 32 layers, "
                    "per-(layer,head) LA density U[0.05,0.35], CA half of it"),
    "llama_32k_ragged": custom_config(
        "llama_32k_ragged", [(_ragged_lengths("llama_32k_ragged", 16, 1024, 3072, 32731), 293)],
        BitSpec(head_density=(0.05, 0.35), head_ca_ratio=0.0625),
        num_layers=32, num_q_heads=32, num_kv_heads=8, head_dim=128, tile=128, page=16,
        description="Llama-3.1-8B, 16 docs of 1024-3072 tokens (seeded, 32731 in all) + 293 "
                    "(33024 tokens) x 32 layers, CA pages of 16 tokens; per-(layer,head) LA "
                    "density U[0.05,0.35], CA page density 1/16 of it (about half of it per "
                    "128-token tile, as in llama_32k)"),
    "qwen3_64k": custom_config(
        "qwen3_64k", [([2048] * 32, 512)],
        BitSpec(la_p=0.15, ca_p=0.08, ca_first_page=True),
        num_layers=1, num_q_heads=64, num_kv_heads=4, head_dim=128, tile=128,
        description="Qwen3-235B-A22B layer, GQA 16:1, 32 docs x 2048 + 512 (66048 tokens), "
                    "LA 0.15, CA 0.08 + first page"),
}
for _p in (0.05, 0.10, 0.20, 0.40, 0.70, 1.00):
    _c = _batch4(_p)
    CONFIGS[_c.name] = _c


def get_config(name: str) -> Config:
    return CONFIGS[name]


def make_layout(cfg: Config) -> Layout:
    B = cfg.tile
    Pg = cfg.page_size
    cu = [0]
    doc_cu = [0]
    doc_end = []
    la_off, ca_off = [], []
    la_pos = ca_pos = 0
    max_tiles = 0
    for docs, suf in cfg.prompts:
        pos = cu[-1]
        tiles = (suf + B - 1) // B  # key tiles of the prompt, each segment tiled on its own
        for n in docs:
            T = (n + B - 1) // B
            W = (T + 63) // 64
            V = ((n + Pg - 1) // Pg + 63) // 64
            tiles += T
            pos += n
            doc_end.append(pos)
            la_off.append(la_pos)
            ca_off.append(ca_pos)
            la_pos += cfg.num_layers * cfg.num_kv_heads * T * W
            ca_pos += cfg.num_layers * cfg.num_kv_heads * V
        pos += suf
        cu.append(pos)
        doc_cu.append(len(doc_end))
        if Pg < B and Pg % 8 == 0:
            # gathered CA pages: each earlier document may add its partial last page
            tiles += len(docs)
        max_tiles = max(max_tiles, tiles)
    return Layout(
        num_prompts=len(cfg.prompts), num_docs=len(doc_end), num_layers=cfg.num_layers,
        num_q_heads=cfg.num_q_heads, num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim,
        tile=B, total_tokens=cu[-1], max_tiles_per_prompt=max(max_tiles, 1),
        cu_seqlens=np.asarray(cu, np.int32), doc_cu=np.asarray(doc_cu, np.int32),
        doc_end=np.asarray(doc_end, np.int32), la_off=np.asarray(la_off, np.int64),
        ca_off=np.asarray(ca_off, np.int64), la_words_len=la_pos, ca_words_len=ca_pos,
        page=cfg.page)


def _pack_rows(bits: np.ndarray) -> np.ndarray:
    """Pack a bool array [..., n] into little-endian uint64 words [..., ceil(n/64)]."""
    n = bits.shape[-1]
    W = (n + 63) // 64
    pad = np.zeros(bits.shape[:-1] + (W * 64,), dtype=bool)
    pad[..., :n] = bits
    by = np.packbits(pad, axis=-1, bitorder="little")
    return by.view("<u8").reshape(bits.shape[:-1] + (W,)).astype(np.uint64)


def make_bits(cfg: Config, layout: Layout):
    """Draw the LA / CA bit vectors of every document, layer and kv head.

    Returns (la_words, ca_words) as uint64 numpy arrays laid out as described
    in the module docstring.
    """
    spec = cfg.bits
    L, Hkv = cfg.num_layers, cfg.num_kv_heads
    la = np.zeros(layout.la_words_len, np.uint64)
    ca = np.zeros(layout.ca_words_len, np.uint64)
    if spec.head_density is not None:
        rng = np.random.Generator(np.random.PCG64(seed_for(cfg.name, "head_density")))
        lo, hi = spec.head_density
        dens = rng.uniform(lo, hi, size=(L, Hkv))
        la_p = dens[:, :, None, None]
        ca_p = (dens * spec.head_ca_ratio)[:, :, None]
    else:
        la_p, ca_p = spec.la_p, spec.ca_p
    for g in range(layout.num_docs):
        T = layout.doc_tiles(g)
        C = layout.doc_pages(g)
        W = (T + 63) // 64
        V = (C + 63) // 64
        i = np.arange(T)[:, None]
        j = np.arange(T)[None, :]
        below = j < i
        if spec.pattern == "random":
            rng = np.random.Generator(np.random.PCG64(seed_for(cfg.name, "doc", g, "bits")))
            la_b = rng.random((L, Hkv, T, T)) < la_p
            ca_b = rng.random((L, Hkv, C)) < ca_p
            if spec.la_window > 0:
                la_b |= ((i - j) >= 1) & ((i - j) <= spec.la_window)
            if spec.ca_first_page and C > 0:
                ca_b[..., 0] = True
        elif spec.pattern == "ones":
            la_b = np.ones((L, Hkv, T, T), bool)
            ca_b = np.ones((L, Hkv, C), bool)
        elif spec.pattern == "zeros":
            la_b = np.zeros((L, Hkv, T, T), bool)
            ca_b = np.zeros((L, Hkv, C), bool)
        elif spec.pattern == "la_only":
            la_b = np.ones((L, Hkv, T, T), bool)
            ca_b = np.zeros((L, Hkv, C), bool)
        elif spec.pattern == "ca_only":
            la_b = np.zeros((L, Hkv, T, T), bool)
            ca_b = np.ones((L, Hkv, C), bool)
        else:
            raise ValueError(spec.pattern)
        # only the strictly-lower triangle of an LA block carries meaning; the
        # generator leaves the rest clear so that stored words stay canonical
        la_b = la_b & below
        la[layout.la_off[g]: layout.la_off[g] + L * Hkv * T * W] = _pack_rows(la_b).reshape(-1)
        ca[layout.ca_off[g]: layout.ca_off[g] + L * Hkv * V] = _pack_rows(ca_b).reshape(-1)
    return la, ca


def make_qkv(cfg: Config, layer: int, device="cpu", dist: str = "normal",
             key_growth: float = 2.5):
    """bf16 Q [tokens, Hq, d], K and V [tokens, Hkv, d], N(0,1) from a per-layer seed.

    dist="growing_keys": the same draws, but every key row is multiplied by
    1 + key_growth * (its position inside its prompt // tile), so that a query row's
    largest score grows from one key tile to the next (by about 4 * key_growth in log2
    units at d = 128): inputs that make an online softmax rescale its running sums
    after the first tile, which N(0,1) inputs almost never do.
    """
    import torch
    if dist not in ("normal", "growing_keys"):
        raise ValueError(f"unknown dist {dist!r}")
    T = cfg.total_tokens
    out = []
    for name, H in (("q", cfg.num_q_heads), ("k", cfg.num_kv_heads), ("v", cfg.num_kv_heads)):
        g = torch.Generator(device=device)
        g.manual_seed(seed_for(cfg.name, layer, name))
        x = torch.randn((T, H, cfg.head_dim), generator=g, device=device, dtype=torch.float32)
        if name == "k" and dist == "growing_keys":
            pos = torch.empty(T, dtype=torch.int64)
            cu = np.cumsum([0] + [sum(d) + s for d, s in cfg.prompts])
            for p in range(len(cfg.prompts)):
                pos[cu[p]:cu[p + 1]] = torch.arange(cu[p + 1] - cu[p])
            f = 1.0 + key_growth * (pos // cfg.tile).to(torch.float32)
            x = x * f.to(device).view(T, 1, 1)
        out.append(x.to(torch.bfloat16))
    return tuple(out)

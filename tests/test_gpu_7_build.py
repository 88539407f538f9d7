"""sift_build_bits: the offline LA / CA bit builder against the oracle's fp64 restatement.

SIFT pages (gist.science/it/paper/2606.09441), "Design del Sistema": each document is
prefilled densely on its own once, and the tiles / pages that draw high attention are
stored as LA / CA bits.  The selection rule is this library's reading (top-k tile mass
per LA row, top-k mean received mass for CA, float32 counts, ties to the lower index).

The CUDA builder takes its masses from the bf16 dense kernel, so tiles whose fp64 masses
are nearly equal may be swapped.  The random cases therefore check that every row keeps
exactly the right number of tiles, nothing at or above the diagonal, and a valid top-k
(no kept tile lighter than a dropped one by more than a small tolerance), and that most
rows equal the oracle's bits exactly.  A case with well separated masses must match the
oracle bit for bit, and its bits then drive the online path.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_attention_close, device_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def _bits(word_array, base, n_words, n_bits):
    """bool[n_bits] from n_words little-endian words starting at base."""
    w = np.ascontiguousarray(np.asarray(word_array[base: base + n_words], np.uint64))
    return np.unpackbits(w.view(np.uint8), bitorder="little")[:n_bits].astype(bool)


def _valid_top(sel, mass, k, rel_tol):
    """sel keeps exactly k candidates and none is lighter than a dropped one by more
    than rel_tol of the mean candidate mass."""
    assert int(sel.sum()) == k, (int(sel.sum()), k)
    if 0 < k < len(mass):
        slack = rel_tol * float(np.mean(mass))
        assert mass[sel].min() >= mass[~sel].max() - slack, (mass[sel].min(), mass[~sel].max())


def _doc_tiles(lay):
    return [lay.doc_tiles(g) for g in range(lay.num_docs)]


def _words_host(t):
    return t.cpu().numpy().view(np.uint64)


# (name, prompts, Hq, Hkv, head_dim, tile, la_fraction, ca_fraction, layers, page)
CASES = [
    ("bg_small", [([256, 512, 384], 128)], 4, 2, 128, 128, 0.25, 0.3, 1, 0),
    # a 70-tile document needs two 64-column windows of one-hot values
    ("bg_windows", [([64 * 70, 64 * 20], 64), ([64 * 12], 64)], 4, 1, 64, 64, 0.2, 0.15, 1, 0),
    ("bg_layers", [([512, 256], 128), ([384], 0)], 8, 2, 128, 128, 0.4, 0.5, 3, 0),
    # general layout: ragged documents; 16-token pages (units of 16, three windows for the
    # longest document), 256-token pages (units of one tile), page = tile
    ("bg_rg16", [([700, 301, 129], 77), ([64], 0)], 4, 2, 128, 128, 0.3, 0.2, 1, 16),
    ("bg_rg256", [([900, 301, 129], 5)], 4, 1, 128, 128, 0.3, 0.4, 2, 256),
    ("bg_rg64", [([333, 130], 40)], 2, 1, 64, 64, 0.25, 0.3, 1, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_build_bits_valid_top_and_mostly_exact(sift, case):
    name, prompts, hq, hkv, d, tile, la_f, ca_f, layers, page = case
    cfg = W.custom_config(name, prompts, W.BitSpec(pattern="zeros"), num_layers=layers,
                          num_q_heads=hq, num_kv_heads=hkv, head_dim=d, tile=tile, page=page)
    lay = W.make_layout(cfg)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(np.zeros(lay.la_words_len, np.uint64),
                             np.zeros(lay.ca_words_len, np.uint64))
    tiles = _doc_tiles(lay)
    max_doc_tiles = max(tiles)
    st = prob.new_status()
    rows = exact = 0
    for layer in range(layers):
        q, k, _ = W.make_qkv(cfg, layer, device="cuda")
        sift.build_bits(prob, layer, q, k, max_doc_tiles, la_f, ca_f, la_d, ca_d, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, sift.status_string(int(st.item()))
        la_g, ca_g = _words_host(la_d), _words_host(ca_d)
        la_o, ca_o, masses, scores = oracle.build_bits(lay, layer, q, k, la_f, ca_f)
        for g, T in enumerate(tiles):
            Wd = (T + 63) // 64
            C = lay.doc_pages(g)
            Vd = (C + 63) // 64
            for h in range(hkv):
                M = masses[(g, h)]
                base = int(lay.la_off[g]) + (layer * hkv + h) * T * Wd
                for i in range(T):
                    row = _bits(la_g, base + i * Wd, Wd, 64 * Wd)
                    assert not row[i:].any(), f"{name} g{g} h{h} row {i}: bits at j >= i"
                    _valid_top(row[:i], M[i, :i], oracle.top_count(la_f, i), 2e-2)
                    rows += 1
                    exact += bool(np.array_equal(row, _bits(la_o, base + i * Wd, Wd, 64 * Wd)))
                cbase = int(lay.ca_off[g]) + (layer * hkv + h) * Vd
                cag = _bits(ca_g, cbase, Vd, 64 * Vd)
                assert not cag[C:].any()
                _valid_top(cag[:C], scores[(g, h)], oracle.top_count(ca_f, C), 2e-2)
                rows += 1
                exact += bool(np.array_equal(cag, _bits(ca_o, cbase, Vd, 64 * Vd)))
    assert exact >= 0.9 * rows, f"{name}: only {exact}/{rows} rows equal the oracle's"


def _separated_qk(cfg, lay, seed):
    """Q and K whose tile masses are far apart: the keys of every document tile point along
    one direction a with a tile strength drawn without repetition, and every query is a
    plus small noise, so mass ranks follow the strengths with large margins."""
    gen = torch.Generator().manual_seed(seed)
    T, d = lay.total_tokens, cfg.head_dim
    a = torch.randn(d, generator=gen)
    a = a / a.norm() * (2.0 * d ** 0.5)
    q = a + 0.05 * torch.randn((T, cfg.num_q_heads, d), generator=gen)
    k = 0.05 * torch.randn((T, cfg.num_kv_heads, d), generator=gen)
    for g in range(lay.num_docs):
        s0 = lay.doc_start(g)
        n = (int(lay.doc_end[g]) - s0) // lay.tile
        for h in range(cfg.num_kv_heads):
            strength = torch.randperm(n, generator=gen).float() / max(n - 1, 1)
            for j in range(n):
                k[s0 + j * lay.tile: s0 + (j + 1) * lay.tile, h] += 0.5 * strength[j] * a
    return q.to(torch.bfloat16).cuda(), k.to(torch.bfloat16).cuda()


def test_build_bits_feeds_the_online_path(sift):
    """Well separated masses: the CUDA bits equal the oracle's bit for bit; decode + sparse
    prefill on them then match the oracle's attention on the oracle's own bits."""
    cfg = W.custom_config("bg_online", [([512, 768], 128), ([640], 256)],
                          W.BitSpec(pattern="zeros"), num_layers=2, num_q_heads=4,
                          num_kv_heads=2, head_dim=128, tile=128)
    lay = W.make_layout(cfg)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(np.zeros(lay.la_words_len, np.uint64),
                             np.zeros(lay.ca_words_len, np.uint64))
    la_o = np.zeros(lay.la_words_len, np.uint64)
    ca_o = np.zeros(lay.ca_words_len, np.uint64)
    st = prob.new_status()
    qk = []
    for layer in range(cfg.num_layers):
        q, k = _separated_qk(cfg, lay, 100 + layer)
        qk.append((q, k))
        sift.build_bits(prob, layer, q, k, max(_doc_tiles(lay)), 0.3, 0.4, la_d, ca_d,
                        dev_status=st)
        la_l, ca_l, _, _ = oracle.build_bits(lay, layer, q, k, 0.3, 0.4)
        la_o |= la_l
        ca_o |= ca_l
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    assert np.array_equal(_words_host(la_d)[:lay.la_words_len], la_o)
    assert np.array_equal(_words_host(ca_d)[:lay.ca_words_len], ca_o)
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    for layer, (q, k) in enumerate(qk):
        _, _, v = W.make_qkv(cfg, layer, device="cuda")
        o, lse = sift.sparse_prefill(prob, layer, q, k, v, kv, cnt, sched, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        O, LSE = oracle.attention_all(lay, la_o, ca_o, layer, q, k, v)
        assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                               f"layer {layer}")


def test_build_bits_rejects_bad_arguments(sift):
    cfg = W.custom_config("bg_args", [([256], 128)], W.BitSpec(pattern="zeros"),
                          num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128)
    lay = W.make_layout(cfg)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(np.zeros(lay.la_words_len, np.uint64),
                             np.zeros(lay.ca_words_len, np.uint64))
    q, k, _ = W.make_qkv(cfg, 0, device="cuda")
    for layer, mdt, la_f, ca_f in ((1, 2, 0.5, 0.5), (0, 0, 0.5, 0.5), (0, 2, 1.5, 0.5),
                                   (0, 2, 0.5, -0.1), (0, 99, 0.5, 0.5)):
        with pytest.raises(sift.SiftError):
            sift.build_bits(prob, layer, q, k, mdt, la_f, ca_f, la_d, ca_d)


def _separated_qk_pages(cfg, lay, seed, unit):
    """As _separated_qk, with a distinct strength for every `unit`-token block of each
    document (so page scores, not only tile masses, are far apart)."""
    gen = torch.Generator().manual_seed(seed)
    T, d = lay.total_tokens, cfg.head_dim
    a = torch.randn(d, generator=gen)
    a = a / a.norm() * (2.0 * d ** 0.5)
    q = a + 0.05 * torch.randn((T, cfg.num_q_heads, d), generator=gen)
    k = 0.05 * torch.randn((T, cfg.num_kv_heads, d), generator=gen)
    for g in range(lay.num_docs):
        s0, e0 = lay.doc_start(g), int(lay.doc_end[g])
        nb = -(-(e0 - s0) // unit)
        for h in range(cfg.num_kv_heads):
            strength = torch.randperm(nb, generator=gen).float() / max(nb - 1, 1)
            for j in range(nb):
                k[s0 + j * unit: min(s0 + (j + 1) * unit, e0), h] += 0.5 * strength[j] * a
    return q.to(torch.bfloat16).cuda(), k.to(torch.bfloat16).cuda()


def test_build_bits_general_layout_feeds_the_online_path(sift):
    """Ragged documents, 16-token pages: the CUDA bits equal the oracle's bit for bit on
    well separated masses, and the general-layout decode + prefill (pages gathered) on them
    match the oracle's attention on the oracle's own bits."""
    cfg = W.custom_config("bg_online_rg", [([300, 411, 200], 77)], W.BitSpec(pattern="zeros"),
                          num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128,
                          page=16)
    lay = W.make_layout(cfg)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(np.zeros(lay.la_words_len, np.uint64),
                             np.zeros(lay.ca_words_len, np.uint64))
    q, k = _separated_qk_pages(cfg, lay, 7, 16)
    st = prob.new_status()
    sift.build_bits(prob, 0, q, k, max(_doc_tiles(lay)), 0.3, 0.1, la_d, ca_d, dev_status=st)
    la_o, ca_o, _, _ = oracle.build_bits(lay, 0, q, k, 0.3, 0.1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    assert np.array_equal(_words_host(la_d)[:lay.la_words_len], la_o)
    assert np.array_equal(_words_host(ca_d)[:lay.ca_words_len], ca_o)
    lists = sift.decode_ragged(prob, la_d, ca_d, dev_status=st)
    _, _, v = W.make_qkv(cfg, 0, device="cuda")
    o, lse = sift.sparse_prefill_ragged(prob, 0, q, k, v, *lists, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O, LSE = oracle.attention_all(lay, la_o, ca_o, 0, q, k, v)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                           "general layout")

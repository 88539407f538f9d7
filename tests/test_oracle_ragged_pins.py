"""Pins for the oracle's general layout: documents of any length (tiles and pages
counted from each document's first token, the last ones partial) and a CA page size
that differs from the LA tile.

* a hand-derived ragged decode fixture (tests/golden/decode_ragged_small.json);
* three routes to one key set: the decoded (first token, info) lists expanded to
  tokens, the C key_visible() rule, and a block-wise numpy token mask;
* the aligned layout as a special case of the ragged decode;
* page-size semantics on single planted CA bits;
* attention: special cases against torch SDPA (fp64) with masks written from the
  plain description, and the numpy dense-mask brute force.

SIFT pages: gist.science/it/paper/2606.09441, "Design del Sistema" (LA flags tiles
of a document's own attention matrix, CA flags KV pages that later documents
attend to) and "Dettagli di Implementazione" (bits decoded into tile indices).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import expand_lists

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "decode_ragged_small.json")) as f:
        g = json.load(f)
    lay = W.Layout(num_prompts=2, num_docs=3, num_layers=g["num_layers"], num_q_heads=2,
                   num_kv_heads=g["num_kv_heads"], head_dim=8, tile=g["tile"],
                   total_tokens=g["cu_seqlens"][-1], max_tiles_per_prompt=6,
                   cu_seqlens=np.array(g["cu_seqlens"], np.int32),
                   doc_cu=np.array(g["doc_cu"], np.int32),
                   doc_end=np.array(g["doc_end"], np.int32),
                   la_off=np.array(g["la_off"], np.int64), ca_off=np.array(g["ca_off"], np.int64),
                   la_words_len=len(g["la_words"]), ca_words_len=len(g["ca_words"]),
                   page=g["page"])
    return g, lay, np.array(g["la_words"], np.uint64), np.array(g["ca_words"], np.uint64)


def test_ragged_golden_fixture():
    g, lay, la, ca = _golden()
    qt, kv, cnt, pg = oracle.decode_ragged(lay, la, ca)
    assert qt.tolist() == g["expected_qtiles"]
    for q, row in enumerate(g["expected_rows"]):
        assert cnt[0, 0, q] == len(row), q
        assert kv[0, 0, q, :len(row)].tolist() == row, q
    # and the fixture's lists are the key set of the token rule
    T = lay.total_tokens
    tok = np.arange(T)
    assert np.array_equal(expand_lists(lay, qt, kv, cnt, pg, 0, 0),
                          oracle.key_mask(lay, la, ca, 0, 0, tok, tok))


def _golden_gather():
    with open(os.path.join(GOLDEN, "decode_gather_small.json")) as f:
        g = json.load(f)
    lay = W.Layout(num_prompts=1, num_docs=3, num_layers=1, num_q_heads=2, num_kv_heads=1,
                   head_dim=8, tile=g["tile"], total_tokens=g["cu_seqlens"][-1],
                   max_tiles_per_prompt=6, cu_seqlens=np.array(g["cu_seqlens"], np.int32),
                   doc_cu=np.array(g["doc_cu"], np.int32),
                   doc_end=np.array(g["doc_end"], np.int32),
                   la_off=np.array(g["la_off"], np.int64), ca_off=np.array(g["ca_off"], np.int64),
                   la_words_len=len(g["la_words"]), ca_words_len=len(g["ca_words"]),
                   page=g["page"])
    return g, lay, np.array(g["la_words"], np.uint64), np.array(g["ca_words"], np.uint64)


def test_gathered_pages_golden_fixture():
    g, lay, la, ca = _golden_gather()
    qt, kv, cnt, pg = oracle.decode_ragged(lay, la, ca, page_cap=g["page_cap"])
    assert qt.tolist() == g["expected_qtiles"]
    for q, row in enumerate(g["expected_rows"]):
        assert cnt[0, 0, q] == len(row), q
        assert kv[0, 0, q, :len(row)].tolist() == row, q
    assert pg[0, 0].tolist() == g["expected_pages"]
    tok = np.arange(lay.total_tokens)
    assert np.array_equal(expand_lists(lay, qt, kv, cnt, pg, 0, 0),
                          oracle.key_mask(lay, la, ca, 0, 0, tok, tok))


RAGGED_CFGS = [
    # tile 16, page 8 (2 pages per tile); odd documents, odd suffix, empty suffix,
    # a suffix-only prompt
    W.custom_config("rg_p8", [([6 * 16 + 5, 16 * 3, 7], 9), ([33], 0), ([], 21)],
                    W.BitSpec(la_p=0.4, ca_p=0.5), num_layers=2, num_q_heads=4,
                    num_kv_heads=2, head_dim=8, tile=16, page=8),
    # tile 16, page 4 (4 pages per tile), one-token documents
    W.custom_config("rg_p4", [([1, 17, 40, 1], 3), ([5, 5], 16)],
                    W.BitSpec(la_p=0.5, ca_p=0.3, la_window=1, ca_first_page=True),
                    num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=8, tile=16, page=4),
    # page = tile (ragged lengths only)
    W.custom_config("rg_eq", [([50, 31, 64], 1)], W.BitSpec(la_p=0.3, ca_p=0.6),
                    num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=8, tile=16),
    # page = 2 and 4 tiles; documents longer than 64 tiles (two LA words per row)
    W.custom_config("rg_p32", [([16 * 70 + 3, 45], 10)], W.BitSpec(la_p=0.1, ca_p=0.5),
                    num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=4, tile=16, page=32),
    W.custom_config("rg_p64", [([200, 130, 64], 0), ([77], 5)],
                    W.BitSpec(head_density=(0.1, 0.7)), num_layers=2, num_q_heads=4,
                    num_kv_heads=2, head_dim=4, tile=16, page=64),
    # many tiny documents with gathered pages: more partial pages than whole tiles
    W.custom_config("rg_tiny", [([17] * 20, 0), ([1, 2, 3, 17, 33], 5)],
                    W.BitSpec(la_p=0.5, ca_p=0.7), num_q_heads=2, num_kv_heads=1, head_dim=4,
                    tile=128, page=16),
    # 65 pages (8 * 64 + 3 tokens): the CA block of each (layer, head) takes two words
    W.custom_config("rg_cross", [([8 * 64 + 3, 20], 4)], W.BitSpec(la_p=0.2, ca_p=0.5),
                    num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=4, tile=16, page=8),
]


@pytest.mark.parametrize("cfg", RAGGED_CFGS, ids=lambda c: c.name)
def test_ragged_lists_token_rule_and_numpy_mask_agree(cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    assert not lay.aligned or cfg.name == "rg_eq"
    qt, kv, cnt, pg = oracle.decode_ragged(lay, la, ca)
    T, B = lay.total_tokens, lay.tile
    tok = np.arange(T)
    # query tiles: every segment cut from its own start, in token order
    exp = []
    for s0, e0, _ in lay.segments():
        exp += [[x, min(B, e0 - x)] for x in range(s0, e0, B)]
    assert qt.tolist() == exp
    for l in range(lay.num_layers):
        for h in range(lay.num_kv_heads):
            A = expand_lists(lay, qt, kv, cnt, pg, l, h)
            Bm = oracle.key_mask(lay, la, ca, l, h, tok, tok)
            C = oracle.token_mask(lay, la, ca, l, h)
            assert np.array_equal(A, Bm), (l, h)
            assert np.array_equal(Bm, C), (l, h)
            for q, (x, rows) in enumerate(qt):
                ent = kv[l, h, q, :cnt[l, h, q]]
                plain = ent[(ent[:, 1] >> 9) & 1 == 0, 0]
                assert np.all(np.diff(plain[:-1]) > 0) if len(plain) > 2 else True
                firsts = ent[:, 0]
                assert firsts[-1] == x and (kv[l, h, q, cnt[l, h, q] - 1, 1] >> 8) & 1 == 1
                assert np.all((kv[l, h, q, :cnt[l, h, q] - 1, 1] >> 8) & 1 == 0)


@pytest.mark.parametrize("name", ["pin_a", "pin_b", "pin_skew"])
def test_ragged_decode_reduces_to_aligned_decode(name):
    """With page == tile and every boundary a multiple of the tile, the ragged lists are
    the aligned lists: first token = global tile index * tile, full tiles, causal last."""
    cfgs = {
        "pin_a": W.custom_config("pin_a", [([256, 512, 128], 128)], W.BitSpec(la_p=0.3, ca_p=0.4),
                                 num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                                 tile=64),
        "pin_b": W.custom_config("pin_b", [([128, 64], 64), ([192], 0), ([], 128)],
                                 W.BitSpec(la_p=0.5, ca_p=0.5, la_window=1, ca_first_page=True),
                                 num_layers=1, num_q_heads=6, num_kv_heads=3, head_dim=8,
                                 tile=64),
        "pin_skew": W.custom_config("pin_skew", [([512] * 4, 64)],
                                    W.BitSpec(head_density=(0.05, 0.6)), num_layers=3,
                                    num_q_heads=4, num_kv_heads=2, head_dim=8, tile=64),
    }
    cfg = cfgs[name]
    lay = W.make_layout(cfg)
    assert lay.aligned
    la, ca = W.make_bits(cfg, lay)
    kv_a, cnt_a = oracle.decode(lay, la, ca)
    qt, kv_r, cnt_r, _ = oracle.decode_ragged(lay, la, ca)
    B = lay.tile
    assert qt.tolist() == [[i * B, B] for i in range(lay.num_tiles)]
    assert np.array_equal(cnt_a, cnt_r)
    full = B | (1 << 16)
    for l in range(lay.num_layers):
        for h in range(lay.num_kv_heads):
            for i in range(lay.num_tiles):
                n = cnt_a[l, h, i]
                assert np.array_equal(kv_r[l, h, i, :n, 0], kv_a[l, h, i, :n] * B)
                info = kv_r[l, h, i, :n, 1]
                assert np.all(info[:-1] == full) and info[-1] == full | (1 << 8)


@pytest.mark.parametrize("page,tile", [(32, 8), (4, 16), (8, 8), (2, 16), (8, 16), (16, 64)])
def test_single_ca_bit_covers_exactly_its_page(page, tile):
    """One CA bit of the first document admits exactly the keys of its page -- tokens
    [j*page, (j+1)*page) of that document, cut at the document's end -- to every query
    of the second document, whatever the tile size."""
    n0 = 3 * page + page // 2 + 1          # a partial last page
    cfg = W.custom_config("pg", [([n0, 2 * tile + 3], 0)], W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=4, tile=tile, page=page)
    lay = W.make_layout(cfg)
    C = lay.doc_pages(0)
    for j in range(C):
        la = np.zeros(lay.la_words_len, np.uint64)
        ca = np.zeros(lay.ca_words_len, np.uint64)
        ca[lay.ca_off[0]] = np.uint64(1 << j)
        q = np.arange(n0, lay.total_tokens)
        M = oracle.key_mask(lay, la, ca, 0, 0, q, np.arange(n0))
        want = np.zeros(n0, bool)
        want[j * page: min((j + 1) * page, n0)] = True
        assert np.all(M == want[None, :]), (page, tile, j)
        qt, kv, cnt, pg = oracle.decode_ragged(lay, la, ca)
        A = expand_lists(lay, qt, kv, cnt, pg, 0, 0)
        assert np.array_equal(A[n0:, :n0], np.broadcast_to(want, (len(q), n0)))


def test_ragged_decode_rejects_pages_that_do_not_nest():
    cfg = W.custom_config("bad", [([40], 8)], W.BitSpec(pattern="ones"), num_q_heads=2,
                          num_kv_heads=1, head_dim=4, tile=16, page=12)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    with pytest.raises(ValueError):
        oracle.decode_ragged(lay, la, ca)
    cfg = W.custom_config("bad2", [([40], 8)], W.BitSpec(pattern="ones"), num_q_heads=2,
                          num_kv_heads=1, head_dim=4, tile=64, page=2)   # 32 pages per tile
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    with pytest.raises(ValueError):
        oracle.decode_ragged(lay, la, ca)


# ---- attention on ragged layouts ---------------------------------------------------

def _qkv(cfg, seed=0):
    return W.make_qkv(cfg, seed)


def _sdpa(q, k, v, mask, scale):
    """fp64 SDPA per query head with kv head qh // G; mask [T, T] bool."""
    qf, kf, vf = (t.double() for t in (q, k, v))
    G = q.shape[1] // k.shape[1]
    out = torch.zeros_like(qf)
    for qh in range(q.shape[1]):
        h = qh // G
        out[:, qh] = torch.nn.functional.scaled_dot_product_attention(
            qf[None, None, :, qh], kf[None, None, :, h], vf[None, None, :, h],
            attn_mask=torch.from_numpy(mask)[None, None], scale=scale)[0, 0]
    return out.numpy()


RG_ATT = W.custom_config("rg_att", [([37, 16 * 2 + 9, 5], 11), ([23], 0), ([], 19)],
                         W.BitSpec(la_p=0.5, ca_p=0.5), num_q_heads=4, num_kv_heads=2,
                         head_dim=8, tile=16, page=8)


def _prompt_causal(lay):
    T = lay.total_tokens
    M = np.zeros((T, T), bool)
    for p in range(lay.num_prompts):
        a, b = int(lay.cu_seqlens[p]), int(lay.cu_seqlens[p + 1])
        M[a:b, a:b] = np.tril(np.ones((b - a, b - a), bool))
    return M


def test_ragged_all_ones_is_dense_causal_per_prompt():
    cfg = W.custom_config("rg_ones", RG_ATT.prompts, W.BitSpec(pattern="ones"), num_q_heads=4,
                          num_kv_heads=2, head_dim=8, tile=16, page=8)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    q, k, v = _qkv(cfg)
    O, _ = oracle.attention_all(lay, la, ca, 0, q, k, v, scale=0.3)
    ref = _sdpa(q, k, v, _prompt_causal(lay), 0.3)
    np.testing.assert_allclose(O, ref, atol=1e-12)


def test_ragged_all_zeros_is_own_document_tile_plus_dense_suffix():
    """No bits: a document token sees the causal keys of its own document tile (tiles cut
    from the document start), a suffix token its whole prompt."""
    cfg = W.custom_config("rg_zero", RG_ATT.prompts, W.BitSpec(pattern="zeros"), num_q_heads=4,
                          num_kv_heads=2, head_dim=8, tile=16, page=8)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    q, k, v = _qkv(cfg)
    T, B = lay.total_tokens, lay.tile
    M = np.zeros((T, T), bool)
    for s0, e0, g in lay.segments():
        for t in range(s0, e0):
            if g < 0:
                p = int(np.searchsorted(lay.cu_seqlens, t, side="right")) - 1
                M[t, int(lay.cu_seqlens[p]): t + 1] = True
            else:
                M[t, s0 + (t - s0) // B * B: t + 1] = True
    O, _ = oracle.attention_all(lay, la, ca, 0, q, k, v)
    ref = _sdpa(q, k, v, M, 1.0 / np.sqrt(8))
    np.testing.assert_allclose(O, ref, atol=1e-12)


def test_ragged_random_bits_match_numpy_brute_force():
    lay = W.make_layout(RG_ATT)
    la, ca = W.make_bits(RG_ATT, lay)
    q, k, v = _qkv(RG_ATT)
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    Ob, LSEb = oracle.brute_force_attention(lay, la, ca, 0, q, k, v)
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_allclose(LSE, LSEb, atol=1e-12)


# ---- the offline bit builder on the general layout -------------------------------------

def test_builder_general_row_sums_and_second_route():
    """Ragged documents, 8-token pages under 16-token tiles: each query tile's masses sum to
    G x its rows, and the unit masses equal the oracle's own attention rows with one-hot
    unit indicators as V (document alone)."""
    cfg = W.custom_config("bb_rg", [([37, 50], 5)], W.BitSpec(pattern="zeros"), num_q_heads=2,
                          num_kv_heads=1, head_dim=8, tile=16, page=8)
    lay = W.make_layout(cfg)
    q, k, _ = W.make_qkv(cfg, 0)
    _, _, masses, scores = oracle.build_bits(lay, 0, q, k, 0.5, 0.5, scale=0.3)
    for g in range(lay.num_docs):
        s0, e0 = lay.doc_start(g), int(lay.doc_end[g])
        n = e0 - s0
        T = -(-n // 16)
        rows = np.array([min(16, n - 16 * i) for i in range(T)])
        np.testing.assert_allclose(masses[(g, 0)].sum(axis=1), 2 * rows, rtol=1e-12)
        # second route: attention rows of the document alone with V = unit indicators
        nu = -(-n // 8)
        sub = W.Layout(num_prompts=1, num_docs=0, num_layers=1, num_q_heads=2, num_kv_heads=1,
                       head_dim=8, tile=16, total_tokens=n, max_tiles_per_prompt=T,
                       cu_seqlens=np.array([0, n], np.int32), doc_cu=np.array([0, 0], np.int32),
                       doc_end=np.zeros(0, np.int32), la_off=np.zeros(0, np.int64),
                       ca_off=np.zeros(0, np.int64), la_words_len=0, ca_words_len=0)
        onehot = torch.zeros((n, 1, 8))
        onehot[torch.arange(n), 0, torch.arange(n) // 8] = 1.0
        tok = np.repeat(np.arange(n, dtype=np.int32), 2)
        head = np.tile(np.arange(2, dtype=np.int32), n)
        o, _ = oracle.attention_rows(sub, np.zeros(0, np.uint64), np.zeros(0, np.uint64), 0,
                                     q[s0:e0], k[s0:e0], onehot.to(torch.bfloat16), tok, head,
                                     scale=0.3)
        per_unit = o.reshape(n, 2, 8).sum(axis=1)[:, :nu]          # [token, unit]
        Mu = np.add.reduceat(per_unit, np.arange(0, n, 16), axis=0)  # [query tile, unit]
        M2 = np.zeros((T, T))
        for u in range(nu):
            M2[:, (8 * u) // 16] += Mu[:, u]
        np.testing.assert_allclose(masses[(g, 0)], M2, atol=1e-10)


@pytest.mark.parametrize("page,tile,hot", [(8, 16, 5), (256, 128, 1), (16, 16, 3)])
def test_builder_general_planted_hot_page(page, tile, hot):
    """Keys of one page aligned with every query draw almost all the mass: it is the only
    page CA keeps at a one-page budget, and LA rows after its tiles keep a tile of it."""
    n = 6 * max(page, tile) + 3                       # a partial last page and tile
    cfg = W.custom_config("bb_hot_rg", [([n], 0)], W.BitSpec(pattern="zeros"), num_q_heads=2,
                          num_kv_heads=1, head_dim=16, tile=tile, page=page)
    lay = W.make_layout(cfg)
    gen = torch.Generator().manual_seed(11)
    a = torch.randn(16, generator=gen)
    q = (a + 0.05 * torch.randn((n, 2, 16), generator=gen)).to(torch.bfloat16)
    k = (0.05 * torch.randn((n, 1, 16), generator=gen)).to(torch.bfloat16)
    k[hot * page: (hot + 1) * page, 0] = (2.0 * a).to(torch.bfloat16)
    C = lay.doc_pages(0)
    la, ca, masses, scores = oracle.build_bits(lay, 0, q, k, 1e-3, 1.0 / C, scale=1.0)
    assert np.argmax(scores[(0, 0)]) == hot
    V = -(-C // 64)
    cab = np.unpackbits(ca[:V].view(np.uint8), bitorder="little")[:C]
    assert cab.sum() == 1 and cab[hot] == 1
    T = lay.doc_tiles(0)
    hot_tiles = set(range((hot * page) // tile, ((hot + 1) * page - 1) // tile + 1))
    W_ = -(-T // 64)
    for i in range(max(hot_tiles) + 1, T):   # one kept tile per row (ceil(1e-3 * i) = 1)
        row = np.unpackbits(la[i * W_: (i + 1) * W_].view(np.uint8), bitorder="little")[:T]
        assert row.sum() == 1 and int(np.nonzero(row)[0][0]) in hot_tiles, (i, row)


def test_builder_general_counts_follow_the_fractions():
    cfg = W.custom_config("bb_cnt_rg", [([16 * 9 + 5, 40], 7)], W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=8, tile=16, page=8)
    lay = W.make_layout(cfg)
    q, k, _ = W.make_qkv(cfg, 0)
    la, ca, _, _ = oracle.build_bits(lay, 0, q, k, 0.3, 0.25)
    for g in range(lay.num_docs):
        T, C = lay.doc_tiles(g), lay.doc_pages(g)
        W_, V = -(-T // 64), -(-C // 64)
        for i in range(T):
            w = la[lay.la_off[g] + i * W_: lay.la_off[g] + (i + 1) * W_]
            assert int(sum(bin(int(x)).count("1") for x in w)) == int(np.ceil(0.3 * i - 1e-4))
        w = ca[lay.ca_off[g]: lay.ca_off[g] + V]
        assert int(sum(bin(int(x)).count("1") for x in w)) == int(np.ceil(0.25 * C - 1e-4))

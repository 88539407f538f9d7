"""Pins for the CPU oracle: checks against things other than the oracle itself.

* a hand-derived decode fixture (tests/golden/decode_small.json);
* popcount identities computed with Python integers;
* special cases that reduce to a library routine (torch SDPA, fp64, CPU) with a
  mask written from the plain description of the case;
* closed forms (first token of a prompt, constant V, a two-token hand example);
* a dense-mask numpy brute force on tiny random inputs.

SIFT pages: gist.science/it/paper/2606.09441, "Design del Sistema" (flagged
tiles/pages computed, the rest skipped) and "Dettagli di Implementazione"
(bits decoded into explicit tile indices).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_layout():
    with open(os.path.join(GOLDEN, "decode_small.json")) as f:
        g = json.load(f)
    lay = W.Layout(num_prompts=2, num_docs=3, num_layers=g["num_layers"], num_q_heads=2,
                   num_kv_heads=g["num_kv_heads"], head_dim=8, tile=g["tile"],
                   total_tokens=g["cu_seqlens"][-1], max_tiles_per_prompt=6,
                   cu_seqlens=np.array(g["cu_seqlens"], np.int32),
                   doc_cu=np.array(g["doc_cu"], np.int32),
                   doc_end=np.array(g["doc_end"], np.int32),
                   la_off=np.array(g["la_off"], np.int64), ca_off=np.array(g["ca_off"], np.int64),
                   la_words_len=len(g["la_words"]), ca_words_len=len(g["ca_words"]))
    return g, lay, np.array(g["la_words"], np.uint64), np.array(g["ca_words"], np.uint64)


def test_decode_golden_fixture():
    g, lay, la, ca = _golden_layout()
    kv, cnt = oracle.decode(lay, la, ca)
    for l in range(2):
        for h in range(2):
            exp = g["expected"][f"l{l}h{h}"]
            for i, row in enumerate(exp):
                assert cnt[l, h, i] == len(row), (l, h, i)
                assert list(kv[l, h, i, :len(row)]) == row, (l, h, i)


SMALL_CFGS = [
    W.custom_config("pin_a", [([256, 512, 128], 128)], W.BitSpec(la_p=0.3, ca_p=0.4),
                    num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=16, tile=64),
    W.custom_config("pin_b", [([128, 64], 64), ([192], 0), ([], 128)],
                    W.BitSpec(la_p=0.5, ca_p=0.5, la_window=1, ca_first_page=True),
                    num_layers=1, num_q_heads=6, num_kv_heads=3, head_dim=8, tile=64),
    # documents longer than 64 tiles: rows span two LA words, CA spans two words
    W.custom_config("pin_wide", [([4 * 130, 4 * 70], 8)], W.BitSpec(la_p=0.1, ca_p=0.2),
                    num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=4, tile=4),
    W.custom_config("pin_skew", [([512] * 4, 64)], W.BitSpec(head_density=(0.05, 0.6)),
                    num_layers=3, num_q_heads=4, num_kv_heads=2, head_dim=8, tile=64),
]


@pytest.mark.parametrize("cfg", SMALL_CFGS, ids=lambda c: c.name)
def test_decode_popcount_identity_and_order(cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    kv, cnt = oracle.decode(lay, la, ca)
    B = lay.tile
    for l in range(lay.num_layers):
        for h in range(lay.num_kv_heads):
            for p in range(lay.num_prompts):
                p0 = int(lay.cu_seqlens[p]) // B
                p1 = int(lay.cu_seqlens[p + 1]) // B
                docs = list(range(lay.doc_cu[p], lay.doc_cu[p + 1]))
                for i in range(p0, p1):
                    row = kv[l, h, i, :cnt[l, h, i]]
                    # lists: strictly increasing, inside the prompt, diagonal last
                    assert row[-1] == i and np.all(np.diff(row) > 0) and row[0] >= p0
                    owner = [g for g in docs if lay.doc_start(g) // B <= i < lay.doc_end[g] // B]
                    if not owner:
                        assert cnt[l, h, i] == i - p0 + 1
                        continue
                    g = owner[0]
                    expect = 1
                    for gp in docs:
                        T = lay.doc_tiles(gp)
                        Wd = (T + 63) // 64
                        if gp < g:
                            base = lay.ca_off[gp] + (l * lay.num_kv_heads + h) * Wd
                            val = sum(int(ca[base + w]) << (64 * w) for w in range(Wd))
                            expect += (val & ((1 << T) - 1)).bit_count()
                    T = lay.doc_tiles(g)
                    Wd = (T + 63) // 64
                    il = i - lay.doc_start(g) // B
                    base = lay.la_off[g] + ((l * lay.num_kv_heads + h) * T + il) * Wd
                    val = sum(int(la[base + w]) << (64 * w) for w in range(Wd))
                    expect += (val & ((1 << il) - 1)).bit_count()
                    assert cnt[l, h, i] == expect, (l, h, i)


@pytest.mark.parametrize("cfg", SMALL_CFGS, ids=lambda c: c.name)
def test_decode_matches_tile_mask_and_token_mask(cfg):
    """Decoded lists == numpy tile mask rows == oracle token mask (three routes)."""
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    kv, cnt = oracle.decode(lay, la, ca)
    B, N = lay.tile, lay.num_tiles
    for l in range(lay.num_layers):
        for h in range(lay.num_kv_heads):
            M = oracle.tile_mask(lay, la, ca, l, h)
            for i in range(N):
                assert list(np.nonzero(M[i])[0]) == list(kv[l, h, i, :cnt[l, h, i]])
            # token route, on the first and last token of each tile
            toks = np.array(sorted({t for i in range(N) for t in (i * B, i * B + B - 1)}))
            keys = np.arange(lay.total_tokens)
            TM = oracle.key_mask(lay, la, ca, l, h, toks, keys)
            for a, t in enumerate(toks):
                expect = np.kron(M[t // B], np.ones(B, bool)) & (keys <= t)
                assert np.array_equal(TM[a], expect), (l, h, t)


def _sdpa_ref(q, k, v, mask, scale):
    """torch SDPA (fp64, CPU) for one prompt; mask [Tq, Tk] bool (True = keep) or 'causal'."""
    G = q.shape[1] // k.shape[1]
    qd = q.double().permute(1, 0, 2)
    kd = k.double().repeat_interleave(G, dim=1).permute(1, 0, 2)
    vd = v.double().repeat_interleave(G, dim=1).permute(1, 0, 2)
    if isinstance(mask, str):
        o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=True,
                                                             scale=scale)
        s = (qd @ kd.transpose(1, 2)) * scale
        s = s.masked_fill(~torch.tril(torch.ones(s.shape[-2:], dtype=torch.bool)), -math.inf)
    else:
        mt = torch.as_tensor(mask)
        o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mt,
                                                             scale=scale)
        s = ((qd @ kd.transpose(1, 2)) * scale).masked_fill(~mt, -math.inf)
    lse = torch.logsumexp(s, dim=-1)  # [H, T]
    return o.permute(1, 0, 2).numpy(), lse.numpy()


def _pattern_cfg(pattern, prompts=(([128, 192, 64], 64), ([64, 128], 128)), Hq=4, Hkv=2, d=16,
                 B=64):
    return W.custom_config(f"pin_{pattern}", list(prompts), W.BitSpec(pattern=pattern),
                           num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, tile=B)


def _oracle_all(cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    q, k, v = W.make_qkv(cfg, 0)
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    return lay, la, ca, q, k, v, O, LSE


def _doc_spans(lay, p):
    return [(lay.doc_start(g), int(lay.doc_end[g])) for g in range(lay.doc_cu[p], lay.doc_cu[p + 1])]


def test_all_ones_equals_dense_causal_sdpa():
    cfg = _pattern_cfg("ones")
    lay, la, ca, q, k, v, O, LSE = _oracle_all(cfg)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    for p in range(lay.num_prompts):
        a, b = int(lay.cu_seqlens[p]), int(lay.cu_seqlens[p + 1])
        o_ref, lse_ref = _sdpa_ref(q[a:b], k[a:b], v[a:b], "causal", scale)
        np.testing.assert_allclose(O[a:b], o_ref, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, a:b], lse_ref, atol=1e-12, rtol=0)


def test_la_only_equals_per_document_causal():
    """LA all ones, CA all zeros: doc rows = causal attention inside their own document;
    suffix rows = causal attention over the whole prompt."""
    cfg = _pattern_cfg("la_only")
    lay, la, ca, q, k, v, O, LSE = _oracle_all(cfg)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    for p in range(lay.num_prompts):
        a, b = int(lay.cu_seqlens[p]), int(lay.cu_seqlens[p + 1])
        for s, e in _doc_spans(lay, p):
            o_ref, lse_ref = _sdpa_ref(q[s:e], k[s:e], v[s:e], "causal", scale)
            np.testing.assert_allclose(O[s:e], o_ref, atol=1e-12, rtol=0)
            np.testing.assert_allclose(LSE[:, s:e], lse_ref, atol=1e-12, rtol=0)
        suf = _doc_spans(lay, p)[-1][1] if _doc_spans(lay, p) else a
        o_ref, lse_ref = _sdpa_ref(q[a:b], k[a:b], v[a:b], "causal", scale)
        np.testing.assert_allclose(O[suf:b], o_ref[suf - a:], atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, suf:b], lse_ref[:, suf - a:], atol=1e-12, rtol=0)


def test_all_zeros_is_block_diagonal_causal():
    """No bits: each document row sees only its own tile (causally)."""
    cfg = _pattern_cfg("zeros")
    lay, la, ca, q, k, v, O, LSE = _oracle_all(cfg)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    B = lay.tile
    for p in range(lay.num_prompts):
        for s, e in _doc_spans(lay, p):
            for t0 in range(s, e, B):
                o_ref, lse_ref = _sdpa_ref(q[t0:t0 + B], k[t0:t0 + B], v[t0:t0 + B], "causal",
                                           scale)
                np.testing.assert_allclose(O[t0:t0 + B], o_ref, atol=1e-12, rtol=0)
                np.testing.assert_allclose(LSE[:, t0:t0 + B], lse_ref, atol=1e-12, rtol=0)


def test_ca_only_sees_earlier_documents_and_own_tile():
    """LA zeros, CA ones: a document row sees every token of the earlier documents of its
    prompt plus its own tile causally; nothing else of its own document."""
    cfg = _pattern_cfg("ca_only")
    lay, la, ca, q, k, v, O, LSE = _oracle_all(cfg)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    B = lay.tile
    for p in range(lay.num_prompts):
        a, b = int(lay.cu_seqlens[p]), int(lay.cu_seqlens[p + 1])
        n = b - a
        mask = np.zeros((n, n), bool)
        for s, e in _doc_spans(lay, p):
            for t in range(s, e):
                mask[t - a, :s - a] = True                      # all earlier documents
                t0 = t - (t - a) % B
                mask[t - a, t0 - a:t - a + 1] = True            # own tile, causal
        suf = _doc_spans(lay, p)[-1][1] if _doc_spans(lay, p) else a
        for t in range(suf, b):
            mask[t - a, :t - a + 1] = True
        o_ref, lse_ref = _sdpa_ref(q[a:b], k[a:b], v[a:b], mask, scale)
        np.testing.assert_allclose(O[a:b], o_ref, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE[:, a:b], lse_ref, atol=1e-12, rtol=0)


def test_closed_forms_first_token_and_constant_v():
    cfg = W.custom_config("pin_closed", [([128, 64], 64), ([64], 0)],
                          W.BitSpec(la_p=0.5, ca_p=0.5), num_q_heads=4, num_kv_heads=2,
                          head_dim=16, tile=64)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    q, k, _ = W.make_qkv(cfg, 0)
    # V constant per (kv head, channel): every row's output equals that constant
    vc = torch.arange(cfg.num_kv_heads * cfg.head_dim, dtype=torch.float32)
    vc = (vc.reshape(1, cfg.num_kv_heads, cfg.head_dim) / 8 - 3).to(torch.bfloat16)
    v = vc.expand(cfg.total_tokens, -1, -1).contiguous()
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    G = cfg.num_q_heads // cfg.num_kv_heads
    for qh in range(cfg.num_q_heads):
        np.testing.assert_allclose(O[:, qh, :], np.broadcast_to(vc[0, qh // G].double().numpy(),
                                                                 O[:, qh, :].shape),
                                   rtol=0, atol=1e-12)
    # first token of each prompt: o = v_0 and lse = scale * <q_0, k_0>
    _, _, v = W.make_qkv(cfg, 0)
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    for p in range(lay.num_prompts):
        t = int(lay.cu_seqlens[p])
        for qh in range(cfg.num_q_heads):
            h = qh // G
            np.testing.assert_array_equal(O[t, qh], v[t, h].double().numpy())
            dot = float((q[t, qh].double() * k[t, h].double()).sum())
            assert abs(LSE[qh, t] - scale * dot) < 1e-12


def test_hand_worked_two_token_example():
    """One prompt of two tokens (a suffix: dense), d = 2, scale 1.
    q1 = (0, 1), k0 = (1, 0), k1 = (0, 1) -> scores 0 and 1 -> weights 1 and e."""
    lay = W.Layout(num_prompts=1, num_docs=0, num_layers=1, num_q_heads=1, num_kv_heads=1,
                   head_dim=2, tile=2, total_tokens=2, max_tiles_per_prompt=1,
                   cu_seqlens=np.array([0, 2], np.int32), doc_cu=np.array([0, 0], np.int32),
                   doc_end=np.zeros(0, np.int32), la_off=np.zeros(0, np.int64),
                   ca_off=np.zeros(0, np.int64), la_words_len=0, ca_words_len=0)
    q = torch.tensor([[[1.0, 0.0]], [[0.0, 1.0]]]).to(torch.bfloat16)
    k = torch.tensor([[[1.0, 0.0]], [[0.0, 1.0]]]).to(torch.bfloat16)
    v = torch.tensor([[[1.0, 2.0]], [[3.0, 4.0]]]).to(torch.bfloat16)
    e = math.e
    o, lse = oracle.attention_rows(lay, np.zeros(0, np.uint64), np.zeros(0, np.uint64), 0,
                                   q, k, v, [0, 1], [0, 0], scale=1.0)
    np.testing.assert_allclose(o[0], [1.0, 2.0], atol=1e-15)
    assert abs(lse[0] - 1.0) < 1e-15
    np.testing.assert_allclose(o[1], [(1 + 3 * e) / (1 + e), (2 + 4 * e) / (1 + e)], atol=1e-14)
    assert abs(lse[1] - math.log(1 + e)) < 1e-14


@pytest.mark.parametrize("cfg", [W.get_config("tiny")] + SMALL_CFGS[:2] + [SMALL_CFGS[3]],
                         ids=lambda c: c.name)
def test_random_bits_match_dense_mask_brute_force(cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    for layer in range(min(cfg.num_layers, 2)):
        q, k, v = W.make_qkv(cfg, layer)
        O, LSE = oracle.attention_all(lay, la, ca, layer, q, k, v)
        O2, LSE2 = oracle.brute_force_attention(lay, la, ca, layer, q, k, v)
        np.testing.assert_allclose(O, O2, atol=1e-12, rtol=0)
        np.testing.assert_allclose(LSE, LSE2, atol=1e-12, rtol=0)


def test_schedule_is_longest_first_permutation():
    cfg = SMALL_CFGS[3]
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    _, cnt = oracle.decode(lay, la, ca)
    sched = oracle.schedule(cnt)
    flat = cnt.reshape(cnt.shape[0], -1)
    for l in range(flat.shape[0]):
        assert sorted(sched[l]) == list(range(flat.shape[1]))
        c = flat[l][sched[l]]
        assert np.all(np.diff(c) <= 0)


# ---- offline bit building (the step before the online path) -------------------------

def test_build_masses_rows_sum_to_group_rows():
    """Every query row's probabilities sum to 1, so row i of M sums to G * tile."""
    cfg = W.custom_config("bb_rows", [([256, 512], 64)], W.BitSpec(la_p=0.3, ca_p=0.3),
                          num_q_heads=4, num_kv_heads=2, head_dim=32, tile=64)
    lay = W.make_layout(cfg)
    q, k, _ = W.make_qkv(cfg, 0)
    _, _, masses, _ = oracle.build_bits(lay, 0, q, k, 0.3, 0.3)
    for (g, h), M in masses.items():
        np.testing.assert_allclose(M.sum(axis=1), 2 * 64, rtol=1e-12)
        assert np.all(np.triu(M, 1) == 0)


def test_build_masses_match_attention_with_one_hot_values():
    """The tile masses equal the oracle's own attention rows when V is the one-hot tile
    indicator of each key (document-alone problem): a second route to M."""
    cfg = W.custom_config("bb_route", [([192, 128], 64)], W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=8, tile=64)
    lay = W.make_layout(cfg)
    q, k, _ = W.make_qkv(cfg, 0)
    _, _, masses, _ = oracle.build_bits(lay, 0, q, k, 0.5, 0.5, scale=0.2)
    for g in range(lay.num_docs):
        s0, e0 = lay.doc_start(g), int(lay.doc_end[g])
        n = e0 - s0
        sub = W.Layout(num_prompts=1, num_docs=0, num_layers=1, num_q_heads=2, num_kv_heads=1,
                       head_dim=8, tile=64, total_tokens=n, max_tiles_per_prompt=n // 64,
                       cu_seqlens=np.array([0, n], np.int32), doc_cu=np.array([0, 0], np.int32),
                       doc_end=np.zeros(0, np.int32), la_off=np.zeros(0, np.int64),
                       ca_off=np.zeros(0, np.int64), la_words_len=0, ca_words_len=0)
        onehot = torch.zeros((n, 1, 8))
        onehot[torch.arange(n), 0, torch.arange(n) // 64] = 1.0
        tok = np.repeat(np.arange(n, dtype=np.int32), 2)
        head = np.tile(np.arange(2, dtype=np.int32), n)
        o, _ = oracle.attention_rows(sub, np.zeros(0, np.uint64), np.zeros(0, np.uint64), 0,
                                     q[s0:e0], k[s0:e0], onehot.to(torch.bfloat16), tok, head,
                                     scale=0.2)
        M2 = o.reshape(n // 64, 64, 2, 8).sum(axis=(1, 2))[:, : n // 64]
        np.testing.assert_allclose(masses[(g, 0)], M2, atol=1e-10)


def test_build_selects_planted_hot_tile():
    """A key tile whose keys align with every query draws almost all the mass: LA keeps it in
    every row below it, and it is the only page CA keeps at a one-page budget."""
    cfg = W.custom_config("bb_hot", [([512], 64)], W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=16, tile=64)
    lay = W.make_layout(cfg)
    gen = torch.Generator().manual_seed(5)
    a = torch.randn(16, generator=gen)
    q = (a + 0.05 * torch.randn((512, 2, 16), generator=gen)).to(torch.bfloat16)
    k = (0.05 * torch.randn((512, 1, 16), generator=gen)).to(torch.bfloat16)
    k[2 * 64: 3 * 64, 0] = (2.0 * a).to(torch.bfloat16)          # tile 2 is hot
    la, ca, _, _ = oracle.build_bits(lay, 0, q, k, 1.0 / 8, 1.0 / 8, scale=1.0)
    for i in range(3, 8):  # rows below the hot tile keep exactly one LA tile (ceil(i/8) = 1)
        assert int(la[i]) == 1 << 2, (i, bin(int(la[i])))
    assert int(ca[0]) == 1 << 2


def test_build_counts_follow_the_fractions():
    cfg = W.custom_config("bb_cnt", [([64 * 20, 64 * 7], 64)], W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=16, tile=64)
    lay = W.make_layout(cfg)
    q, k, _ = W.make_qkv(cfg, 0)
    la, ca, _, _ = oracle.build_bits(lay, 0, q, k, 0.25, 0.4)
    for g, T in ((0, 20), (1, 7)):
        base = lay.la_off[g]
        for i in range(T):
            assert bin(int(la[base + i])).count("1") == int(np.ceil(0.25 * i - 1e-4))
        assert bin(int(ca[lay.ca_off[g]])).count("1") == int(np.ceil(0.4 * T - 1e-4))


# ---- exhaustive decode on tiny prompts ----------------------------------------------

def test_decode_exhaustive_tiny_patterns():
    """Every LA/CA pattern of a two-document prompt against the list rule written out."""
    from helpers import enumerated_prompts, plain_lists
    lay, la, ca, n = enumerated_prompts()
    kv, cnt = oracle.decode(lay, la, ca)
    for pat in range(n):
        for r, want in enumerate(plain_lists(pat, 7 * pat)):
            i = 7 * pat + r
            assert list(kv[0, 0, i, :cnt[0, 0, i]]) == want, (pat, r)

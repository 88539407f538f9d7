"""sift_decode_ragged + sift_sparse_prefill_ragged: documents of any length, each tiled
from its own first token, and CA pages of a size of their own.

* decode: query-tile table, lists and counts bit-exact against the oracle's plain
  ragged decode, and on small layouts the key set the GPU's lists describe, expanded
  to tokens, equal to the token-level rule; the schedule is a longest-first
  permutation;
* attention: every row against the oracle (fp64, key set read from the bits), within
  the tolerances of the aligned path;
* on an aligned layout the general path issues the same MMAs in the same order as the
  aligned one, so its outputs are bitwise identical;
* the 33K-token ragged workload at full size: decode bit-exact, attention on sampled
  query tiles plus whole-output invariants.

SIFT pages (gist.science/it/paper/2606.09441), "Dettagli di Implementazione": bits are
decoded into tile indices that the sparse kernel iterates over; the pages fix no tile
or page size, so documents of any length and the page size are this library's reading.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_attention_close, assert_attention_close_scaled, check_sched,
                     device_bits, expand_lists)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def _setup(sift, cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    assert prob.num_query_tiles == lay.num_query_tiles
    la_d, ca_d = device_bits(la, ca)
    return lay, la, ca, prob, la_d, ca_d


def _check_decode(sift, lay, la, ca, prob, la_d, ca_d):
    st = prob.new_status()
    qt, kv, cnt, sched, pages = sift.decode_ragged(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    qt_o, kv_o, cnt_o, pg_o = oracle.decode_ragged(lay, la, ca, page_cap=prob.page_cap)
    assert np.array_equal(qt.cpu().numpy(), qt_o)
    cnt_h = cnt.cpu().numpy()
    assert np.array_equal(cnt_h, cnt_o)
    kv_h = kv.cpu().numpy()
    L, H, NQ = cnt_h.shape
    for l in range(L):
        for h in range(H):
            for q in range(NQ):
                n = cnt_h[l, h, q]
                assert np.array_equal(kv_h[l, h, q, :n], kv_o[l, h, q, :n]), (l, h, q)
    check_sched(sched.cpu().numpy(), cnt_h)
    if lay.total_tokens <= 6000:
        # beyond the encoding: the key set the GPU's own lists describe, expanded to tokens,
        # is the token-level rule written out block by block (oracle.token_mask)
        pg_e = pages.cpu().numpy() if pages is not None else np.zeros((L, H, 1, 1), np.int32)
        qt_h = qt.cpu().numpy()
        for l in range(L):
            for h in range(H):
                got = expand_lists(lay, qt_h, kv_h, cnt_h, pg_e, l, h)
                assert np.array_equal(got, oracle.token_mask(lay, la, ca, l, h)), (l, h)
    if pages is not None:  # gathered pages: every page a list points at, bit-exact
        pg_h = pages.cpu().numpy()
        for l in range(L):
            for h in range(H):
                for q in range(NQ):
                    for first, info in kv_h[l, h, q, :cnt_h[l, h, q]]:
                        if (int(info) >> 9) & 1:
                            n = (int(info) & 0xFF) // lay.page_size
                            got = pg_h[l].reshape(-1)[first: first + n]
                            want = pg_o[l].reshape(-1)[first: first + n]
                            assert np.array_equal(got, want), (l, h, q, first)
    return qt, kv, cnt, sched, pages


CFGS = [
    # tile 128, d 128, 16-token pages (8 per tile): odd documents, a one-token document,
    # a long document, an empty suffix, a suffix-only prompt
    W.custom_config("rg_a", [([300, 128 * 3 + 1, 77, 1], 50), ([1000], 0), ([], 130)],
                    W.BitSpec(la_p=0.4, ca_p=0.3), num_layers=2, num_q_heads=4,
                    num_kv_heads=2, head_dim=128, tile=128, page=16),
    # tile 64, d 64, 32-token pages, GQA 8:2, many short documents
    W.custom_config("rg_b", [([65, 63, 200, 1], 33), ([5] * 10, 7)],
                    W.BitSpec(la_p=0.5, ca_p=0.5, la_window=1, ca_first_page=True),
                    num_q_heads=8, num_kv_heads=2, head_dim=64, tile=64, page=32),
    # tile 128, d 64, pages of two tiles
    W.custom_config("rg_c", [([700, 260, 129], 100)], W.BitSpec(head_density=(0.1, 0.6)),
                    num_layers=2, num_q_heads=4, num_kv_heads=1, head_dim=64, tile=128,
                    page=256),
    # tile 64, d 128, page = tile: ragged lengths only; 4-token pages of a 64 tile (16 bits)
    W.custom_config("rg_d", [([100, 150], 64)], W.BitSpec(la_p=0.3, ca_p=0.6),
                    num_q_heads=2, num_kv_heads=1, head_dim=128, tile=64),
    W.custom_config("rg_e", [([100, 150, 31], 17)], W.BitSpec(la_p=0.3, ca_p=0.2),
                    num_q_heads=2, num_kv_heads=1, head_dim=128, tile=64, page=4),
    # gathered pages: 16 pages of 8 tokens per tile; 2 pages of 64
    W.custom_config("rg_f", [([333, 250, 129, 64], 40)], W.BitSpec(la_p=0.3, ca_p=0.25),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128, page=8),
    W.custom_config("rg_g", [([333, 250, 129, 64], 40)], W.BitSpec(la_p=0.3, ca_p=0.4),
                    num_q_heads=4, num_kv_heads=2, head_dim=64, tile=128, page=64),
    # many tiny documents: more gathered partial pages than whole tiles
    W.custom_config("rg_tiny", [([17] * 20, 0), ([1, 2, 3, 17, 33], 5)],
                    W.BitSpec(pattern="ones"), num_q_heads=2, num_kv_heads=1, head_dim=128,
                    tile=128, page=16),
    # every bit set / none
    W.custom_config("rg_ones", [([300, 99, 77], 50), ([1000], 5)], W.BitSpec(pattern="ones"),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128, page=16),
    W.custom_config("rg_zeros", [([300, 99, 77], 50), ([1000], 5)], W.BitSpec(pattern="zeros"),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128, page=16),
]


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_ragged_decode_and_attention_match_oracle(sift, cfg):
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    qt, kv, cnt, sched, pages = _check_decode(sift, lay, la, ca, prob, la_d, ca_d)
    st = prob.new_status()
    for layer in range(cfg.num_layers):
        q, k, v = W.make_qkv(cfg, layer, device="cuda")
        o, lse = sift.sparse_prefill_ragged(prob, layer, q, k, v, qt, kv, cnt, sched, pages,
                                            dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, sift.status_string(int(st.item()))
        O, LSE = oracle.attention_all(lay, la, ca, layer, q, k, v)
        assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                               f"{cfg.name} layer {layer}")


def test_ragged_rows_outside_segments_are_not_written(sift):
    """Only rows inside their segment are stored: a sentinel in O survives nowhere, and
    the partial tiles' missing rows are the next segment's, not garbage."""
    cfg = CFGS[0]
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    qt, kv, cnt, sched, pages = sift.decode_ragged(prob, la_d, ca_d)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full((cfg.num_q_heads, lay.total_tokens), float("nan"), device="cuda")
    sift.sparse_prefill_ragged(prob, 0, q, k, v, qt, kv, cnt, sched, pages, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("name", ["tiny", "fu_varlen"])
def test_general_path_equals_aligned_path_on_aligned_layout(sift, name):
    cfg = W.get_config("tiny") if name == "tiny" else W.custom_config(
        "fu_varlen", [([128] * 3, 128), ([256], 0), ([], 128), ([128, 384], 256)],
        W.BitSpec(la_p=0.5, ca_p=0.4, la_window=1, ca_first_page=True),
        num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    assert lay.aligned
    st = prob.new_status()
    kv_a, cnt_a, sch_a = sift.decode(prob, la_d, ca_d, dev_status=st)
    qt, kv_r, cnt_r, sch_r, _ = sift.decode_ragged(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    o1, l1 = sift.sparse_prefill(prob, 0, q, k, v, kv_a, cnt_a, sch_a, dev_status=st)
    o2, l2 = sift.sparse_prefill_ragged(prob, 0, q, k, v, qt, kv_r, cnt_r, sch_r, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(cnt_a, cnt_r)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_ragged_full_size_workload(sift):
    """The 33K-token ragged workload (two of its 32 layers): decode bit-exact, attention on
    sampled query tiles (first, a partial one and the last of every segment kind, plus
    random ones), every row finite and inside the convex hull of V."""
    full = W.get_config("llama_32k_ragged")
    import dataclasses
    cfg = dataclasses.replace(full, num_layers=2)
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    qt, kv, cnt, sched, pages = _check_decode(sift, lay, la, ca, prob, la_d, ca_d)
    qt_h = qt.cpu().numpy()
    rng = np.random.default_rng(7)
    partial = [i for i, (_, r) in enumerate(qt_h) if r < lay.tile]
    picks = sorted(set([0, len(qt_h) - 1] + partial[:4] +
                       list(rng.integers(0, len(qt_h), 12))))
    st = prob.new_status()
    for layer in range(cfg.num_layers):
        q, k, v = W.make_qkv(cfg, layer, device="cuda")
        o, lse = sift.sparse_prefill_ragged(prob, layer, q, k, v, qt, kv, cnt, sched, pages,
                                            dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.isfinite(o.float()).all()
        vmax = v.float().abs().amax(dim=(0, 2))          # per kv head
        G = cfg.num_q_heads // cfg.num_kv_heads
        omax = o.float().abs().amax(dim=(0, 2)).view(cfg.num_kv_heads, G).amax(dim=1)
        assert torch.all(omax <= vmax * (1 + 1e-2))
        tok, head = [], []
        for qi in picks:
            x, r = (int(z) for z in qt_h[qi])
            hq = int(rng.integers(cfg.num_q_heads))
            tok += list(range(x, x + r))
            head += [hq] * r
        tok = np.asarray(tok, np.int32)
        head = np.asarray(head, np.int32)
        O, LSE = oracle.attention_rows(lay, la, ca, layer, q, k, v, tok, head)
        og = o[torch.as_tensor(tok, device="cuda").long(),
               torch.as_tensor(head, device="cuda").long()].double().cpu().numpy()
        lg = lse[torch.as_tensor(head, device="cuda").long(),
                 torch.as_tensor(tok, device="cuda").long()].double().cpu().numpy()
        assert_attention_close(og, lg, O, LSE, f"ragged 33K layer {layer}")


def test_ragged_decode_many_segments_and_prompts(sift):
    """More than 1024 segments (the query-tile scan then runs over several chunks with a
    carry) spread over 350 prompts: decode bit-exact against the oracle."""
    rng = np.random.default_rng(3)
    prompts = []
    for p in range(350):
        docs = [int(x) for x in rng.integers(1, 40, size=int(rng.integers(0, 6)))]
        prompts.append((docs, int(rng.integers(0, 3) * 7)))
    cfg = W.custom_config("rg_many", prompts, W.BitSpec(la_p=0.4, ca_p=0.4), num_layers=1,
                          num_q_heads=2, num_kv_heads=1, head_dim=64, tile=64, page=16)
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    assert lay.num_docs + lay.num_prompts > 1024
    _check_decode(sift, lay, la, ca, prob, la_d, ca_d)


def test_ragged_decode_reports_a_wrong_tile_count(sift):
    """A query-tile count that disagrees with the segments is reported on the device; the
    spare row becomes an empty tile past the end of the batch."""
    import ctypes
    cfg = CFGS[0]
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    NQ = prob.num_query_tiles + 1
    L, H, R = cfg.num_layers, cfg.num_kv_heads, prob.max_tiles_per_prompt
    qt = torch.empty((NQ, 2), dtype=torch.int32, device="cuda")
    kv = torch.empty((L, H, NQ, R, 2), dtype=torch.int32, device="cuda")
    cnt = torch.empty((L, H, NQ), dtype=torch.int32, device="cuda")
    sch = torch.empty((L, H * NQ), dtype=torch.int32, device="cuda")
    pages = torch.empty((L, H, lay.num_docs, prob.page_cap), dtype=torch.int32, device="cuda")
    st = prob.new_status()
    lib = sift.load_library()
    rc = lib.sift_decode_ragged(prob.ref, NQ, la_d.data_ptr(), ca_d.data_ptr(), qt.data_ptr(),
                                kv.data_ptr(), cnt.data_ptr(), sch.data_ptr(), pages.data_ptr(),
                                prob.page_cap, st.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert int(st.item()) == 5  # SIFT_ERR_DEVICE_CHECK
    assert qt[NQ - 1].tolist() == [lay.total_tokens, 0]
    assert cnt[:, :, NQ - 1].eq(1).all()


@pytest.mark.parametrize("name", ["rg_f", "rg_ones"])
def test_ragged_running_max_growth(sift, name):
    """General layout with keys growing in scale tile by tile (rows rescale O mid-row,
    on gathered pages and on masked partial tiles alike) against the oracle."""
    cfg = next(c for c in CFGS if c.name == name)
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    qt, kv, cnt, sched, pages = _check_decode(sift, lay, la, ca, prob, la_d, ca_d)
    st = prob.new_status()
    q, k, v = W.make_qkv(cfg, 0, device="cuda", dist="growing_keys")
    o, lse = sift.sparse_prefill_ragged(prob, 0, q, k, v, qt, kv, cnt, sched, pages,
                                        dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close_scaled(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                           name + " growing keys")


def test_hole_entry_with_128_token_tiles_is_reported(sift):
    """With 128-token tiles the decode writes only entries whose visible keys form a prefix
    of each row (pages below the tile are gathered); an entry whose page mask leaves a hole
    is read there as its first len keys and reported as a device check."""
    cfg = next(c for c in CFGS if c.name == "rg_ones")
    assert cfg.tile == 128 and cfg.page < cfg.tile
    lay, la, ca, prob, la_d, ca_d = _setup(sift, cfg)
    qt, kv, cnt, sched, pages = sift.decode_ragged(prob, la_d, ca_d)
    torch.cuda.synchronize()
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    st = prob.new_status()
    o_ok, l_ok = sift.sparse_prefill_ragged(prob, 0, q, k, v, qt, kv, cnt, sched, pages,
                                            dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the first query tile's only entry is its own tile: drop the first page's bit
    assert int(cnt[0, 0, 0]) == 1
    info = int(kv[0, 0, 0, 0, 1])
    assert info & (1 << 8) and (info >> 16) & 1
    kv_bad = kv.clone()
    kv_bad[0, 0, 0, 0, 1] = info & ~(1 << 16)
    st = prob.new_status()
    o, l = sift.sparse_prefill_ragged(prob, 0, q, k, v, qt, kv_bad, cnt, sched, pages,
                                      dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5, sift.status_string(int(st.item()))  # SIFT_ERR_DEVICE_CHECK
    assert torch.isfinite(o.float()).all() and torch.isfinite(l).all()
    assert torch.equal(o, o_ok) and torch.equal(l, l_ok)  # read as its first len keys

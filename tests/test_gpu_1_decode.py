"""sift_decode on the GPU, bit-exact against the oracle's decode.

SIFT pages (gist.science/it/paper/2606.09441), "Dettagli di Implementazione":
the decoding kernel turns the bit vectors into explicit tile indices.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import check_sched, device_bits, setup

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def _compare(lay, la, ca, kv, cnt, sched):
    kv_o, cnt_o = oracle.decode(lay, la, ca)
    cnt_g = cnt.cpu().numpy()
    kv_g = kv.cpu().numpy()
    assert np.array_equal(cnt_g, cnt_o)
    R = kv_o.shape[-1]
    mask = np.arange(R)[None, None, None, :] < cnt_o[..., None]
    assert np.array_equal(np.where(mask, kv_g, -1), kv_o)
    check_sched(sched.cpu().numpy(), cnt_o)


def test_golden_fixture(sift):
    with open(os.path.join(GOLDEN, "decode_small.json")) as f:
        g = json.load(f)
    prob = sift.SiftProblem(cu_seqlens=g["cu_seqlens"], doc_cu=g["doc_cu"], doc_end=g["doc_end"],
                            la_off=g["la_off"], ca_off=g["ca_off"], num_layers=2,
                            num_q_heads=4, num_kv_heads=2, head_dim=64, tile=g["tile"],
                            la_words_len=len(g["la_words"]), ca_words_len=len(g["ca_words"]),
                            max_tiles_per_prompt=6)
    la_d, ca_d = device_bits(np.array(g["la_words"], np.uint64), np.array(g["ca_words"], np.uint64))
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kv, cnt = kv.cpu().numpy(), cnt.cpu().numpy()
    for l in range(2):
        for h in range(2):
            for i, row in enumerate(g["expected"][f"l{l}h{h}"]):
                assert cnt[l, h, i] == len(row)
                assert list(kv[l, h, i, :len(row)]) == row
    check_sched(sched.cpu().numpy(), cnt)


EDGE_CFGS = [
    W.custom_config("dec_small", [([256, 512, 128], 128)], W.BitSpec(la_p=0.3, ca_p=0.4),
                    num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=64, tile=64),
    # suffix-only prompt, prompt without suffix, one-tile documents, several prompts
    W.custom_config("dec_varlen", [([128, 64], 64), ([192], 0), ([], 128), ([64] * 5, 64)],
                    W.BitSpec(la_p=0.5, ca_p=0.5, la_window=1, ca_first_page=True),
                    num_layers=1, num_q_heads=6, num_kv_heads=3, head_dim=64, tile=64),
    # documents of more than 64 tiles: two words per LA row and per CA vector, > 32 docs
    W.custom_config("dec_wide", [([64 * 130, 64 * 70], 64), ([64] * 40, 128)],
                    W.BitSpec(la_p=0.1, ca_p=0.2), num_layers=1, num_q_heads=2,
                    num_kv_heads=1, head_dim=64, tile=64),
    W.custom_config("dec_ones", [([256] * 3, 128)], W.BitSpec(pattern="ones"),
                    num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=64, tile=64),
    W.custom_config("dec_zeros", [([256] * 3, 128)], W.BitSpec(pattern="zeros"),
                    num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=64, tile=64),
    # 40 kv heads x 1,360 query tiles = 54,400 rows in one layer: the schedule block's
    # counts no longer fit in shared memory beside its tables, so its sort reads them
    # back from the counts array (the batch-of-4 and 262K workloads cover the two-launch
    # form, the 33K one the single launch with the counts in shared memory)
    W.custom_config("dec_many_rows", [([64 * 40] * 34, 0)],
                    W.BitSpec(la_p=0.2, ca_p=0.05, ca_first_page=True), num_layers=1,
                    num_q_heads=80, num_kv_heads=40, head_dim=64, tile=64),
]


@pytest.mark.parametrize("cfg", EDGE_CFGS, ids=lambda c: c.name)
def test_decode_edge_cases(sift, cfg):
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare(lay, la, ca, kv, cnt, sched)


@pytest.mark.parametrize("name", ["tiny", "llama_10doc", "llama_32k", "qwen3_64k", "batch4_p005",
                                  "batch4_p010", "batch4_p020", "batch4_p040", "batch4_p070",
                                  "batch4_p100"])
def test_decode_benchmark_configs(sift, name):
    lay, la, ca, prob, la_d, ca_d = setup(W.get_config(name))
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _compare(lay, la, ca, kv, cnt, sched)


def test_decode_larger_rowcap_and_repeat(sift):
    """rowcap above the need leaves the tail untouched; a second call gives the same result."""
    cfg = EDGE_CFGS[0]
    lay, la, ca, prob0, la_d, ca_d = setup(cfg)
    prob = sift.SiftProblem.from_layout(lay)
    prob = sift.SiftProblem(cu_seqlens=lay.cu_seqlens, doc_cu=lay.doc_cu, doc_end=lay.doc_end,
                            la_off=lay.la_off, ca_off=lay.ca_off, num_layers=lay.num_layers,
                            num_q_heads=lay.num_q_heads, num_kv_heads=lay.num_kv_heads,
                            head_dim=lay.head_dim, tile=lay.tile, la_words_len=lay.la_words_len,
                            ca_words_len=lay.ca_words_len,
                            max_tiles_per_prompt=lay.num_tiles)
    L, H, N = lay.num_layers, lay.num_kv_heads, lay.num_tiles
    kv = torch.full((L, H, N, N), -7, dtype=torch.int32, device="cuda")
    st = prob.new_status()
    for _ in range(2):
        kv, cnt, sched = sift.decode(prob, la_d, ca_d, kv_idx=kv, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kv_o, cnt_o = oracle.decode(lay, la, ca, rowcap=N)
    kv_g = kv.cpu().numpy()
    assert np.array_equal(cnt.cpu().numpy(), cnt_o)
    mask = np.arange(N)[None, None, None, :] < cnt_o[..., None]
    assert np.array_equal(np.where(mask, kv_g, -1), kv_o)
    assert np.all(kv_g[~mask] == -7)


def test_decode_device_check_on_bad_offsets(sift):
    """An LA offset pointing past the words is caught on the device, without a fault."""
    cfg = EDGE_CFGS[0]
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    la_off = lay.la_off.copy()
    la_off[1] = lay.la_words_len + 5
    prob = sift.SiftProblem(cu_seqlens=lay.cu_seqlens, doc_cu=lay.doc_cu, doc_end=lay.doc_end,
                            la_off=la_off, ca_off=lay.ca_off, num_layers=lay.num_layers,
                            num_q_heads=lay.num_q_heads, num_kv_heads=lay.num_kv_heads,
                            head_dim=lay.head_dim, tile=lay.tile, la_words_len=lay.la_words_len,
                            ca_words_len=lay.ca_words_len,
                            max_tiles_per_prompt=lay.max_tiles_per_prompt)
    la_d, ca_d = device_bits(la, ca)
    st = prob.new_status()
    sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # SIFT_ERR_DEVICE_CHECK


def test_decode_device_check_on_prompt_past_the_batch(sift):
    """A prompt end past total_tokens (cu_seqlens lives on the device, so only the kernel
    can see it) is reported; the kernel bounds every index by the batch's tiles."""
    cfg = EDGE_CFGS[0]
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    cu = lay.cu_seqlens.copy()
    cu[-1] = lay.total_tokens + 4 * lay.tile
    prob = sift.SiftProblem(cu_seqlens=cu, doc_cu=lay.doc_cu, doc_end=lay.doc_end,
                            la_off=lay.la_off, ca_off=lay.ca_off, num_layers=lay.num_layers,
                            num_q_heads=lay.num_q_heads, num_kv_heads=lay.num_kv_heads,
                            head_dim=lay.head_dim, tile=lay.tile, la_words_len=lay.la_words_len,
                            ca_words_len=lay.ca_words_len,
                            max_tiles_per_prompt=lay.max_tiles_per_prompt)
    # the struct the kernel reads keeps the batch's real size; only the device array lies
    prob._struct.total_tokens = lay.total_tokens
    la_d, ca_d = device_bits(la, ca)
    st = prob.new_status()
    sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # SIFT_ERR_DEVICE_CHECK


def test_decode_rejects_bad_arguments(sift):
    lay, la, ca, prob, la_d, ca_d = setup(EDGE_CFGS[0])
    with pytest.raises(sift.SiftError) as e:
        sift.decode(prob, None, ca_d)
    assert e.value.code == 1


def test_decode_exhaustive_tiny_patterns_bit_exact(sift):
    """All 512 LA/CA patterns of a two-document, three-tile prompt, as one batch of 512
    prompts: the GPU lists equal the oracle's and the list rule written out."""
    from helpers import enumerated_prompts, plain_lists
    lay, la, ca, n = enumerated_prompts()
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(la, ca)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kv_h, cnt_h = kv.cpu().numpy(), cnt.cpu().numpy()
    kv_o, cnt_o = oracle.decode(lay, la, ca)
    assert np.array_equal(cnt_h, cnt_o)
    for pat in range(n):
        for r, want in enumerate(plain_lists(pat, 7 * pat)):
            i = 7 * pat + r
            assert list(kv_h[0, 0, i, :cnt_h[0, 0, i]]) == want, (pat, r)

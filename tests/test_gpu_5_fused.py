"""sift_fused_prefill: the decode walked inside the prefill.  It issues the same
MMAs on the same tiles in the same order as sift_decode + sift_sparse_prefill, so
its outputs must be bitwise identical; they are also checked against the oracle.

SIFT pages (gist.science/it/paper/2606.09441), "Dettagli di Implementazione": the
bit vectors are decoded into tile indices that the sparse kernel iterates over.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (assert_attention_close, assert_attention_close_scaled, gpu_rows,
                     oracle_rows_for_pairs, sample_pairs, setup)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


CFGS = [
    W.get_config("tiny"),
    W.custom_config("fu_varlen", [([128] * 3, 128), ([256], 0), ([], 128), ([128, 384], 256)],
                    W.BitSpec(la_p=0.5, ca_p=0.4, la_window=1, ca_first_page=True),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("fu_layers", [([256, 384], 128)], W.BitSpec(head_density=(0.05, 0.6)),
                    num_layers=3, num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("fu_wide", [([64 * 70, 64 * 3], 64), ([64] * 40, 64)],
                    W.BitSpec(la_p=0.2, ca_p=0.2), num_q_heads=4, num_kv_heads=1,
                    head_dim=64, tile=64),
    W.custom_config("fu_ones", [([256] * 3, 128)], W.BitSpec(pattern="ones"),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("fu_zeros", [([256] * 3, 128)], W.BitSpec(pattern="zeros"),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
]


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_fused_equals_decode_then_sparse_and_oracle(sift, cfg):
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    for layer in range(cfg.num_layers):
        q, k, v = W.make_qkv(cfg, layer, device="cuda")
        o1, l1 = sift.sparse_prefill(prob, layer, q, k, v, kv, cnt, sched, dev_status=st)
        o2, l2 = sift.fused_prefill(prob, layer, la_d, ca_d, q, k, v, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, sift.status_string(int(st.item()))
        assert torch.equal(o1, o2), f"layer {layer}: outputs differ"
        assert torch.equal(l1, l2), f"layer {layer}: lse differs"
        O, LSE = oracle.attention_all(lay, la, ca, layer, q, k, v)
        assert_attention_close(o2.double().cpu().numpy(), l2.double().cpu().numpy(), O, LSE,
                               f"{cfg.name} layer {layer}")


@pytest.mark.parametrize("name", ["llama_10doc", "qwen3_64k", "batch4_p020"])
def test_fused_full_size(sift, name):
    cfg = W.get_config(name)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    o1, l1 = sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sched, dev_status=st)
    o2, l2 = sift.fused_prefill(prob, 0, la_d, ca_d, q, k, v, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    pairs = sample_pairs(lay, np.random.default_rng(2), n_random=8)
    tok, head, O, LSE = oracle_rows_for_pairs(lay, la, ca, 0, q.cpu(), k.cpu(), v.cpu(), pairs)
    og, lg = gpu_rows(o2, l2, tok, head)
    assert_attention_close(og, lg, O, LSE, name)


def test_fused_rejects_too_many_prompts(sift):
    cfg = W.custom_config("fu_many", [([128], 128)] * 65, W.BitSpec(la_p=0.3, ca_p=0.3),
                          num_q_heads=2, num_kv_heads=1, head_dim=64, tile=64)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    with pytest.raises(sift.SiftError) as e:
        sift.fused_prefill(prob, 0, la_d, ca_d, q, k, v)
    assert e.value.code == 2


def test_fused_running_max_growth(sift):
    """Keys growing in scale tile by tile make rows rescale O mid-row; the fused kernel
    still equals decode + sparse bit for bit and matches the oracle."""
    cfg = W.custom_config("fu_grow", [([256] * 3, 128), ([384], 128)], W.BitSpec(la_p=0.6, ca_p=0.6),
                          num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda", dist="growing_keys")
    o1, l1 = sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sched, dev_status=st)
    o2, l2 = sift.fused_prefill(prob, 0, la_d, ca_d, q, k, v, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close_scaled(o2.double().cpu().numpy(), l2.double().cpu().numpy(), O, LSE, "fu_grow")

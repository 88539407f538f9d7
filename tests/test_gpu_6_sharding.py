"""KV-head shards run through the unchanged C ABI reproduce the head slices of the
unsharded prefill bitwise (each work item reads only its own kv head), and each
shard's decode and attention agree with the oracle run on the unsharded layout,
restricted to the shard's heads (bit-exact lists, outputs within the tolerance)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from bit_vector_guided_gb300.sharding import kv_head_range, shard_bits
from helpers import assert_attention_close, device_bits, setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


@pytest.mark.parametrize("world", [2, 4])
def test_shards_match_unsharded(sift, world):
    cfg = W.custom_config("shard_gpu", [([512, 384], 128), ([256], 128)],
                          W.BitSpec(head_density=(0.05, 0.6)), num_layers=2, num_q_heads=16,
                          num_kv_heads=4, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    G = cfg.num_q_heads // cfg.num_kv_heads
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    kv_o, cnt_o = oracle.decode(lay, la, ca)
    for layer in range(cfg.num_layers):
        q, k, v = W.make_qkv(cfg, layer, device="cuda")
        o, lse = sift.sparse_prefill(prob, layer, q, k, v, kv, cnt, sched, dev_status=st)
        O_ref, LSE_ref = oracle.attention_all(lay, la, ca, layer, q.cpu(), k.cpu(), v.cpu())
        for r in range(world):
            h0, h1 = kv_head_range(r, world, cfg.num_kv_heads)
            la_off, ca_off, la_s, ca_s = shard_bits(lay.cu_seqlens, lay.doc_cu, lay.doc_end,
                                                    lay.la_off, lay.ca_off, la, ca,
                                                    cfg.num_layers, cfg.num_kv_heads, cfg.tile,
                                                    h0, h1)
            sp = sift.SiftProblem(cu_seqlens=lay.cu_seqlens, doc_cu=lay.doc_cu,
                                  doc_end=lay.doc_end, la_off=la_off, ca_off=ca_off,
                                  num_layers=cfg.num_layers, num_q_heads=(h1 - h0) * G,
                                  num_kv_heads=h1 - h0, head_dim=cfg.head_dim, tile=cfg.tile,
                                  la_words_len=len(la_s), ca_words_len=len(ca_s),
                                  max_tiles_per_prompt=lay.max_tiles_per_prompt)
            las, cas = device_bits(la_s, ca_s)
            ss = sp.new_status()
            kv_s, cnt_s, sch_s = sift.decode(sp, las, cas, dev_status=ss)
            qs = q[:, h0 * G:h1 * G].contiguous()
            ks, vs = k[:, h0:h1].contiguous(), v[:, h0:h1].contiguous()
            o_s, lse_s = sift.sparse_prefill(sp, layer, qs, ks, vs, kv_s, cnt_s, sch_s,
                                             dev_status=ss)
            o_f, lse_f = sift.fused_prefill(sp, layer, las, cas, qs, ks, vs, dev_status=ss)
            torch.cuda.synchronize()
            assert int(ss.item()) == 0
            assert torch.equal(cnt_s, cnt[:, h0:h1])
            assert torch.equal(o_s, o[:, h0 * G:h1 * G]) and torch.equal(o_f, o_s)
            assert torch.equal(lse_s, lse[h0 * G:h1 * G]) and torch.equal(lse_f, lse_s)
            # the shard against the oracle of the whole problem, restricted to its heads
            kv_sh, cnt_sh = kv_s.cpu().numpy(), cnt_s.cpu().numpy()
            assert np.array_equal(cnt_sh, cnt_o[:, h0:h1])
            m = np.arange(kv_o.shape[-1])[None, None, None, :] < cnt_o[:, h0:h1, :, None]
            assert np.array_equal(np.where(m, kv_sh, -1), kv_o[:, h0:h1])
            assert_attention_close(o_s.double().cpu().numpy(), lse_s.double().cpu().numpy(),
                                   O_ref[:, h0 * G:h1 * G], LSE_ref[h0 * G:h1 * G],
                                   f"shard {r}/{world} layer {layer}")
        assert int(st.item()) == 0


@pytest.mark.parametrize("world", [2, 4])
def test_general_layout_shards_match_unsharded(sift, world):
    """Ragged documents with 16-token pages gathered: each shard's general-layout prefill
    equals the head slice of the unsharded one, bit for bit."""
    cfg = W.custom_config("shard_gpu_rg", [([300, 411, 77], 50), ([190], 0)],
                          W.BitSpec(la_p=0.4, ca_p=0.3), num_layers=1, num_q_heads=16,
                          num_kv_heads=4, head_dim=128, tile=128, page=16)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    la_d, ca_d = device_bits(la, ca)
    st = prob.new_status()
    lists = sift.decode_ragged(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    o, lse = sift.sparse_prefill_ragged(prob, 0, q, k, v, *lists, dev_status=st)
    G = cfg.num_q_heads // cfg.num_kv_heads
    O_ref, LSE_ref = oracle.attention_all(lay, la, ca, 0, q.cpu(), k.cpu(), v.cpu())
    for r in range(world):
        h0, h1 = kv_head_range(r, world, cfg.num_kv_heads)
        la_off, ca_off, la_s, ca_s = shard_bits(lay.cu_seqlens, lay.doc_cu, lay.doc_end,
                                                lay.la_off, lay.ca_off, la, ca, cfg.num_layers,
                                                cfg.num_kv_heads, cfg.tile, h0, h1, page=16)
        sp = sift.SiftProblem(cu_seqlens=lay.cu_seqlens, doc_cu=lay.doc_cu, doc_end=lay.doc_end,
                              la_off=la_off, ca_off=ca_off, num_layers=cfg.num_layers,
                              num_q_heads=(h1 - h0) * G, num_kv_heads=h1 - h0,
                              head_dim=cfg.head_dim, tile=cfg.tile, la_words_len=len(la_s),
                              ca_words_len=len(ca_s), max_tiles_per_prompt=lay.max_tiles_per_prompt,
                              page=16)
        las, cas = device_bits(la_s, ca_s)
        ss = sp.new_status()
        lists_s = sift.decode_ragged(sp, las, cas, dev_status=ss)
        qs = q[:, h0 * G:h1 * G].contiguous()
        ks, vs = k[:, h0:h1].contiguous(), v[:, h0:h1].contiguous()
        o_s, lse_s = sift.sparse_prefill_ragged(sp, 0, qs, ks, vs, *lists_s, dev_status=ss)
        torch.cuda.synchronize()
        assert int(ss.item()) == 0
        assert torch.equal(o_s, o[:, h0 * G:h1 * G])
        assert torch.equal(lse_s, lse[h0 * G:h1 * G])
        assert_attention_close(o_s.double().cpu().numpy(), lse_s.double().cpu().numpy(),
                               O_ref[:, h0 * G:h1 * G], LSE_ref[h0 * G:h1 * G],
                               f"general-layout shard {r}/{world}")
    assert int(st.item()) == 0

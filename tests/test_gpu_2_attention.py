"""sift_sparse_prefill / sift_dense_prefill on the GPU against the fp64 oracle,
at sizes the oracle computes completely (several tiles, ragged prompt mixes).

SIFT pages (gist.science/it/paper/2606.09441): "Esecuzione Online" and
"Dettagli di Implementazione" (sparse attention over the decoded indices);
"Risultati" (full recompute = dense causal attention).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_attention_close, assert_attention_close_scaled, setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def _run_sparse(sift, cfg, layer=0, qkv=None):
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    q, k, v = qkv if qkv is not None else W.make_qkv(cfg, layer, device="cuda")
    o, lse = sift.sparse_prefill(prob, layer, q, k, v, kv, cnt, sched, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, sift.status_string(int(st.item()))
    return lay, la, ca, prob, (q, k, v), o, lse


SMALL = [
    W.get_config("tiny"),
    W.custom_config("att_b128_d128", [([512, 256, 384], 128)], W.BitSpec(la_p=0.3, ca_p=0.3),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("att_b64_d128", [([256, 192], 64), ([128], 0)], W.BitSpec(la_p=0.4, ca_p=0.3),
                    num_q_heads=4, num_kv_heads=1, head_dim=128, tile=64),
    W.custom_config("att_b128_d64", [([384, 256], 128), ([], 256)], W.BitSpec(la_p=0.4, ca_p=0.3),
                    num_q_heads=8, num_kv_heads=2, head_dim=64, tile=128),
    W.custom_config("att_varlen", [([128] * 3, 128), ([256], 0), ([], 128), ([128, 384], 256)],
                    W.BitSpec(la_p=0.5, ca_p=0.4, la_window=1, ca_first_page=True),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("att_gqa8", [([512, 512], 128)], W.BitSpec(la_p=0.2, ca_p=0.2),
                    num_q_heads=16, num_kv_heads=2, head_dim=128, tile=128),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_sparse_matches_oracle(sift, cfg):
    lay, la, ca, prob, (q, k, v), o, lse = _run_sparse(sift, cfg)
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE, cfg.name)


@pytest.mark.parametrize("cfg", SMALL[:2] + SMALL[4:5], ids=lambda c: c.name)
def test_dense_matches_oracle_all_ones(sift, cfg):
    """The dense kernel equals the oracle with every bit set (dense causal attention)."""
    ones = W.custom_config(cfg.name + "_ones", list(cfg.prompts), W.BitSpec(pattern="ones"),
                           num_q_heads=cfg.num_q_heads, num_kv_heads=cfg.num_kv_heads,
                           head_dim=cfg.head_dim, tile=cfg.tile)
    lay, la, ca, prob, la_d, ca_d = setup(ones)
    q, k, v = W.make_qkv(ones, 0, device="cuda")
    st = prob.new_status()
    o, lse = sift.dense_prefill(prob, q, k, v, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE, "dense")


def test_sparse_all_ones_equals_dense_kernel(sift):
    cfg = W.custom_config("att_ones", [([256] * 4, 128), ([384], 128)], W.BitSpec(pattern="ones"),
                          num_q_heads=8, num_kv_heads=2, head_dim=128, tile=128)
    lay, la, ca, prob, (q, k, v), o, lse = _run_sparse(sift, cfg)
    st = prob.new_status()
    od, lsed = sift.dense_prefill(prob, q, k, v, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    diff = (o.float() - od.float()).abs().max().item()
    assert diff <= 1e-2
    assert (lse - lsed).abs().max().item() <= 1e-4


def test_closed_forms_on_gpu(sift):
    """Constant V -> O is that constant; first token of each prompt -> O = v_0."""
    cfg = W.custom_config("att_closed", [([256, 128], 128), ([128], 0)],
                          W.BitSpec(la_p=0.5, ca_p=0.5), num_q_heads=4, num_kv_heads=2,
                          head_dim=128, tile=128)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    vc = ((torch.arange(2 * 128, device="cuda", dtype=torch.float32).reshape(1, 2, 128) / 64) - 2)
    vconst = vc.to(torch.bfloat16).expand(cfg.total_tokens, -1, -1).contiguous()
    lay, la, ca, prob, _, o, lse = _run_sparse(sift, cfg, qkv=(q, k, vconst))
    exp = vconst.float().repeat_interleave(2, dim=1)
    assert torch.equal(o.float(), exp)
    lay, la, ca, prob, _, o, lse = _run_sparse(sift, cfg, qkv=(q, k, v))
    for p in range(lay.num_prompts):
        t = int(lay.cu_seqlens[p])
        assert torch.equal(o[t].float(), v[t].float().repeat_interleave(2, dim=0))


def test_custom_softmax_scale(sift):
    cfg = SMALL[1]
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    o, lse = sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sched, softmax_scale=0.03,
                                 dev_status=st)
    torch.cuda.synchronize()
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v, scale=0.03)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE, "scale")


def test_multi_layer_slices(sift):
    """Layer l of a 3-layer decode uses its own bits."""
    cfg = W.custom_config("att_layers", [([256, 384], 128)],
                          W.BitSpec(head_density=(0.05, 0.6)), num_layers=3, num_q_heads=4,
                          num_kv_heads=2, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    for layer in range(3):
        q, k, v = W.make_qkv(cfg, layer, device="cuda")
        o, lse = sift.sparse_prefill(prob, layer, q, k, v, kv, cnt, sched, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        O, LSE = oracle.attention_all(lay, la, ca, layer, q, k, v)
        assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                               f"layer {layer}")


def test_unsupported_group_is_rejected(sift):
    cfg = W.custom_config("att_odd", [([256], 128)], W.BitSpec(la_p=0.3, ca_p=0.3),
                          num_q_heads=3, num_kv_heads=1, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    with pytest.raises(sift.SiftError) as e:
        sift.dense_prefill(prob, q, k, v)
    assert e.value.code == 2


def _rescale_events(lay, q, k, scale=None):
    """(row, key tile) pairs of an all-ones layout at which the row's running max (log2
    units, tiles taken in ascending order as the lists hold them) grows by more than 8:
    the case in which the kernel rescales its O accumulator after the first tile."""
    B = lay.tile
    d = q.shape[-1]
    G = q.shape[1] // k.shape[1]
    s = (scale if scale is not None else d ** -0.5) * 1.4426950408889634
    events = 0
    for p in range(lay.num_prompts):
        t0, t1 = int(lay.cu_seqlens[p]), int(lay.cu_seqlens[p + 1])
        qp = q[t0:t1, ::G].float().cpu()           # one query head per kv head
        kp = k[t0:t1].float().cpu()
        sc = torch.einsum("thd,shd->hts", qp, kp) * s
        n = t1 - t0
        causal = torch.arange(n)[None, :] <= torch.arange(n)[:, None]
        sc = sc.masked_fill(~causal, float("-inf"))
        nt = (n + B - 1) // B
        tmax = torch.stack([sc[..., j * B:(j + 1) * B].amax(-1) for j in range(nt)], -1)
        run = tmax[..., 0]
        for j in range(1, nt):
            events += int(((tmax[..., j] > run + 8) & (tmax[..., j] > float("-inf"))).sum())
            run = torch.maximum(run, tmax[..., j])
    return events


GROWTH = [
    W.custom_config("att_grow_ones", [([512, 384], 128), ([256], 128)], W.BitSpec(pattern="ones"),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("att_grow_sparse", [([512, 384, 256], 128)], W.BitSpec(la_p=0.5, ca_p=0.5),
                    num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128),
    W.custom_config("att_grow_b64", [([256, 192], 64), ([128], 64)], W.BitSpec(la_p=0.6, ca_p=0.6),
                    num_q_heads=4, num_kv_heads=1, head_dim=128, tile=64),
]


@pytest.mark.parametrize("cfg", GROWTH, ids=lambda c: c.name)
def test_running_max_growth_matches_oracle(sift, cfg):
    """Keys that grow in scale from tile to tile push each row's running max up by more
    than the lazy-rescale threshold after its first tile, so the O accumulator is rescaled
    in tensor memory mid-row (before that tile's P reaches the P*V MMA); the sparse and
    dense kernels must still match the oracle."""
    q, k, v = W.make_qkv(cfg, 0, device="cuda", dist="growing_keys")
    lay, la, ca, prob, _, o, lse = _run_sparse(sift, cfg, qkv=(q, k, v))
    if cfg.bits.pattern == "ones":
        assert _rescale_events(lay, q, k) > 0
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close_scaled(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                           cfg.name + " sparse")
    if cfg.bits.pattern == "ones":
        st = prob.new_status()
        od, lsed = sift.dense_prefill(prob, q, k, v, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_attention_close_scaled(od.double().cpu().numpy(), lsed.double().cpu().numpy(), O, LSE,
                               cfg.name + " dense")

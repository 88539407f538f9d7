"""The FLOP count behind every TFLOP/s figure of bench.py, pinned to closed forms: with
every LA and CA bit set, each query tile of a prompt of T tiles computes all T(T+1)/2
causal key tiles, so the count must equal the dense causal one; a prompt of one tile is
its diagonal alone, of which (B+1)/(2B) is causal."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads as W  # noqa: E402


def _counts(cfg):
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    _, cnt = oracle.decode(lay, la, ca)
    return lay, cnt


def test_all_bits_set_counts_the_dense_causal_triangle():
    docs = [([256, 128, 384], 128), ([128] * 2, 0)]
    cfg = W.custom_config("flops_ones", docs, W.BitSpec(pattern="ones"), num_layers=2,
                          num_q_heads=8, num_kv_heads=2, head_dim=128, tile=128)
    lay, cnt = _counts(cfg)
    B, d = cfg.tile, cfg.head_dim
    tiles = [(sum(lens) + suffix) // B for lens, suffix in docs]
    triangle = sum(T * (T + 1) // 2 for T in tiles)
    expected = triangle * cfg.num_q_heads * 4.0 * B * B * d  # per layer, all query heads
    flops = bench.computed_flops(cfg, cnt)
    assert flops.shape == (cfg.num_layers,)
    assert np.all(flops == expected)


def test_a_single_tile_prompt_is_its_diagonal():
    cfg = W.custom_config("flops_one_tile", [([], 64)], W.BitSpec(pattern="ones"),
                          num_layers=1, num_q_heads=4, num_kv_heads=1, head_dim=64, tile=64)
    lay, cnt = _counts(cfg)
    assert int(cnt.sum()) == 1
    flops = float(bench.computed_flops(cfg, cnt).sum())
    assert flops == cfg.num_q_heads * 4.0 * 64 * 64 * 64
    frac = bench.useful_fraction(cfg, lay, flops)
    assert abs(frac - (64 + 1) / (2 * 64)) < 1e-12

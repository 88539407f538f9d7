"""KV-head sharding: a rank's re-packed bits describe exactly its heads' rows
(checked with the oracle's decode), the ranks' head ranges tile [0, Hkv), and with
two gloo ranks the job's work adds up over ranks."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as W
from bit_vector_guided_gb300.sharding import kv_head_range, shard_bits

CFG = W.custom_config("shard_cpu", [([256, 512, 128], 128), ([192], 64)],
                      W.BitSpec(head_density=(0.05, 0.6)), num_layers=3, num_q_heads=12,
                      num_kv_heads=6, head_dim=64, tile=64)


def shard_layout(lay, la, ca, h0, h1):
    la_off, ca_off, la_s, ca_s = shard_bits(lay.cu_seqlens, lay.doc_cu, lay.doc_end, lay.la_off,
                                            lay.ca_off, la, ca, lay.num_layers,
                                            lay.num_kv_heads, lay.tile, h0, h1)
    G = lay.num_q_heads // lay.num_kv_heads
    sub = W.Layout(num_prompts=lay.num_prompts, num_docs=lay.num_docs,
                   num_layers=lay.num_layers, num_q_heads=(h1 - h0) * G,
                   num_kv_heads=h1 - h0, head_dim=lay.head_dim, tile=lay.tile,
                   total_tokens=lay.total_tokens, max_tiles_per_prompt=lay.max_tiles_per_prompt,
                   cu_seqlens=lay.cu_seqlens, doc_cu=lay.doc_cu, doc_end=lay.doc_end,
                   la_off=la_off, ca_off=ca_off, la_words_len=len(la_s), ca_words_len=len(ca_s))
    return sub, la_s, ca_s


@pytest.mark.parametrize("world", [1, 2, 3, 4, 6])
def test_shards_decode_to_the_head_slices(world):
    lay = W.make_layout(CFG)
    la, ca = W.make_bits(CFG, lay)
    kv, cnt = oracle.decode(lay, la, ca)
    covered = []
    for r in range(world):
        h0, h1 = kv_head_range(r, world, lay.num_kv_heads)
        covered += list(range(h0, h1))
        sub, la_s, ca_s = shard_layout(lay, la, ca, h0, h1)
        kv_s, cnt_s = oracle.decode(sub, la_s, ca_s)
        assert np.array_equal(cnt_s, cnt[:, h0:h1])
        assert np.array_equal(kv_s, kv[:, h0:h1])
    assert covered == list(range(lay.num_kv_heads))


def test_head_ranges_balanced():
    for world in range(1, 9):
        sizes = [np.subtract(*kv_head_range(r, world, 8)[::-1]) for r in range(world)]
        assert sum(sizes) == 8 and max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        h0, h1 = kv_head_range(rank, world, 8)
        total = bench.sum_over_ranks(float(h1 - h0), dist, "cpu")
        q.put((rank, h0, h1, total))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_cover_all_heads():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [(g[1], g[2]) for g in got] == [(0, 4), (4, 8)]
    assert all(g[3] == 8.0 for g in got)

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


RG = W.custom_config("shard_cpu_rg", [([250, 513, 77], 45), ([190], 0), ([], 30)],
                     W.BitSpec(la_p=0.4, ca_p=0.3), num_layers=2, num_q_heads=12,
                     num_kv_heads=6, head_dim=64, tile=64, page=8)


@pytest.mark.parametrize("world", [2, 3, 6])
def test_general_layout_shards_decode_to_the_head_slices(world):
    """Ragged documents, 8-token pages (gathered): each shard's re-packed words decode to
    the head slice of the unsharded lists, page starts included."""
    lay = W.make_layout(RG)
    la, ca = W.make_bits(RG, lay)
    qt, kv, cnt, pg = oracle.decode_ragged(lay, la, ca)
    G = lay.num_q_heads // lay.num_kv_heads
    for r in range(world):
        h0, h1 = kv_head_range(r, world, lay.num_kv_heads)
        la_off, ca_off, la_s, ca_s = shard_bits(lay.cu_seqlens, lay.doc_cu, lay.doc_end,
                                                lay.la_off, lay.ca_off, la, ca, lay.num_layers,
                                                lay.num_kv_heads, lay.tile, h0, h1, page=8)
        import dataclasses
        sub = dataclasses.replace(lay, num_q_heads=(h1 - h0) * G, num_kv_heads=h1 - h0,
                                  la_off=la_off, ca_off=ca_off, la_words_len=len(la_s),
                                  ca_words_len=len(ca_s))
        qt_s, kv_s, cnt_s, pg_s = oracle.decode_ragged(sub, la_s, ca_s)
        assert np.array_equal(qt_s, qt)
        assert np.array_equal(cnt_s, cnt[:, h0:h1])
        H = h1 - h0
        for l in range(lay.num_layers):
            for hh in range(H):
                for q in range(len(qt)):
                    n = cnt_s[l, hh, q]
                    for (f, info), (f0, info0) in zip(kv_s[l, hh, q, :n], kv[l, h0 + hh, q, :n]):
                        assert info == info0
                        if (int(info) >> 9) & 1:   # gathered: compare the pages themselves
                            npg = (int(info) & 0xFF) // 8
                            a = pg_s[l].reshape(-1)[f: f + npg]
                            b = pg[l].reshape(-1)[f0: f0 + npg]
                            assert np.array_equal(a, b)
                        else:
                            assert f == f0


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

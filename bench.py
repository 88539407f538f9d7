"""Benchmark of the SIFT online-prefill hot path on GB300.

One step = the whole hot path over one batch: ``sift_decode`` of the bit
vectors of every layer (one decode + one schedule launch), then
``sift_sparse_prefill`` for every layer (fresh seeded Q/K/V per layer, resident
in HBM).  Default workload: Llama-3.1-8B heads (32 q / 8 kv, d = 128), one
prompt of 16 docs x 2048 tokens + 256-token query (33,024 tokens), 32 layers,
per-(layer, kv head) LA density U[0.05, 0.35] and CA half of it, tile 128.

Metric: sparse-prefill attention TFLOP/s counting every computed tile at
4*B^2*d per query head (diagonal tiles in full), plus ms per layer against the
dense causal kernel on the same GPU.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload (replicas,
weak scaling, no collective on the data path); timing is the max over ranks.
``--impl reference`` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "sparse-prefill attention TFLOP/s (computed tiles) & % bf16 peak; ms per layer vs dense"
UNIT = "TFLOP/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "sift_sparse_prefill_llama_32k.md")
PROFILE_RAGGED = os.path.join(ROOT, "profiles", "sift_sparse_prefill_ragged_llama_32k_ragged.md")


def profile_summary(workload: str) -> str:
    """Committed ncu summary of the sparse kernel on `workload` (it may not exist)."""
    if workload == "llama_32k":
        return PROFILE_SUMMARY
    if workload == "llama_32k_ragged":
        return PROFILE_RAGGED
    return os.path.join(ROOT, "profiles", f"sift_sparse_prefill_{workload}.md")


def tile_flops(cfg) -> float:
    """FLOPs of one computed tile for one query head: QK^T and PV, 2*B*B*d each."""
    return 4.0 * cfg.tile * cfg.tile * cfg.head_dim


def computed_flops(cfg, counts: np.ndarray) -> np.ndarray:
    """Per-layer FLOPs over computed tiles: sum of row counts x query heads per kv head."""
    G = cfg.num_q_heads // cfg.num_kv_heads
    return counts.reshape(counts.shape[0], -1).sum(axis=1).astype(np.float64) * G * tile_flops(cfg)


def decode_bytes(lay, counts: np.ndarray) -> float:
    """Algorithmic bytes of one decode of all layers: LA/CA words read, kv entries, counts
    and schedule written, counts read again by the schedule."""
    units = counts.size
    return float(8 * (lay.la_words_len + lay.ca_words_len) + 4 * int(counts.sum()) +
                 4 * units + 4 * units + 4 * units)


def decode_launches(lay) -> int:
    """Kernel launches of one sift_decode call (the library's rule): one while the
    schedule blocks' shared memory -- (rowcap + 1 + Hkv*D + 2*D + N) x 4 bytes, plus
    Hkv*N x 4 for the counts when the total stays within 226 KB -- fits in 32 KB, else
    two."""
    base = 4 * (lay.max_tiles_per_prompt + 1 + lay.num_kv_heads * lay.num_docs +
                2 * lay.num_docs + lay.num_tiles)
    cnt = 4 * lay.num_kv_heads * lay.num_tiles
    need = base + (cnt if base + cnt <= 226 * 1024 else 0)
    return 1 if need <= 32 * 1024 else 2


def useful_fraction(cfg, lay, flops_step: float) -> float:
    """Share of the computed-tile FLOPs that are not masked out on the diagonal: every row
    holds one diagonal tile, of which (B+1)/(2B) is causal."""
    B = cfg.tile
    G = cfg.num_q_heads // cfg.num_kv_heads
    diag = cfg.num_layers * cfg.num_kv_heads * lay.num_tiles * G * tile_flops(cfg)
    return (flops_step - diag * (B - 1) / (2 * B)) / flops_step


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def tensor_roofline(achieved: float, kernel: str, traffic, clocks=None) -> dict:
    """Roofline entry of a tensor-bound kernel.  Each launch lasts about a millisecond and
    the timed step tens of milliseconds, so the denominator is the burst bf16 rate (a
    matmul timed on its own); the ratio to the sustained rate (seconds of back-to-back
    matmuls under the power cap, at a lower clock) is kept beside it.  With the clocks
    sampled during the timed region, `achieved_at_max_clock` scales the rate to the
    maximum SM clock (rate / (median MHz / max MHz))."""
    peaks, src = load_peaks()
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    r = {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
         "frac": achieved / burst, "traffic": traffic, "kernel": kernel,
         "peak_source": f"bf16_tflops (burst) of {src}",
         "peak_sustained": sustained, "frac_of_sustained": achieved / sustained}
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        scale = float(clocks["sm_mhz"]) / float(clocks["sm_max_mhz"])
        r["achieved_at_max_clock"] = achieved / scale
        r["frac_at_max_clock"] = achieved / scale / burst
    return r


def _code_only(text: str) -> str:
    """C/C++ source without its comments, whitespace runs collapsed to one space (string
    and character literals are kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest() -> str:
    """Digest of the attention kernel's code (its sources without comments or layout), so
    that a profile summary stays matched to the code it was captured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_vector_guided_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("sift_attention") or name == "ptx.cuh":
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(path, workload):
    """DRAM bytes per launch of the sparse kernel from a committed ncu summary, if it was
    taken on the current kernel source and on this workload (else None)."""
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, _, v = line.strip()[2:].partition(":")
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_digest():
        return None
    if vals.get("workload") != workload:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle legs

def oracle_sample(cfg, lay, la, ca, q, k, v, counts, budget_s: float, seed: int = 7):
    """Time the oracle on (query tile, query head) pairs of layer 0 until ~budget_s of CPU
    work; returns (flops counted as computed tiles, seconds, threads, pairs)."""
    import oracle
    threads = oracle.set_threads(0)
    rng = np.random.default_rng(seed)
    B, G = cfg.tile, cfg.num_q_heads // cfg.num_kv_heads
    N = lay.num_tiles
    flops = secs = 0.0
    pairs = 0
    batch = 1
    while secs < budget_s and pairs < 4096:
        sel = [(int(rng.integers(N)), int(rng.integers(cfg.num_q_heads))) for _ in range(batch)]
        tok = np.concatenate([np.arange(i * B, (i + 1) * B) for i, _ in sel]).astype(np.int32)
        head = np.concatenate([np.full(B, h) for _, h in sel]).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attention_rows(lay, la, ca, 0, q, k, v, tok, head)
        secs += time.perf_counter() - t0
        flops += sum(float(counts[0, h // G, i]) for i, h in sel) * tile_flops(cfg)
        pairs += batch
        batch = min(batch * 2, 64)
    return flops, secs, threads, pairs


def host_inputs_layer0(cfg):
    import torch
    return W.make_qkv(cfg, 0, device="cpu")


def run_reference(args, cfg):
    """--impl reference: the CPU oracle on a bounded sample of the same workload."""
    import oracle
    _, rank, _ = rank_env()
    if rank != 0:
        return 0
    oracle.build()
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    _, counts = oracle.decode(lay, la, ca)
    q, k, v = host_inputs_layer0(cfg)
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(cfg, lay, la, ca, q, k, v, counts, per_step / 4, seed=1)
    tot_f = tot_s = 0.0
    tot_pairs = 0
    threads = 1
    for s in range(args.steps):
        f, sec, threads, pairs = oracle_sample(cfg, lay, la, ca, q, k, v, counts, per_step,
                                               seed=100 + s)
        tot_f += f
        tot_s += sec
        tot_pairs += pairs
    value = tot_f / tot_s / 1e12
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, args, lay),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{tot_pairs} random (query tile, query head) pairs of "
                                   f"layer 0 ({cfg.tile} rows each), ~{per_step:.0f} s per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


def config_dict(cfg, args, lay):
    return {"workload": cfg.name, "description": cfg.description, "tokens": lay.total_tokens,
            "layers": cfg.num_layers, "q_heads": cfg.num_q_heads, "kv_heads": cfg.num_kv_heads,
            "head_dim": cfg.head_dim, "tile": cfg.tile, "prompts": lay.num_prompts,
            "docs": lay.num_docs,
            "l2": "inputs larger than L2: each layer's Q/K/V/O (> 129 MB) is distinct and "
                  "the step cycles through every layer",
            "parallelism": (f"kv-head shards x{args.gpus}" if args.shard == "heads" else
                            f"replicas x{args.gpus}") if args.gpus > 1 else "single GPU"}


# ----------------------------------------------------------------------------- multi-rank helpers

def rank_env():
    """(world, rank, local_rank) from the torchrun environment (1, 0, 0 when absent)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` over all ranks (identity without a process group).  The
    timed region is judged by its slowest rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device) -> float:
    """Sum of `value` over all ranks (identity without a process group)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, steps: int, max_seconds: float,
                     world: int) -> float:
    """Replicas: every rank processes the same per-GPU workload (weak scaling), so the
    job's throughput is all ranks' work over the slowest rank's time."""
    return world * flops_per_rank_step * steps / max_seconds / 1e12


# ----------------------------------------------------------------------------- GPU leg

def run_ours(args, cfg):
    import torch
    import bit_vector_guided_gb300 as sift
    from bit_vector_guided_gb300 import build as sbuild

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        sbuild.build()
    if dist is not None:
        dist.barrier()
    sift.load_library()

    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    L = cfg.num_layers
    shard = args.shard == "heads" and world > 1
    if shard:
        # this rank's kv heads (and their query heads) as an independent problem
        import dataclasses
        from bit_vector_guided_gb300.sharding import kv_head_range, shard_bits
        full = cfg
        h0, h1 = kv_head_range(rank, world, full.num_kv_heads)
        G = full.num_q_heads // full.num_kv_heads
        cfg = dataclasses.replace(full, num_q_heads=(h1 - h0) * G, num_kv_heads=h1 - h0)
        la_off, ca_off, la, ca = shard_bits(lay.cu_seqlens, lay.doc_cu, lay.doc_end, lay.la_off,
                                            lay.ca_off, la, ca, L, full.num_kv_heads,
                                            full.tile, h0, h1)
        lay = dataclasses.replace(lay, num_q_heads=cfg.num_q_heads,
                                  num_kv_heads=cfg.num_kv_heads, la_off=la_off, ca_off=ca_off,
                                  la_words_len=len(la), ca_words_len=len(ca))
        sl = ((h0 * G, h1 * G), (h0, h1), (h0, h1))
        qkv = [tuple(t[:, a:b].contiguous() for t, (a, b) in zip(W.make_qkv(full, l, device=dev), sl))
               for l in range(L)]
    else:
        qkv = [W.make_qkv(cfg, l, device=dev) for l in range(L)]
    prob = sift.SiftProblem.from_layout(lay, dev)
    la_d = torch.from_numpy(np.ascontiguousarray(la).view(np.int64)).to(dev)
    ca_d = torch.from_numpy(np.ascontiguousarray(ca).view(np.int64)).to(dev)
    outs = [(torch.empty_like(q), torch.empty((cfg.num_q_heads, lay.total_tokens),
                                              dtype=torch.float32, device=dev))
            for q, _, _ in qkv]
    H, N, R = cfg.num_kv_heads, lay.num_tiles, lay.max_tiles_per_prompt
    kv_idx = torch.empty((L, H, N, R), dtype=torch.int32, device=dev)
    counts = torch.empty((L, H, N), dtype=torch.int32, device=dev)
    sched = torch.empty((L, H * N), dtype=torch.int32, device=dev)
    status = prob.new_status()
    ws = prob.new_workspace()
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        if events is not None:
            events[0].record(stream)
        sift.decode(prob, la_d, ca_d, kv_idx, counts, sched, dev_status=status, stream=stream)
        if events is not None:
            events[1].record(stream)
        for l in range(L):
            q, k, v = qkv[l]
            o, lse = outs[l]
            sift.sparse_prefill(prob, l, q, k, v, kv_idx, counts, sched, 0.0, o, lse, ws,
                                status, stream)
            if events is not None:
                events[2 + l].record(stream)

    # warm-up (also fills counts for the FLOP count)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError("device status " + sift.status_string(int(status.item())))
    counts_h = counts.cpu().numpy()
    flops_layer = computed_flops(cfg, counts_h)
    flops_step = float(flops_layer.sum())

    # timed region: K steps, events per launch on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(L + 2)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        for s in range(args.steps):
            step(ev[s])
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    if int(status.item()) != 0:
        raise RuntimeError("device status " + sift.status_string(int(status.item())))
    decode_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    layer_ms = np.array([[ev[s][1 + l].elapsed_time(ev[s][2 + l]) for l in range(L)]
                         for s in range(args.steps)])
    ms_per_step = total_ms / args.steps
    if shard:  # strong scaling: the ranks' shards add up to one problem
        job_flops_step = sum_over_ranks(flops_step, dist, dev)
    else:      # replicas: every rank runs the whole workload
        job_flops_step = world * flops_step
    value = whole_job_tflops(job_flops_step, args.steps, total_ms * 1e-3, 1)
    kern_ms = float(layer_ms.mean())
    achieved = float(flops_layer.mean()) / (kern_ms * 1e-3) / 1e12

    traffic = None if shard else profiled_traffic(profile_summary(cfg.name), cfg.name)

    # decode fused into the prefill: the same step without a separate decode, timed over
    # as many steps as the main measurement and alternating with decode + sparse steps
    # (the GPU's speed drifts by a few percent within a run, so the two are compared
    # side by side rather than minutes apart)
    def fused_step():
        for l in range(L):
            q, k, v = qkv[l]
            o, lse = outs[l]
            sift.fused_prefill(prob, l, la_d, ca_d, q, k, v, 0.0, o, lse, ws, status, stream)

    fused_step()
    pair_ms = {"fused": [], "decoded": []}
    for _ in range(max(3, min(args.steps, 10))):
        for name, fn in (("fused", fused_step), ("decoded", step)):
            fz0, fz1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fz0.record(stream)
            fn()
            fz1.record(stream)
            torch.cuda.synchronize(dev)
            pair_ms[name].append(fz0.elapsed_time(fz1))
    if int(status.item()) != 0:
        raise RuntimeError("device status " + sift.status_string(int(status.item())))
    fused_ms_step = float(np.mean(pair_ms["fused"]))
    fused_vs_decoded = fused_ms_step / float(np.mean(pair_ms["decoded"]))

    # offline bit builder (one layer), outside the timed region: into scratch words
    max_doc_tiles = max([(int(lay.doc_end[g]) - lay.doc_start(g)) // cfg.tile
                         for g in range(lay.num_docs)] or [1])
    bl_la, bl_ca = torch.zeros_like(la_d), torch.zeros_like(ca_d)
    bws = torch.empty(max(16, (sift.build_bits_workspace_bytes(prob, max_doc_tiles) + 15)
                          // 16 * 16), dtype=torch.uint8, device=dev)
    build_ms = []
    for rep in range(3):
        q0, k0, _ = qkv[0]
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        sift.build_bits(prob, 0, q0, k0, max_doc_tiles, 0.2, 0.1, bl_la, bl_ca, 0.0, bws,
                        status, stream)
        b1.record(stream)
        torch.cuda.synchronize(dev)
        if rep > 0:
            build_ms.append(b0.elapsed_time(b1))
    build_ms_layer = float(np.mean(build_ms))
    del bws, bl_la, bl_ca

    # dense baseline on the same GPU (a few layers), outside the timed region
    dense_layers = list(range(min(L, 4)))
    dense_ms = []
    for rep in range(3):
        for l in dense_layers:
            q, k, v = qkv[l]
            o, lse = outs[l]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            sift.dense_prefill(prob, q, k, v, 0.0, o, lse, ws, status, stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep > 0:
                dense_ms.append(e0.elapsed_time(e1))
    dense_ms_layer = float(np.mean(dense_ms))
    G = cfg.num_q_heads // cfg.num_kv_heads
    dense_flops_layer = float(sum(
        (n * (n + 1) // 2) for n in np.diff(lay.cu_seqlens) // cfg.tile)) * H * G * tile_flops(cfg)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if shard else "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(cfg, args, lay),
        "gpu_launches": args.steps * (decode_launches(lay) + L),
        "sparse_ms_per_layer": kern_ms,
        "sparse_ms_per_layer_p90": float(np.percentile(layer_ms.mean(axis=0), 90)),
        "dense_ms_per_layer": dense_ms_layer,
        "dense_tflops": dense_flops_layer / (dense_ms_layer * 1e-3) / 1e12,
        "speedup_vs_dense": dense_ms_layer / kern_ms,
        "computed_tile_fraction": float(flops_layer.mean() / dense_flops_layer),
        "decode_us": 1e3 * float(np.median(decode_ms)),
        # decode's algorithmic bytes: every bit word read once; lists, counts and the
        # schedule written once (counts read back by the schedule)
        "decode_gbs": decode_bytes(lay, counts_h) / (float(np.median(decode_ms)) * 1e-3) / 1e9,
        "decode_bytes": decode_bytes(lay, counts_h),
        "decode_note": "decode_gbs: algorithmic bytes over CUDA-event time; the launch's "
                       "duration and DRAM bytes from ncu are in "
                       "profiles/sift_decode_llama_32k.md (the lists stay in L2)",
        # diagonal tiles counted at the (B+1)/(2B) of their entries that are causal
        "useful_tflops": value * useful_fraction(cfg, lay, flops_step),
        "fused_ms_per_step": fused_ms_step,
        "fused_vs_decoded": fused_vs_decoded,
        "fused_ms_per_layer": fused_ms_step / L,
        "fused_tflops": flops_step / (fused_ms_step * 1e-3) / 1e12,
        "decode_launches_per_step": decode_launches(lay),
        "build_bits_ms_per_layer": build_ms_layer,
    }
    clocks = clk.summary()
    result["clocks"] = clocks
    result["roofline"] = tensor_roofline(achieved, "sift_sparse_prefill", traffic, clocks)

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, cfg, lay, prob, la, ca, qkv, outs, kv_idx, counts, sched,
                                status, ws, stream, dev, job_flops_step, dist)
    if not args.no_sweep and rank == 0 and world == 1:
        result["density_sweep"] = run_sweep(args, dev, stream)
    del qkv, outs
    torch.cuda.empty_cache()
    if not args.no_ragged and rank == 0 and world == 1 and not args.layers:
        result["ragged"] = run_ragged(args, dev, stream)
        torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        q0, k0, v0 = host_inputs_layer0(cfg)
        _, counts_o = oracle.decode(lay, la, ca)
        f, sec, thr, pairs = oracle_sample(cfg, lay, la, ca, q0, k0, v0, counts_o,
                                           args.cpu_seconds)
        result["cpu_baseline"] = {
            "value": f / sec / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"{pairs} random (query tile, query head) pairs of layer 0, "
                      f"{cfg.tile} query rows each, {sec:.1f} s on {thr} threads"}
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))
    return 0


def run_e2e(args, cfg, lay, prob, la, ca, qkv, outs, kv_idx, counts, sched, status, ws, stream,
            dev, job_flops_step, dist):
    """Same metric through the public API with host buffers: every step copies that step's
    inputs (bits of all layers + Q/K/V of every layer) from pinned host memory and reads
    every layer's O and LSE back to pinned host memory."""
    import torch
    import bit_vector_guided_gb300 as sift
    L = cfg.num_layers
    la_h = torch.from_numpy(np.ascontiguousarray(la).view(np.int64)).pin_memory()
    ca_h = torch.from_numpy(np.ascontiguousarray(ca).view(np.int64)).pin_memory()
    la_d = torch.empty_like(la_h, device=dev)
    ca_d = torch.empty_like(ca_h, device=dev)
    host_in = [tuple(t.cpu().pin_memory() for t in qkv[l]) for l in range(L)]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                 torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for o, lse in outs]
    h2d = (la_h.numel() + ca_h.numel()) * 8 + sum(t.numel() * t.element_size()
                                                  for tri in host_in for t in tri)
    d2h = sum(o.numel() * o.element_size() + s.numel() * s.element_size() for o, s in host_out)
    up = torch.cuda.Stream(dev)    # host -> device
    down = torch.cuda.Stream(dev)  # device -> host, so both directions of the link overlap
    done_in = [torch.cuda.Event() for _ in range(L)]
    done_kern = [torch.cuda.Event() for _ in range(L)]
    done_down = [torch.cuda.Event() for _ in range(L)]
    done_decode = torch.cuda.Event()

    def step():
        # Each buffer waits only for its own last reader or writer, so consecutive steps
        # pipeline and both copy directions stay busy: a layer's Q/K/V upload waits for that
        # layer's kernel of the previous step, its kernel waits for the previous read-back of
        # its O/LSE, and the bits upload waits for the previous decode.
        up.wait_event(done_decode)
        with torch.cuda.stream(up):
            la_d.copy_(la_h, non_blocking=True)
            ca_d.copy_(ca_h, non_blocking=True)
        ev_bits = torch.cuda.Event()
        ev_bits.record(up)
        for l in range(L):
            up.wait_event(done_kern[l])
            with torch.cuda.stream(up):
                for dst, src in zip(qkv[l], host_in[l]):
                    dst.copy_(src, non_blocking=True)
                done_in[l].record(up)
        stream.wait_event(ev_bits)
        sift.decode(prob, la_d, ca_d, kv_idx, counts, sched, dev_status=status, stream=stream)
        done_decode.record(stream)
        for l in range(L):
            stream.wait_event(done_in[l])
            stream.wait_event(done_down[l])
            q, k, v = qkv[l]
            o, lse = outs[l]
            sift.sparse_prefill(prob, l, q, k, v, kv_idx, counts, sched, 0.0, o, lse, ws,
                                status, stream)
            done_kern[l].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done_kern[l])
                host_out[l][0].copy_(o, non_blocking=True)
                host_out[l][1].copy_(lse, non_blocking=True)
                done_down[l].record(down)

    # The host link's own floor for these bytes: the same copies on the same two streams
    # (uploads on one, read-backs on the other, running at once), with no kernels.
    def copies_only():
        with torch.cuda.stream(up):
            la_d.copy_(la_h, non_blocking=True)
            ca_d.copy_(ca_h, non_blocking=True)
            for l in range(L):
                for dst, src in zip(qkv[l], host_in[l]):
                    dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(down):
            for l in range(L):
                host_out[l][0].copy_(outs[l][0], non_blocking=True)
                host_out[l][1].copy_(outs[l][1], non_blocking=True)

    def copy_reps(n):
        out = []
        for _ in range(n):
            t1 = time.perf_counter()
            copies_only()
            torch.cuda.synchronize(dev)
            out.append(time.perf_counter() - t1)
        return out

    steps = max(1, min(args.steps, 5))
    # The link's speed swings from moment to moment on a shared host (copy repetitions of
    # one run have differed by 40%), so the floor is the median of repetitions timed before
    # and just after the e2e steps; their fastest and their mean are reported too.  The
    # first copy-only repetition after kernels ran, and the first step with kernels after
    # copy-only traffic, each took about 130 ms longer than the rest, so the e2e warm-up
    # steps run after the copy-only repetitions, directly before the timed steps.
    copies_only()
    torch.cuda.synchronize(dev)
    reps = copy_reps(5)
    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    el = max_over_ranks(time.perf_counter() - t0, dist, dev)
    reps += copy_reps(5)
    floor = max_over_ranks(statistics.median(reps), dist, dev)
    floor_min = max_over_ranks(min(reps), dist, dev)
    floor_mean = max_over_ranks(sum(reps) / len(reps), dist, dev)
    return {"value": whole_job_tflops(job_flops_step, steps, el, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": 1e3 * el / steps, "steps": steps,
            "link_floor_ms_per_step": 1e3 * floor,
            "link_fastest_ms_per_step": 1e3 * floor_min,
            "link_mean_ms_per_step": 1e3 * floor_mean,
            "link_reps_ms": [round(1e3 * r, 2) for r in reps],
            "ratio_to_link_mean": (el / steps) / floor_mean,
            "link_gbs": (h2d + d2h) / floor / 1e9,
            "ratio_to_link_floor": (el / steps) / floor,
            "note": "pinned host buffers; H2D of each layer's Q/K/V on one copy stream and "
                    "D2H of its O/LSE on another, both overlapping the kernels; consecutive "
                    "steps pipeline (each buffer waits only for its own last use). "
                    "link_floor_ms_per_step: the same copies alone on the same streams, "
                    "both directions at once, no kernels: the median of 10 repetitions "
                    "timed just before and after the e2e steps (link_fastest / link_mean: "
                    "their fastest and their mean; link_reps_ms: each of them, since the "
                    "link's speed can switch between states during a run)"}


def run_sweep(args, dev, stream):
    """Sparse vs dense at each LA=CA density of the batch-of-4 configuration."""
    import torch
    import bit_vector_guided_gb300 as sift
    rows = []
    base = W.get_config("batch4_p100")
    q, k, v = W.make_qkv(base, 0, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((base.num_q_heads, base.total_tokens), dtype=torch.float32, device=dev)
    dense_ms = None
    for name in ("batch4_p005", "batch4_p010", "batch4_p020", "batch4_p040", "batch4_p070",
                 "batch4_p100"):
        cfg = W.get_config(name)
        lay = W.make_layout(cfg)
        la, ca = W.make_bits(cfg, lay)
        prob = sift.SiftProblem.from_layout(lay, dev)
        la_d = torch.from_numpy(np.ascontiguousarray(la).view(np.int64)).to(dev)
        ca_d = torch.from_numpy(np.ascontiguousarray(ca).view(np.int64)).to(dev)
        st = prob.new_status()
        ws = prob.new_workspace()
        kv, cnt, sch = sift.decode(prob, la_d, ca_d, dev_status=st, stream=stream)

        def timed(fn, reps=5):
            for _ in range(2):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / reps

        sp = timed(lambda: sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sch, 0.0, o, lse, ws,
                                               st, stream))
        if dense_ms is None:
            dense_ms = timed(lambda: sift.dense_prefill(prob, q, k, v, 0.0, o, lse, ws, st,
                                                        stream))
        fl = float(computed_flops(cfg, cnt.cpu().numpy())[0])
        rows.append({"workload": name, "density": cfg.bits.la_p, "sparse_ms": sp,
                     "dense_ms": dense_ms, "speedup": dense_ms / sp,
                     "sparse_tflops": fl / (sp * 1e-3) / 1e12})
        if int(st.item()) != 0:
            raise RuntimeError("sweep device status " + sift.status_string(int(st.item())))
    return rows


def run_ragged(args, dev, stream, cfg=None, steps=3, warmup=2):
    """The general-layout step on a ragged workload (default: the ragged 33K one):
    sift_decode_ragged of all layers, then one sift_sparse_prefill_ragged per layer; dense
    causal attention over the same prompts (documents play no part in it) is timed beside
    it."""
    import torch
    import bit_vector_guided_gb300 as sift
    cfg = cfg or W.get_config("llama_32k_ragged")
    L = cfg.num_layers
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, dev)
    la_d = torch.from_numpy(np.ascontiguousarray(la).view(np.int64)).to(dev)
    ca_d = torch.from_numpy(np.ascontiguousarray(ca).view(np.int64)).to(dev)
    qkv = [W.make_qkv(cfg, l, device=dev) for l in range(L)]
    o = torch.empty_like(qkv[0][0])
    lse = torch.empty((cfg.num_q_heads, lay.total_tokens), dtype=torch.float32, device=dev)
    st = prob.new_status()
    ws = prob.new_workspace()
    H, NQ, R = cfg.num_kv_heads, prob.num_query_tiles, prob.max_tiles_per_prompt
    qt = torch.empty((NQ, 2), dtype=torch.int32, device=dev)
    kv = torch.empty((L, H, NQ, R, 2), dtype=torch.int32, device=dev)
    cnt = torch.empty((L, H, NQ), dtype=torch.int32, device=dev)
    sch = torch.empty((L, H * NQ), dtype=torch.int32, device=dev)
    pages = (torch.empty((L, H, lay.num_docs, prob.page_cap), dtype=torch.int32, device=dev)
             if prob.page_cap > 0 else None)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(L + 2)]

    def step(record=False):
        if record:
            ev[0].record(stream)
        sift.decode_ragged(prob, la_d, ca_d, qt, kv, cnt, sch, pages, dev_status=st,
                           stream=stream)
        if record:
            ev[1].record(stream)
        for l in range(L):
            q, k, v = qkv[l]
            sift.sparse_prefill_ragged(prob, l, q, k, v, qt, kv, cnt, sch, pages, 0.0, o, lse,
                                       ws, st, stream)
            if record:
                ev[2 + l].record(stream)

    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize(dev)
    layer_ms, dec_ms, step_ms = [], [], []
    for _ in range(steps):
        step(record=True)
        torch.cuda.synchronize(dev)
        dec_ms.append(ev[0].elapsed_time(ev[1]))
        layer_ms += [ev[1 + l].elapsed_time(ev[2 + l]) for l in range(L)]
        step_ms.append(ev[0].elapsed_time(ev[L + 1]))
    if int(st.item()) != 0:
        raise RuntimeError("ragged device status " + sift.status_string(int(st.item())))
    fl = computed_flops(cfg, cnt.cpu().numpy())
    kern_ms = float(np.mean(layer_ms))
    # dense causal attention over the same prompts: an aligned problem without documents
    dprob = sift.SiftProblem(cu_seqlens=lay.cu_seqlens,
                             doc_cu=np.zeros(lay.num_prompts + 1, np.int32), doc_end=[],
                             la_off=[], ca_off=[], num_layers=1, num_q_heads=cfg.num_q_heads,
                             num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim,
                             tile=cfg.tile, la_words_len=0, ca_words_len=0, device=dev)
    dws = dprob.new_workspace()
    q, k, v = qkv[0]
    for _ in range(2):
        sift.dense_prefill(dprob, q, k, v, 0.0, o, lse, dws, st, stream)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(3):
        sift.dense_prefill(dprob, q, k, v, 0.0, o, lse, dws, st, stream)
    d1.record(stream)
    torch.cuda.synchronize(dev)
    dense_ms = d0.elapsed_time(d1) / 3
    peak = float(load_peaks()[0].get("bf16_tflops"))
    ktf = float(fl.mean()) / (kern_ms * 1e-3) / 1e12
    return {"workload": cfg.name, "page": cfg.page, "query_tiles": NQ, "layers": L,
            "flops_per_step": float(fl.sum()),
            "ms_per_step": float(np.mean(step_ms)),
            "tflops": float(fl.sum()) / (float(np.mean(step_ms)) * 1e-3) / 1e12,
            "sparse_ms_per_layer": kern_ms, "kernel_tflops": ktf,
            "kernel_frac_of_peak": ktf / peak,
            "decode_us": 1e3 * float(np.median(dec_ms)),
            "dense_ms_per_layer": dense_ms, "speedup_vs_dense": dense_ms / kern_ms,
            "gpu_launches_per_step": 3 + L}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama_32k", choices=sorted(W.CONFIGS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the general-layout leg (ragged documents, 16-token CA pages)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: every rank runs the whole workload (replicas, weak scaling) "
                         "or one range of kv heads of it (heads, strong scaling)")
    ap.add_argument("--decode-only", action="store_true",
                    help="profiling: time only sift_decode of the workload's bits (no Q/K/V "
                         "on the device); prints its own JSON line")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: keep the first N layers of the workload (the JSON "
                         "line then names the reduced workload)")
    args = ap.parse_args(argv)
    if args.warmup < 1:
        ap.error("--warmup must be >= 1 (timed runs use >= 3)")
    cfg = W.get_config(args.config)
    if args.layers and args.layers < cfg.num_layers:
        import dataclasses
        cfg = dataclasses.replace(cfg, num_layers=args.layers,
                                  name=f"{cfg.name}", description=cfg.description +
                                  f" [first {args.layers} layers only]")
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.decode_only:
        return run_decode_only(args, cfg)
    if not W.make_layout(cfg).aligned:
        return run_ragged_line(args, cfg)
    return run_ours(args, cfg)


def run_decode_only(args, cfg):
    """sift_decode of every layer of the workload, alone: W warm-up and K timed calls,
    CUDA events on the launching stream.  Only the bit words,
    the lists, the counts and the schedule live on the device, so a profiler can capture
    these launches at full size cheaply."""
    import torch
    import bit_vector_guided_gb300 as sift
    from bit_vector_guided_gb300 import build as sbuild
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sbuild.build()
    sift.load_library()
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, dev)
    la_d = torch.from_numpy(np.ascontiguousarray(la).view(np.int64)).to(dev)
    ca_d = torch.from_numpy(np.ascontiguousarray(ca).view(np.int64)).to(dev)
    L, H, N, R = cfg.num_layers, cfg.num_kv_heads, lay.num_tiles, lay.max_tiles_per_prompt
    kv = torch.empty((L, H, N, R), dtype=torch.int32, device=dev)
    cnt = torch.empty((L, H, N), dtype=torch.int32, device=dev)
    sch = torch.empty((L, H * N), dtype=torch.int32, device=dev)
    st = prob.new_status()
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        sift.decode(prob, la_d, ca_d, kv, cnt, sch, dev_status=st, stream=stream)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    # keep the GPU busy while the host queues every timed call, so that the events measure
    # the device and not the host's launch rate
    torch.cuda._sleep(int(2e7))
    ev[0].record(stream)
    for s_ in range(args.steps):
        sift.decode(prob, la_d, ca_d, kv, cnt, sch, dev_status=st, stream=stream)
        ev[s_ + 1].record(stream)
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError("device status " + sift.status_string(int(st.item())))
    us = [1e3 * ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    nbytes = decode_bytes(lay, cnt.cpu().numpy())
    med = float(np.median(us))
    print(json.dumps({"metric": "sift_decode us (all layers, one call)", "value": med,
                      "unit": "us", "higher_is_better": False, "steps": args.steps,
                      "warmup": args.warmup, "decode_bytes": nbytes,
                      "decode_gbs": nbytes / (med * 1e-6) / 1e9,
                      "config": config_dict(cfg, args, lay)}))
    return 0


def run_ragged_line(args, cfg):
    """A workload of the general layout as the measured step (one GPU): one JSON line."""
    import torch
    import bit_vector_guided_gb300 as sift
    from bit_vector_guided_gb300 import build as sbuild
    if args.gpus > 1:
        raise SystemExit("the general-layout workloads run on one GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sbuild.build()
    sift.load_library()
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(0) as clk:
        r = run_ragged(args, dev, stream, cfg=cfg, steps=args.steps, warmup=args.warmup)
    lay = W.make_layout(cfg)
    clocks = clk.summary()
    out = {
        "metric": METRIC, "value": r["tflops"], "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(cfg, args, lay),
        "roofline": tensor_roofline(r["kernel_tflops"], "sift_sparse_prefill_ragged",
                                    profiled_traffic(profile_summary(cfg.name), cfg.name),
                                    clocks),
        "gpu_launches": args.steps * r["gpu_launches_per_step"], "ragged": r,
        "clocks": clocks,
    }
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())

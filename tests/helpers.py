"""Shared helpers for the GPU parity tests (inputs from `workloads`, reference from `oracle`)."""
import numpy as np
import torch

import oracle
import workloads as W

# spec tolerances for attention outputs on N(0,1) inputs against the oracle
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_REL = 1e-3


def device_bits(la, ca, device="cuda"):
    """uint64 words -> int64 device tensors holding the same bytes."""
    def up(a):
        a = np.ascontiguousarray(a, np.uint64)
        if a.size == 0:
            a = np.zeros(1, np.uint64)
        return torch.from_numpy(a.view(np.int64)).to(device)
    return up(la), up(ca)


def setup(cfg, device="cuda"):
    import bit_vector_guided_gb300 as sift
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, device)
    la_d, ca_d = device_bits(la, ca, device)
    return lay, la, ca, prob, la_d, ca_d


def check_sched(sched, counts):
    """Each layer's schedule is a permutation of its units with non-increasing counts."""
    L = counts.shape[0]
    flat = counts.reshape(L, -1)
    for l in range(L):
        s = sched[l]
        assert np.array_equal(np.sort(s), np.arange(flat.shape[1])), "sched is not a permutation"
        c = flat[l][s]
        assert np.all(np.diff(c) <= 0), "sched is not longest-first"


def assert_attention_close_scaled(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """The benchmark spec's bounds for inputs that are not N(0,1): each output's error is taken
    relative to max(1, |reference|).  Keys scaled up tile by tile make the softmax peaky,
    so an output row is close to a single value row (|O| up to about 4.5 for N(0,1)
    values), where the bf16 rounding of the output alone reaches half an ulp, 2^-6 =
    0.0156, and that of P (relative 2^-9) adds to it; on N(0,1) inputs (|O| < 1 almost
    everywhere) the bound is the plain one."""
    o = np.asarray(o_gpu, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    rel = np.abs(o - o_ref) / np.maximum(np.abs(o_ref), 1.0)
    _, mean, lrel = attention_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert rel.max() <= MAX_ABS, f"{what}: max scaled error {rel.max():.3g} > {MAX_ABS}"
    assert mean <= MEAN_ABS, f"{what}: mean abs {mean:.3g} > {MEAN_ABS}"
    assert lrel <= LSE_REL, f"{what}: lse rel {lrel:.3g} > {LSE_REL}"
    return float(rel.max()), mean, lrel


def attention_errors(o_gpu, lse_gpu, o_ref, lse_ref):
    """Errors of GPU rows against oracle rows (same shapes, any leading layout)."""
    o = np.asarray(o_gpu, np.float64)
    e = np.abs(o - o_ref)
    lrel = np.abs(np.asarray(lse_gpu, np.float64) - lse_ref) / np.maximum(np.abs(lse_ref), 1e-30)
    return float(e.max()), float(e.mean()), float(lrel.max())


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    mx, mean, lrel = attention_errors(o_gpu, lse_gpu, o_ref, lse_ref)
    assert np.isfinite(np.asarray(o_gpu, np.float64)).all(), f"{what}: non-finite output"
    assert mx <= MAX_ABS, f"{what}: max abs {mx:.3g} > {MAX_ABS}"
    assert mean <= MEAN_ABS, f"{what}: mean abs {mean:.3g} > {MEAN_ABS}"
    assert lrel <= LSE_REL, f"{what}: lse rel {lrel:.3g} > {LSE_REL}"
    return mx, mean, lrel


def sample_pairs(lay, rng, n_random=64):
    """(query tile, query head) pairs to check on a large batch: the first tile of each
    prompt, the last document tile and the last suffix tile of each prompt, plus
    n_random distinct random ones (so at least n_random pairs in all)."""
    B = lay.tile
    Hq = lay.num_q_heads
    pairs = set()
    for p in range(lay.num_prompts):
        t0 = int(lay.cu_seqlens[p]) // B
        t1 = int(lay.cu_seqlens[p + 1]) // B
        docs = range(lay.doc_cu[p], lay.doc_cu[p + 1])
        last_doc_tile = (int(lay.doc_end[docs[-1]]) // B - 1) if len(docs) else t0
        for t in (t0, last_doc_tile, t1 - 1):
            pairs.add((t, int(rng.integers(Hq))))
    N = lay.num_tiles
    target = len(pairs) + min(n_random, N * Hq - len(pairs))
    while len(pairs) < target:
        pairs.add((int(rng.integers(N)), int(rng.integers(Hq))))
    return sorted(pairs)


def compare_decode(lay, kv_gpu, cnt_gpu, kv_o, cnt_o):
    """Decoded lists bit-exact against the oracle's: every count, and every entry up to
    each row's count (entries past it are not written by the kernel)."""
    cnt_g = cnt_gpu.cpu().numpy() if hasattr(cnt_gpu, "cpu") else np.asarray(cnt_gpu)
    kv_g = kv_gpu.cpu().numpy() if hasattr(kv_gpu, "cpu") else np.asarray(kv_gpu)
    assert np.array_equal(cnt_g, cnt_o), "counts differ from the oracle"
    R = kv_o.shape[-1]
    mask = np.arange(R, dtype=np.int32)[None, None, None, :] < cnt_o[..., None]
    assert np.array_equal(np.where(mask, kv_g, -1), kv_o), "lists differ from the oracle"


def oracle_rows_for_pairs(lay, la, ca, layer, q, k, v, pairs):
    B = lay.tile
    tok = np.concatenate([np.arange(i * B, (i + 1) * B) for i, _ in pairs]).astype(np.int32)
    head = np.concatenate([np.full(B, h) for _, h in pairs]).astype(np.int32)
    o, lse = oracle.attention_rows(lay, la, ca, layer, q, k, v, tok, head)
    return tok, head, o, lse


def gpu_rows(o_gpu, lse_gpu, tok, head):
    o = o_gpu[torch.as_tensor(tok, device=o_gpu.device).long(),
              torch.as_tensor(head, device=o_gpu.device).long()].double().cpu().numpy()
    lse = lse_gpu[torch.as_tensor(head, device=o_gpu.device).long(),
                  torch.as_tensor(tok, device=o_gpu.device).long()].double().cpu().numpy()
    return o, lse


def enumerated_prompts():
    """Every LA/CA bit pattern of a prompt with two 3-tile documents and a 1-tile suffix:
    6 meaningful LA bits (rows 1 and 2 of each document) and the 3 CA bits of the first
    document (the second's CA has no later document), 2^9 = 512 patterns, each its own
    prompt in one batch.  Returns (layout, la_words, ca_words, patterns)."""
    B, T = 4, 3
    n = 1 << 9
    cfg = W.custom_config("enum", [([B * T, B * T], B)] * n, W.BitSpec(pattern="zeros"),
                          num_q_heads=2, num_kv_heads=1, head_dim=4, tile=B)
    lay = W.make_layout(cfg)
    la = np.zeros(lay.la_words_len, np.uint64)
    ca = np.zeros(lay.ca_words_len, np.uint64)
    for pat in range(n):
        g0, g1 = 2 * pat, 2 * pat + 1
        bits = [(pat >> b) & 1 for b in range(9)]
        # document 0: LA rows 1 (bit 0 -> j=0) and 2 (bits 1, 2 -> j=0, 1)
        la[lay.la_off[g0] + 1] = np.uint64(bits[0])
        la[lay.la_off[g0] + 2] = np.uint64(bits[1] | bits[2] << 1)
        la[lay.la_off[g1] + 1] = np.uint64(bits[3])
        la[lay.la_off[g1] + 2] = np.uint64(bits[4] | bits[5] << 1)
        ca[lay.ca_off[g0]] = np.uint64(bits[6] | bits[7] << 1 | bits[8] << 2)
    return lay, la, ca, n


def plain_lists(pat, p0):
    """The list rule for one enumerated prompt starting at global tile p0, written out:
    document-0 rows: own LA tiles then the diagonal; document-1 rows: document 0's CA
    pages, own LA tiles, the diagonal; the suffix row: every tile up to itself."""
    bits = [(pat >> b) & 1 for b in range(9)]
    la0 = {1: [0] if bits[0] else [], 2: [j for j, b in ((0, bits[1]), (1, bits[2])) if b]}
    la1 = {1: [0] if bits[3] else [], 2: [j for j, b in ((0, bits[4]), (1, bits[5])) if b]}
    ca0 = [j for j in range(3) if bits[6 + j]]
    rows = []
    for i in range(3):
        rows.append([p0 + j for j in la0.get(i, [])] + [p0 + i])
    for i in range(3):
        rows.append([p0 + j for j in ca0] + [p0 + 3 + j for j in la1.get(i, [])] + [p0 + 3 + i])
    rows.append(list(range(p0, p0 + 7)))
    return rows


def expand_lists(lay, qtiles, kv, counts, pages, layer, h):
    """Token mask implied by the decoded lists: key c of an entry is visible to row r of
    the query tile iff c < len, mask bit c // Pin is set and, when causal, c <= r.  Key c
    is token first + c, or, for a gathered entry, token pages[first + c // page] + c % page
    of the layer's page array."""
    T, B, P = lay.total_tokens, lay.tile, lay.page_size
    pin = min(P, B)
    M = np.zeros((T, T), bool)
    c = np.arange(B)
    flat = pages[layer].reshape(-1)
    for q, (x, rows) in enumerate(qtiles):
        r = np.arange(rows)
        for e in range(counts[layer, h, q]):
            first, info = (int(v) for v in kv[layer, h, q, e])
            ln, causal, mask = info & 0xFF, (info >> 8) & 1, (info >> 16) & 0xFFFF
            col = (c < ln) & (((mask >> (c // pin)) & 1) == 1)
            vis = np.broadcast_to(col[None, :], (rows, B)).copy()
            if causal:
                vis &= c[None, :] <= r[:, None]
            rr, cc = np.nonzero(vis)
            if (info >> 9) & 1:
                keys = flat[first + cc // P] + cc % P
            else:
                keys = first + cc
            M[x + rr, keys] = True
    return M

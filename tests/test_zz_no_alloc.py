"""sift_dense_prefill_noalloc: the dense prefill for callers that cannot allocate
device memory when they call (for example a serving runtime that sizes every
buffer at start-up and forbids allocation on the request path, or code that must
not risk the device-wide synchronisation cudaMalloc/cudaFree can cause).  It
keeps its scratch in the library's fixed per-GPU array instead of a workspace.

Checked through the C ABI against sift_dense_prefill, on two calls in a row
(the second call must not see the first call's scheduler state), and for the
size limit of the scratch array.  Both entry points run the same kernels on the
same rows, so their outputs must be equal bit for bit.  This file runs last so
that a failure here cannot hide the results of the other GPU tests.
"""
import ctypes

import pytest
import torch

import workloads as W
from helpers import setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_dense_prefill_on_two_calls(sift):
    lib = sift.load_library()
    cfg = W.custom_config("noalloc", [([512, 256], 128), ([384], 256)],
                          W.BitSpec(pattern="ones"), num_q_heads=8, num_kv_heads=2,
                          head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    st_ref = prob.new_status()
    o_ref, lse_ref = sift.dense_prefill(prob, q, k, v, dev_status=st_ref)
    torch.cuda.synchronize()
    assert int(st_ref.item()) == 0
    stream = torch.cuda.current_stream()
    for call in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((cfg.num_q_heads, cfg.total_tokens), float("nan"),
                         dtype=torch.float32, device="cuda")
        st = prob.new_status()
        rc = lib.sift_dense_prefill_noalloc(prob.ref, _p(q), _p(k), _p(v), 0.0, _p(o), _p(lse),
                                            _p(st), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, sift.status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: {sift.status_string(int(st.item()))}"
        assert torch.isfinite(o.float()).all().item(), f"call {call}: rows left unwritten"
        assert torch.equal(o, o_ref), f"call {call}: O differs from sift_dense_prefill"
        assert torch.equal(lse, lse_ref), f"call {call}: LSE differs from sift_dense_prefill"


def test_noalloc_rejects_problem_beyond_scratch(sift):
    """A problem needing more scratch than the fixed array is refused on the host."""
    lib = sift.load_library()
    from bit_vector_guided_gb300._native import _Problem
    N = 16400  # 8 kv heads x 16,400 query tiles: 1.05 MB of scratch, above the 1 MiB array
    p = _Problem(num_prompts=1, num_docs=0, num_layers=1, num_q_heads=16, num_kv_heads=8,
                 head_dim=128, tile=128, total_tokens=N * 128, max_tiles_per_prompt=N,
                 page=0, cu_seqlens=16, doc_cu=32, doc_end=None, la_off=None, ca_off=None,
                 la_words_len=0, ca_words_len=0)
    assert lib.sift_workspace_bytes(ctypes.byref(p)) > (1 << 20)
    d = ctypes.c_void_p(256)
    rc = lib.sift_dense_prefill_noalloc(ctypes.byref(p), d, d, d, 0.0, d, d, d, None)
    assert rc == 2  # SIFT_ERR_UNSUPPORTED, nothing enqueued

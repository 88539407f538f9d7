"""Failure detection without a GPU fault: every device-side wait of the attention
kernel is bounded.  The test hook makes the MMA issuer wait on a barrier that
nothing ever signals; the wait must run out after a short limit, the kernel must
unwind (drain its copies, free tensor memory) and report SIFT_ERR_TIMEOUT, and
the context must stay usable for the next, normal launch."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_attention_close, setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sift(cuda_device):
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as s
    s.load_library()
    return s


def test_stalled_wait_times_out_cleanly(sift):
    cfg = W.custom_config("watchdog", [([512, 256], 128)], W.BitSpec(la_p=0.3, ca_p=0.3),
                          num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128)
    lay, la, ca, prob, la_d, ca_d = setup(cfg)
    st = prob.new_status()
    kv, cnt, sched = sift.decode(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sift.debug_set_waits(timeout_ns=2_000_000, stall=True)
    try:
        st = prob.new_status()
        sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sched, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 4, sift.status_string(int(st.item()))  # SIFT_ERR_TIMEOUT
    finally:
        sift.debug_set_waits(0, False)
    # the same context runs the next launch normally
    st = prob.new_status()
    o, lse = sift.sparse_prefill(prob, 0, q, k, v, kv, cnt, sched, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                           "after timeout")


def test_stalled_wait_times_out_cleanly_general_layout(sift):
    """The same on the general layout with gathered pages in flight: the producers' page
    copies are drained like whole-tile ones before the kernel returns."""
    cfg = W.custom_config("watchdog_rg", [([300, 411, 77], 50)], W.BitSpec(la_p=0.3, ca_p=0.4),
                          num_q_heads=4, num_kv_heads=2, head_dim=128, tile=128, page=16)
    lay = W.make_layout(cfg)
    la, ca = W.make_bits(cfg, lay)
    prob = sift.SiftProblem.from_layout(lay, "cuda")
    from helpers import device_bits
    la_d, ca_d = device_bits(la, ca)
    st = prob.new_status()
    lists = sift.decode_ragged(prob, la_d, ca_d, dev_status=st)
    q, k, v = W.make_qkv(cfg, 0, device="cuda")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sift.debug_set_waits(timeout_ns=2_000_000, stall=True)
    try:
        st = prob.new_status()
        sift.sparse_prefill_ragged(prob, 0, q, k, v, *lists, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 4, sift.status_string(int(st.item()))  # SIFT_ERR_TIMEOUT
    finally:
        sift.debug_set_waits(0, False)
    st = prob.new_status()
    o, lse = sift.sparse_prefill_ragged(prob, 0, q, k, v, *lists, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O, LSE = oracle.attention_all(lay, la, ca, 0, q, k, v)
    assert_attention_close(o.double().cpu().numpy(), lse.double().cpu().numpy(), O, LSE,
                           "general layout after timeout")

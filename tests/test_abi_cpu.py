"""The C-ABI library loads here (no GPU), exports every symbol include/sift.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sift.h")


@pytest.fixture(scope="module")
def lib():
    from bit_vector_guided_gb300 import build
    build.build()
    import bit_vector_guided_gb300 as sift
    return sift.load_library()


def test_exports_every_declared_symbol(lib):
    import bit_vector_guided_gb300 as sift
    names = sift.exported_symbols(HEADER)
    assert {"sift_decode", "sift_sparse_prefill", "sift_dense_prefill",
            "sift_status_string", "sift_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libsift.so does not export {n}"


def test_status_strings(lib):
    import bit_vector_guided_gb300 as sift
    for code, name in sift.STATUS.items():
        assert sift.status_string(code) == name
    assert sift.abi_version() == 101


def _struct(**over):
    from bit_vector_guided_gb300._native import _Problem
    f = dict(num_prompts=1, num_docs=0, num_layers=1, num_q_heads=4, num_kv_heads=2,
             head_dim=128, tile=128, total_tokens=256, max_tiles_per_prompt=2, page=0,
             cu_seqlens=16, doc_cu=32, doc_end=None, la_off=None, ca_off=None,
             la_words_len=0, ca_words_len=0)
    f.update(over)
    return _Problem(**f)


@pytest.mark.parametrize("over,code", [
    (dict(num_q_heads=6, num_kv_heads=4), 1),       # Hq % Hkv != 0
    (dict(total_tokens=200), 2),                    # not a multiple of the tile
    (dict(head_dim=96), 2),                         # unsupported head_dim
    (dict(tile=32, total_tokens=256), 2),           # unsupported tile
    (dict(num_q_heads=6, num_kv_heads=2), 2),       # odd GQA group
    (dict(cu_seqlens=None), 1),                     # missing pointer
    (dict(num_docs=2), 1),                          # docs without offsets
    (dict(max_tiles_per_prompt=3), 1),              # rowcap larger than the batch
])
def test_host_validation_rejects_before_launch(lib, over, code):
    p = _struct(**over)
    dummy = ctypes.c_void_p(256)
    rc = lib.sift_dense_prefill(ctypes.byref(p), dummy, dummy, dummy, 0.0, dummy, dummy, dummy,
                                1 << 20, dummy, None)
    assert rc == code


def test_host_validation_pointers_and_sizes(lib):
    p = _struct()
    d = ctypes.c_void_p(256)
    ws = lib.sift_workspace_bytes(ctypes.byref(p))
    assert ws >= 256 + 2 * 2 * 2 * 4
    # misaligned q, too-small workspace, null status, bad layer: all INVALID_ARG
    assert lib.sift_dense_prefill(ctypes.byref(p), ctypes.c_void_p(258), d, d, 0.0, d, d, d,
                                  ws, d, None) == 1
    assert lib.sift_dense_prefill(ctypes.byref(p), d, d, d, 0.0, d, d, d, ws - 1, d, None) == 1
    assert lib.sift_dense_prefill(ctypes.byref(p), d, d, d, 0.0, d, d, d, ws, None, None) == 1
    assert lib.sift_sparse_prefill(ctypes.byref(p), 1, d, d, d, d, d, d, 0.0, d, d, d, ws, d,
                                   None) == 1
    assert lib.sift_decode(None, d, d, d, d, d, d, None) == 1
    assert lib.sift_decode(ctypes.byref(p), d, d, None, d, d, d, None) == 1
    assert lib.sift_workspace_bytes(None) == 0


@pytest.mark.parametrize("over,nq,code", [
    (dict(page=48), 2, 2),                          # page not a power of two
    (dict(page=4), 2, 2),                           # 32 pages per tile: beyond the mask
    (dict(tile=96, total_tokens=200), 3, 2),        # tile not a power of two
    (dict(total_tokens=200), 0, 1),                 # no query tiles
    (dict(total_tokens=200), 9, 1),                 # more query tiles than the segments hold
    (dict(head_dim=96, total_tokens=200), 2, 2),    # unsupported head_dim
    (dict(num_q_heads=6, num_kv_heads=2), 2, 2),    # odd GQA group
])
def test_ragged_host_validation(lib, over, nq, code):
    p = _struct(**over)
    d = ctypes.c_void_p(256)
    rc = lib.sift_sparse_prefill_ragged(ctypes.byref(p), nq, 0, d, d, d, d, d, d, d, d, 1, 0.0,
                                        d, d, d, 1 << 20, d, None)
    assert rc == code
    if code == 2 and "head_dim" not in over and "num_q_heads" not in over:
        assert lib.sift_decode_ragged(ctypes.byref(p), max(nq, 1), d, d, d, d, d, d, d, 1, d,
                                      None) == 2


def test_ragged_layout_rules(lib):
    """A ragged total is fine for the general entry points and for workspace sizing, but
    not for the aligned ones; a page size other than the tile is general-layout only."""
    p = _struct(total_tokens=200)
    assert lib.sift_workspace_bytes(ctypes.byref(p)) > 0
    d = ctypes.c_void_p(256)
    assert lib.sift_decode(ctypes.byref(p), d, d, d, d, d, d, None) == 2
    p = _struct(page=64)
    assert lib.sift_dense_prefill(ctypes.byref(p), d, d, d, 0.0, d, d, d, 1 << 20, d, None) == 2
    # misaligned list pointer (entries are 8-byte pairs)
    p = _struct(total_tokens=200)
    assert lib.sift_sparse_prefill_ragged(ctypes.byref(p), 2, 0, d, d, d, d, ctypes.c_void_p(260),
                                          d, d, d, 1, 0.0, d, d, d, 1 << 20, d, None) == 1
    # gathered pages (page 16 < tile 128) without a page array
    p = _struct(total_tokens=200, page=16, num_docs=1, doc_end=ctypes.c_void_p(64),
                la_off=ctypes.c_void_p(64), ca_off=ctypes.c_void_p(64))
    assert lib.sift_sparse_prefill_ragged(ctypes.byref(p), 2, 0, d, d, d, d, d, d, d, None, 0,
                                          0.0, d, d, d, 1 << 20, d, None) == 1
    assert lib.sift_decode_ragged(ctypes.byref(p), 2, d, d, d, d, d, d, None, 0, d, None) == 1

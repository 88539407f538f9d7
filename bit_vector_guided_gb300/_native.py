"""ctypes binding of libsift.so (include/sift.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers, allocates outputs with torch
when the caller passes none, and raises on a non-OK status.  There is no CPU
fallback: if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import numpy as np

from . import build as _build

__all__ = ["SiftError", "SiftProblem", "load_library", "decode", "sparse_prefill",
           "dense_prefill", "dense_prefill_noalloc", "fused_prefill", "build_bits",
           "decode_ragged", "sparse_prefill_ragged",
           "build_bits_workspace_bytes", "workspace_bytes", "status_string", "debug_set_waits",
           "abi_version", "exported_symbols", "STATUS"]

STATUS = {0: "SIFT_OK", 1: "SIFT_ERR_INVALID_ARG", 2: "SIFT_ERR_UNSUPPORTED", 3: "SIFT_ERR_CUDA",
          4: "SIFT_ERR_TIMEOUT", 5: "SIFT_ERR_DEVICE_CHECK"}


class SiftError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)}")


class _Problem(ctypes.Structure):
    _fields_ = [("num_prompts", ctypes.c_int32), ("num_docs", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("tile", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("max_tiles_per_prompt", ctypes.c_int32), ("page", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("doc_cu", ctypes.c_void_p),
                ("doc_end", ctypes.c_void_p), ("la_off", ctypes.c_void_p),
                ("ca_off", ctypes.c_void_p), ("la_words_len", ctypes.c_int64),
                ("ca_words_len", ctypes.c_int64)]


_lib = None


def load_library(path: Optional[str] = None):
    """Load libsift.so (built in-tree by bit_vector_guided_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libsift.so not found at {path}; run bit_vector_guided_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, u64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_uint64)
    sz = ctypes.c_size_t
    lib.sift_workspace_bytes.argtypes = [P]
    lib.sift_workspace_bytes.restype = sz
    lib.sift_decode.argtypes = [P, P, P, P, P, P, P, P]
    lib.sift_decode.restype = i32
    lib.sift_sparse_prefill.argtypes = [P, i32, P, P, P, P, P, P, f32, P, P, P, sz, P, P]
    lib.sift_sparse_prefill.restype = i32
    lib.sift_dense_prefill.argtypes = [P, P, P, P, f32, P, P, P, sz, P, P]
    lib.sift_dense_prefill.restype = i32
    lib.sift_fused_prefill.argtypes = [P, i32, P, P, P, P, P, f32, P, P, P, sz, P, P]
    lib.sift_fused_prefill.restype = i32
    lib.sift_dense_prefill_noalloc.argtypes = [P, P, P, P, f32, P, P, P, P]
    lib.sift_dense_prefill_noalloc.restype = i32
    lib.sift_build_bits_workspace_bytes.argtypes = [P, i32]
    lib.sift_build_bits_workspace_bytes.restype = sz
    lib.sift_build_bits.argtypes = [P, i32, P, P, i32, f32, f32, f32, P, P, P, sz, P, P]
    lib.sift_build_bits.restype = i32
    lib.sift_decode_ragged.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, P]
    lib.sift_decode_ragged.restype = i32
    lib.sift_sparse_prefill_ragged.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P, i32, f32,
                                               P, P, P, sz, P, P]
    lib.sift_sparse_prefill_ragged.restype = i32
    lib.sift_status_string.argtypes = [i32]
    lib.sift_status_string.restype = ctypes.c_char_p
    lib.sift_debug_set_waits.argtypes = [u64, i32]
    lib.sift_debug_set_waits.restype = None
    lib.sift_abi_version.argtypes = []
    lib.sift_abi_version.restype = i32
    _lib = lib
    return lib


def exported_symbols(header: str) -> list:
    """Names of the functions a header declares (used to check the library's exports)."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sift_[a-z_0-9]+)\s*\(", text)))


def status_string(code: int) -> str:
    return load_library().sift_status_string(int(code)).decode()


def abi_version() -> int:
    return int(load_library().sift_abi_version())


def debug_set_waits(timeout_ns: int = 0, stall: bool = False) -> None:
    """Test hook: limit of device-side waits and a forced stall (see include/sift.h)."""
    load_library().sift_debug_set_waits(int(timeout_ns), 1 if stall else 0)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class SiftProblem:
    """Device-side description of one packed varlen batch (struct sift_problem).

    Host arrays are uploaded once to `device`; the object keeps the device
    tensors alive for as long as it lives.
    """

    def __init__(self, *, cu_seqlens, doc_cu, doc_end, la_off, ca_off, num_layers, num_q_heads,
                 num_kv_heads, head_dim, tile, la_words_len, ca_words_len,
                 max_tiles_per_prompt: Optional[int] = None, page: int = 0, device="cuda"):
        import torch
        cu = np.asarray(cu_seqlens, np.int32)
        self.num_prompts = len(cu) - 1
        self.num_docs = len(np.asarray(doc_end))
        self.num_layers = int(num_layers)
        self.num_q_heads = int(num_q_heads)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = int(head_dim)
        self.tile = int(tile)
        self.total_tokens = int(cu[-1])
        self.num_tiles = self.total_tokens // self.tile
        self.page = int(page)
        # query tiles counted per segment (documents and suffixes tile from their own start),
        # the row count of the general-layout entry points
        dcu = np.asarray(doc_cu, np.int64)
        dend = np.asarray(doc_end, np.int64)
        B = self.tile
        nq = 0
        for p in range(self.num_prompts):
            pos = int(cu[p])
            for g in range(int(dcu[p]), int(dcu[p + 1])):
                nq += (int(dend[g]) - pos + B - 1) // B
                pos = int(dend[g])
            nq += (int(cu[p + 1]) - pos + B - 1) // B
        self.num_query_tiles = nq
        if max_tiles_per_prompt is None:
            max_tiles_per_prompt = int(np.max(np.diff(cu)) // self.tile) if len(cu) > 1 else 1
        self.max_tiles_per_prompt = max(int(max_tiles_per_prompt), 1)
        # gathered CA pages (page below the tile, a multiple of 8): capacity per document
        pg = self.page if self.page > 0 else B
        self.page_cap = self.max_tiles_per_prompt * (B // pg) if (pg < B and pg % 8 == 0) else 0
        self.device = torch.device(device)

        def up(a, dt):
            a = np.ascontiguousarray(np.asarray(a, dt))
            if a.size == 0:
                a = np.zeros(1, dt)
            return torch.from_numpy(a).to(self.device)

        self._cu = up(cu, np.int32)
        self._doc_cu = up(doc_cu, np.int32)
        self._doc_end = up(doc_end, np.int32)
        self._la_off = up(la_off, np.int64)
        self._ca_off = up(ca_off, np.int64)
        self.la_words_len = int(la_words_len)
        self.ca_words_len = int(ca_words_len)
        self._struct = _Problem(self.num_prompts, self.num_docs, self.num_layers,
                                self.num_q_heads, self.num_kv_heads, self.head_dim, self.tile,
                                self.total_tokens, self.max_tiles_per_prompt, self.page,
                                _ptr(self._cu), _ptr(self._doc_cu), _ptr(self._doc_end),
                                _ptr(self._la_off), _ptr(self._ca_off), self.la_words_len,
                                self.ca_words_len)

    @classmethod
    def from_layout(cls, layout, device="cuda"):
        """Build from any object with the attributes of workloads.Layout."""
        return cls(cu_seqlens=layout.cu_seqlens, doc_cu=layout.doc_cu, doc_end=layout.doc_end,
                   la_off=layout.la_off, ca_off=layout.ca_off, num_layers=layout.num_layers,
                   num_q_heads=layout.num_q_heads, num_kv_heads=layout.num_kv_heads,
                   head_dim=layout.head_dim, tile=layout.tile,
                   la_words_len=layout.la_words_len, ca_words_len=layout.ca_words_len,
                   max_tiles_per_prompt=layout.max_tiles_per_prompt,
                   page=int(getattr(layout, "page", 0) or 0), device=device)

    @property
    def ref(self):
        return ctypes.byref(self._struct)

    def workspace_bytes(self) -> int:
        return int(load_library().sift_workspace_bytes(self.ref))

    def new_status(self):
        import torch
        return torch.zeros(1, dtype=torch.int32, device=self.device)

    def new_workspace(self):
        import torch
        n = (self.workspace_bytes() + 15) // 16 * 16
        return torch.empty(max(n, 16), dtype=torch.uint8, device=self.device)


def _check(code: int, where: str):
    if code != 0:
        raise SiftError(code, where)


def workspace_bytes(prob: SiftProblem) -> int:
    return prob.workspace_bytes()


def decode(prob: SiftProblem, la_words, ca_words, kv_idx=None, counts=None, sched=None,
           dev_status=None, stream=None):
    """sift_decode: returns (kv_idx [L,Hkv,N,rowcap], counts [L,Hkv,N], sched [L,Hkv*N])."""
    import torch
    lib = load_library()
    L, H, N, R = prob.num_layers, prob.num_kv_heads, prob.num_tiles, prob.max_tiles_per_prompt
    dev = prob.device
    if kv_idx is None:
        kv_idx = torch.empty((L, H, N, R), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((L, H, N), dtype=torch.int32, device=dev)
    if sched is None:
        sched = torch.empty((L, H * N), dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_decode(prob.ref, _ptr(la_words), _ptr(ca_words), _ptr(kv_idx), _ptr(counts),
                         _ptr(sched), _ptr(dev_status), _stream(stream))
    _check(rc, "sift_decode")
    return kv_idx, counts, sched


def sparse_prefill(prob: SiftProblem, layer: int, q, k, v, kv_idx, counts, sched,
                   softmax_scale: float = 0.0, o=None, lse=None, workspace=None,
                   dev_status=None, stream=None):
    """sift_sparse_prefill: returns (o bf16 [T,Hq,d], lse fp32 [Hq,T])."""
    import torch
    lib = load_library()
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((prob.num_q_heads, prob.total_tokens), dtype=torch.float32,
                          device=q.device)
    if workspace is None:
        workspace = prob.new_workspace()
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_sparse_prefill(prob.ref, int(layer), _ptr(q), _ptr(k), _ptr(v), _ptr(kv_idx),
                                 _ptr(counts), _ptr(sched), float(softmax_scale), _ptr(o),
                                 _ptr(lse), _ptr(workspace), int(workspace.numel()),
                                 _ptr(dev_status), _stream(stream))
    _check(rc, "sift_sparse_prefill")
    return o, lse


def fused_prefill(prob: SiftProblem, layer: int, la_words, ca_words, q, k, v,
                  softmax_scale: float = 0.0, o=None, lse=None, workspace=None,
                  dev_status=None, stream=None):
    """sift_fused_prefill: decode fused into the sparse prefill; returns (o, lse)."""
    import torch
    lib = load_library()
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((prob.num_q_heads, prob.total_tokens), dtype=torch.float32,
                          device=q.device)
    if workspace is None:
        workspace = prob.new_workspace()
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_fused_prefill(prob.ref, int(layer), _ptr(la_words), _ptr(ca_words), _ptr(q),
                                _ptr(k), _ptr(v), float(softmax_scale), _ptr(o), _ptr(lse),
                                _ptr(workspace), int(workspace.numel()), _ptr(dev_status),
                                _stream(stream))
    _check(rc, "sift_fused_prefill")
    return o, lse


def dense_prefill(prob: SiftProblem, q, k, v, softmax_scale: float = 0.0, o=None, lse=None,
                  workspace=None, dev_status=None, stream=None):
    """sift_dense_prefill: returns (o, lse) of dense causal attention per prompt."""
    import torch
    lib = load_library()
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((prob.num_q_heads, prob.total_tokens), dtype=torch.float32,
                          device=q.device)
    if workspace is None:
        workspace = prob.new_workspace()
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_dense_prefill(prob.ref, _ptr(q), _ptr(k), _ptr(v), float(softmax_scale),
                                _ptr(o), _ptr(lse), _ptr(workspace), int(workspace.numel()),
                                _ptr(dev_status), _stream(stream))
    _check(rc, "sift_dense_prefill")
    return o, lse


def dense_prefill_noalloc(prob: SiftProblem, q, k, v, softmax_scale: float = 0.0, o=None,
                          lse=None, dev_status=None, stream=None):
    """sift_dense_prefill_noalloc: dense prefill whose scratch is the library's fixed
    per-GPU array (no workspace argument).  Outputs are allocated here only when the
    caller passes none; callers that cannot allocate pass their own o, lse, dev_status."""
    import torch
    lib = load_library()
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((prob.num_q_heads, prob.total_tokens), dtype=torch.float32,
                          device=q.device)
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_dense_prefill_noalloc(prob.ref, _ptr(q), _ptr(k), _ptr(v), float(softmax_scale),
                                        _ptr(o), _ptr(lse), _ptr(dev_status), _stream(stream))
    _check(rc, "sift_dense_prefill_noalloc")
    return o, lse


def build_bits_workspace_bytes(prob: SiftProblem, max_doc_tiles: int) -> int:
    return int(load_library().sift_build_bits_workspace_bytes(prob.ref, int(max_doc_tiles)))


def build_bits(prob: SiftProblem, layer: int, q, k, max_doc_tiles: int, la_fraction: float,
               ca_fraction: float, la_words, ca_words, softmax_scale: float = 0.0,
               workspace=None, dev_status=None, stream=None):
    """sift_build_bits: writes layer `layer`'s LA / CA words of every document into
    la_words / ca_words (int64 device tensors of the sizes the problem names)."""
    import torch
    lib = load_library()
    if workspace is None:
        n = (build_bits_workspace_bytes(prob, max_doc_tiles) + 15) // 16 * 16
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=prob.device)
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_build_bits(prob.ref, int(layer), _ptr(q), _ptr(k), int(max_doc_tiles),
                             float(la_fraction), float(ca_fraction), float(softmax_scale),
                             _ptr(la_words), _ptr(ca_words), _ptr(workspace),
                             int(workspace.numel()), _ptr(dev_status), _stream(stream))
    _check(rc, "sift_build_bits")
    return la_words, ca_words


def decode_ragged(prob: SiftProblem, la_words, ca_words, qtiles=None, kv=None, counts=None,
                  sched=None, pages=None, dev_status=None, stream=None):
    """sift_decode_ragged: returns (qtiles [NQ,2], kv [L,Hkv,NQ,rowcap,2], counts [L,Hkv,NQ],
    sched [L,Hkv*NQ], pages [L,Hkv,D,page_cap] or None) for documents of any length and a
    CA page size of their own."""
    import torch
    lib = load_library()
    L, H, NQ, R = prob.num_layers, prob.num_kv_heads, prob.num_query_tiles, prob.max_tiles_per_prompt
    dev = prob.device
    if qtiles is None:
        qtiles = torch.empty((NQ, 2), dtype=torch.int32, device=dev)
    if kv is None:
        kv = torch.empty((L, H, NQ, R, 2), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((L, H, NQ), dtype=torch.int32, device=dev)
    if sched is None:
        sched = torch.empty((L, H * NQ), dtype=torch.int32, device=dev)
    if pages is None and prob.page_cap > 0 and prob.num_docs > 0:
        pages = torch.empty((L, H, prob.num_docs, prob.page_cap), dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_decode_ragged(prob.ref, NQ, _ptr(la_words), _ptr(ca_words), _ptr(qtiles),
                                _ptr(kv), _ptr(counts), _ptr(sched), _ptr(pages),
                                prob.page_cap if pages is not None else 0, _ptr(dev_status),
                                _stream(stream))
    _check(rc, "sift_decode_ragged")
    return qtiles, kv, counts, sched, pages


def sparse_prefill_ragged(prob: SiftProblem, layer: int, q, k, v, qtiles, kv, counts, sched,
                          pages=None, softmax_scale: float = 0.0, o=None, lse=None,
                          workspace=None, dev_status=None, stream=None):
    """sift_sparse_prefill_ragged: returns (o bf16 [T,Hq,d], lse fp32 [Hq,T])."""
    import torch
    lib = load_library()
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((prob.num_q_heads, prob.total_tokens), dtype=torch.float32,
                          device=q.device)
    if workspace is None:
        workspace = prob.new_workspace()
    if dev_status is None:
        dev_status = prob.new_status()
    rc = lib.sift_sparse_prefill_ragged(prob.ref, prob.num_query_tiles, int(layer), _ptr(q),
                                        _ptr(k), _ptr(v), _ptr(qtiles), _ptr(kv), _ptr(counts),
                                        _ptr(sched), _ptr(pages),
                                        prob.page_cap if pages is not None else 0,
                                        float(softmax_scale), _ptr(o), _ptr(lse),
                                        _ptr(workspace), int(workspace.numel()), _ptr(dev_status),
                                        _stream(stream))
    _check(rc, "sift_sparse_prefill_ragged")
    return o, lse

"""SIFT online-prefill hot path for GB300 (sm_103a).

``sift_decode`` (bits -> tile lists + longest-first schedule),
``sift_sparse_prefill`` (block-sparse causal GQA flash attention) and
``sift_dense_prefill`` (the dense full-recompute baseline), plus the fused
decode+prefill, the offline bit builder ``sift_build_bits`` and the general-layout
pair ``sift_decode_ragged`` / ``sift_sparse_prefill_ragged`` (documents of any
length, CA pages of their own size), live in the CUDA
library ``libsift.so`` behind the C ABI of ``include/sift.h``; this package is
the Python binding of that library.
"""
from ._native import (STATUS, SiftError, SiftProblem, abi_version, build_bits,
                      build_bits_workspace_bytes, debug_set_waits, decode, decode_ragged,
                      dense_prefill, dense_prefill_noalloc, exported_symbols, fused_prefill,
                      load_library, sparse_prefill, sparse_prefill_ragged, status_string,
                      workspace_bytes)

__all__ = ["STATUS", "SiftError", "SiftProblem", "abi_version", "build_bits",
           "build_bits_workspace_bytes", "debug_set_waits", "decode", "decode_ragged",
           "sparse_prefill_ragged", "dense_prefill",
           "dense_prefill_noalloc", "exported_symbols", "fused_prefill", "load_library",
           "sparse_prefill", "status_string", "workspace_bytes"]

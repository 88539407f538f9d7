"""SIFT online-prefill hot path for GB300 (sm_103a).

``sift_decode`` (bits -> tile lists + longest-first schedule),
``sift_sparse_prefill`` (block-sparse causal GQA flash attention) and
``sift_dense_prefill`` (the dense full-recompute baseline), plus the fused
decode+prefill and the offline bit builder ``sift_build_bits``, live in the CUDA
library ``libsift.so`` behind the C ABI of ``include/sift.h``; this package is
the Python binding of that library.
"""
from ._native import (STATUS, SiftError, SiftProblem, abi_version, build_bits,
                      build_bits_workspace_bytes, debug_set_waits, decode, dense_prefill,
                      dense_prefill_noalloc, exported_symbols, fused_prefill, load_library,
                      sparse_prefill, status_string, workspace_bytes)

__all__ = ["STATUS", "SiftError", "SiftProblem", "abi_version", "build_bits",
           "build_bits_workspace_bytes", "debug_set_waits", "decode", "dense_prefill",
           "dense_prefill_noalloc", "exported_symbols", "fused_prefill", "load_library",
           "sparse_prefill", "status_string", "workspace_bytes"]

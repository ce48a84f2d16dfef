"""Packed-QKV attention prologue for GB300 (sm_103a).

Split a packed qkv projection into heads, per-head RMSNorm of q and k,
rotate-half RoPE (skipped on NoPE layers), contiguous or paged-pool stores;
a one-pass backward that writes the packed gradient; MLA kv latent rows
written straight into a paged pool. All of it runs in the CUDA kernels of
libqkv_prologue.so, reached through its C ABI (include/qkv_prologue.h).

``rope_qkv_prologue_gb300._lib`` holds the ctypes binding with the C names;
``rope_qkv_prologue_gb300.functional`` allocates outputs with torch and calls
it. Importing this package fails if the library has not been built.
"""

from ._lib import *  # noqa: F401,F403
from ._lib import EXPORTED, LIB_PATH, QkvpError, layout  # noqa: F401
from . import functional  # noqa: F401

__all__ = [
    "EXPORTED", "LIB_PATH", "QkvpError", "layout", "functional",
    "qkv_prologue_fwd", "qkv_prologue_pool_write", "qkv_prologue_pool_scatter",
    "qkv_prologue_bwd_workspace_size", "qkv_prologue_bwd", "qkv_prologue_status_string",
    "qkv_prologue_version", "qkvp_layout", "qkvp_variant", "variant",
    "qkv_prologue_fwd_ex", "qkv_prologue_pool_write_ex", "qkv_prologue_bwd_workspace_size_ex",
    "qkv_prologue_bwd_ex", "qkv_prologue_gemm_fwd",
]

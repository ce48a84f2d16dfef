"""fp64 CPU oracle for the packed-QKV attention prologue.

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously correct
definition that the CUDA kernels are checked against. Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it; the library in ``rope_qkv_prologue_gb300`` never
does, and nothing here imports that library.

Sources (page title, then section):

* "[muse_spark][perf] Split the packed qkv inside the q/k region" (torchtitan)
  - Problem 1: the packed projection is viewed as [T, 16 kv heads, 10, 64];
    per kv head, 8 q heads + 1 k + 1 v.
  - Solution 3 / the before/after diagram: split -> per-head norm -> RoPE for q
    and k, v copied; the backward writes the packed grad with no cat.
  - Results, Numerics: moving the split and copies changes no bits.
  - "why is training's q norm kernel slower": training also writes the split q.
* "[muon] Per-head Newton-Schulz for fused QKV projections" (DeepSpeed)
  - What this PR does: the sectioned (q | k | v) and the interleaved-per-KV-
    group packings are the same partition into head_dim blocks in two orders;
    a fused row holds exactly (n_q + 2 n_kv) * head_dim values. The same
    partition of a fused weight's dim 0 is what per-head Newton-Schulz works
    on, one block at a time, with the factor max(1, head_dim / in_features)
    ** 0.5 (newton_schulz.py; the iteration itself is Muon's published one).
* "MLA DSpark: run each drafter layer's kv path beside its q path"
  (TensorRT-LLM #20552)
  - Description: the RMSNorm/RoPE kernel stores the latent rows straight into
    the paged pool at given pages / offsets, instead of staging + scatter.
  - Test Coverage: the direct pool write equals the staged path plus the
    scatter write.

Parity status: the pages print no numeric example (only the block counts and
the split / no-split cases of the Newton-Schulz page, kept in tests/golden/),
so no function here is pinned by printed values. Every function is pinned by
closed forms, invariants, brute force on tiny inputs, finite differences or
the pages' stated layout facts (see tests/test_oracle_pins.py). None is
"parity unpinned".
"""

from .bf16 import bf16_bits_to_f64, to_bf16_rne  # noqa: F401
from .prologue import (  # noqa: F401
    PackedLayout,
    head_blocks,
    split_heads,
    merge_heads,
    rms_norm,
    rms_norm_backward,
    rope_inv_freq,
    rope_angles,
    rope_rotate_half,
    rope_rotate_half_transpose,
    prologue_fwd_f64,
    prologue_fwd,
    prologue_bwd_f64,
    prologue_bwd,
    pool_scatter,
    pool_write,
    mla_rows_f64,
    mla_rows,
    mla_pool_write,
    gemm_prologue_fwd,
)
from .newton_schulz import (  # noqa: F401
    NS_COEFFS,
    NS_STEPS,
    NS_EPS,
    newton_schulz5,
    fused_head_blocks,
    per_head_scale,
    full_matrix_scale,
    per_head_newton_schulz,
    full_matrix_newton_schulz,
    muon_orthogonalize,
    qkv_newton_schulz,
)

"""Per-head Newton-Schulz of a fused QKV update, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the plain definition the
CUDA kernel is checked against. Nothing is blocked, fused or reordered; each
block is a whole matrix and each step is one line.

Source: "[muon] Per-head Newton-Schulz for fused QKV projections" (DeepSpeed),
What this PR does, and the review comment on fused and separate layouts:

* In both packings that ship (sectioned q | k | v and interleaved per KV
  group) every head is head_dim consecutive rows of dim 0, so a fused weight
  [(n_q + 2 n_kv) * head_dim, in_features] is cut into rows // head_dim
  blocks in storage order; which block is a q, k or v head never matters.
* Every block is orthogonalised on its own and multiplied by the same
  factor max(1, head_dim / in_features) ** 0.5.
* The cut is made only when dim 0 is exactly (n_q + 2 n_kv) * head_dim;
  any other weight stays whole and gets max(1, rows / cols) ** 0.5 (up to
  sqrt(3) for a [3h, h] weight, where separately stored q, k, v get 1).

Readings where the page prints no formula:

* The iteration is Muon's quintic Newton-Schulz as published with that
  optimizer (K. Jordan et al., "Muon: An optimizer for hidden layers in
  neural networks", 2024): the matrix is divided by its Frobenius norm plus
  1e-7; a matrix taller than wide is transposed first and the result is
  transposed back; then five times
      A = X X^T,   X <- a X + (b A + c A A) X,
  with (a, b, c) = (3.4445, -4.7750, 2.0315). The page names the per-head
  iteration and its scale, not these constants, so the published defaults
  stand.
* Everything is float64 and nothing is rounded; a caller that compares with a
  bf16 kernel rounds (or not) on its own side.
"""

import numpy as np

from .bf16 import bf16_bits_to_f64

NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
NS_EPS = 1e-7


def newton_schulz5(g, steps=NS_STEPS, coeffs=NS_COEFFS, eps=NS_EPS, rounding=None):
    """Muon's quintic Newton-Schulz of one matrix, float64.

    `rounding` is None for the exact definition. A function given there is
    applied where the published bf16 implementation holds a value in bf16
    (the normalised input, every A, every b A + c A A, every new X); the tests
    use that only to size the parity tolerance of a bf16 kernel.
    """
    r = (lambda v: v) if rounding is None else rounding
    x = np.asarray(g, dtype=np.float64)
    tall = x.shape[0] > x.shape[1]
    if tall:
        x = x.T
    x = r(x / (np.linalg.norm(x) + eps))  # Frobenius norm
    a, b, c = coeffs
    for _ in range(steps):
        A = r(x @ x.T)
        B = r(b * A + c * (A @ A))
        x = r(a * x + B @ x)
    return x.T if tall else x


def fused_head_blocks(rows, n_q, n_kv, head_dim):
    """Number of per-head blocks of a fused weight with `rows` rows in dim 0.

    None when dim 0 is not exactly (n_q + 2 n_kv) * head_dim: such a weight is
    not split (it stays on the full-matrix path).
    """
    if not (n_q and n_kv and head_dim) or n_q <= 0 or n_kv <= 0 or head_dim <= 0:
        return None
    if rows != (n_q + 2 * n_kv) * head_dim:
        return None
    return rows // head_dim


def per_head_scale(head_dim, in_features):
    """The factor every block gets: max(1, head_dim / in_features) ** 0.5."""
    return max(1.0, head_dim / in_features) ** 0.5


def full_matrix_scale(rows, cols):
    """The factor a whole (unsplit) matrix gets: max(1, rows / cols) ** 0.5."""
    return max(1.0, rows / cols) ** 0.5


def per_head_newton_schulz(m, head_dim, **kw):
    """Cut m [rows, cols] into head_dim-row blocks; orthogonalise and scale each."""
    m = np.asarray(m, dtype=np.float64)
    rows, cols = m.shape
    if head_dim <= 0 or rows % head_dim:
        raise ValueError("rows must be a positive multiple of head_dim")
    out = np.empty_like(m)
    s = per_head_scale(head_dim, cols)
    for blk in range(rows // head_dim):
        sl = slice(blk * head_dim, (blk + 1) * head_dim)
        out[sl] = newton_schulz5(m[sl], **kw) * s
    return out


def full_matrix_newton_schulz(m, **kw):
    """The whole matrix as one: Newton-Schulz times max(1, rows / cols) ** 0.5."""
    m = np.asarray(m, dtype=np.float64)
    return newton_schulz5(m, **kw) * full_matrix_scale(*m.shape)


def muon_orthogonalize(m, n_q=None, n_kv=None, head_dim=None):
    """The update a fused QKV weight gets: per head when its dim 0 is the exact
    fused total for (n_q, n_kv, head_dim), else as one matrix."""
    m = np.asarray(m, dtype=np.float64)
    if head_dim and fused_head_blocks(m.shape[0], n_q, n_kv, head_dim) is not None:
        return per_head_newton_schulz(m, head_dim)
    return full_matrix_newton_schulz(m)


def qkv_newton_schulz(layout, m_bits):
    """Per-head Newton-Schulz of a bf16 fused update (uint16 bits, [rows, cols])
    of a PackedLayout; float64 result. The packing (interleaved or sectioned)
    does not enter: only the row count is checked against the fused total."""
    m_bits = np.asarray(m_bits, dtype=np.uint16)
    if fused_head_blocks(m_bits.shape[0], layout.n_q, layout.n_kv, layout.head_dim) is None:
        raise ValueError("dim 0 is not (n_q + 2 n_kv) * head_dim")
    return per_head_newton_schulz(bf16_bits_to_f64(m_bits), layout.head_dim)

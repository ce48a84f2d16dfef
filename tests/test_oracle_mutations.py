"""Plant plausible mistakes in the oracle (on the CPU) and show that a pin catches each.

If one of these stops failing, the pins have lost the power to tell a correct
oracle from a wrong one.
"""

import numpy as np
import pytest

import oracle.bf16 as B
import oracle.newton_schulz as N
import oracle.prologue as P
import oracle_checks as C
import workloads


def _rope_sign_flipped(y, pos, base, inv_freq=None, scale=1.0):
    y = np.asarray(y, dtype=np.float64)
    half = y.shape[-1] // 2
    th = P.rope_angles(pos, y.shape[-1], base, inv_freq)[:, None, :]
    c, s = np.cos(th) * scale, np.sin(th) * scale
    a, b = y[..., :half], y[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def _rope_adjacent_pairs(y, pos, base, inv_freq=None, scale=1.0):
    y = np.asarray(y, dtype=np.float64)
    th = P.rope_angles(pos, y.shape[-1], base, inv_freq)[:, None, :]
    c, s = np.cos(th) * scale, np.sin(th) * scale
    a, b = y[..., 0::2], y[..., 1::2]
    out = np.empty_like(y)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def _rope_factor_on_cos_only(y, pos, base, inv_freq=None, scale=1.0):
    y = np.asarray(y, dtype=np.float64)
    half = y.shape[-1] // 2
    th = P.rope_angles(pos, y.shape[-1], base, inv_freq)[:, None, :]
    c, s = np.cos(th) * scale, np.sin(th)
    a, b = y[..., :half], y[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _angles_ignore_table(pos, head_dim, base, inv_freq=None):
    return np.asarray(pos, dtype=np.float64).reshape(-1, 1) * P.rope_inv_freq(head_dim, base)[None, :]


def _bias_reversed(packed, bias):
    x = np.asarray(packed, dtype=np.float64)
    return x if bias is None else x + np.asarray(bias, dtype=np.float64)[::-1][None, :]


def _bias_dropped(packed, bias):
    return np.asarray(packed, dtype=np.float64)


def _inv_freq_wrong_exponent(head_dim, base):
    return np.power(float(base), -np.arange(head_dim // 2, dtype=np.float64) / head_dim)


def _norm_eps_outside(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * w


def _norm_sum_not_mean(x, w, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * w


def _norm_bwd_missing_term(x, w, g, eps):
    x, g = np.asarray(x, dtype=np.float64), np.asarray(g, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return r * w * g, g * x * r


def _norm_bwd_wrong_power(x, w, g, eps):
    x, g = np.asarray(x, dtype=np.float64), np.asarray(g, dtype=np.float64)
    D = x.shape[-1]
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    dot = np.sum(x * w * g, axis=-1, keepdims=True)
    return r * w * g - x * (r ** 2 / D) * dot, g * x * r


def _blocks_k_v_swapped(layout):
    return [("v" if r == "k" else "k" if r == "v" else r, h) for r, h in _REAL_BLOCKS(layout)]


def _blocks_q_transposed(layout):
    # q head index taken as j * n_kv + g instead of g * G + j
    out = []
    for r, h in _REAL_BLOCKS(layout):
        if r == "q" and layout.kind == "interleaved":
            g, j = divmod(h, layout.group)
            h = j * layout.n_kv + g
        out.append((r, h))
    return out


_REAL_BLOCKS = P.head_blocks


def _bf16_via_float32(x):
    import torch

    with np.errstate(over="ignore"):
        t = torch.from_numpy(np.asarray(x, dtype=np.float64).astype(np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


_REAL_ROPE = P.rope_rotate_half


def _rope_transpose_is_forward(d, pos, base, inv_freq=None, scale=1.0):
    return _REAL_ROPE(d, pos, base, inv_freq, scale)


def _ns_variant(g, norm=lambda x: np.linalg.norm(x) + 1e-7, steps=5, coeffs=(3.4445, -4.7750, 2.0315),
                square=True):
    """Newton-Schulz written out with one planted change at a time."""
    x = np.asarray(g, dtype=np.float64)
    tall = x.shape[0] > x.shape[1]
    x = x.T if tall else x
    x = x / norm(x)
    a, b, c = coeffs
    for _ in range(steps):
        A = x @ x.T
        x = a * x + (b * A + c * (A @ A if square else A)) @ x
    return x.T if tall else x


def _ns_b_sign_flipped(g, **kw):
    return _ns_variant(g, coeffs=(3.4445, 4.7750, 2.0315))


def _ns_four_steps(g, **kw):
    return _ns_variant(g, steps=4)


def _ns_spectral_norm(g, **kw):
    return _ns_variant(g, norm=lambda x: np.linalg.norm(x, 2) + 1e-7)


def _ns_square_dropped(g, **kw):
    return _ns_variant(g, square=False)


def _ns_no_eps(g, **kw):
    return _ns_variant(g, norm=np.linalg.norm)


def _head_scale_whole_matrix(head_dim, in_features):
    return max(1.0, 3.0 * head_dim / in_features) ** 0.5


def _per_head_global_norm(m, head_dim, **kw):
    # the whole fused weight normalised once, no per-block normalisation
    m = np.asarray(m, dtype=np.float64)
    m = m / (np.linalg.norm(m) + 1e-7)
    out = np.empty_like(m)
    for blk in range(m.shape[0] // head_dim):
        sl = slice(blk * head_dim, (blk + 1) * head_dim)
        out[sl] = _ns_variant(m[sl], norm=lambda x: 1.0) * N.per_head_scale(head_dim, m.shape[1])
    return out


def _full_scale_cols_over_rows(rows, cols):
    return max(1.0, cols / rows) ** 0.5


def _blocks_any_multiple(rows, n_q, n_kv, head_dim):
    return rows // head_dim if head_dim and rows % head_dim == 0 else None


def _projection_w_not_transposed(x_bits, w_bits):
    x, w = B.bf16_bits_to_f64(x_bits), B.bf16_bits_to_f64(w_bits)
    return x @ w


def _projection_via_float32(x_bits, w_bits):
    return _bf16_via_float32(P.projection_f64(x_bits, w_bits).astype(np.float32).astype(np.float64))


def _projection_rows_reversed(x_bits, w_bits):
    x, w = B.bf16_bits_to_f64(x_bits), B.bf16_bits_to_f64(w_bits)
    return x @ w[::-1].T


def _checks_all(rng):
    """Every pin, run in turn; raises AssertionError at the first that fails."""
    C.check_to_bf16_rne(B, rng)
    for name in ("head_blocks_8q_over_2kv.txt", "head_blocks_muse_spark_16kv.txt"):
        C.check_head_block_fixture(P, name)
    C.check_rms_norm(P, rng)
    C.check_rope(P, rng)
    C.check_finite_differences(P, P.PackedLayout("interleaved", 2, 1, 8), rng, T=2)
    C.check_backward_invariants(P, P.PackedLayout("interleaved", 8, 2, 64), rng)
    C.check_pool_placement(P, B, rng)
    C.check_mla_rows(P, rng)
    C.check_variant_forward(P, rng)
    C.check_rope_extras(P, rng)
    C.check_variant_backward(P, rng)
    C.check_ns_svd_closed_form(N, rng)
    C.check_ns_equivariance(N, rng)
    C.check_ns_per_head(N, rng)
    C.check_ns_layout_equivalence(N, P, rng)
    C.check_ns_page_facts(N)
    C.check_ns_dispatch(N, rng)
    C.check_projection(P, rng)


def test_unmutated_oracle_passes_every_pin(rng):
    _checks_all(rng)


MUTATIONS = [
    (P, "rope_rotate_half", _rope_sign_flipped),
    (P, "rope_rotate_half", _rope_adjacent_pairs),
    (P, "rope_inv_freq", _inv_freq_wrong_exponent),
    (P, "rms_norm", _norm_eps_outside),
    (P, "rms_norm", _norm_sum_not_mean),
    (P, "rms_norm_backward", _norm_bwd_missing_term),
    (P, "rms_norm_backward", _norm_bwd_wrong_power),
    (P, "rope_rotate_half_transpose", _rope_transpose_is_forward),
    (P, "head_blocks", _blocks_k_v_swapped),
    (P, "head_blocks", _blocks_q_transposed),
    (B, "to_bf16_rne", _bf16_via_float32),
    (P, "rope_rotate_half", _rope_factor_on_cos_only),
    (P, "rope_angles", _angles_ignore_table),
    (P, "add_bias", _bias_reversed),
    (P, "add_bias", _bias_dropped),
    (N, "newton_schulz5", _ns_b_sign_flipped),
    (N, "newton_schulz5", _ns_four_steps),
    (N, "newton_schulz5", _ns_spectral_norm),
    (N, "newton_schulz5", _ns_square_dropped),
    (N, "newton_schulz5", _ns_no_eps),
    (N, "per_head_scale", _head_scale_whole_matrix),
    (N, "per_head_newton_schulz", _per_head_global_norm),
    (N, "fused_head_blocks", _blocks_any_multiple),
    (N, "full_matrix_scale", _full_scale_cols_over_rows),
    (P, "projection_f64", _projection_w_not_transposed),
    (P, "projection", _projection_via_float32),
    (P, "projection_f64", _projection_rows_reversed),
]


@pytest.mark.parametrize("module,name,bad", MUTATIONS, ids=[m[2].__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(module, name, bad, monkeypatch, rng):
    monkeypatch.setattr(module, name, bad)
    with pytest.raises(AssertionError):
        _checks_all(rng)


def test_planted_layout_mistake_breaks_layout_equivalence(monkeypatch):
    # a sectioned table that swaps two q heads must break interleaved == sectioned
    real = P.head_blocks

    def swapped(layout):
        b = real(layout)
        if layout.kind == "sectioned":
            b[0], b[1] = b[1], b[0]
        return b

    monkeypatch.setattr(P, "head_blocks", swapped)
    with pytest.raises(AssertionError):
        C.check_layout_equivalence(P, B, workloads.tiny())

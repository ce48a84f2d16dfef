"""The per-head Newton-Schulz kernels' evaluation order and arithmetic, checked on
the CPU against the fp64 oracle ("[muon] Per-head Newton-Schulz for fused QKV
projections"; Muon's quintic iteration).

1. The kernels evaluate X_5 = M X_0 with M = P_4 P_3 P_2 P_1 P_0,
   P_k = a I + b A_k + c A_k^2 and A_{k+1} = P_k A_k P_k, A_0 = X_0 X_0^T (every
   matrix a polynomial in A_0). In exact arithmetic that is the published
   iteration: here both are evaluated in float64 and must agree to rounding, on
   wide, square and tall blocks, with flat, decaying and low-rank spectra.
2. The kernels hold every matrix operand of the steps as two bf16 terms
   (hi = bf16(v), lo = bf16(v - hi)), form each product as hi.hi + hi.lo + lo.hi
   with float32 accumulation and apply M as hi X + lo X. Emulated here, that
   arithmetic stays well inside the parity bound of the GPU tests (the error of
   the oracle's own bf16 steps); one-term operands (bf16, or tf32) do not on an
   ill-conditioned block, because M is about a^5 on its nearly rank-deficient
   directions and one term loses the small eigenvalues next to it.

The emulation is test code written from the description above; it shares
nothing with the CUDA sources.
"""

import numpy as np
import pytest

import oracle.newton_schulz as N
from oracle.bf16 import bf16_bits_to_f64, to_bf16_rne

A_, B_, C_ = N.NS_COEFFS


def _r16(v):
    return bf16_bits_to_f64(to_bf16_rne(np.asarray(v, dtype=np.float64)))


def _f32(v):
    return np.asarray(v, dtype=np.float32).astype(np.float64)


def _tf32(v):
    """Round to the nearest tf32 (10 explicit mantissa bits), ties away."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x1000) >> 13) << 13
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def gram_polynomial_f64(g, eps=N.NS_EPS):
    """X_5 through the Gram matrix, float64 throughout (no transpose for tall blocks)."""
    g = np.asarray(g, dtype=np.float64)
    inv = 1.0 / (np.linalg.norm(g) + eps)
    A = (g @ g.T) * inv * inv
    eye = np.eye(g.shape[0])
    M = eye
    for _ in range(N.NS_STEPS):
        P = A_ * eye + B_ * A + C_ * (A @ A)
        M = P @ M
        A = P @ A @ P
    return M @ g * inv


def kernel_arithmetic(g, terms="two", eps=N.NS_EPS):
    """The kernels' rounding points, emulated: the Gram matrix from the bf16 block in
    float32; the steps with operands in `terms` ("two": hi + lo bf16, three MMAs per
    product; "bf16" or "tf32": one term) and float32 accumulation; M applied to the
    bf16 block in the same form; the result rounded to bf16."""
    x0 = _r16(g)
    araw = _f32(x0 @ x0.T)
    inv = float(_f32(1.0 / _f32(np.sqrt(_f32(np.trace(araw))) + eps)))
    if terms == "two":
        split = lambda v: (_r16(v), _r16(_f32(v - _r16(v))))  # noqa: E731

        def mm(x, y):  # x y^T from hi/lo terms: hi hi + hi lo + lo hi
            xh, xl = split(x)
            yh, yl = split(y)
            return _f32(xh @ yh.T + xh @ yl.T + xl @ yh.T)
    else:
        rnd = _r16 if terms == "bf16" else _tf32

        def mm(x, y):
            return _f32(rnd(x) @ rnd(y).T)
    A = _f32(_f32(araw * inv) * inv)
    eye = np.eye(A.shape[0])
    M = eye
    for k in range(N.NS_STEPS):
        S = mm(A, A)
        P = _f32(_f32(C_ * S + _f32(B_ * A)) + A_ * eye)
        if k < N.NS_STEPS - 1:
            A = mm(mm(P, A), P)
        M = mm(P, M)
    Mh = _f32(M * inv)
    if terms == "two":
        hi = _r16(Mh)
        lo = _r16(_f32(Mh - hi))
        y = _f32(hi @ x0 + lo @ x0)
    else:
        y = _f32((_r16 if terms == "bf16" else _tf32)(Mh) @ x0)
    return _r16(y)


def _blocks():
    rng = np.random.default_rng(2024)
    out = [("wide N(0,1)", rng.standard_normal((64, 512))),
           ("square N(0,1)", rng.standard_normal((64, 64))),
           ("tall N(0,1)", rng.standard_normal((128, 64)))]
    q1, _ = np.linalg.qr(rng.standard_normal((64, 64)))
    q2, _ = np.linalg.qr(rng.standard_normal((512, 64)))
    out.append(("decaying spectrum", (q1 * np.exp(-np.arange(64) / 6.0)) @ q2.T))
    out.append(("rank 4 + noise", rng.standard_normal((64, 4)) @ rng.standard_normal((4, 512))
                + 1e-3 * rng.standard_normal((64, 512))))
    return out


@pytest.mark.parametrize("name,g", _blocks(), ids=[n for n, _ in _blocks()])
def test_gram_polynomial_is_the_iteration(name, g):
    exact = N.newton_schulz5(g)
    got = gram_polynomial_f64(g)
    assert np.abs(got - exact).max() <= 1e-9 * max(1.0, np.abs(exact).max()), name


def _rel(got, exact):
    return np.linalg.norm(got - exact) / np.linalg.norm(exact)


@pytest.mark.parametrize("name,g", _blocks(), ids=[n for n, _ in _blocks()])
def test_two_term_operands_stay_inside_the_parity_bound(name, g):
    g = _r16(g)
    exact = N.newton_schulz5(g)
    e_bf16_steps = _rel(N.newton_schulz5(g, rounding=_r16), exact)
    e_round = _rel(_r16(exact), exact)
    got = kernel_arithmetic(g, "two")
    # the GPU tests' tight bound: the output's own rounding plus a quarter of the bf16 steps' error
    assert _rel(got, exact) <= 1.25 * e_round + 0.25 * e_bf16_steps, name


@pytest.mark.parametrize("terms", ["bf16", "tf32"])
def test_one_term_operands_fail_an_ill_conditioned_block(terms):
    # the decaying spectrum (singular values e^(-i/6)): with one term the steps
    # lose the small eigenvalues of M next to its a^5 null-space part
    name, g = _blocks()[3]
    g = _r16(g)
    exact = N.newton_schulz5(g)
    bound = 2 * _rel(N.newton_schulz5(g, rounding=_r16), exact) + 2.0 ** -9  # the GPU tests' R29 bound
    assert _rel(kernel_arithmetic(g, "two"), exact) <= bound
    assert _rel(kernel_arithmetic(g, terms), exact) > bound, f"{terms} unexpectedly within R29 on {name}"

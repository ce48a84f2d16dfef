"""Checks that pin the fp64 oracle to facts other than itself.

Each check takes the oracle's modules (``P`` = oracle.prologue, ``B`` =
oracle.bf16) and calls their functions by attribute, so a test can plant a
mistake in one oracle function (monkeypatch) and show that some check fails.
A check raises AssertionError when the oracle disagrees with the fact it pins.

What pins what:
  bf16 rounding     exact rational nearest-even search (fractions.Fraction)
  bf16 widening     struct unpacking of every 16-bit pattern
  split / layouts   the pages' stated head-block orders (tests/golden/), a
                    pure-permutation check, sectioned == interleaved
  RMSNorm           rms == 1 (w=1, eps=0), the eps closed form, one-hot and
                    constant vectors by hand, power-of-two scale invariance
  RoPE              complex-multiplication form, pos 0 identity, pairwise norm,
                    relative position, inv_freq closed values, cos(pos) at i=0
  backward          central finite differences of the forward, eps=0
                    orthogonality, R^T as the adjoint of R, dv passthrough
  pool writes       exact placement and untouched bytes
  variant options   norm off = pure split / pairwise-norm keeping rotation,
                    bias order through the pinned split, bias before the norm
                    (rms 1) and the rotation, one-hot frequency tables, the
                    cos/sin factor at position 0, finite differences of all
  projection       x . W^T against exact rational sums rounded by the exact
                    nearest-even search (square and non-square weights, rows
                    in packed order), a sum one 2**-30 past a bf16 tie (one
                    rounding, not two), W = identity / a row permutation
                    handing the prologue exactly x / x's columns permuted
  per-head Newton-  known-SVD closed forms through a scalar recursion on the
  Schulz            singular values (Muon's published constants, typed here
                    on their own), the 1e-7 on a tiny matrix, orthogonal
                    equivariance, block independence, the tall-block factor,
                    sectioned == interleaved up to the block permutation, the
                    page's split / no-split cases and scales (tests/golden/)
"""

import math
import os
import struct
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 ----

def _exact_bf16_rne(x):
    """Nearest bf16 to x (a float or an exact Fraction) by exact rational
    comparison (ties -> even)."""
    if isinstance(x, Fraction):
        sign = 0x8000 if x < 0 else 0
        X = abs(x)
        ax = float(X)  # within one float64 ulp of X: the candidate window below covers it
    else:
        if math.isnan(x):
            return 0x7FC0
        sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
        ax = abs(x)
        if math.isinf(ax):
            return sign | 0x7F80
        X = Fraction(ax)
    # Candidates: the bf16 patterns around the float32 truncation of |x|.
    f32 = struct.unpack("<I", struct.pack("<f", min(ax, 3.4e38)))[0] >> 16
    best, best_d = None, None
    for b in range(max(0, f32 - 2), min(0x7F80, f32 + 3) + 1):
        if b == 0x7F80:
            val = Fraction(2) ** 128  # overflow rounds like a value at 2**128
        else:
            val = Fraction(struct.unpack("<f", struct.pack("<I", b << 16))[0])
        d = abs(X - val)
        if best is None or d < best_d or (d == best_d and b % 2 == 0):
            best, best_d = b, d
    return sign | best


def bf16_test_values(rng):
    vals = list(rng.standard_normal(4000) * np.exp2(rng.integers(-30, 30, 4000)))
    # exact ties and values one float64 ulp either side of a tie
    for b in rng.integers(0x0001, 0x7F7F, 600):
        lo = struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]
        hi = struct.unpack("<f", struct.pack("<I", (int(b) + 1) << 16))[0]
        mid = (lo + hi) / 2.0
        vals += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, np.inf), -mid]
    vals += [0.0, -0.0, 1e-45, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126,
             3.3895313892515355e38, 3.3961775292304e38, 3.4e38, 1e39, -1e39, 1.0, -1.0]
    return np.array(vals, dtype=np.float64)


def check_to_bf16_rne(B, rng):
    x = bf16_test_values(rng)
    got = B.to_bf16_rne(x)
    want = np.array([_exact_bf16_rne(float(v)) for v in x], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"to_bf16_rne wrong at {x[bad[:5]]}: {got[bad[:5]]} vs {want[bad[:5]]}"


def check_bf16_widen(B):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = B.bf16_bits_to_f64(bits)
    want = np.array([struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in range(65536)])
    ok = (got == want) | (np.isnan(got) & np.isnan(want))
    assert ok.all()


# ------------------------------------------------------------- layouts ----

def read_block_fixture(name):
    """Parse a tests/golden head-block fixture into (n_q, n_kv, D, {kind: [blocks]})."""
    meta, orders = {}, {"interleaved": [], "sectioned": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key in ("n_q", "n_kv", "head_dim"):
                meta[key] = int(rest[0])
            elif key in ("sectioned", "interleaved"):
                orders[key] += rest
            elif key == "interleaved_group":
                orders["interleaved"] += rest[1:]
    parse = lambda tok: (tok[0], int(tok[1:]))  # noqa: E731
    return meta["n_q"], meta["n_kv"], meta["head_dim"], {
        k: [parse(t) for t in v] for k, v in orders.items() if v}


def check_head_block_fixture(P, name):
    n_q, n_kv, D, orders = read_block_fixture(name)
    for kind, want in orders.items():
        got = P.head_blocks(P.PackedLayout(kind, n_q, n_kv, D))
        assert got == want, f"{name} {kind}: {got[:12]} vs {want[:12]}"


def check_split_is_permutation(P, layout, T=3):
    """Each packed element lands in exactly one output slot, unchanged."""
    ids = np.arange(T * layout.row_width, dtype=np.int64).reshape(T, layout.row_width)
    q, k, v = P.split_heads(layout, ids)
    assert q.shape == (T, layout.n_q, layout.head_dim)
    assert k.shape == v.shape == (T, layout.n_kv, layout.head_dim)
    allv = np.concatenate([q.ravel(), k.ravel(), v.ravel()])
    assert np.array_equal(np.sort(allv), ids.ravel())
    # token t's heads come from token t's row only
    for t in range(T):
        lo, hi = t * layout.row_width, (t + 1) * layout.row_width
        for a in (q[t], k[t], v[t]):
            assert a.min() >= lo and a.max() < hi
    # and each head is one contiguous head_dim block of the row
    for a in (q, k, v):
        assert np.all(np.diff(a, axis=-1) == 1)
        assert np.all(a[..., 0] % layout.head_dim == 0)


def check_layout_equivalence(P, B, wl):
    """Interleaved and sectioned packings of the same heads give identical results."""
    from workloads import bits_u16

    Li = P.PackedLayout("interleaved", wl.n_q, wl.n_kv, wl.head_dim)
    Ls = P.PackedLayout("sectioned", wl.n_q, wl.n_kv, wl.head_dim)
    wq, wk = wl.w_q.numpy(), wl.w_k.numpy()
    oi = P.prologue_fwd(Li, bits_u16(wl.packed_rows()), wl.pos.numpy(), wq, wk, wl.eps, wl.rope_base, wl.nope)
    os_ = P.prologue_fwd(Ls, bits_u16(wl.sectioned_rows()), wl.pos.numpy(), wq, wk, wl.eps, wl.rope_base, wl.nope)
    for key in ("q", "k", "v_bits", "q_pre_bits", "k_pre_bits"):
        assert np.array_equal(oi[key], os_[key]), key


# ------------------------------------------------------------- RMSNorm ----

def check_rms_norm(P, rng):
    D = 64
    ones = np.ones(D)
    for scale in (1e-3, 1.0, 37.0):
        x = rng.standard_normal((5, 7, D)) * scale
        y = P.rms_norm(x, ones, 0.0)
        assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=0, atol=1e-14)
        # eps inside the root: rms(y) = sqrt(ms / (ms + eps))
        eps = 0.25 * scale * scale
        ms = np.mean(x * x, axis=-1)
        y = P.rms_norm(x, ones, eps)
        assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + eps)), rtol=1e-13, atol=0)
    # one-hot: mean over D (not a sum, not D-1): y_0 = sqrt(D) * w_0 when eps = 0
    w = rng.uniform(0.5, 1.5, D)
    x = np.zeros(D)
    x[0] = 3.0
    y = P.rms_norm(x, w, 0.0)
    assert abs(y[0] - math.sqrt(D) * w[0]) <= 1e-14 * math.sqrt(D) and np.all(y[1:] == 0)
    # constant vector c: y = c / sqrt(c^2 + eps) * w
    c, eps = -0.75, 1e-6
    y = P.rms_norm(np.full(D, c), w, eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps) * w, rtol=1e-15, atol=0)
    # two-element head, by hand: x = (3, 4): mean square 12.5
    y = P.rms_norm(np.array([3.0, 4.0]), np.array([2.0, 0.5]), 0.5)
    assert np.allclose(y, [3.0 / math.sqrt(13.0) * 2.0, 4.0 / math.sqrt(13.0) * 0.5], rtol=1e-15, atol=0)
    # power-of-two scale invariance with eps = 0 (exact in binary floating point)
    x = rng.standard_normal((4, D))
    assert np.array_equal(P.rms_norm(x * 2.0 ** 9, w, 0.0), P.rms_norm(x, w, 0.0))
    # each head is normalised on its own
    x = rng.standard_normal((2, 3, D))
    x2 = x.copy()
    x2[:, 1, :] *= 10.0
    assert np.array_equal(P.rms_norm(x, w, 1e-6)[:, 0], P.rms_norm(x2, w, 1e-6)[:, 0])


# ---------------------------------------------------------------- RoPE ----

def check_rope(P, rng):
    D = 64
    half = D // 2
    # inverse frequencies: base**(-2i/D); i = 0 is exactly 1, i = D/4 is base**-0.5
    f = P.rope_inv_freq(D, 10000.0)
    assert f.shape == (half,) and f[0] == 1.0
    assert abs(f[D // 4] - 0.01) <= 1e-17
    assert abs(f[half - 1] - 10000.0 ** (-(D - 2) / D)) <= 1e-18
    assert np.all(np.diff(f) < 0)
    pos = rng.integers(0, 400000, 6)
    y = rng.standard_normal((6, 3, D))
    o = P.rope_rotate_half(y, pos, 500000.0)
    # complex form: (y_i + i y_{i+D/2}) * exp(i pos inv_freq_i)
    th = pos[:, None].astype(np.float64) * P.rope_inv_freq(D, 500000.0)[None, :]
    z = (y[..., :half] + 1j * y[..., half:]) * np.exp(1j * th)[:, None, :]
    assert np.allclose(o[..., :half], z.real, rtol=0, atol=1e-12)
    assert np.allclose(o[..., half:], z.imag, rtol=0, atol=1e-12)
    # i = 0 turns by exactly pos radians
    assert np.allclose(o[:, :, 0], y[:, :, 0] * np.cos(pos.astype(float))[:, None]
                       - y[:, :, half] * np.sin(pos.astype(float))[:, None], rtol=0, atol=1e-12)
    # pairwise norm preserved
    assert np.allclose(o[..., :half] ** 2 + o[..., half:] ** 2, y[..., :half] ** 2 + y[..., half:] ** 2,
                       rtol=1e-12, atol=1e-13)
    # position 0 is the identity
    assert np.array_equal(P.rope_rotate_half(y, np.zeros(6, np.int64), 500000.0), y)
    # relative position: <R_m q, R_n k> depends on n - m only
    qv, kv = rng.standard_normal((1, 1, D)), rng.standard_normal((1, 1, D))
    for m, n, s in ((3, 17, 1000), (100, 5, 250000), (0, 393215, -7)):
        a = np.sum(P.rope_rotate_half(qv, [m], 1e4) * P.rope_rotate_half(kv, [n], 1e4))
        b = np.sum(P.rope_rotate_half(qv, [m + s], 1e4) * P.rope_rotate_half(kv, [n + s], 1e4))
        assert abs(a - b) <= 1e-9 * (1 + abs(a))
    # R^T is the adjoint (and the inverse) of R
    g = rng.standard_normal((6, 3, D))
    lhs = np.sum(P.rope_rotate_half(g, pos, 5e5) * y)
    rhs = np.sum(g * P.rope_rotate_half_transpose(y, pos, 5e5))
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs))
    assert np.allclose(P.rope_rotate_half_transpose(o, pos, 500000.0), y, rtol=0, atol=1e-12)


def check_nope_is_rope_at_zero(P, layout, rng, T=4):
    from workloads import norm_weight, _gen

    g = _gen(11)
    x = rng.standard_normal((T, layout.row_width))
    wq, wk = norm_weight(layout.head_dim, g).numpy(), norm_weight(layout.head_dim, g).numpy()
    a = P.prologue_fwd_f64(layout, x, np.zeros(T, np.int64), wq, wk, 1e-6, 5e5, nope=False)
    b = P.prologue_fwd_f64(layout, x, np.arange(T), wq, wk, 1e-6, 5e5, nope=True)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ------------------------------------------------------------ backward ----

def _loss(P, layout, x, wq, wk, pos, eps, base, nope, dq, dk, dv, variant):
    q, k, v = P.prologue_fwd_f64(layout, x, pos, wq, wk, eps, base, nope, **variant)
    return np.sum(dq * q) + np.sum(dk * k) + np.sum(dv * v)


def check_finite_differences(P, layout, rng, T=3, nope=False, n_probe=None, base=10000.0, **variant):
    """Central differences of L = <dq,q> + <dk,k> + <dv,v> against prologue_bwd_f64.

    `variant` (norm / bias / inv_freq / rope_scale) goes to both the forward and
    the backward; with a bias the bias gradient is probed too."""
    D = layout.head_dim
    x = rng.standard_normal((T, layout.row_width))
    wq, wk = rng.uniform(0.5, 1.5, D), rng.uniform(0.5, 1.5, D)
    pos = rng.integers(0, 5000, T)
    eps = 1e-3  # large enough to matter in the derivative
    dq = rng.standard_normal((T, layout.n_q, D))
    dk = rng.standard_normal((T, layout.n_kv, D))
    dv = rng.standard_normal((T, layout.n_kv, D))
    xq, xk, _ = P.split_heads(layout, x)
    got = P.prologue_bwd_f64(layout, dq, dk, dv, xq, xk, pos, wq, wk, eps, base, nope, **variant)
    args = (pos, eps, base, nope, dq, dk, dv)
    h = 1e-6

    def loss(xx, a, b, var):
        return _loss(P, layout, xx, a, b, *args, var)

    idx = [(t, j) for t in range(T) for j in range(layout.row_width)]
    if n_probe is not None:
        pick = rng.choice(len(idx), size=min(n_probe, len(idx)), replace=False)
        idx = [idx[i] for i in pick]
    for t, j in idx:
        xp, xm = x.copy(), x.copy()
        xp[t, j] += h
        xm[t, j] -= h
        fd = (loss(xp, wq, wk, variant) - loss(xm, wq, wk, variant)) / (2 * h)
        an = got["dpacked"][t, j]
        assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (t, j, fd, an)
    for which, w in (("dw_q", wq), ("dw_k", wk)):
        for d in range(D):
            wp, wm = w.copy(), w.copy()
            wp[d] += h
            wm[d] -= h
            if which == "dw_q":
                lp, lm = loss(x, wp, wk, variant), loss(x, wm, wk, variant)
            else:
                lp, lm = loss(x, wq, wp, variant), loss(x, wq, wm, variant)
            fd = (lp - lm) / (2 * h)
            an = got[which][d]
            assert abs(fd - an) <= 1e-6 * (1 + abs(an)), (which, d, fd, an)
    if variant.get("bias") is not None:
        b = np.asarray(variant["bias"], dtype=np.float64)
        cols = range(layout.row_width) if n_probe is None else rng.choice(layout.row_width, n_probe, replace=False)
        for j in cols:
            bp, bm = b.copy(), b.copy()
            bp[j] += h
            bm[j] -= h
            fd = (loss(x, wq, wk, dict(variant, bias=bp)) - loss(x, wq, wk, dict(variant, bias=bm))) / (2 * h)
            an = got["db"][j]
            assert abs(fd - an) <= 1e-6 * (1 + abs(an)), ("db", j, fd, an)
    else:
        assert got["db"] is None


def check_backward_invariants(P, layout, rng, T=5):
    D = layout.head_dim
    x = rng.standard_normal((T, layout.row_width))
    xq, xk, _ = P.split_heads(layout, x)
    wq, wk = rng.uniform(0.5, 1.5, D), rng.uniform(0.5, 1.5, D)
    dq = rng.standard_normal((T, layout.n_q, D))
    dk = rng.standard_normal((T, layout.n_kv, D))
    dv = rng.standard_normal((T, layout.n_kv, D))
    pos = rng.integers(0, 131072, T)
    out = P.prologue_bwd_f64(layout, dq, dk, dv, xq, xk, pos, wq, wk, 0.0, 5e5, False)
    gq, gk, gv = P.split_heads(layout, out["dpacked"])
    # v slots carry dv unchanged
    assert np.array_equal(gv, dv)
    # eps = 0: the norm is scale invariant, so its input gradient is orthogonal to x
    for xs, gs in ((xq, gq), (xk, gk)):
        dots = np.sum(xs * gs, axis=-1)
        scale = np.sqrt(np.sum(xs * xs, axis=-1) * np.sum(gs * gs, axis=-1))
        assert np.all(np.abs(dots) <= 1e-12 * scale)


# --------------------------------------------------------------- pools ----

def check_pool_placement(P, B, rng):
    layout = P.PackedLayout("interleaved", 8, 2, 64)
    T, num_pages, page_size = 7, 5, 4
    bits = B.to_bf16_rne(rng.standard_normal((T, layout.row_width)))
    slots = rng.choice(num_pages * page_size, size=T, replace=False)
    page, off = slots // page_size, slots % page_size
    shape = (num_pages, page_size, layout.n_kv, layout.head_dim)
    kp0 = rng.integers(0, 65536, shape).astype(np.uint16)
    vp0 = rng.integers(0, 65536, shape).astype(np.uint16)
    wq, wk = rng.uniform(0.5, 1.5, 64), rng.uniform(0.5, 1.5, 64)
    pos = rng.integers(0, 131072, T)
    q, k, kp, vp = P.pool_write(layout, bits, pos, wq, wk, 1e-6, 5e5, False, page, off, kp0, vp0)
    ref = P.prologue_fwd(layout, bits, pos, wq, wk, 1e-6, 5e5, False)
    written = np.zeros((num_pages, page_size), bool)
    for t in range(T):
        written[page[t], off[t]] = True
        assert np.array_equal(kp[page[t], off[t]], B.to_bf16_rne(ref["k"][t]))
        # v goes in raw: the packed row's v-slot bits
        assert np.array_equal(vp[page[t], off[t]], bits[t].reshape(-1, 64)[[5, 11]])
    assert np.array_equal(kp[~written], kp0[~written])
    assert np.array_equal(vp[~written], vp0[~written])
    assert np.array_equal(q, ref["q"])


def check_mla_rows(P, rng):
    T = 5
    x = rng.standard_normal((T, 576))
    w = rng.uniform(0.5, 1.5, 512)
    pos = rng.integers(0, 393216, T)
    o = P.mla_rows_f64(x, pos, w, 0.0, 1e4, 512, 64)
    # latent part: rms(y / w) == 1 with eps = 0; it ignores the rope part
    assert np.allclose(np.sqrt(np.mean((o[:, :512] / w) ** 2, axis=-1)), 1.0, rtol=0, atol=1e-14)
    x2 = x.copy()
    x2[:, 512:] *= 100.0
    assert np.array_equal(P.mla_rows_f64(x2, pos, w, 0.0, 1e4, 512, 64)[:, :512], o[:, :512])
    # rope part: complex form with D = 64, base 1e4, not normalised, no weight
    th = pos[:, None].astype(np.float64) * (1e4 ** (-np.arange(32) / 32.0))[None, :]
    z = (x[:, 512:544] + 1j * x[:, 544:576]) * np.exp(1j * th)
    assert np.allclose(o[:, 512:544], z.real, atol=1e-12, rtol=0)
    assert np.allclose(o[:, 544:576], z.imag, atol=1e-12, rtol=0)
    # position 0 leaves the rope part unchanged
    o0 = P.mla_rows_f64(x, np.zeros(T, np.int64), w, 0.0, 1e4, 512, 64)
    assert np.array_equal(o0[:, 512:], x[:, 512:])


# ------------------------------------------------ GQAttention variant ----

def check_variant_forward(P, rng):
    """Norm off, the qkv bias: what each option does, from facts outside the
    oracle's own formulas (the pinned split, pairwise norms, closed values)."""
    for kind in ("interleaved", "sectioned"):
        layout = P.PackedLayout(kind, 8, 2, 64)
        T, D, W, h = 4, layout.head_dim, layout.row_width, layout.head_dim // 2
        x = rng.standard_normal((T, W))
        pos = rng.integers(1, 131072, T)
        ones = np.ones(D)
        xq, xk, xv = P.split_heads(layout, x)
        # norm off and NoPE: a pure split
        q, k, v = P.prologue_fwd_f64(layout, x, pos, ones, ones, 1e-6, 5e5, nope=True, norm=False)
        assert np.array_equal(q, xq) and np.array_equal(k, xk) and np.array_equal(v, xv)
        # norm off with RoPE: the identity at position 0, and it keeps every
        # rotate-half pair's norm elsewhere (with the norm on it would not)
        q0, k0, _ = P.prologue_fwd_f64(layout, x, np.zeros(T, np.int64), ones, ones, 1e-6, 5e5, norm=False)
        assert np.array_equal(q0, xq) and np.array_equal(k0, xk)
        q, k, _ = P.prologue_fwd_f64(layout, x, pos, ones, ones, 1e-6, 5e5, norm=False)
        for o, i in ((q, xq), (k, xk)):
            assert np.allclose(o[..., :h] ** 2 + o[..., h:] ** 2, i[..., :h] ** 2 + i[..., h:] ** 2,
                               rtol=1e-12, atol=1e-13)
            assert not np.allclose(o, i)
        # the bias is in the packed row's order: with x = 0 and nothing else
        # applied the outputs are the bias split by the pinned head-block table
        b = np.arange(W, dtype=np.float64) + 1.0
        z = np.zeros((T, W))
        q, k, v = P.prologue_fwd_f64(layout, z, pos, ones, ones, 1e-6, 5e5, nope=True, norm=False, bias=b)
        bq, bk, bv = P.split_heads(layout, np.tile(b, (T, 1)))
        assert np.array_equal(q, bq) and np.array_equal(k, bk) and np.array_equal(v, bv)
        # the bias goes in before the norm: w = 1, eps = 0 gives every head of the
        # normed bias an rms of exactly 1 (added after the norm it would keep b's)
        q, k, _ = P.prologue_fwd_f64(layout, z, pos, ones, ones, 0.0, 5e5, bias=b)
        for o in (q, k):
            assert np.allclose(np.sqrt(np.mean(o * o, axis=-1)), 1.0, rtol=0, atol=1e-14)
        # and before the rotation: norm off, the roped bias keeps its pairwise norms
        q, k, _ = P.prologue_fwd_f64(layout, z, pos, ones, ones, 1e-6, 5e5, norm=False, bias=b)
        for o, i in ((q, bq), (k, bk)):
            assert np.allclose(o[..., :h] ** 2 + o[..., h:] ** 2, i[..., :h] ** 2 + i[..., h:] ** 2,
                               rtol=1e-12, atol=1e-9)
        # a bias that cancels the input zeroes every output (norm: 0 * r * w = 0)
        q, k, v = P.prologue_fwd_f64(layout, x[:1], pos[:1], ones, ones, 1e-6, 5e5, bias=-x[0])
        assert not np.any(q) and not np.any(k) and not np.any(v)


def check_rope_extras(P, rng):
    """A caller-given frequency table and the cos/sin factor."""
    D, h = 64, 32
    pos = rng.integers(1, 131072, 5)
    y = rng.standard_normal((5, 3, D))
    # the default table passed explicitly changes nothing
    f = P.rope_inv_freq(D, 5e5)
    assert np.array_equal(P.rope_rotate_half(y, pos, 5e5, inv_freq=f), P.rope_rotate_half(y, pos, 5e5))
    # a one-hot table turns pair 0 by pos radians (the base is not used) and
    # leaves every other pair alone
    one = np.zeros(h)
    one[0] = 1.0
    o = P.rope_rotate_half(y, pos, 5e5, inv_freq=one)
    assert np.array_equal(o[..., 1:h], y[..., 1:h]) and np.array_equal(o[..., h + 1:], y[..., h + 1:])
    p = pos.astype(np.float64)[:, None]
    assert np.allclose(o[..., 0], y[..., 0] * np.cos(p) - y[..., h] * np.sin(p), rtol=0, atol=1e-12)
    assert np.allclose(o[..., h], y[..., h] * np.cos(p) + y[..., 0] * np.sin(p), rtol=0, atol=1e-12)
    # cos and sin both carry the factor: position 0 gives factor * y, and every
    # pair's norm is multiplied by factor**2
    assert np.array_equal(P.rope_rotate_half(y, np.zeros(5, np.int64), 5e5, scale=2.0), 2.0 * y)
    o = P.rope_rotate_half(y, pos, 5e5, scale=1.5)
    assert np.allclose(o[..., :h] ** 2 + o[..., h:] ** 2, 2.25 * (y[..., :h] ** 2 + y[..., h:] ** 2),
                       rtol=1e-12, atol=1e-12)
    # the transpose with the same table and factor is the adjoint
    g = rng.standard_normal((5, 3, D))
    ff = rng.uniform(0.0, 1.0, h)
    lhs = np.sum(P.rope_rotate_half(g, pos, 1.0, inv_freq=ff, scale=1.3) * y)
    rhs = np.sum(g * P.rope_rotate_half_transpose(y, pos, 1.0, inv_freq=ff, scale=1.3))
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs))


def check_variant_backward(P, rng):
    """Finite differences of the forward with every option, on tiny shapes."""
    layout = P.PackedLayout("interleaved", 2, 1, 8)
    W = layout.row_width
    b = rng.standard_normal(W)
    ff = rng.uniform(0.0, 1.0, layout.head_dim // 2)
    check_finite_differences(P, layout, rng, T=2, norm=False)
    check_finite_differences(P, layout, rng, T=2, norm=False, bias=b, inv_freq=ff, rope_scale=1.25)
    check_finite_differences(P, layout, rng, T=2, bias=b)
    check_finite_differences(P, P.PackedLayout("sectioned", 2, 1, 8), rng, T=2, bias=b, rope_scale=0.75)
    # without the norm there is nothing for the weights: dw is zero
    x = rng.standard_normal((3, W))
    xq, xk, _ = P.split_heads(layout, x)
    d = [rng.standard_normal((3, n, 8)) for n in (layout.n_q, layout.n_kv, layout.n_kv)]
    out = P.prologue_bwd_f64(layout, *d, xq, xk, [1, 2, 3], np.ones(8), np.ones(8), 1e-6, 1e4, norm=False)
    assert not np.any(out["dw_q"]) and not np.any(out["dw_k"])


# ---------------------------------------------- per-head Newton-Schulz ----

# Muon's quintic constants and step count as published with the optimizer
# (Jordan et al., 2024), typed here independently of the oracle's copy.
_MUON_ABC = (3.4445, -4.7750, 2.0315)
_MUON_STEPS = 5


def _phi5(sigma):
    """What five Newton-Schulz steps do to one singular value."""
    a, b, c = _MUON_ABC
    s = np.asarray(sigma, dtype=np.float64)
    for _ in range(_MUON_STEPS):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def _orthonormal_columns(rng, n, k):
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def _ns_by_svd(g):
    """Newton-Schulz of g through its SVD: U phi5(s / (||g||_F + 1e-7)) V^T."""
    U, s, Vt = np.linalg.svd(np.asarray(g, dtype=np.float64), full_matrices=False)
    return (U * _phi5(s / (np.sqrt(np.sum(s * s)) + 1e-7))) @ Vt


def check_ns_svd_closed_form(N, rng):
    """A matrix built from a known SVD: the iteration acts on each singular value
    alone. Wide, square and tall shapes; a tiny matrix shows the 1e-7."""
    for m, n in [(8, 24), (16, 16), (24, 8), (64, 512)]:
        k = min(m, n)
        U, V = _orthonormal_columns(rng, m, k), _orthonormal_columns(rng, n, k)
        s = np.sort(rng.uniform(0.05, 3.0, k))[::-1]
        for mag in (1.0, 1e-7):
            sm = s * mag
            want = (U * _phi5(sm / (np.sqrt(np.sum(sm * sm)) + 1e-7))) @ V.T
            got = N.newton_schulz5((U * sm) @ V.T)
            err = np.abs(got - want).max()
            assert err <= 1e-9 * max(1.0, np.abs(want).max()), f"svd closed form {m}x{n} mag {mag}: {err}"
    # equal singular values: s Q with orthonormal rows maps to phi5(1/(sqrt(k) + 1e-7/s)) Q
    Q = _orthonormal_columns(rng, 40, 8).T
    got = N.newton_schulz5(3.0 * Q)
    assert np.allclose(got, _phi5(3.0 / (3.0 * np.sqrt(8) + 1e-7)) * Q, rtol=0, atol=1e-12)


def check_ns_equivariance(N, rng):
    """NS(P G Q^T) = P NS(G) Q^T for orthogonal P, Q (order of the products)."""
    for m, n in [(6, 10), (10, 6), (7, 7)]:
        g = rng.standard_normal((m, n))
        Pm, Qm = _orthonormal_columns(rng, m, m), _orthonormal_columns(rng, n, n)
        lhs = N.newton_schulz5(Pm @ g @ Qm.T)
        rhs = Pm @ N.newton_schulz5(g) @ Qm.T
        assert np.abs(lhs - rhs).max() <= 1e-10, f"equivariance {m}x{n}"


def check_ns_per_head(N, rng):
    """Blocks are independent, each normalised on its own, scaled by
    max(1, head_dim / in_features) ** 0.5 (wide: 1; tall: sqrt(D / in))."""
    D, cols = 8, 24
    m = rng.standard_normal((4 * D, cols)) * np.repeat([1e-3, 1.0, 1e3, 7.0], D)[:, None]
    out = N.per_head_newton_schulz(m, D)
    for blk in range(4):
        sl = slice(blk * D, (blk + 1) * D)
        assert np.abs(out[sl] - _ns_by_svd(m[sl])).max() <= 1e-9, f"block {blk}"
    m2 = m.copy()
    m2[:D] = rng.standard_normal((D, cols))
    out2 = N.per_head_newton_schulz(m2, D)
    assert np.array_equal(out2[D:], out[D:]), "a block's result depends on another block"
    # tall blocks (head_dim 16 over 8 inputs): factor sqrt(2)
    t = rng.standard_normal((3 * 16, 8))
    out = N.per_head_newton_schulz(t, 16)
    for blk in range(3):
        sl = slice(blk * 16, (blk + 1) * 16)
        assert np.abs(out[sl] - np.sqrt(2.0) * _ns_by_svd(t[sl])).max() <= 1e-9, f"tall block {blk}"


def check_ns_layout_equivalence(N, P, rng):
    """The same heads packed sectioned and interleaved (block orders pinned by
    the golden head-block fixtures) give the same per-head results, permuted."""
    n_q, n_kv, D, cols = 8, 2, 8, 24
    heads = {("q", h): rng.standard_normal((D, cols)) for h in range(n_q)}
    heads.update({(r, h): rng.standard_normal((D, cols)) for r in "kv" for h in range(n_kv)})
    res = {}
    for kind in ("sectioned", "interleaved"):
        order = P.head_blocks(P.PackedLayout(kind, n_q, n_kv, D))
        w = np.concatenate([heads[b] for b in order], axis=0)
        assert N.fused_head_blocks(w.shape[0], n_q, n_kv, D) == len(order)
        out = N.per_head_newton_schulz(w, D)
        res[kind] = {b: out[i * D:(i + 1) * D] for i, b in enumerate(order)}
    for b in heads:
        assert np.array_equal(res["sectioned"][b], res["interleaved"][b]), f"head {b}"
    # and the per-head update is not the whole-matrix one
    w = np.concatenate([heads[b] for b in P.head_blocks(P.PackedLayout("sectioned", n_q, n_kv, D))])
    assert np.abs(N.per_head_newton_schulz(w, D) - N.full_matrix_newton_schulz(w)).max() > 1e-2


def read_muon_fixture():
    cands, full, head = [], [], []
    with open(os.path.join(GOLDEN, "muon_fused_candidates.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "candidate":
                name, rows, cols, nq, nkv, d, blocks = rest
                cands.append((name, int(rows), int(cols), int(nq), int(nkv), int(d),
                              None if blocks == "-" else int(blocks)))
            elif key == "full_scale":
                full.append((int(rest[0]), int(rest[1]), float(rest[2])))
            elif key == "head_scale":
                head.append((int(rest[0]), int(rest[1]), float(rest[2])))
    return cands, full, head


def check_ns_page_facts(N):
    """The page's split / no-split cases and the scales the review compares."""
    cands, full, head = read_muon_fixture()
    assert cands and full and head
    for name, rows, cols, nq, nkv, d, blocks in cands:
        assert N.fused_head_blocks(rows, nq, nkv, d) == blocks, name
    for rows, cols, f in full:
        assert abs(N.full_matrix_scale(rows, cols) - f) <= 1e-15, (rows, cols)
    for d, cin, f in head:
        assert abs(N.per_head_scale(d, cin) - f) <= 1e-15, (d, cin)


def check_ns_dispatch(N, rng):
    """The update a fused weight gets: per head when dim 0 is the exact fused
    total, else the whole matrix with max(1, rows / cols) ** 0.5 (sqrt(3) for a
    [3h, h] weight), each against the SVD closed form."""
    h = 16
    w = rng.standard_normal((3 * h, h))
    # 1 q head of 16 over 1 kv head: 3 blocks of 16 rows, the exact total
    got = N.muon_orthogonalize(w, n_q=1, n_kv=1, head_dim=16)
    for blk in range(3):
        sl = slice(16 * blk, 16 * blk + 16)
        assert np.abs(got[sl] - _ns_by_svd(w[sl])).max() <= 1e-9, f"per-head block {blk}"
    # a config whose total (4 + 2 * 2) * 16 = 128 is not 48: the whole matrix
    got = N.muon_orthogonalize(w, n_q=4, n_kv=2, head_dim=16)
    assert np.abs(got - np.sqrt(3.0) * _ns_by_svd(w)).max() <= 1e-9, "whole-matrix path"
    got = N.muon_orthogonalize(w)
    assert np.abs(got - np.sqrt(3.0) * _ns_by_svd(w)).max() <= 1e-9, "no head tag: whole matrix"


# ---------------------------------------------------------- projection ----

def _bf16_bits_of(vals):
    """bf16 bits of values that are exactly bf16 (checked)."""
    out = np.array([_exact_bf16_rne(float(v)) for v in np.ravel(vals)], dtype=np.uint16).reshape(np.shape(vals))
    back = np.array([struct.unpack("<f", struct.pack("<I", int(b) << 16))[0] for b in out.ravel()]).reshape(out.shape)
    assert np.array_equal(back, np.asarray(vals, dtype=np.float64)), "test values must be bf16"
    return out


def _bf16_value(bits):
    return Fraction(struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0])


def _exact_projection_bits(x_bits, w_bits):
    """packed[t, c] = sum_k x[t, k] W[c, k], summed exactly in rationals and
    rounded once to the nearest bf16 (ties to even)."""
    T, K = x_bits.shape
    R = w_bits.shape[0]
    xf = [[_bf16_value(b) for b in row] for row in x_bits]
    wf = [[_bf16_value(b) for b in row] for row in w_bits]
    out = np.empty((T, R), dtype=np.uint16)
    for t in range(T):
        for c in range(R):
            out[t, c] = _exact_bf16_rne(sum((xf[t][k] * wf[c][k] for k in range(K)), Fraction(0)))
    return out


def _random_bf16(rng, shape, spread=6):
    v = rng.standard_normal(shape) * np.exp2(rng.integers(-spread, spread + 1, shape))
    return _bf16_bits_of(np.vectorize(lambda a: float(struct.unpack("<f", struct.pack(
        "<I", _exact_bf16_rne(float(a)) << 16))[0]))(v))


def check_projection(P, rng):
    """The projection step and its hand-over to the prologue."""
    L = P.PackedLayout("interleaved", 2, 1, 8)          # packed row of 32 values
    # 1. a square weight (hidden = row width = 32) with no symmetry: x . W^T,
    #    not x . W, against exact rational sums
    x = _random_bf16(rng, (3, L.row_width))
    w = _random_bf16(rng, (L.row_width, L.row_width))
    assert np.array_equal(P.projection(x, w), _exact_projection_bits(x, w)), "square projection"
    # 2. non-square: 5 tokens, hidden 40, wide value spread
    x = _random_bf16(rng, (5, 40), spread=12)
    w = _random_bf16(rng, (L.row_width, 40), spread=12)
    assert np.array_equal(P.projection(x, w), _exact_projection_bits(x, w)), "projection"
    # 3. one rounding: 1 + 2**-8 + 2**-30 is just above the bf16 tie between 1
    #    and 1 + 2**-7 and rounds up; rounded to float32 first it would land on
    #    the tie and go to the even 1.0. Its mirror 1 + 2**-8 - 2**-30 goes to 1.
    xv = np.zeros((2, 40))
    xv[0, :3] = [1.0, 2.0 ** -8, 2.0 ** -30]
    xv[1, :3] = [1.0, 2.0 ** -8, -(2.0 ** -30)]
    wv = np.zeros((L.row_width, 40))
    wv[5, :3] = 1.0
    got = P.projection(_bf16_bits_of(xv), _bf16_bits_of(wv))
    assert got[0, 5] == 0x3F81 and got[1, 5] == 0x3F80, "one rounding to bf16"
    assert not got[:, [c for c in range(L.row_width) if c != 5]].any()
    # 4. hand-over: W = identity gives the prologue exactly x; W = a row
    #    permutation gives it x's columns in that order
    x = _random_bf16(rng, (4, L.row_width), spread=2)
    pos = np.array([0, 1, 7, 300])
    wq, wk = 0.5 + rng.random(8), 0.5 + rng.random(8)
    ident = _bf16_bits_of(np.eye(L.row_width))
    got, packed = P.gemm_prologue_fwd(L, x, ident, pos, wq, wk, 1e-6, 1e4)
    assert np.array_equal(packed, x)
    want = P.prologue_fwd(L, x, pos, wq, wk, 1e-6, 1e4)
    for key in ("q", "k", "v"):
        assert np.array_equal(got[key], want[key]), key
    perm = rng.permutation(L.row_width)
    _, packed = P.gemm_prologue_fwd(L, x, ident[perm], pos, wq, wk, 1e-6, 1e4, nope=True)
    assert np.array_equal(packed, x[:, perm]), "rows of W are the packed columns, in order"

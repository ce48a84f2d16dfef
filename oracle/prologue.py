"""The packed-QKV prologue written out as its plain definition, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring). Nothing here is blocked,
fused or reordered: each function is one step of the method, applied to whole
arrays, in the order the pages give (split -> per-head RMSNorm -> RoPE, v
copied; backward: RoPE^T -> RMSNorm backward -> packed gradient).

Readings taken where the pages print no formula (each one is listed, with its
reason, in the design notes of this repository):

* RMSNorm over one head:  y = x / sqrt(mean(x**2) + eps) * w, eps inside the
  root, a plain weight multiply (no 1 + w, no bias), mean over head_dim.
* RoPE is rotate-half: for i < D/2, inv_freq_i = base**(-2 i / D),
  theta = pos * inv_freq_i,
      o_i       = y_i cos(theta) - y_{i+D/2} sin(theta)
      o_{i+D/2} = y_{i+D/2} cos(theta) + y_i sin(theta).
  No frequency scaling of its own. NoPE layers skip it.
* The GQAttention variant (the follow-up the pages name for Llama 3, Qwen3
  and GPT-OSS: "split -> norm -> RoPE" in GQAttention, GPT-OSS with a qkv
  bias): the norm can be off (split -> RoPE); a bias in the packed row's
  order is added first (before the norm); a caller-given inv_freq table and a
  cos/sin factor stand for those models' frequency scalings. Training saves
  the input heads before the bias; the backward adds it back.
* Norm first, then RoPE ("split -> norm -> RoPE" in the after-diagram of
  "[muse_spark][perf] Split the packed qkv inside the q/k region", Solution).
* One rounding to bf16 at the very end; nothing is rounded between the norm
  and the rotation.
"""

from dataclasses import dataclass

import numpy as np

from .bf16 import bf16_bits_to_f64, to_bf16_rne


# --------------------------------------------------------------------------
# S1: the packing and the split (an index map, no arithmetic)
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class PackedLayout:
    """How the heads of one token sit along a packed row.

    kind "interleaved": per KV group g, G = n_q / n_kv query heads, then one
    key head, then one value head ("[muse_spark][perf] ...", Problem 1:
    [T, 16 kv heads, 10, 64], per kv head 8 q heads + 1 k + 1 v; "[muon]
    Per-head Newton-Schulz ...", What this PR does, second bullet).

    kind "sectioned": all n_q query heads, then n_kv key heads, then n_kv value
    heads, i.e. cat([q_proj, k_proj, v_proj]) ("[muon] ...", What this PR
    does, first bullet).
    """

    kind: str
    n_q: int
    n_kv: int
    head_dim: int

    def __post_init__(self):
        if self.kind not in ("interleaved", "sectioned"):
            raise ValueError(f"unknown packing {self.kind!r}")
        if self.n_kv <= 0 or self.n_q <= 0 or self.n_q % self.n_kv:
            raise ValueError("n_q must be a positive multiple of n_kv")
        if self.head_dim <= 0 or self.head_dim % 2:
            raise ValueError("head_dim must be positive and even")

    @property
    def group(self):
        return self.n_q // self.n_kv

    @property
    def n_blocks(self):
        """Head blocks per row: the exact fused total (n_q + 2 n_kv)."""
        return self.n_q + 2 * self.n_kv

    @property
    def row_width(self):
        return self.n_blocks * self.head_dim


def head_blocks(layout):
    """List of (role, head) for each head_dim-wide block of a packed row."""
    G = layout.group
    blocks = []
    if layout.kind == "interleaved":
        for g in range(layout.n_kv):
            for j in range(G):
                blocks.append(("q", g * G + j))
            blocks.append(("k", g))
            blocks.append(("v", g))
    else:
        blocks += [("q", h) for h in range(layout.n_q)]
        blocks += [("k", h) for h in range(layout.n_kv)]
        blocks += [("v", h) for h in range(layout.n_kv)]
    return blocks


def _block_positions(layout):
    """For each role, the packed block position of head 0, 1, 2, ..."""
    pos = {"q": [None] * layout.n_q, "k": [None] * layout.n_kv, "v": [None] * layout.n_kv}
    for p, (role, h) in enumerate(head_blocks(layout)):
        pos[role][h] = p
    return {role: np.array(v, dtype=np.int64) for role, v in pos.items()}


def split_heads(layout, packed):
    """Split packed rows [T, row_width] (any dtype) into q [T,n_q,D], k, v [T,n_kv,D]."""
    packed = np.asarray(packed)
    T = packed.shape[0]
    rows = packed.reshape(T, layout.n_blocks, layout.head_dim)
    p = _block_positions(layout)
    return rows[:, p["q"], :], rows[:, p["k"], :], rows[:, p["v"], :]


def merge_heads(layout, q, k, v):
    """Inverse of split_heads: place per-head arrays back into packed rows."""
    q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)
    T = q.shape[0]
    out = np.empty((T, layout.n_blocks, layout.head_dim), dtype=q.dtype)
    p = _block_positions(layout)
    out[:, p["q"], :] = q
    out[:, p["k"], :] = k
    out[:, p["v"], :] = v
    return out.reshape(T, layout.row_width)


# --------------------------------------------------------------------------
# S2: per-head RMSNorm
# --------------------------------------------------------------------------

def rms_norm(x, w, eps):
    """y = x / sqrt(mean(x**2) + eps) * w over the last axis (one head)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rms_norm_backward(x, w, g, eps):
    """Gradient of rms_norm given the upstream gradient g of its output.

    With r = (mean(x**2) + eps)**-0.5 and D the head size:
        dx_j = r w_j g_j - x_j (r**3 / D) sum_d x_d w_d g_d
        dw_d = g_d x_d r          (per element; the caller sums it)
    """
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    D = x.shape[-1]
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    dot = np.sum(x * w * g, axis=-1, keepdims=True)
    dx = r * w * g - x * (r ** 3 / D) * dot
    dw_terms = g * x * r
    return dx, dw_terms


# --------------------------------------------------------------------------
# S3: rotate-half RoPE
# --------------------------------------------------------------------------

def rope_inv_freq(head_dim, base):
    """inv_freq_i = base**(-2 i / D) for i < D/2."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / head_dim)


def rope_angles(pos, head_dim, base, inv_freq=None):
    """theta[t, i] = pos[t] * inv_freq_i, float64. A caller-given inv_freq
    (D/2 values) replaces base**(-2 i / D): the frequency scalings of the
    GQAttention users (Llama 3's, YaRN's) only change this table."""
    pos = np.asarray(pos, dtype=np.float64).reshape(-1, 1)
    f = rope_inv_freq(head_dim, base) if inv_freq is None else np.asarray(inv_freq, dtype=np.float64)
    assert f.shape == (head_dim // 2,)
    return pos * f[None, :]


def rope_rotate_half(y, pos, base, inv_freq=None, scale=1.0):
    """Rotate each head of y [T, h, D] by the angles of its token's position.
    cos and sin are both multiplied by `scale` (YaRN's attention factor; 1 for
    plain RoPE)."""
    y = np.asarray(y, dtype=np.float64)
    D = y.shape[-1]
    half = D // 2
    th = rope_angles(pos, D, base, inv_freq)[:, None, :]
    c, s = np.cos(th) * scale, np.sin(th) * scale
    a, b = y[..., :half], y[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_rotate_half_transpose(d, pos, base, inv_freq=None, scale=1.0):
    """Apply (scale R(theta))^T = scale R(-theta): the backward of rope_rotate_half."""
    d = np.asarray(d, dtype=np.float64)
    D = d.shape[-1]
    half = D // 2
    th = rope_angles(pos, D, base, inv_freq)[:, None, :]
    c, s = np.cos(th) * scale, np.sin(th) * scale
    a, b = d[..., :half], d[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


# --------------------------------------------------------------------------
# The GQAttention variant (Llama 3, Qwen3, GPT-OSS): a qkv bias and no norm
# --------------------------------------------------------------------------

def add_bias(packed, bias):
    """packed [T, row_width] + bias [row_width]: the fused linear's bias, given
    in the packed row's own order, added to every token before the split."""
    x = np.asarray(packed, dtype=np.float64)
    if bias is None:
        return x
    b = np.asarray(bias, dtype=np.float64)
    assert b.shape == (x.shape[-1],)
    return x + b[None, :]


# --------------------------------------------------------------------------
# S1-S4: the forward
# --------------------------------------------------------------------------

def prologue_fwd_f64(layout, packed, pos, w_q, w_k, eps, rope_base, nope=False,
                     norm=True, bias=None, inv_freq=None, rope_scale=1.0):
    """Forward on float64 packed rows [T, row_width]: returns exact q, k, v.

    The variant options: `bias` is added to the whole row first; `norm=False`
    skips the RMSNorm (split -> RoPE only); `inv_freq` / `rope_scale` as in
    rope_rotate_half."""
    x = add_bias(packed, bias)
    xq, xk, xv = split_heads(layout, x)
    q = rms_norm(xq, w_q, eps) if norm else xq
    k = rms_norm(xk, w_k, eps) if norm else xk
    if not nope:
        q = rope_rotate_half(q, pos, rope_base, inv_freq, rope_scale)
        k = rope_rotate_half(k, pos, rope_base, inv_freq, rope_scale)
    return q, k, xv


def prologue_fwd(layout, packed_bits, pos, w_q, w_k, eps, rope_base, nope=False,
                 norm=True, bias=None, inv_freq=None, rope_scale=1.0):
    """Forward on bf16 packed rows (uint16 bits [T, row_width]).

    Returns a dict:
      q, k, v  exact float64 outputs [T, n_q, D], [T, n_kv, D] (round with
               to_bf16_rne to get the bf16 bits a kernel should store);
      v_bits   the v heads' output bits: the input bits when there is no bias
               (v is a pure copy), else v rounded once;
      q_pre_bits, k_pre_bits   the split input heads' bits, before any bias
               (what training saves for the backward).
    """
    bits = np.asarray(packed_bits, dtype=np.uint16).reshape(-1, layout.row_width)
    q, k, v = prologue_fwd_f64(layout, bf16_bits_to_f64(bits), pos, w_q, w_k, eps, rope_base, nope,
                               norm, bias, inv_freq, rope_scale)
    qb, kb, vb = split_heads(layout, bits)
    return {"q": q, "k": k, "v": v, "v_bits": vb if bias is None else to_bf16_rne(v),
            "q_pre_bits": qb, "k_pre_bits": kb}


# --------------------------------------------------------------------------
# S5 / S6: paged pool writes
# --------------------------------------------------------------------------

def pool_scatter(pool_bits, rows_bits, page, offset):
    """Staged scatter: copy of pool_bits with row t placed at [page[t], offset[t]].

    pool_bits has shape [num_pages, page_size, ...]; rows_bits [T, ...].
    Every other entry of the pool keeps its bits.
    """
    out = np.array(pool_bits, dtype=np.uint16, copy=True)
    rows = np.asarray(rows_bits, dtype=np.uint16)
    for t in range(rows.shape[0]):
        out[int(page[t]), int(offset[t])] = rows[t]
    return out


def pool_write(layout, packed_bits, pos, w_q, w_k, eps, rope_base, nope,
               page, offset, k_pool_bits, v_pool_bits, **variant):
    """GQA decode write: q contiguous, normed(+roped) k and raw v into the pools.

    Defined as the contiguous forward followed by the staged scatter.
    `variant` takes prologue_fwd's norm / bias / inv_freq / rope_scale.
    Returns (q exact float64, k exact float64, new k pool bits, new v pool bits).
    """
    out = prologue_fwd(layout, packed_bits, pos, w_q, w_k, eps, rope_base, nope, **variant)
    k_pool = pool_scatter(k_pool_bits, to_bf16_rne(out["k"]), page, offset)
    v_pool = pool_scatter(v_pool_bits, out["v_bits"], page, offset)
    return out["q"], out["k"], k_pool, v_pool


def mla_rows_f64(rows, pos, w, eps, rope_base, norm_dim, rope_dim):
    """MLA kv latent row: RMSNorm over [0, norm_dim) with weight w, then
    rotate-half RoPE over [norm_dim, norm_dim + rope_dim) with no norm and no
    weight; the two parts are concatenated back into one row."""
    x = np.asarray(rows, dtype=np.float64).reshape(-1, norm_dim + rope_dim)
    latent = rms_norm(x[:, :norm_dim], w, eps)
    rope = rope_rotate_half(x[:, None, norm_dim:], pos, rope_base)[:, 0, :]
    return np.concatenate([latent, rope], axis=-1)


def mla_rows(rows_bits, pos, w, eps, rope_base, norm_dim=512, rope_dim=64):
    """mla_rows_f64 on bf16 bit rows; returns the exact float64 rows."""
    x = bf16_bits_to_f64(np.asarray(rows_bits, dtype=np.uint16))
    return mla_rows_f64(x, pos, w, eps, rope_base, norm_dim, rope_dim)


def mla_pool_write(rows_bits, pos, w, eps, rope_base, page, offset, pool_bits,
                   norm_dim=512, rope_dim=64):
    """Norm + RoPE of the latent rows, rounded once to bf16, then the staged
    scatter into pool [num_pages, page_size, norm_dim + rope_dim]."""
    exact = mla_rows(rows_bits, pos, w, eps, rope_base, norm_dim, rope_dim)
    return exact, pool_scatter(pool_bits, to_bf16_rne(exact), page, offset)


# --------------------------------------------------------------------------
# S7 / S8: the backward
# --------------------------------------------------------------------------

def prologue_bwd_f64(layout, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, nope=False,
                     norm=True, bias=None, inv_freq=None, rope_scale=1.0):
    """Backward on float64 arrays.

    dq [T,n_q,D], dk/dv [T,n_kv,D] are the gradients of the forward's outputs;
    q_pre/k_pre are the split input heads (before any bias). Returns
      dpacked [T, row_width]  gradient w.r.t. the packed input, in the input
                              layout (v slots hold dv unchanged);
      dw_q, dw_k [D]          gradients of the two RMSNorm weights, summed over
                              every token and head (zero without the norm);
      db [row_width] or None  gradient of the bias: dpacked summed over tokens.
    """
    dq = np.asarray(dq, dtype=np.float64)
    dk = np.asarray(dk, dtype=np.float64)
    if nope:
        gq, gk = dq, dk
    else:
        gq = rope_rotate_half_transpose(dq, pos, rope_base, inv_freq, rope_scale)
        gk = rope_rotate_half_transpose(dk, pos, rope_base, inv_freq, rope_scale)
    if norm:
        # the norm saw the biased input: put the bias back on the saved heads
        bq, bk, _ = split_heads(layout, add_bias(np.zeros((1, layout.row_width)), bias))
        dxq, tq = rms_norm_backward(np.asarray(q_pre, dtype=np.float64) + bq, w_q, gq, eps)
        dxk, tk = rms_norm_backward(np.asarray(k_pre, dtype=np.float64) + bk, w_k, gk, eps)
        dw_q, dw_k = tq.sum(axis=(0, 1)), tk.sum(axis=(0, 1))
    else:
        dxq, dxk = gq, gk
        dw_q = dw_k = np.zeros(layout.head_dim)
    dpacked = merge_heads(layout, dxq, dxk, np.asarray(dv, dtype=np.float64))
    db = None if bias is None else dpacked.sum(axis=0)
    return {"dpacked": dpacked, "dw_q": dw_q, "dw_k": dw_k, "db": db}


def prologue_bwd(layout, dq_bits, dk_bits, dv_bits, q_pre_bits, k_pre_bits,
                 pos, w_q, w_k, eps, rope_base, nope=False, **variant):
    """prologue_bwd_f64 on bf16 bit inputs; results stay exact float64."""
    f = bf16_bits_to_f64
    return prologue_bwd_f64(layout, f(dq_bits), f(dk_bits), f(dv_bits), f(q_pre_bits),
                            f(k_pre_bits), pos, w_q, w_k, eps, rope_base, nope, **variant)


# --------------------------------------------------------------------------
# The projection to the left of the path, with the prologue after it
# --------------------------------------------------------------------------

def projection_f64(x_bits, w_bits):
    """The wqkv projection x . W^T for x [T, hidden] and W [row_width, hidden]
    (nn.Linear's weight layout, rows in the layout's packed order), both bf16
    bits, in float64: every product of two bf16 values is exact in float64."""
    x = bf16_bits_to_f64(np.asarray(x_bits, dtype=np.uint16))
    w = bf16_bits_to_f64(np.asarray(w_bits, dtype=np.uint16))
    return x @ w.T


def projection(x_bits, w_bits):
    """projection_f64 rounded once to bf16: the packed tensor the projection
    hands to the prologue ("[muse_spark][perf] ...", Problem 1)."""
    return to_bf16_rne(projection_f64(x_bits, w_bits))


def gemm_prologue_fwd(layout, x_bits, w_bits, pos, w_q, w_k, eps, rope_base, nope=False, **variant):
    """projection, then prologue_fwd on its packed bits. Returns (prologue_fwd's
    dict, packed bits)."""
    packed = projection(x_bits, w_bits)
    return prologue_fwd(layout, packed, pos, w_q, w_k, eps, rope_base, nope, **variant), packed

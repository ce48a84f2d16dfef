"""Tensor-level helpers over the C ABI: they allocate outputs with torch (device
memory is PyTorch's job here) and call the library. No arithmetic happens in
Python.

The training entry point, ``QKVPrologue.apply``, mirrors the region of
"[muse_spark][perf] Split the packed qkv inside the q/k region" (Solution):
packed qkv in, contiguous q, k, v out; its backward writes the gradient of the
packed tensor in one pass.
"""

import torch

from . import _lib as C


def _layout_of(packed, n_q, n_kv, head_dim, kind):
    T = packed.shape[0]
    row = packed.reshape(T, -1) if packed.is_contiguous() else None
    if row is None:
        raise ValueError("packed must be contiguous ([T, ...] rows)")
    width = row.shape[1]
    if width != (n_q + 2 * n_kv) * head_dim:
        raise ValueError(f"packed row has {width} values, expected (n_q + 2 n_kv) * head_dim = "
                         f"{(n_q + 2 * n_kv) * head_dim}")
    return C.layout(kind, n_q, n_kv, head_dim), T


def _check_dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must live on a CUDA device")


def _variant(bias=None, inv_freq=None, rope_scale=1.0):
    """The qkvp_variant of the GQAttention options, or None for the plain call."""
    if bias is None and inv_freq is None and rope_scale in (None, 0.0, 1.0):
        return None
    if bias is not None:
        _check_dev(bias)
        if bias.dtype != torch.float32 or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous float32 tensor")
    return C.variant(inv_freq=None if inv_freq is None else [float(f) for f in inv_freq],
                     rope_scale=0.0 if rope_scale is None else float(rope_scale), bias=bias)


def _flags(nope=False, save_pre=False, norm=True):
    return (C.QKVP_NOPE if nope else 0) | (C.QKVP_SAVE_PRE if save_pre else 0) | (0 if norm else C.QKVP_NORM_OFF)


def prologue_forward(packed, pos, w_q, w_k, n_q, n_kv, head_dim=64, kind="interleaved", eps=1e-6,
                     rope_base=500000.0, nope=False, save_pre=False, stream=None, norm=True, bias=None,
                     inv_freq=None, rope_scale=1.0):
    """Split + per-head RMSNorm + RoPE. Returns (q, k, v) or (q, k, v, q_pre, k_pre).

    The GQAttention variant options: norm=False (split -> RoPE only; w_q, w_k
    may be None), bias (float32 [(n_q + 2 n_kv) * head_dim] in the packed
    row's order, added first), inv_freq (head_dim / 2 frequencies replacing
    rope_base**(-2i/D)) and rope_scale (factor on cos and sin)."""
    _check_dev(packed, pos, w_q, w_k)
    L, T = _layout_of(packed, n_q, n_kv, head_dim, kind)
    dev = packed.device
    q = torch.empty(T, n_q, head_dim, dtype=torch.bfloat16, device=dev)
    k = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    v = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    q_pre = torch.empty_like(q) if save_pre else None
    k_pre = torch.empty_like(k) if save_pre else None
    C.qkv_prologue_fwd_ex(L, _variant(bias, inv_freq, rope_scale), T, packed, pos, w_q, w_k, eps, rope_base,
                          _flags(nope, save_pre, norm), q, k, v, q_pre, k_pre, stream)
    return (q, k, v, q_pre, k_pre) if save_pre else (q, k, v)


def prologue_backward(dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, n_q, n_kv, head_dim=64,
                      kind="interleaved", eps=1e-6, rope_base=500000.0, nope=False, stream=None,
                      workspace=None, norm=True, bias=None, inv_freq=None, rope_scale=1.0):
    """Packed gradient [T, (n_q + 2 n_kv) * head_dim] and fp32 (dw_q, dw_k), plus
    the fp32 bias gradient when a bias is given: (dpacked, dw_q, dw_k[, dbias]).
    Without the norm dw_q, dw_k are None and q_pre, k_pre, w_q, w_k may be None."""
    _check_dev(dq, dk, dv, q_pre, k_pre, w_q, w_k)
    T = dq.shape[0]
    L = C.layout(kind, n_q, n_kv, head_dim)
    dev = dq.device
    V = _variant(bias, inv_freq, rope_scale)
    dpacked = torch.empty(T, (n_q + 2 * n_kv) * head_dim, dtype=torch.bfloat16, device=dev)
    dw_q = torch.empty(head_dim, dtype=torch.float32, device=dev) if norm else None
    dw_k = torch.empty(head_dim, dtype=torch.float32, device=dev) if norm else None
    dbias = torch.empty((n_q + 2 * n_kv) * head_dim, dtype=torch.float32, device=dev) if bias is not None else None
    need = C.qkv_prologue_bwd_workspace_size_ex(L, V, T)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    C.qkv_prologue_bwd_ex(L, V, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base,
                          _flags(nope, False, norm), dpacked, dw_q, dw_k, dbias, workspace, need, stream)
    return (dpacked, dw_q, dw_k, dbias) if bias is not None else (dpacked, dw_q, dw_k)


def prologue_pool_write(packed, pos, w_q, w_k, page, offset, k_pool, v_pool, n_q, n_kv, head_dim=64,
                        kind="interleaved", eps=1e-6, rope_base=500000.0, nope=False, dev_status=None,
                        stream=None, norm=True, bias=None, inv_freq=None, rope_scale=1.0):
    """q contiguous; normed(+roped) k and raw v into the paged pools. Returns q."""
    _check_dev(packed, pos, w_q, w_k, page, offset, k_pool, v_pool)
    L, T = _layout_of(packed, n_q, n_kv, head_dim, kind)
    q = torch.empty(T, n_q, head_dim, dtype=torch.bfloat16, device=packed.device)
    C.qkv_prologue_pool_write_ex(L, _variant(bias, inv_freq, rope_scale), T, packed, pos, w_q, w_k, eps,
                                 rope_base, _flags(nope, False, norm), q, page, offset, k_pool, v_pool,
                                 k_pool.shape[0], k_pool.shape[1], dev_status, stream)
    return q


def latent_rows(rows, pos, w, eps=1e-6, rope_base=10000.0, norm_dim=512, rope_dim=64, nope=False,
                stream=None, inv_freq=None, rope_scale=1.0):
    """MLA kv latent rows normed/roped into a new contiguous [T, norm_dim + rope_dim] tensor."""
    _check_dev(rows, pos, w)
    T = rows.shape[0]
    L = C.layout("latent", norm_dim=norm_dim, rope_dim=rope_dim)
    out = torch.empty(T, norm_dim + rope_dim, dtype=torch.bfloat16, device=rows.device)
    C.qkv_prologue_fwd_ex(L, _variant(None, inv_freq, rope_scale), T, rows, pos, None, w, eps, rope_base,
                          _flags(nope), None, out, None, None, None, stream)
    return out


def latent_pool_write(rows, pos, w, page, offset, pool, eps=1e-6, rope_base=10000.0, norm_dim=512,
                      rope_dim=64, nope=False, dev_status=None, stream=None, inv_freq=None, rope_scale=1.0):
    """MLA kv latent rows normed/roped straight into pool [num_pages, page_size, 576]."""
    _check_dev(rows, pos, w, page, offset, pool)
    T = rows.shape[0]
    L = C.layout("latent", norm_dim=norm_dim, rope_dim=rope_dim)
    C.qkv_prologue_pool_write_ex(L, _variant(None, inv_freq, rope_scale), T, rows, pos, None, w, eps, rope_base,
                                 _flags(nope), None, page, offset, pool, None, pool.shape[0], pool.shape[1],
                                 dev_status, stream)


def gemm_prologue_forward(x, w_qkv, pos, w_q, w_k, n_q, n_kv, head_dim=64, kind="interleaved", eps=1e-6,
                          rope_base=500000.0, nope=False, save_pre=False, stream=None):
    """The wqkv projection with the prologue in its epilogue: x [T, hidden] bf16,
    w_qkv [(n_q + 2 n_kv) * head_dim, hidden] bf16 (rows in the layout's packed
    order) -> (q, k, v) or (q, k, v, q_pre, k_pre); the packed tensor is never
    materialised."""
    _check_dev(x, w_qkv, pos, w_q, w_k)
    if x.dim() != 2 or w_qkv.dim() != 2 or x.shape[1] != w_qkv.shape[1]:
        raise ValueError("x must be [T, hidden] and w_qkv [rows, hidden]")
    if w_qkv.shape[0] != (n_q + 2 * n_kv) * head_dim:
        raise ValueError("w_qkv must have (n_q + 2 n_kv) * head_dim rows")
    T, hidden = x.shape
    L = C.layout(kind, n_q, n_kv, head_dim)
    dev = x.device
    q = torch.empty(T, n_q, head_dim, dtype=torch.bfloat16, device=dev)
    k = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    v = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    q_pre = torch.empty_like(q) if save_pre else None
    k_pre = torch.empty_like(k) if save_pre else None
    C.qkv_prologue_gemm_fwd(L, T, hidden, x.contiguous(), w_qkv.contiguous(), pos, w_q, w_k, eps, rope_base,
                            _flags(nope, save_pre), q, k, v, q_pre, k_pre, stream)
    return (q, k, v, q_pre, k_pre) if save_pre else (q, k, v)


def per_head_newton_schulz(m, n_q, n_kv, head_dim=64, kind="interleaved", split=0, out=None, workspace=None,
                           stream=None):
    """Per-head Newton-Schulz of a fused QKV weight's update m
    [(n_q + 2 n_kv) * head_dim, in_features] bf16: every head_dim-row block
    orthogonalised on its own (Muon's quintic iteration, five steps) and scaled
    by max(1, head_dim / in_features) ** 0.5 ("[muon] Per-head Newton-Schulz for
    fused QKV projections", What this PR does). `kind` names the packing of the
    rows; the result does not depend on it. A 3-D m [count, rows, cols] (one
    update per layer) is done in one set of launches. `workspace` (a device
    tensor of at least newton_schulz_workspace_bytes bytes) is allocated here
    when not given; `split` fixes the Gram pass's CTAs per 128-row unit."""
    _check_dev(m)
    if m.dim() not in (2, 3) or m.dtype != torch.bfloat16:
        raise ValueError("m must be a bf16 [rows, cols] or [count, rows, cols] tensor")
    if m.shape[-2] != (n_q + 2 * n_kv) * head_dim:
        raise ValueError("m must have (n_q + 2 n_kv) * head_dim rows")
    m = m.contiguous()
    if out is None:
        out = torch.empty_like(m)
    L = C.layout(kind, n_q, n_kv, head_dim)
    count = 1 if m.dim() == 2 else m.shape[0]
    need = C.qkv_newton_schulz_workspace(L, m.shape[-1], split, count)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=m.device)
    nbytes = workspace.numel() * workspace.element_size()
    if m.dim() == 2:
        C.qkv_newton_schulz(L, m.shape[1], m, out, split, workspace, nbytes, stream)
    else:  # every weight of the stack in one set of launches
        C.qkv_newton_schulz_batch(L, count, m.shape[2], m, out, split, workspace, nbytes, stream)
    return out


def newton_schulz_workspace_bytes(m_shape, n_q, n_kv, head_dim=64, kind="interleaved", split=0):
    """Workspace bytes per_head_newton_schulz needs for an update of this shape."""
    count = 1 if len(m_shape) == 2 else m_shape[0]
    return C.qkv_newton_schulz_workspace(C.layout(kind, n_q, n_kv, head_dim), m_shape[-1], split, count)


def on_side_stream(side, fn, *args, **kwargs):
    """Run fn(*args, **kwargs) on CUDA stream `side`, forked from the current
    stream: `side` first waits for everything already queued on the current
    stream, and the returned event is recorded on `side` after fn's work. The
    caller joins with ``torch.cuda.current_stream().wait_event(event)`` before
    anything that reads fn's results.

    This is the drafter-layer pattern of "MLA DSpark: run each drafter layer's
    kv path beside its q path" (Description): the kv path (kv projection ->
    latent norm/RoPE -> direct pool write) forks to an aux stream after the input
    layernorm, the q path runs on the main stream, and attention joins. Works
    under CUDA graph capture (the fork and join become graph edges). Tensors made
    on the current stream and used on `side` must stay alive until the join.
    """
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    with torch.cuda.stream(side):
        out = fn(*args, **kwargs)
        done = torch.cuda.Event()
        done.record(side)
    return out, done


def join(event, stream=None):
    """Make `stream` (default: the current stream) wait for `event`, the join of
    a fork made with on_side_stream or mla_kv_path_beside. Under CUDA graph
    capture this becomes a graph edge."""
    (stream or torch.cuda.current_stream()).wait_event(event)


def mla_kv_path_beside(side, pos, w, page, offset, pool, kv_rows=None, kv_proj=None, eps=1e-6,
                       rope_base=10000.0, norm_dim=512, rope_dim=64, nope=False, dev_status=None,
                       inv_freq=None, rope_scale=1.0):
    """The kv path of one MLA drafter layer on the side stream `side`, beside
    the q path on the current stream ("MLA DSpark: run each drafter layer's kv
    path beside its q path", Description): fork after the layer's input norm,
    run the kv path there, join before attention reads the pool.

    The kv path is: the kv_a rows [T, norm_dim + rope_dim] bf16 (either
    `kv_rows`, already computed, or `kv_proj()`, a callable run on `side` that
    returns them, e.g. the kv_a projection of the layer input), then the
    library's latent norm / RoPE written straight into `pool` [num_pages,
    page_size, norm_dim + rope_dim] at (page, offset) (latent_pool_write).

    Returns (kv_rows, join_event). Everything the caller queued on the current
    stream before the call is visible to the kv path; nothing on the current
    stream waits for it until the caller joins (join(join_event)) -- do that
    before anything reads `pool` or the returned rows. Inputs made on the
    current stream must stay alive until the join. Works under CUDA graph
    capture: the fork and the join become graph edges."""
    if (kv_rows is None) == (kv_proj is None):
        raise ValueError("give exactly one of kv_rows and kv_proj")

    def kv_path():
        rows = kv_proj() if kv_proj is not None else kv_rows
        latent_pool_write(rows, pos, w, page, offset, pool, eps, rope_base, norm_dim, rope_dim, nope,
                          dev_status, None, inv_freq, rope_scale)
        return rows

    return on_side_stream(side, kv_path)


class QKVPrologue(torch.autograd.Function):
    """packed [T, row] -> (q, k, v); backward writes d(packed) in one pass.

    The norm weights w_q, w_k are float32 [head_dim] tensors and receive
    gradients; positions do not.
    """

    @staticmethod
    def forward(ctx, packed, pos, w_q, w_k, n_q, n_kv, head_dim, kind, eps, rope_base, nope):
        q, k, v, q_pre, k_pre = prologue_forward(packed, pos, w_q, w_k, n_q, n_kv, head_dim, kind, eps,
                                                 rope_base, nope, save_pre=True)
        ctx.save_for_backward(q_pre, k_pre, pos, w_q, w_k)
        ctx.cfg = (n_q, n_kv, head_dim, kind, eps, rope_base, nope, packed.shape)
        return q, k, v

    @staticmethod
    def backward(ctx, dq, dk, dv):
        q_pre, k_pre, pos, w_q, w_k = ctx.saved_tensors
        n_q, n_kv, head_dim, kind, eps, rope_base, nope, shape = ctx.cfg
        dq, dk, dv = (g.contiguous() for g in (dq, dk, dv))
        dpacked, dw_q, dw_k = prologue_backward(dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, n_q, n_kv,
                                                head_dim, kind, eps, rope_base, nope)
        return dpacked.view(shape), None, dw_q, dw_k, None, None, None, None, None, None, None


class GQAttentionPrologue(torch.autograd.Function):
    """The GQAttention variant region (Llama 3, Qwen3, GPT-OSS): packed [T, row]
    -> (q, k, v) with the norm optional, an optional qkv bias and a caller's
    RoPE frequency table / cos-sin factor; the backward writes d(packed) in one
    pass and returns the norm-weight and bias gradients where they exist.

    apply(packed, pos, w_q, w_k, bias, n_q, n_kv, head_dim, kind, eps, rope_base,
          nope, norm, inv_freq, rope_scale); w_q / w_k / bias may be None.
    """

    @staticmethod
    def forward(ctx, packed, pos, w_q, w_k, bias, n_q, n_kv, head_dim, kind, eps, rope_base, nope, norm,
                inv_freq, rope_scale):
        out = prologue_forward(packed, pos, w_q, w_k, n_q, n_kv, head_dim, kind, eps, rope_base, nope,
                               save_pre=norm, norm=norm, bias=bias, inv_freq=inv_freq, rope_scale=rope_scale)
        q, k, v = out[:3]
        q_pre, k_pre = (out[3], out[4]) if norm else (None, None)
        ctx.save_for_backward(q_pre, k_pre, pos, w_q, w_k, bias)
        ctx.cfg = (n_q, n_kv, head_dim, kind, eps, rope_base, nope, norm, inv_freq, rope_scale, packed.shape)
        return q, k, v

    @staticmethod
    def backward(ctx, dq, dk, dv):
        q_pre, k_pre, pos, w_q, w_k, bias = ctx.saved_tensors
        n_q, n_kv, head_dim, kind, eps, rope_base, nope, norm, inv_freq, rope_scale, shape = ctx.cfg
        dq, dk, dv = (g.contiguous() for g in (dq, dk, dv))
        out = prologue_backward(dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, n_q, n_kv, head_dim, kind, eps, rope_base,
                                nope, norm=norm, bias=bias, inv_freq=inv_freq, rope_scale=rope_scale)
        dbias = out[3] if bias is not None else None
        return (out[0].view(shape), None, out[1], out[2], dbias) + (None,) * 10

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


def prologue_forward(packed, pos, w_q, w_k, n_q, n_kv, head_dim=64, kind="interleaved", eps=1e-6,
                     rope_base=500000.0, nope=False, save_pre=False, stream=None):
    """Split + per-head RMSNorm + RoPE. Returns (q, k, v) or (q, k, v, q_pre, k_pre)."""
    _check_dev(packed, pos, w_q, w_k)
    L, T = _layout_of(packed, n_q, n_kv, head_dim, kind)
    dev = packed.device
    q = torch.empty(T, n_q, head_dim, dtype=torch.bfloat16, device=dev)
    k = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    v = torch.empty(T, n_kv, head_dim, dtype=torch.bfloat16, device=dev)
    q_pre = torch.empty_like(q) if save_pre else None
    k_pre = torch.empty_like(k) if save_pre else None
    flags = (C.QKVP_NOPE if nope else 0) | (C.QKVP_SAVE_PRE if save_pre else 0)
    C.qkv_prologue_fwd(L, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, k, v, q_pre, k_pre, stream)
    return (q, k, v, q_pre, k_pre) if save_pre else (q, k, v)


def prologue_backward(dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, n_q, n_kv, head_dim=64,
                      kind="interleaved", eps=1e-6, rope_base=500000.0, nope=False, stream=None,
                      workspace=None):
    """Packed gradient [T, (n_q + 2 n_kv) * head_dim] and fp32 (dw_q, dw_k)."""
    _check_dev(dq, dk, dv, q_pre, k_pre, w_q, w_k)
    T = dq.shape[0]
    L = C.layout(kind, n_q, n_kv, head_dim)
    dev = dq.device
    dpacked = torch.empty(T, (n_q + 2 * n_kv) * head_dim, dtype=torch.bfloat16, device=dev)
    dw_q = torch.empty(head_dim, dtype=torch.float32, device=dev)
    dw_k = torch.empty(head_dim, dtype=torch.float32, device=dev)
    need = C.qkv_prologue_bwd_workspace_size(L, T)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    C.qkv_prologue_bwd(L, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base,
                       C.QKVP_NOPE if nope else 0, dpacked, dw_q, dw_k, workspace, need, stream)
    return dpacked, dw_q, dw_k


def prologue_pool_write(packed, pos, w_q, w_k, page, offset, k_pool, v_pool, n_q, n_kv, head_dim=64,
                        kind="interleaved", eps=1e-6, rope_base=500000.0, nope=False, dev_status=None,
                        stream=None):
    """q contiguous; normed(+roped) k and raw v into the paged pools. Returns q."""
    _check_dev(packed, pos, w_q, w_k, page, offset, k_pool, v_pool)
    L, T = _layout_of(packed, n_q, n_kv, head_dim, kind)
    q = torch.empty(T, n_q, head_dim, dtype=torch.bfloat16, device=packed.device)
    C.qkv_prologue_pool_write(L, T, packed, pos, w_q, w_k, eps, rope_base, C.QKVP_NOPE if nope else 0, q,
                              page, offset, k_pool, v_pool, k_pool.shape[0], k_pool.shape[1],
                              dev_status, stream)
    return q


def latent_rows(rows, pos, w, eps=1e-6, rope_base=10000.0, norm_dim=512, rope_dim=64, nope=False,
                stream=None):
    """MLA kv latent rows normed/roped into a new contiguous [T, norm_dim + rope_dim] tensor."""
    _check_dev(rows, pos, w)
    T = rows.shape[0]
    L = C.layout("latent", norm_dim=norm_dim, rope_dim=rope_dim)
    out = torch.empty(T, norm_dim + rope_dim, dtype=torch.bfloat16, device=rows.device)
    C.qkv_prologue_fwd(L, T, rows, pos, None, w, eps, rope_base, C.QKVP_NOPE if nope else 0, None, out,
                       None, None, None, stream)
    return out


def latent_pool_write(rows, pos, w, page, offset, pool, eps=1e-6, rope_base=10000.0, norm_dim=512,
                      rope_dim=64, nope=False, dev_status=None, stream=None):
    """MLA kv latent rows normed/roped straight into pool [num_pages, page_size, 576]."""
    _check_dev(rows, pos, w, page, offset, pool)
    T = rows.shape[0]
    L = C.layout("latent", norm_dim=norm_dim, rope_dim=rope_dim)
    C.qkv_prologue_pool_write(L, T, rows, pos, None, w, eps, rope_base, C.QKVP_NOPE if nope else 0, None,
                              page, offset, pool, None, pool.shape[0], pool.shape[1], dev_status, stream)


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

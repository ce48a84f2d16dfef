"""The two kernel families agree: the shared-memory pipelined kernels (used
wherever a layout fits them) and the general register kernels (forced with
QKVP_FORCE_GENERIC) give the same output bits; and no pipelined kernel ever
gave up on a bounded wait."""

import numpy as np
import pytest
import torch

import workloads
from parity import assert_bf16_close, assert_dw_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu

SHAPES = [  # (T, n_q, n_kv, head_dim)
    (16384, 128, 16, 64),
    (1, 128, 16, 64),
    (3, 128, 16, 64),
    (333, 8, 2, 64),
    (17, 8, 2, 64),
    (129, 32, 8, 128),
    (257, 64, 8, 64),
    (65, 6, 1, 64),
    (40, 16, 16, 128),
]


def _run(C, wl, kind, dev, flags_extra):
    T, n_q, n_kv, D = wl.T, wl.n_q, wl.n_kv, wl.head_dim
    L = C.layout(kind, n_q, n_kv, D)
    rows = (wl.packed_rows() if kind == "interleaved" else wl.sectioned_rows()).to(dev)
    pos, wq, wk = wl.pos.to(dev), wl.w_q.to(dev), wl.w_k.to(dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    q, k, v = torch.empty(T, n_q, D, **bf), torch.empty(T, n_kv, D, **bf), torch.empty(T, n_kv, D, **bf)
    qp, kp = torch.empty(T, n_q, D, **bf), torch.empty(T, n_kv, D, **bf)
    C.qkv_prologue_fwd(L, T, rows, pos, wq, wk, wl.eps, wl.rope_base, C.QKVP_SAVE_PRE | flags_extra, q, k, v, qp, kp)
    need = C.qkv_prologue_bwd_workspace_size(L, T)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
    dp = torch.empty(T, (n_q + 2 * n_kv) * D, **bf)
    dwq, dwk = torch.empty(D, device=dev), torch.empty(D, device=dev)
    C.qkv_prologue_bwd(L, T, wl.dq.to(dev), wl.dk.to(dev), wl.dv.to(dev), qp, kp, pos, wq, wk, wl.eps,
                       wl.rope_base, flags_extra, dp, dwq, dwk, ws, need)
    return q, k, v, qp, kp, dp, dwq, dwk


@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s[0]}_q{s[1]}_kv{s[2]}_d{s[3]}" for s in SHAPES])
@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_pipelined_and_general_kernels_agree(lib, cuda, shape, kind):
    T, n_q, n_kv, D = shape
    wl = workloads.gqa_inputs(T, n_q, n_kv, D, seed=T + n_q, rope_base=5e5, pos_high=393216, with_grads=True)
    a = _run(lib, wl, kind, cuda, 0)
    b = _run(lib, wl, kind, cuda, lib.QKVP_FORCE_GENERIC)
    torch.cuda.synchronize()
    for x, y in zip(a[:6], b[:6]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for x, y in zip(a[6:], b[6:]):
        assert torch.allclose(x, y, rtol=1e-5, atol=1e-5 * float(y.abs().max()))


def test_general_kernels_match_oracle(lib, cuda):
    import oracle.prologue as P

    wl = workloads.gqa_inputs(333, 128, 16, 64, seed=5, rope_base=5e5, pos_high=131072, with_grads=True)
    q, k, v, qp, kp, dp, dwq, dwk = _run(lib, wl, "interleaved", cuda, lib.QKVP_FORCE_GENERIC)
    torch.cuda.synchronize()
    L = P.PackedLayout("interleaved", 128, 16, 64)
    ref = P.prologue_fwd(L, u16(wl.packed_rows()), wl.pos.numpy(), wl.w_q.numpy(), wl.w_k.numpy(), wl.eps,
                         wl.rope_base)
    assert_bf16_close(u16(q), ref["q"], "generic q")
    assert_bf16_close(u16(k), ref["k"], "generic k")
    assert np.array_equal(u16(v), ref["v_bits"])
    rb = P.prologue_bwd(L, u16(wl.dq), u16(wl.dk), u16(wl.dv), ref["q_pre_bits"], ref["k_pre_bits"],
                        wl.pos.numpy(), wl.w_q.numpy(), wl.w_k.numpy(), wl.eps, wl.rope_base)
    assert_bf16_close(u16(dp), rb["dpacked"], "generic dpacked")
    assert_dw_close(dwq.cpu().numpy(), rb["dw_q"])
    assert_dw_close(dwk.cpu().numpy(), rb["dw_k"])


def test_no_pipeline_wait_ever_gave_up(lib, cuda):
    # run a large pipelined forward + backward, then read the device error word
    wl = workloads.train(4096)
    _run(lib, wl, "interleaved", cuda, 0)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=False) == 0


@pytest.mark.parametrize("T", [1, 16, 100, 32768])
@pytest.mark.parametrize("pool", [False, True])
def test_latent_pipelined_and_general_kernels_agree(lib, cuda, T, pool):
    C = lib
    wl = workloads.mla(T)
    L = C.layout("latent", norm_dim=512, rope_dim=64)
    rows, pos, w = wl.rows.to(cuda), wl.pos.to(cuda), wl.w.to(cuda)
    page, off = wl.page.to(cuda), wl.offset.to(cuda)
    outs = []
    for flags in (0, C.QKVP_FORCE_GENERIC):
        if pool:
            dst = workloads.random_pool_bits((wl.num_pages, wl.page_size, 576), 61, cuda)
            C.qkv_prologue_pool_write(L, T, rows, pos, None, w, wl.eps, wl.rope_base, flags, None, page, off, dst,
                                      None, wl.num_pages, wl.page_size)
        else:
            dst = torch.empty(T, 576, dtype=torch.bfloat16, device=cuda)
            C.qkv_prologue_fwd(L, T, rows, pos, None, w, wl.eps, wl.rope_base, flags, None, dst, None)
        outs.append(dst)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))

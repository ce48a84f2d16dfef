"""qkv_prologue_bwd_noalloc, the backward for callers that cannot allocate device
memory (it keeps its partial sums in a fixed array inside the library instead
of a caller workspace), must give what qkv_prologue_bwd gives.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It also runs on its own in a
fresh process (it needs nothing from the other test files).
"""

import pytest
import torch

import workloads
from parity import assert_bf16_close, assert_dw_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu


def _inputs(C, wl, dev, kind="interleaved"):
    T, n_q, n_kv, D = wl.T, wl.n_q, wl.n_kv, wl.head_dim
    L = C.layout(kind, n_q, n_kv, D)
    rows = (wl.packed_rows() if kind == "interleaved" else wl.sectioned_rows()).to(dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    q, k, v = torch.empty(T, n_q, D, **bf), torch.empty(T, n_kv, D, **bf), torch.empty(T, n_kv, D, **bf)
    qp, kp = torch.empty(T, n_q, D, **bf), torch.empty(T, n_kv, D, **bf)
    args = dict(pos=wl.pos.to(dev), w_q=wl.w_q.to(dev), w_k=wl.w_k.to(dev))
    C.qkv_prologue_fwd(L, T, rows, args["pos"], args["w_q"], args["w_k"], wl.eps, wl.rope_base, C.QKVP_SAVE_PRE,
                       q, k, v, qp, kp)
    return L, dict(dq=wl.dq.to(dev), dk=wl.dk.to(dev), dv=wl.dv.to(dev), q_pre=qp, k_pre=kp, **args)


def _outputs(wl, dev):
    D = wl.head_dim
    dp = torch.empty(wl.T, (wl.n_q + 2 * wl.n_kv) * D, dtype=torch.bfloat16, device=dev)
    return dp, torch.empty(D, device=dev), torch.empty(D, device=dev)


def _regular(C, L, wl, a, dev, flags=0):
    dp, dwq, dwk = _outputs(wl, dev)
    need = C.qkv_prologue_bwd_workspace_size(L, wl.T)
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
    C.qkv_prologue_bwd(L, wl.T, a["dq"], a["dk"], a["dv"], a["q_pre"], a["k_pre"], a["pos"], a["w_q"], a["w_k"],
                       wl.eps, wl.rope_base, flags, dp, dwq, dwk, ws, need)
    return dp, dwq, dwk


def _noalloc(C, L, wl, a, dev, flags=0, out=None):
    dp, dwq, dwk = _outputs(wl, dev) if out is None else out
    C.qkv_prologue_bwd_noalloc(L, wl.T, a["dq"], a["dk"], a["dv"], a["q_pre"], a["k_pre"], a["pos"], a["w_q"],
                               a["w_k"], wl.eps, wl.rope_base, flags, dp, dwq, dwk)
    return dp, dwq, dwk


def _same(got, want):
    dp, dwq, dwk = got
    rdp, rdwq, rdwk = want
    # the tolerance the parity tests use, measured against the regular entry point's output
    assert_bf16_close(u16(dp), _widen(rdp), "dpacked")
    assert_dw_close(dwq.cpu().numpy(), rdwq.cpu().numpy(), "dw_q")
    assert_dw_close(dwk.cpu().numpy(), rdwk.cpu().numpy(), "dw_k")
    # and in fact it is the same computation: identical bits
    assert torch.equal(dp.view(torch.int16), rdp.view(torch.int16))
    assert torch.equal(dwq, rdwq) and torch.equal(dwk, rdwk)


def _widen(t):
    from oracle import bf16_bits_to_f64

    return bf16_bits_to_f64(u16(t))


def test_noalloc_backward_matches_regular_backward_twice_in_a_row(lib, cuda):
    C = lib
    cases = [
        workloads.train(4096),                                            # Muse Spark shape
        workloads.gqa_inputs(333, 8, 2, 64, seed=9, rope_base=1e4, pos_high=393216, with_grads=True),
        workloads.gqa_inputs(200, 32, 8, 128, seed=10, rope_base=5e5, pos_high=131072, with_grads=True),
    ]
    for wl in cases:
        L, a = _inputs(C, wl, cuda)
        want = _regular(C, L, wl, a, cuda)
        first = _noalloc(C, L, wl, a, cuda)     # the array holds the previous case's partials here
        second = _noalloc(C, L, wl, a, cuda)    # and this call's own ones here
        torch.cuda.synchronize()
        _same(first, want)
        _same(second, want)
    assert C.qkv_prologue_device_error(clear=False) == 0


def test_noalloc_backward_rejects_work_beyond_its_array(lib, cuda):
    C = lib
    wl = workloads.gqa_inputs(2048, 32, 8, 128, seed=11, rope_base=5e5, with_grads=True)
    L, a = _inputs(C, wl, cuda)
    assert C.qkv_prologue_bwd_workspace_size(L, wl.T) > 512 * 1024
    dp, dwq, dwk = _outputs(wl, cuda)
    dwq.fill_(3.0)
    st = C.qkv_prologue_bwd_noalloc(L, wl.T, a["dq"], a["dk"], a["dv"], a["q_pre"], a["k_pre"], a["pos"], a["w_q"],
                                    a["w_k"], wl.eps, wl.rope_base, 0, dp, dwq, dwk, check=False)
    torch.cuda.synchronize()
    assert st == C.QKVP_ERR_WORKSPACE
    assert torch.all(dwq == 3.0)  # nothing was enqueued


def test_noalloc_backward_nope_and_norm_off(lib, cuda):
    # NoPE and norm-off calls give the regular entry point's bits too; without the
    # norm there are no partial sums, so no scratch is needed and a size that the
    # norm-on call refuses is accepted
    C = lib
    small = workloads.gqa_inputs(257, 16, 4, 64, seed=12, rope_base=5e5, pos_high=131072, with_grads=True)
    big = workloads.gqa_inputs(2048, 32, 8, 128, seed=11, rope_base=5e5, with_grads=True)
    for wl, flags in ((small, C.QKVP_NOPE), (small, C.QKVP_NORM_OFF), (big, C.QKVP_NORM_OFF),
                      (big, C.QKVP_NORM_OFF | C.QKVP_NOPE)):
        L, a = _inputs(C, wl, cuda)
        want = _regular(C, L, wl, a, cuda, flags)
        first = _noalloc(C, L, wl, a, cuda, flags)
        second = _noalloc(C, L, wl, a, cuda, flags)
        torch.cuda.synchronize()
        for got in (first, second):
            assert torch.equal(got[0].view(torch.int16), want[0].view(torch.int16))
            if not flags & C.QKVP_NORM_OFF:
                _same(got, want)
    assert C.qkv_prologue_device_error(clear=False) == 0


def test_noalloc_backward_allocates_no_device_memory(lib, cuda):
    # one warm-up call (it looks up the array's address), then a loop of calls
    # with preallocated outputs: neither the driver's free memory nor torch's
    # allocator may move
    C = lib
    wl = workloads.gqa_inputs(1024, 32, 8, 64, seed=13, rope_base=5e5, pos_high=131072, with_grads=True)
    L, a = _inputs(C, wl, cuda)
    out = _outputs(wl, cuda)
    _noalloc(C, L, wl, a, cuda, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda)
    used0 = torch.cuda.memory_allocated(cuda)
    for _ in range(20):
        _noalloc(C, L, wl, a, cuda, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda)
    assert torch.cuda.memory_allocated(cuda) == used0
    assert free1 == free0

"""The library's bounded wait, made to run out on purpose (no fault, no hang):
qkv_prologue_wait_selftest enqueues a kernel whose only wait is on an mbarrier
phase that nothing completes. Every pipelined kernel waits through the same
code; after the limit (2 s) it must give up, set bit 1 of the device error
word, return, and leave the context usable for the next call."""

import time

import pytest
import torch

import oracle.prologue as P
import workloads
from parity import assert_bf16_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu


def test_wait_gives_up_after_the_limit_and_reports(lib, cuda):
    lib.qkv_prologue_device_error(clear=True)  # start clean
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lib.qkv_prologue_wait_selftest()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 1.9 < waited < 30.0, f"the wait gave up after {waited:.2f} s"
    assert lib.qkv_prologue_device_error(clear=True) == 1  # the timeout bit, nothing else
    assert lib.qkv_prologue_device_error(clear=False) == 0  # cleared

    # the context is still usable: an ordinary forward call is correct afterwards
    F = lib.functional
    wl = workloads.gqa_inputs(16, 8, 2, 64, seed=3, rope_base=10000.0)
    rows = wl.packed_rows()
    q, k, v = F.prologue_forward(rows.to(cuda), wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), 8, 2, 64,
                                 "interleaved", wl.eps, wl.rope_base)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=False) == 0
    ref = P.prologue_fwd(P.PackedLayout("interleaved", 8, 2, 64), u16(rows), wl.pos.numpy(), wl.w_q.numpy(),
                         wl.w_k.numpy(), wl.eps, wl.rope_base)
    assert_bf16_close(u16(q), ref["q"], "q after the timed-out wait")
    assert_bf16_close(u16(k), ref["k"], "k after the timed-out wait")

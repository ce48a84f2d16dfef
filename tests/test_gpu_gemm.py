"""The wqkv projection with the prologue in its epilogue (tcgen05 tensor cores)
against the fp64 oracle: packed = x . W^T rounded once to bf16, then the
prologue. The inputs make every product and partial sum exact in float32, so
the kernel's packed values are the oracle's bit for bit and the outputs are
held to the prologue's tolerance."""

import numpy as np
import pytest
import torch

import oracle.prologue as P
import workloads
from parity import assert_bf16_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu

CASES = [
    # T, hidden, n_q, n_kv, D, kind: tiles with ragged M, N and K edges, both packings and head sizes
    (128, 64, 8, 2, 64, "interleaved"),
    (300, 520, 8, 2, 64, "interleaved"),      # 12 head blocks: 3 N tiles; ragged T and K
    (257, 1024, 128, 16, 64, "interleaved"),  # the Muse Spark row (10240 columns, 40 N tiles)
    (200, 768, 32, 8, 128, "sectioned"),      # Llama 3 / Qwen3 heads
    (64, 4096, 64, 8, 64, "sectioned"),       # GPT-OSS heads, long K
]


@pytest.mark.parametrize("T,hidden,n_q,n_kv,D,kind", CASES)
@pytest.mark.parametrize("save", [False, True])
def test_gemm_prologue_matches_oracle(lib, cuda, T, hidden, n_q, n_kv, D, kind, save):
    F = lib.functional
    x, w = workloads.gemm_inputs(T, hidden, n_q, n_kv, D, seed=T + hidden)
    g = workloads._gen(7)
    pos = torch.randint(0, 393216, (T,), generator=g, dtype=torch.int32)
    w_q, w_k = workloads.norm_weight(D, g), workloads.norm_weight(D, g)
    out = F.gemm_prologue_forward(x.to(cuda), w.to(cuda), pos.to(cuda), w_q.to(cuda), w_k.to(cuda), n_q, n_kv, D,
                                  kind, 1e-6, 5e5, save_pre=save)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=False) == 0
    L = P.PackedLayout(kind, n_q, n_kv, D)
    ref, packed = P.gemm_prologue_fwd(L, u16(x), u16(w), pos.numpy(), w_q.numpy(), w_k.numpy(), 1e-6, 5e5)
    assert_bf16_close(u16(out[0]), ref["q"], "q")
    assert_bf16_close(u16(out[1]), ref["k"], "k")
    assert np.array_equal(u16(out[2]), ref["v_bits"]), "v is the rounded product"
    if save:
        assert np.array_equal(u16(out[3]), ref["q_pre_bits"]) and np.array_equal(u16(out[4]), ref["k_pre_bits"])


def test_gemm_prologue_equals_projection_then_prologue(lib, cuda):
    # with exact inputs cuBLAS's projection gives the same packed bf16 values, so
    # the fused call and cuBLAS + qkv_prologue_fwd agree within one bf16 ulp
    # (their prologues round once from float32 sums taken in different orders)
    F = lib.functional
    T, hidden, n_q, n_kv, D = 512, 2048, 128, 16, 64
    x, w = workloads.gemm_inputs(T, hidden, n_q, n_kv, D, seed=3)
    pos = torch.arange(T, dtype=torch.int32)
    g = workloads._gen(8)
    w_q, w_k = workloads.norm_weight(D, g), workloads.norm_weight(D, g)
    dx, dw = x.to(cuda), w.to(cuda)
    fused = F.gemm_prologue_forward(dx, dw, pos.to(cuda), w_q.to(cuda), w_k.to(cuda), n_q, n_kv, D)
    packed = (dx @ dw.T).contiguous()
    unfused = F.prologue_forward(packed, pos.to(cuda), w_q.to(cuda), w_k.to(cuda), n_q, n_kv, D)
    torch.cuda.synchronize()
    for a, b in zip(fused, unfused):
        assert_bf16_close(u16(a), b.double().cpu().numpy(), "fused vs unfused")

"""Per-head Newton-Schulz of a fused QKV update on the tensor cores against the
fp64 oracle ("[muon] Per-head Newton-Schulz for fused QKV projections").

The kernel holds X, A and b A + c A A in bf16 between its products, as the
published bf16 iteration does, so it cannot match the exact iteration to a
few ulps: its distance from the oracle is that of any bf16 evaluation. Each
block is held to a bound sized on that block: the error of the oracle's own
steps with bf16 rounding at those points (same input, the oracle's rounding
hook), times 2 in relative Frobenius norm and times 3 in the largest element,
plus a floor of 2^-9 (Frobenius) and 2^-8 of the largest element. What is
exact is checked exactly: the two packings give the same bits up to the block
permutation, runs repeat bit for bit, rows past the weight stay untouched.
"""

import numpy as np
import pytest
import torch

import oracle.newton_schulz as N
import workloads
from oracle.bf16 import bf16_bits_to_f64, to_bf16_rne
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu


def _r16(v):
    return bf16_bits_to_f64(to_bf16_rne(v))


def check_blocks(got, m, head_dim, blocks=None, what=""):
    """got, m: bf16 tensors [rows, cols] (CPU); every listed block within its bound."""
    gm, mm = bf16_bits_to_f64(u16(got)), bf16_bits_to_f64(u16(m))
    rows, cols = mm.shape
    s = N.per_head_scale(head_dim, cols)
    worst = 0.0
    for b in (range(rows // head_dim) if blocks is None else blocks):
        sl = slice(b * head_dim, (b + 1) * head_dim)
        exact = N.newton_schulz5(mm[sl]) * s
        nrm = np.linalg.norm(exact)
        if nrm == 0.0:
            assert not np.any(gm[sl]), f"{what} block {b}: a zero block must give zeros"
            continue
        emul = N.newton_schulz5(mm[sl], rounding=_r16) * s
        e_emul = np.linalg.norm(emul - exact) / nrm
        e_got = np.linalg.norm(gm[sl] - exact) / nrm
        assert np.all(np.isfinite(gm[sl])), f"{what} block {b}: non-finite output"
        assert e_got <= 2 * e_emul + 2.0 ** -9, f"{what} block {b}: rel Frobenius {e_got:.4g} vs bf16 steps {e_emul:.4g}"
        big = np.abs(exact).max()
        m_emul, m_got = np.abs(emul - exact).max(), np.abs(gm[sl] - exact).max()
        assert m_got <= 3 * m_emul + 2.0 ** -8 * big, f"{what} block {b}: max abs {m_got:.4g} vs {m_emul:.4g}"
        worst = max(worst, e_got / (e_emul + 1e-30))
    return worst


def run(lib, m, n_q, n_kv, D, kind="interleaved", cluster=0):
    out = lib.functional.per_head_newton_schulz(m, n_q, n_kv, D, kind, cluster=cluster)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    return out


def test_page_model_both_packings(lib, cuda):
    # 8 query heads over 2 KV heads of 64, hidden 512: 12 blocks per layer
    c = workloads.NS_PAGE_MODEL
    for layer in range(2):
        w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=100 + layer)
        ws = workloads.sectioned_weight_from_interleaved(w, c["n_q"], c["n_kv"], c["head_dim"])
        gi = run(lib, w.to(cuda), c["n_q"], c["n_kv"], c["head_dim"], "interleaved").cpu()
        gs = run(lib, ws.to(cuda), c["n_q"], c["n_kv"], c["head_dim"], "sectioned").cpu()
        check_blocks(gi, w, c["head_dim"], what="interleaved")
        # the sectioned result is the interleaved one with its blocks permuted, bit for bit
        want = workloads.sectioned_weight_from_interleaved(gi, c["n_q"], c["n_kv"], c["head_dim"])
        assert torch.equal(gs.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_every_cluster_size(lib, cuda, cluster):
    # 512 columns split 1, 2, 4, 8 ways (512 .. 64 columns per CTA); 20 blocks, odd unit count
    n_q, n_kv, D, cols = 16, 2, 64, 512
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=7 + cluster)
    got = run(lib, w.to(cuda), n_q, n_kv, D, cluster=cluster).cpu()
    check_blocks(got, w, D, what=f"cluster {cluster}")


def test_non_portable_cluster_of_16(lib, cuda):
    L = lib.layout("interleaved", 8, 2, 64)
    try:
        nc, grid = lib.qkv_newton_schulz_plan(L, 1024, 16)
    except lib.QkvpError:
        pytest.skip("the device does not co-schedule clusters of 16 of these CTAs")
    assert nc == 16 and grid == 6 * 16
    w = workloads.fused_qkv_update(8, 2, 64, 1024, seed=21)
    got = run(lib, w.to(cuda), 8, 2, 64, cluster=16).cpu()
    check_blocks(got, w, 64, what="cluster 16")


@pytest.mark.parametrize("cluster", [0, 2])
def test_head_dim_128(lib, cuda, cluster):
    # Llama 3 / Qwen3 heads: one head per 128-row unit, the Gram exchanged in two passes
    n_q, n_kv, D, cols = 4, 2, 128, 1024
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=31)
    got = run(lib, w.to(cuda), n_q, n_kv, D, cluster=cluster).cpu()
    check_blocks(got, w, D, what="head_dim 128")


def test_odd_block_count_leaves_rows_past_the_weight(lib, cuda):
    # 1 q + 1 k + 1 v head of 64: 3 blocks, the second unit half empty
    n_q, n_kv, D, cols = 1, 1, 64, 256
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=41)
    buf = torch.full((4 * D, cols), 7.0, dtype=torch.bfloat16, device=cuda)
    out = buf[: 3 * D]
    lib.functional.per_head_newton_schulz(w.to(cuda), n_q, n_kv, D, out=out)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    assert torch.all(buf[3 * D:] == 7.0), "rows past the weight were written"
    check_blocks(out.cpu(), w, D, what="odd blocks")


def test_tall_blocks(lib, cuda):
    # head_dim 128 over 64 inputs: the published code transposes such a block;
    # the factor is sqrt(128 / 64)
    n_q, n_kv, D, cols = 2, 1, 128, 64
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=51)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what="tall")


def test_zero_tiny_and_large_blocks(lib, cuda):
    n_q, n_kv, D, cols = 4, 2, 64, 384
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=61).float()
    mags = torch.tensor([0.0, 1e-12, 1e3, 1.0, 3e-5, 1.0, 50.0, 1.0])
    w = (w.view(8, D, cols) * mags[:, None, None]).view(8 * D, cols).to(torch.bfloat16)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what="magnitudes")


def test_repeatable_bits(lib, cuda):
    c = workloads.NS_PAGE_MODEL
    w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=71).to(cuda)
    a = run(lib, w, c["n_q"], c["n_kv"], c["head_dim"])
    b = run(lib, w, c["n_q"], c["n_kv"], c["head_dim"])
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_full_size_muse_spark_weight_sampled(lib, cuda):
    # the [10240, 5120] fused weight of the benchmark, in the launch it times;
    # every block finite, sampled blocks against the oracle
    c = workloads.NS_MUSE_SPARK
    w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=81)
    got = run(lib, w.to(cuda), c["n_q"], c["n_kv"], c["head_dim"]).cpu()
    assert torch.isfinite(got.float()).all()
    n_blocks = w.shape[0] // c["head_dim"]
    rng = np.random.default_rng(5)
    sample = sorted(set([0, 1, n_blocks - 1] + list(rng.choice(n_blocks, 5, replace=False))))
    check_blocks(got, w, c["head_dim"], blocks=sample, what="full size")


def test_batch_of_layers_in_one_launch(lib, cuda):
    # the page's model: six layers' updates stacked, one launch; each layer
    # against the oracle, and the same bits as six single calls with the same
    # cluster size (the 128-row units line up with the layers)
    c = workloads.NS_PAGE_MODEL
    ws = [workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=300 + i) for i in range(6)]
    m = torch.stack(ws).to(cuda)
    got = lib.functional.per_head_newton_schulz(m, c["n_q"], c["n_kv"], c["head_dim"], cluster=4)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    for i in range(6):
        one = run(lib, m[i], c["n_q"], c["n_kv"], c["head_dim"], cluster=4)
        assert torch.equal(one.view(torch.int16), got[i].view(torch.int16)), f"layer {i}"
        check_blocks(got[i].cpu(), ws[i], c["head_dim"], what=f"layer {i}")


def test_batch_with_units_across_layers(lib, cuda):
    # 3 blocks per layer (1 q + 1 k + 1 v): the 128-row units straddle layers
    n_q, n_kv, D, cols = 1, 1, 64, 256
    ws = [workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=400 + i) for i in range(3)]
    buf = torch.full((4, 3 * D, cols), 5.0, dtype=torch.bfloat16, device=cuda)
    out = buf[:3]
    lib.functional.per_head_newton_schulz(torch.stack(ws).to(cuda), n_q, n_kv, D, out=out)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    assert torch.all(buf[3] == 5.0), "rows past the stack were written"
    for i in range(3):
        check_blocks(out[i].cpu(), ws[i], D, what=f"layer {i}")


@pytest.mark.parametrize("cluster", [14, 16])
def test_wide_in_features_large_clusters(lib, cuda, cluster):
    # in_features 7168 (112 boxes of 64 columns): clusters of 14 (512 columns per
    # CTA, the fullest receive buffer: 14 slots of 10 rows) and of 16 (448)
    n_q, n_kv, D, cols = 4, 2, 128, 7168
    L = lib.layout("interleaved", n_q, n_kv, D)
    try:
        nc, _ = lib.qkv_newton_schulz_plan(L, cols, cluster)
    except lib.QkvpError:
        pytest.skip(f"the device does not co-schedule clusters of {cluster} of these CTAs")
    assert nc == cluster
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=500 + cluster)
    got = run(lib, w.to(cuda), n_q, n_kv, D, cluster=cluster).cpu()
    check_blocks(got, w, D, what=f"7168 columns, cluster {cluster}")


def test_llama70b_shaped_weight_sampled(lib, cuda):
    # 64 q heads over 8 kv heads of 128, in_features 8192: [10240, 8192], the
    # widest update the kernel takes (16 CTAs of 512 columns per unit)
    n_q, n_kv, D, cols = 64, 8, 128, 8192
    L = lib.layout("interleaved", n_q, n_kv, D)
    try:
        lib.qkv_newton_schulz_plan(L, cols)
    except lib.QkvpError:
        pytest.skip("the device does not co-schedule clusters of 16 of these CTAs")
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=601)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    assert torch.isfinite(got.float()).all()
    check_blocks(got, w, D, blocks=[0, 1, 37, 79], what="[10240, 8192]")

"""Per-head Newton-Schulz of a fused QKV update on the tensor cores against the
fp64 oracle ("[muon] Per-head Newton-Schulz for fused QKV projections").

The kernels evaluate the iteration through each block's Gram matrix (X_5 =
M X_0 with M a product of polynomials in X_0 X_0^T), with every matrix operand
held as two bf16 terms and fp32 accumulation, so they match neither the exact
iteration to a few ulps nor the published bf16 iteration bit for bit. Each
block is held to a bound sized on that block: the error of the oracle's own
steps with bf16 rounding at the published points (same input, the oracle's
rounding hook), times 2 in relative Frobenius norm and times 3 in the largest
element, plus a floor of 2^-9 (Frobenius) and 2^-8 of the largest element.
The two-term arithmetic is much closer to the exact iteration than that; the
`tight` checks hold it to a quarter of the bf16 steps' error plus 1.25 times
the error of rounding the exact result to bf16 (the output's own floor),
also on ill-conditioned blocks (a decaying spectrum, low rank plus noise,
tall blocks), where a one-term (bf16 or tf32) evaluation of M fails by tens
of percent. What is exact is checked exactly: the two packings give the same
bits up to the block permutation, runs repeat bit for bit, rows past the
weight stay untouched, the workspace's prior contents do not matter.
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


def check_blocks(got, m, head_dim, blocks=None, what="", tight=False):
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
        if tight:  # the output's own rounding to bf16 plus a quarter of the bf16 steps' error
            e_round = np.linalg.norm(_r16(exact) - exact) / nrm
            assert e_got <= 1.25 * e_round + 0.25 * e_emul, (
                f"{what} block {b}: rel Frobenius {e_got:.4g}, not well inside the bf16 steps' {e_emul:.4g} "
                f"(rounding the exact result to bf16: {e_round:.4g})")
        worst = max(worst, e_got / (e_emul + 1e-30))
    return worst


def run(lib, m, n_q, n_kv, D, kind="interleaved", split=0):
    out = lib.functional.per_head_newton_schulz(m, n_q, n_kv, D, kind, split=split)
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
        check_blocks(gi, w, c["head_dim"], what="interleaved", tight=True)
        # the sectioned result is the interleaved one with its blocks permuted, bit for bit
        want = workloads.sectioned_weight_from_interleaved(gi, c["n_q"], c["n_kv"], c["head_dim"])
        assert torch.equal(gs.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("split", [1, 2, 3, 8])
def test_every_split(lib, cuda, split):
    # 512 columns (8 boxes) over 1, 2, 3 (ragged: 2, 3, 3 boxes) and 8 Gram
    # CTAs per unit; 20 blocks, an even unit count
    n_q, n_kv, D, cols = 16, 2, 64, 512
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=7 + split)
    got = run(lib, w.to(cuda), n_q, n_kv, D, split=split).cpu()
    check_blocks(got, w, D, what=f"split {split}", tight=True)


def test_split_changes_only_the_summation_order(lib, cuda):
    # splits 1 and 4 sum the Gram partials in different groupings: results
    # differ by rounding only (both within the tight bound)
    n_q, n_kv, D, cols = 8, 2, 64, 1024
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=11)
    a = run(lib, w.to(cuda), n_q, n_kv, D, split=1).cpu()
    b = run(lib, w.to(cuda), n_q, n_kv, D, split=4).cpu()
    check_blocks(a, w, D, what="split 1", tight=True)
    check_blocks(b, w, D, what="split 4", tight=True)
    da = (a.float() - b.float()).abs().max().item()
    assert da < 2.0 ** -6, f"splits 1 and 4 differ by {da}"


def test_largest_split(lib, cuda):
    n_q, n_kv, D, cols = 4, 1, 64, 4096  # 64 boxes, 64 Gram CTAs of one box per unit
    assert lib.qkv_newton_schulz_plan(lib.layout("interleaved", n_q, n_kv, D), cols, 64) == (64, 3 * 64)
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=21)
    got = run(lib, w.to(cuda), n_q, n_kv, D, split=64).cpu()
    check_blocks(got, w, D, what="split 64", tight=True)


@pytest.mark.parametrize("split", [0, 2])
def test_head_dim_128(lib, cuda, split):
    # Llama 3 / Qwen3 heads: one head per 128-row unit, full 128 x 128 products
    n_q, n_kv, D, cols = 4, 2, 128, 1024
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=31)
    got = run(lib, w.to(cuda), n_q, n_kv, D, split=split).cpu()
    check_blocks(got, w, D, what="head_dim 128", tight=True)


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
    check_blocks(out.cpu(), w, D, what="odd blocks", tight=True)


def test_tall_blocks(lib, cuda):
    # head_dim 128 over 64 inputs: the published code transposes such a block
    # (the same polynomial); the Gram matrix X X^T is 128 x 128 of rank 64, so M
    # is large on its null space; the factor is sqrt(128 / 64)
    n_q, n_kv, D, cols = 2, 1, 128, 64
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=51)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what="tall", tight=True)


def _structured(rows, cols, D, kind, seed):
    """Blocks of D rows with a given spectrum, bf16."""
    rng = np.random.default_rng(seed)
    out = np.empty((rows, cols))
    for b in range(rows // D):
        if kind == "decay":  # singular values e^(-i / 6): conditioning ~1e9
            q1, _ = np.linalg.qr(rng.standard_normal((D, D)))
            q2, _ = np.linalg.qr(rng.standard_normal((cols, D)))
            out[b * D:(b + 1) * D] = (q1 * np.exp(-np.arange(D) / 6.0)) @ q2.T
        else:  # rank 4 plus noise 1e-3
            out[b * D:(b + 1) * D] = (rng.standard_normal((D, 4)) @ rng.standard_normal((4, cols))
                                      + 1e-3 * rng.standard_normal((D, cols)))
    return torch.from_numpy(out).to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", ["decay", "low_rank"])
def test_ill_conditioned_blocks(lib, cuda, D, kind):
    n_q, n_kv, cols = 2, 1, 512
    w = _structured((n_q + 2 * n_kv) * D, cols, D, kind, seed=61 + D)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what=f"{kind} D={D}", tight=True)


def test_zero_tiny_and_large_blocks(lib, cuda):
    n_q, n_kv, D, cols = 4, 2, 64, 384
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=61).float()
    mags = torch.tensor([0.0, 1e-12, 1e3, 1.0, 3e-5, 1.0, 50.0, 1.0])
    w = (w.view(8, D, cols) * mags[:, None, None]).view(8 * D, cols).to(torch.bfloat16)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what="magnitudes", tight=True)


def test_repeatable_bits_and_any_workspace_contents(lib, cuda):
    c = workloads.NS_PAGE_MODEL
    F = lib.functional
    w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=71).to(cuda)
    a = run(lib, w, c["n_q"], c["n_kv"], c["head_dim"])
    need = F.newton_schulz_workspace_bytes(w.shape, c["n_q"], c["n_kv"], c["head_dim"])
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=cuda)  # NaN patterns everywhere
    b = F.per_head_newton_schulz(w, c["n_q"], c["n_kv"], c["head_dim"], workspace=ws)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_workspace_too_small_is_refused(lib, cuda):
    c = workloads.NS_PAGE_MODEL
    F = lib.functional
    w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=72).to(cuda)
    need = F.newton_schulz_workspace_bytes(w.shape, c["n_q"], c["n_kv"], c["head_dim"])
    ws = torch.empty(need - 16, dtype=torch.uint8, device=cuda)
    with pytest.raises(lib.QkvpError):
        F.per_head_newton_schulz(w, c["n_q"], c["n_kv"], c["head_dim"], workspace=ws)


def test_full_size_muse_spark_weight_sampled(lib, cuda):
    # the [10240, 5120] fused weight of the benchmark, in the launches it times;
    # every block finite, sampled blocks against the oracle
    c = workloads.NS_MUSE_SPARK
    w = workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=81)
    got = run(lib, w.to(cuda), c["n_q"], c["n_kv"], c["head_dim"]).cpu()
    assert torch.isfinite(got.float()).all()
    n_blocks = w.shape[0] // c["head_dim"]
    rng = np.random.default_rng(5)
    sample = sorted(set([0, 1, n_blocks - 1] + list(rng.choice(n_blocks, 5, replace=False))))
    check_blocks(got, w, c["head_dim"], blocks=sample, what="full size", tight=True)


def test_batch_of_layers_in_one_launch(lib, cuda):
    # the page's model: six layers' updates stacked, one set of launches; each
    # layer against the oracle, and the same bits as six single calls with the
    # same split (the 128-row units line up with the layers)
    c = workloads.NS_PAGE_MODEL
    ws = [workloads.fused_qkv_update(c["n_q"], c["n_kv"], c["head_dim"], c["cols"], seed=300 + i) for i in range(6)]
    m = torch.stack(ws).to(cuda)
    got = lib.functional.per_head_newton_schulz(m, c["n_q"], c["n_kv"], c["head_dim"], split=2)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    for i in range(6):
        one = run(lib, m[i], c["n_q"], c["n_kv"], c["head_dim"], split=2)
        assert torch.equal(one.view(torch.int16), got[i].view(torch.int16)), f"layer {i}"
        check_blocks(got[i].cpu(), ws[i], c["head_dim"], what=f"layer {i}", tight=True)


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
        check_blocks(out[i].cpu(), ws[i], D, what=f"layer {i}", tight=True)


@pytest.mark.parametrize("split", [0, 14])
def test_wide_in_features(lib, cuda, split):
    # in_features 7168 (112 boxes of 64 columns), head_dim 128; split 14: 8
    # boxes per Gram CTA
    n_q, n_kv, D, cols = 4, 2, 128, 7168
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=500 + split)
    got = run(lib, w.to(cuda), n_q, n_kv, D, split=split).cpu()
    check_blocks(got, w, D, what=f"7168 columns, split {split}", tight=True)


def test_llama70b_shaped_weight_sampled(lib, cuda):
    # 64 q heads over 8 kv heads of 128, in_features 8192: [10240, 8192]
    n_q, n_kv, D, cols = 64, 8, 128, 8192
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=601)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    assert torch.isfinite(got.float()).all()
    check_blocks(got, w, D, blocks=[0, 1, 37, 79], what="[10240, 8192]", tight=True)


def test_in_features_beyond_one_smem_slice(lib, cuda):
    # 16384 inputs: wider than any shared-memory-resident slice scheme could
    # hold; the Gram and apply passes stream it
    n_q, n_kv, D, cols = 2, 1, 64, 16384
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=701)
    got = run(lib, w.to(cuda), n_q, n_kv, D).cpu()
    check_blocks(got, w, D, what="16384 columns", tight=True)


def test_under_cuda_graph_capture(lib, cuda):
    # 80 units, the three kernels captured in a graph on a side stream and
    # replayed: the eager call's bits (and the eager call matches the oracle)
    n_q, n_kv, D, cols = 128, 16, 64, 512
    F = lib.functional
    w = workloads.fused_qkv_update(n_q, n_kv, D, cols, seed=91).to(cuda)
    eager = F.per_head_newton_schulz(w, n_q, n_kv, D)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    need = F.newton_schulz_workspace_bytes(w.shape, n_q, n_kv, D)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda)
    out = torch.empty_like(w)
    s = torch.cuda.Stream(cuda)
    s.wait_stream(torch.cuda.current_stream(cuda))
    with torch.cuda.stream(s):
        F.per_head_newton_schulz(w, n_q, n_kv, D, out=out, workspace=ws)  # warm-up outside the graph
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        F.per_head_newton_schulz(w, n_q, n_kv, D, out=out, workspace=ws)
    out.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=True) == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    check_blocks(out.cpu(), w.cpu(), D, blocks=[0, 1, 79, 80, 159], what="graph replay", tight=True)

"""CUDA path (through the C ABI) against the fp64 oracle, on the five workloads
and the edge cases. Every call here reaches the library's kernels; the oracle
runs on the host on the same seeded inputs."""

import numpy as np
import pytest
import torch

import oracle
import oracle.prologue as P
import workloads
from parity import assert_bf16_close, assert_dw_close, bf16_report
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu


def _layout(wl, kind):
    return P.PackedLayout(kind, wl.n_q, wl.n_kv, wl.head_dim)


def _rows(wl, kind):
    return wl.packed_rows() if kind == "interleaved" else wl.sectioned_rows()


def _gpu_fwd(lib, wl, kind, dev, save=False, nope=None):
    F = lib.functional
    nope = wl.nope if nope is None else nope
    return F.prologue_forward(_rows(wl, kind).to(dev), wl.pos.to(dev), wl.w_q.to(dev), wl.w_k.to(dev),
                              wl.n_q, wl.n_kv, wl.head_dim, kind, wl.eps, wl.rope_base, nope, save_pre=save)


def _oracle_fwd(wl, kind, tokens=None, nope=None):
    nope = wl.nope if nope is None else nope
    rows = u16(_rows(wl, kind))
    pos = wl.pos.numpy()
    if tokens is not None:
        rows, pos = rows[tokens], pos[tokens]
    return P.prologue_fwd(_layout(wl, kind), rows, pos, wl.w_q.numpy(), wl.w_k.numpy(), wl.eps,
                          wl.rope_base, nope)


def _check_fwd(wl, kind, out, tokens=None, what=""):
    q, k, v = (u16(t) for t in out[:3])
    if tokens is not None:
        q, k, v = q[tokens], k[tokens], v[tokens]
    ref = _oracle_fwd(wl, kind, tokens)
    rq = assert_bf16_close(q, ref["q"], f"{what} q")
    rk = assert_bf16_close(k, ref["k"], f"{what} k")
    assert np.array_equal(v, ref["v_bits"]), f"{what} v is not a bit copy"
    if len(out) == 5:
        qp_, kp_ = u16(out[3]), u16(out[4])
        if tokens is not None:
            qp_, kp_ = qp_[tokens], kp_[tokens]
        assert np.array_equal(qp_, ref["q_pre_bits"]) and np.array_equal(kp_, ref["k_pre_bits"])
    return rq, rk


def _merge_reports(reports):
    n = sum(r["n"] for r in reports)
    return {"n": n, "exact_match": sum(r["exact_match"] * r["n"] for r in reports) / max(n, 1),
            "max_ulp": max(r["max_ulp"] for r in reports), "max_rel": max(r["max_rel"] for r in reports),
            "all_finite": all(r["all_finite"] for r in reports)}


def _check_fwd_all(wl, kind, out, what="", chunk=2048):
    """_check_fwd over every token, in chunks of the oracle; merged reports."""
    rqs, rks = [], []
    for s in range(0, wl.T, chunk):
        rq, rk = _check_fwd(wl, kind, out, np.arange(s, min(wl.T, s + chunk)), what=f"{what} tokens {s}+")
        rqs.append(rq)
        rks.append(rk)
    return _merge_reports(rqs), _merge_reports(rks)


# ----------------------------------------------------------- workload 1 ----

def test_tiny_forward_both_layouts(lib, cuda):
    wl = workloads.tiny()
    outs = {}
    for kind in ("interleaved", "sectioned"):
        outs[kind] = _gpu_fwd(lib, wl, kind, cuda)
        rq, rk = _check_fwd(wl, kind, outs[kind], what=f"tiny {kind}")
        print(f"tiny {kind}: q {rq} k {rk}")
    for a, b in zip(outs["interleaved"], outs["sectioned"]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ----------------------------------------------------------- workload 2 ----

def _decode_pools(wl, dev):
    shape = (wl.num_pages, wl.page_size, wl.n_kv, wl.head_dim)
    return (workloads.random_pool_bits(shape, 21, dev), workloads.random_pool_bits(shape, 22, dev))


def _restore_slots(pool, ref, slots):
    out = pool.clone()
    S = pool.shape[0] * pool.shape[1]
    out.view(S, -1)[slots] = ref.view(S, -1)[slots]
    return out


@pytest.mark.parametrize("T", [1, 8, 64, 256])
def test_decode_pool_write(lib, cuda, T):
    wl = workloads.decode_pool(T)
    F = lib.functional
    k0, v0 = _decode_pools(wl, cuda)
    kp, vp = k0.clone(), v0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    page, off = wl.page.to(cuda), wl.offset.to(cuda)
    q = F.prologue_pool_write(wl.packed_rows().to(cuda), wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda),
                              page, off, kp, vp, wl.n_q, wl.n_kv, wl.head_dim, "interleaved", wl.eps,
                              wl.rope_base, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = _oracle_fwd(wl, "interleaved")
    assert_bf16_close(u16(q), ref["q"], "decode q")
    slots = (wl.page.long() * wl.page_size + wl.offset.long()).to(cuda)
    S = wl.num_pages * wl.page_size
    assert_bf16_close(u16(kp.view(S, -1)[slots]), ref["k"], "decode k pool")
    assert np.array_equal(u16(vp.view(S, -1)[slots]).reshape(ref["v_bits"].shape), ref["v_bits"])
    # every other pool byte is untouched
    assert torch.equal(_restore_slots(kp, k0, slots).view(torch.int16), k0.view(torch.int16))
    assert torch.equal(_restore_slots(vp, v0, slots).view(torch.int16), v0.view(torch.int16))


@pytest.mark.parametrize("T", [1, 8, 64, 256])
@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_direct_pool_write_equals_staged(lib, cuda, T, kind):
    wl = workloads.decode_pool(T)
    F, C = lib.functional, lib
    k0, v0 = _decode_pools(wl, cuda)
    packed = _rows(wl, kind).to(cuda)
    pos, wq, wk = wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda)
    page, off = wl.page.to(cuda), wl.offset.to(cuda)
    kd, vd = k0.clone(), v0.clone()
    qd = F.prologue_pool_write(packed, pos, wq, wk, page, off, kd, vd, wl.n_q, wl.n_kv, 64, kind, wl.eps,
                               wl.rope_base)
    q, k, v = F.prologue_forward(packed, pos, wq, wk, wl.n_q, wl.n_kv, 64, kind, wl.eps, wl.rope_base)
    ks, vs = k0.clone(), v0.clone()
    L = C.layout(kind, wl.n_q, wl.n_kv, 64)
    C.qkv_prologue_pool_scatter(L, T, k, v, page, off, ks, vs, wl.num_pages, wl.page_size)
    torch.cuda.synchronize()
    assert torch.equal(qd.view(torch.int16), q.view(torch.int16))
    assert torch.equal(kd.view(torch.int16), ks.view(torch.int16))
    assert torch.equal(vd.view(torch.int16), vs.view(torch.int16))


def test_pool_write_bad_indices_set_status_and_skip(lib, cuda):
    wl = workloads.decode_pool(8, num_pages=16, page_size=64)
    F = lib.functional
    k0, v0 = _decode_pools(wl, cuda)
    page, off = wl.page.clone(), wl.offset.clone()
    page[2] = 16        # page out of range
    off[5] = -1         # offset out of range
    kp, vp = k0.clone(), v0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    F.prologue_pool_write(wl.packed_rows().to(cuda), wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda),
                          page.to(cuda), off.to(cuda), kp, vp, wl.n_q, wl.n_kv, 64, "interleaved", wl.eps,
                          wl.rope_base, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.QKVP_DEV_BAD_PAGE | lib.QKVP_DEV_BAD_OFFSET
    good = [t for t in range(8) if t not in (2, 5)]
    slots = torch.tensor([int(page[t]) * 64 + int(off[t]) for t in good], device=cuda)
    assert torch.equal(_restore_slots(kp, k0, slots).view(torch.int16), k0.view(torch.int16))
    ref = _oracle_fwd(wl, "interleaved")
    assert_bf16_close(u16(kp.view(16 * 64, -1)[slots]), ref["k"][good], "k of valid tokens")


# ----------------------------------------------------------- workload 3 ----

@pytest.mark.parametrize("nope", [False, True])
@pytest.mark.parametrize("T", [2048, 16384])
def test_prefill(lib, cuda, T, nope):
    wl = workloads.prefill(T, nope=nope)
    out = _gpu_fwd(lib, wl, "interleaved", cuda)
    torch.cuda.synchronize()
    rq, rk = _check_fwd_all(wl, "interleaved", out, what=f"prefill T={T} nope={nope}")  # every token
    print(f"prefill T={T} nope={nope}: q {rq} k {rk}")
    # at full size: v is the packed v slots, bit for bit, for every token
    packed = wl.packed.to(cuda)
    assert torch.equal(out[2].view(torch.int16), packed[:, :, 9, :].view(torch.int16))


def test_nope_equals_rope_at_position_zero_gpu(lib, cuda):
    wl = workloads.prefill(2048, nope=False)
    wl.pos = torch.zeros_like(wl.pos)
    a = _gpu_fwd(lib, wl, "interleaved", cuda, nope=False)
    b = _gpu_fwd(lib, wl, "interleaved", cuda, nope=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


# ----------------------------------------------------------- workload 4 ----

def _oracle_bwd_chunked(wl, kind, tokens, chunk=512):
    """dpacked of the sampled tokens, dw over all tokens (sum of per-chunk fp64 sums)."""
    L = _layout(wl, kind)
    xq, xk, _ = P.split_heads(L, u16(_rows(wl, kind)))
    dq, dk, dv = u16(wl.dq), u16(wl.dk), u16(wl.dv)
    pos = wl.pos.numpy()
    wq, wk = wl.w_q.numpy(), wl.w_k.numpy()
    dw_q = np.zeros(wl.head_dim)
    dw_k = np.zeros(wl.head_dim)
    for s in range(0, wl.T, chunk):
        sl = slice(s, min(wl.T, s + chunk))
        r = P.prologue_bwd(L, dq[sl], dk[sl], dv[sl], xq[sl], xk[sl], pos[sl], wq, wk, wl.eps, wl.rope_base,
                           wl.nope)
        dw_q += r["dw_q"]
        dw_k += r["dw_k"]
    r = P.prologue_bwd(L, dq[tokens], dk[tokens], dv[tokens], xq[tokens], xk[tokens], pos[tokens], wq, wk,
                       wl.eps, wl.rope_base, wl.nope)
    return r["dpacked"], dw_q, dw_k


def _check_bwd_all(wl, kind, dpacked, dw_q, dw_k, what="", chunk=2048):
    """The packed gradient of every token (element by element, R9) and dw over
    all tokens (R10), the oracle run chunk by chunk (dw: sum of the chunks'
    float64 sums)."""
    L = _layout(wl, kind)
    xq, xk, _ = P.split_heads(L, u16(_rows(wl, kind)))
    dq, dk, dv = u16(wl.dq), u16(wl.dk), u16(wl.dv)
    pos, wq, wk = wl.pos.numpy(), wl.w_q.numpy(), wl.w_k.numpy()
    got = u16(dpacked)
    dwq_ref, dwk_ref = np.zeros(wl.head_dim), np.zeros(wl.head_dim)
    reports = []
    for s in range(0, wl.T, chunk):
        sl = slice(s, min(wl.T, s + chunk))
        r = P.prologue_bwd(L, dq[sl], dk[sl], dv[sl], xq[sl], xk[sl], pos[sl], wq, wk, wl.eps, wl.rope_base,
                           wl.nope)
        reports.append(assert_bf16_close(got[sl], r["dpacked"], f"{what} dpacked tokens {s}+"))
        dwq_ref += r["dw_q"]
        dwk_ref += r["dw_k"]
    eq = assert_dw_close(dw_q.cpu().numpy(), dwq_ref, f"{what} dw_q")
    ek = assert_dw_close(dw_k.cpu().numpy(), dwk_ref, f"{what} dw_k")
    return _merge_reports(reports), eq, ek


@pytest.mark.parametrize("T,kind", [(4096, "interleaved"), (16384, "interleaved"), (16384, "sectioned")])
def test_train_forward_backward(lib, cuda, T, kind):
    # every token of the forward (q, k, v, the pre-norm save) and of the packed
    # gradient against the oracle, dw over all tokens
    wl = workloads.train(T)
    F = lib.functional
    out = _gpu_fwd(lib, wl, kind, cuda, save=True)
    q, k, v, q_pre, k_pre = out
    dpacked, dw_q, dw_k = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), q_pre, k_pre,
                                              wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), wl.n_q,
                                              wl.n_kv, 64, kind, wl.eps, wl.rope_base)
    torch.cuda.synchronize()
    assert lib.qkv_prologue_device_error(clear=False) == 0
    rq, rk = _check_fwd_all(wl, kind, out, what=f"train fwd T={T} {kind}")
    r, eq, ek = _check_bwd_all(wl, kind, dpacked, dw_q, dw_k, what=f"train bwd T={T} {kind}")
    print(f"train T={T} {kind}: q {rq} k {rk} dpacked {r} dw_q err {eq:.2e} dw_k err {ek:.2e}")
    # v slots of the packed gradient carry dv bit for bit, for every token
    L = _layout(wl, kind)
    _, _, dv_slots = P.split_heads(L, u16(dpacked))
    assert np.array_equal(dv_slots, u16(wl.dv))


@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
@pytest.mark.parametrize("nope", [False, True])
def test_backward_small_full_compare(lib, cuda, kind, nope):
    wl = workloads.gqa_inputs(37, 8, 2, 64, seed=41, rope_base=1e4, nope=nope, with_grads=True)
    F = lib.functional
    q, k, v, q_pre, k_pre = _gpu_fwd(lib, wl, kind, cuda, save=True)
    dp, dwq, dwk = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), q_pre, k_pre,
                                       wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), 8, 2, 64, kind,
                                       wl.eps, wl.rope_base, nope)
    torch.cuda.synchronize()
    ref_dp, ref_dwq, ref_dwk = _oracle_bwd_chunked(wl, kind, np.arange(wl.T))
    assert_bf16_close(u16(dp), ref_dp, "dpacked")
    assert_dw_close(dwq.cpu().numpy(), ref_dwq, "dw_q")
    assert_dw_close(dwk.cpu().numpy(), ref_dwk, "dw_k")


def test_backward_deterministic_and_accumulate(lib, cuda):
    wl = workloads.train(4096)
    C = lib
    q, k, v, q_pre, k_pre = _gpu_fwd(lib, wl, "interleaved", cuda, save=True)
    L = C.layout("interleaved", 128, 16, 64)
    T = wl.T
    need = C.qkv_prologue_bwd_workspace_size(L, T)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda)
    args = [wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), q_pre, k_pre, wl.pos.to(cuda), wl.w_q.to(cuda),
            wl.w_k.to(cuda)]
    res = []
    for _ in range(2):
        dp = torch.empty(T, 10240, dtype=torch.bfloat16, device=cuda)
        dwq = torch.empty(64, device=cuda)
        dwk = torch.empty(64, device=cuda)
        C.qkv_prologue_bwd(L, T, *args, wl.eps, wl.rope_base, 0, dp, dwq, dwk, ws, need)
        res.append((dp, dwq, dwk))
    torch.cuda.synchronize()
    for a, b in zip(*res):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    dwq0 = torch.full((64,), 0.5, device=cuda)
    dwk0 = torch.full((64,), -2.0, device=cuda)
    dp = torch.empty(T, 10240, dtype=torch.bfloat16, device=cuda)
    C.qkv_prologue_bwd(L, T, *args, wl.eps, wl.rope_base, C.QKVP_ACCUMULATE_DW, dp, dwq0, dwk0, ws, need)
    torch.cuda.synchronize()
    want_q = (res[0][1].double() + 0.5).float()
    want_k = (res[0][2].double() - 2.0).float()
    assert torch.allclose(dwq0, want_q, rtol=1e-6, atol=1e-5) and torch.allclose(dwk0, want_k, rtol=1e-6, atol=1e-5)


def test_autograd_function_matches_direct_calls(lib, cuda):
    wl = workloads.train(512)
    F = lib.functional
    packed = wl.packed_rows().to(cuda).requires_grad_(True)
    wq = wl.w_q.to(cuda).requires_grad_(True)
    wk = wl.w_k.to(cuda).requires_grad_(True)
    pos = wl.pos.to(cuda)
    q, k, v = F.QKVPrologue.apply(packed, pos, wq, wk, 128, 16, 64, "interleaved", wl.eps, wl.rope_base, False)
    torch.autograd.backward([q, k, v], [wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda)])
    q2, k2, v2, qp_, kp_ = _gpu_fwd(lib, wl, "interleaved", cuda, save=True)
    dp, dwq, dwk = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), qp_, kp_, pos,
                                       wl.w_q.to(cuda), wl.w_k.to(cuda), 128, 16, 64, "interleaved", wl.eps,
                                       wl.rope_base)
    for a, b in ((q, q2), (k, k2), (v, v2), (packed.grad, dp)):
        assert torch.equal(a.detach().view(torch.int16), b.view(torch.int16))
    assert torch.equal(wq.grad, dwq) and torch.equal(wk.grad, dwk)


# ----------------------------------------------------------- workload 5 ----

@pytest.mark.parametrize("T", [16, 64, 32768])
def test_mla_pool_write(lib, cuda, T):
    wl = workloads.mla(T)
    F, C = lib.functional, lib
    W = wl.norm_dim + wl.rope_dim
    pool0 = workloads.random_pool_bits((wl.num_pages, wl.page_size, W), 51, cuda)
    rows, pos, w = wl.rows.to(cuda), wl.pos.to(cuda), wl.w.to(cuda)
    page, off = wl.page.to(cuda), wl.offset.to(cuda)
    direct = pool0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    F.latent_pool_write(rows, pos, w, page, off, direct, wl.eps, wl.rope_base, dev_status=status)
    staged_rows = F.latent_rows(rows, pos, w, wl.eps, wl.rope_base)
    staged = pool0.clone()
    C.qkv_prologue_pool_scatter(C.layout("latent", norm_dim=512, rope_dim=64), T, staged_rows, None, page, off,
                                staged, None, wl.num_pages, wl.page_size)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # (i) the direct write is bitwise the staged norm+RoPE + scatter
    assert torch.equal(direct.view(torch.int16), staged.view(torch.int16))
    # (ii) both within one bf16 ulp of the fp64 oracle
    slots = (wl.page.long() * wl.page_size + wl.offset.long()).to(cuda)
    exact = oracle.mla_rows(u16(wl.rows), wl.pos.numpy(), wl.w.numpy(), wl.eps, wl.rope_base)  # every row
    got = u16(direct.view(-1, W)[slots])
    r = assert_bf16_close(got, exact, f"mla T={T}")
    print(f"mla T={T}: {r}")
    # (iii) untouched bytes
    assert torch.equal(_restore_slots(direct, pool0, slots).view(torch.int16), pool0.view(torch.int16))


# ------------------------------------------------------------ edge cases ----

def test_empty_batch_is_a_no_op(lib, cuda):
    C = lib
    L = C.layout("interleaved", 8, 2, 64)
    buf = torch.full((4, 768), 1.0, dtype=torch.bfloat16, device=cuda)
    w = torch.ones(64, device=cuda)
    pos = torch.zeros(4, dtype=torch.int32, device=cuda)
    assert C.qkv_prologue_fwd(L, 0, buf, pos, w, w, 1e-6, 1e4, 0, buf, buf, buf) == 0
    dwq = torch.full((64,), 7.0, device=cuda)
    dwk = torch.full((64,), 7.0, device=cuda)
    assert C.qkv_prologue_bwd(L, 0, buf, buf, buf, buf, buf, pos, w, w, 1e-6, 1e4, C.QKVP_ACCUMULATE_DW, buf,
                              dwq, dwk, None, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(buf == 1.0) and torch.all(dwq == 7.0)
    assert C.qkv_prologue_bwd(L, 0, buf, buf, buf, buf, buf, pos, w, w, 1e-6, 1e4, 0, buf, dwq, dwk, None, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(dwq == 0.0) and torch.all(dwk == 0.0)


@pytest.mark.parametrize("T", [1, 3, 17, 333, 2731])
@pytest.mark.parametrize("kind", ["interleaved", "sectioned"])
def test_ragged_token_counts(lib, cuda, T, kind):
    # 8 q over 2 kv: 96 chunks per token, so work items straddle tokens
    wl = workloads.gqa_inputs(T, 8, 2, 64, seed=T, rope_base=1e4, pos_high=393216, with_grads=True)
    F = lib.functional
    out = _gpu_fwd(lib, wl, kind, cuda, save=True)
    dp, dwq, dwk = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), out[3], out[4],
                                       wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), 8, 2, 64, kind,
                                       wl.eps, wl.rope_base)
    torch.cuda.synchronize()
    _check_fwd(wl, kind, out, what=f"ragged T={T}")
    ref_dp, ref_dwq, ref_dwk = _oracle_bwd_chunked(wl, kind, np.arange(T))
    assert_bf16_close(u16(dp), ref_dp, "dpacked")
    assert_dw_close(dwq.cpu().numpy(), ref_dwq, "dw_q")
    assert_dw_close(dwk.cpu().numpy(), ref_dwk, "dw_k")


@pytest.mark.parametrize("shape", [(32, 8, 128), (64, 8, 64), (16, 16, 128), (6, 1, 64)])
def test_other_head_shapes(lib, cuda, shape):
    n_q, n_kv, D = shape
    wl = workloads.gqa_inputs(129, n_q, n_kv, D, seed=7, rope_base=5e5, pos_high=131072, with_grads=True)
    F = lib.functional
    for kind in ("interleaved", "sectioned"):
        out = _gpu_fwd(lib, wl, kind, cuda, save=True)
        dp, dwq, dwk = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), out[3], out[4],
                                           wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), n_q, n_kv, D,
                                           kind, wl.eps, wl.rope_base)
        torch.cuda.synchronize()
        _check_fwd(wl, kind, out, what=f"{shape} {kind}")
        ref_dp, ref_dwq, ref_dwk = _oracle_bwd_chunked(wl, kind, np.arange(wl.T))
        assert_bf16_close(u16(dp), ref_dp, "dpacked")
        assert_dw_close(dwq.cpu().numpy(), ref_dwq, "dw_q")
        assert_dw_close(dwk.cpu().numpy(), ref_dwk, "dw_k")


@pytest.mark.parametrize("nope", [False, True])
@pytest.mark.parametrize("shape,T", [((24, 2, 64), 3), ((24, 2, 64), 129), ((16, 8, 64), 3), ((16, 8, 64), 129),
                                     ((128, 16, 64), 333)])
def test_two_step_backward_with_tail_tiles(lib, cuda, shape, T, nope):
    # head_dim 64 rows of 112 / 128 chunk pairs: with one CTA of 10 consumer warps
    # per SM (228 KiB of shared memory) the planner takes 5-token tiles of two steps
    # per thread (the instance that keeps its weight-gradient sums per step), the
    # second step 87.5 % / 100 % full; T = 3 and 129 end in a tile with missing
    # tokens. The Muse Spark rows (640 chunk pairs) take the same instance on
    # 1-token tiles. RoPE and NoPE layers.
    n_q, n_kv, D = shape
    wl = workloads.gqa_inputs(T, n_q, n_kv, D, seed=11 + T, rope_base=5e5, pos_high=131072, nope=nope,
                              with_grads=True)
    F = lib.functional
    for kind in ("interleaved", "sectioned"):
        out = _gpu_fwd(lib, wl, kind, cuda, save=True)
        dp, dwq, dwk = F.prologue_backward(wl.dq.to(cuda), wl.dk.to(cuda), wl.dv.to(cuda), out[3], out[4],
                                           wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), n_q, n_kv, D,
                                           kind, wl.eps, wl.rope_base, nope)
        torch.cuda.synchronize()
        ref_dp, ref_dwq, ref_dwk = _oracle_bwd_chunked(wl, kind, np.arange(wl.T))
        assert_bf16_close(u16(dp), ref_dp, f"dpacked {shape} {kind} T={T} nope={nope}")
        assert_dw_close(dwq.cpu().numpy(), ref_dwq, "dw_q")
        assert_dw_close(dwk.cpu().numpy(), ref_dwk, "dw_k")


def test_padded_rows_and_guard_bands(lib, cuda):
    C = lib
    wl = workloads.gqa_inputs(50, 8, 2, 64, seed=3, rope_base=1e4, pos_high=1000)
    T, W, stride = wl.T, 768, 768 + 64
    rows = torch.full((T, stride), 3.0, dtype=torch.bfloat16)
    rows[:, :W] = wl.packed_rows()
    rows = rows.to(cuda)
    guard = 4096
    sentinel = -12345
    bufs = [torch.full((guard + n + guard,), sentinel, dtype=torch.int16, device=cuda) for n in (T * 512, T * 128, T * 128)]
    q, k, v = (b[guard:-guard].view(torch.bfloat16) for b in bufs)
    L = C.layout("interleaved", 8, 2, 64, row_stride=stride)
    C.qkv_prologue_fwd(L, T, rows, wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), wl.eps, wl.rope_base, 0,
                       q, k, v)
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:guard] == sentinel) and torch.all(b[-guard:] == sentinel)
    _check_fwd(wl, "interleaved", (q.view(T, 8, 64), k.view(T, 2, 64), v.view(T, 2, 64)), what="padded")


def test_extreme_positions(lib, cuda):
    wl = workloads.gqa_inputs(64, 8, 2, 64, seed=9, rope_base=5e5)
    wl.pos = torch.tensor([0, 1, -1, -393215, 2 ** 31 - 1, -(2 ** 31), 2 ** 24 + 1, 393215] * 8, dtype=torch.int32)
    out = _gpu_fwd(lib, wl, "interleaved", cuda)
    torch.cuda.synchronize()
    r = _check_fwd(wl, "interleaved", out, what="extreme positions")
    print("extreme positions", r)


def test_bf16_reports_are_mostly_exact(lib, cuda):
    # not a bound, a sanity figure: most outputs should round exactly like the oracle
    wl = workloads.prefill(2048)
    out = _gpu_fwd(lib, wl, "interleaved", cuda)
    ref = _oracle_fwd(wl, "interleaved")
    r = bf16_report(u16(out[0]), ref["q"])
    assert r["exact_match"] > 0.97, r

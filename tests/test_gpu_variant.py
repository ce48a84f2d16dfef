"""The GQAttention variant (norm off, qkv bias, caller frequency table, cos/sin
factor) through the C ABI against the fp64 oracle, for the three model shapes
it serves (Llama 3 8B, Qwen3 8B, GPT-OSS 20b attention) and both packings,
on the pipelined and the general kernels."""

import numpy as np
import pytest
import torch

import oracle.prologue as P
import workloads
from parity import DW_REL, assert_bf16_close, assert_dw_close
from workloads import bits_u16 as u16

pytestmark = pytest.mark.gpu

KINDS = ["interleaved", "sectioned"]
MODELS = {
    "llama3": workloads.llama3,
    "qwen3": workloads.qwen3,
    "gpt_oss": workloads.gpt_oss,
}


def _layout(wl, kind):
    return P.PackedLayout(kind, wl.n_q, wl.n_kv, wl.head_dim)


def _rows(wl, kind):
    return wl.packed_rows() if kind == "interleaved" else wl.sectioned_rows()


def _dev_opts(wl, kind, dev):
    o = wl.variant(kind)
    if o["bias"] is not None:
        o["bias"] = o["bias"].to(dev)
    return o


def _oracle_opts(wl, kind):
    o = wl.variant(kind)
    if o["bias"] is not None:
        o["bias"] = o["bias"].numpy().astype(np.float64)
    return o


def _gpu_fwd(lib, wl, kind, dev, save=None, generic=False):
    C, F = lib, lib.functional
    save = wl.norm if save is None else save
    opts = _dev_opts(wl, kind, dev)
    rows = _rows(wl, kind).to(dev)
    wq = wl.w_q.to(dev) if wl.norm else None
    wk = wl.w_k.to(dev) if wl.norm else None
    if not generic:
        return F.prologue_forward(rows, wl.pos.to(dev), wq, wk, wl.n_q, wl.n_kv, wl.head_dim, kind, wl.eps,
                                  wl.rope_base, wl.nope, save_pre=save, **opts)
    # the general kernels, through the C call with QKVP_FORCE_GENERIC
    T, D = wl.T, wl.head_dim
    bf = dict(dtype=torch.bfloat16, device=dev)
    q, k, v = torch.empty(T, wl.n_q, D, **bf), torch.empty(T, wl.n_kv, D, **bf), torch.empty(T, wl.n_kv, D, **bf)
    qp = torch.empty_like(q) if save else None
    kp = torch.empty_like(k) if save else None
    V = C.variant(inv_freq=opts["inv_freq"], rope_scale=opts["rope_scale"], bias=opts["bias"])
    flags = (C.QKVP_NOPE if wl.nope else 0) | (C.QKVP_SAVE_PRE if save else 0) | \
        (0 if wl.norm else C.QKVP_NORM_OFF) | C.QKVP_FORCE_GENERIC
    C.qkv_prologue_fwd_ex(C.layout(kind, wl.n_q, wl.n_kv, D), V, T, rows, wl.pos.to(dev), wq, wk, wl.eps,
                          wl.rope_base, flags, q, k, v, qp, kp)
    return (q, k, v, qp, kp) if save else (q, k, v)


def _oracle_fwd(wl, kind, tokens=None):
    rows, pos = u16(_rows(wl, kind)), wl.pos.numpy()
    if tokens is not None:
        rows, pos = rows[tokens], pos[tokens]
    return P.prologue_fwd(_layout(wl, kind), rows, pos, wl.w_q.numpy(), wl.w_k.numpy(), wl.eps, wl.rope_base,
                          wl.nope, **_oracle_opts(wl, kind))


def _check_fwd(wl, kind, out, tokens=None, what=""):
    pick = (lambda a: a) if tokens is None else (lambda a: a[tokens])
    q, k, v = (pick(u16(t)) for t in out[:3])
    ref = _oracle_fwd(wl, kind, tokens)
    assert_bf16_close(q, ref["q"], f"{what} q")
    assert_bf16_close(k, ref["k"], f"{what} k")
    if wl.bias is None:
        assert np.array_equal(v, ref["v_bits"]), f"{what}: v is not a bit copy"
    else:
        assert_bf16_close(v, ref["v"], f"{what} v (biased)")
    if len(out) == 5:  # the saved inputs are the input heads, before any bias
        assert np.array_equal(pick(u16(out[3])), ref["q_pre_bits"])
        assert np.array_equal(pick(u16(out[4])), ref["k_pre_bits"])


def _same_bits(a, b, what):
    for x, y in zip(a, b):
        if x is None:
            assert y is None
            continue
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), what


# ---------------------------------------------------------------- forward ----

@pytest.mark.parametrize("model", list(MODELS))
@pytest.mark.parametrize("kind", KINDS)
def test_variant_forward(lib, cuda, model, kind):
    wl = MODELS[model](131, pos_high=393216, with_grads=False)
    out = _gpu_fwd(lib, wl, kind, cuda)
    gen = _gpu_fwd(lib, wl, kind, cuda, generic=True)
    torch.cuda.synchronize()
    _check_fwd(wl, kind, out, what=f"{model} {kind}")
    # the pipelined and the general kernels give the same bits
    _same_bits(out, gen, f"{model} {kind}: pipelined != general")


@pytest.mark.parametrize("kind", KINDS)
def test_each_option_alone(lib, cuda, kind):
    # the Muse Spark shape with one option at a time, then all of them together
    base = dict(T=77, n_q=128, n_kv=16, head_dim=64, seed=51, rope_base=5e5, pos_high=131072)
    g = workloads._gen(52)
    bias = workloads.qkv_bias((128 + 32) * 64, g)
    table = workloads.llama3_inv_freq(64)
    cases = {
        "norm off": dict(norm=False),
        "norm off, NoPE (a pure split)": dict(norm=False, nope=True),
        "bias, norm on": dict(bias=bias),
        "bias, norm on, NoPE": dict(bias=bias, nope=True),
        "table": dict(inv_freq=table),
        "factor": dict(rope_scale=1.3465735902799727),
        "all": dict(norm=False, bias=bias, inv_freq=table, rope_scale=0.75),
    }
    for name, opts in cases.items():
        wl = workloads.gqa_inputs(base["T"], base["n_q"], base["n_kv"], base["head_dim"], base["seed"],
                                  base["rope_base"], pos_high=base["pos_high"], nope=opts.get("nope", False))
        wl.norm = opts.get("norm", True)
        wl.bias = opts.get("bias")
        wl.inv_freq = opts.get("inv_freq")
        wl.rope_scale = opts.get("rope_scale", 1.0)
        out = _gpu_fwd(lib, wl, kind, cuda)
        gen = _gpu_fwd(lib, wl, kind, cuda, generic=True)
        torch.cuda.synchronize()
        _check_fwd(wl, kind, out, what=f"{name} {kind}")
        _same_bits(out, gen, f"{name} {kind}: pipelined != general")
        if name.startswith("norm off, NoPE"):
            # no norm, no rotation: q and k are the input heads bit for bit
            ref = _oracle_fwd(wl, kind)
            assert np.array_equal(u16(out[0]), ref["q_pre_bits"]) and np.array_equal(u16(out[1]), ref["k_pre_bits"])


def test_plain_options_equal_the_plain_call(lib, cuda):
    # default table passed explicitly, factor 1: the plain call's bits
    wl = workloads.train(300)
    F = lib.functional
    a = F.prologue_forward(wl.packed_rows().to(cuda), wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), 128, 16)
    b = F.prologue_forward(wl.packed_rows().to(cuda), wl.pos.to(cuda), wl.w_q.to(cuda), wl.w_k.to(cuda), 128, 16,
                           inv_freq=P.rope_inv_freq(64, 500000.0), rope_scale=1.0)
    torch.cuda.synchronize()
    _same_bits(a, b, "explicit default table changed the result")


# ------------------------------------------------------------- pool write ----

@pytest.mark.parametrize("model", ["llama3", "gpt_oss"])
@pytest.mark.parametrize("T", [1, 64])
def test_variant_pool_write(lib, cuda, model, T):
    wl = MODELS[model](T, pos_high=131072, with_grads=False)
    num_pages, page_size = 512, 64
    page, off = workloads.random_slots(T, num_pages, page_size, workloads._gen(900 + T))
    shape = (num_pages, page_size, wl.n_kv, wl.head_dim)
    k0, v0 = workloads.random_pool_bits(shape, 31, cuda), workloads.random_pool_bits(shape, 32, cuda)
    kp, vp = k0.clone(), v0.clone()
    F = lib.functional
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    q = F.prologue_pool_write(wl.packed_rows().to(cuda), wl.pos.to(cuda), None, None, page.to(cuda), off.to(cuda),
                              kp, vp, wl.n_q, wl.n_kv, wl.head_dim, "interleaved", wl.eps, wl.rope_base,
                              dev_status=status, **_dev_opts(wl, "interleaved", cuda))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = _oracle_fwd(wl, "interleaved")
    assert_bf16_close(u16(q), ref["q"], "pool q")
    slots = (page.long() * page_size + off.long()).to(cuda)
    S = num_pages * page_size
    assert_bf16_close(u16(kp.view(S, -1)[slots]), ref["k"], "k pool")
    if wl.bias is None:
        assert np.array_equal(u16(vp.view(S, -1)[slots]).reshape(ref["v_bits"].shape), ref["v_bits"])
    else:
        assert_bf16_close(u16(vp.view(S, -1)[slots]), ref["v"], "v pool (biased)")
    for pool, orig in ((kp, k0), (vp, v0)):
        restored = pool.clone()
        restored.view(S, -1)[slots] = orig.view(S, -1)[slots]
        assert torch.equal(restored.view(torch.int16), orig.view(torch.int16))


# --------------------------------------------------------------- backward ----

def _gpu_bwd(lib, wl, kind, dev, saved, generic=False, accumulate_into=None):
    C = lib
    T, D = wl.T, wl.head_dim
    opts = _dev_opts(wl, kind, dev)
    V = C.variant(inv_freq=opts["inv_freq"], rope_scale=opts["rope_scale"], bias=opts["bias"])
    L = C.layout(kind, wl.n_q, wl.n_kv, D)
    W = wl.row_width
    dp = torch.empty(T, W, dtype=torch.bfloat16, device=dev)
    if accumulate_into is not None:
        dwq, dwk, db = accumulate_into
    else:
        dwq = torch.empty(D, device=dev) if wl.norm else None
        dwk = torch.empty(D, device=dev) if wl.norm else None
        db = torch.empty(W, device=dev) if wl.bias is not None else None
    need = C.qkv_prologue_bwd_workspace_size_ex(L, V, T)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    flags = (C.QKVP_NOPE if wl.nope else 0) | (0 if wl.norm else C.QKVP_NORM_OFF) | \
        (C.QKVP_FORCE_GENERIC if generic else 0) | (C.QKVP_ACCUMULATE_DW if accumulate_into is not None else 0)
    qp, kp = saved if wl.norm else (None, None)
    C.qkv_prologue_bwd_ex(L, V, T, wl.dq.to(dev), wl.dk.to(dev), wl.dv.to(dev), qp, kp, wl.pos.to(dev),
                          wl.w_q.to(dev) if wl.norm else None, wl.w_k.to(dev) if wl.norm else None, wl.eps,
                          wl.rope_base, flags, dp, dwq, dwk, db, ws, need)
    return dp, dwq, dwk, db


def _oracle_bwd(wl, kind, tokens, chunk=512):
    """dpacked of the sampled tokens; dw and db over all tokens (sums of per-chunk fp64 sums)."""
    L = _layout(wl, kind)
    xq, xk, _ = P.split_heads(L, u16(_rows(wl, kind)))
    dq, dk, dv = u16(wl.dq), u16(wl.dk), u16(wl.dv)
    pos, opts = wl.pos.numpy(), _oracle_opts(wl, kind)
    wq, wk = wl.w_q.numpy(), wl.w_k.numpy()
    dwq, dwk, db = np.zeros(wl.head_dim), np.zeros(wl.head_dim), np.zeros(wl.row_width)
    for s in range(0, wl.T, chunk):
        sl = slice(s, min(wl.T, s + chunk))
        r = P.prologue_bwd(L, dq[sl], dk[sl], dv[sl], xq[sl], xk[sl], pos[sl], wq, wk, wl.eps, wl.rope_base,
                           wl.nope, **opts)
        dwq += r["dw_q"]
        dwk += r["dw_k"]
        if r["db"] is not None:
            db += r["db"]
    r = P.prologue_bwd(L, dq[tokens], dk[tokens], dv[tokens], xq[tokens], xk[tokens], pos[tokens], wq, wk, wl.eps,
                       wl.rope_base, wl.nope, **opts)
    return r["dpacked"], dwq, dwk, db


def _check_bwd(wl, kind, got, tokens, what):
    dp, dwq, dwk, db = got
    ref_dp, ref_dwq, ref_dwk, ref_db = _oracle_bwd(wl, kind, tokens)
    assert_bf16_close(u16(dp)[tokens], ref_dp, f"{what} dpacked")
    if wl.norm:
        assert_dw_close(dwq.cpu().numpy(), ref_dwq, f"{what} dw_q")
        assert_dw_close(dwk.cpu().numpy(), ref_dwk, f"{what} dw_k")
    if wl.bias is not None:
        assert_dw_close(db.cpu().numpy(), ref_db, f"{what} db")


@pytest.mark.parametrize("model", list(MODELS))
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("T", [1, 257])
def test_variant_backward(lib, cuda, model, kind, T):
    wl = MODELS[model](T, pos_high=393216)
    out = _gpu_fwd(lib, wl, kind, cuda, save=wl.norm)
    saved = out[3:5] if wl.norm else None
    got = _gpu_bwd(lib, wl, kind, cuda, saved)
    gen = _gpu_bwd(lib, wl, kind, cuda, saved, generic=True)
    torch.cuda.synchronize()
    tokens = np.arange(T)
    _check_bwd(wl, kind, got, tokens, f"{model} {kind} T={T}")
    _check_bwd(wl, kind, gen, tokens, f"{model} {kind} T={T} general")
    # the packed gradient has the same bits on both paths; the sums may round differently
    assert torch.equal(got[0].view(torch.int16), gen[0].view(torch.int16))


@pytest.mark.parametrize("kind", KINDS)
def test_bias_backward_with_norm(lib, cuda, kind):
    # bias and norm together: the norm backward must see x + b (Muse Spark shape)
    wl = workloads.gqa_inputs(129, 128, 16, 64, seed=61, rope_base=5e5, pos_high=131072, with_grads=True)
    wl.bias = workloads.qkv_bias(wl.row_width, workloads._gen(62))
    q, k, v, qp, kp = _gpu_fwd(lib, wl, kind, cuda, save=True)
    got = _gpu_bwd(lib, wl, kind, cuda, (qp, kp))
    gen = _gpu_bwd(lib, wl, kind, cuda, (qp, kp), generic=True)
    torch.cuda.synchronize()
    _check_fwd(wl, kind, (q, k, v, qp, kp), what=f"bias+norm {kind}")
    _check_bwd(wl, kind, got, np.arange(wl.T), f"bias+norm {kind}")
    _check_bwd(wl, kind, gen, np.arange(wl.T), f"bias+norm {kind} general")
    assert torch.equal(got[0].view(torch.int16), gen[0].view(torch.int16))


def test_variant_backward_deterministic_and_accumulate(lib, cuda):
    wl = workloads.gpt_oss(1000)
    a = _gpu_bwd(lib, wl, "sectioned", cuda, None)
    b = _gpu_bwd(lib, wl, "sectioned", cuda, None)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[3], b[3])  # the bias gradient: same bits every run
    acc = a[3].clone()
    _gpu_bwd(lib, wl, "sectioned", cuda, None, accumulate_into=(None, None, acc))
    torch.cuda.synchronize()
    ref = (a[3].double() * 2).float()
    assert torch.allclose(acc, ref, rtol=1e-6, atol=1e-6)


def _check_bwd_all(wl, kind, got, what, chunk=2048):
    """The packed gradient of every token (chunk by chunk) and the weight and
    bias gradients over all tokens (sums of the chunks' float64 sums)."""
    dp, dwq, dwk, db = got
    L = _layout(wl, kind)
    xq, xk, _ = P.split_heads(L, u16(_rows(wl, kind)))
    dq, dk, dv = u16(wl.dq), u16(wl.dk), u16(wl.dv)
    pos, opts = wl.pos.numpy(), _oracle_opts(wl, kind)
    wq, wk = wl.w_q.numpy(), wl.w_k.numpy()
    got_dp = u16(dp)
    rq, rk, rb = np.zeros(wl.head_dim), np.zeros(wl.head_dim), np.zeros(wl.row_width)
    for s in range(0, wl.T, chunk):
        sl = slice(s, min(wl.T, s + chunk))
        r = P.prologue_bwd(L, dq[sl], dk[sl], dv[sl], xq[sl], xk[sl], pos[sl], wq, wk, wl.eps, wl.rope_base,
                           wl.nope, **opts)
        assert_bf16_close(got_dp[sl], r["dpacked"], f"{what} dpacked tokens {s}+")
        rq += r["dw_q"]
        rk += r["dw_k"]
        if r["db"] is not None:
            rb += r["db"]
    if wl.norm:
        assert_dw_close(dwq.cpu().numpy(), rq, f"{what} dw_q")
        assert_dw_close(dwk.cpu().numpy(), rk, f"{what} dw_k")
    if wl.bias is not None:
        assert_dw_close(db.cpu().numpy(), rb, f"{what} db")


@pytest.mark.parametrize("model", list(MODELS))
def test_variant_train_full_size(lib, cuda, model):
    # the bench's training step (T = 16384, sectioned rows): every token of the
    # forward and of the packed gradient against the oracle, sums over all tokens
    T = 16384
    wl = MODELS[model](T)
    out = _gpu_fwd(lib, wl, "sectioned", cuda, save=wl.norm)
    got = _gpu_bwd(lib, wl, "sectioned", cuda, out[3:5] if wl.norm else None)
    torch.cuda.synchronize()
    for s in range(0, T, 2048):
        _check_fwd(wl, "sectioned", out, np.arange(s, min(T, s + 2048)), what=f"{model} train fwd tokens {s}+")
    _check_bwd_all(wl, "sectioned", got, f"{model} train bwd")
    if wl.bias is not None:
        # the bias gradient against the written packed gradient: they differ only by
        # dpacked's rounding to bf16 (at most 2^-9 relative per element)
        dps = got[0].double().sum(0).cpu().numpy()
        bound = got[0].double().abs().sum(0).cpu().numpy() * 2.0 ** -8 + DW_REL
        assert np.all(np.abs(got[3].double().cpu().numpy() - dps) <= bound)

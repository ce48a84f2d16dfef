"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any device call.

The argument-check tests pass fake (never dereferenced) addresses, so they only
run where no CUDA device is visible: a check that wrongly passed must not lead
to a kernel launch on fake pointers.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"QKVP_API\s+[\w\s\*]+?\b(qkv_\w+)\s*\(", src))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert {"qkv_prologue_fwd", "qkv_prologue_bwd", "qkv_prologue_pool_write",
            "qkv_prologue_pool_scatter", "qkv_prologue_bwd_workspace_size",
            "qkv_prologue_status_string", "qkv_prologue_version", "qkv_prologue_device_error",
            "qkv_newton_schulz", "qkv_newton_schulz_batch", "qkv_newton_schulz_plan",
            "qkv_newton_schulz_workspace"} <= names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = _declared_functions() - exported
    assert not missing, missing
    # and nothing else of ours leaks out of the library
    ours = {s for s in exported if "qkvp" in s.lower() or s.startswith("qkv_")}
    assert ours == _declared_functions()
    dl = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared_functions():
        assert getattr(dl, name) is not None


def test_binding_exposes_the_same_names(lib):
    for name in _declared_functions():
        assert callable(getattr(lib, name))


def test_version_and_status_strings(lib):
    assert lib.qkv_prologue_version() == lib.QKVP_VERSION == 3
    for code in range(-8, 1):
        s = lib.qkv_prologue_status_string(code)
        assert s and s != "unknown status"
    assert lib.qkv_prologue_status_string(-99) == "unknown status"


def test_constants_match_header(lib):
    src = open(os.path.join(HEADER_DIR, "qkv_prologue.h")).read()
    for name in ("QKVP_OK", "QKVP_ERR_NULL", "QKVP_ERR_SHAPE", "QKVP_ERR_ALIGN", "QKVP_ERR_ARCH",
                 "QKVP_ERR_WORKSPACE", "QKVP_ERR_LAUNCH", "QKVP_ERR_FLAGS", "QKVP_ERR_VALUE",
                 "QKVP_INTERLEAVED", "QKVP_SECTIONED", "QKVP_LATENT", "QKVP_NOPE", "QKVP_SAVE_PRE",
                 "QKVP_ACCUMULATE_DW", "QKVP_FORCE_GENERIC", "QKVP_NORM_OFF", "QKVP_DEV_BAD_PAGE",
                 "QKVP_DEV_BAD_OFFSET"):
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", src)
        assert m, name
        assert int(m.group(1)) == getattr(lib, name), name


def test_variant_struct_matches_c_layout(lib):
    # double* inv_freq; double rope_scale; float* bias
    V = lib.qkvp_variant
    assert ctypes.sizeof(V) == 24
    assert V.inv_freq.offset == 0 and V.rope_scale.offset == 8 and V.bias.offset == 16
    v = lib.variant(inv_freq=[1.0, 0.5], rope_scale=1.25, bias=0x1000)
    assert v.inv_freq[0] == 1.0 and v.inv_freq[1] == 0.5 and v.rope_scale == 1.25 and v.bias == 0x1000


def test_layout_struct_matches_c_layout(lib):
    # int32 kind, n_q, n_kv, head_dim; int64 row_stride; int32 norm_dim, rope_dim
    L = lib.qkvp_layout
    assert ctypes.sizeof(L) == 32
    assert L.row_stride.offset == 16 and L.norm_dim.offset == 24 and L.rope_dim.offset == 28


def test_workspace_size(lib):
    L = lib.layout("interleaved", 128, 16, 64)
    assert lib.qkv_prologue_bwd_workspace_size(L, 0) == 0
    # one partial row [2, 64] fp32 per CTA, at most 1024 rows, then the weight-
    # gradient fold's words: one per possible CTA (1024) and the election word,
    # padded to 16 bytes (4112 bytes)
    fold = 4 * (1024 + 4)
    assert lib.qkv_prologue_bwd_workspace_size(L, 1) == 512 + fold
    for T in range(1, 40):  # at least one row per token up to the cap
        assert lib.qkv_prologue_bwd_workspace_size(L, T) >= 512 * T + fold
    assert lib.qkv_prologue_bwd_workspace_size(L, 16384) == 1024 * 512 + fold
    assert lib.qkv_prologue_bwd_workspace_size(lib.layout("interleaved", 8, 3, 64), 16) == 0
    assert lib.qkv_prologue_bwd_workspace_size(lib.layout("interleaved", 32, 8, 128), 100) > 0


# ----------------------------------------------------- host-side checks ----

def _no_gpu():
    try:
        import torch

        return not torch.cuda.is_available()
    except Exception:
        return True


cpu_only = pytest.mark.skipif(not _no_gpu(), reason="fake-pointer argument checks run only without a GPU")

A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def _fwd(lib, L=None, T=4, packed=A, pos=A, wq=A, wk=A, eps=1e-6, base=1e4, flags=0, q=A, k=A, v=A,
         q_pre=None, k_pre=None):
    L = L or lib.layout("interleaved", 8, 2, 64)
    return lib.qkv_prologue_fwd(L, T, packed, pos, wq, wk, eps, base, flags, q, k, v, q_pre, k_pre, stream=0,
                                check=False)


@cpu_only
def test_fwd_argument_checks(lib):
    C = lib
    assert _fwd(C) == C.QKVP_ERR_ARCH  # valid arguments: it gets as far as the device check
    assert _fwd(C, T=0) == C.QKVP_OK  # empty batch: no device needed
    assert _fwd(C, T=-1) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout("interleaved", 8, 3, 64)) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout("interleaved", 8, 2, 96)) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout("interleaved", 0, 2, 64)) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout(7, 8, 2, 64)) == C.QKVP_ERR_SHAPE
    # the row must hold the exact fused total (n_q + 2 n_kv) * head_dim values
    assert _fwd(C, L=C.layout("interleaved", 8, 2, 64, row_stride=700)) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout("interleaved", 8, 2, 64, row_stride=772)) == C.QKVP_ERR_SHAPE
    assert _fwd(C, L=C.layout("interleaved", 8, 2, 64, row_stride=776)) == C.QKVP_ERR_ARCH
    assert _fwd(C, packed=None) == C.QKVP_ERR_NULL
    assert _fwd(C, q=None) == C.QKVP_ERR_NULL
    assert _fwd(C, pos=None) == C.QKVP_ERR_NULL
    assert _fwd(C, pos=None, flags=C.QKVP_NOPE) == C.QKVP_ERR_ARCH  # NoPE needs no positions
    assert _fwd(C, flags=C.QKVP_SAVE_PRE) == C.QKVP_ERR_NULL
    assert _fwd(C, flags=C.QKVP_SAVE_PRE, q_pre=A, k_pre=A) == C.QKVP_ERR_ARCH
    assert _fwd(C, flags=32) == C.QKVP_ERR_FLAGS
    assert _fwd(C, flags=C.QKVP_FORCE_GENERIC) == C.QKVP_ERR_ARCH
    assert _fwd(C, flags=C.QKVP_ACCUMULATE_DW) == C.QKVP_ERR_FLAGS
    assert _fwd(C, packed=A + 8) == C.QKVP_ERR_ALIGN
    assert _fwd(C, k=A + 2) == C.QKVP_ERR_ALIGN
    assert _fwd(C, pos=A + 2) == C.QKVP_ERR_ALIGN
    assert _fwd(C, eps=-1.0) == C.QKVP_ERR_VALUE
    assert _fwd(C, eps=float("nan")) == C.QKVP_ERR_VALUE
    assert _fwd(C, base=0.0) == C.QKVP_ERR_VALUE
    assert _fwd(C, base=float("inf")) == C.QKVP_ERR_VALUE
    assert _fwd(C, base=0.0, flags=C.QKVP_NOPE) == C.QKVP_ERR_ARCH
    with pytest.raises(C.QkvpError):
        C.qkv_prologue_fwd(C.layout("interleaved", 8, 3, 64), 4, A, A, A, A, 1e-6, 1e4, 0, A, A, A, stream=0)


@cpu_only
def test_latent_argument_checks(lib):
    C = lib
    L = C.layout("latent", norm_dim=512, rope_dim=64)
    ok = dict(L=L, T=4, packed=A, pos=A, wq=None, wk=A, q=None, k=A, v=None)
    assert _fwd(C, **ok) == C.QKVP_ERR_ARCH
    assert _fwd(C, **{**ok, "L": C.layout("latent", norm_dim=500, rope_dim=64)}) == C.QKVP_ERR_SHAPE
    assert _fwd(C, **{**ok, "L": C.layout("latent", norm_dim=512, rope_dim=32)}) == C.QKVP_ERR_SHAPE
    assert _fwd(C, **{**ok, "L": C.layout("latent", norm_dim=2048, rope_dim=64)}) == C.QKVP_ERR_SHAPE
    assert _fwd(C, **{**ok, "wk": None}) == C.QKVP_ERR_NULL
    assert _fwd(C, **{**ok, "flags": C.QKVP_SAVE_PRE}) == C.QKVP_ERR_FLAGS
    pw = C.qkv_prologue_pool_write
    assert pw(L, 4, A, A, None, A, 1e-6, 1e4, 0, None, A, A, A, None, 8192, 64, None, stream=0,
              check=False) == C.QKVP_ERR_ARCH
    assert pw(L, 4, A, A, None, A, 1e-6, 1e4, 0, None, A, A, A, None, 0, 64, None, stream=0,
              check=False) == C.QKVP_ERR_VALUE
    assert pw(L, 4, A, A, None, A, 1e-6, 1e4, 0, None, None, A, A, None, 8192, 64, None, stream=0,
              check=False) == C.QKVP_ERR_NULL


@cpu_only
def test_pool_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 128, 16, 64)

    def pw(**kw):
        a = dict(T=4, packed=A, pos=A, wq=A, wk=A, flags=0, q=A, page=A, off=A, kp=A, vp=A, pages=4096,
                 psize=64, status=None)
        a.update(kw)
        return C.qkv_prologue_pool_write(L, a["T"], a["packed"], a["pos"], a["wq"], a["wk"], 1e-6, 5e5,
                                         a["flags"], a["q"], a["page"], a["off"], a["kp"], a["vp"], a["pages"],
                                         a["psize"], a["status"], stream=0, check=False)

    assert pw() == C.QKVP_ERR_ARCH
    assert pw(vp=None) == C.QKVP_ERR_NULL
    assert pw(page=None) == C.QKVP_ERR_NULL
    assert pw(pages=0) == C.QKVP_ERR_VALUE
    assert pw(psize=-1) == C.QKVP_ERR_VALUE
    assert pw(pages=2 ** 30, psize=64) == C.QKVP_ERR_VALUE
    assert pw(flags=C.QKVP_SAVE_PRE) == C.QKVP_ERR_FLAGS
    assert pw(kp=A + 4) == C.QKVP_ERR_ALIGN
    assert pw(status=A + 1) == C.QKVP_ERR_ALIGN
    sc = C.qkv_prologue_pool_scatter
    assert sc(L, 4, A, A, A, A, A, A, 4096, 64, None, stream=0, check=False) == C.QKVP_ERR_ARCH
    assert sc(L, 4, A, None, A, A, A, A, 4096, 64, None, stream=0, check=False) == C.QKVP_ERR_NULL
    assert sc(L, 0, A, A, A, A, A, A, 4096, 64, None, stream=0, check=False) == C.QKVP_OK


@cpu_only
def test_bwd_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 128, 16, 64)
    need = C.qkv_prologue_bwd_workspace_size(L, 100)

    def bwd(**kw):
        a = dict(L=L, T=100, dq=A, dk=A, dv=A, qp=A, kp=A, pos=A, wq=A, wk=A, flags=0, dp=A, dwq=A, dwk=A,
                 ws=A, wsb=need)
        a.update(kw)
        return C.qkv_prologue_bwd(a["L"], a["T"], a["dq"], a["dk"], a["dv"], a["qp"], a["kp"], a["pos"], a["wq"],
                                  a["wk"], 1e-6, 5e5, a["flags"], a["dp"], a["dwq"], a["dwk"], a["ws"], a["wsb"],
                                  stream=0, check=False)

    assert bwd() == C.QKVP_ERR_ARCH
    assert bwd(wsb=need - 1) == C.QKVP_ERR_WORKSPACE
    assert bwd(ws=None) == C.QKVP_ERR_NULL
    assert bwd(ws=A + 8) == C.QKVP_ERR_ALIGN
    assert bwd(qp=None) == C.QKVP_ERR_NULL
    assert bwd(dwk=None) == C.QKVP_ERR_NULL
    assert bwd(flags=C.QKVP_SAVE_PRE) == C.QKVP_ERR_FLAGS
    assert bwd(flags=C.QKVP_NOPE | C.QKVP_ACCUMULATE_DW, pos=None) == C.QKVP_ERR_ARCH
    assert bwd(L=C.layout("latent", norm_dim=512, rope_dim=64)) == C.QKVP_ERR_SHAPE
    assert bwd(T=0, flags=C.QKVP_ACCUMULATE_DW, ws=None, wsb=0) == C.QKVP_OK
    # T == 0 without ACCUMULATE_DW zeroes dw, which needs the device
    assert bwd(T=0, ws=None, wsb=0) == C.QKVP_ERR_ARCH


@cpu_only
def test_variant_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 8, 2, 64)
    F = (8 + 2 * 2) * 64

    def fwd(V, flags=0, wq=A, wk=A, base=1e4, L=L, **kw):
        a = dict(T=4, packed=A, pos=A, q=A, k=A, v=A)
        a.update(kw)
        return C.qkv_prologue_fwd_ex(L, V, a["T"], a["packed"], a["pos"], wq, wk, 1e-6, base, flags, a["q"],
                                     a["k"], a["v"], None, None, stream=0, check=False)

    assert fwd(None) == C.QKVP_ERR_ARCH
    assert fwd(C.variant(inv_freq=[0.5] * 32, rope_scale=1.3, bias=A)) == C.QKVP_ERR_ARCH
    # norm off needs no weights; with it on they are required
    assert fwd(None, flags=C.QKVP_NORM_OFF, wq=None, wk=None) == C.QKVP_ERR_ARCH
    assert fwd(None, wq=None) == C.QKVP_ERR_NULL
    # a frequency table replaces the base, which is then not checked
    assert fwd(None, base=0.0) == C.QKVP_ERR_VALUE
    assert fwd(C.variant(inv_freq=[1.0] * 32), base=0.0) == C.QKVP_ERR_ARCH
    assert fwd(C.variant(inv_freq=[1.0] * 31 + [float("nan")])) == C.QKVP_ERR_VALUE
    assert fwd(C.variant(rope_scale=-1.0)) == C.QKVP_ERR_VALUE
    assert fwd(C.variant(rope_scale=float("inf"))) == C.QKVP_ERR_VALUE
    assert fwd(C.variant(bias=A + 4)) == C.QKVP_ERR_ALIGN
    # latent rows: frequency table and factor yes, bias and norm-off no
    LL = C.layout("latent", norm_dim=512, rope_dim=64)
    assert fwd(C.variant(inv_freq=[1.0] * 32, rope_scale=2.0), L=LL, wq=None, q=None, v=None) == C.QKVP_ERR_ARCH
    assert fwd(C.variant(bias=A), L=LL, wq=None, q=None, v=None) == C.QKVP_ERR_SHAPE
    assert fwd(None, flags=C.QKVP_NORM_OFF, L=LL, wq=None, q=None, v=None) == C.QKVP_ERR_FLAGS
    pw = C.qkv_prologue_pool_write_ex(L, C.variant(bias=A), 4, A, A, None, None, 1e-6, 1e4, C.QKVP_NORM_OFF, A, A,
                                      A, A, A, 4096, 64, None, stream=0, check=False)
    assert pw == C.QKVP_ERR_ARCH

    # backward
    V = C.variant(bias=A)
    need = C.qkv_prologue_bwd_workspace_size_ex(L, V, 100)
    assert need > C.qkv_prologue_bwd_workspace_size(L, 100)
    # one row per CTA now also holds the bias gradient's F floats
    fold = 4 * (1024 + 4)  # the fold's words after the rows
    rows = (C.qkv_prologue_bwd_workspace_size(L, 100) - fold) // (4 * 2 * 64)
    assert need == rows * 4 * (2 * 64 + F) + fold
    assert C.qkv_prologue_bwd_workspace_size_ex(L, None, 100) == C.qkv_prologue_bwd_workspace_size(L, 100)

    def bwd(V, flags=0, qp=A, kp=A, wq=A, wk=A, dwq=A, dwk=A, db=A, ws=A, wsb=need, L=L):
        return C.qkv_prologue_bwd_ex(L, V, 100, A, A, A, qp, kp, A, wq, wk, 1e-6, 5e5, flags, A, dwq, dwk, db, ws,
                                     wsb, stream=0, check=False)

    assert bwd(V) == C.QKVP_ERR_ARCH
    assert bwd(V, db=None) == C.QKVP_ERR_NULL
    assert bwd(V, db=A + 4) == C.QKVP_ERR_ALIGN
    assert bwd(V, wsb=need - 1) == C.QKVP_ERR_WORKSPACE
    assert bwd(None, db=None) == C.QKVP_ERR_ARCH  # no bias: no dbias needed
    # norm off: no saved inputs, weights or weight gradients needed
    assert bwd(V, flags=C.QKVP_NORM_OFF, qp=None, kp=None, wq=None, wk=None, dwq=None, dwk=None) == C.QKVP_ERR_ARCH
    assert bwd(V, qp=None) == C.QKVP_ERR_NULL
    # norm off and no bias: nothing to reduce, no workspace needed
    assert bwd(None, flags=C.QKVP_NORM_OFF, qp=None, kp=None, wq=None, wk=None, dwq=None, dwk=None, ws=None,
               wsb=0) == C.QKVP_ERR_ARCH
    # a bias gradient longer than one-token work items can hold
    Lbig = C.layout("interleaved", 128, 16, 128)
    assert bwd(V, L=Lbig, wsb=1 << 40) == C.QKVP_ERR_SHAPE


@cpu_only
def test_gemm_fwd_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 128, 16, 64)

    def g(T=256, hidden=5120, x=A, w=A, pos=A, wq=A, wk=A, flags=0, q=A, k=A, v=A, qp=None, kp=None, L=L):
        return C.qkv_prologue_gemm_fwd(L, T, hidden, x, w, pos, wq, wk, 1e-6, 5e5, flags, q, k, v, qp, kp, stream=0,
                                       check=False)

    assert g() == C.QKVP_ERR_ARCH  # valid: reaches the device check
    assert g(T=0) == C.QKVP_OK
    assert g(hidden=5121) == C.QKVP_ERR_SHAPE  # rows of x and W must be 16-byte multiples
    assert g(hidden=4) == C.QKVP_ERR_SHAPE
    assert g(L=C.layout("interleaved", 128, 16, 64, row_stride=10248)) == C.QKVP_ERR_SHAPE  # W is dense
    assert g(L=C.layout("latent", norm_dim=512, rope_dim=64)) == C.QKVP_ERR_SHAPE
    assert g(x=None) == C.QKVP_ERR_NULL
    assert g(w=A + 8) == C.QKVP_ERR_ALIGN
    assert g(flags=C.QKVP_SAVE_PRE) == C.QKVP_ERR_NULL
    assert g(flags=C.QKVP_SAVE_PRE, qp=A, kp=A) == C.QKVP_ERR_ARCH
    assert g(flags=C.QKVP_FORCE_GENERIC) == C.QKVP_ERR_FLAGS
    assert g(pos=None) == C.QKVP_ERR_NULL
    assert g(pos=None, flags=C.QKVP_NOPE) == C.QKVP_ERR_ARCH


@cpu_only
def test_noalloc_backward_argument_checks(lib):
    C = lib

    def bwd(L, T, flags=0):
        return C.qkv_prologue_bwd_noalloc(L, T, A, A, A, A, A, A, A, A, 1e-6, 5e5, flags, A, A, A, stream=0,
                                          check=False)

    # larger than the fixed 512 KiB array: refused before any device call
    assert bwd(C.layout("interleaved", 32, 8, 128), 2048) == C.QKVP_ERR_WORKSPACE
    assert bwd(C.layout("interleaved", 8, 3, 64), 16) == C.QKVP_ERR_SHAPE
    assert bwd(C.layout("interleaved", 128, 16, 64), 0, C.QKVP_ACCUMULATE_DW) == C.QKVP_OK
    assert bwd(C.layout("interleaved", 128, 16, 64), 16384) == C.QKVP_ERR_ARCH   # fits; needs the device


@cpu_only
def test_device_queries_refused_without_a_device(lib):
    C = lib
    # the bounded-wait self-test and the device error word need the device: refused
    assert C.qkv_prologue_wait_selftest(stream=0, check=False) == C.QKVP_ERR_ARCH
    raw = C._lib._lib
    v = ctypes.c_int(7)
    assert raw.qkv_prologue_device_error(0, None) == C.QKVP_ERR_NULL
    assert raw.qkv_prologue_device_error(1, ctypes.byref(v)) == C.QKVP_ERR_ARCH
    assert v.value == 7  # left untouched


def test_binding_fails_loudly_without_the_library(tmp_path):
    # a copy of the package without the .so must refuse to import
    import shutil
    import sys

    pkg = os.path.join(ROOT, "rope_qkv_prologue_gb300")
    dst = tmp_path / "rope_qkv_prologue_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    code = "import rope_qkv_prologue_gb300"
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True)
    assert res.returncode != 0 and "libqkv_prologue.so is missing" in res.stderr


def _ns_ws(units, split, head_dim):
    # the header's formula: per 128-row unit, split fp32 Gram partials of
    # 128 rows of head_dim + 4 and a 64 KiB image of M (bf16 hi and lo planes)
    return units * (split * 128 * (head_dim + 4) * 4 + 65536)


def test_newton_schulz_workspace_size(lib):
    C = lib
    L = C.layout("interleaved", 128, 16, 64)  # 160 blocks of 64 rows: 80 units
    assert C.qkv_newton_schulz_workspace(L, 5120, 4) == _ns_ws(80, 4, 64)
    assert C.qkv_newton_schulz_workspace(L, 5120, 1) == _ns_ws(80, 1, 64)
    L3 = C.layout("interleaved", 3, 1, 64)  # 5 blocks: 3 units, the last half empty
    assert C.qkv_newton_schulz_workspace(L3, 256, 2) == _ns_ws(3, 2, 64)
    assert C.qkv_newton_schulz_workspace(L3, 256, 2, count=3) == _ns_ws(8, 2, 64)  # 15 blocks: 8 units
    L8 = C.layout("sectioned", 8, 2, 128)
    assert C.qkv_newton_schulz_workspace(L8, 1024, 16) == _ns_ws(12, 16, 128)
    assert C.qkv_newton_schulz_workspace(L8, 1024, 2, count=0) == 0
    assert C.qkv_newton_schulz_workspace(L8, 1024, 17, check=False) == C.QKVP_ERR_SHAPE  # more than cols / 64
    assert C.qkv_newton_schulz_workspace(L8, 64 * 65, 65, check=False) == C.QKVP_ERR_SHAPE  # more than 64


@cpu_only
def test_newton_schulz_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 128, 16, 64)
    rows = 160 * 64
    W = A + 2 * rows * 5120 * 2  # a workspace after m and out
    ws4 = _ns_ws(80, 4, 64)

    def ns(L=L, cols=5120, m=A, out=A + rows * 5120 * 2, split=4, ws=W, wsb=ws4):
        return C.qkv_newton_schulz(L, cols, m, out, split, ws, wsb, stream=0, check=False)

    assert ns() == C.QKVP_ERR_ARCH  # valid: reaches the device check
    assert ns(split=0) == C.QKVP_ERR_ARCH  # planning the split needs the device
    assert ns(split=80, wsb=_ns_ws(80, 80, 64)) == C.QKVP_ERR_SHAPE  # at most 64
    assert ns(split=64, wsb=_ns_ws(80, 64, 64)) == C.QKVP_ERR_ARCH
    assert ns(L=C.layout("sectioned", 8, 2, 128), cols=1024, out=A + 1536 * 1024 * 2, split=16,
              wsb=_ns_ws(12, 16, 128)) == C.QKVP_ERR_ARCH
    assert ns(cols=5121) == C.QKVP_ERR_SHAPE    # a multiple of 64
    assert ns(cols=32) == C.QKVP_ERR_SHAPE
    assert ns(cols=(1 << 20) + 64) == C.QKVP_ERR_SHAPE
    assert ns(cols=128, split=3) == C.QKVP_ERR_SHAPE  # more than the 2 boxes of 64 columns
    assert ns(split=-1) == C.QKVP_ERR_SHAPE
    assert ns(L=C.layout("interleaved", 8, 2, 96)) == C.QKVP_ERR_SHAPE
    assert ns(L=C.layout("interleaved", 8, 3, 64)) == C.QKVP_ERR_SHAPE
    assert ns(L=C.layout("latent", norm_dim=512, rope_dim=64)) == C.QKVP_ERR_SHAPE
    assert ns(m=None) == C.QKVP_ERR_NULL
    assert ns(out=None) == C.QKVP_ERR_NULL
    assert ns(m=A + 8) == C.QKVP_ERR_ALIGN
    assert ns(out=A + 16) == C.QKVP_ERR_VALUE   # the output overlaps the input
    assert ns(out=A - rows * 5120 * 2, ws=A + rows * 5120 * 2) == C.QKVP_ERR_ARCH  # just below: no overlap
    assert ns(ws=None) == C.QKVP_ERR_WORKSPACE
    assert ns(wsb=ws4 - 1) == C.QKVP_ERR_WORKSPACE
    assert ns(ws=W + 8) == C.QKVP_ERR_ALIGN
    assert ns(ws=A + 2 * rows * 5120 * 2 - 16) == C.QKVP_ERR_VALUE  # overlaps the output
    assert ns(ws=A - 16) == C.QKVP_ERR_VALUE                     # overlaps the input
    with pytest.raises(C.QkvpError):
        C.qkv_newton_schulz_plan(L, 5120)      # planning needs the device


@cpu_only
def test_newton_schulz_batch_argument_checks(lib):
    C = lib
    L = C.layout("interleaved", 8, 2, 64)
    one = 768 * 512 * 2
    ws = _ns_ws(36, 2, 64)  # six layers of 12 blocks: 36 units

    def nb(count=6, cols=512, m=A, out=A + 6 * one, split=2, w=A + 12 * one, wsb=ws):
        return C.qkv_newton_schulz_batch(L, count, cols, m, out, split, w, wsb, stream=0, check=False)

    assert nb() == C.QKVP_ERR_ARCH            # valid: reaches the device check
    assert nb(count=0) == C.QKVP_OK           # nothing to do
    assert nb(count=-1) == C.QKVP_ERR_SHAPE
    assert nb(count=(1 << 30) // 768 + 1) == C.QKVP_ERR_SHAPE  # more than 2^30 rows
    assert nb(out=A + 5 * one) == C.QKVP_ERR_VALUE  # overlaps the last weight of the stack
    assert nb(out=A + 6 * one, m=None) == C.QKVP_ERR_NULL
    assert nb(cols=500) == C.QKVP_ERR_SHAPE
    assert nb(wsb=ws - 16) == C.QKVP_ERR_WORKSPACE  # sized for 36 units
    assert nb(count=5, wsb=_ns_ws(30, 2, 64)) == C.QKVP_ERR_ARCH

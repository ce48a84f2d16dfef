"""ctypes binding of libqkv_prologue.so: argument marshalling only.

The functions below carry the C names and the C argument order. Tensor
arguments may be torch tensors (their data_ptr() is passed), plain integers
(raw device addresses) or None (NULL). ``stream`` may be a torch.cuda.Stream,
an integer cudaStream_t or None (torch's current stream on the current
device). Every step of the computation runs in the library's CUDA kernels;
there is no Python or CPU fallback: if the library is missing, importing this
module raises.
"""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqkv_prologue.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python rope_qkv_prologue_gb300/_build.py, or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants (mirror include/qkv_prologue.h) ------------------------------
QKVP_VERSION = 3
QKVP_OK = 0
QKVP_ERR_NULL = -1
QKVP_ERR_SHAPE = -2
QKVP_ERR_ALIGN = -3
QKVP_ERR_ARCH = -4
QKVP_ERR_WORKSPACE = -5
QKVP_ERR_LAUNCH = -6
QKVP_ERR_FLAGS = -7
QKVP_ERR_VALUE = -8

QKVP_INTERLEAVED = 0
QKVP_SECTIONED = 1
QKVP_LATENT = 2

QKVP_NOPE = 1
QKVP_SAVE_PRE = 2
QKVP_ACCUMULATE_DW = 4
QKVP_FORCE_GENERIC = 8
QKVP_NORM_OFF = 16

QKVP_DEV_BAD_PAGE = 1
QKVP_DEV_BAD_OFFSET = 2


class qkvp_layout(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("n_q", ctypes.c_int32),
        ("n_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("row_stride", ctypes.c_int64),
        ("norm_dim", ctypes.c_int32),
        ("rope_dim", ctypes.c_int32),
    ]


class qkvp_variant(ctypes.Structure):
    _fields_ = [
        ("inv_freq", ctypes.POINTER(ctypes.c_double)),
        ("rope_scale", ctypes.c_double),
        ("bias", ctypes.c_void_p),
    ]


class QkvpError(RuntimeError):
    def __init__(self, status, func):
        self.status = status
        super().__init__(f"{func}: {qkv_prologue_status_string(status)} (status {status})")


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_u32 = ctypes.c_uint32
_f32 = ctypes.c_float
_f64 = ctypes.c_double
_LP = ctypes.POINTER(qkvp_layout)
_VP = ctypes.POINTER(qkvp_variant)

_SIGS = {
    "qkv_prologue_fwd": ([_LP, _i64, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "qkv_prologue_pool_write": ([_LP, _i64, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp, _vp, _vp,
                                 _i32, _i32, _vp, _vp], ctypes.c_int),
    "qkv_prologue_pool_scatter": ([_LP, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp], ctypes.c_int),
    "qkv_prologue_bwd_workspace_size": ([_LP, _i64], ctypes.c_size_t),
    "qkv_prologue_bwd": ([_LP, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp,
                          _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "qkv_prologue_bwd_noalloc": ([_LP, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp,
                                  _vp, _vp], ctypes.c_int),
    "qkv_prologue_fwd_ex": ([_LP, _VP, _i64, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp, _vp, _vp, _vp],
                            ctypes.c_int),
    "qkv_prologue_pool_write_ex": ([_LP, _VP, _i64, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp, _vp, _vp,
                                    _i32, _i32, _vp, _vp], ctypes.c_int),
    "qkv_prologue_bwd_workspace_size_ex": ([_LP, _VP, _i64], ctypes.c_size_t),
    "qkv_prologue_bwd_ex": ([_LP, _VP, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp,
                             _vp, _vp, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "qkv_prologue_gemm_fwd": ([_LP, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _f32, _f64, _u32, _vp, _vp, _vp, _vp, _vp,
                               _vp], ctypes.c_int),
    "qkv_newton_schulz": ([_LP, _i64, _vp, _vp, _i32, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "qkv_newton_schulz_batch": ([_LP, _i64, _i64, _vp, _vp, _i32, _vp, ctypes.c_size_t, _vp], ctypes.c_int),
    "qkv_newton_schulz_workspace": ([_LP, _i64, _i64, _i32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "qkv_newton_schulz_plan": ([_LP, _i64, _i64, _i32, ctypes.POINTER(ctypes.c_int32),
                                ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "qkv_prologue_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "qkv_prologue_version": ([], ctypes.c_int),
    "qkv_prologue_device_error": ([ctypes.c_int, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "qkv_prologue_wait_selftest": ([_vp], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


def layout(kind="interleaved", n_q=0, n_kv=0, head_dim=64, row_stride=0, norm_dim=0, rope_dim=0):
    """Build a qkvp_layout. kind: 'interleaved' | 'sectioned' | 'latent' or its enum value."""
    kinds = {"interleaved": QKVP_INTERLEAVED, "sectioned": QKVP_SECTIONED, "latent": QKVP_LATENT}
    k = kinds[kind] if isinstance(kind, str) else int(kind)
    return qkvp_layout(k, n_q, n_kv, head_dim, row_stride, norm_dim, rope_dim)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ret(status, func, check):
    if check and status != QKVP_OK:
        raise QkvpError(status, func)
    return status


def variant(inv_freq=None, rope_scale=0.0, bias=None):
    """A qkvp_variant (the GQAttention variant options). inv_freq: a sequence of
    head_dim / 2 floats (kept alive with the struct); bias: a device tensor or
    address, float32 [(n_q + 2 n_kv) * head_dim] in packed-row order."""
    v = qkvp_variant()
    if inv_freq is not None:
        arr = (ctypes.c_double * len(inv_freq))(*[float(f) for f in inv_freq])
        v._inv_freq_keepalive = arr
        v.inv_freq = ctypes.cast(arr, ctypes.POINTER(ctypes.c_double))
    v.rope_scale = float(rope_scale)
    v.bias = _ptr(bias)
    return v


def _vref(v):
    return None if v is None else ctypes.byref(v)


def qkv_prologue_status_string(status):
    return _lib.qkv_prologue_status_string(int(status)).decode()


def qkv_prologue_version():
    return _lib.qkv_prologue_version()


def qkv_prologue_device_error(clear=True, check=True):
    """The library's device error word on the current device (0 = no error)."""
    v = ctypes.c_int(0)
    _ret(_lib.qkv_prologue_device_error(int(bool(clear)), ctypes.byref(v)), "qkv_prologue_device_error", check)
    return v.value


def qkv_prologue_wait_selftest(stream=None, check=True):
    """Enqueue the bounded-wait self-test kernel (gives up after 2 s, sets bit 1
    of the device error word)."""
    return _ret(_lib.qkv_prologue_wait_selftest(_stream(stream)), "qkv_prologue_wait_selftest", check)


def qkv_prologue_fwd(L, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, k, v,
                     q_pre=None, k_pre=None, stream=None, check=True):
    st = _lib.qkv_prologue_fwd(ctypes.byref(L), int(T), _ptr(packed), _ptr(pos), _ptr(w_q), _ptr(w_k),
                               float(eps), float(rope_base), int(flags), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(q_pre), _ptr(k_pre), _stream(stream))
    return _ret(st, "qkv_prologue_fwd", check)


def qkv_prologue_pool_write(L, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, page, offset,
                            k_pool, v_pool, num_pages, page_size, dev_status=None, stream=None,
                            check=True):
    st = _lib.qkv_prologue_pool_write(ctypes.byref(L), int(T), _ptr(packed), _ptr(pos), _ptr(w_q),
                                      _ptr(w_k), float(eps), float(rope_base), int(flags), _ptr(q),
                                      _ptr(page), _ptr(offset), _ptr(k_pool), _ptr(v_pool),
                                      int(num_pages), int(page_size), _ptr(dev_status), _stream(stream))
    return _ret(st, "qkv_prologue_pool_write", check)


def qkv_prologue_pool_scatter(L, T, k_rows, v_rows, page, offset, k_pool, v_pool, num_pages,
                              page_size, dev_status=None, stream=None, check=True):
    st = _lib.qkv_prologue_pool_scatter(ctypes.byref(L), int(T), _ptr(k_rows), _ptr(v_rows), _ptr(page),
                                        _ptr(offset), _ptr(k_pool), _ptr(v_pool), int(num_pages),
                                        int(page_size), _ptr(dev_status), _stream(stream))
    return _ret(st, "qkv_prologue_pool_scatter", check)


def qkv_prologue_bwd_workspace_size(L, T):
    return int(_lib.qkv_prologue_bwd_workspace_size(ctypes.byref(L), int(T)))


def qkv_prologue_bwd(L, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags, dpacked,
                     dw_q, dw_k, workspace, workspace_bytes, stream=None, check=True):
    st = _lib.qkv_prologue_bwd(ctypes.byref(L), int(T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(q_pre),
                               _ptr(k_pre), _ptr(pos), _ptr(w_q), _ptr(w_k), float(eps), float(rope_base),
                               int(flags), _ptr(dpacked), _ptr(dw_q), _ptr(dw_k), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))
    return _ret(st, "qkv_prologue_bwd", check)


def qkv_prologue_bwd_noalloc(L, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags, dpacked,
                             dw_q, dw_k, stream=None, check=True):
    """qkv_prologue_bwd for callers that cannot allocate: the library's own fixed
    512 KiB device array replaces the workspace (see the C header for limits)."""
    st = _lib.qkv_prologue_bwd_noalloc(ctypes.byref(L), int(T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(q_pre),
                                       _ptr(k_pre), _ptr(pos), _ptr(w_q), _ptr(w_k), float(eps),
                                       float(rope_base), int(flags), _ptr(dpacked), _ptr(dw_q), _ptr(dw_k),
                                       _stream(stream))
    return _ret(st, "qkv_prologue_bwd_noalloc", check)


def qkv_prologue_fwd_ex(L, V, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, k, v,
                        q_pre=None, k_pre=None, stream=None, check=True):
    st = _lib.qkv_prologue_fwd_ex(ctypes.byref(L), _vref(V), int(T), _ptr(packed), _ptr(pos), _ptr(w_q),
                                  _ptr(w_k), float(eps), float(rope_base), int(flags), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(q_pre), _ptr(k_pre), _stream(stream))
    return _ret(st, "qkv_prologue_fwd_ex", check)


def qkv_prologue_pool_write_ex(L, V, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, page, offset,
                               k_pool, v_pool, num_pages, page_size, dev_status=None, stream=None, check=True):
    st = _lib.qkv_prologue_pool_write_ex(ctypes.byref(L), _vref(V), int(T), _ptr(packed), _ptr(pos), _ptr(w_q),
                                         _ptr(w_k), float(eps), float(rope_base), int(flags), _ptr(q),
                                         _ptr(page), _ptr(offset), _ptr(k_pool), _ptr(v_pool),
                                         int(num_pages), int(page_size), _ptr(dev_status), _stream(stream))
    return _ret(st, "qkv_prologue_pool_write_ex", check)


def qkv_prologue_bwd_workspace_size_ex(L, V, T):
    return int(_lib.qkv_prologue_bwd_workspace_size_ex(ctypes.byref(L), _vref(V), int(T)))


def qkv_prologue_bwd_ex(L, V, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags, dpacked,
                        dw_q, dw_k, dbias, workspace, workspace_bytes, stream=None, check=True):
    st = _lib.qkv_prologue_bwd_ex(ctypes.byref(L), _vref(V), int(T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(q_pre),
                                  _ptr(k_pre), _ptr(pos), _ptr(w_q), _ptr(w_k), float(eps), float(rope_base),
                                  int(flags), _ptr(dpacked), _ptr(dw_q), _ptr(dw_k), _ptr(dbias),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream))
    return _ret(st, "qkv_prologue_bwd_ex", check)


def qkv_prologue_gemm_fwd(L, T, hidden, x, w_qkv, pos, w_q, w_k, eps, rope_base, flags, q, k, v, q_pre=None,
                          k_pre=None, stream=None, check=True):
    st = _lib.qkv_prologue_gemm_fwd(ctypes.byref(L), int(T), int(hidden), _ptr(x), _ptr(w_qkv), _ptr(pos), _ptr(w_q),
                                    _ptr(w_k), float(eps), float(rope_base), int(flags), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(q_pre), _ptr(k_pre), _stream(stream))
    return _ret(st, "qkv_prologue_gemm_fwd", check)


def qkv_newton_schulz(L, cols, m, out, split=0, workspace=None, workspace_bytes=0, stream=None, check=True):
    st = _lib.qkv_newton_schulz(ctypes.byref(L), int(cols), _ptr(m), _ptr(out), int(split), _ptr(workspace),
                                int(workspace_bytes), _stream(stream))
    return _ret(st, "qkv_newton_schulz", check)


def qkv_newton_schulz_batch(L, count, cols, m, out, split=0, workspace=None, workspace_bytes=0, stream=None,
                            check=True):
    st = _lib.qkv_newton_schulz_batch(ctypes.byref(L), int(count), int(cols), _ptr(m), _ptr(out), int(split),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream))
    return _ret(st, "qkv_newton_schulz_batch", check)


def qkv_newton_schulz_workspace(L, cols, split=0, count=1, check=True):
    """Workspace bytes the Newton-Schulz launches need for these arguments
    (status code instead when check is False and the call fails)."""
    n = ctypes.c_size_t(0)
    st = _lib.qkv_newton_schulz_workspace(ctypes.byref(L), int(count), int(cols), int(split), ctypes.byref(n))
    if not check and st != QKVP_OK:
        return st
    _ret(st, "qkv_newton_schulz_workspace", True)
    return n.value


def qkv_newton_schulz_plan(L, cols, split=0, count=1):
    """(split, Gram grid) the library would launch for these arguments."""
    c, g = ctypes.c_int32(0), ctypes.c_int32(0)
    st = _lib.qkv_newton_schulz_plan(ctypes.byref(L), int(count), int(cols), int(split), ctypes.byref(c),
                                     ctypes.byref(g))
    _ret(st, "qkv_newton_schulz_plan", True)
    return c.value, g.value

"""Plain CPU binary64 oracle of causal streaming-softmax attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
never does, and it shares no code with the CUDA kernels.

The C source (``attn_oracle.c``) holds the arithmetic: the materialised
softmax of StreamingAttentionSM86.alpha (forward-pass and backward-pass
module headers) with the length mask of the self_attn_fwd gist.  This module
only marshals numpy arrays: binary16 inputs are widened to binary64 exactly.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["forward", "backward", "query_rows", "key_rows", "probs_row",
           "inverse_rotate", "num_threads", "set_num_threads"]


class _Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("scale", ctypes.c_double)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER
        d = P(ctypes.c_double)
        i32 = P(ctypes.c_int32)
        sp = P(_Shape)
        lib.oracle_forward.argtypes = [sp, i32, d, d, d, d, d]
        lib.oracle_backward.argtypes = [sp, i32, d, d, d, d, d, d, d, d, d, d]
        lib.oracle_query_rows.argtypes = [sp, i32, d, d, d, d, ctypes.c_int, ctypes.c_int,
                                          i32, ctypes.c_int, d, d, d, d]
        lib.oracle_key_rows.argtypes = [sp, i32, d, d, d, d, ctypes.c_int, ctypes.c_int,
                                        i32, ctypes.c_int, d, d]
        lib.oracle_probs_row.argtypes = [sp, i32, d, d, d, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, d]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _lens(lens):
    if lens is None:
        return None, None
    arr = np.ascontiguousarray(lens, dtype=np.int32)
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _shape(q, k, causal, scale):
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, T, d):
        raise ValueError("k shape %r does not match q %r" % (k.shape, q.shape))
    return _Shape(B, T, H, Hkv, d, 1 if causal else 0, float(scale))


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed (%d)" % (what, rc))


def forward(q, k, vt, *, causal=True, scale=0.125, lens=None):
    """O [B][T][H*d] and base-2 L [B][H][T] in binary64."""
    q, k, vt = _f64(q), _f64(k), _f64(vt)
    s = _shape(q, k, causal, scale)
    B, H, T, d = q.shape
    o = np.empty((B, T, H * d))
    lse = np.empty((B, H, T))
    keep, lp = _lens(lens)
    _check(_load().oracle_forward(ctypes.byref(s), lp, _ptr(q), _ptr(k), _ptr(vt),
                                  _ptr(o), _ptr(lse)), "forward")
    return o, lse


def backward(q, k, vt, dout, *, causal=True, scale=0.125, lens=None):
    """Full pass: dict of o, lse, delta, dq, dk, dvt (binary64, boundary layouts)."""
    q, k, vt, dout = _f64(q), _f64(k), _f64(vt), _f64(dout)
    s = _shape(q, k, causal, scale)
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    out = dict(o=np.empty((B, T, H * d)), lse=np.empty((B, H, T)),
               delta=np.empty((B, H, T)), dq=np.empty((B, H, T, d)),
               dk=np.empty((B, Hkv, T, d)), dvt=np.empty((B, Hkv, d, T)))
    keep, lp = _lens(lens)
    _check(_load().oracle_backward(ctypes.byref(s), lp, _ptr(q), _ptr(k), _ptr(vt),
                                   _ptr(dout), _ptr(out["o"]), _ptr(out["lse"]),
                                   _ptr(out["delta"]), _ptr(out["dq"]), _ptr(out["dk"]),
                                   _ptr(out["dvt"])), "backward")
    return out


def query_rows(q, k, vt, dout, b, h, rows, *, causal=True, scale=0.125, lens=None):
    """Row-local outputs of sampled query rows of head h: o [n][d], lse, delta, dq [n][d]."""
    q, k, vt, dout = _f64(q), _f64(k), _f64(vt), _f64(dout)
    s = _shape(q, k, causal, scale)
    d = q.shape[3]
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    n = rows.size
    o = np.empty((n, d)); lse = np.empty(n); delta = np.empty(n); dq = np.empty((n, d))
    keep, lp = _lens(lens)
    _check(_load().oracle_query_rows(
        ctypes.byref(s), lp, _ptr(q), _ptr(k), _ptr(vt), _ptr(dout), int(b), int(h),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n,
        _ptr(o), _ptr(lse), _ptr(delta), _ptr(dq)), "query_rows")
    return dict(o=o, lse=lse, delta=delta, dq=dq)


def key_rows(q, k, vt, dout, b, kv, keys, *, causal=True, scale=0.125, lens=None):
    """dK [n][d] and dV [n][d] of sampled keys of K/V head kv."""
    q, k, vt, dout = _f64(q), _f64(k), _f64(vt), _f64(dout)
    s = _shape(q, k, causal, scale)
    d = q.shape[3]
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    n = keys.size
    dk = np.empty((n, d)); dv = np.empty((n, d))
    keep, lp = _lens(lens)
    _check(_load().oracle_key_rows(
        ctypes.byref(s), lp, _ptr(q), _ptr(k), _ptr(vt), _ptr(dout), int(b), int(kv),
        keys.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n, _ptr(dk), _ptr(dv)),
        "key_rows")
    return dict(dk=dk, dv=dv)


def probs_row(q, k, vt, b, h, i, *, causal=True, scale=0.125, lens=None):
    """The softmax probability row P[i, :] of head h (length T)."""
    q, k, vt = _f64(q), _f64(k), _f64(vt)
    s = _shape(q, k, causal, scale)
    p = np.empty(q.shape[2])
    keep, lp = _lens(lens)
    _check(_load().oracle_probs_row(ctypes.byref(s), lp, _ptr(q), _ptr(k), _ptr(vt),
                                    int(b), int(h), int(i), _ptr(p)), "probs_row")
    return p


def inverse_rotate(dq, cos, sin):
    """dQ turned back by the inverse half-split rotation, token-major.

    StreamingAttentionSM86.alpha, the rotated epilogue of the dQ-from-scores
    pass: for query row p of head h and column c < 32, with (cos, sin) =
    (cos[p][c], sin[p][c]),
        out[c]      = dq[c] cos + dq[c + 32] sin
        out[c + 32] = dq[c + 32] cos - dq[c] sin,
    stored at row p, columns 64 h + c of a token-major [B][T][H * 64] array.
    Arguments: dq [B][H][T][64] (already scaled by s), cos and sin [T][32];
    all widened to binary64 and computed without intermediate rounding.
    """
    dq = np.asarray(dq, dtype=np.float64)
    cos = np.asarray(cos, dtype=np.float64)
    sin = np.asarray(sin, dtype=np.float64)
    B, H, T, d = dq.shape
    half = d // 2
    x1, x2 = dq[..., :half], dq[..., half:]
    c, s_ = cos[None, None, :, :half], sin[None, None, :, :half]
    out = np.concatenate([x1 * c + x2 * s_, x2 * c - x1 * s_], axis=-1)  # [B][H][T][64]
    return np.ascontiguousarray(out.transpose(0, 2, 1, 3).reshape(B, T, H * d))

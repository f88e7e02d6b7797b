"""Thin Python binding of libattn.so (the C ABI in include/attn.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (device memory and
streams are PyTorch's); the functions check dtypes, shapes, devices and
contiguity, build the ``attn_shape`` struct and call the entry point of the
same name on the current stream (or the one given).  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

_LIB_PATH = _build.LIB

ATTN_OK = 0
ATTN_ERR_SHAPE = -1
ATTN_ERR_NULL = -2
ATTN_ERR_ALIGN = -3
ATTN_ERR_WORKSPACE = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_DEVICE_TIMEOUT = -6
ATTN_ERR_DEVICE = -7
ATTN_ERR_SCRATCH_LIMIT = -8
ATTN_STEP_STORED = 0
ATTN_STEP_FUSED = 1

# lowest bounded-wait limit the library accepts (attn_set_wait_limit_ns)
MIN_WAIT_LIMIT_NS = 10_000_000

HEAD_DIM = 64


class AttnShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("head_begin", ctypes.c_int32), ("head_count", ctypes.c_int32),
                ("v_rows", ctypes.c_int32)]


class AttnDeviceBuffers(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("vt", ctypes.c_void_p),
                ("dout", ctypes.c_void_p), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("delta", ctypes.c_void_p), ("ws", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dvt", ctypes.c_void_p)]


class AttnProjection(ctypes.Structure):
    _fields_ = [("f32", ctypes.c_void_p), ("bf16", ctypes.c_void_p), ("ld", ctypes.c_int64)]


class AttnError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = "%s failed: %s (%d)" % (fn, error_string(code), code)
        if code == ATTN_ERR_CUDA:
            msg += ": " + load_library().attn_last_cuda_error().decode()
        super().__init__(msg)


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libattn.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libattn.so not found at %s: build it with "
                          "causal_streaming_softmax_gb300.build.build()" % p)
    lib = ctypes.CDLL(p)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sp = ctypes.POINTER(AttnShape)
    lib.attn_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp]
    lib.attn_row_terms.argtypes = [sp, vp, vp, vp, vp]
    lib.attn_bwd_workspace_bytes.argtypes = [sp]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_bwd_keys.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.attn_bwd_queries.argtypes = [sp, vp, vp, sz, vp, vp]
    lib.attn_bwd_queries_fused.argtypes = [sp] + [vp] * 9
    lib.attn_bwd_queries_rotated.argtypes = [sp, vp, vp, sz, vp, vp, vp, ctypes.c_int64, vp]
    lib.attn_bwd_queries_rotated.restype = ctypes.c_int
    pp = ctypes.POINTER(AttnProjection)
    lib.attn_bwd_keys_projected.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, sz, pp, pp, vp]
    lib.attn_bwd_keys_projected.restype = ctypes.c_int
    lib.attn_bwd_queries_projected.argtypes = [sp, vp, vp, sz, pp, vp]
    lib.attn_bwd_queries_projected.restype = ctypes.c_int
    lib.attn_bwd_queries_fused.restype = ctypes.c_int
    lib.attn_error_string.argtypes = [ctypes.c_int]
    lib.attn_error_string.restype = ctypes.c_char_p
    lib.attn_last_device_error.argtypes = [vp]
    lib.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.attn_set_wait_limit_ns.restype = None
    lib.attn_wait_limit_ns.argtypes = []
    lib.attn_wait_limit_ns.restype = ctypes.c_uint64
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.attn_version.restype = ctypes.c_int
    lib.attn_last_cuda_error.restype = ctypes.c_char_p
    lib.attn_selftest_arith.argtypes = [vp, vp, vp, ctypes.c_int, vp]
    lib.attn_step_host.argtypes = [ctypes.POINTER(AttnShape), ctypes.POINTER(AttnDeviceBuffers)] + \
        [vp] * 10
    lib.attn_step_host.restype = ctypes.c_int
    lib.attn_step_host_order.argtypes = [ctypes.POINTER(AttnShape),
                                         ctypes.POINTER(AttnDeviceBuffers)]
    lib.attn_step_host_order.restype = ctypes.c_int
    lib.attn_selftest_arith.restype = ctypes.c_int
    for name in ("attn_fwd", "attn_row_terms", "attn_bwd_keys", "attn_bwd_queries",
                 "attn_last_device_error", "attn_selftest_wait_timeout"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def error_string(code: int) -> str:
    return load_library().attn_error_string(int(code)).decode()


def _check(fn, rc):
    if rc != ATTN_OK:
        raise AttnError(fn, rc)


@dataclass
class Shape:
    """Problem shape; ``seq_lens`` is an int32 CUDA tensor [batch] or None."""
    batch: int
    seq: int
    heads: int
    kv_heads: int
    causal: bool = True
    scale: float = 0.125
    seq_lens: Optional[torch.Tensor] = None
    head_begin: int = 0
    head_count: int = 0
    v_rows: bool = False  # V as rows [B][Hkv][T][64] instead of V^T [B][Hkv][64][T]

    def c_struct(self) -> AttnShape:
        lens = 0
        if self.seq_lens is not None:
            t = self.seq_lens
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() \
                    or t.numel() != self.batch:
                raise ValueError("seq_lens must be a contiguous int32 CUDA tensor [batch]")
            lens = t.data_ptr()
        return AttnShape(self.batch, self.seq, self.heads, self.kv_heads, HEAD_DIM,
                         1 if self.causal else 0, lens, float(self.scale),
                         self.head_begin, self.head_count, 1 if self.v_rows else 0)

    def chunk(self, head_begin: int, head_count: int) -> "Shape":
        return Shape(self.batch, self.seq, self.heads, self.kv_heads, self.causal, self.scale,
                     self.seq_lens, head_begin, head_count, self.v_rows)

    def v_shape(self):
        """Shape of the V argument in this layout."""
        if self.v_rows:
            return (self.batch, self.kv_heads, self.seq, HEAD_DIM)
        return (self.batch, self.kv_heads, HEAD_DIM, self.seq)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _want(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def attn_fwd(s: Shape, q, k, vt, o, lse, stream=None) -> None:
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    args = (_want(q, "q", torch.float16, (B, H, T, 64)),
            _want(k, "k", torch.float16, (B, Hkv, T, 64)),
            _want(vt, "vt", torch.float16, s.v_shape()),
            _want(o, "o", torch.float16, (B, T, H * 64)),
            _want(lse, "lse", torch.float32, (B, H, T)))
    shape = s.c_struct()
    _check("attn_fwd", load_library().attn_fwd(ctypes.byref(shape), *args, _stream_ptr(stream)))


def attn_row_terms(s: Shape, o, dout, delta, stream=None) -> None:
    B, T, H = s.batch, s.seq, s.heads
    args = (_want(o, "o", torch.float16, (B, T, H * 64)),
            _want(dout, "dout", torch.float16, (B, H, T, 64)),
            _want(delta, "delta", torch.float32, (B, H, T)))
    shape = s.c_struct()
    _check("attn_row_terms",
           load_library().attn_row_terms(ctypes.byref(shape), *args, _stream_ptr(stream)))


def workspace_bytes(s: Shape) -> int:
    shape = s.c_struct()
    n = load_library().attn_bwd_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise AttnError("attn_bwd_workspace_bytes", ATTN_ERR_SHAPE)
    return n


def alloc_workspace(s: Shape, device=None) -> torch.Tensor:
    """A uint8 CUDA tensor large enough for the dS workspace of ``s``."""
    return torch.empty(workspace_bytes(s), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def _chunk_heads(s: Shape):
    count = s.head_count or s.kv_heads
    return s.head_begin, count


def attn_bwd_keys(s: Shape, q, k, vt, dout, lse, delta, ws, dk, dvt, stream=None) -> None:
    """``ws=None`` runs the key pass without storing dS (for attn_bwd_queries_fused)."""
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    if ws is not None and not (isinstance(ws, torch.Tensor) and ws.is_cuda
                               and ws.dtype == torch.uint8 and ws.is_contiguous()):
        raise TypeError("ws must be a contiguous uint8 CUDA tensor or None")
    args = (_want(q, "q", torch.float16, (B, H, T, 64)),
            _want(k, "k", torch.float16, (B, Hkv, T, 64)),
            _want(vt, "vt", torch.float16, s.v_shape()),
            _want(dout, "dout", torch.float16, (B, H, T, 64)),
            _want(lse, "lse", torch.float32, (B, H, T)),
            _want(delta, "delta", torch.float32, (B, H, T)),
            None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel(),
            _want(dk, "dk", torch.float32, (B, Hkv, T, 64)),
            _want(dvt, "dvt", torch.float32, (B, Hkv, 64, T)))
    shape = s.c_struct()
    _check("attn_bwd_keys",
           load_library().attn_bwd_keys(ctypes.byref(shape), *args, _stream_ptr(stream)))


def attn_bwd_queries(s: Shape, k, ws, dq, stream=None) -> None:
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.dtype == torch.uint8
            and ws.is_contiguous()):
        raise TypeError("ws must be a contiguous uint8 CUDA tensor")
    args = (_want(k, "k", torch.float16, (B, Hkv, T, 64)), ws.data_ptr(), ws.numel(),
            _want(dq, "dq", torch.float32, (B, H, T, 64)))
    shape = s.c_struct()
    _check("attn_bwd_queries",
           load_library().attn_bwd_queries(ctypes.byref(shape), *args, _stream_ptr(stream)))


def attn_bwd_queries_fused(s: Shape, q, k, vt, dout, o, lse, delta, dq, stream=None) -> None:
    """Writes ``delta`` (D = rowsum(dO * O)) and ``dq``; replaces attn_row_terms."""
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    args = (_want(q, "q", torch.float16, (B, H, T, 64)),
            _want(k, "k", torch.float16, (B, Hkv, T, 64)),
            _want(vt, "vt", torch.float16, s.v_shape()),
            _want(dout, "dout", torch.float16, (B, H, T, 64)),
            _want(o, "o", torch.float16, (B, T, H * 64)),
            _want(lse, "lse", torch.float32, (B, H, T)),
            _want(delta, "delta", torch.float32, (B, H, T)),
            _want(dq, "dq", torch.float32, (B, H, T, 64)))
    shape = s.c_struct()
    _check("attn_bwd_queries_fused", load_library().attn_bwd_queries_fused(
        ctypes.byref(shape), *args, _stream_ptr(stream)))


def attn_bwd_queries_rotated(s: Shape, k, ws, cos, sin, out, ld=None, stream=None) -> None:
    """dQ pass with the inverse half-split rotation, bfloat16 token-major
    ``out`` (row stride ``ld`` elements, default heads * 64)."""
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.dtype == torch.uint8
            and ws.is_contiguous()):
        raise TypeError("ws must be a contiguous uint8 CUDA tensor")
    if not (isinstance(out, torch.Tensor) and out.is_cuda and out.dtype == torch.bfloat16):
        raise TypeError("out must be a bfloat16 CUDA tensor")
    ld = H * 64 if ld is None else int(ld)
    args = (_want(k, "k", torch.float16, (B, Hkv, T, 64)), ws.data_ptr(), ws.numel(),
            _want(cos, "cos", torch.float32, (T, 32)), _want(sin, "sin", torch.float32, (T, 32)),
            out.data_ptr(), ld)
    shape = s.c_struct()
    _check("attn_bwd_queries_rotated", load_library().attn_bwd_queries_rotated(
        ctypes.byref(shape), *args, _stream_ptr(stream)))


def projection(f32=None, bf16=None, ld=None) -> AttnProjection:
    """A token-major block of a projection gradient: CUDA tensors (views into
    the wider [B][T][width] gradient, starting at the block's first column),
    float32 and/or bfloat16, row stride ``ld`` elements."""
    for t, dt in ((f32, torch.float32), (bf16, torch.bfloat16)):
        if t is not None and not (t.is_cuda and t.dtype == dt):
            raise TypeError("projection blocks must be CUDA %s tensors" % dt)
    if ld is None:
        raise ValueError("ld (row stride in elements) is required")
    return AttnProjection(None if f32 is None else f32.data_ptr(),
                          None if bf16 is None else bf16.data_ptr(), int(ld))


def attn_bwd_keys_projected(s: Shape, q, k, vt, dout, lse, delta, ws, dk_out: AttnProjection,
                            dv_out: AttnProjection, stream=None) -> None:
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    args = (_want(q, "q", torch.float16, (B, H, T, 64)),
            _want(k, "k", torch.float16, (B, Hkv, T, 64)),
            _want(vt, "vt", torch.float16, s.v_shape()),
            _want(dout, "dout", torch.float16, (B, H, T, 64)),
            _want(lse, "lse", torch.float32, (B, H, T)),
            _want(delta, "delta", torch.float32, (B, H, T)),
            None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel())
    shape = s.c_struct()
    _check("attn_bwd_keys_projected", load_library().attn_bwd_keys_projected(
        ctypes.byref(shape), *args, ctypes.byref(dk_out), ctypes.byref(dv_out),
        _stream_ptr(stream)))


def attn_bwd_queries_projected(s: Shape, k, ws, dq_out: AttnProjection, stream=None) -> None:
    B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
    shape = s.c_struct()
    _check("attn_bwd_queries_projected", load_library().attn_bwd_queries_projected(
        ctypes.byref(shape), _want(k, "k", torch.float16, (B, Hkv, T, 64)), ws.data_ptr(),
        ws.numel(), ctypes.byref(dq_out), _stream_ptr(stream)))


def last_device_error(stream=None) -> int:
    return load_library().attn_last_device_error(_stream_ptr(stream))


def check_device_error(stream=None) -> None:
    _check("device", last_device_error(stream))


def set_wait_limit_ns(ns: int) -> None:
    """Sets the kernels' bounded-wait limit (0: the default; values below
    MIN_WAIT_LIMIT_NS are raised to it)."""
    load_library().attn_set_wait_limit_ns(int(ns))


def wait_limit_ns() -> int:
    return int(load_library().attn_wait_limit_ns())


def selftest_arith(x, stream=None):
    """Runs the library's binary16 packing and exponential over the float32
    CUDA tensor x (even length): returns (packed uint32 words, 2^x)."""
    if not (x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise TypeError("x must be a contiguous float32 CUDA tensor")
    n = x.numel()
    packed = torch.empty(n // 2, dtype=torch.int32, device=x.device)
    e2 = torch.empty(n, dtype=torch.float32, device=x.device)
    _check("attn_selftest_arith", load_library().attn_selftest_arith(
        x.data_ptr(), packed.data_ptr(), e2.data_ptr(), n, _stream_ptr(stream)))
    return packed, e2


def selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> int:
    return load_library().attn_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream))


class Buffers:
    """Device buffers of one forward + backward problem (boundary layouts);
    ``workspace=False`` leaves out the dS workspace (for the fused dQ pass)."""

    def __init__(self, s: Shape, device=None, workspace: bool = True):
        dev = device or torch.device("cuda")
        B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
        self.o = torch.empty((B, T, H * 64), dtype=torch.float16, device=dev)
        self.lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        self.delta = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        self.dq = torch.empty((B, H, T, 64), dtype=torch.float32, device=dev)
        self.dk = torch.empty((B, Hkv, T, 64), dtype=torch.float32, device=dev)
        self.dvt = torch.empty((B, Hkv, 64, T), dtype=torch.float32, device=dev)
        self.ws = alloc_workspace(s, dev) if workspace else None


def forward_backward(s: Shape, q, k, vt, dout, bufs: Buffers, stream=None,
                     fused_dq: bool = False) -> Buffers:
    """One pass of the whole path: attn_fwd, attn_row_terms, attn_bwd_keys,
    attn_bwd_queries; with ``fused_dq``: attn_fwd, attn_bwd_queries_fused
    (D and dQ, S, P, dP recomputed), then attn_bwd_keys storing no dS
    (``bufs.ws`` unused)."""
    attn_fwd(s, q, k, vt, bufs.o, bufs.lse, stream)
    if fused_dq:
        attn_bwd_queries_fused(s, q, k, vt, dout, bufs.o, bufs.lse, bufs.delta, bufs.dq, stream)
        attn_bwd_keys(s, q, k, vt, dout, bufs.lse, bufs.delta, None, bufs.dk, bufs.dvt, stream)
    else:
        attn_row_terms(s, bufs.o, dout, bufs.delta, stream)
        attn_bwd_keys(s, q, k, vt, dout, bufs.lse, bufs.delta, bufs.ws, bufs.dk, bufs.dvt,
                      stream)
        attn_bwd_queries(s, k, bufs.ws, bufs.dq, stream)
    return bufs


class HostProblem:
    """Pinned host copies of one problem's inputs and outputs, for callers
    whose data lives in host memory."""

    def __init__(self, s: Shape, q, k, vt, dout):
        B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
        pin = lambda t: t.contiguous().pin_memory()
        self.q, self.k, self.vt, self.dout = pin(q), pin(k), pin(vt), pin(dout)
        e = lambda shape, dt: torch.empty(shape, dtype=dt).pin_memory()
        self.o = e((B, T, H * 64), torch.float16)
        self.lse = e((B, H, T), torch.float32)
        self.dq = e((B, H, T, 64), torch.float32)
        self.dk = e((B, Hkv, T, 64), torch.float32)
        self.dvt = e((B, Hkv, 64, T), torch.float32)

    def input_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.vt, self.dout))

    def output_bytes(self) -> int:
        return sum(t.numel() * t.element_size()
                   for t in (self.o, self.lse, self.dq, self.dk, self.dvt))


class DeviceInputs:
    def __init__(self, s: Shape, device=None):
        dev = device or torch.device("cuda")
        B, T, H, Hkv = s.batch, s.seq, s.heads, s.kv_heads
        self.q = torch.empty((B, H, T, 64), dtype=torch.float16, device=dev)
        self.k = torch.empty((B, Hkv, T, 64), dtype=torch.float16, device=dev)
        self.vt = torch.empty(s.v_shape(), dtype=torch.float16, device=dev)
        self.dout = torch.empty((B, H, T, 64), dtype=torch.float16, device=dev)


def device_buffers(dev_in: DeviceInputs, bufs: Buffers) -> AttnDeviceBuffers:
    return AttnDeviceBuffers(dev_in.q.data_ptr(), dev_in.k.data_ptr(), dev_in.vt.data_ptr(),
                             dev_in.dout.data_ptr(), bufs.o.data_ptr(), bufs.lse.data_ptr(),
                             bufs.delta.data_ptr(),
                             None if bufs.ws is None else bufs.ws.data_ptr(),
                             0 if bufs.ws is None else bufs.ws.numel() * bufs.ws.element_size(),
                             bufs.dq.data_ptr(), bufs.dk.data_ptr(), bufs.dvt.data_ptr())


def attn_step_host_order(s: Shape, dev: AttnDeviceBuffers) -> str:
    """'stored' or 'fused': the order attn_step_host takes for ``s`` and ``dev``."""
    shape = s.c_struct()
    r = load_library().attn_step_host_order(ctypes.byref(shape), ctypes.byref(dev))
    if r < 0:
        raise AttnError("attn_step_host_order", r)
    return "fused" if r == ATTN_STEP_FUSED else "stored"


def attn_step_host(s: Shape, host: HostProblem, dev_in: DeviceInputs, bufs: Buffers,
                   stream=None) -> None:
    """Host-to-host pass through the C ABI: copies the inputs in, runs the
    forward and backward calls and copies O, L, dQ, dK and dV^T back, the
    copies overlapped with the kernels (asynchronous; synchronise the stream
    before reading ``host``'s outputs).  ``bufs`` without a workspace, or a
    dQ of 8 MiB or more, selects the fused query pass (attn_step_host_order
    says which)."""
    dev = device_buffers(dev_in, bufs)
    shape = s.c_struct()
    _check("attn_step_host", load_library().attn_step_host(
        ctypes.byref(shape), ctypes.byref(dev), host.q.data_ptr(), host.k.data_ptr(),
        host.vt.data_ptr(), host.dout.data_ptr(), host.o.data_ptr(), host.lse.data_ptr(),
        host.dq.data_ptr(), host.dk.data_ptr(), host.dvt.data_ptr(), _stream_ptr(stream)))


forward_backward_host = attn_step_host

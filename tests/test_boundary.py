"""The C ABI without a GPU: the library loads, exports every entry point that
include/attn.h declares, and rejects bad arguments on the host before any
launch (each rejected call here fails validation, so no pointer is ever
dereferenced and nothing reaches a device)."""
import ctypes
import os
import re

import pytest

from causal_streaming_softmax_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"attn_fwd", "attn_row_terms", "attn_bwd_keys", "attn_bwd_queries",
            "attn_bwd_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def shape(**kw):
    base = dict(batch=1, seq=256, heads=4, kv_heads=2, causal=True, scale=0.125)
    base.update(kw)
    return api.Shape(**base).c_struct()


def fwd(lib, s, ptrs=(0x1000,) * 5):
    return lib.attn_fwd(ctypes.byref(s) if s is not None else None, *ptrs, None)


@pytest.mark.parametrize("kw", [
    dict(seq=0), dict(seq=100), dict(seq=-64), dict(heads=3, kv_heads=2),
    dict(heads=70000, kv_heads=1), dict(kv_heads=0), dict(batch=0), dict(batch=70000),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=float("nan")), dict(scale=float("inf")),
    dict(head_begin=1, head_count=0), dict(head_begin=1, head_count=2),
    dict(head_begin=-1, head_count=1),
])
def test_shape_rejected(lib, kw):
    s = shape(**kw)
    assert fwd(lib, s) == api.ATTN_ERR_SHAPE
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(s)) == 0


def test_head_dim_must_be_64(lib):
    s = shape()
    s.head_dim = 128
    assert fwd(lib, s) == api.ATTN_ERR_SHAPE


def test_causal_flag_is_0_or_1(lib):
    s = shape()
    s.causal = 2
    assert fwd(lib, s) == api.ATTN_ERR_SHAPE


def test_null_and_alignment(lib):
    assert lib.attn_fwd(None, *(0x1000,) * 5, None) == api.ATTN_ERR_NULL
    s = shape()
    assert fwd(lib, s, (0x1000, 0, 0x1000, 0x1000, 0x1000)) == api.ATTN_ERR_NULL
    assert fwd(lib, s, (0x1000, 0x1008, 0x1000, 0x1000, 0x1000)) == api.ATTN_ERR_ALIGN
    assert lib.attn_row_terms(ctypes.byref(s), 0x1000, 0x1001, 0x1000, None) == api.ATTN_ERR_ALIGN
    assert lib.attn_row_terms(ctypes.byref(s), 0x1000, None, 0x1000, None) == api.ATTN_ERR_NULL


def test_workspace_checks(lib):
    s = shape()
    need = lib.attn_bwd_workspace_bytes(ctypes.byref(s))
    p = 0x10000
    args = [p] * 6
    assert lib.attn_bwd_keys(ctypes.byref(s), *args, p, need - 1, p, p, None) == \
        api.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_queries(ctypes.byref(s), p, p, need - 16, p, None) == \
        api.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_keys(ctypes.byref(s), *args, None, need, p, p, None) == api.ATTN_ERR_NULL
    assert lib.attn_bwd_queries(ctypes.byref(s), p, p + 8, need, p, None) == api.ATTN_ERR_ALIGN


@pytest.mark.parametrize("B,T,H,Hkv,causal,count", [
    (1, 4096, 32, 8, True, 0), (1, 16384, 32, 4, True, 0), (16, 4096, 16, 16, False, 0),
    (1, 192, 4, 2, True, 0), (2, 4096, 32, 8, True, 3), (1, 64, 1, 1, False, 0),
])
def test_workspace_bytes_closed_form(lib, B, T, H, Hkv, causal, count):
    s = api.Shape(B, T, H, Hkv, causal=causal, head_begin=0, head_count=count).c_struct()
    nt = -(-T // 128)
    pairs = nt * (nt + 1) // 2 if causal else nt * nt
    heads = (count or Hkv) * (H // Hkv)
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(s)) == B * heads * pairs * 128 * 128 * 2


def test_error_strings(lib):
    for code in range(-8, 1):
        msg = api.error_string(code)
        assert msg and msg != "unknown error"
    assert api.error_string(-99) == "unknown error"


def test_python_binding_checks_types():
    import torch
    s = api.Shape(1, 128, 2, 1)
    cpu = torch.zeros(1, 2, 128, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        api.attn_fwd(s, cpu, cpu, cpu, cpu, cpu)


def test_step_host_rejections(lib):
    """attn_step_host refuses a head chunk, missing buffers and misaligned or
    short device buffers before anything is enqueued."""
    p = 0x1000
    h = [p] * 8  # h_q .. h_dk; h_dvt and the stream follow
    dev = api.AttnDeviceBuffers(p, p, p, p, p, p, p, p, 1 << 40, p, p, p)
    chunk = shape(head_begin=0, head_count=1)
    assert lib.attn_step_host(ctypes.byref(chunk), ctypes.byref(dev), *h, p, None) == \
        api.ATTN_ERR_SHAPE
    s = shape()
    assert lib.attn_step_host(ctypes.byref(s), None, *h, p, None) == api.ATTN_ERR_NULL
    assert lib.attn_step_host(ctypes.byref(s), ctypes.byref(dev), *h, None, None) == \
        api.ATTN_ERR_NULL
    no_ws = api.AttnDeviceBuffers(p, p, p, p, p, p, p, None, 1 << 40, p, p, p)
    assert lib.attn_step_host(ctypes.byref(s), ctypes.byref(no_ws), *h, p, None) == \
        api.ATTN_ERR_NULL
    bad = api.AttnDeviceBuffers(p, p, p, p, p, p, p, p + 8, 1 << 40, p, p, p)
    assert lib.attn_step_host(ctypes.byref(s), ctypes.byref(bad), *h, p, None) == \
        api.ATTN_ERR_ALIGN
    short = api.AttnDeviceBuffers(p, p, p, p, p, p, p, p, 16, p, p, p)
    assert lib.attn_step_host(ctypes.byref(s), ctypes.byref(short), *h, p, None) == \
        api.ATTN_ERR_WORKSPACE


def test_step_host_order(lib):
    """attn_step_host takes the fused order without a workspace and for 8 MiB
    of dQ or more, the stored order otherwise (host-side rule, no launch)."""
    p = 0x1000
    with_ws = api.AttnDeviceBuffers(p, p, p, p, p, p, p, p, 1 << 40, p, p, p)
    no_ws = api.AttnDeviceBuffers(p, p, p, p, p, p, p, None, 0, p, p, p)
    small = api.Shape(1, 256, 4, 2, causal=True)            # dQ 256 KiB
    at_switch = api.Shape(1, 2048, 16, 4, causal=True)      # 8 MiB exactly: fused
    below = api.Shape(1, 2048, 15, 5, causal=False)         # 7.5 MiB
    assert api.attn_step_host_order(small, with_ws) == "stored"
    assert api.attn_step_host_order(small, no_ws) == "fused"
    assert api.attn_step_host_order(at_switch, with_ws) == "fused"
    assert api.attn_step_host_order(below, with_ws) == "stored"
    assert api.attn_step_host_order(api.Shape(4, 4096, 16, 16, causal=False), with_ws) == "fused"
    s = shape()
    assert lib.attn_step_host_order(ctypes.byref(s), None) == api.ATTN_ERR_NULL
    bad = shape(heads=3)
    assert lib.attn_step_host_order(ctypes.byref(bad), ctypes.byref(with_ws)) == \
        api.ATTN_ERR_SHAPE


def test_wait_limit_has_a_floor(lib):
    """The bounded-wait limit reads back as set, is raised to the floor when
    set lower, and 0 restores the default; no GPU is touched."""
    default = api.wait_limit_ns()
    try:
        api.set_wait_limit_ns(3_000_000_000)
        assert api.wait_limit_ns() == 3_000_000_000
        for tiny in (1, 1000, api.MIN_WAIT_LIMIT_NS - 1):
            api.set_wait_limit_ns(tiny)
            assert api.wait_limit_ns() == api.MIN_WAIT_LIMIT_NS
        api.set_wait_limit_ns(0)
        assert api.wait_limit_ns() == 2_000_000_000
    finally:
        api.set_wait_limit_ns(default)


def test_header_constants_match_binding():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    codes = dict(re.findall(r"(ATTN_(?:OK|ERR_\w+|STEP_\w+))\s*=\s*(-?\d+)", text))
    for name, value in codes.items():
        assert getattr(api, name) == int(value), name
    floor = re.search(r"ATTN_MIN_WAIT_LIMIT_NS\s+\(\(uint64_t\)(\d+)\)", text)
    assert floor and int(floor.group(1)) == api.MIN_WAIT_LIMIT_NS

"""attn_bwd_noalloc: the backward without a caller-supplied workspace.

Some callers may not allocate device memory while they run: a plugin or
custom-operator execute step that the host framework forbids from
allocating (it owns all device memory), or a latency-bound loop that cannot
take cudaMalloc's implicit device synchronisation.  For them the library
keeps the key pass's dS scratch in a static device array of
ATTN_NOALLOC_SCRATCH_BYTES.

These tests call that entry point through the C ABI and check its dQ, dK and
dV^T against the allocating entry points (attn_bwd_keys then
attn_bwd_queries with a workspace the caller allocated), within the parity
tolerance, on two calls in a row; and that a shape whose dS does not fit the
array is refused before anything is launched.  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest

from causal_streaming_softmax_gb300 import api, build, workloads
from parity_util import GRAD_TOL, rel_fro

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 128 << 20


def _noalloc_fn():
    build.build()
    lib = api.load_library()
    fn = lib.attn_bwd_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(api.AttnShape)] + [vp] * 10
    fn.restype = ctypes.c_int
    return fn


def _device_problem(B, T, H, Hkv, causal, lens, seed):
    import torch
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=seed)
    dev = "cuda"
    t = {n: torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout")}
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    s = api.Shape(B, T, H, Hkv, causal=causal, seq_lens=ln)
    bufs = api.Buffers(s)
    api.attn_fwd(s, t["q"], t["k"], t["vt"], bufs.o, bufs.lse)
    api.attn_row_terms(s, bufs.o, t["dout"], bufs.delta)
    api.attn_bwd_keys(s, t["q"], t["k"], t["vt"], t["dout"], bufs.lse, bufs.delta, bufs.ws,
                      bufs.dk, bufs.dvt)
    api.attn_bwd_queries(s, t["k"], bufs.ws, bufs.dq)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    ref = {n: getattr(bufs, n).cpu().numpy() for n in ("dq", "dk", "dvt")}
    return s, t, bufs, ref, ln


@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", [
    # one K/V head's dS (4 heads x 528 tiles x 32 KiB = 66 MiB) fits once: two
    # passes over the scratch, one per K/V head
    (1, 4096, 8, 2, True, None),
    (2, 640, 4, 4, False, [300, 640]),
])
def test_noalloc_matches_allocating_path(cuda_device, B, T, H, Hkv, causal, lens):
    import torch
    fn = _noalloc_fn()
    s, t, bufs, ref, ln = _device_problem(B, T, H, Hkv, causal, lens, seed=T + H)
    stream = torch.cuda.current_stream().cuda_stream
    shape = s.c_struct()
    for call in range(2):
        dq, dk, dvt = (torch.full_like(getattr(bufs, n), float("nan"))
                       for n in ("dq", "dk", "dvt"))
        rc = fn(ctypes.byref(shape), t["q"].data_ptr(), t["k"].data_ptr(), t["vt"].data_ptr(),
                t["dout"].data_ptr(), bufs.lse.data_ptr(), bufs.delta.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dvt.data_ptr(), stream)
        assert rc == 0, api.error_string(rc)
        torch.cuda.synchronize()
        assert api.last_device_error() == 0
        got = dict(dq=dq.cpu().numpy(), dk=dk.cpu().numpy(), dvt=dvt.cpu().numpy())
        for n in ("dq", "dk", "dvt"):
            assert np.all(np.isfinite(got[n])), (call, n)
            assert rel_fro(got[n], ref[n]) <= GRAD_TOL, (call, n, rel_fro(got[n], ref[n]))


def test_noalloc_refuses_oversized_shape(cuda_device):
    import torch
    fn = _noalloc_fn()
    # one K/V head with 8 query heads at T = 8192 needs 8 x 2080 x 32 KiB of dS
    B, T, H, Hkv = 1, 8192, 8, 1
    nt = T // 128
    assert B * (H // Hkv) * (nt * (nt + 1) // 2) * 32768 > SCRATCH_BYTES
    s = api.Shape(B, T, H, Hkv, causal=True)
    z = lambda *shape, dt=torch.float16: torch.zeros(shape, dtype=dt, device="cuda")
    q, dout = z(B, H, T, 64), z(B, H, T, 64)
    k, vt = z(B, Hkv, T, 64), z(B, Hkv, 64, T)
    lse, delta = z(B, H, T, dt=torch.float32), z(B, H, T, dt=torch.float32)
    dq, dk, dvt = (z(B, H, T, 64, dt=torch.float32), z(B, Hkv, T, 64, dt=torch.float32),
                   z(B, Hkv, 64, T, dt=torch.float32))
    shape = s.c_struct()
    rc = fn(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), vt.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), delta.data_ptr(), dq.data_ptr(), dk.data_ptr(), dvt.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == api.ATTN_ERR_SCRATCH_LIMIT, api.error_string(rc)
    assert "static scratch" in api.error_string(rc)

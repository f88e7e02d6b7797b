"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle,
compare with the tolerances the method's targets state.

Tolerances (stated for the method): O max-abs <= 2e-3; L max-abs <= 1e-4 in
base-2 units; dQ, dK, dV relative Frobenius <= 1e-2.  D (an intermediate of
the backward) has no stated bound; the one used here follows from the O
bound: |D_gpu - D| <= sum_d |dO_d| * 2e-3 + 1e-5 per row.
"""
import numpy as np

O_TOL = 2e-3
L_TOL = 1e-4
GRAD_TOL = 1e-2


def run_gpu(inp, *, causal, scale=0.125, device="cuda", fused_dq=False):
    import torch
    from causal_streaming_softmax_gb300 import api
    q = torch.from_numpy(inp["q"]).to(device)
    k = torch.from_numpy(inp["k"]).to(device)
    vt = torch.from_numpy(inp["vt"]).to(device)
    dout = torch.from_numpy(inp["dout"]).to(device)
    B, H, T, _ = q.shape
    Hkv = k.shape[1]
    lens = None if inp.get("lens") is None else torch.from_numpy(
        np.ascontiguousarray(inp["lens"], dtype=np.int32)).to(device)
    s = api.Shape(B, T, H, Hkv, causal=causal, scale=scale, seq_lens=lens)
    bufs = api.Buffers(s, workspace=not fused_dq)
    api.forward_backward(s, q, k, vt, dout, bufs, fused_dq=fused_dq)
    torch.cuda.synchronize()
    rc = api.last_device_error()
    assert rc == 0, "device error %d" % rc
    return {name: getattr(bufs, name).cpu().numpy()
            for name in ("o", "lse", "delta", "dq", "dk", "dvt")}


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def compare_full(gpu, ref, inp, *, strict=True):
    """Element-wise comparison of a whole problem.  Returns a dict of metrics;
    asserts the tolerances when ``strict``."""
    q = inp["q"]
    B, H, T, d = q.shape
    lens = inp.get("lens")
    valid = np.ones((B, T), dtype=bool)
    if lens is not None:
        valid = np.arange(T)[None, :] < np.asarray(lens)[:, None]
    o_g = gpu["o"].astype(np.float64).reshape(B, T, H, d)
    o_r = ref["o"].reshape(B, T, H, d)
    vmask = valid[:, :, None, None]
    m = {}
    m["o_max_abs"] = float(np.max(np.abs(o_g - o_r) * vmask))
    m["o_pad_nonzero"] = int(np.count_nonzero(o_g * (~vmask)))
    lv = np.broadcast_to(valid[:, None, :], gpu["lse"].shape)
    m["l_max_abs"] = float(np.max(np.abs(gpu["lse"][lv] - ref["lse"][lv]))) if lv.any() else 0.0
    m["l_pad_not_neginf"] = int(np.count_nonzero(~np.isneginf(gpu["lse"][~lv])))
    dabs = np.abs(inp["dout"].astype(np.float64)).sum(-1)  # [B,H,T]
    dtol = O_TOL * dabs + 1e-5
    m["d_excess"] = float(np.max(np.abs(gpu["delta"] - ref["delta"]) - dtol))
    m["dq_rel"] = rel_fro(gpu["dq"], ref["dq"])
    m["dk_rel"] = rel_fro(gpu["dk"], ref["dk"])
    m["dv_rel"] = rel_fro(gpu["dvt"], ref["dvt"])
    m["nonfinite"] = int(sum(np.count_nonzero(~np.isfinite(gpu[k]))
                             for k in ("o", "delta", "dq", "dk", "dvt")))
    if strict:
        assert m["nonfinite"] == 0, m
        assert m["o_max_abs"] <= O_TOL, m
        assert m["o_pad_nonzero"] == 0, m
        assert m["l_max_abs"] <= L_TOL, m
        assert m["l_pad_not_neginf"] == 0, m
        assert m["d_excess"] <= 0, m
        assert m["dq_rel"] <= GRAD_TOL, m
        assert m["dk_rel"] <= GRAD_TOL, m
        assert m["dv_rel"] <= GRAD_TOL, m
    return m

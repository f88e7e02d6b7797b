"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small shapes are compared element by element over the whole problem (they
span several 128-row tiles and ragged tails); the full-size workloads are
compared on sampled rows and keys that the oracle computes one by one, in
the same launch configuration the benchmark times.
"""
import numpy as np
import pytest

import oracle
from causal_streaming_softmax_gb300 import workloads
from parity_util import GRAD_TOL, L_TOL, O_TOL, compare_full, rel_fro, run_gpu

pytestmark = pytest.mark.gpu


def _full(inp, causal, scale=0.125):
    return oracle.backward(inp["q"], inp["k"], inp["vt"], inp["dout"], causal=causal,
                           scale=scale, lens=inp["lens"])


@pytest.mark.parametrize("cfg", [1, 2])
def test_workload_full(cuda_device, cfg):
    w = workloads.WORKLOADS[cfg]
    inp = workloads.make_inputs(w)
    gpu = run_gpu(inp, causal=w.causal, scale=w.scale)
    compare_full(gpu, _full(inp, w.causal, w.scale), inp)


EDGE = [
    # B, T, H, Hkv, causal, lens
    (1, 64, 1, 1, True, None),          # one 64-row block: half of a 128 tile
    (1, 192, 4, 2, True, None),         # ragged tail
    (1, 320, 8, 1, True, None),         # group 8, several tiles + ragged tail
    (2, 256, 4, 4, False, [1, 256]),    # length 1 and full, non-causal
    (4, 256, 2, 1, False, [63, 64, 65, 200]),
    (3, 384, 4, 2, True, [1, 129, 384]),  # causal with lengths
    (2, 512, 2, 2, True, None),
    # non-causal lengths where the second 128-row tile of a 256-row block has
    # no row (it sees no key) while the first sees five key tiles, more than
    # the forward's K/V stage ring holds
    (2, 1024, 2, 2, False, [600, 1000]),
    (1, 1024, 4, 1, True, [600]),
    # empty sequences in a batch: no row and no key of theirs is valid
    (3, 256, 4, 2, True, [0, 100, 256]),
    (2, 128, 2, 1, False, [0, 128]),
    # more forward work units (256 queries of a head) than SMs: the persistent
    # forward walks several units per CTA; the last block's second query tile
    # holds no row (T = 576)
    (1, 576, 80, 8, True, None),
]


@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", EDGE)
def test_edge_shapes(cuda_device, B, T, H, Hkv, causal, lens):
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + H)
    gpu = run_gpu(inp, causal=causal)
    compare_full(gpu, _full(inp, causal), inp)


def test_sharp_softmax_small(cuda_device):
    """Q ~ N(0, 16) as in the GQA workload, small enough for the full oracle."""
    inp = workloads.make_custom_inputs(1, 512, 8, 2, causal=True, q_std=4.0, seed=33)
    gpu = run_gpu(inp, causal=True)
    compare_full(gpu, _full(inp, True), inp)


def test_other_scale(cuda_device):
    inp = workloads.make_custom_inputs(1, 256, 2, 1, causal=True, seed=5)
    gpu = run_gpu(inp, causal=True, scale=0.3)
    compare_full(gpu, _full(inp, True, 0.3), inp)


def test_deterministic(cuda_device):
    w = workloads.WORKLOADS[2]
    inp = workloads.make_inputs(w)
    a = run_gpu(inp, causal=True)
    b = run_gpu(inp, causal=True)
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=True), key


@pytest.mark.parametrize("fused", [False, True])
def test_back_to_back_steps_with_producer_kernels(cuda_device, fused):
    """Every kernel may start while the one before it in the stream finishes
    (programmatic dependent launch) and waits before touching memory.  Steps
    run back to back with no host synchronisation, each fed by torch kernels
    that write the inputs (and the sequence lengths) right before it, give
    the same bits as steps run one at a time."""
    import torch
    from causal_streaming_softmax_gb300 import api
    B, T, H, Hkv = 2, 640, 8, 2
    sets = [workloads.make_custom_inputs(B, T, H, Hkv, causal=True, lens=ln, seed=40 + i)
            for i, ln in enumerate(([640, 300], [129, 640], [640, 640]))]
    ref = [run_gpu(x, causal=True, fused_dq=fused) for x in sets]
    dev = "cuda"
    src = [{n: torch.from_numpy(x[n]).to(dev) for n in ("q", "k", "vt", "dout")} for x in sets]
    src_lens = [torch.tensor(x["lens"], dtype=torch.int32, device=dev) for x in sets]
    q, k, vt, dout = (torch.empty_like(src[0][n]) for n in ("q", "k", "vt", "dout"))
    lens = torch.empty_like(src_lens[0])
    s = api.Shape(B, T, H, Hkv, causal=True, seq_lens=lens)
    bufs = api.Buffers(s, workspace=not fused)
    got = []
    torch.cuda.synchronize()
    for rep in range(2):
        for i in range(len(sets)):
            # torch kernels (not copies) write every input just before the step
            for n, dst in (("q", q), ("k", k), ("vt", vt), ("dout", dout)):
                torch.mul(src[i][n], 1.0, out=dst)
            torch.add(src_lens[i], 0, out=lens)
            api.forward_backward(s, q, k, vt, dout, bufs, fused_dq=fused)
            got.append({n: getattr(bufs, n).clone() for n in ("o", "lse", "dq", "dk", "dvt")})
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    for j, g in enumerate(got):
        for n, v in g.items():
            assert np.array_equal(v.cpu().numpy(), ref[j % len(sets)][n], equal_nan=True), (j, n)


def test_head_chunks_match_whole(cuda_device):
    """The backward walked in K/V-head chunks (workspace per chunk) gives the
    same bits as one call over every head."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(1, 384, 8, 4, causal=True, seed=9)
    whole = run_gpu(inp, causal=True)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    s = api.Shape(1, 384, 8, 4, causal=True)
    bufs = api.Buffers(s)
    api.attn_fwd(s, q, k, vt, bufs.o, bufs.lse)
    api.attn_row_terms(s, bufs.o, dout, bufs.delta)
    for begin, count in ((0, 1), (1, 2), (3, 1)):
        c = s.chunk(begin, count)
        ws = api.alloc_workspace(c)
        assert ws.numel() == api.workspace_bytes(s) * count // 4
        api.attn_bwd_keys(c, q, k, vt, dout, bufs.lse, bufs.delta, ws, bufs.dk, bufs.dvt)
        api.attn_bwd_queries(c, k, ws, bufs.dq)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    for name in ("dq", "dk", "dvt"):
        assert np.array_equal(getattr(bufs, name).cpu().numpy(), whole[name]), name


def test_wait_timeout_selftest(cuda_device):
    """A bounded wait that nothing completes gives up, reports the timeout, and
    the context stays usable."""
    from causal_streaming_softmax_gb300 import api
    assert api.selftest_wait_timeout(1_000_000) == api.ATTN_ERR_DEVICE_TIMEOUT
    assert api.last_device_error() == 0  # reported once, then cleared
    inp = workloads.make_inputs(workloads.WORKLOADS[1])
    gpu = run_gpu(inp, causal=True)
    compare_full(gpu, _full(inp, True), inp)


def test_workspace_too_small_is_rejected(cuda_device):
    import torch
    from causal_streaming_softmax_gb300 import api
    s = api.Shape(1, 256, 2, 1)
    t = lambda *shape, dt=torch.float16: torch.zeros(shape, dtype=dt, device="cuda")
    ws = torch.empty(api.workspace_bytes(s) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.AttnError) as e:
        api.attn_bwd_keys(s, t(1, 2, 256, 64), t(1, 1, 256, 64), t(1, 1, 64, 256),
                          t(1, 2, 256, 64), t(1, 2, 256, dt=torch.float32),
                          t(1, 2, 256, dt=torch.float32), ws, t(1, 1, 256, 64, dt=torch.float32),
                          t(1, 1, 64, 256, dt=torch.float32))
    assert e.value.code == api.ATTN_ERR_WORKSPACE


# ---------------------------------------------------------------------------
# full-size workloads, compared on samples the oracle computes one by one
# ---------------------------------------------------------------------------
def _sample_rows(T, lens_b, rng, n=40):
    cand = {0, 1, 63, 64, 127, 128, 129, T - 1, T - 2}
    if lens_b is not None:
        cand |= {lens_b - 1, lens_b, min(lens_b + 1, T - 1)}
    cand |= set(rng.integers(0, T, size=n).tolist())
    return np.array(sorted(r for r in cand if 0 <= r < T), dtype=np.int32)


def _check_sampled(w, inp, gpu, heads, kv_heads, batches, rng):
    B, H, T, d = inp["q"].shape
    lens = inp["lens"]
    worst = dict(o=0.0, l=0.0)
    dq_num = dq_den = dk_num = dk_den = dv_num = dv_den = 0.0
    o4 = gpu["o"].astype(np.float64).reshape(B, T, H, d)
    for b in batches:
        lb = None if lens is None else int(lens[b])
        rows = _sample_rows(T, lb, rng)
        for h in heads:
            r = oracle.query_rows(inp["q"], inp["k"], inp["vt"], inp["dout"], b, h, rows,
                                  causal=w.causal, scale=w.scale, lens=lens)
            valid = rows < (T if lb is None else lb)
            og = o4[b, rows, h]
            assert np.all(og[~valid] == 0.0)
            assert np.all(np.isneginf(gpu["lse"][b, h, rows[~valid]]))
            if valid.any():
                worst["o"] = max(worst["o"], float(np.max(np.abs(og[valid] - r["o"][valid]))))
                worst["l"] = max(worst["l"], float(np.max(np.abs(
                    gpu["lse"][b, h, rows[valid]] - r["lse"][valid]))))
                dabs = np.abs(inp["dout"][b, h, rows[valid]].astype(np.float64)).sum(-1)
                assert np.all(np.abs(gpu["delta"][b, h, rows[valid]] - r["delta"][valid])
                              <= O_TOL * dabs + 1e-5)
            dq_num += float(np.sum((gpu["dq"][b, h, rows] - r["dq"]) ** 2))
            dq_den += float(np.sum(r["dq"] ** 2))
        for kv in kv_heads:
            keys = _sample_rows(T, lb, rng, n=24)
            r = oracle.key_rows(inp["q"], inp["k"], inp["vt"], inp["dout"], b, kv, keys,
                                causal=w.causal, scale=w.scale, lens=lens)
            dk_num += float(np.sum((gpu["dk"][b, kv, keys] - r["dk"]) ** 2))
            dk_den += float(np.sum(r["dk"] ** 2))
            dv_num += float(np.sum((gpu["dvt"][b, kv][:, keys].T - r["dv"]) ** 2))
            dv_den += float(np.sum(r["dv"] ** 2))
    assert worst["o"] <= O_TOL, worst
    assert worst["l"] <= L_TOL, worst
    assert np.sqrt(dq_num / dq_den) <= GRAD_TOL
    assert np.sqrt(dk_num / dk_den) <= GRAD_TOL
    assert np.sqrt(dv_num / dv_den) <= GRAD_TOL
    for name in ("o", "delta", "dq", "dk", "dvt"):
        assert np.all(np.isfinite(gpu[name])), name
    return worst


def _sample_plan(w, inp, gpu):
    """Which batches, query heads and K/V heads a full-size workload is
    sampled on; for length-masked workloads also checks that every row and
    key at or past a sequence's length got exact zeros."""
    B, H, G = w.batch, w.heads, w.group
    lens = inp["lens"]
    if lens is None:
        return [0], [0, G - 1, H - 1], [w.kv_heads - 1]
    for b in range(B):
        n = int(lens[b])
        assert np.all(gpu["dk"][b, :, n:] == 0.0)
        assert np.all(gpu["dvt"][b, :, :, n:] == 0.0)
        assert np.all(gpu["dq"][b, :, n:] == 0.0)
        assert np.all(gpu["delta"][b, :, n:] == 0.0)
    batches = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 0, B - 1})
    return batches, [0, H - 1], [0]


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_workload_sampled(cuda_device, cfg):
    w = workloads.WORKLOADS[cfg]
    inp = workloads.make_inputs(w)
    gpu = run_gpu(inp, causal=w.causal, scale=w.scale)
    rng = np.random.default_rng(100 + cfg)
    batches, heads, kv_heads = _sample_plan(w, inp, gpu)
    _check_sampled(w, inp, gpu, heads, kv_heads, batches, rng)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", [
    (1, 512, 8, 2, True, None),
    (3, 384, 4, 2, False, [100, 384, 257]),   # batches: the split dQ copy is strided
    (2, 256, 2, 1, True, None),               # one K/V head: dQ in one piece
])
def test_step_host_matches_device_path(cuda_device, B, T, H, Hkv, causal, lens, fused):
    _step_host_against(B, T, H, Hkv, causal, lens, fused, fused)


def test_step_host_large_dq_takes_fused_order(cuda_device):
    """With a workspace but 8 MiB of dQ, attn_step_host runs the fused order:
    the same bits as the forward, the fused query pass and the key pass."""
    _step_host_against(1, 2048, 16, 4, True, None, False, True)


def _step_host_against(B, T, H, Hkv, causal, lens, fused, expect_fused):
    """attn_step_host (host buffers in and out, copies overlapped with the
    kernels) gives the same bits as the four device calls, with the stored
    or the fused dQ pass."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + B)
    ref = run_gpu(inp, causal=causal, fused_dq=expect_fused)
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    s = api.Shape(B, T, H, Hkv, causal=causal, seq_lens=ln)
    host = api.HostProblem(s, *(torch.from_numpy(inp[n]) for n in ("q", "k", "vt", "dout")))
    dev_in = api.DeviceInputs(s)
    bufs = api.Buffers(s, workspace=not fused)
    for out in (host.o, host.lse, host.dq, host.dk, host.dvt):
        out.fill_(float("nan"))
    stream = torch.cuda.Stream()
    for _ in range(2):
        api.attn_step_host(s, host, dev_in, bufs, stream)
        stream.synchronize()
        assert api.last_device_error() == 0
        got = dict(o=host.o.numpy(), lse=host.lse.numpy(), dq=host.dq.numpy(),
                   dk=host.dk.numpy(), dvt=host.dvt.numpy())
        for name, val in got.items():
            assert np.array_equal(val, ref[name], equal_nan=True), name


# ---------------------------------------------------------------------------
# the fused query pass: dQ with S, P, dP recomputed, the key pass storing no dS
# ---------------------------------------------------------------------------
FUSED = [
    (1, 128, 2, 1, True, None),
    (1, 64, 1, 1, True, None),
    (1, 192, 4, 2, True, None),           # ragged tail: the last query tile is half empty
    (2, 256, 4, 4, False, [1, 256]),
    (4, 256, 2, 1, False, [63, 64, 65, 200]),
    (3, 384, 4, 2, True, [1, 129, 384]),
    (2, 1024, 2, 2, False, [600, 1000]),
    (1, 1024, 8, 8, True, None),
    (3, 256, 4, 2, True, [0, 100, 256]),  # an empty sequence
]


@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", FUSED)
def test_fused_dq_against_oracle(cuda_device, B, T, H, Hkv, causal, lens):
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + 7 * H)
    gpu = run_gpu(inp, causal=causal, fused_dq=True)
    compare_full(gpu, _full(inp, causal), inp)


@pytest.mark.parametrize("causal,Hkv", [(True, 4), (False, 16)])
def test_fused_dq_persistent_against_oracle(cuda_device, causal, Hkv):
    """Enough query tiles (at least two per SM) for the persistent fused query
    pass, with a batch of two and a ragged last tile, element by element."""
    B, T, H = 2, 1216, 16
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, seed=77 + Hkv)
    gpu = run_gpu(inp, causal=causal, fused_dq=True)
    compare_full(gpu, _full(inp, causal), inp)


def test_fused_dq_persistent_same_bits_as_per_tile_launch(cuda_device):
    """Lengths equal to T take the one-CTA-per-tile kernel; without lengths the
    same shape takes the persistent one: the products and sums are the same,
    so are the bits."""
    B, T, H, Hkv = 2, 1216, 16, 4
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=True, seed=81)
    pers = run_gpu(inp, causal=True, fused_dq=True)
    inp_l = dict(inp, lens=np.full(B, T, dtype=np.int32))
    tile = run_gpu(inp_l, causal=True, fused_dq=True)
    for name in ("o", "lse", "delta", "dq", "dk", "dvt"):
        assert np.array_equal(pers[name], tile[name], equal_nan=True), name


def test_fused_dq_sharp_softmax(cuda_device):
    inp = workloads.make_custom_inputs(1, 512, 8, 2, causal=True, q_std=4.0, seed=34)
    gpu = run_gpu(inp, causal=True, fused_dq=True)
    compare_full(gpu, _full(inp, True), inp)


def test_key_pass_without_store_same_bits(cuda_device):
    """The key pass that stores no dS gives the same dK and dV^T bits as the
    one that stores it; the fused query pass is deterministic, and its D
    matches the row-terms kernel's to rounding."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(2, 512, 8, 2, causal=True, lens=[300, 512], seed=12)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    ln = torch.tensor([300, 512], dtype=torch.int32, device=dev)
    s = api.Shape(2, 512, 8, 2, causal=True, seq_lens=ln)
    bufs = api.Buffers(s)
    api.attn_fwd(s, q, k, vt, bufs.o, bufs.lse)
    api.attn_row_terms(s, bufs.o, dout, bufs.delta)
    api.attn_bwd_keys(s, q, k, vt, dout, bufs.lse, bufs.delta, bufs.ws, bufs.dk, bufs.dvt)
    dk1, dvt1 = bufs.dk.clone(), bufs.dvt.clone()
    bufs.dk.fill_(float("nan"))
    bufs.dvt.fill_(float("nan"))
    api.attn_bwd_keys(s, q, k, vt, dout, bufs.lse, bufs.delta, None, bufs.dk, bufs.dvt)
    torch.cuda.synchronize()
    assert torch.equal(dk1, bufs.dk) and torch.equal(dvt1, bufs.dvt)
    d_rows = bufs.delta.clone()
    fused = run_gpu(inp, causal=True, fused_dq=True)
    again = run_gpu(inp, causal=True, fused_dq=True)
    for name in fused:
        assert np.array_equal(fused[name], again[name], equal_nan=True), name
    d_rows = d_rows.cpu().numpy()
    assert np.allclose(fused["delta"], d_rows, rtol=1e-5, atol=1e-6)
    assert np.all(fused["delta"][0, :, 300:] == 0.0)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_fused_dq_workload_sampled(cuda_device, cfg):
    w = workloads.WORKLOADS[cfg]
    inp = workloads.make_inputs(w)
    gpu = run_gpu(inp, causal=w.causal, scale=w.scale, fused_dq=True)
    rng = np.random.default_rng(200 + cfg)
    batches, heads, kv_heads = _sample_plan(w, inp, gpu)
    _check_sampled(w, inp, gpu, heads, kv_heads, batches, rng)


def test_fused_dq_head_chunks_match_whole(cuda_device):
    """The fused query pass walked in K/V-head chunks gives the same bits as
    one call over every head."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(2, 384, 8, 4, causal=True, lens=[200, 384], seed=19)
    whole = run_gpu(inp, causal=True, fused_dq=True)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    ln = torch.tensor([200, 384], dtype=torch.int32, device=dev)
    s = api.Shape(2, 384, 8, 4, causal=True, seq_lens=ln)
    bufs = api.Buffers(s, workspace=False)
    api.attn_fwd(s, q, k, vt, bufs.o, bufs.lse)
    bufs.dq.fill_(float("nan"))
    bufs.delta.fill_(float("nan"))
    for begin, count in ((0, 1), (1, 2), (3, 1)):
        api.attn_bwd_queries_fused(s.chunk(begin, count), q, k, vt, dout, bufs.o, bufs.lse,
                                   bufs.delta, bufs.dq)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    assert np.array_equal(bufs.dq.cpu().numpy(), whole["dq"])
    assert np.array_equal(bufs.delta.cpu().numpy(), whole["delta"])


def test_fused_dq_persistent_head_chunks_match_whole(cuda_device):
    """The persistent fused query pass (at least two units per SM in every
    chunk) walked in K/V-head chunks gives the same bits as one call."""
    import torch
    from causal_streaming_softmax_gb300 import api
    B, T, H, Hkv = 2, 1216, 32, 8
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=True, seed=23)
    whole = run_gpu(inp, causal=True, fused_dq=True)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    s = api.Shape(B, T, H, Hkv, causal=True)
    bufs = api.Buffers(s, workspace=False)
    api.attn_fwd(s, q, k, vt, bufs.o, bufs.lse)
    bufs.dq.fill_(float("nan"))
    bufs.delta.fill_(float("nan"))
    for begin, count in ((0, 4), (4, 4)):
        api.attn_bwd_queries_fused(s.chunk(begin, count), q, k, vt, dout, bufs.o, bufs.lse,
                                   bufs.delta, bufs.dq)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    assert np.array_equal(bufs.dq.cpu().numpy(), whole["dq"])
    assert np.array_equal(bufs.delta.cpu().numpy(), whole["delta"])


# ---------------------------------------------------------------------------
# the dQ pass with the inverse half-split rotation (bfloat16, token-major)
# ---------------------------------------------------------------------------
def _bf16_rne(x32):
    b = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", [
    (1, 512, 8, 2, True, None),
    (2, 384, 4, 2, False, [100, 384]),
])
def test_rotated_dq(cuda_device, B, T, H, Hkv, causal, lens):
    """attn_bwd_queries_rotated against the oracle's dQ turned back by the
    inverse rotation, and bit for bit (to one bfloat16 step) against the same
    epilogue applied on the host to the plain pass's binary32 dQ; written as
    a column block of a wider token-major buffer whose other columns stay."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + 3 * H)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    s = api.Shape(B, T, H, Hkv, causal=causal, seq_lens=ln)
    bufs = api.Buffers(s)
    api.forward_backward(s, q, k, vt, dout, bufs)
    rng = np.random.default_rng(5)
    theta = rng.uniform(-np.pi, np.pi, size=(T, 32))
    cos = torch.tensor(np.cos(theta), dtype=torch.float32, device=dev)
    sin = torch.tensor(np.sin(theta), dtype=torch.float32, device=dev)
    width, col0 = H * 64 + 3 * 64 + 16, 64 + 8          # a wider projection gradient
    wide = torch.full((B, T, width), 7.0, dtype=torch.bfloat16, device=dev)
    api.attn_bwd_queries_rotated(s, k, bufs.ws, cos, sin, wide[:, :, col0:], ld=width)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    got = wide.float().cpu().numpy()
    assert np.all(got[:, :, :col0] == 7.0) and np.all(got[:, :, col0 + H * 64:] == 7.0)
    got = got[:, :, col0:col0 + H * 64]
    # against the oracle
    ref = oracle.backward(inp["q"], inp["k"], inp["vt"], inp["dout"], causal=causal,
                          scale=0.125, lens=inp["lens"])
    rot_ref = oracle.inverse_rotate(ref["dq"], cos.cpu().numpy(), sin.cpu().numpy())
    assert rel_fro(got, rot_ref) <= GRAD_TOL
    # against the epilogue on the host, from the plain pass's binary32 dQ
    x = bufs.dq.cpu().numpy().astype(np.float32)              # [B][H][T][64] = s * sum
    c = cos.cpu().numpy()[None, None].astype(np.float64)
    sn = sin.cpu().numpy()[None, None].astype(np.float64)
    x1, x2 = x[..., :32].astype(np.float64), x[..., 32:].astype(np.float64)
    p2 = (x2 * sn).astype(np.float32).astype(np.float64)
    p1 = (x1 * sn).astype(np.float32).astype(np.float64)
    o = np.concatenate([(x1 * c + p2).astype(np.float32), (x2 * c - p1).astype(np.float32)], -1)
    emu = _bf16_rne(o).transpose(0, 2, 1, 3).reshape(B, T, H * 64)
    step = np.abs(emu.astype(np.float64)) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - emu) <= step)
    assert np.mean(got == emu) > 0.999


# ---------------------------------------------------------------------------
# projection-fused epilogues: dQ, dK, dV written token-major, binary32 + bf16
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("store_ds", [True, False])
@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", [
    (1, 384, 8, 2, True, None),
    (2, 320, 4, 4, False, [100, 320]),
])
def test_projection_epilogues(cuda_device, B, T, H, Hkv, causal, lens, store_ds):
    """The projection blocks hold exactly the plain passes' dQ, dK and dV
    (dV untransposed) in binary32, their round-to-nearest-even bfloat16, and
    nothing outside the blocks changes; both blocks also match the oracle's
    gradients laid out token-major within the gradient tolerance."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + H)
    dev = "cuda"
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    s = api.Shape(B, T, H, Hkv, causal=causal, seq_lens=ln)
    bufs = api.Buffers(s)
    api.forward_backward(s, q, k, vt, dout, bufs)
    # a fused QKV gradient [B][T][width]: Q block, then K, then V, with padding
    width = (H + 2 * Hkv) * 64 + 32
    cq, ck, cv = 8, 8 + H * 64, 8 + (H + Hkv) * 64
    g32 = torch.full((B, T, width), -3.0, dtype=torch.float32, device=dev)
    g16 = torch.full((B, T, width), -3.0, dtype=torch.bfloat16, device=dev)
    blk = lambda c0: api.projection(g32[:, :, c0:], g16[:, :, c0:], width)
    ws = bufs.ws if store_ds else None
    api.attn_bwd_keys_projected(s, q, k, vt, dout, bufs.lse, bufs.delta, ws, blk(ck), blk(cv))
    api.attn_bwd_queries_projected(s, k, bufs.ws, blk(cq))
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    a32 = g32.cpu().numpy()
    a16 = g16.float().cpu().numpy()
    want_q = bufs.dq.cpu().numpy().transpose(0, 2, 1, 3).reshape(B, T, H * 64)
    want_k = bufs.dk.cpu().numpy().transpose(0, 2, 1, 3).reshape(B, T, Hkv * 64)
    want_v = bufs.dvt.cpu().numpy().transpose(0, 3, 1, 2).reshape(B, T, Hkv * 64)
    for c0, want in ((cq, want_q), (ck, want_k), (cv, want_v)):
        n = want.shape[2]
        assert np.array_equal(a32[:, :, c0:c0 + n], want)
        assert np.array_equal(a16[:, :, c0:c0 + n], _bf16_rne(want))
    # and against the oracle directly, in the same token-major layout: the
    # blocks must be the gradients, not only equal to another CUDA pass
    ref = _full(inp, causal)
    ref_q = ref["dq"].transpose(0, 2, 1, 3).reshape(B, T, H * 64)
    ref_k = ref["dk"].transpose(0, 2, 1, 3).reshape(B, T, Hkv * 64)
    ref_v = ref["dvt"].transpose(0, 3, 1, 2).reshape(B, T, Hkv * 64)
    for c0, want in ((cq, ref_q), (ck, ref_k), (cv, ref_v)):
        n = want.shape[2]
        assert rel_fro(a32[:, :, c0:c0 + n], want) <= GRAD_TOL
        assert rel_fro(a16[:, :, c0:c0 + n], want) <= GRAD_TOL
    for arr in (a32, a16):
        assert np.all(arr[:, :, :cq] == -3.0) and np.all(arr[:, :, cv + Hkv * 64:] == -3.0)


# ---------------------------------------------------------------------------
# V given as rows [B][Hkv][T][64] instead of V^T
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", [
    (1, 512, 8, 2, True, None),
    (2, 320, 4, 4, False, [100, 320]),
    (2, 1216, 16, 4, True, None),    # enough query tiles for the persistent passes
])
def test_v_rows_layout(cuda_device, B, T, H, Hkv, causal, lens, fused):
    """The whole path with V as rows gives the same bits as with V^T (the
    operands are the same values read through another descriptor), and
    matches the oracle."""
    import torch
    from causal_streaming_softmax_gb300 import api
    inp = workloads.make_custom_inputs(B, T, H, Hkv, causal=causal, lens=lens, seed=T + 9)
    ref = run_gpu(inp, causal=causal, fused_dq=fused)
    dev = "cuda"
    q, k, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "dout"))
    v = torch.from_numpy(np.ascontiguousarray(inp["vt"].transpose(0, 1, 3, 2))).to(dev)
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=dev)
    s = api.Shape(B, T, H, Hkv, causal=causal, seq_lens=ln, v_rows=True)
    bufs = api.Buffers(s, workspace=not fused)
    api.forward_backward(s, q, k, v, dout, bufs, fused_dq=fused)
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    for name in ("o", "lse", "delta", "dq", "dk", "dvt"):
        assert np.array_equal(getattr(bufs, name).cpu().numpy(), ref[name], equal_nan=True), name
    compare_full(ref, _full(inp, causal), inp)

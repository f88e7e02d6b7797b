"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a missing group sum, a wrong
log base) fails at least one of them:

* a hand-worked example (tests/golden/hand_example.json);
* central finite differences of f = sum(O * dO) in binary64;
* torch's scaled_dot_product_attention and autograd in float64 (a library
  routine independent of the oracle's C code);
* closed forms for Q = 0 and for T = 1;
* grouped-query attention equal to multi-head with repeated K/V;
* invariants: probability rows sum to 1, D_i = sum_j P_ij dP_ij,
  sum_j dK_j = 0;
* the sampled entry points equal the full pass.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
LN2 = math.log(2.0)


def rand_inputs(B, T, H, Hkv, d, seed, std=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, H, T, d)) * std, rng.standard_normal((B, Hkv, T, d)),
            rng.standard_normal((B, Hkv, d, T)), rng.standard_normal((B, H, T, d)))


def test_hand_worked_example():
    g = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    inp, exp = g["inputs"], g["expected"]
    out = oracle.backward(np.array(inp["q"]), np.array(inp["k"]), np.array(inp["vt"]),
                          np.array(inp["dout"]), causal=inp["causal"], scale=inp["scale"])
    for key in ("o", "lse", "delta", "dq", "dk", "dvt"):
        np.testing.assert_allclose(out[key], np.array(exp[key]), rtol=0, atol=1e-12,
                                   err_msg=key)


def f_value(q, k, vt, dout, causal, scale, lens):
    """f = sum over valid rows of O . dO (O in [B][T][H*d], dO in [B][H][T][d])."""
    o, _ = oracle.forward(q, k, vt, causal=causal, scale=scale, lens=lens)
    B, H, T, d = q.shape
    o4 = o.reshape(B, T, H, d).transpose(0, 2, 1, 3)
    return float(np.sum(o4 * dout))


FD_CASES = [
    # B, T, H, Hkv, d, causal, lens
    (1, 1, 2, 1, 4, True, None),
    (1, 3, 2, 1, 4, True, None),
    (1, 5, 2, 1, 4, True, None),
    (1, 17, 2, 1, 4, True, None),
    (1, 5, 2, 1, 64, True, None),
    (2, 5, 2, 1, 4, False, [3, 5]),
    (2, 6, 4, 2, 4, True, [4, 6]),
]


@pytest.mark.parametrize("B,T,H,Hkv,d,causal,lens", FD_CASES)
def test_finite_differences(B, T, H, Hkv, d, causal, lens):
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=T * 31 + d + H)
    scale = 0.37
    out = oracle.backward(q, k, vt, dout, causal=causal, scale=scale, lens=lens)
    h = 1e-6
    rng = np.random.default_rng(7)
    for name, arr, grad in (("q", q, out["dq"]), ("k", k, out["dk"]), ("vt", vt, out["dvt"])):
        flat = arr.reshape(-1)
        idx = np.arange(flat.size)
        if flat.size > 160:
            idx = rng.choice(flat.size, 160, replace=False)
        for t in idx:
            old = flat[t]
            flat[t] = old + h
            fp = f_value(q, k, vt, dout, causal, scale, lens)
            flat[t] = old - h
            fm = f_value(q, k, vt, dout, causal, scale, lens)
            flat[t] = old
            fd = (fp - fm) / (2 * h)
            an = grad.reshape(-1)[t]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, t, fd, an)


def torch_reference(q, k, vt, dout, causal, scale, lens):
    """float64 torch SDPA + autograd; returns per-valid-row results."""
    torch = pytest.importorskip("torch")
    B, H, T, d = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(np.swapaxes(vt, 2, 3).copy(), dtype=torch.float64, requires_grad=True)
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    masks = []
    for b in range(B):
        n = T if lens is None else int(lens[b])
        m = (i < n) & (j < n)
        if causal:
            m = m & (j <= i)
        masks.append(m)
    mask = torch.stack(masks)[:, None]  # [B,1,T,T]
    valid_row = mask.any(-1)  # [B,1,T]
    # rows with no valid key: give them one dummy key, zero their outputs after
    safe = mask | (~valid_row)[..., None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=safe, scale=scale)
    o = torch.where(valid_row[..., None], o, torch.zeros_like(o))
    s = (tq @ kk.transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1) / LN2
    (o * torch.tensor(dout)).sum().backward()
    return dict(o=o.detach().numpy(), lse=lse.detach().numpy(), dq=tq.grad.numpy(),
                dk=tk.grad.numpy(), dvt=np.swapaxes(tv.grad.numpy(), 2, 3),
                valid=valid_row[:, 0].numpy())


TORCH_CASES = [
    (1, 64, 2, 1, True, None),
    (1, 96, 4, 4, True, None),
    (2, 80, 4, 2, False, [17, 80]),
    (3, 48, 8, 2, True, [1, 30, 48]),
]


@pytest.mark.parametrize("B,T,H,Hkv,causal,lens", TORCH_CASES)
def test_against_torch_sdpa(B, T, H, Hkv, causal, lens):
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, 64, seed=B * 1000 + T, std=2.0)
    scale = 0.125
    ref = torch_reference(q, k, vt, dout, causal, scale, lens)
    out = oracle.backward(q, k, vt, dout, causal=causal, scale=scale, lens=lens)
    o4 = out["o"].reshape(B, T, H, 64).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(o4, ref["o"], atol=1e-12, rtol=1e-10)
    valid = np.broadcast_to(ref["valid"][:, None, :], out["lse"].shape)
    np.testing.assert_allclose(out["lse"][valid], ref["lse"][valid], atol=1e-12, rtol=1e-12)
    assert np.all(np.isneginf(out["lse"][~valid]))
    for key in ("dq", "dk", "dvt"):
        np.testing.assert_allclose(out[key], ref[key], atol=1e-11, rtol=1e-9, err_msg=key)


def test_q_zero_closed_form_causal():
    B, T, H, Hkv, d = 1, 37, 4, 2, 8
    _, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=3)
    q = np.zeros((B, H, T, d))
    out = oracle.backward(q, k, vt, dout, causal=True, scale=0.3)
    G = H // Hkv
    o4 = out["o"].reshape(B, T, H, d)
    for h in range(H):
        v = vt[0, h // G].T  # [T][d]
        prefix_mean = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
        np.testing.assert_allclose(o4[0, :, h], prefix_mean, atol=1e-12)
        np.testing.assert_allclose(out["lse"][0, h], np.log2(np.arange(1, T + 1)), atol=1e-12)
    # dV_j = sum_{h in group} sum_{i >= j} dO_i / (i + 1)
    for kv in range(Hkv):
        acc = np.zeros((T, d))
        for g in range(G):
            w = dout[0, kv * G + g] / np.arange(1, T + 1)[:, None]
            acc += np.cumsum(w[::-1], axis=0)[::-1]
        np.testing.assert_allclose(out["dvt"][0, kv].T, acc, atol=1e-12)


def test_q_zero_closed_form_varlen_noncausal():
    B, T, H, d = 2, 20, 2, 8
    lens = [7, 20]
    _, k, vt, dout = rand_inputs(B, T, H, H, d, seed=4)
    q = np.zeros((B, H, T, d))
    out = oracle.backward(q, k, vt, dout, causal=False, scale=0.3, lens=lens)
    o4 = out["o"].reshape(B, T, H, d)
    for b in range(B):
        n = lens[b]
        for h in range(H):
            mean = vt[b, h, :, :n].mean(axis=1)
            np.testing.assert_allclose(o4[b, :n, h], np.broadcast_to(mean, (n, d)), atol=1e-12)
            assert np.all(o4[b, n:, h] == 0.0)
            np.testing.assert_allclose(out["lse"][b, h, :n], math.log2(n), atol=1e-12)
            assert np.all(np.isneginf(out["lse"][b, h, n:]))
            assert np.all(out["delta"][b, h, n:] == 0.0)
            assert np.all(out["dq"][b, h, n:] == 0.0)
            assert np.all(out["dk"][b, h, n:] == 0.0)
            assert np.all(out["dvt"][b, h, :, n:] == 0.0)


def test_single_token():
    B, T, H, Hkv, d = 2, 1, 4, 2, 16
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=5)
    scale = 0.125
    out = oracle.backward(q, k, vt, dout, causal=True, scale=scale)
    G = H // Hkv
    o4 = out["o"].reshape(B, T, H, d)
    for b in range(B):
        for h in range(H):
            kv = h // G
            np.testing.assert_allclose(o4[b, 0, h], vt[b, kv, :, 0], atol=1e-14)
            np.testing.assert_allclose(out["lse"][b, h, 0],
                                       scale * q[b, h, 0] @ k[b, kv, 0] / LN2, atol=1e-12)
            np.testing.assert_allclose(out["delta"][b, h, 0], dout[b, h, 0] @ vt[b, kv, :, 0],
                                       atol=1e-12)
    assert np.all(out["dq"] == 0.0)
    np.testing.assert_allclose(out["dk"], 0.0, atol=1e-15)
    for kv in range(Hkv):
        np.testing.assert_allclose(out["dvt"][:, kv, :, 0],
                                   dout[:, kv * G:(kv + 1) * G, 0].sum(axis=1), atol=1e-14)


def test_gqa_equals_mha_with_repeated_kv():
    B, T, H, Hkv, d = 1, 33, 8, 2, 16
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=6)
    G = H // Hkv
    gqa = oracle.backward(q, k, vt, dout, causal=True, scale=0.2)
    mha = oracle.backward(q, np.repeat(k, G, axis=1), np.repeat(vt, G, axis=1), dout,
                          causal=True, scale=0.2)
    for key in ("o", "lse", "delta", "dq"):
        np.testing.assert_allclose(gqa[key], mha[key], atol=1e-13, err_msg=key)
    np.testing.assert_allclose(gqa["dk"], mha["dk"].reshape(B, Hkv, G, T, d).sum(2), atol=1e-12)
    np.testing.assert_allclose(gqa["dvt"], mha["dvt"].reshape(B, Hkv, G, d, T).sum(2), atol=1e-12)


def test_invariants():
    B, T, H, Hkv, d = 2, 29, 4, 2, 16
    lens = [29, 11]
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=8, std=1.5)
    out = oracle.backward(q, k, vt, dout, causal=True, scale=0.25, lens=lens)
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            for i in (0, 5, lens[b] - 1):
                p = oracle.probs_row(q, k, vt, b, h, i, causal=True, scale=0.25, lens=lens)
                assert abs(p.sum() - 1.0) < 1e-13
                assert np.all(p[i + 1:] == 0.0)  # causal: nothing past the diagonal
                dP = vt[b, h // G].T @ dout[b, h, i]  # dP_ij = dO_i . v_j
                np.testing.assert_allclose(out["delta"][b, h, i], p @ dP, atol=1e-12)
        # sum_j dS_ij = 0 for every row, so sum_j dK_j = 0 for every K/V head
        np.testing.assert_allclose(out["dk"][b].sum(axis=1), 0.0, atol=1e-11)


def test_sampled_entry_points_match_full():
    B, T, H, Hkv, d = 2, 45, 4, 2, 64
    lens = [45, 30]
    q, k, vt, dout = rand_inputs(B, T, H, Hkv, d, seed=9)
    for causal in (True, False):
        full = oracle.backward(q, k, vt, dout, causal=causal, scale=0.125, lens=lens)
        rows = np.array([0, 1, 29, 30, 44])
        for b in range(B):
            for h in (0, 3):
                r = oracle.query_rows(q, k, vt, dout, b, h, rows, causal=causal, scale=0.125,
                                      lens=lens)
                o4 = full["o"].reshape(B, T, H, d)
                np.testing.assert_array_equal(r["o"], o4[b, rows, h])
                np.testing.assert_array_equal(r["lse"], full["lse"][b, h, rows])
                np.testing.assert_array_equal(r["delta"], full["delta"][b, h, rows])
                np.testing.assert_array_equal(r["dq"], full["dq"][b, h, rows])
            kr = oracle.key_rows(q, k, vt, dout, b, 1, rows, causal=causal, scale=0.125,
                                 lens=lens)
            np.testing.assert_allclose(kr["dk"], full["dk"][b, 1, rows], atol=1e-13)
            np.testing.assert_allclose(kr["dv"], full["dvt"][b, 1][:, rows].T, atol=1e-13)


# ---------------------------------------------------------------------------
# the inverse half-split rotation of the rotated dQ epilogue
# ---------------------------------------------------------------------------
def _rope_tables(T, seed):
    rng = np.random.default_rng(seed)
    theta = rng.uniform(-np.pi, np.pi, size=(T, 32))
    return np.cos(theta), np.sin(theta), theta


def test_inverse_rotate_identity_and_quarter_turn():
    """cos = 1, sin = 0 is a pure relayout to token-major; a quarter turn
    (cos = 0, sin = 1) maps each pair (a, b) to (b, -a)."""
    rng = np.random.default_rng(3)
    B, H, T = 2, 3, 5
    dq = rng.standard_normal((B, H, T, 64))
    out = oracle.inverse_rotate(dq, np.ones((T, 32)), np.zeros((T, 32)))
    assert np.array_equal(out.reshape(B, T, H, 64), dq.transpose(0, 2, 1, 3))
    out = oracle.inverse_rotate(dq, np.zeros((T, 32)), np.ones((T, 32))).reshape(B, T, H, 64)
    tm = dq.transpose(0, 2, 1, 3)
    assert np.array_equal(out[..., :32], tm[..., 32:])
    assert np.array_equal(out[..., 32:], -tm[..., :32])


def test_inverse_rotate_is_the_pullback_of_the_forward_rotation():
    """The epilogue's rotation is the gradient of the forward half-split
    rotary embedding (each (x_c, x_{c+32}) pair turned by theta_c), taken
    here by torch autograd on that forward map; it also undoes the forward
    map and keeps each pair's length."""
    torch = pytest.importorskip("torch")
    T = 7
    cos, sin, theta = _rope_tables(T, 11)
    rng = np.random.default_rng(12)
    x = torch.tensor(rng.standard_normal((1, 1, T, 64)), dtype=torch.float64,
                     requires_grad=True)
    g = rng.standard_normal((1, 1, T, 64))
    c = torch.tensor(cos, dtype=torch.float64)
    s = torch.tensor(sin, dtype=torch.float64)
    x1, x2 = x[..., :32], x[..., 32:]
    rot = torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)  # forward rotary map
    (rot * torch.tensor(g)).sum().backward()
    pull = oracle.inverse_rotate(g, cos, sin).reshape(1, T, 1, 64).transpose(0, 2, 1, 3)
    assert np.allclose(pull, x.grad.numpy(), rtol=0, atol=1e-14)
    back = oracle.inverse_rotate(rot.detach().numpy(), cos, sin).reshape(1, T, 1, 64)
    assert np.allclose(back.transpose(0, 2, 1, 3), x.detach().numpy(), rtol=0, atol=1e-13)
    gi = oracle.inverse_rotate(g, cos, sin).reshape(T, 64)
    g2 = g.reshape(T, 64)
    assert np.allclose(gi[:, :32] ** 2 + gi[:, 32:] ** 2, g2[:, :32] ** 2 + g2[:, 32:] ** 2)

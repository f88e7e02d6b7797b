"""The two arithmetic steps every kernel builds on, checked on the device.

P is rounded to binary16 before its product with V (the precision contract of
the streaming forward) and P = 2^t is taken with the hardware exponential.
attn_selftest_arith runs exactly the library's inline forms of both over a
float32 array.  The packing must match numpy's binary32 -> binary16 rounding
(round to nearest, ties to even) bit for bit, including signed zeros,
binary16 subnormals, exact ties and overflow to infinity; the exponential must
stay within a relative error of 2^-21 of 2^x over the range a softmax uses
(t <= 0 down to the underflow point), give exactly 1 at 0 and 0 at -inf, and
flush results below the binary32 normal range to zero.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _run(x):
    import torch
    from causal_streaming_softmax_gb300 import api
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    packed, e2 = api.selftest_arith(xt)
    return packed.cpu().numpy().view(np.uint32), e2.cpu().numpy()


def _expected_pack(x):
    with np.errstate(over="ignore"):
        h = x.astype(np.float32).astype(np.float16).view(np.uint16).astype(np.uint32)
    return h[0::2] | (h[1::2] << 16)


def _f16_ties(rng, n):
    """float32 values exactly halfway between neighbouring binary16 numbers."""
    a = rng.integers(0, 0x7BFF, size=n).astype(np.uint16)  # finite, not the largest
    lo = a.view(np.float16).astype(np.float64)
    hi = (a + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)  # exact in binary32
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    return mid * sign


def test_f16_packing_is_round_to_nearest_even(cuda_device):
    rng = np.random.default_rng(7)
    special = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, -65504.0, 65519.996, 65520.0, -65520.0,
                        70000.0, np.inf, -np.inf, 6.1035156e-05, 5.9604645e-08, 2.9802322e-08,
                        2.9802326e-08, -2.9802326e-08, 1e-9, -1e-9, 1.4e-45, 0.5, 2049.0,
                        2051.0, 1.0009766, 1.0004883, 1.0014648, 3.0e-5, -4.5e-6],
                       dtype=np.float32)
    x = np.concatenate([
        special,
        rng.standard_normal(20000).astype(np.float32),
        (rng.random(20000) * 2.0 ** rng.integers(-30, 17, size=20000)).astype(np.float32),
        _f16_ties(rng, 20000),
        rng.uniform(-2.0 ** -14, 2.0 ** -14, size=4000).astype(np.float32),  # f16 subnormals
    ])
    if x.size % 2:
        x = np.append(x, np.float32(0.25))
    got, _ = _run(x)
    want = _expected_pack(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[2 * i]), float(x[2 * i + 1]), hex(got[i]), hex(want[i]))
                           for i in bad[:5]]


def test_f16_packing_nan_stays_nan(cuda_device):
    x = np.array([np.nan, 1.0, -2.0, -np.nan], dtype=np.float32)
    got, _ = _run(x)
    h = np.stack([got & 0xFFFF, got >> 16], axis=1).reshape(-1).astype(np.uint16)
    v = h.view(np.float16)
    assert np.isnan(v[0]) and v[1] == 1.0 and v[2] == -2.0 and np.isnan(v[3])


def test_ex2_relative_error_bound(cuda_device):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.uniform(-126.0, 0.0, size=200000),
        rng.uniform(-1.0, 1.0, size=100000),
        -rng.random(50000) * 2.0 ** -20,      # arguments near 0, where P is near 1
        -np.arange(0, 127, dtype=np.float64),  # exact powers of two
        np.array([0.5, -0.5, 1.0 / 3.0]),
    ]).astype(np.float32)
    if x.size % 2:
        x = np.append(x, np.float32(-3.0))
    _, e2 = _run(x)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(e2.astype(np.float64) - want) / want
    worst = float(rel.max())
    assert worst <= 2.0 ** -21, (worst, float(x[np.argmax(rel)]))


def test_ex2_special_values(cuda_device):
    x = np.array([0.0, -0.0, -np.inf, -200.0, -127.5, -150.0, 1.0, -1.0], dtype=np.float32)
    _, e2 = _run(x)
    assert e2[0] == 1.0 and e2[1] == 1.0
    assert e2[2] == 0.0
    assert e2[3] == 0.0 and e2[5] == 0.0  # below the binary32 normal range: flushed
    assert e2[4] == 0.0 or e2[4] >= np.float32(2.0 ** -126)
    assert abs(e2[6] - 2.0) <= 2.0 ** -20 and abs(e2[7] - 0.5) <= 2.0 ** -22


def test_selftest_arith_rejects_odd_length(cuda_device):
    import ctypes

    from causal_streaming_softmax_gb300 import api
    lib = api.load_library()
    assert lib.attn_selftest_arith(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000),
                                   ctypes.c_void_p(0x1000), 3, None) == api.ATTN_ERR_SHAPE

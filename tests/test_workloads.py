"""The seeded input generator: shapes, dtypes, determinism, length range."""
import numpy as np

from causal_streaming_softmax_gb300 import workloads


def test_shapes_and_dtypes():
    w = workloads.WORKLOADS[1]
    x = workloads.make_inputs(w)
    assert x["q"].shape == (1, 2, 128, 64) and x["q"].dtype == np.float16
    assert x["k"].shape == (1, 1, 128, 64)
    assert x["vt"].shape == (1, 1, 64, 128)
    assert x["dout"].shape == (1, 2, 128, 64)
    assert x["lens"] is None


def test_deterministic_and_seeded():
    w = workloads.WORKLOADS[2]
    a, b = workloads.make_inputs(w), workloads.make_inputs(w)
    for k in ("q", "k", "vt", "dout"):
        assert np.array_equal(a[k], b[k])
    c = workloads.make_inputs(w, seed=99)
    assert not np.array_equal(a["q"], c["q"])


def test_varlen_lengths():
    w = workloads.WORKLOADS[4]
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lens = rng.integers(256, 4096, size=16, endpoint=True)
    assert lens.min() >= 256 and lens.max() <= 4096
    # the generator draws the lengths first, from the same stream
    x = workloads.make_inputs(workloads.Workload("t", 16, 128, 1, 1, False, varlen=True,
                                                 seed=w.seed))
    assert np.array_equal(x["lens"], lens.astype(np.int32))


def test_sharp_q_scaling():
    w = workloads.WORKLOADS[1]
    sharp = workloads.Workload(w.name, w.batch, w.seq, w.heads, w.kv_heads, w.causal,
                               q_std=4.0, seed=w.seed)
    a, b = workloads.make_inputs(w), workloads.make_inputs(sharp)
    np.testing.assert_allclose(b["q"].astype(np.float32), 4 * a["q"].astype(np.float32),
                               rtol=1e-3, atol=1e-3)
    assert np.array_equal(a["k"], b["k"])

"""bench.py's host-side arithmetic without a GPU: the useful-FLOP count the
metric is quoted in, the algorithmic bytes behind the roofline, and the rule
that recorded DRAM traffic is used only for the kernel source it was taken on."""
import ctypes
import os

import numpy as np
import pytest

import bench
from causal_streaming_softmax_gb300 import api, build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_useful_flops_causal_closed_form():
    w = workloads.WORKLOADS[3]
    f = bench.useful_flops(w, None)
    # 4 B H d T^2 / 2 for the forward (two products of 2 d flops per visible pair)
    assert f["fwd"] == 4.0 * 1 * 32 * 64 * 4096 * 4096 / 2
    assert f["keys"] == 2 * f["fwd"] and f["queries"] == 0.5 * f["fwd"]
    assert f["step"] == f["fwd"] + f["keys"] + f["queries"] == 3.5 * f["fwd"]


def test_useful_flops_lengths_count_visible_pairs():
    # non-causal with lengths: every (query, key) pair inside a sequence counts
    w = workloads.Workload("t", 3, 256, 4, 2, False, seed=0)
    lens = np.array([1, 100, 256])
    f = bench.useful_flops(w, lens)
    pairs = sum(int(n) * int(n) for n in lens)
    assert f["fwd"] == 4.0 * 64 * 4 * pairs
    # the same count summed pair by pair on a tiny case
    w2 = workloads.Workload("t", 2, 64, 1, 1, False, seed=0)
    lens2 = np.array([3, 5])
    brute = sum(1 for b, n in enumerate(lens2) for i in range(n) for j in range(n))
    assert bench.useful_flops(w2, lens2)["fwd"] == 4.0 * 64 * brute


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_algorithmic_bytes_workspace_matches_library(lib, cfg):
    # the dS bytes counted for the key and dQ passes are the workspace the
    # library asks for
    w = workloads.WORKLOADS[cfg]
    s = api.Shape(w.batch, w.seq, w.heads, w.kv_heads, causal=w.causal, scale=w.scale)
    ws = lib.attn_bwd_workspace_bytes(ctypes.byref(s.c_struct()))
    b = bench.algorithmic_bytes(w, None)
    B, H, Hkv, T, d = w.batch, w.heads, w.kv_heads, w.seq, 64
    assert b["queries"] == ws + B * Hkv * T * d * 2 + B * H * T * d * 4
    assert b["keys"] - ws == (2 * B * H * T * d * 2 + 2 * B * Hkv * T * d * 2
                              + 2 * B * H * T * 4 + 2 * B * Hkv * T * d * 4)
    # forward: Q, K, V^T in, O and L out, each once
    assert b["fwd"] == 2 * B * H * T * d * 2 + 2 * B * Hkv * T * d * 2 + B * H * T * 4


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    wl = "causal GQA T=4096 H=32 Hkv=8 d=64 Q~N(0,16)"
    h = bench.kernel_source_hash("bwd_keys.cu")
    prof = tmp_path / "profiles"
    prof.mkdir()
    csrc = tmp_path / "causal_streaming_softmax_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "bwd_keys.cu").write_bytes(
        open(os.path.join(ROOT, "causal_streaming_softmax_gb300", "csrc", "bwd_keys.cu"),
             "rb").read())
    (prof / "dram_traffic.txt").write_text(
        "# header\n"
        "kernel=bwd_keys_kernel source=bwd_keys.cu source_sha256=%s workload=%s "
        "bytes_per_launch=123\n" % (h, wl.replace(" ", "_")))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("bwd_keys.cu", wl) == 123.0
    assert bench.recorded_traffic("bwd_keys.cu", "another workload") is None
    # a changed kernel source invalidates the recorded figure
    (csrc / "bwd_keys.cu").write_bytes(b"// edited\n")
    assert bench.recorded_traffic("bwd_keys.cu", wl) is None


def test_peaks_come_from_the_measured_file():
    p = bench.load_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured" and p["tflops"] > 0 and p["hbm_gbs"] > 0
    else:
        assert p["source"] == "fallback"


def test_clock_summary_keeps_only_the_loaded_window():
    """Samples outside the loaded window (an idle GPU before or after) do not
    enter the clock summary; throttle reasons inside it are reported."""
    line = "0, {sm}, 2070, {pw}, 0x0, Not Active, Not Active, Not Active, {cap}\n"
    samples = [(0.0, line.format(sm=2070, pw=200, cap="Not Active")),      # idle, before
               (1.0, line.format(sm=1800, pw=900, cap="Not Active")),
               (1.1, line.format(sm=1700, pw=1300, cap="Active")),
               (1.2, line.format(sm=1750, pw=1200, cap="Not Active")),
               (9.0, line.format(sm=2070, pw=150, cap="Not Active"))]      # idle, after
    c = bench.ClockSampler.summarise(samples, window=(0.5, 2.0), period_ms=50)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 1750.0 and c["sm_mhz_min"] == 1700.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarise(samples, window=(3.0, 4.0))["samples"] == 0

#!/usr/bin/env python3
"""Throughput of causal streaming-softmax attention, forward + backward, on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
attn_fwd, attn_row_terms, attn_bwd_keys, attn_bwd_queries (four launches of
the library's kernels).  Default workload: causal GQA, batch 1, T = 4096,
32 query heads, 8 K/V heads, d = 64, Q ~ N(0, 16), K, V, dO ~ N(0, 1),
scale 1/8, seeded.

Metric: useful TFLOP/s of fwd + bwd, with the causal count 4 B H d T^2 / 2
for the forward and 2.5x that for the backward (3.5x in total); the
non-causal length-masked workload counts 4 d H sum(len^2).

Reported in one JSON line (rank 0): ``value`` is device throughput with the
inputs resident in HBM (L2 flushed before every timed step by a 256 MiB
write, outside the timed events, which sit at step boundaries only; the
per-call split comes from a second leg with an event after every call),
``e2e`` the same metric through the host-buffer C-ABI call attn_step_host
(pinned host -> device copies, the kernels, device -> host copies of O, L,
dQ, dK, dV^T, all inside the timed region, the copies overlapped with the
kernels; ``order`` says whether the call took the stored or the fused
order), ``roofline`` the dominant kernel against the measured tensor peak,
``cpu_baseline`` the binary64 oracle on a bounded sample timed on the host,
and ``fused_dq_variant`` the same step as the pages' two-launch backward:
the fused query pass (D and dQ, recomputing S, P, dP) then the key pass
storing no dS (no workspace), timed separately, with its own host-to-host
``e2e`` when the headline e2e took the stored order.

``--impl reference`` times the oracle (the CPU reference of this method) on
the same workload, one bounded sample per step, and prints the same line
with ``"impl": "reference"``.

Multi-GPU (torchrun): the path has no exchange step, so each rank runs an
independent replica (weak scaling); a host-side barrier brackets the timed
region and the slowest rank's time sets the value.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from causal_streaming_softmax_gb300 import workloads  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
DEFAULT_CONFIG = 3
METRIC = "causal attn fwd+bwd TFLOP/s (fp16, d=64) and % of GB300 dense FP16 tensor peak"


def useful_flops(w: workloads.Workload, lens) -> dict:
    """Useful FLOPs of each call and of the step."""
    d = workloads.HEAD_DIM
    if w.causal and lens is None:
        f_fwd = 4.0 * w.batch * w.heads * d * w.seq * w.seq / 2.0
    else:
        lens = np.full(w.batch, w.seq) if lens is None else np.asarray(lens, dtype=np.float64)
        pairs = float(np.sum(lens.astype(np.float64) ** 2))
        if w.causal:
            pairs /= 2.0
        f_fwd = 4.0 * d * w.heads * pairs
    return dict(fwd=f_fwd, row_terms=0.0, keys=2.0 * f_fwd, queries=0.5 * f_fwd,
                step=3.5 * f_fwd)


def algorithmic_bytes(w: workloads.Workload, lens) -> dict:
    """Minimum bytes each call must move (inputs read once, outputs written once)."""
    B, H, Hkv, T, d = w.batch, w.heads, w.kv_heads, w.seq, workloads.HEAD_DIM
    qb = B * H * T * d * 2
    kb = B * Hkv * T * d * 2
    nt = -(-T // 128)
    pairs = nt * (nt + 1) // 2 if w.causal else nt * nt
    ws = B * H * pairs * 128 * 128 * 2
    return dict(fwd=qb + 2 * kb + qb + B * H * T * 4,
                row_terms=2 * qb + B * H * T * 4,
                keys=2 * qb + 2 * kb + 2 * B * H * T * 4 + ws + 2 * B * Hkv * T * d * 4,
                queries=ws + kb + B * H * T * d * 4)


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(tflops=float(j["bf16_tflops"]),
                    tflops_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    hbm_gbs=float(j["hbm_gbs"]), source="measured")
    return dict(tflops=1900.0, tflops_sustained=1700.0, hbm_gbs=6800.0, source="fallback")


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "causal_streaming_softmax_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel and this workload; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(kernel_file)
    with open(p) as f:
        for line in f:
            if line.startswith("#") or "=" not in line:
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if (kv.get("source") == kernel_file and kv.get("source_sha256") == want
                    and kv.get("workload") == workload.replace(" ", "_")):
                return float(kv["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the GPU works.

    A reader thread stamps each sample with the host clock, so that only the
    samples taken inside a marked window (the loaded region) are summarised.
    """

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        import threading
        self.proc = None
        self.err = None
        self.samples = []  # (host time, line)
        self.period_ms = period_ms
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except (OSError, ValueError) as e:
            self.err = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line))

    def wait_first_sample(self, timeout_s: float = 5.0) -> bool:
        t0 = time.perf_counter()
        while self.proc is not None and not self.samples:
            if time.perf_counter() - t0 > timeout_s:
                return False
            time.sleep(0.01)
        return bool(self.samples)

    def stop(self, window=None) -> dict:
        """Summary of the samples whose host time lies in ``window`` (t0, t1),
        or of all samples."""
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0, note=self.err)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        return self.summarise(self.samples, window, self.period_ms)

    @classmethod
    def summarise(cls, samples, window=None, period_ms=None) -> dict:
        """Median SM clock, the largest maximum clock, median power and the
        throttle reasons seen, over the (host time, csv line) samples whose
        time lies inside ``window``."""
        sm, smax, power, reasons = [], [], [], set()
        for t, line in samples:
            if window is not None and not (window[0] <= t <= window[1]):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(cls.NAMES, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0)
        return dict(sm_mhz=float(statistics.median(sm)), sm_max_mhz=float(max(smax)),
                    sm_mhz_min=float(min(sm)), power_w_median=float(statistics.median(power)),
                    reasons=sorted(reasons), samples=len(sm), period_ms=period_ms)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_sample(w, inp, budget_s: float, max_heads=None):
    """Time the binary64 oracle on whole query heads of the workload (each with
    its K/V head) until the time budget is spent.  Returns (useful FLOP/s,
    heads, seconds, threads)."""
    import oracle
    lens = inp["lens"]
    G = w.group
    one = workloads.Workload(w.name, 1, w.seq, 1, 1, w.causal)
    done, t_total, flops = 0, 0.0, 0.0
    b = 0
    h = 0
    while True:
        kv = h // G
        q = inp["q"][b:b + 1, h:h + 1]
        k = inp["k"][b:b + 1, kv:kv + 1]
        vt = inp["vt"][b:b + 1, kv:kv + 1]
        dout = inp["dout"][b:b + 1, h:h + 1]
        ln = None if lens is None else lens[b:b + 1]
        t0 = time.perf_counter()
        oracle.backward(q, k, vt, dout, causal=w.causal, scale=w.scale, lens=ln)
        t_total += time.perf_counter() - t0
        flops += useful_flops(one, ln)["step"]
        done += 1
        h += 1
        if h == w.heads:
            h, b = 0, (b + 1) % w.batch
        if t_total >= budget_s or (max_heads and done >= max_heads):
            break
    return flops / t_total, done, t_total, oracle.num_threads()


def run_reference(args, w, world, rank):
    """The oracle arm: each step is one whole query head's fwd + bwd."""
    if rank != 0:
        return 0
    import oracle
    inp = workloads.make_inputs(w)
    lens = inp["lens"]
    G = w.group
    one = workloads.Workload(w.name, 1, w.seq, 1, 1, w.causal)
    times, flops = [], []
    for it in range(args.warmup + args.steps):
        h = it % w.heads
        b = (it // w.heads) % w.batch
        kv = h // G
        ln = None if lens is None else lens[b:b + 1]
        t0 = time.perf_counter()
        oracle.backward(inp["q"][b:b + 1, h:h + 1], inp["k"][b:b + 1, kv:kv + 1],
                        inp["vt"][b:b + 1, kv:kv + 1], inp["dout"][b:b + 1, h:h + 1],
                        causal=w.causal, scale=w.scale, lens=ln)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt)
            flops.append(useful_flops(one, ln)["step"])
    total_t = sum(times)
    value = sum(flops) / total_t / 1e12
    sample = ("one query head (with its K/V head) of the %s workload per step, full "
              "forward + backward in binary64" % w.name)
    line = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * total_t / len(times),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic (seeded)", impl="reference",
                config=config_dict(w, lens),
                cpu_baseline=dict(value=value, unit="TFLOP/s", cores=oracle.num_threads(),
                                  kind="oracle", sample=sample),
                e2e=dict(value=value, unit="TFLOP/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))
    print(json.dumps(line))
    return 0


def config_dict(w, lens):
    c = dict(workload=w.name, batch=w.batch, seq=w.seq, heads=w.heads, kv_heads=w.kv_heads,
             head_dim=workloads.HEAD_DIM, causal=w.causal, scale=w.scale,
             q_std=w.q_std, seed=w.seed,
             l2="flushed before every timed step (256 MiB write, outside the timed events)")
    if lens is not None:
        c["seq_lens"] = "uniform [%d, %d], padded to %d" % (w.len_lo, w.len_hi, w.seq)
    return c


def run_ours(args, w, world, rank, local):
    import torch
    from causal_streaming_softmax_gb300 import api
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = workloads.make_inputs(w)
    lens_np = inp["lens"]
    lens = None if lens_np is None else torch.from_numpy(lens_np).to(dev)
    s = api.Shape(w.batch, w.seq, w.heads, w.kv_heads, causal=w.causal, scale=w.scale,
                  seq_lens=lens)
    q, k, vt, dout = (torch.from_numpy(inp[n]).to(dev) for n in ("q", "k", "vt", "dout"))
    bufs = api.Buffers(s, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    calls = (
        ("fwd", "fwd.cu", lambda: api.attn_fwd(s, q, k, vt, bufs.o, bufs.lse, stream)),
        ("row_terms", "row_terms.cu",
         lambda: api.attn_row_terms(s, bufs.o, dout, bufs.delta, stream)),
        ("keys", "bwd_keys.cu",
         lambda: api.attn_bwd_keys(s, q, k, vt, dout, bufs.lse, bufs.delta, bufs.ws, bufs.dk,
                                   bufs.dvt, stream)),
        ("queries", "bwd_queries.cu",
         lambda: api.attn_bwd_queries(s, k, bufs.ws, bufs.dq, stream)),
    )

    for _ in range(args.warmup):
        flush.zero_()
        for _, _, fn in calls:
            fn()
    torch.cuda.synchronize(dev)
    if api.last_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")

    # Clocks are sampled from the start of a sustained leg (the same step back
    # to back for --sustain-s seconds, so that the clocks and the power draw
    # settle at their loaded level) to the end of the timed steps; only the
    # samples inside that loaded window are summarised.
    clocks = ClockSampler(local)
    clocks.wait_first_sample()
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    t_load0 = time.perf_counter()
    sus_ev = []
    while not sus_ev or time.perf_counter() - t_load0 < args.sustain_s:
        for _ in range(20):
            flush.zero_()
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            e[0].record(stream)
            for _, _, fn in calls:
                fn()
            e[1].record(stream)
            sus_ev.append(e)
    torch.cuda.synchronize(dev)
    n_sus = len(sus_ev)
    sus_ms = sum(a.elapsed_time(b) for a, b in sus_ev)
    sus_wall = time.perf_counter() - t_load0

    # The timed steps: events at step boundaries only.  An event recorded
    # between two calls ends the overlap of one launch with the previous
    # kernel's tail (programmatic dependent launch), so the per-call split is
    # taken in a second leg of K steps with an event after every call.
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        for _, _, fn in calls:
            fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.perf_counter()
    t_wall = t_wall1 - t_wall0
    dist_barrier(world)
    if api.last_device_error(stream) != 0:
        raise RuntimeError("device error during the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in ev]

    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
           for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush.zero_()
        sev[i][0].record(stream)
        for c, (_, _, fn) in enumerate(calls):
            fn()
            sev[i][c + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_split1 = time.perf_counter()
    dist_barrier(world)
    clk = clocks.stop(window=(t_load0, t_split1))
    if api.last_device_error(stream) != 0:
        raise RuntimeError("device error during the per-call leg")
    per_call = {name: [sev[i][c].elapsed_time(sev[i][c + 1]) for i in range(K)]
                for c, (name, _, _) in enumerate(calls)}
    split_step_ms = [sev[i][0].elapsed_time(sev[i][-1]) for i in range(K)]
    total_ms = dist_max(sum(step_ms), world)
    ms_per_step = total_ms / K
    fl = useful_flops(w, lens_np)
    value = world * fl["step"] * K / (total_ms / 1e3) / 1e12
    sustained = dict(
        what="the same step (L2 flush, then the four calls) back to back under the clock "
             "sampler just before the timed steps; device time of the calls, flushes excluded",
        steps=n_sus, seconds=sus_wall, ms_per_step=sus_ms / n_sus,
        value=fl["step"] / (sus_ms / n_sus / 1e3) / 1e12, unit="TFLOP/s")
    if clk.get("sm_mhz"):
        # device time x median loaded SM clock: thousands of SM cycles per step
        clk["kcycles_per_step"] = ms_per_step * clk["sm_mhz"]
        clk["window"] = "sustained leg + timed steps + per-call leg (%.1f s)" % (t_split1 - t_load0)

    peaks = load_peaks()
    mean_ms = {n: sum(v) / K for n, v in per_call.items()}
    median_ms = {n: float(statistics.median(v)) for n, v in per_call.items()}
    dom = max(mean_ms, key=mean_ms.get)
    dom_file = dict((n, f) for n, f, _ in calls)[dom]
    nbytes = algorithmic_bytes(w, lens_np)
    if fl[dom] > 0:
        achieved = fl[dom] / (mean_ms[dom] / 1e3) / 1e12
        roof = dict(bound="tensor", achieved=achieved, peak=peaks["tflops"], unit="TFLOP/s",
                    frac=achieved / peaks["tflops"],
                    peak_note="dense bf16 burst peak, %s (fp16 = bf16 rate)" % peaks["source"])
    else:
        achieved = nbytes[dom] / (mean_ms[dom] / 1e3) / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=achieved / peaks["hbm_gbs"], peak_note=peaks["source"])
    roof["kernel"] = dom
    roof["kernel_time"] = ("mean of the %d launches of the per-call leg (an event after every "
                           "call, otherwise the timed step)" % K)
    traffic = recorded_traffic(dom_file, w.name)
    roof["traffic"] = traffic
    roof["algorithmic_bytes"] = nbytes[dom]

    kernels = {}
    for n, f, _ in calls:
        k_ms = mean_ms[n]
        e = dict(ms=k_ms, ms_median=median_ms[n], share=k_ms / sum(mean_ms.values()),
                 gbs=nbytes[n] / (k_ms / 1e3) / 1e9)
        if fl[n] > 0:
            e["tflops"] = fl[n] / (k_ms / 1e3) / 1e12
        kernels[n] = e

    # ---- end to end through the host-buffer API ----
    host = dev_in = None

    def time_e2e(step_bufs):
        # K host-to-host steps through attn_step_host, copies inside the events
        for _ in range(max(1, min(args.warmup, 3))):
            api.forward_backward_host(s, host, dev_in, step_bufs, stream)
        torch.cuda.synchronize(dev)
        Ke = max(1, min(K, 50))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist_barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(Ke):
            api.forward_backward_host(s, host, dev_in, step_bufs, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        dist_barrier(world)
        e_ms = dist_max(e0.elapsed_time(e1), world)
        if api.last_device_error(stream) != 0:
            raise RuntimeError("device error during the end-to-end steps")
        return dict(value=world * fl["step"] * Ke / (e_ms / 1e3) / 1e12, unit="TFLOP/s",
                    h2d_bytes_per_step=host.input_bytes(), d2h_bytes_per_step=host.output_bytes(),
                    steps=Ke, ms_per_step=e_ms / Ke,
                    order=api.attn_step_host_order(s, api.device_buffers(dev_in, step_bufs)))

    e2e = None
    if not args.no_e2e:
        host = api.HostProblem(s, *(torch.from_numpy(inp[n]) for n in ("q", "k", "vt", "dout")))
        dev_in = api.DeviceInputs(s, dev)
        e2e = time_e2e(bufs)

    # ---- the same step with the fused query pass (no dS workspace) ----
    variant = None
    if not args.no_variants:
        fbufs = api.Buffers(s, dev, workspace=False)
        fcalls = (
            ("fwd", lambda: api.attn_fwd(s, q, k, vt, fbufs.o, fbufs.lse, stream)),
            ("queries_fused", lambda: api.attn_bwd_queries_fused(
                s, q, k, vt, dout, fbufs.o, fbufs.lse, fbufs.delta, fbufs.dq, stream)),
            ("keys_nostore", lambda: api.attn_bwd_keys(s, q, k, vt, dout, fbufs.lse, fbufs.delta,
                                                       None, fbufs.dk, fbufs.dvt, stream)),
        )
        for _ in range(args.warmup):
            flush.zero_()
            for _, fn in fcalls:
                fn()
        Kf = max(1, min(K, 100))
        # step-boundary events for the step time, then a per-call leg
        fst = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(Kf)]
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fcalls) + 1)]
               for _ in range(Kf)]
        dist_barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(Kf):
            flush.zero_()
            fst[i][0].record(stream)
            for _, fn in fcalls:
                fn()
            fst[i][1].record(stream)
        for i in range(Kf):
            flush.zero_()
            fev[i][0].record(stream)
            for c, (_, fn) in enumerate(fcalls):
                fn()
                fev[i][c + 1].record(stream)
        torch.cuda.synchronize(dev)
        dist_barrier(world)
        if api.last_device_error(stream) != 0:
            raise RuntimeError("device error during the fused-dQ steps")
        f_ms = dist_max(sum(a.elapsed_time(b) for a, b in fst), world)
        variant = dict(
            what="attn_fwd, attn_bwd_queries_fused (D and dQ, S, P, dP recomputed), then "
                 "attn_bwd_keys storing no dS: no workspace, no row-terms launch",
            value=world * fl["step"] * Kf / (f_ms / 1e3) / 1e12, unit="TFLOP/s", steps=Kf,
            ms_per_step=f_ms / Kf,
            kernels_ms={n: sum(fev[i][c].elapsed_time(fev[i][c + 1]) for i in range(Kf)) / Kf
                        for c, (n, _) in enumerate(fcalls)})
        if host is not None and e2e is not None and e2e["order"] == "stored":
            # the host-to-host step in the fused order (attn_step_host without a
            # workspace), when the headline e2e took the stored order
            variant["e2e"] = time_e2e(fbufs)
        del fbufs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, heads, secs, threads = cpu_oracle_sample(w, inp, args.cpu_budget)
        cpu = dict(value=rate / 1e12, unit="TFLOP/s", cores=threads,
                   host_cores=os.cpu_count(), kind="oracle",
                   sample="%d query head(s) of the %s workload, full forward + backward in "
                          "binary64, %.1f s" % (heads, w.name, secs))

    if rank == 0:
        line = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=K,
                    warmup=args.warmup, ms_per_step=ms_per_step, higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f16",
                    data="synthetic (seeded normal inputs)", config=config_dict(w, lens_np),
                    parallelism="replicas" if world > 1 else "single",
                    frac_of_peak=value / world / peaks["tflops"],
                    ms_per_step_median=float(statistics.median(step_ms)),
                    gpu_launches=len(calls) * K, kernels=kernels, roofline=roof,
                    per_call_leg=dict(
                        what="the timed step again, K times, with an event after every call: "
                             "the per-call split (kernels) and the roofline kernel time",
                        steps=K, ms_per_step=sum(split_step_ms) / K),
                    clocks=clk, sustained=sustained, e2e=e2e, cpu_baseline=cpu, fused_dq_variant=variant,
                    wall_s_timed=t_wall)
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip timing the fused-dQ variant of the step")
    ap.add_argument("--sustain-s", type=float, default=2.0,
                    help="seconds of back-to-back steps under the clock sampler before "
                         "the timed steps")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline")
    args = ap.parse_args()
    # at least three untimed warm-up steps, whatever was asked
    args.warmup = max(3, args.warmup)
    args.sustain_s = max(0.0, args.sustain_s)
    world, rank, local = dist_setup()
    if world != args.gpus and world > 1:
        print("warning: WORLD_SIZE=%d, --gpus=%d" % (world, args.gpus), file=sys.stderr)
    w = workloads.WORKLOADS[args.config]
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    return run_ours(args, w, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

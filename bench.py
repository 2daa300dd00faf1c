"""Benchmark of the Mamba2 recurrent hot path on GB300.

One step = the long-prefill-with-continuation workload: one packed prefill of
65 536 tokens (conv -> chunked scan -> gated norm, 48 heads x 64, d_state 128,
bf16, fresh slot) followed by 64 one-token decode steps on the resulting state.
``value`` is prefill tokens/s; the batched decode workload (256 sequences x 128
steps against a 512-slot pool) is timed in the same run and reported under
``decode``. Inputs are seeded synthetic tensors with the workload's
distributions, resident in HBM before the timed region and larger than L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own independent replica (weak scaling);
the reported time is the maximum over ranks. ``--impl reference`` times the
CPU oracle on the host cores (rank 0 only) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402

METRIC = "Mamba2 layer prefill tokens/s + decode step us; % of HBM/tensor roofline"
WORKLOAD = "long prefill 1x65536 tok + 64 decode steps, 48 heads x 64, d_state 128, 1 group, conv 4, bf16"
TOKENS = 65536
DECODE_TAIL = 64


def peaks():
    f = ROOT / "MEASURED_PEAKS.json"
    if f.exists():
        d = json.loads(f.read_text())
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------------
# algorithmic bytes / flops per launch (bf16 activations, fp32 state)
# --------------------------------------------------------------------------

def conv_bytes(T, d: W.Dims, act_b=2):
    return 2 * T * d.conv_dim * act_b


def scan_bytes(T, d: W.Dims, act_b=2, state_rw=1):
    return T * (d.conv_dim + d.heads + d.d_inner) * act_b + state_rw * d.heads * d.headdim * d.d_state * 4


def scan_flops(T, d: W.Dims, Q=128):
    per_tok = d.heads * 2 * (Q * d.headdim + 2 * d.headdim * d.d_state) + 2 * d.ngroups * Q * d.d_state
    return T * per_tok


def norm_bytes(T, d: W.Dims, act_b=2):
    return 3 * T * d.d_inner * act_b


def prefill_call_bytes(wl: W.Workload, act_b=2):
    """Algorithmic bytes of one conv -> scan -> norm call sequence over a packed
    batch: each op's inputs and outputs once (conv, scan, norm as separate calls),
    the conv history and SSM state of every sequence written once and, when it
    resumes, also read once."""
    d, b = wl.dims, wl.batch
    T = b.rows
    resumed = sum(1 for f in b.fresh if not f)
    n = b.num_seqs
    state = d.heads * d.headdim * d.d_state * 4
    hist = (d.conv_kernel - 1) * d.conv_dim * act_b
    return (conv_bytes(T, d, act_b) + (n + resumed) * hist + scan_bytes(T, d, act_b, state_rw=0)
            + (n + resumed) * state + norm_bytes(T, d, act_b))


def prefill_fused_bytes(wl: W.Workload, act_b=2):
    """The least a fully fused conv -> scan -> norm pass over the batch must move:
    xBC, z and dt read once, the output written once, and the same per-sequence
    conv history and SSM state traffic as the separate calls (no xbc or y round
    trip through HBM). Reported beside the per-call roofline the ABI's separate
    calls are graded on."""
    d, b = wl.dims, wl.batch
    T = b.rows
    resumed = sum(1 for f in b.fresh if not f)
    n = b.num_seqs
    state = d.heads * d.headdim * d.d_state * 4
    hist = (d.conv_kernel - 1) * d.conv_dim * act_b
    per_token = (d.conv_dim + d.d_inner + d.heads + d.d_inner) * act_b
    return T * per_token + (n + resumed) * (hist + state)


def mamba3_bytes(b) -> int:
    """Algorithmic bytes of one Mamba-3 SISO forward call: every input read once, the
    output and the four final states written once (page "Mamba-3 SISO Long-Ragged
    Multi-Chunk Joint States Full VJP", dtype paragraph: bf16 q, k, v, trap, angles, z,
    output, final angle and v; fp32 adt, dt, biases, d, final state and k)."""
    T, H, P, N, R = b.rows, b.heads, b.headdim, b.d_state, b.rot_dim
    n = len(b.cu_seqlens) - 1
    reads = 2 * T * N * 2 + 2 * T * H * P * 2 + T * H * (4 + 4 + 2) + T * R * 2 + 2 * H * N * 4 + H * 4
    writes = T * H * P * 2 + n * H * (R * 2 + P * N * 4 + N * 4 + P * 2)
    return reads + writes


def decode_bytes_per_seq(d: W.Dims, act_b=2):
    return (2 * d.heads * d.headdim * d.d_state * 4 + 2 * (d.conv_kernel - 1) * d.conv_dim * act_b
            + d.conv_dim * act_b + 2 * d.d_inner * act_b + d.heads * act_b)


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    own library, loaded with ctypes) by a background thread every `period_s`
    seconds, so that even a timed region of a few tens of milliseconds gets ten
    or more samples. Reads only; changes no setting. Falls back to nothing
    (summary() returns None) when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device, period_s=0.002):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.period = period_s
        self.rows = []
        self.lib = None
        self.handle = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            bus = None
            if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
                bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
            if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device.index or 0), ctypes.byref(h)) != 0:
                    return
            self.lib, self.handle = lib, h
            self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            self.lib = None

    def _sample(self):
        ct, lib, h = self.ct, self.lib, self.handle
        mhz, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok = lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0  # NVML_CLOCK_SM
        ok = ok and lib.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(mx)) == 0
        ok = ok and self.get_reasons(h, ct.byref(rs)) == 0
        lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw))
        if ok:
            self.rows.append((mhz.value, mx.value, mw.value / 1000.0, rs.value))

    def _loop(self):
        while not self.stop.is_set():
            self._sample()
            self.stop.wait(self.period)

    def __enter__(self):
        if self.lib is not None:
            self.stop = self.threading.Event()
            self.thread = self.threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.lib is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            self._sample()  # at least one sample even for a very short region

    def summary(self):
        if self.lib is None or not self.rows:
            return None
        reasons = sorted({name for r in self.rows for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[0] for r in self.rows), "sm_max_mhz": max(r[1] for r in self.rows),
                "reasons": reasons, "samples": len(self.rows), "power_w_max": max(r[2] for r in self.rows),
                "source": f"NVML every {self.period * 1e3:.0f} ms during the timed region"}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

class Prefill:
    """Device-resident long-prefill workload and its op sequence."""

    def __init__(self, wl: W.Workload, dev):
        import selective_scan_gb300 as ss
        self.ss = ss
        self.wl = wl
        p, d, b = wl.params, wl.dims, wl.batch
        self.dev = dev
        self.x = wl.xBC.to(dev)
        self.z = wl.z.to(dev)
        self.dt = wl.dt.to(dev)
        self.pw = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
        self.conv = wl.conv_state.to(dev)
        self.ssm = wl.ssm_state.to(dev)
        self.xbc = torch.empty_like(self.x)
        self.y = torch.empty((b.rows, d.d_inner), dtype=wl.act, device=dev)
        self.out = torch.empty_like(self.y)
        need = ss.ssd_scan_workspace_bytes(d, b.rows, b.cu_seqlens, b.slots, b.fresh)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        # tensor-core scan: the dt' pre-pass, the state pass when a run is cut into
        # segments (the workspace then holds segment states beyond dt'), the full pass
        segmented = need > b.rows * d.heads * 4 + 256
        self.scan_launches = 3 if segmented else 2
        self.dec_x = wl.dec_xBC.to(dev)
        self.dec_z = wl.dec_z.to(dev)
        self.dec_dt = wl.dec_dt.to(dev)
        self.dec_out = torch.empty((1, d.d_inner), dtype=wl.act, device=dev)
        self.batch = ss.Batch(b.cu_seqlens, b.slots, b.fresh)
        self.dec_batch = ss.Batch(None, [b.slots[0]], [0])
        self.dims = ss.Dims(d.heads, d.headdim, d.d_state, d.ngroups, d.conv_kernel)

    def prefill(self, x=None, z=None, dt=None, out=None, ev=None):
        ss, wl = self.ss, self.wl
        p, d, b = wl.params, wl.dims, wl.batch
        cw, cb, A, dtb, D, nw = self.pw
        x = self.x if x is None else x
        z = self.z if z is None else z
        dt = self.dt if dt is None else dt
        out = self.out if out is None else out
        if ev:
            ev[0].record()
        ss.causal_conv1d(self.xbc, x, cw, cb, self.conv, batch=self.batch)
        if ev:
            ev[1].record()
        ss.ssd_scan(self.y, self.xbc, dt, A, dtb, D, self.ssm, self.dims, workspace=self.ws, batch=self.batch)
        if ev:
            ev[2].record()
        ss.gated_rmsnorm(out, self.y, z, nw, p.norm_groups, p.eps)
        if ev:
            ev[3].record()

    def _decode_steps(self):
        ss, wl = self.ss, self.wl
        p = wl.params
        cw, cb, A, dtb, D, nw = self.pw
        for t in range(self.dec_x.shape[0]):
            ss.decode_step(self.dec_out, self.dec_x[t], self.dec_z[t], self.dec_dt[t], cw, cb, A, dtb, D, nw,
                           p.norm_groups, p.eps, self.conv, self.ssm, self.dims, batch=self.dec_batch)

    def capture_decode(self):
        """Capture the 64 decode steps into a CUDA graph (the batch table is in
        the launch parameters, so the launches replay as they were recorded)."""
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._decode_steps()
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(self.graph):
            self._decode_steps()

    def decode_tail(self, ev=None):
        if getattr(self, "graph", None) is not None:
            self.graph.replay()
        else:
            self._decode_steps()
        if ev:
            ev.record()


def time_decode_batch(dev, reps, warm):
    """256 sequences x 128 carried steps; returns (us/step, events-based)."""
    import selective_scan_gb300 as ss
    wl = W.decode_batch()
    p, d, b = wl.params, wl.dims, wl.batch
    pw = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    conv, ssm = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    xs, zs, dts = wl.dec_xBC.to(dev), wl.dec_z.to(dev), wl.dec_dt.to(dev)
    out = torch.empty((b.num_seqs, d.d_inner), dtype=wl.act, device=dev)
    steps = xs.shape[0]
    batch = ss.Batch(None, b.slots, b.fresh)
    dims = ss.Dims(d.heads, d.headdim, d.d_state, d.ngroups, d.conv_kernel)

    def run_eager():
        for t in range(steps):
            ss.decode_step(out, xs[t], zs[t], dts[t], *pw, p.norm_groups, p.eps, conv, ssm, dims, batch=batch)

    for _ in range(warm):
        run_eager()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_eager()
    run = graph.replay
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
    return us, b.num_seqs, decode_bytes_per_seq(d) * b.num_seqs, reps * steps


def time_decode_device_batch(dev, reps):
    """The same 256 x 128 decode through mamba2_decode_step_device: the batch (slots,
    fresh flags, count) in device memory and checked on the device every step, 128
    steps captured in one CUDA graph; returns us/step."""
    import selective_scan_gb300 as ss
    wl = W.decode_batch()
    p, d, b = wl.params, wl.dims, wl.batch
    pw = [t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w)]
    conv, ssm = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    xs, zs, dts = wl.dec_xBC.to(dev), wl.dec_z.to(dev), wl.dec_dt.to(dev)
    out = torch.empty((b.num_seqs, d.d_inner), dtype=wl.act, device=dev)
    slots = torch.tensor(b.slots, dtype=torch.int32, device=dev)
    fresh = torch.tensor(b.fresh, dtype=torch.uint8, device=dev)
    n = torch.full((1,), b.num_seqs, dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    steps = xs.shape[0]

    def run_eager():
        for t in range(steps):
            ss.decode_step_device(out, xs[t], zs[t], dts[t], *pw, p.norm_groups, p.eps, conv, ssm, d, slots, fresh,
                                  n, status)

    run_eager()
    torch.cuda.synchronize()
    if int(status.item()) != ss.OK:
        raise SystemExit(f"device-batch decode rejected its batch: status {int(status.item())}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_eager()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * steps)


def time_prefill_config(wl: W.Workload, dev, reps, hbm, tf_sus, warm_reps=10):
    """One packed prefill call sequence (conv -> scan -> norm) of a workload, the
    median of `reps` CUDA-event intervals around the three calls: once with L2
    flushed before every call (a 256 MB buffer written between calls, outside
    the interval) and once warm (the same call back to back)."""
    import selective_scan_gb300 as ss
    p, d, b = wl.params, wl.dims, wl.batch
    x, z, dt = wl.xBC.to(dev), wl.z.to(dev), wl.dt.to(dev)
    cw, cb, A, dtb, D, nw = (t.to(dev) for t in (p.conv_w, p.conv_b, p.A_log, p.dt_bias, p.D, p.norm_w))
    conv, ssm = wl.conv_state.to(dev), wl.ssm_state.to(dev)
    xbc = torch.empty_like(x)
    y = torch.empty((b.rows, d.d_inner), dtype=wl.act, device=dev)
    out = torch.empty_like(y)
    batch = ss.Batch(b.cu_seqlens, b.slots, b.fresh)
    dims = ss.Dims(d.heads, d.headdim, d.d_state, d.ngroups, d.conv_kernel)
    need = ss.ssd_scan_workspace_bytes(d, b.rows, b.cu_seqlens, b.slots, b.fresh)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        ss.causal_conv1d(xbc, x, cw, cb, conv, batch=batch)
        ss.ssd_scan(y, xbc, dt, A, dtb, D, ssm, dims, workspace=ws, batch=batch)
        ss.gated_rmsnorm(out, y, z, nw, p.norm_groups, p.eps)

    for _ in range(warm_reps):
        call()
    # the three calls captured once in a CUDA graph (the library's calls are stream-ordered
    # and allocate nothing), so that a replay measures the GPU and not the host's launches
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    res = {}
    for mode, launch in (("l2_flushed", graph.replay), ("warm", graph.replay), ("warm_eager", call)):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            if mode == "l2_flushed":
                flush.fill_(1)
            e0.record()
            launch()
            e1.record()
        torch.cuda.synchronize()
        ts = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
        res[mode] = {"us_median": statistics.median(ts), "us_min": ts[0], "us_max": ts[-1]}
    nbytes = prefill_call_bytes(wl)
    fl = scan_flops(b.rows, d)
    floor_us = max(nbytes / (hbm * 1e9), fl / (tf_sus * 1e12)) * 1e6
    for r in res.values():
        r["tokens_per_s"] = b.rows / (r["us_median"] * 1e-6)
        r["GB/s"] = nbytes / (r["us_median"] * 1e-6) / 1e9
        r["roofline_frac"] = floor_us / r["us_median"]
    return {"workload": wl.name, "tokens": b.rows, "sequences": b.num_seqs, "algorithmic_bytes": nbytes,
            "scan_flops": fl, "roofline_us": floor_us, "reps": reps,
            "launch": "conv -> scan -> norm replayed from one CUDA graph (warm_eager: the three calls launched "
                      "from Python each time)",
            "roofline": "max(algorithmic bytes / measured HBM, SSD flops / sustained bf16)", **res}


def time_mamba3(dev, reps, hbm, seed=5):
    """The Mamba-3 SISO forward on the page's frozen shapes (one seeded batch of 3-5
    sequences), one kernel per call replayed from a CUDA graph: L2 flushed before each
    call and warm, median of `reps` event intervals."""
    import selective_scan_gb300 as ss
    b = W.mamba3_batch(seed=seed)
    n = len(b.cu_seqlens) - 1
    H, P, N, R = b.heads, b.headdim, b.d_state, b.rot_dim
    ins = [t.to(dev).contiguous() for t in b.tensors()]
    out = torch.empty((b.rows, H, P), dtype=torch.bfloat16, device=dev)
    fa = torch.empty((n, H, R), dtype=torch.bfloat16, device=dev)
    fs = torch.empty((n, H, P, N), dtype=torch.float32, device=dev)
    fk = torch.empty((n, H, N), dtype=torch.float32, device=dev)
    fv = torch.empty((n, H, P), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        ss.mamba3_siso_varlen_forward(out, fa, fs, fk, fv, *ins, b.cu_seqlens)

    for _ in range(5):
        call()
    torch.cuda.synchronize()
    digest = output_digest(out)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    res = {}
    for mode in ("l2_flushed", "warm"):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            if mode == "l2_flushed":
                flush.fill_(1)
            e0.record()
            graph.replay()
            e1.record()
        torch.cuda.synchronize()
        ts = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs)
        res[mode] = {"us_median": statistics.median(ts), "us_min": ts[0], "us_max": ts[-1]}
    if output_digest(out) != digest:
        raise SystemExit("mamba3 output changed between calls")
    nbytes = mamba3_bytes(b)
    floor_us = nbytes / (hbm * 1e9) * 1e6
    for r in res.values():
        r["tokens_per_s"] = b.rows / (r["us_median"] * 1e-6)
        r["GB/s"] = nbytes / (r["us_median"] * 1e-6) / 1e9
        r["roofline_frac"] = floor_us / r["us_median"]
    return {"workload": b.name, "tokens": b.rows, "lengths": [b.cu_seqlens[i + 1] - b.cu_seqlens[i] for i in range(n)],
            "algorithmic_bytes": nbytes, "roofline_us": floor_us, "reps": reps,
            "launch": "one kernel per call, replayed from a CUDA graph", "roofline": "algorithmic bytes / measured HBM",
            "output_sha256": digest, **res}


def cpu_baseline(target_s=12.0):
    """The oracle, as it stands, on a bounded prefix of the same workload."""
    import oracle
    oracle.build()
    cores = oracle.num_threads()

    def run(tokens):
        wl = W.long_prefill(tokens=tokens, decode_steps=1)
        p, b, d = wl.params, wl.batch, wl.dims
        conv, ssm = wl.conv_state.clone(), wl.ssm_state.clone()
        t0 = time.perf_counter()
        xbc, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv, b.cu_seqlens, b.slots, b.fresh)
        y, _ = oracle.ssd_scan(xbc, wl.dt, p.A_log, p.dt_bias, p.D, ssm, d.tuple4(), b.cu_seqlens, b.slots,
                               b.fresh)
        oracle.gated_rmsnorm(y, wl.z, p.norm_w, p.norm_groups, p.eps)
        return time.perf_counter() - t0

    probe = 1024
    t = run(probe)
    tokens = int(min(TOKENS, max(probe, (target_s / max(t, 1e-3)) * probe)) // 1024 * 1024)
    t = run(tokens)
    # the same oracle on one host thread, on a shorter prefix (about a third of the time)
    oracle.set_num_threads(1)
    try:
        t1p = run(256)
        tok1 = int(min(TOKENS, max(256, (target_s / 3 / max(t1p, 1e-3)) * 256)) // 256 * 256)
        t1 = run(tok1)
    finally:
        oracle.set_num_threads(cores)
    return {"value": tokens / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"prefill of the first {tokens} of the {TOKENS} tokens (conv -> scan -> norm, "
                      f"48 heads), {t:.1f} s",
            "one_thread": {"value": tok1 / t1, "unit": "tokens/s", "cores": 1,
                           "sample": f"prefill of the first {tok1} tokens, {t1:.1f} s"}}


def output_digest(t) -> str:
    """SHA-256 of a tensor's bytes (device tensors are copied to the host first)."""
    return hashlib.sha256(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes()).hexdigest()


def max_over_ranks(values, world, device):
    """Each rank's timings replaced by their maximum over the ranks (the job ends with
    its slowest replica); the identity on one rank."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world, tokens_per_rank, ms):
    """Whole-job tokens/s: `world` replicas, each processing tokens_per_rank tokens, the
    slowest in `ms` milliseconds (weak scaling: the work per GPU is fixed)."""
    return world * tokens_per_rank / (ms * 1e-3)


def time_link(dev, host_in, host_out, reps=3):
    """The host link alone for one e2e step's bytes: every input tensor copied in
    from pinned host memory and the output copied out, each direction on its own
    stream, and both at once (the floor the streamed host prefill can reach)."""
    dev_in = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in]
    dev_out = torch.empty(host_out.shape, dtype=host_out.dtype, device=dev)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    res = {}
    for mode in ("h2d", "d2h", "both"):
        ms = []
        for _ in range(reps + 1):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if mode in ("h2d", "both"):
                with torch.cuda.stream(s_in):
                    for d_, h_ in zip(dev_in, host_in):
                        d_.copy_(h_, non_blocking=True)
            if mode in ("d2h", "both"):
                with torch.cuda.stream(s_out):
                    host_out.copy_(dev_out, non_blocking=True)
            torch.cuda.synchronize()
            ms.append((time.perf_counter() - t0) * 1e3)
        res[mode + "_ms"] = min(ms[1:])
    bi = sum(t.numel() * t.element_size() for t in host_in)
    bo = host_out.numel() * host_out.element_size()
    res["h2d_GB/s"] = bi / (res["h2d_ms"] * 1e-3) / 1e9
    res["d2h_GB/s"] = bo / (res["d2h_ms"] * 1e-3) / 1e9
    return res


def time_projections(dev, T, d, reps, tf_peak):
    """The layer's projections around the path at T tokens, timed alone (CUDA events on
    the current stream, inputs larger than L2): in_proj [T, d_model] -> z | xBC | dt and
    out_proj [T, d_inner] -> [T, d_model], d_model = d_inner / 2 (the expand factor 2 of
    Mamba2 layers); random-init bf16 weights."""
    import selective_scan_gb300 as ss
    d_model = d.d_inner // 2
    g = torch.Generator("cpu").manual_seed(9)
    w_in, w_out = (t.to(dev) for t in W.draw_proj(g, d, d_model))
    hidden = torch.randn((T, d_model), generator=g).to(torch.bfloat16).to(dev)
    gin = torch.randn((T, d.d_inner), generator=g).to(torch.bfloat16).to(dev)
    z = torch.empty((T, d.d_inner), dtype=torch.bfloat16, device=dev)
    x = torch.empty((T, d.conv_dim), dtype=torch.bfloat16, device=dev)
    dt = torch.empty((T, d.heads), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, d_model), dtype=torch.bfloat16, device=dev)
    calls = {"in_proj": (lambda: ss.in_proj(z, x, dt, hidden, w_in, d), 2.0 * T * d_model * w_in.shape[0]),
             "out_proj": (lambda: ss.out_proj(out, gin, w_out), 2.0 * T * d.d_inner * d_model)}
    res = {"d_model": d_model, "peak_tflops": tf_peak, "peak_kind": "bf16 burst (kernel timed alone)"}
    for name, (fn, flops) in calls.items():
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tf = flops / (ms * 1e-3) / 1e12
        res[name] = {"ms": ms, "flops": flops, "TFLOP/s": tf, "frac_tensor": tf / tf_peak}
    return res


def run_ours(args, rank, world, local_rank):
    import selective_scan_gb300 as ss
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hbm, tf_burst, tf_sus, peak_kind = peaks()
    wl = W.long_prefill(seed=4 + rank, tokens=args.tokens)
    pf = Prefill(wl, dev)
    pf.capture_decode()
    d = wl.dims

    def step(evs=None):
        pf.prefill(ev=evs[:4] if evs else None)
        pf.decode_tail(ev=evs[4] if evs else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # every prefill step is fresh and every kernel reduces in a fixed order, so each
    # step's output is bit-identical: the warm-up digest must survive the timed loop
    digest_warm = output_digest(pf.out)
    if world > 1:
        torch.distributed.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvml = NvmlClockSampler(dev)
    with (nvml if nvml.lib is not None else ClockSampler(local_rank)) as clk:
        torch.cuda.synchronize()
        e_start.record()
        for k in range(args.steps):
            step(evs[k])
        e_end.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = e_start.elapsed_time(e_end)
    t_conv = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    t_scan = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    t_norm = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
    t_tail = sum(e[3].elapsed_time(e[4]) for e in evs) / args.steps
    # the prefill: one interval from before the conv to after the norm (gaps between
    # the launches included)
    prefill_each = [e[0].elapsed_time(e[3]) for e in evs]
    t_prefill = sum(prefill_each) / args.steps
    t_prefill_median = statistics.median(prefill_each)
    total_ms, t_prefill = max_over_ranks([total_ms, t_prefill], world, dev)
    digest_timed = output_digest(pf.out)
    if digest_timed != digest_warm:
        raise SystemExit("prefill output of the timed steps differs from the warm-up output")

    T = args.tokens
    gb = lambda nbytes, ms: nbytes / (ms * 1e-3) / 1e9  # noqa: E731
    kern = {
        "conv": {"ms": t_conv, "bytes": conv_bytes(T, d), "GB/s": gb(conv_bytes(T, d), t_conv)},
        "scan": {"ms": t_scan, "bytes": scan_bytes(T, d), "GB/s": gb(scan_bytes(T, d), t_scan),
                 "TFLOP/s": scan_flops(T, d) / (t_scan * 1e-3) / 1e12, "flops": scan_flops(T, d)},
        "norm": {"ms": t_norm, "bytes": norm_bytes(T, d), "GB/s": gb(norm_bytes(T, d), t_norm)},
    }
    for k in kern.values():
        k["frac_hbm"] = k["GB/s"] / hbm
    kern["scan"]["frac_tensor_sustained"] = kern["scan"]["TFLOP/s"] / tf_sus
    dominant = max(("conv", "scan", "norm"), key=lambda n: kern[n]["ms"])
    dk = kern[dominant]
    traffic = measured_traffic(dominant, T)

    # batched decode (256 sequences x 128 steps), timed separately
    dec_us, dec_n, dec_bytes, dec_steps = time_decode_batch(dev, reps=max(2, args.steps // 100), warm=1)
    dec_gbs = dec_bytes / (dec_us * 1e-6) / 1e9
    dec_dev_us = time_decode_device_batch(dev, reps=max(2, args.steps // 100))

    # the other prefill workloads (130m-shaped 2 048-token prefill, 8-sequence varlen
    # prefill), each call timed alone: L2 flushed and warm, median of the repetitions
    configs = {
        "prefill_130m_2048": time_prefill_config(W.prefill_130m(), dev, args.config_reps, hbm, tf_sus),
        "varlen_130m_8seq": time_prefill_config(W.varlen_130m(), dev, args.config_reps, hbm, tf_sus),
    }

    # the Mamba-3 SISO forward on the page's frozen shapes, timed alone
    configs["mamba3_siso_frozen"] = time_mamba3(dev, args.config_reps, hbm)

    # the layer's projections around the path (tcgen05 GEMMs), timed alone
    proj = time_projections(dev, T, d, reps=max(3, args.steps // 20), tf_peak=tf_burst)
    proj["layer_prefill_ms"] = proj["in_proj"]["ms"] + t_prefill + proj["out_proj"]["ms"]
    proj["layer_tokens_per_s"] = T / (proj["layer_prefill_ms"] * 1e-3)

    # end to end through the C ABI with HOST buffers: mamba2_prefill_host copies each
    # piece's xBC, z and dt in from pinned host memory and its output back, on its own
    # copy streams overlapping the compute, every step inside the timed region
    hx = wl.xBC.pin_memory()
    hz = wl.z.pin_memory()
    hdt = wl.dt.pin_memory()
    hout = torch.empty(tuple(pf.out.shape), dtype=pf.out.dtype).pin_memory()
    cw, cb, A, dtb, Dv, nw = pf.pw
    e2e_need = ss.prefill_host_workspace_bytes(pf.dims, ss.BF16, args.e2e_piece, batch=pf.batch)
    e2e_ws = torch.empty(max(e2e_need, 256), dtype=torch.uint8, device=dev)
    # ten calls at least (about 50 ms), after the warm-up's count of untimed ones: one
    # interval over all of them, so a single slow call weighs a tenth
    e2e_steps = max(10, args.steps // 20)

    def e2e_step():
        ss.prefill_host(hout, hx, hz, hdt, cw, cb, A, dtb, Dv, nw, wl.params.norm_groups, wl.params.eps, pf.conv,
                        pf.ssm, pf.dims, piece_rows=args.e2e_piece, workspace=e2e_ws, batch=pf.batch)

    e2e_step()
    torch.cuda.synchronize()
    e2e_digest_first = output_digest(hout)
    for _ in range(max(1, args.warmup - 1)):
        e2e_step()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(e2e_steps):
        e2e_step()
    a1.record()
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / e2e_steps
    if output_digest(hout) != e2e_digest_first:
        raise SystemExit("streamed host prefill output changed between calls")
    (e2e_ms,) = max_over_ranks([e2e_ms], world, dev)
    link = time_link(dev, [hx, hz, hdt], hout)

    line = {
        "metric": METRIC,
        "value": job_throughput(world, T, t_prefill),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, workload distributions)",
        "config": {"workload": WORKLOAD if T == TOKENS else WORKLOAD.replace(str(TOKENS), str(T)), "tokens": T, "heads": d.heads, "headdim": d.headdim,
                   "d_state": d.d_state, "ngroups": d.ngroups, "conv_kernel": d.conv_kernel,
                   "decode_tail_steps": DECODE_TAIL, "chunk": 128,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
        "prefill_ms": t_prefill,
        "prefill_ms_median": t_prefill_median,
        "prefill_roofline": {"algorithmic_bytes": prefill_call_bytes(wl), "roofline_ms": max(
            prefill_call_bytes(wl) / (hbm * 1e9), scan_flops(T, d) / (tf_sus * 1e12)) * 1e3,
            "frac": max(prefill_call_bytes(wl) / (hbm * 1e9), scan_flops(T, d) / (tf_sus * 1e12)) * 1e3 / t_prefill,
            "fused_minimum": {"algorithmic_bytes": prefill_fused_bytes(wl),
                              "roofline_ms": prefill_fused_bytes(wl) / (hbm * 1e9) * 1e3,
                              "frac": prefill_fused_bytes(wl) / (hbm * 1e9) * 1e3 / t_prefill}},
        "configs": configs,
        "decode_tail_us_per_step": t_tail * 1e3 / DECODE_TAIL,
        "decode_tail_launch": "CUDA graph of the 64 steps",
        "kernels": kern,
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": dk["GB/s"], "peak": hbm, "unit": "GB/s",
                     "frac": dk["GB/s"] / hbm, "traffic": traffic, "peak_kind": peak_kind},
        "decode": {"workload": "256 seqs x 1 token, 128 carried steps, 512-slot pool, 48 heads x 64, d_state 128",
                   "launch": "CUDA graph of the 128 steps",
                   "us_per_step": dec_us, "tokens_per_s": dec_n / (dec_us * 1e-6), "GB/s": dec_gbs,
                   "roofline_frac": dec_gbs / hbm, "roofline_frac_8TBs": dec_gbs / 8000.0,
                   "bytes_per_step": dec_bytes, "steps_timed": dec_steps,
                   "device_batch_us_per_step": dec_dev_us,
                   "device_batch": "mamba2_decode_step_device: batch in device memory, checked on the device "
                                   "every step (one more kernel), 128 steps in one CUDA graph"},
        "layer": proj,
        "e2e": {"value": job_throughput(world, T, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": hx.numel() * 2 + hz.numel() * 2 + hdt.numel() * 2,
                "d2h_bytes_per_step": hout.numel() * 2, "api": "mamba2_prefill_host",
                "piece_rows": args.e2e_piece, "ms_per_step": e2e_ms, "link": link,
                "link_frac": link["both_ms"] / e2e_ms},
        # per step: conv, the scan's launches, norm, and two kernels (state, finish) per decode step
        "gpu_launches": args.steps * (1 + pf.scan_launches + 1 + 2 * DECODE_TAIL),
        "output_digest": {"prefill_sha256": digest_timed, "stable_over_timed_steps": True,
                          "e2e_sha256": e2e_digest_first, "stable_over_e2e_steps": True},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


# --------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# --------------------------------------------------------------------------

def run_reference(args):
    import oracle
    oracle.build()
    sample = 2048
    wl = W.long_prefill(tokens=sample, decode_steps=1)
    p, b, d = wl.params, wl.batch, wl.dims

    def step():
        conv, ssm = wl.conv_state.clone(), wl.ssm_state.clone()
        xbc, _ = oracle.causal_conv1d(wl.xBC, p.conv_w, p.conv_b, conv, b.cu_seqlens, b.slots, b.fresh)
        y, _ = oracle.ssd_scan(xbc, wl.dt, p.A_log, p.dt_bias, p.D, ssm, d.tuple4(), b.cu_seqlens, b.slots,
                               b.fresh)
        oracle.gated_rmsnorm(y, wl.z, p.norm_w, p.norm_groups, p.eps)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = sample / dt
    cores = oracle.num_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": TOKENS, "sample_tokens_per_step": sample},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"prefill of the first {sample} of the {TOKENS} tokens per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


KERNEL_SOURCES = {"conv": "conv1d.cu", "scan": "scan_tc.cu", "norm": "norm.cu"}


def kernel_source_sha(name: str) -> str:
    src = ROOT / "selective_scan_gb300" / "csrc" / KERNEL_SOURCES[name]
    return hashlib.sha256(src.read_bytes()).hexdigest()


def measured_traffic(name: str, tokens: int):
    """DRAM bytes of one launch of `name` from the committed ncu capture, scaled
    to `tokens` (traffic grows with the rows); None when the kernel's source has
    changed since the counters were taken."""
    prof = ROOT / "profiles" / "traffic.json"
    if not prof.exists():
        return None
    rec = json.loads(prof.read_text())
    if name not in rec or rec.get("_sha256", {}).get(name) != kernel_source_sha(name):
        return None
    return int(round(rec[name] * tokens / rec["_tokens"]))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=TOKENS, help="prefill length (profiling captures use less)")
    ap.add_argument("--e2e-piece", type=int, default=8192, help="rows per piece of the streamed host prefill")
    ap.add_argument("--config-reps", type=int, default=60, help="repetitions of each other prefill workload")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

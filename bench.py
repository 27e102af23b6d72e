"""Benchmark: selective-scan forward on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long64k] [--no-extra]

A step is one sscan_fwd call (load, discretise, recurrence, carry, output,
final state) over the workload's whole batch, with inputs resident in HBM.
The headline workload is the largest configuration, long64k (1536 channels x
65536 steps, 16 states, fp32, 1.2 GB per call); the other configurations are
timed the same way under ``per_workload``, each with its own clock record.
Between timed steps a 512 MB buffer is written so that inputs smaller than L2
start from DRAM.  Each step is timed with CUDA events on the launch stream;
``value`` is tokens*channels/s = batch*dim*L / (mean step time), summed over
ranks (every rank runs its own copy of the workload: weak scaling).  The
exponent unit's peak of the roofline is measured in the same run
(``sscan_probe_ex2``); HBM bandwidth comes from MEASURED_PEAKS.json.

``e2e`` is the same metric through the public Python call with pinned host
buffers: per step the inputs are copied host->device, the scan runs, and the
output and final state are copied back, all inside the timed region.  Steps
follow one another on three streams (copy in, compute, copy out) with two
buffer sets, so that one step's inputs travel while the previous step's
outputs come back; ``e2e.serial_value`` is the same with every step's copies
and call in order on one stream.

``--impl reference`` times the double-precision CPU oracle (the plain
sequential definition the GPU path is checked against) on the host cores, on
a bounded channel sample of the same workload; only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import workloads  # noqa: E402

METRIC = ("selective-scan fwd tokens×channels/s, HBM GB/s and % of roofline on 1 GB300")
UNIT = "tokens*channels/s"
SM_COUNT = 152
MUFU_PER_CLK_SM = 32     # ex2 lanes per clock per SM, nominal (used only if the probe fails)
FP32_PER_CLK_SM = 128    # FP32 lanes per clock per SM (unit count)
ISSUE_LANES_PER_CLK_SM = 128  # 4 schedulers x one 32-lane warp instruction per clock
FLUSH_BYTES = 512 << 20  # > 129 MB L2


# ----------------------------------------------------------------- roofline

def peaks():
    """Measured HBM bandwidth and SM clock (MEASURED_PEAKS.json), else the
    profiling recipe's fallback figures."""
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "sm_max_mhz": float(m.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def algorithmic(w: workloads.Workload):
    """Algorithmic bytes, exponentials and FP32 lane-ops of one sscan_fwd pass.

    bytes: read u, delta and write y (B*D*L each), read B and C (B*N*L each),
    read A (D*N fp32) and D (D fp32), write final_state (B*D*N fp32), read h0
    when present.  exps: one 2^x per (b, d, t, n), or per (b, d, t) when every
    state of a channel shares its decay rate.  fp32: 4 per element (delta*A,
    (delta*u)*B, the state FMA, the C FMA), 3 with a shared rate.
    """
    es = 4 if w.dtype == "f32" else 2
    bdl, bnl = w.batch * w.dim * w.L, w.batch * w.N * w.L
    nbytes = 3 * bdl * es + 2 * bnl * es + w.dim * w.N * 4 + w.dim * 4 + w.batch * w.dim * w.N * 4
    if w.h0_std > 0:
        nbytes += w.batch * w.dim * w.N * 4
    elems = bdl * w.N
    scalar = w.A_kind == "scalar"
    exps = bdl if scalar else elems
    fp32 = (3 if scalar else 4) * elems
    return {"bytes": nbytes, "exps": exps, "fp32": fp32, "tokens_channels": bdl, "elements": elems}


def measure_ex2(dev, stream, reps=3):
    """Exponentials per second of the MUFU unit on this GPU, from the
    library's probe (every SM full: 8 CTAs of 256 threads per SM), best of
    ``reps`` CUDA-event timings after a warm-up launch."""
    import torch
    import linear_recurrence_gb300 as lr
    blocks, iters = SM_COUNT * 8, 2000
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    lr.probe_ex2(blocks, iters, sink=sink, stream=stream)
    best = None
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        n = lr.probe_ex2(blocks, iters, sink=sink, stream=stream)
        e.record(stream)
        e.synchronize()
        t = s.elapsed_time(e) * 1e-3
        best = t if best is None else min(best, t)
    return n / best


def measure_element(dev, stream, shared_rate, reps=3):
    """Elements per second that this GPU reaches with the scan's arithmetic,
    from the library's element probe: per element one 2^x and four FP32
    operations (three FP32 when a channel's states share one decay rate and
    the 2^x is taken once per step), independent chains on every SM (two
    resident CTAs of 256 threads, four waves); best of ``reps`` CUDA-event
    timings after a warm-up launch.  Reported beside the roofline: the mix
    issues at about three quarters of the issue slots' peak (dispatch stalls)."""
    import torch
    import linear_recurrence_gb300 as lr
    blocks, iters = SM_COUNT * 8, 2000
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    lr.probe_element(blocks, iters, shared_rate=shared_rate, sink=sink, stream=stream)
    best = None
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        n = lr.probe_element(blocks, iters, shared_rate=shared_rate, sink=sink, stream=stream)
        e.record(stream)
        e.synchronize()
        t = s.elapsed_time(e) * 1e-3
        best = t if best is None else min(best, t)
    return n / best


def roofline(w, t_s, pk):
    """The slower of the HBM bound (algorithmic bytes at the measured copy
    bandwidth) and the issue bound of the arithmetic, derived from unit counts
    and the clock: every exponent and every FP32 operation of the scan takes
    one lane of an issue slot, and an SM issues one 32-lane warp instruction
    per scheduler and clock (four schedulers, 152 SMs, the maximum SM clock).
    Beside it: the exponent unit's and the FP32 pipe's separate bounds, the
    elements at the rate the element probe reaches with this exact mix
    (sscan_probe_element, measured in the run) and the fraction of the HBM
    bound alone."""
    a = algorithmic(w)
    clk = pk["sm_max_mhz"] * 1e6
    bw = pk["hbm_gbs"] * 1e9
    ex2_rate = pk.get("ex2_per_s") or MUFU_PER_CLK_SM * SM_COUNT * clk
    t_hbm = a["bytes"] / bw
    t_exp = a["exps"] / ex2_rate
    t_fp32 = a["fp32"] / (FP32_PER_CLK_SM * SM_COUNT * clk)
    lane_ops = a["exps"] + a["fp32"]
    issue_peak = ISSUE_LANES_PER_CLK_SM * SM_COUNT * clk  # lane operations per second
    t_issue = lane_ops / issue_peak
    t_roof = max(t_hbm, t_issue)
    achieved_gbs = a["bytes"] / t_s / 1e9
    if t_hbm >= t_issue:
        r = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
             "frac": achieved_gbs / pk["hbm_gbs"]}
    else:
        # an arithmetic-bound scan: exponents and FP32 operations per second
        r = {"bound": "alu", "achieved": lane_ops / t_s / 1e12, "peak": issue_peak / 1e12,
             "unit": "T lane-ops/s (exponents + FP32 operations, one issue-slot lane each)",
             "frac": (lane_ops / t_s) / issue_peak,
             "peak_derivation": f"{SM_COUNT} SMs x {ISSUE_LANES_PER_CLK_SM} lanes (4 schedulers x one 32-lane "
                                f"warp instruction) per clock x {pk['sm_max_mhz']:.0f} MHz"}
    shared = a["exps"] < a["elements"]
    elem_rate = pk.get("elem_shared_per_s" if shared else "elem_per_s")
    if elem_rate:
        t_meas = a["elements"] / elem_rate
        r.update({"alu_measured_t_elem_s": elem_rate / 1e12, "t_alu_measured_us": t_meas * 1e6,
                  "frac_of_measured_alu": t_meas / t_s,
                  "alu_measured_source": "sscan_probe_element in this run (the same exponent/FP32 mix)"})
    r.update({"peak_source": pk["source"], "t_roofline_us": t_roof * 1e6,
              "t_hbm_us": t_hbm * 1e6, "t_issue_us": t_issue * 1e6,
              "ex2_peak_source": pk.get("ex2_source", "nominal"), "ex2_peak_texp_s": ex2_rate / 1e12,
              "t_exp_us": t_exp * 1e6, "t_fp32_us": t_fp32 * 1e6,
              "hbm_gbs": achieved_gbs, "frac_of_roofline": t_roof / t_s, "frac_of_hbm": t_hbm / t_s})
    return r


def kernel_source_hash():
    """Hash of the sources of the forward scan (kernel, dispatch, planner): the
    recorded ncu traffic is valid only for the sources it was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(_ROOT, "linear_recurrence_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in ("device_utils.cuh", "sscan_fwd_kernel.cuh",
                                             "sscan_fwd_tma.cuh", "sscan_fwd_tma.cu",
                                             "sscan_dispatch.cuh", "sscan_abi.cu", "sscan_fold.cu")]
    files += glob.glob(os.path.join(csrc, "sscan_fwd_*_*.cu"))
    for p in sorted(files):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(_ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    e = rec.get(workload_name)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_step")


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- GPU timing

def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def physical_gpu(local_index: int) -> str:
    """nvidia-smi id of a local CUDA device (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_index < len(ids):
            return ids[local_index]
    return str(local_index)


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Largest value across ranks (the job takes as long as its slowest rank)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws, device=None):
    if ws > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def time_device(fn, steps, warmup, flush, stream):
    """Mean CUDA-event time (s) of fn over `steps` calls, with the L2 flushed
    before each call; returns (mean seconds, total kernel launches)."""
    import torch
    for _ in range(warmup):
        with torch.cuda.stream(stream):
            flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = []
    launches = 0
    import linear_recurrence_gb300 as lr
    for _ in range(steps):
        with torch.cuda.stream(stream):   # the flush is ordered before the timed call
            flush.zero_()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        launches += lr.last_launch_count()
        evs.append((s, e))
    torch.cuda.synchronize()
    ts = [s.elapsed_time(e) * 1e-3 for s, e in evs]
    return sum(ts) / len(ts), launches, ts


def bench_workload(w, steps, warmup, dev, stream, flush, e2e=False):
    import torch
    import linear_recurrence_gb300 as lr
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    out = torch.empty_like(g["u"])
    fs = torch.empty((w.batch, w.dim, w.N), dtype=torch.float32, device=dev)

    def step():
        lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"],
                     out=out, final_state=fs, stream=stream)

    t, launches, ts = time_device(step, steps, warmup, flush, stream)
    res = {"t": t, "launches": launches, "plan": lr.last_plan(), "ts": ts}
    if e2e:
        host = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        dbuf = {k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in x.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = out_h.numel() * out_h.element_size() + fs_h.numel() * fs_h.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                for k, v in host.items():
                    if v is not None:
                        dbuf[k].copy_(v, non_blocking=True)
                y, hT = lr.sscan_fwd(dbuf["u"], dbuf["delta"], dbuf["A"], dbuf["B"], dbuf["C"],
                                     dbuf["D"], dbuf["h0"], out=out, final_state=fs, stream=stream)
                out_h.copy_(y, non_blocking=True)
                fs_h.copy_(hT, non_blocking=True)

        te_serial, _, _ = time_device(e2e_step, max(3, steps // 2), 2, flush, stream)
        te = time_e2e_pipelined(x, g, steps, warmup, dev, stream)
        res.update({"t_e2e": te, "t_e2e_serial": te_serial, "h2d": h2d, "d2h": d2h})
    return res


def time_e2e_pipelined(x, g, steps, warmup, dev, stream, outputs=None):
    """Seconds per step of a stream of sscan_fwd calls fed from pinned host
    memory: every step copies all its inputs host->device, runs the call and
    copies y and the final state back, on three streams (copy in, compute,
    copy out) with two buffer sets, so that step k+1's inputs travel while
    step k's outputs come back (the link carries both directions at once).
    Timed with CUDA events from the first copy to the last copy out.  A dict
    passed as ``outputs`` receives the host copies of the last step's y and
    final state."""
    import torch
    import linear_recurrence_gb300 as lr
    host = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
    sets = []
    for _ in range(2):
        dbuf = {k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in x.items()}
        out = torch.empty_like(g["u"])
        fs = torch.empty((g["u"].shape[0], g["u"].shape[1], g["A"].shape[1]), dtype=torch.float32, device=dev)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        ev = {n: torch.cuda.Event() for n in ("in_ready", "done", "out_read")}
        sets.append((dbuf, out, fs, out_h, fs_h, ev))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    used = [False, False]

    def step(k):
        i = k % 2
        dbuf, out, fs, out_h, fs_h, ev = sets[i]
        with torch.cuda.stream(s_in):
            if used[i]:
                s_in.wait_event(ev["done"])      # step k-2 no longer reads these inputs
            for n, v in host.items():
                if v is not None:
                    dbuf[n].copy_(v, non_blocking=True)
            ev["in_ready"].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(ev["in_ready"])
            if used[i]:
                stream.wait_event(ev["out_read"])  # step k-2's outputs have left
            lr.sscan_fwd(dbuf["u"], dbuf["delta"], dbuf["A"], dbuf["B"], dbuf["C"], dbuf["D"],
                         dbuf["h0"], out=out, final_state=fs, stream=stream)
            ev["done"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"])
            out_h.copy_(out, non_blocking=True)
            fs_h.copy_(fs, non_blocking=True)
            ev["out_read"].record(s_out)
        used[i] = True

    for k in range(max(warmup, 2)):
        step(k)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for k in range(steps):
        step(k)
    end.record(s_out)  # after every copy out, hence after every step's work
    torch.cuda.synchronize()
    if outputs is not None:
        last = sets[(steps - 1) % 2]
        outputs["y"], outputs["final_state"] = last[3], last[4]
    return start.elapsed_time(end) * 1e-3 / steps


def bench_fused(w, steps, warmup, dev, stream, flush, pk):
    """The scan with its options on workload ``w``: raw delta with a per-channel
    bias and softplus inside the op, and the SiLU output gate z.  Algorithmic
    bytes add z (read, one per (b, d, t)) and the bias (D fp32)."""
    import torch
    import linear_recurrence_gb300 as lr
    x = workloads.make_inputs(w)
    o = workloads.make_option_inputs(w)
    g = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    go = {k: v.to(dev) for k, v in o.items()}
    out = torch.empty_like(g["u"])
    fs = torch.empty((w.batch, w.dim, w.N), dtype=torch.float32, device=dev)

    def step():
        lr.sscan_fwd(g["u"], go["delta_raw"], g["A"], g["B"], g["C"], g["D"], g["h0"],
                     z=go["z"], delta_bias=go["delta_bias"], delta_softplus=True,
                     out=out, final_state=fs, stream=stream)

    t, launches, _ = time_device(step, steps, warmup, flush, stream)
    rf = roofline(w, t, pk)
    es = 4 if w.dtype == "f32" else 2
    extra_bytes = w.batch * w.dim * w.L * es + w.dim * 4
    gbs = (algorithmic(w)["bytes"] + extra_bytes) / t / 1e9
    return {"workload": f"{w.name} + delta_bias + softplus + silu(z) gate", "ms": t * 1e3,
            "value": w.channels * w.L / t, "unit": UNIT, "hbm_gbs": gbs, "bound": rf["bound"],
            "frac_of_plain_roofline": rf["frac_of_roofline"], "plan": lr.last_plan(),
            "launches_per_call": launches / steps}


def bench_bwd(w, steps, warmup, dev, stream, flush, pk, t_fwd):
    """The backward pass (sscan_bwd) on workload ``w`` with random upstream
    gradients of y and the final state.  Algorithmic work per element: the
    recomputed state (1 ex2, 4 FP32) and the reverse sweep (1 ex2, 12 FP32);
    bytes: read u, delta, dy, B, C, A, D, h0 and the final-state gradient, write
    du, ddelta (I/O dtype), dB, dC (fp32), dA, dD, dh0."""
    import torch
    import linear_recurrence_gb300 as lr
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    gen = torch.Generator().manual_seed(w.seed + 200)
    dy = torch.randn((w.batch, w.dim, w.L), generator=gen).to(workloads.io_dtype(w.dtype)).to(dev)
    dhT = torch.randn((w.batch, w.dim, w.N), generator=gen).to(dev)

    def step():
        lr.sscan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"], dy, dhT, stream=stream)

    t, launches, _ = time_device(step, steps, warmup, flush, stream)
    es = 4 if w.dtype == "f32" else 2
    bdl, bnl, dn = w.batch * w.dim * w.L, w.batch * w.N * w.L, w.dim * w.N
    nbytes = (5 * bdl * es + 2 * bnl * es + 2 * bnl * 4 + 2 * dn * 4 + 2 * w.dim * 4
              + 2 * w.batch * w.dim * w.N * 4 + (w.batch * w.dim * w.N * 4 if w.h0_std > 0 else 0))
    elems = bdl * w.N
    clk = pk["sm_max_mhz"] * 1e6
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    t_exp = 2 * elems / (MUFU_PER_CLK_SM * SM_COUNT * clk)
    t_fp32 = 16 * elems / (FP32_PER_CLK_SM * SM_COUNT * clk)
    t_roof = max(t_hbm, t_exp, t_fp32)
    return {"workload": f"{w.name} backward (sscan_bwd)", "ms": t * 1e3, "value": bdl / t, "unit": UNIT,
            "hbm_gbs": nbytes / t / 1e9, "bound": "hbm" if t_hbm >= max(t_exp, t_fp32) else "alu",
            "frac_of_roofline": t_roof / t, "t_roofline_us": t_roof * 1e6,
            "bwd_over_fwd": t / t_fwd if t_fwd else None, "plan": lr.last_plan(),
            "launches_per_call": launches / steps}


def bench_step(steps, warmup, dev, stream, flush, pk):
    """The single-step decode update on DECODE_WORKLOAD: HBM-bound on the fp32
    state (read + write 8 bytes per (b, d, n))."""
    import torch
    import linear_recurrence_gb300 as lr
    w = workloads.DECODE_WORKLOAD
    x = workloads.make_decode_inputs(w)
    g = {k: v.to(dev) for k, v in x.items()}
    out = torch.empty_like(g["u"])
    st = g["state"]
    t, launches, _ = time_device(
        lambda: lr.sscan_step(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], state=st, out=out,
                              stream=stream), steps, warmup, flush, stream)
    es = 2 if w.dtype == "bf16" else 4
    nbytes = (2 * w.batch * w.dim * w.N * 4 + 3 * w.batch * w.dim * es + 2 * w.batch * w.N * es
              + w.dim * w.N * 4 + w.dim * 4)
    gbs = nbytes / t / 1e9
    return {"workload": f"{w.name} (batch={w.batch}, dim={w.dim}, N={w.N}, {w.dtype} I/O, fp32 state)",
            "us": t * 1e6, "hbm_gbs": gbs, "bound": "hbm", "frac": gbs / pk["hbm_gbs"],
            "launches_per_call": launches / steps}


def bench_pscan(steps, warmup, dev, stream, flush):
    import torch
    import linear_recurrence_gb300 as lr
    w = workloads.PSCAN_WORKLOADS["pscan_8k"]
    x = workloads.make_pscan_inputs(w)
    a, b, h0 = x["a"].to(dev), x["b"].to(dev), x["h0"].to(dev)
    h = torch.empty_like(a)
    t, launches, _ = time_device(lambda: lr.pscan(a, b, h0, out=h, stream=stream), steps, warmup,
                                 flush, stream)
    nbytes = 3 * w.rows * w.len * 4 + w.rows * 4
    return {"workload": f"{w.name} (rows={w.rows}, len={w.len}, fp32)", "ms": t * 1e3,
            "hbm_gbs": nbytes / t / 1e9, "plan": lr.last_plan(), "launches_per_call": launches / steps}


# --------------------------------------------------------- CPU oracle leg

def oracle_rate(w, budget_s=10.0, nthreads=None):
    """The oracle (as it stands) on a bounded sample of workload w, on the host
    cores: a channel sample of batch 0 over all L steps, grown (and, once it is
    the whole batch, repeated) until about ``budget_s`` CPU-seconds were spent.
    Returns (tokens*channels/s, cores, sample description, wall seconds)."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    x = workloads.make_inputs(w)
    nch, reps = max(1, min(w.dim, nthreads)), 1
    while True:
        sl = slice(0, nch)
        args = [x["u"][0:1, sl], x["delta"][0:1, sl], x["A"][sl], x["B"][0:1], x["C"][0:1],
                x["D"][sl], None if x["h0"] is None else x["h0"][0:1, sl]]
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.sscan_fwd(*args, nthreads=nthreads)
        dt = time.perf_counter() - t0
        cpu_s = dt * min(nthreads, nch)
        if cpu_s >= budget_s:
            break
        grow = max(1.2, min(8.0, budget_s / max(cpu_s, 1e-3)))
        if nch < w.dim:
            nch = min(w.dim, max(nch + 1, int(nch * grow)))
        else:
            reps = max(reps + 1, int(reps * grow))
    rate = reps * nch * w.L / dt
    sample = (f"{nch} of {w.dim} channels of batch 0 x {reps} repetition(s), all {w.L} steps, "
              f"N={w.N}: {dt:.2f} s wall on {nthreads} threads")
    return rate, nthreads, sample, dt


# --------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long64k", choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads, pscan and the CPU baseline")
    ap.add_argument("--size", default=None,
                    help="BATCHxDIMxL: the workload's recipe at other sizes (smaller cases of the same "
                         "kernels for profiler captures; not a bench line of the configuration)")
    args = ap.parse_args()
    ws, rank, local = _dist()
    w = workloads.WORKLOADS[args.workload]
    if args.size:
        b_, d_, l_ = (int(v) for v in args.size.lower().split("x"))
        w = w.scaled(batch=b_, dim=d_, L=l_)
    wdesc = (f"{w.name}: batch={w.batch}, dim={w.dim}, L={w.L}, N={w.N}, {w.dtype} I/O, "
             f"delta=softplus(N({w.delta_mu},{w.delta_sigma})), A={w.A_kind}"
             + (f", h0~N(0,{w.h0_std}^2)" if w.h0_std > 0 else ""))

    if args.impl == "reference":
        if rank != 0:
            return 0
        rates = []
        for _ in range(args.warmup):
            oracle_rate(w, budget_s=1.0)
        cores = sample = None
        for _ in range(args.steps):
            r, cores, sample, _ = oracle_rate(w, budget_s=10.0)
            rates.append(r)
        v = statistics.mean(rates)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": w.channels * w.L / v * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wdesc, "sample": "per step: " + sample},
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import linear_recurrence_gb300 as lr
    lr.load_library()  # raises if the CUDA library is missing: there is no fallback
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    pk = peaks()
    try:
        pk["ex2_per_s"] = measure_ex2(dev, stream)
        pk["ex2_source"] = "measured in this run (sscan_probe_ex2)"
    except Exception as exc:  # pragma: no cover - reported, nominal figure used
        pk["ex2_source"] = f"nominal 32/clk/SM (probe failed: {exc})"
    try:
        pk["elem_per_s"] = measure_element(dev, stream, False)
        pk["elem_shared_per_s"] = measure_element(dev, stream, True)
    except Exception as exc:  # pragma: no cover - reported, the separate unit peaks used
        print(f"element probe failed: {exc}", file=sys.stderr)

    barrier(ws, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(physical_gpu(dev.index or 0)) as clk:
        res = bench_workload(w, args.steps, args.warmup, dev, stream, flush, e2e=True)
    torch.cuda.synchronize(dev)
    barrier(ws, dev)
    t = max_over_ranks(res["t"], ws, dev)
    te = max_over_ranks(res["t_e2e"], ws, dev)
    value = ws * w.channels * w.L / t
    rf = roofline(w, t, pk)
    rf["traffic"] = recorded_traffic(w.name)
    rf["kernel"] = "sscan_fwd (every launch of one call, timed together)"

    extra = {}
    cpu = None
    if rank == 0 and not args.no_extra:
        per = {}
        for name in ["dim512", "bf16_2k", "long64k", "wide64"]:
            if name == w.name:
                continue
            wx = workloads.WORKLOADS[name]
            with ClockSampler(physical_gpu(dev.index or 0)) as ckx:
                r = bench_workload(wx, max(5, args.steps // 2), 3, dev, stream, flush)
            rfx = roofline(wx, r["t"], pk)
            per[name] = {"ms": r["t"] * 1e3,
                         "value": wx.channels * wx.L / r["t"], "unit": UNIT,
                         "hbm_gbs": rfx["hbm_gbs"], "bound": rfx["bound"],
                         "frac": rfx["frac"], "frac_of_roofline": rfx["frac_of_roofline"],
                         "frac_of_hbm": rfx["frac_of_hbm"],
                         "frac_of_measured_alu": rfx.get("frac_of_measured_alu"),
                         "t_roofline_us": rfx["t_roofline_us"], "plan": r["plan"],
                         "clocks": ckx.summary()}
        with ClockSampler(physical_gpu(dev.index or 0)) as ckx:
            per["bf16_2k_bwd"] = bench_bwd(workloads.WORKLOADS["bf16_2k"], max(5, args.steps // 2), 3, dev,
                                           stream, flush, pk, per.get("bf16_2k", {}).get("ms", 0) * 1e-3)
        per["bf16_2k_bwd"]["clocks"] = ckx.summary()
        with ClockSampler(physical_gpu(dev.index or 0)) as ckx:
            per["bf16_2k_fused"] = bench_fused(workloads.WORKLOADS["bf16_2k"], max(5, args.steps // 2), 3,
                                               dev, stream, flush, pk)
        per["bf16_2k_fused"]["clocks"] = ckx.summary()
        with ClockSampler(physical_gpu(dev.index or 0)) as ckx:
            per["pscan_8k"] = bench_pscan(max(5, args.steps // 2), 3, dev, stream, flush)
        per["pscan_8k"]["clocks"] = ckx.summary()
        with ClockSampler(physical_gpu(dev.index or 0)) as ckx:
            per["decode_step"] = bench_step(max(5, args.steps // 2), 3, dev, stream, flush, pk)
        per["decode_step"]["clocks"] = ckx.summary()
        extra["per_workload"] = per
        rate, cores, sample, _ = oracle_rate(w, budget_s=10.0)
        rate1, _, sample1, _ = oracle_rate(w, budget_s=3.0, nthreads=1)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "one_core": {"value": rate1, "sample": sample1}}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
                "config": {"workload": wdesc,
                           "l2": ("inputs larger than L2; " if algorithmic(w)["bytes"] > (129 << 20) else "")
                           + "a 512 MB buffer written before every step",
                           "plan": res["plan"], "parallelism": f"{ws} independent replicas"},
                "roofline": rf,
                "cpu_baseline": cpu,
                "e2e": {"value": ws * w.channels * w.L / te, "unit": UNIT,
                        "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                        "pipelining": "copy-in, compute and copy-out streams, two buffer sets",
                        "serial_value": ws * w.channels * w.L / max_over_ranks(res["t_e2e_serial"], ws, dev)},
                "gpu_launches": res["launches"],
                "clocks": clk.summary()}
        line.update(extra)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

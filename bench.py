#!/usr/bin/env python3
"""Throughput benchmark: multi-scale deformable attention forward + backward.

One step = msda_forward + msda_backward (all three gradients) over one batch
of the workload, inputs already resident in HBM.  The metric is samples/s
(samples = B*N_q*N_h*N_l*N_p) reported as Gsamples/s, plus the achieved
fraction of the HBM roofline computed from compulsory bytes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the encoder shape in binary32 (B=2, N_q=L=22223, N_h=8,
C_h=32, N_l=4, N_p=4, levels 100x167/50x84/25x42/13x21).  L2 is flushed
(a 2x-L2 buffer is overwritten) before every timed step, outside the timed
interval of that step.  Under torchrun each rank runs an independent replica
on its own GPU (the operator has no cross-GPU exchange); the value is the
samples of all ranks divided by the slowest rank's time.

``--impl reference`` times the CPU oracle (float64 C loops, one process per
host core) on a bounded sample of the same workload: there is no GPU
implementation to compare against.  The default run also reports the
oracle on one core (``cpu_baseline.single_thread``).

Clocks: NVML is polled every millisecond by a child process during the timed
region (``clocks``; ``nvidia-smi`` at 100 ms is kept beside it), after a
warm-up of at least W steps and at least ``--warmup-seconds`` of GPU work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from scale_deformable_attention_forward_gb300 import inputs as gen  # noqa: E402

METRIC = "MSDA fwd+bwd Gsamples/s (q·h·l·p) and achieved HBM GB/s vs GB300 peak"
UNIT = "Gsamples/s"
FALLBACK_HBM_GBS = 6800.0
# binary32 red.global.add payload rate of a GB300, measured with a reduction microbenchmark
# (random 128-byte lines; the same for scalar, vector and TMA bulk reductions)
REDUCTION_GBS = 6710.0
CSRC = os.path.join(ROOT, "scale_deformable_attention_forward_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


# ----------------------------------------------------------------------------- byte model
def compulsory_bytes(w: gen.Workload):
    """Compulsory HBM bytes: each tensor read or written once.

    V = value, O = out / grad_output, Loc = 8 B/sample, A = 4 B/sample.
      fwd = V + Loc + A + O
      bwd = V + Loc + A + O + V(grad_value) + Loc(grad_loc) + A(grad_attn)
    """
    ev = 2 if w.dtype == "bf16" else 4
    V = w.B * w.L * w.N_h * w.C_h * ev
    O = w.B * w.n_queries * w.N_h * w.C_h * ev
    S = w.samples
    fwd = V + 8 * S + 4 * S + O
    bwd = V + 8 * S + 4 * S + O + V + 8 * S + 4 * S
    return fwd, bwd


def gather_roofline(w: gen.Workload, fwd_ms: float, n_sm: int, sm_mhz) -> dict:
    """The forward against its L1 ceiling: samples x 4 corner rows x the
    128-byte lines of one row (C_h values of value's dtype), one line per
    L1 data-pipe wavefront and one wavefront per SM per cycle, at the median
    SM clock sampled during the timed region (the GPU's maximum clock when no
    sample was taken)."""
    ev = 2 if w.dtype == "bf16" else 4
    lines = w.samples * 4 * -(-(w.C_h * ev) // 128)
    mhz = float(sm_mhz) if sm_mhz else 2070.0
    achieved = lines / (fwd_ms * 1e-3) / 1e9
    peak = n_sm * mhz * 1e-3
    return {"what": "forward corner-row reads (samples x 4 corners x 128-byte lines a row) / forward time, against "
                    "one L1 data-pipe wavefront per SM per cycle",
            "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": "Glines/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{n_sm} SMs x {mhz:.0f} MHz" + ("" if sm_mhz else " (maximum clock: no clock sample)")}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("workloads", {}).get(workload)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


_NVML_CHILD = r"""
import ctypes, sys, time
uuid, period = sys.argv[1], float(sys.argv[2])
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    print("fail", flush=True); sys.exit(0)
h = ctypes.c_void_p()
if not uuid or nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
    if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
        print("fail", flush=True); sys.exit(0)
mx = ctypes.c_uint(0)
nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # 1 = NVML_CLOCK_SM
print("ready", mx.value, flush=True)
clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
out = []
import select
while True:
    if select.select([sys.stdin], [], [], 0)[0]:
        break
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
            nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
        out.append("%.6f %d %d" % (time.time(), clk.value, rs.value))
    time.sleep(period)
print("\n".join(out), flush=True)
"""


class NvmlClockSampler:
    """SM clock and clock-event reasons polled through NVML (ctypes on
    libnvidia-ml, read-only queries) every `period` seconds by a child
    process, so that even a timed region of a few milliseconds gets samples
    and the timed process's host thread is not slowed by the polling.
    Samples are kept when their timestamps fall inside the `with` block."""

    # nvmlClocksEventReason* bits (nvml.h); GPU idle and application-clock bits are not throttling
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device, period: float = 0.001):
        self.period = period
        self.samples = []
        self.max_mhz = None
        self.proc = None
        try:
            import torch
            uid = "GPU-" + str(torch.cuda.get_device_properties(torch_device).uuid)
        except Exception:
            uid = ""
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", _NVML_CHILD, uid, str(period)], stdin=subprocess.PIPE,
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline().split()
            if not first or first[0] != "ready":
                self.proc.kill()
                self.proc = None
            else:
                self.max_mhz = float(first[1]) if len(first) > 1 and float(first[1]) > 0 else None
        except Exception:
            self.proc = None

    def __enter__(self):
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        t1 = time.time()
        if self.proc is not None:
            try:
                out, _ = self.proc.communicate(input="stop\n", timeout=30)
            except Exception:
                self.proc.kill()
                out = ""
            for line in out.splitlines():
                parts = line.split()
                if len(parts) == 3:
                    t, c, r = float(parts[0]), float(parts[1]), int(parts[2])
                    if self.t0 <= t <= t1:
                        self.samples.append((c, r))
        return False

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, bits in self.samples:
            for b, n in self.REASONS.items():
                if bits & b:
                    reasons.add(n)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples),
                "source": f"NVML every {self.period * 1e3:.0f} ms during the timed region (a child process)"}


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The maximum of x over all ranks (x itself without torch.distributed)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle leg
def oracle_sample(w: gen.Workload, data: dict, n_queries: int):
    """A bounded slice of the workload for the CPU oracle: batch item 0,
    queries [0, n_queries), every head, level and point; the full value map.
    Arrays are widened to float64 up front (outside any timing)."""
    n = max(1, min(n_queries, w.n_queries))
    loc = data["sampling_locations"]
    loc = loc[0:1, :n] if w.loc_layout == "BQHLP2" else loc[0:1, :, :n]
    sub = {
        "value": np.ascontiguousarray(data["value"][0:1], dtype=np.float64),
        "sampling_locations": np.ascontiguousarray(loc, dtype=np.float64),
        "attention_weights": np.ascontiguousarray(data["attention_weights"][0:1, :n], dtype=np.float64),
        "grad_output": np.ascontiguousarray(data["grad_output"][0:1, :n], dtype=np.float64),
    }
    samples = n * w.N_h * w.N_l * w.N_p
    return sub, samples


def oracle_step(orc, w, data, sub):
    kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
              align_corners=w.align_corners, padding_mode=w.padding_mode)
    orc.forward(sub["value"], data["spatial_shapes"], data["level_start_index"], sub["sampling_locations"],
                sub["attention_weights"], **kw)
    orc.backward(sub["grad_output"], sub["value"], data["spatial_shapes"], data["level_start_index"],
                 sub["sampling_locations"], sub["attention_weights"], **kw)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


_WORKER = {}


def _oracle_worker_init(workload: str):
    """Pool initializer: each process builds the same seeded inputs (outside
    any timing)."""
    import oracle
    w = gen.WORKLOADS[workload]
    _WORKER["w"], _WORKER["data"], _WORKER["orc"] = w, gen.generate(w), oracle.default()


def _oracle_worker_run(job):
    """Forward + backward of queries [q0, q1) of batch item 0, `reps` times
    (the float64 slice is built once per process and kept)."""
    q0, q1, reps = job
    w, data, orc = _WORKER["w"], _WORKER["data"], _WORKER["orc"]
    key = (q0, q1)
    if _WORKER.get("key") != key:
        _WORKER["key"], _WORKER["slice"] = key, oracle_slice(w, data, q0, q1)
    sub, samples = _WORKER["slice"]
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(orc, w, data, sub)
    return samples * reps, time.perf_counter() - t0


def oracle_slice(w, data, q0, q1):
    loc = data["sampling_locations"]
    loc = loc[0:1, q0:q1] if w.loc_layout == "BQHLP2" else loc[0:1, :, q0:q1]
    sub = {
        "value": np.ascontiguousarray(data["value"][0:1], dtype=np.float64),
        "sampling_locations": np.ascontiguousarray(loc, dtype=np.float64),
        "attention_weights": np.ascontiguousarray(data["attention_weights"][0:1, q0:q1], dtype=np.float64),
        "grad_output": np.ascontiguousarray(data["grad_output"][0:1, q0:q1], dtype=np.float64),
    }
    return sub, (q1 - q0) * w.N_h * w.N_l * w.N_p


def time_oracle(w, workload: str, data, target_s: float, cores: int):
    """The oracle, as it stands, on `cores` host processes (a spawn pool: the
    parent has already used the GPU), each on its own query slice of batch
    item 0, for about target_s seconds.  Returns (Gsamples/s, samples, n_q
    per process, seconds, reps)."""
    import multiprocessing as mp
    import oracle
    orc = oracle.default()
    probe_q = max(1, min(w.n_queries, 256))
    sub, s = oracle_sample(w, data, probe_q)
    t0 = time.perf_counter()
    oracle_step(orc, w, data, sub)
    rate = s / max(time.perf_counter() - t0, 1e-6)  # samples/s of one process
    per_q = w.N_h * w.N_l * w.N_p
    n_q = int(max(1, min(w.n_queries // cores, target_s * rate / per_q)))
    reps = max(1, int(target_s * rate / (n_q * per_q)))
    jobs = [(i * n_q, (i + 1) * n_q, reps) for i in range(cores)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(workload,)) as pool:
        pool.map(_oracle_worker_run, [(j[0], j[1], 1) for j in jobs])  # workers up, slices built, warm
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker_run, jobs)
        wall = time.perf_counter() - t0
    samples = sum(r[0] for r in res)
    return samples / wall / 1e9, samples, n_q, wall, reps


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args, w: gen.Workload):
    import torch
    import scale_deformable_attention_forward_gb300 as msda

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    msda.load_library()

    data = gen.generate(w)
    vt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {
        "value": torch.from_numpy(data["value"]).to(vt).pin_memory(),
        "sampling_locations": torch.from_numpy(data["sampling_locations"]).pin_memory(),
        "attention_weights": torch.from_numpy(data["attention_weights"]).pin_memory(),
        "grad_output": torch.from_numpy(data["grad_output"]).to(vt).pin_memory(),
    }
    t = {k: v.to(dev) for k, v in host.items()}
    out = torch.empty((w.B, w.n_queries, w.N_h * w.C_h), dtype=vt, device=dev)
    gv = torch.empty_like(t["value"])
    gl = torch.empty_like(t["sampling_locations"])
    ga = torch.empty_like(t["attention_weights"])
    ws_bytes = msda.msda_backward_workspace_size(t["value"], data["spatial_shapes"], data["level_start_index"],
                                                 t["sampling_locations"], w.value_layout, w.loc_layout)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    kw = dict(value_layout=w.value_layout, sampling_locations_layout=w.loc_layout,
              align_corners=w.align_corners, padding_mode=w.padding_mode)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        msda.msda_forward(t["value"], data["spatial_shapes"], data["level_start_index"], t["sampling_locations"],
                          t["attention_weights"], out=out, **kw)

    def bwd():
        msda.msda_backward(t["grad_output"], t["value"], data["spatial_shapes"], data["level_start_index"],
                           t["sampling_locations"], t["attention_weights"], grad_value=gv,
                           grad_sampling_locations=gl, grad_attention_weights=ga, workspace=ws, **kw)

    # warm-up: W steps, and at least --warmup-seconds of GPU work so clocks settle
    warm_done, t_warm = 0, time.perf_counter()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk_warm:
        while warm_done < args.warmup or time.perf_counter() - t_warm < args.warmup_seconds:
            flush.fill_(1.0)
            fwd()
            bwd()
            warm_done += 1
            if warm_done % 32 == 0:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    nvml = NvmlClockSampler(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk, nvml:
        barrier(world)
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        wall = time.perf_counter() - wall0
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms_local = statistics.mean(f + b for f, b in zip(fwd_ms, bwd_ms))
    step_med_local = statistics.median(f + b for f, b in zip(fwd_ms, bwd_ms))
    step_ms = max_over_ranks(step_ms_local, world, dev)
    value = w.samples * world / (step_ms * 1e-3) / 1e9

    if args.only_step:  # (profiling runs: the step alone, no other legs)
        smi = clk.summary()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
                              "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 6),
                              "fwd_ms": round(statistics.mean(fwd_ms), 6), "bwd_ms": round(statistics.mean(bwd_ms), 6),
                              "config": {"name": args.workload}, "only_step": True,
                              "clocks": nvml.summary() or smi}), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # The staged-level forward (msda_forward_staged) under the same protocol,
    # outside the step: the same output as msda_forward, a different gather.
    out_st = torch.empty_like(out)

    def fwd_staged():
        msda.msda_forward_staged(t["value"], data["spatial_shapes"], data["level_start_index"],
                                 t["sampling_locations"], t["attention_weights"], out=out_st, **kw)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        fwd_staged()
    ev_st = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        ev_st[i][0].record(stream)
        fwd_staged()
        ev_st[i][1].record(stream)
    torch.cuda.synchronize(dev)
    staged_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev_st), world, dev)
    staged_same = bool(torch.equal(out_st, out))
    desc = msda.make_desc((w.B, w.n_queries, w.N_h, w.C_h, w.N_l, w.N_p, w.L), data["spatial_shapes"],
                          data["level_start_index"], w.value_layout, w.loc_layout, w.align_corners,
                          w.padding_mode, msda.DTYPE_BF16 if w.dtype == "bf16" else msda.DTYPE_F32)
    staged_first = msda.staged_levels(desc)
    staged_timeouts = msda.staged_timeouts()

    # The backward with per-level shared-memory grad_value accumulation
    # (msda_backward_staged), same protocol, outside the step.
    gv_st, gl_st, ga_st = torch.empty_like(gv), torch.empty_like(gl), torch.empty_like(ga)

    def bwd_staged():
        msda.msda_backward_staged(t["grad_output"], t["value"], data["spatial_shapes"], data["level_start_index"],
                                  t["sampling_locations"], t["attention_weights"], grad_value=gv_st,
                                  grad_sampling_locations=gl_st, grad_attention_weights=ga_st, workspace=ws, **kw)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        bwd_staged()
    ev_sb = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.fill_(float(i))
        ev_sb[i][0].record(stream)
        bwd_staged()
        ev_sb[i][1].record(stream)
    torch.cuda.synchronize(dev)
    staged_bwd_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev_sb), world, dev)
    staged_bwd_same = bool(torch.equal(gl_st, gl) and torch.equal(ga_st, ga))
    staged_bwd_first = msda.backward_staged_levels(desc)

    # The backward with plain per-corner atomics (the warp-aggregated scatter
    # switched off through MSDA_BWD_AGGREGATE=0), same protocol, outside the step.
    prev = os.environ.get("MSDA_BWD_AGGREGATE")
    os.environ["MSDA_BWD_AGGREGATE"] = "0"
    try:
        for _ in range(args.warmup):
            flush.fill_(1.0)
            bwd_plain_out = msda.msda_backward(t["grad_output"], t["value"], data["spatial_shapes"],
                                               data["level_start_index"], t["sampling_locations"],
                                               t["attention_weights"], grad_value=gv_st, grad_sampling_locations=gl_st,
                                               grad_attention_weights=ga_st, workspace=ws, **kw)
        ev_pl = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.fill_(float(i))
            ev_pl[i][0].record(stream)
            msda.msda_backward(t["grad_output"], t["value"], data["spatial_shapes"], data["level_start_index"],
                               t["sampling_locations"], t["attention_weights"], grad_value=gv_st,
                               grad_sampling_locations=gl_st, grad_attention_weights=ga_st, workspace=ws, **kw)
            ev_pl[i][1].record(stream)
        torch.cuda.synchronize(dev)
    finally:
        if prev is None:
            del os.environ["MSDA_BWD_AGGREGATE"]
        else:
            os.environ["MSDA_BWD_AGGREGATE"] = prev
    plain_bwd_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev_pl), world, dev)
    plain_same = bool(torch.equal(gl_st, gl) and torch.equal(ga_st, ga))

    # The backward for two output subsets (grad_value only: the tile-sorted
    # path on dense problems; grad_sampling_locations + grad_attention_weights
    # only), same protocol, outside the step.
    def bwd_subset(flags):
        msda.msda_backward(t["grad_output"], t["value"], data["spatial_shapes"], data["level_start_index"],
                           t["sampling_locations"], t["attention_weights"], compute_grad_value=flags[0],
                           compute_grad_sampling_locations=flags[1], compute_grad_attention_weights=flags[2],
                           grad_value=gv_st if flags[0] else None, grad_sampling_locations=gl_st if flags[1] else None,
                           grad_attention_weights=ga_st if flags[2] else None, workspace=ws, **kw)

    subset_ms = {}
    for name, flags in (("grad_value_only", (True, False, False)), ("loc_attn_only", (False, True, True))):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            bwd_subset(flags)
        ev_s = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.fill_(float(i))
            ev_s[i][0].record(stream)
            bwd_subset(flags)
            ev_s[i][1].record(stream)
        torch.cuda.synchronize(dev)
        subset_ms[name] = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev_s), world, dev)

    # End to end: pinned host inputs -> device, forward, backward, results ->
    # pinned host, every step.  Two buffer sets and three streams pipeline the
    # steps the way a production loop would: the inputs of step i+1 are copied
    # in and the results of step i-1 copied out while step i computes.
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    outs_shape = {"out": (out.shape, vt), "gv": (gv.shape, vt), "gl": (gl.shape, torch.float32),
                  "ga": (ga.shape, torch.float32)}
    host_out = [{k: torch.empty(s, dtype=dt).pin_memory() for k, (s, dt) in outs_shape.items()} for _ in range(2)]
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    dev_in = [t] + [{k: torch.empty_like(v) for k, v in t.items()}]
    dev_out = [{"out": out, "gv": gv, "gl": gl, "ga": ga},
               {"out": torch.empty_like(out), "gv": torch.empty_like(gv), "gl": torch.empty_like(gl),
                "ga": torch.empty_like(ga)}]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_out:
        e.record(stream)
    K_e2e = max(3, min(K, 200))

    def e2e_step(i):
        k = i % 2
        di, do = dev_in[k], dev_out[k]
        with torch.cuda.stream(s_in):  # inputs of step i (buffer k's last reader: step i-2's compute)
            s_in.wait_event(ev_comp[k])
            for name in host:
                di[name].copy_(host[name], non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_comp):  # compute (buffer k's outputs copied out by step i-2 first)
            s_comp.wait_event(ev_in[k])
            s_comp.wait_event(ev_out[k])
            msda.msda_forward(di["value"], data["spatial_shapes"], data["level_start_index"],
                              di["sampling_locations"], di["attention_weights"], out=do["out"], **kw)
            msda.msda_backward(di["grad_output"], di["value"], data["spatial_shapes"], data["level_start_index"],
                               di["sampling_locations"], di["attention_weights"], grad_value=do["gv"],
                               grad_sampling_locations=do["gl"], grad_attention_weights=do["ga"], workspace=ws,
                               **kw)
            ev_comp[k].record(s_comp)
        with torch.cuda.stream(s_out):  # results of step i
            s_out.wait_event(ev_comp[k])
            for name in host_out[k]:
                host_out[k][name].copy_(do[name], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in (s_in, s_comp, s_out):
        st.wait_event(e0)
    for i in range(K_e2e):
        e2e_step(i)
    for st in (s_in, s_comp, s_out):
        stream.wait_stream(st)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K_e2e, world, dev)
    barrier(world)

    smi = clk.summary()
    clocks = nvml.summary() or dict(smi, source="nvidia-smi every 100 ms during the timed region")
    clocks["nvidia_smi"] = {"timed_region": smi, "warmup": clk_warm.summary()}

    fwd_b, bwd_b = compulsory_bytes(w)
    peak, peak_kind = measured_peaks()
    fwd_mean, bwd_mean = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    dominant = "msda_backward" if bwd_mean >= fwd_mean else "msda_forward"
    dom_bytes, dom_ms = (bwd_b, bwd_mean) if dominant == "msda_backward" else (fwd_b, fwd_mean)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload)
    launches_per_step = 1 + 2 + (1 if w.dtype == "bf16" else 0)  # fwd; zero-fill + bwd; bf16 finalise

    result = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if w.dtype == "f32" else "bf16 storage, f32 arithmetic",
        "data": "synthetic (seeded Deformable-DETR-shaped inputs)",
        "config": {"workload": gen.WORKLOAD_DESCRIPTIONS.get(args.workload, args.workload),
                   "name": args.workload, "samples_per_step_per_gpu": w.samples,
                   "l2": "flushed before every step (2x L2 buffer overwritten, outside the timed interval)",
                   "parallelism": f"replicas x{world} (no cross-GPU exchange)"},
        "fwd_ms": round(fwd_mean, 6),
        "bwd_ms": round(bwd_mean, 6),
        "median": {"ms_per_step": round(max_over_ranks(step_med_local, world, dev), 6),
                   "fwd_ms": round(statistics.median(fwd_ms), 6), "bwd_ms": round(statistics.median(bwd_ms), 6),
                   "what": "medians over the K timed steps (value and ms_per_step use the mean)"},
        "wall_s_timed_region": round(wall, 3),
        "warmup_steps_run": warm_done,
        "clocks": clocks,
        "e2e": {"value": round(w.samples * world / (e2e_ms * 1e-3) / 1e9, 4), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "per step: pinned host -> device copies of the inputs, msda_forward, msda_backward, "
                        "device -> pinned host copies of all four results; double-buffered on three streams "
                        "(copies of neighbouring steps overlap the compute)"},
        "gpu_launches": launches_per_step * K,
        "roofline": {
            "kernel": dominant + (" (zero-fill + fused gather/scatter kernel)" if dominant == "msda_backward"
                                  else " (gather kernel)"),
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes_per_launch": dom_bytes,
            "traffic": (traffic or {}).get(dominant),
        },
        # The backward's real bound: the binary32 reductions of grad_value (four corner rows of
        # C_h values per sample), against the reduction rate a microbenchmark of red.global.add
        # measured on this GPU (6.7 TB/s of payload, whatever the request shape).
        "roofline_reduction": {
            "what": "grad_value reduction payload (samples x 4 corners x C_h x 4 B) / backward time of the "
                    "plain-atomics leg (one reduction line per corner and sample)",
            "achieved": round(w.samples * 4 * w.C_h * 4 / (plain_bwd_ms * 1e-3) / 1e9, 1),
            "peak": REDUCTION_GBS, "unit": "GB/s",
            "frac": round(w.samples * 4 * w.C_h * 4 / (plain_bwd_ms * 1e-3) / 1e9 / REDUCTION_GBS, 4),
            "peak_source": "red.global.add.v4.f32 microbenchmark on GB300 (random 128-byte lines)"},
        "forward_staged": {
            "what": "msda_forward_staged: coarse levels copied to shared memory by TMA, gathered from there",
            "fwd_ms": round(staged_ms, 6), "direct_fwd_ms": round(fwd_mean, 6),
            "speedup_vs_direct": round(fwd_mean / staged_ms, 4) if staged_ms > 0 else None,
            "staged_levels": list(range(staged_first, w.N_l)), "bit_identical_to_direct": staged_same,
            "timeouts": staged_timeouts},
        "backward_subsets": {
            "what": "msda_backward for two output subsets, same protocol, outside the step",
            "grad_value_only_ms": round(subset_ms["grad_value_only"], 6),
            "loc_attn_only_ms": round(subset_ms["loc_attn_only"], 6)},
        "backward_staged": {
            "what": "msda_backward_staged: grad_value of the coarse levels accumulated per block in shared memory",
            "bwd_ms": round(staged_bwd_ms, 6), "direct_bwd_ms": round(bwd_mean, 6),
            "speedup_vs_direct": round(bwd_mean / staged_bwd_ms, 4) if staged_bwd_ms > 0 else None,
            "staged_levels": list(range(staged_bwd_first, w.N_l)),
            "loc_attn_grads_bit_identical_to_direct": staged_bwd_same},
        "backward_plain_atomics": {
            "what": "msda_backward with the warp-aggregated grad_value scatter off (MSDA_BWD_AGGREGATE=0): one "
                    "red.global.add.v4.f32 line per corner and sample",
            "bwd_ms": round(plain_bwd_ms, 6), "aggregated_bwd_ms": round(bwd_mean, 6),
            "aggregated_speedup": round(plain_bwd_ms / bwd_mean, 4) if bwd_mean > 0 else None,
            "loc_attn_grads_bit_identical": plain_same},
        # The forward's own bound: each sample reads four corner rows, and the L1 data pipe
        # serves one line of them (one wavefront) per SM per cycle, whoever reads it.
        "roofline_gather": gather_roofline(w, fwd_mean, torch.cuda.get_device_properties(dev).multi_processor_count,
                                           clocks.get("sm_mhz")),
        "roofline_step": {
            "what": "forward + backward compulsory bytes / step time",
            "achieved": round((fwd_b + bwd_b) / (step_ms * 1e-3) / 1e9, 1), "peak": peak, "unit": "GB/s",
            "frac": round((fwd_b + bwd_b) / (step_ms * 1e-3) / 1e9 / peak, 4),
            "bytes_per_step": fwd_b + bwd_b,
        },
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = max(1, os.cpu_count() or 1)
        v, samples, n_q, dt, reps = time_oracle(w, args.workload, data, args.cpu_seconds, cores)
        result["cpu_baseline"] = {
            "value": round(v, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"batch item 0: {cores} processes, each queries [{n_q}*i, {n_q}*(i+1)) of {w.n_queries} "
                      f"with all heads/levels/points, forward + backward x{reps} in float64; {samples} samples "
                      f"in {dt:.1f} s wall",
            "cpu": cpu_model()}
        v1, samples1, n_q1, dt1, reps1 = time_oracle(w, args.workload, data, args.cpu_seconds / 3, 1)
        result["cpu_baseline"]["single_thread"] = {
            "value": round(v1, 6), "unit": UNIT, "cores": 1,
            "sample": f"batch item 0: one process, queries [0, {n_q1}) of {w.n_queries} with all heads/levels/"
                      f"points, forward + backward x{reps1} in float64; {samples1} samples in {dt1:.1f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, w: gen.Workload):
    """The oracle on all host cores (a spawn pool, one query slice per
    process), a bounded slice of the workload per step."""
    import multiprocessing as mp
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    orc = oracle.default()
    data = gen.generate(w)
    cores = max(1, os.cpu_count() or 1)
    total_steps = args.warmup + args.steps
    per_step_s = max(0.005, args.reference_seconds / max(1, total_steps))
    probe_q = max(1, min(w.n_queries, 64))
    sub, s = oracle_sample(w, data, probe_q)
    t0 = time.perf_counter()
    oracle_step(orc, w, data, sub)
    rate = s / max(time.perf_counter() - t0, 1e-6)
    per_q = w.N_h * w.N_l * w.N_p
    n_q = int(min(max(1, w.n_queries // cores), max(1, per_step_s * rate / per_q)))
    jobs = [(i * n_q, (i + 1) * n_q, 1) for i in range(cores)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(args.workload,)) as pool:
        for _ in range(args.warmup):
            pool.map(_oracle_worker_run, jobs)
        t0 = time.perf_counter()
        done = 0
        for _ in range(args.steps):
            done += sum(r[0] for r in pool.map(_oracle_worker_run, jobs))
        dt = time.perf_counter() - t0
    value = done / dt / 1e9
    result = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Deformable-DETR-shaped inputs)",
        "config": {"workload": gen.WORKLOAD_DESCRIPTIONS.get(args.workload, args.workload), "name": args.workload},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "kind": "oracle", "cores": cores,
                         "sample": f"per step: batch item 0, {cores} processes each on {n_q} queries "
                                   f"(all heads/levels/points; {cores * n_q * per_q} samples), forward + "
                                   f"backward, float64",
                         "cpu": cpu_model()},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "no GPU implementation exists for this operator on the reference pages; the reference arm "
                "is the float64 CPU oracle",
    }
    print(json.dumps(result), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-seconds", type=float, default=0.5,
                    help="keep warming up (untimed) until this much wall time has passed")
    ap.add_argument("--workload", default="encoder32", choices=sorted(gen.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step and print a short line; skip the staged, subset, end-to-end and CPU legs "
                         "(for profiler runs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU work for the cpu_baseline leg (a slice of the workload)")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="total CPU time budget of --impl reference (split over warm-up + steps)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = gen.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

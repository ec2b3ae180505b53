"""Benchmark: selective diagonal scan, forward + backward, on one GB300 per rank.

A step is one pass of the whole path over one batch of the largest workload:
B=16 T=2048 D=5120 DS=16, bf16 I/O, float32 state and gradients, checkpoints
every 256 steps: the forward (y, hT, checkpoints) then the backward (gx,
gdelta, gA, gb, gc, gh0). Inputs are seeded synthetic tensors of that shape
(gen.make_inputs); every input tensor is larger than L2, so no flush is
needed between steps. ``value`` is B*T*D*DS elements per second of
forward+backward over all ranks (weak scaling: every rank runs its own copy).

Also reported: the device time of each kernel group (CUDA events on the launch
stream), the roofline of the dominant kernel, an end-to-end number through the
public API with host buffers (H2D of the inputs and D2H of all outputs inside
the timed region), SM clocks sampled during the timed region, the float64 CPU
oracle timed on a bounded sample (cpu_baseline), and one-line timings of the
other two large workloads (bf16 forward B=8 T=4096 D=1536; float32 forward
B=1 T=65536 D=2048 as 16 chained calls of 4096 steps).

--impl reference times the float64 oracle (the only other implementation of
the method here) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

WORKLOAD = 5
METRIC = "scan elements/s (B*T*D*DS) fwd+bwd"
UNIT = "elem/s"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM bytes (read + write) of one bwd2_kernel launch at workload 5, from an ncu capture of
# the same kernel at T = 512 (344.0 + 344.7 MB): traffic grows with the number of steps, so
# 4 x that at T = 2048. Reset to None whenever the kernel changes until it is captured again.
BWD2_TRAFFIC = {"bytes_per_launch": 4 * 688.759808e6,
                "source": "ncu dram__bytes_read+write of bwd2_kernel at T=512 (688.8 MB) x 4 steps ratio"}

# ---------------------------------------------------------------- algorithmic work per element

def compulsory_bytes(w, direction):
    """Bytes the step must move at least once (inputs read, outputs written)."""
    s = gen.io_bytes(w.io)
    btd, bts, ds = w.B * w.T * w.D, w.B * w.T * w.DS, w.D * w.DS
    state = w.B * w.D * w.DS * 4
    nck = gen.ceil_div(w.T, w.ckpt_interval) if w.ckpt_interval else 0
    if direction == "fwd":   # x, delta in; y out; b, c in; A in; h0 (if any) in; hT out; checkpoints out
        return btd * 3 * s + bts * 2 * s + ds * 4 + (state if w.h0_std > 0 else 0) + state + nck * state
    # bwd: x, delta, dy in; gx, gdelta out (f32); b, c in; gb, gc out (f32); A in, gA out; ckpt in; gh0 out
    return btd * (3 * s + 8) + bts * (2 * s + 8) + 2 * ds * 4 + nck * state + state


# FP32-pipe operations per element the backward needs with one recompute of the
# state from checkpoints: recompute delta*A, a*h, +delta*x*b (3); adjoint
# dy*c, g update, a*g, p = (a g) h_{t-1}, gA, gdelta, <g,b>, gb term, gc term (9).
BWD_OPS_PER_ELEM = 12
# Exponentials per element the method needs (the roofline's algorithmic count): the forward
# one; the backward two (the state recomputed once from its checkpoint, the decay once more
# in the reverse sweep). The kernels execute 1 (forward), 3 (backward: two recompute levels
# and the reverse sweep) and 2 (chunked forward: pass 1 and pass 2); the fractions below use
# the algorithmic counts.
FWD_EX2_PER_ELEM = 1
BWD_EX2_PER_ELEM = 2
BWD_EX2_EXECUTED_PER_ELEM = 3
# Per-SM rates of one GB300 SM, from bench.py --rates (bench_rates.cu: clock64-timed loops of
# independent chains, 152 SMs): ex2.approx 32.0 per clock, scalar FFMA 125 lanes per clock
# (128 nominal), packed FFMA2 62 pairs per clock.
EX2_PER_SM_CLK = 32
FP32_PER_SM_CLK = 128


# ---------------------------------------------------------------- multi-rank aggregation

def max_over_ranks(ms, device=None):
    """The slowest rank's time (ms); the identity on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(elements_per_rank_step, steps, world, max_ms):
    """Whole-job elements/s: every rank processes its own copy of the workload
    (weak scaling), timed by the slowest rank."""
    return world * elements_per_rank_step * steps / (max_ms / 1e3)


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing

def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def oracle_sample(w, budget_s=12.0, seed=0, max_batches=16):
    """Time the float64 oracle (forward with checkpoints + backward) on the first
    B' batches of workload w (all channels), B' grown until one run takes about
    budget_s seconds (at most max_batches). Returns (elements/s, cores, sample)."""
    import oracle
    B1 = 1
    while True:
        inp = gen.make_inputs(gen.workload(WORKLOAD, B=B1), seed=seed)
        args = [inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"]]
        t0 = time.perf_counter()
        oracle.fwd(*args, ckpt_interval=w.ckpt_interval)
        oracle.bwd(*args, inp["dy"])
        dt = time.perf_counter() - t0
        if dt >= budget_s / 2 or B1 >= max_batches:
            break
        B1 = min(max_batches, max(2 * B1, int(B1 * budget_s / max(dt, 1e-3))))
        del inp, args
    el = B1 * w.T * w.D * w.DS
    return el / dt, oracle.threads(), f"B={B1} T={w.T} D={w.D} DS={w.DS} (first {B1} of {w.B} batches, " \
                                      f"fwd+bwd, {dt:.1f} s)"


# ---------------------------------------------------------------- our implementation

def run_ours(args, rank, world, local_rank):
    import torch
    import selective_state_space_03_gb300 as ssm
    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = gen.workload(WORKLOAD)
    inp = gen.make_inputs(w, seed=0)
    el = gen.elements(w)
    K = w.ckpt_interval

    def to_dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    t = {k: to_dev(inp.get(k)) for k in ("x", "delta", "A", "b", "c", "h0", "dy")}
    y, hT, ckpt = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K)
    grads = ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt, t["dy"],
                             ckpt_interval=K)
    desc = ssm.make_desc(w.B, w.T, w.D, w.DS, ssm.SSM_IO_BF16, K, 0)
    import ctypes
    fwd_kernels = 2 if ssm.lib().ssm_scan_fwd_workspace_bytes(ctypes.byref(desc)) else 1
    bwd_kernels = 2 if ssm.lib().ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(desc)) else 1
    kernels_per_step = fwd_kernels + bwd_kernels

    def fwd():
        ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K, y=y, hT=hT,
                         ckpt=ckpt)

    def bwd():
        ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt, t["dy"], ckpt_interval=K,
                         grads=grads)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(el, args.steps, world, total_ms)

    if args.step_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": ms_per_step,
                              "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_only": True}), flush=True)
        return

    # the same backward with fixed-order (bitwise reproducible) gb, gc, gA sums
    ddesc = ssm.make_desc(w.B, w.T, w.D, w.DS, ssm.SSM_IO_BF16, K, 0, ssm.SSM_SCAN_DETERMINISTIC)
    det_ws = torch.empty(ssm.lib().ssm_scan_bwd_ckpt_workspace_bytes(ctypes.byref(ddesc)), dtype=torch.uint8,
                         device=dev)
    g_det = {k: torch.empty_like(v) for k, v in grads.items()}

    def bwd_det():
        ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt, t["dy"], ckpt_interval=K,
                         grads=g_det, workspace=det_ws, deterministic=True)

    bwd_det()
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(5):
        bwd_det()
    d1.record(stream)
    torch.cuda.synchronize()
    bwd_det_ms = d0.elapsed_time(d1) / 5
    del det_ws, g_det

    # the fused variant: softplus applied to delta inside the kernels and the skip y += D x
    # (delta's values are reused as the raw input: the cost does not depend on them)
    Dsk = torch.ones(w.D, dtype=torch.float32, device=dev)
    y_f, hT_f, ck_f = torch.empty_like(y), torch.empty_like(hT), torch.empty_like(ckpt)
    g_f = {k: torch.empty_like(v) for k, v in grads.items()}
    g_f["gD_skip"] = torch.empty_like(Dsk)

    def fwd_fused():
        ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K, y=y_f, hT=hT_f,
                         ckpt=ck_f, D_skip=Dsk, delta_softplus=True)

    def bwd_fused():
        ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck_f, t["dy"], ckpt_interval=K,
                         grads=g_f, D_skip=Dsk, delta_softplus=True)

    fwd_fused()
    bwd_fused()
    torch.cuda.synchronize()
    f0, f1, f2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    f0.record(stream)
    for _ in range(5):
        fwd_fused()
    f1.record(stream)
    for _ in range(5):
        bwd_fused()
    f2.record(stream)
    torch.cuda.synchronize()
    fused_fwd_ms, fused_bwd_ms = f0.elapsed_time(f1) / 5, f1.elapsed_time(f2) / 5
    del y_f, hT_f, ck_f, g_f

    # ---- end to end through the public API with host buffers. Every step copies its inputs
    # from pinned host memory and all its outputs (y, hT and the six gradients) back; the steps
    # are pipelined over three streams (copy in, compute, copy out) with two device buffer sets,
    # so step i's compute overlaps step i+1's upload and step i-1's download.
    pin = {k: (torch.from_numpy(np.ascontiguousarray(inp[k]).view(np.int16)).view(torch.bfloat16)
               if inp[k].dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(inp[k]))).pin_memory()
           for k in ("x", "delta", "A", "b", "c", "dy")}
    outs_h = {"y": torch.empty(y.shape, dtype=y.dtype).pin_memory(),
              "hT": torch.empty(hT.shape, dtype=hT.dtype).pin_memory()}
    for k, v in grads.items():
        outs_h[k] = torch.empty(v.shape, dtype=v.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in outs_h.values())
    sets = []
    for _ in range(2):
        tin = {k: torch.empty_like(t[k]) for k in pin}
        tin["h0"] = t["h0"]
        sets.append({"in": tin, "y": torch.empty_like(y), "hT": torch.empty_like(hT), "ckpt": torch.empty_like(ckpt),
                     "g": {k: torch.empty_like(v) for k, v in grads.items()}})
    s_in, s_comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_outs = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]   # downloads split over two streams
    out_keys = [["y", "gx", "gA", "gh0"], ["gdelta", "gb", "gc", "hT"]]
    assert sorted(sum(out_keys, [])) == sorted(outs_h)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]
    e2e_steps = max(4, min(args.steps, 10))

    def e2e_run(n):
        for i in range(n):
            q = i % 2
            S = sets[q]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[q])          # set q's inputs free again
                for k, v in pin.items():
                    S["in"][k].copy_(v, non_blocking=True)
                ev_in[q].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[q])
                if i >= 2:
                    for o in range(2):
                        s_comp.wait_event(ev_out[o][q])  # set q's outputs downloaded
                ti = S["in"]
                ssm.ssm_scan_fwd(ti["x"], ti["delta"], ti["A"], ti["b"], ti["c"], ti["h0"], ckpt_interval=K,
                                 y=S["y"], hT=S["hT"], ckpt=S["ckpt"])
                ssm.ssm_scan_bwd(ti["x"], ti["delta"], ti["A"], ti["b"], ti["c"], ti["h0"], S["ckpt"], ti["dy"],
                                 ckpt_interval=K, grads=S["g"])
                ev_comp[q].record(s_comp)
            dev_outs = {"y": S["y"], "hT": S["hT"], **S["g"]}
            for o, so in enumerate(s_outs):
                with torch.cuda.stream(so):
                    so.wait_event(ev_comp[q])
                    for k in out_keys[o]:
                        outs_h[k].copy_(dev_outs[k], non_blocking=True)
                    ev_out[o][q].record(so)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(e2e_steps)
    s_last = s_outs[0]
    for st in (s_in, s_comp, s_outs[1]):
        s_last.wait_stream(st)
    e1.record(s_last)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dev)
    # the last step's outputs are on the host: check one of them against the device copy
    assert torch.equal(outs_h["hT"], sets[(e2e_steps - 1) % 2]["hT"].cpu())

    # ---- other large workloads (forward only), one line each
    extra = {}
    if not args.no_extra:
        extra = other_workloads(torch, ssm, dev)

    if rank != 0:
        return
    hbm_peak, peak_kind = load_peaks()
    sm_mhz = clk.get("sm_mhz") or 2070.0
    fp32_peak = FP32_PER_SM_CLK * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6
    ex2_peak = EX2_PER_SM_CLK * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6
    bwd_ops = el * BWD_OPS_PER_ELEM / (bwd_ms / 1e3)
    fwd_ex2 = el * FWD_EX2_PER_ELEM / (fwd_ms / 1e3)
    bwd_ex2 = el * BWD_EX2_PER_ELEM / (bwd_ms / 1e3)
    fwd_bytes, bwd_bytes = compulsory_bytes(w, "fwd"), compulsory_bytes(w, "bwd")
    # the other workloads' fractions, on the same peaks (algorithmic ex2 count, compulsory bytes)
    for wk in (gen.workload(2), gen.workload(3), gen.workload(4)):
        ent = extra.get(wk.name)
        if not ent:
            continue
        elw = gen.elements(wk)
        for direction, key, n_ex2 in (("fwd", "fwd_ms", FWD_EX2_PER_ELEM), ("bwd", "bwd_ms", BWD_EX2_PER_ELEM)):
            if key not in ent:
                continue
            secs = ent[key] / 1e3
            ent[direction + "_ex2_frac"] = elw * n_ex2 / secs / ex2_peak
            ent[direction + "_hbm_frac"] = compulsory_bytes(wk, direction) / secs / 1e9 / hbm_peak
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "io_dtype": w.io,
        "data": "synthetic (seeded Philox normals, gen.make_inputs)",
        "config": workload_config(w, world),
        "kernels": {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "bwd_deterministic_ms": bwd_det_ms,
                    "fused_softplus_skip_fwd_ms": fused_fwd_ms, "fused_softplus_skip_bwd_ms": fused_bwd_ms,
                    "fwd_elem_per_s": el / (fwd_ms / 1e3), "bwd_elem_per_s": el / (bwd_ms / 1e3),
                    "fwd_hbm_gbs": fwd_bytes / (fwd_ms / 1e3) / 1e9, "bwd_hbm_gbs": bwd_bytes / (bwd_ms / 1e3) / 1e9,
                    "fwd_hbm_frac": fwd_bytes / (fwd_ms / 1e3) / 1e9 / hbm_peak,
                    "bwd_hbm_frac": bwd_bytes / (bwd_ms / 1e3) / 1e9 / hbm_peak,
                    "fwd_ex2_frac": fwd_ex2 / ex2_peak, "bwd_ex2_frac": bwd_ex2 / ex2_peak,
                    "bwd_ex2_executed_frac": bwd_ex2 * BWD_EX2_EXECUTED_PER_ELEM / BWD_EX2_PER_ELEM / ex2_peak,
                    "ex2_basis": f"algorithmic MUFU ex2 ({FWD_EX2_PER_ELEM}/element forward, {BWD_EX2_PER_ELEM}/element "
                                 f"backward; the backward executes {BWD_EX2_EXECUTED_PER_ELEM}) vs {EX2_PER_SM_CLK}"
                                 f"/clk/SM x SMs x median SM clock"},
        "roofline": {"kernel": "bwd2_kernel (reverse sweep with recompute, two channels per lane)", "bound": "alu",
                     "achieved": bwd_ops / 1e12, "peak": fp32_peak / 1e12, "unit": "TFLOP/s",
                     "frac": bwd_ops / fp32_peak, "traffic": BWD2_TRAFFIC["bytes_per_launch"],
                     "traffic_source": BWD2_TRAFFIC["source"],
                     "basis": f"{BWD_OPS_PER_ELEM} FP32-pipe ops/element x {el} elements per launch; peak = "
                              f"{FP32_PER_SM_CLK} lanes x SMs x median SM clock {sm_mhz:.0f} MHz",
                     "hbm": {"achieved": bwd_bytes / (bwd_ms / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                             "frac": bwd_bytes / (bwd_ms / 1e3) / 1e9 / hbm_peak, "peak_kind": peak_kind}},
        "e2e": {"value": el / (e2e_ms / 1e3) * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "schedule": "copy-in, compute and two copy-out streams; two device buffer sets"},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clk,
        "other_workloads": extra,
    }
    if not args.no_cpu:
        v, cores, sample = oracle_sample(w)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                                "cpu": cpu_model()}
    print(json.dumps(line), flush=True)


def other_workloads(torch, ssm, dev):
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def dev_t(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    w2 = gen.workload(2)
    i2 = gen.make_inputs(w2)
    t2 = {k: dev_t(i2.get(k)) for k in ("x", "delta", "A", "b", "c", "h0", "dy")}
    K2 = w2.ckpt_interval
    y2, h2, ck2 = ssm.ssm_scan_fwd(t2["x"], t2["delta"], t2["A"], t2["b"], t2["c"], t2["h0"], ckpt_interval=K2)
    ms_f = timed(lambda: ssm.ssm_scan_fwd(t2["x"], t2["delta"], t2["A"], t2["b"], t2["c"], t2["h0"],
                                          ckpt_interval=K2, y=y2, hT=h2, ckpt=ck2))
    g2 = ssm.ssm_scan_bwd(t2["x"], t2["delta"], t2["A"], t2["b"], t2["c"], t2["h0"], ck2, t2["dy"],
                          ckpt_interval=K2)
    ms_b = timed(lambda: ssm.ssm_scan_bwd(t2["x"], t2["delta"], t2["A"], t2["b"], t2["c"], t2["h0"], ck2,
                                          t2["dy"], ckpt_interval=K2, grads=g2))
    ms_f_lb = timed(lambda: ssm.ssm_scan_fwd(t2["x"], t2["delta"], t2["A"], t2["b"], t2["c"], t2["h0"],
                                             ckpt_interval=K2, y=y2, hT=h2, ckpt=ck2, lookback=True))
    ssm.lookback_status()
    out[w2.name] = {"fwd_ms": ms_f, "bwd_ms": ms_b, "elem_per_s": gen.elements(w2) / ((ms_f + ms_b) / 1e3),
                    "fwd_ms_lookback": ms_f_lb, "l2": "flushed"}
    del t2, y2, h2, ck2, g2, i2
    w3 = gen.workload(3)
    i3 = gen.make_inputs(w3)
    t3 = {k: dev_t(i3.get(k)) for k in ("x", "delta", "A", "b", "c", "h0")}
    y3, h3, _ = ssm.ssm_scan_fwd(t3["x"], t3["delta"], t3["A"], t3["b"], t3["c"], t3["h0"])
    ms = timed(lambda: ssm.ssm_scan_fwd(t3["x"], t3["delta"], t3["A"], t3["b"], t3["c"], t3["h0"], y=y3, hT=h3))
    out[w3.name] = {"fwd_ms": ms, "elem_per_s": gen.elements(w3) / (ms / 1e3), "l2": "flushed"}
    del t3, y3, h3, i3
    w4 = gen.workload(4)
    i4 = gen.make_inputs(w4)
    L = w4.chunk_T
    parts = []
    for k in range(w4.T // L):
        sl = slice(L * k, L * (k + 1))
        parts.append(tuple(dev_t(i4[n][:, sl]) for n in ("x", "delta", "b", "c")))
    A4, h04 = dev_t(i4["A"]), dev_t(i4["h0"])
    ys = [torch.empty_like(p[0]) for p in parts]

    def f4():
        h = h04
        for (x, d, b, c), yk in zip(parts, ys):
            _, h, _ = ssm.ssm_scan_fwd(x, d, A4, b, c, h, y=yk)

    ms = timed(f4, reps=3)
    # the same 16 calls captured once in a CUDA graph and replayed (no host launch overhead)
    sg4 = torch.cuda.Stream(dev)
    sg4.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(sg4):
        f4()
    torch.cuda.current_stream().wait_stream(sg4)
    g4 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g4, stream=sg4):
        f4()
    ms_graph = timed(g4.replay, reps=5)

    def f4_lookback():
        h = h04
        for (x, d, b, c), yk in zip(parts, ys):
            _, h, _ = ssm.ssm_scan_fwd(x, d, A4, b, c, h, y=yk, lookback=True)

    ms_lb = timed(f4_lookback, reps=3)
    with torch.cuda.stream(sg4):
        f4_lookback()
    torch.cuda.current_stream().wait_stream(sg4)
    g4lb = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g4lb, stream=sg4):
        f4_lookback()
    ms_lb_graph = timed(g4lb.replay, reps=5)
    ssm.lookback_status()
    out[w4.name] = {"fwd_ms": ms_graph, "elem_per_s": gen.elements(w4) / (ms_graph / 1e3), "calls": w4.T // L,
                    "fwd_ms_eager_calls": ms, "fwd_ms_lookback": ms_lb_graph,
                    "fwd_ms_lookback_eager_calls": ms_lb,
                    "launch": "16 chained calls replayed from one CUDA graph; lookback: one launch per call",
                    "l2": "flushed before the 16 calls"}
    del g4, g4lb
    # single-step decode at workload 5's width: one step per call, state in place; L2 flushed
    # before every step (the 5 MB state would otherwise stay in L2)
    wd = gen.workload(5, T=1)
    idd = gen.make_inputs(wd, with_grad_inputs=False)
    td = {k: dev_t(idd.get(k)) for k in ("x", "delta", "A", "b", "c")}
    xs, ds, bs, cs = (td[k][:, 0].contiguous() for k in ("x", "delta", "b", "c"))
    hd = torch.zeros((wd.B, wd.D, 16), dtype=torch.float32, device=dev)
    yd = torch.empty_like(xs)
    ssm.ssm_scan_step(xs, ds, td["A"], bs, cs, hd, y=yd)
    ts = []
    for _ in range(50):
        flush.zero_()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ssm.ssm_scan_step(xs, ds, td["A"], bs, cs, hd, y=yd)
        b_.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b_))
    us_cold = statistics.median(ts) * 1e3
    nbytes = 2 * wd.B * wd.D * 16 * 4 + 3 * wd.B * wd.D * 2 + 2 * wd.B * 16 * 2 + wd.D * 16 * 4
    # steady state: 32 sessions' states (168 MB, more than L2) stepped round-robin, 64 steps
    # captured in one CUDA graph so host launch overhead is not timed
    # (the sessions' inputs are computed before the steps, so consecutive steps may declare
    # SSM_SCAN_STEP_INPUTS_READY; timed also without it, every load waiting for the step before)
    nsess, nstep = 32, 64
    hss = [torch.zeros_like(hd) for _ in range(nsess)]
    sg = torch.cuda.Stream(dev)

    def graph_us(ready):
        sg.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(sg):
            for k in range(nsess):
                ssm.ssm_scan_step(xs, ds, td["A"], bs, cs, hss[k], y=yd, inputs_ready=ready)
        torch.cuda.current_stream().wait_stream(sg)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=sg):
            for k in range(nstep):
                ssm.ssm_scan_step(xs, ds, td["A"], bs, cs, hss[k % nsess], y=yd, inputs_ready=ready)
        graph.replay()
        torch.cuda.synchronize()
        reps = 10
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b_.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b_) * 1e3 / (reps * nstep)

    us = graph_us(True)
    us_wait = graph_us(False)
    out["decode_step_bf16_B16_D5120"] = {
        "us_per_step": us, "elem_per_s": wd.B * wd.D * 16 / (us / 1e6), "hbm_gbs": nbytes / (us / 1e6) / 1e9,
        "hbm_frac": nbytes / (us / 1e6) / 1e9 / load_peaks()[0], "bytes_per_step": nbytes,
        "schedule": f"{nstep} steps over {nsess} sessions' states in one CUDA graph (states exceed L2), "
                    f"inputs declared ready (SSM_SCAN_STEP_INPUTS_READY)",
        "us_per_step_all_loads_wait": us_wait,
        "us_single_step_after_l2_flush": us_cold}
    del hss
    return out


# ---------------------------------------------------------------- reference arm (the oracle)

def workload_config(w, world):
    """The `config` object of both arms' JSON lines (the same workload, named by its shape)."""
    return {"workload": w.name, "B": w.B, "T": w.T, "D": w.D, "DS": w.DS, "io": w.io,
            "state_and_grads": "f32", "ckpt_interval": w.ckpt_interval,
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = gen.workload(WORKLOAD)
    # size the per-step sample so that warm-up + timed steps take a few minutes at most
    budget = max(2.0, 120.0 / max(1, args.steps + args.warmup))
    _, cores, sample = oracle_sample(w, budget_s=budget)
    B1 = int(sample.split("B=")[1].split()[0])
    inp = gen.make_inputs(gen.workload(WORKLOAD, B=B1), seed=0)
    a = [inp["x"], inp["delta"], inp["A"], inp["b"], inp["c"], inp["h0"]]

    def step():
        oracle.fwd(*a, ckpt_interval=w.ckpt_interval)
        oracle.bwd(*a, inp["dy"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    el = B1 * w.T * w.D * w.DS
    v = el / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Philox normals, gen.make_inputs)",
            "config": workload_config(w, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"B={B1} T={w.T} D={w.D} DS={w.DS} per step (fwd+bwd)", "cpu": cpu_model()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """One warm-up and one more forward(+backward) of workload 5, or of the workload
    --workload names (optionally with B/T replaced), for profilers; prints nothing but 'ok'."""
    import torch
    import selective_state_space_03_gb300 as ssm
    over = {k: v for k, v in (("B", args.B), ("T", args.T)) if v}
    w = gen.workload(args.workload or WORKLOAD, **over)
    inp = gen.make_inputs(w, seed=0)
    dev = torch.device("cuda", 0)

    def to_dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    t = {k: to_dev(inp.get(k)) for k in ("x", "delta", "A", "b", "c", "h0", "dy")}
    K = w.ckpt_interval
    if args.decode:
        # decode steps at the workload's width: the inputs of step 0, the state carried in place
        h = torch.zeros((w.B, w.D, w.DS), dtype=torch.float32, device=dev)
        xs, ds, bs, cs = (t[k][:, 0].contiguous() for k in ("x", "delta", "b", "c"))
        for _ in range(4):
            ssm.ssm_scan_step(xs, ds, t["A"], bs, cs, h)
        torch.cuda.synchronize()
        print("ok")
        return
    for _ in range(2):
        _, _, ck = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ckpt_interval=K)
        if w.bwd:
            ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["b"], t["c"], t["h0"], ck, t["dy"], ckpt_interval=K)
    torch.cuda.synchronize()
    print("ok")


def run_rates():
    """Build and run bench_rates.cu (per-SM ex2, FFMA, FFMA2, shuffle and shared-load rates,
    and a 2 GiB device copy) and print its JSON line: the measurements behind the roofline
    constants above."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "bench_rates")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(ROOT, "bench_rates.cu")], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, check=True)
    print(r.stdout.strip(), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other two workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--step-only", action="store_true",
                    help="time only the forward+backward steps (no other measurements), e.g. under a profiler")
    ap.add_argument("--profile", action="store_true",
                    help="run one warm-up and one forward+backward for a profiler, no timing")
    ap.add_argument("--workload", type=int, default=0, help="with --profile: workload 1-5 instead of 5")
    ap.add_argument("--B", type=int, default=0, help="with --profile: batch size instead of 16")
    ap.add_argument("--T", type=int, default=0, help="with --profile: sequence length instead of 2048")
    ap.add_argument("--decode", action="store_true", help="with --profile: 4 decode steps instead of fwd+bwd")
    ap.add_argument("--rates", action="store_true",
                    help="measure the per-SM unit rates the roofline uses (bench_rates.cu) and exit")
    args = ap.parse_args()
    if args.rates:
        run_rates()
        return
    if args.profile:
        run_profile_case(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

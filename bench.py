#!/usr/bin/env python
"""Benchmark: one training-step attention pass (forward + backward) per step.

Workload (the fwd/bwd configuration): B=2, H=16, N=8192, d=128, BF16, causal,
Q, K, V, dO iid N(0,1) from a fixed seed.  One step = attn_fwd followed by the
three stages of attn_bwd (prepare, dK/dV, dQ) through the C ABI, inputs resident
in HBM.  FLOPs per step are the algorithmic count: forward 4*B*H*N^2*d plus
backward 10*B*H*N^2*d, both halved for causal.  The inputs (4 x 64 MiB) exceed
the 129 MB L2, so no flush runs between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the
workload (the heads are independent; there is no exchange step), the elapsed
time is the max over ranks and `value` counts the work of all ranks.
`--impl reference` times the FP64 CPU oracle on a bounded slice of the same
workload (rank 0 only).

Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s (4*B*H*N^2*d fwd + 10*B*H*N^2*d bwd, halved causal) at 1 GB300"
UNIT = "TFLOP/s"
WORKLOAD = "c5"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="skip the long-sequence forward side numbers")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    p.add_argument("--forward", metavar="WORKLOAD[:causal]",
                   help="time only attn_fwd on one named workload (c1..c5) for a kernel capture, then exit")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def config_dict(w, n_gpus):
    return {"workload": f"training-step attention B={w.B} H={w.H} N={w.N} d={w.d} {w.dtype} causal fwd+bwd",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True, "dtype": w.dtype,
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU",
            "l2": "no flush: inputs 256 MiB > 129 MB L2"}


def step_flops(w):
    return workloads.fwd_flops(w.B, w.H, w.N, w.d, True) + workloads.bwd_flops(w.B, w.H, w.N, w.d, True)


# ---------------------------------------------------------------- clocks


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries) every 2 ms
    while the timed region runs, so that even a timed region of a few tens of
    milliseconds collects a dozen samples or more.  The device is found by its UUID, so
    CUDA_VISIBLE_DEVICES renumbering does not matter."""

    # nvmlClocksEventReasons bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}
    PERIOD_S = 0.002

    def __init__(self, dev):
        import ctypes

        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        self.ct = ctypes
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            return
        self.h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        found = False
        if uuid is not None:
            u = str(uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            found = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) == 0
        if not found and lib.nvmlDeviceGetHandleByIndex_v2(int(dev.index or 0), ctypes.byref(self.h)) != 0:
            return
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
        self.ok = True
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct, lib = self.ct, self.lib
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.time()
            if lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0:  # NVML_CLOCK_SM
                r = int(rs.value) if get_reasons(self.h, ct.byref(rs)) == 0 else 0
                self.samples.append((t, float(clk.value), r))
            time.sleep(self.PERIOD_S)

    def stop(self, t0, t1):
        if not self.ok:
            return None
        self._stop.set()
        self.thread.join(timeout=2)
        rows = [(c, r) for t, c, r in self.samples if t0 <= t <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = sorted({n for _, r in rows for n, b in self.BITS.items() if r & b})
        return {"sm_mhz": statistics.median(c for c, _ in rows), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(rows), "source": "nvml, every 2 ms"}


class SmiClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs
    (used where NVML cannot be loaded directly)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9 or not (t0 - 0.05 <= ts <= t1 + 0.15):
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvidia-smi"}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi, every 100 ms"}


def clock_sampler(dev):
    s = NvmlClockSampler(dev)
    return s if s.ok else SmiClockSampler(dev.index or 0)


# ---------------------------------------------------------------- peaks and profiles


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


KERNEL_SOURCES = {"fwd": ["fwd.cu"], "bwd_prepare": ["bwd.cu"], "bwd_dkdv": ["bwd.cu", "bwd_common.cuh"],
                  "bwd_dq": ["bwd.cu", "bwd_common.cuh"]}


def source_digest(kernel: str):
    """Hash of the source files a kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_online_softmax_attention_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel] + ["ptx.cuh", "common.cuh"]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
    except (OSError, ValueError):
        return None
    ent = d.get(kernel)
    if not ent or ent.get("source_digest") != source_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- our arm


def run_ours(args, w, ws_, rank, local):
    import tiled_online_softmax_attention_gb300 as attn

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    attn.load(build_if_missing=True)
    x = workloads.inputs(WORKLOAD)
    B, H, N, d = w.B, w.H, w.N, w.d
    scale = w.scale
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = attn.attn_bwd_deterministic_workspace_bytes(B, H, N, d)  # the stages below need only this
    wsp = torch.empty(nbytes, device=dev, dtype=torch.uint8)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    dt = q.dtype

    def check(rc, what):
        if rc != attn.ATTN_OK:
            raise RuntimeError(f"{what}: {attn.attn_status_string(rc)}")

    names = ["fwd", "bwd_prepare", "bwd_dkdv", "bwd_dq"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        check(attn.attn_fwd(q, k, v, o, lse, B, H, N, d, dt, True, scale, status, stream), "attn_fwd")
        if ev is not None:
            ev[1].record(stream)
        check(attn.attn_bwd_prepare(o, do, lse, wsp, nbytes, B, H, N, d, dt, stream), "attn_bwd_prepare")
        if ev is not None:
            ev[2].record(stream)
        check(attn.attn_bwd_dkdv(q, k, v, do, wsp, nbytes, dk, dv, B, H, N, d, dt, True, scale, status, stream),
              "attn_bwd_dkdv")
        if ev is not None:
            ev[3].record(stream)
        check(attn.attn_bwd_dq(q, k, v, do, wsp, nbytes, dq, B, H, N, d, dt, True, scale, status, stream),
              "attn_bwd_dq")
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = clock_sampler(dev) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    barrier(ws_)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(ws_)
    clocks = sampler.stop(wall0, wall1) if sampler is not None else None
    if int(status.item()) != 0:
        raise RuntimeError("device-side wait expired in the timed region")
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = allreduce_max(elapsed_ms, ws_, dev)
    per_kernel = {n: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / args.steps for j, n in enumerate(names)}

    # Algorithmic FLOPs per launch (causal halves every N x N product):
    unit = 2.0 * B * H * N * N * d / 2          # one N x N x d product, causal
    kflops = {"fwd": 2 * unit, "bwd_prepare": 0.0, "bwd_dkdv": 4 * unit, "bwd_dq": 1 * unit}
    kbytes = {"bwd_prepare": 2 * B * H * N * d * 2 + B * H * N * 4 + nbytes}   # read O, dO, lse; write D, LSE2
    flops = step_flops(w)
    value = ws_ * args.steps * flops / (elapsed_ms * 1e-3) / 1e12
    pk = peaks()
    dom = max(per_kernel, key=per_kernel.get)
    achieved = kflops[dom] / (per_kernel[dom] * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                "traffic": recorded_traffic(dom), "peak_source": pk["source"] + " bf16 burst",
                "flops_per_launch": kflops[dom]}
    kernels = {}
    for n in names:
        ent = {"ms": round(per_kernel[n], 4)}
        if kflops[n]:
            ent["tflops"] = round(kflops[n] / (per_kernel[n] * 1e-3) / 1e12, 1)
            ent["frac_of_peak"] = round(kflops[n] / (per_kernel[n] * 1e-3) / 1e12 / pk["bf16_tflops"], 4)
        else:
            ent["gbs"] = round(kbytes[n] / (per_kernel[n] * 1e-3) / 1e9, 1)
        kernels[n] = ent

    e2e = None if args.no_e2e else run_e2e(args, w, x, dev, ws_)
    extra = None if args.no_extra else long_forward(attn, dev)
    return {"value": value, "ms_per_step": elapsed_ms / args.steps, "roofline": roofline, "kernels": kernels,
            "clocks": clocks, "e2e": e2e, "gpu_launches": 4 * args.steps, "extra": extra}


def run_e2e(args, w, x, dev, ws_):
    """Same metric through the public API with host buffers: every step copies its Q, K, V,
    dO from pinned host memory to the device and its three gradients back, inside the
    timed region.  Reported two ways: serial (copy in, compute, copy out, one stream) and
    pipelined (double-buffered: step k+1's inputs and step k-1's gradients move on copy
    streams while step k computes, as a training loop would overlap them)."""
    import tiled_online_softmax_attention_gb300 as attn

    hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "dout"))
    hin = (hq, hk, hv, hdo)
    hout = [[torch.empty_like(hq).pin_memory() for _ in range(3)] for _ in range(2)]
    steps = max(3, min(args.steps, 50))
    nb = hq.numel() * hq.element_size()
    B, H, N = w.B, w.H, w.N

    def serial_step():
        q, k, v, do = (t.to(dev, non_blocking=True) for t in hin)
        o, lse = attn.forward(q, k, v, causal=True, scale=w.scale)
        g = attn.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
        for h, t in zip(hout[0], g):
            h.copy_(t, non_blocking=True)

    def timed(fn):
        for i in range(3):
            fn(i, 3)
        torch.cuda.synchronize()
        barrier(ws_)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(steps):
            fn(i, steps)
        torch.cuda.current_stream().wait_stream(h2d)
        torch.cuda.current_stream().wait_stream(d2h)
        b.record()
        torch.cuda.synchronize()
        return allreduce_max(a.elapsed_time(b), ws_, dev)

    # pipelined: two device input sets and two output sets
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = torch.cuda.current_stream(dev)
    din = [[torch.empty_like(t, device=dev) for t in hin] for _ in range(2)]
    dres = [(torch.empty_like(din[0][0]), torch.empty((B, H, N), device=dev, dtype=torch.float32),
             torch.empty_like(din[0][0]), torch.empty_like(din[0][0]), torch.empty_like(din[0][0]))
            for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    for e in in_free + out_free:
        e.record(comp)

    def load(i):
        s = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(in_free[s])
            for dt, ht in zip(din[s], hin):
                dt.copy_(ht, non_blocking=True)
            in_ready[s].record(h2d)

    def pipelined_step(i, n):
        s = i % 2
        if i == 0:
            load(0)
        if i + 1 < n:
            load(i + 1)  # the next step's inputs move while this one computes
        comp.wait_event(in_ready[s])
        comp.wait_event(out_free[s])
        q, k, v, do = din[s]
        o, lse, dq, dk, dv = dres[s]
        attn.forward(q, k, v, causal=True, scale=w.scale, out=(o, lse))
        attn.backward(q, k, v, o, lse, do, causal=True, scale=w.scale, out=(dq, dk, dv))
        in_free[s].record(comp)
        out_ready[s].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(out_ready[s])
            for ht, dt in zip(hout[s], (dq, dk, dv)):
                ht.copy_(dt, non_blocking=True)
            out_free[s].record(d2h)

    ms_serial = timed(lambda i, n: serial_step())
    ms_pipe = timed(pipelined_step)
    flops = step_flops(w)
    return {"value": ws_ * steps * flops / (ms_pipe * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": 4 * nb, "d2h_bytes_per_step": 3 * nb, "steps": steps,
            "mode": "pipelined: step k+1's H2D and step k-1's D2H overlap step k's kernels",
            "serial_value": ws_ * steps * flops / (ms_serial * 1e-3) / 1e12}


def long_forward(attn, dev):
    """Side numbers: the long-sequence forward (B=1, H=32, N=16384, d=128, bf16), both masks."""
    w = workloads.WORKLOADS["c3"]
    x = workloads.inputs("c3")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    out = {}
    for causal in (False, True):
        f = workloads.fwd_flops(w.B, w.H, w.N, w.d, causal)
        for _ in range(3):
            attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, q.dtype, causal, w.scale)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for _ in range(reps):
            attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, q.dtype, causal, w.scale)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        out["causal" if causal else "non_causal"] = {"ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1)}
    res = {"long_forward_B1_H32_N16384_d128": out}
    res["split_kv_B1_H1_N16384_d128"] = split_forward(attn, dev)
    res["decode_B1_H32_Nq128_Nk32768_d128"] = decode_forward(attn, dev)
    res["decode_B1_H16_Nq128_Nk32768_d256"] = decode_forward(attn, dev, 16, 256)
    res["decode_varlen_4seqs_H8_d128"] = decode_varlen_forward(attn, dev)
    res["forward_by_workload"] = forward_by_workload(attn, dev)
    res["forward_d64_vs_d128_grid"] = forward_grid_sweep(attn, dev)
    res["fp8_forward_B1_H32_N16384_d128"] = fp8_forward(attn, dev)
    res["d256_forward_and_step_B1_H16_N16384"] = d256_side(attn, dev)
    res["dropout_training_step_p0.1"] = dropout_step(attn, dev)
    res["backward_paths_B2_H16_N8192"] = backward_modes(attn, dev)
    return res


def backward_modes(attn, dev):
    """The training-step backward alone (B=2, H=16, N=8192, d=128, causal), FLOPs counted
    10*B*H*N^2*d/2: attn_bwd (the two deterministic kernels as one grid), the fused pass
    through its stages (prepare, dK/dV/dQ, dQ finish: five products per tile pair, dQ
    through a float32 accumulator), and attn_bwd_deterministic."""
    w = workloads.WORKLOADS["c5"]
    x = workloads.inputs("c5")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    B, H, N, d, dt, sc = w.B, w.H, w.N, w.d, q.dtype, w.scale
    attn.attn_fwd(q, k, v, o, lse, B, H, N, d, dt, True, sc)
    nb = attn.attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(nb, device=dev, dtype=torch.uint8)
    nbd = attn.attn_bwd_deterministic_workspace_bytes(B, H, N, d)

    def fused():
        attn.attn_bwd_prepare(o, do, lse, ws, nb, B, H, N, d, dt)
        attn.attn_bwd_dkdvdq(q, k, v, do, ws, nb, dk, dv, B, H, N, d, dt, True, sc)
        attn.attn_bwd_dq_finish(ws, nb, dq, B, H, N, d, dt, sc)

    out = {}
    for name, run in (("attn_bwd", lambda: attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, nb, B, H, N, d, dt, True,
                                                          sc)),
                      ("fused_stages", fused),
                      ("deterministic", lambda: attn.attn_bwd_deterministic(q, k, v, o, do, lse, dq, dk, dv, ws, nbd, B,
                                                                            H, N, d, dt, True, sc))):
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for _ in range(reps):
            run()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        f = workloads.bwd_flops(B, H, N, d, True)
        out[name] = {"ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1)}
    return out


def dropout_step(attn, dev):
    """The training-step workload (forward + backward) with dropout p = 0.1, against the
    same step without dropout (the dropout entry points with p = 0), and with the keep
    decisions drawn once (attn_fwd_dropout_bits / attn_bwd_dropout_bits); FLOPs counted as
    without dropout."""
    w = workloads.WORKLOADS["c5"]
    x = workloads.inputs("c5")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    nb = attn.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(nb, device=dev, dtype=torch.uint8)
    out = {}
    for p in (0.0, 0.1):
        def step():
            attn.attn_fwd_dropout(q, k, v, o, lse, w.B, w.H, w.N, w.d, q.dtype, True, w.scale, p, 1234)
            attn.attn_bwd_dropout(q, k, v, o, do, lse, dq, dk, dv, ws, nb, w.B, w.H, w.N, w.d, q.dtype, True,
                                  w.scale, p, 1234)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for _ in range(reps):
            step()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        out[f"p{p}"] = {"ms": round(ms, 4), "tflops": round(step_flops(w) / (ms * 1e-3) / 1e12, 1)}
    # the keep decisions drawn once: the forward stores them, the backward reads them
    nbits = attn.attn_dropout_bits_bytes(w.B, w.H, w.N, w.N)
    bits = torch.empty(nbits, device=dev, dtype=torch.uint8)

    def step_bits():
        attn.attn_fwd_dropout_bits(q, k, v, o, lse, bits, nbits, w.B, w.H, w.N, w.d, q.dtype, True, w.scale, 0.1,
                                   1234)
        attn.attn_bwd_dropout_bits(q, k, v, o, do, lse, bits, nbits, dq, dk, dv, ws, nb, w.B, w.H, w.N, w.d, q.dtype,
                                   True, w.scale, 0.1)
    for _ in range(3):
        step_bits()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    a.record()
    for _ in range(reps):
        step_bits()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    out["p0.1_keep_bits"] = {"ms": round(ms, 4), "tflops": round(step_flops(w) / (ms * 1e-3) / 1e12, 1),
                             "keep_bits_bytes": nbits}
    return out


def d256_side(attn, dev):
    """Head dimension 256: B=1, H=16, N=16384, bf16, both masks; the forward alone (one
    query tile per CTA) and the training step (forward + the three-kernel backward); the
    causal step again with dropout p = 0.1 (FLOPs counted as without dropout)."""
    B, H, N, d = 1, 16, 16384, 256
    x = workloads.draw(B, H, N, d, "bf16", seed=13, with_dout=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    nb = attn.attn_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(nb, device=dev, dtype=torch.uint8)
    scale = 1.0 / math.sqrt(d)

    def timed(call, reps):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            call()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    out = {}
    for causal in (False, True):
        fwd = lambda: attn.attn_fwd(q, k, v, o, lse, B, H, N, d, q.dtype, causal, scale)

        def step():
            fwd()
            attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, nb, B, H, N, d, q.dtype, causal, scale)
        ms = timed(fwd, 10)
        ms_step = timed(step, 5)
        ff = workloads.fwd_flops(B, H, N, d, causal)
        fs = ff + workloads.bwd_flops(B, H, N, d, causal)
        out["causal" if causal else "non_causal"] = {
            "ms": round(ms, 4), "tflops": round(ff / (ms * 1e-3) / 1e12, 1),
            "step_ms": round(ms_step, 4), "step_tflops": round(fs / (ms_step * 1e-3) / 1e12, 1)}
        if causal:
            def step_drop():
                attn.attn_fwd_dropout(q, k, v, o, lse, B, H, N, d, q.dtype, True, scale, 0.1, 1234)
                attn.attn_bwd_dropout(q, k, v, o, do, lse, dq, dk, dv, ws, nb, B, H, N, d, q.dtype, True, scale,
                                      0.1, 1234)
            ms_drop = timed(step_drop, 5)
            out["causal"]["dropout_p0.1_step_ms"] = round(ms_drop, 4)
            out["causal"]["dropout_p0.1_step_tflops"] = round(fs / (ms_drop * 1e-3) / 1e12, 1)
    return out


def fp8_forward(attn, dev):
    """The long-sequence forward on block-scaled E4M3 inputs (attn_fwd_fp8), both masks,
    against the 8-bit tensor peak: the measured bf16 peak times the nominal fp8/bf16
    ratio (4.5 / 2.25 PFLOP/s)."""
    B, H, N, d = 1, 32, 16384, 128
    x = {k: t.to(dev) for k, t in workloads.draw_fp8(B, H, N, d, seed=2).items()}
    o = torch.empty((B, H, N, d), device=dev, dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]
    out = {"peak_tflops": round(fp8_peak, 1), "peak_source": pk["source"] + " bf16 x 2 (nominal fp8/bf16)"}
    for causal in (False, True):
        call = lambda: attn.attn_fwd_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"], x["v_scale"], o, lse,
                                         B, H, N, d, o.dtype, causal, 1.0 / math.sqrt(d))
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for _ in range(reps):
            call()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        tf = workloads.fwd_flops(B, H, N, d, causal) / (ms * 1e-3) / 1e12
        out["causal" if causal else "non_causal"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                                     "frac_of_fp8_peak": round(tf / fp8_peak, 3)}
    return out


def forward_grid_sweep(attn, dev):
    """Non-causal forward at d = 64 and d = 128 over sequence length and head count (B = 1,
    N(0,1) inputs, one call at a time after a 256 MiB L2 flush, median of 15): separates the
    per-CTA cost of short sequences (few key tiles, few waves) from the per-key-tile rate
    that long sequences reach.  d = 64 at N = 1024, 96 heads is the c2 shape."""
    flush = torch.empty(256 << 20, device=dev, dtype=torch.uint8)
    out = {}
    for d in (64, 128):
        for N in (1024, 4096):
            for BH in (96, 768):
                g = torch.Generator().manual_seed(N + BH + d)
                q, k, v = (torch.randn((1, BH, N, d), generator=g).to(torch.bfloat16).to(dev) for _ in range(3))
                o = torch.empty_like(q)
                lse = torch.empty((1, BH, N), device=dev, dtype=torch.float32)
                call = lambda: attn.attn_fwd(q, k, v, o, lse, 1, BH, N, d, q.dtype, False, 1 / math.sqrt(d))
                for _ in range(3):
                    call()
                ts = []
                for _ in range(15):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    call()
                    b.record()
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b))
                ms = sorted(ts)[len(ts) // 2]
                f = workloads.fwd_flops(1, BH, N, d, False)
                out[f"d{d}_N{N}_heads{BH}"] = {"ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1),
                                               "ctas": BH * ((N + 255) // 256)}
                del q, k, v, o, lse
    return out


def forward_by_workload(attn, dev):
    """Forward TFLOP/s on the parity workloads c1, c2, c4 (both masks where they have them).
    c1 and c2 are short sequences: they also get HBM GB/s (algorithmic bytes: Q, K, V read,
    O and the logsumexp written, over the time), timed one call at a time with L2 flushed
    (a 256 MiB write) before each, since their inputs would otherwise stay in the 129 MB L2."""
    out = {}
    flush = torch.empty(256 << 20, device=dev, dtype=torch.uint8)
    for name in ("c1", "c2", "c4"):
        w = workloads.WORKLOADS[name]
        x = workloads.inputs(name)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
        for causal in w.causal:
            call = lambda: attn.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, q.dtype, causal, w.scale)
            for _ in range(5):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 50
            a.record()
            for _ in range(reps):
                call()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            f = workloads.fwd_flops(w.B, w.H, w.N, w.d, causal)
            ent = {"ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1)}
            if name in ("c1", "c2"):
                nbytes = 4 * q.numel() * q.element_size() + lse.numel() * 4  # Q, K, V, O + lse
                tot = 0.0
                for _ in range(20):
                    flush.zero_()
                    a.record()
                    call()
                    b.record()
                    torch.cuda.synchronize()
                    tot += a.elapsed_time(b)
                ms_cold = tot / 20
                ent.update({"ms_l2_flushed": round(ms_cold, 4),
                            "hbm_gbs_l2_flushed": round(nbytes / (ms_cold * 1e-3) / 1e9, 1)})
            out[f"{name}_{'causal' if causal else 'non_causal'}"] = ent
    return out


def split_forward(attn, dev):
    """One head of 16384 tokens: 64 query-tile pairs cannot fill 152 SMs alone; the
    split-KV forward cuts each pair's keys into ranges (then merges them)."""
    B, H, N, d = 1, 1, 16384, 128
    x = workloads.draw(B, H, N, d, "bf16", seed=5)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    sc = 1.0 / math.sqrt(d)
    out = {}
    for causal in (False, True):
        f = workloads.fwd_flops(B, H, N, d, causal)
        ent = {}
        for ns in (1, 2, 4, 8):
            nb = attn.attn_fwd_splitkv_workspace_bytes(B, H, N, d, ns)
            ws = torch.empty(nb, device=dev, dtype=torch.uint8)
            if ns == 1:
                call = lambda: attn.attn_fwd(q, k, v, o, lse, B, H, N, d, q.dtype, causal, sc)
            else:
                call = lambda: attn.attn_fwd_splitkv(q, k, v, o, lse, ws, nb, B, H, N, d, q.dtype, causal, sc, ns)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                call()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / 20
            ent["attn_fwd" if ns == 1 else f"splits_{ns}"] = {"ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1)}
        out["causal" if causal else "non_causal"] = ent
    return out


def decode_forward(attn, dev, H=32, d=128):
    """Decode-like shape: B=1, H heads, 128 new queries against 32768 keys (causal: the
    queries are the last 128 positions), head dimension d.  attn_fwd_rect has one CTA per
    head (a query-tile pair at d <= 128, one query tile at d = 256);
    attn_fwd_splitkv_rect cuts the keys into ranges.  FLOPs: two Nq x Nk x d products
    (causal: the visible part, the last 128 rows of the triangle)."""
    B, Nq, Nk = 1, 128, 32768
    g = torch.Generator().manual_seed(17)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device=dev, dtype=torch.float32)
    sc = 1.0 / math.sqrt(d)
    out = {}
    for causal in (False, True):
        visible = Nq * Nk - (Nq * (Nq - 1) // 2 if causal else 0)
        f = 4.0 * B * H * visible * d
        ent = {}
        for ns in (1, 4, 8, 16):
            nb = attn.attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, ns)
            ws = torch.empty(nb, device=dev, dtype=torch.uint8)
            if ns == 1:
                call = lambda: attn.attn_fwd_rect(q, k, v, o, lse, B, H, Nq, Nk, d, q.dtype, causal, sc)
            else:
                call = lambda: attn.attn_fwd_splitkv_rect(q, k, v, o, lse, ws, nb, B, H, Nq, Nk, d, q.dtype, causal,
                                                          sc, ns)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                call()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / 20
            kv_gbs = 2 * B * H * Nk * d * 2 / (ms * 1e-3) / 1e9
            ent["attn_fwd_rect" if ns == 1 else f"splits_{ns}"] = {
                "ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1), "kv_read_gbs": round(kv_gbs, 1)}
        out["causal" if causal else "non_causal"] = ent
    return out


def decode_varlen_forward(attn, dev):
    """A ragged decode-like batch: 4 sequences of 128 new queries after 8192, 16384, 24576
    and 32768 positions (keys 8320 .. 32896), H = 8, d = 128, bf16, causal and not, packed:
    attn_fwd_varlen (one CTA per sequence and head, 32 CTAs) against
    attn_fwd_varlen_splitkv with 4, 8 and 16 ranges.  FLOPs: the visible part of each
    sequence's 128 x Nk scores, two products."""
    H, d, nq = 8, 128, 128
    lens_k = [8192 + nq, 16384 + nq, 24576 + nq, 32768 + nq]
    B, Tq, Tk = len(lens_k), nq * len(lens_k), sum(lens_k)
    g = torch.Generator().manual_seed(23)
    q = torch.randn((Tq, H, d), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((Tk, H, d), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((Tk, H, d), generator=g).to(torch.bfloat16).to(dev)
    cu_q = torch.arange(0, Tq + 1, nq, dtype=torch.int32, device=dev)
    cu_k = torch.tensor([0] + list(torch.tensor(lens_k).cumsum(0).tolist()), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((H, Tq), device=dev, dtype=torch.float32)
    sc = 1.0 / math.sqrt(d)
    out = {}
    for causal in (False, True):
        visible = sum(nq * n - (nq * (nq - 1) // 2 if causal else 0) for n in lens_k)
        f = 4.0 * H * visible * d
        ent = {}
        for ns in (1, 4, 8, 16):
            nb = attn.attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d, ns)
            ws = torch.empty(nb, device=dev, dtype=torch.uint8)
            if ns == 1:
                call = lambda: attn.attn_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, B, H, nq, max(lens_k), Tq, Tk, d,
                                                    q.dtype, causal, sc)
            else:
                call = lambda: attn.attn_fwd_varlen_splitkv(q, k, v, o, lse, ws, nb, cu_q, cu_k, B, H, nq, max(lens_k),
                                                            Tq, Tk, d, q.dtype, causal, sc, ns)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(20):
                call()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / 20
            kv_gbs = 2 * Tk * H * d * 2 / (ms * 1e-3) / 1e9
            ent["attn_fwd_varlen" if ns == 1 else f"splits_{ns}"] = {
                "ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1), "kv_read_gbs": round(kv_gbs, 1)}
        out["causal" if causal else "non_causal"] = ent
    return out


# ---------------------------------------------------------------- oracle (CPU) timings


def oracle_slice(x, b, h, n_tok):
    """The causal top-left n_tok x n_tok block of one head: exactly the work its first n_tok queries do."""
    return tuple(x[n][b, h, :n_tok] for n in ("q", "k", "v", "dout"))


def time_oracle(x, w, heads, n_tok):
    import oracle

    t0 = time.perf_counter()
    for (b, h) in heads:
        q, k, v, do = oracle_slice(x, b, h, n_tok)
        oracle.attn_fwd(q, k, v, True, w.scale)
        oracle.attn_bwd(q, k, v, do, True, w.scale)
    sec = time.perf_counter() - t0
    flops = len(heads) * (workloads.fwd_flops(1, 1, n_tok, w.d, True) + workloads.bwd_flops(1, 1, n_tok, w.d, True))
    return sec, flops


def cpu_baseline(x, w):
    import oracle

    heads, n_tok = [(0, h) for h in range(12)], w.N
    sec, flops = time_oracle(x, w, heads, n_tok)
    return {"value": flops / sec / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"FP64 oracle forward+backward on 12 whole heads (batch 0, heads 0-11, N={n_tok}) of the "
                      f"workload, {sec:.1f} s"}


def run_reference(args, w):
    import oracle

    x = workloads.inputs(WORKLOAD)
    n_tok = 2048
    for i in range(args.warmup):
        time_oracle(x, w, [(0, i % w.H)], n_tok)
    total_s, total_f = 0.0, 0.0
    for i in range(args.steps):
        s, f = time_oracle(x, w, [(i // w.H % w.B, i % w.H)], n_tok)
        total_s += s
        total_f += f
    value = total_f / total_s / 1e12
    sample = f"FP64 oracle forward+backward, one head per step, first {n_tok} tokens (causal top-left block)"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- distributed plumbing

_PG = None


def init_dist(ws_, local):
    global _PG
    if ws_ > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        _PG = dist


def barrier(ws_):
    if ws_ > 1 and _PG is not None:
        _PG.barrier()


def allreduce_max(val: float, ws_, dev):
    if ws_ > 1 and _PG is not None:
        t = torch.tensor([val], dtype=torch.float64, device=dev)
        _PG.all_reduce(t, op=_PG.ReduceOp.MAX)
        return float(t.item())
    return val


def forward_only(args):
    """attn_fwd alone on one named workload, --warmup untimed and --steps timed calls: the
    command the single-kernel captures of the forward run (a JSON line with the time)."""
    import tiled_online_softmax_attention_gb300 as api

    name, _, mask = args.forward.partition(":")
    w = workloads.WORKLOADS[name]
    causal = mask == "causal"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    api.load(build_if_missing=True)
    x = workloads.inputs(name)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    status = torch.zeros(1, device=dev, dtype=torch.int32)
    call = lambda: api.attn_fwd(q, k, v, o, lse, w.B, w.H, w.N, w.d, q.dtype, causal, w.scale, status)
    for _ in range(args.warmup):
        assert call() == 0
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        call()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / max(args.steps, 1)
    f = workloads.fwd_flops(w.B, w.H, w.N, w.d, causal)
    print(json.dumps({"forward": args.forward, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
                      "ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 1), "status": int(status.item())}),
          flush=True)


def main():
    args = parse()
    if args.forward:
        forward_only(args)
        return
    ws_, rank, local = dist_env()
    w = workloads.WORKLOADS[WORKLOAD]
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return
    init_dist(ws_, local)
    r = run_ours(args, w, ws_, rank, local)
    if rank == 0:
        line = {"metric": METRIC, "value": round(r["value"], 2), "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_dict(w, ws_), "roofline": r["roofline"], "kernels": r["kernels"],
                "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"]}
        if r["extra"]:
            line["extra"] = r["extra"]
        if ws_ == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(workloads.inputs(WORKLOAD), w)
        print(json.dumps(line), flush=True)
    if ws_ > 1 and _PG is not None:
        _PG.barrier()
        _PG.destroy_process_group()


if __name__ == "__main__":
    main()

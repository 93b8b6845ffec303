#!/usr/bin/env python3
"""Benchmark: attention forward + backward TFLOP/s at B8 H32 L4096 D128 fp16.

One step = the whole hot path on one batch of synthetic inputs already in
HBM: forward (O, LSE), Delta preprocess (+ dQ accumulator zeroing), the
backward main pass (dK, dV, dQ accumulator) and the dQ post-process.  FLOPs
follow the usual convention: 4*B*H*L^2*D for the forward, 2.5x that for the
backward, halved under causal masking.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--causal]

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (one (batch, head) unit's forward + backward per
step) and prints the same metric.  Under torchrun (N > 1) every rank runs its
own replica (independent batches, no collective on the data path) and the
reported time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import csv
import datetime
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORK = dict(B=8, L=4096, H=32, Hkv=32, D=128, dtype="fp16")
# Named workloads (the default is the headline one); --causal applies on top.
WORKLOADS = {
    "b8_h32_l4096_d128": dict(B=8, L=4096, H=32, Hkv=32, D=128, dtype="fp16"),
    "b1_h2_l128_d64": dict(B=1, L=128, H=2, Hkv=2, D=64, dtype="fp16"),
    "gqa_b4_h32_hkv8_l4096_d128_bf16": dict(B=4, L=4096, H=32, Hkv=8, D=128, dtype="bf16"),
    "b8_h32_l1024_d64": dict(B=8, L=1024, H=32, Hkv=32, D=64, dtype="fp16"),
    "b1_h32_l1024_d128": dict(B=1, L=1024, H=32, Hkv=32, D=128, dtype="fp16"),
    "b1_h32_l4096_d128": dict(B=1, L=4096, H=32, Hkv=32, D=128, dtype="fp16"),
    "b1_h32_l8192_d128": dict(B=1, L=8192, H=32, Hkv=32, D=128, dtype="fp16"),
    "b1_h32_l16384_d128": dict(B=1, L=16384, H=32, Hkv=32, D=128, dtype="fp16"),
    # prefill of 1024 new queries against an 8192-position key/value sequence
    "prefill_b8_h32_lq1024_lk8192_d128": dict(B=8, L=1024, Lk=8192, H=32, Hkv=32, D=128,
                                              dtype="fp16"),
    # split-KV decoding (forward only): few new queries against a long key/value sequence
    "decode_b16_h32_hkv8_lq1_lk16384_d128_bf16": dict(mode="decode", B=16, L=1, Lk=16384, H=32,
                                                      Hkv=8, D=128, dtype="bf16"),
    "decode_b1_h32_hkv8_lq1_lk131072_d128_bf16": dict(mode="decode", B=1, L=1, Lk=131072, H=32,
                                                      Hkv=8, D=128, dtype="bf16"),
    "decode_b8_h32_hkv8_lq4_lk32768_d128_bf16": dict(mode="decode", B=8, L=4, Lk=32768, H=32,
                                                     Hkv=8, D=128, dtype="bf16"),
    # forward on E4M3 inputs (per-tensor scales), bf16 output
    "fp8_b8_h32_l4096_d128": dict(mode="fp8", B=8, L=4096, H=32, Hkv=32, D=128, dtype="bf16"),
    "fp8_gqa_b4_h32_hkv8_l4096_d128": dict(mode="fp8", B=4, L=4096, H=32, Hkv=8, D=128,
                                           dtype="bf16"),
}
METRIC = "attention fwd/bwd TFLOP/s (fp16 B8 H32 L4096 D128) and % of GB300 TC peak"
# Dense FP16/BF16 tensor rate per GPU from NVIDIA's published HGX B300 figures
# (36 PFLOP/s per 8 GPUs with 2:4 sparsity, i.e. 2.25 PFLOP/s dense per GPU).
DATASHEET_FP16_TFLOPS = 2250.0
DECODE_METRIC = "attention split-KV decode GB/s (Q, K, V read + O, LSE written)"
FP8_METRIC = "attention forward on E4M3 inputs TFLOP/s (4*B*H*L^2*D, halved causal)"
_CSRC = "tiled_attention_fa_gb300/csrc/"
_COMMON = [_CSRC + "ptx.cuh", _CSRC + "common.cuh", _CSRC + "fwd.cuh"]
# Sources each kernel is compiled from (a recorded DRAM figure is valid only
# while these still hash to the value stored beside it).
KERNEL_SOURCES = {
    "fa_fwd_kernel": _COMMON,
    "fa_bwd_prep_kernel": _COMMON + [_CSRC + "bwd.cuh"],
    "fa_bwd_kernel": _COMMON + [_CSRC + "bwd.cuh"],
    "fa_dq_convert_kernel": _COMMON + [_CSRC + "bwd.cuh"],
    "fa_decode_kernel": _COMMON + [_CSRC + "decode.cuh"],
    "fa_decode_combine_kernel": _COMMON + [_CSRC + "decode.cuh"],
    "fa_fwd_kernel_e4m3": _COMMON,
}


def fwd_flops(B, H, L, D, causal, Lk=None):
    """4*B*H*Lq*Lk*D; causal counts the visible (query, key) pairs, i.e. half
    the square for Lq == Lk and Lq*(Lk-Lq) + Lq^2/2 when the queries are the
    last Lq of Lk positions."""
    Lk = L if Lk is None else Lk
    pairs = (L * (Lk - L) + L * L / 2.0) if causal else float(L) * Lk
    return 4.0 * B * H * D * pairs


def step_flops(B, H, L, D, causal, Lk=None):
    return 3.5 * fwd_flops(B, H, L, D, causal, Lk)   # forward + 2.5x backward


def decode_bytes(B, Lq, Lk, H, Hkv, D, esize=2):
    """Bytes decoding must move: Q, K, V read once, O and LSE written once."""
    return esize * (2 * B * Lq * H * D + 2 * B * Lk * Hkv * D) + 4 * B * H * Lq


def is_decode():
    return WORK.get("mode") == "decode"


def is_fp8():
    return WORK.get("mode") == "fp8"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            m = json.load(fh)
        return m["bf16_tflops"], m["bf16_tflops_sustained"], m["hbm_gbs"], "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


def source_hash(kernel):
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary, or
    None when absent or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as fh:
            for line in fh:
                f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
                if f.get("kernel") == kernel and f.get("src") == source_hash(kernel):
                    return float(f["dram_bytes_per_launch"])
    except OSError:
        pass
    return None


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 20 ms; only samples stamped inside the timed
    region (between start() returning and stop() being called) count."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index, enabled=True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.tmp = None
        self.t0 = None

    def start(self):
        if not self.enabled:
            return
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        self.t0 = datetime.datetime.now()

    @staticmethod
    def summarize(rows, t0, t1):
        """Median SM clock, peak clock and active throttle reasons of the rows
        (nvidia-smi CSV, timestamp first) stamped within [t0, t1]."""
        sm, mx, pw, reasons, total = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f")
                clk, cmax = float(r[2]), float(r[3])
            except ValueError:
                continue
            total += 1
            if not (t0 <= ts <= t1):
                continue
            sm.append(clk)
            mx.append(cmax)
            try:
                pw.append(float(r[4]))
            except ValueError:
                pass
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None,
               "reasons": sorted(reasons), "samples": len(sm), "samples_outside": total - len(sm)}
        if pw:
            out["power_w_median"] = statistics.median(pw)
        if not sm:
            out["reasons"] = ["no sample inside the timed region"]
        return out

    def stop(self):
        if not self.enabled:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t1 = datetime.datetime.now()
        time.sleep(3 * self.PERIOD_MS / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = list(csv.reader(io.StringIO(self.tmp.read())))
        os.unlink(self.tmp.name)
        return self.summarize(rows, self.t0, t1)


# --------------------------------------------------------------------- oracle timing

def blas_threads():
    """Threads the host BLAS uses (OpenBLAS query when the library exposes one)."""
    import ctypes
    import numpy as np  # noqa: F401  (loads numpy's BLAS)
    try:
        with open("/proc/self/maps") as fh:
            libs = {ln.split()[-1] for ln in fh if "openblas" in ln.lower() and "/" in ln}
    except OSError:
        libs = set()
    for lib in libs:
        try:
            h = ctypes.CDLL(lib)
        except OSError:
            continue
        for name in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                     "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            fn = getattr(h, name, None)
            if fn is not None:
                return int(fn())
    return len(os.sched_getaffinity(0))


def time_oracle_units(q, k, v, do, causal, n_units, budget_s):
    """Run the oracle's forward+backward on (b, h) units until ``n_units`` or
    ``budget_s`` seconds; returns (units done, seconds)."""
    from oracle import fa_oracle as orc
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    done, t0 = 0, time.perf_counter()
    for u in range(n_units):
        b, h = u % B, (u // B) % H
        hk = orc.kv_head(h, H, Hkv)
        orc.unit_backward(q[b, :, h], k[b, :, hk], v[b, :, hk], do[b, :, h], causal)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def time_oracle_workload(causal, budget_s):
    """Time the oracle's forward+backward over every (b, h) unit of the whole
    workload when one unit's time says that fits in ``budget_s``; returns
    (seconds, units) or None when it would not fit."""
    from oracle import fa_oracle as orc
    from tiled_attention_fa_gb300.inputs import make_qkv
    B, L, H, Hkv, D = WORK["B"], WORK["L"], WORK["H"], WORK["Hkv"], WORK["D"]
    if WORK.get("Lk", L) != L:
        return None
    q1, k1, v1, do1 = cpu_unit_inputs()
    t0 = time.perf_counter()
    orc.unit_backward(q1[0, :, 0], k1[0, :, 0], v1[0, :, 0], do1[0, :, 0], causal)
    if (time.perf_counter() - t0) * B * H > budget_s:
        return None
    q, k, v, do = (t.double().numpy() for t in make_qkv(B, L, H, Hkv, D, WORK["dtype"], seed=0))
    t0 = time.perf_counter()
    for b in range(B):
        for h in range(H):
            hk = orc.kv_head(h, H, Hkv)
            orc.unit_backward(q[b, :, h], k[b, :, hk], v[b, :, hk], do[b, :, h], causal)
    return time.perf_counter() - t0, B * H


def cpu_unit_inputs(seed=0):
    """One (b, h) unit of the workload, [1, L, 1, D] float64 host arrays (same recipe as the tests)."""
    from tiled_attention_fa_gb300.inputs import make_qkv
    q, k, v, do = make_qkv(1, WORK["L"], 1, 1, WORK["D"], WORK["dtype"], seed=seed)
    return tuple(t.double().numpy() for t in (q, k, v, do))


# --------------------------------------------------------------------- arms

def dist_setup():
    from tiled_attention_fa_gb300.replicas import dist_env
    return dist_env()


def reference_arm(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    if is_decode():
        return decode_reference_arm(args, world)
    if is_fp8():
        return fp8_reference_arm(args, world)
    L, D = WORK["L"], WORK["D"]
    qs, ks, vs, dos = cpu_unit_inputs()
    flops_unit = step_flops(1, 1, L, D, args.causal)
    time_oracle_units(qs, ks, vs, dos, args.causal, args.warmup, 1e9)
    n, secs = time_oracle_units(qs, ks, vs, dos, args.causal, args.steps, 1e9)
    value = n * flops_unit / secs / 1e12
    cores = blas_threads()
    sample = (f"oracle fp64 forward+backward of one (batch, head) unit per step "
              f"(L={L}, D={D}, {'causal' if args.causal else 'non-causal'}), {n} steps")
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": secs / n * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(args, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


def config_dict(args, world):
    B, L, H, Hkv, D = WORK["B"], WORK["L"], WORK["H"], WORK["Hkv"], WORK["D"]
    Lk = WORK.get("Lk", L)
    lens = f"L{L}" if Lk == L else f"Lq{L} Lk{Lk}"
    return {"workload": f"attention fwd+bwd B{B} H{H} Hkv{Hkv} {lens} D{D} {WORK['dtype']} "
                        f"{'causal' if args.causal else 'non-causal'}",
            "B": B, "L": L, "Lk": Lk, "H": H, "Hkv": Hkv, "D": D, "causal": bool(args.causal),
            "per_gpu_batch": B, "global_batch": B * world, "parallelism": f"replicas x{world}",
            "l2": ("inputs larger than L2 (Q, K, V, dO %d MB each)" % (B * L * H * D * 2 // 10**6)
                   if B * L * H * D * 2 > 129 * 10**6 else "inputs fit in L2 (no flush)")}


def ours_arm(args):
    if is_decode():
        return decode_arm(args)
    if is_fp8():
        return fp8_arm(args)
    import torch
    import tiled_attention_fa_gb300 as fa
    from tiled_attention_fa_gb300 import _lib, replicas

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    replicas.init("nccl", dev)
    _lib.load()  # fails loudly without the built library

    B, L, H, Hkv, D = WORK["B"], WORK["L"], WORK["H"], WORK["Hkv"], WORK["D"]
    Lk = WORK.get("Lk", L)
    causal = bool(args.causal)
    dt = torch.float16 if WORK["dtype"] == "fp16" else torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(replicas.replica_seed(1234, rank))
    q = torch.randn(B, L, H, D, device=dev, dtype=dt, generator=g)
    k = torch.randn(B, Lk, Hkv, D, device=dev, dtype=dt, generator=g)
    v = torch.randn(B, Lk, Hkv, D, device=dev, dtype=dt, generator=g)
    do = torch.randn(B, L, H, D, device=dev, dtype=dt, generator=g)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, L, device=dev, dtype=torch.float32)
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    acc = fa.alloc_workspace(B, L, H, D, dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        fa.fwd(q, k, v, causal, out=o, lse=lse, stream=stream)
        if ev:
            ev[1].record(stream)
        fa.bwd_preprocess(o, do, delta=delta, dq_accum=acc, stream=stream)
        if ev:
            ev[2].record(stream)
        if Lk == L:
            fa.bwd_main(q, k, v, do, lse, delta, acc, causal, dk=dk, dv=dv, accum_zeroed=True,
                        stream=stream)
            if ev:
                ev[3].record(stream)
            fa.bwd_postprocess(acc, dq, stream=stream)
        else:  # fa_bwd_kv runs both stages; the post-process share is attributed to the main pass
            fa.bwd(q, k, v, o, do, lse, delta, causal, dq=dq, dk=dk, dv=dv, dq_accum=acc,
                   accum_zeroed=True, stream=stream)
            if ev:
                ev[3].record(stream)
        if ev:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    fa.check_device_error()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    replicas.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    replicas.barrier()
    clocks = sampler.stop()
    fa.check_device_error()
    ms = replicas.max_over_ranks(t_start.elapsed_time(t_end), dev)
    ms_per_step = ms / args.steps

    names = ["fa_fwd_kernel", "fa_bwd_prep_kernel", "fa_bwd_kernel", "fa_dq_convert_kernel"]
    per = {n: [e[i].elapsed_time(e[i + 1]) for e in evs] for i, n in enumerate(names)}
    kms = {n: statistics.mean(v) for n, v in per.items()}
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    f_fwd = fwd_flops(B, H, L, D, causal, Lk)
    f_bwd = 2.5 * f_fwd
    Lpad = (L + 127) // 128 * 128
    prep_bytes = 2 * B * L * H * D * 2 + 4 * B * H * L + 4 * B * H * Lpad * D
    conv_bytes = 4 * B * H * Lpad * D + 2 * B * L * H * D
    burst, sustained, hbm, src = peaks()
    kernels = {
        "fa_fwd_kernel": {"ms": kms["fa_fwd_kernel"], "tflops": f_fwd / kms["fa_fwd_kernel"] / 1e9},
        "fa_bwd_prep_kernel": {"ms": kms["fa_bwd_prep_kernel"],
                               "gbs": prep_bytes / kms["fa_bwd_prep_kernel"] / 1e6},
        "fa_bwd_kernel": {"ms": kms["fa_bwd_kernel"], "tflops": f_bwd / kms["fa_bwd_kernel"] / 1e9},
        "fa_dq_convert_kernel": {"ms": kms["fa_dq_convert_kernel"],
                                 "gbs": conv_bytes / kms["fa_dq_convert_kernel"] / 1e6},
    }
    for n in names:  # spread over the timed steps (the mean is "ms")
        kernels[n]["ms_median"] = statistics.median(per[n])
        kernels[n]["ms_min"] = min(per[n])
    for n in ("fa_fwd_kernel", "fa_bwd_kernel"):
        kernels[n]["frac_of_burst"] = kernels[n]["tflops"] / burst
        kernels[n]["frac_of_sustained"] = kernels[n]["tflops"] / sustained
        kernels[n]["frac_of_datasheet"] = kernels[n]["tflops"] / DATASHEET_FP16_TFLOPS
    dom = max(names, key=lambda n: kms[n])
    if dom in ("fa_fwd_kernel", "fa_bwd_kernel"):
        # The kernels run for milliseconds inside a sub-second timed region: the
        # burst figure (a GEMM timed alone) is the matching peak; the
        # sustained figure (seconds back to back, under the power cap) and the
        # datasheet's dense rate are reported beside it.
        ach = kernels[dom]["tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": burst,
                "unit": "TFLOP/s", "frac": ach / burst,
                "peak_source": f"{src} bf16 burst (fp16 dense rate equals bf16)",
                "frac_of_sustained": ach / sustained,
                "frac_of_datasheet": ach / DATASHEET_FP16_TFLOPS}
    else:
        ach = kernels[dom]["gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": f"{src} copy bandwidth"}
    roof["traffic"] = recorded_traffic(dom)

    value = replicas.aggregate_rate(step_flops(B, H, L, D, causal, Lk), world, ms_per_step * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        # HostPipeline: every step uploads its inputs from pinned host memory and
        # reads its results back; one step's copies overlap its neighbours' kernels.
        runner = fa.HostPipeline(B, L, H, Hkv, D, dt, causal, dev, Lk=Lk)
        hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, do))
        for _ in range(2):
            runner.submit(hq, hk, hv, hdo)
        runner.wait()
        n_e2e = max(3, min(args.steps, 10))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        replicas.barrier()
        torch.cuda.synchronize()
        s0.record(runner.up)
        for _ in range(n_e2e):
            runner.submit(hq, hk, hv, hdo)
        s1.record(runner.down)
        runner.wait()
        torch.cuda.synchronize()
        ems = replicas.max_over_ranks(s0.elapsed_time(s1) / n_e2e, dev)
        e2e = {"value": replicas.aggregate_rate(step_flops(B, H, L, D, causal, Lk), world, ems * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": runner.h2d_bytes(),
               "d2h_bytes_per_step": runner.d2h_bytes(), "ms_per_step": ems, "steps": n_e2e}
        del runner

    # ---- oracle on the host cores (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        full = time_oracle_workload(causal, 3 * args.cpu_budget)
        if full is not None:
            secs, n = full
            cpu = {"value": step_flops(B, H, L, D, causal) / secs / 1e12, "unit": "TFLOP/s",
                   "cores": blas_threads(), "kind": "oracle",
                   "sample": f"the whole workload: all {n} (batch, head) units, forward+backward "
                             f"in fp64 ({secs:.1f} s)"}
        else:
            uq, uk, uv, udo = cpu_unit_inputs()
            n, secs = time_oracle_units(uq, uk, uv, udo, causal, 100000, args.cpu_budget)
            cpu = {"value": n * step_flops(1, 1, L, D, causal) / secs / 1e12, "unit": "TFLOP/s",
                   "cores": blas_threads(), "kind": "oracle",
                   "sample": f"{n} (batch, head) unit(s) of the workload, forward+backward in "
                             f"fp64 ({secs:.1f} s)"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": WORK["dtype"],
            "data": "synthetic", "config": config_dict(args, world),
            "frac_of_peak": {"burst": value / world / burst, "sustained": value / world / sustained,
                             "datasheet": value / world / DATASHEET_FP16_TFLOPS, "source": src},
            "step_stats": {"ms_mean": statistics.mean(step_ms), "ms_median": statistics.median(step_ms),
                           "ms_min": min(step_ms), "ms_max": max(step_ms),
                           "note": "this rank's per-step CUDA events; ms_per_step is the "
                                   "max-over-ranks whole-region time / steps"},
            "kernels": kernels, "roofline": roof, "clocks": clocks, "e2e": e2e,
            "cpu_baseline": cpu, "gpu_launches": 4 * args.steps,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0

# --------------------------------------------------------------------- decoding

def decode_config(args, world):
    B, Lq, Lk, H, Hkv, D = (WORK[x] for x in ("B", "L", "Lk", "H", "Hkv", "D"))
    kv = 2 * B * Lk * Hkv * D * 2
    return {"workload": f"attention split-KV decode B{B} H{H} Hkv{Hkv} Lq{Lq} Lk{Lk} D{D} "
                        f"{WORK['dtype']} {'causal' if args.causal else 'non-causal'}",
            "B": B, "Lq": Lq, "Lk": Lk, "H": H, "Hkv": Hkv, "D": D, "causal": bool(args.causal),
            "per_gpu_batch": B, "global_batch": B * world, "parallelism": f"replicas x{world}",
            "l2": (f"inputs larger than L2 (K and V {kv // 10**6} MB)" if kv > 129 * 10**6
                   else "inputs fit in L2 (no flush)")}


def time_oracle_groups(q, k, v, causal, n_groups, budget_s):
    """Oracle forward of whole (batch, K/V head) groups (its g query heads,
    all Lq queries) until ``n_groups`` or ``budget_s``; returns (groups, s)."""
    from oracle import fa_oracle as orc
    H, Hkv = q.shape[2], k.shape[2]
    g = H // Hkv
    done, t0 = 0, time.perf_counter()
    for u in range(n_groups):
        hk = u % Hkv
        for h in range(hk * g, (hk + 1) * g):
            orc.unit_forward(q[0, :, h], k[0, :, hk], v[0, :, hk], causal)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def decode_group_inputs(seed=0):
    """One batch entry of the decode workload as float64 host arrays."""
    from tiled_attention_fa_gb300.inputs import make_qkv_kv
    q, k, v, _ = make_qkv_kv(1, WORK["L"], WORK["Lk"], WORK["H"], WORK["Hkv"], WORK["D"],
                             WORK["dtype"], seed=seed)
    return tuple(t.double().numpy() for t in (q, k, v))


def group_bytes():
    Lq, Lk, H, Hkv, D = (WORK[x] for x in ("L", "Lk", "H", "Hkv", "D"))
    return decode_bytes(1, Lq, Lk, H, Hkv, D) / Hkv


def decode_reference_arm(args, world):
    qs, ks, vs = decode_group_inputs()
    time_oracle_groups(qs, ks, vs, args.causal, args.warmup, 1e9)
    n, secs = time_oracle_groups(qs, ks, vs, args.causal, args.steps, 1e9)
    value = n * group_bytes() / secs / 1e9
    sample = (f"oracle fp64 forward of one (batch, K/V head) group ({WORK['H'] // WORK['Hkv']} "
              f"query heads x Lq={WORK['L']}, Lk={WORK['Lk']}) per step, {n} steps")
    out = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": secs / n * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": decode_config(args, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


def decode_arm(args):
    import torch
    import tiled_attention_fa_gb300 as fa
    from tiled_attention_fa_gb300 import _lib, replicas

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    replicas.init("nccl", dev)
    _lib.load()  # fails loudly without the built library

    B, Lq, Lk, H, Hkv, D = (WORK[x] for x in ("B", "L", "Lk", "H", "Hkv", "D"))
    causal = bool(args.causal)
    dt = torch.float16 if WORK["dtype"] == "fp16" else torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(replicas.replica_seed(4321, rank))
    q = torch.randn(B, Lq, H, D, device=dev, dtype=dt, generator=g)
    k = torch.randn(B, Lk, Hkv, D, device=dev, dtype=dt, generator=g)
    v = torch.randn(B, Lk, Hkv, D, device=dev, dtype=dt, generator=g)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, device=dev, dtype=torch.float32)
    ws = fa.alloc_decode_workspace(B, Lq, Lk, H, Hkv, D, dev)
    kv_bytes = 2 * k.numel() * k.element_size()
    # Between timed steps an L2-sized buffer is rewritten when K/V would fit in L2.
    flush = None if kv_bytes > 129 * 10**6 else torch.empty(256 << 20, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if flush is not None:
            flush.zero_()
        if ev:
            ev[0].record(stream)
        fa.decode_slices(q, k, v, ws, causal, stream=stream)
        if ev:
            ev[1].record(stream)
        fa.decode_merge(ws, o, lse, Lk, Hkv, stream=stream)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    fa.check_device_error()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    replicas.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    replicas.barrier()
    clocks = sampler.stop()
    fa.check_device_error()
    if flush is None:
        ms = t_start.elapsed_time(t_end) / args.steps
    else:  # the L2 flush between steps is not part of a step
        ms = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
    ms_per_step = replicas.max_over_ranks(ms, dev)
    kms = {"fa_decode_kernel": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
           "fa_decode_combine_kernel": statistics.mean(e[1].elapsed_time(e[2]) for e in evs)}
    alg = decode_bytes(B, Lq, Lk, H, Hkv, D)
    part = fa.decode_workspace_size(B, Lq, Lk, H, Hkv, D)
    slice_bytes = kv_bytes + q.numel() * q.element_size() + part
    merge_bytes = part + o.numel() * o.element_size() + lse.numel() * 4
    _, _, hbm, src = peaks()
    kernels = {
        "fa_decode_kernel": {"ms": kms["fa_decode_kernel"],
                             "gbs": slice_bytes / kms["fa_decode_kernel"] / 1e6},
        "fa_decode_combine_kernel": {"ms": kms["fa_decode_combine_kernel"],
                                     "gbs": merge_bytes / kms["fa_decode_combine_kernel"] / 1e6},
    }
    ach = kernels["fa_decode_kernel"]["gbs"]
    roof = {"kernel": "fa_decode_kernel", "bound": "hbm", "achieved": ach, "peak": hbm,
            "unit": "GB/s", "frac": ach / hbm, "peak_source": f"{src} copy bandwidth",
            "traffic": recorded_traffic("fa_decode_kernel"),
            "algorithmic_bytes_per_launch": slice_bytes}
    value = replicas.aggregate_rate(alg, world, ms_per_step * 1e-3) / 1e9
    tflops = fwd_flops(B, H, Lq, D, causal, Lk) / (ms_per_step * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        runner = fa.DecodeHostRunner(B, Lq, Lk, H, Hkv, D, dt, causal, dev)
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        runner.run(hq, hk, hv)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        replicas.barrier()
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(n_e2e):
            runner.run(hq, hk, hv, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize()
        ems = replicas.max_over_ranks(s0.elapsed_time(s1) / n_e2e, dev)
        e2e = {"value": replicas.aggregate_rate(alg, world, ems * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": runner.h2d_bytes(), "d2h_bytes_per_step": runner.d2h_bytes(),
               "ms_per_step": ems, "steps": n_e2e}
        del runner

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qs, ks, vs = decode_group_inputs()
        n, secs = time_oracle_groups(qs, ks, vs, causal, 100000, args.cpu_budget)
        cpu = {"value": n * group_bytes() / secs / 1e9, "unit": "GB/s", "cores": blas_threads(),
               "kind": "oracle",
               "sample": f"{n} (batch, K/V head) group(s) of the workload, forward in fp64 "
                         f"({secs:.1f} s)"}

    if rank == 0:
        out = {
            "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": WORK["dtype"], "data": "synthetic", "config": decode_config(args, world),
            "tflops": tflops, "kernels": kernels, "roofline": roof, "clocks": clocks, "e2e": e2e,
            "cpu_baseline": cpu, "gpu_launches": 2 * args.steps,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------- E4M3 forward

def fp8_config(args, world):
    B, L, H, Hkv, D = (WORK[x] for x in ("B", "L", "H", "Hkv", "D"))
    return {"workload": f"attention forward E4M3 inputs B{B} H{H} Hkv{Hkv} L{L} D{D} -> "
                        f"{WORK['dtype']} {'causal' if args.causal else 'non-causal'}",
            "B": B, "L": L, "H": H, "Hkv": Hkv, "D": D, "causal": bool(args.causal),
            "per_gpu_batch": B, "global_batch": B * world, "parallelism": f"replicas x{world}",
            "l2": (f"inputs larger than L2 (Q {B * L * H * D // 10**6} MB, K and V "
                   f"{2 * B * L * Hkv * D // 10**6} MB)")}


def time_oracle_fp8_units(q8, k8, v8, scales, causal, n_units, budget_s):
    """Oracle FP8 forward of one (b, h) unit at a time (decode + forward)."""
    from oracle import fa_oracle as orc
    qs, ks, vs = scales
    H, Hkv = q8.shape[2], k8.shape[2]
    done, t0 = 0, time.perf_counter()
    for u in range(n_units):
        h = u % H
        hk = orc.kv_head(h, H, Hkv)
        orc.unit_forward(orc.e4m3_decode(q8[0, :, h]) * qs, orc.e4m3_decode(k8[0, :, hk]) * ks,
                         orc.e4m3_decode(v8[0, :, hk]) * vs, causal)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def fp8_unit_inputs(seed=0):
    from tiled_attention_fa_gb300.inputs import make_qkv_fp8
    q8, k8, v8, qs, ks, vs = make_qkv_fp8(1, WORK["L"], WORK["L"], WORK["H"], WORK["Hkv"],
                                          WORK["D"], seed=seed)
    return q8.numpy(), k8.numpy(), v8.numpy(), (qs, ks, vs)


def fp8_reference_arm(args, world):
    L, D = WORK["L"], WORK["D"]
    q8, k8, v8, sc = fp8_unit_inputs()
    time_oracle_fp8_units(q8, k8, v8, sc, args.causal, args.warmup, 1e9)
    n, secs = time_oracle_fp8_units(q8, k8, v8, sc, args.causal, args.steps, 1e9)
    value = n * fwd_flops(1, 1, L, D, args.causal) / secs / 1e12
    sample = (f"oracle fp64 forward of one (batch, head) unit of E4M3 inputs per step (L={L}, "
              f"D={D}, {'causal' if args.causal else 'non-causal'}), {n} steps")
    out = {
        "impl": "reference", "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": secs / n * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": fp8_config(args, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


def fp8_arm(args):
    import torch
    import tiled_attention_fa_gb300 as fa
    from tiled_attention_fa_gb300 import _lib, replicas

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    replicas.init("nccl", dev)
    _lib.load()  # fails loudly without the built library

    B, L, H, Hkv, D = (WORK[x] for x in ("B", "L", "H", "Hkv", "D"))
    causal = bool(args.causal)
    out_dt = torch.bfloat16 if WORK["dtype"] == "bf16" else torch.float16
    g = torch.Generator(device=dev).manual_seed(replicas.replica_seed(777, rank))

    def codes(*shape):
        x = torch.randn(*shape, device=dev, dtype=torch.float32, generator=g)
        s = float(x.abs().max()) / 448.0
        return (x / s).to(torch.float8_e4m3fn).view(torch.uint8), s

    (q8, qs), (k8, ks), (v8, vs) = codes(B, L, H, D), codes(B, L, Hkv, D), codes(B, L, Hkv, D)
    o = torch.empty(B, L, H, D, device=dev, dtype=out_dt)
    lse = torch.empty(B, H, L, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def step():
        fa.fwd_fp8(q8, k8, v8, qs, ks, vs, causal, out_dtype=out_dt, out=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    fa.check_device_error()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    replicas.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    replicas.barrier()
    clocks = sampler.stop()
    fa.check_device_error()
    ms = t_start.elapsed_time(t_end) / args.steps          # one launch per step
    ms_per_step = replicas.max_over_ranks(ms, dev)
    flops = fwd_flops(B, H, L, D, causal)
    ach = flops / (ms * 1e-3) / 1e12
    burst, sustained, hbm, src = peaks()
    # E4M3 dense tensor rate = 2x the 16-bit rate on this part (4.5 vs 2.25 PFLOP/s nominal).
    # A kernel of about a millisecond timed alone: the burst figure applies
    # (sustained beside it), scaled by the nominal E4M3 : BF16 dense ratio of 2.
    peak = 2.0 * burst
    roof = {"kernel": "fa_fwd_kernel (E4M3)", "bound": "tensor", "achieved": ach, "peak": peak,
            "unit": "TFLOP/s", "frac": ach / peak,
            "peak_source": f"{src} bf16 burst x 2 (nominal E4M3 / BF16 dense ratio)",
            "frac_of_sustained": ach / (2.0 * sustained), "frac_of_16bit_burst": ach / burst,
            "traffic": recorded_traffic("fa_fwd_kernel_e4m3")}
    value = replicas.aggregate_rate(flops, world, ms_per_step * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        runner = fa.Fp8HostRunner(B, L, L, H, Hkv, D, out_dt, causal, dev)
        hq, hk, hv = (x.cpu().pin_memory() for x in (q8, k8, v8))
        runner.run(hq, hk, hv, qs, ks, vs)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        replicas.barrier()
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(n_e2e):
            runner.run(hq, hk, hv, qs, ks, vs, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize()
        ems = replicas.max_over_ranks(s0.elapsed_time(s1) / n_e2e, dev)
        e2e = {"value": replicas.aggregate_rate(flops, world, ems * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": runner.h2d_bytes(), "d2h_bytes_per_step": runner.d2h_bytes(),
               "ms_per_step": ems, "steps": n_e2e}
        del runner

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        uq, uk, uv, sc = fp8_unit_inputs()
        n, secs = time_oracle_fp8_units(uq, uk, uv, sc, causal, 100000, args.cpu_budget)
        cpu = {"value": n * fwd_flops(1, 1, L, D, causal) / secs / 1e12, "unit": "TFLOP/s",
               "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n} (batch, head) unit(s) of the workload, E4M3 decode + forward in "
                         f"fp64 ({secs:.1f} s)"}

    if rank == 0:
        out = {
            "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic", "config": fp8_config(args, world),
            "kernels": {"fa_fwd_kernel (E4M3)": {"ms": ms, "tflops": ach}}, "roofline": roof,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--causal", action="store_true", help="causal masking (default: non-causal)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the nvidia-smi clock sampler (for profiler runs)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="b8_h32_l4096_d128")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (smaller values only for profiling captures)")
    args = ap.parse_args()
    WORK.update(WORKLOADS[args.workload])
    if args.batch is not None:
        WORK["B"] = args.batch
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)
    return ours_arm(args)


if __name__ == "__main__":
    sys.exit(main())

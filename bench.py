#!/usr/bin/env python3
"""Attention forward throughput on one GB300 (or N replicas), printed as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one FlashAttention forward pass (the whole hot path: one kernel)
over one batch of the workload.  ``value`` is the attention-forward rate in
TFLOPS with FLOPs = 4 B H T^2 d, halved for a causal mask, inputs resident in
HBM.  Between timed steps the inputs rotate over enough copies that their
total exceeds twice the L2, so no step starts with its operands in L2.
``e2e`` is the same metric through the public Python API with pinned host
buffers: every step copies Q, K, V in and O, LSE out inside the timed region.

``--impl reference`` times the float64 CPU oracle (the slow, plain
definition) on the host cores instead, on a bounded sample of the same
workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fa_inputs as fi  # noqa: E402

DEFAULT_WORKLOAD = "long_causal_b1h32t32768d128"
METRIC = "attention fwd TFLOPS (bf16, 1 GB300) and % of dense BF16 tensor peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
SWEEP_DEFAULT = ["tiny_causal_b1h4t256d64", "gpt2s_causal_b8h12t1024d64", "gpt2m_b16h16t1024d64",
                 "gpt2m_stress_b16h16t1024d64", "llama8b_causal_b1h32t4096d128", "llama8b_b1h32t4096d128",
                 "long_causal_b1h32t32768d128"]
# split-KV (fa_fwd_splitkv, split count chosen by the library) against fa_fwd on the same inputs: shapes
# with fewer work units than SMs, where one head's long rows would otherwise leave SMs idle
SPLITKV_SWEEP = {"splitkv_tiny_causal_b1h4t256d64": dict(B=1, H=4, T=256, d=64, causal=True),
                 "splitkv_prefill_causal_b1h4t8192d128": dict(B=1, H=4, T=8192, d=128, causal=True),
                 "splitkv_single_causal_b1h1t32768d128": dict(B=1, H=1, T=32768, d=128, causal=True)}
# grouped K/V heads: Llama-3.1-8B attention (32 query heads sharing 8 K/V heads), causal and not
GQA_SWEEP = {"llama8b_gqa_causal_b1h32kv8t4096d128": dict(B=1, H=32, Hkv=8, T=4096, d=128, causal=True),
             "llama8b_gqa_b1h32kv8t4096d128": dict(B=1, H=32, Hkv=8, T=4096, d=128, causal=False)}


def metric_flops(B, H, T, d, causal):
    f = 4.0 * B * H * T * T * d
    return f / 2 if causal else f


def floor_bytes(B, H, T, d):
    """Read Q, K, V once and write O (bf16) and LSE (fp32) once."""
    return 4 * B * H * T * d * 2 + B * H * T * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def library_fingerprint():
    """Hash of the library's sources and build flags (identifies the build a number was taken on)."""
    from exact_io_aware_07_gb300 import _build

    return _build._fingerprint(())[:16]


def forward_fingerprint():
    """Hash of the sources that make up the forward kernel and its launch (the backward kernels'
    source is left out), so that recorded ncu traffic of the forward kernel stays matched while
    only the backward changes."""
    import hashlib

    from exact_io_aware_07_gb300 import _build

    h = hashlib.sha256()
    for name in ("fa_kernel.cu", "fa_kernel.h", "ptx.cuh", "fa_api.cu"):
        with open(os.path.join(_build.CSRC, name), "rb") as f:
            h.update(f.read())
    h.update(" ".join(_build.ARCH + _build.CFLAGS).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, fingerprint):
    """DRAM bytes per launch from an ncu summary under profiles/, if taken on this forward-kernel build.

    Returns (bytes, file name) or (None, None).  The figure is dram__bytes_read.sum +
    dram__bytes_write.sum of one launch in a separate ncu capture of the same library build
    (the summary names the command); a bench run under ncu would not give a bench value.
    """
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, None
    pat = re.compile(rf"^traffic_bytes_per_launch\s+{re.escape(workload)}\s+(\d+)\s+fingerprint\s+(\w+)", re.M)
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(pdir, name)) as f:
            for m in pat.finditer(f.read()):
                if m.group(2) == fingerprint:
                    return int(m.group(1)), name
    return None, None


def input_sets(w):
    """Copies of the inputs the timed steps rotate over, so that their total exceeds 2 x L2."""
    set_bytes = floor_bytes(w["B"], w["H"], w["T"], w["d"])
    return max(1, math.ceil(2 * L2_BYTES / set_bytes)) if set_bytes < 2 * L2_BYTES else 1


def workload_config(name, w, world):
    """The `config` object both arms print for a workload."""
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    nsets = input_sets(w)
    return {"workload": name, "B": B, "H": H, "T": T, "d": d, "causal": bool(causal),
            "scale": 1.0 / math.sqrt(d), "qkv_dist": f"Q,K~N(0,{w['sigma_qk']}^2), V~N(0,1), bf16, seed 0",
            "l2": f"inputs rotate over {nsets} copies ({nsets * floor_bytes(B, H, T, d) / 1e6:.0f} MB > 2x L2)"
                  if nsets > 1 else f"one input set of {floor_bytes(B, H, T, d) / 1e6:.0f} MB, larger than 2x L2",
            "parallelism": f"replicas x{world}", "flops_per_step": metric_flops(B, H, T, d, causal)}


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons while the GPU works."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in use for k, v in enumerate(r[4]) if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": max(r[2] for r in use),
                "power_w_max": max(r[3] for r in use), "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")  # host-side barrier and timing reduction only
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x):
    if pg is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def device_inputs(qkv, torch, dev):
    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    return up(qkv.q_bits), up(qkv.k_bits), up(qkv.v_bits)


def time_kernel(fa, torch, dev, w, qkv, steps, warmup, scale, per_step_events=True):
    """Device-timed steps over rotating input copies; returns (total_s, per-launch mean s, nsets)."""
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    q0, k0, v0 = device_inputs(qkv, torch, dev)
    nsets = input_sets(w)
    sets = []
    for s in range(nsets):
        q, k, v = (q0, k0, v0) if s == 0 else (q0.clone(), k0.clone(), v0.clone())
        sets.append((q, k, v, torch.empty_like(q), torch.empty((B, H, T), dtype=torch.float32, device=dev)))
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        q, k, v, o, lse = sets[i % nsets]
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
        if per_step_events else []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    return sets, stream, ev, start, end, nsets


def run_ours(args, world, rank, local, pg):
    import torch

    import exact_io_aware_07_gb300 as fa

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.build()
    fa.load_library()
    name = args.workload
    w = fi.WORKLOADS[name]
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    peaks, peak_src = load_peaks()
    qkv = fi.make_qkv(B, H, T, d, seed=0, sigma_qk=w["sigma_qk"])
    K, W = args.steps, args.warmup
    if K is None:  # about a quarter of a second of timed work
        K = int(min(20000, max(20, 0.25 / max(metric_flops(B, H, T, d, causal) / 1.5e15, 1e-7))))
    # The timed region is K back-to-back calls bracketed by two events: kernels launched with
    # programmatic stream serialization overlap their set-up with the previous call's tail, which
    # an event recorded between calls would prevent.  The isolated launch time (events around each
    # call) is measured after the timed region, for context.
    per_step = False
    sets, stream, ev, start, end, nsets = time_kernel(fa, torch, dev, w, qkv, K, W, scale, per_step)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(K):
        q, k, v, o, lse = sets[i % nsets]
        if per_step:
            ev[i][0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        if per_step:
            ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(pg)
    clk = clocks.stop(t_wall0, t_wall1)
    total_s = start.elapsed_time(end) / 1e3
    launch_s = total_s / K  # the launch rate the timed region sustained
    iso_steps = min(K, 1000)
    iso = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iso_steps)]
    for i in range(iso_steps):
        q, k, v, o, lse = sets[i % nsets]
        iso[i][0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        iso[i][1].record(stream)
    torch.cuda.synchronize(dev)
    launch_iso_s = sum(a.elapsed_time(b) for a, b in iso) / 1e3 / iso_steps
    if fa.fa_device_status(stream) != 0:
        raise RuntimeError("a bounded in-kernel wait ran out during the timed region")
    total_s = max_over_ranks(pg, total_s)
    launch_s = max_over_ranks(pg, launch_s)

    f_step = metric_flops(B, H, T, d, causal)
    value = world * K * f_step / total_s / 1e12
    achieved = f_step / launch_s / 1e12
    fp = library_fingerprint()
    traffic, traffic_file = recorded_traffic(name, forward_fingerprint())
    roofline = {
        "bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
        "traffic_source": (f"recorded: a separate ncu capture of one launch of this forward-kernel build, reads "
                           f"and writes (dram__bytes_read.sum + dram__bytes_write.sum), profiles/{traffic_file}")
                          if traffic else
                          "no ncu capture of this forward-kernel build on record",
        "peak_source": f"{peak_src} bf16 burst", "kernel": "fa_fwd_kernel",
        "floor_bytes": floor_bytes(B, H, T, d),
        "attainable_tflops": round(min(peaks["bf16_tflops"],
                                       f_step / floor_bytes(B, H, T, d) * peaks["hbm_gbs"] / 1e3), 1),
        "hbm_floor_gbs": round(floor_bytes(B, H, T, d) / launch_s / 1e9, 1),
        "achieved_isolated_launch": round(f_step / launch_iso_s / 1e12, 2),
        "launch_us_isolated": round(launch_iso_s * 1e6, 2),
    }
    parity = None
    if rank == 0 and not args.no_parity:
        q, k, v, o, lse = sets[0]  # set 0 holds the seed-0 inputs themselves (the others are copies)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        parity = parity_sample(qkv, o, lse, w, scale, torch)
    # the exponential unit's ceiling: one ex2 per unmasked score against 4 d tensor FLOPs
    ex2_rate = fa.fa_ex2_rate(stream)
    roofline["ex2_per_s"] = float(f"{ex2_rate:.4g}")
    roofline["sfu_limited_tflops"] = round(ex2_rate * 4 * d / 1e12, 1)

    e2e = run_e2e(fa, torch, dev, w, qkv, scale, min(K, args.e2e_steps), pg) if not args.no_e2e else None
    if e2e is not None:
        e2e["value"] = round(world * e2e.pop("steps") * f_step / e2e.pop("seconds") / 1e12, 3)

    sweep = None
    if rank == 0 and world == 1 and not args.no_sweep:
        sweep = run_sweep(fa, torch, dev, [s for s in args.sweep.split(",") if s and s != name], peaks)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, qkv, scale, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(total_s / K * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(name, w, world),
        "pct_of_bf16_peak": round(100 * value / world / peaks["bf16_tflops"], 2),
        "roofline": roofline, "e2e": e2e, "gpu_launches": K, "clocks": clk, "cpu_baseline": cpu,
        "parity": parity, "library_fingerprint": fp, "forward_kernel_fingerprint": forward_fingerprint(),
    }
    if sweep is not None:
        line["sweep"] = sweep
    if rank == 0:
        print(json.dumps(line), flush=True)


def parity_sample(qkv, o, lse, w, scale, torch, per_head=64, seed=7):
    """O and LSE of one launch against the float64 oracle on sampled query rows of every head.

    Rows per head: the first and last 16 and 32 seeded-random ones (all rows when T <= 64).
    Tolerances: max |dO| <= 1e-2 (plus half a bf16 spacing where |O_ref| >= 4, where
    correct rounding alone can exceed 1e-2), mean |dO| <= 1e-3, max |dLSE| <= 1e-3.
    """
    import oracle

    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    torch.cuda.synchronize()
    o_bits = o.view(torch.int16).cpu().numpy().view(np.uint16)
    lse_h = lse.cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    q, k, v = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    o_err_max = o_err_sum = lse_err_max = 0.0
    n = wide = 0
    ok = True
    for b in range(B):
        for h in range(H):
            if T <= per_head:
                rows = np.arange(T)
            else:
                rows = np.unique(np.concatenate([np.arange(16), np.arange(T - 16, T),
                                                 rng.integers(0, T, size=per_head - 32)]))
            o_ref, l_ref = oracle.attention_head(q[b, h], k[b, h], v[b, h], causal, scale, rows=rows)
            o_gpu = fi.bf16_bits_to_f64(o_bits[b, h, rows])
            err = np.abs(o_gpu - o_ref)
            half_ulp = np.ldexp(1.0, np.frexp(np.where(np.abs(o_ref) > 0, np.abs(o_ref), 1.0))[1] - 9)
            tol = np.where(np.abs(o_ref) >= 4.0, 1e-2 + half_ulp, 1e-2)
            ok &= bool((err <= tol).all())
            wide += int((err > 1e-2).sum())
            o_err_max = max(o_err_max, float(err.max()))
            o_err_sum += float(err.sum())
            n += err.size
            lse_err_max = max(lse_err_max, float(np.abs(lse_h[b, h, rows] - l_ref).max()))
    mean = o_err_sum / n
    ok = ok and mean <= 1e-3 and lse_err_max <= 1e-3
    return {"o_max_abs": float(f"{o_err_max:.4g}"), "o_mean_abs": float(f"{mean:.4g}"),
            "lse_max_abs": float(f"{lse_err_max:.4g}"), "o_beyond_1e-2_where_abs_o_ge_4": wide,
            "pass": bool(ok), "rows_checked": n // d, "oracle_s": round(time.perf_counter() - t0, 1),
            "against": f"float64 oracle on {per_head} sampled query rows per head (first 16, last 16, "
                       f"seeded random), seed-0 inputs"}


def run_e2e(fa, torch, dev, w, qkv, scale, steps, pg):
    """Public API with pinned host buffers: H2D of Q, K, V and D2H of O, LSE inside every timed step.

    Consecutive steps alternate between two streams with their own device and host buffers, so one
    step's device-to-host read overlaps the next step's host-to-device copy (the two directions use
    separate copy engines); every step still moves all of its inputs in and its outputs out.
    """
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]

    def pinned(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()

    qh, kh, vh = pinned(qkv.q_bits), pinned(qkv.k_bits), pinned(qkv.v_bits)
    streams = [torch.cuda.current_stream(dev), torch.cuda.Stream(dev)]
    bufs = []
    for _ in range(2):
        bufs.append(dict(q=torch.empty(qh.shape, dtype=torch.bfloat16, device=dev),
                         k=torch.empty(qh.shape, dtype=torch.bfloat16, device=dev),
                         v=torch.empty(qh.shape, dtype=torch.bfloat16, device=dev),
                         oh=torch.empty_like(qh).pin_memory(),
                         lh=torch.empty((B, H, T), dtype=torch.float32).pin_memory()))

    def step(i):
        st, bf = streams[i % 2], bufs[i % 2]
        with torch.cuda.stream(st):
            bf["q"].copy_(qh, non_blocking=True)
            bf["k"].copy_(kh, non_blocking=True)
            bf["v"].copy_(vh, non_blocking=True)
            o, lse = fa.attention(bf["q"], bf["k"], bf["v"], causal=bool(causal), scale=scale, stream=st)
            bf["oh"].copy_(o, non_blocking=True)
            bf["lh"].copy_(lse, non_blocking=True)
            # the device outputs are freed only after this stream's read of them
            o.record_stream(st)
            lse.record_stream(st)

    for i in range(4):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(pg)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(streams[0])
    streams[1].wait_event(a)
    for i in range(steps):
        step(i)
    joined = torch.cuda.Event()
    joined.record(streams[1])
    streams[0].wait_event(joined)
    b.record(streams[0])
    torch.cuda.synchronize(dev)
    barrier(pg)
    sec = max_over_ranks(pg, a.elapsed_time(b) / 1e3)
    return {"unit": "TFLOPS", "steps": steps, "seconds": sec,
            "h2d_bytes_per_step": 3 * qh.numel() * 2,
            "d2h_bytes_per_step": bufs[0]["oh"].numel() * 2 + bufs[0]["lh"].numel() * 4,
            "path": "exact_io_aware_07_gb300.attention() with pinned host buffers, steps alternating on two streams"}


def time_splitkv(fa, torch, dev, g, steps):
    """Device time per call of fa_fwd and of fa_fwd_splitkv (automatic split count), calls alternating."""
    B, H, T, d, causal = g["B"], g["H"], g["T"], g["d"], g["causal"]
    x = fi.make_qkv(B, H, T, d, seed=0)
    q, k, v = device_inputs(x, torch, dev)
    o, lse = torch.empty_like(q), torch.empty((B, H, T), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, 0), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream(dev)
    runs = {"unsplit": lambda: fa.fa_fwd(q, k, v, o, lse, causal, scale, stream),
            "split": lambda: fa.fa_fwd_splitkv(q, k, v, o, lse, causal, scale, 0, ws, stream)}
    for _ in range(5):
        for r in runs.values():
            r()
    torch.cuda.synchronize(dev)
    ev = {n: [] for n in runs}
    for i in range(steps):
        for n, r in runs.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            r()
            b.record(stream)
            ev[n].append((a, b))
    torch.cuda.synchronize(dev)
    if fa.fa_device_status(stream) != 0:
        raise RuntimeError("a bounded in-kernel wait ran out in the split-KV sweep")
    return {n: sorted(a.elapsed_time(b) for a, b in e)[len(e) // 2] / 1e3 for n, e in ev.items()}, ws.numel()


def time_gqa(fa, torch, dev, g, steps):
    """Device time of fa_fwd_gqa per step (inputs rotating past L2)."""
    B, H, Hkv, T, d, causal = g["B"], g["H"], g["Hkv"], g["T"], g["d"], g["causal"]
    x = fi.make_grouped_qkv(B, H, Hkv, T, d, seed=0)

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    q0, k0, v0 = up(x.q_bits), up(x.k_bits), up(x.v_bits)
    set_bytes = (2 * q0.numel() + 2 * k0.numel()) * 2
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    sets = [(q0, k0, v0) if s == 0 else (q0.clone(), k0.clone(), v0.clone()) for s in range(nsets)]
    sets = [(q, k, v, torch.empty_like(q), torch.empty((B, H, T), dtype=torch.float32, device=dev))
            for q, k, v in sets]
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(d)
    for i in range(5):
        fa.fa_fwd_gqa(*sets[i % nsets], causal, scale, stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fa.fa_fwd_gqa(*sets[i % nsets], causal, scale, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in ev]
    return sum(ms) / len(ms) / 1e3


# backward pass: FLOPs counted as 2.5x the forward's (dV, dP, dQ, dK and the recomputed S; the
# kernels also recompute dP and S once more, which is not counted)
BWD_SWEEP = ["gpt2s_causal_b8h12t1024d64", "llama8b_causal_b1h32t4096d128", "llama8b_b1h32t4096d128"]


def time_bwd(fa, torch, dev, w, steps):
    """Device time of fa_bwd (both kernels) per step, inputs rotating past L2."""
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    qkv = fi.make_qkv(B, H, T, d, seed=0, sigma_qk=w["sigma_qk"])
    q0, k0, v0 = device_inputs(qkv, torch, dev)
    do0 = torch.from_numpy(fi.make_grad_out(B, H, T, d, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    scale = 1.0 / math.sqrt(d)
    set_bytes = 9 * q0.numel() * 2
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    sets = []
    for s in range(nsets):
        q, k, v, do = (x if s == 0 else x.clone() for x in (q0, k0, v0, do0))
        o, lse = fa.attention(q, k, v, causal=causal, scale=scale)
        sets.append((q, k, v, o, lse, do, torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, T), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(5):
        fa.fa_bwd(*sets[i % nsets], causal, scale, ws, stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fa.fa_bwd(*sets[i % nsets], causal, scale, ws, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if fa.fa_device_status(stream) != 0:
        raise RuntimeError("a bounded in-kernel wait ran out in the backward pass")
    ms = [a.elapsed_time(b) for a, b in ev]
    return sum(ms) / len(ms) / 1e3


# e4m3 forward (d = 128): the contraction runs at the fp8 rate, so its roofline peak is the measured
# bf16 peak times the nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
FP8_SWEEP = ["llama8b_causal_b1h32t4096d128", "llama8b_b1h32t4096d128"]
FP8_OVER_BF16 = 2.0


def time_fp8(fa, torch, dev, w, steps):
    """Device time of fa_fwd_fp8 (V transpose + attention) per step, inputs rotating past L2."""
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    x = fi.make_qkv_e4m3(B, H, T, d, seed=0)
    q0, k0, v0 = (torch.from_numpy(np.ascontiguousarray(getattr(x, n + "8"))).to(dev) for n in "qkv")
    set_bytes = 3 * q0.numel() + 2 * q0.numel() * 2
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    sets = []
    for s in range(nsets):
        q, k, v = (t if s == 0 else t.clone() for t in (q0, k0, v0))
        sets.append((q, k, v, torch.empty(B, H, T, d, dtype=torch.bfloat16, device=dev),
                     torch.empty(B, H, T, dtype=torch.float32, device=dev)))
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, T, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(d)
    for i in range(5):
        fa.fa_fwd_fp8(*sets[i % nsets], causal, scale, x.descale, ws, stream)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        fa.fa_fwd_fp8(*sets[i % nsets], causal, scale, x.descale, ws, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in ev]
    return sum(ms) / len(ms) / 1e3


def run_sweep(fa, torch, dev, names, peaks, splitkv=SPLITKV_SWEEP, gqa=GQA_SWEEP, bwd=BWD_SWEEP, fp8=FP8_SWEEP):
    """Every other workload, measured the same way with fewer steps (informational)."""
    out = {}
    for name in fp8:
        w = fi.WORKLOADS[name]
        f = metric_flops(w["B"], w["H"], w["T"], w["d"], w["causal"])
        steps = int(min(2000, max(20, 0.5 / max(f / 2.0e15, 1e-6))))
        sec = time_fp8(fa, torch, dev, w, steps)
        peak8 = FP8_OVER_BF16 * peaks["bf16_tflops"]
        out[f"fp8_{name}"] = {"ms_mean": round(sec * 1e3, 4), "tflops": round(f / sec / 1e12, 1),
                              "pct_of_fp8_peak": round(100 * f / sec / 1e12 / peak8, 1),
                              "fp8_peak_tflops": round(peak8, 1), "steps": steps,
                              "kernels": "fa_transpose_e4m3_kernel + fa_fwd_kernel (e4m3)"}
        torch.cuda.empty_cache()
    for name in bwd:
        w = fi.WORKLOADS[name]
        f = 2.5 * metric_flops(w["B"], w["H"], w["T"], w["d"], w["causal"])
        steps = int(min(1000, max(20, 0.5 / max(f / 0.6e15, 1e-6))))
        sec = time_bwd(fa, torch, dev, w, steps)
        out[f"backward_{name}"] = {"ms_mean": round(sec * 1e3, 4), "tflops": round(f / sec / 1e12, 1),
                                   "pct_of_bf16_peak": round(100 * f / sec / 1e12 / peaks["bf16_tflops"], 1),
                                   "steps": steps, "flops": "2.5 x forward",
                                   "kernels": "fa_bwd_kernel (dQ, with the row vectors) + fa_bwd_kernel (dK, dV)"}
        torch.cuda.empty_cache()
    for name, g in gqa.items():
        f = metric_flops(g["B"], g["H"], g["T"], g["d"], g["causal"])
        steps = int(min(2000, max(20, 0.5 / max(f / 1.0e15, 1e-6))))
        sec = time_gqa(fa, torch, dev, g, steps)
        out[name] = {"ms_mean": round(sec * 1e3, 4), "tflops": round(f / sec / 1e12, 1),
                     "pct_of_bf16_peak": round(100 * f / sec / 1e12 / peaks["bf16_tflops"], 1),
                     "steps": steps, "kernels": "fa_fwd_kernel (grouped K/V heads)"}
        torch.cuda.empty_cache()
    for name, g in splitkv.items():
        f = metric_flops(g["B"], g["H"], g["T"], g["d"], g["causal"])
        steps = int(min(1000, max(20, 0.3 / max(f / 1.0e15, 1e-6))))
        sec, ws_bytes = time_splitkv(fa, torch, dev, g, steps)
        out[name] = {"ms_median_split": round(sec["split"] * 1e3, 4), "ms_median_unsplit": round(sec["unsplit"] * 1e3, 4),
                     "tflops_split": round(f / sec["split"] / 1e12, 1),
                     "tflops_unsplit": round(f / sec["unsplit"] / 1e12, 1),
                     "speedup": round(sec["unsplit"] / sec["split"], 3), "steps": steps, "workspace_bytes": ws_bytes,
                     "num_splits": "chosen by the library (0)",
                     "key_ranges_used": fa.fa_fwd_splitkv_count(g["B"], g["H"], g["T"], g["d"], g["causal"], 0),
                     "kernels": "fa_fwd_kernel (partial, last split of each 32-row group merges) vs fa_fwd_kernel"}
        torch.cuda.empty_cache()
    for name in names:
        w = fi.WORKLOADS[name]
        B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
        scale = 1.0 / math.sqrt(d)
        qkv = fi.make_qkv(B, H, T, d, seed=0, sigma_qk=w["sigma_qk"])
        f = metric_flops(B, H, T, d, causal)
        steps = int(min(2000, max(20, 0.5 / max(f / 1.0e15, 1e-6))))
        sets, stream, ev, start, end, nsets = time_kernel(fa, torch, dev, w, qkv, steps, 5, scale, True)
        for i in range(steps):
            q, k, v, o, lse = sets[i % nsets]
            ev[i][0].record(stream)
            fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        mean_s = sum(ms) / len(ms) / 1e3
        out[name] = {"ms_mean": round(mean_s * 1e3, 4), "ms_median": round(ms[len(ms) // 2], 4),
                     "tflops": round(f / mean_s / 1e12, 1),
                     "pct_of_bf16_peak": round(100 * f / mean_s / 1e12 / peaks["bf16_tflops"], 1),
                     "steps": steps}
        del sets
        torch.cuda.empty_cache()
    return out


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info

        n = max((i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"), default=0)
        if n:
            return n
    except ImportError:
        pass
    return os.cpu_count() or 1


def spread_rows(T, count, offset):
    """`count` query rows spread evenly over [0, T), shifted by `offset`: a causal row's cost grows
    with its index, so evenly spread rows cost what the average row of the workload costs."""
    count = max(1, min(T, count))
    stride = T / count
    return np.unique((offset % max(1, int(stride)) + np.floor(np.arange(count) * stride)).astype(np.int64) % T)


def cpu_baseline(w, qkv, scale, seconds):
    """The float64 oracle, as it stands, on heads of the same input until ~`seconds` of CPU work."""
    import oracle

    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    q, k, v = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    rows_per_block = min(T, 256)
    heads = [(b, h) for b in range(B) for h in range(H)]
    done_rows = 0
    t0 = time.perf_counter()
    it = 0
    while True:
        b, h = heads[it % len(heads)]
        rows = spread_rows(T, rows_per_block, it // len(heads))
        oracle.attention_head(q[b, h], k[b, h], v[b, h], causal, scale, rows=rows)
        done_rows += len(rows)
        it += 1
        if time.perf_counter() - t0 >= seconds or done_rows >= 4 * B * H * T:
            break
    dt = time.perf_counter() - t0
    f = metric_flops(1, 1, T, d, causal) / T * done_rows  # metric FLOPs of the rows evaluated
    return {"value": round(f / dt / 1e12, 6), "unit": "TFLOPS", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{done_rows} query rows ({done_rows / (B * H * T):.4f} of the workload) in blocks of "
                      f"{rows_per_block} rows spread evenly over T, {dt:.1f} s, float64 numpy; the metric's FLOPs "
                      f"of those rows over the time"}


def run_reference(args, world, rank):
    """The CPU oracle timed per step on a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return
    import oracle

    name = args.workload
    w = fi.WORKLOADS[name]
    B, H, T, d, causal = w["B"], w["H"], w["T"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    qkv = fi.make_qkv(B, H, T, d, seed=0, sigma_qk=w["sigma_qk"])
    q, k, v = qkv.f64("q"), qkv.f64("k"), qkv.f64("v")
    K = args.steps if args.steps is not None else 20
    W = args.warmup
    # rows per step so that the whole run stays within about `budget` seconds
    t0 = time.perf_counter()
    probe = spread_rows(T, 64, 0)
    oracle.attention_head(q[0, 0], k[0, 0], v[0, 0], causal, scale, rows=probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    rows = int(max(1, min(T, args.reference_budget / max(K + W, 1) / max(per_row, 1e-9))))
    heads = [(b, h) for b in range(B) for h in range(H)]

    def step(i):
        b, h = heads[i % len(heads)]
        rr = spread_rows(T, rows, i // len(heads))
        oracle.attention_head(q[b, h], k[b, h], v[b, h], causal, scale, rows=rr)
        return len(rr)

    for i in range(W):
        step(i)
    t0 = time.perf_counter()
    n_rows = sum(step(W + i) for i in range(K))
    dt = time.perf_counter() - t0
    f = metric_flops(1, 1, T, d, causal) / T * n_rows
    value = f / dt / 1e12
    sample = (f"{rows} query rows of one head per step, spread evenly over T ({n_rows} rows in {K} steps), "
              f"float64 numpy; the metric's FLOPs of those rows over the time")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(dt / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name, w, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 0.25 s of work)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fi.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep", default=",".join(SWEEP_DEFAULT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-budget", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local, pg = dist_setup()
    if args.gpus != world and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark: state-passing conv + scan forward of Mamba-2-like mixer layers on
GB300, tokens/s, with the roofline of the dominant kernel.

A step (the headline) is one forward of the 1.3B-like layer with a random
Gaussian initial state: batch 4, L = 8192, d_inner 4096 (H = 64, P = 64),
N = 128, K = 4, bf16 x / dt / B / C, fp32 h0 ~ N(0, 0.1^2) and a conv state
~ N(0, 1); outputs y and the final conv and SSM states.  It is one
sss_mixer_fwd call (conv + SiLU + chunked scan in one tcgen05 kernel).  Inputs
are resident in HBM when the timed region starts; L2 is flushed (a 256 MiB
write) before every timed step, outside the events.  The same JSON line
carries every other workload as an extra key, each with its own roofline: the
370M-like layer as two 1024-token segments with state passing (and the same
forward as two calls), the 780M-like layer streamed over 64 x 2048-token
segments, the continuous-batching decode update at L_new = 1 and 4, the tiny
fp32 check, and the backward and state-utility kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
work shards by batch with no exchange); ``value`` is the tokens of all ranks
divided by the slowest rank's time.  ``--impl reference`` times the float64
CPU oracle on this machine's host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "m1p3b_8k"
METRIC = "tokens/s per GB300 (conv+scan fwd w/ state passing) and % of HBM/tensor roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


MODEL_LIKE = {"m370m_2k": "370M", "m1p3b_8k": "1.3B", "m780m_128k": "780M"}


def workload_desc(s) -> str:
    if s.name == "tiny_f32":
        return (f"{s.name}: batch {s.Bz}, L={s.L} as {len(s.segments)}x{s.segments[0]}-token "
                f"segments with state passed, H={s.H}, P={s.P}, N={s.N}, K={s.K}, fp32")
    like = MODEL_LIKE.get(s.name, "")
    init = ("Gaussian initial states (h0 ~ N(0,0.1^2), conv state ~ N(0,1))" if s.gaussian_init
            else "zero initial states")
    segs = (f"one {s.L}-token call" if len(s.segments) == 1 else
            f"{len(s.segments)}x{s.segments[0]}-token segments with conv and SSM state passed")
    return (f"{s.name}: Mamba-2 {like}-like mixer layer, batch {s.Bz}, L={s.L} as {segs}, "
            f"H={s.H}, P={s.P}, N={s.N}, K={s.K}, bf16 x/dt/B/C, fp32 state, {init}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak() -> float:
    """Measured dense bf16 TFLOP/s (burst), else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def kernel_source_hash(kernel: str) -> str:
    """sha256 (first 16 hex digits) of the kernel's .cu file followed by every
    local header it includes, directly or through another header, in the
    order first met."""
    import hashlib
    import re
    d = os.path.join(ROOT, "selective_ssm_scan_gb300", "csrc")
    order, todo = [], [f"{kernel}.cu"]
    while todo:
        fn = todo.pop(0)
        if fn in order:
            continue
        order.append(fn)
        with open(os.path.join(d, fn)) as f:
            todo += [m for m in re.findall(r'^#include "([^"]+)"', f.read(), re.M)
                     if os.path.exists(os.path.join(d, m))]
    h = hashlib.sha256()
    for fn in order:
        with open(os.path.join(d, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary of the kernel on
    this workload, if it covers the current build of the kernel (the summary
    states the source hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    import hashlib
    src = None
    val = None
    for line in text.splitlines():
        if line.startswith("source_sha256:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            val = int(float(line.split(":", 1)[1].strip()))
    try:
        cur = kernel_source_hash(kernel)
    except OSError:
        return None
    if src != cur:
        return None
    return val


class Clocks:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.out = out
        else:
            self.out = ""

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(dist, value: float, device) -> float:
    """The slowest rank's value (the job finishes when its last rank does);
    the value itself on one process."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, tokens_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own tokens_per_step each
    step (weak scaling), the job takes the slowest rank's time."""
    return world * tokens_per_step * steps / (total_ms * 1e-3)


def cpu_step_sample(s, nthreads: int = 0, rows: int = 0):
    """The oracle on one step of the workload (or its first ``rows`` batch
    rows, all tokens and heads): conv + scan over every segment with the
    states passed."""
    import oracle
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    rows = slice(0, rows or s.Bz)
    segs = [synth.mixer_segment(s, i, Bz=rows) for i in range(len(s.segments))]
    S = st["conv_state"].f64()[rows]
    h = st["h0"].f64()[rows]
    t0 = time.perf_counter()
    for sg in segs:
        _, S, h = oracle.mixer_fwd(sg["x"], sg["dt"], p["A"], sg["B"], sg["C"], p["w"],
                                   p["bias"], S, h, nthreads=nthreads)
    dt = time.perf_counter() - t0
    tokens = sum(s.segments) * (rows.stop - rows.start)
    return tokens / dt, dt, tokens, oracle.num_threads(nthreads)


# the oracle's sample of a step: one batch row, all its tokens and heads
CPU_SAMPLE_ROWS = 1


def run_reference(args, s):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        cpu_step_sample(s, rows=CPU_SAMPLE_ROWS)
    times = []
    tokens = 0
    cores = None
    for _ in range(args.steps):
        _, dt, tokens, cores = cpu_step_sample(s, rows=CPU_SAMPLE_ROWS)
        times.append(dt)
    total = sum(times)
    value = tokens * len(times) / total
    sample = (f"per step, batch row 0 of {s.name} ({tokens} tokens: {len(s.segments)} "
              f"segment(s) of {s.segments[0]}, all {s.H} heads, states passed)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(s), "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def algorithmic_bytes(s, Lseg: int, x_bytes: int = 2, y_bytes: int = 2) -> int:
    """The method's own HBM traffic for one call over an Lseg-token segment of
    workload s, conv + scan fused (x read once, u never written): x in, y
    out, dt, B and C in, h0 in and hT out, the conv state in and out."""
    a_bytes = 2 if s.dtype == "bf16" else 4
    return (s.Bz * Lseg * s.D * (x_bytes + y_bytes)
            + s.Bz * Lseg * (s.H + 2 * s.G * s.N) * a_bytes
            + 2 * s.Bz * s.H * s.P * s.N * 4
            + 2 * s.Bz * s.D * (s.K - 1) * a_bytes)


def events_timed(torch, stream, flush, fn, steps, sleep_ns=200_000):
    """Per-call device time (ms) of fn() on `stream`, CUDA events on that
    stream, L2 flushed before every call outside the events; the GPU is kept
    busy while the host enqueues the call, so no launch waits for the host."""
    evs = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(sleep_ns)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def roofline_block(byts, ms, hbm, hbm_kind, kernel, workload, traffic_key=None):
    achieved = byts / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm,
            "traffic": traffic_from_profile(*traffic_key) if traffic_key else None,
            "kernel": kernel, "workload": workload,
            "algorithmic_bytes_per_launch": byts, "avg_launch_ms": ms,
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if hbm_kind == "measured"
            else "fallback 6.8 TB/s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-context streaming line")
    ap.add_argument("--no-extra", action="store_true",
                    help="only the headline (no other workloads, backward or utilities)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    s = synth.WORKLOADS[WORKLOAD]
    if args.impl == "reference":
        run_reference(args, s)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import selective_ssm_scan_gb300 as sss

    def T(a):
        if a.dtype == "bf16":
            return torch.from_numpy(a.data.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a.data).to(dev)

    hbm, hbm_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # ---- the headline: one forward of the 1.3B-like layer ------------------
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    sg = {k: T(v) for k, v in synth.mixer_segment(s, 0).items()}
    A, w, bias = T(p["A"]), T(p["w"]), T(p["bias"])
    S0, h0 = T(st["conv_state"]), T(st["h0"])
    L = s.segments[0]
    y = torch.empty((s.Bz, L, s.H, s.P), dtype=torch.bfloat16, device=dev)
    F = torch.empty_like(S0)
    hT = torch.empty_like(h0)
    if not sss.mixer_fwd_supported(s.Bz, L, s.H, s.P, s.N, s.G, s.K, torch.bfloat16,
                                   torch.bfloat16):
        raise SystemExit("the fused forward does not support this workload")
    spans = sss.mixer_fwd_span_count(s.Bz, L, s.H, s.P, s.N, s.G, s.K, torch.bfloat16,
                                     torch.bfloat16)

    def step():
        sss.mixer_fwd(sg["x"], sg["dt"], A, sg["B"], sg["C"], w, bias, S0, h0,
                      conv_state_out=F, hT=hT, y=y, fused=True, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        step_ms = events_timed(torch, stream, flush, step, args.steps)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    assert sss.device_status() == 0, "device status after the headline steps"
    total_ms = max_over_ranks(dist, sum(step_ms), dev)
    tokens_per_step = s.Bz * L
    value = job_rate(world, tokens_per_step, args.steps, total_ms)
    launch_ms = statistics.mean(step_ms)
    fused_bytes = algorithmic_bytes(s, L)
    roofline = roofline_block(
        fused_bytes, launch_ms, hbm, hbm_kind,
        "ssm_scan_pair_kernel<bf16,bf16,fused> (conv+SiLU+chunked scan, two heads per CTA, "
        "one launch per call)", s.name, ("ssm_scan_pair", s.name))
    roofline["traffic_note"] = ("DRAM read + write bytes per launch from the committed ncu "
                                "summary when its source hash matches the current kernel")
    Q = 128
    tc_flops = s.Bz * s.H * (-(-L // Q)) * 2 * Q * (Q * s.N + Q * s.P + 2 * s.P * s.N)
    roofline["tensor_useful_tflops"] = tc_flops / (launch_ms * 1e-3) / 1e12
    # the same kernel against the tensor roofline: the MMAs it issues (per
    # 128-token piece and head pair 64 MMAs of 128x128x16 -- G 8, S' 16, Yo 16,
    # Yd 24, the hi/lo split terms included) over the launch time, against the
    # measured dense bf16 peak (burst: the kernel is timed alone)
    issued = (s.Bz * (s.H // 2)) * (-(-L // Q)) * 64 * 2 * 128 * 128 * 16
    bf16_peak = tensor_peak()
    roofline["tensor"] = {"issued_tflop_per_launch": issued / 1e12,
                          "achieved": issued / (launch_ms * 1e-3) / 1e12,
                          "peak": bf16_peak, "unit": "TFLOP/s",
                          "frac": issued / (launch_ms * 1e-3) / 1e12 / bf16_peak,
                          "useful_frac": tc_flops / (launch_ms * 1e-3) / 1e12 / bf16_peak,
                          "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, burst)"}

    # ---- end to end through the API with host buffers ----------------------
    e2e = bench_e2e(torch, sss, dev, flush, args, s, p, st, dist, world)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(s), "tokens_per_step": tokens_per_step,
                   "path": f"sss_mixer_fwd: one tcgen05 kernel per call (conv+SiLU+scan), two "
                           f"heads per CTA, spans per call {spans}",
                   "l2": "flushed before every timed step (256 MiB write, outside the events); "
                         "inputs 0.3 GB, larger than L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * (1 if spans <= 1 else 4),
        "clocks": clk.summary(),
    }
    if not args.no_extra:
        seg2 = bench_segments(torch, sss, dev, stream, flush, args, hbm, hbm_kind, T)
        out["m370m_2k"] = seg2
        s2 = synth.WORKLOADS["m370m_2k"]
        out["conv_bwd"] = bench_conv_bwd(torch, sss, dev, stream, flush, args, hbm, s2,
                                         s2.segments[0])
        out["scan_bwd"] = bench_scan_bwd(torch, sss, dev, stream, flush, args, hbm, s2,
                                         s2.segments[0])
        out["train_utils"] = bench_train_utils(torch, sss, dev, stream, flush, args, hbm, s2,
                                               s2.segments[0])
        out["tiny_f32"] = bench_tiny(torch, sss, dev, stream, flush, args, hbm, hbm_kind, T)
        out["mamba2_wiring"] = bench_mamba2(torch, sss, dev, stream, flush, args, hbm, s2)
        if not args.no_long:
            out["long_context"] = bench_long_context(torch, sss, dev, stream, flush, args, hbm,
                                                     hbm_kind)
        if not args.no_decode:
            out["decode_256x1"] = bench_decode(torch, sss, dev, stream, flush, args, hbm,
                                               "decode_256x1")
            out["decode_256x4"] = bench_decode(torch, sss, dev, stream, flush, args, hbm,
                                               "decode_256x4")
    if rank == 0 and not args.no_cpu_baseline:
        # whole rows of the step repeated until about 10 s of oracle time has run
        total_t, total_tok, reps, cores = 0.0, 0, 0, None
        while total_t < 10.0 and reps < 200:
            _, dt_, tokens, cores = cpu_step_sample(s, rows=CPU_SAMPLE_ROWS)
            total_t += dt_
            total_tok += tokens
            reps += 1
        out["cpu_baseline"] = {"value": total_tok / total_t, "unit": UNIT, "cores": cores,
                               "kind": "oracle",
                               "sample": f"{reps} repetitions of batch row 0 of {s.name} "
                                         f"({tokens} tokens each, all {s.H} heads, Gaussian "
                                         f"initial states), {total_t:.1f} s wall"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def gpu_local_cpus(torch, dev):
    """The CPUs of the GPU's own NUMA node (the sysfs local_cpulist of its PCI
    function) that this process may run on, or None when that is unknown."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        addr = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        with open(f"/sys/bus/pci/devices/{addr}/local_cpulist") as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except (OSError, ValueError, AttributeError):
        return None


def bench_e2e(torch, sss, dev, flush, args, s, p, st, dist, world):
    """The headline step end to end through the public API: every step copies
    its inputs from pinned host memory to the device and y plus the final
    states back.  The batch rows run as separate calls on four streams, so one
    row's copies overlap another row's kernel."""
    L = s.segments[0]
    seg = synth.mixer_segment(s, 0)
    bf = torch.bfloat16

    def pinned(a):
        if a.dtype == "bf16":
            t = torch.from_numpy(a.data.view(np.int16)).view(bf)
        else:
            t = torch.from_numpy(a.data)
        return torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)

    # the pinned buffers are allocated and first touched from the GPU's own
    # NUMA node, so the copies do not cross between host memory nodes
    local = gpu_local_cpus(torch, dev)
    saved = os.sched_getaffinity(0)
    if local:
        os.sched_setaffinity(0, local)
    try:
        host = {k: pinned(v) for k, v in seg.items()}
        hS0, hh0 = pinned(st["conv_state"]), pinned(st["h0"])
        hy = torch.empty((s.Bz, L, s.H, s.P), dtype=bf, pin_memory=True)
        hF = torch.empty(hS0.shape, dtype=hS0.dtype, pin_memory=True)
        hhT = torch.empty(hh0.shape, dtype=hh0.dtype, pin_memory=True)
        hy.zero_()
        hF.zero_()
        hhT.zero_()
    finally:
        os.sched_setaffinity(0, saved)
    A = torch.from_numpy(p["A"].data).to(dev)
    w = torch.from_numpy(p["w"].data).to(dev)
    bias = torch.from_numpy(p["bias"].data).to(dev)
    dev_in = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host.items()}
    dS0 = torch.empty(hS0.shape, dtype=hS0.dtype, device=dev)
    dh0 = torch.empty(hh0.shape, dtype=hh0.dtype, device=dev)
    dy = torch.empty(hy.shape, dtype=bf, device=dev)
    dF = torch.empty(hF.shape, dtype=hF.dtype, device=dev)
    dhT = torch.empty(hhT.shape, dtype=hhT.dtype, device=dev)
    nstreams = min(4, s.Bz)
    streams = [torch.cuda.Stream(device=dev) for _ in range(nstreams)]
    main = torch.cuda.current_stream()
    rows = [list(range(i, s.Bz, nstreams)) for i in range(nstreams)]

    def e2e_step(e0):
        for sti, rr in zip(streams, rows):
            sti.wait_event(e0)
            with torch.cuda.stream(sti):
                for b in rr:
                    for k in dev_in:
                        dev_in[k][b].copy_(host[k][b], non_blocking=True)
                    dS0[b].copy_(hS0[b], non_blocking=True)
                    dh0[b].copy_(hh0[b], non_blocking=True)
                    sl = slice(b, b + 1)
                    sss.mixer_fwd(dev_in["x"][sl], dev_in["dt"][sl], A, dev_in["B"][sl],
                                  dev_in["C"][sl], w, bias, dS0[sl], dh0[sl],
                                  conv_state_out=dF[sl], hT=dhT[sl], y=dy[sl], fused=True,
                                  stream=sti)
                    hy[b].copy_(dy[b], non_blocking=True)
                    hF[b].copy_(dF[b], non_blocking=True)
                    hhT[b].copy_(dhT[b], non_blocking=True)
        for sti in streams:
            main.wait_stream(sti)

    for _ in range(3):
        e0 = torch.cuda.Event()
        e0.record(main)
        e2e_step(e0)
    torch.cuda.synchronize()
    ms = []
    e2e_steps = max(3, args.steps // 10)
    for _ in range(e2e_steps):
        flush.zero_()
        torch.cuda._sleep(200_000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        e2e_step(e0)
        e1.record(main)
        main.synchronize()
        ms.append(e0.elapsed_time(e1))
    total = max_over_ranks(dist, sum(ms), dev)
    h2d = (sum(t.numel() * t.element_size() for t in host.values())
           + hS0.numel() * hS0.element_size() + hh0.numel() * hh0.element_size())
    d2h = (hy.numel() * hy.element_size() + hF.numel() * hF.element_size()
           + hhT.numel() * hhT.element_size())
    return {"value": job_rate(world, s.Bz * L, e2e_steps, total), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": total / e2e_steps,
            "path": f"sss_mixer_fwd per batch row on {nstreams} streams, pinned host buffers, "
                    "copies in and out inside the timed region",
            "host_buffers": ("allocated from the GPU's NUMA node (CPUs %d-%d)" % (min(local), max(local))
                             if local else "allocated without a NUMA binding (node unknown)")}


def bench_segments(torch, sss, dev, stream, flush, args, hbm, hbm_kind, T):
    """The 370M-like layer: batch 8, L = 2048 as two 1024-token segments with
    conv and SSM state passed (one sss_mixer_fwd per segment), and the same
    forward as two calls per segment (conv with u in fp32, then the scan)."""
    s = synth.WORKLOADS["m370m_2k"]
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    segs = [{k: T(v) for k, v in synth.mixer_segment(s, i).items()} for i in range(len(s.segments))]
    A, w, bias = T(p["A"]), T(p["w"]), T(p["bias"])
    S0, h00 = T(st["conv_state"]), T(st["h0"])
    S = torch.empty_like(S0)
    h = torch.empty_like(h00)
    Lseg = s.segments[0]
    us = [torch.empty((s.Bz, L, s.D), dtype=torch.float32, device=dev) for L in s.segments]
    ys = [torch.empty((s.Bz, L, s.H, s.P), dtype=torch.bfloat16, device=dev) for L in s.segments]
    n_seg = len(segs)

    def run(evs, two_call):
        for i, sg in enumerate(segs):
            evs[i].record(stream)
            if two_call:
                sss.conv_state_fwd(sg["x"], w, bias, S, S, u=us[i], stream=stream)
                evs[n_seg + 1 + i].record(stream)
                sss.ssm_scan_fwd(us[i], sg["dt"], A, sg["B"], sg["C"], h, h, y=ys[i],
                                 stream=stream)
            else:
                sss.mixer_fwd(sg["x"], sg["dt"], A, sg["B"], sg["C"], w, bias, S, h,
                              conv_state_out=S, hT=h, y=ys[i], fused=True, spans=1,
                              stream=stream)
        evs[n_seg].record(stream)

    def timed(two_call, steps):
        all_evs = []
        for _ in range(steps):
            S.copy_(S0)
            h.copy_(h00)
            flush.zero_()
            torch.cuda._sleep(200_000)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_seg + 1)]
            run(evs, two_call)
            all_evs.append(evs)
        stream.synchronize()
        return all_evs

    for _ in range(args.warmup):
        S.copy_(S0)
        h.copy_(h00)
        run([torch.cuda.Event() for _ in range(2 * n_seg + 1)], False)
        S.copy_(S0)
        h.copy_(h00)
        run([torch.cuda.Event() for _ in range(2 * n_seg + 1)], True)
    torch.cuda.synchronize()
    ev1 = timed(False, max(3, args.steps // 2))
    seg_ms = [e[i].elapsed_time(e[i + 1]) for e in ev1 for i in range(n_seg)]
    step_ms = statistics.mean(e[0].elapsed_time(e[n_seg]) for e in ev1)
    ev2 = timed(True, max(3, args.steps // 4))
    conv_ms = statistics.mean(e[i].elapsed_time(e[n_seg + 1 + i]) for e in ev2 for i in range(n_seg))
    scan_ms = statistics.mean(e[n_seg + 1 + i].elapsed_time(e[i + 1] if i + 1 < n_seg else e[n_seg])
                              for e in ev2 for i in range(n_seg))
    two_ms = statistics.mean(e[0].elapsed_time(e[n_seg]) for e in ev2)
    assert sss.device_status() == 0
    fused_bytes = algorithmic_bytes(s, Lseg)
    io = (s.Bz * Lseg * s.H * 2 + 2 * s.Bz * Lseg * s.G * s.N * 2 + s.Bz * Lseg * s.D * 2
          + 2 * s.Bz * s.H * s.P * s.N * 4)
    scan_bytes = s.Bz * Lseg * s.D * 4 + io
    conv_bytes = s.Bz * Lseg * s.D * (2 + 4) + 2 * s.Bz * s.D * (s.K - 1) * 2
    return {"workload": workload_desc(s), "tokens_per_s": s.Bz * s.L / (step_ms * 1e-3),
            "ms_per_step": step_ms,
            "roofline": roofline_block(fused_bytes, statistics.mean(seg_ms), hbm, hbm_kind,
                                       "ssm_scan_pair_kernel<bf16,bf16,fused>", s.name,
                                       ("ssm_scan_pair", s.name)),
            "two_call_path": {
                "ms_per_step": two_ms,
                "conv_state_fwd": {"avg_launch_ms": conv_ms,
                                   "algorithmic_bytes_per_launch": conv_bytes,
                                   "achieved_gbs": conv_bytes / conv_ms / 1e6,
                                   "frac": conv_bytes / conv_ms / 1e6 / hbm},
                "ssm_scan_fwd": {"avg_launch_ms": scan_ms,
                                 "algorithmic_bytes_per_launch": scan_bytes,
                                 "achieved_gbs": scan_bytes / scan_ms / 1e6,
                                 "frac": scan_bytes / scan_ms / 1e6 / hbm}}}


def bench_tiny(torch, sss, dev, stream, flush, args, hbm, hbm_kind, T):
    """The tiny fp32 check (batch 1, L = 64 as two 32-token segments, H = 2,
    P = 4, N = 8): one sss_mixer_fwd per segment on the fp32 path.  Far too
    small to fill the GPU; its time is launch latency."""
    s = synth.WORKLOADS["tiny_f32"]
    p = synth.mixer_params(s)
    st = synth.mixer_initial_states(s)
    segs = [{k: T(v) for k, v in synth.mixer_segment(s, i).items()} for i in range(len(s.segments))]
    A, w, bias = T(p["A"]), T(p["w"]), T(p["bias"])
    S = T(st["conv_state"])
    h = T(st["h0"])
    ys = [torch.empty((s.Bz, L, s.H, s.P), dtype=torch.float32, device=dev) for L in s.segments]

    def call():
        for i, sg in enumerate(segs):
            sss.mixer_fwd(sg["x"], sg["dt"], A, sg["B"], sg["C"], w, bias, S, h,
                          conv_state_out=S, hT=h, y=ys[i], stream=stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ms = statistics.mean(events_timed(torch, stream, flush, call, max(3, args.steps // 10),
                                      sleep_ns=50_000))
    byts = sum(algorithmic_bytes(s, L, 4, 4) for L in s.segments)
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": workload_desc(s), "ms_per_step": ms,
            "tokens_per_s": s.Bz * s.L / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "algorithmic_bytes_per_step": byts,
                         "avg_step_ms": ms, "traffic": None,
                         "kernel": "fp32 path (conv, CUDA-core scan) per segment; far too small "
                                   "to fill the GPU, its time is launch latency"}}


def bench_conv_bwd(torch, sss, dev, stream, flush, args, hbm, s, Lseg):
    """sss_conv_state_bwd on one segment of the workload: bf16 x and state,
    fp32 dy and dF, bf16 dx and dS, fp32 dw and dbias (two kernels: the
    gradient pass and the fixed-order reduction of the weight partials)."""
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    bf = torch.bfloat16
    Bz, D, K = s.Bz, s.D, s.K
    x = torch.randn((Bz, Lseg, D), generator=g, device=dev).to(bf)
    S = torch.randn((Bz, D, K - 1), generator=g, device=dev).to(bf)
    dy = torch.randn((Bz, Lseg, D), generator=g, device=dev)
    q = torch.randn((Bz, D, K - 1), generator=g, device=dev)
    w = torch.randn((D, K), generator=g, device=dev) * (0.5 ** 0.5)
    bias = torch.full((D,), 0.1, device=dev)
    dx = torch.empty((Bz, Lseg, D), dtype=bf, device=dev)
    dS = torch.empty((Bz, D, K - 1), dtype=bf, device=dev)
    dw = torch.empty((D, K), device=dev)
    db = torch.empty((D,), device=dev)
    ws = torch.empty(max(1, sss.conv_state_bwd_workspace_size(Bz, Lseg, D, K)),
                     dtype=torch.uint8, device=dev)

    def call():
        sss.conv_state_bwd(x, w, bias, S, dy, q, dx, dS, dw, db, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    evs = []
    for _ in range(max(3, args.steps // 10)):
        flush.zero_()
        torch.cuda._sleep(200_000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
    stream.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    n_el = Bz * Lseg * D
    byts = (n_el * (2 + 4 + 2)                       # x, dy in; dx out
            + Bz * D * (K - 1) * (2 + 4 + 2)         # S, dF in; dS out
            + D * (K + 1) * 4 * 2)                   # w, bias in; dw, dbias out
    return {"workload": f"one {Lseg}-token segment, Bz={Bz}, D={D}, K={K}",
            "avg_call_ms": ms, "launches_per_call": 2, "algorithmic_bytes_per_call": byts,
            "achieved_gbs": byts / ms / 1e6, "frac": byts / ms / 1e6 / hbm,
            "tokens_per_s": Bz * Lseg / (ms * 1e-3)}


def bench_scan_bwd(torch, sss, dev, stream, flush, args, hbm, s, Lseg):
    """sss_ssm_scan_bwd on one segment of the workload: bf16 x, dt, B, C, fp32
    h0, dy and dhT in; fp32 dx, ddt, dA, dB, dC and dh0 out (four kernels:
    chunk-entry states, chunk-end state gradients, the chunk gradients, the
    fixed-order group and batch sums)."""
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    bf = torch.bfloat16
    Bz, H, P, N, G = s.Bz, s.H, s.P, s.N, 1
    x = torch.randn((Bz, Lseg, H, P), generator=g, device=dev).to(bf)
    dt = torch.nn.functional.softplus(torch.randn((Bz, Lseg, H), generator=g, device=dev) - 2).to(bf)
    A = -torch.rand((H,), generator=g, device=dev) * 0.99 - 0.01
    B = torch.randn((Bz, Lseg, G, N), generator=g, device=dev).to(bf)
    C = torch.randn((Bz, Lseg, G, N), generator=g, device=dev).to(bf)
    h0 = torch.randn((Bz, H, P, N), generator=g, device=dev) * 0.1
    dy = torch.randn((Bz, Lseg, H, P), generator=g, device=dev)
    dhT = torch.randn((Bz, H, P, N), generator=g, device=dev)
    ws = torch.empty(sss.ssm_scan_bwd_workspace_size(Bz, Lseg, H, P, N, G), dtype=torch.uint8,
                     device=dev)

    def call():
        sss.ssm_scan_bwd(x, dt, A, B, C, h0, dy, dhT, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    evs = []
    for _ in range(max(3, args.steps // 50)):
        flush.zero_()
        torch.cuda._sleep(200_000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
    stream.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    tok = Bz * Lseg
    D = H * P
    byts = (tok * (D * (2 + 4 + 4)                   # x bf16, dy fp32 in; dx fp32 out
                   + H * (2 + 4)                     # dt in, ddt out
                   + G * N * (2 * 2 + 2 * 4))        # B, C in; dB, dC out
            + Bz * H * P * N * 4 * 3                 # h0, dhT in; dh0 out
            + H * 4 * 2)                             # A in, dA out
    return {"workload": f"one {Lseg}-token segment, Bz={Bz}, H={H}, P={P}, N={N}, bf16 inputs",
            "avg_call_ms": ms, "launches_per_call": 4, "algorithmic_bytes_per_call": byts,
            "achieved_gbs": byts / ms / 1e6, "frac": byts / ms / 1e6 / hbm,
            "tokens_per_s": tok / (ms * 1e-3),
            "kernel": "fp32 CUDA-core chunked backward (chunks of 64)"}


def bench_mamba2(torch, sss, dev, stream, flush, args, hbm, s):
    """sss_mamba2_mixer_fwd (the full Mamba-2 wiring) on one segment of the
    workload's shape: bf16 xBC over D + 2GN channels, z and dt_raw, fp32
    dt_bias, A, D_skip, conv weights and bias, Gaussian conv state (bf16) and
    h0 (fp32); bf16 y and the final conv and SSM states out.  Two launches: the
    conv over every xBC channel into an fp32 workspace, then the register-tiled
    fp32 CUDA-core scan with the discretisation, skip and gate."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    bf = torch.bfloat16
    Bz, Ls, H, P, N, G, K = s.Bz, s.segments[0], s.H, s.P, s.N, s.G, s.K
    D = H * P
    Dt = D + 2 * G * N
    xBC = torch.randn((Bz, Ls, Dt), generator=g, device=dev).to(bf)
    z = torch.randn((Bz, Ls, D), generator=g, device=dev).to(bf)
    dt_raw = (torch.randn((Bz, Ls, H), generator=g, device=dev) - 2.0).to(bf)
    dt_bias = torch.rand((H,), generator=g, device=dev) - 0.5
    A = -torch.rand((H,), generator=g, device=dev) * 0.99 - 0.01
    D_skip = torch.rand((H,), generator=g, device=dev) + 0.5
    w = torch.randn((Dt, K), generator=g, device=dev) * (0.5 ** 0.5)
    bias = torch.full((Dt,), 0.1, device=dev)
    S = torch.randn((Bz, Dt, K - 1), generator=g, device=dev).to(bf)
    h0 = torch.randn((Bz, H, P, N), generator=g, device=dev) * 0.1
    F = torch.empty_like(S)
    hT = torch.empty_like(h0)
    y = torch.empty((Bz, Ls, H, P), dtype=bf, device=dev)
    ws = torch.empty(max(16, sss.mamba2_mixer_fwd_workspace_size(Bz, Ls, H, P, N, G)),
                     dtype=torch.uint8, device=dev)

    def call():
        sss.mamba2_mixer_fwd(xBC, z, dt_raw, dt_bias, A, D_skip, w, bias, H, G, N,
                             conv_state=S, h0=h0, conv_state_out=F, hT=hT, y=y, workspace=ws,
                             stream=stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ms = statistics.mean(events_timed(torch, stream, flush, call, max(3, args.steps // 10)))
    byts = (Bz * Ls * (Dt * 2 + D * 2 + H * 2 + D * 2)       # xBC, z, dt_raw in; y out
            + 2 * Bz * Dt * (K - 1) * 2                       # conv state in and out
            + 2 * Bz * H * P * N * 4                          # h0 in, hT out
            + Dt * (K + 1) * 4 + 3 * H * 4)                   # weights, bias, dt_bias, A, D
    return {"workload": f"{s.name} shape, one {Ls}-token segment: Bz={Bz}, H={H}, P={P}, N={N}, "
                        f"G={G}, K={K}, xBC over {Dt} channels, bf16, Gaussian states",
            "avg_call_ms": ms, "launches_per_call": 2, "algorithmic_bytes_per_call": byts,
            "achieved_gbs": byts / ms / 1e6, "frac": byts / ms / 1e6 / hbm,
            "tokens_per_s": Bz * Ls / (ms * 1e-3),
            "kernel": "conv_state_fwd_kernel over xBC (fp32 workspace), then "
                      "mamba2_scan_rt_kernel (register-tiled fp32 CUDA cores)"}


def bench_long_context(torch, sss, dev, stream, flush, args, hbm, hbm_kind):
    """The long-context streaming workload: batch 1, 64 consecutive
    2048-token segments of a 780M-like layer (H 48, P 64, N 128, K 4, bf16),
    each sss_mixer_fwd call starting from the previous call's conv and SSM
    states (in place).  Its 24 head pairs fill a sixth of the GPU, so the
    library splits each segment into spans (section 2.5 Eq. (4) of "Understanding
    and Improving Length Generalization in Recurrent Models"); the same stream
    is also timed in one pass per segment.  Inputs of all 64 segments are
    resident (about 0.9 GB, larger than L2); L2 is flushed before each timed
    stream."""
    s = synth.WORKLOADS["m780m_128k"]
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    bf = torch.bfloat16
    Bz, H, P, N, K, G = s.Bz, s.H, s.P, s.N, s.K, s.G
    D, Lseg, nseg = H * P, s.segments[0], len(s.segments)
    L = Lseg * nseg
    x = torch.randn((nseg, Bz, Lseg, D), generator=g, device=dev).to(bf)
    dt = torch.nn.functional.softplus(
        torch.randn((nseg, Bz, Lseg, H), generator=g, device=dev) - 2).to(bf)
    B = torch.randn((nseg, Bz, Lseg, G, N), generator=g, device=dev).to(bf)
    C = torch.randn((nseg, Bz, Lseg, G, N), generator=g, device=dev).to(bf)
    A = -torch.rand((H,), generator=g, device=dev) * 0.99 - 0.01
    w = torch.randn((D, K), generator=g, device=dev) * 0.7
    bias = torch.full((D,), 0.1, device=dev)
    S = torch.zeros((Bz, D, K - 1), dtype=bf, device=dev)
    h = torch.zeros((Bz, H, P, N), device=dev)
    y = torch.empty((Bz, Lseg, H, P), dtype=bf, device=dev)
    ns_auto = sss.mixer_fwd_span_count(Bz, Lseg, H, P, N, G, K, bf, bf)

    def timed(ns):
        ws = (torch.empty(sss.fwd_spans_workspace_size(Bz, Lseg, H, P, N, K, ns),
                          dtype=torch.uint8, device=dev) if ns > 1 else None)

        def stream_once():
            for i in range(nseg):
                sss.mixer_fwd(x[i], dt[i], A, B[i], C[i], w, bias, S, h, conv_state_out=S, hT=h,
                              y=y, fused=True, spans=ns, workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(max(1, min(args.warmup, 3))):
                stream_once()
        torch.cuda.synchronize()
        ms = []
        for _ in range(3):
            flush.zero_()
            torch.cuda._sleep(200_000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                stream_once()
            e1.record(stream)
            stream.synchronize()
            ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    ms_span = timed(ns_auto)
    ms_one = timed(1)
    assert sss.device_status() == 0
    tok = Bz * L
    seg_bytes = algorithmic_bytes(s, Lseg)
    us_seg = ms_span * 1e3 / nseg
    return {"workload": workload_desc(s), "spans_per_segment": ns_auto,
            "ms_per_stream": ms_span, "tokens_per_s": tok / (ms_span * 1e-3),
            "us_per_segment": us_seg,
            "roofline": roofline_block(seg_bytes, us_seg * 1e-3, hbm, hbm_kind,
                                       "the segment's launches together (span kernels and the "
                                       "pair kernel passes)" if ns_auto > 1 else
                                       "ssm_scan_pair_kernel<bf16,bf16,fused>", s.name)
                        | {"per": "2048-token segment, averaged over the 64-segment stream"},
            "one_pass": {"ms_per_stream": ms_one, "tokens_per_s": tok / (ms_one * 1e-3),
                         "us_per_segment": ms_one * 1e3 / nseg,
                         "frac": seg_bytes / (ms_one * 1e-3 / nseg) / 1e9 / hbm},
            "path": "sss_mixer_fwd_spans: conv-state gather + decay sums, state-only pass "
                    "from zero states, warp-shuffle carry, pass from carried states (4 launches "
                    "per segment)" if ns_auto > 1 else "sss_mixer_fwd (one launch per segment)"}


def bench_train_utils(torch, sss, dev, stream, flush, args, hbm, s, Lseg):
    """The state utilities at the workload's state size: a prompt's state
    written into pool rows (circular layout, S_len 4), the zero reset (10% of
    rows), the fitted-noise statistics and sampling, and the per-head
    state-std trace (stride 64) over one segment."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    Bz, H, P, N = s.Bz, s.H, s.P, s.N
    hT = torch.randn((Bz, H, P, N), generator=g, device=dev)
    conv = torch.randn((Bz, s.D, s.K - 1), generator=g, device=dev).to(torch.bfloat16)
    u = torch.rand((Bz,), generator=g, device=dev)
    mu = torch.zeros((H,), device=dev)
    var = torch.ones((H,), device=dev)
    eps = torch.randn((Bz, H, P, N), generator=g, device=dev)
    h0 = torch.empty_like(eps)
    x = torch.randn((Bz, Lseg, H, P), generator=g, device=dev).to(torch.bfloat16)
    dt = torch.nn.functional.softplus(torch.randn((Bz, Lseg, H), generator=g, device=dev) - 2).to(torch.bfloat16)
    A = -torch.rand((H,), generator=g, device=dev) * 0.99 - 0.01
    B = torch.randn((Bz, Lseg, 1, N), generator=g, device=dev).to(torch.bfloat16)
    state = Bz * H * P * N * 4
    xp = torch.randn((Bz, Lseg, s.D), generator=g, device=dev).to(torch.bfloat16)
    cpool = torch.zeros((2 * Bz, s.D, 4), dtype=torch.bfloat16, device=dev)
    spool = torch.zeros((2 * Bz, H, P, N), device=dev)
    pidx = torch.arange(Bz, dtype=torch.int32, device=dev) * 2
    plen = torch.full((Bz,), Lseg, dtype=torch.int32, device=dev)
    calls = {
        "prefill_to_pool": (lambda: sss.prefill_to_pool(xp, conv, s.K, hT, cpool, spool, plen, pidx, H),
                            2 * state + Bz * s.D * 4 * 2 * 2),
        "fitted_noise_update": (lambda: sss.fitted_noise_update(hT, mu, var, 0.1, True), state),
        "fitted_noise_sample": (lambda: sss.fitted_noise_sample(mu, var, eps, h0), 2 * state),
        "state_std_trace": (lambda: sss.state_std_trace(x, dt, A, B, hT, 64),
                            Bz * Lseg * (H * P * 2 + H * 2 + N * 2) + state),
    }
    out = {"workload": f"Bz={Bz}, H={H}, P={P}, N={N} fp32 states; trace over one {Lseg}-token "
                       f"segment, bf16 inputs"}
    for name, (fn, byts) in calls.items():
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(max(3, args.steps // 50)):
            flush.zero_()
            torch.cuda._sleep(100_000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        stream.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        out[name] = {"avg_call_ms": ms, "algorithmic_bytes_per_call": byts,
                     "achieved_gbs": byts / ms / 1e6, "frac": byts / ms / 1e6 / hbm}
    # the reset writes zeros to the rows it resets and touches nothing else
    sss.state_reset(u, 0.1, hT, conv)
    return out


def bench_decode(torch, sss, dev, stream, flush, args, hbm, name):
    """The continuous-batching decode update (sss_mixer_update): 256 of 512
    pool rows by a random permutation, circular conv pool, SSM pool in fp32,
    L_new tokens per call."""
    d = synth.DECODE[name]
    g = torch.Generator(device=dev)
    g.manual_seed(d.seed)
    bf = torch.bfloat16
    conv_pool = torch.randn((d.pool, d.D, d.S_len), generator=g, device=dev).to(bf)
    ssm_pool = torch.randn((d.pool, d.H, d.P, d.N), generator=g, device=dev) * 0.1
    idx = torch.randperm(d.pool, generator=g, device=dev)[: d.Bz].to(torch.int32)
    seqlens = torch.randint(0, d.max_seqlen, (d.Bz,), generator=g, device=dev,
                            dtype=torch.int32)
    x = torch.randn((d.Bz, d.L_new, d.D), generator=g, device=dev).to(bf)
    dt = torch.nn.functional.softplus(
        torch.randn((d.Bz, d.L_new, d.H), generator=g, device=dev) - 2.0).to(bf)
    B = torch.randn((d.Bz, d.L_new, d.G, d.N), generator=g, device=dev).to(bf)
    C = torch.randn((d.Bz, d.L_new, d.G, d.N), generator=g, device=dev).to(bf)
    A = -(torch.rand((d.H,), generator=g, device=dev) * 0.99 + 0.01)
    w = torch.randn((d.D, d.K), generator=g, device=dev) * (0.5 ** 0.5)
    bias = torch.full((d.D,), 0.1, device=dev)
    y = torch.empty((d.Bz, d.L_new, d.H, d.P), dtype=bf, device=dev)

    def call():
        sss.mixer_update(x, w, bias, conv_pool, seqlens, idx, dt, A, B, C, ssm_pool, y)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    evs = []
    for _ in range(max(3, args.steps // 10)):
        flush.zero_()
        torch.cuda._sleep(200_000)  # the host enqueues the call meanwhile
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
    stream.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    avg = statistics.mean(ms)
    byts = (2 * d.Bz * d.H * d.P * d.N * 4
            + d.Bz * d.D * (d.K - 1) * 2 + d.Bz * d.L_new * d.D * 2
            + d.Bz * d.L_new * (2 * d.D * 2 + 2 * d.G * d.N * 2 + d.H * 2))
    gbs = byts / (avg * 1e-3) / 1e9
    return {"workload": f"{name}: 256 of 512 pool rows by a random permutation, circular "
                        f"conv pool [512,4096,4], cache_seqlens ~ U[0,10000), SSM pool "
                        f"[512,64,64,128] fp32, L_new={d.L_new}, H=64, P=64, N=128, K=4, bf16",
            "tokens_per_s": d.Bz * d.L_new / (avg * 1e-3), "avg_launch_ms": avg,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "algorithmic_bytes_per_launch": byts,
                         "kernel": "mixer_update"}}


if __name__ == "__main__":
    main()

"""Benchmark: attention fwd + bwd TFLOP/s on one GB300 (Z128 H8 N1024 D128).

One step = one pass of the whole hot path over one batch: fa_fwd (O, lse)
then fa_bwd (a dQ kernel that also forms Delta, then a dK/dV kernel), fp16
in, fp32 accumulate.  FLOPs are the algorithmic count (forward 4 N^2 D per head, the
backward 2.5x that); the work the method avoids is not counted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  --impl reference times the fp64 CPU oracle (the only
reference this method has) on a bounded sample of the same workload.
Under torchrun each rank runs its own replica of the workload on its GPU (the
heads are independent: no data-path collective); rank 0 prints.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

Z, H, N, D, CAUSAL = 128, 8, 1024, 128, False
HKV, NK = H, N  # K/V heads and key length (grouped heads / unequal lengths; the benchmark has HKV = H, NK = N)
DTYPE = "f16"  # element type of the inputs and outputs: "f16" (benchmark) or "bf16"
WORKLOAD = "attention fwd+bwd, Z128 H8 N1024 D128 non-causal, fp16 inputs ~N(0,1), scale 1/sqrt(D)"
METRIC = "attention fwd / fwd+bwd TFLOP/s at Z128 H8 N1024 D128 on 1 GB300; % of FP16 peak"
UNIT = "TFLOP/s"
SEED = 1002


def set_workload(z, h, n, d, causal, hkv=None, nk=None):
    global Z, H, N, D, CAUSAL, HKV, NK, WORKLOAD
    Z, H, N, D, CAUSAL = z, h, n, d, bool(causal)
    HKV = h if hkv is None else hkv
    NK = n if nk is None else nk
    extra = ""
    if HKV != H:
        extra += f" Hkv{HKV}"
    if NK != N:
        extra += f" Nk{NK}"
    WORKLOAD = (f"attention fwd+bwd, Z{Z} H{H} N{N}{extra} D{D} {'causal' if CAUSAL else 'non-causal'}, "
                "fp16 inputs ~N(0,1), scale 1/sqrt(D)")


def flops_fwd(z, h, n, d, causal, nk=None):
    """4 D FLOPs (two GEMMs) per visible (query, key) pair per query head."""
    nk = n if nk is None else nk
    pairs = n * (n + 1) / 2.0 + n * (nk - n) if causal else float(n) * nk
    return z * h * 4.0 * pairs * d


def flops_step(z=None, h=None, n=None, d=None, causal=None):
    n = N if n is None else n
    return 3.5 * flops_fwd(Z if z is None else z, H if h is None else h, n, D if d is None else d,
                           CAUSAL if causal is None else causal, NK if n == N else n)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            js = json.load(f)
        return {"tflops": js.get("bf16_tflops"), "tflops_sustained": js.get("bf16_tflops_sustained"),
                "hbm_gbs": js.get("hbm_gbs"), "source": "measured"}
    return {"tflops": 1900.0, "tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ CPU oracle


def cpu_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(budget_s=12.0, max_heads=256):
    """Time the fp64 oracle, forward + backward, head by head on the host
    cores until the budget is spent (at least two heads)."""
    from attention_sm_flashattention_gb300.inputs import make_inputs
    from oracle import attention as orc

    q, k, v, do = make_inputs(1, max_heads, N, D, seed=SEED)
    scale = 1.0 / math.sqrt(D)
    done, t_fwd, t_bwd, t0 = 0, 0.0, 0.0, time.perf_counter()
    while done < max_heads and (done < 2 or time.perf_counter() - t0 < budget_s):
        qh, kh, vh, dh = (t[0, done] for t in (q, k, v, do))
        a = time.perf_counter()
        orc.attn_fwd_head(qh, kh, vh, CAUSAL, scale)
        b = time.perf_counter()
        orc.attn_bwd_head(qh, kh, vh, dh, CAUSAL, scale)
        t_fwd += b - a
        t_bwd += time.perf_counter() - b
        done += 1
    el = t_fwd + t_bwd
    fl = flops_step(1, done, N, D, CAUSAL)
    return {"value": fl / el / 1e12, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{done} of the {Z * H} heads (N{N} D{D} {'causal' if CAUSAL else 'non-causal'}), "
                      f"fp64 numpy forward+backward, "
                      f"{el:.1f} s wall",
            "fwd_s_per_head": t_fwd / done, "bwd_s_per_head": t_bwd / done}


def oracle_configs(budget_s=1.5):
    """The oracle on a few heads of every benchmark shape (forward and
    backward timed apart), with its time for all heads of the shape by
    proportion."""
    from attention_sm_flashattention_gb300.inputs import WORKLOADS, make_inputs
    from oracle import attention as orc

    out = {}
    for name, w in WORKLOADS.items():
        nh = min(w.heads, 64)
        q, k, v, do = make_inputs(1, nh, w.N, w.D, seed=w.seed)
        done, t_fwd, t_bwd = 0, 0.0, 0.0
        while done < nh and (done < 2 or t_fwd + t_bwd < budget_s):
            qh, kh, vh, dh = (t[0, done] for t in (q, k, v, do))
            a = time.perf_counter()
            orc.attn_fwd_head(qh, kh, vh, w.causal, w.scale)
            b = time.perf_counter()
            orc.attn_bwd_head(qh, kh, vh, dh, w.causal, w.scale)
            t_fwd += b - a
            t_bwd += time.perf_counter() - b
            done += 1
        out[name] = {"heads_timed": done, "fwd_s_all_heads": t_fwd / done * w.heads,
                     "bwd_s_all_heads": t_bwd / done * w.heads, "cores": cpu_threads()}
    return out


# -------------------------------------------------------------- clock sampler


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                mx.append(float(row[2]))
                pw.append(float(row[3]))
            except ValueError:
                continue
            for nm, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        # under load: samples drawing at least half the peak power seen
        load = [c for c, w in zip(sm, pw) if pw and w >= 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(load) if load else None, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(load)}


# ----------------------------------------------------------------- GPU bench


def smi_index(local_rank):
    """nvidia-smi's index of this rank's GPU."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    return vis.split(",")[local_rank] if vis else local_rank


def gpu_bench(args, rank, world, local_rank):
    import torch

    import attention_sm_flashattention_gb300 as fa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    from attention_sm_flashattention_gb300.inputs import make_inputs

    elem = torch.bfloat16 if DTYPE == "bf16" else torch.float16
    # the seeded recipe the parity tests use (drawn on the CPU, then moved)
    q, k, v, do = make_inputs(Z, H, N, D, SEED, device=dev, dtype=elem, Hkv=HKV, Nk=NK)
    scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((Z, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.bwd_workspace_size(Z, H, N, D, CAUSAL, HKV, NK), device=dev, dtype=torch.uint8)

    def step():
        fa.fwd(q, k, v, causal=CAUSAL, scale=scale, out=(o, lse))
        fa.bwd(q, k, v, o, do, lse, causal=CAUSAL, scale=scale, workspace=ws, out=(dq, dk, dv))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise RuntimeError("device status reports a kernel wait timeout during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    sampler = ClockSampler(smi_index(local_rank))
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    # per-call events on the launching stream: forward kernel and backward call
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        fa.fwd(q, k, v, causal=CAUSAL, scale=scale, out=(o, lse))
        ev[i][1].record(stream)
        fa.bwd(q, k, v, o, do, lse, causal=CAUSAL, scale=scale, workspace=ws, out=(dq, dk, dv))
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    if fa.device_status() != 0:
        raise RuntimeError("device status reports a kernel wait timeout in the timed region")
    total_ms = t_start.elapsed_time(t_end)
    fwd_all = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_all = [e[1].elapsed_time(e[2]) for e in ev]
    fwd_ms = statistics.mean(fwd_all)
    bwd_ms = statistics.mean(bwd_all)

    # ---- end to end through the public API: pinned host in, host out.
    # Every step copies its four inputs in and its four results out.  The
    # copies run on two side streams (the copy engines move both ways at
    # once) into and out of two device buffer sets, so that step i's inputs
    # arrive and step i-1's results leave while the kernels compute.
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, do))
    ho, hdq, hdk, hdv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, dq, dk, dv))
    e2e_steps = max(3, min(args.steps, 20))
    bufs = [(q, k, v, do, o, lse, dq, dk, dv),
            tuple(torch.empty_like(t) for t in (q, k, v, do, o, lse, dq, dk, dv))]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        bq, bk, bv, bdo, bo, blse, bdq, bdk, bdv = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_comp[b])   # step i-2 has finished reading these inputs
            for d, h in ((bq, hq), (bk, hk), (bv, hv), (bdo, hdo)):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])      # step i-2's results have left
        fa.fwd(bq, bk, bv, causal=CAUSAL, scale=scale, out=(bo, blse))
        fa.bwd(bq, bk, bv, bo, bdo, blse, causal=CAUSAL, scale=scale, workspace=ws, out=(bdq, bdk, bdv))
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for h, d in ((ho, bo), (hdq, bdq), (hdk, bdk), (hdv, bdv)):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    def e2e_run(n):
        s_in.wait_stream(stream)
        for i in range(n):
            e2e_step(i)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if fa.device_status() != 0:
        raise RuntimeError("device status reports a kernel wait timeout in the end-to-end leg")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hdq, hdk, hdv))
    del bufs, hq, hk, hv, hdo, ho, hdq, hdk, hdv
    return {"total_ms": total_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "e2e_ms": e2e_ms,
            "fwd_stats": call_stats(fwd_all), "bwd_stats": call_stats(bwd_all),
            "h2d": h2d, "d2h": d2h, "clocks": clocks, "step": step}


def call_stats(ms):
    """Median, min and 90th percentile of per-call times (ms)."""
    xs = sorted(ms)
    return {"median_ms": statistics.median(xs), "min_ms": xs[0],
            "p90_ms": xs[max(0, math.ceil(0.9 * len(xs)) - 1)], "calls": len(xs)}


# The other benchmark shapes, reported beside the headline in the same line:
# (workload, flush L2 before every timed call).  The two D64 shapes' inputs
# (0.1 and 17 MB) fit in L2, so a 256 MB buffer is written before each call.
SIDE_CONFIGS = (("z1h2n128d64", True), ("z4h8n1024d64", True), ("z128h8n1024d128", False),
                ("z128h8n1024d128c", False), ("z128h8n1024d256", False), ("z128h8n1024d256c", False))


def config_bench(name, flush, dev, calls=50, warmup=10):
    """fa_fwd then fa_bwd on one benchmark shape (inputs from the seeded
    recipe): `warmup` untimed calls, then `calls` calls of each, every call
    timed alone with CUDA events on the launching stream."""
    import torch

    import attention_sm_flashattention_gb300 as fa
    from attention_sm_flashattention_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    stream = torch.cuda.current_stream()
    q, k, v, do = make_inputs(w.Z, w.H, w.N, w.D, w.seed, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.Z, w.H, w.N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.bwd_workspace_size(w.Z, w.H, w.N, w.D, w.causal), device=dev, dtype=torch.uint8)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None

    def fwd():
        fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=(o, lse))

    def bwd():
        fa.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, workspace=ws, out=(dq, dk, dv))

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(calls)]
    for e in ev:
        if flush:
            flush_buf.zero_()
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        if flush:
            flush_buf.zero_()
        e[2].record(stream)
        bwd()
        e[3].record(stream)
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise RuntimeError(f"device status reports a kernel wait timeout ({name})")
    f_st = call_stats([e[0].elapsed_time(e[1]) for e in ev])
    b_st = call_stats([e[2].elapsed_time(e[3]) for e in ev])
    peak = measured_peaks()["tflops"]
    f_fl = flops_fwd(w.Z, w.H, w.N, w.D, w.causal)
    f_tf = f_fl / (f_st["median_ms"] * 1e-3) / 1e12
    b_tf = 2.5 * f_fl / (b_st["median_ms"] * 1e-3) / 1e12
    in_mb = 4 * w.Z * w.H * w.N * w.D * 2 / 1e6
    return {
        "workload": f"attention fwd+bwd, {w.describe()}, fp16 inputs ~N(0,1), scale 1/sqrt(D)",
        "fwd": dict(f_st, tflops=f_tf, frac=f_tf / peak),
        "bwd": dict(b_st, tflops=b_tf, frac=b_tf / peak, kernels=bwd_kernel_names(w.D, w.causal)),
        "fwd_bwd_tflops": 3.5 * f_fl / ((f_st["median_ms"] + b_st["median_ms"]) * 1e-3) / 1e12,
        "l2": (f"inputs {in_mb:.0f} MB, smaller than L2: a 256 MB buffer written before every timed call"
               if flush else f"inputs larger than L2 ({in_mb:.0f} MB), no flush needed"),
    }


def side_configs(dev, sampler_index):
    """Every SIDE_CONFIGS shape through config_bench, clocks sampled throughout."""
    sampler = ClockSampler(sampler_index)
    sampler.start()
    time.sleep(0.3)
    out = {name: config_bench(name, flush, dev) for name, flush in SIDE_CONFIGS}
    out["clocks"] = sampler.stop()
    out["timing"] = ("per call: 10 warm-up calls, then 50 calls of fa_fwd and of fa_bwd, each timed alone with "
                     "CUDA events; TFLOP/s and frac (of the measured burst bf16 peak) from the median")
    return out


def sustained_bench(step, ms_per_step, sampler_index, seconds=2.5):
    """The headline step repeated back to back for about `seconds`, against
    the sustained (power-capped) peak."""
    import torch

    stream = torch.cuda.current_stream()
    n = max(50, int(seconds * 1e3 / ms_per_step))
    sampler = ClockSampler(sampler_index)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / n
    val = flops_step() / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    peak = peaks.get("tflops_sustained") or peaks["tflops"]
    return {"steps": n, "seconds": ms * n / 1e3, "ms_per_step": ms, "value": val, "unit": UNIT, "peak": peak,
            "peak_kind": "sustained bf16 cuBLAS (" + peaks["source"] + ")", "frac": val / peak, "clocks": clocks}


def reduce_max(vals, world):
    """Element-wise max of `vals` over the ranks (the slowest rank's times)."""
    if world == 1:
        return vals
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_step_per_rank, world, steps, max_total_ms):
    """Whole-job rate in TFLOP/s: the work of all ranks' steps over the
    slowest rank's time (each rank runs its own replica: weak scaling)."""
    return world * flops_per_step_per_rank * steps / (max_total_ms * 1e-3) / 1e12


def bwd_kernel_names(d, causal):
    c = str(bool(causal)).lower()
    if d == 256:
        return f"fa_bwd call: fa_bwd256_dq_kernel<{c}> (with Delta) + fa_bwd256_dkdv_kernel<{c}>"
    return f"fa_bwd call: fa_bwd_dq_kernel<{d},{c}> (with Delta) + fa_bwd_dkdv_kernel<{d},{c}>"


def bwd_launches(d):
    """Kernels one fa_bwd call launches: a dQ kernel that also forms Delta,
    then a dK/dV kernel (every D)."""
    return 2


def load_traffic():
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        return json.load(f)


def paged_bench(args):
    """Forward over a paged K/V cache (fa_fwd_paged): Z sequences of N queries
    at the end of an NK-token context, HKV K/V heads, pages of args.paged
    tokens assigned from a random permutation.  Times the paged call and, for
    comparison, the dense call on the same shape; prints one JSON line."""
    import torch

    import attention_sm_flashattention_gb300 as fa

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev).manual_seed(SEED)
    elem = torch.bfloat16 if DTYPE == "bf16" else torch.float16
    ps = args.paged
    pages_per_seq = (NK + ps - 1) // ps
    num_pages = Z * pages_per_seq
    q = torch.randn((Z, H, N, D), device=dev, dtype=elem, generator=gen)
    kc = torch.randn((num_pages, ps, HKV, D), device=dev, dtype=elem, generator=gen)
    vc = torch.randn((num_pages, ps, HKV, D), device=dev, dtype=elem, generator=gen)
    table = torch.randperm(num_pages, device=dev, generator=gen).to(torch.int32).view(Z, pages_per_seq)
    lens = torch.full((Z,), NK, dtype=torch.int32, device=dev)
    k = torch.randn((Z, HKV, NK, D), device=dev, dtype=elem, generator=gen)
    v = torch.randn_like(k)
    o = torch.empty_like(q)
    lse = torch.empty((Z, H, N), device=dev, dtype=torch.float32)
    scale = 1.0 / math.sqrt(D)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    sampler = ClockSampler(smi_index(0))
    sampler.start()
    time.sleep(0.3)
    ms = timed(lambda: fa.fwd_paged(q, kc, vc, table, lens, causal=CAUSAL, scale=scale, out=(o, lse)))
    clocks = sampler.stop()
    ms_dense = timed(lambda: fa.fwd(q, k, v, causal=CAUSAL, scale=scale, out=(o, lse)))
    sparse = None
    if args.sparse_keep > 0:
        # selected blocks: the same random share of every sequence's blocks for
        # each K/V head (in shuffled order), the last block always included
        nsel = max(1, min(pages_per_seq, int(round(args.sparse_keep * pages_per_seq))))
        order = torch.argsort(torch.rand((Z, HKV, pages_per_seq), device=dev, generator=gen), dim=2)[:, :, :nsel]
        order[:, :, 0] = pages_per_seq - 1
        sel_blocks = order.to(torch.int32).contiguous()
        sel_pages = torch.gather(table.unsqueeze(1).expand(Z, HKV, pages_per_seq), 2, order).to(torch.int32).contiguous()
        sel_count = torch.full((Z, HKV), nsel, dtype=torch.int32, device=dev)
        ms_sparse = timed(lambda: fa.fwd_sparse(q, kc, vc, sel_pages, sel_blocks, sel_count, lens, causal=CAUSAL,
                                                scale=scale))
        sel_keys = Z * HKV * nsel * ps
        sparse = {"blocks_selected": nsel, "of": pages_per_seq, "ms": ms_sparse,
                  "speedup_vs_paged": ms / ms_sparse,
                  "kv_gbs": 2 * sel_keys * D * q.element_size() / (ms_sparse * 1e-3) / 1e9}
    # the same call with every sequence's key range split into slices
    # (fa_fwd_paged_split), the library's slice count for this shape
    split = None
    nsplit = fa.paged_split_count(Z, H, HKV, N, D, ps, pages_per_seq, CAUSAL)
    if nsplit > 1:
        from attention_sm_flashattention_gb300 import _native
        ws = torch.empty(_native.lib().fa_fwd_paged_split_workspace_size(Z, H, N, D, nsplit), dtype=torch.uint8,
                         device=dev)
        ms_split = timed(lambda: fa.fwd_paged(q, kc, vc, table, lens, causal=CAUSAL, scale=scale, out=(o, lse),
                                              splits=nsplit, workspace=ws))
        split = {"splits": nsplit, "ms": ms_split, "speedup_vs_paged": ms / ms_split,
                 "tflops": flops_fwd(Z, H, N, D, CAUSAL, NK) / (ms_split * 1e-3) / 1e12,
                 "kv_gbs": 2 * Z * HKV * NK * D * q.element_size() / (ms_split * 1e-3) / 1e9}
    # cache write of the Z * N new tokens (ReshapeAndCache) to distinct slots
    toks = Z * N
    k_new = torch.randn((toks, HKV, D), device=dev, dtype=elem, generator=gen)
    v_new = torch.randn_like(k_new)
    slots = torch.randperm(num_pages * ps, device=dev, generator=gen)[:toks].to(torch.int64)
    ms_write = timed(lambda: fa.reshape_and_cache(k_new, v_new, slots, kc, vc))
    if fa.device_status() != 0:
        raise RuntimeError("device status reports a kernel wait timeout")
    fl = flops_fwd(Z, H, N, D, CAUSAL, NK)
    tf = fl / (ms * 1e-3) / 1e12
    kv_bytes = 2 * Z * HKV * NK * D * q.element_size()
    peaks = measured_peaks()
    line = {
        "metric": "attention fwd over a paged K/V cache, TFLOP/s", "value": tf, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
        "config": {"workload": f"paged attention fwd, {Z} sequences, H{H} Hkv{HKV}, {N} queries at the end of "
                               f"{NK}-token contexts, D{D}, pages of {ps} tokens, {'causal' if CAUSAL else 'non-causal'}",
                   "B": Z, "H": H, "Hkv": HKV, "Nq": N, "context": NK, "D": D, "page_size": ps, "causal": CAUSAL},
        "dense_fwd_tflops": fl / (ms_dense * 1e-3) / 1e12, "dense_fwd_ms": ms_dense,
        "kv_cache_gbs": kv_bytes / (ms * 1e-3) / 1e9,
        "sparse": sparse,
        "split": split,
        "cache_write": {"tokens": toks, "ms": ms_write,
                        "gbs": 4 * toks * HKV * D * q.element_size() / (ms_write * 1e-3) / 1e9,
                        "peak_hbm_gbs": peaks["hbm_gbs"]},
        "roofline": {"bound": "tensor", "kernel": f"fa_fwd_kernel<{D},{str(CAUSAL).lower()},paged>", "achieved": tf,
                     "peak": peaks["tflops"], "unit": "TFLOP/s", "frac": tf / peaks["tflops"], "traffic": None},
        "clocks": clocks, "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the other benchmark shapes and the sustained leg (profiling runs)")
    # Workload overrides, for profiling the same step on a smaller case; the
    # default is the benchmark workload above.
    ap.add_argument("--z", type=int, default=Z)
    ap.add_argument("--h", type=int, default=H)
    ap.add_argument("--n", type=int, default=N)
    ap.add_argument("--d", type=int, default=D)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--hkv", type=int, default=None, help="K/V heads (grouped heads; default H)")
    ap.add_argument("--nk", type=int, default=None, help="key length (default N, the query length)")
    ap.add_argument("--paged", type=int, default=0, metavar="PAGE_SIZE",
                    help="time the forward over a paged K/V cache with pages of this many tokens instead")
    ap.add_argument("--sparse-keep", type=float, default=0.0, metavar="FRACTION",
                    help="with --paged: also time the forward over this share of each sequence's blocks")
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="f16",
                    help="element type of the inputs and outputs (the benchmark is f16)")
    args = ap.parse_args()
    global DTYPE
    DTYPE = args.dtype
    args.warmup = max(args.warmup, 3)
    set_workload(args.z, args.h, args.n, args.d, args.causal, args.hkv, args.nk)
    global WORKLOAD
    if DTYPE == "bf16":
        WORKLOAD = WORKLOAD.replace("fp16 inputs", "bf16 inputs")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    in_mb = (2 * Z * H * N + 2 * Z * HKV * NK) * D * 2 / 1e6
    config = {"workload": WORKLOAD, "Z": Z, "H": H, "N": N, "D": D, "causal": CAUSAL,
              "global_batch": Z * world, "seq_len": N, "parallelism": f"replicas{world}",
              "l2": (f"inputs larger than L2 ({in_mb:.0f} MB {DTYPE} per step), no flush needed" if in_mb > 130
                     else f"inputs {in_mb:.0f} MB {DTYPE} per step, smaller than L2: not flushed (profiling case)")}
    if HKV != H or NK != N:
        config.update({"Hkv": HKV, "Nk": NK})

    if args.paged:
        paged_bench(args)
        return

    if args.impl == "reference":
        # The oracle as it stands, on the host cores: each step is one head of
        # the workload (forward + backward in fp64); warm-up steps untimed.
        if rank != 0:
            return
        from attention_sm_flashattention_gb300.inputs import make_inputs
        from oracle import attention as orc

        nh = args.warmup + args.steps
        q, k, v, do = make_inputs(1, min(nh, Z * H), N, D, seed=SEED)
        scale = 1.0 / math.sqrt(D)
        times = []
        for i in range(nh):
            hh = i % q.shape[1]
            t0 = time.perf_counter()
            orc.attn_fwd_head(q[0, hh], k[0, hh], v[0, hh], CAUSAL, scale)
            orc.attn_bwd_head(q[0, hh], k[0, hh], v[0, hh], do[0, hh], CAUSAL, scale)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        per_head = flops_step(1, 1, N, D, CAUSAL)
        el = sum(times)
        val = per_head * len(times) / el / 1e12
        ms = el / len(times) * 1e3  # a timed step is one head
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "step": "one head of the workload (fa_fwd + fa_bwd's arithmetic in fp64 numpy)",
                "ms_all_heads_extrapolated": ms * Z * H,
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                                 "sample": f"{len(times)} heads of the workload ({'causal' if CAUSAL else 'non-causal'}), "
                                           f"one per step, fp64 numpy forward+backward, {el:.1f} s"},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")

    r = gpu_bench(args, rank, world, local_rank)
    total_ms, e2e_ms = reduce_max([r["total_ms"], r["e2e_ms"]], world)
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops_step(), world, args.steps, total_ms)
    e2e_value = job_throughput(flops_step(), world, 1, e2e_ms)
    peaks = measured_peaks()
    fwd_tf = flops_fwd(Z, H, N, D, CAUSAL, NK) / (r["fwd_ms"] * 1e-3) / 1e12
    bwd_tf = 2.5 * flops_fwd(Z, H, N, D, CAUSAL, NK) / (r["bwd_ms"] * 1e-3) / 1e12
    traffic = load_traffic()
    bwd_traffic = traffic.get(f"fa_bwd_d{D}{'c' if CAUSAL else ''}") if traffic else None
    # The roofline's denominator is the cuBLAS bf16 rate measured under the
    # same condition: the sustained (power-capped) figure when the power cap
    # was active during the timed region, else the burst figure.
    capped = "sw_power_cap" in (r["clocks"].get("reasons") or [])
    roof_peak = peaks["tflops_sustained"] if capped and peaks.get("tflops_sustained") else peaks["tflops"]
    roof_kind = ("sustained" if roof_peak != peaks["tflops"] else "burst") + " bf16 cuBLAS (" + peaks["source"] + ")"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE, "data": "synthetic", "config": config,
        "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"], "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_call": r["fwd_stats"], "bwd_call": r["bwd_stats"],
        "pct_of_peak": {"fwd": fwd_tf / peaks["tflops"], "fwd_bwd": value / world / peaks["tflops"],
                        "bwd": bwd_tf / peaks["tflops"], "peak_tflops": peaks["tflops"],
                        "peak_source": peaks["source"]},
        "roofline": {"bound": "tensor", "kernel": bwd_kernel_names(D, CAUSAL),
                     "achieved": bwd_tf, "peak": roof_peak, "unit": "TFLOP/s",
                     "frac": bwd_tf / roof_peak, "peak_kind": roof_kind,
                     "frac_of_burst_peak": bwd_tf / peaks["tflops"], "traffic": bwd_traffic},
        "clocks": r["clocks"],
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": e2e_ms,
                "copies": "pinned host buffers; inputs in and results out on two side streams, two device "
                          "buffer sets, overlapped with the kernels of the neighbouring steps"},
        "gpu_launches": (1 + bwd_launches(D)) * args.steps,
    }
    if world == 1 and not args.no_side:
        # the other benchmark shapes, then the headline step held for seconds
        import torch
        line["configs"] = side_configs(torch.device("cuda", local_rank), smi_index(local_rank))
        line["sustained"] = sustained_bench(r["step"], ms_per_step, smi_index(local_rank))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample()
        if not args.no_side:
            line["cpu_configs"] = oracle_configs()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

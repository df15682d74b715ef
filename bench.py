"""Benchmark of the causal bifocal-RoPE attention path on one B300 (or N replicas).

One step = the whole hot path over one batch of synthetic input:
  * prefill of the 4x-extension workload (L = 131072, G = 4, 32 query / 8 KV
    heads, d = 128, w0 = 4096, theta = 1e6): RoPE stage + routed attention;
  * decode against one absolute-position cache at L = 32767, 32769, 65537,
    131072 (G = 1, 2, 3, 4), one new token each.

`value` is the prefill throughput in TFLOP/s of causal-pair FLOPs (4 * d per
pair per query head), RoPE stage included; decode is reported beside it in
HBM GB/s and tokens/s.  Inputs (1.5 GB per prefill, 0.5 GB of cache) are
larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bifocal_rope_extension_causal_b300 import synth  # noqa: E402
from bifocal_rope_extension_causal_b300 import workloads as W  # noqa: E402

METRIC = "bifocal prefill TFLOP/s & % bf16 tensor peak at 128K; decode HBM GB/s"
PREFILL = W.EXT_128K
DECODE = W.DECODE
KERNELS_PER_PREFILL = 4   # rotation tables, RoPE (Q), RoPE (K), attention
KERNELS_PER_DECODE = 2    # split-K partials, merge


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags)
                          if fl.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
    return rank, local, world


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar (timing only; no data-path collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_rank: float, ms_per_rank: float, world: int) -> float:
    """Whole-job throughput of N independent replicas: the units all ranks
    processed over the slowest rank's time (work units per second)."""
    return world * work_per_rank / (max_over_ranks(ms_per_rank, world) * 1e-3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS = {}


def oracle_sample(n_rows: int = 128, head: int = 0):
    """Time the fp64 oracle on `n_rows` seeded rows of one query head of the
    128K prefill; returns (tflops, seconds, pairs, cores)."""
    import numpy as np
    import oracle
    w = PREFILL
    if head not in _ORACLE_INPUTS:
        q, k, v = synth.prefill_inputs(w.L, w.Hq, w.Hkv, w.d, w.index)
        hk = head // (w.Hq // w.Hkv)
        _ORACLE_INPUTS[head] = (q[:, :, head:head + 1].float().numpy(),
                                k[:, :, hk:hk + 1].float().numpy(),
                                v[:, :, hk:hk + 1].float().numpy())
    qn, kn, vn = _ORACLE_INPUTS[head]
    rows = np.sort(np.random.default_rng(99).choice(w.L, size=n_rows, replace=False))[None]
    t0 = time.perf_counter()
    oracle.bifocal_prefill(qn, kn, vn, w.w0, w.w_pretrained, w.theta, round_rotated_qk=True, rows=rows)
    dt = time.perf_counter() - t0
    pairs = int((rows + 1).sum())
    return 4.0 * w.d * pairs / dt / 1e12, dt, pairs, _cores()


def _cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    rank, _, world = int(os.environ.get("RANK", "0")), 0, int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    vals = []
    for _ in range(args.warmup):
        oracle_sample(32)
    secs, pairs = 0.0, 0
    for _ in range(args.steps):
        v, dt, pr, cores = oracle_sample(32)
        vals.append(v)
        secs += dt
        pairs += pr
    value = 4.0 * PREFILL.d * pairs / secs / 1e12
    sample = (f"fp64 oracle, 4x-extension prefill (L=131072, G=4): 32 seeded query rows of head 0 "
              f"per step ({pairs // max(args.steps, 1)} causal pairs), RoPE tables included")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_dict():
    w, dw = PREFILL, DECODE
    return {"workload": f"{w.name} + {dw.name}", "B": w.B, "L": w.L, "Hq": w.Hq, "Hkv": w.Hkv,
            "d": w.d, "w0": w.w0, "w_pretrained": w.w_pretrained, "rope_theta": w.theta,
            "decode_lengths": list(dw.lengths),
            "l2": "inputs larger than L2 (no flush needed); decode alone alternates two cache copies",
            "parallelism": "replicas"}


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    rank, local, world = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    import ctypes
    import bifocal_rope_extension_causal_b300 as jl
    from bifocal_rope_extension_causal_b300 import _capi
    lib = _capi.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    w, dw = PREFILL, DECODE

    q, k, v = synth.prefill_inputs(w.L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.L), dtype=torch.float32, device=dev)
    ws_bytes = jl.prefill_workspace_size(w.B, w.L, w.Hq, w.Hkv, w.d, w.w_pretrained)
    ws = jl.alloc_workspace(ws_bytes, dev)
    kc, vc, qs = synth.decode_inputs(dw.Lcap, dw.Hq, dw.Hkv, dw.d, dw.index, len(dw.lengths))
    kc, vc, qs = kc.to(dev), vc.to(dev), qs.to(dev)
    od = torch.empty((dw.B, dw.Hq, dw.d), dtype=torch.bfloat16, device=dev)
    lsed = torch.empty((dw.B, dw.Hq), dtype=torch.float32, device=dev)
    dws_bytes = jl.decode_workspace_size(dw.B, dw.Hq, dw.d, dw.Lcap)
    dws = jl.alloc_workspace(dws_bytes, dev)
    P = ctypes.c_void_p

    def rope():
        _capi.check(lib.jl_bifocal_rope(P(qd.data_ptr()), P(kd.data_ptr()), w.B, w.L, w.Hq, w.Hkv,
                                        w.d, w.w_pretrained, w.theta, None, P(ws.data_ptr()),
                                        ws_bytes, sp))

    def attention():
        _capi.check(lib.jl_bifocal_attention(P(vd.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()),
                                             w.B, w.L, w.Hq, w.Hkv, w.d, w.w0, w.w_pretrained, 0.0,
                                             P(ws.data_ptr()), ws_bytes, sp))

    def decode(i, L):
        _capi.check(lib.jl_bifocal_decode(P(qs[i].data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()),
                                          L, dw.Lcap, P(od.data_ptr()), P(lsed.data_ptr()), dw.B,
                                          dw.Hq, dw.Hkv, dw.d, dw.w0, dw.w_pretrained, dw.theta,
                                          0.0, P(dws.data_ptr()), dws_bytes, sp))

    nL = len(dw.lengths)

    def step(ev):
        ev[0].record(stream)
        rope()
        ev[1].record(stream)
        attention()
        ev[2].record(stream)
        for i, L in enumerate(dw.lengths):
            decode(i, L)
            ev[3 + i].record(stream)

    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3 + nL)])
    torch.cuda.synchronize()
    jl.device_status()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3 + nL)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for s in range(args.steps):
            step(events[s])
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    jl.device_status()
    total_ms = start.elapsed_time(stop)
    rope_ms = [e[0].elapsed_time(e[1]) for e in events]
    attn_ms = [e[1].elapsed_time(e[2]) for e in events]
    dec_us = [[1e3 * e[2 + i].elapsed_time(e[3 + i]) for e in events] for i in range(nL)]

    flops = W.prefill_flops(w)
    prefill_ms = statistics.mean(r + a for r, a in zip(rope_ms, attn_ms))
    value = replica_throughput(flops, prefill_ms, world) / 1e12
    total_ms = max_over_ranks(total_ms, world)
    attn_mean = statistics.mean(attn_ms)
    achieved = flops / (attn_mean * 1e-3) / 1e12
    peaks, peak_src = measured_peaks()
    peak_tf = float(peaks.get("bf16_tflops", 1800.0))
    peak_tf_sus = float(peaks.get("bf16_tflops_sustained", 1400.0))
    hbm = float(peaks.get("hbm_gbs", 6400.0))

    dec = {"lengths": list(dw.lengths), "G": [jl.group_size(L, dw.w_pretrained) for L in dw.lengths],
           "us": [], "gbs": [], "tokens_per_s": [], "frac_of_measured_hbm": [],
           "frac_of_8tbs": [], "bytes": []}
    for i, L in enumerate(dw.lengths):
        us = statistics.median(dec_us[i])
        nbytes = W.decode_bytes(L, dw.Hkv, dw.d, dw.Hq, dw.B)
        gbs = nbytes / (us * 1e-6) / 1e9
        dec["us"].append(round(us, 2))
        dec["gbs"].append(round(gbs, 1))
        dec["bytes"].append(nbytes)
        dec["tokens_per_s"].append(round(dw.B / (us * 1e-6), 1))
        dec["frac_of_measured_hbm"].append(round(gbs / hbm, 4))
        dec["frac_of_8tbs"].append(round(gbs / 8000.0, 4))

    # Decode alone, away from the prefill (whose power draw and dirty L2
    # lines slow the first decodes of a step): 20 calls at one length
    # captured in a CUDA graph and replayed, so host call overhead is not
    # timed.  Consecutive calls alternate between two copies of the cache
    # (each at least 134 MB of keys and values, above the 126 MB L2), so no
    # call is served from lines its predecessor left in L2.
    dec["us_alone"], dec["gbs_alone"], dec["frac_alone_of_measured_hbm"] = [], [], []
    n_rep = 20
    caches = [(kc, vc), (kc.clone(), vc.clone())]
    for i, L in enumerate(dw.lengths):
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for r in range(3):  # warm-up on the capture stream
                kx, vx = caches[r % 2]
                jl.decode(qs[i], kx, vx, L, dw.w0, dw.w_pretrained, dw.theta, out=od, lse=lsed,
                          workspace=dws)
        side.synchronize()
        with torch.cuda.graph(graph):
            for r in range(n_rep):
                kx, vx = caches[r % 2]
                jl.decode(qs[i], kx, vx, L, dw.w0, dw.w_pretrained, dw.theta, out=od, lse=lsed,
                          workspace=dws)
        graph.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            reps.append(1e3 * a.elapsed_time(b) / n_rep)
        us = statistics.median(reps)
        gbs = dec["bytes"][i] / (us * 1e-6) / 1e9
        dec["us_alone"].append(round(us, 2))
        dec["gbs_alone"].append(round(gbs, 1))
        dec["frac_alone_of_measured_hbm"].append(round(gbs / hbm, 4))
    jl.device_status()
    del caches

    e2e = run_e2e(jl, q, k, v, w, dev, args.steps, args.warmup, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, dt, pairs, cores = oracle_sample(128)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"fp64 oracle, 4x-extension prefill: 128 seeded query rows of head 0 "
                         f"({pairs} causal pairs) in {dt:.1f} s, RoPE tables included"}
    traffic = load_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16)", "config": config_dict(),
        "pct_bf16_peak": round(value / world / peak_tf, 4),
        "prefill_ms": round(prefill_ms, 3), "rope_ms": round(statistics.mean(rope_ms), 3),
        "attention_ms": round(attn_mean, 3),
        "decode": dec,
        "roofline": {"bound": "tensor", "kernel": "prefill attention", "achieved": round(achieved, 1),
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "traffic": traffic, "peak_source": f"{peak_src} bf16_tflops (burst)",
                     # the step loop runs for seconds under the power cap: the
                     # sustained GEMM figure is the like-for-like denominator
                     "peak_sustained": peak_tf_sus, "frac_of_sustained": round(achieved / peak_tf_sus, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (KERNELS_PER_PREFILL + nL * KERNELS_PER_DECODE),
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(jl, q, k, v, w, dev, steps, warmup, world):
    """Same metric through the public host-buffer call: jl_bifocal_prefill_host
    copies pinned q, k, v in and o, lse out itself (pipelined by query
    chunks), all inside the timed region; `warmup` untimed calls, then
    `steps` timed ones."""
    import torch
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((w.B, w.Hq, w.L), dtype=torch.float32).pin_memory()
    ws = jl.alloc_workspace(jl.load().jl_bifocal_prefill_host_workspace_size(
        w.B, w.L, w.Hq, w.Hkv, w.d, w.w_pretrained), dev)
    stream = torch.cuda.current_stream()

    def once():
        jl.prefill_host(qh, kh, vh, w.w0, w.w_pretrained, w.theta, out=oh, lse=lh, workspace=ws)

    for _ in range(warmup):
        once()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        once()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return {"value": world * W.prefill_flops(w) / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "call": "jl_bifocal_prefill_host (pinned host buffers, copies pipelined with the kernels)"}


def run_profile_prefill(args):
    """Small-case prefill for ncu captures: same heads, d, w0, w_pretrained and
    theta as the 4x-extension workload, sequence length from the flag."""
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    w = PREFILL
    L = int(args.profile_prefill)
    wp = int(args.profile_wp) if args.profile_wp else w.w_pretrained
    dev = torch.device("cuda", 0)
    q, k, v = synth.prefill_inputs(L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = jl.alloc_workspace(jl.prefill_workspace_size(1, L, w.Hq, w.Hkv, w.d, wp), dev)
    for _ in range(args.warmup):
        jl.prefill(qd, kd, vd, w.w0, wp, w.theta, workspace=ws)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        jl.prefill(qd, kd, vd, w.w0, wp, w.theta, workspace=ws)
    b.record()
    torch.cuda.synchronize()
    jl.device_status()
    ms = a.elapsed_time(b) / args.steps
    flops = 4.0 * w.d * (L * (L + 1) // 2) * w.Hq
    print(json.dumps({"profile_prefill_L": L, "w_pretrained": wp, "G": jl.group_size(L, wp), "ms": ms,
                      "tflops": flops / (ms * 1e-3) / 1e12}))
    return 0


def run_profile_three_pass(args):
    """A/B of the two forms of the same prefill on the 4x-extension shapes at
    sequence length L: the routed single pass against the three-pass
    inclusion-exclusion form (two window passes, one full aliased pass, one
    merge).  Reports both times, the single pass's algorithmic TFLOP/s for
    each, and the largest difference between their outputs."""
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    w = PREFILL
    L = int(args.profile_three_pass)
    dev = torch.device("cuda", 0)
    q, k, v = synth.prefill_inputs(L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws1 = jl.alloc_workspace(jl.prefill_workspace_size(1, L, w.Hq, w.Hkv, w.d, w.w_pretrained), dev)
    ws3 = jl.alloc_workspace(jl.load().jl_bifocal_prefill_three_pass_workspace_size(
        1, L, w.Hq, w.Hkv, w.d, w.w_pretrained), dev)
    runs = {"single": lambda: jl.prefill(qd, kd, vd, w.w0, w.w_pretrained, w.theta, workspace=ws1),
            "three_pass": lambda: jl.prefill_three_pass(qd, kd, vd, w.w0, w.w_pretrained, w.theta,
                                                        workspace=ws3)}
    flops = 4.0 * w.d * (L * (L + 1) // 2) * w.Hq
    res, outs = {}, {}
    for name, run in runs.items():
        for _ in range(args.warmup):
            outs[name] = run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            run()
        b.record()
        torch.cuda.synchronize()
        jl.device_status()
        ms = a.elapsed_time(b) / args.steps
        res[name] = {"ms": round(ms, 3), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
    (o1, l1), (o3, l3) = outs["single"], outs["three_pass"]
    do = (o1.float() - o3.float()).abs()
    print(json.dumps({"profile_three_pass_L": L, "G": jl.group_size(L, w.w_pretrained), **res,
                      "ratio_three_over_single": round(res["three_pass"]["ms"] / res["single"]["ms"], 3),
                      "o_maxabs_diff": float(do.max()), "o_meanabs_diff": float(do.mean()),
                      "lse_maxabs_diff": float((l1 - l3).abs().max())}))
    return 0


def run_profile_cta_pair(args):
    """A/B of the two attention kernels on the 4x-extension shapes at sequence
    length L (pretrained length from --profile-wp, else the workload's): the
    default single-CTA kernel (jl_bifocal_attention) against the CTA-pair
    kernel (jl_bifocal_attention_cta_pair), both after one jl_bifocal_rope
    into the same workspace, interleaved per round; min over rounds."""
    import ctypes
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    from bifocal_rope_extension_causal_b300 import _capi
    w = PREFILL
    L = int(args.profile_cta_pair)
    wp = int(args.profile_wp) if args.profile_wp else w.w_pretrained
    dev = torch.device("cuda", 0)
    q, k, v = synth.prefill_inputs(L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    nbytes = jl.prefill_workspace_size(1, L, w.Hq, w.Hkv, w.d, wp)
    ws = jl.alloc_workspace(nbytes, dev)
    lib, P = _capi.load(), ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    _capi.check(lib.jl_bifocal_rope(P(qd.data_ptr()), P(kd.data_ptr()), 1, L, w.Hq, w.Hkv, w.d, wp, w.theta, None,
                                    P(ws.data_ptr()), nbytes, stream))
    outs = {n: (torch.empty_like(qd), torch.empty((1, w.Hq, L), dtype=torch.float32, device=dev))
            for n in ("single_cta", "cta_pair")}
    fns = {"single_cta": lib.jl_bifocal_attention, "cta_pair": lib.jl_bifocal_attention_cta_pair}

    def run(name):
        o, lse = outs[name]
        _capi.check(fns[name](P(vd.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()), 1, L, w.Hq, w.Hkv, w.d, w.w0,
                              wp, 0.0, P(ws.data_ptr()), nbytes, stream))

    for _ in range(args.warmup):
        for name in fns:
            run(name)
    torch.cuda.synchronize()
    times = {n: [] for n in fns}
    for _ in range(args.steps):
        for name in fns:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run(name)
            b.record()
            torch.cuda.synchronize()
            times[name].append(a.elapsed_time(b))
    jl.device_status()
    flops = 4.0 * w.d * (L * (L + 1) // 2) * w.Hq
    res = {}
    for name in fns:
        ms = min(times[name])
        res[name] = {"ms": round(ms, 3), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
    (o1, l1), (o2, l2) = outs["single_cta"], outs["cta_pair"]
    print(json.dumps({"profile_cta_pair_L": L, "w_pretrained": wp, "G": jl.group_size(L, wp), **res,
                      "o_maxabs_diff": float((o1.float() - o2.float()).abs().max()),
                      "lse_maxabs_diff": float((l1 - l2).abs().max())}))
    return 0


def run_profile_decode(args):
    """Decode steps of the decode workload at one cache length, for ncu."""
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    dw = DECODE
    L = int(args.profile_decode)
    dev = torch.device("cuda", 0)
    kc, vc, qs = synth.decode_inputs(dw.Lcap, dw.Hq, dw.Hkv, dw.d, dw.index, 1)
    kc, vc, q = kc.to(dev), vc.to(dev), qs[0].to(dev)
    ws = jl.alloc_workspace(jl.decode_workspace_size(dw.B, dw.Hq, dw.d, dw.Lcap), dev)
    o = torch.empty((dw.B, dw.Hq, dw.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((dw.B, dw.Hq), dtype=torch.float32, device=dev)
    run = lambda: jl.decode(q, kc, vc, L, dw.w0, dw.w_pretrained, dw.theta, out=o, lse=lse, workspace=ws)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        run()
    b.record()
    torch.cuda.synchronize()
    jl.device_status()
    us = 1e3 * a.elapsed_time(b) / args.steps
    nbytes = W.decode_bytes(L, dw.Hkv, dw.d, dw.Hq, dw.B)
    print(json.dumps({"profile_decode_L": L, "G": jl.group_size(L, dw.w_pretrained), "us": us,
                      "gbs": nbytes / (us * 1e-6) / 1e9}))
    return 0


def run_profile_decode_varlen(args):
    """Batched decode with per-sequence lengths: B sequences of the decode
    workload's head layout, lengths spread over [L/2, L], one call per step
    (jl_bifocal_decode_varlen), timed as CUDA-graph replays."""
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    dw = DECODE
    B, L = (int(x) for x in args.profile_decode_varlen)
    dev = torch.device("cuda", 0)
    kc, vc, qs = synth.decode_inputs(L, dw.Hq, dw.Hkv, dw.d, dw.index, 1, B=B)
    kc, vc, q = kc.to(dev), vc.to(dev), qs[0].to(dev)
    lengths = [L - (L // 2) * i // max(1, B - 1) for i in range(B)]
    seq = torch.tensor(lengths, dtype=torch.int32, device=dev)
    ws = jl.alloc_workspace(jl.decode_workspace_size(B, dw.Hq, dw.d, L), dev)
    o = torch.empty((B, dw.Hq, dw.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, dw.Hq), dtype=torch.float32, device=dev)
    run = lambda: jl.decode_varlen(q, kc, vc, seq, dw.w0, dw.w_pretrained, dw.theta, max_len=L, out=o, lse=lse,
                                   workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(max(3, args.warmup)):
            run()
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            run()
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    graph.replay()
    b.record()
    torch.cuda.synchronize()
    jl.device_status()
    us = 1e3 * a.elapsed_time(b) / args.steps
    nbytes = sum(W.decode_bytes(n, dw.Hkv, dw.d, dw.Hq) for n in lengths)
    print(json.dumps({"profile_decode_varlen_B": B, "max_len": L, "lengths": lengths, "us": round(us, 2),
                      "gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "tokens_per_s": round(B / (us * 1e-6), 1)}))
    return 0


def run_profile_chunked(args):
    """Chunked prefill of one sequence: every chunk attends to the cache
    filled by the chunks before it.  Reports the per-chunk times and the
    causal-pair TFLOP/s of the whole sequence."""
    import torch
    import bifocal_rope_extension_causal_b300 as jl
    w = PREFILL
    L, C = (int(x) for x in args.profile_chunked)
    dev = torch.device("cuda", 0)
    q, k, v = synth.prefill_inputs(L, w.Hq, w.Hkv, w.d, w.index)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kc = torch.empty((1, L, w.Hkv, w.d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    ws = jl.alloc_workspace(max(jl.load().jl_bifocal_prefill_chunk_workspace_size(1, C, P0, w.Hq, w.Hkv, w.d,
                                                                                   w.w_pretrained)
                                for P0 in range(0, L, C)), dev)
    starts = list(range(0, L, C))
    outs = [(torch.empty((1, min(C, L - s), w.Hq, w.d), dtype=torch.bfloat16, device=dev),
             torch.empty((1, w.Hq, min(C, L - s)), dtype=torch.float32, device=dev)) for s in starts]

    def sweep(events=None):
        for i, s0 in enumerate(starts):
            e = min(L, s0 + C)
            if events:
                events[i].record()
            jl.prefill_chunk(qd[:, s0:e], kd[:, s0:e], vd[:, s0:e], kc, vc, s0, w.w0, w.w_pretrained, w.theta,
                             out=outs[i][0], lse=outs[i][1], workspace=ws)
        if events:
            events[-1].record()

    for _ in range(args.warmup):
        sweep()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(starts) + 1)]
        sweep(ev)
        torch.cuda.synchronize()
        times.append([ev[i].elapsed_time(ev[i + 1]) for i in range(len(starts))])
    jl.device_status()
    per_chunk = [min(t[i] for t in times) for i in range(len(starts))]
    total = sum(per_chunk)
    flops = 4.0 * w.d * (L * (L + 1) // 2) * w.Hq
    print(json.dumps({"profile_chunked_L": L, "C": C, "chunk_ms": [round(x, 3) for x in per_chunk],
                      "total_ms": total, "tflops": flops / (total * 1e-3) / 1e12,
                      "G_per_chunk": [jl.group_size(min(L, s + C), w.w_pretrained) for s in starts]}))
    return 0


def load_traffic():
    """DRAM bytes per attention launch from the committed ncu capture
    (profiles/prefill_attention_traffic.json), or None if the kernel sources
    changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "prefill_attention_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return d["bytes_per_full_launch"] if h.hexdigest() == d["sources_sha256"] else None
    except (OSError, ValueError, KeyError):
        return None


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-decode", type=int, default=0, metavar="L",
                    help="profiling mode: only decode steps of the decode workload at cache length L")
    ap.add_argument("--profile-chunked", type=int, nargs=2, default=None, metavar=("L", "C"),
                    help="measurement mode: the 4x-extension head layout prefilled in chunks of C "
                         "tokens up to L against the cache (one G per chunk from its total length)")
    ap.add_argument("--profile-decode-varlen", type=int, nargs=2, default=None, metavar=("B", "L"),
                    help="profiling mode: batched decode of B sequences, lengths spread over [L/2, L]")
    ap.add_argument("--profile-three-pass", type=int, default=0, metavar="L",
                    help="A/B mode: single-pass vs three-pass prefill at sequence length L")
    ap.add_argument("--profile-prefill", type=int, default=0, metavar="L",
                    help="profiling mode: only the prefill of the 4x-extension head layout at "
                         "sequence length L (G from L), warm-up + steps calls; prints timings")
    ap.add_argument("--profile-cta-pair", type=int, default=0, metavar="L",
                    help="profiling mode: A/B of the single-CTA and CTA-pair attention kernels on the "
                         "4x-extension head layout at sequence length L; prints both timings")
    ap.add_argument("--profile-wp", type=int, default=0, metavar="W",
                    help="with --profile-prefill or --profile-cta-pair: pretrained length W instead of the workload's "
                         "(G = ceil(L / W); small L with G > 1 exercises the remote phase)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_prefill:
        return run_profile_prefill(args)
    if args.profile_cta_pair:
        return run_profile_cta_pair(args)
    if args.profile_three_pass:
        return run_profile_three_pass(args)
    if args.profile_decode_varlen:
        return run_profile_decode_varlen(args)
    if args.profile_decode:
        return run_profile_decode(args)
    if args.profile_chunked:
        return run_profile_chunked(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

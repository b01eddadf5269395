#!/usr/bin/env python3
"""Benchmark of the cross-token gate aggregation path on GB300.

One step = one TANGO block forward (RMSNorm -> projection GEMM with RoPE/norm/SiLU
epilogues -> TANGO aggregation -> W_o GEMM + residual) at the 70M-tier shape
B=8, T=2048, d=512, m=28480, q/k width 128 (2 heads of 64), bf16 storage, fp32
accumulation, through the C ABI (tango_block_forward).

Printed: ONE JSON line (rank 0).  `value` = tokens/s of the whole job with inputs
resident in HBM; `e2e` = the same through the C ABI with pinned host buffers and every
step's host<->device copies inside the timed region (on a second stream, overlapping the
neighbouring steps' compute); `roofline` = the TANGO aggregation
kernel's algorithmic TFLOP/s against the measured bf16 peak; `cpu_baseline` = the
fp64 oracle on the host cores on a bounded sample.  `also` carries the WANGO and
long-context aggregation measurements.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "aggregation tokens/s and TFLOP/s at T=2k/8k on 1 GB300; % of BF16 tensor-core roofline"
B, T, D, DQK, M, H = 8, 2048, 512, 128, 28480, 2
WORKLOAD = f"TANGO block forward (RMSNorm, q/k/g/v projections, full-prefix aggregation, W_o + residual), " \
           f"B={B} T={T} d={D} m={M} q/k width {DQK} (H={H}, d_h=64), s=10, bf16"
KERNELS_PER_STEP = 4  # rmsnorm, projection GEMM, TANGO aggregation, output GEMM


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true")
    ap.add_argument("--agg-only", choices=["tango", "wango"],
                    help="only run one aggregation kernel (for profiler captures)")
    ap.add_argument("--block-only", action="store_true",
                    help="only run the block forward at batch --agg-B (for profiler captures)")
    ap.add_argument("--decode-only", action="store_true",
                    help="only run WANGO decode steps (W=256) for --agg-B sequences: W + --agg-iters "
                         "steps (for profiler captures)")
    ap.add_argument("--bwd-only", choices=["tango", "wango"],
                    help="only run one aggregation backward at --agg-B, --agg-T (for profiler captures)")
    ap.add_argument("--agg-B", type=int, default=2)
    ap.add_argument("--agg-T", type=int, default=2048)
    ap.add_argument("--agg-iters", type=int, default=3)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_rate(local_ms: float, units_per_rank: float, world: int, device) -> tuple:
    """The job's step time and rate: every rank does `units_per_rank` per step and the job
    is as slow as its slowest rank, so the step time is the maximum over ranks (one
    all-reduce when world > 1) and the rate counts every rank's units."""
    import torch
    t = torch.tensor([local_ms], device=device, dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * units_per_rank / (ms_max * 1e-3)


def measured_traffic(kernel: str, source: str, B_: int, T_: int):
    """DRAM bytes per launch of `kernel` at (B_, T_) from the committed ncu summary
    profiles/traffic.json, or None when there is none or the kernel's source has
    changed since the counters were taken (its SHA-256 is recorded beside them)."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
        src = open(os.path.join(ROOT, "cross_token_gated_gb300", "csrc", source), "rb").read()
        if hashlib.sha256(src).hexdigest() != rec["source_sha256"]:
            return None
        # captured on a smaller batch; DRAM traffic of this kernel grows in proportion to B
        return rec["dram_bytes_per_launch"] * B_ / rec["B"] if rec["T"] == T_ else None
    except Exception:
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return p["bf16_tflops"], p["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


def sustained_peak():
    """The bf16 GEMM rate measured back to back under the power cap, or None."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops_sustained"])
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for nm, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_cpu_baseline(max_seconds: float = 30.0):
    """The fp64 oracle on the host cores: one block forward over the first Tc positions of
    the first nb sequences (causality makes those outputs depend on those positions only).
    Tc grows from 128 to T, then nb from 1 to B, while the sample stays within the budget
    (about 10-30 s of CPU work)."""
    import oracle
    from cross_token_gated_gb300 import synth
    h, w = synth.block_inputs(B, T, D, DQK, M, seed=0, dtype="bf16")
    wv = {n: synth.oracle_view(t) for n, t in w.items()}
    hv = synth.oracle_view(h)
    Tc, nb, spent, result = 128, 1, 0.0, None
    while True:
        t0 = time.perf_counter()
        oracle.block_forward(hv[:nb, :Tc], wv, H=H, tau=10.0, mode=0, window=1)
        dt = time.perf_counter() - t0
        spent += dt
        result = (Tc, nb, dt)
        # the next size costs ~2.5x (longer: projections plus the quadratic pair term) or
        # 2x (more sequences)
        if Tc * 2 <= T:
            if spent + 2.5 * dt > max_seconds:
                break
            Tc *= 2
        elif nb * 2 <= B:
            if spent + 2.0 * dt > max_seconds:
                break
            nb *= 2
        else:
            break
    Tc, nb, dt = result
    return {"value": nb * Tc / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"block forward of sequences 0..{nb - 1}, positions 0..{Tc - 1} (T={Tc} of {T}), "
                      f"{dt:.2f} s, fp64"}


def run_reference(args, rank, world):
    """The oracle timed as it stands on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from cross_token_gated_gb300 import synth
    h, w = synth.block_inputs(1, T, D, DQK, M, seed=0, dtype="bf16")
    wv = {n: synth.oracle_view(t) for n, t in w.items()}
    hv = synth.oracle_view(h)
    # each step is a bounded sample: the first Tc positions of sequence 0, Tc the largest
    # power of two that keeps the whole --steps/--warmup run within about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    Tc = 16
    t0 = time.perf_counter()
    oracle.block_forward(hv[:, :Tc], wv, H=H, tau=10.0)
    per_tok = (time.perf_counter() - t0) / Tc
    while Tc * 2 <= T and per_tok * Tc * 2 <= budget:
        Tc *= 2
    for _ in range(args.warmup):
        oracle.block_forward(hv[:, :Tc], wv, H=H, tau=10.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.block_forward(hv[:, :Tc], wv, H=H, tau=10.0)
    dt = (time.perf_counter() - t0) / args.steps
    val = Tc / dt
    sample = f"each step: block forward of sequence 0, positions 0..{Tc - 1}, fp64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_T": Tc},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.agg_only:
        run_agg_only(args)
        return
    if args.bwd_only:
        run_bwd_only(args)
        return
    if args.block_only:
        run_block_only(args)
        return
    if args.decode_only:
        run_decode_only(args)
        return
    import torch
    import torch.distributed as dist

    import cross_token_gated_gb300 as tg
    from cross_token_gated_gb300 import accounting as acc
    from cross_token_gated_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    tg.load()
    peak_tf, peak_gbs, peak_src = peaks()

    # ---------------------------------------------------------------- inputs
    h, w = synth.block_inputs(B, T, D, DQK, M, seed=rank, dtype="bf16")
    hd = h.to(dev)
    wd = {n: t.to(dev) for n, t in w.items()}
    out = torch.empty_like(hd)
    ws = tg.block_workspace(B, T, D, H, DQK, M, dtype=tg.TG_BF16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        tg.tango_block_forward(hd, wd, out, H=H, ws=ws, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(args.warmup, 3)):
        step()
    st, word = tg.tg_check_device_error(stream)
    if st != tg.TG_OK:
        raise RuntimeError(f"device error after warm-up: {tg.status_string(st)} ({word:#x})")

    # ------------------------------------------------------------- timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
    ms = e0.elapsed_time(e1) / args.steps
    clocks = clk.summary()
    ms_max, value = job_rate(ms, B * T, world, dev)
    st, word = tg.tg_check_device_error(stream)
    if st != tg.TG_OK:
        raise RuntimeError(f"device error in timed region: {tg.status_string(st)} ({word:#x})")

    # ------------------------------------------ dominant kernel: TANGO aggregation
    # The aggregation kernel re-run on the step's own projected q/k/g and u (the
    # workspace regions x, q, k, g, v in that order, each 256-byte aligned, as
    # tango.h documents), timed with events on the same stream.
    L = {"q": 0, "k": 0, "g": 0, "v": 0}
    es = 2
    off = 0
    sz = {"x": B * T * D, "q": B * T * DQK, "k": B * T * DQK, "g": B * T * M, "v": B * T * M}
    base = (ws.data_ptr() + 255) & ~255
    for name in ("x", "q", "k", "g", "v"):
        L[name] = base + off
        off += (sz[name] * es + 255) & ~255
    agg_out = torch.empty(B, T, M, dtype=torch.bfloat16, device=dev)

    def agg_once():
        p = tg.agg_params(B, T, H, DQK, M, dtype=tg.TG_BF16, s=10.0, flags=tg.TG_FLAG_QK_NORMALIZED)
        r = tg.load().tango_aggregate(ctypes.byref(p), L["q"], L["k"], L["g"], L["v"],
                                      agg_out.data_ptr(), None, 0, stream.cuda_stream)
        if r != tg.TG_OK:
            raise tg.TgError(r, "tango_aggregate")

    step()  # refresh the workspace (v was overwritten by gbar * v)
    for _ in range(3):
        agg_once()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(5, args.steps // 2)
    k0.record(stream)
    for _ in range(reps):
        agg_once()
    k1.record(stream)
    torch.cuda.synchronize(dev)
    agg_ms = k0.elapsed_time(k1) / reps
    agg_flops = acc.tango_agg_flops(B, T, DQK, M)
    achieved = agg_flops / (agg_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": measured_traffic("tango_tc_kernel", "tango_tc.cu", B, T),
                "kernel": "tango_tc_kernel", "kernel_ms": agg_ms,
                "algorithmic_flops_per_launch": agg_flops,
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    sus = sustained_peak()
    if sus:  # context: the step runs at the power cap, where the GEMM itself sustains less
        roofline["sustained_peak"] = sus
        roofline["frac_of_sustained"] = achieved / sus

    # ------------------------------------------------------------------ e2e
    # Every step uploads its input from pinned host memory and reads its result back.
    # The copies run on a second stream with two device buffers each way, so step k+1's
    # upload and step k's download overlap step k's block forward, as a serving loop
    # would run them; every copy of every step stays inside the timed region.
    h_host = h.pin_memory()
    o_host = [torch.empty_like(h_host).pin_memory() for _ in range(2)]
    hbuf, obuf = [hd, torch.empty_like(hd)], [out, torch.empty_like(out)]
    cstream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    up, done, down = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n):
        with torch.cuda.stream(cstream):
            hbuf[0].copy_(h_host, non_blocking=True)
            up[0].record(cstream)
        for k in range(n):
            b = k % 2
            stream.wait_event(up[b])
            if k >= 2:
                stream.wait_event(down[b])  # step k-2's result has left obuf[b]
            tg.tango_block_forward(hbuf[b], wd, obuf[b], H=H, ws=ws, stream=stream)
            done[b].record(stream)
            with torch.cuda.stream(cstream):
                if k + 1 < n:
                    if k >= 1:
                        cstream.wait_event(done[1 - b])  # step k-1 has read hbuf[1-b]
                    hbuf[1 - b].copy_(h_host, non_blocking=True)
                    up[1 - b].record(cstream)
                cstream.wait_event(done[b])
                o_host[b].copy_(obuf[b], non_blocking=True)
                down[b].record(cstream)
        stream.wait_stream(cstream)

    e2e_run(4)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    cstream.wait_event(f0)
    e2e_run(args.steps)
    f1.record(stream)
    barrier()
    e2e_ms = f0.elapsed_time(f1) / args.steps
    # the pipelined copies delivered the right result: the last download equals a plain
    # step on the same input, bit for bit (the kernels are deterministic)
    step()
    barrier()
    if not torch.equal(o_host[(args.steps - 1) % 2].to(dev), out):
        raise RuntimeError("pipelined e2e result differs from the plain step")
    e2e = {"value": job_rate(e2e_ms, B * T, world, dev)[1], "unit": "tokens/s",
           "h2d_bytes_per_step": h_host.numel() * 2, "d2h_bytes_per_step": o_host[0].numel() * 2,
           "copies": "second stream, double-buffered, overlapping the neighbouring steps"}

    # -------------------------------------------- other configurations (context)
    also = {}
    if rank == 0 and not args.no_also:
        also = other_configs(tg, acc, dev, stream, peak_tf, peak_gbs)

    step_flops = acc.block_flops(B, T, D, DQK, M)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": T, "d": D, "m": M,
                       "qk_width": DQK, "heads": H, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (g, v are 0.93 GB each)"},
            "step_tflops": step_flops / (ms_max * 1e-3) / 1e12,
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clocks,
            "also": also,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_cpu_baseline()
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def event_ms(f, dev, stream, reps=5, warm=3):
    """Mean device time of f() over `reps` calls, CUDA events on `stream`, after `warm`
    untimed calls."""
    import torch
    for _ in range(warm):
        f()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        f()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def kernel_breakdown(f, dev):
    """Per-kernel device time of one call of f(), from the CUDA profiler's activity
    records (CUPTI): {kernel: {"launches", "ms", "share"}}.  Shares of one call; the
    call's own time is taken separately, without the profiler."""
    import torch
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize(dev)
        for _ in range(2):  # the first session of a process can come back empty: it warms up
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                f()
                torch.cuda.synchronize(dev)
        rows = {}
        for ev in prof.key_averages():
            us = getattr(ev, "self_device_time_total", None)
            if us is None:
                us = getattr(ev, "self_cuda_time_total", 0.0)
            if not us or ev.key.startswith(("cudaLaunch", "cuda", "Memcpy", "Memset")):
                continue
            name = ev.key.replace("(anonymous namespace)::", "").replace("void ", "").replace("tg::", "")
            name = name.split("(")[0].split("<")[0].strip()
            r = rows.setdefault(name, {"launches": 0, "ms": 0.0})
            r["launches"] += int(ev.count)
            r["ms"] += us / 1e3
        total = sum(r["ms"] for r in rows.values()) or 1.0
        for r in rows.values():
            r["share"] = r["ms"] / total
        return dict(sorted(rows.items(), key=lambda kv: -kv[1]["ms"]))
    except Exception as exc:  # the profiler is context only
        return {"unavailable": str(exc)[:200]}


def other_configs(tg, acc, dev, stream, peak_tf, peak_gbs):
    """Context measurements beside the headline step, each event-timed on the device:
    - aggregation only (TANGO, and WANGO with W=256) at B=8 T=2048 and at B=1 over
      T = 1k, 2k, 4k, 8k, with each time's ratio to the T/2 point (the full prefix grows
      quadratically in T, the window linearly); unit-normalised q/k and N(0,1) g, v
      generated on the device;
    - the WANGO block step at B=8 T=2048 (W=256), with v from the projection GEMM and
      with v formed inside the aggregation (TG_FLAG_FUSED_V);
    - the shared-block model forward at B=16 T=1024 (4 TANGO applications, 32,768-entry
      tied embedding): one set of m=28,480 and three sets of m=9,494, with per-kernel
      device times;
    - WANGO decode steps (W=256) at B=1, 8 and 32, timed as one CUDA-graph replay of 64
      consecutive steps;
    - the backward of both aggregations at B=8 T=2048, with per-kernel device times,
      and with the gbar and denominators a saving forward keeps (a training step's
      aggregation: the saving forward plus that backward);
    - the WANGO backward at B=1 T=8192 with the saved forward, on the library's path
      (the running-sum scans for the far older pairs) and on the pair-by-pair path."""
    import torch
    from cross_token_gated_gb300 import synth  # noqa: F401  (the recipe the weights follow)
    res = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)

    def unit(b, t_len):
        x = torch.randn(b, t_len, H, DQK // H, device=dev, generator=gen)
        return (x / x.norm(dim=-1, keepdim=True)).reshape(b, t_len, DQK).bfloat16()

    prev = {}
    for (b, t_len) in ((8, 2048), (1, 1024), (1, 2048), (1, 4096), (1, 8192)):
        q, k = unit(b, t_len), unit(b, t_len)
        g = torch.randn(b, t_len, M, device=dev, generator=gen).bfloat16()
        v = torch.randn(b, t_len, M, device=dev, generator=gen).bfloat16()
        o = torch.empty_like(g)
        for kind in ("tango", "wango"):
            if kind == "tango":
                f = lambda: tg.tango_aggregate(q, k, g, v, o, H=H, flags=tg.TG_FLAG_QK_NORMALIZED, stream=stream)
                fl = acc.tango_agg_flops(b, t_len, DQK, M)
            else:
                f = lambda: tg.wango_aggregate(q, k, g, v, o, H=H, window=256, flags=tg.TG_FLAG_QK_NORMALIZED,
                                               stream=stream)
                fl = acc.wango_agg_flops(b, t_len, DQK, M, H, 256)
            ms = event_ms(f, dev, stream)
            by = acc.agg_bytes(b, t_len, DQK, M)
            rec = {"ms": ms, "tokens_per_s": b * t_len / (ms * 1e-3),
                   "tflops": fl / (ms * 1e-3) / 1e12, "frac_bf16_peak": fl / (ms * 1e-3) / 1e12 / peak_tf,
                   "gbs": by / (ms * 1e-3) / 1e9, "frac_hbm_peak": by / (ms * 1e-3) / 1e9 / peak_gbs}
            if b == 1 and (kind, t_len // 2) in prev:
                rec["ratio_to_half_T"] = ms / prev[(kind, t_len // 2)]
            if b == 1:
                prev[(kind, t_len)] = ms
            res[f"{kind}_B{b}_T{t_len}"] = rec
        del q, k, g, v, o
        torch.cuda.empty_cache()
    res["t_sweep_B1"] = {kind: {str(t): prev[(kind, t)] for t in (1024, 2048, 4096, 8192)}
                         for kind in ("tango", "wango")}
    res["t_sweep_B1"]["unit"] = "ms"

    # ---- the aggregation backward (B=8, T=2048; WANGO with W=256)
    q, k = unit(B, T), unit(B, T)
    g = torch.randn(B, T, M, device=dev, generator=gen).bfloat16()
    v = torch.randn(B, T, M, device=dev, generator=gen).bfloat16()
    dout = torch.randn(B, T, M, device=dev, generator=gen).bfloat16()
    dq, dk, dg, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(g), torch.empty_like(g)
    u, gbar = torch.empty_like(g), torch.empty_like(g)
    den = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    nf = tg.TG_FLAG_QK_NORMALIZED
    for kind in ("tango", "wango"):
        which = tg.TG_WS_TANGO_BWD if kind == "tango" else tg.TG_WS_WANGO_BWD
        p = tg.agg_params(B, T, H, DQK, M, dtype=tg.TG_BF16, window=256, flags=nf)
        wsb = torch.empty(tg.tg_workspace_size(which, p) + 256, dtype=torch.uint8, device=dev)
        kw = {} if kind == "tango" else {"window": 256}
        bwd = tg.tango_aggregate_backward if kind == "tango" else tg.wango_aggregate_backward
        save = tg.tango_aggregate_save if kind == "tango" else tg.wango_aggregate_save
        f = lambda: bwd(q, k, g, v, dout, dq, dk, dg, dv, H=H, flags=nf, ws=wsb, stream=stream, **kw)
        fl = acc.tango_bwd_flops(B, T, DQK, M) if kind == "tango" else acc.wango_bwd_flops(B, T, DQK, M, H, 256)
        ms = event_ms(f, dev, stream, reps=5)
        by = acc.agg_bwd_bytes(B, T, DQK, M)
        # a training step's aggregation: the forward that keeps gbar and the denominators,
        # then the backward that uses them (no recomputation)
        ms_save = event_ms(lambda: save(q, k, g, v, u, gbar, den, H=H, flags=nf, stream=stream, **kw), dev, stream,
                           reps=5)
        f_saved = lambda: bwd(q, k, g, v, dout, dq, dk, dg, dv, H=H, flags=nf, ws=wsb, stream=stream, gbar=gbar,
                              den=den, **kw)
        ms_saved = event_ms(f_saved, dev, stream, reps=5)
        res[f"{kind}_backward_B{B}_T{T}"] = {
            "ms": ms, "tokens_per_s": B * T / (ms * 1e-3), "tflops": fl / (ms * 1e-3) / 1e12,
            "frac_bf16_peak": fl / (ms * 1e-3) / 1e12 / peak_tf, "gbs": by / (ms * 1e-3) / 1e9,
            "algorithmic_tflop": fl / 1e12, "kernels": kernel_breakdown(f, dev),
            "ms_with_saved_forward": ms_saved,
            "frac_bf16_peak_with_saved_forward": fl / (ms_saved * 1e-3) / 1e12 / peak_tf,
            "forward_save_ms": ms_save, "training_step_ms": ms_save + ms_saved}
        del wsb
        torch.cuda.empty_cache()
    del q, k, g, v, dout, dq, dk, dg, dv, u, gbar, den
    torch.cuda.empty_cache()

    # ---- the WANGO backward at long context (B=1, T=8192, W=256): the older pairs beyond
    # the window's band go through the running-sum scans there (the library's choice),
    # timed beside the pair-by-pair path
    b1, t1 = 1, 8192
    q, k = unit(b1, t1), unit(b1, t1)
    g, v, dout = (torch.randn(b1, t1, M, device=dev, generator=gen).bfloat16() for _ in range(3))
    dq, dk, dg, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(g), torch.empty_like(g)
    u, gbar = torch.empty_like(g), torch.empty_like(g)
    den = torch.empty(b1, H, t1, dtype=torch.float32, device=dev)
    ms_save = event_ms(lambda: tg.wango_aggregate_save(q, k, g, v, u, gbar, den, H=H, window=256, flags=nf,
                                                       stream=stream), dev, stream, reps=5)
    rec = {"forward_save_ms": ms_save, "algorithmic_tflop": acc.wango_bwd_flops(b1, t1, DQK, M, H, 256) / 1e12}
    sizes = {}
    for name, ff in (("library", 0), ("scans", tg.TG_FLAG_BWD_FAR_SCAN), ("pairs", tg.TG_FLAG_BWD_FAR_PAIRS)):
        p = tg.agg_params(b1, t1, H, DQK, M, dtype=tg.TG_BF16, window=256, flags=nf | ff)
        sizes[name] = tg.tg_workspace_size(tg.TG_WS_WANGO_BWD, p)
        wsb = torch.empty(sizes[name] + 256, dtype=torch.uint8, device=dev)
        f_saved = lambda: tg.wango_aggregate_backward(q, k, g, v, dout, dq, dk, dg, dv, H=H, window=256,
                                                      flags=nf | ff, ws=wsb, stream=stream, gbar=gbar, den=den)
        rec[f"ms_with_saved_forward_{name}"] = event_ms(f_saved, dev, stream, reps=5)
        if name == "library":
            rec["kernels"] = kernel_breakdown(f_saved, dev)
        del wsb
        torch.cuda.empty_cache()
    rec["library_path"] = "scans" if sizes["library"] == sizes["scans"] else "pairs"
    rec["training_step_ms"] = ms_save + rec["ms_with_saved_forward_library"]
    res[f"wango_backward_B{b1}_T{t1}"] = rec
    del q, k, g, v, dout, dq, dk, dg, dv, u, gbar, den
    torch.cuda.empty_cache()

    # ---- the WANGO block step (B=8, T=2048, W=256)
    def block_weights(d, m, n_sets=1):
        n = lambda r, c: (torch.randn(r, c, device=dev, generator=gen) * c ** -0.5).bfloat16()
        base = {"gamma": torch.ones(d, device=dev).bfloat16(), "Wq": n(DQK, d), "Wk": n(DQK, d)}
        return [dict(base, Wg=n(m, d), Wv=n(m, d), Wo=n(d, m)) for _ in range(n_sets)]

    w = block_weights(D, M)[0]
    h = torch.randn(B, T, D, device=dev, generator=gen).bfloat16()
    out = torch.empty_like(h)
    wsb = tg.block_workspace(B, T, D, H, DQK, M, dtype=tg.TG_BF16, mode=tg.TG_MODE_WANGO, window=256, device=dev)
    f = lambda: tg.tango_block_forward(h, w, out, H=H, mode=tg.TG_MODE_WANGO, window=256, ws=wsb, stream=stream)
    ms = event_ms(f, dev, stream, reps=10)
    fl = acc.block_flops(B, T, D, DQK, M, mode=1, H=H, W=256)
    res[f"wango_block_B{B}_T{T}"] = {"ms": ms, "tokens_per_s": B * T / (ms * 1e-3),
                                     "tflops": fl / (ms * 1e-3) / 1e12, "kernels": kernel_breakdown(f, dev)}
    # the same step with v = W_v x formed inside the aggregation kernel (TG_FLAG_FUSED_V)
    f = lambda: tg.tango_block_forward(h, w, out, H=H, mode=tg.TG_MODE_WANGO, window=256, flags=tg.TG_FLAG_FUSED_V,
                                       ws=wsb, stream=stream)
    ms = event_ms(f, dev, stream, reps=10)
    res[f"wango_block_fused_v_B{B}_T{T}"] = {"ms": ms, "tokens_per_s": B * T / (ms * 1e-3),
                                             "tflops": fl / (ms * 1e-3) / 1e12, "kernels": kernel_breakdown(f, dev)}
    del w, h, out, wsb
    torch.cuda.empty_cache()

    # ---- the shared-block model forward (B=16, T=1024, 4 applications, vocab 32,768)
    Bm, Tm, V = 16, 1024, 32768
    E = (torch.randn(V, D, device=dev, generator=gen) * 0.02).bfloat16()
    gam_f = torch.ones(D, device=dev).bfloat16()
    ids = torch.randint(0, V, (Bm, Tm), device=dev, generator=gen, dtype=torch.int32)
    logits = torch.empty(Bm, Tm, V, device=dev, dtype=torch.bfloat16)
    for m_set, n_sets in ((M, 1), (9494, 3)):
        sets = block_weights(D, m_set, n_sets)
        mp = tg.model_params(Bm, Tm, D, H, DQK, m_set, V, dtype=tg.TG_BF16, n_apps=4, n_sets=n_sets)
        wsm = torch.empty(tg.tg_workspace_size(tg.TG_WS_MODEL, mp) + 256, dtype=torch.uint8, device=dev)
        f = lambda: tg.tango_model_forward(ids, E, gam_f, sets, logits, H=H, n_apps=4, ws=wsm, stream=stream)
        ms = event_ms(f, dev, stream, reps=5)
        fl = acc.model_flops(Bm, Tm, D, DQK, m_set, V, 4)
        res[f"model_B{Bm}_T{Tm}_sets{n_sets}_m{m_set}"] = {
            "ms": ms, "tokens_per_s": Bm * Tm / (ms * 1e-3), "tflops": fl / (ms * 1e-3) / 1e12,
            "frac_bf16_peak": fl / (ms * 1e-3) / 1e12 / peak_tf, "algorithmic_tflop": fl / 1e12,
            "kernels": kernel_breakdown(f, dev)}
        del sets, wsm
        torch.cuda.empty_cache()
    del E, ids, logits

    # ---- WANGO decode steps (W=256), steady state, one graph replay of 64 steps
    for b in (1, 8, 32):
        Wd, n = 256, 64
        q, k = unit(b, 1)[:, 0].contiguous(), unit(b, 1)[:, 0].contiguous()
        g = torch.randn(b, M, device=dev, generator=gen).bfloat16()
        v = torch.randn(b, M, device=dev, generator=gen).bfloat16()
        o = torch.empty_like(g)
        st = tg.decode_state(b, H, DQK, M, window=Wd, dtype=tg.TG_BF16, device=dev)
        for pos in range(Wd + 8):
            tg.wango_decode_step(q, k, g, v, o, st, pos, H=H, window=Wd, flags=tg.TG_FLAG_QK_NORMALIZED,
                                 stream=stream)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(graph, stream=cap):
            for pos in range(Wd + 8, Wd + 8 + n):
                tg.wango_decode_step(q, k, g, v, o, st, pos, H=H, window=Wd, flags=tg.TG_FLAG_QK_NORMALIZED,
                                     stream=cap)
        graph.replay()  # a first replay warms the graph (its upload and the caches)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) / n * 1e3
        by = acc.decode_bytes(b, DQK, M, H, Wd)
        res[f"decode_B{b}_W{Wd}"] = {"us_per_step": us, "tokens_per_s": b / (us * 1e-6),
                                     "gbs": by / (us * 1e-6) / 1e9, "frac_hbm_peak": by / (us * 1e-6) / 1e9 / peak_gbs,
                                     "timing": f"one CUDA-graph replay of {n} consecutive steps, after a warm-up replay"}
        del graph, q, k, g, v, o, st
        torch.cuda.empty_cache()

    st, word = tg.tg_check_device_error(stream)
    if st != tg.TG_OK:
        raise RuntimeError(f"device error in the context measurements ({word:#x})")
    return res


def run_agg_only(args):
    """A few launches of one aggregation kernel on a small case (B, T given), inputs
    larger than L2.  Used for profiler captures; prints one timing line."""
    import torch

    import cross_token_gated_gb300 as tg
    from cross_token_gated_gb300 import accounting as acc
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    b, t_len = args.agg_B, args.agg_T
    q = torch.randn(b, t_len, H, DQK // H, device=dev, generator=gen)
    q = (q / q.norm(dim=-1, keepdim=True)).reshape(b, t_len, DQK).bfloat16()
    k = torch.randn(b, t_len, H, DQK // H, device=dev, generator=gen)
    k = (k / k.norm(dim=-1, keepdim=True)).reshape(b, t_len, DQK).bfloat16()
    g = torch.randn(b, t_len, M, device=dev, generator=gen).bfloat16()
    v = torch.randn(b, t_len, M, device=dev, generator=gen).bfloat16()
    o = torch.empty_like(g)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.agg_iters):
        if args.agg_only == "tango":
            tg.tango_aggregate(q, k, g, v, o, H=H, flags=tg.TG_FLAG_QK_NORMALIZED)
        else:
            tg.wango_aggregate(q, k, g, v, o, H=H, window=256, flags=tg.TG_FLAG_QK_NORMALIZED)
    st, word = tg.tg_check_device_error()
    dt = (time.perf_counter() - t0) / args.agg_iters
    print(json.dumps({"agg_only": args.agg_only, "B": b, "T": t_len, "status": st, "word": word,
                      "wall_ms_per_launch": dt * 1e3}))
    if st != tg.TG_OK:
        sys.exit(1)


def run_bwd_only(args):
    """A few backward calls of one aggregation (W = 256 for WANGO) at --agg-B, --agg-T,
    for profiler captures; prints one timing line."""
    import torch

    import cross_token_gated_gb300 as tg
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    b, t_len = args.agg_B, args.agg_T

    def unit():
        x = torch.randn(b, t_len, H, DQK // H, device=dev, generator=gen)
        return (x / x.norm(dim=-1, keepdim=True)).reshape(b, t_len, DQK).bfloat16()
    q, k = unit(), unit()
    g, v, dout = (torch.randn(b, t_len, M, device=dev, generator=gen).bfloat16() for _ in range(3))
    dq, dk, dg, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(g), torch.empty_like(g)
    fn = tg.tango_aggregate_backward if args.bwd_only == "tango" else tg.wango_aggregate_backward
    kw = {} if args.bwd_only == "tango" else {"window": 256}
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.agg_iters):
        fn(q, k, g, v, dout, dq, dk, dg, dv, H=H, flags=tg.TG_FLAG_QK_NORMALIZED, **kw)
    st, word = tg.tg_check_device_error()
    dt = (time.perf_counter() - t0) / args.agg_iters
    print(json.dumps({"bwd_only": args.bwd_only, "B": b, "T": t_len, "status": st, "word": word,
                      "wall_ms_per_call": dt * 1e3}))
    if st != tg.TG_OK:
        sys.exit(1)


def run_decode_only(args):
    """W + --agg-iters WANGO decode steps (W = 256) for --agg-B sequences, so that the last
    steps run at steady state; prints one timing line for those last steps."""
    import torch

    import cross_token_gated_gb300 as tg
    from cross_token_gated_gb300 import synth
    dev = torch.device("cuda", 0)
    b, W = args.agg_B, 256
    q, k, g, v = (x[:, 0].contiguous().to(dev) for x in synth.agg_inputs(b, 1, DQK, M, seed=0, dtype="bf16"))
    out = torch.empty_like(g)
    st_buf = tg.decode_state(b, H, DQK, M, window=W, dtype=tg.TG_BF16, device=dev)
    for pos in range(W):
        tg.wango_decode_step(q, k, g, v, out, st_buf, pos, H=H, window=W)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for pos in range(W, W + args.agg_iters):
        tg.wango_decode_step(q, k, g, v, out, st_buf, pos, H=H, window=W)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / args.agg_iters
    st, word = tg.tg_check_device_error()
    print(json.dumps({"decode_only": True, "B": b, "W": W, "status": st, "word": word,
                      "wall_us_per_step": dt * 1e6}))
    if st != tg.TG_OK:
        sys.exit(1)


def run_block_only(args):
    """A few block forwards (TANGO) at batch --agg-B and T = --agg-T, for profiler
    captures of the GEMMs; prints one timing line."""
    import torch

    import cross_token_gated_gb300 as tg
    from cross_token_gated_gb300 import synth
    dev = torch.device("cuda", 0)
    b, t_len = args.agg_B, args.agg_T
    h, w = synth.block_inputs(b, t_len, D, DQK, M, seed=0, dtype="bf16")
    hd = h.to(dev)
    wd = {n: x.to(dev) for n, x in w.items()}
    out = torch.empty_like(hd)
    ws = tg.block_workspace(b, t_len, D, H, DQK, M, dtype=tg.TG_BF16, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.agg_iters):
        tg.tango_block_forward(hd, wd, out, H=H, ws=ws)
    st, word = tg.tg_check_device_error()
    dt = (time.perf_counter() - t0) / args.agg_iters
    print(json.dumps({"block_only": True, "B": b, "T": t_len, "status": st, "word": word,
                      "wall_ms_per_launch": dt * 1e3}))
    if st != tg.TG_OK:
        sys.exit(1)


if __name__ == "__main__":
    main()

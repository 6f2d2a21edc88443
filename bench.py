"""Benchmark of block-wise variable-length GQA attention (FCP hot path) on GB300.

One step = one pass of the whole hot path over one batch: fcp_partition + fcp_distribute +
fcp_coalesce (host plan), plan upload, forward tile kernel, LSE merge, backward prologue,
backward tile kernel, dQ conversion. Workload: one 32768-token causal sequence cut into
4096-token blocks (8 blocks, Zig-Zag over 4 simulated workers), 64 query / 8 KV heads,
head_dim 128, bf16 N(0,1) inputs, coalesce degree 16. The rest of the block-size sweep
(512..8192) is reported under "sweep".

Metric: TFLOP/s counting 4*Hq*D per unmasked score pair forward and 2.5x that backward.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fcp|reference] [--no-sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-attn fwd/bwd TFLOP/s & % GB300 dense BF16 peak vs block size (512-8K)"
HEADLINE_BLOCK = 4096
SWEEP = (512, 1024, 2048, 4096, 8192)
L2_FLUSH_BYTES = 512 << 20  # > 129 MB of L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("fcp", "reference"), default="fcp")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="only the headline step (for profiling): no e2e, CPU baseline, reshuffle, sweep, "
                         "configs or merge sections")
    ap.add_argument("--extras", action="store_true",
                    help="also report the planner-level sections: FCP against the ring plan through the kernels, "
                         "the solver's host time, the block-level pipeline by coalesce degree, the balance report")
    ap.add_argument("--with-reshuffle", action="store_true", help="keep the reshuffle section under --step-only")
    ap.add_argument("--block", type=int, default=HEADLINE_BLOCK)
    ap.add_argument("--coalesce", type=int, default=16)
    ap.add_argument("--bwd-band", type=int, default=None,
                    help="rows per backward query band (0: none; default: the plan's choice)")
    ap.add_argument("--seq-len", type=int, default=32768,
                    help="length of the causal sequence (smaller values are for profiler captures)")
    return ap.parse_args()


def workload(args):
    import workloads as W

    if args.seq_len == 32768:
        return W.block_sweep(args.block)
    nb = max(1, args.seq_len // args.block)
    return W.Workload(f"causal {args.seq_len}", [args.seq_len], args.block, 64, 8, 128, max(1, nb // 2), True,
                      token_cap=2 * args.block)


def config_of(w, coalesce, world):
    """The workload description both arms print."""
    return {"workload": f"causal {w.total_tokens}-token sequence, block {w.block_size} "
                        f"({w.total_tokens // w.block_size} blocks, Zig-Zag LPT over {w.n_workers} workers), "
                        f"{w.hq}/{w.hkv} heads, D={w.head_dim}, coalesce {coalesce}, fwd+merge+bwd",
            "block_size": w.block_size, "seq_len": w.total_tokens, "heads_q": w.hq, "heads_kv": w.hkv,
            "head_dim": w.head_dim, "workers_simulated": w.n_workers, "coalesce": coalesce,
            "l2": "flushed between steps (512 MB write, untimed); inputs (Q 512 MiB) also exceed L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank number over the process group (the identity on one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    """Units all ranks processed divided by the slowest rank's step time."""
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


def flops_of(seqlens, causal, hq, d):
    pairs = sum(L * (L + 1) // 2 if causal else L * L for L in seqlens)
    fwd = 4.0 * hq * d * pairs
    return fwd, 2.5 * fwd


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in self.out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------------------- CUDA path
class Step:
    """Buffers and launches of one batch; run() enqueues one whole step on `stream`."""

    def __init__(self, fcp, torch, w, coalesce, device, stream, planner="fcp", pipeline=None, replan=True,
                 bwd_band=None):
        import workloads as W

        self.bwd_band = bwd_band
        self.fcp, self.torch, self.w, self.c, self.dev, self.stream = fcp, torch, w, coalesce, device, stream
        self.planner = planner
        self.pipeline = pipeline  # coalesce degree of the block-level pipeline, or None
        self.replan = replan  # rebuild the plan for every step (host work in the timed region)
        self.next_plan = None
        self.q, self.k, self.v = W.make_qkv(w, device=device)
        self.do = W.make_dout(w, device=device)
        plan = self.make_plan()
        T, hq, hkv, D = w.total_tokens, w.hq, w.hkv, w.head_dim
        rows = plan.view()["partial_rows"]
        self.d_plan = torch.empty(plan.device_bytes() + 256, dtype=torch.uint8, device=device)
        self.part_o = torch.empty((hq, rows, D), dtype=torch.float32, device=device)
        self.part_lse = torch.empty((hq, rows), dtype=torch.float32, device=device)
        self.o = torch.empty((hq, T, D), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((hq, T), dtype=torch.float32, device=device)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.dq_acc = torch.empty((hq, T, D), dtype=torch.float32, device=device)
        self.di = torch.empty((hq, T), dtype=torch.float32, device=device)
        # the backward runs in query bands when the plan has them (long batches)
        self.n_bands = plan.bwd_bands()[0]
        self.dkv_acc = (torch.empty(plan.band_workspace_bytes(hkv, D), dtype=torch.uint8, device=device)
                        if self.n_bands else None)
        self.plan = plan
        self.fwd_flops, self.bwd_flops = flops_of(w.seqlens, w.causal, hq, D)
        self.events = None
        # merge traffic (algorithmic): per (h, token) S partials x (4D+4) read + (2D+4) written
        v = plan.view()
        per_row_parts = {}
        for r in v["runs"]:
            per_row_parts[(int(r[2]), int(r[3]))] = per_row_parts.get((int(r[2]), int(r[3])), 0) + 1
        self.parts_per_row = per_row_parts  # (query range) -> partials of each of its rows
        self.merge_bytes = sum(n * qlen * (4 * D + 4) + qlen * (2 * D + 4) for (_, qlen), n in per_row_parts.items()) * hq
        self.n_stages = int(v["n_exec_stages"])
        # forward stages, merge, prologue, backward tiles (one per query band, then the dK and dV
        # conversions), dQ conversion
        self.n_launches = self.n_stages + 2 + (self.n_bands + 2 if self.n_bands else 1) + 1
        if not replan:
            plan.upload(self.d_plan, stream)

    def make_plan(self):
        w = self.w
        if self.planner == "ring":
            plan = self.fcp.Plan.ring(w.seqlens, w.n_workers, w.causal)
        else:
            plan = self.fcp.Plan(w.seqlens, w.block_size, w.causal)
            if self.bwd_band is not None:
                plan.set_bwd_band(self.bwd_band)
            plan.distribute(w.n_workers, w.token_cap)
        if self.pipeline is not None:
            plan.schedule(self.pipeline)
        elif self.c != 1:
            plan.coalesce(self.c)
        return plan

    def run(self, ev=None, backward=True):
        """One step. ev: optional list of 6 CUDA events recorded between the phases."""
        f, s = self.fcp, self.stream
        rec = (lambda i: ev[i].record(s)) if ev is not None else (lambda i: None)
        rec(0)
        if self.replan:
            # the plan built while the previous step ran (partition + LPT distribute + coalesce
            # or schedule, on the host), uploaded in stream order
            plan = self.next_plan if self.next_plan is not None else self.make_plan()
            self.next_plan = None
            plan.upload(self.d_plan, s)
            self.plan = plan
        plan = self.plan
        if self.n_stages > 1:  # block-level pipeline: one launch per execution stage
            for stg in range(self.n_stages):
                f.block_attn_fwd_stage(plan, self.d_plan, stg, self.q, self.k, self.v, self.part_o, self.part_lse, s)
        else:
            f.block_attn_fwd(plan, self.d_plan, self.q, self.k, self.v, self.part_o, self.part_lse, s)
        rec(1)
        f.block_attn_merge(plan, self.d_plan, self.part_o, self.part_lse, self.o, self.lse, s)
        rec(2)
        if backward:
            f.block_attn_bwd_prologue(plan, self.o, self.do, self.di, self.dq_acc, s)
            rec(3)
            if self.n_bands:
                f.block_attn_bwd_tiles_banded(plan, self.d_plan, self.q, self.k, self.v, self.do, self.lse, self.di,
                                              self.dq_acc, self.dkv_acc, self.dk, self.dv, s)
            else:
                f.block_attn_bwd_tiles(plan, self.d_plan, self.q, self.k, self.v, self.do, self.lse, self.di,
                                       self.dq_acc, self.dk, self.dv, s)
            rec(4)
            f.block_attn_bwd_dq_convert(plan, self.dq_acc, self.dq, s)
        else:  # forward only: the backward phases are empty
            rec(3)
            rec(4)
        rec(5)
        if self.replan:
            # the next batch's plan is built on the host while this step's kernels run, as a
            # training loop would overlap it
            self.next_plan = self.make_plan()


def timed_steps(torch, step, steps, warmup, flush, backward=True):
    """Per-step CUDA-event times of each phase (ms), L2 flushed between steps (not timed)."""
    s = step.stream
    for _ in range(warmup):
        step.run(backward=backward)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for i in range(steps):
        with torch.cuda.stream(s):
            flush.fill_(i & 0xFF)
        step.run(ev=evs[i], backward=backward)
    torch.cuda.synchronize()
    out = []
    for ev in evs:
        t = [ev[j].elapsed_time(ev[j + 1]) for j in range(5)]
        out.append({"fwd": t[0], "merge": t[1], "prologue": t[2], "bwd": t[3], "convert": t[4], "total": sum(t)})
    return out


def oracle_prefix_run(w, S):
    """One oracle forward + backward on the causal prefix of S tokens of the workload's
    sequence (all heads), timed on host cores: (seconds, FLOPs)."""
    import workloads as W
    from oracle import attention as A

    sub = W.Workload("prefix", [S], w.block_size, w.hq, w.hkv, w.head_dim, 1, w.causal, std=w.std)
    q, k, v = W.make_qkv(sub)
    do = W.make_dout(sub)
    t0 = time.perf_counter()
    A.attention_forward(q, k, v, sub.seqlens, sub.causal)
    A.attention_backward(q, k, v, do, sub.seqlens, sub.causal)
    dt = time.perf_counter() - t0
    f, b = flops_of(sub.seqlens, sub.causal, sub.hq, sub.head_dim)
    return dt, f + b


def oracle_prefix_calibrate(w, target_s):
    """Prefix length whose oracle run takes at least a third of target_s (doubling from 256
    tokens, at most half the sequence), with that run's (seconds, FLOPs)."""
    S = 256
    dt, fl = oracle_prefix_run(w, S)
    while dt < target_s / 3 and S < w.total_tokens // 2:
        S *= 2
        dt, fl = oracle_prefix_run(w, S)
    return S, dt, fl


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_sample_desc(w, S, dt):
    return (f"float64 numpy oracle, forward+backward of the first {S} tokens of the causal sequence, "
            f"{w.hq}/{w.hkv} heads, D={w.head_dim} ({dt:.1f} s)")


def cpu_baseline_sample(w, target_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload: a causal prefix of S
    tokens of the same sequence with all heads (forward + backward), timed on host cores."""
    S, dt, fl = oracle_prefix_calibrate(w, target_s)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": oracle_sample_desc(w, S, dt), "seconds": dt}


def traffic_from_profile(kernel_tag, block):
    """DRAM bytes per launch of a kernel on this workload from the committed ncu summary
    (profiles/traffic.txt: tag, source file, sha256/16 of that file at capture, block size,
    bytes), or None if the kernel's source has changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) < 5 or parts[0].startswith("#") or parts[0] != kernel_tag or int(parts[3]) != block:
                continue
            src = os.path.join(ROOT, "context_parallelism_fcp_gb300", "csrc", parts[1])
            with open(src, "rb") as g:
                if hashlib.sha256(g.read()).hexdigest()[:16] == parts[2]:
                    return float(parts[4])
    return None


def bench_fcp(args):
    import torch

    import context_parallelism_fcp_gb300 as fcp
    import workloads as W

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fcp.lib()
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    w = workload(args)
    step = Step(fcp, torch, w, args.coalesce, dev, stream, bwd_band=args.bwd_band)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.step_only:
        cpu = cpu_baseline_sample(w)

    # warm-up, then exactly K timed steps bracketed by barrier + synchronize
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        times = timed_steps(torch, step, args.steps, args.warmup, flush)
        torch.cuda.synchronize()
        barrier()
    code = fcp.device_error(step.d_plan, stream)
    if code:
        raise RuntimeError(f"device error word 0x{code:x}")

    ms = statistics.mean(t["total"] for t in times)
    ms_median = statistics.median(t["total"] for t in times)
    phase = {k: statistics.mean(t[k] for t in times) for k in ("fwd", "merge", "prologue", "bwd", "convert")}
    ms = max_over_ranks(ms, dev)
    value = whole_job_tflops(step.fwd_flops + step.bwd_flops, world, ms)
    sustained = pk["bf16_tflops_sustained"]
    fwd_tf = step.fwd_flops / (phase["fwd"] * 1e-3) / 1e12
    bwd_tf = step.bwd_flops / (phase["bwd"] * 1e-3) / 1e12
    shares = {k: phase[k] / sum(phase.values()) for k in phase}
    dominant = "bwd" if phase["bwd"] >= phase["fwd"] else "fwd"
    dom_tf = bwd_tf if dominant == "bwd" else fwd_tf
    dom_flops = step.bwd_flops if dominant == "bwd" else step.fwd_flops
    traffic = traffic_from_profile("bwd_tile_kernel" if dominant == "bwd" else "fwd_kernel", w.block_size) \
        if w.head_dim == 128 and args.seq_len == 32768 else None

    hq, T, D = w.hq, w.total_tokens, w.head_dim
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "ms_per_step_median": round(ms_median, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_of(w, args.coalesce, world),
        "fwd_tflops": round(fwd_tf, 2),
        "bwd_tflops": round(bwd_tf, 2),
        "fwd_bwd_frac_of_peak": round(value / world / sustained, 4),
        "phase_ms": {k: round(v, 4) for k, v in phase.items()},
        "phase_share": {k: round(v, 4) for k, v in shares.items()},
        "roofline": {"kernel": f"{'bwd_tile_kernel' if dominant == 'bwd' else 'fwd_kernel'}<{w.head_dim}>", "bound": "tensor", "achieved": round(dom_tf, 2),
                     "peak": sustained, "unit": "TFLOP/s", "frac": round(dom_tf / sustained, 4),
                     "traffic": traffic, "algorithmic_flops_per_launch": dom_flops,
                     "peak_source": f"{pk['source']} bf16_tflops_sustained (kernel timed inside a multi-second loop)"},
        "gpu_launches": step.n_launches * args.steps,
        "clocks": clk.summary(),
        "imbalance": None,
    }
    v = step.plan.view()
    loads = [int(x) for x in v["load"]]
    mx = max(loads)
    result["imbalance"] = round((mx - sum(loads) / len(loads)) / mx, 6) if mx else 0.0

    resh = None
    if not args.step_only or args.with_reshuffle:
        # measured here, right after the headline step: after the 524288-token workload of
        # `configs` the same launches ran about 20% slower
        resh = reshuffle_bench(torch, fcp, step, stream, flush, pk)

    # end to end through the public API: pinned host inputs -> device, step, results -> host
    if not args.no_e2e and not args.step_only:
        result["e2e"] = e2e(torch, fcp, w, args, dev, stream, step, flush)
    if cpu is not None:
        result["cpu_baseline"] = cpu
    if args.extras and not args.step_only:
        result["fcp_vs_ring"] = planner_compare(torch, fcp, W, dev, stream, flush, sustained)
        if rank == 0:
            result["solver"] = solver_report(fcp, W)
            result["pipeline"] = pipeline_bench(torch, fcp, W, dev, stream, flush, sustained)
            result["balance"] = balance_report(W)
    # the small sections last, so that the end of the line carries every block size
    if not args.no_sweep and not args.step_only:
        result["configs"] = configs_bench(torch, fcp, W, dev, stream, flush, sustained)
    if resh is not None:
        result["reshuffle_roofline"] = resh
    hbm = pk["hbm_gbs"]
    result["prologue_roofline"] = hbm_roofline(hq * T * (8 * D + 4), phase["prologue"], hbm,
                                               "prologue_kernel: O, dO in; Di, zeroed dQ acc out")
    result["convert_roofline"] = hbm_roofline(hq * T * D * 6, phase["convert"], hbm,
                                              "dq_convert_kernel: f32 dQ in, bf16 dQ out")
    result["merge_roofline_identity"] = hbm_roofline(
        step.merge_bytes, phase["merge"], hbm, "merge_kernel in the step: 1 partial per row (copy path), partly in L2")
    result["fwd_roofline"] = {"kernel": f"fwd_kernel<{D}>", "bound": "tensor", "achieved": round(fwd_tf, 1),
                              "peak": sustained, "unit": "TFLOP/s", "frac": round(fwd_tf / sustained, 4)}
    sw = None
    if not args.no_sweep and not args.step_only:
        sw, merge_general = sweep(torch, fcp, W, args, dev, stream, flush, sustained, hbm)
        result["merge_roofline"] = merge_general
    if sw is not None:
        result["sweep"] = sw
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def hbm_roofline(nbytes, ms, hbm, what, with_bytes=False):
    gbs = nbytes / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
    out = {"bound": "hbm", "achieved": round(gbs), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 3)}
    if with_bytes:
        out["algorithmic_bytes"] = int(nbytes)
    out["what"] = what
    return out


def e2e(torch, fcp, w, args, dev, stream, step, flush):
    """The same metric with host buffers, through the public API (FcpAttention), step for step
    what the device-timed step does: every step plans the batch again on the host
    (FcpAttention.replan: partition, distribute, coalesce, device-image upload), flushes L2,
    copies Q, K, V, dO from pinned host memory, runs forward and backward and copies O, LSE,
    dQ, dK, dV back to pinned host memory. The copies run on their own streams, one per
    direction, into and out of two alternating buffer sets (each with its own FcpAttention,
    so step i+1's plan upload does not touch the image step i reads), so step i+1's inputs
    arrive and step i's results leave while step i computes; dO travels during step i's
    forward and O, LSE during its backward. Every step's planning, flush and copies are inside
    the timed region. `serial` is the same loop with every copy on the compute stream. Under
    several ranks each replica runs this loop after a barrier; the value is every rank's work
    over the slowest rank's time and the byte counts are summed over the ranks, as for the
    headline value."""
    hq, hkv, T, D = w.hq, w.hkv, w.total_tokens, w.head_dim
    world = int(os.environ.get("WORLD_SIZE", "1"))
    hin = [t.cpu().pin_memory() for t in (step.q, step.k, step.v, step.do)]
    outs = (step.o, step.lse, step.dq, step.dk, step.dv)
    hout = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _ in range(2)]
    din = [[torch.empty_like(t) for t in (step.q, step.k, step.v, step.do)] for _ in range(2)]
    dout = [[torch.empty_like(t) for t in outs] for _ in range(2)]
    att = [fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, hq, hkv, D, token_cap=w.token_cap,
                            coalesce=args.coalesce, device=dev) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    qkv_in, do_in, fwd_done, bwd_done, out_free = ([ev() for _ in range(2)] for _ in range(5))

    def pipelined(i):
        b = i & 1
        q, k, v, do = din[b]
        o, lse, dq, dk, dv = dout[b]
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(bwd_done[b])  # set b's plan and inputs were last read by step i-2
            att[b].replan(stream=h2d)
            for d, h in zip(din[b][:3], hin[:3]):
                d.copy_(h, non_blocking=True)
            qkv_in[b].record(h2d)
            do.copy_(hin[3], non_blocking=True)
            do_in[b].record(h2d)
        with torch.cuda.stream(stream):
            flush.fill_(i & 0xFF)
        stream.wait_event(qkv_in[b])
        if i >= 2:
            stream.wait_event(out_free[b])  # set b's outputs were last read by step i-2's copies
        att[b].forward(q, k, v, o=o, lse=lse, stream=stream)
        fwd_done[b].record(stream)
        stream.wait_event(do_in[b])
        att[b].backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, stream=stream)
        bwd_done[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(fwd_done[b])
            for h, d in zip(hout[b][:2], (o, lse)):
                h.copy_(d, non_blocking=True)
            d2h.wait_event(bwd_done[b])
            for h, d in zip(hout[b][2:], (dq, dk, dv)):
                h.copy_(d, non_blocking=True)
            out_free[b].record(d2h)

    def serial(i):
        q, k, v, do = din[0]
        o, lse, dq, dk, dv = dout[0]
        with torch.cuda.stream(stream):
            att[0].replan(stream=stream)
            flush.fill_(i & 0xFF)
            for d, h in zip(din[0], hin):
                d.copy_(h, non_blocking=True)
            att[0].forward(q, k, v, o=o, lse=lse, stream=stream)
            att[0].backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, stream=stream)
            for h, d in zip(hout[0], (o, lse, dq, dk, dv)):
                h.copy_(d, non_blocking=True)

    def timed(one):
        for i in range(args.warmup):
            one(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d.wait_event(e0)
        d2h.wait_event(e0)
        for i in range(args.steps):
            one(args.warmup + i)
        for b in range(2):
            stream.wait_event(out_free[b])
        stream.wait_stream(d2h)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    # whole job, as the headline value: every rank's steps over the slowest rank's time
    ms = max_over_ranks(timed(pipelined), dev)
    ms_serial = max_over_ranks(timed(serial), dev)
    for a in att:
        if fcp.device_error(a.d_plan, stream):
            raise RuntimeError("device error word set in the end-to-end run")
    flops = step.fwd_flops + step.bwd_flops
    return {"value": round(whole_job_tflops(flops, world, ms), 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": world * sum(t.numel() * t.element_size() for t in hin),
            "d2h_bytes_per_step": world * sum(t.numel() * t.element_size() for t in hout[0]),
            "per_step": "plan rebuilt on the host and uploaded, L2 flushed, inputs copied in, results copied out",
            "copies": "h2d and d2h streams, double-buffered: step i+1's inputs and step i's results "
                      "move while step i computes",
            "serial": {"value": round(whole_job_tflops(flops, world, ms_serial), 2),
                       "ms_per_step": round(ms_serial, 3)}}


SWEEP_RUNS = 20  # timed runs per sweep point (the median is reported)


def sweep(torch, fcp, W, args, dev, stream, flush, sustained, hbm):
    """The whole step for every block size (and one partial per pair, c = 1, for b <= 1024):
    medians over SWEEP_RUNS runs, each with L2 flushed and the plan rebuilt. Compact rows:
    fwd = forward + merge, bwd = prologue + tiles + dQ conversion, both TFLOP/s. Returns the
    rows and the merge kernel's roofline on the path that merges (b = 512, c = 1)."""
    cols = ["block", "coalesce", "fwd_tflops", "bwd_tflops", "fwd_bwd_tflops", "frac_of_peak",
            "fwd_kernel_tflops", "bwd_kernel_tflops"]
    rows = []
    merge_general = None
    for b in SWEEP:
        w = W.block_sweep(b)
        for c in ((args.coalesce, 1) if b <= 1024 else (args.coalesce,)):
            st = Step(fcp, torch, w, c, dev, stream)
            times = timed_steps(torch, st, SWEEP_RUNS, 3, flush)
            fwd = statistics.median(t["fwd"] + t["merge"] for t in times)
            bwd = statistics.median(t["prologue"] + t["bwd"] + t["convert"] for t in times)
            fk = statistics.median(t["fwd"] for t in times)
            bk = statistics.median(t["bwd"] for t in times)
            tot = (st.fwd_flops + st.bwd_flops) / ((fwd + bwd) * 1e-3) / 1e12
            rows.append([b, c, round(st.fwd_flops / (fwd * 1e-3) / 1e12), round(st.bwd_flops / (bwd * 1e-3) / 1e12),
                         round(tot), round(tot / sustained, 3),
                         round(st.fwd_flops / (fk * 1e-3) / 1e12), round(st.bwd_flops / (bk * 1e-3) / 1e12)])
            if b == 512 and c == 1:
                merge_general = merge_cold(torch, fcp, st, stream, flush, hbm)
            del st
            torch.cuda.empty_cache()
    return {"cols": cols, "rows": rows, "median_of": SWEEP_RUNS}, merge_general


def merge_cold(torch, fcp, st, stream, flush, hbm, runs=10):
    """The LSE merge alone on a plan with many partials per row, L2 flushed before every
    launch: median GB/s of algorithmic bytes (S partials x (4D+4) read + (2D+4) written per
    head and token)."""
    st.run(backward=False)  # the partials of the step's current plan
    times = []
    for i in range(runs + 2):
        with torch.cuda.stream(stream):
            flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fcp.block_attn_merge(st.plan, st.d_plan, st.part_o, st.part_lse, st.o, st.lse, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    per_row = list(st.parts_per_row.values())
    out = hbm_roofline(st.merge_bytes, ms, hbm, with_bytes=True, what=
                       f"merge_kernel alone, {st.w.name} c=1: {min(per_row)}-{max(per_row)} partials per row, "
                       f"{st.part_o.numel() * 4 / 1e9:.0f} GB of partials, L2 flushed")
    out["ms"] = round(ms, 3)
    return out


def reshuffle_bench(torch, fcp, step, stream, flush, pk):
    """GB/s of the transparent reshuffle of Q (user -> worker layout and back), 2 bytes read
    and written per element, L2 flushed before each timed launch."""
    dst = torch.empty_like(step.q)
    times = []
    for i in range(6):
        with torch.cuda.stream(stream):
            flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fcp.reshuffle(step.plan, step.d_plan, step.q, dst, to_workers=(i % 2 == 0), stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    nbytes = 2 * step.q.numel() * step.q.element_size()
    return hbm_roofline(nbytes, statistics.mean(times), pk["hbm_gbs"], "reshuffle_kernel: Q, user to worker layout")


def planner_compare(torch, fcp, W, dev, stream, flush, sustained):
    """Attention fwd+bwd TFLOP/s of the causal mixed batch (65536 tokens, 16 workers) under
    FCP's plan (4K blocks, LPT) and under the ring baseline's (2N blocks per sequence), with
    one partial per pair (c = 1) and with coalescing (c = 16)."""
    w = W.causal_mixed()
    out = []
    for planner in ("fcp", "ring"):
        for c in (1, 16):
            st = Step(fcp, torch, w, c, dev, stream, planner=planner)
            times = timed_steps(torch, st, 3, 2, flush)
            ms = statistics.mean(t["total"] for t in times)
            tf = (st.fwd_flops + st.bwd_flops) / (ms * 1e-3) / 1e12
            v = st.plan.view()
            out.append({"planner": planner, "coalesce": c, "blocks": v["n_blocks"], "items": v["n_items"],
                        "ms": round(ms, 3), "fwd_bwd_tflops": round(tf, 1), "frac_of_peak": round(tf / sustained, 4)})
            del st
            torch.cuda.empty_cache()
    return out


def pipeline_bench(torch, fcp, W, dev, stream, flush, sustained):
    """The block-level pipeline with the bottom-up coalescer (Section 4.2, Figure 7, Table 2):
    the forward launched one execution stage at a time (local work first, then `degree`
    congestion-free sub-stages per stage), against coalesce degree c. Plans are built once,
    outside the timed region, so the numbers isolate the kernels' side of the trade-off.
    Workloads: the 32K causal sequence at 512-token blocks (64 blocks on 32 workers) and the
    causal mixed batch (4K blocks, 16 workers)."""
    out = []
    for w in (W.block_sweep(512), W.causal_mixed()):
        rows = []
        for degree in (1, 4, 16, 64):
            st = Step(fcp, torch, w, 1, dev, stream, pipeline=degree, replan=False)
            times = timed_steps(torch, st, 3, 2, flush)
            fwd = statistics.mean(t["fwd"] for t in times)
            fm = statistics.mean(t["fwd"] + t["merge"] for t in times)
            tot = statistics.mean(t["total"] for t in times)
            v = st.plan.view()
            rows.append({"degree": degree, "stages": st.n_stages, "runs": v["n_runs"],
                         "fwd_ms": round(fwd, 3), "fwd_tflops": round(st.fwd_flops / (fwd * 1e-3) / 1e12, 1),
                         "fwd_merge_tflops": round(st.fwd_flops / (fm * 1e-3) / 1e12, 1),
                         "fwd_bwd_tflops": round((st.fwd_flops + st.bwd_flops) / (tot * 1e-3) / 1e12, 1),
                         "fwd_bwd_frac_of_peak": round((st.fwd_flops + st.bwd_flops) / (tot * 1e-3) / 1e12
                                                       / sustained, 4)})
            del st
            torch.cuda.empty_cache()
        out.append({"workload": w.name, "workers": w.n_workers, "block": w.block_size, "by_degree": rows})
    return out


def configs_bench(torch, fcp, W, dev, stream, flush, sustained):
    """The other named workloads, through the same step: the full-mask batch (16 lognormal
    sequences, 65536 tokens, 1K blocks, 8 workers; forward + merge only), the causal mixed
    batch (lognormal lengths plus a 32K outlier, 4K blocks, 16 workers) and the 524288-token
    causal sequence (8K blocks, 32 workers; 1 warm-up and 2 timed steps of about 12 s each).
    Coalesce degree 16; L2 flushed between steps; medians of the timed steps. Compact rows:
    TFLOP/s of fwd (+ merge), bwd (prologue + tiles + conversion) and the step, then the
    per-phase milliseconds."""
    cols = ["workload", "tokens", "block", "fwd_tflops", "bwd_tflops", "fwd_bwd_tflops", "frac_of_peak",
            "ms_fwd_kernel", "ms_merge", "ms_prologue", "ms_bwd_kernel", "ms_convert"]
    rows = []
    for w, steps, warm in ((W.full_mask(), 5, 2), (W.causal_mixed(), 5, 2), (W.long_causal(), 2, 1)):
        st = Step(fcp, torch, w, 16, dev, stream)
        times = timed_steps(torch, st, steps, warm, flush, backward=w.backward)
        med = {k: statistics.median(t[k] for t in times) for k in ("fwd", "merge", "prologue", "bwd", "convert")}
        fwd = statistics.median(t["fwd"] + t["merge"] for t in times)
        ftf = st.fwd_flops / (fwd * 1e-3) / 1e12
        btf = tot = None
        if w.backward:
            bwd = statistics.median(t["prologue"] + t["bwd"] + t["convert"] for t in times)
            btf = round(st.bwd_flops / (bwd * 1e-3) / 1e12)
            tot = round((st.fwd_flops + st.bwd_flops) / (statistics.median(t["total"] for t in times) * 1e-3) / 1e12)
        rows.append([w.name, w.total_tokens, w.block_size, round(ftf), btf, tot,
                     round((tot if tot is not None else ftf) / sustained, 3)] +
                    [round(med[k], 2) for k in ("fwd", "merge", "prologue", "bwd", "convert")])
        del st
        torch.cuda.empty_cache()
    return {"cols": cols, "rows": rows}


def solver_report(fcp, W):
    """Host time of the congestion-free solver on the pages' cluster setting (256 workers,
    32K tokens each, 4K blocks) and on the benchmark's own plan."""
    out = {}
    for name, w in (("cluster_256x32k", W.cluster_batch()), ("bench_32k", W.block_sweep(HEADLINE_BLOCK))):
        t0 = time.perf_counter()
        plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers, w.token_cap)
        t1 = time.perf_counter()
        res = plan.solve()
        t2 = time.perf_counter()
        loads = [int(x) for x in plan.view()["load"]]
        mx = max(loads)
        out[name] = {"workers": w.n_workers, "blocks": plan.view()["n_blocks"], "transfers": int(len(res["transfers"])),
                     "stages": res["n_stages"], "plan_ms": round((t1 - t0) * 1e3, 2),
                     "solve_ms": round((t2 - t1) * 1e3, 2),
                     "imbalance": round((mx - sum(loads) / len(loads)) / mx, 6) if mx else 0.0}
    return out


def balance_report(W):
    """FCP vs the ring baseline on the pages' kind of batches (plan level, host only). The
    ring plan of a 256-worker batch has hundreds of thousands of blocks and tens of millions
    of work items, so the cluster comparison runs at 32 workers x 32K tokens."""
    from context_parallelism_fcp_gb300 import balance

    out = {}
    for w in (W.full_mask(), W.causal_mixed(), W.cluster_batch(n_workers=32)):
        out[w.name] = balance.compare(w.seqlens, w.block_size, w.n_workers, w.causal, w.token_cap)
    return out


def bench_reference(args):
    """The oracle as it stands, timed on the host cores on bounded samples of the same
    workload, same metric and unit: the warm-up picks the prefix length (sized so that the
    K timed steps take about two minutes at most), then exactly K steps are timed at that
    length. Under torchrun only rank 0 runs it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args)
    per_step = min(6.0, 120.0 / max(1, args.steps))
    S, _, _ = oracle_prefix_calibrate(w, per_step)  # untimed warm-up and calibration
    for _ in range(max(0, args.warmup - 1)):
        oracle_prefix_run(w, S)
    runs = [oracle_prefix_run(w, S) for _ in range(args.steps)]
    secs = sum(dt for dt, _ in runs)
    val = sum(fl for _, fl in runs) / secs / 1e12
    ms = secs / len(runs) * 1e3
    cpu = {"value": val, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
           "sample": oracle_sample_desc(w, S, secs / len(runs)), "seconds": secs / len(runs)}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": len(runs), "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(w, args.coalesce, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": cpu,
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_fcp(args)


if __name__ == "__main__":
    main()

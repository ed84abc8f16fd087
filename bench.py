#!/usr/bin/env python
"""Throughput of the token-choice MoE FFN block (AFMoE / MiniMax-M3) on GB300.

One step = one moe_forward over one batch of T synthetic tokens (router,
dispatch sort, gate/up + activation, down, combine; with the sandwich norms
also the pre-MLP RMSNorm and, inside the combine, the post-MLP RMSNorm and the
residual add; a dense prefix layer: its MLP GEMMs and the combine), inputs
resident in HBM.
L2 is flushed before every step, outside the timed events: a 256 MiB write, then
a 256 MiB read, so that the step neither finds its inputs in L2 nor pays for
writing back the flush buffer's dirty lines (--flush write: the write alone).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The headline workload is the largest configuration, the MiniMax-M3-shaped block
(T 2048, H 6144, 128 experts of width 3072, packed shared expert); on one GPU
the other configurations (tiny, Nano decode, AFMoE prefill, the Zipf sweep) are
timed after it and reported under "other_configs" of the same line.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
of the block on its own GPU (the block has no cross-GPU exchange): weak scaling.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (bf16) and % of roofline (tensor peak / HBM GB/s at small T)"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def work_model(shape, U: int):
    """Algorithmic FLOPs and HBM bytes of one forward and of its expert kernels.

    FLOPs  F = T (2HE + 6HIk + 6HS); bytes B = U*3HI*2 + 3HS*2 + 4EH + 4E + 2*2TH,
    U = experts that received at least one token (the packed shared expert's
    weights are its 3HS*2 bytes; a dense layer has E = k = U = 0 and its MLP of
    width S as the "shared" term).  With the sandwich norms add the two fp32
    norm weights (8H bytes) and 8TH FLOPs (square, sum, scale and gain per
    element of both norms, and the residual add counted with them).
    Intermediate buffers are implementation traffic and are not counted.
    MX weights: 1 (E4M3) or 1/2 (E2M1) byte per weight plus 1/32 byte of scale
    in place of the 2 bytes of bf16."""
    T, H, E, k, I, S = shape.T, shape.H, shape.E, shape.k, shape.I, shape.S
    # bytes per expert weight: bf16, or an MX element code plus its share of an
    # E8M0 scale byte per 32 weights
    bpw = {"bf16": 2.0, "mxfp8": 1.0 + 1.0 / 32, "mxfp4": 0.5 + 1.0 / 32}[getattr(shape, "weight_format", "bf16")]
    F = T * (2 * H * E + 6 * H * I * k + 6 * H * S)
    B = int((U * 3 * H * I + 3 * H * S) * bpw) + 4 * E * H + 4 * E + 2 * 2 * T * H
    if shape.mlp_norm != "none":
        F += 8 * T * H
        B += 8 * H
    kernels = {
        "gate_up": dict(flops=4 * T * H * (k * I + S), bytes=int((U * 2 * H * I + 2 * H * S) * bpw) + 2 * T * H),
        "down": dict(flops=2 * T * H * (k * I + S), bytes=int((U * H * I + H * S) * bpw) + 2 * T * H),
    }
    kernels["experts"] = dict(flops=kernels["gate_up"]["flops"] + kernels["down"]["flops"],
                              bytes=int((U * 3 * H * I + 3 * H * S) * bpw) + 2 * 2 * T * H)
    return F, B, kernels


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(v: float, world: int, device="cpu") -> float:
    """The largest value any rank reports (every rank must call it: a collective)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank (a replica) processes its own batch in `seconds`,
    the slowest rank's time."""
    return world * tokens_per_rank / seconds


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != gpus:
        raise SystemExit(f"--gpus {gpus} but WORLD_SIZE {world}")
    return world, rank, local


def run_ours(args, shape):
    import torch
    import torch.distributed as dist

    from expert_routed_ffn_gb300 import build as moe_build
    from expert_routed_ffn_gb300 import capi
    from expert_routed_ffn_gb300 import workloads as wl

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        moe_build.build()
    if world > 1:
        dist.barrier()
    dev = torch.device("cuda", local)
    inputs = wl.make_inputs(shape, dev)
    blk = capi.block_from_inputs(shape, inputs, max_tokens=shape.T)
    if args.path:
        blk.set_option(capi.MOE_OPT_PATH, {"decode": capi.PATH_DECODE, "grouped": capi.PATH_GROUPED,
                                           "swapped": capi.PATH_SWAPPED}[args.path])
    if args.gemm_pair is not None:
        blk.set_option(capi.MOE_OPT_GEMM_PAIR, args.gemm_pair)
    if args.two_launch:
        blk.set_option(capi.MOE_OPT_FUSE_EXPERTS, 0)
    if args.no_prefetch:
        blk.set_option(capi.MOE_OPT_PREFETCH, 0)
    X = inputs["X"]
    Y = torch.empty_like(X)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if args.flush == "clean" else None

    def flush_l2():
        flush.fill_(1)  # evicts L2; not inside the timed events
        if flush_rd is not None:  # then replace the dirty lines by clean ones (their write-back happens here)
            flush_rd.sum()

    def step():
        if not args.no_flush:
            flush_l2()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        blk.forward(X, Y)
        e.record()
        return s, e

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if blk.sync_status() != capi.MOE_OK:
        raise SystemExit("device error during warm-up")
    U = 0
    if shape.E > 0:
        idx = blk.inspect(capi.MOE_BUF_TOPK_IDX, shape.T * shape.k, torch.int32)
        U = int(torch.unique(idx).numel())
    launches = blk.stats().kernel_launches
    path = blk.stats().path
    names = blk.stage_names()

    sampler = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "uuid", None) and
                           f"GPU-{torch.cuda.get_device_properties(dev).uuid}")
    t_end = time.perf_counter() + args.preroll  # untimed pre-roll: steady clocks, samples under load
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [step() for _ in range(args.steps)]  # timed steps: no per-kernel events
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    per_step = [s.elapsed_time(e) for s, e in evs]
    clocks = sampler.stop()

    # per-kernel durations: the same steps again with a CUDA event after every
    # kernel (on the launching stream); the events cost the programmatic-launch
    # overlap, so these steps are not the timed ones
    blk.set_option(capi.MOE_OPT_STAGE_EVENTS, 1)
    stage_sum = [0.0] * len(names)
    for _ in range(args.steps):
        step()
        for i, v in enumerate(blk.stage_times()[:len(names)]):
            stage_sum[i] += v
    blk.set_option(capi.MOE_OPT_STAGE_EVENTS, 0)
    # device timeline of the same steps without events: per kernel, first CTA
    # start, first CTA past the wait on its predecessor, last CTA end (us)
    blk.set_option(capi.MOE_OPT_TRACE, 1)
    tl_sum, tl_n, gw_sum, rw_sum = None, 0, None, None
    for _ in range(args.steps):
        step()
        tr = blk.trace()
        if tl_sum is None:
            tl_sum = [[t[0]] + [0.0] * capi.TRACE_FIELDS for t in tr]
        for acc, t in zip(tl_sum, tr):
            for j in range(1, capi.TRACE_FIELDS + 1):
                acc[j] += t[j]
        tl_n += 1
        if "experts_gemm" in names:
            st = blk.inspect(capi.MOE_BUF_GEMM_STATS, 8, torch.int64).cpu().tolist()
            gw_sum = st if gw_sum is None else [a + b for a, b in zip(gw_sum, st)]
        if "router" in names and not shape.dtype == "f32":
            st = blk.inspect(capi.MOE_BUF_ROUTER_STATS, 8, torch.int64).cpu().tolist()
            rw_sum = st if rw_sum is None else [a + b for a, b in zip(rw_sum, st)]
    blk.set_option(capi.MOE_OPT_TRACE, 0)
    gemm_waits = None
    if gw_sum is not None:
        # per CTA and step, us: where the fused expert GEMM's roles spend their time
        per = 1e-3 / (tl_n * torch.cuda.get_device_properties(dev).multi_processor_count)
        keys = ["producer_wait_stage", "producer_wait_rows", "mma_wait_data", "mma_wait_accum",
                "epilogue_wait_accum", "epilogue_work", "cta_busy"]
        gemm_waits = {k: round(v * per, 2) for k, v in zip(keys, gw_sum[:7])}
        gemm_waits["tiles"] = gw_sum[7] // tl_n
    router_phases = None
    if rw_sum is not None and rw_sum[5] > 0:
        # per CTA and step, us: the tensor-core router's phases
        keys = ["main_loop", "cluster_barrier", "push_partials", "sum_and_route", "histogram"]
        router_phases = {k: round(v * 1e-3 / rw_sum[5], 2) for k, v in zip(keys, rw_sum[:5])}
        router_phases["of_which_partial_sums"] = round(rw_sum[6] * 1e-3 / rw_sum[5], 2)
        router_phases["ctas"] = rw_sum[5] // tl_n
    # per kernel: first begin, first ready, last ready, first end, last end
    timeline = ({t[0]: [round(t[j] / tl_n, 2) for j in range(1, capi.TRACE_FIELDS + 1)] for t in tl_sum}
                if tl_sum else None)
    status = blk.sync_status()
    if status != capi.MOE_OK:
        raise SystemExit(f"device error during the timed steps: {capi.STATUS_NAMES[status]}")

    ms = max_over_ranks(sum(per_step) / len(per_step), world, dev)
    value = job_throughput(shape.T, world, ms / 1e3)

    # end to end through the host-buffer entry point: H2D of X, forward, D2H of Y per step
    Xh = X.cpu().pin_memory()
    Yh = torch.empty_like(Xh).pin_memory()
    for _ in range(max(1, args.warmup)):
        blk.forward_host(Xh, Yh)
    e2e_t = []
    for _ in range(args.steps):
        flush_l2()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        blk.forward_host(Xh, Yh)
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(sum(e2e_t) / len(e2e_t), world, dev)
    xbytes = Xh.numel() * Xh.element_size()

    pk, pk_src = peaks()
    F, B, kern = work_model(shape, U)
    t_tc, t_hbm = F / (pk["bf16_tflops"] * 1e12), B / (pk["hbm_gbs"] * 1e9)
    stage_avg = {n: stage_sum[i] / args.steps for i, n in enumerate(names)}
    dom = max(stage_avg, key=stage_avg.get)
    roof = None
    key = {"gate_up_gemm": "gate_up", "decode_gate_up": "gate_up", "gate_up_gemm_swapped": "gate_up",
           "down_gemm": "down", "decode_down": "down", "down_gemm_swapped": "down",
           "experts_gemm": "experts"}.get(dom)
    if key is None:  # report the heavier expert GEMM when a small kernel leads
        gemms = [n for n in stage_avg if "gemm" in n or n.startswith("decode_")]
        if gemms:
            dom = max(gemms, key=stage_avg.get)
            key = "experts" if dom == "experts_gemm" else ("gate_up" if "gate_up" in dom else "down")

    if key is not None:
        kw = kern[key]
        dur = stage_avg[dom] / 1e3
        tensor_time = kw["flops"] / (pk["bf16_tflops"] * 1e12)
        hbm_time = kw["bytes"] / (pk["hbm_gbs"] * 1e9)
        if tensor_time > hbm_time:
            ach = kw["flops"] / dur / 1e12
            roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(ach / pk["bf16_tflops"], 4)}
        else:
            ach = kw["bytes"] / dur / 1e9
            roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(ach / pk["hbm_gbs"], 4)}
        roof.update({"kernel": dom, "dominant_stage": max(stage_avg, key=stage_avg.get),
                     "peak_source": pk_src, "traffic": traffic_of(dom, shape.name),
                     "algorithmic_per_launch": kw["bytes"] if roof["bound"] == "hbm" else kw["flops"]})

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights, U(-0.1,0.1) or Zipf bias)",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H, "E": shape.E, "k": shape.k,
                   "I": shape.I, "S": shape.S, "shared_packed": shape.shared_packed,
                   "hidden_act": shape.hidden_act, "mlp_norm": shape.mlp_norm,
                   "weight_format": shape.weight_format, "path": {1: "decode", 2: "grouped", 3: "swapped"}[path],
                   "parallelism": f"replicas{world}",
                   "l2": ("not flushed: inputs larger than L2" if args.no_flush else
                          "flushed before every step (256 MiB write), flush outside the timed events" +
                          ("; then a 256 MiB read, so the step starts with no dirty L2 lines"
                           if args.flush == "clean" else ""))},
        "roofline": roof,
        "block_roofline": {"t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2), "t_meas_us": round(ms * 1e3, 2),
                           "frac": round(max(t_tc, t_hbm) / (ms / 1e3), 4),
                           "bound": "tensor" if t_tc > t_hbm else "hbm", "flops": F, "bytes": B,
                           "experts_touched": U, "tflops": round(F / (ms / 1e3) / 1e12, 2),
                           "gbs": round(B / (ms / 1e3) / 1e9, 1), "peak_source": pk_src},
        "stage_us": {n: round(v * 1e3, 2) for n, v in stage_avg.items()},
        "timeline_us": timeline,
        "gemm_role_us": gemm_waits,
        "router_phase_us": router_phases,
        "e2e": {"value": round(job_throughput(shape.T, world, e2e_s), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": xbytes, "d2h_bytes_per_step": xbytes},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(shape, inputs, budget_s=args.cpu_seconds)
    blk.close()
    del inputs, X, Y, blk
    if world == 1 and args.other_configs:
        out["other_configs"] = other_configs(args, shape.name, dev, flush_l2)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# the other workloads of the block's configuration list, timed after the headline one
OTHER_CONFIGS = ("tiny", "nano_decode", "afmoe_prefill", "zipf_T1", "zipf_T8", "zipf_T64", "zipf_T512",
                 "zipf_T4096", "zipf_T16384")


def other_configs(args, headline: str, dev, flush_l2):
    """Step time, tokens/s, block roofline fraction and clocks of each other
    workload: the same timed steps as the headline (L2 flushed before each,
    CUDA events around the forward), repeated for at least 0.4 s."""
    import torch

    from expert_routed_ffn_gb300 import capi
    from expert_routed_ffn_gb300 import workloads as wl
    pk, _ = peaks()
    res = {}
    for name in OTHER_CONFIGS:
        shape = wl.WORKLOADS[name]
        if shape.name == headline:
            continue
        inputs = wl.make_inputs(shape, dev)
        blk = capi.block_from_inputs(shape, inputs, max_tokens=shape.T)
        X = inputs["X"]
        Y = torch.empty_like(X)

        def step():
            flush_l2()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            blk.forward(X, Y)
            e.record()
            return s, e

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        U = int(torch.unique(blk.inspect(capi.MOE_BUF_TOPK_IDX, shape.T * shape.k, torch.int32)).numel())
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            step()
            torch.cuda.synchronize()
        # at least other_steps timed steps and at least 0.4 s of them, so that the
        # clock sampler (every 100 ms) sees this workload under load
        sampler = ClockSampler(f"GPU-{torch.cuda.get_device_properties(dev).uuid}")
        evs = []
        t_end = time.perf_counter() + 0.4
        while len(evs) < args.other_steps or time.perf_counter() < t_end:
            evs.extend(step() for _ in range(args.other_steps))
            torch.cuda.synchronize()
        clocks = sampler.stop()
        if blk.sync_status() != capi.MOE_OK:
            raise SystemExit(f"device error while timing {name}")
        ms = sum(s.elapsed_time(e) for s, e in evs) / len(evs)
        F, B, _ = work_model(shape, U)
        t_tc, t_hbm = F / (pk["bf16_tflops"] * 1e12), B / (pk["hbm_gbs"] * 1e9)
        res[shape.name] = {"ms_per_step": round(ms, 5), "tokens_per_s": round(shape.T / (ms / 1e3), 1),
                           "block_roofline_frac": round(max(t_tc, t_hbm) / (ms / 1e3), 4),
                           "bound": "tensor" if t_tc > t_hbm else "hbm", "t_roof_us": round(max(t_tc, t_hbm) * 1e6, 2),
                           "experts_touched": U, "steps": len(evs), "clocks": clocks}
        blk.close()
        del inputs, X, Y, blk
        torch.cuda.empty_cache()
    return res


def traffic_of(stage: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel; else None."""
    import hashlib
    src = {"gate_up_gemm": "gemm_tc.cu", "down_gemm": "gemm_tc.cu", "experts_gemm": "gemm_tc.cu",
           "decode_gate_up": "stream.cu",
           "decode_down": "stream.cu", "gate_up_gemm_swapped": "gemm_sab.cu",
           "down_gemm_swapped": "gemm_sab.cu"}.get(stage)
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if src is None or not os.path.exists(path):
        return None
    with open(os.path.join(ROOT, "expert_routed_ffn_gb300", "csrc", src), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == stage and parts[1] == workload \
                    and parts[3] == sha:
                return int(float(parts[2]))
    return None


def cpu_baseline(shape, inputs, budget_s=10.0):
    """The fp64 oracle, as it stands, on the host cores: whole-workload passes
    (or a token sample of it) until about budget_s of wall time."""
    import torch

    import oracle
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}
    cores = os.cpu_count() or 1
    n = shape.T
    t0 = time.perf_counter()
    oracle.block_output(shape, host, tokens=list(range(min(n, cores))), nthreads=cores)
    per_tok = (time.perf_counter() - t0) / min(n, cores)
    n = max(1, min(shape.T, int(budget_s / 3 / max(per_tok, 1e-9))))
    toks = list(range(n))
    times = []
    t_start = time.perf_counter()
    while len(times) < 3 or time.perf_counter() - t_start < budget_s:
        t0 = time.perf_counter()
        oracle.block_output(shape, host, tokens=toks, nthreads=cores)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > 3 * budget_s:
            break
    med = statistics.median(times)
    # the same oracle on one thread, on a smaller token sample (about budget_s / 3)
    n1 = max(1, min(shape.T, int(budget_s / 9 / max(per_tok * min(shape.T, cores), 1e-9))))
    t1 = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.block_output(shape, host, tokens=list(range(n1)), nthreads=1)
        t1.append(time.perf_counter() - t0)
    return {"value": round(n / med, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"tokens 0..{n - 1} of the {shape.name} workload, {len(times)} passes, median",
            "one_thread": {"value": round(n1 / statistics.median(t1), 2), "unit": "tokens/s",
                           "sample": f"tokens 0..{n1 - 1}, 3 passes, median"}}


def run_reference(args, shape):
    """The fp64 CPU oracle as the reference arm, on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from expert_routed_ffn_gb300 import workloads as wl
    oracle.build()
    inputs = wl.make_inputs(shape, "cpu")
    cores = os.cpu_count() or 1
    # size each step to about one second of oracle work
    t0 = time.perf_counter()
    oracle.block_output(shape, inputs, tokens=list(range(min(shape.T, cores))), nthreads=cores)
    per_tok = (time.perf_counter() - t0) / min(shape.T, cores)
    n = max(1, min(shape.T, int(1.0 / max(per_tok, 1e-9))))
    toks = list(range(n))
    for _ in range(args.warmup):
        oracle.block_output(shape, inputs, tokens=toks, nthreads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.block_output(shape, inputs, tokens=toks, nthreads=cores)
        times.append(time.perf_counter() - t0)
    s = sum(times) / len(times)
    value = n / s
    sample = f"tokens 0..{n - 1} of the {shape.name} workload per step"
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H, "E": shape.E, "k": shape.k,
                   "I": shape.I, "S": shape.S, "mlp_norm": shape.mlp_norm, "tokens_per_step": n},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="m3",
                    help="workload of the headline line (default: the largest configuration, the MiniMax-M3 block)")
    ap.add_argument("--other-configs", type=int, choices=[0, 1], default=1,
                    help="also time the other configurations (one GPU only), under other_configs")
    ap.add_argument("--other-steps", type=int, default=20)
    ap.add_argument("--shape", action="append", default=[], metavar="KEY=VALUE",
                    help="override a field of the workload (e.g. T=256, num_experts=16) for a smaller "
                         "case of the same kernels, such as a profiler capture")
    ap.add_argument("--path", choices=["decode", "grouped", "swapped"], default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-pair", type=int, choices=[0, 1, 2], default=None,
                    help="CTA-pair expert GEMM: 0 never, 1 always, 2 by size (the default)")
    ap.add_argument("--two-launch", action="store_true", help="gate/up and down GEMMs as two launches")
    ap.add_argument("--no-prefetch", action="store_true", help="no L2 prefetch of expert weights while routing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--preroll", type=float, default=1.0, help="seconds of untimed steps before timing")
    ap.add_argument("--flush", choices=["write", "clean"], default="clean",
                    help="L2 flush before each step: a 256 MiB write, or the write and then a 256 MiB read")
    ap.add_argument("--no-flush", action="store_true",
                    help="skip the L2 flush between steps (only valid when the inputs exceed L2)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    from expert_routed_ffn_gb300 import workloads as wl
    shape = wl.WORKLOADS[args.workload]
    if args.shape:
        kw = {}
        for item in args.shape:
            key, val = item.split("=", 1)
            cur = getattr(shape, key)
            kw[key] = val in ("1", "true", "True") if isinstance(cur, bool) else type(cur)(val)
        shape = shape.replace(name=shape.name + "_" + "_".join(args.shape), **kw)
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the EFLA chunked forward (and decode step) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one efla_fwd_chunked call over the language-model-layer workload
(B=8, H=16, T=2048, d_k=d_v=128, bf16 q/k/v, fp32 beta, S0 = 0, o in the dtype
of q (bf16), fp32 S_T, chunk 64) with inputs resident in HBM.  L2 is flushed (a 512 MiB write)
before every timed step; each step is bracketed by CUDA events on the
launching stream.  Prints ONE JSON line on rank 0.

Under torchrun (N > 1) every rank runs an independent replica of the workload
(the (sequence, head) units are independent, no collective is needed); value =
tokens of all ranks / max-over-ranks time.

--impl reference times the fp64 CPU oracle on the host cores (rank 0 only) on
a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "EFLA chunked fwd tokens/s & TFLOP/s (H16 d128 T2048), % roofline; decode GB/s"
WORKLOAD = "lm"
CHUNK = 64


def flops_per_token_head(dk: int, dv: int, C: int = CHUNK) -> float:
    """Algorithmic flop count per token-head: 6 d_k d_v (state products) +
    3 C d_k + 2 C d_v (intra-chunk products) + C^2/3 (triangular inverse)."""
    return 6 * dk * dv + 3 * C * dk + 2 * C * dv + C * C / 3.0


def fwd_bytes(B, T, H, dk, dv, N, in_bytes=2, o_bytes=2, s0=False, s_t=True) -> int:
    """Algorithmic bytes: every input read once, every output written once (o in the
    input dtype: 1028 B per token-head at d = 128 bf16, plus S0 and S_T per unit)."""
    th = B * T * H
    b = th * (2 * dk * in_bytes + dv * in_bytes + 4 + dv * o_bytes)
    st = N * H * dk * dv * 4
    return b + (st if s0 else 0) + (st if s_t else 0)


def decode_bytes(B, H, dk, dv, in_bytes=2, o_bytes=2) -> int:
    u = B * H
    return u * ((2 * dk + dv) * in_bytes + 4 + dv * o_bytes + 2 * dk * dv * 4)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def profile_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of the kernel (every source_file / source_sha256 pair it
    lists, the kernel's file and the headers it includes; else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    pairs = re.findall(r"source_file:\s*(\S+)\s*\nsource_sha256:\s*([0-9a-f]{64})", text)
    if not (m_b and pairs):
        return None
    for f, sha in pairs:
        src = os.path.join(ROOT, f)
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != sha:
            return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"efla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


def dist_init():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(inp, units, threads, min_seconds=0.0, max_reps=1):
    """Time the fp64 oracle on a list of (b, h) units of a fixed-length workload, repeated
    until `min_seconds` of CPU work (at most `max_reps` passes); returns (seconds, token-heads)."""
    import oracle
    q, k, v, beta = inp["q"], inp["k"], inp["v"], inp["beta"]
    bs = sorted({b for b, _ in units})
    hs = sorted({h for _, h in units})
    # contiguous fp64 copies of the sampled rows/heads (not timed)
    sub = [x[bs][:, :, hs].double().numpy() for x in (q, k, v)]
    sb = beta[bs][:, :, hs].double().numpy()
    reps, dt = 0, 0.0
    while reps < max(1, max_reps) and (reps == 0 or dt < min_seconds):
        t0 = time.perf_counter()
        oracle.fwd(sub[0], sub[1], sub[2], sb, None, threads=threads)
        dt += time.perf_counter() - t0
        reps += 1
    return dt, reps * len(bs) * len(hs) * q.shape[1]


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    import workloads
    cfg = workloads.FWD_WORKLOADS[WORKLOAD]
    inp = workloads.make_fwd_inputs(cfg)
    cores = os.cpu_count() or 1
    oracle.build()
    # each step: 2 batch rows x 8 heads = 16 (b, h) units = 32768 token-heads
    units = [(b, h) for b in (0, 1) for h in range(8)]
    for _ in range(args.warmup):
        oracle_sample(inp, units[:cores] if len(units) > cores else units, cores)
    times, toks = [], 0
    for _ in range(args.steps):
        dt, n = oracle_sample(inp, units, cores)
        times.append(dt)
        toks += n
    total = sum(times)
    value = toks / total / cfg.H  # tokens/s: a token is one position of all H heads
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: EFLA forward B8 H16 T2048 d128 (sample: 16 (b,h) units per step)",
                   "sample_units_per_step": len(units)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "16 (batch row, head) units x 2048 tokens per step, fp64 C oracle, "
                                   "OpenMP over units"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    import exact_delta_rule_gb300 as efla
    import workloads
    from exact_delta_rule_gb300 import build as libbuild

    libbuild.build()
    efla.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = workloads.FWD_WORKLOADS[WORKLOAD]
    inp = workloads.make_fwd_inputs(cfg)
    B, T, H, dk, dv, N = inp["B"], inp["T"], inp["H"], cfg.dk, cfg.dv, inp["N"]
    q, k, v, beta = (inp[x].to(dev) for x in ("q", "k", "v", "beta"))
    o = torch.empty((B, T, H, dv), dtype=q.dtype, device=dev)  # o in the dtype of q
    S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    if args.leg != "all":  # one secondary figure alone (profiling runs); no contract line
        print(json.dumps({args.leg: run_leg(args, efla, dev, stream, flush, q, k, v, beta)}), flush=True)
        return

    def step():
        efla.fwd_chunked(q, k, v, beta, None, None, o=o, S_T=S_T, chunk=CHUNK, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if efla.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    per_step = [a.elapsed_time(b) / 1e3 for a, b in evs]
    t_local = sum(per_step)
    t_max = max_over_ranks(t_local, world)
    tokens = B * T * H  # token-heads per step
    value = world * tokens * args.steps / t_max / H  # tokens/s (a token = one position of all H heads)
    ms_per_step = 1e3 * t_max / args.steps

    peaks = read_peaks()
    nbytes = fwd_bytes(B, T, H, dk, dv, N)
    avg = t_local / args.steps
    achieved_gbs = nbytes / avg / 1e9
    flops = flops_per_token_head(dk, dv) * tokens
    traffic = profile_traffic("chunk_tc_lm")

    # ---- end to end through host buffers (pinned), copies inside the timed region
    hq, hk, hv, hb = (x.cpu().pin_memory() for x in (inp["q"], inp["k"], inp["v"], inp["beta"]))
    # Two sets of device buffers and of pinned host outputs: the copy-in of step i + 1 and the
    # copy-out of step i - 1 run on their own streams while step i computes (a serving
    # pipeline).  Every step still moves its inputs in and its results out inside the timed
    # region.
    e_steps = max(3, min(args.steps, 10))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    dev_sets = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v), b=torch.empty_like(beta),
                     o=torch.empty_like(o), S=torch.empty_like(S_T)) for _ in range(2)]
    host_out = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(), torch.empty(S_T.shape, dtype=S_T.dtype).pin_memory())
                for _ in range(2)]
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "comp", "out")}

    def e2e_run(n):
        for i in range(n):
            d, (ho, hs) = dev_sets[i % 2], host_out[i % 2]
            if i >= 2:
                s_in.wait_event(ev["comp"][i % 2])  # step i-2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                d["q"].copy_(hq, non_blocking=True)
                d["k"].copy_(hk, non_blocking=True)
                d["v"].copy_(hv, non_blocking=True)
                d["b"].copy_(hb, non_blocking=True)
            ev["in"][i % 2].record(s_in)
            stream.wait_event(ev["in"][i % 2])
            if i >= 2:
                stream.wait_event(ev["out"][i % 2])  # step i-2's outputs have left these buffers
            efla.fwd_chunked(d["q"], d["k"], d["v"], d["b"], None, None, o=d["o"], S_T=d["S"], chunk=CHUNK,
                             stream=stream)
            ev["comp"][i % 2].record(stream)
            s_out.wait_event(ev["comp"][i % 2])
            with torch.cuda.stream(s_out):
                ho.copy_(d["o"], non_blocking=True)
                hs.copy_(d["S"], non_blocking=True)
            ev["out"][i % 2].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    e2e_run(e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    ho, hs = host_out[0]
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hb))
    d2h = ho.numel() * ho.element_size() + hs.numel() * hs.element_size()

    # ---- decode step (secondary figure): B256 H32 d128, CUDA graph of chained steps
    dec = decode_figures(efla, dev, stream)

    # ---- the same forward with the delta-rule (DeltaNet) gate, L2-normalised keys
    kn = (k.float() / k.float().norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(k.dtype)
    t_dn = time_steps(lambda: efla.fwd_chunked(q, kn, v, beta, None, None, o=o, S_T=S_T, chunk=CHUNK,
                                               stream=stream, update="euler"), args.steps, flush, stream)
    deltanet = {"workload": "lm shape, delta-rule gate alpha = beta, unit-norm keys",
                "ms_per_step": 1e3 * t_dn, "tokens_per_s": tokens / H / t_dn,
                "efla_time_over_deltanet_time": avg / t_dn}

    # ---- prep kernel: lambda, alpha, alpha*k, alpha*v for every token-head of the lm workload
    t_pr = time_steps(lambda: efla.prep(k, beta, v, lam=True, alpha=True, ak=True, av=True, stream=stream),
                      args.steps, flush, stream)
    pr_bytes = tokens * (2 * dk * 2 + 2 * dv * 2 + 12)
    prep_fig = {"workload": "lm: 262144 token-head rows, bf16 k, v in, lambda/alpha fp32 and alpha*k, alpha*v bf16 out",
                "us_per_call": 1e6 * t_pr, "GB/s": pr_bytes / t_pr / 1e9, "bytes_per_call": pr_bytes,
                "frac_hbm": pr_bytes / t_pr / 1e9 / peaks["hbm_gbs"]}

    # ---- multi-token decode: 16 tokens per sequence appended to the B256 H32 state
    dt_fig = decode_tokens_figure(efla, dev, stream, args.steps, flush, peaks)

    # ---- backward pass on the lm shape (dO random, dS_T random)
    bwd_fig = bwd_figure(efla, dev, stream, q, k, v, beta, flush, peaks)

    # ---- the stiff/long configuration: one sequence per head, unsplit and split along time
    stiff_fig = stiff_figure(efla, dev, stream, max(3, args.steps // 2), flush, peaks)

    # ---- the packed variable-length configuration
    varlen_fig = varlen_figure(efla, dev, stream, max(3, args.steps // 2), flush, peaks)

    # ---- CPU baseline: the oracle on a bounded sample of the same workload
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "precision": "bf16 inputs and o; tensor-core operands split into bf16 hi+lo; fp32 state and accumulation",
            "data": "synthetic",
            "config": {"workload": "lm: EFLA chunked forward B=8 H=16 T=2048 d_k=d_v=128, bf16 q,k,v, fp32 beta, "
                                   "S0=0, o bf16 (the dtype of q), S_T fp32, chunk 64",
                       "B": B, "T": T, "H": H, "d_k": dk, "d_v": dv, "chunk": CHUNK,
                       "l2": "flushed (512 MiB write) before every timed step",
                       "parallelism": f"replicas x{world}"},
            "token_heads_per_s": world * tokens * args.steps / t_max,
            "tflops": flops / avg / 1e12,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes_per_launch": nbytes,
                         "bytes_per_token_head": "q,k,v 768 + beta 4 + o 256 = 1028 (bf16), plus S_T 64 KiB per unit",
                         "peak_source": f"{peaks['source']} hbm_gbs (copy burst)",
                         "kernel": "efla chunk kernel (one launch per step)",
                         "t_roof_us": 1e6 * max(nbytes / (peaks["hbm_gbs"] * 1e9),
                                                flops / (peaks["bf16_tflops"] * 1e12))},
            "e2e": {"value": world * tokens * e_steps / t_e2e / H, "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
                    "pipeline": "pinned host inputs -> device, fwd_chunked, o and S_T -> pinned host, on three "
                                "streams with double-buffered device and host tensors"},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "decode": dec,
            "deltanet": deltanet,
            "prep": prep_fig,
            "decode_tokens": dt_fig,
            "stiff": stiff_fig,
            "varlen": varlen_fig,
            "bwd": bwd_fig,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_leg(args, efla, dev, stream, flush, q, k, v, beta):
    peaks = read_peaks()
    if args.leg == "decode":
        return decode_figures(efla, dev, stream)
    if args.leg == "decode_tokens":
        return decode_tokens_figure(efla, dev, stream, args.steps, flush, peaks)
    if args.leg == "bwd":
        return bwd_figure(efla, dev, stream, q, k, v, beta, flush, peaks)
    if args.leg == "stiff":
        return stiff_figure(efla, dev, stream, max(3, args.steps // 2), flush, peaks)
    return varlen_figure(efla, dev, stream, max(3, args.steps // 2), flush, peaks)


def time_steps(fn, steps, flush, stream):
    """Average seconds of `fn` over `steps` calls, L2 flushed before each, CUDA events."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    total = 0.0
    for i in range(steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        total += a.elapsed_time(b) / 1e3
    return total / steps


def decode_figures(efla, dev, stream):
    """Decode: 1000 chained efla_decode_step calls on the B256 H32 state, each step with its
    own inputs (drawn on the device beforehand from seed (4 << 32) + step, the workload's laws),
    captured in one CUDA graph; the state (512 MiB) exceeds L2."""
    import torch

    import workloads
    cfg = workloads.DECODE
    S = workloads.make_decode_state(cfg).to(dev)
    n = cfg.steps
    shp = (cfg.B, cfg.H)
    ins = []
    for i in range(n):
        gen = torch.Generator(device=dev)
        gen.manual_seed((cfg.seed << 32) + i)
        ins.append([torch.randn(shp + (cfg.dk,), generator=gen, device=dev).to(torch.bfloat16),
                    torch.randn(shp + (cfg.dk,), generator=gen, device=dev).to(torch.bfloat16),
                    torch.randn(shp + (cfg.dv,), generator=gen, device=dev).to(torch.bfloat16),
                    torch.sigmoid(torch.randn(shp, generator=gen, device=dev))])
    o = torch.empty((cfg.B, cfg.H, cfg.dv), dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(3):
            efla.decode_step(*ins[i], S, o=o, stream=side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(n):
            efla.decode_step(*ins[i], S, o=o, stream=side)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 2
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / (reps * n)
    nbytes = decode_bytes(cfg.B, cfg.H, cfg.dk, cfg.dv)
    peaks = read_peaks()
    del ins
    return {"workload": f"decode: B=256 H=32 d=128 bf16 q,k,v and o, fp32 S in place; a CUDA graph of {n} "
                        f"chained steps, each with its own inputs (drawn on the device from seed (4<<32)+step); "
                        f"S (512 MiB) exceeds L2",
            "us_per_step": 1e6 * t, "GB/s": nbytes / t / 1e9, "bytes_per_step": nbytes,
            "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"], "gpu_launches": reps * n}


def bwd_figure(efla, dev, stream, q, k, v, beta, flush, peaks, steps=3):
    import torch
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    g = torch.Generator(device=dev).manual_seed(7)
    dO = torch.randn((B, T, H, dv), generator=g, device=dev)
    dST = torch.randn((B, H, dk, dv), generator=g, device=dev)
    ws = torch.empty(efla.bwd_workspace(B, T, H, dk, dv), dtype=torch.uint8, device=dev)
    t = time_steps(lambda: efla.bwd_chunked(q, k, v, beta, None, dO, dST, workspace=ws, stream=stream), steps,
                   flush, stream)
    t_rec = time_steps(lambda: efla.bwd_recurrent(q, k, v, beta, None, dO, dST, stream=stream), 1, flush, stream)
    # training: the forward that keeps the chunk-start states and T'' for the backward, and the
    # backward from them (the workspace is not changed by the backward, so the timed calls reuse it)
    o_t = torch.empty_like(q)
    S_t = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    t_train = time_steps(lambda: efla.fwd_chunked_train(q, k, v, beta, None, workspace=ws, o=o_t, S_T=S_t,
                                                        stream=stream), steps, flush, stream)
    t_saved = time_steps(lambda: efla.bwd_chunked(q, k, v, beta, None, dO, dST, workspace=ws, saved=True,
                                                  stream=stream), steps, flush, stream)
    th = B * T * H
    # each input read once and each output written once: q, k, v bf16 + beta + dO fp32 in; dq, dk, dv fp32 +
    # dbeta out; dS_T in and dS0 out per (b, h)
    nbytes = th * ((dk + dk + dv) * 2 + 4 + dv * 4 + (dk + dk + dv) * 4 + 4) + 2 * B * H * dk * dv * 4
    ws_bytes = ws.numel()
    return {"workload": "lm shape backward (B=8 H=16 T=2048 d=128, bf16 q,k,v): dq, dk, dv, dbeta, dS0 (fp32) "
                        "from random dO and dS_T (fp32), chunks of 64",
            "ms_per_call": 1e3 * t, "tokens_per_s": B * T / t, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
            "workspace_bytes": ws_bytes,
            "path": "forward on the tensor cores writing every chunk-start state and T'' (workspace); dO split "
                    "into bf16 hi/lo; reverse pass over chunks for the end-state gradients on the tensor cores (one "
                    "CTA per (b, h)), also writing G, dv and -dR (hi/lo); per-chunk gradients on the tensor cores "
                    "(persistent CTAs over the (b, h, chunk) items)",
            "ms_recurrent": 1e3 * t_rec,
            "training": {"ms_forward_keeping_states": 1e3 * t_train, "ms_backward_from_saved": 1e3 * t_saved,
                         "ms_step": 1e3 * (t_train + t_saved),
                         "note": "efla_fwd_chunked_train then efla_bwd_chunked_saved: the backward does not "
                                 "run the forward again"},
            "gpu_launches": 4 * steps + 1 + steps + 3 * steps}


def stiff_figure(efla, dev, stream, steps, flush, peaks):
    import torch

    import workloads
    cfg = workloads.FWD_WORKLOADS["stiff"]
    inp = workloads.make_fwd_inputs(cfg)
    g = {x: inp[x].to(dev) for x in ("q", "k", "v", "beta", "S0")}
    B, T, H, dk, dv = cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    need, G = efla.scan_workspace(B, T, H, dk, dv, 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    t_plain = time_steps(lambda: efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o=o, S_T=S_T,
                                                  stream=stream), steps, flush, stream)
    t_scan = time_steps(lambda: efla.fwd_chunked_scan(g["q"], g["k"], g["v"], g["beta"], g["S0"], o=o, S_T=S_T,
                                                      workspace=ws, stream=stream), steps, flush, stream)
    tokens = B * T
    nbytes = fwd_bytes(B, T, H, dk, dv, B, s0=True)
    return {"workload": "stiff: B=1 H=16 T=65536 d=128 bf16, key norms U[0.1,10], beta=sigmoid(N(2,1)), "
                        "S0~0.1 N(0,1), o bf16, S_T fp32",
            "ms_unsplit": 1e3 * t_plain, "tokens_per_s_unsplit": tokens / t_plain,
            "ms_split": 1e3 * t_scan, "tokens_per_s_split": tokens / t_scan, "segments": G,
            "speedup": t_plain / t_scan, "algorithmic_bytes": nbytes,
            "frac_hbm_unsplit": nbytes / t_plain / 1e9 / peaks["hbm_gbs"],
            "frac_hbm_split": nbytes / t_scan / 1e9 / peaks["hbm_gbs"],
            "gpu_launches": 3 * steps + steps}


def varlen_figure(efla, dev, stream, steps, flush, peaks):
    """The packed variable-length workload: 64 sequences of U{1..8192} tokens, H8 d128 bf16,
    per-sequence S0; one launch, one CTA per (sequence, head), in sequence order (no
    longest-first ordering)."""
    import torch

    import workloads
    cfg = workloads.FWD_WORKLOADS["varlen"]
    inp = workloads.make_fwd_inputs(cfg)
    g = {x: inp[x].to(dev) for x in ("q", "k", "v", "beta", "S0", "cu_seqlens")}
    B, T, H, N, dk, dv = inp["B"], inp["T"], inp["H"], inp["N"], cfg.dk, cfg.dv
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    t = time_steps(lambda: efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["cu_seqlens"], o=o,
                                            S_T=S_T, stream=stream), steps, flush, stream)
    nbytes = fwd_bytes(B, T, H, dk, dv, N, s0=True) + (N + 1) * 4
    lens = [int(inp["cu_seqlens"][i + 1] - inp["cu_seqlens"][i]) for i in range(N)]
    return {"workload": f"varlen: {N} sequences, lengths U{{1..8192}} (seeded; {T} tokens, longest {max(lens)}), "
                        f"H=8 d=128 bf16, per-sequence S0~0.1 N(0,1), o bf16, S_T fp32",
            "ms_per_call": 1e3 * t, "tokens_per_s": T / t, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
            "tflops": flops_per_token_head(dk, dv) * T * H / t / 1e12,
            "scheduling": "one CTA per (sequence, head), longest sequence first (each CTA ranks the lengths)",
            "gpu_launches": steps}


def decode_tokens_figure(efla, dev, stream, steps, flush, peaks, m=16):
    import workloads
    cfg = workloads.DECODE
    S = workloads.make_decode_state(cfg).to(dev)
    inp = workloads.make_decode_tokens(m, cfg)
    g = [inp[x].to(dev) for x in ("q", "k", "v", "beta")]
    import torch
    o = torch.empty((cfg.B, m, cfg.H, cfg.dv), dtype=torch.bfloat16, device=dev)
    t = time_steps(lambda: efla.decode_tokens(*g, S, o=o, stream=stream), steps, flush, stream)
    u = cfg.B * cfg.H
    nbytes = u * (m * ((2 * cfg.dk + cfg.dv) * 2 + 4 + cfg.dv * 2) + 2 * cfg.dk * cfg.dv * 4)
    return {"workload": f"decode_tokens: B=256 H=32 d=128, {m} tokens per sequence per call, bf16 q,k,v and o, "
                        f"fp32 S in place (read and written once)",
            "us_per_call": 1e6 * t, "tokens_per_s": cfg.B * m / t, "GB/s": nbytes / t / 1e9,
            "bytes_per_call": nbytes, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
            "gpu_launches": steps}


def cpu_baseline(inp):
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    units = [(b, h) for b in range(8) for h in range(16)]
    dt, th = oracle_sample(inp, units, cores, min_seconds=10.0, max_reps=60)
    reps = th // (len(units) * 2048)
    return {"value": th / dt / 16, "unit": "tokens/s", "token_heads_per_s": th / dt,
            "cores": cores, "kind": "oracle",
            "sample": f"all {len(units)} (batch row, head) units x 2048 tokens of one lm step, repeated {reps}x "
                      f"(>= 10 s of CPU work), fp64 C oracle, OpenMP over units", "seconds": dt}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--leg", choices=["all", "decode", "decode_tokens", "bwd", "stiff", "varlen"], default="all",
                    help="run one secondary figure alone and print it (for profiling); 'all' is the bench")
    args = ap.parse_args()
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

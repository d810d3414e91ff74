"""Benchmark of the NVFP4 routed-MoE expert forward (route + forward) on GB300.

Default workload: the Qwen3.6-35B-A3B-shaped MoE layer in the decode regime (H=2048,
E=256, top-8, I=512, shared expert 512, group 16), T=64 tokens, seed 0. One step
runs 40 distinct layer copies (same bytes, distinct addresses, each with its own
routing), so the touched weights of a step (~16 GB) are far larger than the 129 MB
L2 and every layer streams its experts from HBM. One step is captured once in a
CUDA graph and replayed.

Metric: MoE-layer tokens/s = T * layers / step time. The JSON line also carries the
roofline of the dominant kernel (algorithmic weight bytes / its average launch
duration, from CUDA events recorded on the launch stream inside the graph), the
oracle's CPU throughput, an end-to-end number with host buffers, and SM clocks.

`--impl reference` times the CPU oracle (the reference arm of this build) on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s; decode weight-stream HBM GB/s & prefill TFLOPS vs roofline"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.lines, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(value: float, dev=None) -> float:
    """Largest value over the ranks of the default process group (the value itself when
    there is none): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev if dev is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(tokens_per_step_per_rank: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput under weak scaling: all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_step_per_rank * steps / (max_ms / 1e3)


def run_reference(args, world, rank):
    """CPU oracle on a bounded sample of the workload (the reference arm)."""
    import oracle
    oracle.build()
    if rank != 0:
        return
    shape = synth.SHAPES[args.shape]
    routed = synth.make_pieces(shape, 0)
    shared = synth.make_pieces(shape, 0, shared=True)
    rb, sb = oracle.slice_bank(routed, shape.group), oracle.slice_bank(shared, shape.group)
    cores = oracle.default_threads()
    T = args.T
    tok = min(T, args.ref_tokens)
    times = []
    for step in range(args.warmup + args.steps):
        logits = synth.make_logits(T, shape.num_experts, seed=step % args.layers)
        x = synth.make_activations(T, shape.hidden, seed=step % args.layers)
        t0 = time.perf_counter()
        ids, w = oracle.route(logits, shape.top_k)
        oracle.moe_forward(rb, sb, shape.group, x, ids, w, tokens=np.arange(tok), nthreads=cores)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    value = tok * len(times) / sum(times)
    sample = f"{tok} of the {T} tokens of one layer per step, route + forward, {cores} threads"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _expert_bytes(shape, inter):
    """Algorithmic bytes of one NVFP4 expert of intermediate width `inter` (tp=1): gate_up and
    down codes, e4m3 block scales and fp32 row globals."""
    H, g = shape.hidden, shape.group
    gate_up = 2 * inter * H // 2 + 2 * inter * H // g + 2 * inter * 4
    down = H * inter // 2 + H * inter // g + H * 4
    return gate_up, down


def _sources_sha256(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic(stage):
    """DRAM bytes (read + write) per launch of the stage's kernel from the committed ncu
    capture (profiles/kernel_traffic.json), or None when that kernel's sources have
    changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "kernel_traffic.json")) as f:
            rec = json.load(f).get(stage)
        if rec and _sources_sha256(rec["sources"]) == rec["sources_sha256"]:
            return rec
    except (OSError, ValueError, KeyError):
        pass
    return None


def _config(args):
    sh = synth.SHAPES[args.shape]
    return {"workload": f"{args.shape}-moe-decode-T{args.T}", "T": args.T, "layers": args.layers,
            "hidden": sh.hidden, "num_experts": sh.num_experts, "top_k": sh.top_k, "intermediate": sh.intermediate,
            "shared_intermediate": sh.shared_intermediate, "group": sh.group,
            "tp": 1, "seed": 0, "routing": "N(0,1) logits",
            "l2": f"inputs larger than L2: {args.layers} distinct layer copies per step"}


def cpu_baseline(T, shape, budget_s=10.0):
    import oracle
    oracle.build()
    routed = synth.make_pieces(shape, 0)
    shared = synth.make_pieces(shape, 0, shared=True)
    rb, sb = oracle.slice_bank(routed, shape.group), oracle.slice_bank(shared, shape.group)
    cores = oracle.default_threads()
    tokens, layers, t_total = 0, 0, 0.0
    while t_total < budget_s and layers < 40:
        logits = synth.make_logits(T, shape.num_experts, seed=layers)
        x = synth.make_activations(T, shape.hidden, seed=layers)
        t0 = time.perf_counter()
        ids, w = oracle.route(logits, shape.top_k)
        oracle.moe_forward(rb, sb, shape.group, x, ids, w, nthreads=cores)
        t_total += time.perf_counter() - t0
        tokens += T
        layers += 1
    return {"value": tokens / t_total, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{layers} layers x {T} tokens (route + forward, fp64), {t_total:.1f} s"}


def _cold_l2(buf, r):
    """Evicts L2 before a timed repetition: writes the whole 512 MB buffer, then reads its
    first 256 MB back, so that the dirty lines the writes leave are written back here and
    L2 holds clean lines of an unrelated buffer when the timed work starts."""
    import torch
    buf.fill_(r & 0xFF)
    buf[: 256 << 20].view(torch.int32).sum()


def measure_prefill(ft, dev, cfg, shape, routed_d, shared_d, T, reps=6):
    """One layer of `shape` at T tokens (Zipf routing), L2 flushed before every repetition."""
    import torch
    rb, sb = ft.alloc_banks(cfg, 0, dev), ft.alloc_banks(cfg, 1, dev)
    ft.ft_moe_pack(cfg, 0, routed_d, rb)
    ft.ft_moe_pack(cfg, 1, shared_d, sb)
    H, E, k = shape.hidden, shape.num_experts, shape.top_k
    x = torch.from_numpy(synth.make_activations(T, H, seed=7).view(np.int16)).to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(synth.zipf_logits(T, E, seed=7)).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(ft.ft_moe_workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    n_ev = ft.FT_NSTAGES + 1
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream(dev)
    for e_ in ev:
        e_.record(stream)
    times, stages = [], []
    for r in range(reps + 2):
        _cold_l2(flush, r)
        start.record(stream)
        ft.ft_moe_route(lg, k, ids, w)
        ft.ft_moe_set_stage_events(ev)
        ft.ft_moe_forward(cfg, rb, sb, x, ids, w, out, ws)
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if r >= 2:
            times.append(start.elapsed_time(stop))
            stages.append([ev[i].elapsed_time(ev[i + 1]) for i in range(ft.FT_NSTAGES)])
    assert ft.ft_moe_read_status(ws) == 0
    ms = float(np.median(times))
    # 2 * 3 * H * I per routed expert x k, plus the shared expert's 2 * 3 * H * I_s, per token
    flops = 6.0 * H * (k * shape.intermediate + shape.shared_intermediate) * T
    _, tfl, peak_kind = _peaks()
    st = np.median(np.array(stages), axis=0)
    counts = np.bincount(ids.cpu().numpy().reshape(-1), minlength=E)
    del rb, sb, ws, flush
    return {"T": T, "routing": "zipf(1.1)", "us": ms * 1e3, "tokens_per_s": T / (ms / 1e3),
            "tflops": flops / (ms / 1e3) / 1e12, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / tfl,
            "peak_source": f"{peak_kind} bf16 dense", "l2": "512 MB written, then 256 MB read back, before every repetition",
            "stage_us": {n: float(v * 1e3) for n, v in zip(ft.STAGES, st)},
            "expert_tokens_max_over_mean": float(counts.max() / counts.mean())}


def measure_w4a4(ft, dev, cfg, rb, sb, shape, T, reps=5):
    """The W4A4 variant (NVFP4 activations, block-scaled FP4 tensor cores) on one prefill layer,
    Zipf routing, L2 flushed before every repetition; TFLOP/s against the FP4 dense peak taken
    as the measured bf16 peak times the nominal FP4 / bf16 ratio (13.5 / 2.25)."""
    import torch
    H, E, k = shape.hidden, shape.num_experts, shape.top_k
    x = torch.from_numpy(synth.make_activations(T, H, seed=7).view(np.int16)).to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(synth.zipf_logits(T, E, seed=7)).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(ft.ft_moe_workspace_size_w4a4(cfg, T), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    n_ev = ft.FT_NSTAGES + 1
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream(dev)
    for e_ in ev:
        e_.record(stream)
    times, stages = [], []
    for r in range(reps + 2):
        _cold_l2(flush, r)
        start.record(stream)
        ft.ft_moe_route(lg, k, ids, w)
        ft.ft_moe_set_stage_events(ev)
        ft.ft_moe_forward_w4a4(cfg, rb, sb, x, ids, w, out, ws)
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if r >= 2:
            times.append(start.elapsed_time(stop))
            stages.append([ev[i].elapsed_time(ev[i + 1]) for i in range(ft.FT_NSTAGES)])
    assert ft.ft_moe_read_status(ws) == 0
    ms = float(np.median(times))
    flops = 6.0 * H * (k * shape.intermediate + shape.shared_intermediate) * T
    _, tfl, kind = _peaks()
    fp4_peak = tfl * 13.5 / 2.25
    st = np.median(np.array(stages), axis=0)
    del ws, flush
    return {"T": T, "routing": "zipf(1.1)", "us": ms * 1e3, "tokens_per_s": T / (ms / 1e3),
            "tflops": flops / (ms / 1e3) / 1e12, "fp4_peak_tflops": fp4_peak,
            "frac_of_fp4_peak": flops / (ms / 1e3) / 1e12 / fp4_peak,
            "peak_source": f"{kind} bf16 dense x 13.5 / 2.25 (nominal FP4 / bf16)",
            "stage_us": {n: float(v * 1e3) for n, v in zip(ft.STAGES, st)},
            "kernel": "tcgen05 kind::mxf4nvf4 (e2m1 x e2m1, ue4m3 block scales), NVFP4 activations"}


def measure_router(ft, dev, T, E=256, H=2048, reps=6):
    """ft_moe_route_gemm (router logit GEMM + top-8) for one layer's router, L2 flushed."""
    import torch
    x = torch.from_numpy(synth.make_activations(T, H, seed=5).view(np.int16)).to(dev).view(torch.bfloat16)
    wr = torch.from_numpy(synth.make_router_weights(E, H, seed=5).view(np.int16)).to(dev).view(torch.bfloat16)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
    w = torch.empty((T, 8), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream(dev)
    times = []
    for r in range(reps + 2):
        _cold_l2(flush, r)
        start.record(stream)
        ft.ft_moe_route_gemm(x, wr, 8, logits, ids, w)
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if r >= 2:
            times.append(start.elapsed_time(stop))
    us = float(np.median(times)) * 1e3
    del flush
    return {"T": T, "E": E, "H": H, "us": us, "weight_gbs": E * H * 2 / (us * 1e-6) / 1e9,
            "tflops": 2.0 * T * E * H / (us * 1e-6) / 1e12, "l2": "512 MB written, then 256 MB read back, before every repetition"}


def measure_fp8(ft, dev, T=64, L=16, reps=20, T_prefill=2048):
    """fp8_block experts (the Qwen3.6-FP8 geometry): decode layer time over L distinct layer
    copies (captured in a CUDA graph, inputs larger than L2) and one prefill layer."""
    import torch
    shape = synth.SHAPES["qwen36_fp8"]
    cfg = ft.MoEConfig.of(shape)
    H, E, k = shape.hidden, shape.num_experts, shape.top_k
    routed = {n: torch.from_numpy(v).to(dev) for n, v in synth.make_fp8_pieces(shape, 0).items()}
    shared = {n: torch.from_numpy(v).to(dev) for n, v in synth.make_fp8_pieces(shape, 0, shared=True).items()}
    layers = []
    for _ in range(L):
        rb, sb = ft.alloc_banks(cfg, 0, dev), ft.alloc_banks(cfg, 1, dev)
        ft.ft_moe_pack(cfg, 0, routed, rb)
        ft.ft_moe_pack(cfg, 1, shared, sb)
        layers.append((rb, sb))
    del routed, shared
    x = torch.from_numpy(np.stack([synth.make_activations(T, H, seed=l) for l in range(L)]).view(np.int16)).to(dev)
    x = x.view(torch.bfloat16)
    lg = torch.from_numpy(np.stack([synth.make_logits(T, E, seed=l) for l in range(L)])).to(dev)
    ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    out = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(ft.ft_moe_workspace_size(cfg, T_prefill), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        for l in range(L):
            ft.ft_moe_route(lg[l], k, ids[l], w[l])
            ft.ft_moe_forward(cfg, layers[l][0], layers[l][1], x[l], ids[l], w[l], out[l], ws)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize(dev)
    assert ft.ft_moe_read_status(ws) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for _ in range(3):
            g.replay()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        stop.record(stream)
    torch.cuda.synchronize(dev)
    us_layer = start.elapsed_time(stop) * 1e3 / (reps * L)
    ids_np = ids.cpu().numpy()
    per_expert = 2 * 512 * 2048 + 8 * 16 * 4 + 2048 * 512 + 16 * 4 * 4
    layer_bytes = float(np.mean([(len(np.unique(ids_np[l])) + 1) * per_expert for l in range(L)]))
    hbm, _, kind = _peaks()
    decode = {"T": T, "layers": L, "us_per_layer": us_layer, "tokens_per_s": T / (us_layer * 1e-6),
              "weight_gbs": layer_bytes / (us_layer * 1e-6) / 1e9,
              "frac_of_hbm": layer_bytes / (us_layer * 1e-6) / 1e9 / hbm,
              "weight_bytes_per_layer": layer_bytes, "bytes_per_expert": per_expert,
              "peak_source": f"{kind} HBM copy bandwidth"}
    # one prefill layer, L2 flushed before every repetition
    xp = torch.from_numpy(synth.make_activations(T_prefill, H, seed=7).view(np.int16)).to(dev).view(torch.bfloat16)
    lgp = torch.from_numpy(synth.zipf_logits(T_prefill, E, seed=7)).to(dev)
    idp = torch.empty((T_prefill, k), dtype=torch.int32, device=dev)
    wp = torch.empty((T_prefill, k), dtype=torch.float32, device=dev)
    outp = torch.empty((T_prefill, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    times = []
    cur = torch.cuda.current_stream(dev)
    for r in range(6):
        _cold_l2(flush, r)
        start.record(cur)
        ft.ft_moe_route(lgp, k, idp, wp)
        ft.ft_moe_forward(cfg, layers[0][0], layers[0][1], xp, idp, wp, outp, ws)
        stop.record(cur)
        torch.cuda.synchronize(dev)
        if r >= 2:
            times.append(start.elapsed_time(stop))
    assert ft.ft_moe_read_status(ws) == 0
    ms = float(np.median(times))
    _, tfl, _ = _peaks()
    flops = 56623104.0 * T_prefill
    prefill = {"T": T_prefill, "routing": "zipf(1.1)", "us": ms * 1e3, "tokens_per_s": T_prefill / (ms / 1e3),
               "tflops": flops / (ms / 1e3) / 1e12, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / tfl,
               "kernel": "tcgen05 grouped GEMM (f16 operands, block scale folded into A per 128-row tile)"}
    del layers, flush
    torch.cuda.empty_cache()
    return {"format": "fp8_block (e4m3 weights, fp32 scale_inv per 128x128 block)", "decode": decode,
            "prefill": prefill}


def _rank_bytes(ft, cfg):
    """Algorithmic weight bytes of one routed expert and of the shared expert for this
    rank's banks (codes, block scales and row globals, from the library's own layout)."""
    E = cfg.num_experts
    routed = sum(b for *_, b in ft.ft_moe_layout(cfg, 0)) / E
    shared = sum(b for *_, b in ft.ft_moe_layout(cfg, 1)) if cfg.shared_intermediate else 0
    return float(routed), float(shared)


def _ranks(ft, dev, shape, tp, pieces_d):
    """Packed banks of every tp rank of one layer copy: [(cfg, routed, shared)]."""
    out = []
    for r in range(tp):
        cfg = ft.MoEConfig.of(shape, r, tp)
        rb, sb = ft.alloc_banks(cfg, 0, dev), ft.alloc_banks(cfg, 1, dev)
        ft.ft_moe_pack(cfg, 0, pieces_d[0], rb)
        ft.ft_moe_pack(cfg, 1, pieces_d[1], sb)
        out.append((cfg, rb, sb))
    return out


def measure_decode_row(ft, dev, shape, copies, T, zipf, reps=20, seed=100):
    """Decode regime: one step = for every layer copy, route once (the router is
    replicated) and run every tp rank's forward in sequence. Inputs larger than L2: the
    copies are distinct allocations of the full layer. Returns per-layer time (summed over
    ranks), touched-expert bytes and the fraction of the measured HBM bandwidth."""
    import torch
    L, tp = len(copies), len(copies[0])
    H, E, k = shape.hidden, shape.num_experts, shape.top_k
    mk = synth.zipf_logits if zipf else synth.make_logits
    x = torch.from_numpy(np.stack([synth.make_activations(T, H, seed=seed + l) for l in range(L)]).view(np.int16))
    x = x.to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(np.stack([mk(T, E, seed=seed + l) for l in range(L)])).to(dev)
    ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    out = torch.empty((L, tp, T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(ft.ft_moe_workspace_size(c[0], T) for c in copies[0]), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        for l in range(L):
            ft.ft_moe_route(lg[l], k, ids[l], w[l])
            for r, (cfg, rb, sb) in enumerate(copies[l]):
                ft.ft_moe_forward(cfg, rb, sb, x[l], ids[l], w[l], out[l, r], ws)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize(dev)
    assert ft.ft_moe_read_status(ws) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        stop.record(stream)
    torch.cuda.synchronize(dev)
    us_layer = start.elapsed_time(stop) * 1e3 / (reps * L)
    ids_np = ids.cpu().numpy()
    per_rank = [_rank_bytes(ft, c[0]) for c in copies[0]]
    layer_bytes = float(np.mean([sum(len(np.unique(ids_np[l])) * re + se for re, se in per_rank)
                                 for l in range(L)]))
    hbm, _, kind = _peaks()
    gbs = layer_bytes / (us_layer * 1e-6) / 1e9
    del x, lg, ids, w, out, ws, g
    return {"T": T, "tp": tp, "layers": L, "routing": "zipf(1.1)" if zipf else "N(0,1)",
            "us_per_layer": us_layer, "tokens_per_s": T / (us_layer * 1e-6), "weight_bytes_per_layer": layer_bytes,
            "gbs": gbs, "frac_of_hbm": gbs / hbm, "peak_source": f"{kind} HBM copy bandwidth",
            "timing": "CUDA graph of all layer copies, CUDA events, inputs larger than L2"}


def measure_prefill_row(ft, dev, shape, ranks, T, reps=5, seed=7):
    """Prefill regime, one layer: route once, then every tp rank's forward in sequence, L2
    flushed (512 MB written, then 256 MB read back) before the route and before each rank; the layer time is the
    sum of the route and rank times (CUDA events on the launch stream)."""
    import torch
    H, E, k = shape.hidden, shape.num_experts, shape.top_k
    x = torch.from_numpy(synth.make_activations(T, H, seed=seed).view(np.int16)).to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(synth.zipf_logits(T, E, seed=seed)).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(ft.ft_moe_workspace_size(c, T) for c, _, _ in ranks), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * (len(ranks) + 1))]
    totals = []
    for rep in range(reps + 2):
        parts = []
        _cold_l2(flush, rep)
        evs[0].record(stream)
        ft.ft_moe_route(lg, k, ids, w)
        evs[1].record(stream)
        for r, (cfg, rb, sb) in enumerate(ranks):
            _cold_l2(flush, (rep + r + 1))
            evs[2 * r + 2].record(stream)
            ft.ft_moe_forward(cfg, rb, sb, x, ids, w, out, ws)
            evs[2 * r + 3].record(stream)
        torch.cuda.synchronize(dev)
        assert ft.ft_moe_read_status(ws) == 0
        parts = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(len(ranks) + 1)]
        if rep >= 2:
            totals.append(parts)
    med = np.median(np.array(totals), axis=0)
    ms = float(med.sum())
    flops = 6.0 * H * (k * shape.intermediate + shape.shared_intermediate) * T
    _, tfl, kind = _peaks()
    del x, lg, ids, w, out, ws, flush
    return {"T": T, "tp": len(ranks), "routing": "zipf(1.1)", "us": ms * 1e3, "route_us": float(med[0] * 1e3),
            "rank_us": [float(v * 1e3) for v in med[1:]], "tokens_per_s": T / (ms / 1e3),
            "tflops": flops / (ms / 1e3) / 1e12, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / tfl,
            "peak_source": f"{kind} bf16 dense", "l2": "512 MB written, then 256 MB read back, before the route and before each rank"}


def measure_configs(ft, dev, qwen_pieces_d, qwen_copies, args):
    """The benchmark's other configurations, each with its roofline fraction: qwen36 decode
    at T = 1, 8, 32 (N(0,1) routing); the rank-local tp slices (tp = 2, 4) at decode T = 32
    and prefill T = 2048; and the DeepSeek-V4-like layer (H = 4096, I = I_s = 2048, g = 32)
    at T = 1, 16 (decode) and 4096 (prefill), tp = 1 and 4."""
    import torch
    qwen = synth.SHAPES["qwen36"]
    rows = {"qwen36_decode": [measure_decode_row(ft, dev, qwen, qwen_copies, T, False) for T in (1, 8, 32)]}
    tp_rows = []
    for tp in (2, 4):
        copies = [_ranks(ft, dev, qwen, tp, qwen_pieces_d) for _ in range(16)]
        tp_rows.append(measure_decode_row(ft, dev, qwen, copies, 32, False))
        tp_rows.append(measure_prefill_row(ft, dev, qwen, copies[0], 2048))
        del copies
        torch.cuda.empty_cache()
    rows["qwen36_tp_slices"] = tp_rows
    if not args.no_dsv4:
        ds = synth.SHAPES["dsv4"]
        pieces = synth.make_pieces(ds, 0), synth.make_pieces(ds, 0, shared=True)
        pieces_d = tuple({n: torch.from_numpy(v).to(dev) for n, v in p.items()} for p in pieces)
        del pieces
        ds_rows = []
        for tp in (1, 4):
            copies = [_ranks(ft, dev, ds, tp, pieces_d) for _ in range(8)]
            for T in (1, 16):
                ds_rows.append(measure_decode_row(ft, dev, ds, copies, T, True))
            ds_rows.append(measure_prefill_row(ft, dev, ds, copies[0], 4096))
            del copies
            torch.cuda.empty_cache()
        rows["dsv4"] = ds_rows
        del pieces_d
        torch.cuda.empty_cache()
    return rows


def run_ours(args, world, rank, local):
    import torch
    import nvfp4_quantized_moe_gb300 as ft
    from nvfp4_quantized_moe_gb300 import build as ftbuild

    if rank == 0 or world == 1:
        ftbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        dist.barrier()
        ftbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ft.load()
    shape = synth.SHAPES[args.shape]
    cfg = ft.MoEConfig.of(shape)
    T, L, H, E, k = args.T, args.layers, shape.hidden, shape.num_experts, shape.top_k
    routed_np = synth.make_pieces(shape, 0)
    shared_np = synth.make_pieces(shape, 0, shared=True)
    routed_d = {n: torch.from_numpy(v).to(dev) for n, v in routed_np.items()}
    shared_d = {n: torch.from_numpy(v).to(dev) for n, v in shared_np.items()}
    layers = []
    for l in range(L):
        rb, sb = ft.alloc_banks(cfg, 0, dev), ft.alloc_banks(cfg, 1, dev)
        ft.ft_moe_pack(cfg, 0, routed_d, rb)
        ft.ft_moe_pack(cfg, 1, shared_d, sb)
        layers.append((rb, sb))
    prefill = None
    if not args.no_prefill:
        prefill = [measure_prefill(ft, dev, cfg, shape, routed_d, shared_d, int(T_))
                   for T_ in args.prefill_T.split(",")]
    w4a4 = None
    if not args.no_w4a4:
        w4a4 = [measure_w4a4(ft, dev, cfg, layers[0][0], layers[0][1], shape, int(T_))
                for T_ in args.prefill_T.split(",")]
    router = [measure_router(ft, dev, T_, E=E, H=H) for T_ in (T, 2048)]
    fp8 = None if args.no_fp8 else measure_fp8(ft, dev)
    configs = None
    if not args.no_configs:
        configs = measure_configs(ft, dev, (routed_d, shared_d), [[(cfg, rb, sb)] for rb, sb in layers], args)
    del routed_d, shared_d
    x_host = [synth.make_activations(T, H, seed=l) for l in range(L)]
    lg_host = [synth.make_logits(T, E, seed=l) for l in range(L)]
    x = torch.from_numpy(np.stack(x_host).view(np.int16)).to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(np.stack(lg_host)).to(dev)
    ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    out = torch.empty((L, T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(ft.ft_moe_workspace_size(cfg, T), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    n_stage = ft.FT_NSTAGES + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage)] for _ in range(L)]
    for row in ev:
        for e_ in row:
            e_.record(stream)  # torch creates the CUDA event lazily, on first record

    def step(profile: bool):
        for l in range(L):
            ft.ft_moe_route(lg[l], k, ids[l], w[l])
            if profile:
                ft.ft_moe_set_stage_events(ev[l])
            ft.ft_moe_forward(cfg, layers[l][0], layers[l][1], x[l], ids[l], w[l], out[l], ws)

    with torch.cuda.stream(stream):
        step(False)  # eager warm-up (also checks the status word below)
    torch.cuda.synchronize(dev)
    assert ft.ft_moe_read_status(ws) == 0
    graphs = {}
    for profile in (False, True):
        g = torch.cuda.CUDAGraph()
        n0 = ft.ft_moe_launch_count()
        with torch.cuda.graph(g, stream=stream):
            step(profile)
        graphs[profile] = (g, ft.ft_moe_launch_count() - n0)
    g_plain, launches_per_step = graphs[False]

    # touched experts per layer (algorithmic bytes)
    ids_np = ids.cpu().numpy()
    touched = [len(np.unique(ids_np[l])) for l in range(L)]
    gu_bytes_per_expert, dn_bytes_per_expert = _expert_bytes(shape, shape.intermediate)
    gu_sh, dn_sh = _expert_bytes(shape, shape.shared_intermediate) if shape.shared_intermediate else (0, 0)
    per_expert = gu_bytes_per_expert + dn_bytes_per_expert
    layer_bytes = [t * per_expert + gu_sh + dn_sh for t in touched]

    for _ in range(args.warmup):
        g_plain.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                g_plain.replay()
            stop.record(stream)
        torch.cuda.synchronize(dev)
    elapsed_ms = _max_over_ranks(start.elapsed_time(stop), dev)
    ms_step = elapsed_ms / args.steps
    value = _job_value(T * L, world, args.steps, elapsed_ms)

    # per-stage durations from the profiled graph
    g_prof = graphs[True][0]
    reps = 5
    stage_ms = np.zeros((reps, L, ft.FT_NSTAGES))
    for r in range(reps):
        g_prof.replay()
        torch.cuda.synchronize(dev)
        for l in range(L):
            for s in range(ft.FT_NSTAGES):
                stage_ms[r, l, s] = ev[l][s].elapsed_time(ev[l][s + 1])
    stage_mean_us = {name: float(stage_ms[:, :, i].mean() * 1e3) for i, name in enumerate(ft.STAGES)}
    hbm, tfl, peak_kind = _peaks()
    # the routed and the shared expert run in the same launch per stage (decode regime)
    gu_alg = float(np.mean([t * gu_bytes_per_expert + gu_sh for t in touched]))
    dn_alg = float(np.mean([t * dn_bytes_per_expert + dn_sh for t in touched]))
    alg = {"gate_up": gu_alg, "down": dn_alg, "shared_gate_up": float(gu_sh), "shared_down": float(dn_sh)}
    if stage_mean_us["down"] < 0.5 and stage_mean_us["combine"] < 0.5:
        # one fused launch (gate_up, down, combine) between the gate_up and the next stage
        # marks: it streams every touched expert's gate_up and down bytes
        stage_mean_us = {"align": stage_mean_us["align"], "decode_fused": stage_mean_us["gate_up"]}
        alg = {"decode_fused": gu_alg + dn_alg}
    dominant = max(stage_mean_us, key=stage_mean_us.get)
    dom_bytes = alg.get(dominant, 0.0)
    dom_s = stage_mean_us[dominant] * 1e-6
    achieved = dom_bytes / dom_s / 1e9 if dom_bytes else None
    tr = _traffic(dominant)
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm if achieved else None,
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "traffic_alg_bytes": tr["alg_bytes_of_captured_launch"] if tr else None,
                "peak_source": f"{peak_kind} HBM copy bandwidth",
                "alg_bytes_per_launch": dom_bytes, "avg_launch_us": stage_mean_us[dominant]}
    layer_us = ms_step * 1e3 / L
    layer_gbs = float(np.mean(layer_bytes)) / (layer_us * 1e-6) / 1e9

    # end to end: pinned host inputs in, bf16 outputs back, every step
    x_pin = torch.from_numpy(np.stack(x_host).view(np.int16)).pin_memory()
    lg_pin = torch.from_numpy(np.stack(lg_host)).pin_memory()
    out_pin = torch.empty((L, T, H), dtype=torch.bfloat16).pin_memory()
    x16 = x.view(torch.int16)
    for _ in range(2):
        with torch.cuda.stream(stream):
            x16.copy_(x_pin, non_blocking=True)
            lg.copy_(lg_pin, non_blocking=True)
            g_plain.replay()
            out_pin.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, args.steps // 2)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            x16.copy_(x_pin, non_blocking=True)
            lg.copy_(lg_pin, non_blocking=True)
            g_plain.replay()
            out_pin.copy_(out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    wall_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e = {"value": world * T * L / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_pin.numel() * 2 + lg_pin.numel() * 4),
           "d2h_bytes_per_step": int(out_pin.numel() * 2), "ms_per_step": e2e_ms, "host_wall_ms_per_step": wall_ms}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": _config(args),
        "roofline": roofline, "layer": {"us": layer_us, "touched_experts_mean": float(np.mean(touched)),
                                        "weight_bytes_mean": float(np.mean(layer_bytes)), "gbs": layer_gbs,
                                        "frac_of_hbm": layer_gbs / hbm},
        "stage_us": stage_mean_us, "prefill": prefill, "w4a4": w4a4, "configs": configs, "router_gemm": router,
        "fp8_block": fp8, "e2e": e2e,
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(T, shape)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the fp8_block expert measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (decode T=1/8/32, tp slices, the DeepSeek-V4-like layer)")
    ap.add_argument("--no-dsv4", action="store_true", help="skip the DeepSeek-V4-like layer among the configurations")
    ap.add_argument("--no-w4a4", action="store_true", help="skip the W4A4 (NVFP4 activations) prefill measurement")
    ap.add_argument("--shape", choices=["qwen36", "dsv4"], default="qwen36",
                    help="NVFP4 layer family of the decode and prefill measurements")
    ap.add_argument("--prefill-T", default="2048,8192", help="comma-separated prefill token counts")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the Engram forward hot path (one layer, dim 5120, hc 4) on GB300.

One step = one pass of the whole path over one batch of synthetic input, through the public call
engram_forward: n-gram hash with the look-back cache and table-row gather + dequantisation (one
kernel), then the projection with the gate-and-add (one kernel at this size). Default workload:
prefill, B=1, T=4096. The dominant kernel is also timed alone for the roofline, and a decode
workload (B=64 after a 2048-token prefill) is reported beside it.

Prints one JSON line (rank 0). With torchrun (N > 1) every rank runs its own batch of B
sequences on its own GPU (sequences are independent: weak scaling, no collective on the data
path); the step time is the max over ranks.

--impl reference times the CPU oracle (oracle/) on the host cores instead, on a bounded sample of
the same workload per step, and prints the same line with "impl": "reference".
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Engram tokens/s per layer (dim5120, hc4), prefill+decode; % of roofline"
FLOPS_PER_TOKEN = 2 * 1536 * 25600           # wkv projection
BYTES_PER_TOKEN = 40960 + 40960 + 1536 + 48  # x in, out, gathered fp8 rows, e8m0 scales
WKV_BYTES = 25600 * 1536 * 2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20                   # > 129 MB L2


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("native", "reference"), default="native")
    p.add_argument("--batch", type=int, default=1, help="sequences per GPU")
    p.add_argument("--seq", type=int, default=4096, help="new tokens per sequence")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the masked batched prefill and the T sweep")
    return p.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(base: int, rank: int) -> int:
    """Each rank draws its own sequences: a disjoint shard of the global batch."""
    return base + 1000 * rank


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
        h = hashlib.sha256()
        for src in d["sources"]:   # every file the kernel is compiled from, in order
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != d["source_sha"]:
            return None
        return {"bytes_per_launch": d["bytes_per_launch"], "tokens_per_launch": d["tokens"]}
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------- native arm


def run_native(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from deepseek_v4_engram_gb300 import build as _build
    _build.build()
    import deepseek_v4_engram_gb300 as eg
    import synth

    geom = synth.FULL
    B, T = args.batch, args.seq
    M = B * T
    model = synth.make_model(geom, synth.BASE_SEED + 1)
    batch = synth.make_batch(geom, B, T, shard_seed(synth.BASE_SEED + 101, rank))
    t = model.tables

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        elif a.dtype == np.uint64:
            a = a.view(np.int64)
        return torch.from_numpy(a).cuda()

    desc = eg.make_desc(geom.dim, geom.hc_mult, geom.n_heads, geom.max_ngram_size, geom.head_dim,
                        t.num_embeddings, model.eps)
    tables = eg.DeviceTables(dev(t.token_map), t.pad_id, dev(t.multipliers), dev(t.primes),
                             dev(t.offsets))
    weights = eg.DeviceWeights(dev(model.table), dev(model.scales), dev(model.wkv), dev(model.q),
                               dev(model.k))
    x = dev(batch.x)
    tokens = dev(batch.tokens)
    out = torch.empty_like(x)
    steps_total = args.warmup + args.steps + 2
    cache = torch.zeros((B, T * steps_total), dtype=torch.int32, device="cuda")
    cache_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(eg.engram_forward_workspace_size(desc, M), dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():   # the public call: hash + row gather (one kernel), projection + gate (one kernel)
        eg.engram_forward(desc, tables, weights, x, tokens, cache, cache_len, None, out, ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set during warm-up")
    # Each timed step replays a CUDA graph of that call, as a serving loop would, so that the
    # events bracket device work only (the host-side argument checks and launches are not in
    # the step's critical path there).
    step_graph = capture_graph(step)
    cache_len.zero_()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()                       # L2 flush between timed steps (not timed)
            ev[i][0].record(stream)
            step_graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    wall = time.time() - wall0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    errors = eg.engram_check_errors()
    total_ms = reduce_max(sum(step_ms), device="cuda")
    value = world * M * args.steps / (total_ms / 1e3)

    # The dominant kernel, timed alone with CUDA events on the same stream: engram_wkv_gate (the
    # projection + gate kernel the step runs at this size) on the rows the step gathered.
    rows = ws[: M * geom.K * 2].view(torch.int16).view(M, geom.K)
    kws = torch.empty(eg.api.engram_wkv_gate_workspace_size(desc, M), dtype=torch.uint8,
                      device="cuda")
    kern_graph = capture_graph(
        lambda: eg.engram_wkv_gate(desc, rows, weights.wkv, x.view(M, geom.hc_mult, geom.dim),
                                   weights.q_weight, weights.k_weight, None,
                                   out.view(M, geom.hc_mult, geom.dim), workspace=kws))
    kern_ms = []
    for i in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kern_graph.replay()
        b.record(stream)
        kern_ms.append((a, b))
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in kern_ms]

    peaks, peak_kind = load_peaks()
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    achieved = FLOPS_PER_TOKEN * M / kern_avg_s / 1e12
    traffic = kernel_traffic("engram_fused_kernel")
    roofline = {
        "kernel": "engram_fused_kernel (projection + gate, tcgen05)",
        "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
        "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
        "peak_kind": f"{peak_kind} bf16 dense (burst)",
        "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
        "kernel_us": round(kern_avg_s * 1e6, 2),
        "kernel_timing": "engram_wkv_gate alone on the step's rows (CUDA graph replay: counter "
                         "memset + kernel), L2 flushed before each launch",
        "kernel_share_of_step": round(statistics.mean(kern_ms) / statistics.mean(step_ms), 4),
        # the captured bytes hold for the captured token count only (the weight's share of the
        # traffic does not grow with the tokens)
        "traffic": (None if traffic is None or traffic["tokens_per_launch"] != M else
                    traffic["bytes_per_launch"]),
        "algorithmic_bytes": M * BYTES_PER_TOKEN + WKV_BYTES,
    }
    # whole-step roofline: max(FLOPs at bf16 peak, bytes at HBM peak)
    t_roof = max(FLOPS_PER_TOKEN * M / (peaks["bf16_tflops"] * 1e12),
                 (M * BYTES_PER_TOKEN + WKV_BYTES) / (peaks["hbm_gbs"] * 1e9))
    step_s = total_ms / args.steps / 1e3
    decode = None if args.no_decode else run_decode(eg, desc, tables, weights, model, geom, args,
                                                    flush, peaks)

    configs = None
    if not args.no_configs and world == 1:
        configs = run_configs(eg, desc, tables, weights, model, geom, flush, peaks)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(eg, desc, tables, weights, batch, geom, args, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(model, batch, budget_s=10.0)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"prefill B{B} T{T} per GPU, dim 5120, hc 4, 24 rows x hd 64, "
                               "fp8 table 12.6M rows (~805 MB), wkv 25600x1536 bf16",
                   "global_batch": B * world, "seq_len": T, "parallelism": f"replicas x{world}",
                   "l2": "flushed (256 MB write) between timed steps",
                   "timing": "CUDA graph replay of engram_forward per step"},
        "roofline": roofline,
        "step_roofline_frac": round(t_roof / step_s, 4),
        "gpu_launches": 2 * args.steps,
        "decode": decode,
        "configs": configs,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "device_errors": errors,
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def capture_graph(fn):
    """A CUDA graph of fn(), captured on a side stream after one eager run there (which resolves
    every lazy setup outside the capture)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


def time_forward(eg, desc, tables, weights, x, tokens, mask, B, T, flush, steps, warmup,
                 in_graph=False):
    """Mean ms per step of engram_forward on B sequences of T new tokens: a captured graph
    replayed per step, L2 flushed before each step (outside the events). With in_graph, also the
    mean ms per step of 8 steps captured in one graph (time_steps_in_graph): (ms, ms or None)."""
    import torch
    M = B * T
    cache = torch.zeros((B, T * (steps + warmup + 2 + (40 if in_graph else 0))), dtype=torch.int32,
                        device="cuda")
    cache_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x)
    ws = torch.empty(eg.engram_forward_workspace_size(desc, M), dtype=torch.uint8, device="cuda")

    def step():
        eg.engram_forward(desc, tables, weights, x, tokens, cache, cache_len, mask, out, ws)

    graph = capture_graph(step)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    ev = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms_graph = time_steps_in_graph(step, flush, 8) if in_graph else None
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set")
    return (ms, ms_graph) if in_graph else ms


def roofline_of(M, ms, peaks):
    t_flop = FLOPS_PER_TOKEN * M / (peaks["bf16_tflops"] * 1e12)
    t_byte = (M * BYTES_PER_TOKEN + WKV_BYTES) / (peaks["hbm_gbs"] * 1e9)
    return ("tensor" if t_flop >= t_byte else "hbm"), max(t_flop, t_byte) / (ms / 1e3)


def run_configs(eg, desc, tables, weights, model, geom, flush, peaks):
    """The masked batched prefill (B8 T8192: pow2 block scales, Student-t x, ~10% of positions
    masked in contiguous spans) and the T sweep at B1; each step through engram_forward."""
    import numpy as np
    import torch
    import synth

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    res = {}
    w = synth.WORKLOADS["masked_b8_t8192"]
    pm = synth.make_model(geom, w["model_seed"], scale_mode=w["scale_mode"])
    pw = eg.DeviceWeights(dev(pm.table), dev(pm.scales), weights.wkv, weights.q_weight,
                          weights.k_weight)
    # tokens and mask from the host generators; x (2.7 GB) drawn on the device
    rng = np.random.default_rng(w["batch_seed"])
    tokens = synth.make_tokens(geom, w["B"], w["T"], rng)
    mask = synth.make_span_mask(w["B"], w["T"], w["mask_frac"], rng)
    x = synth.make_x_device((w["B"], w["T"], geom.hc_mult, geom.dim), w["batch_seed"],
                            w["x_dist"])
    M = w["B"] * w["T"]
    ms = time_forward(eg, desc, tables, pw, x, dev(tokens), dev(mask.astype(np.uint8)), w["B"],
                      w["T"], flush, steps=5, warmup=3)
    bound, frac = roofline_of(M, ms, peaks)
    res["masked"] = {"workload": "masked prefill B8 T8192 (pow2 scales, Student-t x, ~10% masked "
                                 "spans)", "value": round(M / (ms / 1e3), 1), "unit": "tokens/s",
                     "ms_per_step": round(ms, 4), "bound": bound, "roofline_frac": round(frac, 4)}
    del pw, x
    w = synth.WORKLOADS["sweep_b1"]
    tmax = max(w["T_list"])
    tok_all = dev(synth.make_tokens(geom, 1, tmax, np.random.default_rng(w["batch_seed"])))
    x_all = synth.make_x_device((1, tmax, geom.hc_mult, geom.dim), w["batch_seed"])
    sweep, between = [], []
    # the configured points, then the plan boundaries between them (256: small-batch projection;
    # 1024, 2048: fused kernel with deferred output)
    for T in tuple(w["T_list"]) + (256, 1024, 2048):
        steps = 20 if T <= 4096 else 5
        small = T <= 512   # where the graph launch per step is a visible share of the step
        # short steps get more warm-up steps, so that every point is timed after some
        # milliseconds of the same work (the first point follows the 2.7 GB generation of x)
        r = time_forward(eg, desc, tables, weights, x_all[:, :T].contiguous(),
                         tok_all[:, :T].contiguous(), None, 1, T, flush, steps=steps,
                         warmup=50 if small else 3, in_graph=small)
        ms, ms_graph = r if small else (r, None)
        bound, frac = roofline_of(T, ms, peaks)
        point = {"T": T, "value": round(T / (ms / 1e3), 1), "us_per_step": round(ms * 1e3, 2),
                 "bound": bound, "roofline_frac": round(frac, 4)}
        if ms_graph is not None:
            point["in_graph"] = {"us_per_step": round(ms_graph * 1e3, 2),
                                 "roofline_frac": round(roofline_of(T, ms_graph, peaks)[1], 4)}
        (sweep if T in w["T_list"] else between).append(point)
    res["layers"] = run_layers(eg, desc, tables, geom, flush, peaks)
    res["layers"]["workload"] = ("stages 1+2 for 4 Engram layers (own constants and tables), one "
                                 "launch vs one call per layer")
    res["sweep"] = {"workload": "prefill B1, T = 1 .. 65536", "unit": "tokens/s",
                    "points": sweep, "between": between,
                    "in_graph_timing": "T <= 512: also 8 steps in one CUDA graph, L2 flushed "
                                       "before each, event record nodes around each step",
                    "crossover_tokens": round(WKV_BYTES / (FLOPS_PER_TOKEN / (peaks["bf16_tflops"]
                                              * 1e12) * peaks["hbm_gbs"] * 1e9 - BYTES_PER_TOKEN))}
    return res


def time_graph(fn, flush, steps, warmup):
    """Mean ms of a captured CUDA graph of fn(), replayed per step with L2 flushed before each."""
    import torch
    graph = capture_graph(fn)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    ev = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def time_launches(launch, flush, steps, warmup):
    """Mean ms of launch() (one graph launch the library owns) with L2 flushed before each."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        launch()
    ev = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def run_layers(eg, desc, tables, geom, flush, peaks, n_layers=4, steps=20, warmup=3):
    """Stages 1 + 2 for several Engram layers: n_layers layers (each with its own hash constants
    and a 0.8-1.1 GB fp8 table) hashed and gathered by one engram_hash_rows_layers launch, against
    one single-layer call per layer, each layer with its own copy of the look-back cache (what
    separate per-layer hash states would do); at decode B64 (2048-token caches) and prefill B1
    T4096. Algorithmic bytes per (token, layer): the 24 fp8 rows and their e8m0 scales read, the 24
    bf16 rows written."""
    import numpy as np
    import torch
    import synth

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int64) if a.dtype == np.uint64 else a).cuda()

    S, hd = geom.n_hash_cols, geom.head_dim
    layers = []
    for i, lh in enumerate(synth.make_layer_hashes(geom, n_layers, synth.BASE_SEED + 800,
                                                   with_tables=False)):
        rows = lh.num_embeddings
        layers.append(dict(
            multipliers=dev(lh.multipliers), primes=dev(lh.primes), offsets=dev(lh.offsets),
            table=synth.make_fp8_rows_device(rows, hd, synth.BASE_SEED + 810 + i),
            scales=torch.full((rows, hd // 32), 127, dtype=torch.uint8, device="cuda")))
    bytes_per = S * (hd + hd // 32 + 2 * hd)
    res = {"n_layers": n_layers, "table_rows": [int(d["table"].shape[0]) for d in layers]}
    rng = np.random.default_rng(synth.BASE_SEED + 820)
    for name, B, T, prefill in (("decode_b64", 64, 1, 2048), ("prefill_b1_t4096", 1, 4096, 0)):
        M = B * T
        cap = prefill + T * (warmup + steps + 4)
        tok = dev(synth.make_tokens(geom, B, T, rng))
        caches = [(torch.zeros((B, cap), dtype=torch.int32, device="cuda"),
                   torch.zeros(B, dtype=torch.int32, device="cuda")) for _ in range(n_layers + 1)]
        recs = [eg.DeviceLayerHash(**d, rows=torch.empty((M, S * hd), dtype=torch.int16,
                                                         device="cuda")) for d in layers]
        if prefill:
            pre = dev(synth.make_tokens(geom, B, prefill, rng))
            pre_rows = torch.empty((B * prefill, S * hd), dtype=torch.int16, device="cuda")
            for c, ln in caches:
                eg.engram_hash_rows_layers(desc, tables, [eg.DeviceLayerHash(
                    **layers[0], rows=pre_rows)], pre, c, ln)
            del pre_rows

        def shared():
            eg.engram_hash_rows_layers(desc, tables, recs, tok, *caches[0])

        def separate():
            for i, r in enumerate(recs):
                eg.engram_hash_rows_layers(desc, tables, [r], tok, *caches[i + 1])

        ms_sh = time_graph(shared, flush, steps, warmup)
        ms_sep = time_graph(separate, flush, steps, warmup)
        if eg.engram_check_errors() != 0:
            raise RuntimeError("device error word set during the layers workload")
        nbytes = M * n_layers * bytes_per
        gbs = nbytes / (ms_sh / 1e3) / 1e9
        res[name] = {"tokens": M, "us_one_launch": round(ms_sh * 1e3, 2),
                     "us_one_call_per_layer": round(ms_sep * 1e3, 2),
                     "layer_tokens_per_s": round(M * n_layers / (ms_sh / 1e3), 1),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(gbs / peaks["hbm_gbs"], 4),
                                  "algorithmic_bytes": nbytes}}
        del recs, caches
    return res


def run_decode(eg, desc, tables, weights, model, geom, args, flush, peaks, B=64, prefill=2048):
    """Decode: B sequences whose 2048-token prefill is already hashed into the device cache, then
    one new token per sequence per step. Each step is one captured CUDA graph of engram_forward
    (as a serving loop would replay it); L2 is flushed before every timed step."""
    import numpy as np
    import torch
    import synth
    rng = np.random.default_rng(synth.BASE_SEED + 102)
    n = args.warmup + args.steps + 4
    pre = torch.from_numpy(rng.integers(0, geom.vocab, (B, prefill), dtype=np.int32)).cuda()
    cache = torch.zeros((B, prefill + 16 * n + 256), dtype=torch.int32, device="cuda")
    cache_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    ids = torch.empty((B, prefill, geom.n_hash_cols), dtype=torch.int32, device="cuda")
    eg.engram_hash(desc, tables, pre, cache, cache_len, ids)
    batch = synth.make_batch(geom, B, 1, synth.BASE_SEED + 702)
    x = torch.from_numpy(batch.x.view(np.int16)).cuda()
    tok = torch.from_numpy(batch.tokens).cuda()
    out = torch.empty_like(x)
    ws = torch.empty(eg.engram_forward_workspace_size(desc, B), dtype=torch.uint8, device="cuda")

    def step():
        eg.engram_forward(desc, tables, weights, x, tok, cache, cache_len, None, out, ws)

    # the decode loop as a serving loop runs it: the library's own graph of the step
    # (engram_forward_graph_create), one engram_graph_launch per step
    graph = eg.EngramGraph(desc, tables, weights, x, tok, cache, cache_len, None, out, ws)
    ms = time_launches(graph.launch, flush, args.steps, args.warmup)
    graph.destroy()
    in_graph_ms = time_steps_in_graph(step, flush, 8)
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set during decode")
    bytes_step = WKV_BYTES + B * BYTES_PER_TOKEN
    gbs = bytes_step / (ms / 1e3) / 1e9
    res = {"workload": f"decode B{B} x 1 token, {prefill}-token cache per sequence",
           "value": round(B / (ms / 1e3), 1), "unit": "tokens/s", "us_per_step": round(ms * 1e3, 2),
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                        "algorithmic_bytes": bytes_step},
           "gpu_launches_per_step": 3,
           "timing": "engram_graph_launch per step (the library's CUDA graph of engram_forward: "
                     "3 kernels), L2 flushed (256 MB write) before each"}
    # What the weight stream alone costs in this setting: the step's projection kernel by itself
    # (engram_wkv on the step's gathered rows: weight stream and kv stores, no hash and no
    # gate), after the same flush. The flush leaves L2 full of dirty lines, so every line the
    # stream brings in also writes one back.
    rows = ws[: B * geom.K * 2].view(torch.int16).view(B, geom.K)
    kv_alone = torch.empty((B, geom.N), dtype=torch.int16, device="cuda")
    alone_ms = time_graph(lambda: eg.engram_wkv(rows, weights.wkv, kv_alone), flush, args.steps,
                          args.warmup)
    res["projection_alone"] = {
        "us": round(alone_ms * 1e3, 2),
        "weight_gbs": round(WKV_BYTES / (alone_ms / 1e3) / 1e9, 1),
        "frac_of_hbm_peak": round(WKV_BYTES / (alone_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
        "timing": "engram_wkv (the decode projection kernel) alone on the step's rows, CUDA graph "
                  "replay, L2 flushed before each as for the steps"}
    # The floor under that: one read of the weight over every SM that does nothing with the bytes
    # (engram_probe_stream_read: bulk copies into the projection's ring depth, or plain loads),
    # after the same flush.
    floor = {}
    for method, name in ((0, "bulk_copies"), (1, "plain_loads"), (2, "bulk_copies_evict_first")):
        f_ms = time_graph(lambda m=method: eg.api.engram_probe_stream_read(weights.wkv, m), flush,
                          args.steps, args.warmup)
        floor[name] = {"us": round(f_ms * 1e3, 2),
                       "gbs": round(WKV_BYTES / (f_ms / 1e3) / 1e9, 1),
                       "frac_of_hbm_peak": round(WKV_BYTES / (f_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                                 4)}
    floor["timing"] = ("engram_probe_stream_read over the 78.6 MB wkv weight, CUDA graph replay, "
                       "L2 flushed before each as for the steps")
    res["stream_floor"] = floor
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set by the stream probe")
    res["inputs_larger_than_l2"] = decode_rotating(eg, desc, tables, weights, geom, cache,
                                                   cache_len, B, args, peaks, bytes_step)
    # Stages 2-4 from given hash ids (engram_forward_ids): in a model decode step the hash of
    # every Engram layer is resolved once (engram_hash_rows_layers or engram_hash) and each layer
    # then runs only the gather, projection and gate.
    hid = torch.empty((B, 1, geom.n_hash_cols), dtype=torch.int32, device="cuda")
    eg.engram_forward(desc, tables, weights, x, tok, cache, cache_len, None, out, ws,
                      hash_ids_out=hid)
    x3 = x.view(B, geom.hc_mult, geom.dim)
    out3 = out.view(B, geom.hc_mult, geom.dim)
    ids2 = hid.view(B, geom.n_hash_cols)
    ids_ms = time_graph(lambda: eg.engram_forward_ids(desc, weights, x3, ids2, None, out3, ws),
                        flush, args.steps, args.warmup)
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set during decode from ids")
    gbs_ids = bytes_step / (ids_ms / 1e3) / 1e9
    res["from_ids"] = {
        "workload": f"decode B{B} x 1 token from given hash ids (engram_forward_ids: gather, "
                    "projection, gate)",
        "value": round(B / (ids_ms / 1e3), 1), "unit": "tokens/s",
        "us_per_step": round(ids_ms * 1e3, 2),
        "roofline": {"bound": "hbm", "achieved": round(gbs_ids, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs_ids / peaks["hbm_gbs"], 4),
                     "algorithmic_bytes": bytes_step},
        "timing": "CUDA graph replay per step, L2 flushed (256 MB write) before each"}
    # Stages 3-4 from rows already gathered (a model step whose engram_hash_rows_layers launch has
    # gathered every Engram layer's rows): the projection (engram_wkv) and the gate
    # (engram_gate_and_add) of one layer.
    kv_rows = torch.empty((B, geom.N), dtype=torch.int16, device="cuda")

    def rows_step():
        eg.engram_wkv(rows, weights.wkv, kv_rows)
        eg.engram_gate_and_add(desc, x3, kv_rows, weights.q_weight, weights.k_weight, None, out3)

    rows_ms = time_graph(rows_step, flush, args.steps, args.warmup)
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set during decode from rows")
    gbs_rows = bytes_step / (rows_ms / 1e3) / 1e9
    res["from_rows"] = {
        "workload": f"decode B{B} x 1 token from rows already gathered (engram_wkv + "
                    "engram_gate_and_add: projection, gate)",
        "value": round(B / (rows_ms / 1e3), 1), "unit": "tokens/s",
        "us_per_step": round(rows_ms * 1e3, 2),
        "roofline": {"bound": "hbm", "achieved": round(gbs_rows, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs_rows / peaks["hbm_gbs"], 4),
                     "algorithmic_bytes": bytes_step},
        "timing": "CUDA graph replay per step, L2 flushed (256 MB write) before each"}
    if in_graph_ms is not None:
        # the same steps without a graph launch per step: what a serving loop that captures many
        # layers or steps in one graph sees
        res["in_graph"] = {
            "us_per_step": round(in_graph_ms * 1e3, 2),
            "frac": round(bytes_step / (in_graph_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "timing": "8 steps in one CUDA graph, L2 flushed (256 MB write) before each, event "
                      "record nodes around each step"}
    return res


def decode_rotating(eg, desc, tables, weights, geom, cache, cache_len, B, args, peaks,
                    bytes_step, copies=3):
    """The decode step with no flush between steps: each step reads its own copy of the wkv
    weight, x and tokens, and the copies rotate, so the inputs of the steps add up to more than
    L2 (3 x 78.6 MB of weight): every step reads its weight from HBM, and L2 holds no dirty lines
    from a flush (as in a model, where a decode step streams other layers' weights in between)."""
    import numpy as np
    import torch
    import synth
    graphs = []
    keep = []
    for c in range(copies):
        w = weights.wkv.clone()
        wts = eg.DeviceWeights(weights.table, weights.scales, w, weights.q_weight,
                               weights.k_weight)
        batch = synth.make_batch(geom, B, 1, synth.BASE_SEED + 710 + c)
        x = torch.from_numpy(batch.x.view(np.int16)).cuda()
        tok = torch.from_numpy(batch.tokens).cuda()
        out = torch.empty_like(x)
        ws = torch.empty(eg.engram_forward_workspace_size(desc, B), dtype=torch.uint8,
                         device="cuda")
        keep.append((w, wts, x, tok, out, ws))

        def step(wts=wts, x=x, tok=tok, out=out, ws=ws):
            eg.engram_forward(desc, tables, wts, x, tok, cache, cache_len, None, out, ws)
        graphs.append(capture_graph(step))
    for i in range(args.warmup * copies):
        graphs[i % copies].replay()
    torch.cuda.synchronize()
    ev = []
    n = args.steps - args.steps % copies or copies
    for i in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graphs[i % copies].replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    if eg.engram_check_errors() != 0:
        raise RuntimeError("device error word set during decode")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    gbs = bytes_step / (ms / 1e3) / 1e9
    del keep
    return {"value": round(B / (ms / 1e3), 1), "unit": "tokens/s",
            "us_per_step": round(ms * 1e3, 2),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)},
            "timing": f"CUDA graph replay per step, no flush: {copies} copies of the weight, x "
                      "and tokens rotated (inputs larger than L2)"}


def time_steps_in_graph(step, flush, k, replays=3):
    """Mean ms per step of `step` captured k times in one CUDA graph, each preceded by an L2
    flush and bracketed by event record nodes (events recorded inside the graph), so that the
    per-step time excludes the graph launch. None where torch cannot record events in a graph."""
    import torch
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(k)]
    except TypeError:
        return None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for a, b in evs:
            flush.zero_()
            a.record()
            step()
            b.record()
    graph.replay()   # warm-up
    torch.cuda.synchronize()
    samples = []
    for _ in range(replays):
        graph.replay()
        torch.cuda.synchronize()
        samples += [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(samples)


def run_e2e(eg, desc, tables, weights, batch, geom, args, world):
    """Same metric through engram_forward from pinned host buffers: every step copies its inputs
    host -> device, runs the forward and copies its output device -> host, all inside the timed
    region. As a serving loop would, the steps are pipelined over three streams with double
    device buffers: step i's upload, step i-1's forward and step i-2's download overlap (the
    forwards run in order on one stream, so the look-back cache is updated in order)."""
    import numpy as np
    import torch
    B, T = batch.tokens.shape
    M = B * T
    x_h = torch.from_numpy(np.ascontiguousarray(batch.x).view(np.int16)).pin_memory()
    tok_h = torch.from_numpy(np.ascontiguousarray(batch.tokens)).pin_memory()
    out_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x_h, device="cuda") for _ in range(2)]
    tok_d = [torch.empty_like(tok_h, device="cuda") for _ in range(2)]
    out_d = [torch.empty_like(x_d[0]) for _ in range(2)]
    n = args.warmup + args.steps + 2
    cache = torch.zeros((B, T * n), dtype=torch.int32, device="cuda")
    cache_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(eg.engram_forward_workspace_size(desc, M), dtype=torch.uint8, device="cuda")
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("up", "comp", "down")}
    for k in ev:   # every event starts out recorded, so the first waits pass
        for e in ev[k]:
            e.record()
    torch.cuda.synchronize()

    def step(i):
        j = i % 2
        with torch.cuda.stream(up):                  # inputs into buffer j once step i-2 is done
            up.wait_event(ev["comp"][j])
            x_d[j].copy_(x_h, non_blocking=True)
            tok_d[j].copy_(tok_h, non_blocking=True)
            ev["up"][j].record(up)
        with torch.cuda.stream(comp):                # forward i once its inputs are in and
            comp.wait_event(ev["up"][j])             # step i-2's output has been copied out
            comp.wait_event(ev["down"][j])
            eg.engram_forward(desc, tables, weights, x_d[j], tok_d[j], cache, cache_len, None,
                              out_d[j], ws, stream=comp)
            ev["comp"][j].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev["comp"][j])
            out_h[j].copy_(out_d[j], non_blocking=True)
            ev["down"][j].record(down)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(up)
    for i in range(args.steps):
        step(args.warmup + i)
    for st in (up, comp):
        down.wait_stream(st)
    e.record(down)
    torch.cuda.synchronize()
    ms = reduce_max(s.elapsed_time(e), device="cuda")
    return {"value": round(world * M * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x_h.numel() * 2 + tok_h.numel() * 4),
            "d2h_bytes_per_step": int(out_h[0].numel() * 2),
            "api": "engram_forward (pinned host -> device -> host, every step; uploads, forwards "
                   "and downloads of consecutive steps overlap on three streams)"}


# ---------------------------------------------------------------------------- oracle timing


def oracle_tokens_per_s(model, batch, budget_s: float, chunk: int = 128):
    """Run the oracle over the first tokens of sequence 0 in chunks until budget_s has passed."""
    from oracle import engram as E
    t = model.tables
    g = model.geom
    st = E.NgramHashState(t.token_map, t.pad_id, t.multipliers, t.primes, t.offsets,
                          g.n_heads, g.max_ngram_size, 1)
    done, t0 = 0, time.perf_counter()
    T = batch.tokens.shape[1]
    while done < T:
        n = min(chunk, T - done)
        E.forward(st, model.table, model.scales, model.wkv, model.q, model.k,
                  batch.x[:1, done:done + n], batch.tokens[:1, done:done + n], None, model.eps)
        done += n
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return done / el, done, el


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(model, batch, budget_s: float):
    tps, n, el = oracle_tokens_per_s(model, batch, budget_s)
    return {"value": round(tps, 2), "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"first {n} tokens of the same prefill workload, {el:.1f} s; float64 numpy "
                      "(matmul through the host BLAS on all cores)"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import synth
    geom = synth.FULL
    model = synth.make_model(geom, synth.BASE_SEED + 1)
    batch = synth.make_batch(geom, args.batch, args.seq, synth.BASE_SEED + 101)
    per_step = []
    sample = 128
    for i in range(args.warmup + args.steps):
        tps, n, el = oracle_tokens_per_s(model, batch, budget_s=0.0, chunk=sample)
        if i >= args.warmup:
            per_step.append(el)
    total = sum(per_step)
    value = sample * args.steps / total
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": f"prefill B{args.batch} T{args.seq} per GPU, dim 5120, hc 4; each "
                               f"step the oracle runs a {sample}-token sample of it",
                   "global_batch": args.batch, "seq_len": args.seq, "parallelism": "host CPU"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": host_cores(),
                         "kind": "oracle", "sample": f"{sample} tokens per step"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()

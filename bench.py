#!/usr/bin/env python
"""Benchmark: Maple MoE layer, batch-1 decode (route + expert FFN), on one B300.

Workload (the metric's configuration): hidden 2048, 256 experts, top-8, no shared
expert, intermediate 512; ternary experts packed 5 trits/byte with fp32 row scales;
bf16 router [256 x 2048]; one bf16 N(0,1) token per step.  One step = route + expert
FFN of one token on one layer (one maple_moe_layer call).  The timed steps walk over
1000 distinct seeded tokens and LAYERS independently seeded layers (10.5 GB packed) in
order, so a layer is revisited only after 63 others (inputs larger than L2); every
timed graph is replayed once untimed first and L2 is flushed before the timed region.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead, on a
bounded sample of the same workload.  Under torchrun with N > 1 every rank runs an
independent replica (the path has no exchange step) and `value` sums all ranks.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, E, I, K_TOP = 2048, 256, 512, 8
N_TOKENS = 1000
LAYERS = 64
L2_FLUSH_BYTES = 256 << 20  # twice the B300's 126 MB L2
LAUNCHES_PER_STEP = 1       # maple_moe_layer at T = 1: one launch of the fused kernel
METRIC = "ternary MoE layer tokens/s (batch 1 & 64 decode); packed-weight HBM GB/s vs peak"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
# the batch-1 layer kernel and the device helpers it is built from
LAYER_KERNEL_SOURCES = ("ternary_weight_moe_02_b300/csrc/layer_decode.cu",
                        "ternary_weight_moe_02_b300/csrc/common.cuh")
EXPERT_BYTES = 2 * I * ((H + 4) // 5) + H * ((I + 4) // 5) + 4 * (2 * I + H)  # 643,072


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(units_per_rank: float, elapsed_s: float, world: int) -> float:
    """Whole-job rate of `world` replicas that each processed units_per_rank units:
    all units over the slowest rank's time (every rank gets the same value)."""
    return world * units_per_rank / _max_over_ranks(elapsed_s, world)


# ----------------------------------------------------------------------------- inputs

def sources_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel: str, sources) -> float | None:
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu summary,
    or None when there is none or the kernel's sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256") != sources_sha256(sources):
        return None
    return float(rec["dram_bytes_per_launch"])


def build_layers(maple, synth, n_layers: int, seed0: int = 1000):
    """n_layers independent Maple layers: bf16 N(0,0.02) experts drawn on the GPU and
    packed by maple_ternarize_pack (untimed set-up), bf16 router weights."""
    layers = []
    Bh, Bi = (H + 4) // 5, (I + 4) // 5
    for l in range(n_layers):
        w = synth.expert_weights(E, H, I, seed=seed0 + l, device="cuda")
        gate = torch.empty((E, I, Bh), dtype=torch.uint8, device="cuda")
        up = torch.empty((E, I, Bh), dtype=torch.uint8, device="cuda")
        down = torch.empty((E, H, Bi), dtype=torch.uint8, device="cuda")
        sg = torch.empty((E, I), device="cuda")
        su = torch.empty((E, I), device="cuda")
        sd = torch.empty((E, H), device="cuda")
        maple.maple_ternarize_pack(w["gate"].view(E * I, H), gate.view(E * I, Bh), sg.view(-1))
        maple.maple_ternarize_pack(w["up"].view(E * I, H), up.view(E * I, Bh), su.view(-1))
        maple.maple_ternarize_pack(w["down"].view(E * H, I), down.view(E * H, Bi), sd.view(-1))
        del w
        router = synth.router_weights(E, H, seed=seed0 + l, device="cuda")
        layers.append((maple.Experts(gate, up, down, sg, su, sd, clamp=7.0), router))
    torch.cuda.synchronize()
    return layers


# ------------------------------------------------------------------------ GPU arm

def run_gpu(args, world, rank, local):
    from ternary_weight_moe_02_b300 import maple, synth
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n_layers = args.layers
    layers = build_layers(maple, synth, n_layers, seed0=1000 + 97 * rank)
    x_all = synth.tokens(N_TOKENS, H, seed=7 + rank, device="cuda")
    logits = torch.empty((1, E), device=dev)
    idx = torch.empty((1, K_TOP), dtype=torch.int32, device=dev)
    wts = torch.empty((1, K_TOP), device=dev)
    y = torch.empty((1, H), device=dev)
    # maple_moe_layer wants the first 256 bytes zero before its first call
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(1, K_TOP, layers[0][0]), dtype=torch.uint8,
                     device=dev)
    ws_ffn = torch.empty(maple.maple_moe_ffn_workspace_size(1, K_TOP, layers[0][0]),
                         dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, s, events=None):
        # one layer step: route + FFN of one token (a single fused launch)
        ex, router = layers[i % n_layers]
        x = x_all[i % N_TOKENS: i % N_TOKENS + 1]
        if events is not None:
            events[0].record(s)
        maple.maple_moe_layer(x, router, None, ex, K_TOP, logits, idx, wts, y, ws, stream=s)
        if events is not None:
            events[1].record(s)

    def step_two_calls(i, s):
        ex, router = layers[i % n_layers]
        x = x_all[i % N_TOKENS: i % N_TOKENS + 1]
        maple.maple_route_topk(x, router, None, K_TOP, logits, idx, wts, stream=s)
        maple.maple_moe_ffn(ex, x, idx, wts, y, ws_ffn, stream=s)

    # The timed steps are one continuous walk i = 0 .. K-1 over layers i % n_layers and
    # tokens i % N_TOKENS.  Graphs of `chunk` steps (a multiple of n_layers when K is
    # larger, so that back-to-back replays continue the walk seamlessly) are replayed.
    K = args.steps
    chunk = K if K <= args.chunk else max(n_layers, args.chunk // n_layers * n_layers)
    reps, rem = divmod(K, chunk)
    l2_flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        # writes a buffer twice the size of L2: no layer data stays cached
        l2_flush.zero_()

    def capture(n_steps, start, fn=step):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):  # warm the launch path before capture
                fn(start + i, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_steps):
                    fn(start + i, stream)
        return g

    g_chunk = capture(chunk, 0)
    g_rem = capture(rem, 0) if rem else None
    # warm-up on steps the timed walk does not start with (layers from the middle of the
    # cycle), then one untimed replay of every timed graph (its first launch and upload),
    # then an L2 flush: the timed region starts cold
    g_warm = capture(args.warmup, K + n_layers // 2)
    with torch.cuda.stream(stream):
        g_warm.replay()
        g_chunk.replay()
        if g_rem is not None:
            g_rem.replay()
        flush()
    torch.cuda.synchronize()
    _barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        torch.cuda.synchronize()
        _barrier(world)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                g_chunk.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        _barrier(world)
    elapsed_s = ev0.elapsed_time(ev1) / 1e3
    elapsed_max = _max_over_ranks(elapsed_s, world)
    value = _job_rate(K, elapsed_s, world)
    launches = K * LAUNCHES_PER_STEP

    # The same steps through the two separate calls (route_topk, moe_ffn), from a flushed
    # L2 after one untimed replay.
    n_two = min(K, chunk)
    g_two = capture(n_two, 0, step_two_calls)
    with torch.cuda.stream(stream):
        g_two.replay()
        flush()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        g_two.replay()
        t1.record(stream)
    t1.synchronize()
    two_call_value = n_two / (t0.elapsed_time(t1) / 1e3)

    # Roofline pass: the same walk with graph-captured events around each step's launch
    # (the events are graph nodes of their own, so each launch runs alone), from a
    # flushed L2, giving the live average duration of the dominant launch.
    n_roof = min(K, 2000)
    pairs = [(torch.cuda.Event(enable_timing=True, external=True),
              torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n_roof)]
    g_roof = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_roof, stream=stream):
            for i in range(n_roof):
                step(i, stream, pairs[i])
    with torch.cuda.stream(stream):
        flush()
        g_roof.replay()
    torch.cuda.synchronize()
    ffn_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs)
    peak, peak_kind = _peaks()
    packed_bytes = K_TOP * EXPERT_BYTES  # 8 distinct experts per batch-1 token
    # everything one launch must move: packed experts + scales, router, x, y, logits/idx/w
    alg_bytes = packed_bytes + E * H * 2 + H * 2 + H * 4 + E * 4 + K_TOP * 8
    achieved = alg_bytes / (ffn_ms / 1e3) / 1e9

    # End-to-end through the public API with host buffers: every step, maple_moe_layer_host
    # copies the step's token from pinned host memory, runs the layer and copies y back
    # into pinned host memory.  The calls are bound (arguments checked and marshalled)
    # before the timed region; the loop makes one C call per step.
    n_e2e = min(K, 2000)
    x_host = x_all[:N_TOKENS].cpu().pin_memory()
    y_host = torch.empty((1, H), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((1, H), dtype=torch.bfloat16, device=dev)

    def bound(i):
        ex, router = layers[i % n_layers]
        t = i % N_TOKENS
        return maple.bind_moe_layer_host(x_host[t:t + 1], x_dev, router, None, ex, K_TOP, logits, idx, wts, y,
                                         y_host, ws, stream=stream)
    warm_calls = [bound(K + i) for i in range(3)]
    calls = [bound(i) for i in range(n_e2e)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for c in warm_calls:
            c()
        flush()
        stream.synchronize()
        e0.record(stream)
        for c in calls:
            c()
        e1.record(stream)
    e1.synchronize()
    e2e_value = _job_rate(n_e2e, e0.elapsed_time(e1) / 1e3, world)

    legs = tuple(args.legs.split(",")) if args.legs else SECONDARY_LEGS
    secondary = (run_secondary(maple, synth, layers, dev, stream, legs, flush=flush,
                               cpu=(rank == 0 and world == 1 and args.cpu_tokens > 0))
                 if args.secondary else None)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_max * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic (seeded bf16 N(0,0.02) weights, ternarized and packed on the GPU)",
        "config": {"workload": "maple_moe_layer_decode_b1", "hidden": H, "experts": E,
                   "top_k": K_TOP, "moe_intermediate": I, "tokens_per_step": 1,
                   "distinct_tokens": N_TOKENS, "layers_cycled": n_layers,
                   "packed_gb": round(n_layers * E * EXPERT_BYTES / 1e9, 2),
                   "l2": "inputs larger than L2 (64 layers walked in order, a layer revisited "
                         "only after 63 others); L2 flushed before the timed region",
                   "graph": f"CUDA graph of {chunk} steps, replayed once untimed first",
                   "parallelism": f"replicas{world}"},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "kernel": "moe_layer_b1_kernel (whole step, one launch)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": alg_bytes, "avg_launch_us": ffn_ms * 1e3,
                     "packed_weight_gbs": packed_bytes / (ffn_ms / 1e3) / 1e9,
                     "traffic": measured_traffic("moe_layer_b1_kernel", LAYER_KERNEL_SOURCES)},
        "two_call_path": {"value": two_call_value, "unit": "tokens/s",
                          "calls": "maple_route_topk + maple_moe_ffn (4 launches per step)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": n_e2e,
                "h2d_bytes_per_step": H * 2, "d2h_bytes_per_step": H * 4,
                "call": "maple_moe_layer_host (token in from pinned host memory, y out to it)"},
        "clocks": clocks.summary(),
    }
    if secondary is not None:
        result["secondary"] = secondary
    return result


# ------------------------------------------------------------- secondary workloads

SECONDARY_LEGS = ("decode_b1", "decode_b8", "decode_b32", "decode_b64", "decode_b1_streamed", "prefill_4096",
                  "ternarize_pack", "pack_ternary")
STREAM_SLOTS = 64    # HBM expert slots of the streamed-decode leg
STREAM_STEPS = 200   # timed tokens of the streamed-decode leg
DECODE_BATCHES = (1, 8, 32, 64)


def expert_bytes(H: int, I: int) -> int:
    """Packed rows and fp32 scales of one expert: gate and up [I][ceil(H/5)], down
    [H][ceil(I/5)], scales 2I + H (643,072 B at the Maple shape)."""
    return 2 * I * ((H + 4) // 5) + H * ((I + 4) // 5) + 4 * (2 * I + H)


def distinct_expert_bytes(idx_per_layer, E: int, H: int, I: int) -> int:
    """Bytes of the distinct experts each layer's routing touches, summed over layers
    (ids outside [0, E) touch nothing)."""
    total = 0
    for idx in idx_per_layer:
        ids = idx.reshape(-1)
        ids = ids[(ids >= 0) & (ids < E)]
        total += int(torch.unique(ids).numel()) * expert_bytes(H, I)
    return total


def run_secondary(maple, synth, layers, dev, stream, legs=SECONDARY_LEGS, flush=None, cpu=True):
    """Other configurations of the same path, measured briefly (not the headline):
    decode batches of 1, 8, 32 and 64 tokens over 24 stacked layers with a N(0,0.5)
    router bias (with the packed-weight rate over the distinct experts each layer
    touches), the 4096-token prefill with a Zipf(1.1) bias, ternarize + pack throughput
    on whole layers, and (after it, on its output) the packing of already-ternary
    matrices.  Each timed graph replay starts from a flushed L2 (the flush is outside
    the events).  With cpu=True each leg also carries the oracle's figure on a bounded
    sample of the same workload (single-threaded, the sample stated)."""
    out = {}
    n_stack = min(24, len(layers))

    def timed_graph(fn, n_steps, reps=3):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(2):
                fn(i)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_steps):
                    fn(i)
            g.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for a, b in evs:
                if flush is not None:
                    flush()
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / 1e3 / (reps * n_steps)

    for T in DECODE_BATCHES:
        if f"decode_b{T}" not in legs:
            continue
        xs = [synth.tokens(T, H, seed=100 + l, device=dev) for l in range(n_stack)]
        biases = [synth.bias_normal(E, seed=200 + l).to(dev) for l in range(n_stack)]
        logits = torch.empty((T, E), device=dev)
        idx = torch.empty((T, K_TOP), dtype=torch.int32, device=dev)
        w = torch.empty((T, K_TOP), device=dev)
        y = torch.empty((T, H), device=dev)
        ws = torch.zeros(maple.maple_moe_layer_workspace_size(T, K_TOP, layers[0][0]), dtype=torch.uint8,
                         device=dev)

        def layer(i, T=T, xs=xs, biases=biases, logits=logits, idx=idx, w=w, y=y, ws=ws):
            ex, router = layers[i % n_stack]
            maple.maple_moe_layer(xs[i % n_stack], router, biases[i % n_stack], ex, K_TOP, logits, idx,
                                  w, y, ws, stream=stream)
        sec = timed_graph(layer, n_stack)
        # the experts each layer's routing touches (routed again, outside the timed graph)
        idx_layers = []
        with torch.cuda.stream(stream):
            for i in range(n_stack):
                maple.maple_route_topk(xs[i], layers[i][1], biases[i], K_TOP, logits, idx, w, stream=stream)
                idx_layers.append(idx.clone())
        stream.synchronize()
        packed = distinct_expert_bytes(idx_layers, E, H, I) / n_stack
        leg = {"value": T / sec, "unit": "tokens/s", "ms_per_layer": sec * 1e3,
               "layers": n_stack, "bias": "N(0, 0.5) per expert",
               "distinct_expert_mb_per_layer": packed / 1e6,
               "packed_weight_gbs": packed / sec / 1e9}
        if cpu:
            leg["cpu_baseline"] = oracle_decode_sample(T, min(T, 4), dev)
        out[f"decode_b{T}"] = leg

    if "decode_b1_streamed" in legs:
        out["decode_b1_streamed"] = streamed_leg(maple, layers[0], dev, stream, flush, cpu)

    if "prefill_4096" not in legs and "ternarize_pack" not in legs:
        return out
    T = 4096
    x = synth.tokens(T, H, seed=300, device=dev)
    bias = synth.bias_zipf(E, seed=0, gamma=1.0).to(dev)
    logits = torch.empty((T, E), device=dev)
    idx = torch.empty((T, K_TOP), dtype=torch.int32, device=dev)
    w = torch.empty((T, K_TOP), device=dev)
    y = torch.empty((T, H), device=dev)
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(T, K_TOP, layers[0][0]), dtype=torch.uint8,
                     device=dev)

    def prefill(i):
        ex, router = layers[i % n_stack]
        maple.maple_moe_layer(x, router, bias, ex, K_TOP, logits, idx, w, y, ws, stream=stream)
    if "prefill_4096" in legs:
        sec = timed_graph(prefill, 2, reps=2)
        flops = 2 * 3 * I * H * T * K_TOP
        out["prefill_4096"] = {"value": T / sec, "unit": "tokens/s", "ms_per_layer": sec * 1e3,
                               "dense_equiv_tflops": flops / sec / 1e12, "bias": "Zipf(1.1) ranking"}
        if cpu:
            out["prefill_4096"]["cpu_baseline"] = oracle_prefill_sample(x, layers[0], bias, 32)
    if "ternarize_pack" not in legs:
        return out

    # ternarize + pack of whole layers (all 768 matrices of a layer per chunk)
    n_pack = 2
    wts = [synth.expert_weights(E, H, I, seed=5000 + l, device=dev) for l in range(n_pack)]
    Bh, Bi = (H + 4) // 5, (I + 4) // 5
    pk = {"gate": torch.empty((E * I, Bh), dtype=torch.uint8, device=dev),
          "up": torch.empty((E * I, Bh), dtype=torch.uint8, device=dev),
          "down": torch.empty((E * H, Bi), dtype=torch.uint8, device=dev)}
    sc = {"gate": torch.empty(E * I, device=dev), "up": torch.empty(E * I, device=dev),
          "down": torch.empty(E * H, device=dev)}

    def pack(i):
        wl = wts[i % n_pack]
        for name, K in (("gate", H), ("up", H), ("down", I)):
            maple.maple_ternarize_pack(wl[name].view(-1, K), pk[name], sc[name], stream=stream)
    sec = timed_graph(pack, n_pack, reps=3)
    weights = 3 * E * H * I
    bytes_moved = weights * 2 + E * (2 * I * Bh + H * Bi) + 4 * E * (2 * I + H)
    peak, kind = _peaks()
    out["ternarize_pack"] = {"value": bytes_moved / sec / 1e9, "unit": "GB/s",
                             "frac_of_peak": bytes_moved / sec / 1e9 / peak,
                             "ms_per_layer": sec * 1e3, "bytes_per_layer": bytes_moved,
                             "weights_per_layer": weights, "peak_source": f"{kind} hbm_gbs"}
    if cpu:
        out["ternarize_pack"]["cpu_baseline"] = oracle_pack_sample(wts[0], 96, exact=False)
    del wts
    if "pack_ternary" not in legs:
        return out

    # packing of already-ternary bf16 matrices (a whole layer, as a released checkpoint
    # stores them): the trits of the pack leg times each row's scale rounded to bf16
    tern = {}
    with torch.cuda.stream(stream):
        for name, K in (("gate", H), ("up", H), ("down", I)):
            f32 = torch.empty((pk[name].shape[0], K), device=dev)
            maple.maple_unpack(pk[name], sc[name], K, f32, stream=stream)
            tern[name] = f32.to(torch.bfloat16)
            del f32
    stream.synchronize()
    pk2 = {name: torch.empty_like(t) for name, t in pk.items()}
    sc2 = {name: torch.empty_like(t) for name, t in sc.items()}
    bad = torch.zeros(1, dtype=torch.int32, device=dev)

    def pack_ternary(i):
        for name in ("gate", "up", "down"):
            maple.maple_pack_ternary(tern[name], pk2[name], sc2[name], bad, stream=stream)
    sec = timed_graph(pack_ternary, 1, reps=3)
    same = all(torch.equal(pk2[name], pk[name]) for name in pk)
    out["pack_ternary"] = {"value": bytes_moved / sec / 1e9, "unit": "GB/s",
                           "frac_of_peak": bytes_moved / sec / 1e9 / peak,
                           "ms_per_layer": sec * 1e3, "bytes_per_layer": bytes_moved,
                           "non_ternary_rows": int(bad.item()), "bytes_equal_absmean_pack": same,
                           "peak_source": f"{kind} hbm_gbs"}
    if cpu:
        out["pack_ternary"]["cpu_baseline"] = oracle_pack_sample(tern, 48, exact=True)
    del tern, pk2, sc2
    return out


def streamed_leg(maple, layer, dev, stream, flush, cpu):
    """Batch-1 decode with the layer's experts in pinned host memory and STREAM_SLOTS
    expert slots in HBM: per token, route (device), maple_cache_fetch (copies the
    missing experts across the host link) and the FFN on the cache, all in one CUDA
    graph of STREAM_STEPS distinct tokens.  Reports tokens/s, the host-link rate of the
    expert copies (the cache's own count of copied experts x their bytes, over the
    timed region) and, for comparison, the measured rate of a pinned host-to-device
    copy of 256 MB."""
    from ternary_weight_moe_02_b300 import synth
    ex, router = layer
    pool = maple.Experts(*[t.cpu().pin_memory() for t in ex.tensors], clamp=ex.clamp)
    cache = maple.ExpertCache(STREAM_SLOTS, E, H, I, clamp=ex.clamp, device=dev)
    xs = synth.tokens(2 * STREAM_STEPS, H, seed=400, device=dev)
    logits = torch.empty((1, E), device=dev)
    idx = torch.empty((1, K_TOP), dtype=torch.int32, device=dev)
    w = torch.empty((1, K_TOP), device=dev)
    idx_slot = torch.empty((1, K_TOP), dtype=torch.int32, device=dev)
    y = torch.empty((1, H), device=dev)
    ws_c = torch.empty(maple.maple_cache_fetch_workspace_size(1, K_TOP), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(maple.maple_moe_ffn_workspace_size(1, K_TOP, cache.experts), dtype=torch.uint8, device=dev)

    def step(i):
        x = xs[i:i + 1]
        maple.maple_route_topk(x, router, None, K_TOP, logits, idx, w, stream=stream)
        maple.maple_cache_fetch(pool, cache, idx, idx_slot, ws_c, stream=stream)
        maple.maple_moe_ffn(cache.experts, x, idx_slot, w, y, ws_f, stream=stream)

    def graph(start):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(STREAM_STEPS):
                    step(start + i)
        return g
    g_warm, g_time = graph(STREAM_STEPS), graph(0)
    with torch.cuda.stream(stream):
        g_warm.replay()  # fills the cache with other tokens' experts
        flush()
    stream.synchronize()
    c0 = cache.counters()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        g_time.replay()
        b.record(stream)
    b.synchronize()
    sec = a.elapsed_time(b) / 1e3
    c1 = cache.counters()
    copied = (c1["experts_copied"] - c0["experts_copied"]) * EXPERT_BYTES
    hits, misses = c1["hits"] - c0["hits"], c1["misses"] - c0["misses"]
    # the host link's plain copy rate, for comparison
    src = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    dst = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        dst.copy_(src, non_blocking=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
    b.synchronize()
    link = (256 << 20) / (a.elapsed_time(b) / 1e3) / 1e9
    del src, dst
    leg = {"value": STREAM_STEPS / sec, "unit": "tokens/s", "ms_per_token": sec * 1e3 / STREAM_STEPS,
           "cache_slots": STREAM_SLOTS, "hit_rate": hits / max(1, hits + misses),
           "experts_copied_per_token": (c1["experts_copied"] - c0["experts_copied"]) / STREAM_STEPS,
           "host_link_gbs": copied / sec / 1e9, "pinned_h2d_copy_gbs": link,
           "link_frac": copied / sec / 1e9 / link,
           "steps": "route_topk + cache_fetch + moe_ffn per token, one CUDA graph"}
    if cpu:
        leg["cpu_baseline"] = oracle_decode_sample(1, 1, dev)
    del pool, cache
    return leg


# ------------------------------------------------------------------- CPU (oracle) arm

def oracle_sample(n_tokens: int, seed_layer: int = 1000):
    """Oracle route + FFN on n_tokens of layer 0 (bf16 weights drawn on the GPU when one
    is present, else on the CPU; the oracle packs the experts it needs, untimed).
    Returns (tokens/s, seconds)."""
    import oracle
    from ternary_weight_moe_02_b300 import synth
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.expert_weights(E, H, I, seed=seed_layer, device=gen_dev)
    router = synth.bf16_bits(synth.router_weights(E, H, seed=seed_layer, device=gen_dev))
    x = synth.bf16_bits(synth.tokens(N_TOKENS, H, seed=7, device=gen_dev))[:n_tokens]
    _, idx0, _ = oracle.route(x, router, None, K_TOP)
    packed = {}
    for name, rows, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        packed[name] = np.full((E, rows, (K + 4) // 5), 121, np.uint8)
        packed["s_" + name] = np.zeros((E, rows), np.float32)
        for e in sorted(set(idx0.reshape(-1).tolist())):
            p, s = oracle.ternarize_pack(synth.bf16_bits(w[name][e]))
            packed[name][e], packed["s_" + name][e] = p, s
    del w
    t0 = time.perf_counter()
    for t in range(n_tokens):
        _, idx, wt = oracle.route(x[t:t + 1], router, None, K_TOP)
        oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                       packed["s_up"], packed["s_down"], x[t:t + 1], idx, wt)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def _oracle_layer(seed_layer: int, experts_needed, gen_dev):
    """Oracle-packed experts (only those needed; the others are never read) and the bf16
    router of the bench's layer `seed_layer` (weights drawn as build_layers draws them)."""
    import oracle
    from ternary_weight_moe_02_b300 import synth
    w = synth.expert_weights(E, H, I, seed=seed_layer, device=gen_dev)
    router = synth.bf16_bits(synth.router_weights(E, H, seed=seed_layer, device=gen_dev))
    packed = {}
    for name, rows, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        packed[name] = np.full((E, rows, (K + 4) // 5), 121, np.uint8)
        packed["s_" + name] = np.zeros((E, rows), np.float32)
        for e in sorted(set(int(v) for v in experts_needed)):
            p, s = oracle.ternarize_pack(synth.bf16_bits(w[name][e]))
            packed[name][e], packed["s_" + name][e] = p, s
    return packed, router


def _oracle_route_ffn(packed, router, x_bits, bias):
    import oracle
    _, idx, wt = oracle.route(x_bits, router, bias, K_TOP)
    oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"], packed["s_up"],
                   packed["s_down"], x_bits, idx, wt)


def oracle_decode_sample(T: int, n_tokens: int, dev) -> dict:
    """Oracle route + FFN of n_tokens of the decode leg's first stacked layer (its N(0,0.5)
    bias and token batch), as layer-tokens/s: the oracle's cost is linear in tokens, so a
    T-token layer step costs T times the per-token time, on each of the 24 layers."""
    import oracle
    from ternary_weight_moe_02_b300 import synth
    gen_dev = dev if torch.cuda.is_available() else "cpu"
    x = synth.bf16_bits(synth.tokens(T, H, seed=100, device=gen_dev))[:n_tokens]
    bias = synth.bias_normal(E, seed=200).double().numpy()
    router_bits = synth.bf16_bits(synth.router_weights(E, H, seed=1000, device=gen_dev))
    _, idx0, _ = oracle.route(x, router_bits, bias, K_TOP)
    packed, router = _oracle_layer(1000, idx0.reshape(-1), gen_dev)
    t0 = time.perf_counter()
    _oracle_route_ffn(packed, router, x, bias)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_tokens} of the {T} tokens of one 256-expert layer (route + FFN, "
                      f"{dt:.2f} s); per-token cost, the same on each of the 24 layers"}


def oracle_prefill_sample(x, layer, bias, n_ffn: int) -> dict:
    """Oracle of the 4096-token prefill: routing of all tokens timed in full, the FFN on
    n_ffn tokens stratified by the load of their first expert, scaled to all tokens."""
    import oracle
    from ternary_weight_moe_02_b300 import synth
    T = x.shape[0]
    xb = synth.bf16_bits(x)
    b = bias.double().cpu().numpy()
    router = synth.bf16_bits(layer[1])
    t0 = time.perf_counter()
    _, idx, wt = oracle.route(xb, router, b, K_TOP)
    t_route = time.perf_counter() - t0
    load = np.bincount(idx.reshape(-1), minlength=E)
    order = np.argsort(-load[idx[:, 0]], kind="stable")
    pick = order[np.linspace(0, T - 1, n_ffn).astype(np.int64)]
    ex = layer[0]
    packed = {name: t.cpu().numpy() for name, t in zip(("gate", "up", "down", "s_gate", "s_up", "s_down"),
                                                       ex.tensors)}
    t0 = time.perf_counter()
    oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"], packed["s_up"],
                   packed["s_down"], xb[pick], idx[pick], wt[pick])
    t_ffn = time.perf_counter() - t0
    est = t_route + t_ffn * T / n_ffn
    return {"value": T / est, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"routing of all {T} tokens ({t_route:.1f} s) + the FFN on {n_ffn} tokens "
                      f"stratified by expert load ({t_ffn:.1f} s), scaled to {T} tokens"}


def oracle_pack_sample(wts, n_mats: int, exact: bool) -> dict:
    """Oracle ternarize + pack (exact=False) or already-ternary pack (exact=True) of n_mats
    of a layer's matrices (a third each of gate, up and down), as GB/s of the same
    algorithmic bytes as the GPU leg (2 B read + 0.2 B written per weight + 4 B per row)."""
    import oracle
    from ternary_weight_moe_02_b300 import synth
    per = max(1, n_mats // 3)
    mats = []
    for name, K in (("gate", H), ("up", H), ("down", I)):
        src = wts[name].view(-1, I if name != "down" else H, K)
        mats += [synth.bf16_bits(src[e]) for e in range(per)]
    nbytes, dt = 0, 0.0
    for m in mats:
        t0 = time.perf_counter()
        q, s = (oracle.ternary_exact(m)[:2] if exact else oracle.ternarize(m))
        oracle.pack(q)
        dt += time.perf_counter() - t0
        rows, K = m.shape
        nbytes += rows * K * 2 + rows * ((K + 4) // 5) + 4 * rows
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(mats)} matrices of one layer ({dt:.1f} s)"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    per_step = []
    for _ in range(args.warmup):
        oracle_sample(1)
    for _ in range(args.steps):
        v, dt = oracle_sample(args.ref_tokens)
        per_step.append(dt / args.ref_tokens)
    value = 1.0 / statistics.mean(per_step)
    sample = f"{args.ref_tokens} tokens of one 256-expert layer per step (route + FFN, oracle)"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(per_step) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "maple_moe_layer_decode_b1", "hidden": H, "experts": E,
                   "top_k": K_TOP, "moe_intermediate": I, "tokens_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1000)
    ap.add_argument("--impl", default="maple", choices=["maple", "reference"])
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--chunk", type=int, default=1024,
                    help="steps per captured graph (rounded to a multiple of --layers)")
    ap.add_argument("--ref-tokens", type=int, default=4, help="oracle tokens per reference step")
    ap.add_argument("--cpu-tokens", type=int, default=40, help="oracle tokens for cpu_baseline")
    ap.add_argument("--legs", default="", help="comma-separated subset of the secondary legs "
                    + ",".join(SECONDARY_LEGS))
    ap.add_argument("--secondary", type=int, default=1,
                    help="also time decode b8/b64, the 4096-token prefill and ternarize+pack")
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        out = run_gpu(args, world, rank, local)
        if rank == 0 and world == 1 and args.cpu_tokens > 0:
            v, dt = oracle_sample(args.cpu_tokens)
            out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                   "sample": f"{args.cpu_tokens} tokens of one 256-expert layer "
                                             f"(route + FFN, single-threaded C, {dt:.1f} s)",
                                   "host_cpus": os.cpu_count()}
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

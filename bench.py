#!/usr/bin/env python
"""SlimKV decode-attention benchmark: prints ONE JSON line.

The headline workload is 128K context at 16x compression on the Llama-3.1-8B
attention shape (batch 8, 32 query / 8 KV heads, d = 128, 8192 beacon states at
latent rank 256 plus a 2048-token raw window, 32 layers). One "step" is one
decode step: the slimkv_decode_attn call of each of the 32 layers, each layer
with its own cache buffers in HBM (4 GiB of cache per step, far larger than L2,
so no flush is needed between steps).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl slimkv|reference]
                  [--config 2] [--mode latent|reconstruct|reconstruct_rope|full] [--loop 128]
                  [--layers N] [--no-companions]

Besides the device-timed step (`value`), the line carries the split-decode
kernel's roofline (CUDA events around its launch; DRAM traffic from the committed
ncu capture while the kernel sources match it), the end-to-end time through the
public API with one packed host copy of every layer's inputs in and of every
output out per step (`e2e`), the CPU oracle's time on a sample of the step
(`cpu_baseline`), the SM clocks sampled during the timed region, and a
multi-step decode of `--loop` generated tokens (window append + decode per layer,
`decode_loop`), and, for the headline workload, the comparison kernels timed on the
same layers (`baselines`: the reconstruction baseline without and with beacon-key
RoPE, full-KV attention over the 131072-token uncompressed cache) and the other two
workloads' decode steps (`configs`). Under torchrun each rank decodes its own share
of the batch.

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the pages describe a method, not a program).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & HBM GB/s (frac of 8 TB/s), 128K ctx @16x, 1 B300"
NOMINAL_HBM_GBS = 8000.0


def _measured_traffic(w, mode):
    """DRAM bytes per decode launch from the committed ncu capture, or None.

    The capture is only used while the decode kernel's sources are unchanged
    since it was taken (hashes recorded beside it) and for the workload it was
    taken on."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "tc_decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        for rel, digest in rec["source_sha256"].items():
            with open(os.path.join(ROOT, rel), "rb") as src:
                if hashlib.sha256(src.read()).hexdigest() != digest:
                    return None
    except (OSError, KeyError, ValueError):
        return None
    if mode != "latent" or not rec["workload"].startswith(w.name + ","):
        return None
    return rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def _workload(cfg: int, layers: int = 0):
    import dataclasses
    from latent_kv_cache_decode_b300 import workloads as wl
    w = wl.config(cfg)
    if layers and layers < w.layers:
        w = dataclasses.replace(w, layers=layers,
                                ranks=w.ranks[:layers] if w.ranks is not None else None)
    return w


def build_layers(w, device, unique: int = 4, batch=None):
    """Device buffers for every layer. Values come from the seeded generator for
    `unique` distinct layers (every distinct rank for variable-rank workloads);
    every layer still gets buffers of its own, so each step streams the whole
    cache from HBM. `batch` lists the global batch elements this rank owns."""
    from latent_kv_cache_decode_b300 import workloads as wl
    src = {}
    layers = []
    for l in range(w.layers):
        key = w.r(l) if w.ranks is not None else l % unique
        if key not in src:
            src[key] = wl.layer_tensors(w, l, batch=batch)
        layers.append({k: v.to(device).clone() for k, v in src[key].items()})
    return layers


def _cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


def oracle_layer_seconds(w, layers_sample):
    """Wall time of the float64 oracle on the given layers (host cores)."""
    import oracle
    from latent_kv_cache_decode_b300 import workloads as wl
    secs = []
    for l in layers_sample:
        t = wl.layer_tensors(w, l)
        f = {k: (wl.as_f64(v) if k != "q_pos" else v.numpy()) for k, v in t.items()}
        t0 = time.perf_counter()
        oracle.decode_attn(f["q"], f["C_K"], f["C_V"], f["K_raw"], f["V_raw"], f["U_K"], f["U_V"],
                           f["q_pos"], w.scale, w.rope_base)
        secs.append(time.perf_counter() - t0)
    return secs


def time_layer_graph(calls, dev, steps: int, warmup: int):
    """Device time (us) of one step: every call of `calls` once, in a CUDA graph on a
    stream of its own, CUDA events around `steps` replays after `warmup`."""
    import torch
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for c in calls:
            c(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c(stream)
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) * 1e3 / steps


def companion_measurements(args, w, layers, dev, peak):
    """The comparison kernels on the headline workload's own layers (the reconstruction
    baseline without and with beacon-key RoPE, full-KV attention over the uncompressed
    131072-token cache), and the other two workloads' decode steps, each timed as a CUDA
    graph of all layers (device time per step)."""
    import torch
    from latent_kv_cache_decode_b300 import binding as bd
    from latent_kv_cache_decode_b300 import workloads as wl
    steps, warm = max(3, min(args.steps, 10)), 3
    ws = bd.Workspace(dev)
    outs = [torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev) for _ in layers]
    kw = lambda l, st: dict(scale=w.scale, rope_base=w.rope_base, out=outs[l], workspace=ws, stream=st)
    rec = [lambda st, l=l, t=t: bd.decode_attn_reconstruct(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"],
                                                             t["U_K"], t["U_V"], t["q_pos"], **kw(l, st))
           for l, t in enumerate(layers)]
    rec_rope = [lambda st, l=l, t=t: bd.decode_attn_reconstruct_rope(t["q"], t["C_K"], t["C_V"], t["K_raw"],
                                                                       t["V_raw"], t["U_K"], t["U_V"], t["q_pos"],
                                                                       w.ratio, **kw(l, st))
                for l, t in enumerate(layers)]
    base = {"workload": w.name, "layers": w.layers,
            "reconstruct_us": time_layer_graph(rec, dev, steps, warm),
            "reconstruct_rope_us": time_layer_graph(rec_rope, dev, steps, warm)}
    # full KV: the uncompressed cache the beacons stand for (N_b x ratio = 131072 tokens),
    # two distinct per-layer buffers of 4 GiB each (>> L2) cycled over the layers
    T = w.T_full or w.N_b * w.ratio
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    full = [(torch.randn((w.B, T, w.Hkv, w.d), generator=g, device=dev, dtype=torch.bfloat16),
             torch.randn((w.B, T, w.Hkv, w.d), generator=g, device=dev, dtype=torch.bfloat16)) for _ in range(2)]
    fkv = [lambda st, l=l, t=t: bd.decode_attn_full_kv(t["q"], full[l % 2][0], full[l % 2][1], t["q_pos"],
                                                         **kw(l, st))
           for l, t in enumerate(layers)]
    base["full_kv_us"] = time_layer_graph(fkv, dev, max(3, steps // 2), warm)
    base["full_kv_cache_tokens"] = T
    base["full_kv_buffers"] = "2 distinct per-layer buffers of 4 GiB, cycled"
    del full
    torch.cuda.empty_cache()
    cfgs = {}
    for cfg in (1, 3):
        wc = _workload(cfg, args.layers)
        lc = build_layers(wc, dev)
        oc = [torch.empty((wc.B, wc.Hq, wc.d), dtype=torch.float32, device=dev) for _ in lc]
        wsc = bd.Workspace(dev)
        calls = [lambda st, l=l, t=t: bd.decode_attn(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"],
                                                      t["U_V"], t["q_pos"], scale=wc.scale, rope_base=wc.rope_base,
                                                      out=oc[l], workspace=wsc, stream=st)
                 for l, t in enumerate(lc)]
        us = time_layer_graph(calls, dev, steps, warm)
        cache_b = sum(wl.cache_bytes(wc, l) for l in range(wc.layers))
        cfgs[wc.name] = {"us_per_step": us, "layers": wc.layers, "batch": wc.B, "cache_bytes_per_step": cache_b,
                         "hbm_gbs": cache_b / (us * 1e-6) / 1e9,
                         "frac_of_measured_copy": cache_b / (us * 1e-6) / 1e9 / peak}
        del lc, oc, wsc
        torch.cuda.empty_cache()
    return base, cfgs


def prefill_flops(w, layer: int, T: int) -> float:
    """Algorithmic flops of one prefill chunk of T tokens for one layer, all batch
    elements: latent scores and values (2 T Hq N_b (r_k + r_v)), the causal chunk
    (scores and values over T (T + 1) / 2 pairs: 4 Hq d T (T + 1) / 2), and the query
    and value projections (2 T Hq d (r_k + r_v))."""
    r = w.r(layer)
    per_b = (2 * T * w.Hq * w.N_b * 2 * r + 4 * w.Hq * w.d * T * (T + 1) / 2 + 2 * T * w.Hq * w.d * 2 * r)
    return w.B * per_b


def prefill_measurement(args, w, layers, dev, chunk: int = 1024):
    """Prefill-side attention on the headline workload's layers: one chunk of `chunk`
    tokens per batch element attends to the layer's 8192 beacons and, causally, to
    itself (the chunk right after the beacons' span), timed as a CUDA graph of all
    layers. Chunk queries, keys and values are seeded device draws, four distinct sets
    cycled over the layers."""
    import torch
    from latent_kv_cache_decode_b300 import binding as bd
    steps, warm = 3, 2
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 100)
    sets = []
    for _ in range(4):
        q = torch.randn((w.B, chunk, w.Hq, w.d), generator=g, device=dev).to(torch.bfloat16)
        k = torch.randn((w.B, chunk, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
        v = torch.randn((w.B, chunk, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
        sets.append((q, k, v))
    p0 = torch.full((w.B,), w.N_b * w.ratio, dtype=torch.int32, device=dev)
    out = torch.empty((w.B, chunk, w.Hq, w.d), dtype=torch.float32, device=dev)
    ws = bd.Workspace(dev)
    calls = [lambda st, l=l, t=t: bd.prefill_attn(sets[l % 4][0], t["C_K"], t["C_V"], sets[l % 4][1], sets[l % 4][2],
                                                   t["U_K"], t["U_V"], p0, scale=w.scale, rope_base=w.rope_base,
                                                   out=out, workspace=ws, stream=st)
             for l, t in enumerate(layers)]
    us = time_layer_graph(calls, dev, steps, warm)
    fl = sum(prefill_flops(w, l, chunk) for l in range(len(layers)))
    tf = fl / (us * 1e-6) / 1e12
    peak_tf = None
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        with open(pp) as f:
            peak_tf = float(json.load(f)["bf16_tflops_sustained"])
    del sets, out, ws
    torch.cuda.empty_cache()
    return {"workload": w.name, "chunk_tokens": chunk, "beacons": w.N_b, "layers": len(layers),
            "us_per_step": us, "us_per_layer": us / len(layers),
            "tokens_per_s": w.B * chunk / (us * 1e-6),
            "flops_per_step": fl, "tflops": tf,
            "peak_tflops": peak_tf, "peak_kind": "measured bf16 sustained (cuBLAS, long loop)",
            "frac": tf / peak_tf if peak_tf else None,
            "how": "CUDA graph of all layers (staging kernel + tensor-core prefill kernel per layer), "
                   "CUDA events over 3 replays after 2"}


def run_reference(args):
    """CPU oracle arm: each step is one sampled layer, reported per full step."""
    w = _workload(args.config, args.layers)
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    n = args.warmup + args.steps
    layers = [(i * 7) % w.layers for i in range(n)]
    secs = oracle_layer_seconds(w, layers)
    timed = secs[args.warmup:]
    us_step = statistics.mean(timed) * w.layers * 1e6
    sample = (f"{len(timed)} sampled layers of {w.layers} (one per step, after {args.warmup} "
              f"warm-up layers), float64 numpy oracle, mean per layer x{w.layers}")
    return {"impl": "reference", "metric": METRIC, "value": us_step, "unit": "us/step",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": {"workload": w.name, "batch": w.B, "layers": w.layers, "N_b": w.N_b,
                       "W": w.W, "rank": w.rank or "per-layer", "mode": "latent"},
            "cpu_baseline": {"value": us_step, "unit": "us/step", "cores": _cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": us_step, "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_slimkv(args):
    import torch
    import torch.distributed as dist
    from latent_kv_cache_decode_b300 import binding as bd
    from latent_kv_cache_decode_b300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = bd.load()
    w = _workload(args.config, args.layers)
    mode = args.mode
    from latent_kv_cache_decode_b300.sharding import batch_shard, max_over_ranks
    layers = build_layers(w, dev, batch=batch_shard(w.B, world, rank))
    full = []
    n_buf = 0
    if mode == "full":
        # uncompressed cache of T_full tokens per layer (the context the compressed cache
        # stands for, N_b x ratio, when the workload names none), drawn on the device from
        # a seeded generator; cycled over distinct buffers when HBM is short
        if not w.T_full:
            w = dataclasses.replace(w, T_full=w.N_b * w.ratio)
        free, _ = torch.cuda.mem_get_info()
        per_layer = 2 * w.B * w.T_full * w.Hkv * w.d * 2
        n_buf = max(2, min(w.layers, int(0.8 * free // per_layer)))
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        for _ in range(n_buf):
            K = torch.randn((w.B, w.T_full, w.Hkv, w.d), generator=g, device=dev, dtype=torch.bfloat16)
            V = torch.randn((w.B, w.T_full, w.Hkv, w.d), generator=g, device=dev, dtype=torch.bfloat16)
            full.append((K, V))
    stream = torch.cuda.Stream(device=dev)
    ws = bd.Workspace(dev)
    outs = [torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev) for _ in layers]

    def call(l, t):
        kw = dict(scale=w.scale, rope_base=w.rope_base, out=outs[l], workspace=ws, stream=stream)
        if mode == "latent":
            bd.decode_attn(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"], t["U_V"],
                           t["q_pos"], **kw)
        elif mode == "reconstruct":
            bd.decode_attn_reconstruct(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"],
                                       t["U_V"], t["q_pos"], **kw)
        elif mode == "reconstruct_rope":
            bd.decode_attn_reconstruct_rope(t["q"], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"],
                                            t["U_V"], t["q_pos"], w.ratio, **kw)
        else:
            K, V = full[l % n_buf]
            bd.decode_attn_full_kv(t["q"], K, V, t["q_pos"], **kw)

    def step():
        for l, t in enumerate(layers):
            call(l, t)

    # size the workspace and build the plans outside the capture
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist if world > 1 else None, dev)

    # dominant kernel (split decode) timed alone: CUDA events recorded by the library on
    # the launching stream right before and after each layer's decode launch, captured
    # with the layer calls in a CUDA graph of their own (as the timed step is), so that
    # the events bracket the device-side launch and run of the kernel, not the host's
    # submission of it; the event nodes also break the programmatic-launch overlap with
    # the query projection, so the kernel's prologue is inside the bracket
    from cuda.bindings import runtime as rt
    evs = [(rt.cudaEventCreate()[1], rt.cudaEventCreate()[1]) for _ in layers]

    def timed_step():
        for l, t in enumerate(layers):
            lib.slimkv_time_next_decode(int(evs[l][0]), int(evs[l][1]))
            call(l, t)

    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph, stream=stream):
        timed_step()
    torch.cuda.synchronize()
    kern_ms = []
    for rep in range(1 + max(1, min(args.steps, 5))):
        with torch.cuda.stream(stream):
            tgraph.replay()
        torch.cuda.synchronize()
        if rep == 0:
            continue   # warm-up replay
        for a, b in evs:
            err, t_ms = rt.cudaEventElapsedTime(a, b)
            if err != rt.cudaError_t.cudaSuccess:
                raise RuntimeError(f"cudaEventElapsedTime: {err}")
            kern_ms.append(t_ms)
    for a, b in evs:
        rt.cudaEventDestroy(a)
        rt.cudaEventDestroy(b)
    del tgraph
    kern_avg_ms = statistics.mean(kern_ms)

    # end to end through the public API with host buffers: every step copies every
    # layer's q and q_pos from pinned host memory, runs the layer calls, and reads every
    # output back, inside the timed region (the cache is device-resident state, like
    # model weights); the step runs as a captured graph (`e2e`) and, separately, issued
    # call by call (`eager_value`)
    L = len(layers)
    q_dev = torch.stack([t["q"] for t in layers])            # [L, B, Hq, d]
    pos_dev = torch.stack([t["q_pos"] for t in layers])      # [L, B]
    out_dev = torch.empty((L,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=dev)
    q_host = q_dev.cpu().pin_memory()
    pos_host = pos_dev.cpu().pin_memory()
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    e2e_layers = [dict(t, q=q_dev[l], q_pos=pos_dev[l]) for l, t in enumerate(layers)]
    h2d = q_host.numel() * q_host.element_size() + pos_host.numel() * pos_host.element_size()
    d2h = out_host.numel() * out_host.element_size()
    outs_saved = outs[:]
    outs[:] = [out_dev[l] for l in range(L)]
    e2e_steps = max(1, args.steps)
    with torch.cuda.stream(stream):   # one untimed pass (host-side caches)
        for l, t in enumerate(e2e_layers):
            call(l, t)
    torch.cuda.synchronize()
    # the step's transfers are pipelined with its layers, as a serving loop would: the
    # layers run in chunks of CH; each chunk's q / q_pos go up on a copy stream ahead of
    # it (the first chunk before any layer), and its outputs come back on that stream
    # while the later chunks compute; the step ends when the last outputs are on the host
    CH = 4
    chunks = [(c, min(c + CH, L)) for c in range(0, L, CH)]
    cstream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_out = [torch.cuda.Event() for _ in chunks]

    def e2e_step():
        cstream.wait_stream(stream)   # the previous step is done with q_dev / out_dev
        with torch.cuda.stream(cstream):
            for i, (a, z) in enumerate(chunks):
                q_dev[a:z].copy_(q_host[a:z], non_blocking=True)
                pos_dev[a:z].copy_(pos_host[a:z], non_blocking=True)
                ev_in[i].record(cstream)
        for i, (a, z) in enumerate(chunks):
            stream.wait_event(ev_in[i])
            for l in range(a, z):
                call(l, e2e_layers[l])
            ev_out[i].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(ev_out[i])
                out_host[a:z].copy_(out_dev[a:z], non_blocking=True)
        stream.wait_stream(cstream)   # the step's outputs are on the host

    with torch.cuda.stream(stream):   # one untimed step (first use of the copy stream and events)
        e2e_step()
    torch.cuda.synchronize()
    # eager: the 32 library calls issued from Python every step
    # each step waits for its outputs on the host before the next is issued, as a decode
    # loop must (the next token's input depends on them)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            e2e_step()
            stream.synchronize()
    e2e_eager_us = (time.perf_counter() - t0) / e2e_steps * 1e6
    # graph: the same step (calls and transfers) captured once in a CUDA graph, replayed
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            g_e2e.replay()
            stream.synchronize()
    e2e_us = (time.perf_counter() - t0) / e2e_steps * 1e6
    torch.cuda.synchronize()
    if not torch.equal(out_host, out_dev.cpu()):
        raise RuntimeError("end-to-end step: the outputs read back differ from the device outputs")
    del g_e2e
    outs[:] = outs_saved

    # multi-step decode: args.loop generated tokens, each appending its key and value
    # to every layer's window ring and running the layer's decode at its position
    # (append + query projection + decode + combine per layer), one CUDA graph per
    # token replayed with the position buffer advanced in between; run last, as the
    # appends overwrite the windows
    loop = None
    if args.loop > 0 and mode == "latent":
        # every (token, layer) gets its own query, key and value: seeded device draws for
        # all tokens, copied into the graph's input buffers before each token's replay
        # (inside the timed region, like the position)
        Bl = layers[0]["q"].shape[0]
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed * 1000 + 17 + rank)
        q_all = torch.randn((args.loop, w.layers, Bl, w.Hq, w.d), generator=gen, device=dev).to(w.torch_dtype())
        kv_all = torch.randn((args.loop, 2, w.layers, Bl, w.Hkv, w.d), generator=gen, device=dev).to(w.torch_dtype())
        q_cur = q_all[0].clone()
        kv_cur = kv_all[0].clone()
        pos_all = (layers[0]["q_pos"].to(torch.int64)[None, :] +
                   torch.arange(args.loop + 1, device=dev)[:, None]).to(torch.int32)
        pos_cur = pos_all[0].clone()

        def token_step():
            for l, t in enumerate(layers):
                bd.append_kv(kv_cur[0, l], kv_cur[1, l], t["K_raw"], t["V_raw"], pos_cur, rope_base=w.rope_base,
                             stream=stream)
                bd.decode_attn(q_cur[l], t["C_K"], t["C_V"], t["K_raw"], t["V_raw"], t["U_K"], t["U_V"], pos_cur,
                               scale=w.scale, rope_base=w.rope_base, out=outs[l], workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            token_step()
        torch.cuda.synchronize()
        g_tok = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_tok, stream=stream):
            token_step()
        torch.cuda.synchronize()
        la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            la.record(stream)
            for i in range(args.loop):
                pos_cur.copy_(pos_all[i + 1], non_blocking=True)
                q_cur.copy_(q_all[i], non_blocking=True)
                kv_cur.copy_(kv_all[i], non_blocking=True)
                g_tok.replay()
            lb.record(stream)
        torch.cuda.synchronize()
        us_tok = la.elapsed_time(lb) * 1e3 / args.loop
        loop = {"tokens": args.loop, "us_per_token": us_tok, "tokens_per_s": world * w.B / (us_tok * 1e-6),
                "per_token": f"{w.layers} layers x (window append + decode), CUDA graph per token; each token's "
                             "queries, keys and values (distinct per token and layer) copied into the graph's "
                             "inputs before its replay",
                "gpu_launches_per_token": w.layers * 4}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peak, peak_kind = _peaks()
    if mode == "full":
        cache_b = w.layers * 2 * w.B * w.T_full * w.Hkv * w.d * 2
    else:
        cache_b = sum(wl.cache_bytes(w, l) for l in range(w.layers))
    us = ms * 1e3
    layer_bytes = cache_b / w.layers
    achieved = layer_bytes / (kern_avg_ms * 1e-3) / 1e9
    launches_per_call = {"latent": 3, "reconstruct": 5, "reconstruct_rope": 5, "full": 3}[mode]
    res = {
        "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator)",
        "config": {"workload": w.name, "batch": w.B, "layers": w.layers, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, "N_b": w.N_b, "rank": w.rank or "per-layer", "W": w.W, "mode": mode,
                   "parallelism": f"batch-sharded dp{world}" if world > 1 else "1 GPU",
                   "global_batch": world * w.B,
                   "l2": "no flush: each step streams the whole per-layer cache (>> 126 MB L2)"},
        "tokens_per_s": world * w.B / (ms * 1e-3),
        "cache_bytes_per_step": cache_b,
        "hbm_gbs": cache_b / (ms * 1e-3) / 1e9,
        "frac_of_8tbs": cache_b / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "frac_of_measured_copy": cache_b / (ms * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": "tc_decode_kernel", "achieved": achieved,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _measured_traffic(w, mode),
                     "launch_us": kern_avg_ms * 1e3, "bytes_per_launch": layer_bytes},
        "clocks": clk.summary(),
        "e2e": {"value": e2e_us, "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": f"host clock over {max(1, args.steps)} steps, each ended by a stream sync (the host "
                       "holds the step's outputs before it issues the next): pinned H2D of every layer's "
                       "q and q_pos and D2H of every output, pipelined in chunks of 4 layers on a copy "
                       f"stream with the {w.layers} library calls, all captured in one CUDA graph",
                "eager_value": e2e_eager_us,
                "eager_how": f"the same, with the {w.layers} library calls and the transfers issued "
                             "from Python every step"},
        "gpu_launches": args.steps * w.layers * launches_per_call,
    }
    if loop is not None:
        res["decode_loop"] = loop
    if args.companions and world == 1 and mode == "latent" and args.config == 2:
        res["baselines"], res["configs"] = companion_measurements(args, w, layers, dev, peak)
        res["prefill"] = prefill_measurement(args, w, layers, dev)
    if not args.no_cpu_baseline and world == 1:
        sample_layers = [0, w.layers // 2]
        secs = oracle_layer_seconds(w, sample_layers)
        v = statistics.mean(secs) * w.layers * 1e6
        res["cpu_baseline"] = {"value": v, "unit": "us/step", "cores": _cpu_cores(), "kind": "oracle",
                               "sample": f"layers {sample_layers} of {w.layers}, float64 numpy "
                                         f"oracle, mean per layer x{w.layers}"}
    if world > 1:
        dist.destroy_process_group()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="slimkv", choices=["slimkv", "reference"])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--mode", default="latent", choices=["latent", "reconstruct", "reconstruct_rope", "full"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--loop", type=int, default=128,
                    help="generated tokens of the multi-step decode measurement (0: skip)")
    ap.add_argument("--no-companions", dest="companions", action="store_false",
                    help="skip the comparison kernels and the other workloads in the line")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (small profiling captures; 0 = all)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    res = run_reference(args) if args.impl == "reference" else run_slimkv(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the GB300 CacheBlend per-layer KV blend.

Metric: context tokens blended per second per layer = n_ctx * layers / step
time, where one step is the whole hot path (deviation, top-k under the
gradual filter, fused cache, query encoding, causal GQA attention) over every
layer of one synthetic request. Default workload: the long-context
Mistral-7B-shaped 32-layer blend (16 x 2048 cached tokens + 128 suffix
tokens, 32 q / 8 kv heads, head_dim 128, r1 = 30% -> r2 = 15%), the largest
of the blend workloads that fits one GPU.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Our arm: inputs resident in HBM (per-layer buffers, 17 GB per step at the
default workload, far larger than L2); each step is one cb_blend_request call
through the C ABI (all layers, pipelined over the plan's streams), replayed as
a CUDA graph. Per-kernel times come from one more CUDA graph per stage
(cb_blend_stage): that stage's kernel for every layer that has it, back to
back on one stream, replayed `steps` times; a kernel's time is the graph's
time over its launches (no events between kernels, which would serialise
their programmatic launch overlap). `e2e` repeats the metric through the C ABI
from pinned host buffers with the host-to-device copies of every layer's
inputs and the device-to-host copy of its outputs inside the timed region.
`cpu_baseline` times the CPU oracle on a bounded sample (seeded row samples
of layers 1, 2 and 3; each part's time scaled by its work, then per-step time
t1 + t2 + (layers - 2) t3). The reference arm (--impl reference) times the
CPU oracle itself the same way, one sampled layer per step.
Under torchrun each rank runs an independent replica (the blend of one
request does not shard); value = all ranks' tokens / the slowest rank's time.
`--path sweep` times the single-layer blend at every recompute ratio of the
ratio-sweep workload.
"""

from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "context tokens blended/s per layer"
UNIT = "tokens/s"
STAGES = ("deviation", "topk", "fuse", "attention")
DEFAULT_WORKLOAD = {"blend": "long32k", "sweep": "sweep", "decode": "long32k", "diagnostics": "sweep",
                    "projection": "mistral7b"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    help="workload name (default: long32k for the blend and decode paths, sweep for the sweep "
                         "and diagnostics paths, mistral7b for the projection path)")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--path", choices=["blend", "sweep", "decode", "diagnostics", "projection"], default="blend",
                    help="blend: the per-layer blend (default); sweep: the single-layer blend at every "
                         "recompute ratio of the ratio-sweep workload, L2 flushed between repetitions; "
                         "decode: one decode step's attention over "
                         "every layer's cache after the request; diagnostics: attention deviation of the "
                         "fused cache from a full prefill over the recompute ratios, and attention sparsity; "
                         "projection: the gathered QKV projection of every layer's recomputed rows")
    ap.add_argument("--eps", type=float, default=1e-3, help="sparsity threshold of the diagnostics path")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (smaller captures for profiling; not a bench line)")
    ap.add_argument("--deviation", choices=["v", "kv"], default="v",
                    help="rank by the V deviation (default) or by the K+V deviation")
    ap.add_argument("--filter", choices=["keep", "reselect"], default="keep",
                    help="layers >= 3 keep S_{l-1} (default) or re-select from the layer-1 pool")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device, world):
    """The largest value of x over the ranks (the slowest rank's time); x itself on one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units all ranks processed per second, over the slowest rank's time in ms."""
    return units_per_rank * world / (ms / 1e3)


def workload_desc(cfg):
    return (f"{cfg.name}: {cfg.n_chunks}x{cfg.chunk_len} cached + {cfg.n_suffix} suffix tokens, "
            f"{cfg.hq} q / {cfg.hkv} kv heads, head_dim {cfg.head_dim}, RoPE theta {cfg.rope_theta:g}, "
            f"{cfg.layers} layers, r1 {cfg.r1_pct}% -> r2 {cfg.r2_pct}%")


def data_desc(cfg):
    noise = (f"sigma {cfg.sigma_hi} on a seeded {cfg.hkvd_frac:.0%} set, {cfg.sigma_lo} elsewhere, "
             f"{cfg.swap_frac:.0%} of the set swapped per layer" if cfg.noise == "set"
             else f"lognormal per-token scale (mu {cfg.lognormal_mu}, sigma {cfg.lognormal_sigma})")
    return f"synthetic: seeded N(0,1) bf16 caches and queries; recomputed K/V = cached + noise ({noise})"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm", "clocks.max.sm", "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- oracle (CPU)
def oracle_chain(cfg, inputs, deviation="v", filter="keep"):
    """The oracle's own selection chain over the given layers (inputs of layers 1, 2, ...):
    ([(layer, C_l, k_l, selects)], {layer: S_l})."""
    from oracle.blend import candidate_layer, gradual_filter_schedule
    from oracle.deviation import deviation_canonical_f32, kv_deviation_canonical_f32
    from oracle.positions import chunk_local_positions
    from oracle.topk import hkvd_topk

    sched = gradual_filter_schedule(cfg.n_ctx, cfg.layers, cfg.r1_pct, cfg.r2_pct, filter)
    p_old = chunk_local_positions(cfg.n_chunks, cfg.chunk_len)
    sels = {0: np.arange(cfg.n_ctx)}
    chain = []
    for (layer, k, selects), inp in zip(sched, inputs):
        cand = sels[candidate_layer(layer, filter)]
        chain.append((layer, cand, k, selects))
        sels[layer] = cand
        if selects:
            if deviation == "kv":
                dev = kv_deviation_canonical_f32(inp.k_new[cand], inp.k_old[cand], inp.v_new[cand], inp.v_old[cand],
                                                 p_old[cand], cfg.rope_theta)
            else:
                dev = deviation_canonical_f32(inp.v_new[cand], inp.v_old[cand])
            sels[layer], _ = hkvd_topk(dev, cand, k)
    return chain, sels


def generate_inputs(cfg, layer_ids, sets, workers=None, consume=None):
    """Inputs of the given layers, generated on the host cores in parallel (each layer's
    random streams are independent, and numpy's generators release the GIL). With `consume`,
    each layer is handed to consume(LayerInputs) as soon as it is ready and its result kept
    instead (so the raw arrays of all layers need not be held at once)."""
    from concurrent.futures import ThreadPoolExecutor, as_completed

    from workloads.generator import generate_layer

    workers = max(1, min(len(layer_ids), workers or os.cpu_count() or 1))
    out = {}
    with ThreadPoolExecutor(max_workers=workers) as ex:
        futs = {ex.submit(generate_layer, cfg, layer, sets): layer for layer in layer_ids}
        for f in as_completed(futs):
            inp = f.result()
            out[futs[f]] = consume(inp) if consume else inp
            del inp
    return [out[layer] for layer in layer_ids]


def _attention_blocks(q_pos, block):
    """[(first row, rows, key rows)] of the oracle's row blocks of causal_gqa_attention: each block
    of `block` consecutive query rows computes scores against keys 0 .. (its last position)."""
    return [(b0, min(block, q_pos.size - b0), int(q_pos[min(q_pos.size, b0 + block) - 1]) + 1)
            for b0 in range(0, q_pos.size, block)]


def oracle_layer_sample(cfg, inp, entry, sel_tok, rng, row_frac, n_blocks, deviation="v", block=256):
    """Time the CPU oracle on a seeded sample of one layer.

    Returns (cpu seconds spent, estimated seconds of the whole layer). Every part runs the
    oracle's own functions on a seeded fraction row_frac of its rows: the deviation and top-k of
    a filtering layer (over that fraction of the candidates, k scaled alike), the re-rotation of
    cached keys, the encoding of recomputed keys (rows of S_l and the suffix), the fuse (the row
    copies it defines) and the query encoding; these times are scaled by 1 / row_frac. The
    attention runs the oracle's causal_gqa_attention on n_blocks of the row blocks it forms over
    Q_l (blocks of `block` consecutive query rows against the full cache), and its time is scaled
    by the score entries of all blocks over those of the sampled ones. The rows of the attention's
    cache that the sample did not fuse keep their cached values: the oracle's time does not depend
    on the values, and its outputs are discarded here."""
    from oracle.attention import causal_gqa_attention
    from oracle.deviation import bf16_bits_to_f64, deviation_canonical_f32, kv_deviation_canonical_f32
    from oracle.positions import chunk_local_positions
    from oracle.rope import rerotate, rope_rotate, round_bf16
    from oracle.topk import hkvd_topk

    layer, cand, k, selects = entry
    n_ctx, n = cfg.n_ctx, cfg.n_tokens
    p_old = chunk_local_positions(cfg.n_chunks, cfg.chunk_len)
    q_tok = np.concatenate([np.asarray(sel_tok, dtype=np.int64), np.arange(n_ctx, n)])

    def pick(arr, frac):
        arr = np.asarray(arr, dtype=np.int64)
        m = min(arr.size, max(1, int(round(frac * arr.size))))
        return np.sort(rng.choice(arr, size=m, replace=False)) if m < arr.size else arr

    c_s = pick(cand, row_frac) if selects and len(cand) else None
    r_s = pick(np.arange(n_ctx), row_frac) if n_ctx else np.zeros(0, np.int64)
    n_s = pick(q_tok, row_frac) if q_tok.size else np.zeros(0, np.int64)
    blocks = _attention_blocks(q_tok, block)
    chosen = sorted(rng.choice(len(blocks), size=min(n_blocks, len(blocks)), replace=False)) if blocks else []
    # untimed: the attention's full-length cache, and its sampled blocks' encoded queries
    kbuf = bf16_bits_to_f64(np.concatenate([inp.k_old, inp.k_new[n_ctx:]]))
    vbuf = bf16_bits_to_f64(np.concatenate([inp.v_old, inp.v_new[n_ctx:]]))
    q_blocks = [(q_tok[b0:b0 + m], round_bf16(rope_rotate(bf16_bits_to_f64(inp.q[q_tok[b0:b0 + m]]),
                                                          q_tok[b0:b0 + m], cfg.rope_theta)))
                for b0, m, _ in (blocks[i] for i in chosen)]

    t0 = time.perf_counter()
    if c_s is not None:
        if deviation == "kv":
            dev = kv_deviation_canonical_f32(inp.k_new[c_s], inp.k_old[c_s], inp.v_new[c_s], inp.v_old[c_s],
                                             p_old[c_s], cfg.rope_theta)
        else:
            dev = deviation_canonical_f32(inp.v_new[c_s], inp.v_old[c_s])
        hkvd_topk(dev, c_s, (k * c_s.size) // len(cand))
    if r_s.size:
        kbuf[r_s] = round_bf16(rerotate(bf16_bits_to_f64(inp.k_old[r_s]), p_old[r_s], r_s, cfg.rope_theta))
    if n_s.size:
        kbuf[n_s] = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new[n_s]), n_s, cfg.rope_theta))
        vbuf[n_s] = bf16_bits_to_f64(inp.v_new[n_s])
        round_bf16(rope_rotate(bf16_bits_to_f64(inp.q[n_s]), n_s, cfg.rope_theta))
    t1 = time.perf_counter()
    for pos, q_rot in q_blocks:
        causal_gqa_attention(q_rot, pos, kbuf, vbuf, block=block)
    t2 = time.perf_counter()
    # work of each part over the work sampled
    stream_scale = 1.0 / row_frac
    w_all = sum(m * kend for _, m, kend in blocks)
    w_s = sum(blocks[i][1] * blocks[i][2] for i in chosen)
    attn_scale = w_all / w_s if w_s else 0.0
    return t2 - t0, (t1 - t0) * stream_scale + (t2 - t1) * attn_scale


def oracle_step_estimate(cfg, layer_times):
    """Per-step time of the whole request from per-layer estimates of layers 1, 2 and 3: layers
    >= 3 all do the work of layer 3 (same candidate and query counts)."""
    t = {layer: statistics.mean(v) for layer, v in layer_times.items()}
    if cfg.layers >= 3:
        return t[1] + t[2] + (cfg.layers - 2) * t[3]
    return sum(t[layer] for layer in range(1, cfg.layers + 1))


def sampled_layers(cfg):
    return list(range(1, min(3, cfg.layers) + 1))


def cpu_baseline(cfg, inputs, deviation="v", filter="keep"):
    """The oracle on seeded samples of layers 1, 2 and 3 (inputs: their LayerInputs)."""
    layer_ids = sampled_layers(cfg)
    chain, sels = oracle_chain(cfg, inputs[:len(layer_ids)], deviation, filter)
    rng = np.random.default_rng(cfg.seed + 17)
    row_frac = min(1.0, 8192.0 / max(1, cfg.n_ctx))
    n_blocks = 4
    spent, est = 0.0, {}
    for i, layer in enumerate(layer_ids):
        s, e = oracle_layer_sample(cfg, inputs[i], chain[i], sels[layer], rng, row_frac, n_blocks, deviation)
        spent += s
        est[layer] = [e]
    t_step = oracle_step_estimate(cfg, est)
    sample = (f"oracle on seeded samples of layers {', '.join(map(str, layer_ids))} of {cfg.name}: "
              f"{row_frac:.3g} of the rows of deviation, top-k, re-rotation, encoding and fuse (time x "
              f"{1 / row_frac:.3g}) and {n_blocks} of its 256-query-row attention blocks per layer (time x the "
              f"score entries of all blocks / sampled); {spent:.1f} s of CPU work; per-step time "
              f"t1 + t2 + {max(0, cfg.layers - 2)} t3 = {t_step:.1f} s")
    return {"value": cfg.n_ctx * cfg.layers / t_step, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": sample + "; numpy fp64 with its BLAS on all host cores"}


def run_reference(args, cfg):
    from workloads.generator import hkvd_noise_sets

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    sets = hkvd_noise_sets(cfg)
    layer_ids = sampled_layers(cfg)
    inputs = generate_inputs(cfg, layer_ids, sets)
    chain, sels = oracle_chain(cfg, inputs, args.deviation, args.filter)
    rng = np.random.default_rng(cfg.seed + 29)
    row_frac = min(1.0, 2048.0 / max(1, cfg.n_ctx))
    # steps cycle over layers 1, 3, 2, 3 (layers >= 3 all do layer 3's work)
    cycle = [x for x in (1, 3, 2, 3) if x in layer_ids]

    def one(i):
        j = layer_ids.index(cycle[i % len(cycle)])
        return oracle_layer_sample(cfg, inputs[j], chain[j], sels[layer_ids[j]], rng, row_frac, 1, args.deviation)

    for i in range(args.warmup):
        one(i)
    spent, est = 0.0, {}
    for i in range(args.steps):
        s, e = one(i)
        spent += s
        est.setdefault(cycle[i % len(cycle)], []).append(e)
    for layer in layer_ids:  # too few steps to reach a layer: time one more sample of it
        if layer not in est:
            s, e = oracle_layer_sample(cfg, inputs[layer_ids.index(layer)], chain[layer_ids.index(layer)],
                                       sels[layer], rng, row_frac, 1, args.deviation)
            est[layer] = [e]
    t_step = oracle_step_estimate(cfg, est)
    value = cfg.n_ctx * cfg.layers / t_step
    sample = (f"each step the oracle on a seeded sample of one layer of {cfg.name} (layers 1, 3, 2, 3, ... in "
              f"turn; layers >= 3 all do layer 3's work): {row_frac:.3g} of the rows of deviation, top-k, "
              f"re-rotation, encoding and fuse (time x {1 / row_frac:.3g}) and one 256-query-row attention block "
              f"(time x the score entries of all blocks / sampled); per-layer estimates averaged per layer, "
              f"per-step time t1 + t2 + {max(0, cfg.layers - 2)} t3 = {t_step:.1f} s; "
              f"{spent:.1f} s of CPU work in the timed steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / max(1, args.steps),
            "est_ms_per_request": 1e3 * t_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": data_desc(cfg), "config": {"workload": workload_desc(cfg), "n_ctx": cfg.n_ctx,
                                               "n_tokens": cfg.n_tokens, "layers": cfg.layers,
                                               "deviation": args.deviation, "filter": args.filter},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm
def attention_flops(cfg, sel_tok):
    q_pos = np.concatenate([np.asarray(sel_tok, dtype=np.int64), np.arange(cfg.n_ctx, cfg.n_tokens)])
    return 4.0 * cfg.hq * cfg.head_dim * float(np.sum(q_pos + 1))


def stage_bytes(cfg, n_cand, k, mq, selects, deviation="v"):
    """Algorithmic HBM bytes of one layer's streaming kernels: deviation reads V_new and V_old of
    the candidates (and K_new, K_old for the K+V deviation); the fuse pass reads and writes K and
    V of every row and reads and writes the query rows it encodes."""
    row_kv = cfg.hkv * cfg.head_dim * 2
    row_q = cfg.hq * cfg.head_dim * 2
    reads = 4.0 if deviation == "kv" else 2.0
    return {"deviation": reads * n_cand * row_kv if selects else 0.0,
            "fuse": 4.0 * cfg.n_tokens * row_kv + 2.0 * mq * row_q}


def stage_applies(name, size):
    n_cand, k, mq, selects = size
    return {"deviation": bool(selects), "topk": bool(selects), "fuse": True, "attention": mq > 0}[name]


def traffic_for(kernel_src, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel source on this
    workload, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        src = open(os.path.join(ROOT, "rag_kv_cache_gb300", "csrc", kernel_src), "rb").read()
        entry = rec.get(f"{kernel_src}@{workload}")
        if entry and entry.get("source_sha256") == hashlib.sha256(src).hexdigest():
            return entry
    except (OSError, ValueError):
        pass
    return None


def pinned_layer(inp):
    """A LayerInputs whose five tensors now live in pinned host memory: `.pinned` holds them as
    torch bf16 tensors and the numpy fields become uint16 views of the same bytes."""
    import torch

    from workloads.torch_io import bf16_tensor

    pinned = {}
    for name in ("k_old", "v_old", "k_new", "v_new", "q"):
        t = bf16_tensor(getattr(inp, name), "cpu", pin=True)
        pinned[name] = t
        setattr(inp, name, t.view(torch.int16).numpy().view(np.uint16))
    inp.pinned = pinned
    return inp


def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    import rag_kv_cache_gb300 as cb
    from rag_kv_cache_gb300.build import build
    from workloads.generator import hkvd_noise_sets

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)

    sets = hkvd_noise_sets(cfg)
    # Inputs go straight to pinned host memory (the source of both the device copies and the
    # end-to-end run); the oracle samples read layers 1-3 through numpy views of the same bytes.
    host_inputs = generate_inputs(cfg, list(range(1, cfg.layers + 1)), sets,
                                  workers=max(1, (os.cpu_count() or 1) // world), consume=pinned_layer)
    d_in = [{name: t.to(dev) for name, t in h.pinned.items()} for h in host_inputs]
    plan = cb.Plan.from_config(cfg, deviation=args.deviation, filter=args.filter)
    bufs = [cb.LayerBuffers(plan, dev) for _ in range(cfg.layers)]

    def cand_of(li):  # C of layer li + 1: the selection of the layer the plan's filter names
        c = plan.candidate_layer(li + 1)
        return None if c == 0 else bufs[c - 1].sel_tok
    sizes = [plan.layer_sizes(layer) for layer in range(1, cfg.layers + 1)]
    stream = torch.cuda.Stream(dev)

    layers_spec = [dict(bufs=bufs[li], **d_in[li]) for li in range(cfg.layers)]

    def step():
        # the whole request in one call: layers pipelined over the plan's streams
        cb.cb_blend_request(plan, layers_spec, stream=stream)

    # warm up eagerly (first launches configure the kernels), check the device error word
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    stream.synchronize()
    plan.check()

    use_graph = not args.no_graph
    chunk = 32
    plain_graphs = []
    if use_graph:
        try:
            warm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(warm, stream=stream):
                step()
            for s0 in range(0, args.steps, chunk):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(s0, min(args.steps, s0 + chunk)):
                        step()
                plain_graphs.append(g)
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    warm.replay()
            stream.synchronize()
        except Exception as e:  # capture unsupported: fall back to eager launches
            print(f"bench: CUDA graph capture failed ({e}); timing eager launches", file=sys.stderr)
            use_graph, plain_graphs = False, []

    def timed(fn):
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            start.record(stream)
            fn()
            stop.record(stream)
        stream.synchronize()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        return start.elapsed_time(stop)

    def run_steps():
        if use_graph:
            for g in plain_graphs:
                g.replay()
        else:
            for _ in range(args.steps):
                step()

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    with ClockSampler(gpu_index) as clocks:
        elapsed_ms = timed(run_steps)
    plan.check()
    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(cfg.n_ctx * cfg.layers * args.steps, world, elapsed_ms)

    # Per-kernel times: one graph per stage holding that stage's kernel for every layer that has
    # it (cb_blend_stage; each stage rewrites its outputs from its inputs, so replays are idempotent).
    stage_ms, stage_launches = {}, {}
    for name in STAGES:
        layer_ids = [li for li in range(cfg.layers) if stage_applies(name, sizes[li])]
        if not layer_ids:
            continue

        def stage_pass(name=name, layer_ids=layer_ids):
            for li in layer_ids:
                cb.cb_blend_stage(plan, li + 1, name, cand=cand_of(li), bufs=bufs[li], stream=stream, **d_in[li])

        if use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                stage_pass()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
            ms = timed(lambda: [g.replay() for _ in range(args.steps)])
        else:
            with torch.cuda.stream(stream):
                stage_pass()
            ms = timed(lambda: [stage_pass() for _ in range(args.steps)])
        stage_ms[name] = ms / args.steps
        stage_launches[name] = len(layer_ids)
    plan.check()

    flops = np.array([attention_flops(cfg, bufs[li].sel_tok[: sizes[li][1]].cpu().numpy())
                      for li in range(cfg.layers)])
    peaks = load_peaks()
    attn_s = stage_ms["attention"] / 1e3
    achieved_tf = float(flops.sum()) / attn_s / 1e12
    peak_tf = peaks["bf16_tflops_sustained"]
    # the kernel the request's attention launches run (all layers of a workload take the same one here)
    paired = cb.cb_attention_uses_paired_tiles(plan, sizes[-1][2])
    traffic = traffic_for("attention_pp.cu" if paired else "attention.cu", cfg.name)
    roofline = {"kernel": "hkvd_attention_pp (two query tiles per CTA)" if paired else "hkvd_attention",
                "bound": "tensor", "achieved": achieved_tf, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": achieved_tf / peak_tf,
                "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                "peak_source": f"{peaks['source']} bf16 sustained (kernel timed inside a long step)",
                "flops_per_step": float(flops.sum()), "launches_per_step": stage_launches["attention"],
                "avg_launch_us": 1e3 * stage_ms["attention"] / stage_launches["attention"],
                "timed_as": "the attention launches of every layer back to back in one CUDA graph (the kernel "
                            "alone); `step_implied` divides the same FLOPs by the whole pipelined step, whose "
                            "other kernels overlap the attention on other streams",
                "step_implied": {"achieved": float(flops.sum()) / (ms_per_step / 1e3) / 1e12,
                                 "frac": float(flops.sum()) / (ms_per_step / 1e3) / 1e12 / peak_tf}}
    stages = {}
    for name, per_step_ms in stage_ms.items():
        entry = {"ms_per_step": per_step_ms, "launches_per_step": stage_launches[name],
                 "us_per_launch": 1e3 * per_step_ms / stage_launches[name]}
        if name in ("deviation", "fuse"):
            b = sum(stage_bytes(cfg, *sizes[li], args.deviation)[name] for li in range(cfg.layers))
            gbs = b / (per_step_ms / 1e3) / 1e9
            entry.update({"bytes_per_step": b, "achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]})
        stages[name] = entry
    launches_per_step = sum(stage_launches.values())

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": data_desc(cfg),
            "config": {"workload": workload_desc(cfg), "n_ctx": cfg.n_ctx, "n_tokens": cfg.n_tokens,
                       "layers": cfg.layers, "deviation": args.deviation, "filter": args.filter,
                       "l2": f"inputs larger than L2: {sum(sum(t.numel() * 2 for t in d.values()) for d in d_in) / 1e9:.2f} GB per step",
                       "cuda_graph": use_graph, "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "stages": stages,
            "stage_sum_ms_per_step": sum(stage_ms.values()),
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary()}

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, cfg, cb, plan, [h.pinned for h in host_inputs], bufs, sizes, dev, world)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, host_inputs[:3], args.deviation, args.filter)
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_sweep(args, cfg):
    """Sweep path: the single-layer blend at every recompute ratio r of the workload (r1 = r2 = r),
    each repetition timed alone with the L2 flushed before it (a 512 MB write), median over
    `steps` repetitions. Per r: the whole layer (cb_blend_layer) and each stage alone
    (cb_blend_stage). At r = 100% every context row is recomputed, so the blend must equal a full
    prefill's attention: the encoded cache, and the attention of every row over it by the same
    kernels outside the blend, are compared bit for bit."""
    import dataclasses

    import torch

    import rag_kv_cache_gb300 as cb
    from rag_kv_cache_gb300.build import build
    from workloads.generator import generate_layer

    rank, world, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)
    ratios = list(cfg.sweep_pct) or [cfg.r1_pct]
    inp = generate_layer(cfg, 1)
    d_in = {name: t.to(dev) for name, t in pinned_layer(inp).pinned.items()}
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    peaks = load_peaks()
    rows, check, launches = [], None, 0
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]

    def timed_median(fn_graph):
        ts = []
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                flush.fill_(1)
                a.record(stream)
                fn_graph.replay()
                b.record(stream)
        stream.synchronize()
        ts = [a.elapsed_time(b) for a, b in ev]
        return statistics.median(ts)

    with ClockSampler(gpu_index) as clocks:
        for r in ratios:
            rcfg = dataclasses.replace(cfg, r1_pct=r, r2_pct=r, layers=1)
            plan = cb.Plan.from_config(rcfg)
            bufs = cb.LayerBuffers(plan, dev)
            n_cand, k, mq, selects = plan.layer_sizes(1)

            def layer(plan=plan, bufs=bufs):
                cb.cb_blend_layer(plan, 1, cand=None, bufs=bufs, stream=stream, **d_in)

            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    layer()
            stream.synchronize()
            plan.check()
            graphs = {}
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer()
            graphs["layer"] = g
            for name in STAGES:
                if not stage_applies(name, (n_cand, k, mq, selects)):
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    cb.cb_blend_stage(plan, 1, name, cand=None, bufs=bufs, stream=stream, **d_in)
                graphs[name] = g
            ms = {name: timed_median(g) for name, g in graphs.items()}
            launches += args.steps * 2 * (len(graphs) - 1)  # the layer graph holds one launch per stage
            plan.check()
            flops = attention_flops(rcfg, bufs.sel_tok[:k].cpu().numpy())
            b = stage_bytes(rcfg, n_cand, k, mq, selects)
            row = {"r_pct": r, "k": k, "mq": mq, "ms_layer": ms["layer"],
                   "tokens_per_s": cfg.n_ctx / (ms["layer"] / 1e3),
                   "attention_flops": flops, "attention_us": 1e3 * ms["attention"],
                   "attention_tflops": flops / (ms["attention"] / 1e3) / 1e12,
                   "attention_frac": flops / (ms["attention"] / 1e3) / 1e12 / peaks["bf16_tflops"],
                   "fuse_us": 1e3 * ms["fuse"],
                   "fuse_frac_hbm": b["fuse"] / (ms["fuse"] / 1e3) / 1e9 / peaks["hbm_gbs"]}
            if "deviation" in ms:
                row.update({"deviation_us": 1e3 * ms["deviation"],
                            "deviation_frac_hbm": b["deviation"] / (ms["deviation"] / 1e3) / 1e9 / peaks["hbm_gbs"],
                            "topk_us": 1e3 * ms["topk"]})
            rows.append(row)
            if r == 100:
                # full prefill by the same kernels outside the blend: every key and query encoded at
                # its position, then causal attention of all rows over the recomputed cache
                n = cfg.n_tokens
                pos = torch.arange(n, dtype=torch.int32, device=dev)
                k_full = torch.empty_like(d_in["k_new"])
                q_all = torch.empty((n, cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device=dev)
                o_full = torch.empty_like(q_all)
                with torch.cuda.stream(stream):
                    layer()
                    cb.cb_rope_rerotate(plan, k_full, d_in["k_new"], pos, stream=stream)
                    cb.cb_rope_rerotate(plan, q_all, d_in["q"], pos, stream=stream)
                    cb.cb_hkvd_attention(plan, q_all, pos, n, k_full, d_in["v_new"], n, o_full, stream=stream)
                stream.synchronize()
                plan.check()
                same = lambda a, b_: bool(torch.equal(a.view(torch.int16), b_.view(torch.int16)))
                check = {"fused_k_equals_encoded_k_new": same(bufs.k_fused, k_full),
                         "fused_v_equals_v_new": same(bufs.v_fused, d_in["v_new"]),
                         "out_equals_full_prefill": same(bufs.out[:mq], o_full),
                         "max_abs_diff": float((bufs.out[:mq].float() - o_full.float()).abs().max())}
            plan.close()
    base = next((x for x in rows if x["r_pct"] == cfg.r1_pct), rows[0])
    line = {"metric": METRIC, "value": base["tokens_per_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": base["ms_layer"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": data_desc(cfg),
            "config": {"workload": workload_desc(cfg), "path": "sweep", "n_ctx": cfg.n_ctx,
                       "value_at_r_pct": base["r_pct"], "cuda_graph": True,
                       "l2": "flushed before every repetition (512 MB write, outside the timed region)",
                       "attention_peak": "measured bf16 burst (one launch timed alone)"},
            "sweep": rows, "r100_full_recompute_check": check,
            "gpu_launches": launches, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, cfg):
    """Decode path: per step, the newest token's attention over each layer's cache (n_tokens + 1 keys)."""
    import torch
    import torch.distributed as dist

    import rag_kv_cache_gb300 as cb
    from rag_kv_cache_gb300.build import build
    from workloads.generator import generate_decode
    from workloads.torch_io import bf16_tensor

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)
    ins = [generate_decode(cfg, layer) for layer in range(1, cfg.layers + 1)]
    n_keys = cfg.n_tokens + 1
    d_k = [bf16_tensor(x.k, dev) for x in ins]
    d_v = [bf16_tensor(x.v, dev) for x in ins]
    d_q = [bf16_tensor(x.q, dev) for x in ins]
    outs = [torch.empty((cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device=dev) for _ in ins]
    plan = cb.Plan.from_config(cfg)
    stream = torch.cuda.Stream(dev)

    def step():
        for li in range(cfg.layers):
            cb.cb_decode_attention(plan, d_q[li], d_k[li], d_v[li], n_keys, outs[li], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    plan.check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_index) as clocks:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                g.replay()
            stop.record(stream)
        stream.synchronize()
    ms = start.elapsed_time(stop)
    plan.check()
    ms = max_over_ranks(ms, dev, world)
    ms_step = ms / args.steps
    row_kv = cfg.hkv * cfg.head_dim * 2
    bytes_launch = 2.0 * n_keys * row_kv + 2.0 * cfg.hq * cfg.head_dim * 2
    us_launch = 1e3 * ms_step / cfg.layers
    gbs = bytes_launch / (us_launch * 1e-6) / 1e9
    peaks = load_peaks()
    line = {"metric": "decode steps/s (one new token, attention of every layer)", "value": world * 1e3 / ms_step,
            "unit": "steps/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) bf16 caches and queries",
            "config": {"workload": workload_desc(cfg), "path": "decode", "n_keys": n_keys,
                       "l2": f"inputs larger than L2: {cfg.layers * bytes_launch / 1e9:.2f} GB per step",
                       "cuda_graph": True},
            "roofline": {"kernel": "decode_tc", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": (traffic_for("decode_tc.cu", cfg.name) or {}).get("dram_bytes_per_launch"),
                         "peak_source": f"{peaks['source']} copy bandwidth", "bytes_per_launch": bytes_launch,
                         "launches_per_step": cfg.layers, "avg_launch_us": us_launch},
            "gpu_launches": cfg.layers * args.steps, "clocks": clocks.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_diagnostics(args, cfg):
    """Diagnostics path on one layer: for every recompute ratio of the workload's sweep (else r1),
    blend the layer and measure ||Attn(Q, K_fused, V_fused) - Attn(Q, K_new, V_new)|| over all
    query rows against a full prefill, and the full prefill's Sparsity(A, eps). Both attentions of
    the deviation run through cb_hkvd_attention (the same kernel for the same launch size), so the
    deviation holds only what the blend changes: zero at r = 100%. Times the diagnostics of one
    ratio: both encodes, the two attentions, the two passes of the sparsity count and the
    reductions."""
    import dataclasses

    import torch

    import rag_kv_cache_gb300 as cb
    from rag_kv_cache_gb300.build import build
    from workloads.generator import generate_layer
    from workloads.torch_io import layer_tensors

    rank, world, local = dist_env()
    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)
    ratios = list(cfg.sweep_pct) or [cfg.r1_pct]
    inp = generate_layer(cfg, 1)
    t = layer_tensors(inp, dev)
    n, hq, d = cfg.n_tokens, cfg.hq, cfg.head_dim
    pos = torch.arange(n, dtype=torch.int32, device=dev)
    k_full = torch.empty((n, cfg.hkv, d), dtype=torch.bfloat16, device=dev)
    q_all = torch.empty((n, hq, d), dtype=torch.bfloat16, device=dev)
    o_full, o_fused, o_count = torch.empty_like(q_all), torch.empty_like(q_all), torch.empty_like(q_all)
    stats = torch.empty((n, hq, 2), dtype=torch.float32, device=dev)
    counts = torch.empty((n, hq), dtype=torch.int32, device=dev)
    total = torch.empty(1, dtype=torch.int64, device=dev)
    sums = torch.empty(2, dtype=torch.float64, device=dev)
    stream = torch.cuda.Stream(dev)
    series, timed_plan = {}, None
    for r in ratios:
        plan = cb.Plan.from_config(dataclasses.replace(cfg, r1_pct=r, r2_pct=r))
        bufs = cb.LayerBuffers(plan, dev)

        def diag(plan=plan, bufs=bufs):
            cb.cb_rope_rerotate(plan, k_full, t["k_new"], pos, stream=stream)
            cb.cb_rope_rerotate(plan, q_all, t["q"], pos, stream=stream)
            cb.cb_hkvd_attention(plan, q_all, pos, n, bufs.k_fused, bufs.v_fused, n, o_fused, stream=stream)
            cb.cb_hkvd_attention(plan, q_all, pos, n, k_full, t["v_new"], n, o_full, stream=stream)
            cb.cb_attention_sparsity(plan, q_all, pos, n, k_full, t["v_new"], n, args.eps, o_count, stats, counts,
                                     total, stream=stream)
            cb.cb_output_deviation(plan, o_fused, o_full, n, sums, stream=stream)

        with torch.cuda.stream(stream):
            cb.cb_blend_layer(plan, 1, cand=None, bufs=bufs, stream=stream, **t)
            diag()
        stream.synchronize()
        plan.check()
        s2 = sums.cpu().numpy()
        series[str(r)] = {"dev": float(np.sqrt(s2[0])), "ref": float(np.sqrt(s2[1])),
                          "rel": float(np.sqrt(s2[0] / s2[1]))}
        sparsity = int(total.item()) / float(hq * n * n)
        if r == ratios[-1]:
            timed_plan = plan
            # time the diagnostics of this ratio, and the counting pass alone
            for _ in range(args.warmup):
                with torch.cuda.stream(stream):
                    diag()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                diag()
            gc = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gc, stream=stream):
                cb.cb_attention_sparsity(plan, q_all, pos, n, k_full, t["v_new"], n, args.eps, o_count, stats,
                                         counts, total, stream=stream)
            start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]
            with ClockSampler(gpu_index) as clocks:
                with torch.cuda.stream(stream):
                    start.record(stream)
                    for _ in range(args.steps):
                        g.replay()
                    stop.record(stream)
                stream.synchronize()
                ms = start.elapsed_time(stop) / args.steps
                with torch.cuda.stream(stream):
                    start.record(stream)
                    for _ in range(args.steps):
                        gc.replay()
                    stop.record(stream)
                stream.synchronize()
                ms_count = start.elapsed_time(stop) / args.steps
        else:
            plan.close()
    timed_plan.check()
    flops = 4.0 * hq * d * n * (n + 1) / 2.0  # one causal attention over all n rows
    peaks = load_peaks()
    achieved = 2 * flops / (ms_count * 1e-3) / 1e12  # the sparsity count runs the attention twice
    line = {"metric": "diagnostics time per layer (deviation over all rows + sparsity)", "value": ms,
            "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": data_desc(cfg),
            "config": {"workload": workload_desc(cfg), "path": "diagnostics", "n_tokens": n, "eps": args.eps,
                       "timed_ratio_pct": ratios[-1], "cuda_graph": True},
            "deviation_vs_r": series, "sparsity": sparsity,
            "roofline": {"kernel": "hkvd_attention (statistics and counting passes)", "bound": "tensor",
                         "achieved": achieved, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops_sustained"], "traffic": None,
                         "peak_source": f"{peaks['source']} bf16 sustained", "ms_sparsity_count": ms_count},
            "gpu_launches": 8 * args.steps, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)
    timed_plan.close()
    return 0


def run_projection(args, cfg):
    """Projection path: per step, the QKV projection (RoPE-encoded q and k) of every layer's
    recomputed rows, at the blend's row counts: layer 1 all tokens, layer l >= 2 the candidates
    C_l (= S_{l-1}) and the suffix. A layer's hidden rows are the outputs the previous layer's
    attention produced, which are exactly its query rows S_{l-1} and the suffix, in that list
    order; so row i of x is token tokens[i] and the rows are read in place
    (cb_qkv_projection_indexed with x_index = NULL). The same step with every layer's rows
    gathered from a full [n_tokens, d_model] matrix (cb_qkv_projection with a row list: the
    gather kernel plus the GEMM) is timed too and reported under "gathered_rows". Four distinct
    hidden-state / weight sets (random, of the model's shape) are cycled over the layers, so a
    layer's weights are not in L2 from the layer before."""
    import torch
    import torch.distributed as dist

    import rag_kv_cache_gb300 as cb
    from rag_kv_cache_gb300.build import build
    from workloads.generator import generate_projection
    from workloads.torch_io import bf16_tensor

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build()
    dev = torch.device("cuda", local)
    plan = cb.Plan.from_config(cfg)
    sets = [generate_projection(cfg, s + 1) for s in range(min(4, cfg.layers))]
    xs = [bf16_tensor(x, dev) for x, _ in sets]
    ws = [bf16_tensor(w, dev) for _, w in sets]
    rng = np.random.default_rng(cfg.config_id)
    tokens, sizes = [], []
    cand = np.arange(cfg.n_ctx)
    for layer in range(1, cfg.layers + 1):
        n_cand, k, mq, selects = plan.layer_sizes(layer)
        if layer == 1:
            r = np.arange(cfg.n_tokens)  # layer 1 recomputes every token
        else:
            if n_cand < cand.size:  # C_l = S_{l-1}: a subset of the previous candidates
                cand = np.sort(rng.choice(cand, n_cand, replace=False))
            r = np.concatenate([cand, np.arange(cfg.n_ctx, cfg.n_tokens)])
        tokens.append(torch.as_tensor(r.astype(np.int32), device=dev))
        sizes.append(r.size)
    d_model = cfg.d_model
    xg = torch.empty((cfg.n_tokens, d_model), dtype=torch.bfloat16, device=dev)
    q = torch.empty((cfg.n_tokens, cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device=dev)
    k = torch.empty((cfg.n_tokens, cfg.hkv, cfg.head_dim), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    stream = torch.cuda.Stream(dev)

    def step_in_place():
        for li in range(cfg.layers):
            s_ = li % len(sets)
            cb.cb_qkv_projection_indexed(plan, xs[s_][: sizes[li]], None, tokens[li], sizes[li], ws[s_], q, k, v,
                                         encode=True, stream=stream)

    def step_gathered():
        for li in range(cfg.layers):
            s_ = li % len(sets)
            cb.cb_qkv_projection(plan, xs[s_], tokens[li], sizes[li], ws[s_], q, k, v, encode=True, x_gathered=xg,
                                 stream=stream)

    def timed(step, clocked):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step()
        stream.synchronize()
        plan.check()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        stream.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(gpu_index) if clocked else contextlib.nullcontext() as clocks:
            with torch.cuda.stream(stream):
                start.record(stream)
                for _ in range(args.steps):
                    g.replay()
                stop.record(stream)
            stream.synchronize()
        ms = start.elapsed_time(stop) / args.steps
        plan.check()
        return max_over_ranks(ms, dev, world), clocks

    ms, clocks = timed(step_in_place, True)
    ms_gathered, _ = timed(step_gathered, False)
    n_out = (cfg.hq + 2 * cfg.hkv) * cfg.head_dim
    flops = sum(2.0 * m_ * d_model * n_out for m_ in sizes)
    peaks = load_peaks()
    peak = peaks["bf16_tflops_sustained"]
    tf = flops / (ms * 1e-3) / 1e12
    tf_g = flops / (ms_gathered * 1e-3) / 1e12
    line = {"metric": "QKV projection TFLOP/s (recomputed rows of every layer)", "value": world * tf,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) hidden rows, N(0, 1/d_model) weights of the model's shape",
            "config": {"workload": workload_desc(cfg), "path": "projection", "d_model": d_model, "n_out": n_out,
                       "rows_per_layer": sorted(set(sizes)), "cuda_graph": True,
                       "rows": "in place: row i of a layer's x is token tokens[i] (the previous layer's "
                               "attention rows, in list order); layer 1 all tokens",
                       "l2": "four weight sets cycled (4 x %.0f MB)" % (n_out * d_model * 2 / 1e6)},
            "roofline": {"kernel": "qkv_projection_pair", "bound": "tensor", "achieved": tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": tf / peak,
                         "traffic": (traffic_for("qkv.cu", cfg.name) or {}).get("dram_bytes_per_launch"),
                         "peak_source": f"{peaks['source']} bf16 sustained", "flops_per_step": flops},
            "gathered_rows": {"ms_per_step": ms_gathered, "achieved": tf_g, "frac": tf_g / peak,
                              "how": "every layer's rows gathered from a full [n_tokens, d_model] matrix first "
                                     "(row gather kernel + GEMM per layer)"},
            "gpu_launches": cfg.layers * args.steps, "clocks": clocks.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(args, cfg, cb, plan, h_in, bufs, sizes, dev, world):
    """Metric through the C ABI with host buffers: H2D of every layer's inputs (h_in: pinned
    tensors per layer) and D2H of its outputs (attention rows and S_l) timed. The fused K/V
    stay on the device, where the layer's consumers (the next layers' decode) read them."""
    import torch
    import torch.distributed as dist

    d_in = [{k: torch.empty_like(v, device=dev) for k, v in h.items()} for h in h_in]
    h_out = [torch.empty((s[2], cfg.hq, cfg.head_dim), dtype=torch.bfloat16, pin_memory=True) for s in sizes]
    h_sel = [torch.empty((max(s[1], 1),), dtype=torch.int32, pin_memory=True) for s in sizes]
    comp = torch.cuda.Stream(dev)
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    layer_done = [torch.cuda.Event() for _ in range(cfg.layers)]
    copied = [torch.cuda.Event() for _ in range(cfg.layers)]
    drained = [torch.cuda.Event() for _ in range(cfg.layers)]
    for e in layer_done + drained:
        e.record(comp)
    h2d_bytes = sum(sum(t.numel() * 2 for t in h.values()) for h in h_in)
    d2h_bytes = sum(o.numel() * 2 + (s[1] * 4) for o, s in zip(h_out, sizes))

    def step():
        for li in range(cfg.layers):
            with torch.cuda.stream(h2d):
                h2d.wait_event(layer_done[li])  # the previous step's layer li has consumed these buffers
                for k, t in h_in[li].items():
                    d_in[li][k].copy_(t, non_blocking=True)
                copied[li].record(h2d)
        for li in range(cfg.layers):
            comp.wait_event(copied[li])
            comp.wait_event(drained[li])
            c = plan.candidate_layer(li + 1)
            cb.cb_blend_layer(plan, li + 1, cand=None if c == 0 else bufs[c - 1].sel_tok, bufs=bufs[li],
                              stream=comp, **d_in[li])
            layer_done[li].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(layer_done[li])
                h_out[li].copy_(bufs[li].out[: sizes[li][2]], non_blocking=True)
                if sizes[li][1] > 0:
                    h_sel[li][: sizes[li][1]].copy_(bufs[li].sel_tok[: sizes[li][1]], non_blocking=True)
                drained[li].record(d2h)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(comp)
    for _ in range(args.e2e_steps):
        step()
    comp.wait_stream(d2h)
    comp.wait_stream(h2d)
    stop.record(comp)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(start.elapsed_time(stop), dev, world)
    if world > 1:
        dist.barrier()
    plan.check()
    return {"value": cfg.n_ctx * cfg.layers * args.e2e_steps * world / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
            "ms_per_step": ms / args.e2e_steps, "steps": args.e2e_steps,
            "copies": "every layer's five input tensors host to device; its attention output rows and "
                      "S_l device to host; the fused K/V stay on the device for the layer's consumers"}


def main():
    args = parse_args()
    if args.warmup < 3:
        print("bench: --warmup below 3 raised to 3", file=sys.stderr)
        args.warmup = 3
    from workloads import get_config

    if args.workload is None:
        args.workload = DEFAULT_WORKLOAD[args.path]
    cfg = get_config(args.workload)
    if args.layers is not None:
        import dataclasses

        cfg = dataclasses.replace(cfg, layers=max(1, min(cfg.layers, args.layers)))
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.path == "sweep":
        return run_sweep(args, cfg)
    if args.path == "decode":
        return run_decode(args, cfg)
    if args.path == "diagnostics":
        return run_diagnostics(args, cfg)
    if args.path == "projection":
        return run_projection(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())

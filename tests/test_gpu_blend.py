"""Whole-layer parity: cb_blend_layer against the oracle's blend, on the five workloads.

HKVD sets, candidate rows, deviations and fused V are compared bit for bit;
fused K, encoded queries and attention outputs within 2e-2 abs + 1e-2 rel.
At full size the attention is checked on seeded samples of query rows (the
oracle computes those rows one by one); everything else is checked whole.
"""

import dataclasses

import numpy as np
import pytest
import torch

from conftest import assert_close_attention, assert_close_bf16, record_strict_attention
from oracle.blend import blend_layer, candidate_layer, gradual_filter_schedule
from oracle.deviation import bf16_bits_to_f64
from workloads import get_config
from workloads.generator import generate_layer, hkvd_noise_sets
from workloads.torch_io import bf16_bits, layer_tensors

pytestmark = pytest.mark.gpu


def run_gpu_layers(cb, cfg, layers, style="half", r1=None, r2=None, deviation="v", filter="keep"):
    """Run layers 1..max(layers) on the GPU; return {layer: outputs} for the requested ones."""
    plan = cb.Plan.from_config(cfg, rope_style=style, r1_pct=r1, r2_pct=r2, deviation=deviation, filter=filter)
    sets = hkvd_noise_sets(cfg)
    bufs = [cb.LayerBuffers(plan), cb.LayerBuffers(plan)]  # ping-pong
    sels = {0: None}  # kept copies of each layer's S_l: C_l is one of them
    results = {}
    for layer in range(1, max(layers) + 1):
        inp = generate_layer(cfg, layer, sets)
        t = layer_tensors(inp)
        b = bufs[layer % 2]
        cand = sels[plan.candidate_layer(layer)]
        cb.cb_blend_layer(plan, layer, cand=cand, bufs=b, **t)
        n_cand, k, mq, selects = plan.layer_sizes(layer)
        plan.check()
        if layer in layers:
            results[layer] = dict(
                inp=inp, k=k, mq=mq, selects=selects,
                dev=b.dev[:n_cand].cpu().numpy().copy() if selects else None,
                sel_tok=b.sel_tok[:k].cpu().numpy().copy(), sel_row=b.sel_row[:k].cpu().numpy().copy(),
                k_fused=bf16_bits(b.k_fused), v_fused=bf16_bits(b.v_fused),
                q_rot=bf16_bits(b.q_rot[:mq]), out=bf16_bits(b.out[:mq]))
        sels[layer] = b.sel_tok[:k].clone()
    plan.close()
    return results


def oracle_layers(cfg, layers, style="half", attention_rows=None, deviation="v", filter="keep", full_rows=()):
    """The oracle's blend for the requested layers (selection chain followed from layer 1).

    Layers that are not requested only carry the chain forward: a layer that keeps its
    candidates passes them on unchanged, one that selects runs only its deviation and top-k.
    attention_rows(mq, layer) picks the query rows whose attention the oracle computes; layers
    in full_rows compute every row."""
    from oracle.deviation import deviation_canonical_f32, kv_deviation_canonical_f32
    from oracle.positions import chunk_local_positions
    from oracle.topk import hkvd_topk

    sets = hkvd_noise_sets(cfg)
    sched = gradual_filter_schedule(cfg.n_ctx, cfg.layers, cfg.r1_pct, cfg.r2_pct, filter)
    p_old = chunk_local_positions(cfg.n_chunks, cfg.chunk_len)
    sels = {0: np.arange(cfg.n_ctx)}
    out = {}
    for layer, k, selects in sched[: max(layers)]:
        cand = sels[candidate_layer(layer, filter)]
        if layer in layers:
            inp = generate_layer(cfg, layer, sets)
            rows = None if (layer in full_rows or attention_rows is None) else attention_rows(k + cfg.n_suffix, layer)
            res = blend_layer(cfg, inp, layer, cand, k, selects, style, attention_rows=rows, deviation=deviation)
            out[layer] = res
            sels[layer] = res.sel_tok
        elif selects:
            inp = generate_layer(cfg, layer, sets)
            if deviation == "kv":
                dev = kv_deviation_canonical_f32(inp.k_new[cand], inp.k_old[cand], inp.v_new[cand], inp.v_old[cand],
                                                 p_old[cand], cfg.rope_theta, style)
            else:
                dev = deviation_canonical_f32(inp.v_new[cand], inp.v_old[cand])
            sels[layer], _ = hkvd_topk(dev, cand, k)
        else:
            sels[layer] = cand
    return out


def run_gpu_request(cb, cfg, layers, deviation="v", filter="keep"):
    """All layers of the request in one cb_blend_request call; {layer: outputs} for the requested
    layers. Inputs are generated on the host cores in parallel and moved to the device at once."""
    import bench

    plan = cb.Plan.from_config(cfg, deviation=deviation, filter=filter)
    sets = hkvd_noise_sets(cfg)
    keep = {}

    def to_device(inp):
        if inp.layer in layers:
            keep[inp.layer] = inp
        return layer_tensors(inp)

    d_in = bench.generate_inputs(cfg, list(range(1, cfg.layers + 1)), sets, consume=to_device)
    bufs = [cb.LayerBuffers(plan) for _ in range(cfg.layers)]
    cb.cb_blend_request(plan, [dict(bufs=bufs[i], **d_in[i]) for i in range(cfg.layers)])
    torch.cuda.synchronize()
    plan.check()
    results = {}
    for layer in layers:
        b = bufs[layer - 1]
        n_cand, k, mq, selects = plan.layer_sizes(layer)
        results[layer] = dict(
            inp=keep[layer], k=k, mq=mq, selects=selects,
            dev=b.dev[:n_cand].cpu().numpy().copy() if selects else None,
            sel_tok=b.sel_tok[:k].cpu().numpy().copy(), sel_row=b.sel_row[:k].cpu().numpy().copy(),
            k_fused=bf16_bits(b.k_fused), v_fused=bf16_bits(b.v_fused),
            q_rot=bf16_bits(b.q_rot[:mq]), out=bf16_bits(b.out[:mq]))
    plan.close()
    del d_in, bufs
    torch.cuda.empty_cache()
    return results


def compare(g, o, cfg, rows=None, what=""):
    assert np.array_equal(g["sel_tok"], o.sel_tok)
    assert np.array_equal(g["sel_row"], o.sel_row)
    if o.dev is not None:
        assert np.array_equal(g["dev"].view(np.uint32), o.dev.view(np.uint32))
    assert np.array_equal(bf16_bits_to_f64(g["v_fused"]), o.v_fused)
    assert_close_bf16(bf16_bits_to_f64(g["k_fused"]), o.k_fused, what="fused K")
    assert_close_bf16(bf16_bits_to_f64(g["q_rot"]), o.q_rot, what="encoded Q")
    got = bf16_bits_to_f64(g["out"])
    if rows is None:
        rows = np.arange(got.shape[0])
    record_strict_attention(what or cfg.name, got[rows], o.out[rows])
    assert_close_attention(got[rows], o.out[rows], o.out_vscale[rows], what=f"attention ({rows.size} rows)")


def sampled_rows(cfg, seed, n=256):
    """n seeded query rows plus the first and last HKVD rows and the first and last suffix rows."""
    rng = np.random.default_rng(seed)

    def pick(mq, layer):
        k = mq - cfg.n_suffix
        fixed = [0, mq - 1] + ([k - 1] if k > 0 else []) + ([k] if cfg.n_suffix > 0 else [])
        return np.unique(np.concatenate([np.asarray(fixed), rng.choice(mq, size=min(mq, n), replace=False)]))
    return pick


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_tiny_layer_exact(cb, style):
    cfg = get_config("tiny")
    g = run_gpu_layers(cb, cfg, [1], style)[1]
    o = oracle_layers(cfg, [1], style)[1]
    compare(g, o, cfg)
    # the noise model's high-deviation set is what the selection finds
    assert set(g["sel_tok"].tolist()) == set(g["inp"].hkvd_set.tolist())


def test_small_multilayer_gradual_filter(cb):
    cfg = dataclasses.replace(get_config("mistral7b"), name="small5", config_id=91, n_chunks=5, chunk_len=96,
                              n_suffix=24, layers=5)
    g = run_gpu_layers(cb, cfg, [1, 2, 3, 4, 5])
    o = oracle_layers(cfg, [1, 2, 3, 4, 5])
    for layer in range(1, 6):
        compare(g[layer], o[layer], cfg, what=f"small5 layer {layer}")
    assert np.array_equal(g[4]["sel_tok"], g[2]["sel_tok"])


@pytest.mark.parametrize("deviation,filter,style", [("kv", "keep", "half"), ("kv", "keep", "interleaved"),
                                                   ("v", "reselect", "half"), ("kv", "reselect", "interleaved")])
def test_small_multilayer_variants(cb, deviation, filter, style):
    # the K+V deviation and the per-layer re-selection reading of the gradual filter
    cfg = dataclasses.replace(get_config("mistral7b"), name="small5", config_id=91, n_chunks=5, chunk_len=96,
                              n_suffix=24, layers=5)
    g = run_gpu_layers(cb, cfg, [1, 2, 3, 4, 5], style, deviation=deviation, filter=filter)
    o = oracle_layers(cfg, [1, 2, 3, 4, 5], style, deviation=deviation, filter=filter)
    for layer in range(1, 6):
        assert o[layer].dev is not None or filter == "keep"
        compare(g[layer], o[layer], cfg)


@pytest.mark.parametrize("r", [5, 10, 15, 30, 50, 100])
def test_ratio_sweep(cb, r):
    cfg = get_config("sweep").with_ratio(r)
    rng = np.random.default_rng(r)
    pick = lambda mq, layer: np.sort(rng.choice(mq, size=min(mq, 192), replace=False))
    g = run_gpu_layers(cb, cfg, [1])[1]
    o = oracle_layers(cfg, [1], attention_rows=pick)[1]
    compare(g, o, cfg, rows=np.flatnonzero(~np.isnan(o.out[:, 0, 0])), what=f"sweep r={r}%")
    if r == 100:
        assert g["sel_tok"].tolist() == list(range(cfg.n_ctx))


@pytest.mark.parametrize("name,layers,full_rows", [("mistral7b", [1, 2, 3, 32], [3]), ("llama70b", [1, 2, 3, 80], []),
                                                ("long32k", [1, 2, 3, 32], [])])
def test_full_size_requests(cb, name, layers, full_rows):
    # every layer of the request through cb_blend_request (the selection chain on the device);
    # the oracle checks the first three layers and the last: sets, rows, deviations and fused V
    # bit for bit, K, queries and >= 256 seeded attention rows (plus the first and last HKVD and
    # suffix rows) within tolerance; the layers in full_rows check every attention row
    cfg = get_config(name)
    g = run_gpu_request(cb, cfg, layers)
    o = oracle_layers(cfg, layers, attention_rows=sampled_rows(cfg, cfg.config_id), full_rows=full_rows)
    for layer in layers:
        compare(g[layer], o[layer], cfg, rows=np.flatnonzero(~np.isnan(o[layer].out[:, 0, 0])),
                what=f"{name} layer {layer}")
    assert np.array_equal(g[layers[-1]]["sel_tok"], g[2]["sel_tok"])  # kept from layer 3 on


def test_full_size_kv_reselect(cb):
    # Mistral-7B-shaped, layers 1-4 with the K+V deviation and re-selection at every layer
    cfg = get_config("mistral7b")
    rng = np.random.default_rng(77)
    pick = lambda mq, layer: np.unique(np.concatenate([[0, mq - 1], rng.choice(mq, size=48, replace=False)]))
    g = run_gpu_layers(cb, cfg, [1, 2, 3, 4], deviation="kv", filter="reselect")
    o = oracle_layers(cfg, [1, 2, 3, 4], attention_rows=pick, deviation="kv", filter="reselect")
    for layer in (1, 2, 3, 4):
        compare(g[layer], o[layer], cfg, rows=np.flatnonzero(~np.isnan(o[layer].out[:, 0, 0])))


@pytest.mark.parametrize("name,layers,deviation,filter", [("mistral7b", 4, "v", "keep"), ("tiny", 1, "v", "keep"),
                                                          ("mistral7b", 4, "kv", "reselect"),
                                                          ("mistral7b", 20, "v", "reselect"),  # two selection batches
                                                          ("mistral7b", 18, "kv", "reselect")])
def test_request_scheduling_matches_layer_by_layer(cb, name, layers, deviation, filter):
    # cb_blend_request overlaps layers on several streams; its outputs must be the same bytes
    # as calling cb_blend_layer layer after layer.
    cfg = get_config(name)
    plan = cb.Plan.from_config(cfg, deviation=deviation, filter=filter)
    sets = hkvd_noise_sets(cfg)
    ins = [layer_tensors(generate_layer(cfg, layer, sets)) for layer in range(1, layers + 1)]
    seq = [cb.LayerBuffers(plan) for _ in range(layers)]
    req = [cb.LayerBuffers(plan) for _ in range(layers)]
    for li in range(layers):
        c = plan.candidate_layer(li + 1)
        cb.cb_blend_layer(plan, li + 1, cand=None if c == 0 else seq[c - 1].sel_tok, bufs=seq[li], **ins[li])
    for _ in range(2):  # twice: the second call reuses the plan's streams and events
        cb.cb_blend_request(plan, [dict(bufs=req[li], **ins[li]) for li in range(layers)])
    torch.cuda.synchronize()
    plan.check()
    for li in range(layers):
        _, k, mq, _ = plan.layer_sizes(li + 1)
        a, b = seq[li], req[li]
        assert torch.equal(a.sel_tok[:k], b.sel_tok[:k]) and torch.equal(a.sel_row[:k], b.sel_row[:k])
        for f in ("k_fused", "v_fused"):
            assert torch.equal(getattr(a, f).view(torch.int16), getattr(b, f).view(torch.int16))
        for f in ("q_rot", "out"):
            assert torch.equal(getattr(a, f)[:mq].view(torch.int16), getattr(b, f)[:mq].view(torch.int16))
    plan.close()


def test_stages_one_by_one_match_the_layer_call(cb):
    # cb_blend_stage runs each stage alone; in order they must give cb_blend_layer's bytes.
    cfg = get_config("mistral7b")
    plan = cb.Plan.from_config(cfg)
    sets = hkvd_noise_sets(cfg)
    ins = [layer_tensors(generate_layer(cfg, layer, sets)) for layer in (1, 2, 3)]
    whole = [cb.LayerBuffers(plan) for _ in range(3)]
    staged = [cb.LayerBuffers(plan) for _ in range(3)]
    for li in range(3):
        cb.cb_blend_layer(plan, li + 1, cand=None if li == 0 else whole[li - 1].sel_tok, bufs=whole[li], **ins[li])
        for stage in ("deviation", "topk", "fuse", "attention"):
            cb.cb_blend_stage(plan, li + 1, stage, cand=None if li == 0 else staged[li - 1].sel_tok,
                              bufs=staged[li], **ins[li])
    torch.cuda.synchronize()
    plan.check()
    for li in range(3):
        _, k, mq, _ = plan.layer_sizes(li + 1)
        a, b = whole[li], staged[li]
        assert torch.equal(a.sel_tok[:k], b.sel_tok[:k]) and torch.equal(a.sel_row[:k], b.sel_row[:k])
        for f in ("k_fused", "v_fused"):
            assert torch.equal(getattr(a, f).view(torch.int16), getattr(b, f).view(torch.int16))
        for f in ("q_rot", "out"):
            assert torch.equal(getattr(a, f)[:mq].view(torch.int16), getattr(b, f)[:mq].view(torch.int16))
    with pytest.raises(cb.CacheBlendError):
        cb.cb_blend_stage(plan, 1, "fuse", cand=None, bufs=staged[0], **dict(ins[0], q=None))
    plan.close()


@pytest.mark.parametrize("case", ["no_hkvd", "no_suffix", "ragged", "single_chunk"])
def test_degenerate_requests(cb, case):
    # r = 0 (only the suffix attends), no suffix (only the HKVD rows attend), chunk lengths and
    # suffixes that fill no tile, and a single chunk (nothing is re-rotated)
    base = get_config("mistral7b")
    kw = dict(no_hkvd=dict(n_chunks=3, chunk_len=100, n_suffix=20, r1_pct=0, r2_pct=0),
              no_suffix=dict(n_chunks=3, chunk_len=100, n_suffix=0),
              ragged=dict(n_chunks=3, chunk_len=77, n_suffix=5, hq=8, hkv=2, head_dim=64),
              single_chunk=dict(n_chunks=1, chunk_len=300, n_suffix=12))[case]
    cfg = dataclasses.replace(base, name=case, config_id=95, layers=3, **kw)
    g = run_gpu_layers(cb, cfg, [1, 2, 3])
    o = oracle_layers(cfg, [1, 2, 3])
    for layer in (1, 2, 3):
        compare(g[layer], o[layer], cfg)
        if case == "no_hkvd":
            assert g[layer]["k"] == 0 and g[layer]["mq"] == cfg.n_suffix
        if case == "no_suffix":
            assert g[layer]["mq"] == g[layer]["k"]

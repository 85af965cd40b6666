"""Pins of the oracle's whole layer: the fused cache definition, the r = 100% identity
and the gradual filter's structure, on the seeded workloads."""

import dataclasses
import os

import numpy as np
import pytest
import torch

from oracle.blend import blend_layer, blend_request, candidate_layer, gradual_filter_schedule
from oracle.deviation import bf16_bits_to_f64
from oracle.rope import rerotate, rope_rotate, round_bf16
from oracle.topk import k_for_ratio
from workloads import get_config
from workloads.generator import generate_layer


def _small_multilayer():
    # Mistral-like structure at a size the oracle runs in seconds: 4 chunks x 64 + 16,
    # 8 q / 2 kv heads, 4 layers, r1 = 30% -> r2 = 15%.
    base = get_config("mistral7b")
    return dataclasses.replace(base, name="small4", config_id=90, n_chunks=4, chunk_len=64,
                               n_suffix=16, hq=8, hkv=2, head_dim=64, layers=4)


def test_fused_cache_is_new_on_selection_and_old_elsewhere():
    cfg = get_config("tiny")
    inp = generate_layer(cfg, 1)
    k = k_for_ratio(cfg.r1_pct, cfg.n_ctx)
    res = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), k, True, attention_rows=False)
    n_ctx, n = cfg.n_ctx, cfg.n_tokens
    assert res.sel_tok.size == k and np.all(np.diff(res.sel_tok) > 0)
    p_new = np.arange(n)
    p_old = np.arange(n_ctx) % cfg.chunk_len
    old_rot = round_bf16(rerotate(bf16_bits_to_f64(inp.k_old), p_old, p_new[:n_ctx], cfg.rope_theta))
    new_enc = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new), p_new, cfg.rope_theta))
    is_new = np.zeros(n, bool)
    is_new[res.sel_tok] = True
    is_new[n_ctx:] = True
    assert np.array_equal(res.is_new, is_new)
    for t in range(n):
        if is_new[t]:
            assert np.array_equal(res.k_fused[t], new_enc[t])
            assert np.array_equal(res.v_fused[t], bf16_bits_to_f64(inp.v_new[t]))
        else:
            assert np.array_equal(res.k_fused[t], old_rot[t])
            assert np.array_equal(res.v_fused[t], bf16_bits_to_f64(inp.v_old[t]))
    # chunk 0 keys are not moved (delta 0): bitwise the cached bytes
    first = ~is_new[: cfg.chunk_len]
    assert np.array_equal(res.k_fused[: cfg.chunk_len][first], bf16_bits_to_f64(inp.k_old[: cfg.chunk_len])[first])


def test_full_ratio_equals_full_recompute_attention():
    # "数学推导" §形式化: with S = every token, Attention(Q, K_fused, V_fused) is
    # Attention(Q, K_new, V_new). Checked against torch's causal attention.
    cfg = get_config("tiny").with_ratio(100)
    inp = generate_layer(cfg, 1)
    res = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), cfg.n_ctx, True)
    n = cfg.n_tokens
    assert res.q_tok.tolist() == list(range(n))
    pos = np.arange(n)
    q = round_bf16(rope_rotate(bf16_bits_to_f64(inp.q), pos, cfg.rope_theta))
    k = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new), pos, cfg.rope_theta))
    v = bf16_bits_to_f64(inp.v_new)
    g = cfg.hq // cfg.hkv
    t = lambda x, rep: torch.from_numpy(np.repeat(x, rep, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q, 1), t(k, g), t(v, g), is_causal=True)
    np.testing.assert_allclose(res.out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_selection_finds_the_high_deviation_tokens():
    # With sigma 1.0 on 15% of tokens and 0.01 elsewhere, the r = 15% selection is
    # exactly the noisy set (the deviation gap is ~10^4).
    cfg = get_config("tiny")
    inp = generate_layer(cfg, 1)
    res = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), k_for_ratio(15, cfg.n_ctx), True, attention_rows=False)
    assert set(res.sel_tok.tolist()) == set(inp.hkvd_set.tolist())


def test_gradual_filter_structure_over_layers():
    cfg = _small_multilayer()
    from workloads.generator import hkvd_noise_sets
    sets = hkvd_noise_sets(cfg)
    inputs = (generate_layer(cfg, layer, sets) for layer in range(1, cfg.layers + 1))
    sched = gradual_filter_schedule(cfg.n_ctx, cfg.layers, cfg.r1_pct, cfg.r2_pct)
    prev = None
    results = list(blend_request(cfg, inputs, attention_rows=False))
    for (layer, k, selects), res in zip(sched, results):
        assert res.sel_tok.size == k
        assert set(res.sel_tok.tolist()) <= set(res.cand.tolist())
        assert np.array_equal(res.cand[res.sel_row], res.sel_tok)
        if prev is not None:
            assert np.array_equal(res.cand, prev.sel_tok)
        if not selects:
            assert res.dev is None and np.array_equal(res.sel_tok, prev.sel_tok)
        prev = res
    assert results[0].cand.size == cfg.n_ctx


def test_workload_generator_is_deterministic_and_shaped():
    cfg = get_config("tiny")
    a, b = generate_layer(cfg, 1), generate_layer(cfg, 1)
    for f in ("k_old", "v_old", "k_new", "v_new", "q"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert a.k_old.shape == (512, 2, 64) and a.k_new.shape == (544, 2, 64) and a.q.shape == (544, 4, 64)
    assert a.hkvd_set.size == 76


def test_reselect_schedule_and_candidate_layers():
    s = gradual_filter_schedule(3072, 32, 30, 15, filter="reselect")
    assert s[0] == (1, 921, True) and all(x == (i + 2, 460, True) for i, x in enumerate(s[1:]))
    assert [candidate_layer(l, "reselect") for l in (1, 2, 3, 9)] == [0, 1, 1, 1]
    assert [candidate_layer(l, "keep") for l in (1, 2, 3, 9)] == [0, 1, 2, 8]


def test_reselect_follows_each_layers_high_deviation_set():
    # With filter="reselect" every layer >= 2 re-ranks the layer-1 pool by its own deviation,
    # so it keeps the tokens of that layer's high-noise set that lie in the pool (the noise
    # model: sigma 1.0 on the set, 0.01 elsewhere, 10% of the set swapped per layer).
    cfg = dataclasses.replace(_small_multilayer(), name="small4r", config_id=92, layers=5)
    from workloads.generator import hkvd_noise_sets
    sets = hkvd_noise_sets(cfg)
    inputs = [generate_layer(cfg, layer, sets) for layer in range(1, cfg.layers + 1)]
    res = list(blend_request(cfg, iter(inputs), attention_rows=False, filter="reselect"))
    pool = set(res[0].sel_tok.tolist())
    k2 = k_for_ratio(cfg.r2_pct, cfg.n_ctx)
    moved = False
    for layer in range(2, cfg.layers + 1):
        r = res[layer - 1]
        assert np.array_equal(r.cand, res[0].sel_tok) and r.dev is not None and r.sel_tok.size == k2
        want = pool & set(sets[layer - 1].tolist())
        assert len(want) <= k2 and want <= set(r.sel_tok.tolist())
        moved |= not np.array_equal(r.sel_tok, res[1].sel_tok)
    assert moved  # the keep reading would have frozen S_2


def test_kv_deviation_mode_ranks_by_the_kv_number():
    cfg = _small_multilayer()
    inp = generate_layer(cfg, 1)
    from oracle.deviation import kv_deviation_canonical_f32
    from oracle.positions import chunk_local_positions
    cand = np.arange(cfg.n_ctx)
    k = k_for_ratio(cfg.r1_pct, cfg.n_ctx)
    res = blend_layer(cfg, inp, 1, cand, k, True, attention_rows=False, deviation="kv")
    dev = kv_deviation_canonical_f32(inp.k_new[:cfg.n_ctx], inp.k_old, inp.v_new[:cfg.n_ctx], inp.v_old,
                                     chunk_local_positions(cfg.n_chunks, cfg.chunk_len), cfg.rope_theta)
    np.testing.assert_array_equal(res.dev.view(np.uint32), dev.view(np.uint32))
    kth = np.sort(dev)[::-1][k - 1]
    assert np.all(dev[res.sel_tok] >= kth) and np.sum(dev > kth) <= k


@pytest.mark.parametrize("fixture,filter", [("gradual_filter.txt", "keep"), ("gradual_filter_reselect.txt", "reselect")])
def test_gradual_filter_golden_example(fixture, filter):
    # tests/golden/gradual_filter*.txt: three layers worked by hand from the page's description,
    # in the default reading and in the re-selection reading
    from oracle.topk import hkvd_topk

    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", fixture)
    lines = [ln for ln in open(path, encoding="utf-8").read().splitlines() if ln and not ln.startswith("#")]
    n_ctx = int(lines[0].split("|")[1])
    r1, r2 = (int(x) for x in lines[1].split("|")[1].split())
    layers = []
    for ln in lines[2:]:
        f = [x.strip() for x in ln.split("|")]
        layers.append((int(f[0]), np.array(f[1].split(), dtype=np.int64),
                       None if f[2] == "-" else np.array(f[2].split(), dtype=np.float64),
                       np.array(f[3].split(), dtype=np.int64)))
    schedule = gradual_filter_schedule(n_ctx, len(layers), r1, r2, filter)
    selections = {0: np.arange(n_ctx)}
    for (layer, cand_want, dev, sel_want), (l2, k, selects) in zip(layers, schedule):
        assert layer == l2
        cand = selections[candidate_layer(layer, filter)]
        assert np.array_equal(cand, cand_want)
        if selects:
            sel, rows = hkvd_topk(dev, cand, k)
            assert np.array_equal(cand[rows], sel)
        else:
            assert dev is None and k == cand.size
            sel = cand
        assert np.array_equal(sel, sel_want)
        selections[layer] = sel

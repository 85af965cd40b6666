"""Gathered QKV projection (the step before the blend, "rag的kvcache问题" §阶段一) against the oracle.

Written rows within 2e-2 abs + 1e-2 rel of the oracle's fp64 product rounded to bf16 (fp32
accumulation, bf16 output); rows outside the list are left as they were, bit for bit.
"""

import dataclasses

import numpy as np
import pytest
import torch

from conftest import assert_close_bf16
from oracle.deviation import bf16_bits_to_f64
from oracle.projection import qkv_projection
from workloads import get_config
from workloads.generator import generate_projection
from workloads.torch_io import bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _run(cb, cfg, rows, m, encode, style="half", d_model=None):
    plan = cb.Plan.from_config(cfg, rope_style=style)
    x, w = generate_projection(cfg, 1, d_model)
    n = cfg.n_tokens
    sentinel = lambda h: torch.full((n, h, cfg.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    q, k, v = sentinel(cfg.hq), sentinel(cfg.hkv), sentinel(cfg.hkv)
    xg = torch.empty((max(m, 1), x.shape[1]), dtype=torch.bfloat16, device="cuda") if rows is not None else None
    cb.cb_qkv_projection(plan, bf16_tensor(x), None if rows is None else _i32(rows), m, bf16_tensor(w), q, k, v,
                         encode=encode, x_gathered=xg)
    plan.check()
    plan.close()
    tok = np.arange(m) if rows is None else np.asarray(rows)
    oq, ok, ov = qkv_projection(bf16_bits_to_f64(x), tok, bf16_bits_to_f64(w), cfg.hq, cfg.hkv, cfg.head_dim,
                                cfg.rope_theta, encode, style)
    got = [bf16_bits_to_f64(bf16_bits(t)) for t in (q, k, v)]
    for g, o, what in zip(got, (oq, ok, ov), "qkv"):
        assert_close_bf16(g[tok], o, what=what)
        untouched = np.setdiff1d(np.arange(n), tok)
        assert np.all(g[untouched] == 7.0)
    return got


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("encode", [True, False])
def test_tiny_gathered_rows(cb, style, encode):
    cfg = get_config("tiny")
    rng = np.random.default_rng(5)
    rows = np.concatenate([np.sort(rng.choice(cfg.n_ctx, 81, replace=False)), np.arange(cfg.n_ctx, cfg.n_tokens)])
    _run(cb, cfg, rows, rows.size, encode, style)


@pytest.mark.parametrize("m", [1, 127, 129, 300])
def test_row_counts_and_in_place_rows(cb, m):
    cfg = dataclasses.replace(get_config("tiny"), hq=8, hkv=1, head_dim=128, n_chunks=1, chunk_len=292, n_suffix=8)
    _run(cb, cfg, None, m, True, d_model=64)  # one K slice; 1280 outputs = 5 tiles


def test_partial_last_tile_of_w(cb):
    cfg = dataclasses.replace(get_config("tiny"), hq=4, hkv=1, head_dim=64)  # 384 outputs: 1.5 tiles
    rows = np.arange(0, cfg.n_tokens, 3)
    _run(cb, cfg, rows, rows.size, True)


@pytest.mark.parametrize("name,m", [("mistral7b", 985), ("llama70b", 300)])
def test_model_shapes(cb, name, m):
    cfg = get_config(name)
    rng = np.random.default_rng(m)
    n_suf = cfg.n_suffix
    rows = np.concatenate([np.sort(rng.choice(cfg.n_ctx, m - n_suf, replace=False)),
                           np.arange(cfg.n_ctx, cfg.n_tokens)])
    _run(cb, cfg, rows, rows.size, True)


def test_bad_row_is_recorded_and_skipped(cb):
    cfg = get_config("tiny")
    plan = cb.Plan.from_config(cfg)
    x, w = generate_projection(cfg, 1)
    q = torch.zeros((cfg.n_tokens, cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((cfg.n_tokens, cfg.hkv, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    xg = torch.empty((3, x.shape[1]), dtype=torch.bfloat16, device="cuda")
    cb.cb_qkv_projection(plan, bf16_tensor(x), _i32([5, cfg.n_tokens + 3, 9]), 3, bf16_tensor(w), q, k, v, x_gathered=xg)
    with pytest.raises(cb.CacheBlendError):
        plan.check()
    assert torch.count_nonzero(q[5]) > 0 and torch.count_nonzero(q[9]) > 0
    with pytest.raises(cb.CacheBlendError):  # d_model not a multiple of 64
        cb.cb_qkv_projection(plan, bf16_tensor(x[:, :100].copy()), None, 4, bf16_tensor(w[:, :100].copy()), q, k, v)
    plan.close()


def test_gathered_rows_repeat_bit_identical(cb):
    # Back-to-back launches share the gather workspace and the tiles' shared-memory staging (the
    # epilogue reuses the TMA ring); a read of stale rows or staging would show as launches
    # that differ. Two inputs alternate over 16 launches at the Mistral-7B shape (524 rows =
    # 4 full tiles and a 12-row tail): every launch equals the first one on its input bit for bit.
    cfg = get_config("mistral7b")
    plan = cb.Plan.from_config(cfg)
    rng = np.random.default_rng(524)
    rows = _i32(np.concatenate([np.sort(rng.choice(cfg.n_ctx, 460, replace=False)),
                                np.arange(cfg.n_ctx, cfg.n_tokens)]))
    inputs = [tuple(bf16_tensor(a) for a in generate_projection(cfg, s)) for s in (1, 2)]
    shape = lambda h: (cfg.n_tokens, h, cfg.head_dim)
    xg = torch.empty((524, cfg.d_model), dtype=torch.bfloat16, device="cuda")
    first = [None, None]
    for it in range(16):
        x, w = inputs[it % 2]
        q = torch.zeros(shape(cfg.hq), dtype=torch.bfloat16, device="cuda")
        k = torch.zeros(shape(cfg.hkv), dtype=torch.bfloat16, device="cuda")
        v = torch.zeros(shape(cfg.hkv), dtype=torch.bfloat16, device="cuda")
        cb.cb_qkv_projection(plan, x, rows, 524, w, q, k, v, encode=True, x_gathered=xg)
        got = torch.cat([q.flatten(), k.flatten(), v.flatten()])
        if first[it % 2] is None:
            first[it % 2] = got
        else:
            assert torch.equal(got.view(torch.int16), first[it % 2].view(torch.int16)), f"launch {it}"
    plan.check()
    assert not torch.equal(first[0], first[1])
    plan.close()


def _run_indexed(cb, cfg, x_full, w, x_in, x_index, tokens, encode=True):
    """cb_qkv_projection_indexed on x_in (rows x_in[x_index[i]] or x_in[i]) written at tokens; the
    oracle takes the same hidden rows from x_full, where x_full[tokens[i]] is that row."""
    plan = cb.Plan.from_config(cfg)
    n, m = cfg.n_tokens, len(tokens)
    sentinel = lambda h: torch.full((n, h, cfg.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    q, k, v = sentinel(cfg.hq), sentinel(cfg.hkv), sentinel(cfg.hkv)
    xg = torch.empty((m, x_in.shape[1]), dtype=torch.bfloat16, device="cuda") if x_index is not None else None
    cb.cb_qkv_projection_indexed(plan, bf16_tensor(x_in), None if x_index is None else _i32(x_index), _i32(tokens), m,
                                 bf16_tensor(w), q, k, v, encode=encode, x_gathered=xg)
    plan.check()
    plan.close()
    tok = np.asarray(tokens)
    oq, ok, ov = qkv_projection(bf16_bits_to_f64(x_full), tok, bf16_bits_to_f64(w), cfg.hq, cfg.hkv, cfg.head_dim,
                                cfg.rope_theta, encode, "half")
    got = [bf16_bits_to_f64(bf16_bits(t)) for t in (q, k, v)]
    for g, o, what in zip(got, (oq, ok, ov), "qkv"):
        assert_close_bf16(g[tok], o, what=what)
        assert np.all(g[np.setdiff1d(np.arange(n), tok)] == 7.0)


def test_indexed_rows_in_place_written_at_tokens(cb):
    # Layers 4.. of the kept set: the previous layer left the hidden rows of S and the suffix in
    # list order, so row i of x is token tokens[i] (Mistral-7B shape, 460 + 64 rows).
    cfg = get_config("mistral7b")
    x, w = generate_projection(cfg, 3)
    rng = np.random.default_rng(46)
    tokens = np.concatenate([np.sort(rng.choice(cfg.n_ctx, 460, replace=False)), np.arange(cfg.n_ctx, cfg.n_tokens)])
    _run_indexed(cb, cfg, x, w, x[tokens], None, tokens)


def test_indexed_rows_by_position_in_a_compact_list(cb):
    # Layer 3 of the kept set: x holds the rows of the candidate list C (and the suffix) in list
    # order; S is a subset, taken by position. Unsorted positions, tiny shape with a 256-wide model.
    cfg = get_config("tiny")
    x, w = generate_projection(cfg, 4)
    rng = np.random.default_rng(47)
    cand = np.concatenate([np.sort(rng.choice(cfg.n_ctx, 150, replace=False)), np.arange(cfg.n_ctx, cfg.n_tokens)])
    pos = rng.permutation(cand.size)[:90]
    _run_indexed(cb, cfg, x, w, x[cand], pos, cand[pos])


def test_indexed_bad_index_and_token_are_recorded(cb):
    cfg = get_config("tiny")
    plan = cb.Plan.from_config(cfg)
    x, w = generate_projection(cfg, 1)
    q = torch.zeros((cfg.n_tokens, cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((cfg.n_tokens, cfg.hkv, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    xg = torch.empty((3, x.shape[1]), dtype=torch.bfloat16, device="cuda")
    xd, wd = bf16_tensor(x[:10]), bf16_tensor(w)
    # a token outside the plan: recorded, that row not written, the others written
    cb.cb_qkv_projection_indexed(plan, xd, None, _i32([4, cfg.n_tokens, 6]), 3, wd, q, k, v)
    with pytest.raises(cb.CacheBlendError):
        plan.check()
    assert torch.count_nonzero(q[4]) > 0 and torch.count_nonzero(q[6]) > 0
    plan.close()
    plan = cb.Plan.from_config(cfg)
    q.zero_()
    # an index outside x: recorded
    cb.cb_qkv_projection_indexed(plan, xd, _i32([1, 10, 2]), _i32([4, 5, 6]), 3, wd, q, k, v, x_gathered=xg)
    with pytest.raises(cb.CacheBlendError):
        plan.check()
    assert torch.count_nonzero(q[4]) > 0 and torch.count_nonzero(q[6]) > 0
    with pytest.raises(cb.CacheBlendError):  # in place needs m <= x_rows
        cb.cb_qkv_projection_indexed(plan, xd, None, None, 11, wd, q, k, v)
    plan.close()

"""Pins of the oracle's quality diagnostics ("数学推导" §形式化: the attention deviation the
selection minimises; §注意力稀疏性的量化分析: Sparsity(A, eps))."""

import dataclasses

import numpy as np
import pytest
import torch

from oracle.blend import blend_layer
from oracle.diagnostics import attention_deviation, attention_sparsity, blend_diagnostics, full_prefill_cache
from oracle.topk import k_for_ratio
from workloads import get_config
from workloads.generator import generate_layer


def test_deviation_is_the_frobenius_norm():
    a = np.zeros((2, 1, 2))
    b = np.zeros((2, 1, 2))
    a[0, 0] = [3.0, 0.0]
    a[1, 0] = [0.0, 4.0]
    assert attention_deviation(a, b) == (5.0, 0.0)
    assert attention_deviation(b, a) == (5.0, 5.0)


@pytest.mark.parametrize("n,eps,want", [(10, 0.3, 49 + 45), (10, 2.0, 100), (10, 0.0, 0), (7, 0.21, 18 + 21)])
def test_equal_scores_closed_form(n, eps, want):
    # q = 0: row i gives 1/(i+1) to keys 0..i and 0 to the i masked keys after it, so with
    # 0 < eps <= 1 the count is sum over rows with 1/(i+1) < eps of (i+1), plus n(n-1)/2.
    q = np.zeros((n, 1, 8))
    k = np.random.default_rng(0).standard_normal((n, 1, 8))
    count, near, total = attention_sparsity(q, np.arange(n), k, eps)
    assert (count, total) == (want, n * n)


@pytest.mark.parametrize("hq,hkv,n", [(4, 2, 40), (2, 1, 33)])
def test_counts_match_library_softmax_matrix(hq, hkv, n):
    rng = np.random.default_rng(n)
    q = rng.standard_normal((n, hq, 16)) * 2.0
    k = rng.standard_normal((n, hkv, 16))
    eps = 0.01
    count, near, total = attention_sparsity(q, np.arange(n), k, eps)
    g = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).permute(1, 0, 2)
    s = qt @ kt.transpose(1, 2) / np.sqrt(16)
    s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
    a = torch.softmax(s, dim=-1).numpy()
    assert count == int(np.sum(a < eps)) and total == hq * n * n
    assert near == int(np.sum(np.abs(a - eps) <= 1e-3 * eps))


def test_full_ratio_has_zero_deviation_and_low_ratio_does_not():
    cfg = dataclasses.replace(get_config("tiny"), name="tinyd", config_id=93, n_chunks=2, chunk_len=64, n_suffix=16)
    inp = generate_layer(cfg, 1)
    full = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), cfg.n_ctx, True, attention_rows=False)
    k_full, v_full = full_prefill_cache(cfg, inp)
    assert np.array_equal(full.k_fused, k_full) and np.array_equal(full.v_fused, v_full)
    d100 = blend_diagnostics(cfg, inp, full, 1e-3)
    assert d100["dev"] == 0.0 and d100["ref"] > 0
    part = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), k_for_ratio(15, cfg.n_ctx), True, attention_rows=False)
    d15 = blend_diagnostics(cfg, inp, part, 1e-3)
    assert 0 < d15["dev"] < d15["ref"]
    assert d15["count"] == d100["count"]  # sparsity is a property of the full prefill only

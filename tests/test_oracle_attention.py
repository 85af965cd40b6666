"""Pins of the oracle's causal GQA attention against the library routine and special cases.

"数学推导" §形式化 (Attention(Q, K, V)); "rag的kvcache问题" §transformer训练与推理并行计算的差异
(causal mask) and §阶段二 (row independence).
"""

import numpy as np
import pytest
import torch

from oracle.attention import causal_gqa_attention


def _sdpa_causal(q, k, v):
    # torch's causal attention in fp64 over all rows; q [N, Hq, D], k/v [N, Hkv, D]
    g = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1).permute(1, 0, 2)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 64, 300), (8, 8, 32, 130), (8, 1, 16, 77), (16, 2, 128, 260)])
def test_all_rows_equal_library_causal_attention(hq, hkv, d, n):
    rng = np.random.default_rng(hq * 100 + n)
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    ours = causal_gqa_attention(q, np.arange(n), k, v, block=64)
    np.testing.assert_allclose(ours, _sdpa_causal(q, k, v), rtol=1e-10, atol=1e-12)


def test_query_subset_equals_rows_of_full():
    rng = np.random.default_rng(7)
    n = 200
    q = rng.standard_normal((n, 4, 32))
    k = rng.standard_normal((n, 2, 32))
    v = rng.standard_normal((n, 2, 32))
    full = _sdpa_causal(q, k, v)
    rows = np.sort(rng.choice(n, size=37, replace=False))
    np.testing.assert_allclose(causal_gqa_attention(q[rows], rows, k, v, block=16), full[rows], rtol=1e-10, atol=1e-12)


def test_first_position_returns_its_own_value():
    rng = np.random.default_rng(8)
    k = rng.standard_normal((50, 2, 16))
    v = rng.standard_normal((50, 2, 16))
    q = rng.standard_normal((1, 4, 16)) * 30
    o = causal_gqa_attention(q, np.array([0]), k, v)
    np.testing.assert_allclose(o[0], np.repeat(v[0], 2, axis=0), rtol=0, atol=0)


def test_equal_scores_give_mean_of_visible_values():
    rng = np.random.default_rng(9)
    k = rng.standard_normal((40, 2, 16))
    v = rng.standard_normal((40, 2, 16))
    pos = np.array([0, 5, 39])
    o = causal_gqa_attention(np.zeros((3, 4, 16)), pos, k, v)
    for i, p in enumerate(pos):
        np.testing.assert_allclose(o[i], np.repeat(v[: p + 1].mean(axis=0), 2, axis=0), atol=1e-14)


def test_weights_sum_to_one():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((20, 8, 16)) * 5
    k = rng.standard_normal((90, 2, 16))
    o = causal_gqa_attention(q, np.sort(rng.choice(90, 20, replace=False)), k, np.ones((90, 2, 16)))
    np.testing.assert_allclose(o, 1.0, atol=1e-13)


# ---------------------------------------------------------------- decode ("rag的kvcache问题" §阶段 2)
from oracle.attention import decode_attention  # noqa: E402


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 64, 300), (8, 1, 16, 77), (16, 2, 128, 260)])
def test_decode_is_the_last_row_of_library_causal_attention(hq, hkv, d, n):
    rng = np.random.default_rng(hq + n)
    q = rng.standard_normal((n, hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    got = decode_attention(q[-1], k, v)
    np.testing.assert_allclose(got, _sdpa_causal(q, k, v)[-1], rtol=1e-12, atol=1e-12)


def test_decode_with_one_key_returns_its_value():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((8, 64)), rng.standard_normal((1, 2, 64)), rng.standard_normal((1, 2, 64))
    got = decode_attention(q, k, v)
    np.testing.assert_array_equal(got, np.repeat(v[0], 4, axis=0))


def test_decode_zero_query_averages_all_values():
    # q = 0 gives equal scores: every key weighs 1/n (nothing is masked in decode)
    rng = np.random.default_rng(6)
    k, v = rng.standard_normal((2, 37, 2, 32))
    got = decode_attention(np.zeros((4, 32)), k, v)
    np.testing.assert_allclose(got, np.repeat(v.mean(axis=0), 2, axis=0), rtol=1e-13)

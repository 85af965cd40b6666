"""Pins of the oracle's gathered QKV projection ("rag的kvcache问题" §阶段一, §渐进式过滤机制)."""

import numpy as np
import pytest

from oracle.projection import qkv_projection
from oracle.rope import rope_rotate, round_bf16


def _loops(x, rows, w):
    # the product written out element by element
    out = np.zeros((len(rows), w.shape[0]))
    for i, t in enumerate(rows):
        for o in range(w.shape[0]):
            out[i, o] = sum(x[t, c] * w[o, c] for c in range(x.shape[1]))
    return out


def test_gathered_product_matches_loops_and_splits_heads():
    rng = np.random.default_rng(1)
    hq, hkv, d, dm = 4, 2, 8, 16
    x = rng.standard_normal((10, dm))
    w = rng.standard_normal(((hq + 2 * hkv) * d, dm))
    rows = np.array([7, 2, 9])
    q, k, v = qkv_projection(x, rows, w, hq, hkv, d, 1e4, encode=False)
    ref = round_bf16(_loops(x, rows, w))
    np.testing.assert_array_equal(q.reshape(3, -1), ref[:, : hq * d])
    np.testing.assert_array_equal(k.reshape(3, -1), ref[:, hq * d: (hq + hkv) * d])
    np.testing.assert_array_equal(v.reshape(3, -1), ref[:, (hq + hkv) * d:])


def test_one_hot_rows_pick_weight_columns():
    hq, hkv, d, dm = 2, 1, 8, 8
    w = np.arange((hq + 2 * hkv) * d * dm, dtype=np.float64).reshape(-1, dm) / 64.0
    x = np.eye(dm)
    q, k, v = qkv_projection(x, [3], w, hq, hkv, d, 1e4, encode=False)
    np.testing.assert_array_equal(np.concatenate([q.ravel(), k.ravel(), v.ravel()]), round_bf16(w[:, 3]))


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_encoding_rotates_q_and_k_at_the_token_position_only(style):
    rng = np.random.default_rng(2)
    hq, hkv, d, dm = 2, 1, 16, 32
    x = rng.standard_normal((50, dm))
    w = rng.standard_normal(((hq + 2 * hkv) * d, dm))
    rows = np.array([0, 13, 49])
    q0, k0, v0 = qkv_projection(x, rows, w, hq, hkv, d, 1e4, encode=False, style=style)
    q1, k1, v1 = qkv_projection(x, rows, w, hq, hkv, d, 1e4, encode=True, style=style)
    np.testing.assert_array_equal(v0, v1)
    np.testing.assert_array_equal(q1[0], q0[0])  # position 0: no turn
    y = x[rows] @ w.T
    np.testing.assert_array_equal(q1, round_bf16(rope_rotate(y[:, : hq * d].reshape(3, hq, d), rows, 1e4, style)))
    # turning keeps each pair's length
    i0, i1 = (np.arange(d // 2), np.arange(d // 2) + d // 2) if style == "half" else (np.arange(0, d, 2), np.arange(1, d, 2))
    kf = rope_rotate(y[:, hq * d: (hq + hkv) * d].reshape(3, hkv, d), rows, 1e4, style)
    kr = y[:, hq * d: (hq + hkv) * d].reshape(3, hkv, d)
    np.testing.assert_allclose(kf[..., i0] ** 2 + kf[..., i1] ** 2, kr[..., i0] ** 2 + kr[..., i1] ** 2, rtol=1e-12)

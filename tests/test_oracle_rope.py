"""Pins of the oracle's RoPE and re-rotation against closed forms and identities.

"数学推导" §RoPE 位置编码的相对位置不变性证明 and §CacheBlend 中的应用.
"""

import os

import numpy as np
import pytest
import torch

from oracle.rope import inv_freq, pair_indices, rerotate, rope_rotate, round_bf16
from workloads.generator import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_closed_form.txt")


def _golden():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, vals = (s.strip() for s in line.split("|"))
        out[name] = np.array([float(v) for v in vals.split()])
    return out


def test_inv_freq_closed_form():
    np.testing.assert_allclose(inv_freq(8, 1e4), _golden()["inv_freq_d8_theta1e4"], rtol=1e-15)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_d2_is_the_textbook_rotation(style):
    g = _golden()
    np.testing.assert_allclose(rope_rotate(np.array([[[1.0, 0.0]]]), 1, 1e4, style)[0, 0], g["d2_x10_p1"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rope_rotate(np.array([[[1.0, 0.0]]]), -1, 1e4, style)[0, 0], g["d2_x10_pm1"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rope_rotate(np.array([[[0.0, 1.0]]]), 1, 1e4, style)[0, 0], g["d2_x01_p1"], rtol=0, atol=1e-15)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 1, 2))
    p = rng.integers(-50, 50, size=5)
    for i in range(5):
        r = np.array([[np.cos(p[i]), -np.sin(p[i])], [np.sin(p[i]), np.cos(p[i])]])
        np.testing.assert_allclose(rope_rotate(x[i:i + 1], p[i], 1e4, style)[0, 0], r @ x[i, 0], atol=1e-14)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_complex_multiplication_form(style):
    # RoFormer: rotating a pair by angle a is multiplying x0 + i x1 by e^{i a}.
    rng = np.random.default_rng(1)
    d, theta = 16, 1e4
    x = rng.standard_normal((7, 3, d))
    pos = rng.integers(0, 5000, size=7)
    out = rope_rotate(x, pos, theta, style)
    if style == "half":
        z, zo = x[..., : d // 2] + 1j * x[..., d // 2:], out[..., : d // 2] + 1j * out[..., d // 2:]
    else:
        z, zo = x[..., 0::2] + 1j * x[..., 1::2], out[..., 0::2] + 1j * out[..., 1::2]
    freqs = np.array([theta ** (-2.0 * j / d) for j in range(d // 2)])
    expect = z * np.exp(1j * pos[:, None, None] * freqs[None, None, :])
    np.testing.assert_allclose(zo, expect, atol=1e-12)


def test_pair_indices_cover_all_dims():
    for style in ("half", "interleaved"):
        i0, i1 = pair_indices(128, style)
        assert sorted(np.concatenate([i0, i1]).tolist()) == list(range(128))


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_relative_position_invariance(style):
    # q~_m . k~_n = q_m^T R_{n-m} k_n depends on n - m only.
    rng = np.random.default_rng(2)
    d, theta = 128, 1e4
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    for m, n, s in [(0, 5, 100), (17, 3, 4000), (1000, 1000, 31000), (32000, 12, 777)]:
        a = float(np.sum(rope_rotate(q, m, theta, style) * rope_rotate(k, n, theta, style)))
        b = float(np.sum(rope_rotate(q, m + s, theta, style) * rope_rotate(k, n + s, theta, style)))
        c = float(np.sum(q * rope_rotate(k, n - m, theta, style)))
        assert abs(a - b) <= 1e-11 * max(1.0, abs(a))
        assert abs(a - c) <= 1e-11 * max(1.0, abs(a))


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("theta", [1e4, 5e5])
def test_rerotation_equals_direct_encoding(style, theta):
    # k_new = R_{p_new} k_base = R_{p_new - p_old} (R_{p_old} k_base)
    rng = np.random.default_rng(3)
    base = rng.standard_normal((64, 2, 128))
    p_old = rng.integers(0, 2048, size=64)
    p_new = p_old + 2048 * rng.integers(0, 16, size=64)
    k_old = rope_rotate(base, p_old, theta, style)
    np.testing.assert_allclose(rerotate(k_old, p_old, p_new, theta, style),
                               rope_rotate(base, p_new, theta, style), atol=1e-11)


def test_zero_delta_is_identity_bitwise():
    x = np.random.default_rng(4).standard_normal((9, 2, 64))
    assert np.array_equal(rerotate(x, np.arange(9), np.arange(9), 1e4), x)


def test_rotation_preserves_pair_norms():
    x = np.random.default_rng(5).standard_normal((11, 4, 64))
    y = rope_rotate(x, np.arange(11) * 997, 1e4, "half")
    i0, i1 = pair_indices(64, "half")
    np.testing.assert_allclose(x[..., i0] ** 2 + x[..., i1] ** 2, y[..., i0] ** 2 + y[..., i1] ** 2, rtol=1e-13)


def test_round_bf16_matches_bit_rounding_and_torch():
    rng = np.random.default_rng(6)
    x32 = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ours = round_bf16(x32.astype(np.float64))
    bits = bf16_bits_to_f32(f32_to_bf16_bits(x32)).astype(np.float64)
    assert np.array_equal(ours, bits)
    tt = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, tt)
    # ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert round_bf16(np.array([-(1 + 3 * 2.0 ** -8)]))[0] == -(1 + 2.0 ** -6)

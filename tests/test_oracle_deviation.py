"""Pins of the oracle's V deviation ("数学推导" §近似解).

The canonical fp32 order is pinned by hand-derived rounding cases; the value
by the exact rational sum within the fp32 summation error bound.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle.deviation import deviation_canonical_f32, deviation_fp64
from workloads.generator import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "deviation_rounding.txt")


def _cases():
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, e, entries, expect = (s.strip() for s in line.split("|"))
        yield name, int(e), entries.split(), float.fromhex(expect)


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: c[0])
def test_hand_derived_rounding_order(case):
    _, e, entries, expect = case
    vn = np.zeros(e, np.float32)
    vo = np.zeros(e, np.float32)
    for ent in entries:
        idx, a, b = ent.split(":")
        vn[int(idx)] = float.fromhex(a) if "x" in a else float(a)
        vo[int(idx)] = float.fromhex(b) if "x" in b else float(b)
    # E elements as one token of Hkv = E / 128 heads of D = 128 (or one head)
    shape = (1, e // 128, 128) if e % 128 == 0 else (1, 1, e)
    got = deviation_canonical_f32(f32_to_bf16_bits(vn).reshape(shape), f32_to_bf16_bits(vo).reshape(shape))
    assert got.dtype == np.float32
    assert float(got[0]) == expect


def test_equal_rows_give_exact_zero():
    bits = f32_to_bf16_bits(np.random.default_rng(0).standard_normal((5, 8, 128)).astype(np.float32))
    dev = deviation_canonical_f32(bits, bits)
    assert np.all(dev == 0) and not np.any(np.signbit(dev))


@pytest.mark.parametrize("d", [3.0, 1.5, -0.375, 2.0 ** -60, 1.0 + 2.0 ** -7])
def test_single_nonzero_element_is_its_square(d):
    vn = np.zeros((1, 2, 64), np.float32)
    vo = np.zeros((1, 2, 64), np.float32)
    vn[0, 1, 17] = d
    got = deviation_canonical_f32(f32_to_bf16_bits(vn), f32_to_bf16_bits(vo))
    assert float(got[0]) == float(np.float32(d) * np.float32(d))


@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (1, 8), (3, 40)])
def test_within_fp32_bound_of_exact_sum(hkv, d):
    rng = np.random.default_rng(hkv * 1000 + d)
    m = 6
    vo = f32_to_bf16_bits(rng.standard_normal((m, hkv, d)).astype(np.float32))
    scale = np.exp(rng.uniform(-8, 2, size=(m, 1, 1))).astype(np.float32)
    vn = f32_to_bf16_bits(bf16_bits_to_f32(vo) + scale * rng.standard_normal((m, hkv, d)).astype(np.float32))
    dev = deviation_canonical_f32(vn, vo)
    a = bf16_bits_to_f32(vn).astype(np.float64).reshape(m, -1)
    b = bf16_bits_to_f32(vo).astype(np.float64).reshape(m, -1)
    e = hkv * d
    n_seq = -(-e // 256) * 8  # sequential adds per lane
    u = 2.0 ** -24
    for t in range(m):
        exact = sum((Fraction(float(x)) - Fraction(float(y))) ** 2 for x, y in zip(a[t], b[t]))
        # d rounding (1u, doubled by squaring), product rounding (1u), n_seq + 5 adds
        bound = (n_seq + 5 + 3) * u * 1.01 * float(exact)
        assert abs(Fraction(float(dev[t])) - exact) <= Fraction(bound)
    np.testing.assert_allclose(dev, deviation_fp64(bf16_bits_to_f32(vn), bf16_bits_to_f32(vo)), rtol=1e-5)

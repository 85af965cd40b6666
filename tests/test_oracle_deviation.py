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


# ---------------------------------------------------------------------------
# K+V deviation ("rag的kvcache问题" §核心发现: Δkv on the whole KV of a token).

from oracle.deviation import (key_deviation_fp64, kv_deviation_canonical_f32, kv_deviation_fp64,  # noqa: E402
                              rotate_f32)
from oracle.rope import rope_rotate, rope_table_f32  # noqa: E402


def _bits(rng, *shape, scale=1.0):
    return f32_to_bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


def test_rope_table_zero_position_and_closed_form():
    c, s = rope_table_f32([0, 1, 7], 8, 1e4)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    # pair 0 turns by p radians (theta^0 = 1); pair j of D = 8 by p * theta^(-j/4)
    assert c[1, 0] == np.float32(np.cos(1.0)) and s[2, 0] == np.float32(np.sin(7.0))
    np.testing.assert_allclose(c[2, 2], np.cos(7.0 * 1e4 ** -0.5), rtol=1e-7)


def test_rope_table_matches_library_cos_within_half_ulp():
    pos = np.arange(0, 4096, 37)
    c, s = rope_table_f32(pos, 128, 5e5)
    ang = pos[:, None] * (5e5 ** (-2.0 * np.arange(64) / 128))[None, :]
    for got, ref in ((c, np.cos(ang)), (s, np.sin(ang))):
        ulp = np.spacing(np.abs(got)).astype(np.float64)
        assert np.all(np.abs(got.astype(np.float64) - ref) <= 0.5 * ulp + 1e-15)


@pytest.mark.parametrize("p_old", [1, 3, 300])
def test_key_term_closed_form_single_pair(p_old):
    # one head of D = 8, k_new = k_old = e_0 (pair 0 turns by one radian per position):
    # ||R_{p_new} e_0 - R_{p_new - p_old} e_0||^2 = |e^{i p_old} - 1|^2 = 2 - 2 cos(p_old)
    e0 = np.zeros((1, 1, 8))
    e0[0, 0, 0] = 1.0
    p_new = p_old + 5000
    got = key_deviation_fp64(e0, e0, [p_old], [p_new], 1e4)
    assert got[0] == pytest.approx(2.0 - 2.0 * np.cos(p_old), rel=1e-12, abs=1e-15)
    bits = f32_to_bf16_bits(e0.astype(np.float32))
    zero = np.zeros_like(bits)
    got32 = kv_deviation_canonical_f32(bits, bits, zero, zero, np.array([p_old]), 1e4)
    assert float(got32[0]) == pytest.approx(2.0 - 2.0 * np.cos(p_old), rel=1e-6)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_key_term_is_frame_invariant(style):
    # R_{p_new} = R_{p_new - p_old} R_{p_old} and rotations keep norms, so the key term in the
    # global frame equals ||R_{p_old} k_new - k_old||^2 (a wrong sign of either turn breaks this).
    rng = np.random.default_rng(11)
    kn, ko = rng.standard_normal((2, 9, 3, 64))
    p_old = rng.integers(0, 2048, 9)
    p_new = p_old + rng.integers(0, 30000, 9)
    glob = key_deviation_fp64(kn, ko, p_old, p_new, 1e4, style)
    local = ((rope_rotate(kn, p_old, 1e4, style) - ko) ** 2).reshape(9, -1).sum(1)
    np.testing.assert_allclose(glob, local, rtol=1e-11)
    # and it is not the same as comparing without moving the cached key
    unmoved = ((rope_rotate(kn, p_new, 1e4, style) - ko) ** 2).reshape(9, -1).sum(1)
    assert np.all(np.abs(unmoved - glob) > 1e-6 * glob)


def test_kv_is_key_term_plus_v_term():
    rng = np.random.default_rng(12)
    kn, ko, vn, vo = rng.standard_normal((4, 5, 2, 64))
    p_old = np.arange(5) * 100
    got = kv_deviation_fp64(kn, ko, vn, vo, p_old, p_old + 512, 1e4)
    ref = key_deviation_fp64(kn, ko, p_old, p_old + 512, 1e4) + deviation_fp64(vn, vo)
    np.testing.assert_array_equal(got, ref)


def test_kv_at_position_zero_is_the_canonical_sum_of_k_then_v():
    # at p_old = 0 the table gives c = 1, s = 0 exactly, so the key part is k_new - k_old and the
    # K+V number is the pinned V-only canonical sum over the rows [K heads, V heads]
    # (Hkv * D = 256: no padding between the two parts).
    rng = np.random.default_rng(13)
    kn, ko, vn, vo = (_bits(rng, 7, 2, 128) for _ in range(4))
    got = kv_deviation_canonical_f32(kn, ko, vn, vo, np.zeros(7, np.int64), 1e4)
    ref = deviation_canonical_f32(np.concatenate([kn, vn], axis=1), np.concatenate([ko, vo], axis=1))
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    same = kv_deviation_canonical_f32(ko, ko, vn, vo, np.zeros(7, np.int64), 1e4)
    np.testing.assert_array_equal(same.view(np.uint32), deviation_canonical_f32(vn, vo).view(np.uint32))


def _kv_canonical_scalar(kn, ko, vn, vo, p_old, theta, style):
    """Element-by-element restatement (numpy fp32 scalars, plain loops) for tiny inputs."""
    f32 = np.float32
    m, hkv, d = kn.shape
    out = []
    for t in range(m):
        c_t, s_t = rope_table_f32([p_old[t]], d, theta)
        seq = []
        for h in range(hkv):
            for j in range(d):
                if style == "half":
                    pair, first = (j, True) if j < d // 2 else (j - d // 2, False)
                    x, y = kn[t, h, pair], kn[t, h, pair + d // 2]
                else:
                    pair, first = j // 2, j % 2 == 0
                    x, y = kn[t, h, 2 * pair], kn[t, h, 2 * pair + 1]
                c, s = c_t[0, pair], s_t[0, pair]
                r = f32(f32(x * c) - f32(y * s)) if first else f32(f32(x * s) + f32(y * c))
                seq.append(f32(r - ko[t, h, j]))
        seq += [f32(0)] * (-len(seq) % 256)
        seq += [f32(a - b) for a, b in zip(vn[t].reshape(-1), vo[t].reshape(-1))]
        seq += [f32(0)] * (-len(seq) % 256)
        acc = [f32(0)] * 32
        for c0 in range(len(seq) // 8):
            lane = c0 % 32
            for e in range(8):
                v = seq[c0 * 8 + e]
                acc[lane] = f32(acc[lane] + f32(v * v))
        for off in (16, 8, 4, 2, 1):
            acc = [f32(acc[l] + acc[l ^ off]) for l in range(32)]
        out.append(acc[0])
    return np.array(out, np.float32)


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("hkv,d", [(2, 64), (1, 64), (3, 128)])
def test_kv_canonical_matches_plain_loops(style, hkv, d):
    rng = np.random.default_rng(hkv * 7 + d)
    kn, ko, vn, vo = (_bits(rng, 4, hkv, d) for _ in range(4))
    p_old = rng.integers(0, 4000, 4)
    got = kv_deviation_canonical_f32(kn, ko, vn, vo, p_old, 1e4, style)
    f = bf16_bits_to_f32
    ref = _kv_canonical_scalar(f(kn), f(ko), f(vn), f(vo), p_old, 1e4, style)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("noise", [1.0, 0.01])
def test_kv_canonical_within_rounding_bound_of_fp64(style, noise):
    # cached keys encoded at p_old from a pre-RoPE key, recomputed key = pre-RoPE key + noise:
    # the key term is then about noise^2 * E, where cancellation makes the fp32 error relative
    # to |k|, not to the difference. Bound per element: table entries (u/2 each), two products
    # and a sum (u each) and the difference (u) give |error of d| <= 4u (|x| + |y|) + u |d|.
    rng = np.random.default_rng(int(noise * 100) + (style == "half"))
    m, hkv, d, theta = 6, 2, 128, 1e4
    p_old = rng.integers(0, 2048, m)
    pre = rng.standard_normal((m, hkv, d))
    ko = f32_to_bf16_bits(rope_rotate(pre, p_old, theta, style).astype(np.float32))
    kn = f32_to_bf16_bits((pre + noise * rng.standard_normal((m, hkv, d))).astype(np.float32))
    vo = _bits(rng, m, hkv, d)
    vn = f32_to_bf16_bits(bf16_bits_to_f32(vo) + np.float32(noise) * rng.standard_normal((m, hkv, d)).astype(np.float32))
    got = kv_deviation_canonical_f32(kn, ko, vn, vo, p_old, theta, style).astype(np.float64)
    f = lambda b: bf16_bits_to_f32(b).astype(np.float64)
    exact = kv_deviation_fp64(f(kn), f(ko), f(vn), f(vo), p_old, p_old + 3000, theta, style)
    u = 2.0 ** -24
    x = np.abs(f(kn))
    from oracle.rope import pair_indices
    i0, i1 = pair_indices(d, style)
    pair_mag = np.empty_like(x)
    pair_mag[..., i0] = x[..., i0] + x[..., i1]
    pair_mag[..., i1] = pair_mag[..., i0]
    dk = rope_rotate(f(kn), p_old, theta, style) - f(ko)
    err_d = 4 * u * pair_mag + u * np.abs(dk)
    key_bound = (2 * np.abs(dk) * err_d + err_d ** 2).reshape(m, -1).sum(1)
    n_seq = 2 * (-(-hkv * d // 256)) * 8
    bound = key_bound + (n_seq + 8) * u * 1.01 * exact
    assert np.all(np.abs(got - exact) <= bound), (got - exact, bound)


def test_rotate_f32_identity_turn_is_bitwise():
    # c = 1, s = 0 leaves rows unchanged bit for bit, whatever the sign of the other member
    x = np.array([[[1.5, -2.0, -0.0, 3.0]]], np.float32)
    out = rotate_f32(x, np.ones((1, 2), np.float32), np.zeros((1, 2), np.float32), "interleaved")
    np.testing.assert_array_equal(out.view(np.uint32), x.view(np.uint32))


def test_empty_candidate_set_has_no_deviations():
    # a layer whose candidate set is empty (r = 0 selects nothing at layer 1) ranks nothing
    empty = np.zeros((0, 8, 128), np.uint16)
    assert deviation_canonical_f32(empty, empty).shape == (0,)
    assert deviation_fp64(empty.astype(np.float64), empty.astype(np.float64)).shape == (0,)
    got = kv_deviation_canonical_f32(empty, empty, empty, empty, np.zeros(0, np.int64), 1e4)
    assert got.shape == (0,)

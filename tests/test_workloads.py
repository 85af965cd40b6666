"""The seeded input generator: bf16 rounding against torch's conversion, determinism, shapes and
the noise model of the workloads (CPU)."""

import numpy as np
import pytest
import torch

from workloads import get_config
from workloads.generator import bf16_bits_to_f32, f32_to_bf16_bits, generate_layer, hkvd_noise_sets


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(3_000_003).astype(np.float32),
        (rng.standard_normal(10_000) * 1e30).astype(np.float32),
        (rng.standard_normal(10_000) * 1e-30).astype(np.float32),
        # exact ties between two bf16 values: the 16 dropped bits are 0x8000
        (np.arange(1, 5000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 1e-45, -1e-45], dtype=np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f32_to_bf16_bits(x)
    assert got.dtype == np.uint16 and np.array_equal(got, want)
    # widening is exact
    assert np.array_equal(bf16_bits_to_f32(got), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_rounding_keeps_shape_and_accepts_strided_input():
    x = np.random.default_rng(6).standard_normal((6, 8)).astype(np.float32)[:, ::2]
    got = f32_to_bf16_bits(x)
    assert got.shape == (6, 4)
    assert np.array_equal(got, f32_to_bf16_bits(np.ascontiguousarray(x)))


def test_layers_are_deterministic_and_shaped():
    cfg = get_config("tiny")
    a, b = generate_layer(cfg, 1), generate_layer(cfg, 1)
    for name in ("k_old", "v_old", "k_new", "v_new", "q"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    assert a.k_old.shape == (cfg.n_ctx, cfg.hkv, cfg.head_dim)
    assert a.k_new.shape == (cfg.n_tokens, cfg.hkv, cfg.head_dim)
    assert a.q.shape == (cfg.n_tokens, cfg.hq, cfg.head_dim)


@pytest.mark.parametrize("name", ["mistral7b", "llama70b"])
def test_noise_sets_have_the_stated_size_and_swap_a_tenth_per_layer(name):
    cfg = get_config(name)
    sets = hkvd_noise_sets(cfg)
    size = int(np.floor(cfg.hkvd_frac * cfg.n_ctx))
    assert all(len(s) == size and np.all(np.diff(s) > 0) for s in sets)
    n_swap = int(np.floor(cfg.swap_frac * size))
    assert cfg.swap_frac == pytest.approx(0.1)
    for prev, cur in zip(sets[:-1], sets[1:]):
        # a tenth of the set leaves for tokens that were outside it
        assert len(np.setdiff1d(prev, cur)) == n_swap and len(np.setdiff1d(cur, prev)) == n_swap

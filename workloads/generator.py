"""Seeded input generator: the bytes both the CUDA path and the oracle consume.

Every tensor is drawn in fp32 from numpy's PCG64 and rounded once to bf16
(round to nearest, ties to even); arrays hold raw bf16 bit patterns as uint16.
Streams are keyed by (workload seed, layer, tensor id), so any one layer can be
regenerated alone.

What is drawn, per layer (the input recipe):
  k_old, v_old   [n_ctx, hkv, d]    ~ N(0, 1)   the reused chunk caches
  k_new, v_new   [n_tokens, hkv, d] token-indexed recomputed K (before RoPE)
                                    and V. Context rows: old + s_t * eps with
                                    eps ~ N(0, 1); suffix rows: fresh N(0, 1)
  q              [n_tokens, hq, d]  ~ N(0, 1), before RoPE
where s_t is the per-token noise scale of the workload: sigma_hi on the
high-deviation set H_l and sigma_lo elsewhere, or a lognormal scale.
H_1 is a seeded random subset; H_{l+1} is H_l with a seeded fraction of its
members swapped for tokens outside it.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .configs import BlendConfig

_T_K_OLD, _T_V_OLD, _T_K_EPS, _T_V_EPS, _T_Q = 0, 1, 2, 3, 4
_T_K_SUF, _T_V_SUF, _T_LOGN, _T_SETS = 5, 6, 7, 100
_T_DEC_K, _T_DEC_V, _T_DEC_Q = 200, 201, 202
_T_PROJ_X, _T_PROJ_W = 300, 301


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Per element: (b + 0x7FFF + ((b >> 16) & 1)) >> 16 on the fp32 bit pattern b, modulo 2^32. Done
    in blocks of 2^20 elements with one scratch buffer, so large tensors do not allocate several
    full-size temporaries."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    b = a.view(np.uint32).reshape(-1)
    out = np.empty(b.shape, dtype=np.uint16)
    block = 1 << 20
    t = np.empty(min(block, b.size), dtype=np.uint32)
    for i in range(0, b.size, block):
        src = b[i:i + block]
        w = t[:src.size]
        np.right_shift(src, np.uint32(16), out=w)
        np.bitwise_and(w, np.uint32(1), out=w)
        np.add(w, np.uint32(0x7FFF), out=w)
        np.add(w, src, out=w)
        np.right_shift(w, np.uint32(16), out=w)
        out[i:i + block] = w
    return out.reshape(a.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(cfg: BlendConfig, layer: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, layer, tensor])))


def hkvd_noise_sets(cfg: BlendConfig) -> list:
    """Per-layer high-deviation token sets H_1 .. H_layers (sorted int64 arrays).

    Empty list entries never occur for the "set" noise model; the lognormal
    model has no set and returns a list of None.
    """
    if cfg.noise != "set":
        return [None] * cfg.layers
    rng = _rng(cfg, 0, _T_SETS)
    size = int(np.floor(cfg.hkvd_frac * cfg.n_ctx))
    cur = np.sort(rng.choice(cfg.n_ctx, size=size, replace=False)).astype(np.int64)
    sets = [cur]
    for _ in range(1, cfg.layers):
        n_swap = int(np.floor(cfg.swap_frac * cur.size))
        if n_swap > 0:
            out = rng.choice(cur, size=n_swap, replace=False)
            outside = np.setdiff1d(np.arange(cfg.n_ctx, dtype=np.int64), cur, assume_unique=True)
            inn = rng.choice(outside, size=n_swap, replace=False)
            cur = np.sort(np.concatenate([np.setdiff1d(cur, out, assume_unique=True), inn]))
        sets.append(cur)
    return sets


@dataclass
class LayerInputs:
    layer: int
    k_old: np.ndarray        # uint16 bf16 bits [n_ctx, hkv, d]
    v_old: np.ndarray        # uint16 bf16 bits [n_ctx, hkv, d]
    k_new: np.ndarray        # uint16 bf16 bits [n_tokens, hkv, d]
    v_new: np.ndarray        # uint16 bf16 bits [n_tokens, hkv, d]
    q: np.ndarray            # uint16 bf16 bits [n_tokens, hq, d]
    noise_scale: np.ndarray  # float32 [n_ctx]
    hkvd_set: np.ndarray | None


def noise_scales(cfg: BlendConfig, layer: int, hset) -> np.ndarray:
    if cfg.noise == "set":
        s = np.full(cfg.n_ctx, cfg.sigma_lo, dtype=np.float32)
        s[hset] = cfg.sigma_hi
        return s
    if cfg.noise == "lognormal":
        z = _rng(cfg, layer, _T_LOGN).standard_normal(cfg.n_ctx, dtype=np.float32)
        return np.exp(np.float32(cfg.lognormal_mu) + np.float32(cfg.lognormal_sigma) * z).astype(np.float32)
    raise ValueError(f"unknown noise model {cfg.noise!r}")


def generate_layer(cfg: BlendConfig, layer: int, sets: list | None = None) -> LayerInputs:
    """Inputs of one layer (1-based). Pass `sets` from hkvd_noise_sets to avoid recomputing it."""
    if not 1 <= layer <= cfg.layers:
        raise ValueError(f"layer {layer} outside 1..{cfg.layers}")
    if sets is None:
        sets = hkvd_noise_sets(cfg)
    hset = sets[layer - 1]
    n_ctx, n, hkv, hq, d = cfg.n_ctx, cfg.n_tokens, cfg.hkv, cfg.hq, cfg.head_dim
    s = noise_scales(cfg, layer, hset)[:, None, None]

    k_old = f32_to_bf16_bits(_rng(cfg, layer, _T_K_OLD).standard_normal((n_ctx, hkv, d), dtype=np.float32))
    v_old = f32_to_bf16_bits(_rng(cfg, layer, _T_V_OLD).standard_normal((n_ctx, hkv, d), dtype=np.float32))

    k_new = np.empty((n, hkv, d), dtype=np.uint16)
    v_new = np.empty((n, hkv, d), dtype=np.uint16)
    # recomputed = cached + s * eps, in fp32 (in place on eps), rounded once to bf16
    k_eps = _rng(cfg, layer, _T_K_EPS).standard_normal((n_ctx, hkv, d), dtype=np.float32)
    np.multiply(k_eps, s, out=k_eps)
    np.add(k_eps, bf16_bits_to_f32(k_old), out=k_eps)
    k_new[:n_ctx] = f32_to_bf16_bits(k_eps)
    del k_eps
    v_eps = _rng(cfg, layer, _T_V_EPS).standard_normal((n_ctx, hkv, d), dtype=np.float32)
    np.multiply(v_eps, s, out=v_eps)
    np.add(v_eps, bf16_bits_to_f32(v_old), out=v_eps)
    v_new[:n_ctx] = f32_to_bf16_bits(v_eps)
    del v_eps
    n_suf = cfg.n_suffix
    k_new[n_ctx:] = f32_to_bf16_bits(_rng(cfg, layer, _T_K_SUF).standard_normal((n_suf, hkv, d), dtype=np.float32))
    v_new[n_ctx:] = f32_to_bf16_bits(_rng(cfg, layer, _T_V_SUF).standard_normal((n_suf, hkv, d), dtype=np.float32))

    q = f32_to_bf16_bits(_rng(cfg, layer, _T_Q).standard_normal((n, hq, d), dtype=np.float32))
    return LayerInputs(layer, k_old, v_old, k_new, v_new, q, s[:, 0, 0].copy(), hset)


@dataclass
class DecodeInputs:
    layer: int
    k: np.ndarray  # uint16 bf16 bits [n_keys, hkv, d]: the layer's cache after the request, plus one token
    v: np.ndarray  # uint16 bf16 bits [n_keys, hkv, d]
    q: np.ndarray  # uint16 bf16 bits [hq, d]: the newest token's query (taken as already encoded)


def generate_decode(cfg: BlendConfig, layer: int, extra: int = 1) -> DecodeInputs:
    """One decode step's inputs for a layer: N(0, 1) caches of n_tokens + extra rows and a query."""
    n = cfg.n_tokens + extra
    k = f32_to_bf16_bits(_rng(cfg, layer, _T_DEC_K).standard_normal((n, cfg.hkv, cfg.head_dim), dtype=np.float32))
    v = f32_to_bf16_bits(_rng(cfg, layer, _T_DEC_V).standard_normal((n, cfg.hkv, cfg.head_dim), dtype=np.float32))
    q = f32_to_bf16_bits(_rng(cfg, layer, _T_DEC_Q).standard_normal((cfg.hq, cfg.head_dim), dtype=np.float32))
    return DecodeInputs(layer, k, v, q)


def generate_projection(cfg: BlendConfig, layer: int, d_model: int | None = None):
    """The QKV projection's inputs for a layer: hidden rows x [n_tokens, d_model] ~ N(0, 1) and
    a fused weight w [(hq + 2 hkv) * head_dim, d_model] ~ N(0, 1 / d_model) (random weights of
    the model's shape; no trained weights), both as bf16 bits."""
    dm = d_model or cfg.d_model
    if dm <= 0:
        raise ValueError("the workload has no hidden size")
    n_out = (cfg.hq + 2 * cfg.hkv) * cfg.head_dim
    x = f32_to_bf16_bits(_rng(cfg, layer, _T_PROJ_X).standard_normal((cfg.n_tokens, dm), dtype=np.float32))
    w = f32_to_bf16_bits(_rng(cfg, layer, _T_PROJ_W).standard_normal((n_out, dm), dtype=np.float32)
                         * np.float32(1.0 / np.sqrt(dm)))
    return x, w

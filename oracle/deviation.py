"""Per-token V deviation, the key of the HKVD selection.

"数学推导" §近似解: the greedy selection ranks token i by the squared L2
distance ||V_new[i] - V_old[i]||_2^2 between its recomputed and its cached V
("rag的kvcache问题" §核心发现 calls the per-token distance the KV deviation).
For a layer with Hkv kv heads of dimension D the token's V is the Hkv*D
vector of all its heads, so one token gets one number.

The exact value is a real number; the selection that ranks these numbers is
an integer result decided by floating point, so the oracle and the CUDA
kernel must form the same fp32 number. ``deviation_canonical_f32`` writes out
that number's summation order (the order the kernel also follows):

  * the E = Hkv*D elements of a token, in memory order e = h*D + j, are cut
    into 8-element chunks c = e // 8; E is padded with zeros to a multiple of
    256 (adding +0 leaves every partial sum unchanged);
  * lane l in 0..31 owns the chunks c = l, l+32, l+64, ... in that order and,
    inside a chunk, the elements in order; for each element it forms
    d = fl32(v_new - v_old), p = fl32(d*d), acc_l = fl32(acc_l + p), with
    acc_l starting at +0 (bf16 to fp32 is exact; no fused multiply-add);
  * the 32 partial sums are combined by a butterfly: for off = 16, 8, 4, 2, 1,
    acc_l = fl32(acc_l + acc_(l xor off)); the result is acc_0.

fl32 is IEEE binary32 round-to-nearest-even with subnormals kept.

K+V variant. "rag的kvcache问题" §核心发现 writes the deviation on the whole
KV of a token, Δkv = |KV_i[j] - KV_i^full[j]|. Read here as the squared
distance of K and of V summed: dev = ||K~_new - K~_old||^2 + ||V_new - V_old||^2,
where the keys are compared as attention sees them, both at the global
position p_new: K~_new = R_{p_new} k_new (the recomputed key before RoPE) and
K~_old = R_{p_new - p_old} k_old (the cached key, encoded at its chunk-local
position p_old, moved). Because every R is a rotation, R_{p_new} = R_{p_new -
p_old} R_{p_old} and ||R x|| = ||x||, the key term equals ||R_{p_old} k_new -
k_old||^2 exactly; the fp32 form below uses that chunk-local frame (one
rotation instead of two). ``kv_deviation_canonical_f32`` fixes the number:
  * the K part: each element of R_{p_old} k_new is formed in fp32 from the
    table of ``rope.rope_table_f32`` (c, s at p_old) as
    x' = fl32(fl32(x c) - fl32(y s)) for the first member x of a pair and
    y' = fl32(fl32(x s) + fl32(y c)) for the second member y; then
    d = fl32(x' - k_old) per element;
  * the V part: d = fl32(v_new - v_old) per element;
  * each part has E = Hkv*D elements, padded with zeros to a multiple of 256;
    the K part, then the V part, form one sequence that is cut into 8-element
    chunks and summed by the canonical order above (so every lane adds its K
    chunks before its V chunks).
"""

from __future__ import annotations

import numpy as np

from .rope import pair_indices, rerotate, rope_rotate, rope_table_f32


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def deviation_fp64(v_new: np.ndarray, v_old: np.ndarray) -> np.ndarray:
    """sum over heads and dims of (v_new - v_old)^2 per token, in fp64 (plain order)."""
    d = np.asarray(v_new, dtype=np.float64) - np.asarray(v_old, dtype=np.float64)
    return (d * d).reshape(d.shape[0], int(np.prod(d.shape[1:]))).sum(axis=1)


def key_deviation_fp64(k_new, k_old, p_old, p_new, theta: float, style: str = "half") -> np.ndarray:
    """sum over heads and dims of (R_{p_new} k_new - R_{p_new - p_old} k_old)^2 per token, fp64.

    k_new: recomputed keys before RoPE, k_old: cached keys encoded at p_old, both [m, Hkv, D]
    values; p_old, p_new: [m] positions.
    """
    a = rope_rotate(k_new, p_new, theta, style)
    b = rerotate(k_old, p_old, p_new, theta, style)
    d = a - b
    return (d * d).reshape(d.shape[0], int(np.prod(d.shape[1:]))).sum(axis=1)


def kv_deviation_fp64(k_new, k_old, v_new, v_old, p_old, p_new, theta: float, style: str = "half") -> np.ndarray:
    """K+V deviation per token in fp64: the key term plus the V term."""
    return key_deviation_fp64(k_new, k_old, p_old, p_new, theta, style) + deviation_fp64(v_new, v_old)


def _canonical_sum(parts) -> np.ndarray:
    """Canonical fp32 sum of squares of the per-element differences (list of [m, E] fp32 arrays)."""
    m = parts[0].shape[0]
    padded_parts = []
    for d in parts:
        e = d.shape[1]
        if e % 8:
            raise ValueError("Hkv*D must be a multiple of 8")
        pad = -(-e // 256) * 256 - e
        padded_parts.append(np.concatenate([d, np.zeros((m, pad), np.float32)], axis=1) if pad else d)
    d = np.concatenate(padded_parts, axis=1) if len(padded_parts) > 1 else padded_parts[0]
    # element e = (k*32 + lane)*8 + i  ->  axes (k, lane, i)
    d = d.reshape(m, d.shape[1] // 256, 32, 8)
    p = d * d
    acc = np.zeros((m, 32), dtype=np.float32)
    for k in range(p.shape[1]):
        for i in range(8):
            acc = acc + p[:, k, :, i]
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        acc = acc + acc[:, lanes ^ off]
    return acc[:, 0].copy()


def deviation_canonical_f32(v_new_bits: np.ndarray, v_old_bits: np.ndarray) -> np.ndarray:
    """fp32 deviation per token in the canonical order; inputs are bf16 bits [m, Hkv, D]."""
    m, e = v_new_bits.shape[0], int(np.prod(v_new_bits.shape[1:]))
    vn = _bf16_bits_to_f32(v_new_bits).reshape(m, e)
    vo = _bf16_bits_to_f32(v_old_bits).reshape(m, e)
    return _canonical_sum([vn - vo])


def rotate_f32(x: np.ndarray, cos_t: np.ndarray, sin_t: np.ndarray, style: str = "half") -> np.ndarray:
    """R x in fp32 per row from an fp32 table ([m, D/2] each), each product and sum rounded to fp32."""
    i0, i1 = pair_indices(x.shape[-1], style)
    c = cos_t[:, None, :]
    s = sin_t[:, None, :]
    x0, x1 = x[..., i0], x[..., i1]
    out = np.empty_like(x)
    out[..., i0] = (x0 * c) - (x1 * s)
    out[..., i1] = (x0 * s) + (x1 * c)
    return out


def kv_deviation_canonical_f32(k_new_bits, k_old_bits, v_new_bits, v_old_bits, p_old, theta: float,
                               style: str = "half") -> np.ndarray:
    """fp32 K+V deviation per token in the canonical order; bf16 bits [m, Hkv, D], p_old [m]."""
    m, hkv, d = k_new_bits.shape
    cos_t, sin_t = rope_table_f32(p_old, d, theta)
    kn = _bf16_bits_to_f32(k_new_bits).reshape(m, hkv, d)
    ko = _bf16_bits_to_f32(k_old_bits).reshape(m, hkv, d)
    e = hkv * d
    dk = (rotate_f32(kn, cos_t, sin_t, style) - ko).reshape(m, e)
    dv = _bf16_bits_to_f32(v_new_bits).reshape(m, e) - _bf16_bits_to_f32(v_old_bits).reshape(m, e)
    return _canonical_sum([dk, dv])

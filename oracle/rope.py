"""RoPE encoding and re-rotation of cached keys, in fp64.

"数学推导" §RoPE 位置编码的相对位置不变性证明: a query or key at position m is
rotated pair by pair, q~_m = R_m q_m, with the 2x2 rotation
R = [[cos a, -sin a], [sin a, cos a]]. The angle of pair j at position p is
p * theta^(-2j/D) (RoFormer, which that page cites).

"数学推导" §CacheBlend 中的应用: a key cached at p_old is moved to p_new by
k_new = R_{p_new} R_{p_old}^-1 k_old = R_{p_new - p_old} k_old.

Which two of the D coordinates form pair j is not fixed by the pages:
  "half"        pairs (j, j + D/2)   (the GPT-NeoX / Llama / Mistral layout; default)
  "interleaved" pairs (2j, 2j + 1)
"""

from __future__ import annotations

import math

import numpy as np

STYLES = ("half", "interleaved")


def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2j/D) for j = 0 .. D/2 - 1, fp64."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * j / head_dim)


def pair_indices(head_dim: int, style: str):
    """The two coordinate indices of each rotation pair."""
    half = head_dim // 2
    j = np.arange(half)
    if style == "half":
        return j, j + half
    if style == "interleaved":
        return 2 * j, 2 * j + 1
    raise ValueError(f"unknown RoPE style {style!r}")


def rope_rotate(x: np.ndarray, pos, theta: float, style: str = "half") -> np.ndarray:
    """Apply R_pos to every row of x [n, H, D]; pos is a scalar or [n] (may be negative)."""
    x = np.asarray(x, dtype=np.float64)
    n, _, d = x.shape
    pos = np.broadcast_to(np.asarray(pos, dtype=np.float64), (n,))
    angle = pos[:, None] * inv_freq(d, theta)[None, :]          # [n, D/2]
    c = np.cos(angle)[:, None, :]                                 # [n, 1, D/2]
    s = np.sin(angle)[:, None, :]
    i0, i1 = pair_indices(d, style)
    x0, x1 = x[..., i0], x[..., i1]
    out = np.empty_like(x)
    out[..., i0] = c * x0 - s * x1
    out[..., i1] = s * x0 + c * x1
    return out


def rerotate(k_old: np.ndarray, p_old, p_new, theta: float, style: str = "half") -> np.ndarray:
    """Move keys encoded at p_old to p_new: R_{p_new - p_old} k_old."""
    delta = np.asarray(p_new, dtype=np.int64) - np.asarray(p_old, dtype=np.int64)
    return rope_rotate(k_old, delta, theta, style)


def rope_table_f32(positions, head_dim: int, theta: float):
    """fl32(cos a), fl32(sin a) of every pair j at every given position, [n, D/2] each.

    a = fl64(p * fl64(theta^(-2j/D))) with the exponent formed as (-2 j) / D
    in fp64, and theta^x, cos and sin from the C library's fp64 routines
    (Python's math module calls them one value at a time). The result is the
    per-pair rotation that fp32 RoPE arithmetic starts from; where a
    computation must be reproduced bit for bit in fp32, it starts here.
    """
    pos = [int(p) for p in np.asarray(positions).reshape(-1)]
    half = head_dim // 2
    inv = [math.pow(float(theta), (-2.0 * j) / head_dim) for j in range(half)]
    cos_t = np.empty((len(pos), half), np.float32)
    sin_t = np.empty((len(pos), half), np.float32)
    cache = {}
    for r, p in enumerate(pos):
        row = cache.get(p)
        if row is None:
            ang = [float(p) * f for f in inv]
            row = (np.array([math.cos(a) for a in ang], np.float64).astype(np.float32),
                   np.array([math.sin(a) for a in ang], np.float64).astype(np.float32))
            cache[p] = row
        cos_t[r], sin_t[r] = row
    return cos_t, sin_t


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits: with x = m * 2^e and 0.5 <= |m| < 1, the
    result is rint(m * 2^8) * 2^(e - 8). Values below the bf16 normal range
    (|x| < 2^-126) are outside what this oracle is used for.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)

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
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def deviation_fp64(v_new: np.ndarray, v_old: np.ndarray) -> np.ndarray:
    """sum over heads and dims of (v_new - v_old)^2 per token, in fp64 (plain order)."""
    d = np.asarray(v_new, dtype=np.float64) - np.asarray(v_old, dtype=np.float64)
    return (d * d).reshape(d.shape[0], -1).sum(axis=1)


def deviation_canonical_f32(v_new_bits: np.ndarray, v_old_bits: np.ndarray) -> np.ndarray:
    """fp32 deviation per token in the canonical order; inputs are bf16 bits [m, Hkv, D]."""
    m = v_new_bits.shape[0]
    vn = _bf16_bits_to_f32(v_new_bits).reshape(m, -1)
    vo = _bf16_bits_to_f32(v_old_bits).reshape(m, -1)
    e = vn.shape[1]
    if e % 8:
        raise ValueError("Hkv*D must be a multiple of 8")
    padded = -(-e // 256) * 256
    if padded != e:
        vn = np.concatenate([vn, np.zeros((m, padded - e), np.float32)], axis=1)
        vo = np.concatenate([vo, np.zeros((m, padded - e), np.float32)], axis=1)
    # element e = (k*32 + lane)*8 + i  ->  axes (k, lane, i)
    d = (vn - vo).reshape(m, padded // 256, 32, 8)
    p = d * d
    acc = np.zeros((m, 32), dtype=np.float32)
    for k in range(p.shape[1]):
        for i in range(8):
            acc = acc + p[:, k, :, i]
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        acc = acc + acc[:, lanes ^ off]
    return acc[:, 0].copy()

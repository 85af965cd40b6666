"""Quality diagnostics of the blend: the attention deviation it minimises and attention sparsity.

"数学推导" §形式化 states the goal of the selection S as the attention deviation
    || Attention(Q, K_fused, V_fused) - Attention(Q, K_new, V_new) ||,
where K_new, V_new are the cache of a full prefill: every recomputed key encoded
at its global position, every recomputed value. Read here as the Frobenius norm
over all query rows of the layer (Q: every token's query, encoded at its
position, causal attention); the norm of the full-prefill output is returned
beside it for a relative figure.

"数学推导" §注意力稀疏性的量化分析 defines, for the attention weights
A in R^{n x n}, Sparsity(A, eps) = |{(i, j): A_ij < eps}| / n^2. A is the causal
softmax matrix of one head (entries above the diagonal are 0 and count when
eps > 0); over several heads the counts and the n^2 add up. Whether an entry
lies below eps is decided by floating point, so ``attention_sparsity`` also
returns how many entries lie within a relative band of eps, where another
correct evaluation (fp32 scores, a different summation order) may decide the
other way.
"""

from __future__ import annotations

import numpy as np

from .attention import causal_gqa_attention
from .deviation import bf16_bits_to_f64
from .rope import rope_rotate, round_bf16


def full_prefill_cache(cfg, inp, style: str = "half"):
    """K_new, V_new of a full prefill: all n_tokens recomputed rows, keys encoded at p_new = i."""
    n = cfg.n_tokens
    k_full = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new), np.arange(n), cfg.rope_theta, style))
    return k_full, bf16_bits_to_f64(inp.v_new)


def all_queries(cfg, inp, style: str = "half"):
    """Every token's query encoded at its position (bf16 values), [n_tokens, Hq, D]."""
    return round_bf16(rope_rotate(bf16_bits_to_f64(inp.q), np.arange(cfg.n_tokens), cfg.rope_theta, style))


def attention_deviation(o, o_ref):
    """(||o - o_ref||_F, ||o_ref||_F) in fp64."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    return float(np.sqrt(np.sum((o - o_ref) ** 2))), float(np.sqrt(np.sum(o_ref ** 2)))


def attention_sparsity(q, q_pos, k, eps: float, scale: float | None = None, band: float = 1e-3,
                       per_row: bool = False):
    """Count of causal attention weights below eps over rows q_pos and keys 0..n_keys-1.

    q [mq, Hq, D] (encoded), k [n_keys, Hkv, D]. Returns (count, near, total): count of
    entries A_ij < eps (masked entries are 0), entries with |A_ij - eps| <= band * eps,
    and total = Hq * mq * n_keys; with per_row, also the [mq, Hq] arrays of both counts.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    mq, hq, d = q.shape
    n, hkv, _ = k.shape
    group = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    visible = np.arange(n)[None, :] <= q_pos[:, None]
    rows_count = np.zeros((mq, hq), dtype=np.int64)
    rows_near = np.zeros((mq, hq), dtype=np.int64)
    for h in range(hq):
        s = (q[:, h, :] @ k[:, h // group, :].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        a = np.exp(s)
        a = a / a.sum(axis=1, keepdims=True)
        rows_count[:, h] = np.sum(a < eps, axis=1)
        rows_near[:, h] = np.sum(np.abs(a - eps) <= band * eps, axis=1)
    out = (int(rows_count.sum()), int(rows_near.sum()), hq * mq * n)
    return out + (rows_count, rows_near) if per_row else out


def blend_diagnostics(cfg, inp, res, eps: float, style: str = "half"):
    """Deviation of the layer's fused cache from a full prefill, and the full prefill's sparsity.

    res: the layer's ``blend.LayerResult`` (its k_fused / v_fused). Returns a dict with
    dev, ref (Frobenius norms), and the sparsity count / near / total.
    """
    n = cfg.n_tokens
    k_full, v_full = full_prefill_cache(cfg, inp, style)
    q_all = all_queries(cfg, inp, style)
    pos = np.arange(n)
    o_full = causal_gqa_attention(q_all, pos, k_full, v_full)
    o_fused = causal_gqa_attention(q_all, pos, res.k_fused, res.v_fused)
    dev, ref = attention_deviation(o_fused, o_full)
    count, near, total = attention_sparsity(q_all, pos, k_full, eps)
    return {"dev": dev, "ref": ref, "count": count, "near": near, "total": total,
            "o_full": o_full, "o_fused": o_fused}

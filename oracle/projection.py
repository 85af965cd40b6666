"""The step before the blend: the QKV projection of the rows a layer recomputes.

"rag的kvcache问题" §阶段一 (QKV 矩阵的生成): each token's q, k, v is its hidden vector
times the projection weights, row by row, computed in practice as one product of the
stacked rows X [N, d] with W. "rag的kvcache问题" §渐进式过滤机制: at layer l only the
candidate tokens (and the query suffix) are recomputed, so the rows of X are the
candidates' rows. Read here with one fused weight W_qkv [(Hq + 2 Hkv) D, d] (an
nn.Linear weight: one output feature per row), output features ordered Q heads, K
heads, V heads; optional RoPE encoding of q and k at each token's position
("数学推导" §RoPE 位置编码的相对位置不变性证明), applied to the fp64 product.
Results are rounded once to bf16.
"""

from __future__ import annotations

import numpy as np

from .rope import rope_rotate, round_bf16


def qkv_projection(x, rows, w, hq: int, hkv: int, head_dim: int, theta: float, encode: bool,
                   style: str = "half"):
    """q [m, Hq, D], k [m, Hkv, D], v [m, Hkv, D] (bf16 values) of the token rows `rows` of x."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    y = x[rows] @ w.T                                   # [m, (Hq + 2 Hkv) D]
    m = rows.size
    q = y[:, : hq * head_dim].reshape(m, hq, head_dim)
    k = y[:, hq * head_dim: (hq + hkv) * head_dim].reshape(m, hkv, head_dim)
    v = y[:, (hq + hkv) * head_dim:].reshape(m, hkv, head_dim)
    if encode:
        q = rope_rotate(q, rows, theta, style)
        k = rope_rotate(k, rows, theta, style)
    return round_bf16(q), round_bf16(k), round_bf16(v)

"""Causal grouped-query attention for a subset of query rows, in fp64.

"数学推导" §形式化 states the target Attention(Q, K_fused, V_fused);
"rag的kvcache问题" §渐进式过滤机制 hands the spliced cache to the layer's
self-attention. The same page (§transformer训练与推理并行计算的差异) fixes the
causal mask: a token sees only tokens before it (and itself), masked with -inf
before the softmax. §阶段二 of that page notes that row i of Q K^T needs only
q_i and all of K, so computing only the selected query rows is the same
computation restricted to those rows; rows are processed in blocks for memory
only. The softmax scale 1/sqrt(D) and the grouping "q head h reads kv head
h // (Hq/Hkv)" are the standard readings (the pages state neither).
"""

from __future__ import annotations

import numpy as np


def causal_gqa_attention(q, q_pos, k, v, scale: float | None = None, block: int = 256,
                         return_vscale: bool = False):
    """O[i, h] = sum_{j <= q_pos[i]} softmax_j(q[i,h] . k[j,g] * scale) v[j,g], g = h // G.

    q [mq, Hq, D], q_pos [mq]; k, v [N, Hkv, D] with key j at position j.
    With return_vscale, also returns sum_j softmax_j |v[j,g]| per output element:
    the magnitude that rounding the softmax weights multiplies (an error scale
    for comparisons, not part of the attention).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    mq, hq, d = q.shape
    n, hkv, _ = k.shape
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((mq, hq, d), dtype=np.float64)
    vscale = np.zeros((mq, hq, d), dtype=np.float64) if return_vscale else None
    for b0 in range(0, mq, block):
        b1 = min(mq, b0 + block)
        pos = q_pos[b0:b1]
        # keys past the block's last query are masked for every row of the block
        kend = min(n, int(pos.max()) + 1)
        visible = np.arange(kend)[None, :] <= pos[:, None]      # [b, kend]
        for h in range(hq):
            g = h // group
            s = (q[b0:b1, h, :] @ k[:kend, g, :].T) * scale
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[b0:b1, h, :] = p @ v[:kend, g, :]
            if return_vscale:
                vscale[b0:b1, h, :] = p @ np.abs(v[:kend, g, :])
    return (out, vscale) if return_vscale else out


def decode_attention(q, k, v, scale: float | None = None, return_vscale: bool = False):
    """One decode step ("rag的kvcache问题" §阶段 2 (Decode)): the newest token is the only query.

    Its query row q [Hq, D] (RoPE-encoded at its position n_keys - 1) attends over the whole
    cache k, v [n_keys, Hkv, D], whose last row is the newest token's own key and value, so
    no key is masked: O[h] = sum_{j < n_keys} softmax_j(q[h] . k[j, g] * scale) v[j, g].
    This is the causal attention above for the single row at position n_keys - 1.
    """
    q = np.asarray(q, dtype=np.float64)
    n = np.asarray(k).shape[0]
    if n < 1:
        raise ValueError("decode needs at least the newest token's own key")
    res = causal_gqa_attention(q[None], np.array([n - 1]), k, v, scale=scale, return_vscale=return_vscale)
    if return_vscale:
        return res[0][0], res[1][0]
    return res[0]

"""Fused KV of one layer.

"数学推导" §形式化: K_fused[i] = K_new[i] if i is in S, else K_old[i] (and
likewise for V). Here K_old is the cached key after re-rotation to its global
position, and K_new is the recomputed key encoded at its global position.
The query suffix has no cache, so its rows are always new
("rag的kvcache问题" §渐进式过滤机制: the recomputed rows are spliced into the
reused cache before the layer's attention).
"""

from __future__ import annotations

import numpy as np


def fused_kv(k_old_rot, v_old, k_new_enc, v_new, sel_tok, n_ctx: int):
    """Return (K_fused, V_fused, is_new) over all n_tokens rows.

    k_old_rot, v_old  [n_ctx, Hkv, D]     cached rows (K already at global positions)
    k_new_enc, v_new  [n_tokens, Hkv, D]  recomputed rows, indexed by token
    sel_tok           selected context token ids
    """
    n_tokens = k_new_enc.shape[0]
    is_new = np.zeros(n_tokens, dtype=bool)
    is_new[np.asarray(sel_tok, dtype=np.int64)] = True
    is_new[n_ctx:] = True
    k_f = np.where(is_new[:n_ctx, None, None], k_new_enc[:n_ctx], k_old_rot)
    v_f = np.where(is_new[:n_ctx, None, None], v_new[:n_ctx], v_old)
    k_f = np.concatenate([k_f, k_new_enc[n_ctx:]], axis=0)
    v_f = np.concatenate([v_f, v_new[n_ctx:]], axis=0)
    return k_f, v_f, is_new

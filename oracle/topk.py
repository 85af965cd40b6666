"""HKVD top-k selection and the gradual-filter budget.

"数学推导" §近似解: S = TopK_i ||V_new[i] - V_old[i]||_2^2, the k tokens of
largest V deviation. Ties are broken toward the lower token index. The
selection is returned in ascending token order together with each selected
token's row in the candidate list.
"""

from __future__ import annotations

import numpy as np


def hkvd_topk(dev: np.ndarray, cand: np.ndarray, k: int):
    """Select k of the m candidates.

    dev  [m] deviation per candidate (compared as given)
    cand [m] strictly ascending token ids
    Returns (sel_tok [k] ascending token ids, sel_row [k] indices into cand).
    """
    dev = np.asarray(dev)
    cand = np.asarray(cand, dtype=np.int64)
    m = dev.shape[0]
    if not 0 <= k <= m:
        raise ValueError(f"k={k} outside 0..{m}")
    # primary key: deviation, largest first; secondary key: token id, smallest first
    order = np.lexsort((cand, -dev))
    rows = np.sort(order[:k])
    return cand[rows], rows


def k_for_ratio(r_pct: int, n_ctx: int) -> int:
    """Budget of an r% filter: floor(r * n_ctx / 100) over the cached context tokens."""
    return (int(r_pct) * int(n_ctx)) // 100

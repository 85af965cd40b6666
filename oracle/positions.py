"""Token positions before and after the blend.

"rag的kvcache问题" §独立编码: each chunk's cache is computed alone, so its keys
carry chunk-local positions (taken here to start at 0 in every chunk). After
the chunks are concatenated, token i sits at global position i; the query
suffix follows the last chunk.
"""

from __future__ import annotations

import numpy as np


def global_positions(n_tokens: int) -> np.ndarray:
    """p_new[i] = i for every token of the request (chunks, then suffix)."""
    return np.arange(n_tokens, dtype=np.int64)


def chunk_local_positions(n_chunks: int, chunk_len: int) -> np.ndarray:
    """p_old[i] = i mod chunk_len for the cached context tokens."""
    return np.arange(n_chunks * chunk_len, dtype=np.int64) % chunk_len

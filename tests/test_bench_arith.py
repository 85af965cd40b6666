"""The bench's roofline arithmetic against independent counts on small shapes (CPU)."""

import dataclasses

import numpy as np

import bench
from workloads import get_config


def test_attention_flops_counts_visible_query_key_pairs():
    cfg = dataclasses.replace(get_config("tiny"), n_chunks=2, chunk_len=40, n_suffix=5, hq=4, hkv=2, head_dim=8)
    rng = np.random.default_rng(0)
    sel = np.sort(rng.choice(cfg.n_ctx, size=11, replace=False))
    q_pos = np.concatenate([sel, np.arange(cfg.n_ctx, cfg.n_tokens)])
    visible = np.arange(cfg.n_tokens)[None, :] <= q_pos[:, None]  # causal mask by global position
    # per visible (query, head, key): D multiply-adds for q.k and D for p v, two flops each
    want = int(visible.sum()) * cfg.hq * 2 * cfg.head_dim * 2
    assert bench.attention_flops(cfg, sel) == want


def test_stage_bytes_match_the_rows_the_kernels_move():
    cfg = get_config("mistral7b")
    row_kv = cfg.hkv * cfg.head_dim * 2
    row_q = cfg.hq * cfg.head_dim * 2
    n_cand, k = cfg.n_ctx, 921
    mq = k + cfg.n_suffix
    b = bench.stage_bytes(cfg, n_cand, k, mq, True)
    # deviation: one V_new and one V_old row per candidate
    assert b["deviation"] == n_cand * 2 * row_kv
    # fuse: every token's K and V row read once and written once, every query row read and written
    assert b["fuse"] == cfg.n_tokens * (2 * row_kv) * 2 + mq * row_q * 2
    assert bench.stage_bytes(cfg, n_cand, k, mq, True, "kv")["deviation"] == n_cand * 4 * row_kv
    assert bench.stage_bytes(cfg, k, k, mq, False)["deviation"] == 0.0


def test_whole_job_rate_and_slowest_rank():
    # value = all ranks' units / the slowest rank's time
    assert bench.whole_job_rate(1000, 4, 2.0) == 1000 * 4 / 2e-3

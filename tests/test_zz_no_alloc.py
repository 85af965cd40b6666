"""The allocation-free HKVD selection gives the oracle's tokens, and allocates nothing.

cb_hkvd_select_noalloc serves callers that cannot allocate device memory where
they pick tokens (for example a serving engine whose own pool owns all free
HBM, or a request path that must not pay cudaMalloc's device synchronisation):
it keeps its deviations in a fixed array inside the library instead of a
caller or plan buffer. Each result is compared with the oracle's canonical
deviation and top-k (oracle.deviation, oracle.topk), bit for bit, and with
cb_kv_deviation + cb_hkvd_topk; calls come in pairs on different problems, so
the second call reuses the array the first one filled. This file sorts last
so that a run stopping at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from oracle.deviation import deviation_canonical_f32
from oracle.topk import hkvd_topk
from workloads import get_config
from workloads.generator import bf16_bits_to_f32, f32_to_bf16_bits
from workloads.torch_io import bf16_tensor

pytestmark = pytest.mark.gpu

MAX_CANDIDATES = 65536  # CB_NOALLOC_MAX_CANDIDATES in include/cacheblend.h


def _problem(seed, n_rows, m, hkv, d, with_cand=True):
    """Seeded V caches with a wide spread of per-token deviations and exact ties (rows whose
    recomputed V equals the cached one have deviation 0; copied rows share a value)."""
    rng = np.random.default_rng(seed)
    old = rng.standard_normal((n_rows, hkv, d)).astype(np.float32)
    v_old = f32_to_bf16_bits(old)
    scale = np.exp(rng.uniform(-8, 1, size=(n_rows, 1, 1))).astype(np.float32)
    scale[rng.random(n_rows) < 0.05] = 0.0
    v_new = f32_to_bf16_bits(bf16_bits_to_f32(v_old) + scale * rng.standard_normal((n_rows, hkv, d)).astype(np.float32))
    dup = rng.choice(n_rows - 1, size=n_rows // 50, replace=False)
    v_new[dup + 1], v_old[dup + 1] = v_new[dup], v_old[dup]
    cand = np.sort(rng.choice(n_rows, size=m, replace=False)).astype(np.int32) if with_cand else None
    return v_new, v_old, cand


def _oracle(v_new, v_old, cand, m, k):
    rows = np.arange(m) if cand is None else cand.astype(np.int64)
    dev = deviation_canonical_f32(v_new[rows], v_old[rows])
    return hkvd_topk(dev, rows, k)


def _regular(cb, plan, v_new, v_old, cand, m, k):
    dev = torch.empty(m, dtype=torch.float32, device="cuda")
    st = torch.empty(k, dtype=torch.int32, device="cuda")
    sr = torch.empty(k, dtype=torch.int32, device="cuda")
    cb.cb_kv_deviation(plan, v_new, v_old, cand, m, dev)
    cb.cb_hkvd_topk(plan, dev, cand, m, k, st, sr)
    plan.check()
    return st.cpu().numpy(), sr.cpu().numpy()


def _noalloc(cb, v_new, v_old, cand, m, k, n_rows):
    st = torch.full((k,), -1, dtype=torch.int32, device="cuda")
    sr = torch.full((k,), -1, dtype=torch.int32, device="cuda")
    cb.cb_hkvd_select_noalloc(v_new, v_old, cand, m, k, n_rows, st, sr)
    return st.cpu().numpy(), sr.cpu().numpy()


def test_noalloc_selection_matches_oracle_and_regular_path_twice(cb):
    cfg = get_config("mistral7b")
    n_rows = cfg.n_ctx
    plan = cb.Plan.from_config(cfg)
    for seed, m, k in ((1, 3000, 921), (2, 1200, 460)):
        v_new, v_old, cand = _problem(seed, n_rows, m, cfg.hkv, cfg.head_dim)
        d_new, d_old, d_cand = bf16_tensor(v_new), bf16_tensor(v_old), torch.as_tensor(cand).cuda()
        tok, row = _noalloc(cb, d_new, d_old, d_cand, m, k, n_rows)
        want_tok, want_row = _oracle(v_new, v_old, cand, m, k)
        assert np.array_equal(tok, want_tok) and np.array_equal(row, want_row)
        reg_tok, reg_row = _regular(cb, plan, d_new, d_old, d_cand, m, k)
        assert np.array_equal(tok, reg_tok) and np.array_equal(row, reg_row)
    plan.close()


def test_noalloc_whole_array_without_candidate_list(cb):
    # m = CB_NOALLOC_MAX_CANDIDATES fills the whole array; cand = NULL means tokens 0 .. m - 1.
    hkv, d = 8, 128
    cfg = get_config("long32k")
    plan = cb.Plan.from_config(cfg)
    for seed, n_rows, m, k in ((3, MAX_CANDIDATES, MAX_CANDIDATES, 9830), (4, 40000, 32768, 4915)):
        v_new, v_old, _ = _problem(seed, n_rows, m, hkv, d, with_cand=False)
        d_new, d_old = bf16_tensor(v_new), bf16_tensor(v_old)
        tok, row = _noalloc(cb, d_new, d_old, None, m, k, n_rows)
        want_tok, want_row = _oracle(v_new, v_old, None, m, k)
        assert np.array_equal(tok, want_tok) and np.array_equal(row, want_row)
        if m <= cfg.n_ctx:  # the plan's path without a list takes at most its n_ctx tokens
            reg_tok, reg_row = _regular(cb, plan, d_new, d_old, None, m, k)
            assert np.array_equal(tok, reg_tok) and np.array_equal(row, reg_row)
    plan.close()


def test_noalloc_allocates_nothing(cb):
    n_rows, m, k, hkv, d = 8192, 8192, 1228, 8, 128
    v_new, v_old, cand = _problem(5, n_rows, m, hkv, d)
    d_new, d_old, d_cand = bf16_tensor(v_new), bf16_tensor(v_old), torch.as_tensor(cand).cuda()
    st = torch.empty(k, dtype=torch.int32, device="cuda")
    sr = torch.empty(k, dtype=torch.int32, device="cuda")
    cb.cb_hkvd_select_noalloc(d_new, d_old, d_cand, m, k, n_rows, st, sr)  # first call on the device
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for _ in range(3):
        cb.cb_hkvd_select_noalloc(d_new, d_old, d_cand, m, k, n_rows, st, sr)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0  # cudaMemGetInfo: no device memory taken
    want_tok, want_row = _oracle(v_new, v_old, cand, m, k)
    assert np.array_equal(st.cpu().numpy(), want_tok) and np.array_equal(sr.cpu().numpy(), want_row)


def test_noalloc_out_of_range_candidate_ranks_first(cb):
    # With no plan there is no error word: a candidate id past n_rows is skipped by the deviation
    # kernel's bounds check and gets a NaN deviation, which the top-k ranks above every number.
    n_rows, m, k, hkv, d = 4096, 2000, 300, 8, 128
    v_new, v_old, cand = _problem(6, n_rows, m, hkv, d)
    cand = cand.copy()
    cand[-1] = n_rows + 7  # still strictly ascending
    d_new, d_old, d_cand = bf16_tensor(v_new), bf16_tensor(v_old), torch.as_tensor(cand).cuda()
    tok, row = _noalloc(cb, d_new, d_old, d_cand, m, k, n_rows)
    dev = deviation_canonical_f32(v_new[cand[:-1]], v_old[cand[:-1]])
    want_tok, want_row = hkvd_topk(np.append(dev, np.float32(np.inf)), cand.astype(np.int64), k)
    assert np.array_equal(tok, want_tok) and np.array_equal(row, want_row)
    assert tok[-1] == n_rows + 7 and row[-1] == m - 1


def test_noalloc_rejects_more_candidates_than_its_array(cb):
    v = torch.zeros(70000, 1, 8, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_hkvd_select_noalloc(v, v, None, MAX_CANDIDATES + 1, 1, 70000, out, out)
    assert e.value.status == 1 and "65536" in str(e.value)

"""Pins of the oracle's HKVD top-k ("数学推导" §近似解) and the gradual-filter budget."""

import os

import numpy as np
import pytest

from oracle.blend import gradual_filter_schedule
from oracle.topk import hkvd_topk, k_for_ratio

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "topk_ties.txt")


def _golden():
    cand = dev = None
    rows = []
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        parts = [s.strip() for s in line.split("|")]
        if parts[0] == "cand":
            cand = np.array([int(v) for v in parts[1].split()])
        elif parts[0] == "dev":
            dev = np.array([float(v) for v in parts[1].split()], np.float32)
        else:
            rows.append((int(parts[0]), [int(v) for v in parts[1].split()], [int(v) for v in parts[2].split()]))
    return cand, dev, rows


def test_hand_worked_ties():
    cand, dev, rows = _golden()
    for k, tok, row in rows:
        st, sr = hkvd_topk(dev, cand, k)
        assert st.tolist() == tok and sr.tolist() == row


def _brute_force(dev, cand, k):
    # token t is selected iff fewer than k candidates outrank it, where u outranks t
    # when dev[u] > dev[t], or dev[u] == dev[t] and cand[u] < cand[t]
    m = len(dev)
    sel = []
    for t in range(m):
        rank = sum(1 for u in range(m) if dev[u] > dev[t] or (dev[u] == dev[t] and cand[u] < cand[t]))
        if rank < k:
            sel.append(t)
    return np.array(cand)[sel], np.array(sel, dtype=np.int64)


@pytest.mark.parametrize("seed", range(20))
def test_matches_rank_counting_with_forced_ties(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(1, 65))
    cand = np.sort(rng.choice(500, size=m, replace=False))
    dev = rng.choice(np.array([0.0, 0.25, 1.0, 1.5, 7.0], np.float32), size=m)
    for k in sorted({0, 1, m // 3, m // 2, m - 1 if m > 1 else 0, m}):
        st, sr = hkvd_topk(dev, cand, k)
        bt, br = _brute_force(dev, cand, k)
        assert st.tolist() == bt.tolist() and sr.tolist() == br.tolist()
        assert np.all(np.diff(st) > 0)


def test_all_equal_takes_lowest_ids():
    cand = np.arange(10, 40)
    st, _ = hkvd_topk(np.zeros(30, np.float32), cand, 7)
    assert st.tolist() == list(range(10, 17))


def test_k_bounds():
    with pytest.raises(ValueError):
        hkvd_topk(np.zeros(3, np.float32), np.arange(3), 4)


def test_budget_floor():
    assert k_for_ratio(15, 512) == 76
    assert k_for_ratio(30, 3072) == 921 and k_for_ratio(15, 3072) == 460
    assert k_for_ratio(30, 32768) == 9830 and k_for_ratio(15, 32768) == 4915
    assert k_for_ratio(20, 8192) == 1638 and k_for_ratio(10, 8192) == 819
    assert [k_for_ratio(r, 8192) for r in (5, 10, 15, 30, 50, 100)] == [409, 819, 1228, 2457, 4096, 8192]


def test_schedule_structure():
    s = gradual_filter_schedule(3072, 32, 30, 15)
    assert s[0] == (1, 921, True) and s[1] == (2, 460, True)
    assert all(x == (i + 3, 460, False) for i, x in enumerate(s[2:]))
    with pytest.raises(ValueError):
        gradual_filter_schedule(100, 3, 10, 20)

"""The allocation-free HKVD selection gives the same tokens as the regular path.

cb_hkvd_select_noalloc serves callers that cannot allocate device memory where
they pick tokens (for example a serving engine whose own pool owns all free
HBM, or a request path that must not pay cudaMalloc's device synchronisation):
it keeps its deviations in a fixed array inside the library instead of a
caller or plan buffer. Here it is called twice in a row on different problems
(so the second call reuses the array the first one filled) and each result is
compared with cb_kv_deviation + cb_hkvd_topk. This file sorts last so that a
run stopping at the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from workloads import get_config
from workloads.generator import bf16_bits_to_f32, f32_to_bf16_bits
from workloads.torch_io import bf16_tensor

pytestmark = pytest.mark.gpu


def _problem(seed, n_rows, m, hkv, d):
    rng = np.random.default_rng(seed)
    v_old = f32_to_bf16_bits(rng.standard_normal((n_rows, hkv, d)).astype(np.float32))
    scale = np.exp(rng.uniform(-8, 1, size=(n_rows, 1, 1))).astype(np.float32)
    v_new = f32_to_bf16_bits(bf16_bits_to_f32(v_old) + scale * rng.standard_normal((n_rows, hkv, d)).astype(np.float32))
    cand = np.sort(rng.choice(n_rows, size=m, replace=False)).astype(np.int32)
    return bf16_tensor(v_new), bf16_tensor(v_old), torch.as_tensor(cand).cuda()


def _regular(cb, plan, v_new, v_old, cand, m, k):
    dev = torch.empty(m, dtype=torch.float32, device="cuda")
    st = torch.empty(k, dtype=torch.int32, device="cuda")
    sr = torch.empty(k, dtype=torch.int32, device="cuda")
    cb.cb_kv_deviation(plan, v_new, v_old, cand, m, dev)
    cb.cb_hkvd_topk(plan, dev, cand, m, k, st, sr)
    return st.cpu().numpy(), sr.cpu().numpy()


def test_noalloc_selection_matches_regular_path_twice(cb):
    cfg = get_config("mistral7b")
    n_rows = cfg.n_ctx
    plan = cb.Plan.from_config(cfg)
    problems = [(_problem(1, n_rows, 3000, cfg.hkv, cfg.head_dim), 3000, 921),
                (_problem(2, n_rows, 1200, cfg.hkv, cfg.head_dim), 1200, 460)]
    for (v_new, v_old, cand), m, k in problems:
        st = torch.full((k,), -1, dtype=torch.int32, device="cuda")
        sr = torch.full((k,), -1, dtype=torch.int32, device="cuda")
        cb.cb_hkvd_select_noalloc(v_new, v_old, cand, m, k, n_rows, st, sr)
        want_tok, want_row = _regular(cb, plan, v_new, v_old, cand, m, k)
        assert np.array_equal(st.cpu().numpy(), want_tok)
        assert np.array_equal(sr.cpu().numpy(), want_row)
    plan.check()
    plan.close()


def test_noalloc_rejects_more_candidates_than_its_array(cb):
    v = torch.zeros(70000, 1, 8, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_hkvd_select_noalloc(v, v, None, 65537, 1, 70000, out, out)
    assert e.value.status == 1 and "65536" in str(e.value)

"""Quality diagnostics on the GPU against the oracle: attention sparsity ("数学推导"
§注意力稀疏性的量化分析) and the attention deviation of the fused cache from a full prefill
("数学推导" §形式化).

Sparsity counts are integers decided by floating point: per row, the GPU count may differ from
the oracle's only by weights the oracle finds within 1e-3 (relative) of eps.
"""

import dataclasses

import numpy as np
import pytest
import torch

from conftest import assert_close_attention
from oracle.attention import causal_gqa_attention
from oracle.blend import blend_layer
from oracle.deviation import bf16_bits_to_f64
from oracle.diagnostics import attention_sparsity, blend_diagnostics
from oracle.topk import k_for_ratio
from workloads import get_config
from workloads.generator import f32_to_bf16_bits, generate_layer
from workloads.torch_io import bf16_bits, bf16_tensor, layer_tensors

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _plan(cb, hq, hkv, d, n):
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1, chunk_len=max(n - 8, 8),
                              n_suffix=8)
    return cb.Plan.from_config(cfg)


def _gpu_sparsity(cb, plan, q, q_pos, k, v, n_keys, eps):
    mq, hq, d = q.shape
    out = torch.empty((mq, hq, d), dtype=torch.bfloat16, device="cuda")
    stats = torch.empty((mq, hq, 2), dtype=torch.float32, device="cuda")
    counts = torch.empty((mq, hq), dtype=torch.int32, device="cuda")
    total = torch.empty(1, dtype=torch.int64, device="cuda")
    cb.cb_attention_sparsity(plan, q, _i32(q_pos), mq, k, v, n_keys, eps, out, stats, counts, total)
    plan.check()
    return int(total.item()), counts.cpu().numpy(), stats.cpu().numpy(), out


@pytest.mark.parametrize("hq,hkv,d,n,rows", [(4, 2, 64, 300, "all"), (32, 8, 128, 1000, "all"),
                                             (64, 8, 128, 700, "sparse"), (16, 16, 64, 129, "all")])
@pytest.mark.parametrize("eps", [1e-3, 2e-2])
def test_sparsity_counts(cb, hq, hkv, d, n, rows, eps):
    rng = np.random.default_rng(n + hq)
    draw = lambda *s: f32_to_bf16_bits((2.0 * rng.standard_normal(s)).astype(np.float32))
    k, v = draw(n, hkv, d), draw(n, hkv, d)
    q_pos = np.arange(n) if rows == "all" else np.sort(rng.choice(n, size=n // 3, replace=False))
    q = draw(q_pos.size, hq, d)
    plan = _plan(cb, hq, hkv, d, n)
    total, counts, stats, out = _gpu_sparsity(cb, plan, bf16_tensor(q), q_pos, bf16_tensor(k), bf16_tensor(v), n, eps)
    qf, kf, vf = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    count, near, tot, rows_count, rows_near = attention_sparsity(qf, q_pos, kf, eps, per_row=True)
    assert np.all(np.abs(counts.astype(np.int64) - rows_count) <= rows_near)
    assert abs(total - count) <= near and near < 1e-3 * tot
    # the first pass is the plain attention, and its (max, sum) describe that softmax
    ref, vs = causal_gqa_attention(qf, q_pos, kf, vf, return_vscale=True)
    assert_close_attention(bf16_bits_to_f64(bf16_bits(out)), ref, vs)
    g = hq // hkv
    for i in (0, q_pos.size - 1):
        for h in (0, hq - 1):
            s2 = (qf[i, h] @ kf[: q_pos[i] + 1, h // g].T) / np.sqrt(d) / np.log(2.0)
            m, ssum = stats[i, h]
            np.testing.assert_allclose(np.sum(np.exp2(s2 - m)), ssum, rtol=2e-5)
    plan.close()


def test_output_deviation_reduction(cb):
    rng = np.random.default_rng(3)
    plan = _plan(cb, 32, 8, 128, 64)
    a = f32_to_bf16_bits(rng.standard_normal((777, 32, 128)).astype(np.float32))
    b = f32_to_bf16_bits(rng.standard_normal((777, 32, 128)).astype(np.float32))
    sums = torch.empty(2, dtype=torch.float64, device="cuda")
    cb.cb_output_deviation(plan, bf16_tensor(a), bf16_tensor(b), 777, sums)
    plan.check()
    af, bfv = bf16_bits_to_f64(a), bf16_bits_to_f64(b)
    np.testing.assert_allclose(sums.cpu().numpy(), [np.sum((af - bfv) ** 2), np.sum(bfv ** 2)], rtol=1e-12)
    plan.close()


def gpu_blend_diagnostics(cb, plan, cfg, bufs, t, eps):
    """The GPU side of the diagnostics for one blended layer (bufs: its LayerBuffers)."""
    n = cfg.n_tokens
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    k_full = torch.empty_like(bufs.k_fused)
    q_all = torch.empty((n, cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    cb.cb_rope_rerotate(plan, k_full, t["k_new"], pos)  # the full prefill's keys, at p = i
    cb.cb_rope_rerotate(plan, q_all, t["q"], pos)
    o_full = torch.empty_like(q_all)
    o_fused = torch.empty_like(q_all)
    cb.cb_hkvd_attention(plan, q_all, pos, n, bufs.k_fused, bufs.v_fused, n, o_fused)
    stats = torch.empty((n, cfg.hq, 2), dtype=torch.float32, device="cuda")
    counts = torch.empty((n, cfg.hq), dtype=torch.int32, device="cuda")
    total = torch.empty(1, dtype=torch.int64, device="cuda")
    cb.cb_attention_sparsity(plan, q_all, pos, n, k_full, t["v_new"], n, eps, o_full, stats, counts, total)
    sums = torch.empty(2, dtype=torch.float64, device="cuda")
    cb.cb_output_deviation(plan, o_fused, o_full, n, sums)
    plan.check()
    s = sums.cpu().numpy()
    return dict(dev=float(np.sqrt(s[0])), ref=float(np.sqrt(s[1])), count=int(total.item()),
                o_full=bf16_bits_to_f64(bf16_bits(o_full)), o_fused=bf16_bits_to_f64(bf16_bits(o_fused)))


@pytest.mark.parametrize("r", [15, 100])
def test_blend_diagnostics_match_the_oracle(cb, r):
    cfg = dataclasses.replace(get_config("mistral7b"), name="diag", config_id=94, n_chunks=4, chunk_len=120,
                              n_suffix=24, layers=1, r1_pct=r, r2_pct=r)
    inp = generate_layer(cfg, 1)
    t = layer_tensors(inp)
    plan = cb.Plan.from_config(cfg)
    bufs = cb.LayerBuffers(plan)
    cb.cb_blend_layer(plan, 1, cand=None, bufs=bufs, **t)
    eps = 1e-3
    g = gpu_blend_diagnostics(cb, plan, cfg, bufs, t, eps)
    res = blend_layer(cfg, inp, 1, np.arange(cfg.n_ctx), k_for_ratio(r, cfg.n_ctx), True, attention_rows=False)
    o = blend_diagnostics(cfg, inp, res, eps)
    # the reduction is the norm of the GPU's own outputs ...
    np.testing.assert_allclose(g["dev"], np.sqrt(np.sum((g["o_fused"] - g["o_full"]) ** 2)), rtol=1e-9, atol=1e-12)
    # ... which are the attention outputs within tolerance, so the norms differ at most by their errors
    bound = (np.sqrt(np.sum((g["o_fused"] - o["o_fused"]) ** 2)) + np.sqrt(np.sum((g["o_full"] - o["o_full"]) ** 2)))
    assert abs(g["dev"] - o["dev"]) <= bound + 1e-9
    assert abs(g["ref"] - o["ref"]) <= np.sqrt(np.sum((g["o_full"] - o["o_full"]) ** 2)) + 1e-9
    if r == 100:
        assert g["dev"] <= 1e-3 * g["ref"]  # same cache up to the two encoders' rounding
    else:
        assert g["dev"] > 0.01 * g["ref"]
    assert abs(g["count"] - o["count"]) <= o["near"]
    plan.close()

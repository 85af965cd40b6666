"""Decode attention ("rag的kvcache问题" §阶段 2 (Decode)) through the C ABI against the oracle.

The newest token's query row attends over the whole cache (its own key and value in the last
row). Outputs within 2e-2 * max(1, sum_j p_j |v_j|) + 1e-2 |ref| (bf16 output, fp32 softmax).
"""

import dataclasses

import numpy as np
import pytest
import torch

from conftest import assert_close_attention
from oracle.attention import decode_attention
from oracle.blend import blend_layer
from oracle.deviation import bf16_bits_to_f64
from workloads import get_config
from workloads.generator import f32_to_bf16_bits, generate_layer, hkvd_noise_sets
from workloads.torch_io import bf16_bits, bf16_tensor, layer_tensors

pytestmark = pytest.mark.gpu


def _plan(cb, hq, hkv, d, n_tokens=64):
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1, chunk_len=n_tokens - 8,
                              n_suffix=8)
    return cb.Plan.from_config(cfg)


def _draw(rng, *shape, scale=1.0):
    return f32_to_bf16_bits((scale * rng.standard_normal(shape)).astype(np.float32))


def _check(cb, plan, q, k, v, n_keys, scale=0.0, what="decode"):
    hq, d = q.shape
    out = torch.empty((hq, d), dtype=torch.bfloat16, device="cuda")
    cb.cb_decode_attention(plan, bf16_tensor(q), bf16_tensor(k), bf16_tensor(v), n_keys, out, scale=scale)
    plan.check()
    ref, vs = decode_attention(bf16_bits_to_f64(q), bf16_bits_to_f64(k[:n_keys]), bf16_bits_to_f64(v[:n_keys]),
                               scale=None if scale <= 0 else scale, return_vscale=True)
    assert_close_attention(bf16_bits_to_f64(bf16_bits(out)), ref, vs, what=what)
    return out


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (32, 8, 128), (64, 8, 128), (16, 16, 128), (32, 16, 64),
                                      (16, 1, 64), (32, 2, 128)])
@pytest.mark.parametrize("n_keys", [1, 7, 9, 33, 127, 128, 129, 256, 300, 3137])
def test_decode_shapes_and_lengths(cb, hq, hkv, d, n_keys):
    rng = np.random.default_rng(hq * 1000 + hkv * 10 + n_keys)
    plan = _plan(cb, hq, hkv, d)
    q = _draw(rng, hq, d, scale=1.5)
    k, v = _draw(rng, n_keys, hkv, d), _draw(rng, n_keys, hkv, d)
    _check(cb, plan, q, k, v, n_keys)
    plan.close()


def test_decode_long_cache_peaked_scores_and_repeat(cb):
    # 32,897 keys (the long-context workload plus one token) with a few keys far above the rest,
    # so the max moves late; a second call on the same plan reuses the split counters.
    rng = np.random.default_rng(4)
    hq, hkv, d, n = 32, 8, 128, 32897
    plan = _plan(cb, hq, hkv, d)
    q = _draw(rng, hq, d)
    k, v = _draw(rng, n, hkv, d), _draw(rng, n, hkv, d)
    kf = bf16_bits_to_f64(k)
    qf = bf16_bits_to_f64(q).reshape(hkv, hq // hkv, d)
    for j in (17, 20000, n - 1):  # keys aligned with their heads' queries
        k[j] = f32_to_bf16_bits((4.0 * qf.mean(axis=1) / np.linalg.norm(qf.mean(axis=1), axis=1, keepdims=True)
                                 * np.sqrt(d)).astype(np.float32))
    first = _check(cb, plan, q, k, v, n)
    second = _check(cb, plan, q, k, v, n)
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))
    _check(cb, plan, q, k, v, 5000, scale=0.05, what="decode (shorter cache, custom scale)")
    plan.close()


def test_decode_over_the_blended_cache(cb):
    # the step after the blend: layer 3 of the Mistral-7B-shaped request is blended on the GPU,
    # the first generated token's key and value are appended, and its query attends over it.
    cfg = get_config("mistral7b")
    sets = hkvd_noise_sets(cfg)
    plan = cb.Plan.from_config(cfg)
    rng = np.random.default_rng(8)
    inputs = [generate_layer(cfg, layer, sets) for layer in (1, 2, 3)]
    bufs = [cb.LayerBuffers(plan) for _ in range(3)]
    cand = None
    for li in range(3):
        cb.cb_blend_layer(plan, li + 1, cand=cand, bufs=bufs[li], **layer_tensors(inputs[li]))
        cand = bufs[li].sel_tok
    plan.check()
    new_k, new_v = _draw(rng, 1, cfg.hkv, cfg.head_dim), _draw(rng, 1, cfg.hkv, cfg.head_dim)
    q = _draw(rng, cfg.hq, cfg.head_dim)
    k_cache = torch.cat([bufs[2].k_fused, bf16_tensor(new_k)])
    v_cache = torch.cat([bufs[2].v_fused, bf16_tensor(new_v)])
    n = cfg.n_tokens + 1
    out = torch.empty((cfg.hq, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    cb.cb_decode_attention(plan, bf16_tensor(q), k_cache, v_cache, n, out)
    plan.check()
    # oracle: its own blend of the same layers, then the same appended row
    sel = np.arange(cfg.n_ctx)
    from oracle.blend import gradual_filter_schedule
    for (layer, k, selects), inp in zip(gradual_filter_schedule(cfg.n_ctx, 3, cfg.r1_pct, cfg.r2_pct), inputs):
        res = blend_layer(cfg, inp, layer, sel, k, selects, attention_rows=False)
        sel = res.sel_tok
    kc = np.concatenate([res.k_fused, bf16_bits_to_f64(new_k)])
    vc = np.concatenate([res.v_fused, bf16_bits_to_f64(new_v)])
    ref, vs = decode_attention(bf16_bits_to_f64(q), kc, vc, return_vscale=True)
    assert_close_attention(bf16_bits_to_f64(bf16_bits(out)), ref, vs, what="decode after blend")
    plan.close()


def test_decode_rejects_bad_arguments(cb):
    plan = _plan(cb, 4, 2, 64)
    q = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((8, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cb.CacheBlendError):
        cb.cb_decode_attention(plan, q, k, k, -1, q.clone())
    with pytest.raises(cb.CacheBlendError):
        cb.cb_decode_attention(plan, None, k, k, 8, q.clone())
    cb.cb_decode_attention(plan, q, k, k, 0, q.clone())  # nothing to do
    plan.close()

"""The attention kernel's failure path: a bounded wait that runs out is reported, and the
device stays usable.

cb_test_attention_wait_timeout runs the attention kernel in a form whose K-tile producer never
requests key tile 1 and whose waits give up after 100 us (a barrier that nothing completes, no
fault, trap or endless loop). Every CTA whose queries reach that tile must record CB_ERR_TIMEOUT
in the plan's error word, drain what it started, free its tensor memory and return; a normal
attention call right after must then give the oracle's result on the same SMs.
"""

import dataclasses
import time

import numpy as np
import pytest
import torch

from conftest import assert_close_bf16
from oracle.attention import causal_gqa_attention
from oracle.deviation import bf16_bits_to_f64
from workloads import get_config
from workloads.generator import f32_to_bf16_bits
from workloads.torch_io import bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu


def test_attention_wait_timeout_is_reported_and_the_device_stays_usable(cb):
    hq, hkv, d, n_keys = 32, 8, 128, 640
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1, chunk_len=n_keys - 1,
                              n_suffix=1)
    plan = cb.Plan.from_config(cfg)
    rng = np.random.default_rng(404)
    q_pos = np.sort(rng.choice(np.arange(128, n_keys), size=96, replace=False))  # every tile reaches key tile 1
    mq = q_pos.size
    q = f32_to_bf16_bits(rng.standard_normal((mq, hq, d)).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    dq, dk, dv = bf16_tensor(q), bf16_tensor(k), bf16_tensor(v)
    pos = torch.as_tensor(q_pos.astype(np.int32)).cuda()
    out = torch.zeros((mq, hq, d), dtype=torch.bfloat16, device="cuda")
    ref = causal_gqa_attention(bf16_bits_to_f64(q), q_pos, bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    for _ in range(2):  # the failure and the recovery, twice in a row
        t0 = time.perf_counter()
        cb.cb_test_attention_wait_timeout(plan, dq, pos, mq, dk, dv, n_keys, out)
        with pytest.raises(cb.CacheBlendError) as e:
            plan.check()  # synchronises: the kernel has returned
        assert e.value.status == 4 and "flags 0x8 " in str(e.value)
        assert time.perf_counter() - t0 < 30.0
        plan.check()  # the error word was read and cleared
        out.zero_()
        cb.cb_hkvd_attention(plan, dq, pos, mq, dk, dv, n_keys, out)
        plan.check()
        assert_close_bf16(bf16_bits_to_f64(bf16_bits(out)), ref, what="attention after a timed-out launch")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_test_attention_wait_timeout(plan, dq, pos, mq, dk, dv, 128, out)  # no key tile 1 to miss
    assert e.value.status == 1
    plan.close()


def test_decode_wait_timeout_is_reported_and_the_plan_stays_usable(cb):
    # cb_test_decode_wait_timeout: the decode kernel whose producer never copies key tile 1 of its
    # split and whose waits give up after 100 us. Every CTA with a second tile records the timeout,
    # drains, frees its tensor memory and still takes its ticket; a normal decode on the same plan
    # right after (same split counters) must then match the oracle.
    from oracle.attention import decode_attention

    hq, hkv, d, n_keys = 32, 8, 128, 3137
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1, chunk_len=n_keys - 1,
                              n_suffix=1)
    plan = cb.Plan.from_config(cfg)
    rng = np.random.default_rng(405)
    q = f32_to_bf16_bits(rng.standard_normal((hq, d)).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    dq, dk, dv = bf16_tensor(q), bf16_tensor(k), bf16_tensor(v)
    out = torch.zeros((hq, d), dtype=torch.bfloat16, device="cuda")
    ref = decode_attention(bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    for _ in range(2):  # the failure and the recovery, twice in a row
        t0 = time.perf_counter()
        cb.cb_test_decode_wait_timeout(plan, dq, dk, dv, n_keys, out)
        with pytest.raises(cb.CacheBlendError) as e:
            plan.check()
        assert e.value.status == 4 and "flags 0x8 " in str(e.value)
        assert time.perf_counter() - t0 < 30.0
        plan.check()
        out.zero_()
        cb.cb_decode_attention(plan, dq, dk, dv, n_keys, out)
        plan.check()
        assert_close_bf16(bf16_bits_to_f64(bf16_bits(out)), ref, what="decode after a timed-out launch")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_test_decode_wait_timeout(plan, dq, dk, dv, 128, out)  # no key tile 1 to miss
    assert e.value.status == 1
    plan.close()


def test_projection_wait_timeout_is_reported_and_the_device_stays_usable(cb):
    # cb_test_projection_wait_timeout: the CTA-pair projection kernel whose first CTA of each pair
    # never copies its share of K step 1 (the pair's barrier for it cannot complete) and whose
    # waits give up after 100 us. Both CTAs of every pair must record the timeout, drain, free
    # their tensor memory and meet at the cluster barrier; a normal projection right after must
    # match the oracle.
    from oracle.projection import qkv_projection
    from workloads.generator import generate_projection

    cfg = dataclasses.replace(get_config("tiny"), hq=8, hkv=2, head_dim=128, d_model=512, n_chunks=1, chunk_len=392,
                              n_suffix=8)
    plan = cb.Plan.from_config(cfg)
    m = 300  # three row tiles: two CTA pairs, one of them half past m
    x, w = generate_projection(cfg, 3)
    dx, dw = bf16_tensor(x[:m]), bf16_tensor(w)
    shape = lambda h: (cfg.n_tokens, h, cfg.head_dim)
    q, k, v = (torch.zeros(shape(h), dtype=torch.bfloat16, device="cuda") for h in (cfg.hq, cfg.hkv, cfg.hkv))
    oq, ok, ov = qkv_projection(bf16_bits_to_f64(x), np.arange(m), bf16_bits_to_f64(w), cfg.hq, cfg.hkv,
                                cfg.head_dim, cfg.rope_theta, False)
    for _ in range(2):  # the failure and the recovery, twice in a row
        t0 = time.perf_counter()
        cb.cb_test_projection_wait_timeout(plan, dx, m, dw, q, k, v)
        with pytest.raises(cb.CacheBlendError) as e:
            plan.check()
        assert e.value.status == 4 and "flags 0x8 " in str(e.value)
        assert time.perf_counter() - t0 < 30.0
        plan.check()
        cb.cb_qkv_projection_indexed(plan, dx, None, None, m, dw, q, k, v)
        plan.check()
        for got, want, what in ((q, oq, "q"), (k, ok, "k"), (v, ov, "v")):
            assert_close_bf16(bf16_bits_to_f64(bf16_bits(got[:m])), want, what=f"projection {what} after a timeout")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_test_projection_wait_timeout(plan, bf16_tensor(x[:m, :64].copy()), m, bf16_tensor(w[:, :64].copy()),
                                           q, k, v)  # d_model 64: no K step 1 to miss
    assert e.value.status == 1
    plan.close()

"""Per-kernel parity of the CUDA library against the CPU oracle, through the C ABI.

Integer and byte results (deviation bits, selected sets, copied V rows) are
compared bit for bit; rotated keys and attention outputs within
2e-2 absolute + 1e-2 relative (bf16 storage, fp32 accumulation).
"""

import dataclasses

import numpy as np
import pytest
import torch

from conftest import assert_close_bf16
from oracle.attention import causal_gqa_attention
from oracle.deviation import bf16_bits_to_f64, deviation_canonical_f32, kv_deviation_canonical_f32
from oracle.rope import rerotate, rope_rotate, round_bf16
from oracle.topk import hkvd_topk
from workloads import get_config
from workloads.generator import f32_to_bf16_bits, generate_layer
from workloads.torch_io import bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _shape(name, **kw):
    return dataclasses.replace(get_config(name), **kw)


def _plan(cb, cfg, style="half", r1=None, r2=None):
    return cb.Plan.from_config(cfg, rope_style=style, r1_pct=r1, r2_pct=r2)


# ---------------------------------------------------------------- rotation
@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("name", ["tiny", "mistral7b", "llama70b"])
def test_rerotate_cached_keys(cb, name, style):
    cfg = get_config(name)
    if name != "tiny":
        cfg = dataclasses.replace(cfg, n_chunks=3, chunk_len=200, n_suffix=40)
    plan = _plan(cb, cfg, style)
    inp = generate_layer(cfg, 1)
    n_ctx = cfg.n_ctx
    p_old = np.arange(n_ctx) % cfg.chunk_len
    p_new = np.arange(n_ctx)
    x = bf16_tensor(inp.k_old)
    out = torch.zeros_like(x)
    cb.cb_rope_rerotate(plan, out, x, _i32(p_new), pos_from=_i32(p_old))
    plan.check()
    ref = round_bf16(rerotate(bf16_bits_to_f64(inp.k_old), p_old, p_new, cfg.rope_theta, style))
    got = bf16_bits_to_f64(bf16_bits(out))
    assert_close_bf16(got, ref, what="re-rotated keys")
    assert np.mean(got == ref) > 0.99  # fp32 math vs fp64: at most rare 1-ulp differences
    # chunk 0 has delta 0: the bytes are copied unchanged
    assert np.array_equal(bf16_bits(out)[: cfg.chunk_len], inp.k_old[: cfg.chunk_len])


def test_encode_in_place_and_negative_delta(cb):
    cfg = get_config("tiny")
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(11)
    bits = f32_to_bf16_bits(rng.standard_normal((300, 4, 64)).astype(np.float32))
    pos = rng.integers(0, cfg.n_tokens, size=300)
    x = bf16_tensor(bits)
    cb.cb_rope_rerotate(plan, x, x, _i32(pos))  # in place, encode at pos
    ref = round_bf16(rope_rotate(bf16_bits_to_f64(bits), pos, cfg.rope_theta))
    assert_close_bf16(bf16_bits_to_f64(bf16_bits(x)), ref, what="encode in place")
    # rotating back by -pos recovers the input within bf16 rounding
    back = torch.empty_like(x)
    cb.cb_rope_rerotate(plan, back, x, _i32(np.zeros(300)), pos_from=_i32(pos))
    plan.check()
    assert_close_bf16(bf16_bits_to_f64(bf16_bits(back)), bf16_bits_to_f64(bits), what="inverse rotation")


def test_gather_scatter_rows_and_range_check(cb):
    cfg = get_config("tiny")
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(12)
    src = f32_to_bf16_bits(rng.standard_normal((50, 2, 64)).astype(np.float32))
    x = bf16_tensor(src)
    out = torch.zeros(80, 2, 64, dtype=torch.bfloat16, device="cuda")
    in_rows = rng.choice(50, 20, replace=False)
    out_rows = rng.choice(80, 20, replace=False)
    pos = rng.integers(0, 500, 20)
    cb.cb_rope_rerotate(plan, out, x, _i32(pos), in_rows=_i32(in_rows), out_rows=_i32(out_rows))
    plan.check()
    got = bf16_bits_to_f64(bf16_bits(out))
    ref = round_bf16(rope_rotate(bf16_bits_to_f64(src[in_rows]), pos, cfg.rope_theta))
    assert_close_bf16(got[out_rows], ref, what="gathered rows")
    untouched = np.setdiff1d(np.arange(80), out_rows)
    assert np.all(got[untouched] == 0)
    # a delta beyond the table and a row beyond the tensor are skipped and reported
    bad_pos = pos.copy()
    bad_pos[3] = cfg.n_tokens + 5
    bad_in = in_rows.copy()
    bad_in[7] = 50
    before = bf16_bits(out).copy()
    cb.cb_rope_rerotate(plan, out, x, _i32(bad_pos), in_rows=_i32(bad_in), out_rows=_i32(out_rows))
    with pytest.raises(cb.CacheBlendError) as e:
        plan.check()
    assert e.value.status == 5
    after = bf16_bits(out)
    assert np.array_equal(after[out_rows[3]], before[out_rows[3]])
    assert np.array_equal(after[out_rows[7]], before[out_rows[7]])
    plan.check()  # the error word was cleared


# ---------------------------------------------------------------- deviation
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (16, 128), (1, 64), (3, 64)])
def test_deviation_bit_exact(cb, hkv, d):
    cfg = dataclasses.replace(get_config("tiny"), hkv=hkv, hq=hkv * 2, head_dim=d, n_chunks=4, chunk_len=333)
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(hkv * 100 + d)
    n_ctx = cfg.n_ctx
    v_old = f32_to_bf16_bits(rng.standard_normal((n_ctx, hkv, d)).astype(np.float32))
    scale = np.exp(rng.uniform(-9, 1, size=(n_ctx, 1, 1))).astype(np.float32)
    v_new = np.concatenate([
        f32_to_bf16_bits((v_old.astype(np.uint32) << 16).view(np.float32)
                         + scale * rng.standard_normal((n_ctx, hkv, d)).astype(np.float32)),
        f32_to_bf16_bits(rng.standard_normal((cfg.n_suffix, hkv, d)).astype(np.float32))])
    v_new[5] = v_old[5]  # an exact-zero deviation
    cand = np.sort(rng.choice(n_ctx, size=n_ctx // 3, replace=False))
    dev = torch.empty(cand.size, dtype=torch.float32, device="cuda")
    cb.cb_kv_deviation(plan, bf16_tensor(v_new), bf16_tensor(v_old), _i32(cand), cand.size, dev)
    ref = deviation_canonical_f32(v_new[cand], v_old[cand])
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # identity candidate list
    dev_all = torch.empty(n_ctx, dtype=torch.float32, device="cuda")
    cb.cb_kv_deviation(plan, bf16_tensor(v_new), bf16_tensor(v_old), None, n_ctx, dev_all)
    plan.check()
    ref_all = deviation_canonical_f32(v_new[:n_ctx], v_old)
    assert np.array_equal(dev_all.cpu().numpy().view(np.uint32), ref_all.view(np.uint32))
    assert dev_all[5].item() == 0.0


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (16, 128), (3, 64)])
def test_kv_deviation_bit_exact(cb, hkv, d, style):
    # K+V deviation: the recomputed key turned to p_old = t mod chunk_len (chunk_len 333, so the
    # table rows differ from the token ids) in fp32 from the plan's table, then the canonical sum.
    cfg = dataclasses.replace(get_config("tiny"), hkv=hkv, hq=hkv * 2, head_dim=d, n_chunks=4, chunk_len=333)
    plan = _plan(cb, cfg, style)
    rng = np.random.default_rng(hkv * 100 + d + (style == "half"))
    n_ctx, n = cfg.n_ctx, cfg.n_tokens
    draw = lambda rows, sc=1.0: f32_to_bf16_bits((sc * rng.standard_normal((rows, hkv, d))).astype(np.float32))
    k_old, v_old = draw(n_ctx), draw(n_ctx)
    scale = np.exp(rng.uniform(-9, 1, size=(n, 1, 1))).astype(np.float32)
    k_new = f32_to_bf16_bits(np.concatenate([(k_old.astype(np.uint32) << 16).view(np.float32),
                                             np.zeros((cfg.n_suffix, hkv, d), np.float32)])
                             + scale * rng.standard_normal((n, hkv, d)).astype(np.float32))
    v_new = draw(n)
    v_new[7] = v_old[7]
    cand = np.sort(rng.choice(n_ctx, size=n_ctx // 3, replace=False))
    dev = torch.empty(cand.size, dtype=torch.float32, device="cuda")
    cb.cb_kv_deviation_kv(plan, bf16_tensor(k_new), bf16_tensor(k_old), bf16_tensor(v_new), bf16_tensor(v_old),
                          _i32(cand), cand.size, dev)
    plan.check()
    ref = kv_deviation_canonical_f32(k_new[cand], k_old[cand], v_new[cand], v_old[cand], cand % cfg.chunk_len,
                                     cfg.rope_theta, style)
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # identity candidate list, and a token whose key part is exactly zero (p_old = 0, same key)
    k_new[0] = k_old[0]
    dev_all = torch.empty(n_ctx, dtype=torch.float32, device="cuda")
    cb.cb_kv_deviation_kv(plan, bf16_tensor(k_new), bf16_tensor(k_old), bf16_tensor(v_new), bf16_tensor(v_old),
                          None, n_ctx, dev_all)
    plan.check()
    ref_all = kv_deviation_canonical_f32(k_new[:n_ctx], k_old, v_new[:n_ctx], v_old,
                                         np.arange(n_ctx) % cfg.chunk_len, cfg.rope_theta, style)
    assert np.array_equal(dev_all.cpu().numpy().view(np.uint32), ref_all.view(np.uint32))
    assert dev_all[0].item() == float(deviation_canonical_f32(v_new[:1], v_old[:1])[0])


def test_deviation_golden_rounding_cases(cb):
    # the hand-derived cases that pin the summation order, run on the GPU
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "deviation_rounding.txt")
    cfg = dataclasses.replace(get_config("tiny"), hkv=4, hq=8, head_dim=128)
    plan = _plan(cb, cfg)
    for line in open(path, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, e, entries, expect = (s.strip() for s in line.split("|"))
        vn = np.zeros(512, np.float32)
        vo = np.zeros(512, np.float32)
        for ent in entries.split():
            i, a, b = ent.split(":")
            vn[int(i)] = float.fromhex(a) if "x" in a else float(a)
            vo[int(i)] = float.fromhex(b) if "x" in b else float(b)
        dev = torch.empty(1, dtype=torch.float32, device="cuda")
        cb.cb_kv_deviation(plan, bf16_tensor(f32_to_bf16_bits(vn).reshape(1, 4, 128)),
                           bf16_tensor(f32_to_bf16_bits(vo).reshape(1, 4, 128)), None, 1, dev)
        assert dev.item() == float.fromhex(expect), name


# ---------------------------------------------------------------- top-k
@pytest.mark.parametrize("m", [1, 7, 64, 256, 257, 1000, 1024, 1025, 3072, 4096, 4097, 32768, 40000])
def test_topk_bit_exact_with_ties(cb, m):
    plan = _plan(cb, get_config("tiny"))
    rng = np.random.default_rng(m)
    cand = np.sort(rng.choice(max(2 * m, 10), size=m, replace=False))
    pools = [rng.choice(np.array([0.0, 0.5, 1.0, 3.0], np.float32), size=m),
             rng.standard_normal(m).astype(np.float32) ** 2,
             np.zeros(m, np.float32)]
    for dev in pools:
        for k in sorted({1, m // 7, m // 2, m - 1, m} - {0}):
            d = torch.as_tensor(dev).cuda()
            st = torch.full((k,), -1, dtype=torch.int32, device="cuda")
            sr = torch.full((k,), -1, dtype=torch.int32, device="cuda")
            cb.cb_hkvd_topk(plan, d, _i32(cand), m, k, st, sr)
            rt, rr = hkvd_topk(dev, cand, k)
            assert np.array_equal(st.cpu().numpy(), rt) and np.array_equal(sr.cpu().numpy(), rr), (m, k)
    plan.check()


def test_topk_lognormal_near_ties(cb):
    # the ratio-sweep noise model: per-token scales spread over decades, so the
    # selection boundary falls among closely spaced deviations
    cfg = get_config("sweep")
    inp = generate_layer(cfg, 1)
    plan = _plan(cb, cfg, r1=100, r2=100)
    n = cfg.n_ctx
    dev = torch.empty(n, dtype=torch.float32, device="cuda")
    cb.cb_kv_deviation(plan, bf16_tensor(inp.v_new), bf16_tensor(inp.v_old), None, n, dev)
    ref_dev = deviation_canonical_f32(inp.v_new[:n], inp.v_old)
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), ref_dev.view(np.uint32))
    for r in cfg.sweep_pct:
        k = r * n // 100
        st = torch.empty(k, dtype=torch.int32, device="cuda")
        sr = torch.empty(k, dtype=torch.int32, device="cuda")
        cb.cb_hkvd_topk(plan, dev, None, n, k, st, sr)
        rt, _ = hkvd_topk(ref_dev, np.arange(n), k)
        assert np.array_equal(st.cpu().numpy(), rt), r
    plan.check()


# ---------------------------------------------------------------- fuse / scatter
@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_fuse_scatter(cb, style):
    cfg = get_config("tiny")
    plan = _plan(cb, cfg, style)
    inp = generate_layer(cfg, 1)
    rng = np.random.default_rng(5)
    sel = np.sort(rng.choice(cfg.n_ctx, 76, replace=False))
    kf = bf16_tensor(np.zeros((cfg.n_tokens, 2, 64), np.uint16))
    vf = bf16_tensor(np.zeros((cfg.n_tokens, 2, 64), np.uint16))
    cb.cb_fuse_scatter(plan, kf, vf, bf16_tensor(inp.k_new), bf16_tensor(inp.v_new), _i32(sel), sel.size)
    plan.check()
    rows = np.concatenate([sel, np.arange(cfg.n_ctx, cfg.n_tokens)])
    others = np.setdiff1d(np.arange(cfg.n_tokens), rows)
    kb, vb = bf16_bits(kf), bf16_bits(vf)
    assert np.array_equal(vb[rows], inp.v_new[rows]) and np.all(vb[others] == 0) and np.all(kb[others] == 0)
    ref = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new[rows]), rows, cfg.rope_theta, style))
    assert_close_bf16(bf16_bits_to_f64(kb[rows]), ref, what="scattered keys")


# ---------------------------------------------------------------- attention
def _attention_case(cb, hq, hkv, d, n_keys, q_pos, seed, scale_q=1.0):
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=max(n_keys - 1, 1), n_suffix=1)
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(seed)
    mq = len(q_pos)
    q = f32_to_bf16_bits((scale_q * rng.standard_normal((mq, hq, d))).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    ref = causal_gqa_attention(bf16_bits_to_f64(q), q_pos, bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    return bf16_bits_to_f64(bf16_bits(out)), ref


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (32, 8, 128), (64, 8, 128), (8, 8, 128), (16, 1, 64)])
def test_attention_sparse_queries(cb, hq, hkv, d):
    rng = np.random.default_rng(hq + d)
    n_keys = 1000
    q_pos = np.sort(rng.choice(n_keys, size=150, replace=False))
    got, ref = _attention_case(cb, hq, hkv, d, n_keys, q_pos, seed=hq * 7 + d)
    assert_close_bf16(got, ref, what=f"attention hq={hq} hkv={hkv} d={d}")


@pytest.mark.parametrize("n_keys", [1, 2, 127, 128, 129, 300, 2049])
def test_attention_all_positions(cb, n_keys):
    # every position queried: the full-recompute case (r = 100%)
    q_pos = np.arange(n_keys)
    got, ref = _attention_case(cb, 32, 8, 128, n_keys, q_pos, seed=n_keys)
    assert_close_bf16(got, ref, what=f"attention n_keys={n_keys}")


def test_attention_peaked_scores_force_rescale(cb):
    # large query norms make the running max jump between key tiles (O rescaling path)
    rng = np.random.default_rng(3)
    q_pos = np.sort(rng.choice(1500, size=100, replace=False))
    got, ref = _attention_case(cb, 8, 2, 64, 1500, q_pos, seed=9, scale_q=6.0)
    assert_close_bf16(got, ref, what="peaked attention")


def test_attention_score_jumps_between_key_tiles(cb):
    # Keys whose scores exceed everything earlier by far more than 2^64 (in base-2 units of the
    # scaled score), in both halves of the key tiles: the softmax must move its reference and
    # rescale what it accumulated instead of overflowing.
    hq, hkv, d, n_keys = 8, 2, 128, 1000
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=n_keys - 1, n_suffix=1)
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(21)
    q_pos = np.sort(np.concatenate([rng.choice(np.arange(0, 300), 20, replace=False),
                                    rng.choice(np.arange(300, 700), 40, replace=False),
                                    rng.choice(np.arange(700, n_keys), 40, replace=False)]))
    mq = q_pos.size
    q = f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal((mq, hq, d))).astype(np.float32))
    kf = rng.standard_normal((n_keys, hkv, d)).astype(np.float32)
    kf[300] = 6.0   # tile 2 (even tiles)
    kf[450] = 8.0   # tile 3 (odd tiles)
    kf[705] = 12.0  # tile 5 (odd tiles), far above the tile-3 spike
    k = f32_to_bf16_bits(kf)
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    ref = causal_gqa_attention(bf16_bits_to_f64(q), q_pos, bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    got = bf16_bits_to_f64(bf16_bits(out))
    assert np.all(np.isfinite(got))
    assert_close_bf16(got, ref, what="attention with score jumps")


def test_attention_first_tile_scores_far_below_zero(cb):
    # Rows whose scores in the first key tiles lie far below 0 (2^score would underflow fp32): the
    # softmax reference must follow the row max, not start from 0.
    hq, hkv, d, n_keys = 8, 2, 128, 600
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=n_keys - 1, n_suffix=1)
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(31)
    q_pos = np.sort(np.concatenate([rng.choice(np.arange(0, 128), 30, replace=False),
                                    rng.choice(np.arange(128, 256), 30, replace=False),
                                    rng.choice(np.arange(256, n_keys), 30, replace=False)]))
    mq = q_pos.size
    q = f32_to_bf16_bits((-1.0 - 0.05 * rng.standard_normal((mq, hq, d))).astype(np.float32))
    kf = rng.standard_normal((n_keys, hkv, d)).astype(np.float32)
    kf[:256] = 5.0 + 0.1 * kf[:256]  # tiles 0 and 1: scores near -640 (raw), far below 0
    k = f32_to_bf16_bits(kf)
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    ref = causal_gqa_attention(bf16_bits_to_f64(q), q_pos, bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    got = bf16_bits_to_f64(bf16_bits(out))
    assert np.all(np.isfinite(got))
    assert_close_bf16(got, ref, what="attention with very negative first-tile scores")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64)])
def test_attention_tiles_mixing_early_and_late_rows(cb, hq, hkv, d):
    # Query tiles that mix rows at the start of the cache with rows near its end: the early rows
    # see only the first key tile and are masked in every later one, while the late rows attend
    # to the whole cache. A second call on the same plan must give the same bits.
    n_keys = 3100
    tq = 128 // (hq // hkv)
    q_pos = np.concatenate([np.arange(0, tq // 2), np.arange(n_keys - tq // 2 - 40, n_keys - 40),
                            np.arange(1000, 1000 + tq), np.arange(n_keys - tq, n_keys)])
    q_pos = np.unique(q_pos)
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=n_keys - 1, n_suffix=1)
    plan = _plan(cb, cfg)
    rng = np.random.default_rng(hq + hkv)
    mq = q_pos.size
    q = f32_to_bf16_bits((2.0 * rng.standard_normal((mq, hq, d))).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    outs = []
    for _ in range(2):
        out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
        plan.check()
        outs.append(bf16_bits(out))
    assert np.array_equal(outs[0], outs[1])
    ref = causal_gqa_attention(bf16_bits_to_f64(q), q_pos, bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    assert_close_bf16(bf16_bits_to_f64(outs[0]), ref, what="attention with early and late rows in one tile")


# ---------------------------------------------------------------- paired-tile attention (large launches)
def _attention_sampled(cb, hq, hkv, d, n_keys, q_pos, seed, rows=256, scale_q=1.0, peaked=False):
    """Attention of len(q_pos) query rows (a launch large enough for the paired-tile kernel),
    checked against the oracle on `rows` seeded rows plus the first and last rows."""
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=max(n_keys - 1, 1), n_suffix=1)
    plan = _plan(cb, cfg)
    mq = len(q_pos)
    assert cb.cb_attention_uses_paired_tiles(plan, mq)
    rng = np.random.default_rng(seed)
    q = f32_to_bf16_bits((scale_q * rng.standard_normal((mq, hq, d))).astype(np.float32))
    k = rng.standard_normal((n_keys, hkv, d)).astype(np.float32)
    if peaked:  # a few keys far above the rest, spread over the range: the running max jumps
        k[rng.choice(n_keys, size=8, replace=False)] *= 6.0
    k = f32_to_bf16_bits(k)
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    got = bf16_bits_to_f64(bf16_bits(out))
    assert not np.isnan(got).any()  # every row written, including the ragged last tile
    pick = np.unique(np.concatenate([[0, mq - 1], rng.choice(mq, size=min(rows, mq), replace=False)]))
    ref = causal_gqa_attention(bf16_bits_to_f64(q[pick]), np.asarray(q_pos)[pick], bf16_bits_to_f64(k),
                               bf16_bits_to_f64(v))
    plan.close()
    return got[pick], ref


@pytest.mark.parametrize("hq,hkv,mq,n_keys", [(32, 8, 2500, 4000),   # odd tile count: the last pair has no tile 1
                                              (64, 8, 2600, 9000),   # Llama-70B grouping
                                              (8, 8, 10000, 12000),  # one query head per kv head
                                              (16, 1, 5500, 6000)])  # sixteen query heads per kv head
def test_paired_tile_attention_sparse_rows(cb, hq, hkv, mq, n_keys):
    rng = np.random.default_rng(mq)
    q_pos = np.sort(rng.choice(n_keys, size=mq, replace=False))
    got, ref = _attention_sampled(cb, hq, hkv, 128, n_keys, q_pos, seed=hq + mq)
    assert_close_bf16(got, ref, what=f"paired-tile attention hq={hq} hkv={hkv} mq={mq}")


@pytest.mark.parametrize("hq,hkv,mq,n_keys,paired", [(32, 8, 2500, 4000, True), (8, 2, 120, 1500, False)])
def test_attention_moderate_score_jumps(cb, hq, hkv, mq, n_keys, paired):
    # Later key tiles whose max passes a row's first-tile max by 2^9 - 2^15 (base-2 units of the
    # scaled score): below the P-sum limit, so the kernels keep the reference and P reaches
    # 2^9 - 2^15 unrescaled (the old rule rescaled at 2^8). One spike key per half tile.
    d = 128
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=n_keys - 1, n_suffix=1)
    plan = _plan(cb, cfg)
    assert bool(cb.cb_attention_uses_paired_tiles(plan, mq)) == paired
    rng = np.random.default_rng(51 + mq)
    q_pos = np.sort(rng.choice(np.arange(128, n_keys), size=mq, replace=False))  # every row sees tile 0 whole
    q = f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal((mq, hq, d))).astype(np.float32))
    kf = (0.25 * rng.standard_normal((n_keys, hkv, d))).astype(np.float32)
    spikes = [k for k in range(160, n_keys, 128)] + [k for k in range(230, n_keys, 256)]
    kf[spikes] = rng.uniform(0.72, 0.90, size=(len(spikes), 1, 1)).astype(np.float32)
    k = f32_to_bf16_bits(kf)
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    # the regime holds: for every query row, spike keys it sees score 2^9 - 2^15 above its tile-0 max
    qd, kd = bf16_bits_to_f64(q), bf16_bits_to_f64(k)
    c = np.log2(np.e) / np.sqrt(d)
    g = hq // hkv
    s0 = np.einsum("qhd,khd->qhk", qd, kd[:128].repeat(g, axis=1)).max(axis=2) * c
    ss = np.einsum("qhd,khd->qhk", qd, kd[spikes].repeat(g, axis=1)) * c
    jump = ss - s0[:, :, None]
    seen = np.asarray(spikes)[None, :] <= q_pos[:, None]
    assert seen.any()
    assert np.all((jump[seen.nonzero()[0], :, seen.nonzero()[1]] > 9) & (jump[seen.nonzero()[0], :, seen.nonzero()[1]] < 15))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    got = bf16_bits_to_f64(bf16_bits(out))
    pick = np.unique(np.concatenate([[0, mq - 1], rng.choice(mq, size=min(mq, 160), replace=False)]))
    ref = causal_gqa_attention(qd[pick], q_pos[pick], kd, bf16_bits_to_f64(v))
    plan.close()
    assert_close_bf16(got[pick], ref, what=f"attention with moderate score jumps ({'paired' if paired else 'one-tile'})")


def test_paired_tile_attention_score_jumps(cb):
    # The paired-tile kernel runs a row's later key tiles against its running reference and
    # takes a max only when a half tile's P sum passes its limit. Keys whose scores exceed
    # everything before them by far more than 2^32 (base-2 units of the scaled score), in the
    # first and second half of odd and even key tiles, make that sum overflow: a first half is
    # redone before the issuer is told, a second half after the first half of P V has completed,
    # both against a moved reference with O rescaled.
    hq, hkv, d, n_keys, mq = 32, 8, 128, 4000, 2500
    cfg = dataclasses.replace(get_config("tiny"), hq=hq, hkv=hkv, head_dim=d, n_chunks=1,
                              chunk_len=n_keys - 1, n_suffix=1)
    plan = _plan(cb, cfg)
    assert cb.cb_attention_uses_paired_tiles(plan, mq)
    rng = np.random.default_rng(33)
    q_pos = np.sort(rng.choice(n_keys, size=mq, replace=False))
    q = f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal((mq, hq, d))).astype(np.float32))
    kf = rng.standard_normal((n_keys, hkv, d)).astype(np.float32)
    # each spike passes the previous one by about 2^33 or more; key % 128 < 64 is a tile's first half
    spikes = {356: 4.0,    # tile 2, second half
              1410: 6.0,   # tile 11, first half
              1734: 8.0,   # tile 13, second half
              2705: 10.0,  # tile 21, first half
              3440: 12.0}  # tile 26, second half
    for key, val in spikes.items():
        kf[key] = val
    k = f32_to_bf16_bits(kf)
    v = f32_to_bf16_bits(rng.standard_normal((n_keys, hkv, d)).astype(np.float32))
    out = torch.full((mq, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    cb.cb_hkvd_attention(plan, bf16_tensor(q), _i32(q_pos), mq, bf16_tensor(k), bf16_tensor(v), n_keys, out)
    plan.check()
    got = bf16_bits_to_f64(bf16_bits(out))
    assert np.all(np.isfinite(got))
    # rows on both sides of every spike, plus seeded rows
    near = [np.searchsorted(q_pos, t) + o for t in spikes for o in (-1, 0, 1)]
    pick = np.unique(np.clip(np.concatenate([near, [0, mq - 1], rng.choice(mq, size=160, replace=False)]), 0, mq - 1))
    ref = causal_gqa_attention(bf16_bits_to_f64(q[pick]), q_pos[pick], bf16_bits_to_f64(k), bf16_bits_to_f64(v))
    plan.close()
    assert_close_bf16(got[pick], ref, what="paired-tile attention with score jumps")


def test_paired_tile_attention_dense_suffix_and_rescale(cb):
    # every position from 0 (causal diagonal in every key tile), keys that force the running max
    # up by more than 2^8 inside the loop
    n_keys = 3000
    q_pos = np.arange(n_keys)
    got, ref = _attention_sampled(cb, 32, 8, 128, n_keys, q_pos, seed=7, scale_q=2.0, peaked=True)
    assert_close_bf16(got, ref, what="paired-tile attention, all positions, peaked keys")

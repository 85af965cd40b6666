"""GB300 (sm_103a) CacheBlend per-layer KV blend.

Thin PyTorch-facing binding of the C ABI in include/cacheblend.h: the same
call names, tensors passed as device pointers, the current torch stream as
the CUDA stream. PyTorch only allocates device memory and provides streams;
every step of the blend runs in the library's CUDA kernels.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import CacheBlendError, check

__all__ = ["Plan", "CacheBlendError", "cb_rope_rerotate", "cb_kv_deviation", "cb_kv_deviation_kv", "cb_hkvd_topk",
           "cb_fuse_scatter", "cb_hkvd_attention", "cb_decode_attention", "cb_attention_sparsity",
           "cb_output_deviation", "cb_qkv_projection", "cb_qkv_projection_indexed", "cb_blend_layer", "cb_blend_stage",
           "cb_blend_request", "cb_hkvd_select_noalloc", "cb_attention_uses_paired_tiles",
           "cb_test_attention_wait_timeout", "cb_test_decode_wait_timeout", "cb_test_projection_wait_timeout",
           "cb_check", "cb_version",
           "LayerBuffers"]


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class Plan:
    """A cb_plan: one blend request's shapes, RoPE table and scratch on the current device."""

    def __init__(self, n_chunks, chunk_len, n_suffix, hq, hkv, head_dim, rope_theta, rope_style="half",
                 r1_pct=15, r2_pct=15, deviation="v", filter="keep"):
        lib = _lib.load()
        self.cfg = _lib.CbConfig(n_chunks, chunk_len, n_suffix, hq, hkv, head_dim, float(rope_theta),
                                 _lib.ROPE_STYLES[rope_style], r1_pct, r2_pct, _lib.DEVIATIONS[deviation],
                                 _lib.FILTERS[filter])
        self.deviation, self.filter = deviation, filter
        self.n_ctx = n_chunks * chunk_len
        self.n_tokens = self.n_ctx + n_suffix
        self.hq, self.hkv, self.head_dim = hq, hkv, head_dim
        self._h = ctypes.c_void_p()
        check(lib.cb_plan_create(ctypes.byref(self.cfg), ctypes.byref(self._h)))

    @classmethod
    def from_config(cls, cfg, rope_style="half", r1_pct=None, r2_pct=None, deviation="v", filter="keep"):
        """From a workloads.BlendConfig (or anything with the same fields)."""
        return cls(cfg.n_chunks, cfg.chunk_len, cfg.n_suffix, cfg.hq, cfg.hkv, cfg.head_dim, cfg.rope_theta,
                   rope_style, cfg.r1_pct if r1_pct is None else r1_pct, cfg.r2_pct if r2_pct is None else r2_pct,
                   deviation, filter)

    def candidate_layer(self, layer):
        """The layer whose selection is C_layer (0: all context tokens), per the plan's filter."""
        if layer <= 1:
            return 0
        return 1 if self.filter == "reselect" else layer - 1

    @property
    def handle(self):
        if not self._h:
            raise RuntimeError("plan is closed")
        return self._h

    def layer_sizes(self, layer):
        v = [ctypes.c_int32() for _ in range(4)]
        check(_lib.load().cb_layer_sizes(self.handle, layer, *[ctypes.byref(x) for x in v]))
        return tuple(x.value for x in v)  # (n_cand, k, mq, selects)

    def check(self):
        check(_lib.load().cb_check(self.handle))

    def close(self):
        if getattr(self, "_h", None):
            _lib.load().cb_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def cb_version() -> int:
    return _lib.load().cb_version()


def cb_check(plan: Plan) -> None:
    plan.check()


def cb_rope_rerotate(plan, out, x, pos_to, pos_from=None, in_rows=None, out_rows=None, n=None, stream=None):
    """out[out_rows[i]] = R_{pos_to[i] - pos_from[i]} x[in_rows[i]] (see cacheblend.h)."""
    n = pos_to.numel() if n is None else n
    n_heads = x.shape[1]
    check(_lib.load().cb_rope_rerotate(
        plan.handle, _ptr(out, torch.bfloat16, "out"), _ptr(x, torch.bfloat16, "x"),
        _ptr(in_rows, torch.int32, "in_rows"), _ptr(out_rows, torch.int32, "out_rows"),
        _ptr(pos_from, torch.int32, "pos_from"), _ptr(pos_to, torch.int32, "pos_to"), n, n_heads,
        x.shape[0], out.shape[0], _stream(stream)))


def cb_kv_deviation(plan, v_new, v_old, cand, m, dev, stream=None):
    check(_lib.load().cb_kv_deviation(
        plan.handle, _ptr(v_new, torch.bfloat16, "v_new"), _ptr(v_old, torch.bfloat16, "v_old"),
        _ptr(cand, torch.int32, "cand"), m, _ptr(dev, torch.float32, "dev"), _stream(stream)))


def cb_kv_deviation_kv(plan, k_new, k_old, v_new, v_old, cand, m, dev, stream=None):
    check(_lib.load().cb_kv_deviation_kv(
        plan.handle, _ptr(k_new, torch.bfloat16, "k_new"), _ptr(k_old, torch.bfloat16, "k_old"),
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(v_old, torch.bfloat16, "v_old"),
        _ptr(cand, torch.int32, "cand"), m, _ptr(dev, torch.float32, "dev"), _stream(stream)))


def cb_hkvd_topk(plan, dev, cand, m, k, sel_tok, sel_row, stream=None):
    check(_lib.load().cb_hkvd_topk(
        plan.handle, _ptr(dev, torch.float32, "dev"), _ptr(cand, torch.int32, "cand"), m, k,
        _ptr(sel_tok, torch.int32, "sel_tok"), _ptr(sel_row, torch.int32, "sel_row"), _stream(stream)))


def cb_fuse_scatter(plan, k_fused, v_fused, k_new, v_new, sel_tok, k, stream=None):
    check(_lib.load().cb_fuse_scatter(
        plan.handle, _ptr(k_fused, torch.bfloat16, "k_fused"), _ptr(v_fused, torch.bfloat16, "v_fused"),
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(sel_tok, torch.int32, "sel_tok"), k, _stream(stream)))


def cb_hkvd_attention(plan, q, q_pos, mq, k, v, n_keys, out, scale=0.0, stream=None):
    check(_lib.load().cb_hkvd_attention(
        plan.handle, _ptr(q, torch.bfloat16, "q"), _ptr(q_pos, torch.int32, "q_pos"), mq,
        _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"), n_keys, float(scale),
        _ptr(out, torch.bfloat16, "out"), _stream(stream)))


def cb_decode_attention(plan, q, k, v, n_keys, out, scale=0.0, stream=None):
    """One decode step's attention: q [Hq, D] at position n_keys - 1 over k, v [>= n_keys, Hkv, D]."""
    check(_lib.load().cb_decode_attention(
        plan.handle, _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        n_keys, float(scale), _ptr(out, torch.bfloat16, "out"), _stream(stream)))


def cb_attention_sparsity(plan, q, q_pos, mq, k, v, n_keys, eps, out, row_stats, counts, total, scale=0.0,
                          stream=None):
    """Counts of attention weights below eps (see cacheblend.h); row_stats float32 [mq, hq, 2],
    counts int32 [mq, hq], total int64 [1] (device, written as an unsigned count)."""
    check(_lib.load().cb_attention_sparsity(
        plan.handle, _ptr(q, torch.bfloat16, "q"), _ptr(q_pos, torch.int32, "q_pos"), mq,
        _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"), n_keys, float(scale), float(eps),
        _ptr(out, torch.bfloat16, "out"), _ptr(row_stats, torch.float32, "row_stats"),
        _ptr(counts, torch.int32, "counts"), _ptr(total, torch.int64, "total"), _stream(stream)))


def cb_output_deviation(plan, o, o_ref, rows, sums, stream=None):
    """sums (float64 [2], device) = (sum (o - o_ref)^2, sum o_ref^2) over rows x hq x D."""
    check(_lib.load().cb_output_deviation(
        plan.handle, _ptr(o, torch.bfloat16, "o"), _ptr(o_ref, torch.bfloat16, "o_ref"), rows,
        _ptr(sums, torch.float64, "sums"), _stream(stream)))


def cb_qkv_projection(plan, x, rows, m, w_qkv, q, k, v, encode=False, x_gathered=None, stream=None):
    """q / k / v rows of the tokens `rows` (int32, or None: tokens 0..m-1) from x [x_rows, d_model]
    times w_qkv^T, RoPE-encoded q and k when `encode` (see cacheblend.h)."""
    check(_lib.load().cb_qkv_projection(
        plan.handle, _ptr(x, torch.bfloat16, "x"), x.shape[0], x.shape[1], _ptr(rows, torch.int32, "rows"), m,
        _ptr(w_qkv, torch.bfloat16, "w_qkv"), 1 if encode else 0, _ptr(x_gathered, torch.bfloat16, "x_gathered"),
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"), _stream(stream)))


def cb_qkv_projection_indexed(plan, x, x_index, tokens, m, w_qkv, q, k, v, encode=False, x_gathered=None,
                              stream=None):
    """q / k / v at tokens[i] (int32, or None: token i) from x[x_index[i]] W^T (x_index int32, or
    None: x[i] read in place), RoPE-encoded q and k when `encode` (see cacheblend.h)."""
    check(_lib.load().cb_qkv_projection_indexed(
        plan.handle, _ptr(x, torch.bfloat16, "x"), x.shape[0], x.shape[1], _ptr(x_index, torch.int32, "x_index"),
        _ptr(tokens, torch.int32, "tokens"), m, _ptr(w_qkv, torch.bfloat16, "w_qkv"), 1 if encode else 0,
        _ptr(x_gathered, torch.bfloat16, "x_gathered"), _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"),
        _ptr(v, torch.bfloat16, "v"), _stream(stream)))


def cb_hkvd_select_noalloc(v_new, v_old, cand, m, k, n_rows, sel_tok, sel_row, stream=None):
    """HKVD selection with no allocation anywhere (see cacheblend.h): the deviations
    between its two kernels live in a fixed array inside the library, so this call
    needs no plan. For callers that must not allocate device memory where they
    select tokens. m is at most 65536; calls that overlap on the GPU race."""
    check(_lib.load().cb_hkvd_select_noalloc(
        _ptr(v_new, torch.bfloat16, "v_new"), _ptr(v_old, torch.bfloat16, "v_old"),
        _ptr(cand, torch.int32, "cand"), m, k, n_rows, v_new.shape[1], v_new.shape[2],
        _ptr(sel_tok, torch.int32, "sel_tok"), _ptr(sel_row, torch.int32, "sel_row"), _stream(stream)))


def cb_attention_uses_paired_tiles(plan, mq) -> bool:
    """True if an attention call of mq query rows runs the paired-tile kernel (see cacheblend.h)."""
    return bool(_lib.load().cb_attention_uses_paired_tiles(plan.handle, mq))


def cb_test_decode_wait_timeout(plan, q, k, v, n_keys, out, stream=None):
    """Decode attention in a form whose bounded waits run out (see cacheblend.h; test support)."""
    check(_lib.load().cb_test_decode_wait_timeout(
        plan.handle, _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
        n_keys, _ptr(out, torch.bfloat16, "out"), _stream(stream)))


def cb_test_projection_wait_timeout(plan, x, m, w_qkv, q, k, v, stream=None):
    """The QKV projection in a form whose bounded waits run out (see cacheblend.h; test support)."""
    check(_lib.load().cb_test_projection_wait_timeout(
        plan.handle, _ptr(x, torch.bfloat16, "x"), x.shape[1], m, _ptr(w_qkv, torch.bfloat16, "w_qkv"),
        _ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"), _stream(stream)))


def cb_test_attention_wait_timeout(plan, q, q_pos, mq, k, v, n_keys, out, stream=None):
    """Test support: the attention kernel in a form whose waits run out (see cacheblend.h); the
    plan's next check() raises with CB_ERR_TIMEOUT."""
    check(_lib.load().cb_test_attention_wait_timeout(
        plan.handle, _ptr(q, torch.bfloat16, "q"), _ptr(q_pos, torch.int32, "q_pos"), mq,
        _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"), n_keys, _ptr(out, torch.bfloat16, "out"),
        _stream(stream)))


class LayerBuffers:
    """Device buffers of one layer's outputs, sized for the plan's largest layer."""

    def __init__(self, plan: Plan, device="cuda"):
        n1, k1, mq1, _ = plan.layer_sizes(1)
        bf = dict(dtype=torch.bfloat16, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.dev = torch.empty(max(n1, 1), dtype=torch.float32, device=device)
        self.sel_tok = torch.empty(max(k1, 1), **i32)
        self.sel_row = torch.empty(max(k1, 1), **i32)
        self.k_fused = torch.empty(plan.n_tokens, plan.hkv, plan.head_dim, **bf)
        self.v_fused = torch.empty(plan.n_tokens, plan.hkv, plan.head_dim, **bf)
        self.q_rot = torch.empty(max(mq1, 1), plan.hq, plan.head_dim, **bf)
        self.out = torch.empty(max(mq1, 1), plan.hq, plan.head_dim, **bf)


def _layer_io(k_old, v_old, k_new, v_new, q, cand, bufs):
    return _lib.CbLayerIO(
        _ptr(k_old, torch.bfloat16, "k_old"), _ptr(v_old, torch.bfloat16, "v_old"),
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(q, torch.bfloat16, "q"), _ptr(cand, torch.int32, "cand"), _ptr(bufs.dev, torch.float32, "dev"),
        _ptr(bufs.sel_tok, torch.int32, "sel_tok"), _ptr(bufs.sel_row, torch.int32, "sel_row"),
        _ptr(bufs.k_fused, torch.bfloat16, "k_fused"), _ptr(bufs.v_fused, torch.bfloat16, "v_fused"),
        _ptr(bufs.q_rot, torch.bfloat16, "q_rot"), _ptr(bufs.out, torch.bfloat16, "out"))


def cb_blend_request(plan, layers, stream=None):
    """All layers of one request (cb_blend_request): `layers` lists, for layers 1..n, dicts with
    k_old, v_old, k_new, v_new, q and bufs (a LayerBuffers per layer; buffers must not alias).
    Layer l reads the candidates layers[l-2]["bufs"].sel_tok (filter "reselect": layers[0]["bufs"].sel_tok)."""
    n = len(layers)
    arr = (_lib.CbLayerIO * n)()
    for i, L in enumerate(layers):
        arr[i] = _layer_io(L["k_old"], L["v_old"], L["k_new"], L["v_new"], L["q"], None, L["bufs"])
    check(_lib.load().cb_blend_request(plan.handle, n, arr, _stream(stream)))


def cb_blend_layer(plan, layer, *, k_old, v_old, k_new, v_new, q, cand, bufs: LayerBuffers, stream=None):
    """One layer of the blend; outputs land in `bufs` (sizes from plan.layer_sizes(layer))."""
    io = _layer_io(k_old, v_old, k_new, v_new, q, cand, bufs)
    check(_lib.load().cb_blend_layer(plan.handle, layer, ctypes.byref(io), _stream(stream)))


def cb_blend_stage(plan, layer, stage, *, k_old, v_old, k_new, v_new, q, cand, bufs: LayerBuffers, stream=None):
    """One stage ("deviation", "topk", "fuse" or "attention") of cb_blend_layer alone, reading
    what the layer's earlier stages wrote into `bufs` (cb_blend_stage)."""
    io = _layer_io(k_old, v_old, k_new, v_new, q, cand, bufs)
    check(_lib.load().cb_blend_stage(plan.handle, layer, ctypes.byref(io), _lib.STAGES[stage], _stream(stream)))

"""One layer of the CacheBlend blend, and the gradual filter across layers.

Per layer l (all steps are the definitions in the sibling modules):
  1. cached keys are re-rotated from chunk-local to global positions
     ("数学推导" §CacheBlend 中的应用);
  2. at a filtering layer, the V deviation of every candidate token is formed
     and the k_l largest are selected ("数学推导" §近似解);
  3. the selected and suffix rows take their recomputed K (encoded at the
     global position) and V; all other rows keep the cache ("数学推导" §形式化);
  4. the selected tokens and the suffix attend causally over the fused cache.

Gradual filter ("rag的kvcache问题" §渐进式过滤机制), as read here:
  layer 1: candidates = all context tokens, keep k_1 = floor(r1 * n_ctx / 100);
  layer 2: candidates = the layer-1 selection, keep k_2 = floor(r2 * n_ctx / 100);
  layer >= 3: candidates = the previous selection, which is kept whole
              (no deviation, no top-k).
A second reading (filter="reselect"), which the page leaves open: the
layer-2 step repeats at every layer >= 2, i.e. candidates = the layer-1
selection and k_2 kept by that layer's own deviation; the page's "stable from
layer 3" is then an observation about the selections, not a rule.
A single-layer workload runs layer 1 with r1 as its ratio.

Deviation ("deviation" argument): "v" ranks by the V distance of
"数学推导" §近似解, "kv" by the K+V distance (see oracle.deviation).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .attention import causal_gqa_attention
from .deviation import bf16_bits_to_f64, deviation_canonical_f32, kv_deviation_canonical_f32
from .fuse import fused_kv
from .positions import chunk_local_positions, global_positions
from .rope import rerotate, rope_rotate, round_bf16
from .topk import hkvd_topk, k_for_ratio


FILTERS = ("keep", "reselect")
DEVIATIONS = ("v", "kv")


def gradual_filter_schedule(n_ctx: int, layers: int, r1_pct: int, r2_pct: int, filter: str = "keep"):
    """[(layer, k_l, selects)] for layers 1..layers."""
    if filter not in FILTERS:
        raise ValueError(f"unknown filter {filter!r}")
    if not 0 <= r2_pct <= r1_pct <= 100:
        raise ValueError("need 0 <= r2 <= r1 <= 100")
    k1, k2 = k_for_ratio(r1_pct, n_ctx), k_for_ratio(r2_pct, n_ctx)
    out = []
    for layer in range(1, layers + 1):
        if layer == 1:
            out.append((1, k1, True))
        elif layer == 2:
            out.append((2, k2, True))
        else:
            out.append((layer, k2, filter == "reselect"))
    return out


def candidate_layer(layer: int, filter: str = "keep") -> int:
    """The layer whose selection is C_l (0: all context tokens)."""
    if layer <= 1:
        return 0
    return 1 if filter == "reselect" else layer - 1


@dataclass
class LayerResult:
    layer: int
    cand: np.ndarray
    k: int
    dev: np.ndarray | None      # fp32 canonical deviation per candidate (filtering layers)
    sel_tok: np.ndarray         # S_l, ascending token ids
    sel_row: np.ndarray         # rows of S_l in cand
    k_fused: np.ndarray         # fp64 holding bf16 values [N, Hkv, D]
    v_fused: np.ndarray         # fp64 holding bf16 values [N, Hkv, D]
    is_new: np.ndarray          # bool [N]: row taken from the recomputed K/V
    q_tok: np.ndarray           # query tokens: S_l then the suffix
    q_rot: np.ndarray           # fp64 holding bf16 values [mq, Hq, D]
    out: np.ndarray | None      # fp64 [mq, Hq, D] (rows not requested are NaN)
    out_vscale: np.ndarray | None = None  # sum_j softmax_j |v_j| per output element (error scale)


def blend_layer(cfg, inp, layer: int, cand, k: int, selects: bool, style: str = "half",
                attention_rows=None, deviation: str = "v") -> LayerResult:
    """One layer. `inp` is a workloads.LayerInputs; attention_rows=None computes all
    query rows, an index array computes only those rows, and False skips attention."""
    n_ctx, n = cfg.n_ctx, cfg.n_tokens
    cand = np.asarray(cand, dtype=np.int64)
    p_new = global_positions(n)
    p_old = chunk_local_positions(cfg.n_chunks, cfg.chunk_len)

    if selects:
        if deviation == "v":
            dev = deviation_canonical_f32(inp.v_new[cand], inp.v_old[cand])
        elif deviation == "kv":
            dev = kv_deviation_canonical_f32(inp.k_new[cand], inp.k_old[cand], inp.v_new[cand], inp.v_old[cand],
                                             p_old[cand], cfg.rope_theta, style)
        else:
            raise ValueError(f"unknown deviation {deviation!r}")
        sel_tok, sel_row = hkvd_topk(dev, cand, k)
    else:
        if k != cand.size:
            raise ValueError("a non-filtering layer keeps its whole candidate set")
        dev, sel_tok, sel_row = None, cand, np.arange(cand.size)

    k_old_rot = round_bf16(rerotate(bf16_bits_to_f64(inp.k_old), p_old, p_new[:n_ctx],
                                    cfg.rope_theta, style))
    rows_new = np.concatenate([sel_tok, np.arange(n_ctx, n)])
    k_new_enc = np.zeros((n, cfg.hkv, cfg.head_dim))
    k_new_enc[rows_new] = round_bf16(rope_rotate(bf16_bits_to_f64(inp.k_new[rows_new]),
                                                 p_new[rows_new], cfg.rope_theta, style))
    k_f, v_f, is_new = fused_kv(k_old_rot, bf16_bits_to_f64(inp.v_old), k_new_enc,
                                bf16_bits_to_f64(inp.v_new), sel_tok, n_ctx)

    q_tok = rows_new
    q_rot = round_bf16(rope_rotate(bf16_bits_to_f64(inp.q[q_tok]), q_tok, cfg.rope_theta, style))
    out = vs = None
    if attention_rows is None:
        out, vs = causal_gqa_attention(q_rot, q_tok, k_f, v_f, return_vscale=True)
    elif attention_rows is not False:
        rows = np.asarray(attention_rows, dtype=np.int64)
        out = np.full(q_rot.shape, np.nan)
        vs = np.full(q_rot.shape, np.nan)
        out[rows], vs[rows] = causal_gqa_attention(q_rot[rows], q_tok[rows], k_f, v_f, return_vscale=True)
    return LayerResult(layer, cand, k, dev, sel_tok, sel_row, k_f, v_f, is_new, q_tok, q_rot, out, vs)


def blend_request(cfg, layer_inputs, style: str = "half", attention_rows=None, deviation: str = "v",
                  filter: str = "keep"):
    """Run the gradual filter over the layers whose inputs are given (in order from layer 1).

    layer_inputs: iterable of workloads.LayerInputs for layers 1, 2, ...
    Yields one LayerResult per layer.
    """
    sched = gradual_filter_schedule(cfg.n_ctx, cfg.layers, cfg.r1_pct, cfg.r2_pct, filter)
    sel = {0: np.arange(cfg.n_ctx, dtype=np.int64)}
    for (layer, k, selects), inp in zip(sched, layer_inputs):
        if inp.layer != layer:
            raise ValueError("layer inputs must start at layer 1 and be consecutive")
        cand = sel[candidate_layer(layer, filter)]
        res = blend_layer(cfg, inp, layer, cand, k, selects, style, attention_rows, deviation)
        sel[layer] = res.sel_tok
        yield res

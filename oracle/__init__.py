"""CPU oracle for the CacheBlend per-layer KV blend.

TEST INFRASTRUCTURE. This package is a plain, slow CPU statement of what the
blend computes, used only to check the CUDA library. Only the test suite, the
smoke check in ``__graft_entry__`` and the CPU-baseline / reference legs of
``bench.py`` may import it. The CUDA library and its Python binding never
import it, and it imports nothing from them: the two sides share only the
seeded input bytes made by the ``workloads`` package.

Arithmetic is fp64 (numpy) except where the method's result is an integer
decided by floating point (the top-k over the V deviation): there both sides
take the decision on the same fp32 values, summed in one documented order
(``oracle.deviation.deviation_canonical_f32``).

Sources: "数学推导" (CacheBlend appendix C) for RoPE, the re-rotation of
cached keys, the fused KV and the top-k selection; "rag的kvcache问题" for
the gradual filtering scheme, independent chunk encoding, the causal mask and
row-parallel attention.

Parity status per function:
  rope.rope_rotate / rope.rerotate     pinned (closed-form identities, textbook 2-D rotation)
  deviation.deviation_canonical_f32    pinned (exact sum within bound, hand-derived rounding cases)
  topk.hkvd_topk                       pinned (brute-force rank counting, ties, k = 0 / m)
  fuse.fused_kv                        pinned (definition, provenance)
  attention.causal_gqa_attention       pinned (library causal attention, single key, equal scores)
  blend.gradual_filter_schedule        pinned (three-layer examples worked by hand from the page's
                                       illustration, one per reading; structure)
  deviation.kv_deviation_canonical_f32 pinned (closed form, frame invariance, plain loops, bound)
  attention.decode_attention           pinned (last row of library causal attention, special cases)
  diagnostics.attention_deviation      pinned (definition, r = 100% gives exactly 0)
  diagnostics.attention_sparsity       pinned (closed form for equal scores, library softmax matrix)
  projection.qkv_projection            pinned (element loops, one-hot rows, RoPE at the row position)
"""

from . import attention, blend, deviation, diagnostics, fuse, positions, projection, rope, topk  # noqa: F401

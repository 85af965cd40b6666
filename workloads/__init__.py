"""Seeded synthetic workloads for the CacheBlend per-layer KV blend.

This package produces input bytes only. It holds none of the blend's
arithmetic (no rotation, no deviation, no selection, no attention): the
CUDA library and the CPU oracle both consume exactly the bytes made here and
compute everything else on their own.
"""

from .configs import CONFIGS, BlendConfig, get_config  # noqa: F401
from .generator import (  # noqa: F401
    LayerInputs,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    generate_layer,
    hkvd_noise_sets,
)

"""The five blend workloads: shapes, RoPE base, recompute ratios and noise model.

Shapes follow the CacheBlend setting described on "rag的kvcache问题"
(section 独立编码): a request is a list of cached chunks, each encoded on its own
at chunk-local positions starting from 0, followed by a query suffix that has
no cache. Recompute ratios r1 (layer 1) and r2 (layer 2 on) follow the same
page's gradual filtering scheme (section 渐进式过滤机制). The noise model
(about 15% of tokens with a large KV deviation, the rest near zero, and a
high-deviation set that persists across layers) follows the same page's
sections 核心发现 and 跨层相关性.
"""

from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class BlendConfig:
    name: str
    config_id: int
    n_chunks: int
    chunk_len: int
    n_suffix: int
    hq: int
    hkv: int
    head_dim: int
    rope_theta: float
    layers: int
    r1_pct: int
    r2_pct: int
    # "set": sigma_hi on a seeded set of hkvd_frac of the context tokens,
    # sigma_lo elsewhere. "lognormal": per-token scale exp(mu + sigma * z).
    noise: str = "set"
    hkvd_frac: float = 0.15
    swap_frac: float = 0.10
    sigma_hi: float = 1.0
    sigma_lo: float = 0.01
    lognormal_mu: float = -4.0
    lognormal_sigma: float = 2.0
    sweep_pct: tuple = field(default_factory=tuple)
    # hidden size of the model (the QKV projection's input width)
    d_model: int = 0

    @property
    def n_ctx(self) -> int:
        return self.n_chunks * self.chunk_len

    @property
    def n_tokens(self) -> int:
        return self.n_ctx + self.n_suffix

    @property
    def seed(self) -> int:
        return 1234 + 1000 * self.config_id

    def with_ratio(self, r_pct: int) -> "BlendConfig":
        """Single-layer variant selecting r_pct% (used by the ratio sweep)."""
        return BlendConfig(**{**self.__dict__, "r1_pct": r_pct, "r2_pct": r_pct})


CONFIGS = {
    # 2 chunks x 256 + 32 suffix, 4 q / 2 kv heads, head_dim 64: small enough
    # for the CPU oracle to finish in seconds.
    "tiny": BlendConfig("tiny", 1, 2, 256, 32, 4, 2, 64, 1e4, 1, 15, 15,
                        noise="set", hkvd_frac=0.15, swap_frac=0.0, d_model=256),
    # Mistral-7B-shaped: 6 x 512 + 64, 32 q / 8 kv heads, head_dim 128, 32 layers.
    "mistral7b": BlendConfig("mistral7b", 2, 6, 512, 64, 32, 8, 128, 1e4, 32, 30, 15,
                             noise="set", hkvd_frac=0.15, swap_frac=0.10, d_model=4096),
    # Long-context Mistral-7B-shaped: 16 x 2048 + 128 (32,896 tokens), 32 layers.
    "long32k": BlendConfig("long32k", 3, 16, 2048, 128, 32, 8, 128, 1e4, 32, 30, 15,
                           noise="set", hkvd_frac=0.15, swap_frac=0.10, d_model=4096),
    # Llama-70B-shaped: 8 x 1024 + 256, 64 q / 8 kv heads, theta 5e5, 80 layers.
    "llama70b": BlendConfig("llama70b", 4, 8, 1024, 256, 64, 8, 128, 5e5, 80, 20, 10,
                            noise="set", hkvd_frac=0.10, swap_frac=0.10, d_model=8192),
    # Recompute-ratio sweep at Mistral shape, 16 x 512 + 64, one layer; the
    # lognormal per-token noise scale makes the top-k boundary dense with ties.
    "sweep": BlendConfig("sweep", 5, 16, 512, 64, 32, 8, 128, 1e4, 1, 15, 15,
                         noise="lognormal", sweep_pct=(5, 10, 15, 30, 50, 100), d_model=4096),
}


def get_config(name: str) -> BlendConfig:
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    return CONFIGS[name]

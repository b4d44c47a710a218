"""The five synthetic engram workloads, as plain data.

Shapes follow DeepSeek-V4.1-Flash as the pages give them: engram before model
layers 1 and 14, four-gram windows over eight heads (24 hash columns, 48 ids a
token over two layers), 256-wide rows, dim 4096 and four hyper-connection
streams (page "spark_model/layers/engram_v41.rs", module doc).
Nothing here computes any part of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class EngramConfig:
    name: str
    vocab: int
    n_compressed: int            # token_map range [0, n_compressed)
    unmapped_5pct: bool          # 5% of tokens map to -1
    pad_token_id: int
    pad_compressed: object       # force token_map[pad_token_id] to this value (or None)
    layer_ids: tuple
    max_ngram: int
    n_heads: int
    prime_target: int            # per-slot primes: the first L*C primes >= this
    head_dim: int
    scale_block: int
    dim: int
    hc: int
    fmt: str                     # "fp8" (e4m3 + pow2 f32 scales), "fp8_e8m0" (one-byte scales) or "q2k"
    batch: int                   # independent sequences
    prefix: int                  # positions hashed before the measured call
    T: int                       # tokens per sequence per call
    ids: str                     # "zipf" or "uniform"
    zipf_s: float = 1.1
    seed: int = 0
    eps: float = 1e-6
    decode_steps: int = 0        # single-token steps after the prefill
    wkv_fmt: str = "bf16"        # "q2k": wkv also held as Q2_K blocks (its bf16 form is their dequantisation)
    layer_fmts: tuple = ()       # per-layer table formats overriding `fmt` (mixed-format tests)

    def fmt_of(self, layer: int) -> str:
        """The table format of layer `layer`."""
        return self.layer_fmts[layer] if self.layer_fmts else self.fmt

    @property
    def n_layers(self) -> int:
        return len(self.layer_ids)

    @property
    def cols(self) -> int:
        return (self.max_ngram - 1) * self.n_heads

    @property
    def K(self) -> int:
        return self.cols * self.head_dim

    @property
    def N(self) -> int:
        return self.dim * (self.hc + 1)

    @property
    def max_seq(self) -> int:
        return self.prefix + self.T + self.decode_steps + 8192

    def with_(self, **kw) -> "EngramConfig":
        return replace(self, **kw)


TINY = EngramConfig(
    name="tiny", vocab=1000, n_compressed=600, unmapped_5pct=True, pad_token_id=0,
    pad_compressed=0, layer_ids=(0,), max_ngram=3, n_heads=2, prime_target=509,
    head_dim=64, scale_block=32, dim=128, hc=2, fmt="fp8", batch=1, prefix=0, T=16,
    ids="uniform")

V41_DECODE = EngramConfig(
    name="v41_decode_T1", vocab=129280, n_compressed=65536, unmapped_5pct=False,
    pad_token_id=0, pad_compressed=None, layer_ids=(1, 14), max_ngram=4, n_heads=8,
    prime_target=1 << 17, head_dim=256, scale_block=32, dim=4096, hc=4, fmt="fp8",
    batch=1, prefix=2048, T=1, ids="zipf")

V41_PREFILL = V41_DECODE.with_(name="v41_prefill_T4096", prefix=0, T=4096)

V41_Q2K = V41_DECODE.with_(name="v41_q2k_T512", prime_target=1 << 18, fmt="q2k",
                           prefix=0, T=512)

STRESS = V41_DECODE.with_(name="large_table_stress", prime_target=1 << 20, batch=8,
                          prefix=0, T=1536, ids="uniform", decode_steps=512)

# The single-token step projecting from Q2_K-quantised wkv (6x fewer weight bytes).
V41_DECODE_WKVQ2K = V41_DECODE.with_(name="v41_decode_T1_wkv_q2k", wkv_fmt="q2k")

# The decode step with one-byte e8m0 scales (264 instead of 288 bytes a row).
V41_DECODE_E8M0 = V41_DECODE.with_(name="v41_decode_T1_e8m0", fmt="fp8_e8m0")

CONFIGS = {c.name: c for c in (TINY, V41_DECODE, V41_PREFILL, V41_Q2K, STRESS, V41_DECODE_WKVQ2K,
                               V41_DECODE_E8M0)}

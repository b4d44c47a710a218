"""Glue between the seeded generator and the CPU oracle for the parity tests.

The oracle's inputs are always regenerated on the CPU by the numpy twin of the
generator (deepseek_v4_engram_hash_gb300.synth) -- never copied from the GPU
path under test -- except where a test checks one stage on the GPU's own
output of the previous stage (stage-wise parity), which it says.
"""
import numpy as np

import oracle
from deepseek_v4_engram_hash_gb300 import synth


def hash_state(cfg, batch=None, max_seq=None):
    t = synth.hash_tables(cfg)
    return oracle.HashState(t["token_map"], t["pad_id"], t["multipliers"], t["primes"],
                            t["offsets"], cfg.n_layers, cfg.max_ngram, cfg.n_heads,
                            batch or cfg.batch, max_seq or cfg.max_seq)


def rows(cfg, layer, ids) -> np.ndarray:
    """Dequantised rows [len(ids), hd] (bf16 bits) of layer `layer` for row ids `ids`."""
    ids = np.asarray(ids, dtype=np.int64).ravel()
    uniq, inv = np.unique(ids, return_inverse=True)
    if cfg.fmt == "fp8":
        codes, scales = synth.table_fp8_rows(cfg, layer, uniq)
        return oracle.rows_fp8(codes, scales, cfg.head_dim, cfg.scale_block, inv)
    blocks = synth.table_q2k_rows(cfg, layer, uniq)
    return oracle.rows_q2k(blocks, inv)


def x_of(cfg, layer, row_ids) -> np.ndarray:
    """x [M, K] bf16 bits from row ids [M, L, C]: the C rows concatenated in column order."""
    M = row_ids.shape[0]
    r = rows(cfg, layer, row_ids[:, layer, :].reshape(-1))
    return r.reshape(M, cfg.cols * cfg.head_dim)


def kv(cfg, layer, x_bits, out_rows=None) -> np.ndarray:
    """kv [M, len(out_rows)] bf16 bits; out_rows defaults to all N outputs."""
    if out_rows is None:
        out_rows = np.arange(cfg.N)
    w = synth.wkv_rows(cfg, layer, out_rows)
    return oracle.linear_bf16(x_bits, w)


def gate(cfg, layer, h, kv_bits):
    q, k = synth.qk_weights(cfg, layer)
    return oracle.gate(h, kv_bits, q, k, cfg.hc, cfg.dim, cfg.eps)


def kv_rel_err(got_bits, want_bits) -> float:
    """max |g - r| / max(|r|, 1e-3 max|r|) over bf16 outputs."""
    g = oracle.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = oracle.bf16_bits_to_f32(want_bits).astype(np.float64)
    floor = 1e-3 * max(np.abs(r).max(), 1e-30)
    return float((np.abs(g - r) / np.maximum(np.abs(r), floor)).max())


KV_TOL = 2e-2
H_TOL = 1e-3

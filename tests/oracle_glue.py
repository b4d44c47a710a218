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
    fmt = cfg.fmt_of(layer)
    if fmt == "fp8":
        codes, scales = synth.table_fp8_rows(cfg, layer, uniq)
        return oracle.rows_fp8(codes, scales, cfg.head_dim, cfg.scale_block, inv)
    if fmt == "fp8_e8m0":
        codes, scales = synth.table_fp8_rows(cfg, layer, uniq)
        e8 = ((scales.view(np.int32) >> 23) & 0xFF).astype(np.uint8)      # exact powers of two
        return oracle.rows_fp8_e8m0(codes, e8, cfg.head_dim, cfg.scale_block, inv)
    blocks = synth.table_q2k_rows(cfg, layer, uniq)
    return oracle.rows_q2k(blocks, inv)


def x_of(cfg, layer, row_ids) -> np.ndarray:
    """x [M, K] bf16 bits from row ids [M, L, C]: the C rows concatenated in column order."""
    M = row_ids.shape[0]
    r = rows(cfg, layer, row_ids[:, layer, :].reshape(-1))
    return r.reshape(M, cfg.cols * cfg.head_dim)


def wkv(cfg, layer, out_rows) -> np.ndarray:
    """wkv rows [len(out_rows), K] as bf16 bits; with Q2_K wkv, the oracle's
    decode of the row's K / 256 blocks."""
    out_rows = np.asarray(out_rows, dtype=np.int64).ravel()
    if getattr(cfg, "wkv_fmt", "bf16") == "q2k":
        nb = cfg.K // 256
        blk_ids = (out_rows[:, None] * nb + np.arange(nb)[None, :]).ravel()
        blocks = synth.table_q2k_rows(cfg, layer, blk_ids, tag="wkvq2k")
        return oracle.rows_q2k(blocks, np.arange(blk_ids.size)).reshape(out_rows.size, cfg.K)
    return synth.wkv_rows(cfg, layer, out_rows)


_WKV_FULL = {}


def wkv_full(cfg, layer) -> np.ndarray:
    """All N rows of wkv (bf16 bits), regenerated on the CPU once per
    (seed, layer, shape, format) and kept for the session."""
    key = (cfg.seed, layer, cfg.N, cfg.K, getattr(cfg, "wkv_fmt", "bf16"))
    w = _WKV_FULL.get(key)
    if w is None:
        if len(_WKV_FULL) >= 4:
            _WKV_FULL.clear()
        w = wkv(cfg, layer, np.arange(cfg.N))
        _WKV_FULL[key] = w
    return w


def kv(cfg, layer, x_bits, out_rows=None) -> np.ndarray:
    """kv [M, len(out_rows)] bf16 bits; out_rows defaults to all N outputs."""
    if out_rows is None:
        return oracle.linear_bf16(x_bits, wkv_full(cfg, layer))
    return oracle.linear_bf16(x_bits, wkv(cfg, layer, out_rows))


def e2e_highway(cfg, h0, kv_gpu, kv_orc, h_gpu):
    """The end-to-end highway check: the oracle's gates run on the oracle's
    own kv (kv_orc, one [M, N] bf16 array a layer) from h0, and the GPU's
    highway h_gpu is compared with that result against the bound the
    projection's rounding allows.  With the stage-wise chain s (the oracle's
    gates on the GPU's kv, kv_gpu) and the end-to-end chain o, layer l adds
    sigma_s v_s - sigma_o v_o = sigma_s (v_s - v_o) + (sigma_s - sigma_o) v_o
    to the difference of the two chains, so

      |h_gpu - h_o| <= |h_gpu - h_s| + sum_l (sigma_s |dv| + |dsigma| |v_o|) + rounding

    with |h_gpu - h_s| <= H_TOL (the stage-wise bar) and the rounding of the
    two chains' f32 updates (a half-ulp of each product sigma v and of each
    sum, per chain and layer).  Returns (max |h_gpu - h_o|, the smallest bound - |h_gpu - h_o|)."""
    q_k = [synth.qk_weights(cfg, l) for l in range(cfg.n_layers)]
    hs = np.array(h0, dtype=np.float32, copy=True)
    ho = hs.copy()
    D, hc = cfg.dim, cfg.hc
    bound = np.full(hs.shape, H_TOL, dtype=np.float64)
    for l in range(cfg.n_layers):
        q, k = q_k[l]
        hs_n, gs = oracle.gate(hs, kv_gpu[l], q, k, hc, D, cfg.eps, return_gate=True)
        ho_n, go = oracle.gate(ho, kv_orc[l], q, k, hc, D, cfg.eps, return_gate=True)
        vs = oracle.bf16_bits_to_f32(np.asarray(kv_gpu[l])[:, hc * D:]).astype(np.float64)
        vo = oracle.bf16_bits_to_f32(np.asarray(kv_orc[l])[:, hc * D:]).astype(np.float64)
        gs64, go64 = gs.astype(np.float64), go.astype(np.float64)
        bound += (gs64[:, :, None] * np.abs(vs - vo)[:, None, :]
                  + np.abs(gs64 - go64)[:, :, None] * np.abs(vo)[:, None, :]
                  + 2.0 ** -24 * (np.abs(hs_n) + np.abs(ho_n)
                                  + gs64[:, :, None] * np.abs(vs)[:, None, :]
                                  + go64[:, :, None] * np.abs(vo)[:, None, :]))
        hs, ho = hs_n, ho_n
    dh = np.abs(np.asarray(h_gpu, dtype=np.float64) - ho)
    return float(dh.max()), float((bound - dh).min())


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

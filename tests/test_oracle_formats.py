"""Pins of the oracle's number formats and table-row decoders (CPU only).

e4m3 decode/encode, bf16 and binary16 are checked against library routines
(torch / numpy conversions), e8m0 against an exact rational rule, fp8 rows
against the exactness of e4m3 x 2^k in bf16, and Q2_K rows against a block
decoded by hand (tests/golden/q2k_hand.json).
"""
import json
import os
from fractions import Fraction

import numpy as np
import torch

from conftest import GOLDEN


def _torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_all_codes(orc):
    ref = _torch_e4m3_values()
    for b in range(256):
        v = orc.e4m3_to_f32(b)
        if np.isnan(ref[b]):
            assert np.isnan(v), b
        else:
            assert v == ref[b] and np.signbit(v) == np.signbit(ref[b]), b


def test_e4m3_encode_matches_library_rne(orc):
    vals = _torch_e4m3_values()
    finite = np.sort(np.unique(np.abs(vals[~np.isnan(vals)])))
    mids = (finite[:-1] + finite[1:]) / 2                 # exact ties
    xs = np.concatenate([finite, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                         np.random.default_rng(0).uniform(0, 448, 4000)]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.f32_to_e4m3(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # the page's own rules beyond the library's range
    assert orc.f32_to_e4m3(500.0) == 0x7E and orc.f32_to_e4m3(-1e30) == 0xFE
    assert orc.f32_to_e4m3(float("nan")) == 0x7F
    assert orc.f32_to_e4m3(1e-40) == 0x00 and orc.f32_to_e4m3(-1e-40) == 0x80


def test_e4m3_round_trip(orc):
    for b in range(256):
        if b & 0x7F == 0x7F:
            continue
        assert orc.f32_to_e4m3(orc.e4m3_to_f32(b)) == b


def test_bf16_matches_library(orc):
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 10.0 ** rng.integers(-40, 38, 3000),
                         np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, np.inf, -np.inf,
                                   3.3895314e38, 1e-45, -1e-39], dtype=np.float32)]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # a NaN stays a NaN whatever its sign and payload (IEEE 754 conversion); the
    # library returns one canonical NaN, so only NaN-ness is compared
    nans = np.array([0x7FC00000, 0x7FFFFFFF, 0xFFFFFFFF, 0xFFC00001, 0x7FC0FFFF], dtype=np.uint32).view(np.float32)
    for x in nans:
        b = orc.f32_to_bf16(float(x))
        assert (b & 0x7F80) == 0x7F80 and (b & 0x007F) != 0, hex(b)


def test_f16_decode_all_codes(orc):
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    for h in range(0, 65536, 7):
        v = orc.f16_to_f32(h)
        assert (np.isnan(v) and np.isnan(ref[h])) or (v == ref[h] and np.signbit(v) == np.signbit(ref[h])), h


def test_e8m0_nearest_power_ties_to_even_code(orc):
    rng = np.random.default_rng(2)
    xs = list(np.float32(rng.uniform(0.01, 100, 500))) + [np.float32(1.5 * 2.0 ** e) for e in range(-10, 10)]
    for x in xs:
        fx = Fraction(float(x))
        e = int(np.floor(np.log2(float(x))))
        lo, hi = Fraction(2) ** e, Fraction(2) ** (e + 1)
        if fx - lo < hi - fx:
            want = lo
        elif fx - lo > hi - fx:
            want = hi
        else:                                  # tie: the even biased code
            want = lo if (e + 127) % 2 == 0 else hi
        assert Fraction(orc.f32_to_e8m0(float(x))) == want, x


def test_fp8_rows_exact_for_every_code_and_scale(orc):
    """e4m3 value x 2^k is bf16-exact (CPU reference page, `regen_table`):
    every non-NaN code times every 2^k, k in [-10, 10]."""
    codes = np.array([b for b in range(256) if b & 0x7F != 0x7F], dtype=np.uint8)
    hd = 256
    table = np.zeros((21, hd), dtype=np.uint8)
    table[:, :codes.size] = codes
    scales = np.array([[2.0 ** k] * (hd // 32) for k in range(-10, 11)], dtype=np.float32)
    out = orc.rows_fp8(table, scales, hd, 32, np.arange(21))
    vals = _torch_e4m3_values()
    for r, k in enumerate(range(-10, 11)):
        want = vals[codes].astype(np.float64) * 2.0 ** k
        got = orc.bf16_bits_to_f32(out[r, :codes.size]).astype(np.float64)
        assert np.array_equal(got, want)
        assert np.array_equal(np.signbit(got), np.signbit(want))


def test_fp8_rows_scale_blocks_and_gather(orc):
    """Scale block d // blk, row gather by id (repeated ids, order kept)."""
    hd, blk = 64, 16
    table = np.full((5, hd), 0x38, dtype=np.uint8)        # 1.0 everywhere
    scales = np.array([[2.0 ** (r + b) for b in range(hd // blk)] for r in range(5)], dtype=np.float32)
    out = orc.bf16_bits_to_f32(orc.rows_fp8(table, scales, hd, blk, [3, 0, 3]))
    for i, r in enumerate([3, 0, 3]):
        assert np.array_equal(out[i], np.repeat(2.0 ** (r + np.arange(hd // blk)), blk))


def test_q2k_hand_decoded_block(orc):
    g = json.load(open(os.path.join(GOLDEN, "q2k_hand.json")))
    blk = np.frombuffer(bytes.fromhex(g["block_hex"]), dtype=np.uint8)[None, :]
    out = orc.bf16_bits_to_f32(orc.rows_q2k(blk, [0]))[0]
    for v, want in g["expected"].items():
        assert out[int(v)] == want, (v, out[int(v)], want)


def test_q2k_gather_and_bounds(orc):
    g = json.load(open(os.path.join(GOLDEN, "q2k_hand.json")))
    blk = np.frombuffer(bytes.fromhex(g["block_hex"]), dtype=np.uint8)
    zero = np.zeros(84, dtype=np.uint8)
    blocks = np.stack([zero, blk, zero])
    out = orc.rows_q2k(blocks, [1, 0])
    assert np.array_equal(out[0], orc.rows_q2k(blk[None], [0])[0])
    assert not out[1].any()
    import pytest
    with pytest.raises(ValueError):
        orc.rows_q2k(blocks, [3])


def test_e8m0_decode_exact_powers(orc):
    """code c -> 2^(c - 127) exactly (c = 0 is the f32 subnormal 2^-127), 255 -> NaN;
    and the page's encoder maps every such power back to itself."""
    for c in range(255):
        v = orc.e8m0_to_f32(c)
        assert Fraction(v) == Fraction(2) ** (c - 127), c
        if c >= 1:
            assert orc.f32_to_e8m0(v) == v
    assert np.isnan(orc.e8m0_to_f32(255))


def test_fp8_rows_e8m0_scales_exact(orc):
    """One-byte scales give the float64 product e4m3 x 2^(code-127) exactly."""
    codes = np.array([b for b in range(256) if b & 0x7F != 0x7F], dtype=np.uint8)
    hd, blk = 256, 32
    table = np.zeros((15, hd), dtype=np.uint8)
    table[:, :codes.size] = codes
    sc = np.array([[117 + r] * (hd // blk) for r in range(15)], dtype=np.uint8)   # 2^-10 .. 2^4
    out = orc.rows_fp8_e8m0(table, sc, hd, blk, np.arange(15))
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for r in range(15):
        want = vals[codes].astype(np.float64) * 2.0 ** (r - 10)
        got = orc.bf16_bits_to_f32(out[r, :codes.size]).astype(np.float64)
        assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))

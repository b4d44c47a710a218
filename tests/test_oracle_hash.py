"""Pins of the oracle's n-gram hash (CPU only).

The hash follows `NgramHashState::forward` on the CPU reference page
"metrale_model_arch/deepseek_v41_ref/engram.rs".  It is pinned by hand-worked
windows (tests/golden/hash_hand.json), by brute force over every window of a
tiny vocabulary against an independent Python big-integer statement, by the
range invariant, by the split/one-shot equivalence and by window locality.
"""
import itertools
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import hash_bigint


def _state(orc, case, B=1, max_seq=64, L=1):
    return orc.HashState(case["token_map"], case["token_map"][case["pad_token_id"]],
                         case["multipliers"], case["primes"], case["offsets"], L,
                         case["max_ngram"], case["n_heads"], B, max_seq)


@pytest.mark.parametrize("idx", [0, 1])
def test_hand_worked_windows(orc, idx):
    case = json.load(open(os.path.join(GOLDEN, "hash_hand.json")))["cases"][idx]
    st = _state(orc, case)
    out = st.forward(np.array([case["ids"]]), case["start_pos"])
    assert out[0, :, 0, :].tolist() == case["expected"]


def test_brute_force_tiny_vocab(orc):
    """Every length-4 sequence over an 8-token vocabulary (with -1 entries),
    two layers, trigram, two heads, multipliers that overflow i64."""
    token_map = [0, 1, 2, 3, 4, 5, -1, -1]
    ng, H, L = 3, 2, 2
    rng = np.random.default_rng(7)
    mult = [int(v) | 1 for v in rng.integers(1 << 40, 1 << 62, size=L * ng)]
    mult[1] = -mult[1]                      # a negative multiplier too
    primes = [5, 7, 11, 13, 17, 19, 23, 29]
    offsets = [0, 5, 12, 23, 0, 17, 36, 59]
    seqs = np.array(list(itertools.product(range(8), repeat=4)), dtype=np.int64)
    st = orc.HashState(token_map, 0, mult, primes, offsets, L, ng, H, len(seqs), 4)
    out = st.forward(seqs, 0)
    for b in range(0, len(seqs), 37):       # every 37th sequence in Python big ints
        ref = hash_bigint.hash_sequence(token_map, 0, mult, primes, offsets, L, ng, H, seqs[b])
        assert out[b].tolist() == ref, f"sequence {seqs[b].tolist()}"


def test_ids_in_slot_range_v41(orc):
    """Every id of column c lies in [offset_c, offset_c + prime_c)."""
    from deepseek_v4_engram_hash_gb300 import configs, synth
    cfg = configs.V41_DECODE
    t = synth.hash_tables(cfg)
    ids = synth.token_ids(cfg, "range", 3000)[None, :]
    st = orc.HashState(t["token_map"], t["pad_id"], t["multipliers"], t["primes"],
                       t["offsets"], cfg.n_layers, cfg.max_ngram, cfg.n_heads, 1, 4096)
    out = st.forward(ids, 0)[0]                      # [T, L, C]
    lo = t["offsets"].reshape(cfg.n_layers, cfg.cols)
    hi = lo + t["primes"].reshape(cfg.n_layers, cfg.cols)
    assert (out >= lo[None]).all() and (out < hi[None]).all()
    # the hash spreads: most slots are hit by many distinct ids
    assert len(np.unique(out[:, 0, 0])) > 2000


def test_prefill_decode_split_equals_one_shot(orc):
    from deepseek_v4_engram_hash_gb300 import configs, synth
    cfg = configs.TINY
    t = synth.hash_tables(cfg)
    B, T = 3, 40
    ids = np.stack([synth.token_ids(cfg, f"split{b}", T) for b in range(B)])
    mk = lambda: orc.HashState(t["token_map"], t["pad_id"], t["multipliers"], t["primes"],
                               t["offsets"], cfg.n_layers, cfg.max_ngram, cfg.n_heads, B, 64)
    one = mk().forward(ids, 0)
    st = mk()
    parts = [st.forward(ids[:, a:b], a) for a, b in ((0, 17), (17, 18), (18, 19), (19, 40))]
    assert np.array_equal(np.concatenate(parts, axis=1), one)


def test_window_locality(orc):
    """Position p depends on the ids at p-ng+1 .. p only."""
    from deepseek_v4_engram_hash_gb300 import configs, synth
    cfg = configs.V41_DECODE
    t = synth.hash_tables(cfg)
    ids = synth.token_ids(cfg, "loc", 12)
    mk = lambda: orc.HashState(t["token_map"], t["pad_id"], t["multipliers"], t["primes"],
                               t["offsets"], cfg.n_layers, cfg.max_ngram, cfg.n_heads, 1, 16)
    base = mk().forward(ids[None], 0)[0]
    far = ids.copy()
    far[:8] = (far[:8] + 1) % cfg.vocab                # positions <= 7 change
    out = mk().forward(far[None], 0)[0]
    assert np.array_equal(out[11], base[11])           # window of 11 is 8..11
    near = ids.copy()
    near[8] = (near[8] + 1) % cfg.vocab
    out2 = mk().forward(near[None], 0)[0]
    assert not np.array_equal(out2[11, :, 2 * cfg.n_heads:], base[11, :, 2 * cfg.n_heads:])
    assert np.array_equal(out2[11, :, :2 * cfg.n_heads], base[11, :, :2 * cfg.n_heads])


def test_fresh_cache_reads_zero_lookback(orc):
    """A fresh cache holds 0 (not -1): hashing one token at start_pos 5 sees
    compressed id 0 behind it."""
    case = json.load(open(os.path.join(GOLDEN, "hash_hand.json")))["cases"][0]
    st = _state(orc, case, max_seq=8)
    out = st.forward(np.array([[2]]), 5)[0, 0, 0]
    win = hash_bigint.window([0, 0, 0, 0, 0, 3], 5, 3, 0)
    assert win == [3, 0, 0]
    ref = hash_bigint.hash_window(win, case["multipliers"], case["primes"], case["offsets"], 2)
    assert out.tolist() == ref


def test_errors(orc):
    case = json.load(open(os.path.join(GOLDEN, "hash_hand.json")))["cases"][0]
    st = _state(orc, case, max_seq=4)
    with pytest.raises(ValueError, match="-1"):
        st.forward(np.array([[1, 2, 3, 4, 5]]), 0)       # capacity
    with pytest.raises(ValueError, match="-2"):
        st.forward(np.array([[6]]), 0)                   # outside token_map
    with pytest.raises(ValueError, match="-2"):
        st.forward(np.array([[-1]]), 0)
    bad = dict(case, primes=[11, 0, 17, 19])
    with pytest.raises(ValueError, match="-4"):
        _state(orc, bad).forward(np.array([[1]]), 0)

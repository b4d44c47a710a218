"""Second, independent statement of the engram n-gram hash, in Python integers.

TEST INFRASTRUCTURE.  It pins the C oracle's hash: Python integers do not
overflow, so the i64 wrap is written as an explicit reduction mod 2**64 and a
re-signing, and Python's ``%`` is already the Euclidean remainder for a
positive modulus.  Neither the C oracle nor the CUDA path is used here.

Follows `NgramHashState::forward` on the CPU reference page
"metrale_model_arch/deepseek_v41_ref/engram.rs".
"""
from __future__ import annotations

_M64 = 1 << 64


def to_i64(v: int) -> int:
    """Reduce an integer to the signed 64-bit two's-complement range."""
    v %= _M64
    return v - _M64 if v >= (1 << 63) else v


def window(cache_row, pos: int, ng: int, pad_id: int) -> list:
    """The ng compressed ids at shifts 0..ng-1 behind `pos` (shift 0 = pos)."""
    out = []
    blocked = False
    for shift in range(ng):
        src = cache_row[max(pos - shift, 0)]
        blocked = blocked or pos < shift or src == -1
        out.append(pad_id if blocked else src)
    return out


def hash_window(tokens, mult_layer, primes_layer, offsets_layer, n_heads: int) -> list:
    """Row ids of one layer for one window: [(ng - 1) * n_heads]."""
    ng = len(tokens)
    ids = [0] * ((ng - 1) * n_heads)
    rolling = to_i64(tokens[0] * mult_layer[0])
    for n in range(1, ng):
        rolling = to_i64(rolling ^ to_i64(tokens[n] * mult_layer[n]))
        for h in range(n_heads):
            col = (n - 1) * n_heads + h
            ids[col] = (rolling % primes_layer[col]) + offsets_layer[col]
    return ids


def hash_sequence(token_map, pad_id, multipliers, primes, offsets, n_layers, max_ngram,
                  n_heads, seq_ids) -> list:
    """One-shot hash of a whole sequence from position 0 with a zeroed cache.

    multipliers [L * ng], primes / offsets [L * C] (flat, as the GGUF metadata
    ships them).  Returns [T][L][C].
    """
    ng, C = max_ngram, (max_ngram - 1) * n_heads
    cache = [int(token_map[int(t)]) for t in seq_ids]
    out = []
    for pos in range(len(cache)):
        toks = window(cache, pos, ng, int(pad_id))
        per_layer = []
        for li in range(n_layers):
            m = [int(v) for v in multipliers[li * ng:(li + 1) * ng]]
            p = [int(v) for v in primes[li * C:(li + 1) * C]]
            o = [int(v) for v in offsets[li * C:(li + 1) * C]]
            per_layer.append(hash_window(toks, m, p, o, n_heads))
        out.append(per_layer)
    return out

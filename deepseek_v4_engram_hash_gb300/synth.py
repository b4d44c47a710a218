"""Seeded synthetic inputs for the engram forward (numpy and CUDA twins).

This module is the ONLY code that both the CPU oracle's tests and the CUDA path
draw on, and it holds none of the method's arithmetic: it draws integers from a
counter-based generator and converts them with library routines (numpy, torch
and CUDA's own float16 / bfloat16 / fp8 conversions).

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: element `i` of a stream
with key `k` is the mix of `k + (i + 1) * 0x9E3779B97F4A7C15`.  Any single
element of any input can therefore be regenerated on its own, which lets the
oracle rebuild only the table rows and weight rows it checks.

Normal variates are N(0, 1) by the Box-Muller transform (Box & Muller, "A note
on the generation of random normal deviates", Ann. Math. Stat. 1958) of one
64-bit output: u1 = (high 32 bits + 1) / 2^32 in (0, 1], u2 = low 32 bits /
2^32, z = sqrt(-2 ln u1) cos(2 pi u2), so |z| <= 6.66.  The logarithm and the
cosine are evaluated here in float64 from their series with a fixed sequence of
correctly rounded IEEE operations (no fused multiply-add) -- ln m = 2 atanh(s),
s = (m - 1) / (m + 1), after an exact reduction of u1 to m in [sqrt(1/2),
sqrt(2)); cos and sin of (pi/2) f, |f| <= 1/2, after an exact reduction of
4 u2 by its nearest integer -- so that the CUDA twin, doing the same
operations, gets the same bits; the result is rounded to f32 and scaled to the
requested sigma by one f32 multiply.  (Library log and cos may differ in the
last place between machines; these do not.)  Every other step is integer or a
single correctly rounded IEEE operation, so the numpy and CUDA twins produce
the same bits on any machine.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1

# Float64 constants of the Box-Muller evaluation, written as exact binary
# values (the CUDA twin holds the same literals): ln 2, pi / 2, sqrt(1/2), and
# the series coefficients 1 / (2k + 1) (atanh), (-1)^k / (2k)! (cos) and
# (-1)^k / (2k + 1)! (sin), each the double nearest the exact rational.
_LN2 = float.fromhex("0x1.62e42fefa39efp-1")
_PI_2 = float.fromhex("0x1.921fb54442d18p+0")
_SQRT_HALF = float.fromhex("0x1.6a09e667f3bcdp-1")
_ATANH = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "0x1.5555555555555p-2", "0x1.999999999999ap-3", "0x1.2492492492492p-3",
    "0x1.c71c71c71c71cp-4", "0x1.745d1745d1746p-4", "0x1.3b13b13b13b14p-4", "0x1.1111111111111p-4",
    "0x1.e1e1e1e1e1e1ep-5", "0x1.af286bca1af28p-5", "0x1.8618618618618p-5")]
_COS = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.0000000000000p-1", "0x1.5555555555555p-5", "-0x1.6c16c16c16c17p-10",
    "0x1.a01a01a01a01ap-16", "-0x1.27e4fb7789f5cp-22", "0x1.1eed8eff8d898p-29", "-0x1.93974a8c07c9dp-37",
    "0x1.ae7f3e733b81fp-45", "-0x1.6827863b97d97p-53")]
_SIN = [float.fromhex(h) for h in (
    "0x1.0000000000000p+0", "-0x1.5555555555555p-3", "0x1.1111111111111p-7", "-0x1.a01a01a01a01ap-13",
    "0x1.71de3a556c734p-19", "-0x1.ae64567f544e4p-26", "0x1.6124613a86d09p-33", "-0x1.ae7f3e733b81fp-41",
    "0x1.952c77030ad4ap-49", "-0x1.2f49b46814157p-57")]


# ---------------------------------------------------------------------------
# SplitMix64
# ---------------------------------------------------------------------------

def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def _fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h = ((h ^ b) * 0x100000001B3) & _M64
    return h


def stream_key(seed: int, tag: str) -> int:
    """The 64-bit key of the named input stream under `seed`."""
    return _mix64_int(((seed * GAMMA) & _M64) ^ _fnv1a64(tag))


def splitmix64(key: int, idx) -> np.ndarray:
    """Element(s) `idx` of the SplitMix64 stream keyed `key` (uint64 array)."""
    i = np.atleast_1d(np.asarray(idx, dtype=np.uint64))
    z = (i + np.uint64(1)) * np.uint64(GAMMA) + np.uint64(key)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def normal_scale(sigma: float) -> np.float32:
    """The f32 constant that scales a standard normal to std `sigma`."""
    return np.float32(sigma)


def std_normal_f64(z) -> np.ndarray:
    """N(0, 1) from SplitMix64 outputs z (uint64) by Box-Muller, in float64 with
    the fixed operation sequence the CUDA twin repeats (in-place numpy ops
    round exactly as the separate ones would)."""
    z = np.asarray(z, dtype=np.uint64)
    # -2 ln u1, u1 = (a + 1) 2^-32: n = a + 1 = m0 2^e exactly, m0 in [sqrt(1/2), sqrt(2))
    nd = ((z >> np.uint64(32)) + np.uint64(1)).astype(np.float64)
    m0, e = np.frexp(nd)
    low = m0 < _SQRT_HALF
    m0[low] *= 2.0
    e = e.astype(np.float64)
    e[low] -= 1.0
    s = m0 - 1.0
    m0 += 1.0
    s /= m0
    s2 = s * s
    p = np.full_like(s, _ATANH[10])
    for k in range(9, -1, -1):
        p *= s2
        p += _ATANH[k]
    p *= s
    p *= 2.0                          # ln m
    e -= 32.0
    e *= _LN2
    e += p                            # ln u1
    e *= -2.0
    r = np.sqrt(e, out=e)
    # cos(2 pi u2) = cos((pi/2) w), w = 4 u2 = b 2^-30 = q + f, q the nearest integer
    w = (z & np.uint64(0xFFFFFFFF)).astype(np.float64)
    w *= 2.0 ** -30
    q = np.floor(w + 0.5)
    w -= q                            # f
    w *= _PI_2                        # x
    x2 = w * w
    c = np.full_like(w, _COS[9])
    sn = np.full_like(w, _SIN[9])
    for k in range(8, -1, -1):
        c *= x2
        c += _COS[k]
        sn *= x2
        sn += _SIN[k]
    sn *= w
    qi = q.astype(np.int64)
    odd = (qi & 1).astype(bool)
    c[odd] = sn[odd]
    neg = (qi == 1) | (qi == 2)
    c[neg] = -c[neg]
    r *= c
    return r


def normal_f32(key: int, idx, sigma: float) -> np.ndarray:
    """N(0, sigma^2) as f32: the float64 standard normal rounded to f32, times sigma."""
    return std_normal_f64(splitmix64(key, idx)).astype(np.float32) * normal_scale(sigma)


def _torch():
    import torch
    return torch


def to_bf16_bits(x) -> np.ndarray:
    """f32 -> bf16 bit patterns by torch's round-to-nearest-even conversion."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x) -> np.ndarray:
    """f32 (|x| <= 448) -> e4m3fn codes by torch's round-to-nearest-even conversion."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ---------------------------------------------------------------------------
# Hash tables
# ---------------------------------------------------------------------------

def _is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    f = 3
    while f * f <= n:
        if n % f == 0:
            return False
        f += 2
    return True


def primes_from(target: int, count: int) -> list:
    """The first `count` primes >= target, ascending."""
    out, n = [], max(2, target)
    while len(out) < count:
        if _is_prime(n):
            out.append(n)
        n += 1
    return out


def hash_tables(cfg) -> dict:
    """token_map, pad id, multipliers, per-slot primes and cumulative offsets.

    primes: the first L*C primes >= cfg.prime_target, assigned in (layer,
    n-gram, head) order.  offsets[l][c] = sum of the primes of the earlier
    columns of layer l, so each layer's table has rows_per_layer[l] rows.
    """
    L, ng, C = cfg.n_layers, cfg.max_ngram, cfg.cols
    v = np.arange(cfg.vocab, dtype=np.uint64)
    z = splitmix64(stream_key(cfg.seed, "token_map"), v)
    tm = ((z & np.uint64(0xFFFFFFFF)) % np.uint64(cfg.n_compressed)).astype(np.int64)
    if cfg.unmapped_5pct:
        tm[((z >> np.uint64(32)) % np.uint64(20)) == 0] = -1
    if cfg.pad_compressed is not None:
        tm[cfg.pad_token_id] = cfg.pad_compressed
    zm = splitmix64(stream_key(cfg.seed, "mult"), np.arange(L * ng, dtype=np.uint64))
    mult = ((zm >> np.uint64(2)) | np.uint64(1)).astype(np.int64)
    primes = np.array(primes_from(cfg.prime_target, L * C), dtype=np.int64).reshape(L, C)
    offsets = np.zeros((L, C), dtype=np.int64)
    offsets[:, 1:] = np.cumsum(primes[:, :-1], axis=1)
    rows = primes.sum(axis=1)
    return dict(token_map=tm, pad_token_id=cfg.pad_token_id, pad_id=int(tm[cfg.pad_token_id]),
                multipliers=mult, primes=primes.reshape(-1), offsets=offsets.reshape(-1),
                rows_per_layer=[int(r) for r in rows])


def token_ids(cfg, tag: str, n: int) -> np.ndarray:
    """n token ids (int32): Zipf(s) over ranks 1..vocab (id = rank - 1) by
    inverse-CDF sampling, or uniform."""
    z = splitmix64(stream_key(cfg.seed, "ids." + tag), np.arange(n, dtype=np.uint64))
    if cfg.ids == "uniform":
        return (z % np.uint64(cfg.vocab)).astype(np.int32)
    w = np.arange(1, cfg.vocab + 1, dtype=np.float64) ** (-cfg.zipf_s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.minimum(np.searchsorted(cdf, u, side="right"), cfg.vocab - 1).astype(np.int32)


# ---------------------------------------------------------------------------
# Tables, weights, highway (numpy twins; any subset of rows)
# ---------------------------------------------------------------------------

def _chunked(n: int, step: int, fn) -> None:
    """fn(a, b) over [0, n) in chunks of `step`, on a few threads when there
    are several chunks (numpy and torch release the GIL on large arrays; each
    chunk writes its own slice, so the result does not depend on the order)."""
    starts = list(range(0, n, step))
    if len(starts) <= 1:
        for a in starts:
            fn(a, min(n, a + step))
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1, 16)) as ex:
        list(ex.map(lambda a: fn(a, min(n, a + step)), starts))


def table_fp8_rows(cfg, layer: int, rows):
    """Rows of layer `layer`'s fp8 table: codes [n, hd] u8 and scales [n, hd/blk] f32.

    Values are e4m3(N(0,1)) (never near the +-448 clamp); scales are 2^k,
    k uniform in {-4..2}, per scale_block values."""
    rows = np.atleast_1d(np.asarray(rows, dtype=np.uint64)).ravel()
    hd, nb = cfg.head_dim, cfg.head_dim // cfg.scale_block
    codes = np.empty((rows.size, hd), dtype=np.uint8)
    scales = np.empty((rows.size, nb), dtype=np.float32)
    kt, ks = stream_key(cfg.seed, f"table.{layer}"), stream_key(cfg.seed, f"scales.{layer}")

    def fill(a, b):
        r = rows[a:b]
        idx = r[:, None] * np.uint64(hd) + np.arange(hd, dtype=np.uint64)[None, :]
        x = normal_f32(kt, idx, 1.0)
        codes[a:b] = to_e4m3_codes(np.clip(x, -448.0, 448.0)).reshape(r.size, hd)
        sidx = r[:, None] * np.uint64(nb) + np.arange(nb, dtype=np.uint64)[None, :]
        k = (splitmix64(ks, sidx) % np.uint64(7)).astype(np.int64) - 4
        scales[a:b] = ((k + 127) << 23).astype(np.uint32).view(np.float32).reshape(r.size, nb)

    _chunked(rows.size, max(1, (1 << 20) // hd), fill)
    return codes, scales


Q2K_D_LO = np.float32(1e-3)
Q2K_D_STEP = np.float32(9e-3 / (1 << 24))


def table_q2k_rows(cfg, layer: int, rows, tag: str = "q2k") -> np.ndarray:
    """Rows of layer `layer`'s Q2_K table: [n, 84] u8.  Bytes 0..79 (sub-block
    scale/min nibbles and 2-bit quants) uniform; d and dmin uniform in
    (1e-3, 1e-2), stored as binary16.  tag "wkvq2k" gives Q2_K wkv blocks
    ([N * K / 256] of them, a row's blocks contiguous)."""
    rows = np.atleast_1d(np.asarray(rows, dtype=np.uint64)).ravel()
    key = stream_key(cfg.seed, f"{tag}.{layer}")
    idx = rows[:, None] * np.uint64(12) + np.arange(12, dtype=np.uint64)[None, :]
    z = splitmix64(key, idx).reshape(rows.size, 12)
    out = np.zeros((rows.size, 84), dtype=np.uint8)
    out[:, :80] = np.ascontiguousarray(z[:, :10]).astype("<u8").view(np.uint8).reshape(rows.size, 80)
    u = (z[:, 10:12] >> np.uint64(40)).astype(np.float32)
    d = (u * Q2K_D_STEP + Q2K_D_LO).astype(np.float16)
    out[:, 80:84] = np.ascontiguousarray(d).astype("<f2").view(np.uint8).reshape(rows.size, 4)
    return out


def wkv_rows(cfg, layer: int, rows, sigma: float = 0.02) -> np.ndarray:
    """Rows of wkv [N, K] as bf16 bits, N(0, sigma^2)."""
    rows = np.atleast_1d(np.asarray(rows, dtype=np.uint64)).ravel()
    K = cfg.K
    key = stream_key(cfg.seed, f"wkv.{layer}")
    out = np.empty((rows.size, K), dtype=np.uint16)

    def fill(a, b):
        r = rows[a:b]
        idx = r[:, None] * np.uint64(K) + np.arange(K, dtype=np.uint64)[None, :]
        out[a:b] = to_bf16_bits(normal_f32(key, idx, sigma)).reshape(r.size, K)

    _chunked(rows.size, max(1, (1 << 20) // K), fill)
    return out


def qk_weights(cfg, layer: int):
    """q and k [hc, dim] as f32 values of bf16: bf16(1 + 0.05 N(0,1))."""
    n = cfg.hc * cfg.dim
    out = []
    for name in ("q", "k"):
        a = normal_f32(stream_key(cfg.seed, f"{name}.{layer}"), np.arange(n, dtype=np.uint64), 0.05)
        bits = to_bf16_bits(a + np.float32(1.0))
        out.append((bits.astype(np.uint32) << 16).view(np.float32).reshape(cfg.hc, cfg.dim))
    return out[0], out[1]


def highway(cfg, tokens, tag: str = "h") -> np.ndarray:
    """h [len(tokens), hc, dim] f32 N(0,1) for the given global token indices."""
    tokens = np.atleast_1d(np.asarray(tokens, dtype=np.uint64)).ravel()
    w = cfg.hc * cfg.dim
    idx = tokens[:, None] * np.uint64(w) + np.arange(w, dtype=np.uint64)[None, :]
    return normal_f32(stream_key(cfg.seed, tag), idx, 1.0).reshape(tokens.size, cfg.hc, cfg.dim)


# ---------------------------------------------------------------------------
# CUDA twin (libengram_synth.so): fills whole device buffers
# ---------------------------------------------------------------------------

_SYNTH = None


def _synth_lib():
    global _SYNTH
    if _SYNTH is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libengram_synth.so")
        if not os.path.exists(path):
            raise RuntimeError("libengram_synth.so is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        u64, i64, P, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
        L.synth_fp8_table.argtypes = [u64, u64, i64, ctypes.c_int, ctypes.c_int, f32, P, P, P]
        L.synth_q2k_table.argtypes = [u64, i64, f32, f32, P, P]
        L.synth_bf16_normal.argtypes = [u64, i64, f32, P, P]
        L.synth_f32_normal.argtypes = [u64, i64, i64, f32, P, P]
        for f in (L.synth_fp8_table, L.synth_q2k_table, L.synth_bf16_normal, L.synth_f32_normal):
            f.restype = ctypes.c_int
        _SYNTH = L
    return _SYNTH


def _stream_of(t):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def fill_table_fp8_cuda(cfg, layer: int, codes, scales):
    """codes: uint8 CUDA tensor [R, hd]; scales: float32 CUDA tensor [R, hd/blk]."""
    _check(_synth_lib().synth_fp8_table(
        stream_key(cfg.seed, f"table.{layer}"), stream_key(cfg.seed, f"scales.{layer}"),
        codes.shape[0], cfg.head_dim, cfg.scale_block, float(normal_scale(1.0)),
        ctypes.c_void_p(codes.data_ptr()),
        ctypes.c_void_p(scales.data_ptr()), _stream_of(codes)), "synth_fp8_table")


def fill_table_q2k_cuda(cfg, layer: int, blocks, tag: str = "q2k"):
    """blocks: uint8 CUDA tensor [R, 84]."""
    _check(_synth_lib().synth_q2k_table(
        stream_key(cfg.seed, f"{tag}.{layer}"), blocks.shape[0], float(Q2K_D_STEP), float(Q2K_D_LO),
        ctypes.c_void_p(blocks.data_ptr()), _stream_of(blocks)), "synth_q2k_table")


def fill_wkv_cuda(cfg, layer: int, wkv, sigma: float = 0.02):
    """wkv: bfloat16 CUDA tensor [N, K]."""
    _check(_synth_lib().synth_bf16_normal(
        stream_key(cfg.seed, f"wkv.{layer}"), wkv.numel(), float(normal_scale(sigma)),
        ctypes.c_void_p(wkv.data_ptr()), _stream_of(wkv)), "synth_bf16_normal")


def fill_highway_cuda(cfg, h, first_token: int = 0, tag: str = "h"):
    """h: float32 CUDA tensor [n_tok, hc, dim] holding global tokens first_token.."""
    w = cfg.hc * cfg.dim
    _check(_synth_lib().synth_f32_normal(
        stream_key(cfg.seed, tag), first_token * w, h.numel(), float(normal_scale(1.0)),
        ctypes.c_void_p(h.data_ptr()), _stream_of(h)), "synth_f32_normal")

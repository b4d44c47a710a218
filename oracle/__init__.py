"""CPU oracle of the DeepSeek-V4.1 engram forward (test infrastructure).

This package is TEST INFRASTRUCTURE, not product code.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA path: ``oracle.c`` is plain scalar C
compiled by gcc, and ``hash_bigint.py`` is an independent Python big-integer
restatement of the hash used to pin it.

The functions follow the CPU reference page
"metrale_model_arch/deepseek_v41_ref/engram.rs" stage by stage; see the
comments in ``oracle.c`` for the equations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
E_CAPACITY = -1
E_TOKEN = -2
E_ROW = -3
E_PRIME = -4


def compile_source(src: str, out: str) -> str:
    """Compile the C source `src` into the shared library `out` with gcc
    (OpenMP if available), with the flags the oracle is built with."""
    tmp = out + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so``."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


def load(path: str) -> ctypes.CDLL:
    """The library at `path` (built from ``oracle.c`` or a copy of it) with
    the signatures of its functions declared."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    L.orc_num_threads.restype = i32
    L.orc_set_num_threads.argtypes = [i32]
    L.orc_set_num_threads.restype = None
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    L.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_to_f32.restype = ctypes.c_float
    L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
    L.orc_f32_to_e4m3.restype = ctypes.c_uint8
    L.orc_f32_to_e8m0.argtypes = [ctypes.c_float]
    L.orc_f32_to_e8m0.restype = ctypes.c_float
    L.orc_e8m0_to_f32.argtypes = [ctypes.c_uint8]
    L.orc_e8m0_to_f32.restype = ctypes.c_float
    L.orc_rows_fp8_e8m0.argtypes = [P, P, i64, i32, i32, P, i64, P]
    L.orc_rows_fp8_e8m0.restype = i32
    L.orc_hash.argtypes = [P, i64, i64, P, P, P, i32, i32, i32, P, i32, i64, P, i32, i64, P]
    L.orc_hash.restype = i32
    L.orc_rows_fp8.argtypes = [P, P, i64, i32, i32, P, i64, P]
    L.orc_rows_fp8.restype = i32
    L.orc_rows_q2k.argtypes = [P, i64, P, i64, P]
    L.orc_rows_q2k.restype = i32
    L.orc_linear_bf16.argtypes = [P, i64, i64, P, i64, P, P]
    L.orc_linear_bf16.restype = None
    L.orc_gate.argtypes = [P, P, P, P, i64, i32, i32, ctypes.c_float, i32, P]
    L.orc_gate.restype = None
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load(_LIB)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---- scalar codecs ---------------------------------------------------------

def f32_to_bf16(x: float) -> int:
    return int(lib().orc_f32_to_bf16(float(x)))


def bf16_to_f32(b: int) -> float:
    return float(lib().orc_bf16_to_f32(int(b)))


def f16_to_f32(b: int) -> float:
    return float(lib().orc_f16_to_f32(int(b)))


def e4m3_to_f32(b: int) -> float:
    return float(lib().orc_e4m3_to_f32(int(b)))


def f32_to_e4m3(x: float) -> int:
    return int(lib().orc_f32_to_e4m3(float(x)))


def f32_to_e8m0(x: float) -> float:
    return float(lib().orc_f32_to_e8m0(float(x)))


def e8m0_to_f32(code: int) -> float:
    return float(lib().orc_e8m0_to_f32(int(code)))


# ---- stages ----------------------------------------------------------------

class HashState:
    """The look-back cache of `NgramHashState` (zero-initialised) and its tables."""

    def __init__(self, token_map, pad_id, multipliers, primes, offsets,
                 n_layers, max_ngram, n_heads, batch, max_seq):
        self.token_map = _c(token_map, np.int64)
        self.pad_id = int(pad_id)
        self.mult = _c(multipliers, np.int64)
        self.primes = _c(primes, np.int64)
        self.offsets = _c(offsets, np.int64)
        self.L, self.ng, self.H = int(n_layers), int(max_ngram), int(n_heads)
        self.C = (self.ng - 1) * self.H
        self.B, self.max_seq = int(batch), int(max_seq)
        self.cache = np.zeros(self.B * self.max_seq, dtype=np.int64)

    def reset(self):
        self.cache[:] = 0

    def forward(self, ids, start_pos: int) -> np.ndarray:
        """ids [B, T] -> row ids [B, T, L, C] (int64)."""
        ids = _c(ids, np.int64)
        assert ids.ndim == 2 and ids.shape[0] == self.B
        T = ids.shape[1]
        out = np.zeros((self.B, T, self.L, self.C), dtype=np.int64)
        rc = lib().orc_hash(_p(self.token_map), self.token_map.size, self.pad_id,
                            _p(self.mult), _p(self.primes), _p(self.offsets),
                            self.L, self.ng, self.H, _p(self.cache), self.B, self.max_seq,
                            _p(ids), T, int(start_pos), _p(out))
        if rc != OK:
            raise ValueError(f"oracle hash error {rc}")
        return out


def rows_fp8(table, scales, hd: int, scale_block: int, ids) -> np.ndarray:
    """table [R, hd] e4m3 codes, scales [R, hd/blk] f32, ids [n] -> [n, hd] bf16 bits."""
    table = _c(table, np.uint8)
    scales = _c(scales, np.float32)
    ids = _c(ids, np.int64).ravel()
    R = table.size // hd
    out = np.zeros((ids.size, hd), dtype=np.uint16)
    rc = lib().orc_rows_fp8(_p(table), _p(scales), R, hd, scale_block, _p(ids), ids.size, _p(out))
    if rc != OK:
        raise ValueError(f"oracle rows_fp8 error {rc}")
    return out


def rows_fp8_e8m0(table, scales_u8, hd: int, scale_block: int, ids) -> np.ndarray:
    """table [R, hd] e4m3 codes, scales [R, hd/blk] e8m0 bytes, ids [n] -> [n, hd] bf16 bits."""
    table = _c(table, np.uint8)
    scales = _c(scales_u8, np.uint8)
    ids = _c(ids, np.int64).ravel()
    R = table.size // hd
    out = np.zeros((ids.size, hd), dtype=np.uint16)
    rc = lib().orc_rows_fp8_e8m0(_p(table), _p(scales), R, hd, scale_block, _p(ids), ids.size, _p(out))
    if rc != OK:
        raise ValueError(f"oracle rows_fp8_e8m0 error {rc}")
    return out


def rows_q2k(blocks, ids) -> np.ndarray:
    """blocks [R, 84] u8, ids [n] -> [n, 256] bf16 bits."""
    blocks = _c(blocks, np.uint8)
    ids = _c(ids, np.int64).ravel()
    R = blocks.size // 84
    out = np.zeros((ids.size, 256), dtype=np.uint16)
    rc = lib().orc_rows_q2k(_p(blocks), R, _p(ids), ids.size, _p(out))
    if rc != OK:
        raise ValueError(f"oracle rows_q2k error {rc}")
    return out


def linear_bf16(x_bits, w_bits, return_acc: bool = False):
    """x [rows, in] and w [out, in] bf16 bits -> y [rows, out] bf16 bits (and f32 sums)."""
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    rows, in_f = x.shape
    out_f = w.shape[0]
    assert w.shape[1] == in_f
    y = np.zeros((rows, out_f), dtype=np.uint16)
    acc = np.zeros((rows, out_f), dtype=np.float32) if return_acc else None
    lib().orc_linear_bf16(_p(x), rows, in_f, _p(w), out_f, _p(acc), _p(y))
    return (y, acc) if return_acc else y


def gate(h, kv_bits, q, k, hc: int, D: int, eps: float, bf16_out: bool = False,
         return_gate: bool = False):
    """h [T, hc, D] f32 (copied, not modified), kv [T, (hc+1) D] bf16 bits,
    q, k [hc, D] f32 -> updated h (and the [T, hc] gate values)."""
    hout = np.array(h, dtype=np.float32, copy=True, order="C")
    kv = _c(kv_bits, np.uint16)
    q = _c(q, np.float32)
    k = _c(k, np.float32)
    T = hout.size // (hc * D)
    assert kv.size == T * (hc + 1) * D and q.size == hc * D and k.size == hc * D
    g = np.zeros((T, hc), dtype=np.float32) if return_gate else None
    lib().orc_gate(_p(hout), _p(kv), _p(q), _p(k), T, hc, D, float(eps), int(bf16_out), _p(g))
    return (hout, g) if return_gate else hout


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Widen bf16 bit patterns to f32 values (a plain bit shift)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)

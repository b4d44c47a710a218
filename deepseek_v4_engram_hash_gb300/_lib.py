"""Thin Python binding of libengram's C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls and does
nothing but turn torch tensors into device pointers and the current torch
stream into a `cudaStream_t`; every step of the engram path runs in
libengram's CUDA kernels.  If libengram.so is missing the import fails
loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libengram.so")

ENGRAM_FMT_FP8 = 0
ENGRAM_FMT_Q2K = 1
ENGRAM_FMT_FP8_E8M0 = 2


class EngramError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class engram_geom(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("max_ngram", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dim", ctypes.c_int32), ("hc", ctypes.c_int32),
                ("scale_block", ctypes.c_int32), ("vocab", ctypes.c_int64)]


class engram_layer(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("fmt", ctypes.c_int32),
                ("wkv", ctypes.c_void_p), ("qk", ctypes.c_void_p), ("wkv_q2k", ctypes.c_void_p),
                ("wkv_tiled", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                               "(the engram path has no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        sz, st = ctypes.c_size_t, ctypes.c_void_p
        sig = {
            "engram_tables_create": ([ctypes.POINTER(engram_geom), P, i64, u64p, u64p, u64p,
                                      ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
            "engram_tables_destroy": ([P], None),
            "engram_hasher_create": ([P, i32, i64, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
            "engram_hasher_reset": ([P, st], ctypes.c_int),
            "engram_hasher_destroy": ([P], None),
            "engram_hash": ([P, P, i32, i64, P, st], ctypes.c_int),
            "engram_rows_fp8": ([P, P, i64, i32, i32, P, i64, i64, i32, P, st], ctypes.c_int),
            "engram_rows_q2k": ([P, i64, P, i64, i64, i32, P, st], ctypes.c_int),
            "engram_rows_fp8_e8m0": ([P, P, i64, i32, i32, P, i64, i64, i32, P, st], ctypes.c_int),
            "engram_project": ([P, P, i32, i32, i32, P, st], ctypes.c_int),
            "engram_gate": ([P, P, P, i32, i32, i32, ctypes.c_float, st], ctypes.c_int),
            "engram_project_q2k": ([P, P, i32, i32, P, st], ctypes.c_int),
            "engram_tiled_wkv_bytes": ([i32, i32], ctypes.c_size_t),
            "engram_selftest_wait_timeout": ([i32, st], ctypes.c_int),
            "engram_tile_wkv": ([P, i32, i32, P, st], ctypes.c_int),
            "engram_forward": ([P, ctypes.POINTER(engram_layer), P, i32, i64, P, ctypes.c_float,
                                P, sz, st], ctypes.c_int),
            "engram_forward_host": ([P, ctypes.POINTER(engram_layer), P, P, i32, i64, P, P,
                                     ctypes.c_float, P, sz, st], ctypes.c_int),
            "engram_forward_noalloc": ([P, ctypes.POINTER(engram_layer), P, i32, i64, P, ctypes.c_float,
                                        st], ctypes.c_int),
            "engram_forward_dpos": ([P, ctypes.POINTER(engram_layer), P, i32, P, P, ctypes.c_float,
                                     P, sz, st], ctypes.c_int),
            "engram_graph_create": ([P, ctypes.POINTER(engram_layer), P, i32, P, P, ctypes.c_float,
                                     P, sz, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
            "engram_graph_create_steps": ([P, ctypes.POINTER(engram_layer), P, i32, i32, P, P, ctypes.c_float,
                                           P, sz, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
            "engram_graph_launch": ([P, st], ctypes.c_int),
            "engram_graph_destroy": ([P], None),
            "engram_workspace_bytes": ([ctypes.POINTER(engram_geom), i64], sz),
            "engram_workspace_layout": ([ctypes.POINTER(engram_geom), i64, ctypes.POINTER(sz)],
                                        ctypes.c_int),
            "engram_set_profile_events": ([P, i32], ctypes.c_int),
            "engram_check": ([st], ctypes.c_int),
            "engram_strerror": ([ctypes.c_int], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().engram_strerror(int(code)).decode()


def _ok(rc: int, what: str):
    if rc != 0:
        raise EngramError(rc, what)


def _ptr(t) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(None)
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_geom(n_layers, max_ngram, n_heads, head_dim, dim, hc, scale_block, vocab) -> engram_geom:
    return engram_geom(n_layers, max_ngram, n_heads, head_dim, dim, hc, scale_block, vocab)


# ---- handles ---------------------------------------------------------------

class Tables:
    """Device copies of the hash tables (`engram_tables_create`)."""

    def __init__(self, geom: engram_geom, token_map, pad_token_id, multipliers, primes, offsets):
        import numpy as np
        self.geom = geom
        self._keep = [np.ascontiguousarray(token_map, dtype=np.int64),
                      np.ascontiguousarray(multipliers, dtype=np.int64).view(np.uint64),
                      np.ascontiguousarray(primes, dtype=np.int64).view(np.uint64),
                      np.ascontiguousarray(offsets, dtype=np.int64).view(np.uint64)]
        h = ctypes.c_void_p()
        tm, mu, pr, of = (a.ctypes.data_as(ctypes.c_void_p) for a in self._keep)
        _ok(lib().engram_tables_create(ctypes.byref(geom), tm, int(pad_token_id), mu, pr, of,
                                       ctypes.byref(h)), "engram_tables_create")
        self.handle = h

    def close(self):
        if self.handle:
            lib().engram_tables_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Hasher:
    """The look-back cache (`engram_hasher_create`); keeps its tables alive."""

    def __init__(self, tables: Tables, batch: int, max_seq: int):
        self.tables = tables
        self.batch, self.max_seq = int(batch), int(max_seq)
        h = ctypes.c_void_p()
        _ok(lib().engram_hasher_create(tables.handle, self.batch, self.max_seq, ctypes.byref(h)),
            "engram_hasher_create")
        self.handle = h

    def close(self):
        if self.handle:
            lib().engram_hasher_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- entry points (same names as the C ABI) --------------------------------

def engram_hasher_reset(hs: Hasher, stream=None):
    _ok(lib().engram_hasher_reset(hs.handle, _stream(stream)), "engram_hasher_reset")


def engram_hash(hs: Hasher, d_ids, T: int, start_pos: int, d_row_ids, stream=None):
    _ok(lib().engram_hash(hs.handle, _ptr(d_ids), int(T), int(start_pos), _ptr(d_row_ids),
                          _stream(stream)), "engram_hash")


def engram_rows_fp8(d_table, d_scales, R, head_dim, scale_block, d_row_ids, n_tok, id_stride, C,
                    d_rows, stream=None):
    _ok(lib().engram_rows_fp8(_ptr(d_table), _ptr(d_scales), int(R), int(head_dim), int(scale_block),
                              _ptr(d_row_ids), int(n_tok), int(id_stride), int(C), _ptr(d_rows),
                              _stream(stream)), "engram_rows_fp8")


def engram_rows_fp8_e8m0(d_table, d_scales_u8, R, head_dim, scale_block, d_row_ids, n_tok, id_stride, C,
                         d_rows, stream=None):
    _ok(lib().engram_rows_fp8_e8m0(_ptr(d_table), _ptr(d_scales_u8), int(R), int(head_dim), int(scale_block),
                                   _ptr(d_row_ids), int(n_tok), int(id_stride), int(C), _ptr(d_rows),
                                   _stream(stream)), "engram_rows_fp8_e8m0")


def engram_rows_q2k(d_blocks, R, d_row_ids, n_tok, id_stride, C, d_rows, stream=None):
    _ok(lib().engram_rows_q2k(_ptr(d_blocks), int(R), _ptr(d_row_ids), int(n_tok), int(id_stride),
                              int(C), _ptr(d_rows), _stream(stream)), "engram_rows_q2k")


def engram_project(d_x, d_wkv, T, K, N, d_kv, stream=None):
    _ok(lib().engram_project(_ptr(d_x), _ptr(d_wkv), int(T), int(K), int(N), _ptr(d_kv),
                             _stream(stream)), "engram_project")


def engram_project_q2k(d_x, d_wkv_q2k, K, N, d_kv, stream=None):
    _ok(lib().engram_project_q2k(_ptr(d_x), _ptr(d_wkv_q2k), int(K), int(N), _ptr(d_kv), _stream(stream)),
        "engram_project_q2k")


def engram_selftest_wait_timeout(limit_us, stream=None):
    _ok(lib().engram_selftest_wait_timeout(int(limit_us), _stream(stream)), "engram_selftest_wait_timeout")


def engram_tiled_wkv_bytes(N, K) -> int:
    return int(lib().engram_tiled_wkv_bytes(int(N), int(K)))


def engram_tile_wkv(d_wkv, N, K, d_tiled, stream=None):
    _ok(lib().engram_tile_wkv(_ptr(d_wkv), int(N), int(K), _ptr(d_tiled), _stream(stream)), "engram_tile_wkv")


def engram_gate(d_h, d_kv, d_qk, T, hc, dim, eps, stream=None):
    _ok(lib().engram_gate(_ptr(d_h), _ptr(d_kv), _ptr(d_qk), int(T), int(hc), int(dim), float(eps),
                          _stream(stream)), "engram_gate")


def layers_array(layers) -> ctypes.Array:
    """layers: list of dicts with table, scales, rows, fmt, wkv, qk (tensors or ints)."""
    arr = (engram_layer * len(layers))()
    for i, ly in enumerate(layers):
        arr[i] = engram_layer(_ptr(ly["table"]).value, _ptr(ly.get("scales")).value, int(ly["rows"]),
                              int(ly["fmt"]), _ptr(ly.get("wkv")).value, _ptr(ly["qk"]).value,
                              _ptr(ly.get("wkv_q2k")).value, _ptr(ly.get("wkv_tiled")).value)
    return arr


def engram_forward(hs: Hasher, layers, d_ids, T, start_pos, d_h, eps, d_ws, ws_bytes, stream=None):
    arr = layers if isinstance(layers, ctypes.Array) else layers_array(layers)
    _ok(lib().engram_forward(hs.handle, arr, _ptr(d_ids), int(T), int(start_pos), _ptr(d_h), float(eps),
                             _ptr(d_ws), int(ws_bytes), _stream(stream)), "engram_forward")


def engram_forward_host(hs: Hasher, layers, h_ids, d_ids, T, start_pos, h_h, d_h, eps, d_ws, ws_bytes,
                        stream=None):
    arr = layers if isinstance(layers, ctypes.Array) else layers_array(layers)
    _ok(lib().engram_forward_host(hs.handle, arr, _ptr(h_ids), _ptr(d_ids), int(T), int(start_pos),
                                  _ptr(h_h), _ptr(d_h), float(eps), _ptr(d_ws), int(ws_bytes),
                                  _stream(stream)), "engram_forward_host")


def engram_forward_noalloc(hs: Hasher, layers, d_ids, T, start_pos, d_h, eps, stream=None):
    """engram_forward with the library's fixed device scratch (no allocation)."""
    arr = layers if isinstance(layers, ctypes.Array) else layers_array(layers)
    _ok(lib().engram_forward_noalloc(hs.handle, arr, _ptr(d_ids), int(T), int(start_pos), _ptr(d_h),
                                     float(eps), _stream(stream)), "engram_forward_noalloc")


def engram_forward_dpos(hs: Hasher, layers, d_ids, T, d_start_pos, d_h, eps, d_ws, ws_bytes, stream=None):
    arr = layers if isinstance(layers, ctypes.Array) else layers_array(layers)
    _ok(lib().engram_forward_dpos(hs.handle, arr, _ptr(d_ids), int(T), _ptr(d_start_pos), _ptr(d_h),
                                  float(eps), _ptr(d_ws), int(ws_bytes), _stream(stream)), "engram_forward_dpos")


class Graph:
    """Captured decode steps (`engram_graph_create_steps`; steps = 1 is
    `engram_graph_create`); replay with launch()."""

    def __init__(self, hs: Hasher, layers, d_ids, T, d_start_pos, d_h, eps, d_ws, ws_bytes, steps: int = 1):
        self._keep = (hs, layers if isinstance(layers, ctypes.Array) else layers_array(layers))
        g = ctypes.c_void_p()
        if steps == 1:
            _ok(lib().engram_graph_create(hs.handle, self._keep[1], _ptr(d_ids), int(T), _ptr(d_start_pos),
                                          _ptr(d_h), float(eps), _ptr(d_ws), int(ws_bytes), ctypes.byref(g)),
                "engram_graph_create")
        else:
            _ok(lib().engram_graph_create_steps(hs.handle, self._keep[1], _ptr(d_ids), int(T), int(steps),
                                                _ptr(d_start_pos), _ptr(d_h), float(eps), _ptr(d_ws),
                                                int(ws_bytes), ctypes.byref(g)),
                "engram_graph_create_steps")
        self.handle = g

    def launch(self, stream=None):
        _ok(lib().engram_graph_launch(self.handle, _stream(stream)), "engram_graph_launch")

    def close(self):
        if self.handle:
            lib().engram_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def engram_workspace_bytes(geom: engram_geom, max_tokens: int) -> int:
    return int(lib().engram_workspace_bytes(ctypes.byref(geom), int(max_tokens)))


def engram_workspace_layout(geom: engram_geom, tokens: int) -> list:
    off = (ctypes.c_size_t * (2 + 2 * geom.n_layers))()
    _ok(lib().engram_workspace_layout(ctypes.byref(geom), int(tokens), off), "engram_workspace_layout")
    return list(off)


def prepare_events(events) -> None:
    """Create the cudaEvent_t behind torch events (record each once, then sync)."""
    for e in events:
        e.record()
    torch.cuda.synchronize()


def engram_set_profile_events(events) -> None:
    """events: 5 torch.cuda.Event already created (prepare_events), or None."""
    global _prof_keep
    if events is None:
        _prof_keep = None
        _ok(lib().engram_set_profile_events(None, 0), "engram_set_profile_events")
        return
    handles = [e.cuda_event for e in events]
    if not all(handles):
        raise ValueError("profile events must be created first (prepare_events)")
    _prof_keep = (ctypes.c_uint64 * len(handles))(*handles)
    _ok(lib().engram_set_profile_events(ctypes.cast(_prof_keep, ctypes.c_void_p), len(handles)),
        "engram_set_profile_events")


_prof_keep = None


def engram_check(stream=None) -> int:
    return int(lib().engram_check(_stream(stream)))

"""libengram on the CPU: the library loads, exports every symbol include/engram.h
declares, and its host-side validation refuses bad arguments before it
touches the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def E():
    from deepseek_v4_engram_hash_gb300 import build
    build.build()
    from deepseek_v4_engram_hash_gb300 import _lib
    _lib.lib()
    return _lib


def _declared():
    src = open(os.path.join(ROOT, "include", "engram.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(engram_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(E):
    names = _declared()
    assert len(names) >= 17
    L = ctypes.CDLL(E.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_strerror(E):
    assert E.strerror(0) == "ok"
    assert "hc" in E.strerror(-6)
    assert E.strerror(-999) == "unknown engram error"


def _geom(E, **kw):
    d = dict(n_layers=2, max_ngram=4, n_heads=8, head_dim=256, dim=4096, hc=4, scale_block=32,
             vocab=129280)
    d.update(kw)
    return E.make_geom(**d)


def test_workspace_layout(E):
    g = _geom(E)
    off = E.engram_workspace_layout(g, 1)
    C, N = 24, 4096 * 5
    assert off[0] == 0
    assert off[1] == 256 * ((1 * 2 * C * 8 + 255) // 256)
    assert off[2] - off[1] == 256 * ((N * 2 + 255) // 256)
    assert off[-1] == E.engram_workspace_bytes(g, 1)
    # prefill adds the gathered x per layer, and (from 256 tokens) the CTA-pair
    # GEMM's 24 MiB of last-wave partial tiles at the end
    big = E.engram_workspace_layout(g, 4096)
    assert big[-1] - big[3] == 2 * 4096 * C * 256 * 2 + 96 * 256 * 256 * 4
    small = E.engram_workspace_layout(g, 255)
    assert small[-1] - small[3] == 2 * 255 * C * 256 * 2
    assert E.engram_workspace_bytes(_geom(E, hc=5), 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(hc=5), -6), (dict(hc=0), -6), (dict(n_layers=0), -1), (dict(n_layers=5), -1),
    (dict(max_ngram=1), -1), (dict(head_dim=24), -1), (dict(scale_block=24), -1),
    (dict(dim=12), -1), (dict(vocab=0), -1),
])
def test_tables_create_refuses_bad_geometry(E, kw, code):
    g = _geom(E, **kw)
    h = ctypes.c_void_p()
    buf = (ctypes.c_int64 * 64)()
    rc = E.lib().engram_tables_create(ctypes.byref(g), buf, 0, buf, buf, buf, ctypes.byref(h))
    assert rc == code and not h.value


def test_tables_create_refuses_bad_values(E):
    g = _geom(E, n_layers=1, max_ngram=2, n_heads=1, vocab=4, head_dim=64)
    h = ctypes.c_void_p()
    tm = (ctypes.c_int64 * 4)(0, 1, 2, 3)
    ok = (ctypes.c_uint64 * 2)(3, 5)
    zero = (ctypes.c_uint64 * 2)(0, 0)
    big = (ctypes.c_uint64 * 2)(1 << 63, 1)
    L = E.lib()
    assert L.engram_tables_create(ctypes.byref(g), tm, 4, ok, ok, ok, ctypes.byref(h)) == -1
    assert L.engram_tables_create(ctypes.byref(g), tm, 0, big, ok, ok, ctypes.byref(h)) == -1
    assert L.engram_tables_create(ctypes.byref(g), tm, 0, ok, zero, ok, ctypes.byref(h)) == -1
    assert L.engram_tables_create(ctypes.byref(g), None, 0, ok, ok, ok, ctypes.byref(h)) == -2


def test_compute_calls_refuse_before_launch(E):
    L = E.lib()
    P = ctypes.c_void_p
    a16 = P(1 << 20)            # aligned fake addresses: never dereferenced, refused first
    odd = P((1 << 20) + 2)
    assert L.engram_project(None, a16, 1, 256, 384, a16, None) == -2
    assert L.engram_project(a16, a16, 1, 250, 384, a16, None) == -1
    assert L.engram_project(a16, a16, 1, 256, 380, a16, None) == -1
    assert L.engram_project(odd, a16, 1, 256, 384, a16, None) == -3
    assert L.engram_gate(a16, a16, a16, 1, 5, 128, ctypes.c_float(1e-6), None) == -6
    assert L.engram_gate(a16, a16, a16, 1, 2, 100, ctypes.c_float(1e-6), None) == -1
    assert L.engram_gate(odd, a16, a16, 1, 2, 128, ctypes.c_float(1e-6), None) == -3
    assert L.engram_rows_fp8(a16, a16, 10, 64, 24, a16, 1, 4, 4, a16, None) == -1
    assert L.engram_rows_fp8(odd, a16, 10, 64, 32, a16, 1, 4, 4, a16, None) == -3
    assert L.engram_rows_fp8(a16, a16, 10, 64, 32, a16, 1, 3, 4, a16, None) == -1
    assert L.engram_rows_q2k(P((1 << 20) + 1), 10, a16, 1, 4, 4, a16, None) == -3
    # Q2_K weights are copied by the bulk-copy engine: 16-byte aligned, K % 256, K <= 6144
    assert L.engram_project_q2k(a16, P((1 << 20) + 4), 256, 16, a16, None) == -3
    assert L.engram_project_q2k(a16, a16, 320, 16, a16, None) == -1
    assert L.engram_project_q2k(a16, a16, 6400, 16, a16, None) == -11
    assert L.engram_hash(None, a16, 1, 0, a16, None) == -2
    assert L.engram_set_profile_events(a16, 3) == -1


def test_selftest_wait_timeout_refuses_bad_limits(E):
    L = E.lib()
    assert L.engram_selftest_wait_timeout(0, None) == -1
    assert L.engram_selftest_wait_timeout(2000000, None) == -1


def test_tiled_wkv_size_and_refusals(E):
    """engram_tiled_wkv_bytes: 16-row x 2048-column tiles, ragged edges padded;
    engram_tile_wkv refuses null, misaligned and overlapping buffers and bad
    shapes before it launches anything."""
    L = E.lib()
    L.engram_tiled_wkv_bytes.restype = ctypes.c_size_t
    assert L.engram_tiled_wkv_bytes(20480, 6144) == 1280 * 3 * 16 * 2048 * 2   # = wkv bytes, no padding
    assert L.engram_tiled_wkv_bytes(120, 4800) == 8 * 3 * 16 * 2048 * 2
    assert L.engram_tiled_wkv_bytes(1, 8) == 16 * 2048 * 2
    assert L.engram_tiled_wkv_bytes(0, 64) == 0 and L.engram_tiled_wkv_bytes(16, 12) == 0
    P = ctypes.c_void_p
    w, t = P(1 << 30), P(1 << 34)      # far apart, aligned, never dereferenced
    assert L.engram_tile_wkv(None, 16, 64, t, None) == -2
    assert L.engram_tile_wkv(w, 16, 64, None, None) == -2
    assert L.engram_tile_wkv(w, 0, 64, t, None) == -1
    assert L.engram_tile_wkv(w, 16, 60, t, None) == -1
    assert L.engram_tile_wkv(P((1 << 30) + 8), 16, 64, t, None) == -3
    assert L.engram_tile_wkv(w, 16, 64, P((1 << 34) + 2), None) == -3
    assert L.engram_tile_wkv(w, 16, 64, P((1 << 30) + 1024), None) == -1    # overlaps wkv


def test_missing_library_fails_loudly(monkeypatch):
    """Without libengram.so the binding raises; nothing falls back to the CPU."""
    from deepseek_v4_engram_hash_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", _lib.LIB_PATH + ".absent")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.strerror(0)

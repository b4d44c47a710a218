"""The oracle and the CUDA path share no code (CPU only): nothing in the
package imports the oracle, no CUDA source includes anything of it, the
oracle's C source includes only the C library, and the oracle package
imports nothing of the CUDA path.  Only the seeded input generators
(deepseek_v4_engram_hash_gb300/synth.py) serve both sides."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "deepseek_v4_engram_hash_gb300")


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def test_package_never_imports_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b)", re.M)
    for f in _files(PKG, (".py",)):
        assert not pat.search(open(f).read()), f


def test_cuda_sources_include_nothing_of_the_oracle():
    for f in _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")):
        for inc in re.findall(r'#include\s+[<"]([^>"]+)[>"]', open(f).read()):
            assert "oracle" not in inc, (f, inc)


def test_oracle_c_includes_only_the_c_library():
    incs = set(re.findall(r'#include\s+<([^>]+)>', open(os.path.join(ROOT, "oracle", "oracle.c")).read()))
    assert not re.search(r'#include\s+"', open(os.path.join(ROOT, "oracle", "oracle.c")).read())
    assert incs <= {"math.h", "stdint.h", "string.h", "omp.h"}, incs


def test_oracle_package_imports_nothing_of_the_cuda_path():
    pat = re.compile(r"^\s*(import|from)\s+deepseek_v4_engram_hash_gb300", re.M)
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        assert not pat.search(open(f).read()), f

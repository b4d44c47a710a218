"""The seeded generator's normals (CPU): the float64 Box-Muller evaluation
agrees with the library's log and cos to double precision, and the variates
have the moments and tails of N(0, 1) (not a bounded approximation)."""
import numpy as np

from deepseek_v4_engram_hash_gb300 import synth


def test_box_muller_series_matches_library_functions():
    z = synth.splitmix64(synth.stream_key(0, "normal-check"), np.arange(1 << 20, dtype=np.uint64))
    got = synth.std_normal_f64(z)
    u1 = ((z >> np.uint64(32)).astype(np.float64) + 1.0) * 2.0 ** -32
    u2 = (z & np.uint64(0xFFFFFFFF)).astype(np.float64) * 2.0 ** -32
    want = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    assert np.abs(got - want).max() < 1e-13


def test_normal_moments_and_tails():
    z = synth.splitmix64(synth.stream_key(1, "normal-moments"), np.arange(1 << 22, dtype=np.uint64))
    x = synth.std_normal_f64(z)
    n = x.size
    assert abs(x.mean()) < 4 / np.sqrt(n)
    assert abs(x.std() - 1.0) < 4 * np.sqrt(0.5 / n)
    kurt = np.mean(x ** 4) / np.mean(x ** 2) ** 2 - 3.0
    assert abs(kurt) < 0.02                                 # 0 for N(0,1); -0.3 for a 4-term uniform sum
    assert np.abs(x).max() > 4.8                            # tails beyond any sum of four uniforms
    # the share beyond 3 sigma: 0.27 % for N(0,1)
    assert abs(np.mean(np.abs(x) > 3.0) - 0.0026998) < 0.0004


def test_extremes_of_the_transform():
    """u1 = 1 gives 0; the largest radius sqrt(-2 ln 2^-32) = 6.66 bounds every variate."""
    z = np.array([0xFFFFFFFF_00000000, 0x00000000_00000000, 0x00000000_40000000, 0x00000000_80000000],
                 dtype=np.uint64)
    x = synth.std_normal_f64(z)
    assert x[0] == 0.0
    r = np.sqrt(-2.0 * np.log(2.0 ** -32))
    assert abs(x[1] - r) < 1e-13                            # cos 0 = 1
    assert abs(x[2]) < 1e-13                                # cos(pi/2) = 0 at 4 u2 = 1
    assert abs(x[3] + r) < 1e-13                            # cos(pi) = -1


def test_cuda_twin_holds_the_same_constants():
    """The CUDA twin's series coefficients and constants are the numpy twin's
    (read from its source: the two evaluate the same operations on the same
    doubles)."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(synth.__file__), "csrc", "synth.cu")).read()

    def arr(name):
        body = re.search(name + r"\[\d+\] = \{(.*?)\};", src, re.S).group(1)
        return [float.fromhex(t.strip()) for t in body.split(",") if t.strip()]

    assert arr("kAtanh") == synth._ATANH
    assert arr("kCos") == synth._COS
    assert arr("kSin") == synth._SIN
    for name, val in (("kLn2", synth._LN2), ("kPi2", synth._PI_2), ("kSqrtHalf", synth._SQRT_HALF)):
        lit = re.search(name + r" = (0x[0-9a-fp.+-]+)", src).group(1)
        assert float.fromhex(lit) == val, name

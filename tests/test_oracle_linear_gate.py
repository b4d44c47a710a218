"""Pins of the oracle's projection and gate (CPU only).

The projection (`linear_bf16` on the CPU reference page) is checked against
numpy's float64 matrix product within the f32 summation error bound and
against torch's bf16 rounding of the f32 sums.  The gate (`gate_and_add`) is
checked against closed forms for constant inputs, against its value = 0 and
sign-symmetry special cases, and against one-hot q*k weights.
"""
import math

import numpy as np
import torch


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_linear_matches_f64_product(orc):
    rng = np.random.default_rng(3)
    rows, in_f, out_f = 5, 384, 7                        # non-square: a transposed w fails
    x = _bf16(rng.standard_normal((rows, in_f)))
    w = _bf16(0.02 * rng.standard_normal((out_f, in_f)))
    y, acc = orc.linear_bf16(x, w, return_acc=True)
    xf, wf = _f(x).astype(np.float64), _f(w).astype(np.float64)
    exact = xf @ wf.T
    bound = in_f * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
    assert (np.abs(acc - exact) <= bound).all()
    assert np.array_equal(y, _bf16(acc))


def test_linear_accumulates_in_f32_in_index_order(orc):
    """x = (1, 2^-24, 2^-24), w = (1, 1, 1): in f32 from the left each 2^-24 is
    half an ulp of 1 and rounds away (ties to even), so the sum is exactly 1;
    the exact sum, a wider accumulator or a pairwise order give 1 + 2^-23."""
    x = _bf16(np.array([[1.0, 2.0 ** -24, 2.0 ** -24]]))
    w = _bf16(np.ones((1, 3)))
    _, acc = orc.linear_bf16(x, w, return_acc=True)
    assert acc[0, 0] == np.float32(1.0)
    x2 = _bf16(np.array([[2.0 ** -24, 2.0 ** -24, 1.0]]))      # small terms first: they add up
    _, acc2 = orc.linear_bf16(x2, w, return_acc=True)
    assert acc2[0, 0] == np.float32(1.0 + 2.0 ** -23)


def test_linear_picks_rows_of_w(orc):
    in_f = 64
    x = _bf16(np.eye(3, in_f))                              # x_r = e_r
    w = _bf16(np.arange(4 * in_f, dtype=np.float32).reshape(4, in_f) / 64)
    y = _f(orc.linear_bf16(x, w))
    assert np.array_equal(y, _f(w)[:, :3].T)               # y[r, o] = w[o, r]


def _gate_closed_form(a, b, r, D, eps):
    s = math.sqrt(D) * a * r * b / (math.sqrt(a * a + eps) * math.sqrt(b * b + eps))
    g = math.copysign(math.sqrt(max(abs(s), 1e-6)), s)
    return 1.0 / (1.0 + math.exp(-g))


def test_gate_closed_form_constant_streams(orc):
    """h[c] = a_c, key_c = b_c, q k = r_c: s_c = sqrt(D) a r b / (sqrt(a^2+e) sqrt(b^2+e))."""
    D, hc, eps = 128, 4, 1e-6
    a = [0.5, -1.25, 2.0, 0.0]                            # a = 0: s = +0, the 1e-6 floor
    b = [0.75, 0.5, -0.25, 1.0]
    r = [1.0, 0.5, 0.001, 1.0]
    value = np.linspace(-2, 2, D).astype(np.float32)
    h = np.stack([np.full(D, ai, np.float32) for ai in a])[None]
    kv = np.concatenate([np.full(D, bi, np.float32) for bi in b] + [value])[None]
    q = np.stack([np.full(D, ri, np.float32) for ri in r])
    k = np.ones((hc, D), np.float32)
    out, gate = orc.gate(h, _bf16(kv), q, k, hc, D, eps, return_gate=True)
    vbf = _f(_bf16(value))
    for c in range(hc):
        want = _gate_closed_form(a[c], b[c], r[c], D, eps)
        assert abs(gate[0, c] - want) < 2e-6, (c, gate[0, c], want)
        assert np.allclose(out[0, c], a[c] + gate[0, c] * vbf, atol=1e-6, rtol=0)


def test_gate_value_zero_leaves_h(orc):
    rng = np.random.default_rng(4)
    D, hc = 64, 4
    h = rng.standard_normal((3, hc, D)).astype(np.float32)
    kv = np.concatenate([rng.standard_normal((3, hc * D)), np.zeros((3, D))], axis=1)
    q = np.ones((hc, D), np.float32)
    out = orc.gate(h, _bf16(kv), q, q, hc, D, 1e-6)
    assert np.array_equal(out.view(np.uint32), h.view(np.uint32))


def test_gate_sign_symmetry(orc):
    """Negating the keys negates s, and sigma(-g) = 1 - sigma(g)."""
    rng = np.random.default_rng(5)
    D, hc, T = 96, 2, 4
    h = rng.standard_normal((T, hc, D)).astype(np.float32)
    keys = _f(_bf16(rng.standard_normal((T, hc * D))))
    value = _f(_bf16(rng.standard_normal((T, D))))
    q = _f(_bf16(1 + 0.05 * rng.standard_normal((hc, D))))
    k = _f(_bf16(1 + 0.05 * rng.standard_normal((hc, D))))
    _, g1 = orc.gate(h, _bf16(np.concatenate([keys, value], 1)), q, k, hc, D, 1e-6, return_gate=True)
    _, g2 = orc.gate(h, _bf16(np.concatenate([-keys, value], 1)), q, k, hc, D, 1e-6, return_gate=True)
    assert np.allclose(g1 + g2, 1.0, atol=1e-6)
    assert ((g1 > 0) & (g1 < 1)).all()


def test_gate_one_hot_qk_selects_coordinate(orc):
    """q k = e_j: dot = h_j key_j, so s = h_j key_j / (rms(h) rms(key) sqrt(D))."""
    rng = np.random.default_rng(6)
    D, hc, j = 64, 2, 17
    h = rng.standard_normal((1, hc, D)).astype(np.float32)
    keys = _f(_bf16(rng.standard_normal((hc, D))))
    kv = _bf16(np.concatenate([keys.ravel(), np.ones(D)]))[None]
    q = np.zeros((hc, D), np.float32)
    q[:, j] = 1.0
    _, g = orc.gate(h, kv, q, np.ones_like(q), hc, D, 0.0, return_gate=True)
    for c in range(hc):
        hr, kr = h[0, c].astype(np.float64), keys[c].astype(np.float64)
        s = hr[j] * kr[j] / (math.sqrt((hr ** 2).mean()) * math.sqrt((kr ** 2).mean()) * math.sqrt(D))
        gg = math.copysign(math.sqrt(max(abs(s), 1e-6)), s)
        assert abs(g[0, c] - 1 / (1 + math.exp(-gg))) < 1e-5


def test_gate_bf16_out_mode(orc):
    rng = np.random.default_rng(8)
    D, hc = 32, 1
    h = rng.standard_normal((2, hc, D)).astype(np.float32)
    kv = _bf16(rng.standard_normal((2, 2 * D)))
    q = np.ones((hc, D), np.float32)
    out = orc.gate(h, kv, q, q, hc, D, 1e-6, bf16_out=True)
    assert np.array_equal(out, _f(_bf16(out)))
    full = orc.gate(h, kv, q, q, hc, D, 1e-6)
    assert np.array_equal(_bf16(full), _bf16(out))

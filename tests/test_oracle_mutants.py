"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake -- a dropped term, a wrong sign, index, shift or
rounding, a transposed operand -- in a scratch copy of ``oracle/oracle.c``,
compiles it into a scratch library, and runs the pins of that stage against
it: at least one pin must fail.  The committed oracle is never touched; the
mutant library replaces it only inside the test (monkeypatched).
"""
import inspect
import os

import pytest

import oracle
import test_oracle_formats as pins_formats
import test_oracle_hash as pins_hash
import test_oracle_linear_gate as pins_linear_gate

HASH, FORMATS, LINGATE = pins_hash, pins_formats, pins_linear_gate

# (name, text in oracle.c, replacement, pin modules that must catch it)
MUTANTS = [
    # stage 1: the hash
    ("hash: XOR combine dropped (last slot only)", "X ^= wrapping_mul(w, mult[(int64_t)l * ng + j]);",
     "X = wrapping_mul(w, mult[(int64_t)l * ng + j]);", [HASH]),
    ("hash: products added instead of XOR-combined", "X ^= wrapping_mul(w, mult[(int64_t)l * ng + j]);",
     "X = wrapping_add(X, wrapping_mul(w, mult[(int64_t)l * ng + j]));", [HASH]),
    ("hash: truncated remainder", "if (r < 0) r += P;", "", [HASH]),
    ("hash: unsigned remainder", "__int128 r = (__int128)x % (__int128)P;",
     "__int128 r = (__int128)((uint64_t)x % (uint64_t)P);", [HASH]),
    ("hash: window shifted by one", "const int64_t w = j < cut ? seq_cache[p - j] : pad_id;",
     "const int64_t w = j < cut && p > j ? seq_cache[p - j - 1] : pad_id;", [HASH]),
    ("hash: blocking not carried to larger shifts", "const int64_t w = j < cut ? seq_cache[p - j] : pad_id;",
     "const int64_t w = j <= p && seq_cache[p - j] != -1 ? seq_cache[p - j] : pad_id;", [HASH]),
    ("hash: unmapped id not blocked", "if (j > p || seq_cache[p - j] == -1) return j;",
     "if (j > p) return j;", [HASH]),
    ("hash: first layer's offsets for every layer", "offsets[(int64_t)l * C + c]);",
     "offsets[c]);", [HASH]),
    ("hash: multipliers indexed [shift][layer]", "X ^= wrapping_mul(w, mult[(int64_t)l * ng + j]);",
     "X ^= wrapping_mul(w, mult[(int64_t)j * L + l]);", [HASH]),
    ("hash: columns head-major", "const int c = (g - 2) * H + h;",
     "const int c = h * (ng - 1) + (g - 2);", [HASH]),
    ("hash: the window's first slot left out", "for (int j = 0; j < g; ++j) {",
     "for (int j = 1; j < g; ++j) {", [HASH]),
    ("hash: the (n+1)-gram one slot short", "for (int j = 0; j < g; ++j) {",
     "for (int j = 0; j < g - 1; ++j) {", [HASH]),
    ("hash: new positions never enter the cache",
     "cache[(int64_t)b * max_seq + start_pos + s] = token_map[ids[(int64_t)b * T + s]];", "(void)0;", [HASH]),
    # number formats and table rows
    ("bf16: truncation", "u += 0x7FFFu + ((u >> 16) & 1u);", "", [FORMATS, LINGATE]),
    ("bf16: ties away from zero", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;", [FORMATS]),
    ("e4m3: exponent bias 8", "return sign * (1.0f + m / 8.0f) * ldexpf(1.0f, e - 7);",
     "return sign * (1.0f + m / 8.0f) * ldexpf(1.0f, e - 8);", [FORMATS]),
    ("e4m3: subnormal scale 2^-7", "return sign * m / 8.0f * ldexpf(1.0f, -6);",
     "return sign * m / 8.0f * ldexpf(1.0f, -7);", [FORMATS]),
    ("e4m3: no NaN code", "if (e == 15 && m == 7.0f) return NAN;", "", [FORMATS]),
    ("e4m3 encode: saturates to the NaN code", "if (a > 448.0) return sign | 0x7E;",
     "if (a > 448.0) return sign | 0x7F;", [FORMATS]),
    ("f16: subnormals off by a factor two", "if (e == 0) v = ldexpf((float)m, -24);",
     "if (e == 0) v = ldexpf((float)m, -25);", [FORMATS]),
    ("e8m0: rounds down", "if (m > 0x400000u || (m == 0x400000u && (e & 1u) == 1u)) e += 1;", "", [FORMATS]),
    ("e8m0: ties to the odd code", "(m == 0x400000u && (e & 1u) == 1u)",
     "(m == 0x400000u && (e & 1u) == 0u)", [FORMATS]),
    ("fp8 rows: scale block d % nblk", "const float s = scales[id * nblk + d / blk];",
     "const float s = scales[id * nblk + d % nblk];", [FORMATS]),
    ("fp8 rows: scale not applied", "const float s = scales[id * nblk + d / blk];",
     "const float s = 1.0f + 0.0f * scales[id * nblk + d / blk];", [FORMATS]),
    ("e8m0 rows: scale byte off by one", "const float s = orc_e8m0_to_f32(scales[id * nblk + d / blk]);",
     "const float s = orc_e8m0_to_f32((uint8_t)(scales[id * nblk + d / blk] + 1));", [FORMATS]),
    ("q2k: d and dmin swapped", "const float y = d * (float)(s & 15) * (float)q - dmin * (float)(s >> 4);",
     "const float y = dmin * (float)(s & 15) * (float)q - d * (float)(s >> 4);", [FORMATS]),
    ("q2k: scale and min nibbles swapped",
     "const float y = d * (float)(s & 15) * (float)q - dmin * (float)(s >> 4);",
     "const float y = d * (float)(s >> 4) * (float)q - dmin * (float)(s & 15);", [FORMATS]),
    ("q2k: min added", "const float y = d * (float)(s & 15) * (float)q - dmin * (float)(s >> 4);",
     "const float y = d * (float)(s & 15) * (float)q + dmin * (float)(s >> 4);", [FORMATS]),
    ("q2k: quant shift j", "const int q = (qs[32 * half + l] >> (2 * j)) & 3;",
     "const int q = (qs[32 * half + l] >> j) & 3;", [FORMATS]),
    ("q2k: quant byte ignores the half", "const int q = (qs[32 * half + l] >> (2 * j)) & 3;",
     "const int q = (qs[l] >> (2 * j)) & 3;", [FORMATS]),
    ("q2k: one sub-block per 32 values", "const int s = sc[8 * half + 2 * j + l / 16];",
     "const int s = sc[8 * half + 2 * j];", [FORMATS]),
    ("e4m3 encode: truncation", "int mant = (int)round_ties_even((a * ldexp(1.0, -e) - 1.0) * 8.0);",
     "int mant = (int)((a * ldexp(1.0, -e) - 1.0) * 8.0);", [FORMATS]),
    ("e4m3 encode: subnormal threshold", "if (e < -6) return sign | (uint8_t)round_ties_even(a * 512.0);",
     "if (e < -7) return sign | (uint8_t)round_ties_even(a * 512.0);", [FORMATS]),
    ("e4m3 encode: mantissa carry dropped", "if (mant == 8) { e += 1; mant = 0; }", "", [FORMATS]),
    ("rounding: ties up", "return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f + 1.0;", [FORMATS]),
    ("f16: normal exponent bias", "else v = ldexpf((float)(1024 + m), e - 25);",
     "else v = ldexpf((float)(1024 + m), e - 24);", [FORMATS]),
    ("bf16: NaN not kept quiet", "if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);",
     "", [FORMATS]),
    ("e8m0 decode: code 255 not NaN", "if (code == 255) return NAN;", "", [FORMATS]),
    ("hash: token range off by one", "if (ids[i] < 0 || ids[i] >= vocab) return ORC_E_TOKEN;",
     "if (ids[i] < 0 || ids[i] > vocab) return ORC_E_TOKEN;", [HASH]),
    ("hash: capacity off by one", "if (start_pos < 0 || start_pos + T > max_seq) return ORC_E_CAPACITY;",
     "if (start_pos < 0 || start_pos + T > max_seq + 1) return ORC_E_CAPACITY;", [HASH]),
    # stage 3: the projection
    ("linear: w transposed", "sum += orc_bf16_to_f32(xr[i]) * orc_bf16_to_f32(wr[i]);",
     "sum += orc_bf16_to_f32(xr[i]) * orc_bf16_to_f32(w[i * out_f + o]);", [LINGATE]),
    ("linear: last term dropped", "for (int64_t i = 0; i < in_f; ++i)",
     "for (int64_t i = 0; i + 1 < in_f; ++i)", [LINGATE]),
    ("linear: accumulated in double", "float sum = 0.0f;\n            for (int64_t i = 0; i < in_f; ++i)",
     "double sum = 0.0;\n            for (int64_t i = 0; i < in_f; ++i)", [LINGATE]),
    ("linear: summed from the last term", "sum += orc_bf16_to_f32(xr[i]) * orc_bf16_to_f32(wr[i]);",
     "sum += orc_bf16_to_f32(xr[in_f - 1 - i]) * orc_bf16_to_f32(wr[in_f - 1 - i]);", [LINGATE]),
    ("linear: output truncated to bf16", "y[r * out_f + o] = orc_f32_to_bf16(sum);",
     "y[r * out_f + o] = (uint16_t)(f2u(sum) >> 16);", [LINGATE]),
    # stage 4: the gate
    ("gate: sign of s dropped", "const float g = copysignf(sqrtf(fmaxf(fabsf(s), 1e-6f)), s);",
     "const float g = sqrtf(fmaxf(fabsf(s), 1e-6f));", [LINGATE]),
    ("gate: no floor on |s|", "const float g = copysignf(sqrtf(fmaxf(fabsf(s), 1e-6f)), s);",
     "const float g = copysignf(sqrtf(fabsf(s)), s);", [LINGATE]),
    ("gate: no square root", "const float g = copysignf(sqrtf(fmaxf(fabsf(s), 1e-6f)), s);",
     "const float g = copysignf(fmaxf(fabsf(s), 1e-6f), s);", [LINGATE]),
    ("gate: eps dropped", "const float rstd = (1.0f / sqrtf(hh / (float)D + eps)) *",
     "const float rstd = (1.0f / sqrtf(hh / (float)D)) *", [LINGATE]),
    ("gate: D^-1/2 dropped", "const float s = dot * rstd * inv_sqrt_dim;", "const float s = dot * rstd;",
     [LINGATE]),
    ("gate: q*k not applied", "dot += hr[d] * (q[c * D + d] * k[c * D + d]) * kd;", "dot += hr[d] * kd;",
     [LINGATE]),
    ("gate: hh from the key", "hh += hr[d] * hr[d];", "hh += kd * kd;", [LINGATE]),
    ("gate: stream 0's key for every stream", "const uint16_t *key = kv + t * kv_w + (int64_t)c * D;",
     "const uint16_t *key = kv + t * kv_w;", [LINGATE]),
    ("gate: value from the key columns", "const uint16_t *value = kv + t * kv_w + (int64_t)hc * D;",
     "const uint16_t *value = kv + t * kv_w;", [LINGATE]),
    ("gate: kk from the highway", "kk += kd * kd;", "kk += hr[d] * hr[d];", [LINGATE]),
    ("gate: key norm dropped", "(1.0f / sqrtf(kk / (float)D + eps));", "1.0f;", [LINGATE]),
    ("gate: key added instead of the value", "float o = hr[d] + gate * orc_bf16_to_f32(value[d]);",
     "float o = hr[d] + gate * orc_bf16_to_f32(key[d]);", [LINGATE]),
    ("gate: every stream updates stream 0", "float *hr = h + (t * hc + c) * D;", "float *hr = h + t * hc * D;",
     [LINGATE]),
    ("gate: sigmoid of -g", "const float gate = 1.0f / (1.0f + expf(-g));",
     "const float gate = 1.0f / (1.0f + expf(g));", [LINGATE]),
    ("gate: highway rounded to bf16 always", "if (bf16_out) o = orc_bf16_to_f32(orc_f32_to_bf16(o));",
     "o = orc_bf16_to_f32(orc_f32_to_bf16(o));", [LINGATE]),
]


def _pin_calls(modules):
    """Every pin of the modules as a zero-argument call (parametrised pins once
    per parameter value)."""
    calls = []
    for mod in modules:
        for name, fn in sorted(vars(mod).items()):
            if not (name.startswith("test_") and callable(fn)):
                continue
            params = [p for p in inspect.signature(fn).parameters if p != "orc"]
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            if not params:
                calls.append((f"{mod.__name__}.{name}", lambda fn=fn: fn(oracle)))
                continue
            assert len(params) == 1 and len(marks) == 1 and marks[0].args[0] == params[0]
            for v in marks[0].args[1]:
                calls.append((f"{mod.__name__}.{name}[{v}]", lambda fn=fn, v=v: fn(oracle, v)))
    return calls


def test_every_mutant_text_occurs_once():
    src = open(oracle._SRC).read()
    for name, old, new, _ in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(idx, tmp_path, monkeypatch):
    name, old, new, modules = MUTANTS[idx]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1
    path = os.path.join(tmp_path, "oracle_mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.compile_source(path, os.path.join(tmp_path, f"liboracle_mutant{idx}.so"))
    monkeypatch.setattr(oracle, "_lib", oracle.load(so))
    caught = []
    for pin, call in _pin_calls(modules):
        try:
            call()
        except (AssertionError, ValueError, IndexError, pytest.fail.Exception):
            caught.append(pin)
    assert caught, f"no pin catches the planted mistake: {name}"


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    """The control: the same machinery on an unchanged copy fails no pin, so
    a caught mutant was caught by its planted mistake."""
    path = os.path.join(tmp_path, "oracle_copy.c")
    with open(path, "w") as f:
        f.write(open(oracle._SRC).read())
    so = oracle.compile_source(path, os.path.join(tmp_path, "liboracle_copy.so"))
    monkeypatch.setattr(oracle, "_lib", oracle.load(so))
    failed = []
    for pin, call in _pin_calls([HASH, FORMATS, LINGATE]):
        try:
            call()
        except (Exception, pytest.fail.Exception) as e:         # noqa: BLE001 -- any failure counts
            failed.append(f"{pin}: {type(e).__name__}")
    assert not failed, failed
    assert len(_pin_calls([HASH, FORMATS, LINGATE])) >= 25

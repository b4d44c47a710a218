"""GPU parity of each stage through the C ABI against the CPU oracle.

Hash ids and dequantised rows must be bit-exact; the bf16 projection within
2e-2 max relative error (floored at 1e-3 of the largest output); the FP32
highway after the gate within 1e-3 absolute, the oracle gate being run on the
same kv the GPU gate reads (stage-wise).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_glue as G
from deepseek_v4_engram_hash_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import __graft_entry__
    __graft_entry__.build()
    from deepseek_v4_engram_hash_gb300 import _lib
    assert torch.cuda.is_available()
    return _lib


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _hash_setup(E, cfg, batch):
    t = synth.hash_tables(cfg)
    g = E.make_geom(cfg.n_layers, cfg.max_ngram, cfg.n_heads, cfg.head_dim, cfg.dim, cfg.hc,
                    cfg.scale_block, cfg.vocab)
    tabs = E.Tables(g, t["token_map"], t["pad_token_id"], t["multipliers"], t["primes"], t["offsets"])
    return E.Hasher(tabs, batch, 4096), G.hash_state(cfg, batch, 4096)


# ---------------------------------------------------------------- hash ----

@pytest.mark.parametrize("cfg,batch,splits", [
    (configs.TINY, 1, [16]),
    (configs.TINY, 3, [7, 1, 1, 30, 1]),                 # ragged prefill + decode steps
    (configs.V41_DECODE, 2, [300, 1, 1, 1, 700]),
    (configs.STRESS, 8, [1536, 1, 1]),
])
def test_hash_bit_exact(E, cfg, batch, splits):
    hs, ref = _hash_setup(E, cfg, batch)
    pos = 0
    for i, T in enumerate(splits):
        ids = np.stack([synth.token_ids(cfg, f"h{i}.{b}", T) for b in range(batch)])
        d_ids = torch.from_numpy(ids).cuda()
        out = torch.empty((batch, T, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        E.engram_hash(hs, d_ids, T, pos, out)
        want = ref.forward(ids, pos)
        assert E.engram_check() == 0
        assert np.array_equal(out.cpu().numpy(), want), f"split {i} at {pos}"
        pos += T


def test_hash_wrapping_and_negative_tokens(E):
    """Multipliers with the top bit region set, tokens of every map class."""
    cfg = configs.TINY
    g = E.make_geom(2, 3, 2, 64, 128, 2, 32, 8)
    tm = np.array([0, 1, 2, 3, 4, 5, -1, 600], dtype=np.int64)
    mult = np.array([(1 << 62) + 1, (1 << 62) - 1, 3, 7, (1 << 61) + 5, 11], dtype=np.int64)
    primes = np.array([5, 7, 11, 13, 17, 19, 23, 29], dtype=np.int64)
    offs = np.array([0, 5, 12, 23, 0, 17, 36, 59], dtype=np.int64)
    hs = E.Hasher(E.Tables(g, tm, 0, mult, primes, offs), 512, 8)
    ref = oracle.HashState(tm, 0, mult, primes, offs, 2, 3, 2, 512, 8)
    ids = np.array(np.unravel_index(np.arange(512), (8, 8, 8))).T.astype(np.int32)  # all 3-windows
    out = torch.empty((512, 3, 2, 4), dtype=torch.int64, device="cuda")
    E.engram_hash(hs, torch.from_numpy(np.ascontiguousarray(ids)).cuda(), 3, 0, out)
    assert np.array_equal(out.cpu().numpy(), ref.forward(ids, 0))
    del cfg


def test_hash_token_out_of_range_sets_error(E):
    hs, _ = _hash_setup(E, configs.TINY, 1)
    ids = torch.tensor([[3, 1000, 5]], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 3, 1, 4), dtype=torch.int64, device="cuda")
    E.engram_hash(hs, ids, 3, 0, out)
    assert E.engram_check() == -7
    assert E.engram_check() == 0                          # read-and-clear
    with pytest.raises(E.EngramError) as e:
        E.engram_hash(hs, ids, 3, 4094, out)              # 4094 + 3 > max_seq 4096
    assert e.value.code == -4


# ---------------------------------------------------------------- rows ----

@pytest.mark.parametrize("hd,blk", [(64, 32), (256, 32), (256, 16), (128, 64), (32, 32)])
def test_rows_fp8_every_code_bit_exact(E, hd, blk):
    codes = np.array([b for b in range(256) if b & 0x7F != 0x7F], dtype=np.uint8)
    R = 40
    rng = np.random.default_rng(hd + blk)
    table = rng.choice(codes, size=(R, hd)).astype(np.uint8)
    table[0, :] = np.resize(codes, hd)
    k = rng.integers(-10, 11, size=(R, hd // blk))
    scales = (2.0 ** k).astype(np.float32)
    C, n_tok = 3, 17
    ids = rng.integers(0, R, size=(n_tok, 5)).astype(np.int64)   # id_stride 5 > C
    ids[0, :C] = 0
    d_rows = torch.empty((n_tok * C, hd), dtype=torch.bfloat16, device="cuda")
    E.engram_rows_fp8(torch.from_numpy(table).cuda(), torch.from_numpy(scales).cuda(), R, hd, blk,
                      torch.from_numpy(ids).cuda(), n_tok, 5, C, d_rows)
    assert E.engram_check() == 0
    want = oracle.rows_fp8(table, scales, hd, blk, ids[:, :C].reshape(-1))
    assert np.array_equal(_u16(d_rows).reshape(-1, hd), want)


def test_rows_fp8_synth_table_and_bad_id(E):
    cfg = configs.V41_DECODE
    rows = np.array([0, 5, 77, 3_000_000, 123_456], dtype=np.int64)
    codes, scales = synth.table_fp8_rows(cfg, 1, rows)
    ids = np.array([[0, 1, 2, 3, 4, 1], [4, 3, 2, 1, 0, 99]], dtype=np.int64)
    d_rows = torch.empty((12, 256), dtype=torch.bfloat16, device="cuda")
    E.engram_rows_fp8(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), 5, 256, 32,
                      torch.from_numpy(ids).cuda(), 2, 6, 6, d_rows)
    assert E.engram_check() == -8                         # id 99 outside 5 rows
    got = _u16(d_rows).reshape(2, 6, 256)
    assert np.array_equal(got[0], oracle.rows_fp8(codes, scales, 256, 32, ids[0]))
    assert not got[1, 5].any()                            # the bad row reads as zeros


def test_rows_q2k_bit_exact(E):
    import json
    import os
    from conftest import GOLDEN
    cfg = configs.V41_Q2K
    blocks = synth.table_q2k_rows(cfg, 0, np.arange(200))
    g = json.load(open(os.path.join(GOLDEN, "q2k_hand.json")))
    blocks[7] = np.frombuffer(bytes.fromhex(g["block_hex"]), dtype=np.uint8)
    rng = np.random.default_rng(9)
    ids = rng.integers(0, 200, size=(33, 24)).astype(np.int64)
    ids[0, 0] = 7
    d_rows = torch.empty((33 * 24, 256), dtype=torch.bfloat16, device="cuda")
    E.engram_rows_q2k(torch.from_numpy(blocks).cuda(), 200, torch.from_numpy(ids).cuda(), 33, 24, 24,
                      d_rows)
    assert E.engram_check() == 0
    got = _u16(d_rows).reshape(-1, 256)
    assert np.array_equal(got, oracle.rows_q2k(blocks, ids.reshape(-1)))
    hand = oracle.bf16_bits_to_f32(got[0])
    for v, want in g["expected"].items():
        assert hand[int(v)] == want


# ---------------------------------------------------------- projection ----

@pytest.mark.parametrize("T,K,N", [(1, 6144, 2048), (3, 6144, 1040), (8, 1024, 512),
                                   (9, 256, 384), (100, 1024, 528), (300, 512, 1024)])
def test_project_vs_oracle(E, T, K, N):
    rng = np.random.default_rng(T * 7 + K)
    x = synth.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32) * 2)
    w = synth.to_bf16_bits(0.02 * rng.standard_normal((N, K)).astype(np.float32))
    d_kv = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    E.engram_project(torch.from_numpy(x.view(np.int16)).cuda(), torch.from_numpy(w.view(np.int16)).cuda(),
                     T, K, N, d_kv)
    assert E.engram_check() == 0
    want = oracle.linear_bf16(x, w)
    assert G.kv_rel_err(_u16(d_kv), want) <= G.KV_TOL


@pytest.mark.parametrize("T,N", [(512, 20480), (300, 1040)])
def test_project_cta_pairs_bit_identical_to_one_cta(E, T, N):
    """From 256 tokens the projection runs on CTA pairs (256 x 256 tiles); its
    kv equals, bit for bit, the one-CTA tensor-core GEMM's on the same rows
    (computed here 250 rows at a time, each call below 256 tokens), and the
    oracle's within tolerance on sampled rows."""
    K = 6144
    rng = np.random.default_rng(T + N)
    x = synth.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    w = synth.to_bf16_bits(0.02 * rng.standard_normal((N, K)).astype(np.float32))
    d_x = torch.from_numpy(x.view(np.int16)).cuda()
    d_w = torch.from_numpy(w.view(np.int16)).cuda()
    kv2 = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    E.engram_project(d_x, d_w, T, K, N, kv2)
    kv1 = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, T, 250):
        r1 = min(T, r0 + 250)
        assert r1 - r0 > 8                           # stays on the GEMM, not the GEMV
        E.engram_project(d_x[r0:r1].contiguous(), d_w, r1 - r0, K, N, kv1[r0:r1])
    assert E.engram_check() == 0
    assert torch.equal(kv1.view(torch.int16), kv2.view(torch.int16))
    rows = np.unique(np.concatenate([np.arange(0, T, 37), [T - 1]]))
    want = oracle.linear_bf16(x[rows], w)
    assert G.kv_rel_err(_u16(kv2)[rows], want) <= G.KV_TOL


# ---------------------------------------------------------------- gate ----

# rows = T x hc: up to 512 the layer-pipelined variant, above it the
# register-lean one (four CTAs an SM), D from 8 to 16384
@pytest.mark.parametrize("N,K", [(120, 4800), (1040, 6144), (7, 16), (20480, 2056)])
def test_tile_wkv_layout(E, N, K):
    """engram_tile_wkv against the layout written out in numpy: 16-row x
    2048-column tiles, g-major, zero past the last row and column."""
    g = torch.Generator(device="cpu").manual_seed(N * 7 + K)
    w = torch.randint(-32768, 32767, (N, K), generator=g, dtype=torch.int32).to(torch.int16)
    d_w = w.cuda().view(torch.bfloat16)
    nbytes = E.engram_tiled_wkv_bytes(N, K)
    G, C = -(-N // 16), -(-K // 2048)
    assert nbytes == G * C * 16 * 2048 * 2
    d_t = torch.full((nbytes // 2,), -1, dtype=torch.int16, device="cuda")   # poison: every slot written
    E.engram_tile_wkv(d_w, N, K, d_t.view(torch.bfloat16))
    torch.cuda.synchronize()
    want = np.zeros((G * 16, C * 2048), dtype=np.int16)
    want[:N, :K] = w.numpy()
    want = want.reshape(G, 16, C, 2048).transpose(0, 2, 1, 3).ravel()
    assert np.array_equal(d_t.cpu().numpy(), want)


@pytest.mark.parametrize("T,hc,D", [(16, 2, 128), (5, 4, 4096), (3, 1, 8), (2, 3, 16384), (7, 4, 1000),
                                   (200, 4, 4096), (300, 2, 1000), (129, 4, 16384), (700, 4, 4096),
                                   (150, 4, 3000)])
def test_gate_vs_oracle(E, T, hc, D):
    rng = np.random.default_rng(T + hc + D)
    h = rng.standard_normal((T, hc, D)).astype(np.float32)
    kv = synth.to_bf16_bits(rng.standard_normal((T, (hc + 1) * D)).astype(np.float32) * 0.5)
    q = oracle.bf16_bits_to_f32(synth.to_bf16_bits(1 + 0.05 * rng.standard_normal((hc, D)).astype(np.float32)))
    k = oracle.bf16_bits_to_f32(synth.to_bf16_bits(1 + 0.05 * rng.standard_normal((hc, D)).astype(np.float32)))
    d_h = torch.from_numpy(h).cuda()
    E.engram_gate(d_h, torch.from_numpy(kv.view(np.int16)).cuda(), torch.from_numpy(q * k).cuda(), T, hc, D,
                  1e-6)
    want = oracle.gate(h, kv, q, k, hc, D, 1e-6)
    assert np.abs(d_h.cpu().numpy() - want).max() <= G.H_TOL


def test_gate_value_zero_keeps_h_bits(E):
    T, hc, D = 4, 4, 512
    rng = np.random.default_rng(1)
    h = rng.standard_normal((T, hc, D)).astype(np.float32)
    kv = np.zeros((T, (hc + 1) * D), dtype=np.uint16)
    kv[:, :hc * D] = synth.to_bf16_bits(rng.standard_normal((T, hc * D)).astype(np.float32))
    d_h = torch.from_numpy(h).cuda()
    qk = torch.ones((hc, D), dtype=torch.float32, device="cuda")
    E.engram_gate(d_h, torch.from_numpy(kv.view(np.int16)).cuda(), qk, T, hc, D, 1e-6)
    assert np.array_equal(d_h.cpu().numpy().view(np.uint32), h.view(np.uint32))


def test_hash_remainder_extreme_primes(E):
    """The Euclidean remainder for moduli from 1 to just below 2^63, on wrapped
    products of both signs: bit-exact against the oracle."""
    primes = np.array([1, 2, 3, (1 << 31) - 1, (1 << 40) + 15, (1 << 62) + 135, (1 << 63) - 25, 509],
                      dtype=np.int64)
    L, ng, H = 2, 3, 2
    offs = np.zeros(8, dtype=np.int64)
    rng = np.random.default_rng(3)
    mult = rng.integers(1, 1 << 62, size=L * ng, dtype=np.int64) | 1
    tm = rng.integers(0, 1 << 40, size=64, dtype=np.int64)
    g = E.make_geom(L, ng, H, 64, 128, 2, 32, 64)
    hs = E.Hasher(E.Tables(g, tm, 0, mult, primes, offs), 16, 64)
    ref = oracle.HashState(tm, tm[0], mult, primes, offs, L, ng, H, 16, 64)
    ids = rng.integers(0, 64, size=(16, 40)).astype(np.int32)
    out = torch.empty((16, 40, L, 4), dtype=torch.int64, device="cuda")
    E.engram_hash(hs, torch.from_numpy(ids).cuda(), 40, 0, out)
    assert np.array_equal(out.cpu().numpy(), ref.forward(ids, 0))

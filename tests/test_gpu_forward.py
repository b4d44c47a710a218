"""End-to-end parity of engram_forward on the five workloads.

For every call: the row ids in the workspace equal the oracle's hash exactly;
the kv of each layer in the workspace is within 2e-2 of the oracle projection
of the oracle's own rows (all outputs on the tiny workload, a seeded sample of
tokens x outputs on the V4.1-shaped ones); the highway is within 1e-3 of the
oracle gates applied layer after layer to the GPU's kv (stage-wise).
"""
import numpy as np
import pytest
import torch

import oracle_glue as G
from deepseek_v4_engram_hash_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import __graft_entry__
    __graft_entry__.build()
    from deepseek_v4_engram_hash_gb300 import _lib
    return _lib


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_call(eng, ref, ids, start_pos, d_h, h0_rows, tok_sample, out_sample, first_token, e2e=True):
    """Run one forward and check it.  h0_rows: f32 [len(tok_sample), hc, D] of
    the highway rows tok_sample before the call (regenerated on the CPU).
    With e2e, the oracle projects the sampled tokens onto every output: kv is
    checked on all N outputs and the highway end to end (oracle kv) against
    the derived bound, besides stage-wise."""
    cfg = eng.cfg
    B, T = ids.shape
    M = B * T
    eng.forward(ids, start_pos, d_h)
    from deepseek_v4_engram_hash_gb300 import _lib as E
    assert E.engram_check() == 0
    want_ids = ref.forward(ids, start_pos).reshape(M, cfg.n_layers, cfg.cols)
    got_ids = eng.row_ids(M).cpu().numpy()
    assert np.array_equal(got_ids, want_ids), "row ids"
    h = h0_rows.copy()
    lay = eng.workspace_layout(M)
    x_kept = lay[1 + 2 * cfg.n_layers] > lay[1 + cfg.n_layers]     # GEMM steps keep x in the workspace
    kv_g, kv_o = [], []
    for l in range(cfg.n_layers):
        kv_gpu = _u16(eng.kv(M, l))[tok_sample]                     # [S, N]
        x = G.x_of(cfg, l, want_ids[tok_sample])
        if x_kept:
            assert np.array_equal(_u16(eng.x(M, l))[tok_sample], x), f"layer {l} x rows"
        if e2e:
            want_kv = G.kv(cfg, l, x)                               # every output
            err = G.kv_rel_err(kv_gpu, want_kv)
            kv_o.append(want_kv)
        else:
            want_kv = G.kv(cfg, l, x, out_sample)
            err = G.kv_rel_err(kv_gpu[:, out_sample], want_kv)
        assert err <= G.KV_TOL, f"layer {l} kv rel err {err}"
        kv_g.append(kv_gpu)
        h = G.gate(cfg, l, h, kv_gpu)                               # stage-wise
    got_h = d_h.view(M, cfg.hc, cfg.dim)[torch.as_tensor(tok_sample, device=d_h.device)].cpu().numpy()
    dh = np.abs(got_h - h).max()
    assert dh <= G.H_TOL, f"highway |dh| {dh}"
    if e2e:
        dh_e2e, margin = G.e2e_highway(cfg, h0_rows, kv_g, kv_o, got_h)
        print(f"[e2e] {cfg.name} T={T} B={B}: stage-wise |dh| {dh:.3g}; end-to-end |dh| {dh_e2e:.3g}, "
              f"smallest margin to the bound {margin:.3g}")
        assert margin >= 0.0, f"end-to-end highway outside the derived bound by {-margin}"
    return dh


def _h_device(cfg, first_token, M, numpy_ok):
    if numpy_ok:
        return torch.from_numpy(synth.highway(cfg, np.arange(first_token, first_token + M))).cuda()
    d_h = torch.empty((M, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    synth.fill_highway_cuda(cfg, d_h, first_token)
    return d_h


def test_forward_tiny_full(E):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    ref = G.hash_state(cfg, 1)
    pos, first = 0, 0
    for T in (cfg.T, 1, 1, 1, 5):                       # prefill (tensor path), decode (GEMV path)
        ids = eng.ids_for(f"tiny{pos}", T)
        d_h = _h_device(cfg, first, T, True)
        h0 = d_h.cpu().numpy()
        _check_call(eng, ref, ids, pos, d_h, h0, np.arange(T), np.arange(cfg.N), first)
        pos += T
        first += T


def _sample(rng, n, k):
    return np.sort(rng.choice(n, size=min(n, k), replace=False))


@pytest.mark.parametrize("name", ["v41_decode_T1", "v41_prefill_T4096", "v41_q2k_T512"])
def test_forward_v41(E, name):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.CONFIGS[name]
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=max(cfg.T, 1))
    ref = G.hash_state(cfg, 1)
    rng = np.random.default_rng(11)
    pos = 0
    if cfg.prefix:
        from deepseek_v4_engram_hash_gb300 import _lib as EL
        pre = eng.ids_for("prefix", cfg.prefix)
        out = torch.empty((1, cfg.prefix, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        EL.engram_hash(eng.hasher, torch.from_numpy(pre).cuda(), cfg.prefix, 0, out)
        assert np.array_equal(out.cpu().numpy(), ref.forward(pre, 0))
        pos = cfg.prefix
    calls = 3 if cfg.T == 1 else 1
    outs = np.concatenate([np.arange(0, cfg.N, 97), [cfg.dim - 1, cfg.dim, cfg.hc * cfg.dim,
                                                       cfg.N - 1]])
    outs = np.unique(outs)
    for i in range(calls):
        T = cfg.T
        ids = eng.ids_for(f"call{i}", T)
        d_h = _h_device(cfg, pos, T, T <= 64)
        toks = _sample(rng, T, 24) if T > 24 else np.arange(T)
        h0 = synth.highway(cfg, pos + toks)
        _check_call(eng, ref, ids, pos, d_h, h0, toks, outs, pos)
        pos += T


def test_forward_stress_batch8_prefill_then_decode(E):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.STRESS
    B = cfg.batch
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * cfg.T)
    ref = G.hash_state(cfg, B)
    rng = np.random.default_rng(12)
    outs = np.unique(np.concatenate([np.arange(5, cfg.N, 211), [cfg.N - 1]]))
    ids = eng.ids_for("prefill", cfg.T)
    M = B * cfg.T
    d_h = _h_device(cfg, 0, M, False)
    toks = _sample(rng, M, 256)
    _check_call(eng, ref, ids, 0, d_h, synth.highway(cfg, toks), toks, outs, 0)
    pos, first = cfg.T, M
    for step in range(3):                               # single-token decode of all 8 sequences
        ids = eng.ids_for(f"dec{step}", 1)
        d_h = _h_device(cfg, first, B, True)
        _check_call(eng, ref, ids, pos, d_h, d_h.cpu().numpy(), np.arange(B), outs, first)
        pos += 1
        first += B


@pytest.mark.parametrize("tables,weights,B", [("fp8", "bf16", 1), ("e8m0", "bf16", 1), ("q2k", "bf16", 1),
                                              ("q2k", "q2k", 1), ("fp8", "q2k", 1), ("fp8", "bf16", 8),
                                              ("q2k", "q2k", 8)])
def test_forward_fused_gemv_matches_staged_calls(E, tables, weights, B):
    """A decode step of B sequences (B tokens, the GEMV path): the forward's
    fused gather + GEMV gives the same kv bits as the row kernel
    (engram_rows_fp8, engram_rows_fp8_e8m0 or engram_rows_q2k) followed by
    engram_project (or engram_project_q2k, one token a call): the rows decoded
    into the mma fragments in registers equal the row kernel's, bit for bit,
    and each token's column of the mma is independent of the others."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = {"fp8": configs.V41_DECODE, "e8m0": configs.V41_DECODE_E8M0, "q2k": configs.V41_Q2K.with_(T=1)}[tables]
    if weights == "q2k":
        cfg = cfg.with_(wkv_fmt="q2k")
    cfg = cfg.with_(batch=B)
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B)
    ids = eng.ids_for("fused", 1)                                            # [B, 1]
    d_h = _h_device(cfg, 0, B, True)
    eng.forward(ids, 7, d_h)
    assert E.engram_check() == 0
    row_ids = eng.row_ids(B).clone()                                         # [B, L, C]
    for l in range(cfg.n_layers):
        d = eng.layer_data[l]
        x = torch.empty((B * cfg.cols, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
        rid = row_ids[:, l, :].contiguous()
        if tables == "fp8":
            E.engram_rows_fp8(d["table"], d["scales"], d["rows"], cfg.head_dim, cfg.scale_block, rid, B,
                              cfg.cols, cfg.cols, x)
        elif tables == "e8m0":
            E.engram_rows_fp8_e8m0(d["table"], d["scales"], d["rows"], cfg.head_dim, cfg.scale_block, rid, B,
                                   cfg.cols, cfg.cols, x)
        else:
            E.engram_rows_q2k(d["table"], d["rows"], rid, B, cfg.cols, cfg.cols, x)
        xt = x.view(B, cfg.K)
        kv = torch.empty((B, cfg.N), dtype=torch.bfloat16, device="cuda")
        if weights == "q2k":
            for t in range(B):
                E.engram_project_q2k(xt[t:t + 1], d["wkv_q2k"], cfg.K, cfg.N, kv[t:t + 1])
        else:
            E.engram_project(xt, d["wkv"], B, cfg.K, cfg.N, kv)
        assert E.engram_check() == 0
        assert torch.equal(kv.view(torch.int16), eng.kv(B, l).view(torch.int16)), f"layer {l}"


@pytest.mark.parametrize("name", ["v41", "odd_n", "wide_c"])
def test_forward_tiled_wkv_bit_identical(E, name):
    """The 1..8-token projection reading the tiled wkv gives the same kv and
    highway bits as reading row-major wkv (V4.1 at 1, 2 and 8 tokens; N = 120
    with a short last row group; K = 4800 with a part-filled last tile)."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = {"v41": configs.V41_DECODE.with_(batch=1, T=8), "odd_n": ODD_N, "wide_c": WIDE_C}[name]
    B = 1 if name == "v41" else cfg.batch
    engs = [runner.EngramSetup(cfg, batch=B, max_tokens=8 * B, tiled_wkv=t) for t in (True, False)]
    assert "wkv_tiled" in engs[0].layer_data[0] and "wkv_tiled" not in engs[1].layer_data[0]
    pos, first = 0, 0
    for T in (1, 2, 8, 1):
        M = B * T
        if M > 8:
            continue
        ids = engs[0].ids_for(f"tiled{pos}", T)
        outs = []
        for eng in engs:
            d_h = _h_device(cfg, first, M, True)
            eng.forward(ids, pos, d_h)
            assert E.engram_check() == 0
            outs.append((d_h.clone(), [eng.kv(M, l).clone() for l in range(cfg.n_layers)]))
        assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32)), "highway"
        for l in range(cfg.n_layers):
            assert torch.equal(outs[0][1][l].view(torch.int16), outs[1][1][l].view(torch.int16)), f"kv {l}"
        pos += T
        first += M


def test_hasher_reset_clears_the_lookback(E):
    """engram_hasher_reset returns the look-back cache to zeros (and the
    projection's work counters): a decode step after a prefill and a reset
    hashes its window over zeros, as a fresh oracle state does, and every
    output of that step checks."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    pre = eng.ids_for("reset-prefill", cfg.T)
    eng.forward(pre, 0, _h_device(cfg, 0, cfg.T, True))
    assert E.engram_check() == 0
    E.engram_hasher_reset(eng.hasher)
    ids = eng.ids_for("reset-step", 2)
    kept = G.hash_state(cfg, 1)
    kept.forward(pre, 0)
    fresh = G.hash_state(cfg, 1)
    assert not np.array_equal(kept.forward(ids, cfg.T), G.hash_state(cfg, 1).forward(ids, cfg.T)), \
        "the windows must reach into the prefill for the reset to show"
    d_h = _h_device(cfg, cfg.T, 2, True)
    _check_call(eng, fresh, ids, cfg.T, d_h, d_h.cpu().numpy(), np.arange(2), np.arange(cfg.N), cfg.T)


ODD_FP8 = configs.TINY.with_(
    name="odd_fp8", vocab=5000, n_compressed=3000, unmapped_5pct=True, pad_token_id=7,
    pad_compressed=-1, layer_ids=(2, 9, 30), max_ngram=5, n_heads=3, prime_target=1000,
    head_dim=128, scale_block=64, dim=256, hc=3, batch=2, T=37, ids="uniform", seed=5)

ODD_Q2K = configs.TINY.with_(
    name="odd_q2k", vocab=700, n_compressed=400, unmapped_5pct=True, pad_token_id=3,
    pad_compressed=None, layer_ids=(1, 4), max_ngram=2, n_heads=5, prime_target=300,
    head_dim=256, scale_block=32, dim=64, hc=1, fmt="q2k", batch=3, T=9, ids="uniform", seed=6)


# N = 40 x 3 = 120: the last 16-row group of wkv holds 8 rows (the GEMV's
# short last group, the GEMM's partial column tile).
ODD_N = configs.TINY.with_(name="odd_n", dim=40, hc=2, batch=3, T=7, seed=7)

# C = 15 x 20 = 300 columns: 8 tokens are 2400 row ids, more than a GEMV CTA
# hashes itself, so the hash kernel runs first and the GEMV gathers from the
# ids in the workspace (4 tokens stay fused); K = 300 x 16 = 4800.
WIDE_C = configs.TINY.with_(name="wide_c", layer_ids=(3,), max_ngram=16, n_heads=20, prime_target=97,
                            head_dim=16, scale_block=16, dim=64, hc=1, batch=4, T=12, seed=8)


# Table formats differing between layers: fp8, Q2_K and e8m0 layers (the
# larger steps then hash in their own launch and gather layer by layer), and
# f32 beside e8m0 scales (one fused hash + gather launch reading both).
MIXED_Q2K = configs.TINY.with_(name="mixed_q2k", layer_ids=(1, 4, 7), head_dim=256, scale_block=32,
                               layer_fmts=("fp8", "q2k", "fp8_e8m0"), batch=2, T=11, seed=9)
MIXED_E8M0 = configs.TINY.with_(name="mixed_e8m0", layer_ids=(2, 5), head_dim=128, scale_block=16,
                                layer_fmts=("fp8_e8m0", "fp8"), batch=2, T=13, seed=10)


@pytest.mark.parametrize("cfg", [ODD_FP8, ODD_Q2K, ODD_N, WIDE_C, MIXED_Q2K, MIXED_E8M0], ids=lambda c: c.name)
def test_forward_odd_geometry_all_paths(E, cfg):
    """Three layers / pad id -1 / 5-grams / 64-wide scale blocks, Q2_K at
    C = 5, N = 120 (a short last row group), and table formats that differ
    between layers; the call sequence crosses both projection paths (GEMM
    above 8 tokens, fused GEMV at or below) and checks every output."""
    from deepseek_v4_engram_hash_gb300 import runner
    B = cfg.batch
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * cfg.T)
    ref = G.hash_state(cfg, B)
    pos, first = 0, 0
    for T in (cfg.T, 1, 2, 0, 1, 4, 1):
        M = B * T
        if B * T > B * cfg.T:
            continue
        ids = eng.ids_for(f"odd{pos}", T)
        d_h = _h_device(cfg, first, max(M, 1), True)[:M]
        h0 = d_h.cpu().numpy()
        if M == 0:
            eng.forward(ids, pos, d_h)
            assert E.engram_check() == 0
            continue
        _check_call(eng, ref, ids, pos, d_h, h0, np.arange(M), np.arange(cfg.N), first)
        pos += T
        first += M


def test_forward_all_unmapped_tokens_use_pad_windows(E):
    """Every token maps to -1: every window is all pad, so every id equals
    rem_euclid(rolling(pad, ..., pad)) + offset, identical at every position."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=12)
    unmapped = int(np.flatnonzero(eng.hash_np["token_map"] == -1)[0])
    ids = np.full((1, 12), unmapped, dtype=np.int32)
    d_h = _h_device(cfg, 0, 12, True)
    ref = G.hash_state(cfg, 1)
    _check_call(eng, ref, ids, 0, d_h, d_h.cpu().numpy(), np.arange(12), np.arange(cfg.N), 0)
    got = eng.row_ids(12).cpu().numpy()
    assert (got == got[0]).all()


@pytest.mark.parametrize("T,pinned", [(1, True), (6, True), (1, False), (6, False)])
def test_forward_host_buffers_match_device_forward(E, T, pinned):
    """engram_forward_host gives the same highway as engram_forward: from
    page-locked buffers (read and updated in place by the kernels) and from
    pageable ones (staged through device buffers)."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY.with_(batch=2)
    eng = runner.EngramSetup(cfg, batch=2, max_tokens=2 * T)
    hs2 = E.Hasher(eng.tables, 2, cfg.max_seq)
    pos = 0
    for step in range(3):
        ids = eng.ids_for(f"host{step}", T)
        h0 = synth.highway(cfg, np.arange(2 * T * step, 2 * T * (step + 1)))
        d_h = torch.from_numpy(h0).cuda()
        eng.forward(ids, pos, d_h)
        h_ids = torch.from_numpy(ids.copy())
        h_h = torch.from_numpy(h0.copy())
        if pinned:
            h_ids, h_h = h_ids.pin_memory(), h_h.pin_memory()
        d_ids2 = torch.empty((2, T), dtype=torch.int32, device="cuda")
        d_h2 = torch.empty((2 * T, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
        E.engram_forward_host(hs2, eng.layers, h_ids, d_ids2, T, pos, h_h, d_h2, cfg.eps, eng.ws, eng.ws_bytes)
        torch.cuda.synchronize()
        assert E.engram_check() == 0
        assert torch.equal(h_h, d_h.cpu())
        pos += T


MAX_GEO = configs.TINY.with_(
    name="max_geometry", layer_ids=(1, 2, 3, 4), max_ngram=16, n_heads=1, prime_target=97,
    head_dim=64, scale_block=32, dim=64, hc=4, batch=1, T=20, seed=9)


def test_forward_maximum_geometry(E):
    """Four layers (the most the kernels take), 16-gram windows (C = 15), hc = 4;
    300 tokens take the CTA-pair GEMM with four layers in one launch, a
    half-empty pair row tile and a 64-column partial column tile (N = 320)."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = MAX_GEO
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=300)
    ref = G.hash_state(cfg, 1)
    pos = 0
    for T in (cfg.T, 1, 3, 300):
        ids = eng.ids_for(f"max{pos}", T)
        d_h = _h_device(cfg, pos, T, True)
        _check_call(eng, ref, ids, pos, d_h, d_h.cpu().numpy(), np.arange(T), np.arange(cfg.N), pos)
        pos += T


def test_long_decode_carries_lookback(E):
    """512 single-token steps of 8 sequences after a 1536-token prefill (the
    large-table workload's decode, on V4.1-sized tables): every step's row
    ids equal the oracle's."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.V41_DECODE.with_(batch=8, prefix=0, T=1536, ids="uniform", decode_steps=512)
    B = cfg.batch
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * cfg.T)
    ref = G.hash_state(cfg, B)
    ids = eng.ids_for("prefill", cfg.T)
    d_h = _h_device(cfg, 0, B * cfg.T, False)
    eng.forward(ids, 0, d_h)
    assert np.array_equal(eng.row_ids(B * cfg.T).cpu().numpy(),
                          ref.forward(ids, 0).reshape(B * cfg.T, cfg.n_layers, cfg.cols))
    steps = eng.ids_for("decode", 512)
    d_h = _h_device(cfg, 0, B, True)
    got = []
    for k in range(512):
        eng.forward(np.ascontiguousarray(steps[:, k:k + 1]), cfg.T + k, d_h)
        got.append(eng.row_ids(B).clone())
    assert E.engram_check() == 0
    for k in range(512):
        want = ref.forward(steps[:, k:k + 1], cfg.T + k).reshape(B, cfg.n_layers, cfg.cols)
        assert np.array_equal(got[k].cpu().numpy(), want), f"step {k}"
    # the last step's projection, one output row from every 16-row group of both
    # layers: after 512 launches the groups still all get computed
    last = got[-1].cpu().numpy()
    rows = np.arange(0, cfg.N, 16) + np.arange(cfg.N // 16) % 16
    for l in range(cfg.n_layers):
        kv_gpu = _u16(eng.kv(B, l))[:, rows]
        want_kv = G.kv(cfg, l, G.x_of(cfg, l, last), rows)
        assert G.kv_rel_err(kv_gpu, want_kv) <= G.KV_TOL, f"layer {l} kv after 512 steps"


@pytest.mark.parametrize("name,T", [("v41_decode_T1", 1), ("tiny", 16), ("v41_prefill_T4096", 4096)])
def test_forward_is_bit_reproducible(E, name, T):
    """Fixed reduction orders everywhere: two runs give the same bits."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.CONFIGS[name]
    outs = []
    for _ in range(2):
        eng = runner.EngramSetup(cfg, batch=1, max_tokens=T)
        d_h = _h_device(cfg, 0, T, False)
        eng.forward(eng.ids_for("repro", T), 0, d_h)
        outs.append((d_h.clone(), [eng.kv(T, l).clone() for l in range(cfg.n_layers)]))
        del eng
    assert torch.equal(outs[0][0], outs[1][0])
    for a, b in zip(outs[0][1], outs[1][1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# One layer, N = 20480 (80 column tiles of 256) at 256 tokens: 80 pair tiles on
# the GPU's pairs leave a last wave of 4 tiles, which the forward cuts along K
# (K = 512: 8 ranges of one k step); every output of every token is checked.
KSPLIT = configs.TINY.with_(name="ksplit_tail", layer_ids=(0,), max_ngram=3, n_heads=1, prime_target=509,
                            head_dim=256, scale_block=32, dim=4096, hc=4, batch=1, T=256, seed=13)


def test_forward_ksplit_last_wave(E):
    """The CTA-pair GEMM's last wave cut along K (f32 partial tiles added in
    range order by the fix-up launch): kv within tolerance of the oracle on
    every output, the highway stage-wise and end to end, and two runs
    bit-identical (the fix-up's order is fixed)."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = KSPLIT
    outs = []
    for rep in range(2):
        eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
        ids = eng.ids_for("ksplit", cfg.T)
        d_h = _h_device(cfg, 0, cfg.T, True)
        if rep == 0:
            _check_call(eng, G.hash_state(cfg, 1), ids, 0, d_h, d_h.cpu().numpy(), np.arange(cfg.T),
                        np.arange(cfg.N), 0)
        else:
            eng.forward(ids, 0, d_h)
            assert E.engram_check() == 0
        outs.append((d_h.clone(), eng.kv(cfg.T, 0).clone()))
        del eng
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))


# Two layers, N = 4000 (a 160-column last column tile), 768 tokens (three pair
# rows): 96 pair tiles leave a last wave of 20 tiles, cut into K ranges; the
# fix-up must stop at column N.
KSPLIT_RAGGED = configs.TINY.with_(name="ksplit_ragged", layer_ids=(0, 3), max_ngram=3, n_heads=1,
                                   prime_target=509, head_dim=128, scale_block=32, dim=1000, hc=3,
                                   batch=3, T=256, seed=14)


def test_forward_ksplit_ragged_columns_two_layers(E):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = KSPLIT_RAGGED
    eng = runner.EngramSetup(cfg, batch=cfg.batch, max_tokens=cfg.batch * cfg.T)
    ids = eng.ids_for("ksplit-ragged", cfg.T)
    M = cfg.batch * cfg.T
    d_h = _h_device(cfg, 0, M, True)
    _check_call(eng, G.hash_state(cfg, cfg.batch), ids, 0, d_h, d_h.cpu().numpy(), np.arange(M),
                np.arange(cfg.N), 0)


def test_forward_ksplit_inside_a_multi_step_graph(E):
    """Two 256-token steps captured in one graph: the pair GEMM's K-split last
    wave and its fix-up launch replay bit-identically to eager calls."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = KSPLIT
    K = 2
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    hs2 = E.Hasher(eng.tables, 1, cfg.max_seq)
    ws2 = torch.empty_like(eng.ws)
    ids = np.stack([eng.ids_for(f"ksg{k}", cfg.T) for k in range(K)])                   # [K, 1, T]
    h0 = torch.from_numpy(synth.highway(cfg, np.arange(K * cfg.T))).view(K, cfg.T, cfg.hc, cfg.dim)
    d_he = [h0[k].clone().cuda() for k in range(K)]
    for k in range(K):
        eng.forward(ids[k], k * cfg.T, d_he[k])
    d_pos = torch.zeros((1,), dtype=torch.int64, device="cuda")
    d_ids = torch.from_numpy(ids).cuda()
    d_hg = h0.clone().cuda()
    graph = E.Graph(hs2, eng.layers, d_ids, cfg.T, d_pos, d_hg, cfg.eps, ws2, eng.ws_bytes, steps=K)
    graph.launch()
    assert E.engram_check() == 0
    for k in range(K):
        assert torch.equal(d_he[k].view(torch.int32), d_hg[k].view(torch.int32)), f"step {k}"
    assert d_pos.item() == K * cfg.T
    graph.close()

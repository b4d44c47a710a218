"""The single-token projection from Q2_K-quantised wkv (`wkv_q2k`, 84-byte
blocks, 6x fewer weight bytes): bit-identical to the bf16 GEMV on the
dequantised weights, as the GPU module page states, and within tolerance of
the oracle; the forward with it gives bit-identical highways."""
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
    return _lib


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# (narrower K: warps past the last block decode a clamped block against zero x,
# which must add exact zeros, so those shapes with N % 16 == 0 check the bits too)
@pytest.mark.parametrize("K,N", [(6144, 20480), (256, 100), (1536, 777), (256, 96), (1536, 784), (4352, 160)])
def test_project_q2k_bit_identical_to_bf16_on_dequantised(E, K, N):
    cfg = configs.V41_DECODE
    nb = N * (K // 256)
    blocks = torch.empty((nb, 84), dtype=torch.uint8, device="cuda")
    synth.fill_table_q2k_cuda(cfg, 3, blocks, tag="wkvq2k")
    w = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    E.engram_rows_q2k(blocks, nb, torch.arange(nb, device="cuda"), nb, 1, 1, w)
    rng = np.random.default_rng(K + N)
    x = torch.from_numpy(synth.to_bf16_bits(rng.standard_normal((1, K)).astype(np.float32)).view(np.int16)).cuda()
    kv_q = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    kv_b = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    E.engram_project_q2k(x, blocks, K, N, kv_q)
    if N % 16 == 0:
        E.engram_project(x, w, 1, K, N, kv_b)
        assert torch.equal(kv_q.view(torch.int16), kv_b.view(torch.int16))
    assert E.engram_check() == 0
    rows = np.unique(np.concatenate([np.arange(0, N, max(1, N // 97)), [N - 1]]))
    blk_ids = (rows[:, None] * (K // 256) + np.arange(K // 256)[None]).ravel()
    cpu_blocks = synth.table_q2k_rows(cfg, 3, blk_ids, tag="wkvq2k")        # regenerated on the CPU
    wq = oracle.rows_q2k(cpu_blocks, np.arange(blk_ids.size))
    want = oracle.linear_bf16(x.cpu().numpy().view(np.uint16), wq.reshape(rows.size, K))
    assert G.kv_rel_err(_u16(kv_q)[:, rows], want) <= G.KV_TOL


@pytest.mark.parametrize("B", [1, 2, 3, 8])
def test_forward_wkv_q2k_matches_bf16_path_and_oracle(E, B):
    """Decode steps of B sequences (B tokens a call): the projection from Q2_K
    wkv gives the bf16 path's kv and highway bit for bit, and the oracle's
    within tolerance."""
    from deepseek_v4_engram_hash_gb300 import _lib, runner
    cfg = configs.V41_DECODE_WKVQ2K.with_(batch=B)
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B)
    plain = _lib.layers_array([{k: v for k, v in d.items() if k != "wkv_q2k"} for d in eng.layer_data])
    hs2 = _lib.Hasher(eng.tables, B, cfg.max_seq)
    ref = G.hash_state(cfg, B)
    pos = 0
    for step in range(3):
        ids = torch.from_numpy(eng.ids_for(f"q{step}", 1)).cuda()
        h0 = synth.highway(cfg, pos * B + np.arange(B))
        d_q = torch.from_numpy(h0).cuda()
        d_b = torch.from_numpy(h0).cuda()
        eng.forward(ids, pos, d_q)                                   # Q2_K wkv
        kv_q = [_u16(eng.kv(B, l)) for l in range(cfg.n_layers)]
        _lib.engram_forward(hs2, plain, ids, 1, pos, d_b, cfg.eps, eng.ws, eng.ws_bytes)   # bf16 wkv
        assert E.engram_check() == 0
        assert torch.equal(d_q, d_b)
        want_ids = ref.forward(ids.cpu().numpy(), pos).reshape(B, cfg.n_layers, cfg.cols)
        h = h0
        outs = np.unique(np.concatenate([np.arange(0, cfg.N, 211), [cfg.N - 1]]))
        for l in range(cfg.n_layers):
            assert np.array_equal(kv_q[l], _u16(eng.kv(B, l)))
            x = G.x_of(cfg, l, want_ids)
            assert G.kv_rel_err(kv_q[l][:, outs], G.kv(cfg, l, x, outs)) <= G.KV_TOL
            h = G.gate(cfg, l, h, kv_q[l])
        assert np.abs(d_q.cpu().numpy() - h).max() <= G.H_TOL
        pos += 1

"""The decode step as a CUDA graph with a device-resident position (NEXT: the
pages' single-token graph capture and its eager-versus-graph comparison):
replays are bit-identical to eager calls at the same positions, the position
advances by itself, and a position past the cache is reported, not written."""
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


@pytest.mark.parametrize("cfg,B,T", [(configs.V41_DECODE, 1, 1), (configs.TINY, 2, 3), (configs.TINY, 1, 12)],
                         ids=["v41_T1", "tiny_B2_T3", "tiny_T12_gemm"])
def test_graph_replay_bit_identical_to_eager(E, cfg, B, T):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = cfg.with_(batch=B)
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * T)
    hs2 = E.Hasher(eng.tables, B, cfg.max_seq)
    ws2 = torch.empty_like(eng.ws)
    pos = cfg.prefix
    if pos:
        pre = torch.from_numpy(eng.ids_for("prefix", pos)).cuda()
        out = torch.empty((B, pos, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        E.engram_hash(eng.hasher, pre, pos, 0, out)
        E.engram_hash(hs2, pre, pos, 0, out)
    d_pos = torch.tensor([pos], dtype=torch.int64, device="cuda")
    d_ids = torch.zeros((B, T), dtype=torch.int32, device="cuda")
    d_hg = torch.zeros((B * T, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    graph = E.Graph(hs2, eng.layers, d_ids, T, d_pos, d_hg, cfg.eps, ws2, eng.ws_bytes)
    ref = G.hash_state(cfg, B)
    if cfg.prefix:
        ref.forward(eng.ids_for("prefix", pos), 0)
    for step in range(5):
        ids = eng.ids_for(f"g{step}", T)
        h0 = torch.from_numpy(synth.highway(cfg, np.arange(step * B * T, (step + 1) * B * T)))
        d_he = h0.cuda()
        eng.forward(ids, pos, d_he)                               # eager
        d_ids.copy_(torch.from_numpy(ids))
        d_hg.copy_(h0)
        graph.launch()                                            # replay
        assert E.engram_check() == 0
        assert torch.equal(d_he, d_hg), f"step {step}"
        assert torch.equal(eng.row_ids(B * T), (ws2[:B * T * cfg.n_layers * cfg.cols * 8]
                                                .view(torch.int64).view(B * T, cfg.n_layers, cfg.cols)))
        want = ref.forward(ids, pos).reshape(B * T, cfg.n_layers, cfg.cols)
        assert np.array_equal(eng.row_ids(B * T).cpu().numpy(), want)
        pos += T
    assert d_pos.item() == pos
    graph.close()


@pytest.mark.parametrize("T", [4, 16])      # hash inside the GEMV; hash inside the row gather
def test_device_position_past_the_cache_is_reported(E, T):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY.with_(prefix=0, T=T, decode_steps=0)
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=T)
    cache_len = cfg.max_seq
    d_pos = torch.tensor([cache_len - 2], dtype=torch.int64, device="cuda")     # 2 + T > remaining
    ids = torch.ones((1, T), dtype=torch.int32, device="cuda")
    d_h = torch.zeros((T, cfg.hc, cfg.dim), device="cuda")
    E.engram_forward_dpos(eng.hasher, eng.layers, ids, T, d_pos, d_h, cfg.eps, eng.ws, eng.ws_bytes)
    assert E.engram_check() == -4
    # a valid call afterwards still hashes exactly (the failed step wrote nothing)
    d_pos.fill_(0)
    E.engram_forward_dpos(eng.hasher, eng.layers, ids, T, d_pos, d_h, cfg.eps, eng.ws, eng.ws_bytes)
    assert E.engram_check() == 0
    ref = G.hash_state(cfg, 1)
    assert np.array_equal(eng.row_ids(T).cpu().numpy(),
                          ref.forward(ids.cpu().numpy(), 0).reshape(T, cfg.n_layers, cfg.cols))
    assert d_pos.item() == T


@pytest.mark.parametrize("cfg,B,T,K", [(configs.V41_DECODE, 1, 1, 8), (configs.TINY, 2, 3, 4),
                                       (configs.TINY, 1, 12, 3), (configs.V41_DECODE_WKVQ2K, 1, 1, 8),
                                       (configs.V41_DECODE_E8M0, 2, 1, 4)],
                         ids=["v41_T1_8steps", "tiny_B2_T3_4steps", "tiny_T12_gemm_3steps", "v41_q2k_wkv_8steps",
                              "v41_e8m0_B2_4steps"])
def test_multi_step_graph_bit_identical_to_eager(E, cfg, B, T, K):
    """K decode steps in one graph (each step hashing at *d_pos + k T, only the
    last step's gate advancing the position): every step's highway rows equal
    K eager calls at the same positions bit for bit, the last step's row ids
    too, and every step's ids equal the oracle's."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = cfg.with_(batch=B)
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * T)
    hs2 = E.Hasher(eng.tables, B, cfg.max_seq)
    ws2 = torch.empty_like(eng.ws)
    pos = cfg.prefix
    ref = G.hash_state(cfg, B)
    if pos:
        pre = eng.ids_for("prefix", pos)
        out = torch.empty((B, pos, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        E.engram_hash(eng.hasher, torch.from_numpy(pre).cuda(), pos, 0, out)
        E.engram_hash(hs2, torch.from_numpy(pre).cuda(), pos, 0, out)
        ref.forward(pre, 0)
    M = B * T
    d_pos = torch.tensor([pos], dtype=torch.int64, device="cuda")
    d_ids = torch.zeros((K, B, T), dtype=torch.int32, device="cuda")
    d_hg = torch.zeros((K, M, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    graph = E.Graph(hs2, eng.layers, d_ids, T, d_pos, d_hg, cfg.eps, ws2, eng.ws_bytes, steps=K)
    first = 0
    for replay in range(3):
        ids = np.stack([eng.ids_for(f"ms{replay}.{k}", T) for k in range(K)])           # [K, B, T]
        h0 = torch.from_numpy(synth.highway(cfg, np.arange(first, first + K * M))).view(K, M, cfg.hc, cfg.dim)
        d_he = [h0[k].clone().cuda() for k in range(K)]
        for k in range(K):                                                              # eager, back to back
            eng.forward(ids[k], pos + k * T, d_he[k])
        d_ids.copy_(torch.from_numpy(ids))
        d_hg.copy_(h0)
        graph.launch()
        assert E.engram_check() == 0
        for k in range(K):
            assert torch.equal(d_he[k].view(torch.int32), d_hg[k].view(torch.int32)), f"replay {replay} step {k}"
            want = ref.forward(ids[k], pos + k * T).reshape(M, cfg.n_layers, cfg.cols)
            if k == K - 1:
                got = ws2[:M * cfg.n_layers * cfg.cols * 8].view(torch.int64).view(M, cfg.n_layers, cfg.cols)
                assert np.array_equal(got.cpu().numpy(), want)
                assert np.array_equal(eng.row_ids(M).cpu().numpy(), want)
        pos += K * T
        first += K * M
    assert d_pos.item() == pos
    graph.close()


def test_multi_step_graph_past_the_cache_is_reported(E):
    """Steps of a multi-step graph that would run past the cache report
    ENGRAM_E_CAPACITY on the device and touch no cache entry."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY.with_(prefix=0, T=1, decode_steps=0)
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=1)
    K = 3
    d_pos = torch.tensor([cfg.max_seq - 2], dtype=torch.int64, device="cuda")    # steps 0, 1 fit; step 2 not
    d_ids = torch.ones((K, 1, 1), dtype=torch.int32, device="cuda")
    d_h = torch.zeros((K, 1, cfg.hc, cfg.dim), device="cuda")
    graph = E.Graph(eng.hasher, eng.layers, d_ids, 1, d_pos, d_h, cfg.eps, eng.ws, eng.ws_bytes, steps=K)
    graph.launch()
    assert E.engram_check() == -4
    graph.close()

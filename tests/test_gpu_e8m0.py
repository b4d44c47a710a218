"""One-byte e8m0 table scales (NEXT: `f32_to_e8m0_rne`'s byte storage): the
rows are bit-exact against the oracle for every e4m3 code and scale byte, equal
to the f32-scale rows, and the forward gives the same highway as with f32
scales and matches the oracle."""
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


@pytest.mark.parametrize("hd,blk", [(256, 32), (64, 16)])
def test_rows_e8m0_every_code_and_scale_byte(E, hd, blk):
    codes = np.array([b for b in range(256) if b & 0x7F != 0x7F], dtype=np.uint8)
    scale_bytes = np.array([0, 1, 100, 117, 120, 127, 130, 131, 140, 200, 254], dtype=np.uint8)
    R = scale_bytes.size
    table = np.resize(codes, (R, hd)).astype(np.uint8)
    sc = np.repeat(scale_bytes[:, None], hd // blk, axis=1)
    ids = np.arange(R, dtype=np.int64)[:, None]
    d_rows = torch.empty((R, hd), dtype=torch.bfloat16, device="cuda")
    E.engram_rows_fp8_e8m0(torch.from_numpy(table).cuda(), torch.from_numpy(sc).cuda(), R, hd, blk,
                           torch.from_numpy(ids).cuda(), R, 1, 1, d_rows)
    assert E.engram_check() == 0
    want = oracle.rows_fp8_e8m0(table, sc, hd, blk, ids.ravel())
    assert np.array_equal(_u16(d_rows), want)
    # the same values as f32 scales
    f32 = np.array([oracle.e8m0_to_f32(int(c)) for c in scale_bytes], dtype=np.float32)
    d2 = torch.empty_like(d_rows)
    E.engram_rows_fp8(torch.from_numpy(table).cuda(), torch.from_numpy(np.repeat(f32[:, None], hd // blk, 1)).cuda(),
                      R, hd, blk, torch.from_numpy(ids).cuda(), R, 1, 1, d2)
    assert torch.equal(d_rows.view(torch.int16), d2.view(torch.int16))


TINY_E8M0 = configs.TINY.with_(name="tiny_e8m0", fmt="fp8_e8m0", batch=2, T=9)


@pytest.mark.parametrize("cfg", [TINY_E8M0, configs.V41_DECODE_E8M0], ids=lambda c: c.name)
def test_forward_e8m0_matches_f32_scales_and_oracle(E, cfg):
    from deepseek_v4_engram_hash_gb300 import runner
    B = cfg.batch
    e8 = runner.EngramSetup(cfg, batch=B, max_tokens=B * cfg.T)
    f32 = runner.EngramSetup(cfg.with_(fmt="fp8"), batch=B, max_tokens=B * cfg.T)
    ref = G.hash_state(cfg, B)
    pos = 0
    for T in ((cfg.T, 1, 1) if cfg.T > 1 else (1, 1)):
        M = B * T
        ids = e8.ids_for(f"e8{pos}", T)
        h0 = synth.highway(cfg, np.arange(pos * B, pos * B + M))
        d1, d2 = torch.from_numpy(h0).cuda(), torch.from_numpy(h0).cuda()
        e8.forward(ids, pos, d1)
        f32.forward(ids, pos, d2)
        assert E.engram_check() == 0
        assert torch.equal(d1, d2)
        want_ids = ref.forward(ids, pos).reshape(M, cfg.n_layers, cfg.cols)
        assert np.array_equal(e8.row_ids(M).cpu().numpy(), want_ids)
        outs = np.unique(np.concatenate([np.arange(0, cfg.N, max(1, cfg.N // 150)), [cfg.N - 1]]))
        h = h0
        for l in range(cfg.n_layers):
            kv = _u16(e8.kv(M, l))
            assert G.kv_rel_err(kv[:, outs], G.kv(cfg, l, G.x_of(cfg, l, want_ids), outs)) <= G.KV_TOL
            h = G.gate(cfg, l, h, kv)
        assert np.abs(d1.cpu().numpy() - h).max() <= G.H_TOL
        pos += T

"""Tables in page-locked host memory, read by row in place by the kernels
(NEXT: host-resident tables larger than HBM, as the pages' page-locked,
device-visible arena): identical results to device-resident tables, and a
pointer the device cannot read is refused before any launch."""
import numpy as np
import pytest
import torch

from deepseek_v4_engram_hash_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import __graft_entry__
    __graft_entry__.build()
    from deepseek_v4_engram_hash_gb300 import _lib
    return _lib


@pytest.mark.parametrize("cfg", [configs.V41_DECODE.with_(prefix=64, T=1),
                                 configs.V41_Q2K.with_(T=40),
                                 configs.TINY.with_(fmt="fp8_e8m0", T=12)], ids=lambda c: c.name)
def test_host_tables_match_device_tables(E, cfg):
    from deepseek_v4_engram_hash_gb300 import runner
    dev = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    host = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T, tables_on_host=True)
    assert not host.layer_data[0]["table"].is_cuda and host.layer_data[0]["table"].is_pinned()
    pos = 0
    for T in (cfg.T, 1):
        ids = dev.ids_for(f"host{pos}", T)
        h0 = synth.highway(cfg, np.arange(pos, pos + T))
        d1, d2 = torch.from_numpy(h0).cuda(), torch.from_numpy(h0).cuda()
        dev.forward(ids, pos, d1)
        host.forward(ids, pos, d2)
        assert E.engram_check() == 0
        assert torch.equal(d1, d2)
        for l in range(cfg.n_layers):
            assert torch.equal(dev.kv(T, l).view(torch.int16), host.kv(T, l).view(torch.int16))
        pos += T


def test_unreadable_table_pointer_is_refused(E):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=4)
    pageable = np.zeros((eng.layer_data[0]["rows"], cfg.head_dim), dtype=np.uint8)   # not page-locked
    bad = [dict(d) for d in eng.layer_data]
    bad[0]["table"] = pageable.ctypes.data
    d_h = torch.zeros((4, cfg.hc, cfg.dim), device="cuda")
    with pytest.raises(E.EngramError) as e:
        E.engram_forward(eng.hasher, bad, torch.zeros((1, 4), dtype=torch.int32, device="cuda"), 4, 0, d_h,
                         cfg.eps, eng.ws, eng.ws_bytes)
    assert e.value.code == -1
    assert not d_h.any().item()

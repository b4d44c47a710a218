"""engram_forward_noalloc: the forward for callers that cannot allocate device
memory (a host that owns every allocation, a loop that must not enter the
allocator).  Its scratch is the library's fixed 4 MiB device array; it runs
the kernels of engram_forward with a caller-allocated workspace, so its results
must equal that forward's bit for bit.

This file is collected last so that a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
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


def _twin_hashers(E, eng, cfg, batch, prefix):
    """Two hashers on the same tables with the same look-back."""
    hs2 = E.Hasher(eng.tables, batch, cfg.max_seq)
    if prefix:
        pre = torch.from_numpy(eng.ids_for("prefix", prefix)).cuda()
        out = torch.empty((batch, prefix, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        E.engram_hash(eng.hasher, pre, prefix, 0, out)
        E.engram_hash(hs2, pre, prefix, 0, out)
    return hs2


@pytest.mark.parametrize("name,batch,T", [("v41_decode_T1", 1, 1), ("tiny", 2, 5)])
def test_noalloc_matches_forward_two_calls_in_a_row(E, name, batch, T):
    """Both entry points run the same kernels on the same inputs; only where
    the scratch lives differs, so the highway must agree bit for bit on each
    of two calls in a row (a stale or misplaced scratch region would show),
    and both hashers must carry the same look-back afterwards."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.CONFIGS[name]
    eng = runner.EngramSetup(cfg, batch=batch, max_tokens=batch * T)
    prefix = cfg.prefix
    hs2 = _twin_hashers(E, eng, cfg, batch, prefix)
    pos = prefix
    for call in range(2):
        ids = torch.from_numpy(eng.ids_for(f"noalloc{call}", T)).cuda()
        h0 = synth.highway(cfg, np.arange(pos * batch, pos * batch + batch * T))
        d_h_ref = torch.from_numpy(h0).cuda()
        d_h_new = torch.from_numpy(h0).cuda()
        E.engram_forward(eng.hasher, eng.layers, ids, T, pos, d_h_ref, cfg.eps, eng.ws, eng.ws_bytes)
        E.engram_forward_noalloc(hs2, eng.layers, ids, T, pos, d_h_new, cfg.eps)
        assert E.engram_check() == 0
        assert torch.equal(d_h_ref.view(torch.int32), d_h_new.view(torch.int32)), \
            f"call {call}: |dh| {(d_h_ref - d_h_new).abs().max().item()}"
        assert not torch.equal(d_h_new, torch.from_numpy(h0).cuda())      # the gate did run
        pos += T
    # the look-back each hasher carries: the next window's row ids agree
    nxt = torch.from_numpy(eng.ids_for("noalloc-next", 1)).cuda()
    a = torch.empty((batch, 1, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
    b = torch.empty_like(a)
    E.engram_hash(eng.hasher, nxt, 1, pos, a)
    E.engram_hash(hs2, nxt, 1, pos, b)
    assert E.engram_check() == 0
    assert torch.equal(a, b)


def test_noalloc_zero_tokens_is_a_no_op(E):
    """T = 0 is a valid no-op here as in engram_forward; a position past the
    hasher's capacity is refused the same way by both."""
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    d_h = torch.zeros((1, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    E.engram_forward_noalloc(eng.hasher, eng.layers, ids, 0, 0, d_h, cfg.eps)
    assert E.engram_check() == 0
    assert not d_h.any().item()
    for call in (lambda: E.engram_forward(eng.hasher, eng.layers, ids, 0, cfg.max_seq + 1, d_h, cfg.eps,
                                          eng.ws, eng.ws_bytes),
                 lambda: E.engram_forward_noalloc(eng.hasher, eng.layers, ids, 0, cfg.max_seq + 1, d_h, cfg.eps)):
        with pytest.raises(E.EngramError) as e:
            call()
        assert e.value.code == -4


def test_noalloc_refuses_more_than_its_scratch(E):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.V41_DECODE
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=1)
    T = 64                                             # ~6.8 MB of workspace at this shape
    ids = torch.zeros((1, T), dtype=torch.int32, device="cuda")
    d_h = torch.zeros((T, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    with pytest.raises(E.EngramError) as e:
        E.engram_forward_noalloc(eng.hasher, eng.layers, ids, T, 0, d_h, cfg.eps)
    assert e.value.code == -12
    assert "fixed scratch" in str(e.value)
    assert not d_h.any().item()                        # nothing ran

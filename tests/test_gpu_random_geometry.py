"""Seeded random geometries through the whole forward, every output checked
against the oracle: layers 1..4, n-grams 2..16, 1..8 heads, head_dim 16..256
with its scale blocks, dim a multiple of 8, hc 1..4, fp8 / e8m0 / Q2_K tables,
bf16 or (where K is a multiple of 256) Q2_K-quantised wkv, batch 1..5, and a call sequence that crosses the GEMV (<= 8 tokens) and the
GEMM paths.  Row ids must be bit-exact, kv within 2e-2, the highway within
1e-3 (stage-wise)."""
import numpy as np
import pytest

import oracle_glue as G
from deepseek_v4_engram_hash_gb300 import configs

from test_gpu_forward import _check_call, _h_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    import __graft_entry__
    __graft_entry__.build()
    from deepseek_v4_engram_hash_gb300 import _lib
    return _lib


def _geometry(seed: int):
    rng = np.random.default_rng(1000 + seed)
    while True:
        L = int(rng.integers(1, 5))
        ng = int(rng.integers(2, 17))
        H = int(rng.integers(1, 9))
        fmt = ["fp8", "fp8_e8m0", "q2k"][int(rng.integers(0, 3))]
        hd = 256 if fmt == "q2k" else int(rng.choice([16, 32, 48, 64, 128, 256]))
        blks = [b for b in (16, 32, 64) if hd % b == 0]
        blk = int(rng.choice(blks))
        C = (ng - 1) * H
        if (C * hd) % 64 or C * hd > 8192:
            continue
        dim = 8 * int(rng.integers(1, 33))
        hc = int(rng.integers(1, 5))
        B = int(rng.integers(1, 6))
        T = int(rng.integers(9, 40))
        # Q2_K-quantised wkv (the <= 8-token projection reads its blocks) where K allows it
        wkv_fmt = "q2k" if (C * hd) % 256 == 0 and C * hd <= 6144 and int(rng.integers(0, 2)) else "bf16"
        return configs.TINY.with_(
            name=f"rand{seed}", vocab=int(rng.integers(50, 3000)), n_compressed=int(rng.integers(20, 2000)),
            unmapped_5pct=bool(rng.integers(0, 2)), pad_token_id=int(rng.integers(0, 20)),
            layer_ids=tuple(range(L)), max_ngram=ng, n_heads=H, prime_target=int(rng.integers(50, 400)),
            head_dim=hd, scale_block=blk, dim=dim, hc=hc, fmt=fmt, batch=B, T=T, ids="uniform",
            seed=seed, wkv_fmt=wkv_fmt)


@pytest.mark.parametrize("seed", range(16))
def test_forward_random_geometry(E, seed):
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = _geometry(seed)
    B = cfg.batch
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=B * cfg.T)
    ref = G.hash_state(cfg, B)
    pos, first = 0, 0
    for T in (cfg.T, 1, 2, 1, 5):
        M = B * T
        ids = eng.ids_for(f"r{pos}", T)
        d_h = _h_device(cfg, first, M, True)
        _check_call(eng, ref, ids, pos, d_h, d_h.cpu().numpy(), np.arange(M), np.arange(cfg.N), first)
        pos += T
        first += M

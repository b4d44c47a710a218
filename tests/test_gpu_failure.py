"""Failure detection on the GPU without a fault: the bounded mbarrier wait
that every copy ring and GEMM of the library uses gives up after its limit,
raises ENGRAM_E_TIMEOUT in the device error word and returns; the device
stays usable afterwards."""
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


def test_bounded_wait_gives_up_and_reports(E):
    import time
    t0 = time.perf_counter()
    E.engram_selftest_wait_timeout(50000)          # 50 ms on a barrier nothing arrives at
    assert E.engram_check() == -10                 # ENGRAM_E_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert E.engram_check() == 0                   # read and cleared
    # the context is intact: a whole forward still checks against the oracle
    from deepseek_v4_engram_hash_gb300 import runner
    cfg = configs.TINY
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    ids = eng.ids_for("after-timeout", cfg.T)
    d_h = _h_device(cfg, 0, cfg.T, True)
    _check_call(eng, G.hash_state(cfg, 1), ids, 0, d_h, d_h.cpu().numpy(), np.arange(cfg.T),
                np.arange(cfg.N), 0)

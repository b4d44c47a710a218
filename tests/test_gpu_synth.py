"""The CUDA twin of the seeded input generator reproduces the numpy twin bit
for bit (so oracle inputs regenerated on the CPU equal what the GPU path
reads)."""
import numpy as np
import pytest
import torch

from deepseek_v4_engram_hash_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("cfg", [configs.TINY, configs.V41_DECODE])
def test_fp8_table(cfg):
    R, hd = 5000, cfg.head_dim
    codes = torch.empty((R, hd), dtype=torch.uint8, device="cuda")
    scales = torch.empty((R, hd // cfg.scale_block), dtype=torch.float32, device="cuda")
    synth.fill_table_fp8_cuda(cfg, 1, codes, scales)
    c, s = synth.table_fp8_rows(cfg, 1, np.arange(R))
    assert np.array_equal(codes.cpu().numpy(), c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_q2k_table():
    cfg = configs.V41_Q2K
    R = 3001
    blocks = torch.empty((R, 84), dtype=torch.uint8, device="cuda")
    synth.fill_table_q2k_cuda(cfg, 0, blocks)
    assert np.array_equal(blocks.cpu().numpy(), synth.table_q2k_rows(cfg, 0, np.arange(R)))


def test_wkv_and_highway():
    cfg = configs.TINY
    w = torch.empty((cfg.N, cfg.K), dtype=torch.bfloat16, device="cuda")
    synth.fill_wkv_cuda(cfg, 0, w)
    assert np.array_equal(w.view(torch.int16).cpu().numpy().view(np.uint16),
                          synth.wkv_rows(cfg, 0, np.arange(cfg.N)))
    h = torch.empty((40, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    synth.fill_highway_cuda(cfg, h, first_token=17)
    assert np.array_equal(h.cpu().numpy().view(np.uint32),
                          synth.highway(cfg, np.arange(17, 57)).view(np.uint32))


def test_normals_bit_identical_at_scale():
    """Four million N(0, 1) f32 values (the Box-Muller series evaluation in
    float64) agree bit for bit between the twins, tails included."""
    cfg = configs.TINY
    n_tok = 16384                                          # x hc 2 x dim 128 = 4.2 M values
    h = torch.empty((n_tok, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    synth.fill_highway_cuda(cfg, h, first_token=3)
    want = synth.highway(cfg, np.arange(3, 3 + n_tok))
    got = h.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.abs(want).max() > 4.5

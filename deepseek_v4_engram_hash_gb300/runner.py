"""Set-up of one synthetic engram workload on a device, and its forward call.

`EngramSetup` builds everything a workload needs in HBM -- hash tables
(libengram handles), per-layer tables (fp8 codes + scales, or Q2_K blocks),
wkv, q*k and the forward workspace -- from the seeded generator, then calls
the C ABI.  It holds no part of the method: every stage runs in libengram.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as E
from . import synth


class EngramSetup:
    def __init__(self, cfg, device="cuda", batch: int | None = None, max_tokens: int | None = None,
                 tables_on_host: bool = False, tiled_wkv: bool = True):
        """tables_on_host: keep the per-layer tables in page-locked host memory,
        read row by row in place by the kernels (tables larger than HBM).
        tiled_wkv: also hold each layer's wkv in the engram_tile_wkv layout,
        which the 1..8-token projection then reads."""
        self.cfg = cfg
        self.tables_on_host = tables_on_host
        self.device = torch.device(device)
        self.batch = int(batch or cfg.batch)
        t = synth.hash_tables(cfg)
        self.hash_np = t
        self.geom = E.make_geom(cfg.n_layers, cfg.max_ngram, cfg.n_heads, cfg.head_dim, cfg.dim,
                                cfg.hc, cfg.scale_block, cfg.vocab)
        with torch.cuda.device(self.device):
            self.tables = E.Tables(self.geom, t["token_map"], t["pad_token_id"], t["multipliers"],
                                   t["primes"], t["offsets"])
            self.hasher = E.Hasher(self.tables, self.batch, cfg.max_seq)
            self.layer_data = []
            for l in range(cfg.n_layers):
                R = t["rows_per_layer"][l]
                d = {"rows": R}
                fmt = cfg.fmt_of(l)
                if fmt in ("fp8", "fp8_e8m0"):
                    d["table"] = torch.empty((R, cfg.head_dim), dtype=torch.uint8, device=self.device)
                    d["scales"] = torch.empty((R, cfg.head_dim // cfg.scale_block), dtype=torch.float32,
                                              device=self.device)
                    synth.fill_table_fp8_cuda(cfg, l, d["table"], d["scales"])
                    d["fmt"] = E.ENGRAM_FMT_FP8
                    if fmt == "fp8_e8m0":
                        # the scales are exact powers of two: store their biased exponent bytes
                        d["scales"] = ((d["scales"].view(torch.int32) >> 23) & 0xFF).to(torch.uint8)
                        d["fmt"] = E.ENGRAM_FMT_FP8_E8M0
                else:
                    d["table"] = torch.empty((R, 84), dtype=torch.uint8, device=self.device)
                    d["scales"] = None
                    synth.fill_table_q2k_cuda(cfg, l, d["table"])
                    d["fmt"] = E.ENGRAM_FMT_Q2K
                d["wkv"] = torch.empty((cfg.N, cfg.K), dtype=torch.bfloat16, device=self.device)
                if cfg.wkv_fmt == "q2k":
                    # Q2_K blocks, and their bf16 dequantisation (by libengram) for multi-token calls
                    nb = cfg.N * (cfg.K // 256)
                    d["wkv_q2k"] = torch.empty((nb, 84), dtype=torch.uint8, device=self.device)
                    synth.fill_table_q2k_cuda(cfg, l, d["wkv_q2k"], tag="wkvq2k")
                    ids = torch.arange(nb, dtype=torch.int64, device=self.device)
                    E.engram_rows_q2k(d["wkv_q2k"], nb, ids, nb, 1, 1, d["wkv"])
                else:
                    synth.fill_wkv_cuda(cfg, l, d["wkv"])
                if tiled_wkv:
                    d["wkv_tiled"] = torch.empty(E.engram_tiled_wkv_bytes(cfg.N, cfg.K) // 2, dtype=torch.bfloat16,
                                                 device=self.device)
                    E.engram_tile_wkv(d["wkv"], cfg.N, cfg.K, d["wkv_tiled"])
                if tables_on_host:
                    for key in ("table", "scales"):
                        if d.get(key) is not None:
                            d[key] = d[key].cpu().pin_memory()      # device-visible, read in place
                    torch.cuda.empty_cache()
                q, k = synth.qk_weights(cfg, l)
                d["q"], d["k"] = q, k
                d["qk"] = torch.from_numpy(q * k).to(self.device)   # exact: bf16 x bf16 fits f32
                self.layer_data.append(d)
            self.layers = E.layers_array(self.layer_data)
            self.max_tokens = int(max_tokens or self.batch * cfg.T)
            self.ws_bytes = E.engram_workspace_bytes(self.geom, self.max_tokens)
            self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)
            torch.cuda.synchronize(self.device)

    def ids_for(self, tag: str, T: int) -> np.ndarray:
        """[batch, T] int32 token ids of sequence-specific streams."""
        return np.stack([synth.token_ids(self.cfg, f"{tag}.{b}", T) for b in range(self.batch)])

    def workspace_layout(self, tokens: int) -> list:
        return E.engram_workspace_layout(self.geom, tokens)

    def row_ids(self, tokens: int) -> torch.Tensor:
        off = self.workspace_layout(tokens)[0]
        n = tokens * self.cfg.n_layers * self.cfg.cols * 8
        return self.ws[off:off + n].view(torch.int64).view(tokens, self.cfg.n_layers, self.cfg.cols)

    def kv(self, tokens: int, layer: int) -> torch.Tensor:
        off = self.workspace_layout(tokens)[1 + layer]
        n = tokens * self.cfg.N * 2
        return self.ws[off:off + n].view(torch.bfloat16).view(tokens, self.cfg.N)

    def x(self, tokens: int, layer: int) -> torch.Tensor:
        """The gathered rows [tokens, K] bf16 of one layer (steps that run the
        projection as a GEMM keep them in the workspace)."""
        off = self.workspace_layout(tokens)[1 + self.cfg.n_layers + layer]
        n = tokens * self.cfg.K * 2
        return self.ws[off:off + n].view(torch.bfloat16).view(tokens, self.cfg.K)

    def forward(self, ids, start_pos: int, d_h, stream=None):
        """ids: [batch, T] int32 (numpy or CUDA tensor); d_h: [batch*T, hc, dim] f32 CUDA."""
        if isinstance(ids, np.ndarray):
            ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(self.device)
        T = ids.shape[1]
        E.engram_forward(self.hasher, self.layers, ids, T, start_pos, d_h, self.cfg.eps, self.ws,
                         self.ws_bytes, stream)
        return ids


def highway_host(cfg, tokens) -> np.ndarray:
    """Initial highway rows [len(tokens), hc, dim] from the seeded generator."""
    return synth.highway(cfg, tokens)

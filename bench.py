"""Benchmark of the engram forward on one GB300 (one JSON line on stdout).

Default workload: the DeepSeek-V4.1-Flash-shaped single-token decode step
(T = 1, both engram layers {1, 14}, hash included), after a 2048-token
prefilled look-back; each timed step is one decode position.  A second
measurement runs the T = 4096 prefill of the same geometry.

  python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--no-prefill]

Under torchrun (WORLD_SIZE > 1) each rank runs its own replica on its own
sequence (no data-path collective): value = all ranks' tokens / max rank time.
--impl reference times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "engram tokens/s at T=1 and T=4096 (1 GB300); % of HBM / bf16 TC roofline"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _src_hash(*names) -> str:
    h = hashlib.sha1()
    for n in names:
        h.update(open(os.path.join(ROOT, "deepseek_v4_engram_hash_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:12]


# GB300 datasheet rates (dense bf16 tensor, HBM3e), for the fractions beside
# the measured peaks.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0
# Tensor pipe active share of the prefill GEMM in its ncu capture
# (profiles/gemm_tc2_v41_prefill_T4096.md).
TENSOR_PIPE_ACTIVE = 0.947

# DRAM bytes (read + write) per launch from one ncu capture, keyed by the
# source hash of the kernel they were taken on; a changed kernel reports null.
NCU_TRAFFIC = {("gemv", "a87084ccbf2f"): 506553088}   # 503.45 MB read + 3.10 MB written
# Integer-pipe (ALU) warp instructions of one Q2_K-weight decode launch (T = 1,
# both layers) from one ncu capture (sm__inst_executed_pipe_alu.sum), keyed the same way.
NCU_ALU = {("gemv_q2k", "a87084ccbf2f"): 15024147}


def _sm_count() -> int:
    import torch
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def q2k_alu_roofline(r, clocks, hbm, sms):
    """The Q2_K-weight decode is bound by its integer pipe, not by HBM: its
    ALU instructions (ncu, one launch) over the launch's event-timed duration,
    against the pipe's peak -- 16 lanes a cycle in each of the 4 sub-partitions
    of every SM (one warp instruction every 2 cycles) at the SM clock sampled
    during the benchmark.  The HBM fraction of the same launch beside it."""
    mhz = (clocks or {}).get("sm_mhz") or 2070.0
    peak = sms * 4 * 0.5 * mhz * 1e6 / 1e12                       # T warp instructions / s
    gemv_s = r["stage_ms"]["gemv"] * 1e-3
    n = NCU_ALU.get(("gemv_q2k", _src_hash("gemv.cu", "common.cuh")))
    wbytes = r["step_algorithmic_bytes"]
    out = {"bound": "alu", "unit": "T integer-pipe warp instructions/s", "peak": peak,
           "peak_source": f"{sms} SMs x 4 sub-partitions x 0.5 warp instructions a cycle x {mhz:.0f} MHz",
           "kernel": "gemv_mma_kernel<1, 1> (fused hash, row gather, Q2_K decode and wkv GEMV, both layers)",
           "kernel_ms": r["stage_ms"]["gemv"],
           "hbm_frac": wbytes / gemv_s / 1e9 / hbm}
    if n is None:                       # the kernel changed since the count was taken
        out.update(achieved=None, frac=None, instructions=None)
    else:
        out.update(achieved=n / gemv_s / 1e12, frac=n / gemv_s / 1e12 / peak, instructions=n)
    return out


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.rows, self.proc = gpu, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------------
# Algorithmic work
# ---------------------------------------------------------------------------

def row_bytes(cfg) -> int:
    if cfg.fmt == "q2k":
        return 84
    return cfg.head_dim + (cfg.head_dim // cfg.scale_block) * (1 if cfg.fmt == "fp8_e8m0" else 4)


def gemv_bytes(cfg, M) -> int:
    """Fused gather + GEMV launch, all layers: wkv once, the rows, kv written."""
    L = cfg.n_layers
    return L * (cfg.N * cfg.K * 2 + M * cfg.cols * row_bytes(cfg) + M * cfg.N * 2)


def step_bytes(cfg, M) -> int:
    """Whole step (the roofline of the method): wkv once, rows, highway read +
    write, q*k, ids and token_map entries; intermediates excluded."""
    L = cfg.n_layers
    return (L * (cfg.N * cfg.K * 2 + M * cfg.cols * row_bytes(cfg) + cfg.hc * cfg.dim * 4)
            + M * cfg.hc * cfg.dim * 8 + M * 12)


def gemm_flops(cfg, M) -> float:
    return 2.0 * M * cfg.N * cfg.K * cfg.n_layers


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_decode(args, rank, world):
    import torch
    from deepseek_v4_engram_hash_gb300 import _lib as E
    from deepseek_v4_engram_hash_gb300 import configs, runner, synth

    cfg = configs.V41_DECODE.with_(seed=rank_seed(rank))
    cfg = cfg.with_(decode_steps=4 * args.steps + 4 * args.warmup)
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=1)
    n = args.warmup + 2 * args.steps
    pre = eng.ids_for("prefix", cfg.prefix)
    out = torch.empty((1, cfg.prefix, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
    E.engram_hash(eng.hasher, torch.from_numpy(pre).cuda(), cfg.prefix, 0, out)
    ids_all = torch.from_numpy(eng.ids_for("decode", n).reshape(n, 1, 1)).cuda()
    d_h = torch.from_numpy(synth.highway(cfg, [cfg.prefix])).cuda()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    E.prepare_events([e for row in ev for e in row])
    pos = cfg.prefix
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(torch.cuda.current_device()) as clk:
        time.sleep(0.3)                         # let the clock sampler start
        # the W warm-up steps run right before the timed ones, so that the timed
        # region starts from a GPU whose clocks are up
        for i in range(args.warmup):
            eng.forward(ids_all[i], pos, d_h)
            pos += 1
        _barrier(world)
        torch.cuda.synchronize()
        t0.record()
        for i in range(args.steps):
            eng.forward(ids_all[args.warmup + i], pos, d_h)
            pos += 1
        t1.record()
        torch.cuda.synchronize()
        _barrier(world)
        assert E.engram_check() == 0
        ms = t0.elapsed_time(t1) / args.steps
        # Same steps again with an event between the stages of every step (the
        # events stop the projection -> gate launch overlap, so this pass gives
        # each kernel's own duration; the step time above is taken without them).
        for i in range(args.steps):
            E.engram_set_profile_events(ev[i])
            eng.forward(ids_all[args.warmup + args.steps + i], pos, d_h)
            pos += 1
        torch.cuda.synchronize()
    E.engram_set_profile_events(None)
    assert E.engram_check() == 0
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in ev])  # ms
    gemv_ms = float(stage[:, 2].mean())

    # end to end through the host-buffer entry point: ids and highway copied in, highway out
    h_ids = torch.from_numpy(eng.ids_for("e2e", n).reshape(n, 1, 1)).pin_memory()
    h_h = torch.from_numpy(synth.highway(cfg, [0])).pin_memory()
    d_ids = torch.empty((1, 1), dtype=torch.int32, device="cuda")
    for i in range(args.warmup):
        E.engram_forward_host(eng.hasher, eng.layers, h_ids[i], d_ids, 1, pos, h_h, d_h, cfg.eps, eng.ws,
                              eng.ws_bytes)
        pos += 1
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        E.engram_forward_host(eng.hasher, eng.layers, h_ids[args.warmup + i], d_ids, 1, pos, h_h, d_h,
                              cfg.eps, eng.ws, eng.ws_bytes)
        pos += 1
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    return dict(cfg=cfg, eng=eng, ms=ms, gemv_ms=gemv_ms, stage_ms=stage.mean(0).tolist(), clocks=clk.summary(),
                e2e_ms=e2e_ms, h2d=4 + cfg.hc * cfg.dim * 4, d2h=cfg.hc * cfg.dim * 4)


def run_prefill(args):
    import torch
    from deepseek_v4_engram_hash_gb300 import _lib as E
    from deepseek_v4_engram_hash_gb300 import configs, runner, synth

    cfg = configs.V41_PREFILL
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=cfg.T)
    T = cfg.T
    d_h = torch.empty((T, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    synth.fill_highway_cuda(cfg, d_h)
    ids = torch.from_numpy(eng.ids_for("prefill", T)).cuda()
    steps, warm = args.prefill_steps, 3
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    E.prepare_events([e for row in ev for e in row])
    for _ in range(warm):
        eng.forward(ids, 0, d_h)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        E.engram_set_profile_events(ev[i])
        eng.forward(ids, 0, d_h)
    t1.record()
    torch.cuda.synchronize()
    E.engram_set_profile_events(None)
    assert E.engram_check() == 0
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in ev])
    ms = t0.elapsed_time(t1) / steps
    return dict(cfg=cfg, ms=ms, stage_ms=stage.mean(0).tolist())


def run_other(cfg, prefill_steps, decode_steps, warm=3, tables_on_host=False):
    """Prefill (batch x T tokens in one call) and, if asked, single-token decode
    steps of every sequence, for the Q2_K and large-table workloads."""
    import torch
    from deepseek_v4_engram_hash_gb300 import _lib as E
    from deepseek_v4_engram_hash_gb300 import runner, synth

    B, T = cfg.batch, cfg.T
    M = B * T
    eng = runner.EngramSetup(cfg, batch=B, max_tokens=M, tables_on_host=tables_on_host)
    d_h = torch.empty((M, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
    synth.fill_highway_cuda(cfg, d_h)
    ids = torch.from_numpy(eng.ids_for("prefill", T)).cuda()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(prefill_steps)]
    E.prepare_events([e for row in ev for e in row])
    for _ in range(warm):
        eng.forward(ids, 0, d_h)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(prefill_steps):
        eng.forward(ids, 0, d_h)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / prefill_steps
    for i in range(prefill_steps):
        E.engram_set_profile_events(ev[i])
        eng.forward(ids, 0, d_h)
    torch.cuda.synchronize()
    E.engram_set_profile_events(None)
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in ev]).mean(0)
    rows_rw = M * cfg.n_layers * cfg.cols * (row_bytes(cfg) + cfg.head_dim * 2)
    out = {"prefill": {"tokens_per_step": M, "ms_per_step": ms, "tokens_per_s": M / (ms * 1e-3),
                       "stage_ms": dict(zip(["hash", "gather", "gemm", "gate"], stage.tolist())),
                       "gemm_tflops": gemm_flops(cfg, M) / (stage[2] * 1e-3) / 1e12,
                       "gather_gbs": rows_rw / (stage[1] * 1e-3) / 1e9}}
    if decode_steps:
        n = warm + decode_steps
        dids = torch.from_numpy(eng.ids_for("decode", n).T.copy().reshape(n, B, 1)).cuda()
        dh = torch.empty((B, cfg.hc, cfg.dim), dtype=torch.float32, device="cuda")
        synth.fill_highway_cuda(cfg, dh, M)
        pos = T
        for i in range(warm):
            eng.forward(dids[i], pos, dh)
            pos += 1
        torch.cuda.synchronize()
        t0.record()
        for i in range(decode_steps):
            eng.forward(dids[warm + i], pos, dh)
            pos += 1
        t1.record()
        torch.cuda.synchronize()
        dms = t0.elapsed_time(t1) / decode_steps
        sb = step_bytes(cfg, B)
        out["decode"] = {"tokens_per_step": B, "ms_per_step": dms, "tokens_per_s": B / (dms * 1e-3),
                         "step_gbs": sb / (dms * 1e-3) / 1e9, "step_algorithmic_bytes": sb}
    assert E.engram_check() == 0
    del eng
    torch.cuda.empty_cache()
    return out


def run_decode_only(cfg, steps, warm=10, tables_on_host=False, batch=1, stage_steps=0):
    """Single-token decode steps of `batch` sequences after the configured look-back
    (and, with stage_steps, as many more with events between the stages)."""
    import torch
    from deepseek_v4_engram_hash_gb300 import _lib as E
    from deepseek_v4_engram_hash_gb300 import runner, synth

    cfg = cfg.with_(decode_steps=steps + warm + stage_steps + 8, batch=batch)
    eng = runner.EngramSetup(cfg, batch=batch, max_tokens=batch, tables_on_host=tables_on_host)
    if cfg.prefix:
        pre = torch.from_numpy(eng.ids_for("prefix", cfg.prefix)).cuda()
        out = torch.empty((batch, cfg.prefix, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
        E.engram_hash(eng.hasher, pre, cfg.prefix, 0, out)
    n = warm + steps + stage_steps
    ids = torch.from_numpy(eng.ids_for("decode", n).T.copy().reshape(n, batch, 1)).cuda()
    d_h = torch.from_numpy(synth.highway(cfg, np.arange(batch))).cuda()
    pos = cfg.prefix
    for i in range(warm):
        eng.forward(ids[i], pos, d_h)
        pos += 1
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        eng.forward(ids[warm + i], pos, d_h)
        pos += 1
    t1.record()
    torch.cuda.synchronize()
    assert E.engram_check() == 0
    ms = t0.elapsed_time(t1) / steps
    out = {}
    if stage_steps:
        # the projection's own duration: further steps with an event between the stages
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(stage_steps)]
        E.prepare_events([e for row in ev for e in row])
        for i in range(stage_steps):
            E.engram_set_profile_events(ev[i])
            eng.forward(ids[warm + steps + i], pos, d_h)
            pos += 1
        torch.cuda.synchronize()
        E.engram_set_profile_events(None)
        assert E.engram_check() == 0
        stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in ev])  # ms
        out["stage_ms"] = dict(zip(["hash", "gather", "gemv", "gate"], stage.mean(0).tolist()))
    wbytes = cfg.n_layers * cfg.N * (cfg.K // 256) * 84 if cfg.wkv_fmt == "q2k" else cfg.n_layers * cfg.N * cfg.K * 2
    sb = step_bytes(cfg, batch) - cfg.n_layers * cfg.N * cfg.K * 2 + wbytes
    del eng
    torch.cuda.empty_cache()
    return {"tokens_per_step": batch, "ms_per_step": ms, "tokens_per_s": batch / (ms * 1e-3),
            "step_algorithmic_bytes": sb, "step_gbs": sb / (ms * 1e-3) / 1e9, **out}


def run_decode_graph(cfg, steps, warm=32, per_graph=32):
    """Single-token decode steps replayed from one captured graph of
    `per_graph` consecutive steps; each replay's ids are copied into the
    graph's id buffer on the device first."""
    import torch
    from deepseek_v4_engram_hash_gb300 import _lib as E
    from deepseek_v4_engram_hash_gb300 import runner, synth

    steps = max(per_graph, steps // per_graph * per_graph)
    warm = max(per_graph, warm // per_graph * per_graph)
    cfg = cfg.with_(decode_steps=steps + warm + 8)
    eng = runner.EngramSetup(cfg, batch=1, max_tokens=1)
    pre = torch.from_numpy(eng.ids_for("prefix", cfg.prefix)).cuda()
    out = torch.empty((1, cfg.prefix, cfg.n_layers, cfg.cols), dtype=torch.int64, device="cuda")
    E.engram_hash(eng.hasher, pre, cfg.prefix, 0, out)
    n = warm + steps
    ids = torch.from_numpy(eng.ids_for("decode", n).reshape(n // per_graph, per_graph, 1, 1)).cuda()
    d_ids = torch.zeros((per_graph, 1, 1), dtype=torch.int32, device="cuda")
    d_pos = torch.tensor([cfg.prefix], dtype=torch.int64, device="cuda")
    d_h = torch.from_numpy(synth.highway(cfg, np.arange(per_graph))).cuda().view(per_graph, 1, cfg.hc, cfg.dim)
    graph = E.Graph(eng.hasher, eng.layers, d_ids, 1, d_pos, d_h, cfg.eps, eng.ws, eng.ws_bytes, steps=per_graph)
    for i in range(warm // per_graph):
        d_ids.copy_(ids[i])
        graph.launch()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps // per_graph):
        d_ids.copy_(ids[warm // per_graph + i])
        graph.launch()
    t1.record()
    torch.cuda.synchronize()
    assert E.engram_check() == 0
    ms = t0.elapsed_time(t1) / steps
    graph.close()
    del eng
    torch.cuda.empty_cache()
    return {"tokens_per_step": 1, "ms_per_step": ms, "tokens_per_s": 1.0 / (ms * 1e-3),
            "note": f"graphs of {per_graph} consecutive steps, one replay plus a device copy of its ids "
                    f"every {per_graph} steps"}


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world):
    """The largest per-rank value (step time) over all ranks; CPU tensors
    under gloo, device tensors under NCCL."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank_step: int, max_ms_per_step: float, world: int) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank_step / (max_ms_per_step * 1e-3)


def rank_seed(rank: int) -> int:
    """Each rank runs its own replica on its own synthetic sequence."""
    return rank


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_mods():
    import oracle
    from deepseek_v4_engram_hash_gb300 import configs, synth
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle_glue as G
    return oracle, configs, synth, G


def host_inputs(cfg, eng=None):
    """The oracle's stored inputs for fp8-table workloads: each layer's table
    (codes, scales) and wkv as host arrays -- copied from a set-up workload's
    device memory when given (the numpy twin generates the same bits), else
    generated on the host by the seeded generator.  Input preparation, untimed."""
    import torch
    oracle, configs, synth, G = _oracle_mods()
    tables, wkv = [], []
    rows = synth.hash_tables(cfg)["rows_per_layer"]
    for l in range(cfg.n_layers):
        if eng is not None:
            d = eng.layer_data[l]
            tables.append((d["table"].cpu().numpy(), d["scales"].cpu().numpy()))
            wkv.append(d["wkv"].view(torch.int16).cpu().numpy().view(np.uint16))
        else:
            tables.append(synth.table_fp8_rows(cfg, l, np.arange(rows[l])))
            wkv.append(synth.wkv_rows(cfg, l, np.arange(cfg.N)))
    return tables, wkv


def oracle_forward(cfg, st, ids, pos, h, wkv, qk, tables=None):
    """One oracle forward of ids [B, T] at position pos: the hash, every layer's
    row gather (from the stored tables, or -- without them -- the touched rows
    regenerated by the seeded generator and decoded by the oracle), the
    projection and the gate, in the oracle's order.  Returns the new highway."""
    oracle, configs, synth, G = _oracle_mods()
    B, T = ids.shape
    M = B * T
    rid = st.forward(ids, pos).reshape(M, cfg.n_layers, cfg.cols)
    for l in range(cfg.n_layers):
        if tables is not None:
            codes, scales = tables[l]
            x = oracle.rows_fp8(codes, scales, cfg.head_dim, cfg.scale_block, rid[:, l, :].ravel())
            x = x.reshape(M, cfg.K)
        else:
            x = G.x_of(cfg, l, rid)
        kv = oracle.linear_bf16(x, wkv[l])
        h = oracle.gate(h, kv, qk[l][0], qk[l][1], cfg.hc, cfg.dim, cfg.eps)
    return h


def oracle_decode_rate(budget_s: float, tables, wkv, steps=None, warm=0):
    """Oracle decode steps (T = 1) of the single-token workload on the host
    cores, each step whole (hash, row gather from the stored tables,
    projection, gate of both layers): for about budget_s seconds, or -- with
    `steps` -- `warm` untimed steps and then exactly `steps` timed ones.
    Returns (tokens/s, threads, timed steps)."""
    oracle, configs, synth, G = _oracle_mods()
    cfg = configs.V41_DECODE
    qk = [synth.qk_weights(cfg, l) for l in range(cfg.n_layers)]
    total = 4096 if steps is None else warm + steps
    st = G.hash_state(cfg, 1, cfg.prefix + total + 16)
    st.forward(synth.token_ids(cfg, "prefix.0", cfg.prefix)[None], 0)
    h = synth.highway(cfg, [cfg.prefix])
    ids = synth.token_ids(cfg, "decode.0", total)
    pos, n, t_used = cfg.prefix, 0, 0.0
    while n < total and (steps is not None or t_used < budget_s):
        t = time.perf_counter()
        h = oracle_forward(cfg, st, ids[n:n + 1][None], pos, h, wkv, qk, tables)
        if n >= warm:
            t_used += time.perf_counter() - t
        pos += 1
        n += 1
    timed = n - warm
    return timed / t_used, oracle.num_threads(), timed


def oracle_sample_rate(cfg, wkv, tables=None, prefill_tokens=0, decode_steps=0, batch=1):
    """The oracle on a bounded sample of a workload: the first prefill_tokens
    tokens of each sequence in one call, or (after hashing the workload's
    prefill, untimed) decode_steps single-token steps of every sequence.
    Returns (tokens/s over the timed calls, threads)."""
    oracle, configs, synth, G = _oracle_mods()
    qk = [synth.qk_weights(cfg, l) for l in range(cfg.n_layers)]
    st = G.hash_state(cfg, batch)
    ids = np.stack([synth.token_ids(cfg, f"prefill.{b}", cfg.T) for b in range(batch)])
    if prefill_tokens:
        h = synth.highway(cfg, np.arange(batch * prefill_tokens))
        t = time.perf_counter()
        oracle_forward(cfg, st, ids[:, :prefill_tokens], 0, h, wkv, qk, tables)
        return batch * prefill_tokens / (time.perf_counter() - t), oracle.num_threads()
    st.forward(ids, 0)
    dec = np.stack([synth.token_ids(cfg, f"decode.{b}", decode_steps) for b in range(batch)])
    h = synth.highway(cfg, np.arange(batch))
    t_used = 0.0
    for k in range(decode_steps):
        t = time.perf_counter()
        h = oracle_forward(cfg, st, dec[:, k:k + 1], cfg.T + k, h, wkv, qk, tables)
        t_used += time.perf_counter() - t
    return batch * decode_steps / t_used, oracle.num_threads()


def cpu_baselines(eng):
    """The oracle as it stands on the host cores, on bounded samples (about
    20 s of CPU work in all): the single-token step (all threads, then one),
    a 256-token sample of the 4096-token prefill, a 64-token sample of the
    Q2_K-table prefill and decode steps of the large-table workload."""
    oracle, configs, synth, G = _oracle_mods()
    cfg = configs.V41_DECODE
    tables, wkv = host_inputs(cfg, eng)
    rate, threads, n = oracle_decode_rate(8.0, tables, wkv)
    oracle.set_num_threads(1)
    rate1, _, n1 = oracle_decode_rate(4.0, tables, wkv)
    oracle.set_num_threads(threads)
    prate, _ = oracle_sample_rate(configs.V41_PREFILL, wkv, tables, prefill_tokens=256)
    qrate, _ = oracle_sample_rate(configs.V41_Q2K, wkv, None, prefill_tokens=64)
    srate, _ = oracle_sample_rate(configs.STRESS, wkv, None, decode_steps=3, batch=configs.STRESS.batch)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} whole V4.1 decode steps (T=1) of the plain C oracle: hash, row gather from the "
                      f"stored fp8 tables, projection and gate of both layers",
            "single_thread": {"value": rate1, "unit": "tokens/s", "cores": 1, "steps": n1},
            "prefill": {"value": prate, "unit": "tokens/s", "cores": threads,
                        "sample": "the first 256 tokens of the 4096-token prefill in one whole call (hash, "
                                  "row gather from the stored tables, projection, gate); every stage costs "
                                  "the same per token, so this rate extrapolates linearly to the full prefill "
                                  "(4096 tokens: about %.0f s)" % (4096 / prate)},
            "v41_q2k_T512": {"value": qrate, "unit": "tokens/s", "cores": threads,
                             "sample": "the first 64 tokens of the 512-token Q2_K-table prefill in one whole "
                                       "call; the touched Q2_K rows regenerated by the seeded generator and "
                                       "decoded by the oracle (no stored table); extrapolates linearly"},
            "large_table_stress": {"value": srate, "unit": "tokens/s", "cores": threads,
                                   "sample": "3 single-token decode steps of all 8 sequences after the "
                                             "1536-token prefill (hashed untimed); touched rows regenerated "
                                             "by the seeded generator"}}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    # W untimed and K timed whole oracle decode steps of the single-token
    # workload (about 21 ms a step on the 16 host cores); the stored tables
    # and wkv are generated on the host first (input preparation, untimed)
    oracle, configs, synth, G = _oracle_mods()
    tables, wkv = host_inputs(configs.V41_DECODE)
    rate, threads, n = oracle_decode_rate(0.0, tables, wkv, steps=args.steps, warm=args.warmup)
    line = {"metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 / rate, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "v41_decode_T1", "tokens_per_step": 1},
            "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n} timed whole decode steps (after {args.warmup} untimed) of the plain "
                                       f"C oracle: hash, row gather from the stored fp8 tables, projection and "
                                       f"gate of both layers"},
            "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill-steps", type=int, default=5)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the Q2_K and large-table lines")
    ap.add_argument("--only", choices=["decode", "prefill", "wkvq2k", "wkvq2k8", "decode8", "q2k512", "stress"],
                    default=None,
                    help="run one workload only (for profiling); prints its own JSON line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    # one build a node: local rank 0 compiles (when anything is stale), the
    # others wait for it and then only load the libraries
    if world > 1 and local != 0:
        dist.barrier()
    __graft_entry__.build()
    if world > 1 and local == 0:
        dist.barrier()

    hbm, bf16_burst, bf16_sust, peak_src = _peaks()
    if args.only == "decode8":
        from deepseek_v4_engram_hash_gb300 import configs
        print(json.dumps(run_decode_only(configs.V41_DECODE, args.steps, batch=8)), flush=True)
        return
    if args.only in ("wkvq2k", "wkvq2k8"):
        from deepseek_v4_engram_hash_gb300 import configs
        r = run_decode_only(configs.V41_DECODE_WKVQ2K, args.steps, batch=8 if args.only == "wkvq2k8" else 1,
                            stage_steps=min(args.steps, 100))
        if args.only == "wkvq2k":
            r["roofline"] = q2k_alu_roofline(r, None, hbm, _sm_count())
        print(json.dumps(r), flush=True)
        return
    if args.only in ("q2k512", "stress"):
        from deepseek_v4_engram_hash_gb300 import configs
        c = configs.V41_Q2K if args.only == "q2k512" else configs.STRESS
        r = run_other(c, args.prefill_steps, 0)
        r["workload"] = c.name
        print(json.dumps(r), flush=True)
        return
    if args.only == "prefill":
        p = run_prefill(args)
        print(json.dumps({"workload": p["cfg"].name, "ms_per_step": p["ms"], "stage_ms": p["stage_ms"],
                          "tokens_per_s": p["cfg"].T / (p["ms"] * 1e-3)}), flush=True)
        return
    d = run_decode(args, rank, world)
    cfg, M = d["cfg"], 1
    ms = _max_over_ranks(d["ms"], world)
    e2e_ms = _max_over_ranks(d["e2e_ms"], world)
    gemv_gbs = gemv_bytes(cfg, M) / (d["gemv_ms"] * 1e-3) / 1e9
    step_gbs = step_bytes(cfg, M) / (ms * 1e-3) / 1e9
    key = _src_hash("gemv.cu", "common.cuh")
    traffic = NCU_TRAFFIC.get(("gemv", key))

    pre = None
    if not args.no_prefill and rank == 0 and args.only is None:
        p = run_prefill(args)
        pc = p["cfg"]
        gemm_ms = p["stage_ms"][2]
        pre = {"workload": pc.name, "tokens_per_step": pc.T, "ms_per_step": p["ms"],
               "value": pc.T / (p["ms"] * 1e-3), "unit": "tokens/s",
               "stage_ms": dict(zip(["hash", "gather", "gemm", "gate"], p["stage_ms"])),
               "stage_note": "fp8 tables hash inside the row-gather launch: 'hash' is the empty interval "
                             "before it and 'gather' covers hash and gather of both layers",
               "roofline": {"bound": "tensor", "achieved": gemm_flops(pc, pc.T) / (gemm_ms * 1e-3) / 1e12,
                            "peak": bf16_burst, "unit": "TFLOP/s",
                            "frac": gemm_flops(pc, pc.T) / (gemm_ms * 1e-3) / 1e12 / bf16_burst,
                            "peak_source": f"{peak_src} bf16 burst (GEMM timed in short back-to-back steps)",
                            "peak_nominal": NOMINAL_BF16_TFLOPS,
                            "frac_of_nominal": gemm_flops(pc, pc.T) / (gemm_ms * 1e-3) / 1e12 / NOMINAL_BF16_TFLOPS,
                            "tensor_pipe_active": TENSOR_PIPE_ACTIVE,
                            "note": "the measured peak is cuBLAS bf16 at 8192^3, so a kernel can read a little "
                                    "above 1.0 of it; frac_of_nominal is against the dense bf16 datasheet rate",
                            "kernel": "gemm_tc2_kernel (tcgen05 on CTA pairs, both layers in one launch)"}}

    others = None
    if rank == 0 and args.only is None and not args.no_others:
        from deepseek_v4_engram_hash_gb300 import configs
        others = {}
        for name, c, ps, ds in (("v41_q2k_T512", configs.V41_Q2K, 10, 0),
                                ("large_table_stress", configs.STRESS, 3, 200)):
            r = run_other(c, ps, ds)
            r["workload"] = name
            others[name] = r
        r = run_decode_only(configs.V41_DECODE_E8M0, 2000)
        r["workload"] = configs.V41_DECODE_E8M0.name
        r["note"] = "one-byte e8m0 table scales (264 B a row instead of 288 B)"
        others[configs.V41_DECODE_E8M0.name] = r
        r = run_decode_graph(configs.V41_DECODE, 2000)
        r1 = run_decode_graph(configs.V41_DECODE, 2000, per_graph=1)
        r["single_step_graph"] = {"ms_per_step": r1["ms_per_step"], "tokens_per_s": r1["tokens_per_s"]}
        r["workload"] = "v41_decode_T1_graph"
        others["v41_decode_T1_graph"] = r
        r = run_decode_only(configs.V41_DECODE, 2000, tables_on_host=True)
        r["workload"] = "v41_decode_T1_host_tables"
        r["note"] = "tables in page-locked host memory, rows read in place over the CPU-GPU link"
        others["v41_decode_T1_host_tables"] = r
        r = run_other(configs.V41_PREFILL, 5, 0, tables_on_host=True)
        r["workload"] = "v41_prefill_T4096_host_tables"
        others["v41_prefill_T4096_host_tables"] = r
        r = run_decode_only(configs.V41_DECODE_WKVQ2K, 2000, stage_steps=200)
        r["workload"] = configs.V41_DECODE_WKVQ2K.name
        r["note"] = "projection read from Q2_K-quantised wkv (82.6 MB a step instead of 503.3 MB)"
        r["roofline"] = q2k_alu_roofline(r, d["clocks"], hbm, _sm_count())
        others[configs.V41_DECODE_WKVQ2K.name] = r
        r = run_decode_only(configs.V41_DECODE_WKVQ2K, 1000, batch=8)
        r["workload"] = "v41_decode_B8_wkv_q2k"
        r["note"] = "8 sequences x 1 token a step, projection from Q2_K-quantised wkv"
        others["v41_decode_B8_wkv_q2k"] = r

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and args.only is None:
        cpu = cpu_baselines(d["eng"])

    if rank == 0:
        line = {
            "metric": METRIC, "value": whole_job_rate(M, ms, world), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "v41_decode_T1: V4.1-Flash engram decode step, T=1 per sequence, "
                                   "layers {1,14}, 2048-token look-back, fp8 tables, dim 4096, hc 4",
                       "tokens_per_step": M * world, "l2": "inputs larger than L2 (wkv 503 MB read per step)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": {"bound": "hbm", "achieved": gemv_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gemv_gbs / hbm, "traffic": traffic,
                         "kernel": "gemv_mma_kernel<1, 0> (fused hash, row gather and wkv GEMV, both layers)",
                         "algorithmic_bytes": gemv_bytes(cfg, M), "peak_source": f"{peak_src} hbm_gbs",
                         "peak_nominal": NOMINAL_HBM_GBS, "frac_of_nominal": gemv_gbs / NOMINAL_HBM_GBS},
            "step_roofline": {"achieved": step_gbs, "frac": step_gbs / hbm, "algorithmic_bytes": step_bytes(cfg, M)},
            "stage_ms": dict(zip(["hash", "gather", "gemv", "gate"], d["stage_ms"])),
            "stage_note": "per-kernel times from a second pass with events between the stages; "
                          "the hash and the gather run inside the gemv launch",
            "gpu_launches": 2 * args.steps,
            "clocks": d["clocks"],
            "e2e": {"value": whole_job_rate(M, e2e_ms, world), "unit": "tokens/s",
                    "h2d_bytes_per_step": d["h2d"], "d2h_bytes_per_step": d["d2h"]},
            "cpu_baseline": cpu,
            "prefill": pre,
            "other_workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

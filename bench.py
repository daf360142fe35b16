#!/usr/bin/env python
"""Benchmark of the DDTree verify step on GB300.

One step = the whole hot path over one batch: ancestor masks, tree-verify
attention over the paged committed prefix, per-node vocab argmax, greedy
acceptance and the commit copy, all through the C-ABI library.  Default
workload: one sequence with 131,072 committed tokens, 24 query / 4 KV heads,
head dim 256, bf16, a 22-node random tree (branching <= 4), 151,936-entry
vocabulary, 64-token pages placed by a random permutation.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is algorithmic bytes of the step
(committed K/V, queries, tree K/V, outputs, page table, logits, commit copy)
per second; under torchrun every rank runs its own sequence (weak scaling)
and the time is the maximum over ranks.  ``--impl reference`` times the fp64
CPU oracle on the host cores on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-verify HBM GB/s (% of peak) and verify steps/s, budget 22 @128K ctx"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
KERNELS_PER_STEP = 2  # lucetree_verify_step: the prefix attention kernel, then the finish kernel


# ----------------------------------------------------------------------------- bytes

def attn_bytes(cfg: W.VerifyConfig) -> int:
    """Algorithmic bytes of one lucetree_verify_attn call."""
    s = 2
    kv = sum(cfg.ctx) * cfg.Hkv * cfg.D * 2 * s
    q = cfg.B * cfg.N * cfg.Hq * cfg.D * s
    out = cfg.B * cfg.N * cfg.Hq * (cfg.D + 1) * 4
    tree = cfg.B * cfg.N * cfg.Hkv * cfg.D * 2 * s
    pt = sum(-(-L // 64) for L in cfg.ctx) * 4
    anc = cfg.B * cfg.N * 8
    return kv + q + out + tree + pt + anc


def step_bytes(cfg: W.VerifyConfig, accepted_total: int) -> int:
    logits = cfg.B * (cfg.N + 1) * cfg.vocab * 4
    commit = 2 * accepted_total * cfg.Hkv * cfg.D * 2 * 2
    small = cfg.B * cfg.N * 4 * 6
    return attn_bytes(cfg) + logits + commit + small


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha(prefix: str = "attn_prefix") -> str:
    """Hash of one kernel's sources (files starting with `prefix`) and the
    shared device headers."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_tree_ddtree_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.startswith(prefix) or fn in ("internal.cuh", "tc_ptx.cuh"):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def prefix_kernel_sha() -> str:
    return kernel_sha("attn_prefix")


def profiled_traffic(summary: str = "attn_prefix_verify-128k-b22.md", prefix: str = "attn_prefix"):
    """dram bytes per launch of a kernel from its committed ncu summary, or None
    when the kernel's sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", summary)
    try:
        txt = open(p).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s*\(source sha\s*([0-9a-f]+)\)", txt)
    if not m or m.group(2) != kernel_sha(prefix):
        return None
    return int(m.group(1))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str | None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------- oracle timing

def oracle_step_sample(inp, cfg, rows, threads):
    """One bounded oracle step: sampled attention rows, then argmax, acceptance
    and commit of the whole batch.  Returns (attention seconds, rest seconds)."""
    import oracle
    did = oracle.BF16 if cfg.dtype == W.BF16 else oracle.F16
    t0 = time.perf_counter()
    oracle.verify_attn(inp, did, rows=rows, threads=threads)
    t1 = time.perf_counter()
    am = oracle.argmax(inp["logits"])
    acc, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    oracle.commit(inp, acc, alen, inplace=True)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def cpu_baseline(inp, cfg, acc_total, budget_s=15.0):
    threads = os.cpu_count() or 1
    total_rows = cfg.B * cfg.N * cfg.Hq
    # calibrate on one row per thread, then size the sample to the budget
    rows = W.sample_rows(cfg, threads, seed=7)
    ta, tr = oracle_step_sample(inp, cfg, rows, threads)
    per_row = ta / len(rows)
    n = int(min(total_rows, max(len(rows), (budget_s - ta) / max(per_row, 1e-9))))
    rows = W.sample_rows(cfg, n, seed=8)
    ta, tr = oracle_step_sample(inp, cfg, rows, threads)
    step_s = ta * total_rows / len(rows) + tr
    return {"value": step_bytes(cfg, acc_total) / step_s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {total_rows} attention rows (fp64 C, {threads} threads) scaled to the "
                      f"full step, plus argmax/accept/commit of the whole batch",
            "ms_per_step": step_s * 1e3}


def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = W.generate(cfg, seed=0)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    total_rows = cfg.B * cfg.N * cfg.Hq
    am = oracle.argmax(inp["logits"])
    _, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    acc_total = int(alen.sum())
    # size each step's row sample so warmup + steps stay within ~150 s
    rows = W.sample_rows(cfg, threads, seed=7)
    ta, _ = oracle_step_sample(inp, cfg, rows, threads)
    per_row = ta / len(rows)
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(total_rows, per_step_budget / max(per_row, 1e-9))))
    rows = W.sample_rows(cfg, n, seed=9)
    for _ in range(args.warmup):
        oracle_step_sample(inp, cfg, rows, threads)
    equiv = []
    for _ in range(args.steps):
        ta, tr = oracle_step_sample(inp, cfg, rows, threads)
        equiv.append(ta * total_rows / len(rows) + tr)
    step_s = float(np.mean(equiv))
    value = step_bytes(cfg, acc_total) / step_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_dict(cfg),
        "verify_steps_per_s": 1.0 / step_s,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(rows)} of {total_rows} attention rows per step (fp64 C, {threads} "
                                   f"threads) scaled to the full step, plus argmax/accept/commit of the batch"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(cfg):
    return {"workload": f"{cfg.name}: {cfg.B} seq x {','.join(str(x) for x in cfg.ctx)} committed tokens, "
                        f"{cfg.Hq}q/{cfg.Hkv}kv heads, D={cfg.D}, {cfg.dtype}, {cfg.N}-node {cfg.tree} tree, "
                        f"vocab {cfg.vocab}, 64-token pages ({cfg.paged})",
            "global_batch": cfg.B, "seq_len": cfg.ctx[0], "tree_budget": cfg.N, "heads_q": cfg.Hq,
            "heads_kv": cfg.Hkv, "head_dim": cfg.D, "vocab": cfg.vocab, "page_size": 64,
            "parallelism": "replicas (one sequence per rank)",
            "l2": (f"inputs larger than L2: committed K/V {cfg.kv_bytes() >> 20} MiB > 129 MB L2"
                   if cfg.kv_bytes() > L2_BYTES else
                   f"inputs smaller than L2 (committed K/V {cfg.kv_bytes() / 2**20:g} MiB, L2 not flushed "
                   f"between steps): an L2-resident timing, not a contract figure")}


# ----------------------------------------------------------------------------- timing helpers

def ms_stats(ms) -> dict:
    """Mean, median and 90th percentile of per-iteration device times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"mean": float(a.mean()), "p50": float(np.percentile(a, 50)), "p90": float(np.percentile(a, 90)),
            "n": int(a.size)}


def issue_step(step, dd, stream):
    """One whole verify step through the C-ABI on `stream`: one call of
    lucetree_verify_step (ancestor masks, tree attention, argmax, acceptance,
    commit)."""
    step.run(dd["q"], dd["k_pool"], dd["v_pool"], dd["page_table"], dd["ctx_len"], dd["k_tree"], dd["v_tree"],
             dd["parent"], dd["draft"], dd["logits"], stream=stream)


def time_attention(LT, step, dd, stream, n, flush=None, group=10):
    """n lucetree_verify_attn calls (the split-K prefix kernel and the merge
    launch) on the step's inputs; returns ms per call, one value per timed
    span.  Without `flush` the calls run back to back, as in a loop of steps,
    in spans of `group` calls between CUDA events on `stream` (an event between
    two calls would stop the next call's programmatic launch from overlapping
    this one's tail).  With `flush` (a buffer written between calls to empty
    L2) every call is bracketed by its own events, the write outside them."""
    import torch
    LT.lucetree_build_anc_mask(dd["parent"], step.anc, step.status, stream)

    def call():
        LT.lucetree_verify_attn(dd["q"], dd["k_pool"], dd["v_pool"], dd["page_table"], dd["ctx_len"],
                                dd["k_tree"], dd["v_tree"], step.anc, step.out, step.status, step.ws_attn,
                                lse=step.lse, stream=stream)

    span = 1 if flush is not None else max(1, min(group, n))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(max(1, n // span))]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            if flush is not None:
                flush.fill_(1)
            e0.record(stream)
            for _ in range(span):
                call()
            e1.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / span for a, b in ev]


def time_spans(call, stream, dev, n, group=10):
    """ms per call of `call` on `stream`, one value per span of `group` calls
    run back to back between CUDA events (as the headline call is timed: an
    event between two calls would stop the next call's programmatic launch
    from overlapping this one's tail), after five untimed calls."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(5):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(max(1, n // group))]
        torch.cuda.synchronize(dev)
        for e0, e1 in ev:
            e0.record(stream)
            for _ in range(group):
                call()
            e1.record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) / group for a, b in ev]


def attn_flops(cfg: W.VerifyConfig) -> int:
    """Algorithmic flops of one attention call: Q.K^T and P.V over the
    committed prefix, 4 * N * Hq * L * D per sequence."""
    return sum(4 * cfg.N * cfg.Hq * L * cfg.D for L in cfg.ctx)


def peak_tensor_sustained():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return 1700.0, "fallback (sustained)"


def device_inputs(cfg: W.VerifyConfig, dev, seed: int, pool_cfg: W.VerifyConfig | None = None, pools: bool = True):
    """A verify workload on the device: the tree, draft tokens and planted
    logits from the seeded generator, the committed K/V pools and queries as
    seeded N(0, 1) draws made on the device (the same distribution the
    generator uses; the attention time does not depend on the values).
    pool_cfg: the configuration whose page geometry the pools follow (a
    larger budget reserves more pages), by default cfg itself."""
    import torch
    pc = pool_cfg or cfg
    meta = W.generate(cfg, seed=seed, with_pools=False)
    geo = W.generate(pc, seed=seed, with_pools=False, with_logits=False) if pool_cfg is not None else meta
    tdt = torch.bfloat16 if cfg.dtype == W.BF16 else torch.float16
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + seed)
    num_pages = sum(W.pages_needed(L, pc.N) for L in pc.ctx) + pc.spare_pages

    def normal(shape):
        t = torch.empty(shape, dtype=tdt, device=dev)
        flat = t.view(-1)
        step = 1 << 26
        for i in range(0, flat.numel(), step):
            j = min(flat.numel(), i + step)
            flat[i:j] = torch.randn(j - i, device=dev, generator=g).to(tdt)
        return t

    d = dict(q=normal((cfg.B, cfg.N, cfg.Hq, cfg.D)), k_tree=normal((cfg.B, cfg.N, cfg.Hkv, cfg.D)),
             v_tree=normal((cfg.B, cfg.N, cfg.Hkv, cfg.D)),
             page_table=torch.from_numpy(geo["page_table"]).to(dev),
             ctx_len=torch.from_numpy(meta["ctx_len"]).to(dev), parent=torch.from_numpy(meta["parent"]).to(dev),
             draft=torch.from_numpy(meta["draft"]).to(dev), logits=torch.from_numpy(meta["logits"]).to(dev))
    if pools:
        d["k_pool"] = normal((num_pages, cfg.Hkv, W.PAGE, cfg.D))
        d["v_pool"] = normal((num_pages, cfg.Hkv, W.PAGE, cfg.D))
    return d


def measure_configs(args, dev, stream, rank):
    """The other workloads, each timed as whole verify steps through the C-ABI
    with CUDA events around the step and around its attention call: the
    27B-class 32K / budget 22 (its 128 MiB of K/V about fills L2, so L2 is
    flushed between steps here, for every workload), 128K / budget 40,
    256K on permuted pages / budget 22 with the commit into reserved pages,
    and the 4-sequence sweep {4K, 32K, 128K, 256K} at budgets 1 / 22 / 40 / 64
    as chains and random trees (planted match 0.7).  Budget 64 is reported
    against the sustained bf16 tensor peak as well (384 flop per K/V byte)."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    peak, peak_kind = peak_hbm()
    tpeak, tpeak_kind = peak_tensor_sustained()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MiB > L2
    n = max(5, min(20, args.steps // 100 or 5))
    todo = [W.GQA27B_32K, W.LONG_128K, W.PAGED_256K]
    sweep = [c for c in W.sweep_points() if c.p_plant == 0.7 and c.N in (1, 22, 40, 64)]
    pool64 = [c for c in W.sweep_points() if c.N == 64 and c.tree == "random" and c.p_plant == 0.7][0]
    out = {}
    shared = None
    for cfg in todo + sweep:
        is_sweep = cfg in sweep
        if is_sweep:
            if shared is None:
                shared = device_inputs(pool64, dev, seed=rank, pool_cfg=pool64)
            meta = device_inputs(cfg, dev, seed=rank, pool_cfg=pool64, pools=False) if cfg is not pool64 else shared
            d = dict(meta, k_pool=shared["k_pool"], v_pool=shared["v_pool"])
            del meta
        else:
            d = device_inputs(cfg, dev, seed=rank)
        step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab, device=dev)
        ctx0 = d["ctx_len"].clone()
        # the inputs were drawn (and the step's counters zeroed) on the current
        # stream: the side stream must not start before they are complete
        stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(stream):
            for _ in range(3):
                issue_step(step, d, stream)
            stream.synchronize()
            ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(n)]
            for e in ev:
                flush.fill_(1)
                e[0].record(stream)
                issue_step(step, d, stream)
                e[1].record(stream)
        torch.cuda.synchronize(dev)
        assert torch.equal(d["ctx_len"], ctx0)  # the step writes ctx_out, the committed length stays
        stp = ms_stats([a.elapsed_time(b) for a, b in ev])
        attn = ms_stats(time_attention(LT, step, d, stream, n, flush))
        ab = attn_bytes(cfg)
        rec = {"workload": config_dict(cfg)["workload"], "attn_ms": attn, "step_ms": stp,
               "kv_bytes": cfg.kv_bytes(), "attn_bytes": ab,
               "attn_GBps": ab / (attn["p50"] * 1e-3) / 1e9,
               "frac_of_hbm_peak": ab / (attn["p50"] * 1e-3) / 1e9 / peak,
               "verify_steps_per_s": 1e3 / stp["p50"], "accepted": int(step.acc_len.sum().item()),
               "device_status": int(step.status.item()),
               "l2": "a 256 MiB buffer is written between timed steps (L2 flushed)"}
        if cfg.N == 64:
            fl = attn_flops(cfg)
            rec["tensor"] = {"flops": fl, "achieved_tflops": fl / (attn["p50"] * 1e-3) / 1e12, "peak": tpeak,
                             "peak_kind": tpeak_kind, "frac": fl / (attn["p50"] * 1e-3) / 1e12 / tpeak}
        out[cfg.name] = rec
        del d, step
        torch.cuda.empty_cache()
    out["peak"], out["peak_kind"] = peak, peak_kind
    return out


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, cfg):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    LT.load()

    inp = W.generate(cfg, seed=rank)
    tdt = torch.bfloat16 if cfg.dtype == W.BF16 else torch.float16

    def h16(a, pin=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt)
        return t.pin_memory() if pin else t.to(dev)

    d = dict(q=h16(inp["q"]), k_pool=h16(inp["k_pool"]), v_pool=h16(inp["v_pool"]), k_tree=h16(inp["k_tree"]),
             v_tree=h16(inp["v_tree"]), page_table=torch.from_numpy(inp["page_table"]).to(dev),
             ctx_len=torch.from_numpy(inp["ctx_len"]).to(dev), parent=torch.from_numpy(inp["parent"]).to(dev),
             draft=torch.from_numpy(inp["draft"]).to(dev), logits=torch.from_numpy(inp["logits"]).to(dev))
    stream = torch.cuda.Stream(device=dev)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab, device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # inputs and the zeroed counters are ready first

    def one(dd=None):
        issue_step(step, d if dd is None else dd, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            one()
    stream.synchronize()
    status = int(step.status.item())
    acc_total = int(step.acc_len.sum().item())

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    # events every `grp` steps give the spread of the per-step time without
    # putting an event between every pair of programmatically dependent launches
    grp = 10 if args.steps >= 40 else 1
    bounds = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps // grp + 1)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for k in range(args.steps):
        if k % grp == 0 and k // grp < len(bounds) - 1:
            bounds[k // grp].record(stream)
        one()
        if k + 1 == (args.steps // grp) * grp:
            bounds[-1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = t_start.elapsed_time(t_end)
    step_st = ms_stats([bounds[k].elapsed_time(bounds[k + 1]) / grp for k in range(len(bounds) - 1)])
    step_st["group"] = grp
    # the dominant kernel alone: lucetree_verify_attn calls back to back on the
    # same resident inputs (512 MiB of K/V > L2), ten calls between CUDA events
    attn_st = ms_stats(time_attention(LT, step, d, stream, args.steps))
    attn_st["group"] = 10
    attn_ms = attn_st["mean"]
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    ms_per_step = elapsed_ms / args.steps

    # the same step replayed from a CUDA graph (launch overhead off the host)
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        with torch.cuda.stream(stream):
            g0.record(stream)
            for _ in range(args.steps):
                g.replay()
            g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = max_over_ranks(g0.elapsed_time(g1), dev) / args.steps
        del g
    except Exception as e:  # capture is an extra measurement; the timed loop above is the contract
        print(f"[bench] CUDA graph replay not measured: {e}", file=sys.stderr)

    # end to end: pinned host inputs -> device, the step, results -> host, every step
    # The step's inputs (queries, tree K/V, parents, draft tokens, logits) sit in
    # one pinned host buffer and go up in one copy into one of two device
    # buffers, whose typed views the step reads; its result (accepted path,
    # count, bonus token, new length) is one contiguous device buffer that one
    # copy reads back.
    up_keys = ("q", "k_tree", "v_tree", "parent", "draft", "logits")
    src = dict(q=h16(inp["q"], True), k_tree=h16(inp["k_tree"], True), v_tree=h16(inp["v_tree"], True),
               parent=torch.from_numpy(inp["parent"]), draft=torch.from_numpy(inp["draft"]),
               logits=torch.from_numpy(inp["logits"]))
    offs, pos = {}, 0
    for k in up_keys:
        offs[k] = pos
        pos += -(-src[k].numel() * src[k].element_size() // 256) * 256
    host_pack = torch.empty(pos, dtype=torch.uint8).pin_memory()

    def views(pack):
        return {k: pack[offs[k]:offs[k] + src[k].numel() * src[k].element_size()].view(src[k].dtype).view(src[k].shape)
                for k in up_keys}

    for k, v in views(host_pack).items():
        v.copy_(src[k])
    n_buf = 3
    dev_packs = [torch.empty(pos, dtype=torch.uint8, device=dev) for _ in range(n_buf)]
    res = dict(results=torch.empty_like(step.results, device="cpu").pin_memory())
    h2d = sum(src[k].numel() * src[k].element_size() for k in up_keys)
    d2h = sum(t.numel() * t.element_size() for t in res.values())
    e2e_steps = min(args.steps, 500)
    # Every step copies its own inputs from pinned host memory and the host
    # reads every step's result back.  The inputs go into three rotating
    # device buffers, copied on a second stream two steps ahead, so a step's
    # upload overlaps the two steps before it.  Two VerifyStep objects take
    # turns, so step i's result is read back on a third stream while step i+1
    # runs (a copy on the compute stream would sit between two steps and keep
    # the next step's programmatic launch from overlapping this one's tail);
    # the host enqueues step i before it waits for step i-1's result.
    copy_stream = torch.cuda.Stream(device=dev)
    rb_stream = torch.cuda.Stream(device=dev)
    steps2 = [step, LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab, device=dev)]
    stream.wait_stream(torch.cuda.current_stream(dev))  # the second step's zeroed counters
    bufs = []
    for pk in dev_packs:
        b = dict(d)
        b.update(views(pk))
        bufs.append(b)
    ev_in = [torch.cuda.Event() for _ in range(n_buf)]
    ev_used = [torch.cuda.Event() for _ in range(n_buf)]
    ev_res = [torch.cuda.Event(), torch.cuda.Event()]
    for e in ev_res:
        e.record(rb_stream)
    # every tenth upload is timed (its own event pair, read after the loop)
    ev_copy = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(-(-e2e_steps // 10))]
    results = [res, {k: torch.empty_like(t).pin_memory() for k, t in res.items()}]

    def upload(i):
        b = i % n_buf
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_used[b])  # the step that last read this buffer has finished
            if i % 10 == 0:
                ev_copy[i // 10][0].record(copy_stream)
            dev_packs[b].copy_(host_pack, non_blocking=True)
            if i % 10 == 0:
                ev_copy[i // 10][1].record(copy_stream)
            ev_in[b].record(copy_stream)

    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    upload(0)
    if e2e_steps > 1:
        upload(1)
    for i in range(e2e_steps):
        if i + 2 < e2e_steps:
            upload(i + 2)
        st = steps2[i % 2]
        with torch.cuda.stream(stream):
            stream.wait_event(ev_in[i % n_buf])
            stream.wait_event(ev_res[i % 2])  # step i-2's result (same object) has been read back
            issue_step(st, bufs[i % n_buf], stream)
            ev_used[i % n_buf].record(stream)
        with torch.cuda.stream(rb_stream):
            rb_stream.wait_event(ev_used[i % n_buf])
            results[i % 2]["results"].copy_(st.results, non_blocking=True)
            ev_res[i % 2].record(rb_stream)
        if i >= 1:
            ev_res[(i - 1) % 2].synchronize()  # the host has step i-1's result
    ev_res[(e2e_steps - 1) % 2].synchronize()  # and the last step's
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev) / e2e_steps
    torch.cuda.synchronize(dev)
    copy_ms = [a.elapsed_time(b) for a, b in ev_copy]
    barrier()

    sb = step_bytes(cfg, acc_total)
    value = world * sb / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = peak_hbm()
    achieved = attn_bytes(cfg) / (attn_ms * 1e-3) / 1e9
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic", "config": config_dict(cfg),
        "verify_steps_per_s": world * 1e3 / ms_per_step,
        "verify_steps_per_s_graph": (world * 1e3 / graph_ms) if graph_ms else None,
        "hbm_pct_of_peak": 100.0 * (sb / (ms_per_step * 1e-3) / 1e9) / peak,
        "attn_ms_per_call": attn_ms, "attn_ms_stats": attn_st, "step_ms_stats": step_st,
        "accepted_per_step": acc_total, "device_status": status,
        "clocks": clocks,
        "e2e": {"value": world * sb / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "h2d_ms_per_copy_p50": float(np.median(copy_ms)) if copy_ms else None,
                "pipeline": "each step's inputs (one packed pinned buffer, one copy) upload on a second stream two "
                            "steps ahead into one of three device buffers; two VerifyStep objects take turns and "
                            "each step's result (one copy, on a third stream) is read by the host one step later"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "roofline": {"bound": "hbm", "kernel": "lucetree_verify_attn (split-K prefix + tree/merge launch)",
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "algorithmic_bytes_per_launch": attn_bytes(cfg)},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, cfg, acc_total)
    if not args.no_lmhead:
        # the lm_head row is measured apart from the step: the step takes the
        # generator's logits, this call produces the argmax from hidden states
        line["lmhead_argmax"] = measure_lmhead(args, dev, stream, rank, with_cpu=world == 1 and not args.no_cpu_baseline)
    if not args.no_delta:
        # the recurrent-state row of hybrid targets, measured apart from the attention step
        line["delta_rule"] = measure_delta(args, dev, stream, rank, with_cpu=world == 1 and not args.no_cpu_baseline)
    if not args.no_stage:
        line["stage_pages"] = measure_stage(args, dev, stream, rank)
    if not args.no_vq and cfg.D == 256:
        line["quantised_v"] = measure_vq(args, dev, stream, rank, d, step, cfg)
        line["quantised_k"] = measure_kq(args, dev, stream, rank, d, step, cfg)
    if not args.no_configs:
        for held in (d, bufs[0], bufs[1]):
            held.clear()  # the other workloads need the device memory
        dev_packs.clear()
        del steps2[1:]
        torch.cuda.empty_cache()
        line["configs"] = measure_configs(args, dev, stream, rank)
    print(json.dumps(line), flush=True)
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


def measure_lmhead(args, dev, stream, rank, with_cpu=True):
    """The fused lm_head projection + argmax on the 27B-class workload (23 verify
    rows, d_model 5120, vocabulary 151936, bf16): each call streams the
    1.56 GB weight once, so it is timed alone with CUDA events on its stream
    (the weight is larger than L2; nothing to flush).  Inputs are seeded
    normals drawn on the device; parity is the tests' business."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    lc = W.LMHEAD_27B_B22
    if getattr(args, "lmhead_vocab", None):
        lc = dataclasses.replace(lc, name=f"{lc.name}-v{args.lmhead_vocab}", vocab=args.lmhead_vocab)
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + rank)
    hidden = torch.randn(lc.rows, lc.d_model, device=dev, generator=g).to(torch.bfloat16)
    weight = torch.empty(lc.vocab, lc.d_model, dtype=torch.bfloat16, device=dev)
    for v0 in range(0, lc.vocab, 16384):
        v1 = min(lc.vocab, v0 + 16384)
        weight[v0:v1] = (torch.randn(v1 - v0, lc.d_model, device=dev, generator=g) * lc.w_std).to(torch.bfloat16)
    out = torch.empty(lc.rows, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(LT.lucetree_lmhead_argmax_workspace(lc.rows), dtype=torch.uint8, device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))  # the weights are drawn on the current stream
    for _ in range(3):
        LT.lucetree_lmhead_argmax(hidden, weight, out, st, ws, stream=stream)
    n = max(10, min(100, args.steps // 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize(dev)
    for k in range(n):
        evs[k][0].record(stream)
        LT.lucetree_lmhead_argmax(hidden, weight, out, st, ws, stream=stream)
        evs[k][1].record(stream)
    torch.cuda.synchronize(dev)
    st_ms = ms_stats([a.elapsed_time(b) for a, b in evs])
    ms = st_ms["mean"]
    nbytes = lc.weight_bytes() + lc.rows * lc.d_model * 2 + lc.rows * 4
    peak, peak_kind = peak_hbm()
    achieved = nbytes / (ms * 1e-3) / 1e9
    res = {
        "workload": f"{lc.name}: rows {lc.rows}, d_model {lc.d_model}, vocab {lc.vocab}, bf16",
        "ms_per_call": ms, "ms_stats": st_ms, "calls_timed": n, "device_status": int(st.item()),
        "tflops": 2.0 * lc.rows * lc.d_model * lc.vocab / (ms * 1e-3) / 1e12,
        "roofline": {"bound": "hbm", "kernel": "lucetree_lmhead_argmax", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic("lmhead_argmax_lmhead-27b-b22.md", "lmhead")
                     if lc.vocab == W.LMHEAD_27B_B22.vocab else None,
                     "algorithmic_bytes_per_launch": nbytes},
    }
    if with_cpu:
        import oracle
        threads = os.cpu_count() or 1
        hb = hidden.view(torch.int16).cpu().numpy().view(np.uint16)
        wb = weight.view(torch.int16).cpu().numpy().view(np.uint16)
        sample = 2
        t0 = time.perf_counter()
        oracle.lmhead_argmax(hb[:sample], wb, oracle.BF16, threads=threads)
        cpu_ms = (time.perf_counter() - t0) * 1e3 * lc.rows / sample
        res["cpu_baseline"] = {"ms_per_call": cpu_ms, "cores": threads, "kind": "oracle",
                               "sample": f"{sample} of {lc.rows} rows over the full vocabulary, scaled to {lc.rows}"}
    return res


def measure_delta(args, dev, stream, rank, with_cpu=True):
    """The recurrent-state (gated delta rule) tree pass and its commit on the
    27B-class hybrid-layer workload (22-node tree, 16 q/k and 32 v heads of
    128 dims, fp32 state), timed alone with CUDA events on their stream.  The
    commit replays the deepest root path.  Inputs are the seeded workload."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    dc = W.DELTA_27B_B22
    inp = W.generate_delta(dc, seed=rank)
    tdt = torch.bfloat16
    d = {k: torch.from_numpy(np.ascontiguousarray(inp[k]).view(np.int16)).view(tdt).to(dev) for k in ("q", "k", "v")}
    for k in ("alpha", "beta", "state", "parent"):
        d[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev)
    out = torch.empty(dc.B, dc.N, dc.Hv, dc.dv, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    par = inp["parent"][0]
    depth = np.zeros(dc.N, int)
    for i in range(dc.N):
        depth[i] = 0 if par[i] < 0 else depth[par[i]] + 1
    path, i = [], int(np.argmax(depth))
    while i >= 0:
        path.append(i)
        i = int(par[i])
    path = path[::-1]
    acc = np.full((dc.B, dc.N), -1, np.int32)
    acc[0, :len(path)] = path
    acc_d = torch.from_numpy(acc).to(dev)
    len_d = torch.tensor([len(path)], dtype=torch.int32, device=dev)
    state_work = d["state"].clone()
    stream.wait_stream(torch.cuda.current_stream(dev))  # the copies above run on the current stream

    def tree():
        LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["state"], out, st,
                               stream=stream)

    def commit():
        LT.lucetree_delta_commit(d["k"], d["v"], d["alpha"], d["beta"], acc_d, len_d, state_work, st, stream=stream)

    def timed(fn, n):
        # a few microseconds of GPU work per call: the calls are captured in a
        # CUDA graph (20 per graph) and replayed, so host-side argument
        # marshalling does not leak into the device time
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(20):
                fn()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (20 * n)

    n = max(20, min(200, args.steps // 10))
    tree_ms, commit_ms = timed(tree, n), timed(commit, n)
    qkv = dc.B * dc.N * (2 * dc.Hk * dc.dk + dc.Hv * dc.dv) * 2 + dc.B * dc.N * dc.Hv * 8 + dc.B * dc.N * 4
    tree_bytes = dc.state_bytes() + qkv + dc.B * dc.N * dc.Hv * dc.dv * 4
    a = len(path)
    commit_bytes = 2 * dc.state_bytes() + dc.B * a * (dc.Hk * dc.dk + dc.Hv * dc.dv) * 2 + dc.B * a * dc.Hv * 8
    peak, peak_kind = peak_hbm()
    res = {
        "workload": f"{dc.name}: B {dc.B}, N {dc.N} (random tree, depth {int(depth.max()) + 1}), Hk {dc.Hk}, "
                    f"Hv {dc.Hv}, dk {dc.dk}, dv {dc.dv}, bf16 q/k/v, fp32 state; commit of {a} nodes",
        "tree_ms_per_call": tree_ms, "commit_ms_per_call": commit_ms, "calls_timed": 20 * n,
        "timing": "CUDA graph of 20 calls replayed; device time per call",
        "device_status": int(st.item()),
        "roofline": {"bound": "latency", "kernel": "lucetree_delta_tree",
                     "achieved": tree_bytes / (tree_ms * 1e-3) / 1e9, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": tree_bytes / (tree_ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": tree_bytes},
        "commit_roofline": {"bound": "latency", "kernel": "lucetree_delta_commit",
                            "achieved": commit_bytes / (commit_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                            "frac": commit_bytes / (commit_ms * 1e-3) / 1e9 / peak,
                            "algorithmic_bytes_per_launch": commit_bytes},
    }
    if with_cpu:
        import oracle
        t0 = time.perf_counter()
        oracle.delta_tree(inp, oracle.BF16)
        oracle.delta_commit(inp, oracle.BF16, acc, np.array([a], np.int32))
        res["cpu_baseline"] = {"ms_per_call": (time.perf_counter() - t0) * 1e3, "cores": 1, "kind": "oracle",
                               "sample": "the whole workload: tree pass plus commit, one thread"}
    return res


def measure_vq(args, dev, stream, rank, d, step, cfg):
    """The headline attention call with V stored quantised (int8 and int4 codes,
    one power-of-two exponent per token and head; K stays bf16), timed with
    CUDA events on the stream over the same resident inputs as the step, in
    spans of ten back-to-back calls like the 16-bit call."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    res = {}
    L = sum(cfg.ctx)
    peak, peak_kind = peak_hbm()
    for name, fmt, vbytes in (("int8", W.V_INT8, 1.0), ("int4", W.V_INT4, 0.5)):
        vq = W.generate_vq(cfg, fmt, seed=rank)
        codes = torch.from_numpy(vq["v_codes"]).to(dev)
        vexp = torch.from_numpy(vq["v_exp"]).to(dev)
        stream.wait_stream(torch.cuda.current_stream(dev))

        def call():
            LT.lucetree_verify_attn_vq(d["q"], d["k_pool"], codes, vexp, fmt, d["page_table"], d["ctx_len"],
                                       d["k_tree"], d["v_tree"], step.anc, step.out, step.status, step.ws_attn,
                                       stream=stream)

        st_ms = ms_stats(time_spans(call, stream, dev, max(20, min(200, args.steps // 10))))
        ms = st_ms["mean"]
        nbytes = int(L * cfg.Hkv * cfg.D * (2 + vbytes) + L * cfg.Hkv
                     + cfg.B * cfg.N * cfg.Hq * cfg.D * 2 + cfg.B * cfg.N * cfg.Hq * cfg.D * 4 + 4 * L // 64)
        res[name] = {"ms_per_call": ms, "ms_stats": st_ms, "device_status": int(step.status.item()),
                     "algorithmic_bytes_per_launch": nbytes, "achieved_GBps": nbytes / (ms * 1e-3) / 1e9,
                     "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
                     "kv_bytes_per_token": cfg.Hkv * cfg.D * (2 + vbytes) + cfg.Hkv}
    res["workload"] = f"{cfg.name} attention call, K bf16, V as int8 / int4 codes with per-token exponents"
    res["peak"], res["peak_kind"] = peak, peak_kind
    return res


def measure_kq(args, dev, stream, rank, d, step, cfg):
    """The headline attention call with K stored as FP8 E4M3 codes (one
    power-of-two exponent per token and head) and V in bf16 or as int8 codes,
    timed with CUDA events on the stream over resident inputs, in spans of ten
    back-to-back calls like the 16-bit call.  The codes
    are drawn on the device from N(0, 160^2) values, the exponents uniform in
    [119, 120] (keys of about unit spread: the generator's default)."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    res = {}
    L = sum(cfg.ctx)
    P = d["k_pool"].shape[0]
    peak, peak_kind = peak_hbm()
    g = torch.Generator(device=dev)
    g.manual_seed(99 + rank)
    # codes of N(0, 160^2) values (a row's largest magnitude near the top of E4M3's range, as a per-token
    # scale puts it), the distribution of the generator's default
    kc = torch.empty((P, cfg.Hkv, W.PAGE, cfg.D), dtype=torch.uint8, device=dev)
    flat = kc.view(-1)
    for i in range(0, flat.numel(), 1 << 26):
        j = min(flat.numel(), i + (1 << 26))
        x = (torch.randn(j - i, generator=g, device=dev) * 160.0).clamp_(-448.0, 448.0)
        flat[i:j] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    ke = torch.randint(119, 121, (P, cfg.Hkv, W.PAGE), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    vq = W.generate_vq(cfg, W.V_INT8, seed=rank)
    vcodes = torch.from_numpy(vq["v_codes"]).to(dev)
    vexp = torch.from_numpy(vq["v_exp"]).to(dev)
    ws = torch.empty(LT.lucetree_verify_attn_kq_workspace(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D), dtype=torch.uint8,
                     device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    for name, fmt, vbytes in (("e4m3_k_bf16_v", LT.LUCETREE_V_SAME, 2.0), ("e4m3_k_int8_v", LT.LUCETREE_V_INT8, 1.0)):
        vp, vx = (d["v_pool"], None) if fmt == LT.LUCETREE_V_SAME else (vcodes, vexp)

        def call():
            LT.lucetree_verify_attn_kq(d["q"], kc, ke, vp, d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
                                       step.anc, step.out, step.status, ws, v_format=fmt, v_exp=vx, stream=stream)

        st_ms = ms_stats(time_spans(call, stream, dev, max(20, min(200, args.steps // 10))))
        per_tok = cfg.Hkv * (cfg.D * (1 + vbytes) + 1 + (1 if fmt != LT.LUCETREE_V_SAME else 0))
        nbytes = int(L * per_tok + cfg.B * cfg.N * cfg.Hq * cfg.D * 2 + cfg.B * cfg.N * cfg.Hq * cfg.D * 4
                     + 4 * L // 64)
        res[name] = {"ms_per_call": st_ms["mean"], "ms_stats": st_ms, "device_status": int(step.status.item()),
                     "algorithmic_bytes_per_launch": nbytes, "achieved_GBps": nbytes / (st_ms["mean"] * 1e-3) / 1e9,
                     "frac_of_hbm_peak": nbytes / (st_ms["mean"] * 1e-3) / 1e9 / peak, "kv_bytes_per_token": per_tok}
    res["workload"] = f"{cfg.name} attention call, K as E4M3 codes with per-token exponents, V bf16 or int8 codes"
    res["peak"], res["peak_kind"] = peak, peak_kind
    return res


def measure_stage(args, dev, stream, rank):
    """Host-resident cold pages: a quarter of the 128K-token sequence's pages
    (512 pages of [4 heads][64][256] bf16, K and V: 128 MiB) staged from
    page-locked host pools into device pool pages, timed with CUDA events on
    the stream, against a plain pinned host-to-device copy of the same bytes
    (the link's copy rate, measured here)."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    cfg = W.HEADLINE_128K_B22
    n = (cfg.ctx[0] // W.PAGE) // 4
    shape = (n, cfg.Hkv, W.PAGE, cfg.D)
    g = torch.Generator()
    g.manual_seed(777 + rank)
    host_k = torch.randint(-32768, 32767, shape, dtype=torch.int16, generator=g).pin_memory()
    host_v = torch.randint(-32768, 32767, shape, dtype=torch.int16, generator=g).pin_memory()
    pool_k = torch.empty((n + 64,) + shape[1:], dtype=torch.int16, device=dev)
    pool_v = torch.empty_like(pool_k)
    src = torch.arange(n, dtype=torch.int32, device=dev)
    dst = torch.randperm(n + 64, generator=g)[:n].to(torch.int32).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    nbytes = 2 * host_k.numel() * 2
    stream.wait_stream(torch.cuda.current_stream(dev))

    def stage():
        LT.lucetree_stage_pages(host_k, host_v, src, dst, pool_k, pool_v, st, stream=stream)

    def copy():
        pool_k[:n].copy_(host_k, non_blocking=True)
        pool_v[:n].copy_(host_v, non_blocking=True)

    res = {}
    for name, fn in (("stage", stage), ("h2d_copy", copy)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
            torch.cuda.synchronize(dev)
            for e0, e1 in evs:
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = float(np.median([e0.elapsed_time(e1) for e0, e1 in evs]))
    gbs = nbytes / (res["stage"] * 1e-3) / 1e9
    peak = nbytes / (res["h2d_copy"] * 1e-3) / 1e9
    return {
        "workload": f"{n} cold pages of {cfg.Hkv}x{W.PAGE}x{cfg.D} bf16, K and V ({nbytes / 2**20:.0f} MiB), "
                    "page-locked host pools -> device pool pages",
        "ms_per_call": res["stage"], "device_status": int(st.item()),
        "roofline": {"bound": "host link", "kernel": "lucetree_stage_pages", "achieved": gbs, "peak": peak,
                     "peak_kind": "measured here: pinned host-to-device copy of the same bytes", "unit": "GB/s",
                     "frac": gbs / peak, "algorithmic_bytes_per_launch": nbytes},
    }


def run_vq_only(args):
    """Only the quantised-V attention calls on the headline workload (for
    profiler captures): inputs, ancestor masks, then measure_vq."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    cfg = W.CONFIGS[args.config]
    inp = W.generate(cfg, seed=0, with_logits=False)
    tdt = torch.bfloat16 if cfg.dtype == W.BF16 else torch.float16
    h16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(dev)
    d = dict(q=h16(inp["q"]), k_pool=h16(inp["k_pool"]), k_tree=h16(inp["k_tree"]), v_tree=h16(inp["v_tree"]),
             page_table=torch.from_numpy(inp["page_table"]).to(dev), ctx_len=torch.from_numpy(inp["ctx_len"]).to(dev),
             parent=torch.from_numpy(inp["parent"]).to(dev))
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab, device=dev)
    LT.lucetree_build_anc_mask(d["parent"], step.anc, step.status, stream)
    d["v_pool"] = h16(inp["v_pool"])
    print(json.dumps({"quantised_v": measure_vq(args, dev, stream, 0, d, step, cfg),
                      "quantised_k": measure_kq(args, dev, stream, 0, d, step, cfg)}), flush=True)
    return 0


def run_stage_only(args):
    import torch
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    print(json.dumps({"stage_pages": measure_stage(args, dev, stream, 0)}), flush=True)
    return 0


def run_delta_only(args):
    import torch
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    print(json.dumps({"delta_rule": measure_delta(args, dev, stream, 0, with_cpu=False)}), flush=True)
    return 0


def run_lmhead_only(args):
    import torch
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    print(json.dumps({"lmhead_argmax": measure_lmhead(args, dev, stream, 0, with_cpu=False)}), flush=True)
    return 0


def run_configs_only(args):
    import torch
    from speculative_decoding_tree_ddtree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    print(json.dumps({"configs": measure_configs(args, dev, stream, 0)}), flush=True)
    return 0


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=W.HEADLINE_128K_B22.name, choices=sorted(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-lmhead", action="store_true", help="skip the fused lm_head + argmax measurement")
    ap.add_argument("--lmhead-only", action="store_true", help="time only the fused lm_head + argmax")
    ap.add_argument("--lmhead-vocab", type=int, default=None,
                    help="with --lmhead-only: a smaller vocabulary (profiler captures)")
    ap.add_argument("--no-delta", action="store_true", help="skip the recurrent-state (delta rule) measurement")
    ap.add_argument("--delta-only", action="store_true", help="time only the recurrent-state tree pass and commit")
    ap.add_argument("--no-stage", action="store_true", help="skip the host-resident page staging measurement")
    ap.add_argument("--no-vq", action="store_true", help="skip the quantised-V attention measurement")
    ap.add_argument("--vq-only", action="store_true", help="time only the quantised-V attention calls")
    ap.add_argument("--stage-only", action="store_true", help="time only the host-resident page staging")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (32K, 128K/b40, 256K paged, the 4-sequence sweep)")
    ap.add_argument("--configs-only", action="store_true", help="time only the other workloads")
    return ap


def main(argv=None):
    args = build_parser().parse_args(argv)
    if args.lmhead_only:
        return run_lmhead_only(args)
    if args.delta_only:
        return run_delta_only(args)
    if args.stage_only:
        return run_stage_only(args)
    if args.vq_only:
        return run_vq_only(args)
    if args.configs_only:
        return run_configs_only(args)
    cfg = W.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())

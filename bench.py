#!/usr/bin/env python3
"""Benchmark of the bounded-tree speculative decoding hot path on GB300.

One step = the whole path on one batch of synthetic input, resident in HBM:
  tsd_build_tree  (drafter top-k + log-normaliser, best-first heap)
  tsd_tree_mask   (ancestor bitmask + position ids)
  tsd_verify_tev  (node-row reduction, per-node combination, exit and bonus draws)
Workload (per GPU): 32 independent trees, V=151936, L=16, k=8, B=256, T=0.6,
bf16 logits -- the batched verification configuration.  The metric is TEV
rounds (trees verified) per second; the dominant kernel is the node-row
reduction, reported against the measured HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
trees (weak scaling, no data-path collective); the step time is the max over
ranks.  --impl reference times the float64 CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TEV verify rounds/sec and logits HBM GB/s (% of peak) at V=151936, B=64/256"
WORKLOAD = dict(workload="batched verification: 32 independent trees, V=151936, L=16, "
                         "top-k=8, B=256, T=0.6, bf16 (Gumbel-perturbed Zipf drafter; "
                         "target = drafter row at node depth + N(0, 1.5^2))",
                trees_per_gpu=32, V=151936, L=16, topk=8, B=256, temperature=0.6,
                step="tsd_build_tree, then tsd_tree_mask (side stream) alongside tsd_verify_tev",
                l2="inputs larger than L2: 2.66 GB of logits read per step per GPU, no flush")
HBM_PEAK_FALLBACK = 6800.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_PEAK_FALLBACK, "fallback"


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "rows_kernel_b256_traffic.json")
ROWS_SOURCES = ("tree_speculative_decoding_position_gb300/csrc/k_rows.cu",
                "tree_speculative_decoding_position_gb300/csrc/chunk_reduce.cuh",
                "tree_speculative_decoding_position_gb300/csrc/tsd_internal.cuh")


def rows_source_digest() -> str:
    """SHA-256 over the source files that define the node-row reduction."""
    import hashlib
    h = hashlib.sha256()
    for rel in ROWS_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def committed_traffic():
    """Per-launch DRAM bytes (read + write) of the node-row reduction on the
    workload's launch, from the ncu capture recorded in
    profiles/rows_kernel_b256_traffic.json, and a note.  The figure is null
    when no capture is recorded or when the kernel's sources have changed
    since it was taken (the record carries their digest)."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no ncu capture recorded"
    if rec.get("source_sha256") != rows_source_digest():
        return None, "the kernel's sources changed since the recorded ncu capture"
    return float(rec["dram_bytes_per_launch"]), rec.get("how", "")


# ---------------------------------------------------------------------------
# Clocks: NVML read-only queries, polled during the timed region.
# ---------------------------------------------------------------------------
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, uuid: str, period_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.period = period_s
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            return

    def _poll(self):
        mhz, reasons, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(reasons))
            self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
            self.samples.append((int(mhz.value), int(reasons.value), pw.value / 1000.0))
            time.sleep(self.period)

    def start(self):
        self.samples = []
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()

    def stop(self) -> dict:
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        self._stop.set()
        self._t.join()
        s = self.samples
        reasons = set()
        for _, r, _ in s:
            for bit, name in _REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in s) if s else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(s),
                "power_w_max": max((x[2] for x in s), default=None)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def rank_seeds(rank: int, nt: int) -> list:
    """Seeds of one rank's trees: each rank verifies its own trees (replicas
    over disjoint inputs)."""
    import synth
    return [synth.seed_for(2, t) + 100000 * rank for t in range(nt)]


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: every rank's elapsed time, all-reduced by max."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, nt: int, ms_per_step: float) -> float:
    """Trees verified per second by the whole job: every rank's trees per step
    over the slowest rank's step time."""
    return world * nt / (ms_per_step * 1e-3)


def run_ours(args):
    import torch

    import synth
    import tree_speculative_decoding_position_gb300 as tsd

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tsd.load()

    W = WORKLOAD
    nt, V, L, k, B, T = W["trees_per_gpu"], W["V"], W["L"], W["topk"], W["B"], W["temperature"]
    if args.trees:
        nt = args.trees  # a smaller batch, for profiler captures only
    seeds = rank_seeds(rank, nt)
    drafter = synth.zipf_drafter(nt, L, V, 0, device=dev, seeds=seeds)          # [nt,1,L,V]
    tr = tsd.tsd_build_tree(drafter, topk=k, B=B)
    target = torch.empty(nt, B + 1, V, dtype=torch.bfloat16, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(drafter[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1,
                               out=target[t, :n])
        target[t, n:] = 0
    torch.cuda.synchronize()
    ws_b = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, nt, 1, L, V, k, B,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    ws_v = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, nt, 1, 1, V, 1, B,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)  # the mask does not depend on TEV: run it alongside

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        t_ = tsd.tsd_build_tree(drafter, topk=k, B=B, workspace=ws_b)
        if ev is not None:
            ev[1].record(stream)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            tsd.tsd_tree_mask(t_["parent"], t_["n_nodes"], prefix_len=1024)
        if ev is not None:
            out = tsd.tsd_verify_tev_timed(target, t_["parent"], t_["token"], t_["n_nodes"], T,
                                           seed=i, stage_events=ev[2:7], workspace=ws_v)
        else:
            out = tsd.tsd_verify_tev(target, t_["parent"], t_["token"], t_["n_nodes"], T,
                                     seed=i, workspace=ws_v)
        stream.wait_stream(side)
        return t_, out

    for i in range(args.warmup):
        step(i)
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    # the headline: K steps of the plain public calls, nothing recorded between
    # their kernels
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = new_events(2)
    clocks.start()
    start.record(stream)
    last = None
    for i in range(args.steps):
        last = step(1000 + i)
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    assert int((last[1]["status"] != 0).sum()) == 0, "a tree failed in the timed region"

    # the stage breakdown, from a second timed region of K steps in which TEV
    # is the instrumented call (events recorded between its kernels)
    evsets = [new_events(7) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(3000 + i, evsets[i])
    torch.cuda.synchronize()

    def avg(a, b):
        return statistics.mean(evsets[i][a].elapsed_time(evsets[i][b]) for i in range(args.steps))
    stage = dict(build=avg(0, 1), tev_prep=avg(2, 3), tev_rows=avg(3, 4),
                 tev_combine=avg(4, 5), tev_draws=avg(5, 6))  # the mask runs on a side stream
    n_nodes_total = int(last[0]["n_nodes"].sum())
    rows_bytes = n_nodes_total * V * 2
    peak, peak_kind = measured_peaks()
    achieved = rows_bytes / (stage["tev_rows"] * 1e-3) / 1e9
    ms_per_step = total_ms / args.steps
    value = whole_job_value(world, nt, ms_per_step)

    # end to end through the public API with host buffers: the drafter and
    # target logits sit in page-locked host memory and the library's kernels
    # read them there over the host link (they are the host->device transfer,
    # inside the timed region); the three result vectors are read back.  The
    # same step with explicit copies into device buffers is recorded beside it.
    e2e = None
    e2e_copy = None
    if not args.no_e2e:
        drafter_h = torch.empty(drafter.shape, dtype=drafter.dtype, pin_memory=True)
        target_h = torch.empty(target.shape, dtype=target.dtype, pin_memory=True)
        drafter_h.copy_(drafter)
        target_h.copy_(target)
        res_h = torch.empty(3, nt, dtype=torch.int32, pin_memory=True)
        ke = max(3, min(args.steps, 20))

        def step_host(i):
            t_ = tsd.tsd_build_tree(drafter_h, topk=k, B=B, workspace=ws_b, device=dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                tsd.tsd_tree_mask(t_["parent"], t_["n_nodes"], prefix_len=1024)
            o_ = tsd.tsd_verify_tev(target_h, t_["parent"], t_["token"], t_["n_nodes"], T,
                                    seed=i, workspace=ws_v)
            stream.wait_stream(side)
            return t_, o_

        def step_copy(i):
            drafter.copy_(drafter_h, non_blocking=True)
            target.copy_(target_h, non_blocking=True)
            return step(i)

        def timed(fn):
            for i in range(2):
                fn(i)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            s2, e2 = new_events(2)
            s2.record(stream)
            for i in range(ke):
                _, o = fn(2000 + i)
                res_h[0].copy_(o["exit_node"], non_blocking=True)
                res_h[1].copy_(o["bonus_token"], non_blocking=True)
                res_h[2].copy_(o["accept_len"], non_blocking=True)
            e2.record(stream)
            torch.cuda.synchronize()
            assert int((o["status"] != 0).sum()) == 0, "a tree failed in the end-to-end run"
            e_ms = max_over_ranks(s2.elapsed_time(e2) / ke, dist, dev)
            return {"value": whole_job_value(world, nt, e_ms), "unit": "rounds/s",
                    "h2d_bytes_per_step": drafter.numel() * 2 + target.numel() * 2,
                    "d2h_bytes_per_step": res_h.numel() * 4, "steps": ke,
                    "ms_per_step": e_ms}

        e2e = timed(step_host)
        e2e["how"] = "logits in pinned host memory, read by the kernels over the host link"
        e2e_copy = timed(step_copy)
        e2e_copy["how"] = "explicit copies of the logits into device buffers, then the device step"

    # secondary measurements (not the headline): TEV alone vs predraw on the
    # same trees, and the batch-1 Qwen-vocabulary round at B=64
    extra = {"stage_ms": {k_: round(v, 4) for k_, v in stage.items()}}
    if e2e_copy is not None:
        extra["e2e_explicit_copies"] = e2e_copy
    if rank == 0 and not args.no_extra:
        extra.update(secondary(tsd, torch, synth, dev, stream, dict(last[0], _drafter=drafter),
                               target, T, ws_v, V))
        extra.update(exit_loss_bench(tsd, torch, stream, drafter, last[0], last[1], V))
        extra.update(forest_bench(tsd, torch, stream, drafter, k, B))

    if rank != 0:
        return
    traffic, traffic_note = committed_traffic()
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(drafter, target, last[0], k, B, T, out=last[1], seed=1000 + args.steps - 1)
    line = {
        "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(W, parallelism="replicas: dp%d over trees" % world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "rows_kernel (node-row reduction)",
                     "algorithmic_bytes_per_launch": rows_bytes,
                     "duration_ms": stage["tev_rows"],
                     "duration_from": "CUDA events around the kernel on its stream, mean over a "
                                      "second timed region of K steps with the instrumented TEV "
                                      "call (the headline steps record nothing between kernels)",
                     "traffic_note": traffic_note, "peak_kind": peak_kind},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 8 * args.steps,
        "clocks": clk, "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def oracle_ms(fn) -> float:
    """Wall time of one call of the float64 oracle on the host (one thread)."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    fn(oracle)
    return 1e3 * (time.perf_counter() - t0)


def exit_loss_bench(tsd, torch, stream, drafter, tree, tev, V):
    """The exit-guided loss on the workload's drafter rows (32 trees x 16 rows),
    weighted by the step's TEV exit masses: loss alone, and loss with its
    gradient (an fp32 row per drafter row).  Algorithmic bytes: one read of
    the drafter logits for the loss; for the gradient a second read plus the
    fp32 write."""
    out = {}
    rows = drafter.shape[0] * drafter.shape[2]
    dbytes = rows * V * 2
    nt, L = drafter.shape[0], drafter.shape[2]
    ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_EXIT_LOSS, nt, 1, L, V, 1,
                                            tree["token"].shape[1] - 1, drafter.dtype),
                     dtype=torch.uint8, device=drafter.device)
    for grad in (False, True):
        fn = lambda: tsd.tsd_exit_loss(drafter, tree["token"], tree["depth"], tree["n_nodes"],
                                       tev["exit_mass"], with_grad=grad, workspace=ws)
        # captured once in a CUDA graph and replayed, as a training step would
        cap = torch.cuda.Stream(drafter.device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for i in range(3):
                fn()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        for i in range(3):
            graph.replay()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for i in range(20):
            graph.replay()
        e.record(stream)
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / 20
        del graph
        nbytes = dbytes + (dbytes + rows * V * 4 if grad else 0)
        out["exit_loss" + ("_with_grad" if grad else "")] = {
            "ms": ms, "algorithmic_gb": nbytes / 1e9, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac_of_measured": nbytes / (ms * 1e-3) / 1e9 / measured_peaks()[0]}
    # the oracle beside it: one tree's loss and gradient, float64, one host thread
    z0 = drafter[0, 0].float().cpu().numpy()
    tk, dp = tree["token"][0].cpu().numpy(), tree["depth"][0].cpu().numpy()
    n0, w0 = int(tree["n_nodes"][0]), tev["exit_mass"][0].float().cpu().numpy()
    o_ms = oracle_ms(lambda orc: orc.exit_loss(z0, 1.0, tk, dp, n0, w0, with_grad=True))
    out["exit_loss_with_grad"].update(oracle_ms_per_tree=o_ms,
                                      ms_per_tree=out["exit_loss_with_grad"]["ms"] / nt,
                                      oracle_sample="one tree (16 rows), loss and gradient")
    return out


def forest_bench(tsd, torch, stream, drafter, k, B):
    """Shared-budget widths on the workload's 32 requests, each built to the
    cap B = 256 and then cut to the globally best M* prefixes under a
    synthetic linear round-time law t(M) = l0 + c1 M, l0 = 1 (one target
    call) and c1 = 1/S for a target that doubles its latency at S extra
    tree tokens.  Times the whole call (builder + selection + trim) against
    the plain builder on the same inputs, and reports M*, the width spread and
    the law's objective (G + R) / t(M*)."""
    out = {}
    nt, L, V = drafter.shape[0], drafter.shape[2], drafter.shape[3]
    ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_FOREST, nt, 1, L, V, k, B,
                                            drafter.dtype), dtype=torch.uint8, device=drafter.device)
    wsb = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, nt, 1, L, V, k, B,
                                             drafter.dtype), dtype=torch.uint8, device=drafter.device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(3):
        tsd.tsd_build_tree(drafter, topk=k, B=B, workspace=wsb)
    s.record(stream)
    for i in range(10):
        tsd.tsd_build_tree(drafter, topk=k, B=B, workspace=wsb)
    e.record(stream)
    torch.cuda.synchronize()
    out["forest_build_tree_ms"] = s.elapsed_time(e) / 10
    for S in (512, 2048, 8192):
        c1, M_max = 1.0 / S, nt * B
        for i in range(3):
            f = tsd.tsd_build_forest(drafter, topk=k, B=B, M_max=M_max, l0=1.0, c1=c1, workspace=ws)
        s.record(stream)
        for i in range(10):
            f = tsd.tsd_build_forest(drafter, topk=k, B=B, M_max=M_max, l0=1.0, c1=c1, workspace=ws)
        e.record(stream)
        torch.cuda.synchronize()
        w = (f["n_nodes"] - 1).clamp(min=0)
        M = int(f["total"])
        G = float(torch.where(f["score"][:, 1:] > -float("inf"), f["score"][:, 1:].double().exp(),
                              torch.zeros((), dtype=torch.float64, device=w.device)).sum())
        out["forest_S%d" % S] = {"ms": s.elapsed_time(e) / 10, "M_star": M,
                                 "width_min": int(w.min()), "width_max": int(w.max()),
                                 "objective": (G + nt) / (1.0 + c1 * M)}
    # the oracle beside it: one request's tree, and the selection over all 32
    # requests' builder trees (S = 2048)
    import numpy as np
    z0 = drafter[0, 0].float().cpu().numpy()
    tb = tsd.tsd_build_tree(drafter, topk=k, B=B, workspace=wsb)
    sc = tb["score"].double().cpu().numpy()
    dp, nn = tb["depth"].cpu().numpy(), tb["n_nodes"].cpu().numpy()
    b_ms = oracle_ms(lambda orc: orc.build_tree(orc.drafter_lists(z0, 1.0, k), B))
    s_ms = oracle_ms(lambda orc: orc.forest_select(sc, dp, nn, nt * B, 1.0, 1.0 / 2048))
    out["forest_S2048"].update(oracle_ms=b_ms * nt + s_ms, oracle_select_ms=s_ms,
                               oracle_sample="one request's tree (x 32 requests) plus the selection "
                                             "over 32 trees; float64, one host thread")
    return out


def secondary(tsd, torch, synth, dev, stream, tree, target, T, ws_v, V):
    out = {}
    # verifier stage: TEV vs predraw-and-follow, sequential residual and
    # proposal-aware verification on the same 32 trees; the proposal is the
    # drafter's own probability of each child's token (setup, not timed)
    drafter = tree["_drafter"]
    depth = tree["depth"].clamp(min=1).long() - 1
    logq = torch.log_softmax(drafter[:, 0].float(), dim=-1)           # [nt, L, V]
    q = torch.stack([logq[t, depth[t], tree["token"][t].clamp(min=0).long()].exp()
                     for t in range(drafter.shape[0])]).float().contiguous()
    del logq
    verifiers = (("tev", tsd.tsd_verify_tev), ("predraw", tsd.tsd_verify_ddtree),
                 ("seqres", tsd.tsd_verify_seqres),
                 ("proposal", lambda x, p_, t_, n_, T_, seed, workspace:
                  tsd.tsd_verify_proposal(x, p_, t_, n_, q, T_, seed=seed, workspace=workspace)))
    for name, fn in verifiers:
        for i in range(3):
            fn(target, tree["parent"], tree["token"], tree["n_nodes"], T, seed=i, workspace=ws_v)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for i in range(10):
            fn(target, tree["parent"], tree["token"], tree["n_nodes"], T, seed=i, workspace=ws_v)
        e.record(stream)
        torch.cuda.synchronize()
        out["verifier_ms_b256_x32_" + name] = s.elapsed_time(e) / 10
    # the oracle beside them: one tree of the 32, float64, one host thread
    n0 = int(tree["n_nodes"][0])
    z0 = target[0, :n0].float().cpu().numpy()
    p0, t0_ = tree["parent"][0].cpu().numpy(), tree["token"][0].cpu().numpy()
    q0 = q[0].double().cpu().numpy()
    out["verifier_oracle_ms_per_tree"] = {
        "seqres": oracle_ms(lambda orc: orc.seqres(z0, p0, t0_, n0, T, 1)),
        "proposal": oracle_ms(lambda orc: orc.proposal(z0, p0, t0_, n0, T, q0, 1)),
        "tev": oracle_ms(lambda orc: orc.tev(z0, p0, t0_, n0, T, 1)),
        "sample": "tree 0 of the 32 (B=256, V=151936)"}
    # batch-1 round, V=151936, B=64, T=1: 32 rotating copies (632 MB > 4x L2)
    B1 = 64
    dr = synth.zipf_drafter(1, 16, V, synth.seed_for(1), device=dev)
    t1 = tsd.tsd_build_tree(dr, topk=8, B=B1)
    n = int(t1["n_nodes"][0])
    copies = []
    for c in range(32):
        x = torch.zeros(1, B1 + 1, V, dtype=torch.bfloat16, device=dev)
        synth.target_from_rows(dr[0, 0], t1["depth"][0, :n], 1.5, synth.seed_for(1, 1) + c,
                               out=x[0, :n])
        copies.append(x)
    ws1 = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 1, 1, 1, V, 1, B1,
                                             torch.bfloat16), dtype=torch.uint8, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(48)]
    for ev in evs:
        for e in ev:
            e.record(stream)
    for i in range(8):
        tsd.tsd_verify_tev(copies[i % 32], t1["parent"], t1["token"], t1["n_nodes"], 1.0,
                           seed=i, workspace=ws1)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(48):
        tsd.tsd_verify_tev_timed(copies[i % 32], t1["parent"], t1["token"], t1["n_nodes"], 1.0,
                                 seed=i, stage_events=evs[i], workspace=ws1)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / 48
    rows_ms = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs)
    out["b64_single_tree"] = {"tev_rounds_per_s": 1000.0 / ms, "tev_ms": ms,
                              "row_reduction_ms": rows_ms,
                              "row_reduction_gbs": n * V * 2 / (rows_ms * 1e-3) / 1e9,
                              "row_reduction_kernel": "tev_stream_kernel (a launch this small "
                                                      "takes the two-kernel path)"}
    # the same round, greedy (T = 0)
    s.record(stream)
    for i in range(48):
        tsd.tsd_verify_tev(copies[i % 32], t1["parent"], t1["token"], t1["n_nodes"], 0.0,
                           seed=i, workspace=ws1)
    e.record(stream)
    torch.cuda.synchronize()
    out["b64_single_tree"]["tev_ms_T0"] = s.elapsed_time(e) / 48
    # the same round as a decode loop would issue it: build + mask + TEV captured
    # once in a CUDA graph and replayed (GPU latency without the Python calls),
    # L2 flushed before every replay
    ws1b = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 1, 1, 16, V, 8, B1,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024,
                        dtype=torch.float32, device=dev)

    def round1(i):
        t_ = tsd.tsd_build_tree(dr, topk=8, B=B1, workspace=ws1b)
        tsd.tsd_tree_mask(t_["parent"], t_["n_nodes"], prefix_len=1024)
        return tsd.tsd_verify_tev(copies[0], t_["parent"], t_["token"], t_["n_nodes"], 1.0,
                                  seed=i, workspace=ws1)

    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(3):
            round1(i)
    stream.wait_stream(cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        round1(0)
    lat = []
    for i in range(45):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 5:
            lat.append(a.elapsed_time(b))
    out["b64_single_tree"]["round_graph_ms"] = statistics.median(lat)
    out["b64_single_tree"]["round_graph_ms_best"] = min(lat)
    del graph
    # the verifier stage alone at batch 1: TEV against predraw-and-follow on
    # the same tree and logits, each captured in a CUDA graph and replayed with
    # L2 flushed first (the pages compare the two at batch 1)
    for name, vfn in (("tev", tsd.tsd_verify_tev), ("predraw", tsd.tsd_verify_ddtree)):
        with torch.cuda.stream(cap):
            for i in range(3):
                vfn(copies[0], t1["parent"], t1["token"], t1["n_nodes"], 1.0, seed=i,
                    workspace=ws1)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            vfn(copies[0], t1["parent"], t1["token"], t1["n_nodes"], 1.0, seed=0, workspace=ws1)
        lat = []
        for i in range(45):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 5:
                lat.append(a.elapsed_time(b))
        out["b64_single_tree"]["verify_graph_ms_" + name] = statistics.median(lat)
        del graph
    out["batch1_tev_vs_predraw"] = batch1_grid(tsd, torch, synth, dev, stream, flush, cap, V)
    # the oracle beside it: the same round, float64, one host thread
    z1 = dr[0, 0].float().cpu().numpy()
    tg1 = copies[0][0, :n].float().cpu().numpy()
    out["b64_single_tree"].update(
        oracle_round_ms=oracle_ms(lambda orc: oracle_round(orc, z1, tg1, 8, B1, 1.0, 0)),
        oracle_sample="one round (drafter statistics, heap, mask, TEV at T=1), float64, one thread")
    del copies
    # mixture-of-futures workload: 16 trees, K = 8 modes from two latent
    # futures, B = 128; the mixture builder, then TEV at T = 1 on its trees
    nt_m, K_m, B_m = 16, 8, 128
    mix, _, choice = synth.mixture_drafter(nt_m, K_m, 16, V, synth.seed_for(3), device=dev)
    ws_m = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, nt_m, K_m, 16, V, 8, B_m,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    for i in range(3):
        tm = tsd.tsd_build_tree(mix, topk=8, B=B_m, workspace=ws_m)
    s.record(stream)
    for i in range(10):
        tm = tsd.tsd_build_tree(mix, topk=8, B=B_m, workspace=ws_m)
    e.record(stream)
    torch.cuda.synchronize()
    build_eager_ms = s.elapsed_time(e) / 10  # back-to-back calls, host launch rate included
    # the device time of one call: CUDA-graph replay, L2 flushed before each
    build_ms, _ = graph_latency(torch, stream, flush, cap,
                                lambda: tsd.tsd_build_tree(mix, topk=8, B=B_m, workspace=ws_m))
    tgt_m = torch.zeros(nt_m, B_m + 1, V, dtype=torch.bfloat16, device=dev)
    for t in range(nt_m):
        n_t = int(tm["n_nodes"][t])
        # the target follows the future the tree's seed chose, at its node depths
        fut = synth.mixture_drafter(1, 2, 16, V, synth.seed_for(3) + t, device=dev)[1][0, choice[t]]
        synth.target_from_rows(fut, tm["depth"][t, :n_t], 1.5, synth.seed_for(3, 500 + t),
                               out=tgt_m[t, :n_t])
    for i in range(3):
        tsd.tsd_verify_tev(tgt_m, tm["parent"], tm["token"], tm["n_nodes"], 1.0, seed=i)
    s.record(stream)
    for i in range(10):
        ov = tsd.tsd_verify_tev(tgt_m, tm["parent"], tm["token"], tm["n_nodes"], 1.0, seed=i)
    e.record(stream)
    torch.cuda.synchronize()
    tev_ms = s.elapsed_time(e) / 10
    out["mixture_k8_b128_x16"] = {
        "build_ms": build_ms, "build_eager_ms": build_eager_ms, "tev_ms": tev_ms,
        "rounds_per_s": nt_m / ((build_ms + tev_ms) * 1e-3),
        "mean_accept_len": float(ov["accept_len"].float().mean()),
        "mean_coverage_plus_1": float(ov["coverage"].mean()) + 1.0,
        "status_ok": int((ov["status"] == 0).sum()),
        "ms_per_tree": (build_ms + tev_ms) / nt_m}
    # the oracle beside it: tree 0's round (merged-heap build over K = 8 modes, TEV)
    zm0 = mix[0].float().cpu().numpy()
    n0 = int(tm["n_nodes"][0])
    tg0 = tgt_m[0, :n0].float().cpu().numpy()

    def mix_round(orc):
        ref = orc.build_tree(orc.drafter_lists(zm0, 1.0, 8), B_m)
        orc.tev(tg0[:ref["n_nodes"]], ref["parent"], ref["token"], ref["n_nodes"], 1.0, seed=0)

    out["mixture_k8_b128_x16"].update(
        oracle_ms_per_tree=oracle_ms(mix_round),
        oracle_sample="tree 0 of the 16 (K=8, B=128): build and TEV, float64, one host thread")
    # the same workload under the log-sum-exp score ([MFD] Eq. 6): build time,
    # and TEV at T = 1 on its trees against targets built the same way
    ws_l = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_LSE, nt_m, K_m, 16, V, 8, B_m,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    for i in range(3):
        tl = tsd.tsd_build_lse_tree(mix, topk=8, B=B_m, workspace=ws_l)
    s.record(stream)
    for i in range(10):
        tl = tsd.tsd_build_lse_tree(mix, topk=8, B=B_m, workspace=ws_l)
    e.record(stream)
    torch.cuda.synchronize()
    lse_eager_ms = s.elapsed_time(e) / 10
    lse_ms, _ = graph_latency(torch, stream, flush, cap,
                              lambda: tsd.tsd_build_lse_tree(mix, topk=8, B=B_m, workspace=ws_l))
    tgt_l = torch.zeros(nt_m, B_m + 1, V, dtype=torch.bfloat16, device=dev)
    for t in range(nt_m):
        n_t = int(tl["n_nodes"][t])
        fut = synth.mixture_drafter(1, 2, 16, V, synth.seed_for(3) + t, device=dev)[1][0, choice[t]]
        synth.target_from_rows(fut, tl["depth"][t, :n_t], 1.5, synth.seed_for(3, 500 + t),
                               out=tgt_l[t, :n_t])
    acc_l, cov_l = [], []
    for i in range(8):
        o = tsd.tsd_verify_tev(tgt_l, tl["parent"], tl["token"], tl["n_nodes"], 1.0, seed=100 + i)
        acc_l.append(float(o["accept_len"].float().mean()))
        cov_l.append(float(o["coverage"].mean()))
    acc_m = []
    for i in range(8):
        o = tsd.tsd_verify_tev(tgt_m, tm["parent"], tm["token"], tm["n_nodes"], 1.0, seed=100 + i)
        acc_m.append(float(o["accept_len"].float().mean()))
    out["mixture_lse_k8_b128_x16"] = {
        "build_ms": lse_ms, "build_eager_ms": lse_eager_ms, "max_rule_build_ms": build_ms,
        "timing": "build_ms: CUDA-graph replay, L2 flushed before each; build_eager_ms: 10 calls "
                  "back to back (host launch rate included)",
        "mean_accept_len": statistics.mean(acc_l), "max_rule_mean_accept_len": statistics.mean(acc_m),
        "mean_coverage_plus_1": statistics.mean(cov_l) + 1.0,
        "mean_candidates": float(tl["n_cand"].float().mean()),
        "status_ok": int((tl["status"] == 0).sum()),
        "ms_per_tree": lse_ms / nt_m}
    zm = mix[0].float().cpu().numpy()
    out["mixture_lse_k8_b128_x16"].update(
        oracle_ms_per_tree=oracle_ms(lambda orc: orc.lse_tree(zm, 1.0, 8, B_m)),
        oracle_sample="tree 0 of the 16 (K=8, L=16, B=128), float64, one host thread")
    return out


# [EXIT] App. D.1: verifier-stage latency reductions of TEV against
# predraw-and-follow at batch 1 (H20, Qwen3-4B target), context only
PAGES_TEV_VS_PREDRAW = {0.6: {32: -12.9, 64: -15.2, 128: -24.3}, 1.0: {32: -12.0, 64: -14.0, 128: -17.1}}


def graph_latency(torch, stream, flush, cap, fn, reps=40):
    """Median (and best) latency of fn captured in a CUDA graph and replayed,
    L2 flushed before every replay; CUDA events on the launching stream."""
    with torch.cuda.stream(cap):
        for i in range(3):
            fn()
    stream.wait_stream(cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    lat = []
    for i in range(reps + 5):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 5:
            lat.append(a.elapsed_time(b))
    del graph
    return statistics.median(lat), min(lat)


def batch1_grid(tsd, torch, synth, dev, stream, flush, cap, V):
    """The pages' batch-1 comparison ([EXIT] App. D.1): the verifier stage of
    TEV against predraw-and-follow on one tree, B in {32, 64, 128} x T in
    {0.6, 1.0}, each call captured in a CUDA graph and replayed with L2
    flushed first.  Both verifiers share the row reduction; they differ in
    the draws (one exit draw and one bonus draw, against a draw at every
    node)."""
    rows = []
    for B in (32, 64, 128):
        dr = synth.zipf_drafter(1, 16, V, synth.seed_for(1, 300 + B), device=dev)
        tr = tsd.tsd_build_tree(dr, topk=8, B=B)
        n = int(tr["n_nodes"][0])
        x = torch.zeros(1, B + 1, V, dtype=torch.bfloat16, device=dev)
        synth.target_from_rows(dr[0, 0], tr["depth"][0, :n], 1.5, synth.seed_for(1, 400 + B),
                               out=x[0, :n])
        ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 1, 1, 1, V, 1, B,
                                                torch.bfloat16), dtype=torch.uint8, device=dev)
        for T in (0.6, 1.0):
            tev = graph_latency(torch, stream, flush, cap, lambda: tsd.tsd_verify_tev(
                x, tr["parent"], tr["token"], tr["n_nodes"], T, seed=1, workspace=ws))
            pre = graph_latency(torch, stream, flush, cap, lambda: tsd.tsd_verify_ddtree(
                x, tr["parent"], tr["token"], tr["n_nodes"], T, seed=1, workspace=ws))
            rows.append({"B": B, "T": T, "tev_ms": tev[0], "tev_ms_best": tev[1],
                         "predraw_ms": pre[0], "predraw_ms_best": pre[1],
                         "tev_vs_predraw_pct": 100.0 * (tev[0] / pre[0] - 1.0),
                         "pages_pct_h20": PAGES_TEV_VS_PREDRAW[T][B],
                         "logits_mb": n * V * 2 / 1e6})
        del x, ws, tr, dr
    return {"points": rows,
            "how": "one tree, V=151936 bf16, CUDA graph replay with L2 flushed before each, "
                   "median of 40; pages_pct_h20 is [EXIT] App. D.1 on an H20 (context only)"}


def run_sweep(args):
    """TEV throughput over B x trees x T (V = 151936, bf16): one JSON table
    written to --sweep-out.  Trees come from the GPU builder on Zipf drafter
    logits; target rows are the drafter row at node depth + N(0, 1.5^2).
    Per point: 10 warm-up launches, then 50 timed ones, each bracketed by
    CUDA events (median and best reported); when the point's logits are
    under 4x the L2 size, a 2x-L2 write flushes L2 before every launch.  At
    the points with at most 8 trees the float64 oracle is timed on every
    tree, single-threaded on the host."""
    import numpy as np
    import torch

    import oracle
    import synth
    import tree_speculative_decoding_position_gb300 as tsd
    oracle.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    V, L = 151936, 16
    peak = measured_peaks()[0]
    rows = []
    for B in (16, 64, 256, 512):
        for nt in (1, 8, 64, 256):
            need = nt * (B + 1) * V * 2
            free = torch.cuda.mem_get_info(dev)[0]
            if need * 1.2 > free:
                rows.append(dict(B=B, trees=nt, skipped="needs %.1f GB, %.1f GB free" % (need / 1e9, free / 1e9)))
                continue
            seeds = [synth.seed_for(4, 1000 * B + t) for t in range(nt)]
            dr = synth.zipf_drafter(nt, L, V, 0, device=dev, seeds=seeds)
            tr = tsd.tsd_build_tree(dr, topk=8, B=B)
            x = torch.zeros(nt, B + 1, V, dtype=torch.bfloat16, device=dev)
            for t in range(nt):
                n = int(tr["n_nodes"][t])
                synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=x[t, :n])
            del dr
            ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, nt, 1, 1, V, 1, B,
                                                    torch.bfloat16), dtype=torch.uint8, device=dev)
            nbytes = int(tr["n_nodes"].sum()) * V * 2
            small = nbytes < 4 * l2
            host = None
            if nt <= 8:  # the oracle's inputs, copied once
                host = [(x[t, :int(tr["n_nodes"][t])].float().cpu().numpy().astype(np.float64),
                         tr["parent"][t].cpu().numpy(), tr["token"][t].cpu().numpy(),
                         int(tr["n_nodes"][t])) for t in range(nt)]
            for T in (0.0, 0.6, 1.0):
                for i in range(10):
                    tsd.tsd_verify_tev(x, tr["parent"], tr["token"], tr["n_nodes"], T, seed=i,
                                       workspace=ws, with_masses=False)
                evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(50)]
                for ev in evs:
                    for e_ in ev:
                        e_.record(stream)
                torch.cuda.synchronize()
                for i in range(50):
                    if small:
                        flush.fill_(float(i))
                    tsd.tsd_verify_tev_timed(x, tr["parent"], tr["token"], tr["n_nodes"], T,
                                             seed=i, stage_events=evs[i], workspace=ws,
                                             with_masses=False)
                torch.cuda.synchronize()
                tot = [ev[0].elapsed_time(ev[4]) for ev in evs]
                rk = [ev[1].elapsed_time(ev[2]) for ev in evs]
                med, best, rmed = statistics.median(tot), min(tot), statistics.median(rk)
                pt = dict(B=B, trees=nt, T=T, tev_ms=med, tev_ms_best=best,
                          rounds_per_s=nt / (med * 1e-3), rounds_per_s_best=nt / (best * 1e-3),
                          rows_kernel_ms=rmed, rows_kernel_gbs=nbytes / (rmed * 1e-3) / 1e9,
                          rows_frac_of_measured=nbytes / (rmed * 1e-3) / 1e9 / peak,
                          logits_gb=nbytes / 1e9, launches=50,
                          l2="flushed before each launch" if small else "inputs >= 4x L2")
                if host is not None:
                    t0 = time.perf_counter()
                    for t, (z, par, tok, n) in enumerate(host):
                        oracle.tev(z, par, tok, n, T, seed=0, tree=t)
                    o_s = time.perf_counter() - t0
                    pt.update(oracle_ms_per_tree=1e3 * o_s / nt, oracle_rounds_per_s=nt / o_s,
                              oracle_threads=1, gpu_over_oracle=(nt / (med * 1e-3)) / (nt / o_s))
                rows.append(pt)
            del x, ws, tr, host
            torch.cuda.empty_cache()
    with open(args.sweep_out, "w") as f:
        json.dump(rows, f, indent=1)
    print(json.dumps({"sweep_points": len(rows), "out": args.sweep_out}))


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_round(oracle, z, tg, k, B, T, t, seed=0, keep_lists=False):
    """One round of the workload in the float64 oracle: drafter statistics and
    heap, mask, TEV.  z: [L, V] drafter logits, tg: [n, V] target rows.
    Returns the oracle's tree and TEV result (and the drafter lists)."""
    lists = oracle.drafter_lists(z, 1.0, k)
    ref = oracle.build_tree(lists, B)
    oracle.tree_mask(ref["parent"], ref["n_nodes"], B, 1024)
    o = oracle.tev(tg, ref["parent"], ref["token"], ref["n_nodes"], T, seed=seed, tree=t)
    return (ref, o, lists) if keep_lists else (ref, o)


SCORE_TOL = 1e-6   # builder order may differ only between prefixes this close (relative)
FLIP_TOL = 1e-6    # a draw may differ only where the CDF is this close to u * total


def _prefix_score(seq, lists):
    """float64 score of a token sequence in the one-mode capped universe
    (path sum of z / T_d minus the summed log-normalisers), None outside it."""
    import numpy as np
    z, c = 0.0, 0.0
    for j, x in enumerate(seq):
        hit = np.nonzero(lists["top_id"][0, j] == x)[0]
        if hit.size == 0:
            return None
        z += lists["top_zt"][0, j, hit[0]]
        c += lists["lse"][0, j]
    return z - c


def _sequences(parent, token, n):
    seqs = [()]
    for u in range(1, n):
        seqs.append(seqs[int(parent[u])] + (int(token[u]),))
    return seqs


def builder_flips(ref, lists, par, tok, n):
    """Node-by-node comparison of a GPU tree with the oracle's: the number of
    positions whose prefixes differ, each allowed only between prefixes whose
    float64 scores are within SCORE_TOL; None if any difference is not such a
    near-tie (a builder error)."""
    if n != ref["n_nodes"]:
        return None
    sg, so = _sequences(par, tok, n), _sequences(ref["parent"], ref["token"], n)
    flips = 0
    for a, b in zip(sg, so):
        if a == b:
            continue
        sa, sb = _prefix_score(a, lists), _prefix_score(b, lists)
        if sa is None or sb is None or abs(sa - sb) > SCORE_TOL * max(1.0, abs(sb)):
            return None
        flips += 1
    return flips


def _draw_flip(got, want, masses, u):
    """0 if the two inverse-CDF draws agree, 1 if they differ only across a
    CDF boundary within FLIP_TOL of u * total, None otherwise."""
    import numpy as np
    if got == want:
        return 0
    if got < 0 or want < 0:
        return None
    cum = np.cumsum(np.asarray(masses, dtype=np.float64))
    lo, hi = min(got, want), max(got, want)
    if hi >= cum.size:
        return None
    ok = abs(cum[lo] - u * cum[-1]) <= FLIP_TOL * cum[-1] and \
        cum[hi - 1] - cum[lo] <= FLIP_TOL * cum[-1]
    return 1 if ok else None


def agreement(oracle, ref, lists, tg, tree, out, t, T, seed):
    """The GPU's tree t and its TEV outputs against the float64 oracle, for
    the benchmark line.  The builder: node by node, near-tie flips counted
    (builder_flips).  TEV: the oracle's TEV on the GPU's own tree and target
    rows, against the GPU's exit node, bonus token and accepted length (exact
    up to counted near-boundary draw flips) and exit masses (largest relative
    error; values below 1e-30 compared absolutely).  Returns a dict."""
    import numpy as np
    n = int(tree["n_nodes"][t])
    par = tree["parent"][t, :n].cpu().numpy()
    tok = tree["token"][t, :n].cpu().numpy()
    bf = builder_flips(ref, lists, par, tok, n)
    o = oracle.tev(tg[:n], par, tok, n, T, seed=seed, tree=t)
    ex, by = int(out["exit_node"][t]), int(out["bonus_token"][t])
    df = _draw_flip(ex, o["exit_node"], o["w"], o["u_exit"])
    if df == 0:
        p = oracle.row_probs(tg[ex].astype(np.float64), T)
        p[[int(tok[u]) for u in range(1, n) if int(par[u]) == ex]] = 0.0
        bflip = _draw_flip(by, o["bonus"], p, o["u_bonus"])
        df = None if bflip is None else bflip
        if df is not None and int(out["accept_len"][t]) != o["accept_len"]:
            df = None
    w = out["exit_mass"][t, :n].double().cpu().numpy()
    err = np.abs(w - o["w"]) / np.maximum(np.abs(o["w"]), 1e-30)
    small = np.abs(o["w"]) < 1e-30
    err[small] = np.abs(w - o["w"])[small]
    return {"builder_flips": bf, "draw_flips": df, "err": float(err.max())}


def cpu_baseline(drafter, target, tree, k, B, T, budget_s=8.0, out=None, seed=0):
    """The float64 oracle as it stands on the host, on a bounded sample of the
    same workload (whole rounds: drafter statistics, heap, mask, TEV): first
    single-threaded, then with one thread per host core over trees (the
    oracle's C code runs outside the interpreter lock).  About budget_s
    seconds each.  The single-threaded rounds use the timed step's last seed,
    and their results are compared, outside the timing, with that step's GPU
    outputs `out` on the same trees."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.build()
    nt = drafter.shape[0]
    inputs = []
    for t in range(nt):
        n = int(tree["n_nodes"][t])
        inputs.append((drafter[t, 0].float().cpu().numpy(), target[t, :n].float().cpu().numpy()))
    done, spent = 0, 0.0
    same_tree, builder_err, flips_b, flips_d, draw_err, max_err = 0, 0, 0, 0, 0, 0.0
    for t in range(nt):
        t0 = time.perf_counter()
        ref, o, lists = oracle_round(oracle, *inputs[t], k, B, T, t, seed=seed, keep_lists=True)
        spent += time.perf_counter() - t0
        done += 1
        if out is not None:  # outside the timing
            a = agreement(oracle, ref, lists, inputs[t][1], tree, out, t, T, seed)
            if a["builder_flips"] is None:
                builder_err += 1
            else:
                same_tree += a["builder_flips"] == 0
                flips_b += a["builder_flips"]
            if a["draw_flips"] is None:
                draw_err += 1
            else:
                flips_d += a["draw_flips"]
            max_err = max(max_err, a["err"])
        if spent >= budget_s and done >= 2:
            break
    single = {"value": done / spent, "cores": 1,
              "sample": "%d of the %d trees of one step, %.1f s" % (done, nt, spent)}
    agree = None
    if out is not None:
        agree = {"trees": done, "same_tree": same_tree, "builder_mismatch": builder_err,
                 "builder_flips": flips_b, "draw_mismatch": draw_err, "draw_flips": flips_d,
                 "max_rel_err_exit_mass": max_err,
                 "note": "the first trees of the timed step's last call: the oracle's float64 "
                         "build against the GPU's tree node by node (flips = positions that "
                         "differ between prefixes whose oracle scores are within 1e-6), and the "
                         "oracle's TEV on the GPU's tree with that call's seed against its "
                         "outputs (flips = draws that differ across a CDF boundary within 1e-6 "
                         "of u * total)"}
    nth = host_threads()
    n_rounds = max(nth, int(round(budget_s * single["value"] * nth)))
    with ThreadPoolExecutor(max_workers=nth) as pool:
        t0 = time.perf_counter()
        list(pool.map(lambda t: oracle_round(oracle, *inputs[t % nt], k, B, T, t), range(n_rounds)))
        wall = time.perf_counter() - t0
    return {"value": n_rounds / wall, "unit": "rounds/s", "cores": nth, "kind": "oracle",
            "sample": "%d rounds over the workload's %d trees (build + mask + TEV per tree), "
                      "float64, %d threads over trees, %.1f s wall" % (n_rounds, nt, nth, wall),
            "single_thread": single, "agreement_with_gpu": agree}


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import numpy as np
    import torch

    import oracle
    import synth
    oracle.build()
    W = WORKLOAD
    nt, V, L, k, B, T = W["trees_per_gpu"], W["V"], W["L"], W["topk"], W["B"], W["temperature"]

    cache = {}

    def inputs(t):
        """Synthetic inputs of tree t (generated once, outside the timing)."""
        if t not in cache:
            seed = synth.seed_for(2, t)
            dr = synth.zipf_drafter(1, L, V, 0, device="cpu", seeds=[seed])[0, 0]
            ref = oracle.build_tree(oracle.drafter_lists(dr.float().numpy(), 1.0, k), B)
            n = ref["n_nodes"]
            tg = synth.target_from_rows(dr, ref["depth"][:n], 1.5, seed + 1).float().numpy()
            cache[t] = (dr.float().numpy(), tg)
        return cache[t]

    from concurrent.futures import ThreadPoolExecutor
    nth = host_threads()
    for t in range(4):
        inputs(t)  # generated before any timing

    def step(i):
        """One step: `nth` rounds of the workload, one tree per host thread."""
        t0 = time.perf_counter()
        list(pool.map(lambda j: oracle_round(oracle, *inputs((i * nth + j) % 4), k, B, T, j),
                      range(nth)))
        return time.perf_counter() - t0

    with ThreadPoolExecutor(max_workers=nth) as pool:
        for i in range(args.warmup):
            step(i)
        spent = sum(step(args.warmup + i) for i in range(args.steps))
    value = args.steps * nth / spent
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rounds/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(W, parallelism="host cores: %d threads, one tree each per step" % nth),
        "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": nth, "kind": "oracle",
                         "sample": "%d trees per step, one per host thread (build + mask + TEV; "
                                   "four trees' inputs in rotation), float64 oracle" % nth},
        "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _op_setup(name, tsd, torch, synth, dev):
    """The workload of one secondary operation, as the extras time it; returns
    a callable that issues one call."""
    V = WORKLOAD["V"]
    if name in ("tev_b64", "build_b64"):
        # the batch-1 round: one tree, L=16, top-k 8, B=64, TEV at T=1
        dr = synth.zipf_drafter(1, 16, V, synth.seed_for(1), device=dev)
        t1 = tsd.tsd_build_tree(dr, topk=8, B=64)
        n = int(t1["n_nodes"][0])
        x = torch.zeros(1, 65, V, dtype=torch.bfloat16, device=dev)
        synth.target_from_rows(dr[0, 0], t1["depth"][0, :n], 1.5, synth.seed_for(1, 1), out=x[0, :n])
        wv = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 1, 1, 1, V, 1, 64,
                                                torch.bfloat16), dtype=torch.uint8, device=dev)
        wb = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 1, 1, 16, V, 8, 64,
                                                torch.bfloat16), dtype=torch.uint8, device=dev)
        if name == "build_b64":
            return lambda: tsd.tsd_build_tree(dr, topk=8, B=64, workspace=wb)
        return lambda: tsd.tsd_verify_tev(x, t1["parent"], t1["token"], t1["n_nodes"], 1.0, seed=1,
                                          workspace=wv)
    if name in ("build_lse", "build_mixture"):
        mix, _, _ = synth.mixture_drafter(16, 8, 16, V, synth.seed_for(3), device=dev)
        op = tsd.TSD_OP_BUILD_LSE if name == "build_lse" else tsd.TSD_OP_BUILD_TREE
        ws = torch.empty(tsd.tsd_workspace_size(op, 16, 8, 16, V, 8, 128, torch.bfloat16),
                         dtype=torch.uint8, device=dev)
        if name == "build_lse":
            return lambda: tsd.tsd_build_lse_tree(mix, topk=8, B=128, workspace=ws)
        return lambda: tsd.tsd_build_tree(mix, topk=8, B=128, workspace=ws)
    nt, L, k, B = WORKLOAD["trees_per_gpu"], WORKLOAD["L"], WORKLOAD["topk"], WORKLOAD["B"]
    drafter = synth.zipf_drafter(nt, L, V, 0, device=dev,
                                 seeds=[synth.seed_for(2, t) for t in range(nt)])
    if name == "build_forest":
        ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_FOREST, nt, 1, L, V, k, B,
                                                torch.bfloat16), dtype=torch.uint8, device=dev)
        return lambda: tsd.tsd_build_forest(drafter, topk=k, B=B, M_max=nt * B, l0=1.0,
                                            c1=1.0 / 2048, workspace=ws)
    tr = tsd.tsd_build_tree(drafter, topk=k, B=B)
    if name.startswith("verify_"):
        # the workload's verification: its 32 trees, targets as the step's
        T = WORKLOAD["temperature"]
        target = torch.zeros(nt, B + 1, V, dtype=torch.bfloat16, device=dev)
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            synth.target_from_rows(drafter[t, 0], tr["depth"][t, :n], 1.5, synth.seed_for(2, t) + 1,
                                   out=target[t, :n])
        wv = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, nt, 1, 1, V, 1, B,
                                                torch.bfloat16), dtype=torch.uint8, device=dev)
        args = (target, tr["parent"], tr["token"], tr["n_nodes"], T)
        if name == "verify_tev":
            return lambda: tsd.tsd_verify_tev(*args, seed=1, workspace=wv)
        if name == "verify_seqres":
            return lambda: tsd.tsd_verify_seqres(*args, seed=1, workspace=wv)
        if name == "verify_ddtree":
            return lambda: tsd.tsd_verify_ddtree(*args, seed=1, workspace=wv)
        d = tr["depth"].clamp(min=1).long() - 1
        logq = torch.log_softmax(drafter[:, 0].float(), dim=-1)
        q = torch.stack([logq[t, d[t], tr["token"][t].clamp(min=0).long()].exp()
                         for t in range(nt)]).float().contiguous()
        del logq
        return lambda: tsd.tsd_verify_proposal(target, tr["parent"], tr["token"], tr["n_nodes"], q,
                                               T, seed=1, workspace=wv)
    w = torch.rand(nt, B + 1, generator=torch.Generator(device=dev).manual_seed(5),
                   device=dev) * (tr["depth"] >= 0)
    ws = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_EXIT_LOSS, nt, 1, L, V, 1, B,
                                            torch.bfloat16), dtype=torch.uint8, device=dev)
    grad = name == "exit_loss_grad"
    return lambda: tsd.tsd_exit_loss(drafter, tr["token"], tr["depth"], tr["n_nodes"], w,
                                     with_grad=grad, workspace=ws)


OPS = ("build_lse", "build_mixture", "build_forest", "exit_loss", "exit_loss_grad", "tev_b64",
       "build_b64", "verify_tev", "verify_seqres", "verify_proposal", "verify_ddtree")


def run_op(args):
    import torch

    import synth
    import tree_speculative_decoding_position_gb300 as tsd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    tsd.load()
    fn = _op_setup(args.op, tsd, torch, synth, dev)
    for i in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for i in range(args.steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    print(json.dumps({"op": args.op, "calls": args.steps, "ms_per_call": s.elapsed_time(e) / args.steps}),
          flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trees", type=int, default=0,
                    help="trees per GPU (default: the workload's 32); for profiler captures")
    ap.add_argument("--sweep", action="store_true",
                    help="time TEV over B x trees x T instead (writes --sweep-out)")
    ap.add_argument("--sweep-out", default="sweep.json")
    ap.add_argument("--op", choices=sorted(OPS), default=None,
                    help="run one secondary operation alone on its workload (for profiler "
                         "captures): warm-up calls, then --steps timed calls")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.op:
        run_op(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

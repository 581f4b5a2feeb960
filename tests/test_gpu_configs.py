"""GPU parity on the rest of the workload grid: the builder and TEV against the
float64 oracle at the full Qwen-size vocabulary (V = 151936, L = 16, top-k 8,
bf16), in the launches the benchmark and the throughput sweep run.

* the mixture-of-futures workload: 16 trees, K = 8 modes from two latent
  futures, B = 128 ([MFD] App. B "Merged heap"), TEV at T = 1;
* the batched workload at T = 1 (32 trees, B = 256);
* the sweep's budgets B = 16 and B = 512 at 1 and 8 trees, T in {0, 0.6, 1};
* the sweep's large launches: 64 and 256 trees at B = 64, 256 trees at
  B = 16, 64 trees at B = 256.

In every launch the builder's sampled trees are compared with the oracle's
node by node, TEV's outputs on sampled trees with the oracle's TEV on the same
tree and logits ([EXIT] App. B; masses within 1e-5 relative, draws exact up to
counted near-boundary flips), and every tree of the launch is checked for
validity (status, sum of exit masses, exit node, accepted length, bonus token
not a drafted child).  Flips are counted and reported in the test summary.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_batch_valid, check_tev, compare_trees, oracle_build, to_np, tree_np

pytestmark = pytest.mark.gpu

V_Q = synth.V_QWEN


@pytest.fixture(scope="module")
def tsd():
    import tree_speculative_decoding_position_gb300 as m
    from tree_speculative_decoding_position_gb300 import build
    build.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _zipf_launch(tsd, dev, cfg, nt, B):
    """cfg's Zipf drafter for nt trees, the GPU trees, and target rows at the
    nodes' depths (drafter row + N(0, 1.5^2)), as the benchmark builds them."""
    seeds = [synth.seed_for(cfg, 100 * B + t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, V_Q, 0, device=dev, seeds=seeds)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B)
    x = torch.zeros(nt, B + 1, V_Q, dtype=torch.bfloat16, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=x[t, :n])
    return dr, tr, x


def _check_launch(tsd, orc, dr, tr, x, B, temps, sample, seed0):
    """Builder parity on the sampled trees, then TEV at each temperature:
    whole-launch validity and oracle parity on the sampled trees.  Returns
    (builder flips, draw flips)."""
    nt = x.shape[0]
    assert to_np(tr["status"]).tolist() == [0] * nt
    bflips = 0
    for t in sample:
        ref, lists = oracle_build(orc, dr[t], 8, B)
        bflips += compare_trees(tree_np(tr, t), ref, lists)
    host = {}
    for t in sample:
        n = int(tr["n_nodes"][t])
        host[t] = (x[t, :n].float().cpu().numpy().astype(np.float64), to_np(tr["parent"][t]),
                   to_np(tr["token"][t]), n)
    dflips = 0
    for i, T in enumerate(temps):
        seed = seed0 + i
        out = tsd.tsd_verify_tev(x, tr["parent"], tr["token"], tr["n_nodes"], T, seed=seed)
        check_batch_valid(out, tr, T)
        for t in sample:
            z64, par, tok, n = host[t]
            o = orc.tev(z64, par, tok, n, T, seed=seed, tree=t)
            dflips += check_tev(out, t, o, z64, par, tok, n, T)
    return bflips, dflips


def test_mixture_workload_build_and_tev(tsd, dev, orc, flip_log):
    """The mixture-of-futures workload as the benchmark launches it: 16 trees,
    K = 8 modes, B = 128, one build call (merged heap, best-mode score), then
    TEV at T = 1 on targets that follow the future each tree's seed chose.
    Four sampled trees against the oracle's merged-heap build and TEV."""
    nt, K, B = 16, 8, 128
    mix, futures, choice = synth.mixture_drafter(nt, K, 16, V_Q, synth.seed_for(3), device=dev)
    tr = tsd.tsd_build_tree(mix, topk=8, B=B)
    x = torch.zeros(nt, B + 1, V_Q, dtype=torch.bfloat16, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(futures[t, choice[t]], tr["depth"][t, :n], 1.5,
                               synth.seed_for(3, 500 + t), out=x[t, :n])
    bf, df = _check_launch(tsd, orc, mix, tr, x, B, (1.0,), (0, 5, 10, 15), 40)
    flip_log("builder", bf)
    flip_log("draw", df)
    assert bf <= 2 and df <= 1, (bf, df)


def test_batched_workload_at_t1(tsd, dev, orc, flip_log):
    """The batched workload's launch (32 trees, B = 256) at T = 1: four sampled
    trees against the oracle, every tree valid."""
    dr, tr, x = _zipf_launch(tsd, dev, 2, 32, 256)
    bf, df = _check_launch(tsd, orc, dr, tr, x, 256, (1.0,), (0, 11, 20, 31), 61)
    flip_log("builder", bf)
    flip_log("draw", df)
    assert bf <= 2 and df <= 1, (bf, df)


@pytest.mark.parametrize("B", [16, 512])
@pytest.mark.parametrize("nt", [1, 8])
def test_sweep_budgets(tsd, dev, orc, flip_log, B, nt):
    """The sweep's smallest and largest budgets, one tree and eight trees per
    launch, at T = 0, 0.6 and 1: the builder and TEV on sampled trees against
    the oracle."""
    dr, tr, x = _zipf_launch(tsd, dev, 4, nt, B)
    sample = (0,) if nt == 1 else (0, 3, 7)
    bf, df = _check_launch(tsd, orc, dr, tr, x, B, (0.0, 0.6, 1.0), sample, 71)
    flip_log("builder", bf)
    flip_log("draw", df)
    assert bf <= 2 and df <= 2, (bf, df)


@pytest.mark.parametrize("nt,B,temps", [(64, 64, (0.6,)), (256, 64, (0.0, 1.0)),
                                         (256, 16, (0.6,)), (64, 256, (1.0,))])
def test_sweep_large_launches(tsd, dev, orc, flip_log, nt, B, temps):
    """The sweep's large launches (64 and 256 trees per call): every tree
    valid, and two sampled trees (the first and the last) against the oracle's
    build and TEV."""
    dr, tr, x = _zipf_launch(tsd, dev, 5, nt, B)
    bf, df = _check_launch(tsd, orc, dr, tr, x, B, temps, (0, nt - 1), 81)
    flip_log("builder", bf)
    flip_log("draw", df)
    assert bf <= 2 and df <= 1, (bf, df)

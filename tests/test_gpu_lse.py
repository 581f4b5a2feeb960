"""GPU parity of the mixture tree under the log-sum-exp score ([MFD] App. B
"Max or log-sum-exp", Eq. 6) against the oracle on the same seeded inputs.

The per-mode lists are decided by float64 path sums of z/T on both sides, bit
for bit, so the candidate count matches exactly.  The GPU sums the modes'
exp terms in fp32 (the oracle in float64), so two prefixes may swap only when
their float64 mixture scores differ by at most SCORE_TOL relative (floor 1)."""
import numpy as np
import pytest
import scipy.special
import torch

import synth
from gpu_helpers import SCORE_TOL, compare_trees, sequences

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


def _lse_score(seq, z, lse, lp, T):
    a = [lp[m] + sum(z[m, j, x] / T for j, x in enumerate(seq)) - sum(lse[m, :len(seq)])
         for m in range(z.shape[0])]
    return float(scipy.special.logsumexp(a))


def _compare(out, t, ref, z, T, k, lp):
    """Returns the number of order swaps (each between near-equal scores)."""
    n_g, n_o = int(out["n_nodes"][t]), ref["n_nodes"]
    assert n_g == n_o, ("node count", n_g, n_o)
    par = out["parent"][t].cpu().numpy()
    tok = out["token"][t].cpu().numpy()
    sg, so = sequences(par, tok, n_g), sequences(ref["parent"], ref["token"], n_o)
    for u in range(1, n_g):
        assert 0 <= par[u] < u
    if sg == so:
        got = out["score"][t].cpu().numpy()[1:n_g].astype(np.float64)
        want = ref["score"][1:n_o]
        assert np.all(np.abs(got - want) <= SCORE_TOL * np.maximum(1.0, np.abs(want)))
        assert np.array_equal(out["depth"][t].cpu().numpy()[:n_g], ref["depth"][:n_o])
        return 0
    lse = __import__("oracle").drafter_lists(z, T, k)["lse"]
    lpv = np.full(z.shape[0], -np.log(z.shape[0])) if lp is None else lp
    flips = 0
    for i in range(1, n_g):
        if sg[i] == so[i]:
            continue
        a, b = _lse_score(sg[i], z, lse, lpv, T), _lse_score(so[i], z, lse, lpv, T)
        assert abs(a - b) <= SCORE_TOL * max(1.0, abs(b)), ("order", i, sg[i], so[i], a, b)
        flips += 1
    return flips


@pytest.mark.parametrize("case", ["bf16_qwen_k4", "fp32_misaligned_prior", "mixture_k8_b128"])
def test_lse_tree_matches_oracle(tsd, dev, orc, case):
    T = 1.0
    if case == "bf16_qwen_k4":
        nt, K, L, V, k, B, dtype, prior = 3, 4, 6, V_Q, 8, 64, torch.bfloat16, False
    elif case == "fp32_misaligned_prior":
        nt, K, L, V, k, B, dtype, prior, T = 2, 8, 5, 4099, 4, 128, torch.float32, True, 0.8
    else:  # the bench's launch: 16 trees, three of them sampled
        nt, K, L, V, k, B, dtype, prior = 16, 8, 16, V_Q, 8, 128, torch.bfloat16, False
    dr, _, _ = synth.mixture_drafter(nt, K, L, V, synth.seed_for(11, K), dtype=dtype)
    lp = None
    if prior:
        g = torch.Generator().manual_seed(synth.seed_for(11, 99))
        lp = torch.randn(nt, K, generator=g).float()
    out = tsd.tsd_build_lse_tree(dr.to(dev), topk=k, B=B, drafter_temp=T,
                                 log_prior=None if lp is None else lp.to(dev))
    assert out["status"].cpu().tolist() == [0] * nt
    flips = 0
    for t in (range(nt) if nt <= 4 else (0, 7, 15)):
        z = dr[t].double().numpy()
        lpt = None if lp is None else lp[t].double().numpy()
        ref = orc.lse_tree(z, T, k, B, log_prior=lpt)
        assert int(out["n_cand"][t]) == ref["n_cand"]
        flips += _compare(out, t, ref, z, T, k, lpt)
    assert flips <= 4


def test_lse_tree_one_mode(tsd, dev, orc):
    """K = 1: the key is log Q exactly (no fp32 sum), so the tree equals the
    oracle's node for node, and DDTree's builder tree up to exact ties."""
    nt, L, k, B = 3, 8, 8, 200
    dr = synth.zipf_drafter(nt, L, V_Q, synth.seed_for(12), device="cpu")
    out = tsd.tsd_build_lse_tree(dr.to(dev), topk=k, B=B)
    bt = tsd.tsd_build_tree(dr.to(dev), topk=k, B=B)
    for t in range(nt):
        z = dr[t].double().numpy()
        ref = orc.lse_tree(z, 1.0, k, B)
        assert _compare(out, t, ref, z, 1.0, k, None) == 0
        lists = orc.drafter_lists(z, 1.0, k)
        got = {key: out[key][t].cpu().numpy() for key in ("parent", "token", "depth", "score")}
        got["n_nodes"] = int(out["n_nodes"][t])
        bld = {key: bt[key][t].cpu().numpy() for key in ("parent", "token", "depth", "score")}
        bld["n_nodes"] = int(bt["n_nodes"][t])
        compare_trees(got, bld, lists)  # swaps only between exactly tied prefixes


def test_lse_tree_edges(tsd, dev, orc):
    # a small universe: two finite tokens per row, every candidate taken
    z = torch.full((1, 2, 3, 64), -float("inf"))
    z[0, 0, :, :2] = torch.tensor([1.0, 0.5])
    z[0, 1, :, 1:3] = torch.tensor([0.7, 0.2])
    out = tsd.tsd_build_lse_tree(z.to(dev), topk=4, B=100)
    ref = orc.lse_tree(z[0].double().numpy(), 1.0, 4, 100)
    assert int(out["n_cand"][0]) == ref["n_cand"] and int(out["n_nodes"][0]) == ref["n_cand"] + 1
    # constant rows make many prefixes tie exactly under s_lse; the fp32 and
    # float64 sums break those ties differently, each swap checked in _compare
    assert _compare(out, 0, ref, z[0].double().numpy(), 1.0, 4, None) <= 8
    # a non-finite row fails its tree only; B = 0 is the root alone
    z = torch.randn(2, 3, 4, 32)
    z[1, 2, 1, 5] = float("nan")
    out = tsd.tsd_build_lse_tree(z.to(dev), topk=4, B=8)
    assert out["status"].cpu().tolist() == [0, 5]
    assert int(out["n_nodes"][1]) == 0 and int(out["n_nodes"][0]) == 9
    assert torch.all(out["parent"][1] == -1)
    out = tsd.tsd_build_lse_tree(z[:1].to(dev), topk=4, B=0)
    assert int(out["n_nodes"][0]) == 1 and int(out["status"][0]) == 0
    # sizes past the limits are refused on the host
    with pytest.raises(tsd.TsdError):
        tsd.tsd_build_lse_tree(torch.zeros(1, 8, 2, 64, device=dev), topk=4, B=600)
    with pytest.raises(tsd.TsdError):
        tsd.tsd_build_lse_tree(torch.zeros(1, 1, 2, 64, device=dev), topk=4, B=2049)


def test_lse_tree_large_budget_from_pinned_host(tsd, dev, orc):
    """B = 1024 with two modes: several entries per thread in the dedupe and a
    4096-entry sort per depth; the logits are read from page-locked host
    memory, and the result equals the device-resident one."""
    nt, K, L, V, k, B = 2, 2, 4, 5000, 8, 1024
    dr, _, _ = synth.mixture_drafter(nt, K, L, V, synth.seed_for(13), dtype=torch.float32)
    host = dr.pin_memory()
    out = tsd.tsd_build_lse_tree(host, topk=k, B=B, device=dev)
    same = tsd.tsd_build_lse_tree(dr.to(dev), topk=k, B=B)
    torch.cuda.synchronize()
    for key in ("parent", "token", "depth", "score", "n_nodes", "n_cand"):
        assert torch.equal(out[key], same[key]), key
    flips = 0
    for t in range(nt):
        z = dr[t].double().numpy()
        ref = orc.lse_tree(z, 1.0, k, B)
        assert int(out["n_cand"][t]) == ref["n_cand"]
        flips += _compare(out, t, ref, z, 1.0, k, None)
    assert flips <= 4


@pytest.mark.parametrize("case", ["k8_b128_l11", "k3_b100_l28", "k8_b256_l12", "k4_b64_l1"])
def test_lse_tree_merge_groups(tsd, dev, orc, case):
    """The selection runs on a pair of CTAs per tree, each merging half the
    depths in groups of kGroupSlots / (2 K B): a last group shorter than the
    others (K = 8, B = 128, L = 11), a K B that does not divide the table
    (K = 3, B = 100, L = 28), candidates too many for shared memory, kept in
    the workspace (K = 8, B = 256, L = 12: 24576 entries, groups of 4
    depths), and one depth, the second CTA holding none (L = 1)."""
    if case == "k8_b128_l11":
        nt, K, L, V, k, B = 2, 8, 11, 3000, 8, 128
    elif case == "k3_b100_l28":
        nt, K, L, V, k, B = 2, 3, 28, 2000, 4, 100  # L ceil(log2 k) <= 56
    elif case == "k8_b256_l12":
        nt, K, L, V, k, B = 2, 8, 12, 3000, 8, 256
    else:
        nt, K, L, V, k, B = 3, 4, 1, 500, 8, 64
    dr, _, _ = synth.mixture_drafter(nt, K, L, V, synth.seed_for(14, K), dtype=torch.float32)
    out = tsd.tsd_build_lse_tree(dr.to(dev), topk=k, B=B)
    assert out["status"].cpu().tolist() == [0] * nt
    flips = 0
    for t in range(nt):
        z = dr[t].double().numpy()
        ref = orc.lse_tree(z, 1.0, k, B)
        assert int(out["n_cand"][t]) == ref["n_cand"]
        flips += _compare(out, t, ref, z, 1.0, k, None)
    assert flips <= 4

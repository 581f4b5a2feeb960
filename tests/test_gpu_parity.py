"""GPU parity: the CUDA library (through the C ABI binding) against the
float64 oracle on the same seeded inputs, element by element.

Sizes: the tiny configuration (V=32, L=4, k=4, B=8); a mid-size vocabulary
that spans several 8 KB chunks plus a ragged tail; and the full Qwen-size
vocabulary V=151936 with B=64 (one tree) and B=256 (32 trees, sampled trees
checked against the oracle one by one).  Tolerances live in gpu_helpers.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_draw, check_tev as _check_tev, compare_trees
from gpu_helpers import oracle_build, to_np as _np, tree_np as _tree_np

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


# ---------------------------------------------------------------------------
# builder
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_build_tiny(tsd, dev, orc, seed):
    dr = synth.tiny_drafter(synth.seed_for(0, seed))
    out = tsd.tsd_build_tree(dr[None, None].to(dev), topk=4, B=8)
    ref, lists = oracle_build(orc, dr[None], 4, 8)
    g = _tree_np(out)
    assert int(out["status"][0]) == 0
    assert compare_trees(g, ref, lists) == 0
    n = g["n_nodes"]
    assert np.array_equal(g["rank"][:n], ref["rank"][:n])
    assert np.array_equal(g["mode"][:n], ref["mode"][:n])
    assert np.all(g["parent"][n:] == -1) and np.all(np.isneginf(g["score"][n:]))


@pytest.mark.parametrize("V,B,k,temp", [(12805, 64, 8, 1.0), (4096 * 3, 200, 8, 0.7),
                                         (1001, 40, 5, 1.0), (V_Q, 64, 8, 1.0)])
def test_build_single_mode(tsd, dev, orc, flip_log, V, B, k, temp):
    dr = synth.zipf_drafter(1, 16, V, synth.seed_for(1), device="cpu")  # [1, 1, 16, V] bf16
    out = tsd.tsd_build_tree(dr.to(dev), topk=k, B=B, drafter_temp=temp)
    ref, lists = oracle_build(orc, dr[0], k, B, temp)
    flips = compare_trees(_tree_np(out), ref, lists)
    flip_log("builder", flips)
    assert flips <= 2, flips


def test_build_batched_b256(tsd, dev, orc, flip_log):
    """The bench's launch: 32 trees, V=151936, L=16, top-k 8, B=256, one call;
    every tree prefix-closed with falling scores, four sampled trees against
    the oracle node by node."""
    nt, B = 32, 256
    seeds = [synth.seed_for(2, t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, V_Q, 0, device=dev, seeds=seeds)
    out = tsd.tsd_build_tree(dr, topk=8, B=B)
    assert _np(out["status"]).tolist() == [0] * nt
    assert _np(out["n_nodes"]).tolist() == [B + 1] * nt
    par, sc = _np(out["parent"]), _np(out["score"])
    for t in range(nt):
        assert np.all((par[t, 1:] >= 0) & (par[t, 1:] < np.arange(1, B + 1)))
        assert np.all(sc[t, 1:] <= sc[t, par[t, 1:]] + 1e-6)
    flips = 0
    for t in (0, 7, 19, 31):
        ref, lists = oracle_build(orc, dr[t].cpu(), 8, B)
        flips += compare_trees(_tree_np(out, t), ref, lists)
    flip_log("builder", flips)
    assert flips <= 2, flips


@pytest.mark.parametrize("B", [99, 100, 127, 128, 129])
def test_build_crowded_bound(tsd, dev, orc, flip_log, B):
    """A drafter whose best prefixes crowd the B-th score (an exact tie
    between two depth-4 prefixes at places 98 and 99, many candidates just
    below): once the taken list holds B prefixes the frontier must stay
    within its buffer.  Before the frontier was capped at K*B entries there,
    these budgets overflowed it and the tree came back empty (status 5)."""
    dr = synth.zipf_drafter(1, 16, V_Q, 0, device=dev, seeds=[synth.seed_for(4, 127000)])
    out = tsd.tsd_build_tree(dr, topk=8, B=B)
    assert int(out["status"][0]) == 0 and int(out["n_nodes"][0]) == B + 1
    ref, lists = oracle_build(orc, dr[0].cpu(), 8, B)
    flips = compare_trees(_tree_np(out), ref, lists)
    flip_log("builder", flips)
    assert flips <= 1, flips


def test_build_budget_sweep(tsd, dev, orc):
    """Every budget from 90 to 140 on four drafters, one call per budget with
    the four trees: each tree full (B+1 nodes, status 0) and the first of
    them equal to the oracle's."""
    seeds = [synth.seed_for(4, 127000)] + [synth.seed_for(8, t) for t in range(3)]
    dr = synth.zipf_drafter(4, 16, V_Q, 0, device=dev, seeds=seeds)
    for B in range(90, 141):
        out = tsd.tsd_build_tree(dr, topk=8, B=B)
        assert _np(out["status"]).tolist() == [0] * 4, (B, _np(out["status"]))
        assert _np(out["n_nodes"]).tolist() == [B + 1] * 4, B
        if B % 10 == 0:
            ref, lists = oracle_build(orc, dr[1].cpu(), 8, B)
            assert compare_trees(_tree_np(out, 1), ref, lists) <= 1, B


def test_build_fp32_and_misaligned(tsd, dev, orc):
    """fp32 logits, and a row start that is not 16-byte aligned (generic path)."""
    dr = synth.zipf_drafter(1, 6, 5000, synth.seed_for(1, 3), device="cpu", dtype=torch.float32)
    buf = torch.empty(1 + dr.numel(), dtype=torch.float32, device=dev)
    buf[1:] = dr.reshape(-1).to(dev)
    view = buf[1:].view(dr.shape)
    out = tsd.tsd_build_tree(view, topk=6, B=50)
    ref, lists = oracle_build(orc, dr[0], 6, 50)
    assert compare_trees(_tree_np(out), ref, lists) <= 1


def test_build_mixture(tsd, dev, orc, flip_log):
    """K=8 modes from two latent futures (the mixture workload), B=128."""
    dr, _, _ = synth.mixture_drafter(2, 8, 16, V_Q, synth.seed_for(3), device="cpu")
    out = tsd.tsd_build_tree(dr.to(dev), topk=8, B=128)
    flips = 0
    for t in range(2):
        ref, lists = oracle_build(orc, dr[t], 8, 128)
        flips += compare_trees(_tree_np(out, t), ref, lists)
    flip_log("builder", flips)
    assert flips <= 2


def test_build_masked_and_small_universe(tsd, dev, orc):
    """-inf logits outside a few tokens: only finite-score prefixes become
    nodes, so n_nodes < B+1."""
    z = torch.full((1, 1, 3, 64), -float("inf"))
    z[0, 0, :, :2] = torch.tensor([1.0, 0.5])
    out = tsd.tsd_build_tree(z.to(dev), topk=4, B=50)
    ref, lists = oracle_build(orc, z[0], 4, 50)
    assert ref["n_nodes"] == 1 + 2 + 4 + 8
    assert compare_trees(_tree_np(out), ref, lists) == 0


@pytest.mark.parametrize("V,L,k,B", [(V_Q, 16, 8, 256), (V_Q, 16, 8, 64), (5000, 16, 2, 200),
                                     (5000, 16, 4, 340), (5000, 12, 16, 256), (5000, 16, 8, 1),
                                     (5000, 16, 8, 700), (5000, 16, 8, 1500)])
def test_build_one_mode_equals_duplicated_modes(tsd, dev, V, L, k, B):
    """One mode takes the threshold expansion where it applies; the same
    drafter given as two identical modes takes the rounds, whose merged heap
    keeps each prefix's first (mode 0) entry, in the one-mode order.  The two
    trees must be identical bit for bit: nodes, parents, tokens, depths,
    ranks and scores.  Budgets span one node, several depths
    of full enumeration (k = 2, 4, 16), and budgets past the expansion's
    capacity (the rounds on both sides)."""
    seeds = [synth.seed_for(4, 500 + t) for t in range(3)]
    dr = synth.zipf_drafter(3, L, V, 0, device=dev, seeds=seeds)
    one = tsd.tsd_build_tree(dr, topk=k, B=B)
    two = tsd.tsd_build_tree(torch.cat([dr, dr], dim=1), topk=k, B=B)
    assert _np(one["status"]).tolist() == [0] * 3
    assert _np(two["status"]).tolist() == [0] * 3
    for key in ("n_nodes", "parent", "token", "depth", "rank", "score"):
        assert np.array_equal(_np(one[key]), _np(two[key])), key


@pytest.mark.parametrize("case", ["peaked_then_flat", "uniform", "flat_deep"])
def test_build_threshold_edge_drafters(tsd, dev, orc, case):
    """Drafters at the edges of the one-mode threshold expansion, against the
    oracle: near-certain first three positions then eight equal tokens a
    position (the candidates within the bound multiply by eight a depth, the
    pair lists can outgrow their capacity and the rounds take the tree);
    every logit equal (all prefixes of a depth tie, one key bin holds
    hundreds of candidates ranked by their tie keys); and eight equal tokens
    at every position of a 16-row drafter with B = 1000 (the rounds)."""
    V, L = 64, 12
    z = torch.zeros(1, 1, L, V)
    B = 256
    if case == "peaked_then_flat":
        z[0, 0, :3, 0] = 30.0
        z[0, 0, 3:, :] = -30.0
        z[0, 0, 3:, :8] = 5.0
    elif case == "flat_deep":
        L = 16
        z = torch.full((1, 1, L, V), -30.0)
        z[0, 0, :, :8] = 1.0
        B = 1000
    out = tsd.tsd_build_tree(z.to(dev), topk=8, B=B)
    assert int(out["status"][0]) == 0
    ref, lists = oracle_build(orc, z[0], 8, B)
    assert compare_trees(_tree_np(out), ref, lists) == 0


def test_build_nonfinite_status(tsd, dev):
    z = torch.randn(2, 1, 4, 32)
    z[1, 0, 2, 5] = float("nan")
    out = tsd.tsd_build_tree(z.to(dev), topk=4, B=8)
    assert _np(out["status"]).tolist() == [0, 5]
    assert int(out["n_nodes"][1]) == 0 and int(out["n_nodes"][0]) == 9


# ---------------------------------------------------------------------------
# mask
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,P", [(8, 0), (64, 1024), (300, 17)])
def test_tree_mask(tsd, dev, orc, B, P):
    dr = synth.zipf_drafter(3, 16, 2048, synth.seed_for(4, B), device="cpu")
    parents, nn = [], []
    for t in range(3):
        ref, _ = oracle_build(orc, dr[t], 8, B)
        parents.append(ref["parent"])
        nn.append(ref["n_nodes"])
    nn[2] = max(1, nn[2] - 5)  # a ragged tree: trailing slots are padding
    par = torch.tensor(np.stack(parents), dtype=torch.int32, device=dev)
    n_nodes = torch.tensor(nn, dtype=torch.int32, device=dev)
    out = tsd.tsd_tree_mask(par, n_nodes, prefix_len=P, additive=True)
    for t in range(3):
        bits, pos, add = orc.tree_mask(parents[t], nn[t], B, P, with_additive=True)
        assert np.array_equal(_np(out["anc_bits"][t]).view(np.uint32), bits)
        assert np.array_equal(_np(out["position_ids"][t]), pos)
        assert np.array_equal(_np(out["additive_mask"][t]), add.astype(np.float32))
    assert _np(out["status"]).tolist() == [0, 0, 0]


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tev_and_mask_at_the_largest_budget(tsd, dev, orc, flip_log, T):
    """B = TSD_MAX_B (4096 nodes per tree, the largest child-list sort and
    bit rows of 128 words): a random recursive tree (parent of u uniform
    below u), one ragged tree, bf16 target logits at V = 5000.  TEV against
    the oracle (masses within tolerance, draws exact up to counted flips)
    and the mask bit for bit."""
    V, B = 5000, 4095
    rng = np.random.default_rng(synth.seed_for(4, 4095))
    nt = 2
    parent = np.full((nt, B + 1), -1, dtype=np.int32)
    token = np.full((nt, B + 1), -1, dtype=np.int32)
    nn = [B + 1, 3001]
    for t in range(nt):
        parent[t, 1:nn[t]] = [int(rng.integers(u)) for u in range(1, nn[t])]
        token[t, 1:nn[t]] = rng.permutation(V)[:nn[t] - 1]
    g = torch.Generator().manual_seed(int(synth.seed_for(4, 4096)))
    z = (torch.randn(nt, B + 1, V, generator=g) * 2).to(torch.bfloat16)
    for t in range(nt):  # raise about a third of the drafted tokens so that paths carry mass
        for u in range(1, nn[t]):
            if int(parent[t, u]) >= 0 and rng.random() < 0.3:
                z[t, int(parent[t, u]), int(token[t, u])] = 6.0
    pd, xd = torch.tensor(parent, device=dev), torch.tensor(token, device=dev)
    nd = torch.tensor(nn, dtype=torch.int32, device=dev)
    out = tsd.tsd_verify_tev(z.to(dev), pd, xd, nd, T, seed=3)
    flips = 0
    for t in range(nt):
        n = nn[t]
        z64 = z[t, :n].float().numpy().astype(np.float64)
        o = orc.tev(z64, parent[t], token[t], n, T, seed=3, tree=t)
        flips += _check_tev(out, t, o, z64, parent[t], token[t], n, T)
    flip_log("draw", flips)
    assert flips <= 1, flips
    m = tsd.tsd_tree_mask(pd, nd, prefix_len=77)
    for t in range(nt):
        bits, pos, _ = orc.tree_mask(parent[t], nn[t], B, 77)
        assert np.array_equal(_np(m["anc_bits"][t]).view(np.uint32), bits)
        assert np.array_equal(_np(m["position_ids"][t]), pos)
    assert _np(m["status"]).tolist() == [0] * nt


def test_tree_mask_bad_tree(tsd, dev):
    par = torch.tensor([[-1, 0, 2, 1]], dtype=torch.int32, device=dev)  # parent after child
    out = tsd.tsd_tree_mask(par, torch.tensor([4], dtype=torch.int32, device=dev))
    assert int(out["status"][0]) == 4
    assert _np(out["position_ids"][0]).tolist() == [0, 0, 0, 0]


# ---------------------------------------------------------------------------
# TEV and predraw
# ---------------------------------------------------------------------------
def _target_for(orc, tree, drafter_rows, sigma, seed, B, dtype):
    n = tree["n_nodes"]
    rows = synth.target_from_rows(drafter_rows.float(), tree["depth"][:n], sigma, seed, dtype=dtype)
    full = torch.zeros(B + 1, rows.shape[1], dtype=dtype)
    full[:n] = rows
    return full


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
@pytest.mark.parametrize("seed", range(4))
def test_tev_tiny(tsd, dev, orc, T, seed):
    s = synth.seed_for(0, seed)
    dr = synth.tiny_drafter(s)
    ref, _ = oracle_build(orc, dr[None], 4, 8)
    n = ref["n_nodes"]
    tgt = synth.tiny_target(dr, ref["depth"][:n], s + 7)
    full = torch.zeros(1, 9, 32)
    full[0, :n] = tgt
    par = torch.tensor(ref["parent"][None], dtype=torch.int32, device=dev)
    tok = torch.tensor(ref["token"][None], dtype=torch.int32, device=dev)
    nn = torch.tensor([n], dtype=torch.int32, device=dev)
    for sd in range(5):
        out = tsd.tsd_verify_tev(full.to(dev), par, tok, nn, T, seed=sd)
        o = orc.tev(tgt.numpy(), ref["parent"], ref["token"], n, T, seed=sd)
        assert _check_tev(out, 0, o, tgt.numpy().astype(np.float64), ref["parent"],
                          ref["token"], n, T) == 0
        d = tsd.tsd_verify_ddtree(full.to(dev), par, tok, nn, T, seed=sd)
        od = orc.predraw(tgt.numpy(), ref["parent"], ref["token"], n, T, seed=sd)
        assert _np(d["draws"][0])[:n].tolist() == od["draws"].tolist()
        assert (int(d["exit_node"][0]), int(d["bonus_token"][0]), int(d["accept_len"][0])) == \
            (od["exit_node"], od["bonus"], od["accept_len"])


@pytest.mark.parametrize("V,dtype", [(12805, torch.bfloat16), (4096 * 2 + 100, torch.float32),
                                     (3001, torch.bfloat16)])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tev_midsize(tsd, dev, orc, flip_log, V, dtype, T):
    """Several chunks and a ragged tail (V=3001 bf16 is not a multiple of 8:
    the generic path)."""
    B = 64
    dr = synth.zipf_drafter(1, 16, V, synth.seed_for(1, 7), device="cpu")
    ref, _ = oracle_build(orc, dr[0], 8, B)
    tgt = _target_for(orc, ref, dr[0, 0], 1.5, synth.seed_for(1, 8), B, dtype)
    par = torch.tensor(ref["parent"][None], dtype=torch.int32, device=dev)
    tok = torch.tensor(ref["token"][None], dtype=torch.int32, device=dev)
    nn = torch.tensor([ref["n_nodes"]], dtype=torch.int32, device=dev)
    n = ref["n_nodes"]
    z64 = tgt.float().numpy().astype(np.float64)
    flips = 0
    for sd in range(6):
        out = tsd.tsd_verify_tev(tgt[None].to(dev), par, tok, nn, T, seed=sd)
        o = orc.tev(z64[:n], ref["parent"], ref["token"], n, T, seed=sd)
        flips += _check_tev(out, 0, o, z64, ref["parent"], ref["token"], n, T)
        d = tsd.tsd_verify_ddtree(tgt[None].to(dev), par, tok, nn, T, seed=sd)
        od = orc.predraw(z64[:n], ref["parent"], ref["token"], n, T, seed=sd)
        for v in range(n):
            if int(d["draws"][0, v]) != int(od["draws"][v]):
                p = orc.row_probs(z64[v], T)
                flips += check_draw(int(d["draws"][0, v]), int(od["draws"][v]), p,
                                    orc.uniform(sd, 0, v, 2))
    flip_log("draw", flips)
    assert flips <= 2, flips


@pytest.mark.parametrize("T", [1.0, 0.0])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tev_qwen_vocab_b64(tsd, dev, orc, flip_log, T, dtype):
    """The batch-1 Qwen-vocabulary round: V=151936, L=16, k=8, B=64, target
    logits in bf16 (38 chunks per row) and fp32 (75 chunks: the per-chunk
    warp loops take three rounds)."""
    B = 64
    dr = synth.zipf_drafter(1, 16, V_Q, synth.seed_for(1), device="cpu")
    ref, _ = oracle_build(orc, dr[0], 8, B)
    tgt = _target_for(orc, ref, dr[0, 0], 1.5, synth.seed_for(1, 1), B, dtype)
    n = ref["n_nodes"]
    par = torch.tensor(ref["parent"][None], dtype=torch.int32, device=dev)
    tok = torch.tensor(ref["token"][None], dtype=torch.int32, device=dev)
    nn = torch.tensor([n], dtype=torch.int32, device=dev)
    z64 = tgt.float().numpy().astype(np.float64)
    flips = 0
    for sd in range(3):
        out = tsd.tsd_verify_tev(tgt[None].to(dev), par, tok, nn, T, seed=sd)
        o = orc.tev(z64[:n], ref["parent"], ref["token"], n, T, seed=sd)
        flips += _check_tev(out, 0, o, z64, ref["parent"], ref["token"], n, T)
    flip_log("draw", flips)
    assert flips <= 1


def test_tev_batched_b256(tsd, dev, orc, flip_log):
    """32 independent trees, V=151936, B=256, T=0.6, bf16: every tree checked
    for validity, four sampled trees against the oracle element by element."""
    nt, B, T = 32, 256, 0.6
    seeds = [synth.seed_for(2, t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, V_Q, 0, device=dev, seeds=seeds)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B)
    assert _np(tr["status"]).tolist() == [0] * nt
    tgt = torch.empty(nt, B + 1, V_Q, dtype=torch.bfloat16, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=tgt[t, :n])
        tgt[t, n:] = 0
    out = tsd.tsd_verify_tev(tgt, tr["parent"], tr["token"], tr["n_nodes"], T, seed=123)
    assert _np(out["status"]).tolist() == [0] * nt
    w = _np(out["exit_mass"])
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-4)
    for t in range(nt):
        ex = int(out["exit_node"][t])
        kids = [int(tr["token"][t, u]) for u in range(1, B + 1) if int(tr["parent"][t, u]) == ex]
        assert int(out["bonus_token"][t]) not in kids
    # sampled trees, element by element (the tree itself is the GPU's here; its
    # parity with the oracle builder is checked in the builder tests)
    flips = 0
    for t in (0, 9, 22, 31):
        n = int(tr["n_nodes"][t])
        par, tok = _np(tr["parent"][t]), _np(tr["token"][t])
        z64 = tgt[t, :n].float().cpu().numpy().astype(np.float64)
        o = orc.tev(z64, par, tok, n, T, seed=123, tree=t)
        flips += _check_tev(out, t, o, z64, par, tok, n, T)
    flip_log("draw", flips)
    assert flips <= 1


def test_tev_edge_cases(tsd, dev, orc):
    """Root-only tree, a chain, a star, a tree with masked tokens, and per-tree
    error codes (bad tree, NaN logits) next to valid trees."""
    V, B = 640, 12
    g = torch.Generator().manual_seed(5)
    z = torch.randn(5, B + 1, V, generator=g) * 2
    parent = np.full((5, B + 1), -1, dtype=np.int32)
    token = np.full((5, B + 1), -1, dtype=np.int32)
    nn = [1, B + 1, B + 1, 6, 4]
    for u in range(1, B + 1):  # tree 1: chain; tree 2: star
        parent[1, u], token[1, u] = u - 1, (7 * u) % V
        parent[2, u], token[2, u] = 0, 3 * u
    parent[3, 1:6] = [0, 0, 1, 1, 2]
    token[3, 1:6] = [5, 9, 5, 100, 639]
    z[3, 1, 10:600] = -float("inf")  # masked tokens
    parent[4, 1:4] = [0, 1, 1]
    token[4, 1:4] = [1, 2, 2]  # repeated sibling token: a malformed tree
    zz = z.clone()
    zz[0, 0, 17] = float("nan")  # tree 0 gets a NaN
    for T in (1.0, 0.0):
        out = tsd.tsd_verify_tev(zz.to(dev), torch.tensor(parent, device=dev),
                                 torch.tensor(token, device=dev),
                                 torch.tensor(nn, dtype=torch.int32, device=dev), T, seed=9)
        st = _np(out["status"]).tolist()
        assert st == [5, 0, 0, 0, 4], st
        assert int(out["exit_node"][4]) == -1 and int(out["accept_len"][4]) == 0
        for t in (1, 2, 3):
            n = nn[t]
            z64 = z[t, :n].numpy().astype(np.float64)
            o = orc.tev(z64, parent[t], token[t], n, T, seed=9, tree=t)
            assert _check_tev(out, t, o, z64, parent[t], token[t], n, T) == 0
        # the NaN-free copy of tree 0 (root only): exit at the root, bonus ~ p_root
        out0 = tsd.tsd_verify_tev(z[:1].to(dev), torch.tensor(parent[:1], device=dev),
                                  torch.tensor(token[:1], device=dev),
                                  torch.tensor([1], dtype=torch.int32, device=dev), T, seed=9)
        o = orc.tev(z[0, :1].numpy().astype(np.float64), parent[0], token[0], 1, T, seed=9)
        assert (int(out0["exit_node"][0]), int(out0["bonus_token"][0]), int(out0["accept_len"][0])) \
            == (0, o["bonus"], 1)


def _greedy_tie_case(V, B, rng):
    """A random tree and integer-valued target logits whose row maxima tie
    exactly at several tokens spread over lanes, vectors and chunks.  At
    about 70% of the nodes with children, a drafted child is the smallest id
    among the tied maxima (accepted at T = 0); elsewhere a smaller id ties
    with it (rejected).  Two rows have maxima of 0 tied between -0.0 and
    +0.0; one row has its only maximum at the last token."""
    parent = np.full(B + 1, -1, dtype=np.int32)
    token = np.full(B + 1, -1, dtype=np.int32)
    for u in range(1, B + 1):
        parent[u] = rng.integers(max(0, u - 5), u) if u > 3 else u - 1
        used = {int(token[s]) for s in range(1, u) if parent[s] == parent[u]}
        while True:
            x = int(rng.integers(0, V))
            if x not in used:
                break
        token[u] = x
    z = rng.integers(-8, 1, size=(B + 1, V)).astype(np.float32)
    for v in range(B + 1):
        kids = [int(token[u]) for u in range(1, B + 1) if parent[u] == v]
        ties = set(int(x) for x in rng.integers(0, V, size=int(rng.integers(1, 5))))
        if kids:
            c = kids[int(rng.integers(0, len(kids)))]
            if rng.random() < 0.7:  # the child is the first of the tied maxima
                ties = {x for x in ties if x > c} | {c}
            else:  # a smaller id ties with it
                ties |= {c, int(rng.integers(0, c))} if c > 0 else {c}
        z[v, sorted(ties)] = 3.0
    # rows 1 and 2: maxima of 0, signed zeros tied
    for v, first_neg in ((1, True), (2, False)):
        z[v] = np.minimum(z[v], -1.0)
        pos = np.sort(rng.choice(V, size=6, replace=False))
        z[v, pos] = 0.0
        z[v, pos[0::2] if first_neg else pos[1::2]] = -0.0
    # row 3: one maximum, at the last token
    z[3] = np.minimum(z[3], 2.0)
    z[3, V - 1] = 5.0
    return parent, token, z


@pytest.mark.parametrize("V,dtype", [(3 * 4096 + 512, torch.bfloat16), (2 * 2048 + 256, torch.float32),
                                     (3001, torch.bfloat16)])
def test_tev_greedy_exact_ties(tsd, dev, orc, V, dtype):
    """T = 0 with exact ties at the row maxima: the arg-max must be the
    smallest tied id on both sides, so exit node, bonus token, accepted
    length and the predraw-and-follow draws are bit-exact."""
    B, nt = 24, 6
    rng = np.random.default_rng(synth.seed_for(1, 40))
    cases = [_greedy_tie_case(V, B, rng) for _ in range(nt)]
    par = torch.tensor(np.stack([c[0] for c in cases]), device=dev)
    tok = torch.tensor(np.stack([c[1] for c in cases]), device=dev)
    zt = torch.tensor(np.stack([c[2] for c in cases])).to(dtype)
    nn = torch.full((nt,), B + 1, dtype=torch.int32, device=dev)
    out = tsd.tsd_verify_tev(zt.to(dev), par, tok, nn, 0.0, seed=3)
    d = tsd.tsd_verify_ddtree(zt.to(dev), par, tok, nn, 0.0, seed=3)
    accepted = 0
    for t, (parent, token, _) in enumerate(cases):
        z64 = zt[t].float().numpy().astype(np.float64)
        o = orc.tev(z64, parent, token, B + 1, 0.0, seed=3, tree=t)
        assert _check_tev(out, t, o, z64, parent, token, B + 1, 0.0) == 0
        assert int(out["exit_node"][t]) == o["exit_node"] and int(out["bonus_token"][t]) == o["bonus"]
        od = orc.predraw(z64, parent, token, B + 1, 0.0, seed=3, tree=t)
        assert _np(d["draws"][t]).tolist() == od["draws"].tolist()
        assert (int(d["exit_node"][t]), int(d["bonus_token"][t])) == (od["exit_node"], od["bonus"])
        accepted += o["accept_len"] - 1
    assert accepted > 0  # some drafted children were accepted


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tev_greedy_nonfinite_rows(tsd, dev, orc, dtype):
    """At T = 0 as at T > 0, a node row holding +inf or NaN, or with every
    token at -inf, is an error for its tree (status 5); other trees are
    unaffected."""
    V, B = 4096 + 1024, 3
    g = torch.Generator().manual_seed(11)
    z = torch.randn(4, B + 1, V, generator=g)
    parent = np.array([[-1, 0, 0, 1]] * 4, dtype=np.int32)
    token = np.array([[-1, 5, 9, 7]] * 4, dtype=np.int32)
    z[0, 2, 4500] = float("inf")
    z[1, 3, :] = -float("inf")
    z[2, 1, 77] = float("nan")
    zt = z.to(dtype)
    nn = torch.full((4,), B + 1, dtype=torch.int32, device=dev)
    for T in (0.0, 1.0):
        out = tsd.tsd_verify_tev(zt.to(dev), torch.tensor(parent, device=dev),
                                 torch.tensor(token, device=dev), nn, T, seed=1)
        st = _np(out["status"]).tolist()
        assert st == [5, 5, 5, 0], (T, st)
        for t in range(3):  # the oracle rejects the same rows
            with pytest.raises(orc.OracleError):
                orc.tev(zt[t].float().numpy().astype(np.float64), parent[t], token[t], B + 1, T, seed=1)


def test_tev_outputs_fully_written(tsd, dev, orc):
    """Every output slot is written (sentinel fill through a caller workspace
    filled with NaN bytes)."""
    V, B = 300, 10
    z = torch.randn(2, B + 1, V)
    parent = torch.tensor([[-1, 0, 0, 1] + [-1] * 7, [-1] + [-1] * 10], dtype=torch.int32)
    token = torch.tensor([[-1, 4, 8, 15] + [-1] * 7, [-1] * 11], dtype=torch.int32)
    nn = torch.tensor([4, 1], dtype=torch.int32)
    nbytes = tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 2, 1, 1, V, 1, B, torch.float32)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)
    out = tsd.tsd_verify_tev(z.to(dev), parent.to(dev), token.to(dev), nn.to(dev), 1.0, seed=3,
                             workspace=ws)
    assert _np(out["status"]).tolist() == [0, 0]
    w = _np(out["exit_mass"])
    assert np.all(np.isfinite(w)) and np.all(w[0, 4:] == 0) and np.all(w[1, 1:] == 0)
    assert w[1, 0] == 1.0


def test_tev_and_predraw_law_on_gpu(tsd, dev, orc):
    """10^6 GPU draws of each verifier on one tiny tree (replicated over
    100000 tree slots with their own uniforms) against the exact joint law
    from the oracle's masses: chi-square, as the pages' saturation theorem
    requires of both."""
    import scipy.stats
    s = synth.seed_for(0, 99)
    dr = synth.tiny_drafter(s)
    ref, _ = oracle_build(orc, dr[None], 4, 8)
    n = ref["n_nodes"]
    tgt = synth.tiny_target(dr, ref["depth"][:n], s + 7).numpy().astype(np.float64)
    o = orc.tev(tgt, ref["parent"], ref["token"], n, 1.0, seed=0)
    law = np.zeros((n, 32))
    for v in range(n):
        p = orc.row_probs(tgt[v], 1.0)
        kids = [int(ref["token"][u]) for u in range(1, n) if int(ref["parent"][u]) == v]
        p[kids] = 0.0
        law[v] = o["w"][v] * p / p.sum()
    R = 100000
    full = torch.zeros(R, 9, 32, device=dev)
    full[:, :n] = torch.tensor(tgt, dtype=torch.float32, device=dev)
    par = torch.tensor(ref["parent"], dtype=torch.int32, device=dev).expand(R, 9).contiguous()
    tok = torch.tensor(ref["token"], dtype=torch.int32, device=dev).expand(R, 9).contiguous()
    nn = torch.full((R,), n, dtype=torch.int32, device=dev)
    for fn in (tsd.tsd_verify_tev, tsd.tsd_verify_ddtree):
        counts = np.zeros(n * 32)
        for rep in range(10):
            out = fn(full, par, tok, nn, 1.0, seed=1000 + rep)
            cell = _np(out["exit_node"]).astype(np.int64) * 32 + _np(out["bonus_token"])
            counts += np.bincount(cell, minlength=n * 32)
        exp = law.ravel() * counts.sum()
        assert counts[exp == 0].sum() == 0
        keep = exp >= 5
        obs = np.append(counts[keep], counts[~keep].sum())
        ex = np.append(exp[keep], exp[~keep].sum())
        assert scipy.stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue > 1e-4, fn.__name__


def test_build_edge_budgets(tsd, dev, orc, flip_log):
    """B = 0 (the root alone); budgets whose search buffers spill from shared
    to global memory (8 modes at B = 512, one mode at the largest B); and rows
    of equal logits, where every token ties (the drafter kernel's exact
    fallback for an overflowing candidate set)."""
    dr = synth.zipf_drafter(1, 6, 2048, synth.seed_for(5), device="cpu")
    out = tsd.tsd_build_tree(dr.to(dev), topk=8, B=0)
    assert int(out["n_nodes"][0]) == 1 and int(out["status"][0]) == 0
    assert _np(out["parent"][0]).tolist() == [-1]
    mix, _, _ = synth.mixture_drafter(1, 8, 6, 1024, synth.seed_for(5, 1), device="cpu")
    out = tsd.tsd_build_tree(mix.to(dev), topk=8, B=512)
    ref, lists = oracle_build(orc, mix[0], 8, 512)
    assert compare_trees(_tree_np(out), ref, lists) <= 1
    out = tsd.tsd_build_tree(dr.to(dev), topk=8, B=4095)
    ref, lists = oracle_build(orc, dr[0], 8, 4095)
    flips = compare_trees(_tree_np(out), ref, lists)  # each within SCORE_TOL
    flip_log("builder", flips)
    assert flips <= 2
    flat = torch.zeros(2, 1, 5, 9000)
    flat[1, 0, 2, 4444] = 1.0
    out = tsd.tsd_build_tree(flat.to(dev), topk=8, B=100)
    for t in range(2):
        ref, lists = oracle_build(orc, flat[t], 8, 100)
        g = _tree_np(out, t)
        assert compare_trees(g, ref, lists) == 0
        assert np.array_equal(g["rank"][:g["n_nodes"]], ref["rank"][:ref["n_nodes"]])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_build_topk_selection_paths(tsd, dev, orc, dtype):
    """The drafter top-k through each of its selection paths, checked against
    the oracle builder tree for tree: a handful of tokens at or above the
    bound (one warp sort); dozens of tokens tied at the row maximum, spread
    over every chunk (the bound admits all of them: a longer list); a row
    with fewer than k chunks (the bound is -inf: every token is scanned);
    and a row whose top tokens all sit in one chunk."""
    V, L = 40960, 4
    g = torch.Generator().manual_seed(synth.seed_for(5, 9))
    z = torch.randint(-20, 1, (4, 1, L, V), generator=g).float()
    # row pattern 1: 60 tokens tied at 5.0, spread over all chunks
    ties = torch.randperm(V, generator=g)[:60]
    z[1, 0, :, ties] = 5.0
    # pattern 3: the 30 largest logits packed into chunk 2
    z[3, 0, :, 2 * 4096 + 100: 2 * 4096 + 130] = torch.arange(30, dtype=torch.float32) * 0.25 + 3.0
    # pattern 0: Zipf-like distinct values
    z[0] = synth.zipf_drafter(1, L, V, synth.seed_for(5, 10), device="cpu", dtype=torch.float32)[0]
    small = synth.zipf_drafter(1, L, 3000, synth.seed_for(5, 11), device="cpu", dtype=torch.float32)
    zz = z.to(dtype)
    out = tsd.tsd_build_tree(zz.to(dev), topk=8, B=40)
    for t in range(4):
        ref, lists = oracle_build(orc, zz[t], 8, 40)
        assert compare_trees(_tree_np(out, t), ref, lists) == 0, t
    zs = small.to(dtype)  # 3000 tokens: one chunk in bf16, two in fp32 (fewer than k)
    out = tsd.tsd_build_tree(zs.to(dev), topk=8, B=40)
    ref, lists = oracle_build(orc, zs[0], 8, 40)
    assert compare_trees(_tree_np(out, 0), ref, lists) == 0


def test_logits_in_pinned_host_memory(tsd, dev, orc):
    """Drafter and target logits read straight from page-locked host memory
    give the same trees and the same verification outputs as the same logits
    in device memory."""
    nt, V, B = 3, 20000, 24
    seeds = [synth.seed_for(6, t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 6, V, 0, device="cpu", seeds=seeds)
    dr_h = dr.pin_memory()
    tr_d = tsd.tsd_build_tree(dr.to(dev), topk=8, B=B)
    tr_h = tsd.tsd_build_tree(dr_h, topk=8, B=B, device=dev)
    for key in ("parent", "token", "depth", "score", "n_nodes", "status"):
        assert torch.equal(tr_d[key], tr_h[key]), key
    tgt = torch.zeros(nt, B + 1, V, dtype=torch.bfloat16)
    for t in range(nt):
        n = int(tr_d["n_nodes"][t])
        tgt[t, :n] = synth.target_from_rows(dr[t, 0].float(), _np(tr_d["depth"][t, :n]), 1.5,
                                            seeds[t] + 1)
    tgt_h = tgt.pin_memory()
    for T in (0.6, 0.0):
        o_d = tsd.tsd_verify_tev(tgt.to(dev), tr_d["parent"], tr_d["token"], tr_d["n_nodes"], T, seed=5)
        o_h = tsd.tsd_verify_tev(tgt_h, tr_d["parent"], tr_d["token"], tr_d["n_nodes"], T, seed=5)
        for key in o_d:
            assert torch.equal(o_d[key], o_h[key]), (T, key)
        p_h = tsd.tsd_verify_ddtree(tgt_h, tr_d["parent"], tr_d["token"], tr_d["n_nodes"], T, seed=5)
        p_d = tsd.tsd_verify_ddtree(tgt.to(dev), tr_d["parent"], tr_d["token"], tr_d["n_nodes"], T, seed=5)
        for key in p_d:
            assert torch.equal(p_d[key], p_h[key]), (T, key)


def test_deep_trees(tsd, dev, orc):
    """The deepest shapes the limits allow: L = 28 with top-4 (56 bits of rank
    sequence) in the builder; L = 31 with top-2 in the log-sum-exp tree (two
    modes) and in the exit loss."""
    dr = synth.zipf_drafter(2, 28, 5000, synth.seed_for(6), device="cpu")
    out = tsd.tsd_build_tree(dr.to(dev), topk=4, B=300)
    for t in range(2):
        ref, lists = oracle_build(orc, dr[t], 4, 300)
        assert compare_trees(_tree_np(out, t), ref, lists) <= 1
        assert int(out["depth"][t].max()) <= 28
    mix, _, _ = synth.mixture_drafter(1, 2, 31, 3000, synth.seed_for(6, 1), device="cpu")
    lt = tsd.tsd_build_lse_tree(mix.to(dev), topk=2, B=200)
    ref = orc.lse_tree(mix[0].double().numpy(), 1.0, 2, 200)
    assert int(lt["n_cand"][0]) == ref["n_cand"] and int(lt["n_nodes"][0]) == ref["n_nodes"]
    seq_g = sequences_of(_np(lt["parent"][0]), _np(lt["token"][0]), ref["n_nodes"])
    seq_o = sequences_of(ref["parent"], ref["token"], ref["n_nodes"])
    assert len(set(seq_g) ^ set(seq_o)) <= 2  # a near-tie at the cut may swap one prefix
    z = synth.zipf_drafter(2, 31, 3000, synth.seed_for(6, 2), device="cpu", dtype=torch.float32)
    tr = tsd.tsd_build_tree(z.to(dev), topk=2, B=120)
    w = torch.rand(2, 121, generator=torch.Generator().manual_seed(3)).to(dev) * (tr["depth"] >= 0)
    ex = tsd.tsd_exit_loss(z.to(dev), tr["token"], tr["depth"], tr["n_nodes"], w)
    for t in range(2):
        n = int(tr["n_nodes"][t])
        num = orc.exit_loss(z[t, 0].double().numpy(), 1.0, _np(tr["token"][t]), _np(tr["depth"][t]),
                            n, w[t].double().cpu().numpy())
        assert abs(float(ex["loss_tree"][t]) - num) <= 1e-5 * abs(num)


def sequences_of(parent, token, n):
    seqs = [()]
    for u in range(1, n):
        seqs.append(seqs[int(parent[u])] + (int(token[u]),))
    return seqs

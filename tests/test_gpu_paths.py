"""Both Tree Exit Verification paths (and both predraw-and-follow paths) on
the same trees.

tsd_verify_tev runs small budgets (B <= 64, 16-byte aligned rows) as two
kernels (a streaming row kernel, then one block per tree) and larger ones as
the batched four-kernel chain.  Here the same trees and logits go through
both: as given (B small: the two-kernel path) and padded with unused slots to
B = 140 (the batched chain).  The two must agree exactly on exit node, bonus
token, accepted length and status, and within the parity tolerance on the
masses; both are also checked against the float64 oracle ([EXIT] App. B).
The cases include the malformed-tree and non-finite-row statuses, greedy ties
and rows whose children fill a whole chunk.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import RTOL, check_tev, close, to_np

pytestmark = pytest.mark.gpu

B_CHAIN = 140  # above the two-kernel path's largest budget


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


def _pad(z, parent, token, B_new):
    nt, R, V = z.shape
    zp = torch.zeros(nt, B_new + 1, V, dtype=z.dtype)
    zp[:, :R] = z
    pp = np.full((nt, B_new + 1), -1, dtype=np.int32)
    tp = np.full((nt, B_new + 1), -1, dtype=np.int32)
    pp[:, :R] = parent
    tp[:, :R] = token
    return zp, pp, tp


def _both(tsd, dev, z, parent, token, nn, T, seed):
    """(two-kernel outputs, batched-chain outputs cut back to B+1 slots)."""
    R = z.shape[1]
    nd = torch.tensor(nn, dtype=torch.int32, device=dev)
    a = tsd.tsd_verify_tev(z.to(dev), torch.tensor(parent, device=dev),
                           torch.tensor(token, device=dev), nd, T, seed=seed)
    zp, pp, tp = _pad(z, parent, token, B_CHAIN)
    b = tsd.tsd_verify_tev(zp.to(dev), torch.tensor(pp, device=dev), torch.tensor(tp, device=dev),
                           nd, T, seed=seed)
    b = dict(b)
    for k in ("exit_mass", "prefix_prob"):
        assert float(b[k][:, R:].abs().max()) == 0.0
        b[k] = b[k][:, :R]
    return a, b


def _both_predraw(tsd, dev, z, parent, token, nn, T, seed):
    R = z.shape[1]
    nd = torch.tensor(nn, dtype=torch.int32, device=dev)
    a = tsd.tsd_verify_ddtree(z.to(dev), torch.tensor(parent, device=dev),
                              torch.tensor(token, device=dev), nd, T, seed=seed)
    zp, pp, tp = _pad(z, parent, token, B_CHAIN)
    b = dict(tsd.tsd_verify_ddtree(zp.to(dev), torch.tensor(pp, device=dev),
                                   torch.tensor(tp, device=dev), nd, T, seed=seed))
    assert int((b["draws"][:, R:] != -1).sum()) == 0
    b["draws"] = b["draws"][:, :R]
    for k in ("exit_node", "bonus_token", "accept_len", "status", "draws"):
        assert torch.equal(a[k], b[k]), (k, to_np(a[k]), to_np(b[k]))
    return a


def _agree(a, b):
    for k in ("exit_node", "bonus_token", "accept_len", "status"):
        assert torch.equal(a[k], b[k]), (k, to_np(a[k]), to_np(b[k]))
    for k in ("exit_mass", "prefix_prob", "coverage"):
        ok, err = close(to_np(a[k]), to_np(b[k]), rtol=RTOL)
        assert ok, (k, err)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
def test_paths_agree_on_builder_trees(tsd, dev, orc, dtype, T):
    """Four GPU-built trees (V = 12800: four bf16 / seven fp32 chunks, rows
    aligned), B = 48; both paths against each other and the oracle."""
    V, B, nt = 12800, 48, 4
    seeds = [synth.seed_for(7, t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, V, 0, device=dev, seeds=seeds)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B)
    z = torch.zeros(nt, B + 1, V, dtype=dtype)
    par, tok = to_np(tr["parent"]), to_np(tr["token"])
    nn = to_np(tr["n_nodes"]).tolist()
    for t in range(nt):
        z[t, :nn[t]] = synth.target_from_rows(dr[t, 0].cpu().float(), to_np(tr["depth"][t, :nn[t]]),
                                              1.5, seeds[t] + 1, dtype=dtype)
    for seed in (3, 4):
        a, b = _both(tsd, dev, z, par, tok, nn, T, seed)
        _agree(a, b)
        d = _both_predraw(tsd, dev, z, par, tok, nn, T, seed)
        for t in range(nt):
            z64 = z[t, :nn[t]].float().numpy().astype(np.float64)
            o = orc.tev(z64, par[t], tok[t], nn[t], T, seed=seed, tree=t)
            assert check_tev(a, t, o, z64, par[t], tok[t], nn[t], T) == 0
            od = orc.predraw(z64, par[t], tok[t], nn[t], T, seed=seed, tree=t)
            assert to_np(d["draws"][t])[:nn[t]].tolist() == od["draws"].tolist()
            assert (int(d["exit_node"][t]), int(d["bonus_token"][t]), int(d["accept_len"][t])) == \
                (od["exit_node"], od["bonus"], od["accept_len"])


def test_paths_agree_on_edge_cases(tsd, dev, orc):
    """Root-only tree, chain, star (children spread over a chunk), masked
    tokens, a repeated sibling token (malformed), a parent after its child
    (malformed), n_nodes out of range (malformed), a NaN row, a row at -inf:
    statuses 0, 4 and 5 side by side, identical on both paths."""
    V, B = 4096, 12
    g = torch.Generator().manual_seed(synth.seed_for(7, 100))
    z = torch.randn(9, B + 1, V, generator=g) * 2
    parent = np.full((9, B + 1), -1, dtype=np.int32)
    token = np.full((9, B + 1), -1, dtype=np.int32)
    nn = [1, B + 1, B + 1, 6, 4, 4, B + 5, 3, 3]
    for u in range(1, B + 1):  # tree 1: chain; tree 2: star
        parent[1, u], token[1, u] = u - 1, (7 * u) % V
        parent[2, u], token[2, u] = 0, 300 * u
    parent[3, 1:6] = [0, 0, 1, 1, 2]
    token[3, 1:6] = [5, 9, 5, 100, 4095]
    z[3, 1, 10:3000] = -float("inf")  # masked tokens
    parent[4, 1:4] = [0, 1, 1]
    token[4, 1:4] = [1, 2, 2]  # repeated sibling token
    parent[5, 1:4] = [0, 2, 1]
    token[5, 1:4] = [1, 2, 3]  # node 2's parent comes after it
    parent[6, 1:] = 0
    token[6, 1:] = np.arange(1, B + 1)
    parent[7, 1:3] = [0, 0]
    token[7, 1:3] = [8, 9]
    z[7, 2, 17] = float("nan")
    parent[8, 1:3] = [0, 1]
    token[8, 1:3] = [3, 4]
    z[8, 1, :] = -float("inf")
    for T in (1.0, 0.0):
        a, b = _both(tsd, dev, z, parent, token, nn, T, seed=9)
        _agree(a, b)
        assert to_np(a["status"]).tolist() == [0, 0, 0, 0, 4, 4, 4, 5, 5], to_np(a["status"])
        d = _both_predraw(tsd, dev, z, parent, token, nn, T, seed=9)
        assert to_np(d["status"]).tolist() == [0, 0, 0, 0, 4, 4, 4, 5, 5], to_np(d["status"])
        for t in (0, 1, 2, 3):
            n = nn[t]
            z64 = z[t, :n].numpy().astype(np.float64)
            o = orc.tev(z64, parent[t], token[t], n, T, seed=9, tree=t)
            assert check_tev(a, t, o, z64, parent[t], token[t], n, T) == 0


def test_paths_agree_on_greedy_ties(tsd, dev, orc):
    """T = 0 with the row maxima tied across lanes and chunks, and a drafted
    child as the first of the tied maxima at most nodes."""
    V, B, nt = 3 * 4096, 24, 4
    rng = np.random.default_rng(synth.seed_for(7, 200))
    parent = np.full((nt, B + 1), -1, dtype=np.int32)
    token = np.full((nt, B + 1), -1, dtype=np.int32)
    z = rng.integers(-8, 1, size=(nt, B + 1, V)).astype(np.float32)
    for t in range(nt):
        for u in range(1, B + 1):
            parent[t, u] = rng.integers(max(0, u - 5), u) if u > 3 else u - 1
            used = {int(token[t, s]) for s in range(1, u) if parent[t, s] == parent[t, u]}
            x = int(rng.integers(0, V))
            while x in used:
                x = int(rng.integers(0, V))
            token[t, u] = x
        for v in range(B + 1):
            kids = [int(token[t, u]) for u in range(1, B + 1) if parent[t, u] == v]
            ties = {int(x) for x in rng.integers(0, V, size=3)}
            if kids and rng.random() < 0.7:
                c = kids[0]
                ties = {x for x in ties if x > c} | {c}
            z[t, v, sorted(ties)] = 3.0
    zt = torch.tensor(z).to(torch.bfloat16)
    a, b = _both(tsd, dev, zt, parent, token, [B + 1] * nt, 0.0, seed=2)
    _agree(a, b)
    _both_predraw(tsd, dev, zt, parent, token, [B + 1] * nt, 0.0, seed=2)
    for t in range(nt):
        z64 = zt[t].float().numpy().astype(np.float64)
        o = orc.tev(z64, parent[t], token[t], B + 1, 0.0, seed=2, tree=t)
        assert check_tev(a, t, o, z64, parent[t], token[t], B + 1, 0.0) == 0

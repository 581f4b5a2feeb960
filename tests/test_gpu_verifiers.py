"""GPU parity of the sequential residual verifier ([EXIT] App. A.4.2) and the
proposal-aware verifier ([CAST] App. B.1 Thm. 3) against the float64 oracle:
the same trees, logits and uniforms give the same exit node, bonus token and
accepted length, up to counted decisions that fall within 1e-6 of their
threshold (the kernel decides in fp32, the oracle in fp64); at T = 0 they are
bit-exact.  The GPU draws also follow the exact joint law."""
import numpy as np
import pytest
import scipy.special
import torch

import synth

pytestmark = pytest.mark.gpu


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


def _np(t):
    return t.detach().cpu().numpy()


def _q_child(dr, tr, t, n, B, T_d=1.0):
    """q_{pa(u)}(x_u): the drafter's probability of node u's token at its position."""
    q = np.ones(B + 1)
    for u in range(1, n):
        d = int(tr["depth"][t, u])
        q[u] = scipy.special.softmax(dr[t, 0, d - 1].double().cpu().numpy() / T_d)[int(tr["token"][t, u])]
    return q


def _seqres_margin(orc, z64, par, tok, n, T, seed, t):
    """Smallest |u (1 - M) - p_j| over the decisions on the oracle's walk (and
    the bonus draw's CDF gap): how close the run came to a threshold."""
    p = [orc.row_probs(z64[v], T) for v in range(n)]
    kids = {v: sorted([u for u in range(1, n) if par[u] == v], key=lambda u: tok[u]) for v in range(n)}
    v, margin = 0, 1.0
    while True:
        M, nxt = 0.0, None
        for j, u in enumerate(kids[v]):
            pj = p[v][tok[u]]
            lhs = orc.uniform_sub(seed, t, v, 3, j) * (1.0 - M)
            margin = min(margin, abs(lhs - pj))
            if lhs < pj:
                nxt = u
                break
            M += pj
        if nxt is None:
            break
        v = nxt
    res = p[v].copy()
    res[[tok[u] for u in kids[v]]] = 0.0
    cum = np.cumsum(res)
    margin = min(margin, float(np.min(np.abs(cum - orc.uniform_sub(seed, t, v, 4, 0) * cum[-1]))))
    return margin


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
@pytest.mark.parametrize("V,dtype", [(32, torch.float32), (12805, torch.bfloat16),
                                     (4096 * 2 + 100, torch.float32), (synth.V_QWEN, torch.bfloat16)])
def test_verifiers_match_oracle(tsd, dev, orc, T, V, dtype):
    nt, B = (24, 8) if V == 32 else (4, 48)
    seeds = [synth.seed_for(8, 1000 * V % 977 + t) for t in range(nt)]
    if V == 32:
        drs = [synth.tiny_drafter(s) for s in seeds]
        dr = torch.stack(drs)[:, None].to(dev)
        tr = tsd.tsd_build_tree(dr, topk=4, B=B)
        tgt = torch.zeros(nt, B + 1, V, device=dev)
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            tgt[t, :n] = synth.tiny_target(drs[t], _np(tr["depth"][t, :n]), seeds[t] + 7).to(dev)
    else:
        dr = synth.zipf_drafter(nt, 8, V, 0, device=dev, seeds=seeds, dtype=dtype)
        tr = tsd.tsd_build_tree(dr, topk=8, B=B)
        tgt = torch.zeros(nt, B + 1, V, dtype=dtype, device=dev)
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1,
                                   out=tgt[t, :n], dtype=dtype)
    q = np.stack([_q_child(dr, tr, t, int(tr["n_nodes"][t]), B) for t in range(nt)])
    qd = torch.tensor(q, dtype=torch.float32, device=dev)
    flips = 0
    for seed in range(3):
        s_out = tsd.tsd_verify_seqres(tgt, tr["parent"], tr["token"], tr["n_nodes"], T, seed=seed)
        p_out = tsd.tsd_verify_proposal(tgt, tr["parent"], tr["token"], tr["n_nodes"], qd, T, seed=seed)
        assert _np(s_out["status"]).tolist() == [0] * nt
        assert _np(p_out["status"]).tolist() == [0] * nt
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            par, tok = _np(tr["parent"][t]), _np(tr["token"][t])
            z64 = tgt[t, :n].float().cpu().numpy().astype(np.float64)
            o = orc.seqres(z64, par, tok, n, T, seed=seed, tree=t)
            got = (int(s_out["exit_node"][t]), int(s_out["bonus_token"][t]), int(s_out["accept_len"][t]))
            if got != (o["exit_node"], o["bonus"], o["accept_len"]):
                assert T > 0 and _seqres_margin(orc, z64, par, tok, n, T, seed, t) < 1e-6, (t, got, o)
                flips += 1
            o = orc.proposal(z64, par, tok, n, T, q[t], seed=seed, tree=t)
            got = (int(p_out["exit_node"][t]), int(p_out["bonus_token"][t]), int(p_out["accept_len"][t]))
            if got != (o["exit_node"], o["bonus"], o["accept_len"]):
                assert T > 0, (t, got, o)  # greedy is bit-exact
                flips += 1
    assert flips <= 2, flips


def test_verifiers_law_on_gpu(tsd, dev, orc):
    """GPU draws of both verifiers on one tiny tree, replicated over 100000
    tree slots with their own uniforms: chi-square against the exact joint
    law of (exit node, bonus token)."""
    import scipy.stats
    s = synth.seed_for(0, 98)
    dr = synth.tiny_drafter(s)
    z = dr.numpy().astype(np.float64)
    ref = orc.build_tree(orc.drafter_lists(z, 1.0, 4), 8)
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
    q = np.ones(9)
    for u in range(1, n):
        q[u] = scipy.special.softmax(z[int(ref["depth"][u]) - 1])[int(ref["token"][u])]
    qd = torch.tensor(q, dtype=torch.float32, device=dev).expand(R, 9).contiguous()
    for name in ("seqres", "proposal"):
        counts = np.zeros(n * 32)
        for rep in range(10):
            if name == "seqres":
                out = tsd.tsd_verify_seqres(full, par, tok, nn, 1.0, seed=2000 + rep)
            else:
                out = tsd.tsd_verify_proposal(full, par, tok, nn, qd, 1.0, seed=3000 + rep)
            cell = _np(out["exit_node"]).astype(np.int64) * 32 + _np(out["bonus_token"])
            counts += np.bincount(cell, minlength=n * 32)
        exp = law.ravel() * counts.sum()
        assert counts[exp == 0].sum() == 0, name
        keep = exp >= 5
        obs = np.append(counts[keep], counts[~keep].sum())
        ex = np.append(exp[keep], exp[~keep].sum())
        assert scipy.stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue > 1e-4, name


def test_proposal_rejects_non_positive_q(tsd, dev, orc):
    """A proposal that is zero or NaN on a child marks its tree 5; other
    trees are unaffected; bad trees still report 4."""
    s = synth.seed_for(0, 97)
    dr = synth.tiny_drafter(s)
    ref = orc.build_tree(orc.drafter_lists(dr.numpy().astype(np.float64), 1.0, 4), 8)
    n = ref["n_nodes"]
    tgt = synth.tiny_target(dr, ref["depth"][:n], s + 7)
    full = torch.zeros(3, 9, 32, device=dev)
    full[:, :n] = tgt.to(dev)
    par = torch.tensor(ref["parent"], dtype=torch.int32, device=dev).expand(3, 9).contiguous().clone()
    tok = torch.tensor(ref["token"], dtype=torch.int32, device=dev).expand(3, 9).contiguous().clone()
    par[2, 1] = 5  # parent after child: a malformed tree
    nn = torch.full((3,), n, dtype=torch.int32, device=dev)
    q = torch.full((3, 9), 0.3, device=dev)
    q[1, 1:n] = 0.0
    out = tsd.tsd_verify_proposal(full, par, tok, nn, q, 1.0, seed=1)
    assert _np(out["status"]).tolist() == [0, 5, 4]
    assert int(out["exit_node"][1]) == -1


def test_verifiers_in_the_bench_launch(tsd, dev, orc):
    """32 trees, V=151936, B=256, T=0.6, bf16 (the bench's verification
    launch): four sampled trees against the oracle for both walk rules."""
    nt, B, T = 32, 256, 0.6
    seeds = [synth.seed_for(2, t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, synth.V_QWEN, 0, device=dev, seeds=seeds)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B)
    tgt = torch.zeros(nt, B + 1, synth.V_QWEN, dtype=torch.bfloat16, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=tgt[t, :n])
    sample = (0, 11, 20, 31)
    q = np.ones((nt, B + 1))
    for t in sample:
        q[t] = _q_child(dr, tr, t, int(tr["n_nodes"][t]), B)
    qd = torch.tensor(q, dtype=torch.float32, device=dev)
    flips = 0
    for seed in (5, 6):
        s_out = tsd.tsd_verify_seqres(tgt, tr["parent"], tr["token"], tr["n_nodes"], T, seed=seed)
        p_out = tsd.tsd_verify_proposal(tgt, tr["parent"], tr["token"], tr["n_nodes"], qd, T,
                                        seed=seed)
        assert _np(s_out["status"]).tolist() == [0] * nt
        assert _np(p_out["status"]).tolist() == [0] * nt
        for t in sample:
            n = int(tr["n_nodes"][t])
            par, tok = _np(tr["parent"][t]), _np(tr["token"][t])
            z64 = tgt[t, :n].float().cpu().numpy().astype(np.float64)
            o = orc.seqres(z64, par, tok, n, T, seed=seed, tree=t)
            got = (int(s_out["exit_node"][t]), int(s_out["bonus_token"][t]), int(s_out["accept_len"][t]))
            if got != (o["exit_node"], o["bonus"], o["accept_len"]):
                assert _seqres_margin(orc, z64, par, tok, n, T, seed, t) < 1e-6, (t, got, o)
                flips += 1
            o = orc.proposal(z64, par, tok, n, T, q[t], seed=seed, tree=t)
            got = (int(p_out["exit_node"][t]), int(p_out["bonus_token"][t]), int(p_out["accept_len"][t]))
            flips += got != (o["exit_node"], o["bonus"], o["accept_len"])
    assert flips <= 1, flips


def _wide_trees(rng, V, B):
    """Three hand-shaped trees in one B = 4095 launch: a star of 4095 children
    (the largest budget; more than 32 children per node), a 40-wide root whose
    three largest-token children hold 50 children each, and a chain into a
    70-wide node.  Node order is not token order: tokens are drawn at random,
    distinct among siblings."""
    trees = []
    # star
    toks = rng.permutation(V)[:B]
    trees.append(([-1] + [0] * B, [-1] + toks.tolist()))
    # two wide levels
    par, tok = [-1], [-1]
    kids = rng.permutation(V)[:40]
    for x in kids:
        par.append(0)
        tok.append(int(x))
    for u in sorted(range(1, 41), key=lambda u: -tok[u])[:3]:
        for x in rng.permutation(V)[:50]:
            par.append(u)
            tok.append(int(x))
    trees.append((par, tok))
    # chain into a wide node
    par, tok = [-1, 0, 1], [-1, int(rng.integers(V)), int(rng.integers(V))]
    for x in rng.permutation(V)[:70]:
        par.append(2)
        tok.append(int(x))
    trees.append((par, tok))
    return trees


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_verifiers_wide_nodes_and_largest_budget(tsd, dev, orc, T):
    """Nodes with 40 to 4095 children (the walks' lanes cover several
    32-child chunks per node) at B = TSD_MAX_B (the largest staging), bf16,
    V = 5000.  Each internal node's row favours its largest-token child, so
    the sequential rule rejects most siblings before it accepts and the
    proposal rule draws many candidates; both match the oracle."""
    V, B = 5000, 4095
    rng = np.random.default_rng(synth.seed_for(8, 4095))
    trees = _wide_trees(rng, V, B)
    nt = len(trees)
    par = np.full((nt, B + 1), -1, dtype=np.int32)
    tok = np.full((nt, B + 1), -1, dtype=np.int32)
    nn = np.zeros(nt, dtype=np.int32)
    for t, (p_, x_) in enumerate(trees):
        nn[t] = len(p_)
        par[t, :nn[t]] = p_
        tok[t, :nn[t]] = x_
    g = torch.Generator(device="cpu").manual_seed(int(synth.seed_for(8, 4096)))
    z = torch.randn(nt, B + 1, V, generator=g)
    for t in range(nt):
        for v in range(nn[t]):
            ch = [int(tok[t, u]) for u in range(1, nn[t]) if par[t, u] == v]
            if ch:
                z[t, v, max(ch)] += 10.0
    tgt = z.to(torch.bfloat16).to(dev)
    q = rng.uniform(0.5, 1.5, size=(nt, B + 1))
    pd, xd = torch.tensor(par, device=dev), torch.tensor(tok, device=dev)
    nd = torch.tensor(nn, device=dev)
    qd = torch.tensor(q, dtype=torch.float32, device=dev)
    flips, deep = 0, 0
    for seed in range(3):
        s_out = tsd.tsd_verify_seqres(tgt, pd, xd, nd, T, seed=seed)
        p_out = tsd.tsd_verify_proposal(tgt, pd, xd, nd, qd, T, seed=seed)
        assert _np(s_out["status"]).tolist() == [0] * nt
        assert _np(p_out["status"]).tolist() == [0] * nt
        for t in range(nt):
            n = int(nn[t])
            z64 = tgt[t, :n].float().cpu().numpy().astype(np.float64)
            o = orc.seqres(z64, par[t], tok[t], n, T, seed=seed, tree=t)
            got = (int(s_out["exit_node"][t]), int(s_out["bonus_token"][t]), int(s_out["accept_len"][t]))
            if got != (o["exit_node"], o["bonus"], o["accept_len"]):
                assert T > 0 and _seqres_margin(orc, z64, par[t], tok[t], n, T, seed, t) < 1e-6, (t, got, o)
                flips += 1
            deep += o["accept_len"] > 1
            o = orc.proposal(z64, par[t], tok[t], n, T, q[t], seed=seed, tree=t)
            got = (int(p_out["exit_node"][t]), int(p_out["bonus_token"][t]), int(p_out["accept_len"][t]))
            if got != (o["exit_node"], o["bonus"], o["accept_len"]):
                assert T > 0, (t, got, o)
                flips += 1
    assert flips <= 1, flips
    assert deep >= 3  # the walks do pass the wide nodes

"""Comparison helpers for the GPU parity tests: the CUDA path against the
float64 oracle on the same seeded inputs.

Tolerances (stated once, used by every GPU test):
  * integer structure (tree, mask, greedy outputs, sampled indices given the
    same uniforms): bit-exact, except that a sampled index may flip where the
    oracle's CDF lies within FLIP_TOL (relative to the distribution's total) of
    the threshold u * total; such flips are counted and reported, and the
    tests bound their number;
  * builder order: two prefixes may swap only when their oracle scores differ
    by at most SCORE_TOL relative (the kernel's log-normaliser is accumulated
    in fp32, the oracle's in fp64); builder scores agree within SCORE_TOL
    relative, absolute below magnitude 1 (the normaliser's error is at the
    scale of the logits, while a path of near-certain tokens scores near 0);
  * probabilities, exit masses, coverage: RTOL relative; values below TINY
    compared absolutely.
"""
import numpy as np

RTOL = 1e-5
TINY = 1e-30
FLIP_TOL = 1e-6
SCORE_TOL = 1e-6


def close(got, want, rtol=RTOL, tiny=TINY):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if got.size == 0 and want.size == 0:
        return True, 0.0
    err = np.abs(got - want)
    ok = (err <= rtol * np.abs(want)) | ((np.abs(want) < tiny) & (np.abs(got) < tiny * 1e3))
    return bool(np.all(ok)), float(np.max(err / np.maximum(np.abs(want), tiny)))


def sequences(parent, token, n):
    seqs = [()]
    for u in range(1, n):
        seqs.append(seqs[int(parent[u])] + (int(token[u]),))
    return seqs


def prefix_score(seq, lists):
    """Best-mode score of a token sequence in the capped universe (fp64),
    evaluated like the builder (path sum of z/T minus the summed row
    log-normalisers), or None if no mode holds it."""
    top_id, top_zt, lse = lists["top_id"], lists["top_zt"], lists["lse"]
    K, L, k = top_id.shape
    best = None
    for m in range(K):
        z, c = 0.0, 0.0
        for j, x in enumerate(seq):
            hit = np.nonzero(top_id[m, j] == x)[0]
            if hit.size == 0:
                z = None
                break
            z = z + top_zt[m, j, hit[0]]
            c = c + lse[m, j]
        if z is not None and (best is None or z - c > best):
            best = z - c
    return best


def compare_trees(gpu, ref, lists):
    """Compare a GPU-built tree (numpy arrays for one tree) with the oracle's.
    Returns the number of order flips (each within SCORE_TOL); raises on
    anything else."""
    n_g, n_o = int(gpu["n_nodes"]), int(ref["n_nodes"])
    assert n_g == n_o, ("node count", n_g, n_o)
    sg = sequences(gpu["parent"], gpu["token"], n_g)
    so = sequences(ref["parent"], ref["token"], n_o)
    if sg == so:
        assert np.array_equal(gpu["depth"][:n_g], ref["depth"][:n_o])
        g = np.asarray(gpu["score"][1:n_g], dtype=np.float64)
        w = np.asarray(ref["score"][1:n_o], dtype=np.float64)
        err = np.abs(g - w)
        assert np.all(err <= SCORE_TOL * np.maximum(1.0, np.abs(w))), ("scores", float(err.max(initial=0.0)))
        return 0
    flips = 0
    for i in range(1, n_g):
        if sg[i] == so[i]:
            continue
        a = prefix_score(sg[i], lists)
        b = prefix_score(so[i], lists)
        assert a is not None, ("gpu node outside the universe", sg[i])
        assert abs(a - b) <= SCORE_TOL * max(1.0, abs(b)), ("order", i, sg[i], so[i], a, b)
        flips += 1
    # same prefix-closed shape: every GPU node's parent precedes it
    for u in range(1, n_g):
        assert 0 <= gpu["parent"][u] < u
    return flips


def check_draw(idx_gpu, idx_ref, masses, u, tol=FLIP_TOL):
    """Inverse-CDF draw check.  masses: the oracle's (fp64) masses in draw
    order; u: the uniform.  Returns 0 if equal, 1 for an accepted near-
    boundary flip; raises otherwise."""
    if idx_gpu == idx_ref:
        return 0
    masses = np.asarray(masses, dtype=np.float64)
    cum = np.cumsum(masses)
    total = cum[-1]
    thr = u * total
    lo, hi = min(idx_gpu, idx_ref), max(idx_gpu, idx_ref)
    assert abs(cum[lo] - thr) <= tol * total, ("draw", idx_gpu, idx_ref, cum[lo], thr)
    assert masses[lo + 1:hi].sum() <= tol * total, ("draw skips mass", idx_gpu, idx_ref)
    return 1


def to_np(t):
    return t.detach().cpu().numpy()


def tree_np(out, t=0):
    """One tree of a tsd_build_tree result as numpy arrays."""
    return {k: to_np(out[k][t]) for k in ("parent", "token", "depth", "score", "rank", "mode")} | \
        {"n_nodes": int(out["n_nodes"][t])}


def oracle_build(orc, drafter, k, B, temp=1.0):
    """drafter: [K, L, V] torch (any float dtype) -> oracle tree + lists."""
    z = drafter.float().cpu().numpy().astype(np.float64)
    lists = orc.drafter_lists(z, temp, k)
    return orc.build_tree(lists, B), lists


def check_tev(out, t, o, tgt64, parent, token, n, T):
    """One tree of a tsd_verify_tev result against the oracle's TEV `o` on the
    same tree: masses within RTOL; exit node, bonus token and accepted length
    exact up to counted near-boundary draw flips (returned)."""
    import oracle
    ok, err = close(to_np(out["exit_mass"][t])[:n], o["w"])
    assert ok, ("w", err)
    ok, err = close(to_np(out["prefix_prob"][t])[:n], o["P"])
    assert ok, ("P", err)
    ok, err = close(float(out["coverage"][t]), o["coverage"])
    assert ok, ("C_p", err)
    assert int(out["status"][t]) == 0
    ex = int(out["exit_node"][t])
    flips = check_draw(ex, o["exit_node"], o["w"], o["u_exit"])
    if ex == o["exit_node"]:
        p = oracle.row_probs(tgt64[ex], T)
        kids = [int(token[u]) for u in range(1, n) if int(parent[u]) == ex]
        p[kids] = 0.0
        flips += check_draw(int(out["bonus_token"][t]), o["bonus"], p, o["u_bonus"])
        assert int(out["accept_len"][t]) == o["accept_len"]
    return flips


def check_batch_valid(out, tree, T):
    """Whole-launch validity of a TEV result on GPU-built trees: every tree's
    status is ok, its exit masses sum to one, its exit node is a node, its
    accepted length is the exit node's depth + 1, and its bonus token is not a
    drafted child of the exit node (at T = 0 as well: the arg-max is then not a
    child)."""
    nt = int(tree["n_nodes"].shape[0])
    st = to_np(out["status"])
    assert st.tolist() == [0] * nt, st
    w = to_np(out["exit_mass"]).astype(np.float64)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-4), w.sum(axis=1)
    nn = to_np(tree["n_nodes"])
    par, tok, dep = to_np(tree["parent"]), to_np(tree["token"]), to_np(tree["depth"])
    ex, bon, acc = to_np(out["exit_node"]), to_np(out["bonus_token"]), to_np(out["accept_len"])
    for t in range(nt):
        n = int(nn[t])
        assert 0 <= ex[t] < n and w[t, ex[t]] > 0.0
        assert acc[t] == dep[t, ex[t]] + 1
        kids = tok[t, 1:n][par[t, 1:n] == ex[t]]
        assert bon[t] >= 0 and bon[t] not in kids, (t, bon[t])

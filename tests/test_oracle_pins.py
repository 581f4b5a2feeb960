"""Pins for the float64 oracle: each check compares it with something other
than itself -- a library routine, brute force on tiny inputs, a closed form
the pages print, or a fixture worked by hand from the definitions.

Page titles cited below:
  [EXIT] Where Draft Trees Lose Target Mass: Exit-Guided Speculative Decoding
  [CAST] CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters
  [MFD]  Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
         Speculative Decoding
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers written independently of the oracle
# --------------------------------------------------------------------------
def children_of(parent, n):
    ch = {v: [] for v in range(n)}
    for u in range(1, n):
        ch[int(parent[u])].append(u)
    return ch


def depths_of(parent, n):
    d = [0] * n
    for u in range(1, n):
        d[u] = d[int(parent[u])] + 1
    return d


def probs_library(z, T):
    """p_v = softmax(z/T) via scipy, or one-hot at the lowest arg-max at T=0."""
    z = np.asarray(z, dtype=np.float64)
    if T == 0:
        p = np.zeros_like(z)
        p[int(np.argmax(z))] = 1.0  # numpy argmax returns the first maximum
        return p
    return scipy.special.softmax(z / T)


def brute_force_continuations(z, parent, token, n, T):
    """Enumerate every target continuation through the tree: the joint law of
    (exit node, next token) and the reach probability of every node."""
    ch = children_of(parent, n)
    probs = [probs_library(z[v], T) for v in range(n)]
    joint = np.zeros((n, z.shape[1]))
    reach = np.zeros(n)

    def walk(v, q):
        reach[v] += q
        kids = {int(token[u]): u for u in ch[v]}
        for a in range(z.shape[1]):
            pa = q * probs[v][a]
            if a in kids:
                walk(kids[a], pa)
            else:
                joint[v, a] += pa

    walk(0, 1.0)
    return joint, reach, probs


def tiny_tree(orc, seed, B=8, k=4, T_d=1.0):
    dr = synth.tiny_drafter(seed).numpy().astype(np.float64)
    tr = orc.build_tree(orc.drafter_lists(dr, T_d, k), B)
    n = tr["n_nodes"]
    tgt = synth.tiny_target(synth.tiny_drafter(seed), tr["depth"][:n], seed + 7).numpy()
    return dr, tr, n, tgt.astype(np.float64)


# --------------------------------------------------------------------------
# Philox4x64-10 and the uniforms
# --------------------------------------------------------------------------
def _numpy_philox_block(counter, key):
    """numpy's Philox (4x64, 10 rounds) pre-increments its 256-bit counter, so
    the block at counter c is produced from a generator set to c - 1."""
    c = sum(int(x) << (64 * i) for i, x in enumerate(counter))
    c = (c - 1) % (1 << 256)
    words = np.array([(c >> (64 * i)) & ((1 << 64) - 1) for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=words)
    return bg.random_raw(4).astype(np.uint64)


@pytest.mark.parametrize("counter,key", [
    ((0, 0, 0, 0), (0, 0)),
    ((1, 0, 0, 0), (0, 0)),
    ((5, 6, 7, 8), (123456789, 987654321)),
    ((31, 512, 2, 0), (20261202, 0)),
    ((2**64 - 1, 2**64 - 1, 3, 0), (2**64 - 1, 17)),
])
def test_philox_matches_numpy(orc, counter, key):
    """The generator's published known-answer vectors are not available to
    these tests, so the pin is an independent implementation instead:
    numpy's Philox4x64-10, including a carry through all four counter words."""
    ours = orc.philox4x64_10(counter, key)
    ref = _numpy_philox_block(counter, key)
    assert [int(x) for x in ours] == [int(x) for x in ref]


def test_uniform_grid_and_uniformity(orc):
    us = np.array([orc.uniform(99, t, 0, 0) for t in range(40000)])
    assert us.min() >= 0.0 and us.max() < 1.0
    assert np.all(us * 2**24 == np.floor(us * 2**24))
    # the stream and node fields change the draw
    assert orc.uniform(1, 2, 3, 0) != orc.uniform(1, 2, 3, 1)
    assert orc.uniform(1, 2, 3, 0) != orc.uniform(1, 2, 4, 0)
    hist = np.histogram(us, bins=64, range=(0, 1))[0]
    assert scipy.stats.chisquare(hist).pvalue > 1e-4
    # lag-1 correlation near zero
    assert abs(np.corrcoef(us[:-1], us[1:])[0, 1]) < 0.03


# --------------------------------------------------------------------------
# Drafter statistics [CAST Sec. 2 Eq. 1, App. C]
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.6, 2.5])
def test_drafter_stats_vs_library(orc, T):
    rng = np.random.default_rng(5)
    z = np.round(rng.normal(0, 3, size=(6, 200)) * 2) / 2  # quantised: many exact ties
    z[2, 17] = -np.inf  # a masked token
    lse, tid, tlq = orc.drafter_stats(z, T, 8)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z / T, axis=1), rtol=0, atol=1e-12)
    for r in range(z.shape[0]):
        order = np.lexsort((np.arange(z.shape[1]), -z[r]))  # logit desc, id asc
        assert list(tid[r]) == list(order[:8])
        np.testing.assert_allclose(tlq[r], scipy.special.log_softmax(z[r] / T)[order[:8]], atol=1e-12)


def test_drafter_stats_rejects_nonfinite(orc):
    z = np.zeros((2, 16))
    z[1, 3] = np.nan
    with pytest.raises(orc.OracleError) as e:
        orc.drafter_stats(z, 1.0, 4)
    assert e.value.code == orc.ERR_NONFINITE


# --------------------------------------------------------------------------
# Builder [CAST Thm. 1, App. C; MFD Sec. 4.3, App. B Prop. 6]
# --------------------------------------------------------------------------
def exhaustive_topB(lists, B):
    """Enumerate every prefix of every mode's capped universe, score it, keep
    each distinct token sequence at its best entry in the order (score desc,
    depth asc, mode asc, rank sequence asc), and return the first B.  A score
    is the left-to-right sum of the scaled logits along the prefix minus the
    sum of the rows' log-normalisers up to its depth (the sum of log q)."""
    top_id, top_zt, lse = lists["top_id"], lists["top_zt"], lists["lse"]
    K, L, k = top_id.shape
    entries = []
    for m in range(K):
        cum = [0.0]
        for j in range(L):
            cum.append(cum[-1] + lse[m, j])
        for d in range(1, L + 1):
            for ranks in itertools.product(range(k), repeat=d):
                z = 0.0
                for j, r in enumerate(ranks):
                    z = z + top_zt[m, j, r]
                s = z - cum[d]
                if s == -np.inf:
                    continue
                toks = tuple(int(top_id[m, j, r]) for j, r in enumerate(ranks))
                entries.append((-s, d, m, ranks, toks, s))
    entries.sort(key=lambda e: (e[0], e[1], e[2], e[3]))
    seen, out = set(), []
    for e in entries:
        if e[4] in seen:
            continue
        seen.add(e[4])
        out.append(e)
        if len(out) == B:
            break
    return out


def tree_sequences(tr):
    n = tr["n_nodes"]
    seqs = {0: ()}
    for u in range(1, n):
        seqs[u] = seqs[int(tr["parent"][u])] + (int(tr["token"][u]),)
    return [seqs[u] for u in range(n)]


def _random_lists(rng, K, L, k, V, quantise=False):
    tid = np.zeros((K, L, k), dtype=np.int32)
    tzt = np.zeros((K, L, k))
    lse = np.zeros((K, L))
    for m in range(K):
        for j in range(L):
            z = rng.normal(0, 2, size=V)
            if quantise:
                z = np.round(z * 2) / 2
            order = np.lexsort((np.arange(V), -z))[:k]
            tid[m, j], tzt[m, j], lse[m, j] = order, z[order], scipy.special.logsumexp(z)
    return dict(top_id=tid, top_zt=tzt, lse=lse)


def _sub(lists, m0, m1):
    return {key: v[m0:m1] for key, v in lists.items()}


def _cat(a, b):
    return {key: np.concatenate([a[key], b[key]]) for key in a}


@pytest.mark.parametrize("seed", range(12))
def test_builder_single_mode_equals_exhaustive(orc, seed):
    rng = np.random.default_rng(seed)
    L, k, V = 4, 4, 12
    ls = _random_lists(rng, 1, L, k, V, quantise=(seed % 2 == 1))
    B = int(rng.integers(1, 60))
    tr = orc.build_tree(ls, B)
    ref = exhaustive_topB(ls, B)
    seqs = tree_sequences(tr)
    assert tr["n_nodes"] == len(ref) + 1
    assert seqs[1:] == [e[4] for e in ref]
    np.testing.assert_array_equal(tr["score"][1:tr["n_nodes"]], [e[5] for e in ref])
    # prefix-closed [CAST Thm. 1]: every parent precedes its child
    for u in range(1, tr["n_nodes"]):
        assert 0 <= tr["parent"][u] < u
        assert tr["depth"][u] == tr["depth"][tr["parent"][u]] + 1


def test_builder_scores_never_rise_along_a_path(orc):
    """A prefix's sum of log q cannot exceed its parent's ([CAST] Sec. 2
    Eq. 1: every log q is at most 0).  Fixture: depth 1 has z/T = 0.8758...
    under LSE 3.5232... (log q < 0); depth 2's only token has z/T equal to
    its LSE (q = 1).  Evaluated as (path sum) - C(d), the depth-2 score
    rounds 4.4e-16 above the depth-1 score; the builder takes the parent's
    score there, under both push rules, so the child ties its parent and
    follows it.  Found by a random search over float64 values."""
    a, b, x = 0.8758060614355943, 3.5232430639311674, 3.461974184283127
    assert (a + x) - (b + x) > a - b  # the fixture does round upward
    ls = dict(top_id=np.array([[[5], [9]]], dtype=np.int32),
              top_zt=np.array([[[a], [x]]]), lse=np.array([[b, x]]))
    for rule in (0, 1):
        tr = orc.build_tree(ls, 2, push_rule=rule)
        assert tr["n_nodes"] == 3
        assert tr["parent"][1:3].tolist() == [0, 1]
        assert tr["token"][1:3].tolist() == [5, 9]
        assert tr["score"][1] == a - b and tr["score"][2] == tr["score"][1]


@pytest.mark.parametrize("seed", range(4))
def test_builder_scores_never_rise_random(orc, seed):
    """The same property on random lists whose rows are certain (q = 1,
    z/T = LSE) at random positions: every node's score is at most its
    parent's, and parents precede children."""
    rng = np.random.default_rng(900 + seed)
    K, L, k = 1 + seed % 2, 6, 3
    zt = rng.uniform(-8.0, 8.0, size=(K, L, k))
    zt = -np.sort(-zt, axis=-1)
    lse = zt[..., 0] + rng.uniform(0.0, 2.0, size=(K, L))
    certain = rng.random((K, L)) < 0.5
    lse = np.where(certain, zt[..., 0], lse)  # rank 0 carries all the mass
    ids = np.broadcast_to(np.arange(k, dtype=np.int32), (K, L, k)).copy()
    tr = orc.build_tree(dict(top_id=ids, top_zt=zt, lse=lse), 60)
    for u in range(1, tr["n_nodes"]):
        p = tr["parent"][u]
        assert 0 <= p < u
        if p > 0:
            assert tr["score"][u] <= tr["score"][p]


@pytest.mark.parametrize("seed", range(8))
def test_push_rules_agree(orc, seed):
    """Sibling+first-child pushes [MFD App. B] and push-all-k-children
    [CAST App. C] pop the same prefixes in the same order."""
    rng = np.random.default_rng(100 + seed)
    K = 1 + seed % 3
    ls = _random_lists(rng, K, 5, 6, 20, quantise=(seed % 2 == 0))
    for B in (1, 7, 40, 90):
        a = orc.build_tree(ls, B, push_rule=0)
        b = orc.build_tree(ls, B, push_rule=1)
        for key in ("parent", "token", "depth", "rank", "mode"):
            np.testing.assert_array_equal(a[key], b[key])
        np.testing.assert_array_equal(a["score"], b["score"])


def test_mixture_equals_exhaustive_random_instances(orc):
    """Random instances in the manner of [MFD App. B] (up to 8 modes, small
    positions and vocabularies, budgets up to 40, cap = whole vocabulary so
    Prop. 6 is exact): the merged heap returns the B best distinct prefixes
    under the best-mode score."""
    rng = np.random.default_rng(2026)
    for inst in range(120):
        K = int(rng.integers(1, 9))
        L = int(rng.integers(1, 4))
        V = int(rng.integers(2, 6))
        ls = _random_lists(rng, K, L, V, V, quantise=(inst % 3 == 0))
        B = int(rng.integers(1, 41))
        tr = orc.build_tree(ls, B)
        ref = exhaustive_topB(ls, B)
        assert tree_sequences(tr)[1:] == [e[4] for e in ref], inst
        np.testing.assert_array_equal(tr["score"][1:tr["n_nodes"]], [e[5] for e in ref])
    # two instances at the page's full size: 5 positions, 10 tokens each
    for inst in range(2):
        K = 2 + inst
        ls = _random_lists(rng, K, 5, 10, 10)
        tr = orc.build_tree(ls, 40)
        ref = exhaustive_topB(ls, 40)
        assert tree_sequences(tr)[1:] == [e[4] for e in ref]


def test_mixture_single_mode_is_ddtree(orc):
    """With K = 1 the merged heap is DDTree's builder [MFD App. B Prop. 6]:
    check the K = 1 call against the mixture call with the one mode duplicated
    under a second copy -- the duplicate reuses every node."""
    rng = np.random.default_rng(7)
    ls = _random_lists(rng, 1, 6, 8, 40)
    single = orc.build_tree(ls, 64)
    dup = orc.build_tree(_cat(ls, ls), 64)
    for key in ("parent", "token", "depth", "score"):
        np.testing.assert_array_equal(single[key], dup[key])
    assert np.all(dup["mode"][1:dup["n_nodes"]] == 0)


def test_mixture_is_union_of_mode_trees(orc):
    """[MFD Sec. 3.4 Prop. 4]: without ties the mixture tree is the union of
    the per-mode top-n_k trees, n_k = #{v : log Q_k(v) >= theta}."""
    rng = np.random.default_rng(11)
    for _ in range(10):
        K = int(rng.integers(2, 6))
        ls = _random_lists(rng, K, 3, 5, 5)
        B = int(rng.integers(5, 40))
        tr = orc.build_tree(ls, B)
        n = tr["n_nodes"]
        theta = tr["score"][n - 1]
        union = set()
        for m in range(K):
            one = exhaustive_topB(_sub(ls, m, m + 1), 10**9)
            nk = sum(1 for e in one if e[5] >= theta)
            sub = orc.build_tree(_sub(ls, m, m + 1), nk)
            union |= set(tree_sequences(sub)[1:])
        assert union == set(tree_sequences(tr)[1:])


def test_product_tree_holds_chimeras(orc):
    """[MFD Sec. 3.2 Lemma 1]: if a product's top-B tree (no ties) holds two
    depth-d prefixes differing in m positions, it holds at least 2^(m-1) of
    their splices."""
    rng = np.random.default_rng(3)
    for _ in range(6):
        ls = _random_lists(rng, 1, 4, 4, 4)
        tr = orc.build_tree(ls, 60)
        seqs = set(tree_sequences(tr)[1:])
        by_depth = {}
        for s in seqs:
            by_depth.setdefault(len(s), []).append(s)
        for d, group in by_depth.items():
            for v, w in itertools.combinations(group, 2):
                diff = [i for i in range(d) if v[i] != w[i]]
                m = len(diff)
                splices = set()
                for mask in range(1 << m):
                    u = list(w)
                    for b, i in enumerate(diff):
                        if mask >> b & 1:
                            u[i] = v[i]
                    splices.add(tuple(u))
                assert len(splices & seqs) >= 2 ** (m - 1)


def _separation_lists(futures, modes_on, k, D):
    """Point-mass modes: mode m puts all mass on future modes_on[m]."""
    K = len(modes_on)
    tid = np.zeros((K, D, k), dtype=np.int32)
    tlq = np.full((K, D, k), -np.inf)
    for m, f in enumerate(modes_on):
        for i in range(D):
            others = [t for t in range(k + len(futures)) if t != futures[f][i]][:k - 1]
            tid[m, i] = [futures[f][i]] + others
            tlq[m, i, 0] = 0.0
    return {"top_id": tid, "top_zt": tlq, "lse": np.zeros((K, D))}


def _acceptance(tr, futures, mu):
    """E[alpha] = sum over tree nodes of the target prefix mass [MFD Prop. 1]."""
    acc = 0.0
    for s in tree_sequences(tr)[1:]:
        for f, m in zip(futures, mu):
            if tuple(f[:len(s)]) == s:
                acc += m
    return acc


def test_separation_model_closed_forms(orc):
    cases = json.load(open(os.path.join(GOLDEN, "mfd_separation.json")))["cases"]
    # case 1: M=2, D=15, B=256
    c = cases[0]
    M, D, B = c["M"], c["D"], c["B"]
    futures = [[2 * i for i in range(D)], [2 * i + 1 for i in range(D)]]
    mix = orc.build_tree(_separation_lists(futures, [0, 1], 2, D), B)
    assert _acceptance(mix, futures, [0.5, 0.5]) == pytest.approx(c["optimal"])
    rng = np.random.default_rng(1)
    for _ in range(20):  # random products over the two futures' tokens, no ties
        tid = np.zeros((1, D, 2), dtype=np.int32)
        tlq = np.zeros((1, D, 2))
        for i in range(D):
            a = rng.uniform(0.05, 0.95)
            pair = sorted([(a, futures[0][i]), (1 - a, futures[1][i])], reverse=True)
            tid[0, i] = [pair[0][1], pair[1][1]]
            tlq[0, i] = [math.log(pair[0][0]), math.log(pair[1][0])]
        prod = orc.build_tree(orc.lists_from_logq(tid, tlq), B)
        assert _acceptance(prod, futures, [0.5, 0.5]) <= c["product_bound"] + 1e-12
        assert D / M + (1 - 1 / M) * (1 + math.log2(B)) == pytest.approx(c["product_bound"])
    # case 2: unequal futures
    c = cases[1]
    D, B, mu = c["D"], c["B"], c["mu"]
    futures = [[2 * i for i in range(D)], [2 * i + 1 for i in range(D)]]
    mix = orc.build_tree(_separation_lists(futures, [0, 1], 2, D), B)
    assert _acceptance(mix, futures, mu) == pytest.approx(c["uniform_prior_mixture"])
    eps = 1e-3
    tid = np.zeros((1, D, 2), dtype=np.int32)
    tlq = np.zeros((1, D, 2))
    for i in range(D):
        tid[0, i] = [futures[0][i], futures[1][i]]
        tlq[0, i] = [math.log(1 - eps), math.log(eps)]
    prod = orc.build_tree(orc.lists_from_logq(tid, tlq), B)
    assert _acceptance(prod, futures, mu) == pytest.approx(c["product_on_first"])
    # case 3: point-mass mixture accepts min(B, K D)/M
    c = cases[2]
    M, K, D = c["M"], c["K"], c["D"]
    futures = [[M * i + f for i in range(D)] for f in range(M)]
    for B in c["B_list"]:
        mix = orc.build_tree(_separation_lists(futures, list(range(K)), 2, D), B)
        assert _acceptance(mix, futures, [1 / M] * M) == pytest.approx(min(B, K * D) / M)
        assert mix["n_nodes"] == min(B, K * D) + 1  # zero-mass prefixes are never kept


# --------------------------------------------------------------------------
# Ancestor mask and position ids [CAST App. C, Lemma 1]
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_tree_mask_vs_ancestor_sets(orc, seed):
    rng = np.random.default_rng(seed)
    ls = _random_lists(rng, 1, 6, 4, 10)
    B = 40
    tr = orc.build_tree(ls, B)
    n = tr["n_nodes"]
    P = int(rng.integers(0, 50))
    bits, pos, add = orc.tree_mask(tr["parent"], n, B, P, with_additive=True)
    dep = depths_of(tr["parent"], n)
    for v in range(B + 1):
        got = {u for u in range(B + 1) if bits[v, u // 32] >> (u % 32) & 1}
        if v < n:
            anc, u = set(), v
            while u >= 0:
                anc.add(u)
                u = int(tr["parent"][u])
            assert got == anc and len(got) == dep[v] + 1
            assert pos[v] == P + dep[v]
        else:
            assert got == {v} and pos[v] == P
        assert np.all(add[v, :P] == 0.0)
        for u in range(B + 1):
            assert add[v, P + u] == (0.0 if u in got else -np.inf)
    # transitively closed: an ancestor's ancestors are ancestors
    for v in range(n):
        for u in range(n):
            if bits[v, u // 32] >> (u % 32) & 1:
                for x in range(n):
                    if bits[u, x // 32] >> (x % 32) & 1:
                        assert bits[v, x // 32] >> (x % 32) & 1


# --------------------------------------------------------------------------
# TEV [EXIT Sec. 3, App. A, App. B Algorithm 1]
# --------------------------------------------------------------------------
def test_tev_hand_fixture(orc):
    g = json.load(open(os.path.join(GOLDEN, "tev_hand_v3.json")))
    par, tok = g["tree"]["parent"], g["tree"]["token"]
    z = np.log(np.array(g["p"]))
    r = orc.tev(z, par, tok, 4, 1.0, seed=1)
    e = g["expected"]
    np.testing.assert_allclose(r["P"], e["P"], atol=1e-14)
    np.testing.assert_allclose(r["rho"], e["rho"], atol=1e-14)
    np.testing.assert_allclose(r["w"], e["w"], atol=1e-14)
    assert r["coverage"] == pytest.approx(e["coverage"], abs=1e-14)
    # the residual law the bonus is drawn from, by exhaustive draws over the
    # uniform grid is too costly; check it through the brute-force joint law
    joint, _, _ = brute_force_continuations(z, par, tok, 4, 1.0)
    for v in range(4):
        np.testing.assert_allclose(joint[v] / joint[v].sum(), e["residual"][v], atol=1e-14)


@pytest.mark.parametrize("T", [1.0, 0.6, 0.0])
@pytest.mark.parametrize("seed", range(5))
def test_tev_exit_law_by_brute_force(orc, T, seed):
    """Enumerating target continuations [EXIT Lemma 1, Eq. 5-6, 24-29]."""
    _, tr, n, tgt = tiny_tree(orc, 1000 + seed)
    par, tok = tr["parent"], tr["token"]
    r = orc.tev(tgt, par, tok, n, T, seed=seed)
    joint, reach, _ = brute_force_continuations(tgt, par, tok, n, T)
    dep = depths_of(par, n)
    ch = children_of(par, n)
    np.testing.assert_allclose(r["w"], joint.sum(axis=1), atol=1e-13)   # Lemma 1
    assert r["w"].sum() == pytest.approx(1.0, abs=1e-13)                  # Eq. 5
    np.testing.assert_allclose(r["P"], reach, atol=1e-13)                # Eq. 2, 20
    exp_len = sum(joint[v].sum() * (dep[v] + 1) for v in range(n))
    assert exp_len == pytest.approx(1.0 + r["coverage"], abs=1e-12)       # Thm. 1 at equality
    assert r["coverage"] == pytest.approx(sum(r["w"][v] * dep[v] for v in range(n)), abs=1e-12)
    for v in range(n):  # local conservation, Eq. 24-25
        assert r["w"][v] + sum(r["P"][u] for u in ch[v]) == pytest.approx(r["P"][v], abs=1e-13)
        # Eq. 4 directly: rho = 1 - sum of child probabilities
        assert r["rho"][v] == pytest.approx(1.0 - sum(r["pedge"][u] for u in ch[v]), abs=1e-12)
    for u in range(n):  # subtree sums, Eq. 26
        sub = [v for v in range(n) if _in_subtree(v, u, par)]
        assert sum(r["w"][v] for v in sub) == pytest.approx(r["P"][u], abs=1e-12)
    assert r["accept_len"] == dep[r["exit_node"]] + 1


def _in_subtree(v, u, par):
    while v >= 0:
        if v == u:
            return True
        v = int(par[v])
    return False


def test_one_step_coverage_gain(orc):
    """[EXIT Eq. 12-13]: adding child (v, a) raises C_p by P(v) p_v(a); the
    sum over the missing tokens is w(v)."""
    _, tr, n, tgt = tiny_tree(orc, 77)
    par, tok = list(tr["parent"][:n]), list(tr["token"][:n])
    base = orc.tev(tgt, par, tok, n, 1.0, seed=3)
    ch = children_of(par, n)
    v = max(range(n), key=lambda x: base["w"][x])
    taken = {tok[u] for u in ch[v]}
    gains = 0.0
    p_v = probs_library(tgt[v], 1.0)
    for a in range(tgt.shape[1]):
        if a in taken:
            continue
        z2 = np.vstack([tgt, tgt[:1]])  # the new node's own row does not enter C_p
        r2 = orc.tev(z2, par + [v], tok + [a], n + 1, 1.0, seed=3)
        gain = r2["coverage"] - base["coverage"]
        assert gain == pytest.approx(base["P"][v] * p_v[a], abs=1e-13)
        gains += gain
    assert gains == pytest.approx(base["w"][v], abs=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_greedy_is_argmax_walk(orc, seed):
    """T = 0 reduces to following the target arg-max [CAST Sec. 2, Sec. 3.4]."""
    _, tr, n, tgt = tiny_tree(orc, 500 + seed)
    par, tok = tr["parent"], tr["token"]
    ch = children_of(par, n)
    v = 0
    while True:
        a = int(np.argmax(tgt[v]))
        nxt = [u for u in ch[v] if int(tok[u]) == a]
        if not nxt:
            break
        v = nxt[0]
    for s in range(3):
        r = orc.tev(tgt, par, tok, n, 0.0, seed=s)
        assert (r["exit_node"], r["bonus"]) == (v, int(np.argmax(tgt[v])))
        d = orc.predraw(tgt, par, tok, n, 0.0, seed=s)
        assert (d["exit_node"], d["bonus"]) == (v, int(np.argmax(tgt[v])))


def test_tev_and_predraw_share_the_exact_law(orc):
    """Chi-square over 10^6 seeded draws of each sampler against the exact
    joint law P(v) rho(v) p_v^res(a) from brute force [EXIT Thm. 1, Cor. 1,
    Eq. 10, 56], and against each other; acceptance frequency = P(u) [Eq. 58]."""
    _, tr, n, tgt = tiny_tree(orc, 4242)
    par, tok = tr["parent"], tr["token"]
    T = 1.0
    joint, _, _ = brute_force_continuations(tgt, par, tok, n, T)
    N = 1_000_000
    draws = {}
    for kind in ("tev", "predraw"):
        ex, bo = orc.sample_many(kind, tgt, par, tok, n, T, seed=31337, n_draws=N)
        draws[kind] = (ex, bo)
        cells = ex.astype(np.int64) * tgt.shape[1] + bo
        obs = np.bincount(cells, minlength=joint.size).astype(float)
        exp = joint.ravel() * N
        assert obs[exp == 0].sum() == 0, kind  # zero-mass events never happen
        keep = exp >= 5
        rest_o, rest_e = obs[~keep].sum(), exp[~keep].sum()
        o = np.append(obs[keep], rest_o)
        e = np.append(exp[keep], rest_e)
        assert scipy.stats.chisquare(o, e * o.sum() / e.sum()).pvalue > 1e-4, kind
        # exit-node law alone
        eo = np.bincount(ex, minlength=n).astype(float)
        ew = joint.sum(axis=1) * N
        k2 = ew > 0
        assert scipy.stats.chisquare(eo[k2], ew[k2] * eo[k2].sum() / ew[k2].sum()).pvalue > 1e-4
    # the two samplers against each other (two-sample chi-square on exit nodes)
    a = np.bincount(draws["tev"][0], minlength=n)
    b = np.bincount(draws["predraw"][0], minlength=n)
    m = (a + b) > 0
    assert scipy.stats.chi2_contingency(np.vstack([a[m], b[m]]))[1] > 1e-4
    # acceptance frequency of every node equals P(u)
    r = orc.tev(tgt, par, tok, n, T, seed=0)
    ex = draws["tev"][0]
    for u in range(1, n):
        sub = np.array([_in_subtree(v, u, par) for v in range(n)])
        f = sub[ex].mean()
        sd = math.sqrt(r["P"][u] * (1 - r["P"][u]) / N) + 1e-12
        assert abs(f - r["P"][u]) < 5 * sd


def test_tev_rejects_bad_trees(orc):
    z = np.zeros((3, 8))
    with pytest.raises(orc.OracleError):
        orc.tev(z, [-1, 0, 0], [-1, 2, 2], 3, 1.0, 0)  # sibling tokens repeat
    with pytest.raises(orc.OracleError):
        orc.tev(z, [-1, 2, 0], [-1, 1, 2], 3, 1.0, 0)  # parent after child
    with pytest.raises(orc.OracleError):
        orc.tev(z, [-1, 0, 0], [-1, 1, 8], 3, 1.0, 0)  # token out of range


def _numpy_uniform(seed, tree, node, stream):
    """The uniform of the stated reading, from numpy's Philox: the top 24 bits
    of the first output word of counter (tree, node, stream, 0), key (seed, 0)."""
    x0 = int(_numpy_philox_block((tree, node, stream, 0), (seed, 0))[0])
    return (x0 >> 40) * 2.0**-24


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_draws_are_inverse_cdf_of_the_stated_uniforms(orc, T):
    """The reading of TEV's two draws [EXIT App. B]: inverse CDF over nodes
    in index order (exit) and over non-child token ids ascending (bonus), with
    the uniforms of the counter layout above.  Exit law and residual law come
    from brute force, the uniforms from numpy -- nothing from the oracle."""
    _, tr, n, tgt = tiny_tree(orc, 9090)
    par, tok = tr["parent"], tr["token"]
    joint, _, probs = brute_force_continuations(tgt, par, tok, n, T)
    w = joint.sum(axis=1)
    ch = children_of(par, n)
    for tree in range(300):
        u1 = _numpy_uniform(5, tree, 0, 0)
        u2 = _numpy_uniform(5, tree, 0, 1)
        cw = np.cumsum(w)
        ex = int(np.argmax(cw > u1 * cw[-1]))
        kids = {int(tok[u]) for u in ch[ex]}
        res = np.array([0.0 if a in kids else probs[ex][a] for a in range(tgt.shape[1])])
        cr = np.cumsum(res)
        bo = int(np.argmax(cr > u2 * cr[-1]))
        r = orc.tev(tgt, par, tok, n, T, seed=5, tree=tree)
        assert (r["exit_node"], r["bonus"]) == (ex, bo), tree
        # predraw: R_v is the inverse CDF of p_v at the node's own uniform
        d = orc.predraw(tgt, par, tok, n, T, seed=5, tree=tree)
        for v in range(n):
            cp = np.cumsum(probs[v])
            assert d["draws"][v] == int(np.argmax(cp > _numpy_uniform(5, tree, v, 2) * cp[-1]))


# ---------------------------------------------------------------------------
# Exit-guided loss ([EXIT] Sec. 5 Eq. 14, App. C.2 Eq. 66)
# ---------------------------------------------------------------------------
def _exit_loss_case(seed, L=4, V=50, n=12):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2, size=(L, V))
    depth = np.zeros(n, dtype=np.int32)
    token = np.full(n, -1, dtype=np.int32)
    for v in range(1, n):
        depth[v] = int(rng.integers(1, L + 1))
        token[v] = int(rng.integers(0, V))
    omega = rng.random(n)
    return z, token, depth, omega


def test_exit_loss_hand_fixture(orc):
    g = json.load(open(os.path.join(GOLDEN, "exit_loss_hand.json")))
    num, grad = orc.exit_loss(np.array(g["z"]), g["T"], g["token"], g["depth"], len(g["token"]),
                              g["omega"], with_grad=True)
    assert num == pytest.approx(g["numerator"], rel=1e-14)
    assert np.allclose(grad, np.array(g["grad"]), rtol=1e-13, atol=1e-15)


def test_exit_loss_constant_rows_cost_log_V(orc):
    """Every token equally likely: -log q = log V at every node."""
    z, token, depth, omega = _exit_loss_case(3)
    z[:] = 1.7
    num = orc.exit_loss(z, 0.8, token, depth, len(token), omega)
    assert num == pytest.approx(np.log(z.shape[1]) * omega[1:].sum(), rel=1e-12)


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_exit_loss_matches_library_log_softmax(orc, T):
    from scipy.special import log_softmax
    z, token, depth, omega = _exit_loss_case(5)
    want = -sum(omega[v] * log_softmax(z[depth[v] - 1] / T)[token[v]] for v in range(1, len(token)))
    assert orc.exit_loss(z, T, token, depth, len(token), omega) == pytest.approx(want, rel=1e-12)


def test_exit_loss_per_row_regrouping(orc):
    """Eq. 67: one log-normaliser per row, weighted by the row's summed weight,
    minus a gather -- equal to the node-by-node sum of Eq. 66."""
    from scipy.special import logsumexp
    z, token, depth, omega = _exit_loss_case(7)
    W = np.zeros(z.shape[0])
    gather = 0.0
    for v in range(1, len(token)):
        W[depth[v] - 1] += omega[v]
        gather += omega[v] * z[depth[v] - 1, token[v]]
    want = sum(W[m] * logsumexp(z[m]) for m in range(z.shape[0])) - gather
    assert orc.exit_loss(z, 1.0, token, depth, len(token), omega) == pytest.approx(want, rel=1e-12)


def test_exit_loss_gradient_by_finite_differences(orc):
    z, token, depth, omega = _exit_loss_case(9, L=3, V=20)
    T = 0.9
    _, grad = orc.exit_loss(z, T, token, depth, len(token), omega, with_grad=True)
    rng = np.random.default_rng(1)
    h = 1e-6
    for _ in range(12):
        m, a = int(rng.integers(0, z.shape[0])), int(rng.integers(0, z.shape[1]))
        zp, zm = z.copy(), z.copy()
        zp[m, a] += h
        zm[m, a] -= h
        fd = (orc.exit_loss(zp, T, token, depth, len(token), omega)
              - orc.exit_loss(zm, T, token, depth, len(token), omega)) / (2 * h)
        assert fd == pytest.approx(grad[m, a], rel=1e-5, abs=1e-8)


def test_exit_loss_temperature_is_a_logit_scale(orc):
    z, token, depth, omega = _exit_loss_case(11)
    a = orc.exit_loss(z, 1.6, token, depth, len(token), omega)
    b = orc.exit_loss(z / 1.6, 1.0, token, depth, len(token), omega)
    assert a == pytest.approx(b, rel=1e-12)


# ---------------------------------------------------------------------------
# Sequential residual ([EXIT] App. A.4.2) and proposal-aware ([CAST] App. B.1
# Thm. 3) verification
# ---------------------------------------------------------------------------
def _proposal_for(tr, n, dr, T_d=1.0, flat=False):
    """q_child[u]: the drafter's probability of node u's token at u's position,
    or (flat) a deliberately mismatched proposal -- the same for every child."""
    q = np.zeros(n)
    for u in range(1, n):
        d = int(tr["depth"][u])
        q[u] = 1.0 if flat else scipy.special.softmax(dr[d - 1] / T_d)[int(tr["token"][u])]
    return q


@pytest.mark.parametrize("kind,flat", [("seqres", False), ("proposal", False), ("proposal", True)])
def test_new_verifiers_realise_the_exact_law(orc, kind, flat):
    """Chi-square over 10^6 seeded draws against the brute-force joint law of
    (exit node, bonus token), and against TEV's draws [EXIT Eq. 51-53; CAST
    Thm. 3: each committed token follows p_v]."""
    dr, tr, n, tgt = tiny_tree(orc, 4243)
    par, tok = tr["parent"], tr["token"]
    T = 1.0
    joint, _, _ = brute_force_continuations(tgt, par, tok, n, T)
    N = 1_000_000
    q = _proposal_for(tr, n, dr, flat=flat) if kind == "proposal" else None
    ex, bo = orc.sample_many(kind, tgt, par, tok, n, T, seed=777, n_draws=N, q_child=q)
    cells = ex.astype(np.int64) * tgt.shape[1] + bo
    obs = np.bincount(cells, minlength=joint.size).astype(float)
    exp = joint.ravel() * N
    assert obs[exp == 0].sum() == 0
    keep = exp >= 5
    o = np.append(obs[keep], obs[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    assert scipy.stats.chisquare(o, e * o.sum() / e.sum()).pvalue > 1e-4
    ta, _ = orc.sample_many("tev", tgt, par, tok, n, T, seed=778, n_draws=N)
    a, b = np.bincount(ta, minlength=n), np.bincount(ex, minlength=n)
    m = (a + b) > 0
    assert scipy.stats.chi2_contingency(np.vstack([a[m], b[m]]))[1] > 1e-4


@pytest.mark.parametrize("seed", range(4))
def test_new_verifiers_greedy_is_argmax_walk(orc, seed):
    dr, tr, n, tgt = tiny_tree(orc, 600 + seed)
    par, tok = tr["parent"], tr["token"]
    ch = children_of(par, n)
    v = 0
    while True:
        a = int(np.argmax(tgt[v]))
        nxt = [u for u in ch[v] if int(tok[u]) == a]
        if not nxt:
            break
        v = nxt[0]
    q = _proposal_for(tr, n, dr)
    for s in range(3):
        r = orc.seqres(tgt, par, tok, n, 0.0, seed=s)
        assert (r["exit_node"], r["bonus"]) == (v, int(np.argmax(tgt[v])))
        r = orc.proposal(tgt, par, tok, n, 0.0, q, seed=s)
        assert (r["exit_node"], r["bonus"]) == (v, int(np.argmax(tgt[v])))


def _numpy_uniform_sub(seed, tree, node, stream, sub):
    x0 = int(_numpy_philox_block((tree, node, stream, sub), (seed, 0))[0])
    return (x0 >> 40) * 2.0**-24


def test_seqres_decisions_from_the_stated_uniforms(orc):
    """The walk recomputed from brute-force probabilities and numpy-Philox
    uniforms (stream 3 sub j for child j in token order, stream 4 for the
    bonus): nothing from the oracle."""
    _, tr, n, tgt = tiny_tree(orc, 9191)
    par, tok = tr["parent"], tr["token"]
    T = 0.8
    probs = [probs_library(tgt[v], T) for v in range(n)]
    ch = children_of(par, n)
    for tree in range(200):
        v = 0
        while True:
            kids = sorted(ch[v], key=lambda u: int(tok[u]))
            M, nxt = 0.0, None
            for j, u in enumerate(kids):
                pj = probs[v][int(tok[u])]
                if _numpy_uniform_sub(3, tree, v, 3, j) * (1.0 - M) < pj:
                    nxt = u
                    break
                M += pj
            if nxt is None:
                break
            v = nxt
        res = probs[v].copy()
        res[[int(tok[u]) for u in ch[v]]] = 0.0
        cr = np.cumsum(res)
        bo = int(np.argmax(cr > _numpy_uniform_sub(3, tree, v, 4, 0) * cr[-1]))
        r = orc.seqres(tgt, par, tok, n, T, seed=3, tree=tree)
        assert (r["exit_node"], r["bonus"]) == (v, bo), tree


# ---------------------------------------------------------------------------
# Shared budget under load ([CAST] Sec. 3.3 Thm. 2, App. B.4 Prop. 2-3)
# ---------------------------------------------------------------------------
def _forest_instance(rng, R, max_n=12):
    """R requests with random nonincreasing prefix scores (node 0 the root)."""
    stride = max_n + 1
    scores = np.full((R, stride), -np.inf)
    depth = np.zeros((R, stride), dtype=np.int32)
    n = np.zeros(R, dtype=np.int32)
    for r in range(R):
        k = int(rng.integers(0, max_n + 1))
        s = -rng.exponential(1.0, size=k).cumsum() * rng.uniform(0.05, 0.6)  # decreasing
        scores[r, 0] = 0.0
        scores[r, 1:k + 1] = s
        depth[r, 1:k + 1] = rng.integers(1, 5, size=k)
        n[r] = k + 1
    return scores, depth, n


def _throughput(masses_sorted, R, l0, c1, M):
    return (masses_sorted[:M].sum() + R) / (l0 + c1 * M)


@pytest.mark.parametrize("seed", range(40))
def test_forest_select_maximises_batch_throughput(orc, seed):
    """Prop. 3 / Thm. 2: the stopping rule's M* maximises (G(M) + R) / l(M)
    over every allowed total M, G from a brute-force sort of all masses."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    scores, depth, n = _forest_instance(rng, R)
    l0, c1 = float(rng.uniform(0.5, 5)), float(rng.uniform(0.0, 0.4))
    total = int((n - 1).sum())
    M_max = int(rng.integers(0, total + 3))
    out = orc.forest_select(scores, depth, n, M_max, l0, c1)
    masses = np.sort(np.concatenate([np.exp(scores[r, 1:n[r]]) for r in range(R)]))[::-1]
    best = max(_throughput(masses, R, l0, c1, M) for M in range(0, min(M_max, total) + 1))
    assert _throughput(masses, R, l0, c1, out["M"]) == pytest.approx(best, rel=1e-12)
    assert out["G"] == pytest.approx(masses[:out["M"]].sum(), rel=1e-12)
    assert out["width"].sum() == out["M"]


def test_forest_select_cost_slope_limits(orc):
    rng = np.random.default_rng(3)
    scores, depth, n = _forest_instance(rng, 3)
    total = int((n - 1).sum())
    assert orc.forest_select(scores, depth, n, 10**6, 1.0, 0.0)["M"] == total  # width is free
    assert orc.forest_select(scores, depth, n, 5, 1.0, 0.0)["M"] == min(5, total)
    assert orc.forest_select(scores, depth, n, 10**6, 1.0, 1e9)["M"] == 0  # width is ruinous


@pytest.mark.parametrize("seed", range(25))
def test_forest_select_is_the_best_split(orc, seed):
    """Prop. 2: at its total M*, the selection's summed mass equals the best
    over every split of M* among the requests (each taking a prefix of its
    own best-first list), found by exhaustive enumeration."""
    import itertools
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(2, 4))
    scores, depth, n = _forest_instance(rng, R, max_n=6)
    out = orc.forest_select(scores, depth, n, 10**6, float(rng.uniform(0.5, 3)),
                            float(rng.uniform(0.0, 0.3)))
    M = out["M"]
    best = -1.0
    for split in itertools.product(*[range(int(n[r])) for r in range(R)]):
        if sum(split) == M:
            best = max(best, sum(np.exp(scores[r, 1:1 + split[r]]).sum() for r in range(R)))
    got = sum(np.exp(scores[r, 1:1 + out["width"][r]]).sum() for r in range(R))
    assert got == pytest.approx(best, rel=1e-12)


def test_forest_select_with_builder_trees_is_prefix_closed(orc):
    """Composed with the oracle builder: every request keeps the first
    width[r] nodes of its pop order, a prefix-closed tree."""
    R, B = 4, 30
    scores = np.full((R, B + 1), -np.inf)
    depth = np.zeros((R, B + 1), dtype=np.int32)
    parents, n = [], np.zeros(R, dtype=np.int32)
    for r in range(R):
        dr = synth.tiny_drafter(synth.seed_for(0, 300 + r)).numpy().astype(np.float64)
        tr = orc.build_tree(orc.drafter_lists(dr, 1.0, 4), B)
        scores[r, :tr["n_nodes"]] = tr["score"][:tr["n_nodes"]]
        depth[r, :tr["n_nodes"]] = tr["depth"][:tr["n_nodes"]]
        n[r] = tr["n_nodes"]
        parents.append(tr["parent"])
    out = orc.forest_select(scores, depth, n, 60, 2.0, 0.05)
    assert 0 < out["M"] <= 60
    for r in range(R):
        for u in range(1, 1 + int(out["width"][r])):
            assert parents[r][u] < 1 + out["width"][r]


def test_forest_select_tie_order(orc):
    """Equal masses: the shorter prefix first, then the lower request index."""
    scores = np.array([[0.0, -0.5, -0.5], [0.0, -0.5, -0.5]])
    depth = np.array([[0, 2, 2], [0, 1, 2]], dtype=np.int32)
    out = orc.forest_select(scores, depth, np.array([3, 3]), 1, 1.0, 0.0)
    assert out["width"].tolist() == [0, 1]  # request 1's depth-1 node comes first
    out = orc.forest_select(scores, depth, np.array([3, 3]), 2, 1.0, 0.0)
    assert out["width"].tolist() == [1, 1]  # then request 0 (depth 2, lower index) before request 1's depth 2


# --------------------------------------------------------------------------
# mixture tree under the log-sum-exp score ([MFD] App. B Eq. 6)
# --------------------------------------------------------------------------
def _paths(tr):
    return sequences_of(tr["parent"], tr["token"], tr["n_nodes"])[1:]


def sequences_of(parent, token, n):
    seqs = [()]
    for u in range(1, n):
        seqs.append(seqs[int(parent[u])] + (int(token[u]),))
    return seqs


def _brute_lse_tree(z, T, k, B, log_prior=None):
    """From the definitions: each mode's capped universe enumerated, its
    per-depth top-B by the product of softmax probabilities, the union ranked
    by log sum_m pi_m prod_j p_{m,j}(x_j)."""
    K, L, V = z.shape
    with np.errstate(divide="ignore"):
        p = scipy.special.softmax(z / T, axis=-1)
    pi = np.full(K, 1.0 / K) if log_prior is None else np.exp(np.asarray(log_prior, dtype=float))
    caps = [[np.lexsort((np.arange(V), -z[m, j]))[:k] for j in range(L)] for m in range(K)]
    cands = set()
    for m in range(K):
        for d in range(1, L + 1):
            seqs = [s for s in itertools.product(*caps[m][:d])]
            q = [float(np.prod([p[m, j, x] for j, x in enumerate(s)])) for s in seqs]
            ranked = sorted([(qq, tuple(int(x) for x in s)) for qq, s in zip(q, seqs) if qq > 0],
                            key=lambda t: -t[0])
            cands.update(s for _, s in ranked[:B])

    def qbar(s):
        return sum(pi[m] * np.prod([p[m, j, x] for j, x in enumerate(s)]) for m in range(K))

    scored = sorted(((math.log(qbar(s)), s) for s in cands), key=lambda t: -t[0])
    return scored[:B], len(cands), qbar


def test_lse_tree_hand_fixture(orc):
    g = json.load(open(os.path.join(GOLDEN, "lse_tree_hand.json")))
    for ex in g["examples"]:
        z = np.log(np.array(ex["p"]))
        for case in ex["cases"]:
            tr = orc.lse_tree(z, 1.0, ex["k"], case["B"])
            assert tr["n_cand"] == case["n_cand"]
            assert [list(s) for s in _paths(tr)] == case["paths"]
            np.testing.assert_allclose(tr["score"][1:tr["n_nodes"]], np.log(case["qbar"]), rtol=0,
                                       atol=1e-12)


@pytest.mark.parametrize("seed", range(30))
def test_lse_tree_matches_brute_force(orc, seed):
    rng = np.random.default_rng(800 + seed)
    K, L, V = int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(3, 8))
    k, B = int(rng.integers(1, min(V, 4) + 1)), int(rng.integers(1, 13))
    z = rng.normal(size=(K, L, V)) * 1.5
    if seed % 5 == 4:
        z[rng.random(z.shape) < 0.2] = -np.inf      # masked tokens: zero-probability prefixes
        z[..., 0] = np.maximum(z[..., 0], 0.0)      # every row keeps a finite token
    log_prior = None if seed % 2 == 0 else rng.normal(size=K)
    T = [1.0, 0.7, 1.8][seed % 3]
    tr = orc.lse_tree(z, T, k, B, log_prior=log_prior)
    want, n_cand, _ = _brute_lse_tree(z, T, k, B, log_prior)
    assert tr["n_cand"] == n_cand
    assert _paths(tr) == [s for _, s in want]
    np.testing.assert_allclose(tr["score"][1:tr["n_nodes"]], [s for s, _ in want], rtol=0, atol=1e-11)


@pytest.mark.parametrize("seed", range(6))
def test_lse_tree_one_mode_is_the_ddtree_builder(orc, seed):
    rng = np.random.default_rng(900 + seed)
    L, V, k, B = 4, 40, 6, 30
    z = rng.normal(size=(1, L, V)) * 2
    tr = orc.lse_tree(z, 1.0, k, B)
    ref = orc.build_tree(orc.drafter_lists(z, 1.0, k), B)
    assert tr["n_nodes"] == ref["n_nodes"]
    for key in ("parent", "token", "depth"):
        assert np.array_equal(tr[key], ref[key]), key
    assert np.array_equal(tr["score"][1:], ref["score"][1:])


def test_lse_tree_identical_modes_and_prior_shift(orc):
    rng = np.random.default_rng(950)
    z1 = rng.normal(size=(1, 3, 25)) * 2
    one = orc.lse_tree(z1, 1.0, 5, 20)
    for K in (2, 5):
        many = orc.lse_tree(np.repeat(z1, K, axis=0), 1.0, 5, 20)
        assert many["n_cand"] == one["n_cand"]
        assert _paths(many) == _paths(one)
        np.testing.assert_allclose(many["score"], one["score"], rtol=0, atol=1e-12)
    z = rng.normal(size=(3, 3, 25)) * 2
    lp = rng.normal(size=3)
    a = orc.lse_tree(z, 1.0, 5, 20, log_prior=lp)
    b = orc.lse_tree(z, 1.0, 5, 20, log_prior=lp + 2.5)
    assert _paths(a) == _paths(b)
    np.testing.assert_allclose(b["score"][1:], a["score"][1:] + 2.5, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(10))
def test_lse_tree_bounds_and_coverage_against_max_rule(orc, seed):
    """s(v) <= s_lse(v) <= s(v) + log K for every node, with s the best-mode
    score; the tree is prefix-closed with scores falling along paths; its
    mixture mass is at least that of the max rule's tree of the same budget,
    which lies inside the candidate set."""
    rng = np.random.default_rng(1000 + seed)
    K, L, V, k, B = int(rng.integers(2, 6)), 3, 12, 4, int(rng.integers(4, 25))
    z = rng.normal(size=(K, L, V)) * 2
    tr = orc.lse_tree(z, 1.0, k, B)
    _, _, qbar = _brute_lse_tree(z, 1.0, k, B)
    p = scipy.special.softmax(z, axis=-1)
    n = tr["n_nodes"]
    seqs = sequences_of(tr["parent"], tr["token"], n)
    for u in range(1, n):
        s = seqs[u]
        best = max(math.log(np.prod([p[m, j, x] for j, x in enumerate(s)]) / K) for m in range(K))
        assert best - 1e-12 <= tr["score"][u] <= best + math.log(K) + 1e-12
        assert 0 <= tr["parent"][u] < u
        assert tr["score"][u] <= tr["score"][tr["parent"][u]] or tr["parent"][u] == 0
    mx = orc.build_tree(orc.drafter_lists(z, 1.0, k), B)
    mseqs = sequences_of(mx["parent"], mx["token"], mx["n_nodes"])
    assert sum(qbar(s) for s in seqs[1:]) >= sum(qbar(s) for s in mseqs[1:]) - 1e-12


def test_lse_tree_edge_budgets(orc):
    rng = np.random.default_rng(1100)
    z = rng.normal(size=(2, 3, 6))
    assert orc.lse_tree(z, 1.0, 2, 0)["n_nodes"] == 1
    big = orc.lse_tree(z, 1.0, 2, 200)                   # every candidate taken
    assert big["n_nodes"] == big["n_cand"] + 1

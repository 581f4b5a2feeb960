"""GPU parity of the shared-budget width selection ([CAST] Sec. 3.3 Thm. 2,
App. B.4 Prop. 2-3) against the oracle: the oracle builder's tree per
request, merged and cut by the oracle's stopping rule.  The GPU decides the
rule with fp32 masses and float64 sums, so M* may differ by one only where
the rule's two sides are within 1e-6 of each other; the kept trees then
match node for node."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import compare_trees

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


def _oracle_forest(orc, dr, k, B, M_max, l0, c1):
    R = dr.shape[0]
    scores = np.full((R, B + 1), -np.inf)
    depth = np.zeros((R, B + 1), dtype=np.int32)
    n = np.zeros(R, dtype=np.int32)
    trees, lists = [], []
    for r in range(R):
        ls = orc.drafter_lists(dr[r].float().cpu().numpy().astype(np.float64), 1.0, k)
        tr = orc.build_tree(ls, B)
        trees.append(tr)
        lists.append(ls)
        scores[r, :tr["n_nodes"]] = tr["score"][:tr["n_nodes"]]
        depth[r, :tr["n_nodes"]] = tr["depth"][:tr["n_nodes"]]
        n[r] = tr["n_nodes"]
    sel = orc.forest_select(scores, depth, n, M_max, l0, c1)
    return sel, trees, lists, scores, depth, n


def _margin(scores, depth, n, M, l0, c1):
    """|lhs - rhs| of the rule at the oracle's stopping point, relative."""
    masses = np.sort(np.concatenate([np.exp(scores[r, 1:n[r]]) for r in range(len(n))]))[::-1]
    if M >= len(masses):
        return 1.0
    G = masses[:M].sum()
    rhs = c1 * (G + len(n)) / (l0 + c1 * M)
    return abs(masses[M] - rhs) / max(rhs, 1e-300)


@pytest.mark.parametrize("V,dtype,c1", [(synth.V_QWEN, torch.bfloat16, 0.002),
                                        (synth.V_QWEN, torch.bfloat16, 0.02),
                                        (synth.V_QWEN, torch.bfloat16, 0.2),
                                        (4096 + 128, torch.float32, 0.01)])
def test_forest_matches_oracle(tsd, dev, orc, V, dtype, c1):
    R, L, k, B, M_max, l0 = 8, 12, 8, 64, 400, 1.0
    seeds = [synth.seed_for(9, r) for r in range(R)]
    dr = synth.zipf_drafter(R, L, V, 0, device=dev, seeds=seeds, dtype=dtype)
    out = tsd.tsd_build_forest(dr, topk=k, B=B, M_max=M_max, l0=l0, c1=c1)
    sel, trees, lists, scores, depth, n = _oracle_forest(orc, dr[:, 0], k, B, M_max, l0, c1)
    M = int(out["total"])
    assert out["status"].cpu().tolist() == [0] * R
    if M != sel["M"]:
        assert abs(M - sel["M"]) == 1 and _margin(scores, depth, n, min(M, sel["M"]), l0, c1) < 1e-6
        return
    width = (out["n_nodes"] - 1).cpu().numpy()
    assert width.tolist() == sel["width"].tolist()
    assert 0 <= M <= M_max and (M > 0 or c1 * R > l0)   # c1 R > l0: no candidate pays (M* = 0)
    flips = 0
    for r in range(R):
        w = int(width[r])
        got = {key: out[key][r].cpu().numpy() for key in ("parent", "token", "depth", "score")}
        got["n_nodes"] = w + 1
        ref = {key: trees[r][key] for key in ("parent", "token", "depth", "score")}
        ref["n_nodes"] = w + 1
        flips += compare_trees(got, ref, lists[r])
        assert np.all(got["parent"][w + 1:] == -1) and np.all(np.isneginf(got["score"][w + 1:]))
    assert flips <= 2


def test_forest_limits_and_failed_requests(tsd, dev, orc):
    """c1 = 0 keeps every candidate up to M_max; a request with a NaN logit
    fails (status 5, n_nodes 0) and takes no share; too many candidates are
    refused on the host."""
    R, L, k, B, V = 4, 6, 8, 30, 3000
    dr = synth.zipf_drafter(R, L, V, 0, device=dev, seeds=[synth.seed_for(9, 50 + r) for r in range(R)],
                            dtype=torch.float32)
    out = tsd.tsd_build_forest(dr, topk=k, B=B, M_max=10**6, l0=1.0, c1=0.0)
    assert int(out["total"]) == int((out["n_nodes"] - 1).sum()) == R * B
    out = tsd.tsd_build_forest(dr, topk=k, B=B, M_max=37, l0=1.0, c1=0.0)
    assert int(out["total"]) == 37
    dr2 = dr.clone()
    dr2[2, 0, 3, 11] = float("nan")
    out = tsd.tsd_build_forest(dr2, topk=k, B=B, M_max=10**6, l0=1.0, c1=0.0)
    assert out["status"].cpu().tolist() == [0, 0, 5, 0]
    assert int(out["n_nodes"][2]) == 0 and int(out["total"]) == 3 * B
    with pytest.raises(tsd.TsdError):
        tsd.tsd_build_forest(torch.zeros(64, 1, 4, 512, device=dev), topk=4, B=200, M_max=10, l0=1.0, c1=0.1)


def test_forest_in_the_bench_launch(tsd, dev, orc):
    """The bench's launch: 32 requests, V=151936, L=16, top-k 8, cap B=256
    (8192 candidates), l(M) = 1 + M/2048: the oracle builds every request's
    tree and selects; M* and every width must agree."""
    R, L, k, B, l0, c1 = 32, 16, 8, 256, 1.0, 1.0 / 2048
    seeds = [synth.seed_for(2, t) for t in range(R)]
    dr = synth.zipf_drafter(R, L, synth.V_QWEN, 0, device=dev, seeds=seeds)
    out = tsd.tsd_build_forest(dr, topk=k, B=B, M_max=R * B, l0=l0, c1=c1)
    sel, trees, lists, scores, depth, n = _oracle_forest(orc, dr[:, 0], k, B, R * B, l0, c1)
    M = int(out["total"])
    assert out["status"].cpu().tolist() == [0] * R
    if M != sel["M"]:
        assert abs(M - sel["M"]) == 1 and _margin(scores, depth, n, min(M, sel["M"]), l0, c1) < 1e-6
        return
    assert (out["n_nodes"] - 1).cpu().numpy().tolist() == sel["width"].tolist()

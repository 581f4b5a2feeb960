"""GPU parity of the exit-guided loss ([EXIT] Sec. 5 Eq. 14, evaluated via
App. C.2 Eq. 67) against the float64 oracle, which forms Eq. 66 node by
node.  Trees come from the GPU builder and the weights from TEV's exit
masses, as in ExitTrain."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

RTOL = 1e-5


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


def _case(tsd, dev, nt, L, V, B, dtype, seed, temp=1.0):
    seeds = [synth.seed_for(7, seed * 100 + t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, L, V, 0, device=dev, seeds=seeds, dtype=dtype)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B, drafter_temp=temp)
    tgt = torch.zeros(nt, B + 1, V, dtype=dtype, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=tgt[t, :n],
                               dtype=dtype)
    ov = tsd.tsd_verify_tev(tgt, tr["parent"], tr["token"], tr["n_nodes"], 1.0, seed=3)
    return dr, tr, ov["exit_mass"]


def _oracle(orc, dr, tr, omega, temp, grad=False):
    nums, grads = [], []
    for t in range(dr.shape[0]):
        n = int(tr["n_nodes"][t])
        z = dr[t, 0].float().cpu().numpy().astype(np.float64)
        r = orc.exit_loss(z, temp, tr["token"][t].cpu().numpy(), tr["depth"][t].cpu().numpy(), n,
                          omega[t].double().cpu().numpy(), with_grad=grad)
        if grad:
            nums.append(r[0])
            grads.append(r[1])
        else:
            nums.append(r)
    return np.array(nums), grads


@pytest.mark.parametrize("V,dtype,temp", [(12800, torch.bfloat16, 1.0), (4096 + 256, torch.float32, 0.8),
                                          (3001, torch.bfloat16, 1.0)])
def test_exit_loss_and_gradient(tsd, dev, orc, V, dtype, temp):
    """Several chunks with a tail; fp32; V=3001 is not a multiple of 8 (the
    generic path)."""
    nt, L, B = 3, 6, 40
    dr, tr, w = _case(tsd, dev, nt, L, V, B, dtype, 1, temp)
    out = tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, drafter_temp=temp,
                            with_grad=True)
    assert out["status"].cpu().tolist() == [0] * nt
    nums, grads = _oracle(orc, dr, tr, w, temp, grad=True)
    assert np.allclose(out["loss_tree"].cpu().numpy(), nums, rtol=RTOL, atol=0)
    N = float((tr["n_nodes"] - 1).sum())
    assert float(out["loss"]) == pytest.approx(nums.sum() / N, rel=RTOL)
    g = out["grad"].cpu().numpy().astype(np.float64)
    for t in range(nt):
        want = grads[t] / N
        scale = np.abs(want).max()
        assert np.allclose(g[t], want, rtol=1e-4, atol=1e-6 * scale), t


def test_exit_loss_qwen_vocab(tsd, dev, orc):
    """V=151936, L=16, B=64, 4 trees, bf16: the numerators element by element;
    the gradient on the rows a node scores, at sampled columns and at every
    gathered token."""
    nt, L, V, B = 4, 16, synth.V_QWEN, 64
    dr, tr, w = _case(tsd, dev, nt, L, V, B, torch.bfloat16, 2)
    out = tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, with_grad=True)
    nums, grads = _oracle(orc, dr, tr, w, 1.0, grad=True)
    assert np.allclose(out["loss_tree"].cpu().numpy(), nums, rtol=RTOL, atol=0)
    N = float((tr["n_nodes"] - 1).sum())
    g = out["grad"]
    rng = np.random.default_rng(0)
    cols = rng.integers(0, V, 2000)
    for t in range(nt):
        want = grads[t] / N
        scale = np.abs(want).max()
        got = g[t].cpu().numpy().astype(np.float64)
        n = int(tr["n_nodes"][t])
        toks = tr["token"][t, 1:n].cpu().numpy()
        for m in range(L):
            assert np.allclose(got[m, cols], want[m, cols], rtol=1e-4, atol=1e-6 * scale)
            assert np.allclose(got[m, toks], want[m, toks], rtol=1e-4, atol=1e-6 * scale)


def test_exit_loss_statuses_and_host_logits(tsd, dev, orc):
    """A depth outside [1, L] or a token outside [0, V) marks its tree 4; a NaN
    logit marks it 5; valid trees are unaffected and the scalar counts only
    them.  Logits in page-locked host memory give the same results."""
    nt, L, V, B = 4, 5, 5000, 20
    dr, tr, w = _case(tsd, dev, nt, L, V, B, torch.float32, 3)
    depth = tr["depth"].clone()
    token = tr["token"].clone()
    depth[1, 3] = L + 1
    token[2, 2] = V
    dr2 = dr.clone()
    dr2[3, 0, :, 17] = float("nan")
    out = tsd.tsd_exit_loss(dr2, token, depth, tr["n_nodes"], w, with_grad=True)
    assert out["status"].cpu().tolist() == [0, 4, 4, 5]
    nums, _ = _oracle(orc, dr, tr, w, 1.0)
    assert float(out["loss_tree"][0]) == pytest.approx(nums[0], rel=RTOL)
    assert float(out["loss"]) == pytest.approx(nums[0] / float(tr["n_nodes"][0] - 1), rel=RTOL)
    assert float(out["grad"][1:].abs().max()) == 0.0
    host = tsd.tsd_exit_loss(dr.cpu().pin_memory(), tr["token"], tr["depth"], tr["n_nodes"], w,
                             with_grad=True)
    dev_out = tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, with_grad=True)
    for k in ("loss_tree", "loss", "status"):
        assert torch.equal(host[k], dev_out[k]), k
    # the gathered terms are added with float atomics, whose order may vary
    assert torch.allclose(host["grad"], dev_out["grad"], rtol=1e-6, atol=0)


def test_exit_loss_in_the_bench_launch(tsd, dev, orc):
    """32 trees x 16 rows, V=151936, B=256, bf16 (the bench's launch), weighted
    by TEV's exit masses: every tree's numerator and the scalar loss against
    the oracle; the gradient of two sampled trees at sampled columns and at
    every gathered token."""
    nt, L, V, B = 32, 16, synth.V_QWEN, 256
    dr, tr, w = _case(tsd, dev, nt, L, V, B, torch.bfloat16, 4)
    out = tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, with_grad=True)
    nums, _ = _oracle(orc, dr, tr, w, 1.0)
    assert np.allclose(out["loss_tree"].cpu().numpy(), nums, rtol=RTOL, atol=0)
    N = float((tr["n_nodes"] - 1).sum())
    assert abs(float(out["loss"]) - nums.sum() / N) <= RTOL * abs(nums.sum() / N)
    cols = np.random.default_rng(1).integers(0, V, 2000)
    for t in (3, 30):
        sub = {k: v[t:t + 1] for k, v in tr.items()}
        _, grads = _oracle(orc, dr[t:t + 1], sub, w[t:t + 1], 1.0, grad=True)
        want = grads[0] / N
        scale = np.abs(want).max()
        got = out["grad"][t].cpu().numpy().astype(np.float64)
        toks = tr["token"][t, 1:int(tr["n_nodes"][t])].cpu().numpy()
        for m in range(L):
            assert np.allclose(got[m, cols], want[m, cols], rtol=1e-4, atol=1e-6 * scale)
            assert np.allclose(got[m, toks], want[m, toks], rtol=1e-4, atol=1e-6 * scale)


def test_exit_loss_non_finite_rows_and_terms(tsd, dev, orc):
    """The kernel forms a tree's numerator as sum_m LSE_m W_m - sum_v w z / T
    (Eq. 67).  A row whose logits hold a NaN makes its tree non-finite only if
    some node lies on that row, as in the oracle's node-by-node Eq. 66; a
    drafted token at -inf makes its tree non-finite whatever its weight."""
    L, V, B = 5, 3000, 6
    g = torch.Generator().manual_seed(synth.seed_for(7, 900))
    z = torch.randn(4, 1, L, V, generator=g) * 2
    parent = torch.full((4, B + 1), -1, dtype=torch.int32)
    token = torch.full((4, B + 1), -1, dtype=torch.int32)
    depth = torch.full((4, B + 1), -1, dtype=torch.int32)
    depth[:, 0] = 0
    # every tree: root, two children (depth 1), one grandchild each (depth 2)
    parent[:, 1:5] = torch.tensor([0, 0, 1, 2], dtype=torch.int32)
    token[:, 1:5] = torch.tensor([11, 22, 33, 44], dtype=torch.int32)
    depth[:, 1:5] = torch.tensor([1, 1, 2, 2], dtype=torch.int32)
    n_nodes = torch.full((4,), 5, dtype=torch.int32)
    z[1, 0, 4, 100] = float("nan")  # row 5: no node there
    z[2, 0, 1, 7] = float("nan")  # row 2: the grandchildren's
    z[3, 0, 0, 22] = -float("inf")  # a drafted token at -inf
    w = torch.rand(4, B + 1, generator=g) * (depth >= 1)
    w[3, 2] = 0.0  # weight zero on the -inf token: still non-finite
    out = tsd.tsd_exit_loss(z.to(dev), token.to(dev), depth.to(dev), n_nodes.to(dev), w.to(dev))
    assert out["status"].cpu().tolist() == [0, 0, 5, 5]
    for t in (0, 1):
        want = orc.exit_loss(z[t, 0].double().numpy(), 1.0, token[t].numpy(), depth[t].numpy(), 5,
                             w[t].double().numpy())
        assert float(out["loss_tree"][t]) == pytest.approx(want, rel=RTOL)
    for t in (2, 3):
        with pytest.raises(Exception):
            orc.exit_loss(z[t, 0].double().numpy(), 1.0, token[t].numpy(), depth[t].numpy(), 5,
                          w[t].double().numpy())

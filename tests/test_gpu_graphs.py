"""Every entry point is capturable in a CUDA graph: the library allocates
nothing, keeps no host-side state between calls and never synchronises, so a
captured step replayed on new inputs (copied into the captured buffers) gives
exactly what eager calls give on those inputs."""
import pytest
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


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def _inputs(nt, L, V, B, seed, dev):
    seeds = [synth.seed_for(14, seed * 100 + t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, L, V, 0, device=dev, seeds=seeds)
    tgt = torch.zeros(nt, B + 1, V, dtype=torch.bfloat16, device=dev)
    return dr, tgt, seeds


def test_step_replays_from_a_graph(tsd, dev):
    nt, L, V, B, T = 4, 16, 12805, 64, 0.6
    dr, tgt, seeds = _inputs(nt, L, V, B, 1, dev)
    wb = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, nt, 1, L, V, 8, B, torch.bfloat16),
                     dtype=torch.uint8, device=dev)
    wv = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, nt, 1, 1, V, 1, B, torch.bfloat16),
                     dtype=torch.uint8, device=dev)

    def fill_targets(d, x, tr):
        x.zero_()
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            synth.target_from_rows(d[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=x[t, :n])

    def step():
        tr = tsd.tsd_build_tree(dr, topk=8, B=B, workspace=wb)
        mk = tsd.tsd_tree_mask(tr["parent"], tr["n_nodes"], prefix_len=7)
        out = tsd.tsd_verify_tev(tgt, tr["parent"], tr["token"], tr["n_nodes"], T, seed=9,
                                 workspace=wv)
        return tr, mk, out

    fill_targets(dr, tgt, tsd.tsd_build_tree(dr, topk=8, B=B))
    g, (tr_g, mk_g, out_g) = _capture(step)
    # new inputs into the captured buffers, then replay
    dr2, _, _ = _inputs(nt, L, V, B, 2, dev)
    dr.copy_(dr2)
    fill_targets(dr, tgt, tsd.tsd_build_tree(dr, topk=8, B=B))
    g.replay()
    torch.cuda.synchronize()
    tr_e, mk_e, out_e = step()
    torch.cuda.synchronize()
    for key in ("parent", "token", "depth", "score", "n_nodes", "status"):
        assert torch.equal(tr_g[key], tr_e[key]), key
    assert torch.equal(mk_g["anc_bits"], mk_e["anc_bits"])
    assert torch.equal(mk_g["position_ids"], mk_e["position_ids"])
    for key in ("exit_node", "bonus_token", "accept_len", "exit_mass", "status"):
        assert torch.equal(out_g[key], out_e[key]), key


def test_secondary_operations_replay_from_a_graph(tsd, dev):
    """The log-sum-exp tree (its kernels set shared-memory attributes at
    launch) and the exit loss with its gradient (a memset node in the graph)."""
    mix, _, _ = synth.mixture_drafter(2, 4, 8, 6000, synth.seed_for(14, 7), device=dev)
    wl = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_LSE, 2, 4, 8, 6000, 8, 64,
                                            torch.bfloat16), dtype=torch.uint8, device=dev)
    g, lg = _capture(lambda: tsd.tsd_build_lse_tree(mix, topk=8, B=64, workspace=wl))
    mix2, _, _ = synth.mixture_drafter(2, 4, 8, 6000, synth.seed_for(14, 8), device=dev)
    mix.copy_(mix2)
    g.replay()
    le = tsd.tsd_build_lse_tree(mix, topk=8, B=64, workspace=wl)
    torch.cuda.synchronize()
    for key in ("parent", "token", "score", "n_nodes", "n_cand"):
        assert torch.equal(lg[key], le[key]), key
    dr, _, _ = _inputs(3, 8, 9000, 40, 3, dev)
    tr = tsd.tsd_build_tree(dr, topk=8, B=40)
    w = torch.rand(3, 41, generator=torch.Generator(device=dev).manual_seed(4), device=dev)
    w = w * (tr["depth"] >= 0)
    we = torch.empty(tsd.tsd_workspace_size(tsd.TSD_OP_EXIT_LOSS, 3, 1, 8, 9000, 1, 40,
                                            torch.bfloat16), dtype=torch.uint8, device=dev)
    g2, eg = _capture(lambda: tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w,
                                                with_grad=True, workspace=we))
    w.mul_(0.5)
    g2.replay()
    torch.cuda.synchronize()
    ref = tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, with_grad=True,
                            workspace=we)
    torch.cuda.synchronize()
    assert torch.allclose(eg["loss_tree"], ref["loss_tree"], rtol=1e-12, atol=0)
    assert torch.allclose(eg["grad"], ref["grad"], rtol=1e-5, atol=1e-9)


def test_calls_on_concurrent_streams(tsd, dev):
    """Two independent batches issued on two streams from two host threads at
    once, each with its own workspace, give what one stream gives."""
    import threading
    nt, L, V, B, T = 3, 16, 9000, 48, 1.0
    jobs = []
    for j in range(2):
        dr, tgt, seeds = _inputs(nt, L, V, B, 20 + j, dev)
        tr = tsd.tsd_build_tree(dr, topk=8, B=B)
        for t in range(nt):
            n = int(tr["n_nodes"][t])
            synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=tgt[t, :n])
        jobs.append((dr, tgt))
    torch.cuda.synchronize()

    def run(dr, tgt):
        tr = tsd.tsd_build_tree(dr, topk=8, B=B)
        out = tsd.tsd_verify_tev(tgt, tr["parent"], tr["token"], tr["n_nodes"], T, seed=4)
        return tr, out

    want = [run(*j) for j in jobs]
    torch.cuda.synchronize()
    got = [None, None]
    streams = [torch.cuda.Stream(dev) for _ in range(2)]

    def worker(i):
        with torch.cuda.stream(streams[i]):
            for _ in range(5):
                got[i] = run(*jobs[i])

    ths = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    torch.cuda.synchronize()
    for i in range(2):
        for key in ("parent", "token", "n_nodes"):
            assert torch.equal(got[i][0][key], want[i][0][key]), (i, key)
        for key in ("exit_node", "bonus_token", "accept_len", "exit_mass"):
            assert torch.equal(got[i][1][key], want[i][1][key]), (i, key)

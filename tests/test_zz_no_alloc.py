"""tsd_verify_tev_noalloc: Tree Exit Verification for callers that cannot
allocate device memory (for example a plug-in that an inference engine hands
only its input and output pointers, or a decode loop that must not call
cudaMalloc because cudaMalloc can synchronise the device).  Its scratch is a
static array inside the library instead of a caller workspace.

The test calls the entry point through the C ABI (ctypes, with PyTorch only
holding the inputs and outputs) three times in a row, and each call meets the
previous call's leftovers in the shared scratch: a large launch (12 trees,
B = 200, bf16), then a smaller one (3 trees, B = 16, fp32 logits, so every
array of the scratch layout sits at another offset and the large call's data
lies past the small call's extent), then the large launch again at another
temperature.  Each result is checked against tsd_verify_tev with a freshly
allocated workspace, within the parity tests' tolerance.  The file is named so
that pytest collects it last.
"""
import ctypes

import pytest
import torch

import synth
from gpu_helpers import close

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, x, par, tok, nn, T, seed):
    nt, Bp1, V = x.shape
    dev = x.device
    o = {k: torch.full((nt,), -7, dtype=torch.int32, device=dev)
         for k in ("exit_node", "bonus_token", "accept_len", "status")}
    o["exit_mass"] = torch.full((nt, Bp1), -7.0, device=dev)
    o["prefix_prob"] = torch.full((nt, Bp1), -7.0, device=dev)
    o["coverage"] = torch.full((nt,), -7.0, device=dev)
    P = ctypes.c_void_p
    st = lib.tsd_verify_tev_noalloc(
        P(x.data_ptr()), 0 if x.dtype == torch.bfloat16 else 1, P(par.data_ptr()),
        P(tok.data_ptr()), P(nn.data_ptr()), nt, Bp1 - 1, V, T, seed,
        P(o["exit_node"].data_ptr()), P(o["bonus_token"].data_ptr()),
        P(o["accept_len"].data_ptr()), P(o["exit_mass"].data_ptr()),
        P(o["prefix_prob"].data_ptr()), P(o["coverage"].data_ptr()), P(o["status"].data_ptr()),
        P(torch.cuda.current_stream(dev).cuda_stream))
    torch.cuda.synchronize()
    return st, o


def _case(tsd, dev, nt, B, V, dtype, cfg):
    seeds = [synth.seed_for(cfg, 50 + t) for t in range(nt)]
    dr = synth.zipf_drafter(nt, 16, V, 0, device=dev, seeds=seeds)
    tr = tsd.tsd_build_tree(dr, topk=8, B=B)
    x = torch.zeros(nt, B + 1, V, dtype=dtype, device=dev)
    for t in range(nt):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, seeds[t] + 1, out=x[t, :n])
    return x, tr


def test_noalloc_matches_workspace_entry_point():
    import tree_speculative_decoding_position_gb300 as tsd
    from tree_speculative_decoding_position_gb300 import build
    build.build()
    lib = tsd.load()
    dev = torch.device("cuda:0")
    big = _case(tsd, dev, 12, 200, 12805, torch.bfloat16, 1)
    small = _case(tsd, dev, 3, 16, 12805, torch.float32, 7)
    for call, ((x, tr), T, seed) in enumerate([(big, 1.0, 77), (small, 0.6, 78), (big, 0.0, 79)]):
        st, got = _call_noalloc(lib, x, tr["parent"], tr["token"], tr["n_nodes"], T, seed)
        assert st == tsd.TSD_OK, (call, st)
        ref = tsd.tsd_verify_tev(x, tr["parent"], tr["token"], tr["n_nodes"], T, seed=seed)
        torch.cuda.synchronize()
        for k in ("exit_node", "bonus_token", "accept_len", "status"):
            assert torch.equal(got[k], ref[k]), (call, k)
        for k in ("exit_mass", "prefix_prob", "coverage"):
            ok, err = close(got[k].cpu().numpy(), ref[k].cpu().numpy())
            assert ok, (call, k, err)
        assert int((got["status"] != 0).sum()) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import tree_speculative_decoding_position_gb300 as tsd
    lib = tsd.load()
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: the size check comes first
    # 512 trees of B = 512 at V = 151936 need far more than 16 MiB of scratch
    st = lib.tsd_verify_tev_noalloc(fake, 0, fake, fake, fake, 512, 512, 151936, 1.0, 0, fake,
                                    fake, fake, None, None, None, fake, None)
    assert st == tsd.TSD_ERR_WORKSPACE

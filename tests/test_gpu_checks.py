"""The bounds-checked build (-DTSD_CHECKS, libtsd_checks.so): every entry
point on representative and edge-case inputs must pass every check, and give
the same outputs as the product library.  Each library runs in its own
process (the binding loads one library per process).

The checked build also narrows the log-sum-exp selection's group hash to 6
bits, so that its exact check fails and the depth-by-depth merge runs; the
outputs of that merge are compared here with the default build's grouped
merge."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import synth
import tree_speculative_decoding_position_gb300 as tsd
tsd.load()
dev = torch.device("cuda:0")
out = {"lib": tsd.LIB_PATH.rsplit("/", 1)[-1]}

def keep(name, d, keys):
    for k in keys:
        if k in d:
            out[name + "." + k] = d[k].detach().cpu().double().numpy().round(6).tolist()

for V, dtype in ((synth.V_QWEN, torch.bfloat16), (12805, torch.bfloat16), (4097, torch.float32)):
    dr = synth.zipf_drafter(2, 8, V, 0, device=dev, seeds=[synth.seed_for(11, V + t) for t in range(2)],
                            dtype=dtype)
    tr = tsd.tsd_build_tree(dr, topk=8, B=64)
    keep("build%d" % V, tr, ("parent", "token", "depth", "n_nodes", "status"))
    m = tsd.tsd_tree_mask(tr["parent"], tr["n_nodes"], prefix_len=10, additive=True)
    keep("mask%d" % V, m, ("anc_bits", "position_ids", "status"))
    tgt = torch.zeros(2, 65, V, dtype=dtype, device=dev)
    for t in range(2):
        n = int(tr["n_nodes"][t])
        synth.target_from_rows(dr[t, 0], tr["depth"][t, :n], 1.5, synth.seed_for(11, t), out=tgt[t, :n])
    q = torch.full((2, 65), 0.5, device=dev)
    for T in (1.0, 0.0):
        a = (tgt, tr["parent"], tr["token"], tr["n_nodes"], T)
        keep("tev%d_%g" % (V, T), tsd.tsd_verify_tev(*a, seed=3),
             ("exit_node", "bonus_token", "accept_len", "exit_mass", "status"))
        keep("ddtree%d_%g" % (V, T), tsd.tsd_verify_ddtree(*a, seed=3),
             ("exit_node", "bonus_token", "accept_len", "status"))
        keep("seqres%d_%g" % (V, T), tsd.tsd_verify_seqres(*a, seed=3),
             ("exit_node", "bonus_token", "accept_len", "status"))
        keep("proposal%d_%g" % (V, T), tsd.tsd_verify_proposal(tgt, tr["parent"], tr["token"],
             tr["n_nodes"], q, T, seed=3), ("exit_node", "bonus_token", "accept_len", "status"))
        keep("noalloc%d_%g" % (V, T), tsd.tsd_verify_tev_noalloc(*a, seed=3),
             ("exit_node", "bonus_token", "accept_len", "status"))
    w = torch.rand(2, 65, generator=torch.Generator(device=dev).manual_seed(5), device=dev) * (tr["depth"] >= 0)
    keep("exit%d" % V, tsd.tsd_exit_loss(dr, tr["token"], tr["depth"], tr["n_nodes"], w, with_grad=True),
         ("loss_tree", "status"))

mix, _, _ = synth.mixture_drafter(3, 4, 6, 3000, synth.seed_for(11, 1), device=dev)
keep("mixture", tsd.tsd_build_tree(mix, topk=8, B=100), ("parent", "token", "n_nodes", "status"))
keep("lse", tsd.tsd_build_lse_tree(mix, topk=8, B=100), ("parent", "token", "n_nodes", "status", "n_cand"))
# the mixture workload's shape (two groups of eight depths in the selection's
# merge); the checked build always takes the depth-by-depth merge
mix, _, _ = synth.mixture_drafter(2, 8, 16, synth.V_QWEN, synth.seed_for(11, 2), device=dev)
keep("lse_k8", tsd.tsd_build_lse_tree(mix, topk=8, B=128), ("parent", "token", "depth", "n_nodes", "status",
                                                           "n_cand"))
dr = synth.zipf_drafter(6, 8, 3000, 0, device=dev, seeds=[synth.seed_for(11, 50 + t) for t in range(6)])
keep("forest", tsd.tsd_build_forest(dr, topk=8, B=64, M_max=200, l0=1.0, c1=1.0 / 256),
     ("parent", "n_nodes", "status", "total"))

# edge trees in one B = 4095 launch: a 4095-child star, a malformed tree, NaN logits
V, B = 5000, 4095
rng = np.random.default_rng(7)
par = np.full((3, B + 1), -1, dtype=np.int32)
tok = np.full((3, B + 1), -1, dtype=np.int32)
par[:, 1:] = 0
tok[:, 1:] = rng.permutation(V)[:B]
par[1, 5] = 9  # parent after child
nn = torch.full((3,), B + 1, dtype=torch.int32, device=dev)
z = torch.randn(3, B + 1, V, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
z[2, 0, 17] = float("nan")
z = z.to(dev)
pd, xd = torch.tensor(par, device=dev), torch.tensor(tok, device=dev)
qd = torch.full((3, B + 1), 0.25, device=dev)
for T in (1.0, 0.0):
    keep("edge_tev_%g" % T, tsd.tsd_verify_tev(z, pd, xd, nn, T, seed=1), ("exit_node", "bonus_token", "status"))
    keep("edge_seqres_%g" % T, tsd.tsd_verify_seqres(z, pd, xd, nn, T, seed=1), ("exit_node", "status"))
    keep("edge_prop_%g" % T, tsd.tsd_verify_proposal(z, pd, xd, nn, qd, T, seed=1), ("exit_node", "status"))
    keep("edge_dd_%g" % T, tsd.tsd_verify_ddtree(z, pd, xd, nn, T, seed=1), ("exit_node", "status"))
keep("edge_mask", tsd.tsd_tree_mask(pd, nn, prefix_len=3), ("position_ids", "status"))
out["check_failures"] = tsd.tsd_debug_check_failures()
print(json.dumps(out))
"""


def _run(library):
    env = dict(os.environ)
    env.pop("TSD_LIBRARY", None)
    if library:
        env["TSD_LIBRARY"] = library
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_passes_every_check_and_matches():
    from tree_speculative_decoding_position_gb300 import build
    build.build()
    build.build(checks=True)
    checked = _run("checks")
    plain = _run(None)
    assert checked["lib"] == "libtsd_checks.so" and plain["lib"] == "libtsd.so"
    assert checked.pop("check_failures") == 0
    assert plain.pop("check_failures") == 0  # the default build has no checks
    checked.pop("lib")
    plain.pop("lib")
    assert checked.keys() == plain.keys()
    import numpy as np
    for k in plain:  # integers exactly; floats up to contraction order
        a, b = np.asarray(checked[k], dtype=np.float64), np.asarray(plain[k], dtype=np.float64)
        assert a.shape == b.shape and np.allclose(a, b, rtol=1e-5, atol=1e-7, equal_nan=True), k
    # the edge trees: star valid, malformed tree 4, NaN tree 5
    assert checked["edge_tev_1.status"] == [0, 4, 5]
    assert checked["edge_seqres_0.status"] == [0, 4, 5]

"""Float64 CPU oracle for bounded-tree speculative decoding.

TEST INFRASTRUCTURE ONLY.  A plain, slow, obviously-correct restatement of
what the CUDA library computes (``tsd_oracle.c``), loaded through ctypes.
Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import it.  It shares no code with the CUDA library, and
the product path never calls it.

Every function takes and returns numpy arrays; floating inputs are converted
to float64 exactly (bf16 and fp32 values are representable in float64).

Parity status: each function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsd_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

OK, ERR_ARG, ERR_BAD_TREE, ERR_NONFINITE = 0, 1, 4, 5


def build(force: bool = False) -> str:
    """Compile ``tsd_oracle.c`` into ``liboracle.so`` next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, f64, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_uint64
        lib.orc_philox4x64_10.argtypes = [P, P, P]
        lib.orc_philox4x64_10.restype = None
        lib.orc_uniform.argtypes = [u64, u64, u64, u64]
        lib.orc_uniform.restype = f64
        lib.orc_drafter_stats.argtypes = [P, i64, i64, f64, i32, P, P, P, P]
        lib.orc_build_tree.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        lib.orc_tree_mask.argtypes = [P, i32, i32, i32, P, P, P, i64]
        lib.orc_row_probs.argtypes = [P, i64, f64, P]
        lib.orc_tev.argtypes = [P, P, P, i32, i64, f64, u64, u64, P, P, P, P, P, P, P, P, P, P]
        lib.orc_predraw.argtypes = [P, P, P, i32, i64, f64, u64, u64, P, P, P, P]
        lib.orc_tev_sample_many.argtypes = [P, P, P, i32, i64, f64, u64, u64, i64, P, P]
        lib.orc_predraw_sample_many.argtypes = [P, P, P, i32, i64, f64, u64, u64, i64, P, P]
        lib.orc_exit_loss.argtypes = [P, i32, i64, f64, P, P, i32, P, P, P]
        lib.orc_forest_select.argtypes = [P, P, P, i32, i32, i32, f64, f64, P, P, P]
        lib.orc_uniform_sub.argtypes = [u64, u64, u64, u64, u64]
        lib.orc_lse_tree.argtypes = [P, i32, i32, i64, f64, i32, i32, P, P, P, P, P, P, P]
        lib.orc_uniform_sub.restype = f64
        lib.orc_seqres.argtypes = [P, P, P, i32, i64, f64, u64, u64, P, P, P]
        lib.orc_proposal.argtypes = [P, P, P, i32, i64, f64, P, u64, u64, P, P, P]
        lib.orc_seqres_sample_many.argtypes = [P, P, P, i32, i64, f64, u64, u64, i64, P, P]
        lib.orc_proposal_sample_many.argtypes = [P, P, P, i32, i64, f64, P, u64, u64, i64, P, P]
        for f in ("orc_forest_select", "orc_seqres", "orc_proposal", "orc_seqres_sample_many",
                  "orc_proposal_sample_many", "orc_exit_loss", "orc_drafter_stats", "orc_build_tree", "orc_tree_mask", "orc_row_probs",
                  "orc_tev", "orc_predraw", "orc_tev_sample_many", "orc_predraw_sample_many"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s failed with status %d" % (what, code))
        self.code = code


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


def philox4x64_10(counter, key) -> np.ndarray:
    """Philox4x64-10 block: 4 uint64 outputs for a 4-word counter, 2-word key."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.zeros(4, dtype=np.uint64)
    _load().orc_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, tree: int, node: int, stream: int) -> float:
    """The uniform the method uses for (seed; tree, node, stream)."""
    return _load().orc_uniform(seed, tree, node, stream)


def drafter_stats(z, temp: float, k: int):
    """Per row: LSE of z/temp, top-k ids by (logit desc, id asc), their log q."""
    d = drafter_lists(z, temp, k)
    return d["lse"], d["top_id"], d["top_logq"]


def drafter_lists(z, temp: float, k: int) -> dict:
    """The builder's input, per row: lse (log-normaliser of z/temp), top_id
    (top-k by logit desc, id asc), top_logq (their log q) and top_zt (their
    z/temp).  z: [..., V]; leading dims are kept (e.g. [K, L])."""
    z = _f64(z)
    V = z.shape[-1]
    rows = z.size // V
    lse = np.zeros(rows)
    tid = np.zeros((rows, k), dtype=np.int32)
    tlq = np.zeros((rows, k))
    tzt = np.zeros((rows, k))
    _check(_load().orc_drafter_stats(_ptr(z), rows, V, temp, k, _ptr(lse), _ptr(tid), _ptr(tlq),
                                     _ptr(tzt)), "drafter_stats")
    shp = z.shape[:-1]
    return dict(lse=lse.reshape(shp), top_id=tid.reshape(shp + (k,)),
                top_logq=tlq.reshape(shp + (k,)), top_zt=tzt.reshape(shp + (k,)))


def build_tree(lists: dict, B: int, push_rule: int = 0) -> dict:
    """Best-first builder on one tree.  lists: top_id, top_zt [K, L, k] (or
    [L, k]) and lse [K, L] (or [L]), as drafter_lists returns them."""
    tid = _i32(lists["top_id"])
    tzt = _f64(lists["top_zt"])
    lse = _f64(lists["lse"])
    if tid.ndim == 2:
        tid, tzt, lse = tid[None], tzt[None], lse[None]
    K, L, k = tid.shape
    out = {n: np.zeros(B + 1, dtype=np.int32) for n in ("parent", "token", "depth", "rank", "mode")}
    out["score"] = np.zeros(B + 1)
    nn = np.zeros(1, dtype=np.int32)
    _check(_load().orc_build_tree(_ptr(tid), _ptr(tzt), _ptr(np.ascontiguousarray(lse)), K, L, k,
                                  B, push_rule, _ptr(out["parent"]), _ptr(out["token"]),
                                  _ptr(out["depth"]), _ptr(out["score"]), _ptr(out["rank"]),
                                  _ptr(out["mode"]), _ptr(nn)), "build_tree")
    out["n_nodes"] = int(nn[0])
    return out


def lists_from_logq(top_id, top_logq) -> dict:
    """Builder lists from log-probabilities alone (z/T = log q, LSE = 0): for
    tests that state a universe directly by its log q."""
    tlq = _f64(top_logq)
    return dict(top_id=_i32(top_id), top_zt=tlq, lse=np.zeros(tlq.shape[:-1]))


def tree_mask(parent, n_nodes: int, B: int, prefix_len: int, with_additive: bool = False):
    parent = _i32(parent)
    W = (B + 1 + 31) // 32
    bits = np.zeros((B + 1, W), dtype=np.uint32)
    pos = np.zeros(B + 1, dtype=np.int32)
    ld = prefix_len + B + 1
    add = np.zeros((B + 1, ld)) if with_additive else None
    _check(_load().orc_tree_mask(_ptr(parent), n_nodes, B, prefix_len, _ptr(bits), _ptr(pos),
                                 _ptr(add) if add is not None else None, ld), "tree_mask")
    return bits, pos, add


def row_probs(z, T: float) -> np.ndarray:
    z = _f64(z)
    p = np.zeros_like(z)
    _check(_load().orc_row_probs(_ptr(z), z.size, T, _ptr(p)), "row_probs")
    return p


def tev(z, parent, token, n_nodes: int, T: float, seed: int, tree: int = 0) -> dict:
    """Tree Exit Verification on one tree; z: [>= n_nodes, V] target logits."""
    z = _f64(z)
    V = z.shape[-1]
    z = np.ascontiguousarray(z.reshape(-1, V)[:n_nodes])
    parent, token = _i32(parent), _i32(token)
    n = n_nodes
    P, rho, w, pedge = (np.zeros(n) for _ in range(4))
    cov = np.zeros(1)
    ex, bo, al = (np.zeros(1, dtype=np.int32) for _ in range(3))
    ue, ub = np.zeros(1), np.zeros(1)
    _check(_load().orc_tev(_ptr(z), _ptr(parent), _ptr(token), n, V, T, seed, tree, _ptr(P),
                           _ptr(rho), _ptr(w), _ptr(pedge), _ptr(cov), _ptr(ex), _ptr(bo),
                           _ptr(al), _ptr(ue), _ptr(ub)), "tev")
    return dict(P=P, rho=rho, w=w, pedge=pedge, coverage=float(cov[0]), exit_node=int(ex[0]),
                bonus=int(bo[0]), accept_len=int(al[0]), u_exit=float(ue[0]), u_bonus=float(ub[0]))


def predraw(z, parent, token, n_nodes: int, T: float, seed: int, tree: int = 0) -> dict:
    """Predraw-and-follow on one tree; z: [>= n_nodes, V] target logits."""
    z = _f64(z)
    V = z.shape[-1]
    z = np.ascontiguousarray(z.reshape(-1, V)[:n_nodes])
    parent, token = _i32(parent), _i32(token)
    draws = np.zeros(n_nodes, dtype=np.int32)
    ex, bo, al = (np.zeros(1, dtype=np.int32) for _ in range(3))
    _check(_load().orc_predraw(_ptr(z), _ptr(parent), _ptr(token), n_nodes, V, T, seed, tree,
                               _ptr(draws), _ptr(ex), _ptr(bo), _ptr(al)), "predraw")
    return dict(draws=draws, exit_node=int(ex[0]), bonus=int(bo[0]), accept_len=int(al[0]))


def sample_many(kind: str, z, parent, token, n_nodes: int, T: float, seed: int, n_draws: int,
                first_tree: int = 0, q_child=None):
    """(exit node, bonus token) of n_draws independent draws of the sampler
    `kind` ("tev", "predraw", "seqres" or "proposal", the last with
    q_child) on one tree; draw i uses tree index first_tree + i."""
    z = _f64(z)
    V = z.shape[-1]
    z = np.ascontiguousarray(z.reshape(-1, V)[:n_nodes])
    parent, token = _i32(parent), _i32(token)
    ex = np.zeros(n_draws, dtype=np.int32)
    bo = np.zeros(n_draws, dtype=np.int32)
    lib = _load()
    if kind == "proposal":
        q = _f64(q_child)
        _check(lib.orc_proposal_sample_many(_ptr(z), _ptr(parent), _ptr(token), n_nodes, V, T,
                                            _ptr(q), seed, first_tree, n_draws, _ptr(ex), _ptr(bo)),
               "proposal_sample_many")
        return ex, bo
    fn = {"tev": lib.orc_tev_sample_many, "predraw": lib.orc_predraw_sample_many,
          "seqres": lib.orc_seqres_sample_many}[kind]
    _check(fn(_ptr(z), _ptr(parent), _ptr(token), n_nodes, V, T, seed, first_tree, n_draws,
              _ptr(ex), _ptr(bo)), kind + "_sample_many")
    return ex, bo


def uniform_sub(seed: int, tree: int, node: int, stream: int, sub: int) -> float:
    return float(_load().orc_uniform_sub(seed, tree, node, stream, sub))


def seqres(z, parent, token, n_nodes: int, T: float, seed: int, tree: int = 0) -> dict:
    """Exact sequential residual verification ([EXIT] App. A.4.2) on one tree."""
    z = _f64(z)
    V = z.shape[-1]
    z = np.ascontiguousarray(z.reshape(-1, V)[:n_nodes])
    parent, token = _i32(parent), _i32(token)
    ex, bo, al = (np.zeros(1, dtype=np.int32) for _ in range(3))
    _check(_load().orc_seqres(_ptr(z), _ptr(parent), _ptr(token), n_nodes, V, T, seed, tree,
                              _ptr(ex), _ptr(bo), _ptr(al)), "seqres")
    return dict(exit_node=int(ex[0]), bonus=int(bo[0]), accept_len=int(al[0]))


def proposal(z, parent, token, n_nodes: int, T: float, q_child, seed: int, tree: int = 0) -> dict:
    """Proposal-aware verification ([CAST] App. B.1 Thm. 3) on one tree;
    q_child[u] = the proposal's probability of node u's token (u >= 1)."""
    z = _f64(z)
    V = z.shape[-1]
    z = np.ascontiguousarray(z.reshape(-1, V)[:n_nodes])
    parent, token = _i32(parent), _i32(token)
    q = _f64(q_child)
    ex, bo, al = (np.zeros(1, dtype=np.int32) for _ in range(3))
    _check(_load().orc_proposal(_ptr(z), _ptr(parent), _ptr(token), n_nodes, V, T, _ptr(q), seed,
                                tree, _ptr(ex), _ptr(bo), _ptr(al)), "proposal")
    return dict(exit_node=int(ex[0]), bonus=int(bo[0]), accept_len=int(al[0]))


def exit_loss(z, T: float, token, depth, n_nodes: int, omega, with_grad: bool = False):
    """Exit-guided loss numerator of one example ([EXIT] Eq. 14 / 66) and,
    optionally, its gradient with respect to the drafter logits z [L, V]."""
    z = _f64(z)
    L, V = z.shape
    token, depth = _i32(token), _i32(depth)
    omega = _f64(omega)
    num = np.zeros(1)
    grad = np.zeros((L, V)) if with_grad else None
    _check(_load().orc_exit_loss(_ptr(z), L, V, T, _ptr(token), _ptr(depth), n_nodes, _ptr(omega),
                                 _ptr(num), _ptr(grad) if grad is not None else None), "exit_loss")
    return (float(num[0]), grad) if with_grad else float(num[0])


def forest_select(scores, depth, n_nodes, M_max: int, l0: float, c1: float) -> dict:
    """Shared-budget selection over R requests ([CAST] App. B.4 Prop. 2-3):
    scores, depth [R, stride] in each request's pop order (node 0 the root);
    returns the per-request widths, the total M* and G(M*)."""
    scores = _f64(scores)
    depth = _i32(depth)
    n_nodes = _i32(n_nodes)
    R, stride = scores.shape
    width = np.zeros(R, dtype=np.int32)
    ms = np.zeros(1, dtype=np.int32)
    g = np.zeros(1)
    _check(_load().orc_forest_select(_ptr(scores), _ptr(depth), _ptr(n_nodes), R, stride, M_max,
                                     l0, c1, _ptr(width), _ptr(ms), _ptr(g)), "forest_select")
    return dict(width=width, M=int(ms[0]), G=float(g[0]))


def lse_tree(z, temp: float, k: int, B: int, log_prior=None) -> dict:
    """Mixture tree under the log-sum-exp score ([MFD] App. B Eq. 6): the B
    best distinct prefixes of the modes' per-depth top-B lists, ranked by
    log sum_m pi_m Q_m(v).  z: [K, L, V] drafter logits; log_prior: [K] or
    None (uniform).  Returns parent, token, depth, score ([B+1]; score = the
    ranking key), n_nodes and n_cand (distinct candidates)."""
    z = _f64(z)
    K, L, V = z.shape
    lp = None if log_prior is None else _f64(log_prior)
    out = {n: np.zeros(B + 1, dtype=np.int32) for n in ("parent", "token", "depth")}
    out["score"] = np.zeros(B + 1)
    nn = np.zeros(1, dtype=np.int32)
    nc = np.zeros(1, dtype=np.int32)
    _check(_load().orc_lse_tree(_ptr(z), K, L, V, temp, k, B, _ptr(lp) if lp is not None else None,
                                _ptr(out["parent"]), _ptr(out["token"]), _ptr(out["depth"]),
                                _ptr(out["score"]), _ptr(nn), _ptr(nc)), "lse_tree")
    out["n_nodes"] = int(nn[0])
    out["n_cand"] = int(nc[0])
    return out

"""GB300 (sm_103a) library for the data-parallel hot path of bounded-tree
speculative decoding: the best-first draft-tree builder (with the mixture
variant), the ancestor mask and position ids, and exact Tree Exit
Verification, plus a predraw-and-follow verifier kept as an equivalence check.

This module is a thin binding over the C ABI in ``include/tsd.h`` (loaded
from ``libtsd.so`` with ctypes): it checks tensor dtypes, shapes, devices and
contiguity, allocates outputs and the workspace with PyTorch, and passes raw
pointers and the current CUDA stream.  Every step of the path runs in the
library's CUDA kernels; there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["TsdError", "load", "tsd_status_string", "tsd_workspace_size", "tsd_build_tree",
           "tsd_tree_mask", "tsd_verify_tev", "tsd_verify_tev_timed", "tsd_verify_ddtree",
           "tsd_verify_tev_noalloc", "tsd_exit_loss", "tsd_verify_seqres",
           "tsd_verify_proposal", "tsd_build_forest", "tsd_debug_check_failures", "LIB_PATH"]

# TSD_LIBRARY=checks selects the bounds-checked build (libtsd_checks.so, made by
# build.build(checks=True)); the default is the product library.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libtsd_checks.so" if os.environ.get("TSD_LIBRARY") == "checks"
                        else "libtsd.so")

TSD_OK, TSD_ERR_INVALID_ARG, TSD_ERR_CUDA, TSD_ERR_WORKSPACE = 0, 1, 2, 3
TSD_ERR_BAD_TREE, TSD_ERR_NONFINITE, TSD_ERR_TIMEOUT = 4, 5, 6
TSD_BF16, TSD_F32 = 0, 1
TSD_OP_BUILD_TREE, TSD_OP_VERIFY_TEV, TSD_OP_VERIFY_DDTREE, TSD_OP_EXIT_LOSS = 0, 1, 2, 3
TSD_OP_BUILD_FOREST, TSD_OP_BUILD_LSE = 4, 5

_lib = None


class TsdError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, tsd_status_string(code), code))
        self.code = code


def load():
    """Load the library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("%s is missing: build it with "
                           "`python -m tree_speculative_decoding_position_gb300.build%s`"
                           % (os.path.basename(LIB_PATH),
                              " --checks" if LIB_PATH.endswith("_checks.so") else ""))
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_uint64, ctypes.c_size_t)
    lib.tsd_status_string.argtypes = [i32]
    lib.tsd_status_string.restype = ctypes.c_char_p
    lib.tsd_debug_check_failures.argtypes = []
    lib.tsd_debug_check_failures.restype = ctypes.c_uint
    lib.tsd_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32]
    lib.tsd_workspace_size.restype = sz
    lib.tsd_build_tree.argtypes = [P, i32, i32, i32, i32, i64, i32, i32, f32,
                                   P, P, P, P, P, P, P, P, P, sz, P]
    lib.tsd_tree_mask.argtypes = [P, P, i32, i32, i32, P, P, P, i64, P, P]
    lib.tsd_verify_tev.argtypes = [P, i32, P, P, P, i32, i32, i64, f32, u64,
                                   P, P, P, P, P, P, P, P, sz, P]
    lib.tsd_verify_tev_timed.argtypes = lib.tsd_verify_tev.argtypes + [P]
    lib.tsd_verify_tev_noalloc.argtypes = [P, i32, P, P, P, i32, i32, i64, f32, u64,
                                           P, P, P, P, P, P, P, P]
    lib.tsd_verify_ddtree.argtypes = [P, i32, P, P, P, i32, i32, i64, f32, u64,
                                      P, P, P, P, P, P, sz, P]
    lib.tsd_exit_loss.argtypes = [P, i32, i32, i32, i64, f32, P, P, P, i32, P, P, P, P, P, P,
                                  sz, P]
    lib.tsd_verify_seqres.argtypes = [P, i32, P, P, P, i32, i32, i64, f32, u64, P, P, P, P, P, sz, P]
    lib.tsd_verify_proposal.argtypes = [P, i32, P, P, P, P, i32, i32, i64, f32, u64, P, P, P, P, P,
                                        sz, P]
    f64 = ctypes.c_double
    lib.tsd_build_forest.argtypes = [P, i32, i32, i32, i64, i32, i32, f32, i32, f64, f64,
                                     P, P, P, P, P, P, P, P, sz, P]
    lib.tsd_build_lse_tree.argtypes = [P, i32, i32, i32, i32, i64, i32, i32, f32, P,
                                       P, P, P, P, P, P, P, P, sz, P]
    for f in ("tsd_build_tree", "tsd_tree_mask", "tsd_verify_tev", "tsd_verify_tev_timed",
              "tsd_verify_ddtree", "tsd_verify_tev_noalloc", "tsd_exit_loss", "tsd_verify_seqres",
              "tsd_verify_proposal", "tsd_build_forest", "tsd_build_lse_tree"):
        getattr(lib, f).restype = i32
    _lib = lib
    return lib


def tsd_debug_check_failures() -> int:
    """Bits of the bounds-check site classes that failed since the last call
    (a checked build only; 0 in the default build).  Synchronises the device."""
    return int(load().tsd_debug_check_failures())


def tsd_status_string(code: int) -> str:
    return load().tsd_status_string(int(code)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return TSD_BF16
    if t.dtype == torch.float32:
        return TSD_F32
    raise TypeError("logits must be bfloat16 or float32, got %s" % t.dtype)


def tsd_workspace_size(op: int, n_trees: int, n_modes: int, L: int, V: int, topk: int, B: int,
                       dtype: torch.dtype) -> int:
    code = TSD_BF16 if dtype == torch.bfloat16 else TSD_F32
    return int(load().tsd_workspace_size(op, n_trees, n_modes, L, V, topk, B, code))


def _cuda(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _logits(t: torch.Tensor, name: str) -> torch.Tensor:
    """Logits may sit in device memory or in page-locked host memory, which
    the kernels read directly over the host link (the library checks that the
    host memory is mapped for the device)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
        raise ValueError("%s must be a CUDA tensor or a pinned (page-locked) CPU tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace holds fewer than %d bytes" % nbytes)
        return workspace
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def tsd_build_tree(drafter_logits: torch.Tensor, topk: int, B: int, drafter_temp: float = 1.0,
                   workspace=None, device=None) -> dict:
    """Best-first tree builder.  drafter_logits: [n_trees, n_modes, L, V]
    (bf16/fp32), on the GPU or in pinned host memory (then the outputs go to
    `device`, default the current CUDA device).  Returns parent, token,
    depth, score, rank, mode ([n_trees, B+1]), n_nodes and status
    ([n_trees])."""
    x = _logits(drafter_logits, "drafter_logits")
    if x.dim() != 4:
        raise ValueError("drafter_logits must be [n_trees, n_modes, L, V]")
    n_trees, n_modes, L, V = x.shape
    if x.is_cuda:
        dev = x.device
    else:
        dev = torch.device(device) if device is not None else \
            torch.device("cuda", torch.cuda.current_device())
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, B + 1, **i32) for k in ("parent", "token", "depth", "rank", "mode")}
    out["score"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
    out["n_nodes"] = torch.empty(n_trees, **i32)
    out["status"] = torch.empty(n_trees, **i32)
    nbytes = tsd_workspace_size(TSD_OP_BUILD_TREE, n_trees, n_modes, L, V, topk, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_build_tree")
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = load().tsd_build_tree(_ptr(x), _dtype_code(x), n_trees, n_modes, L, V, topk, B,
                                   drafter_temp, _ptr(out["parent"]), _ptr(out["token"]),
                                   _ptr(out["depth"]), _ptr(out["score"]), _ptr(out["rank"]),
                                   _ptr(out["mode"]), _ptr(out["n_nodes"]), _ptr(out["status"]),
                                   _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_build_tree")
    return out


def tsd_build_lse_tree(drafter_logits: torch.Tensor, topk: int, B: int, drafter_temp: float = 1.0,
                       log_prior=None, workspace=None, device=None) -> dict:
    """Mixture tree under the log-sum-exp score ([MFD] App. B Eq. 6): the B
    best distinct prefixes of the modes' per-depth lists, ranked by
    log sum_m pi_m Q_m(v).  drafter_logits: [n_trees, n_modes, L, V]
    (bf16/fp32, GPU or pinned host); log_prior: None (uniform) or
    [n_trees, n_modes] float32.  Returns parent, token, depth, score
    ([n_trees, B+1]), n_nodes, status and n_cand ([n_trees])."""
    x = _logits(drafter_logits, "drafter_logits")
    if x.dim() != 4:
        raise ValueError("drafter_logits must be [n_trees, n_modes, L, V]")
    n_trees, n_modes, L, V = x.shape
    dev = x.device if x.is_cuda else (torch.device(device) if device is not None else
                                      torch.device("cuda", torch.cuda.current_device()))
    lp = None
    if log_prior is not None:
        lp = log_prior
        if not (lp.dtype == torch.float32 and lp.shape == (n_trees, n_modes) and lp.is_contiguous()
                and (lp.is_cuda or lp.is_pinned())):
            raise ValueError("log_prior must be a contiguous float32 [n_trees, n_modes] tensor on "
                             "the GPU or in pinned host memory")
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, B + 1, **i32) for k in ("parent", "token", "depth")}
    out["score"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
    for k in ("n_nodes", "status", "n_cand"):
        out[k] = torch.empty(n_trees, **i32)
    nbytes = tsd_workspace_size(TSD_OP_BUILD_LSE, n_trees, n_modes, L, V, topk, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_build_lse_tree")
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = load().tsd_build_lse_tree(_ptr(x), _dtype_code(x), n_trees, n_modes, L, V, topk, B,
                                       drafter_temp, _ptr(lp) if lp is not None else None,
                                       _ptr(out["parent"]), _ptr(out["token"]), _ptr(out["depth"]),
                                       _ptr(out["score"]), _ptr(out["n_nodes"]), _ptr(out["status"]),
                                       _ptr(out["n_cand"]), _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_build_lse_tree")
    return out


def tsd_tree_mask(parent: torch.Tensor, n_nodes: torch.Tensor, prefix_len: int = 0,
                  additive: bool = False) -> dict:
    """Ancestor bitmask [n_trees, B+1, W], position ids [n_trees, B+1] and,
    if `additive`, the float mask [n_trees, B+1, prefix_len+B+1]."""
    parent = _cuda(parent, "parent", torch.int32)
    n_nodes = _cuda(n_nodes, "n_nodes", torch.int32)
    n_trees, Bp1 = parent.shape
    B = Bp1 - 1
    W = (B + 32) // 32
    dev = parent.device
    bits = torch.empty(n_trees, Bp1, W, dtype=torch.int32, device=dev)
    pos = torch.empty(n_trees, Bp1, dtype=torch.int32, device=dev)
    status = torch.empty(n_trees, dtype=torch.int32, device=dev)
    ld = prefix_len + B + 1
    add = torch.empty(n_trees, Bp1, ld, dtype=torch.float32, device=dev) if additive else None
    with torch.cuda.device(dev):
        st = load().tsd_tree_mask(_ptr(parent), _ptr(n_nodes), n_trees, B, prefix_len, _ptr(bits),
                                  _ptr(pos), _ptr(add), ld, _ptr(status), _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_tree_mask")
    return dict(anc_bits=bits, position_ids=pos, additive_mask=add, status=status)


def _verify_common(target_logits, parent, token, n_nodes):
    x = _logits(target_logits, "target_logits")
    if x.dim() != 3:
        raise ValueError("target_logits must be [n_trees, B+1, V]")
    n_trees, Bp1, V = x.shape
    parent = _cuda(parent, "parent", torch.int32)
    token = _cuda(token, "token", torch.int32)
    n_nodes = _cuda(n_nodes, "n_nodes", torch.int32)
    if tuple(parent.shape) != (n_trees, Bp1) or tuple(token.shape) != (n_trees, Bp1) \
            or tuple(n_nodes.shape) != (n_trees,):
        raise ValueError("parent/token must be [n_trees, B+1] and n_nodes [n_trees]")
    if x.is_cuda and x.device != parent.device:
        raise ValueError("target_logits and the tree must be on one device")
    return x, parent, token, n_nodes, n_trees, Bp1 - 1, V


def tsd_verify_tev(target_logits: torch.Tensor, parent: torch.Tensor, token: torch.Tensor,
                   n_nodes: torch.Tensor, temperature: float, seed: int, workspace=None,
                   with_masses: bool = True, out: dict | None = None) -> dict:
    """Tree Exit Verification.  Returns exit_node, bonus_token, accept_len,
    status ([n_trees]) and, with `with_masses`, exit_mass, prefix_prob
    ([n_trees, B+1]) and coverage ([n_trees]).  `out` may hold preallocated
    output tensors of those shapes (int32 / float32)."""
    return _tev(target_logits, parent, token, n_nodes, temperature, seed, workspace,
                with_masses, out, None)


def tsd_verify_tev_timed(target_logits: torch.Tensor, parent: torch.Tensor, token: torch.Tensor,
                         n_nodes: torch.Tensor, temperature: float, seed: int, stage_events,
                         workspace=None, with_masses: bool = True,
                         out: dict | None = None) -> dict:
    """tsd_verify_tev that records five torch.cuda.Event objects (each recorded
    once before, so that it exists) around its four kernels: before the tree
    preparation, before and after the node-row reduction, after the per-node
    combination, after the draws."""
    if len(stage_events) != 5:
        raise ValueError("stage_events must hold five CUDA events")
    handles = (ctypes.c_void_p * 5)(*[int(e.cuda_event) for e in stage_events])
    if not all(handles):
        raise ValueError("record each event once before passing it")
    return _tev(target_logits, parent, token, n_nodes, temperature, seed, workspace,
                with_masses, out, handles)


def _tev(target_logits, parent, token, n_nodes, temperature, seed, workspace, with_masses, out,
         handles) -> dict:
    x, parent, token, n_nodes, n_trees, B, V = _verify_common(target_logits, parent, token, n_nodes)
    dev = parent.device
    i32 = dict(dtype=torch.int32, device=dev)
    if out is None:
        out = {k: torch.empty(n_trees, **i32) for k in ("exit_node", "bonus_token", "accept_len", "status")}
        if with_masses:
            out["exit_mass"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
            out["prefix_prob"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
            out["coverage"] = torch.empty(n_trees, dtype=torch.float32, device=dev)
    nbytes = tsd_workspace_size(TSD_OP_VERIFY_TEV, n_trees, 1, 1, V, 1, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_verify_tev")
    ws = _workspace(nbytes, dev, workspace)
    args = [_ptr(x), _dtype_code(x), _ptr(parent), _ptr(token), _ptr(n_nodes), n_trees, B, V,
            temperature, seed, _ptr(out["exit_node"]), _ptr(out["bonus_token"]),
            _ptr(out["accept_len"]), _ptr(out.get("exit_mass")), _ptr(out.get("prefix_prob")),
            _ptr(out.get("coverage")), _ptr(out["status"]), _ptr(ws), nbytes, _stream(dev)]
    with torch.cuda.device(dev):
        if handles is None:
            st = load().tsd_verify_tev(*args)
        else:
            st = load().tsd_verify_tev_timed(*args, handles)
    if st != TSD_OK:
        raise TsdError(st, "tsd_verify_tev")
    return out


def tsd_verify_tev_noalloc(target_logits: torch.Tensor, parent: torch.Tensor,
                           token: torch.Tensor, n_nodes: torch.Tensor, temperature: float,
                           seed: int, with_masses: bool = True) -> dict:
    """tsd_verify_tev without a workspace, for callers that cannot allocate
    device memory: the library's static scratch is used instead (see
    include/tsd.h for its size limit and the one-time set-up per device).
    The outputs are allocated here only because this binding returns new
    tensors."""
    x, parent, token, n_nodes, n_trees, B, V = _verify_common(target_logits, parent, token, n_nodes)
    dev = parent.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, **i32) for k in ("exit_node", "bonus_token", "accept_len", "status")}
    if with_masses:
        out["exit_mass"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
        out["prefix_prob"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
        out["coverage"] = torch.empty(n_trees, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = load().tsd_verify_tev_noalloc(
            _ptr(x), _dtype_code(x), _ptr(parent), _ptr(token), _ptr(n_nodes), n_trees, B, V,
            temperature, seed, _ptr(out["exit_node"]), _ptr(out["bonus_token"]),
            _ptr(out["accept_len"]), _ptr(out.get("exit_mass")), _ptr(out.get("prefix_prob")),
            _ptr(out.get("coverage")), _ptr(out["status"]), _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_verify_tev_noalloc")
    return out


def tsd_verify_ddtree(target_logits: torch.Tensor, parent: torch.Tensor, token: torch.Tensor,
                      n_nodes: torch.Tensor, temperature: float, seed: int,
                      workspace=None) -> dict:
    """Predraw-and-follow.  Returns exit_node, bonus_token, accept_len, status
    ([n_trees]) and the per-node draws ([n_trees, B+1])."""
    x, parent, token, n_nodes, n_trees, B, V = _verify_common(target_logits, parent, token, n_nodes)
    dev = parent.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, **i32) for k in ("exit_node", "bonus_token", "accept_len", "status")}
    out["draws"] = torch.empty(n_trees, B + 1, **i32)
    nbytes = tsd_workspace_size(TSD_OP_VERIFY_DDTREE, n_trees, 1, 1, V, 1, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_verify_ddtree")
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = load().tsd_verify_ddtree(_ptr(x), _dtype_code(x), _ptr(parent), _ptr(token),
                                      _ptr(n_nodes), n_trees, B, V, temperature, seed,
                                      _ptr(out["exit_node"]), _ptr(out["bonus_token"]),
                                      _ptr(out["accept_len"]), _ptr(out["draws"]),
                                      _ptr(out["status"]), _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_verify_ddtree")
    return out


def tsd_exit_loss(drafter_logits: torch.Tensor, token: torch.Tensor, depth: torch.Tensor,
                  n_nodes: torch.Tensor, omega: torch.Tensor, drafter_temp: float = 1.0,
                  with_grad: bool = False, workspace=None) -> dict:
    """Exit-guided loss ([EXIT] Eq. 14 via Eq. 67).  drafter_logits:
    [n_trees, L, V] (or [n_trees, 1, L, V]); token, depth: [n_trees, B+1];
    n_nodes: [n_trees]; omega: [n_trees, B+1] float32 (TEV's exit_mass).
    Returns loss (float64 scalar tensor), loss_tree ([n_trees] float64
    numerators), status and, with `with_grad`, grad ([n_trees, L, V] float32,
    d loss / d drafter_logits)."""
    x = _logits(drafter_logits, "drafter_logits")
    if x.dim() == 4:
        if x.shape[1] != 1:
            raise ValueError("the exit loss takes one mode")
        x = x.reshape(x.shape[0], x.shape[2], x.shape[3])
    if x.dim() != 3:
        raise ValueError("drafter_logits must be [n_trees, L, V]")
    n_trees, L, V = x.shape
    token = _cuda(token, "token", torch.int32)
    depth = _cuda(depth, "depth", torch.int32)
    n_nodes = _cuda(n_nodes, "n_nodes", torch.int32)
    omega = _cuda(omega, "omega", torch.float32)
    Bp1 = token.shape[1]
    if tuple(token.shape) != (n_trees, Bp1) or tuple(depth.shape) != (n_trees, Bp1) \
            or tuple(omega.shape) != (n_trees, Bp1) or tuple(n_nodes.shape) != (n_trees,):
        raise ValueError("token/depth/omega must be [n_trees, B+1] and n_nodes [n_trees]")
    dev = token.device
    out = {"loss_tree": torch.empty(n_trees, dtype=torch.float64, device=dev),
           "loss": torch.empty((), dtype=torch.float64, device=dev),
           "status": torch.empty(n_trees, dtype=torch.int32, device=dev)}
    if with_grad:
        out["grad"] = torch.empty(n_trees, L, V, dtype=torch.float32, device=dev)
    nbytes = tsd_workspace_size(TSD_OP_EXIT_LOSS, n_trees, 1, L, V, 1, Bp1 - 1, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_exit_loss")
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = load().tsd_exit_loss(_ptr(x), _dtype_code(x), n_trees, L, V, drafter_temp, _ptr(token),
                                  _ptr(depth), _ptr(n_nodes), Bp1 - 1, _ptr(omega),
                                  _ptr(out["loss_tree"]), _ptr(out["loss"]), _ptr(out.get("grad")),
                                  _ptr(out["status"]), _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_exit_loss")
    return out


def _walk_verifier(name, target_logits, parent, token, n_nodes, temperature, seed, workspace,
                   q_child=None):
    x, parent, token, n_nodes, n_trees, B, V = _verify_common(target_logits, parent, token, n_nodes)
    dev = parent.device
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, **i32) for k in ("exit_node", "bonus_token", "accept_len", "status")}
    nbytes = tsd_workspace_size(TSD_OP_VERIFY_TEV, n_trees, 1, 1, V, 1, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, name)
    ws = _workspace(nbytes, dev, workspace)
    lib = load()
    with torch.cuda.device(dev):
        head = [_ptr(x), _dtype_code(x), _ptr(parent), _ptr(token), _ptr(n_nodes)]
        if q_child is not None:
            q_child = _cuda(q_child, "q_child", torch.float32)
            if tuple(q_child.shape) != (n_trees, B + 1):
                raise ValueError("q_child must be [n_trees, B+1]")
            head.append(_ptr(q_child))
        st = getattr(lib, name)(*head, n_trees, B, V, temperature, seed, _ptr(out["exit_node"]),
                                _ptr(out["bonus_token"]), _ptr(out["accept_len"]),
                                _ptr(out["status"]), _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, name)
    return out


def tsd_verify_seqres(target_logits: torch.Tensor, parent: torch.Tensor, token: torch.Tensor,
                      n_nodes: torch.Tensor, temperature: float, seed: int,
                      workspace=None) -> dict:
    """Exact sequential residual verification ([EXIT] App. A.4.2).  Returns
    exit_node, bonus_token, accept_len, status ([n_trees])."""
    return _walk_verifier("tsd_verify_seqres", target_logits, parent, token, n_nodes, temperature,
                          seed, workspace)


def tsd_verify_proposal(target_logits: torch.Tensor, parent: torch.Tensor, token: torch.Tensor,
                        n_nodes: torch.Tensor, q_child: torch.Tensor, temperature: float, seed: int,
                        workspace=None) -> dict:
    """Proposal-aware verification ([CAST] App. B.1 Thm. 3).  q_child:
    [n_trees, B+1] float32, the proposal's probability of each node's token
    under its parent.  Returns exit_node, bonus_token, accept_len, status."""
    return _walk_verifier("tsd_verify_proposal", target_logits, parent, token, n_nodes, temperature,
                          seed, workspace, q_child=q_child)


def tsd_build_forest(drafter_logits: torch.Tensor, topk: int, B: int, M_max: int, l0: float,
                     c1: float, drafter_temp: float = 1.0, workspace=None, device=None) -> dict:
    """Cost-aware widths under a shared budget ([CAST] App. B.4): one tree per
    request, built to the cap B, then the globally best M* <= M_max prefixes
    by the batched stopping rule with round time l0 + c1 M.  drafter_logits:
    [n_trees, L, V] or [n_trees, 1, L, V].  Returns parent, token, depth,
    score ([n_trees, B+1]), n_nodes, status ([n_trees]) and total (M*)."""
    x = _logits(drafter_logits, "drafter_logits")
    if x.dim() == 3:
        x = x.reshape(x.shape[0], 1, x.shape[1], x.shape[2])
    if x.dim() != 4 or x.shape[1] != 1:
        raise ValueError("drafter_logits must be [n_trees, L, V] (one mode)")
    n_trees, _, L, V = x.shape
    dev = x.device if x.is_cuda else (torch.device(device) if device is not None else
                                      torch.device("cuda", torch.cuda.current_device()))
    i32 = dict(dtype=torch.int32, device=dev)
    out = {k: torch.empty(n_trees, B + 1, **i32) for k in ("parent", "token", "depth")}
    out["score"] = torch.empty(n_trees, B + 1, dtype=torch.float32, device=dev)
    out["n_nodes"] = torch.empty(n_trees, **i32)
    out["status"] = torch.empty(n_trees, **i32)
    out["total"] = torch.empty((), **i32)
    nbytes = tsd_workspace_size(TSD_OP_BUILD_FOREST, n_trees, 1, L, V, topk, B, x.dtype)
    if nbytes == 0:
        raise TsdError(TSD_ERR_INVALID_ARG, "tsd_build_forest")
    ws = _workspace(nbytes, dev, workspace)
    with torch.cuda.device(dev):
        st = load().tsd_build_forest(_ptr(x), _dtype_code(x), n_trees, L, V, topk, B, drafter_temp,
                                     int(M_max), float(l0), float(c1), _ptr(out["parent"]),
                                     _ptr(out["token"]), _ptr(out["depth"]), _ptr(out["score"]),
                                     _ptr(out["n_nodes"]), _ptr(out["status"]), _ptr(out["total"]),
                                     _ptr(ws), nbytes, _stream(dev))
    if st != TSD_OK:
        raise TsdError(st, "tsd_build_forest")
    return out

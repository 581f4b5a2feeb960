"""CPU-only checks of the C ABI: the library builds and loads, exports every
entry point include/tsd.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

import tree_speculative_decoding_position_gb300 as tsd
from tree_speculative_decoding_position_gb300 import build as tsd_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tsd.h")


@pytest.fixture(scope="module")
def lib():
    tsd_build.build()
    return tsd.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tsd_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted([
        "tsd_build_forest", "tsd_build_lse_tree", "tsd_build_tree", "tsd_debug_check_failures",
        "tsd_status_string", "tsd_tree_mask", "tsd_verify_ddtree",
        "tsd_exit_loss", "tsd_verify_proposal", "tsd_verify_seqres", "tsd_verify_tev",
        "tsd_verify_tev_noalloc", "tsd_verify_tev_timed", "tsd_workspace_size"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_default_build_has_no_checks(lib):
    """The product library compiles the bounds checks out: the reader returns 0
    without touching a device (this runs with no GPU)."""
    assert tsd.tsd_debug_check_failures() == 0


def test_status_strings(lib):
    for code in range(7):
        assert tsd.tsd_status_string(code)
    assert tsd.tsd_status_string(0) == "ok"
    assert tsd.tsd_status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    import torch
    V = 151936
    n = tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 32, 1, 1, V, 1, 256, torch.bfloat16)
    # per node: CSR/depth/stat arrays plus one 16-byte record per 4096-token chunk
    assert n >= 32 * 257 * 38 * 16
    assert n % 256 == 0
    assert tsd.tsd_workspace_size(tsd.TSD_OP_VERIFY_TEV, 0, 1, 1, V, 1, 256, torch.bfloat16) == 0
    assert tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 16, 8, 16, V, 8, 128, torch.bfloat16) > 0
    # top-k above the cap, or rank digits that do not fit the 56-bit tie key
    assert tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 1, 1, 16, V, 33, 64, torch.bfloat16) == 0
    assert tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 1, 1, 20, V, 16, 64, torch.bfloat16) == 0
    assert tsd.tsd_workspace_size(tsd.TSD_OP_BUILD_TREE, 1, 9, 16, V, 8, 64, torch.bfloat16) == 0


def test_invalid_arguments_are_rejected_on_the_host(lib):
    """Null pointers and out-of-range sizes return TSD_ERR_INVALID_ARG before
    anything touches a GPU (this runs on a machine without one)."""
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: the checks fail first
    st = lib.tsd_verify_tev(None, 0, fake, fake, fake, 1, 8, 32, 1.0, 0, fake, fake, fake,
                            None, None, None, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG
    st = lib.tsd_verify_tev(fake, 0, fake, fake, fake, 1, 8, 32, -1.0, 0, fake, fake, fake,
                            None, None, None, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG
    st = lib.tsd_verify_tev(fake, 7, fake, fake, fake, 1, 8, 32, 1.0, 0, fake, fake, fake,
                            None, None, None, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG
    st = lib.tsd_verify_tev(fake, 0, fake, fake, fake, 1, 5000, 32, 1.0, 0, fake, fake, fake,
                            None, None, None, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG
    # workspace too small
    st = lib.tsd_verify_tev(fake, 0, fake, fake, fake, 1, 8, 32, 1.0, 0, fake, fake, fake,
                            None, None, None, fake, fake, 16, None)
    assert st == tsd.TSD_ERR_WORKSPACE
    st = lib.tsd_verify_tev_timed(fake, 0, fake, fake, fake, 1, 8, 32, 1.0, 0, fake, fake, fake,
                                  None, None, None, fake, fake, 1 << 20, None, None)
    assert st == tsd.TSD_ERR_INVALID_ARG  # no stage events
    st = lib.tsd_verify_ddtree(fake, 0, fake, fake, None, 1, 8, 32, 1.0, 0, fake, fake, fake,
                               None, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG
    st = lib.tsd_build_tree(fake, 0, 1, 1, 4, 32, 4, 8, 0.0, fake, fake, fake, fake, None, None,
                            fake, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG  # drafter temperature must be > 0
    st = lib.tsd_build_tree(fake, 0, 1, 1, 4, 32, 64, 8, 1.0, fake, fake, fake, fake, None, None,
                            fake, fake, fake, 1 << 20, None)
    assert st == tsd.TSD_ERR_INVALID_ARG  # top-k above V
    st = lib.tsd_tree_mask(fake, fake, 1, 8, 3, fake, fake, fake, 5, fake, None)
    assert st == tsd.TSD_ERR_INVALID_ARG  # mask_ld < P + B + 1
    st = lib.tsd_tree_mask(fake, fake, 1, 8, -1, fake, fake, None, 0, fake, None)
    assert st == tsd.TSD_ERR_INVALID_ARG


def test_pageable_host_logits_are_refused(lib):
    """Logits may live on the GPU or in page-locked host memory; ordinary
    (pageable) host tensors are refused before any CUDA call."""
    import torch
    with pytest.raises(ValueError):
        tsd.tsd_build_tree(torch.zeros(1, 1, 4, 32), topk=4, B=8)
    with pytest.raises(ValueError):
        tsd.tsd_verify_tev(torch.zeros(1, 9, 32), torch.zeros(1, 9, dtype=torch.int32),
                           torch.zeros(1, 9, dtype=torch.int32), torch.ones(1, dtype=torch.int32),
                           1.0, seed=0)


def test_newer_operations_check_sizes_and_arguments_on_the_host(lib):
    """Workspace sizes and argument errors of the exit loss, the shared-budget
    widths, the log-sum-exp tree and the two walk verifiers, with no GPU."""
    import torch
    V, bf = 151936, torch.bfloat16
    ws = tsd.tsd_workspace_size
    assert ws(tsd.TSD_OP_EXIT_LOSS, 32, 1, 16, V, 1, 256, bf) > 0
    assert ws(tsd.TSD_OP_EXIT_LOSS, 32, 1, 32, V, 1, 256, bf) == 0        # L above TSD_MAX_L
    assert ws(tsd.TSD_OP_BUILD_FOREST, 32, 1, 16, V, 8, 256, bf) > 0
    assert ws(tsd.TSD_OP_BUILD_FOREST, 33, 1, 16, V, 8, 256, bf) == 0     # > 8192 candidates
    assert ws(tsd.TSD_OP_BUILD_FOREST, 2, 2, 16, V, 8, 64, bf) == 0       # one mode only
    assert ws(tsd.TSD_OP_BUILD_LSE, 16, 8, 16, V, 8, 128, bf) > 0
    assert ws(tsd.TSD_OP_BUILD_LSE, 1, 8, 16, V, 8, 600, bf) == 0         # n_modes * B > 4096
    assert ws(tsd.TSD_OP_BUILD_LSE, 1, 1, 16, V, 8, 2049, bf) == 0        # B > 2048
    assert ws(tsd.TSD_OP_BUILD_LSE, 1, 1, 16, V, 32, 2048, bf) == 0       # lists beyond shared memory
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: the checks fail first
    big = 1 << 30
    st = lib.tsd_build_forest(fake, 0, 4, 4, 32, 4, 8, 1.0, 10, 1.0, -0.5, fake, fake, fake, fake,
                              fake, fake, fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # c1 < 0
    st = lib.tsd_build_forest(fake, 0, 4, 4, 32, 4, 8, 1.0, 10, 0.0, 0.5, fake, fake, fake, fake,
                              fake, fake, fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # l0 must be > 0
    st = lib.tsd_build_forest(fake, 0, 64, 4, 512, 4, 200, 1.0, 10, 1.0, 0.5, fake, fake, fake,
                              fake, fake, fake, fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # 12800 candidates
    st = lib.tsd_build_lse_tree(fake, 0, 1, 2, 4, 512, 4, 2049, 1.0, None, fake, fake, fake, fake,
                                fake, fake, None, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # B > 2048
    st = lib.tsd_build_lse_tree(fake, 0, 1, 8, 4, 512, 4, 600, 1.0, None, fake, fake, fake, fake,
                                fake, fake, None, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # n_modes * B > 4096
    st = lib.tsd_build_lse_tree(fake, 0, 1, 2, 4, 512, 4, 64, 0.0, None, fake, fake, fake, fake,
                                fake, fake, None, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # drafter temperature 0
    st = lib.tsd_exit_loss(fake, 0, 1, 4, 32, 1.0, None, fake, fake, 8, fake, fake, fake, None,
                           fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # no tokens
    st = lib.tsd_verify_seqres(fake, 0, fake, fake, fake, 1, 8, 32, -1.0, 0, fake, fake, fake,
                               fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # negative temperature
    st = lib.tsd_verify_proposal(fake, 0, fake, fake, fake, None, 1, 8, 32, 1.0, 0, fake, fake,
                                 fake, fake, fake, big, None)
    assert st == tsd.TSD_ERR_INVALID_ARG                                   # no proposal

"""sv_accept_tree_noalloc: tree acceptance for callers that cannot allocate device
memory (the library keeps its per-row statistics in a fixed device array).

Called through the C ABI with raw pointers and compared with sv_accept_tree (which
takes a caller workspace) on the same inputs, twice in a row, so that a second call
that reuses the fixed array's leftover contents is covered.  This file is collected
last so that a run stopping at its first failure has run every other test already.
"""
import ctypes

import pytest
import torch

import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import build as svbuild
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KEYS = ("path_nodes", "tokens", "num_emitted", "num_accepted", "near_ties")


def _noalloc_call(lib, mode, tl, q, parent, toks, seed, rnd, outs):
    par = (ctypes.c_int32 * len(parent))(*parent)
    B, N, V = tl.shape
    Dq = 0 if q is None else q.shape[1]
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sv_accept_tree_noalloc(mode, 1, B, N, V, par, 0, P(toks), P(tl), P(q), sv.Q_LOGITS, Dq,
                                      1.0, 0, 1.0, seed, rnd, P(outs["path_nodes"]), P(outs["tokens"]),
                                      P(outs["num_emitted"]), P(outs["num_accepted"]),
                                      P(outs["near_ties"]), stream)


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_noalloc_matches_workspace_entry_point(cuda_ok, mode):
    svbuild.build()
    lib = sv.load_library()
    parent = wl.TREE_T26
    B, V = 48, 4000
    W = max(wl.depths(parent)) + 1
    lg = wl.medusa_logits(B, parent, V, sigma=3.0, seed=77, coverage=True, coverage_sigma=0.7)
    dev = torch.device("cuda")
    tl = lg["target_logits"].to(dev)
    q = lg["draft_logits"].to(dev) if mode == sv.EXACT else None
    toks = lg["node_tokens"].to(dev)
    for call in range(2):
        seed, rnd = 5 + call, call
        ref = sv.sv_accept_tree(mode, tl, q, sv.Q_LOGITS, parent, toks, seed=seed, round_=rnd)
        outs = {k: torch.full((B, W) if k in ("path_nodes", "tokens") else (B,), -7,
                              dtype=torch.int32, device=dev) for k in KEYS}
        assert _noalloc_call(lib, mode, tl, q, parent, toks, seed, rnd, outs) == sv.SV_OK, \
            lib.sv_last_error().decode()
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(outs[k], ref[k]), (call, k)
    assert sv.sv_read_device_status() == 0


def test_noalloc_rejects_rows_beyond_its_scratch(cuda_ok):
    svbuild.build()
    lib = sv.load_library()
    par = (ctypes.c_int32 * 5)(-1, 0, 1, 2, 3)
    P = ctypes.c_void_p(16)
    # 20000 * (5 + 4) rows > 65536: rejected before anything is launched
    rc = lib.sv_accept_tree_noalloc(sv.EXACT, 1, 20000, 5, 64, par, 0, P, P, P, sv.Q_LOGITS, 4, 1.0,
                                    0, 1.0, 0, 0, P, P, P, P, P, None)
    assert rc == sv.SV_ERR_UNSUPPORTED
    assert "fixed scratch" in lib.sv_last_error().decode()

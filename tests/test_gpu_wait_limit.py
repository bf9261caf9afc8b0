"""The tensor-core attention kernel's bounded waits, made to run out.

A unit cut across every CTA (one sequence and kv head, a 32K prefix) makes CTAs wait for
copies, MMAs and each other's partial results.  With the wait limit set far below the time
the first tile takes to arrive, the waits give up: the call returns, the kernel reports
SV_DEV_TIMEOUT, and -- with the limit restored -- the next call on the same workspace
matches the oracle.  Nothing is hung or faulted: the waits are bounded by design and the
test only shortens their bound.
"""
import math

import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_returns_and_leaves_the_workspace_usable(cuda_ok):
    par = wl.chain_parent(3)
    B, N, Hq, Hkv, D = 1, 4, 8, 1, 128
    inp = wl.attention_inputs(B, N, Hq, Hkv, D, [32768], dtype=torch.bfloat16, seed=13)
    assert sv.sv_tree_attention_path(torch.bfloat16, N, Hq, Hkv, D) == 1
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cache = sv.KVCache(g["cache_k"], g["cache_v"], g["prefix_len"])
    size = sv.sv_tree_attention_workspace_size(torch.bfloat16, B, N, Hq, Hkv, D, 32768 + 8)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(D)
    sv.sv_read_device_status()
    try:
        sv.sv_set_wait_limit_ns(100)  # 100 ns: far below the first tile's arrival
        sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, par, scale, workspace=ws)
        torch.cuda.synchronize()
        st = sv.sv_read_device_status()
    finally:
        sv.sv_set_wait_limit_ns(0)
    assert st & sv.SV_DEV_TIMEOUT, f"status {st:#x}"
    # the default limit again: the same workspace serves the next calls, which match the oracle
    ref = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], par, scale)
    for _ in range(2):
        out = sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, par, scale,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert sv.sv_read_device_status() == 0
        err = (out.double().cpu() - ref).abs().max().item()
        assert err < 2e-2, f"max-abs error {err} after the timed-out call"

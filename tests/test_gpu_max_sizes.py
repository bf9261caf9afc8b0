"""The largest sizes the ABI accepts, against the CPU oracle: top-k at SV_MAX_TOP_K, the
longest chain (63 drafts, a 64-node tree of depth 63) and the longest tree-attention chain
over ragged prefixes."""
import math

import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_TOP_K = 1024  # SV_MAX_TOP_K
MAX_GAMMA = 63    # SV_MAX_TREE_NODES - 1


def _chain(mode, lg, T=1.0, top_k=0, seed=3, rnd=1):
    dev = torch.device("cuda")
    q = None if mode == sv.GREEDY else lg["draft_logits"].to(dev)
    out = sv.sv_accept_chain(mode, lg["target_logits"].to(dev), q, sv.Q_LOGITS,
                             lg["draft_tokens"].to(dev), temperature=T, top_k=top_k, seed=seed,
                             round_=rnd)
    torch.cuda.synchronize()
    ref = oracle.accept_chain(mode, lg["target_logits"], None if q is None else lg["draft_logits"],
                              oracle.Q_LOGITS, lg["draft_tokens"], temperature=T, top_k=top_k,
                              seed=seed, round_=rnd)
    return out, ref


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_top_k_at_its_maximum(cuda_ok, mode):
    lg = wl.chain_logits(16, 4, 32768, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16,
                         temperature=0.8, top_k=MAX_TOP_K, seed=91)
    out, ref = _chain(mode, lg, T=0.8, top_k=MAX_TOP_K, seed=4, rnd=2)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_longest_chain(cuda_ok, mode):
    """63 drafts: the draft logits stay close to the target's, so that long prefixes of the
    chain are accepted and the deepest decisions are reached."""
    lg = wl.chain_logits(8, MAX_GAMMA, 4000, sigma=2.0, draft_sigma=0.05, dtype=torch.bfloat16, seed=92)
    out, ref = _chain(mode, lg, seed=6, rnd=3)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"])
    if mode == sv.EXACT:
        assert int(ref["num_accepted"].max()) > 8  # the deep nodes are decided
    assert sv.sv_read_device_status() == 0


def test_longest_chain_attention(cuda_ok):
    """A 64-node chain (depth 63) over ragged prefixes: every node sees the prefix and all
    the nodes before it."""
    parent = wl.chain_parent(MAX_GAMMA)
    lens = [0, 5, 128, 300]
    inp = wl.attention_inputs(len(lens), len(parent), 8, 2, 128, lens, dtype=torch.bfloat16,
                              seed=93, device="cuda")
    cache = sv.KVCache(inp["cache_k"], inp["cache_v"], inp["prefix_len"])
    out = sv.sv_tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], cache, parent, 1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    ref = oracle.tree_attention(inp["q"].cpu(), inp["k_tree"].cpu(), inp["v_tree"].cpu(),
                                inp["cache_k"].cpu(), inp["cache_v"].cpu(), inp["prefix_len"].cpu(),
                                parent, 1.0 / math.sqrt(128))
    err = (out.double().cpu() - ref).abs().max().item()
    assert err < 2e-2, err
    assert sv.sv_read_device_status() == 0

"""Typical acceptance on the GPU against the oracle (the Medusa paper's rule: accept x iff
p_parent(x) > min(epsilon, delta * exp(-H(p_parent)))).  Decisions, paths and the greedy
token after the kept node are integers and must be identical outside the reported near ties
(decision class only: the rule draws no uniforms)."""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KEYS = ["path_nodes", "tokens", "num_emitted", "num_accepted"]


@pytest.mark.parametrize("parent,V,dtype,T,eps,delta", [
    (wl.TREE_T26, 2000, torch.bfloat16, 1.0, 0.3, 0.09),
    (wl.TREE_T64, 32000, torch.bfloat16, 0.7, 0.2, 0.3),
    (wl.chain_parent(5), 128256, torch.bfloat16, 1.0, 0.09, 0.3),
    (wl.TREE_EXAMPLE7, 4000, torch.float32, 1.3, 0.5, 1.0),
])
def test_typical_matches_oracle(cuda_ok, parent, V, dtype, T, eps, delta):
    B = 32
    lg = wl.medusa_logits(B, parent, V, sigma=3.0, dtype=dtype, seed=61, coverage=True,
                          coverage_sigma=0.5)
    dev = torch.device("cuda")
    sv.sv_read_device_status()
    out = sv.sv_accept_typical(lg["target_logits"].to(dev), parent, lg["node_tokens"].to(dev),
                               temperature=T, epsilon=eps, delta=delta)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ref = oracle.accept_typical(lg["target_logits"], parent, lg["node_tokens"], temperature=T,
                                epsilon=eps, delta=delta)
    compare(out, ref, KEYS, max_exempt_frac=0.03)
    assert int((out["near_ties"].cpu() >> 16).sum()) == 0  # no sample ties: no sampling
    assert int(ref["num_accepted"].sum()) > 0


def test_typical_per_sequence_trees(cuda_ok):
    trees = [list(wl.TREE_T26), list(wl.TREE_T64[:26]), list(wl.TREE_EXAMPLE7) + [0] * 19]
    B, V = 12, 3000
    par = [trees[b % 3] for b in range(B)]
    tl, tk = [], []
    for b in range(B):
        lg = wl.medusa_logits(1, par[b], V, sigma=3.0, seed=70 + b, coverage=True, coverage_sigma=0.5)
        tl.append(lg["target_logits"])
        tk.append(lg["node_tokens"])
    tl, tk = torch.cat(tl), torch.cat(tk)
    dev = torch.device("cuda")
    out = sv.sv_accept_typical(tl.to(dev), torch.tensor(par, dtype=torch.int32, device=dev),
                               tk.to(dev), epsilon=0.3, delta=0.09)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ref = oracle.accept_typical(tl, par, tk, epsilon=0.3, delta=0.09)
    compare(out, ref, KEYS, max_exempt_frac=0.1)


def test_typical_limits(cuda_ok):
    """epsilon = 0: every candidate with mass is accepted (the deepest node wins); a
    threshold of 1 accepts none and emits the root row's argmax."""
    parent = wl.TREE_T26
    B, V = 16, 1000
    lg = wl.medusa_logits(B, parent, V, sigma=2.0, seed=81)
    dev = torch.device("cuda")
    out = sv.sv_accept_typical(lg["target_logits"].to(dev), parent, lg["node_tokens"].to(dev),
                               epsilon=0.0, delta=0.0)
    torch.cuda.synchronize()
    assert bool((out["num_accepted"].cpu() == max(wl.depths(parent))).all())
    out = sv.sv_accept_typical(lg["target_logits"].to(dev), parent, lg["node_tokens"].to(dev),
                               epsilon=1.0, delta=1e9)
    torch.cuda.synchronize()
    assert bool((out["num_accepted"].cpu() == 0).all())
    am = lg["target_logits"][:, 0].float().argmax(dim=-1).to(torch.int32)
    assert torch.equal(out["tokens"][:, 0].cpu(), am)

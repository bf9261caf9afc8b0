"""Pins of the oracle's LM-head projection and of acceptance over its double logits (CPU).

* Weight rows that are unit vectors pick single hidden entries (a transposed operand or a
  wrong index fails), and a hand-computed 1 x 3 by 4 x 3 example.
* Rows do not mix: changing one hidden row changes only that row's logits.
* Scaling the weight by 2 scales every logit by 2 exactly (bf16 inputs, double sums).
* Acceptance over the float64 logits equals acceptance over the same values stored as
  float32 when the values are exactly representable (integers), for chains and trees, so
  the double reading of the logits is the same procedure.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_sv_gb300 import workloads as wl


def test_unit_weight_rows_pick_hidden_entries():
    rows, Dm, V = 5, 12, 40
    g = torch.Generator().manual_seed(1)
    h = torch.randn((rows, Dm), generator=g).to(torch.bfloat16)
    pick = torch.randint(0, Dm, (V,), generator=g)
    w = torch.zeros((V, Dm), dtype=torch.bfloat16)
    w[torch.arange(V), pick] = 1.0
    z = oracle.lm_head(h, w)
    assert z.shape == (rows, V) and z.dtype == torch.float64
    assert torch.equal(z, h.double()[:, pick])


def test_hand_computed_example():
    h = torch.tensor([[1.0, 2.0, 3.0]], dtype=torch.float32)
    w = torch.tensor([[1, 0, 0], [0, 1, 0], [1, 1, 1], [2, -1, 0.5]], dtype=torch.float32)
    assert oracle.lm_head(h, w).tolist() == [[1.0, 2.0, 6.0, 1.5]]
    # leading dimensions are kept: [B, N, Dm] -> [B, N, V]
    h3 = h.view(1, 1, 3).expand(2, 3, 3).contiguous()
    assert oracle.lm_head(h3, w).shape == (2, 3, 4)


def test_rows_do_not_mix_and_scaling_is_exact():
    rows, Dm, V = 6, 64, 96
    g = torch.Generator().manual_seed(2)
    h = torch.randn((rows, Dm), generator=g).to(torch.bfloat16)
    w = torch.randn((V, Dm), generator=g).to(torch.bfloat16)
    z = oracle.lm_head(h, w)
    h2 = h.clone()
    h2[3] = torch.randn(Dm, generator=g).to(torch.bfloat16)
    z2 = oracle.lm_head(h2, w)
    keep = [r for r in range(rows) if r != 3]
    assert torch.equal(z[keep], z2[keep]) and not torch.equal(z[3], z2[3])
    assert torch.equal(oracle.lm_head(h, (w.float() * 2).to(torch.bfloat16)), 2 * z)


def test_shape_errors():
    with pytest.raises(ValueError):
        oracle.lm_head(torch.zeros((2, 8)), torch.zeros((16, 7)))
    with pytest.raises(TypeError):
        oracle.lm_head(torch.zeros((2, 8), dtype=torch.float64), torch.zeros((16, 8)))


def _integer_inputs(B, N, Dm, V, seed):
    """Small-integer hidden states and weights: every logit is an integer below 2^24, exact
    in float32 and in double."""
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(-3, 4, (B, N, Dm), generator=g).to(torch.bfloat16)
    w = torch.randint(-2, 3, (V, Dm), generator=g).to(torch.bfloat16)
    return h, w


@pytest.mark.parametrize("T,top_k", [(1.0, 0), (2.5, 12)])
def test_chain_acceptance_over_double_logits(T, top_k):
    B, gamma, Dm, V = 200, 4, 16, 64
    h, w = _integer_inputs(B, gamma + 1, Dm, V, seed=3)
    z64 = oracle.lm_head(h, w)
    z32 = z64.float()
    assert torch.equal(z32.double(), z64)
    qh, _ = _integer_inputs(B, gamma, Dm, V, seed=4)
    q64 = oracle.lm_head(qh, w)
    toks = torch.randint(0, V, (B, gamma), generator=torch.Generator().manual_seed(5),
                         dtype=torch.int32)
    a = oracle.accept_chain(oracle.EXACT, z64, q64, oracle.Q_LOGITS, toks, temperature=T,
                            top_k=top_k, seed=7, round_=1)
    b = oracle.accept_chain(oracle.EXACT, z32, q64.float(), oracle.Q_LOGITS, toks,
                            temperature=T, top_k=top_k, seed=7, round_=1)
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties"):
        assert torch.equal(a[k], b[k]), k
    # greedy: the first emitted token is row 0's argmax whether or not draft 1 passed
    # (integer logits tie often: the lowest id wins, as torch.argmax returns it)
    g = oracle.accept_chain(oracle.GREEDY, z64, None, oracle.Q_LOGITS, toks)
    assert torch.equal(g["tokens"][:, 0], z64[:, 0].argmax(-1).int())


def test_tree_acceptance_over_double_logits():
    parent = wl.TREE_T26
    N, B, Dm, V = len(parent), 64, 16, 64
    h, w = _integer_inputs(B, N, Dm, V, seed=8)
    z64 = oracle.lm_head(h, w)
    Dq = max(wl.depths(parent))
    qh, _ = _integer_inputs(B, Dq, Dm, V, seed=9)
    q64 = oracle.lm_head(qh, w)
    toks = torch.randint(0, V, (B, N), generator=torch.Generator().manual_seed(10),
                         dtype=torch.int32)
    for fn in (lambda z, q: oracle.accept_tree(oracle.EXACT, z, q, oracle.Q_LOGITS, parent, toks,
                                               temperature=3.0, seed=2),
               lambda z, q: oracle.accept_tree_recursive(z, q, oracle.Q_LOGITS, parent, toks,
                                                         temperature=3.0, seed=2)):
        a, b = fn(z64, q64), fn(z64.float(), q64.float())
        for k in ("tokens", "num_emitted", "num_accepted", "path_nodes"):
            assert torch.equal(a[k], b[k]), k
    assert np.isfinite(z64.numpy()).all()

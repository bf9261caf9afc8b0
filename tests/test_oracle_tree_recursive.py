"""Pins of the oracle's exact tree acceptance with siblings tried in rank order (CPU only).

* On a chain (one child per node) it must be the chain procedure, bit for bit.
* With sibling drafts sampled independently from q, the first emitted token must follow the
  target distribution p (the multi-candidate form of the acceptance rule's guarantee,
  hncyxsy.com section 2.1): a chi-square test over many sequences.
* Special cases: p == q accepts the first child; disjoint supports reject every child and
  sample from p; a rejected first child leaves the residual to the second.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verify_sv_gb300 import workloads as wl


def _log(p):
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -np.inf)


@pytest.mark.parametrize("top_k,T,top_p", [(0, 1.0, 1.0), (5, 0.7, 1.0), (8, 0.9, 0.85)])
def test_chain_is_the_chain_procedure(top_k, T, top_p):
    B, gamma, V = 300, 5, 64
    lg = wl.chain_logits(B, gamma, V, sigma=2.0, draft_sigma=0.7, dtype=torch.bfloat16,
                         temperature=T, top_k=top_k, top_p=top_p, seed=41)
    ch = oracle.accept_chain(oracle.EXACT, lg["target_logits"], lg["draft_logits"], oracle.Q_LOGITS,
                             lg["draft_tokens"], temperature=T, top_k=top_k, top_p=top_p, seed=9,
                             round_=2)
    nt = torch.zeros((B, gamma + 1), dtype=torch.int32)
    nt[:, 1:] = lg["draft_tokens"]
    tr = oracle.accept_tree_recursive(lg["target_logits"], lg["draft_logits"], oracle.Q_LOGITS,
                                      wl.chain_parent(gamma), nt, temperature=T, top_k=top_k,
                                      top_p=top_p, seed=9, round_=2)
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties", "flags"):
        assert torch.equal(ch[k], tr[k]), k


def _one_level(B, p, q, m, seed):
    """A root with m children whose tokens are drawn independently from q (probabilities)."""
    V = p.shape[0]
    rng = np.random.default_rng(seed)
    tl = torch.from_numpy(_log(p).astype(np.float32)).view(1, 1, V).expand(B, m + 1, V).contiguous()
    qq = torch.from_numpy(q.astype(np.float32)).view(1, 1, V).expand(B, 1, V).contiguous()
    toks = np.zeros((B, m + 1), dtype=np.int32)
    toks[:, 1:] = rng.choice(V, size=(B, m), p=q / q.sum())
    return tl, qq, torch.from_numpy(toks), [-1] + [0] * m


@pytest.mark.parametrize("m", [2, 3])
def test_first_token_follows_p_with_independent_sibling_drafts(m):
    V, B = 16, 400_000
    rng = np.random.default_rng(11 + m)
    p = rng.dirichlet(np.full(V, 0.7))
    q = rng.dirichlet(np.full(V, 0.7))
    tl, qq, toks, parent = _one_level(B, p, q, m, seed=5)
    out = oracle.accept_tree_recursive(tl, qq, oracle.Q_PROBS_F32, parent, toks, seed=3, round_=1)
    first = out["tokens"][:, 0].numpy()
    counts = np.bincount(first, minlength=V)
    p0 = np.exp(_log(p).astype(np.float32).astype(np.float64))
    p0 /= p0.sum()
    chi2, pval = stats.chisquare(counts, B * p0)
    assert pval > 1e-4, (chi2, pval)
    # the independent-decision rule of accept_tree does not preserve p here: its first
    # token over-represents the drafts (a check that the test can tell the two apart)
    ind = oracle.accept_tree(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, parent, toks, seed=3, round_=1)
    c2 = np.bincount(ind["tokens"][:, 0].numpy(), minlength=V)
    assert stats.chisquare(c2, B * p0)[1] < 1e-6


def test_special_cases():
    V, B = 8, 2000
    p = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0])
    # p == q: the first child is always accepted
    tl, qq, toks, parent = _one_level(B, p, p.copy(), 3, seed=1)
    out = oracle.accept_tree_recursive(tl, qq, oracle.Q_PROBS_F32, parent, toks, seed=2)
    assert torch.all(out["path_nodes"][:, 1] == 1)
    # disjoint supports: every child rejected, the token comes from p
    q = np.array([0, 0, 0, 0, 0.25, 0.25, 0.25, 0.25])
    tl, qq, toks, parent = _one_level(B, p, q, 3, seed=1)
    out = oracle.accept_tree_recursive(tl, qq, oracle.Q_PROBS_F32, parent, toks, seed=2)
    assert torch.all(out["num_accepted"] == 0)
    assert torch.all(out["tokens"][:, 0] < 4)
    # a rejected first child hands the residual to the second: q puts all mass on token 0
    # (p = 0.4 there), the first child drafts 0 and the second drafts 1.  The second is
    # accepted iff the first was rejected, with probability p'(1)/q(1) where q(1) = 0 ->
    # ratio +inf (accepted, reported in the flags)
    q = np.zeros(V)
    q[0] = 1.0
    tl = torch.from_numpy(_log(p).astype(np.float32)).view(1, 1, V).expand(B, 3, V).contiguous()
    qq = torch.from_numpy(q.astype(np.float32)).view(1, 1, V).expand(B, 1, V).contiguous()
    toks = torch.tensor([[0, 0, 1]], dtype=torch.int32).expand(B, 3).contiguous()
    out = oracle.accept_tree_recursive(tl, qq, oracle.Q_PROBS_F32, [-1, 0, 0], toks, seed=4)
    first_acc = (out["path_nodes"][:, 1] == 1).double().mean().item()
    assert abs(first_acc - 0.4) < 4 * np.sqrt(0.24 / B)
    assert torch.all(out["num_accepted"] == 1)  # the second is accepted whenever reached

"""Pins of the oracle's verification of deterministic drafts (CPU only).

Prompt-lookup drafts are copies, not samples: the jennyma11 blog ("投机解码的五条路线",
section "Prompt Lookup / N-gram") sends them to the target's verification like any other
drafts.  Their draft distribution is a point mass, q = e_x, so the rule of hncyxsy.com
sections 2.1-2.2 accepts x iff u < p(x) and, after a rejection, samples norm([p - e_x]+),
which is p with x removed.  Pinned here:
  - distribution preservation: the first emitted token follows p_0 whatever the fixed draft
    (chi-square), and the second follows p_1 once the first draft passed;
  - the pages' closed form: with p_i(x_i) = alpha at every position the mean emitted count
    is (1 - alpha^(gamma+1)) / (1 - alpha) = 3.3616 at alpha = 0.8, gamma = 4;
  - the residual never returns the rejected draft;
  - a draft of -1 ends the chain: [x1, -1, -1, -1] equals the one-draft chain [x1].
"""
import math

import numpy as np
import torch
from scipy import stats

import oracle

V = 16


def _log(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -np.inf)


def _rows(B, p_rows):
    return torch.from_numpy(_log(p_rows).astype(np.float32)).unsqueeze(0).expand(
        B, len(p_rows), V).contiguous()


def _run(tl, drafts, seed=7, rnd=0, mode=oracle.EXACT):
    return oracle.accept_chain(mode, tl, None, oracle.Q_DRAFT_ONEHOT, drafts, seed=seed,
                               round_=rnd)


def test_first_token_follows_the_target_with_fixed_drafts():
    gamma, B = 3, 300_000
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.full(V, 0.8), size=gamma + 1)
    x = np.array([int(np.argsort(p[i])[V // 2]) for i in range(gamma)], dtype=np.int32)
    drafts = torch.from_numpy(np.tile(x, (B, 1)))
    out = _run(_rows(B, p), drafts)
    p32 = np.exp(_log(p).astype(np.float32).astype(np.float64))
    p32 /= p32.sum(axis=1, keepdims=True)
    first = out["tokens"][:, 0].numpy()
    assert stats.chisquare(np.bincount(first, minlength=V), B * p32[0]).pvalue > 1e-4
    # the second emitted token, given the first draft passed and a second token exists
    sel = (first == x[0]) & (out["num_emitted"].numpy() >= 2)
    second = out["tokens"][:, 1].numpy()[sel]
    assert stats.chisquare(np.bincount(second, minlength=V), sel.sum() * p32[1]).pvalue > 1e-4


def test_closed_form_with_constant_acceptance():
    """p_i(x_i) = alpha at every position: each draft passes with probability alpha."""
    alpha, gamma, B = 0.8, 4, 400_000
    p = np.zeros((gamma + 1, V))
    p[:, 3] = alpha
    p[:, 4:] = (1 - alpha) / (V - 4)
    drafts = torch.full((B, gamma), 3, dtype=torch.int32)
    out = _run(_rows(B, p), drafts, seed=11)
    probs = [alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma]
    vals = np.arange(gamma + 1) + 1
    mean = float(np.dot(probs, vals))
    sd = math.sqrt(float(np.dot(probs, vals ** 2)) - mean ** 2)
    assert abs(mean - 3.3616) < 1e-9
    em = out["num_emitted"].double().mean().item()
    assert abs(em - mean) < 4 * sd / math.sqrt(B)


def test_residual_excludes_the_rejected_draft():
    B = 50_000
    rng = np.random.default_rng(9)
    p = rng.dirichlet(np.full(V, 0.5), size=2)
    x = int(np.argmax(p[0]))  # a likely draft, rejected with probability 1 - p(x)
    out = _run(_rows(B, p), torch.full((B, 1), x, dtype=torch.int32), seed=3)
    rej = out["num_accepted"] == 0
    assert int(rej.sum()) > 1000
    assert not bool((out["tokens"][rej, 0] == x).any())
    # and the residual is p without x, renormalised
    p32 = np.exp(_log(p[0]).astype(np.float32).astype(np.float64))
    r = p32.copy()
    r[x] = 0.0
    r /= r.sum()
    hist = np.bincount(out["tokens"][rej, 0].numpy(), minlength=V)
    keep = r > 0
    assert stats.chisquare(hist[keep], int(rej.sum()) * r[keep]).pvalue > 1e-4


def test_end_marker_equals_the_shorter_chain():
    B = 4000
    rng = np.random.default_rng(13)
    p = rng.dirichlet(np.full(V, 0.7), size=5)
    x1 = torch.from_numpy(rng.integers(0, V, size=(B, 1)).astype(np.int32))
    short = _run(_rows(B, p[:2]), x1, seed=21, rnd=4)
    drafts = torch.full((B, 4), -1, dtype=torch.int32)
    drafts[:, :1] = x1
    long = _run(_rows(B, p), drafts, seed=21, rnd=4)
    assert torch.equal(long["num_emitted"], short["num_emitted"])
    assert torch.equal(long["num_accepted"], short["num_accepted"])
    assert torch.equal(long["tokens"][:, :2], short["tokens"])
    assert bool((long["tokens"][:, 2:] == -1).all())
    assert torch.equal(long["near_ties"], short["near_ties"])
    assert int(long["flags"].sum()) == 0  # -1 is not a bad token
    # greedy as well
    g_long = _run(_rows(B, p), drafts, mode=oracle.GREEDY)
    g_short = _run(_rows(B, p[:2]), x1, mode=oracle.GREEDY)
    assert torch.equal(g_long["tokens"][:, :2], g_short["tokens"])


def test_one_hot_equals_one_hot_probability_rows():
    """The one-hot kind gives what the same drafts give with q passed as e_x rows."""
    gamma, B = 3, 2000
    rng = np.random.default_rng(17)
    p = rng.dirichlet(np.full(V, 0.6), size=gamma + 1)
    drafts = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    q = np.zeros((B, gamma, V), dtype=np.float32)
    for i in range(gamma):
        q[np.arange(B), i, drafts[:, i]] = 1.0
    tl = _rows(B, p)
    a = _run(tl, torch.from_numpy(drafts), seed=2, rnd=1)
    b = oracle.accept_chain(oracle.EXACT, tl, torch.from_numpy(q), oracle.Q_PROBS_F32,
                            torch.from_numpy(drafts), seed=2, round_=1)
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties"):
        assert torch.equal(a[k], b[k]), k

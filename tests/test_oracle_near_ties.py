"""Pins of the oracle's near-tie reports on hand-built cases.

The acceptance rule reports, not hides, every decision whose |u_acc - p/q| is below
1e-6 (hncyxsy.com sections 2.1-2.2 give the rule u < p/q; the 1e-6 window is the
reading of "bit-exact decisions, near ties reported").  Three windows are pinned here, each
with the tested quantity placed 5e-7 inside and 2e-6 outside it, on both sides where the
window has two:
  - the decision window |u_acc - ratio| < 1e-6, counted only when the decision matters
    (its parent lies on an accepted path);
  - the inverse-CDF window: u_smp * sum(w) within 1e-6 of a CDF boundary around the chosen
    token, absolute in probability units (not relative to sum(w));
  - the top-p cut window: the cumulative mass at the cut within 1e-6 of top_p.
Probabilities are given exactly: target logits are float64 logs of a chosen distribution
(softmax returns it to within 1e-16) and q is a float32 probability row with values exact
in float32.  The packed word carries decision ties in its low 16 bits and sample ties in
its high 16 bits.
"""
import math

import numpy as np
import pytest
import torch

import oracle

V = 16
SEED, RND = 4242, 7
SAMPLE_TIE = 65536
DEC_IN, DEC_OUT = 5e-7, 2e-6


def _logits(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -np.inf)


def _spread(p, fixed):
    """Fill the entries of p not in `fixed` with equal shares of the remaining mass."""
    p = np.array(p, dtype=np.float64)
    free = [j for j in range(len(p)) if j not in fixed]
    rest = 1.0 - sum(p[j] for j in fixed)
    for j in free:
        p[j] = rest / len(free)
    return p


def _chain(p_rows, q_rows, drafts, top_k=0, top_p=1.0, seed=SEED, rnd=RND):
    tl = torch.from_numpy(np.stack([_logits(r) for r in p_rows])[None]).contiguous()
    qq = torch.from_numpy(np.stack(q_rows).astype(np.float32)[None]).contiguous()
    toks = torch.tensor([drafts], dtype=torch.int32)
    return oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, temperature=1.0,
                               top_k=top_k, top_p=top_p, seed=seed, round_=rnd)


def _q_row(x, qx):
    """A float32-exact q row with q(x) = qx and the rest spread evenly (rounded to f32)."""
    q = np.full(V, (1.0 - qx) / (V - 1), dtype=np.float32)
    q[x] = np.float32(qx)
    assert float(q[x]) == qx
    return q


# ------------------------------------------------------------ decision window

@pytest.mark.parametrize("delta,near", [(DEC_IN, 1), (-DEC_IN, 1), (DEC_OUT, 0), (-DEC_OUT, 0)])
def test_decision_window(delta, near):
    """ratio = u_acc + delta for the one draft: near iff |delta| < 1e-6; accepted iff delta > 0."""
    x = 3
    u_acc, _ = oracle.uniforms(SEED, RND, 0, 1)
    p0 = _spread(np.zeros(V), [x])
    p0[x] = 0.5 * (u_acc + delta)  # q(x) = 0.5 exactly
    p0 = _spread(p0, [x])
    p1 = _spread(np.zeros(V), [])
    out = _chain([p0, p1], [_q_row(x, 0.5)], [x])
    w = int(out["near_ties"][0])
    assert w & 0xFFFF == near
    assert w >> 16 == 0  # this seed's final sample is far from every boundary
    assert int(out["num_accepted"][0]) == (1 if delta > 0 else 0)


def test_decision_window_counts_only_on_accepted_paths():
    """Chain 0 -> 1 -> 2 as a tree: node 2's decision sits 5e-7 from its ratio.  It counts
    when node 1 is accepted and not when node 1 is rejected (then it cannot matter)."""
    parent = [-1, 0, 1]
    x1, x2 = 4, 5
    u2, _ = oracle.uniforms(SEED, RND, 0, 2)
    q = np.stack([_q_row(x1, 0.5), _q_row(x2, 0.5)])
    p1 = _spread(np.zeros(V), [x2])
    p1[x2] = 0.5 * (u2 + DEC_IN)
    p1 = _spread(p1, [x2])
    p2 = _spread(np.zeros(V), [])
    toks = torch.tensor([[0, x1, x2]], dtype=torch.int32)
    qq = torch.from_numpy(q[None]).contiguous()
    res = {}
    for accept_1 in (True, False):
        p0 = np.zeros(V)
        if accept_1:
            p0[x1] = 0.75  # ratio 1.5: accepted whatever u
        else:
            p0[x1] = 0.0   # ratio 0: rejected
        p0 = _spread(p0, [x1])
        if not accept_1:
            p0[x1] = 0.0
            p0 = p0 / p0.sum()
        tl = torch.from_numpy(np.stack([_logits(p0), _logits(p1), _logits(p2)])[None]).contiguous()
        out = oracle.accept_tree(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, parent, toks,
                                 seed=SEED, round_=RND)
        res[accept_1] = out
    # node 1 accepted: node 2's near decision matters and is counted
    assert int(res[True]["near_ties"][0]) & 0xFFFF == 1
    assert int(res[True]["num_accepted"][0]) == 2  # u2 < ratio (delta > 0)
    # node 1 rejected: the same near decision is off the accepted path and not counted
    assert int(res[False]["near_ties"][0]) & 0xFFFF == 0
    assert int(res[False]["num_accepted"][0]) == 0
    assert int(res[True]["acc"][0, 2]) == 1 and int(res[False]["acc"][0, 2]) == 1


# ------------------------------------------------------- inverse-CDF window

@pytest.mark.parametrize("delta,near,tok", [(DEC_IN, 1, 0), (-DEC_IN, 1, 1), (DEC_OUT, 0, 0),
                                            (-DEC_OUT, 0, 1)])
def test_sample_window_bonus(delta, near, tok):
    """Every draft accepted, the bonus drawn from p_1 with C_0 = u_smp + delta: the
    sample is near iff |delta| < 1e-6, on either side of the boundary."""
    x = 2
    _, u_smp = oracle.uniforms(SEED, RND, 0, 1)  # the bonus uses node gamma = 1
    p0 = _spread(np.zeros(V), [x])
    p0[x] = 0.75
    p0 = _spread(p0, [x])  # ratio 1.5: accepted
    p1 = np.zeros(V)
    p1[0] = u_smp + delta
    p1 = _spread(p1, [0])
    out = _chain([p0, p1], [_q_row(x, 0.5)], [x])
    w = int(out["near_ties"][0])
    assert int(out["num_accepted"][0]) == 1
    assert w & 0xFFFF == 0
    assert w >> 16 == near
    assert int(out["tokens"][0, 1]) == tok


@pytest.mark.parametrize("delta,near,tok", [(DEC_IN, 1, 0), (-DEC_IN, 1, 1), (DEC_OUT, 0, 0)])
def test_sample_window_is_absolute(delta, near, tok):
    """The draft is rejected (p(x) = 0) and the residual [p - q]+ = (p_0, p_1, 0, ...)
    has mass 0.2, with p_0 = u_smp * 0.2 + delta.  At delta = 5e-7 the sample is near
    in absolute units (5e-7 < 1e-6) though not relative to the mass (5e-7 > 2e-7)."""
    x = 3
    mass = 0.2
    _, u_smp = oracle.uniforms(SEED, RND, 0, 0)  # the first rejection samples with node 0
    p0 = np.zeros(V)
    p0[0] = u_smp * mass + delta
    p0[1] = mass - p0[0]
    p0[2] = 1.0 - mass
    q = np.zeros(V, dtype=np.float32)
    q[2] = np.float32(0.875)  # >= p0[2]: no residual there
    q[3:] = np.float32(0.125 / (V - 3))
    p1 = _spread(np.zeros(V), [])
    out = _chain([p0, p1], [q], [x])
    w = int(out["near_ties"][0])
    assert int(out["num_accepted"][0]) == 0
    assert w & 0xFFFF == 0  # ratio 0 and u_acc far above 1e-6 for this seed
    assert w >> 16 == near
    assert int(out["tokens"][0, 0]) == tok


# ------------------------------------------------------------ top-p window

@pytest.mark.parametrize("delta,near", [(DEC_IN, 1), (-DEC_IN, 1), (DEC_OUT, 0), (-DEC_OUT, 0)])
def test_top_p_cut_window(delta, near):
    """top_k = 4, top_p = 0.75: the ranked masses 0.5, 0.25 + delta, 0.15, 0.1 - delta put
    the cumulative mass at rank 1 at top_p + delta.  The cut is a near tie (a decision
    class tie: it changes the kept set) iff |delta| < 1e-6."""
    x = 0  # the draft: ratio = p(0) / q(0), far from u
    p0 = np.zeros(V)
    p0[0], p0[1], p0[2], p0[3] = 0.5, 0.25 + delta, 0.15, 0.1 - delta
    # the bonus row's own cut (ranked 0.4, 0.3, 0.2, 0.1) is far from top_p
    p1 = np.zeros(V)
    p1[0], p1[1], p1[2], p1[3] = 0.4, 0.3, 0.2, 0.1
    out = _chain([p0, p1], [_q_row(x, 0.5)], [x], top_k=4, top_p=0.75)
    w = int(out["near_ties"][0])
    assert w & 0xFFFF == near
    # the kept set: ranks 0..1 when delta >= 0, ranks 0..2 when delta < 0; p(0) after the
    # renormalisation is 0.5 / (0.75 + delta) or 0.5 / (0.9): > q(0) = 0.5, accepted
    assert int(out["num_accepted"][0]) == 1


def test_top_p_cut_keeps_the_crossing_entry():
    """The kept set is the smallest ranked prefix whose mass reaches top_p: with masses
    0.5, 0.25 + 2e-6 the bonus can only be token 0 or 1, never 2 or 3."""
    p0 = _spread(np.zeros(V), [0])
    p0[0] = 0.75
    p0 = _spread(p0, [0])
    toks = []
    for seed in range(40):
        p1 = np.zeros(V)
        p1[0], p1[1], p1[2], p1[3] = 0.5, 0.25 + DEC_OUT, 0.15, 0.1 - DEC_OUT
        out = _chain([p0, p1], [_q_row(0, 0.5)], [0], top_k=4, top_p=0.75, seed=seed)
        if int(out["num_accepted"][0]) == 1:
            toks.append(int(out["tokens"][0, 1]))
    assert toks and set(toks) <= {0, 1} and len(set(toks)) == 2

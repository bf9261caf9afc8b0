"""Pins of the oracle's typical acceptance (CPU only).

The rule (Medusa paper, Cai et al. 2024, section "Typical Acceptance"; named without a rule
by the jennyma11 blog, section "Medusa"): a candidate x is accepted iff
p(x) > min(epsilon, delta * exp(-H(p))), p the parent's target distribution, H its entropy
in nats.  Pinned by closed forms: the entropy of uniform and two-point distributions, the
threshold on either side of p(x), the two limits (epsilon = 0 accepts every token with mass,
a threshold of 1 accepts none), the 1e-6 near-tie window on either side, and ties counted
only on accepted paths.
"""
import math

import numpy as np
import pytest
import torch

import oracle

V = 16


def _logits(p_rows):
    p = np.asarray(p_rows, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return torch.from_numpy(np.where(p > 0, np.log(p), -np.inf))


def _uniform(k):
    p = np.zeros(V)
    p[:k] = 1.0 / k
    return p


def test_entropy_closed_forms():
    two = np.zeros(V)
    two[3], two[9] = 0.3, 0.7
    rows = [_uniform(1), _uniform(4), _uniform(16), two]
    tl = _logits(rows).unsqueeze(0)  # one sequence, a 4-node chain
    out = oracle.accept_typical(tl, [-1, 0, 1, 2], torch.zeros((1, 4), dtype=torch.int32))
    H = out["entropy"][0]
    assert abs(float(H[0]) - 0.0) < 1e-12
    assert abs(float(H[1]) - math.log(4)) < 1e-12
    assert abs(float(H[2]) - math.log(16)) < 1e-12
    assert abs(float(H[3]) - (-0.3 * math.log(0.3) - 0.7 * math.log(0.7))) < 1e-12


def test_temperature_enters_the_distribution():
    """Two tokens with logits 0 and ln 3: p = (1/4, 3/4) at T = 1 and (1/(1+3^(1/2)), ...)
    at T = 2."""
    z = torch.full((1, 2, V), -math.inf, dtype=torch.float64)
    z[0, :, 0], z[0, :, 1] = 0.0, math.log(3.0)
    for T in (1.0, 2.0):
        out = oracle.accept_typical(z, [-1, 0], torch.zeros((1, 2), dtype=torch.int32), temperature=T)
        a = 1.0 / (1.0 + 3.0 ** (1.0 / T))
        assert abs(float(out["entropy"][0, 0]) - (-a * math.log(a) - (1 - a) * math.log(1 - a))) < 1e-12


@pytest.mark.parametrize("eps,delta,accepted", [
    (0.3, 0.9, 1),    # threshold min(0.3, 0.9/4 = 0.225): p(x) = 0.25 passes
    (0.3, 1.1, 0),    # threshold min(0.3, 1.1/4 = 0.275): fails
    (0.2, 1.1, 1),    # threshold min(0.2, 0.275) = 0.2: passes
    (0.24, 5.0, 1),   # epsilon decides
    (0.26, 5.0, 0),
])
def test_threshold_on_either_side(eps, delta, accepted):
    """The root row is uniform over 4 tokens (H = ln 4, exp(-H) = 1/4): the draft token 2
    has p = 1/4 against the threshold min(epsilon, delta / 4)."""
    tl = _logits([_uniform(4), _uniform(2)]).unsqueeze(0)
    out = oracle.accept_typical(tl, [-1, 0], torch.tensor([[0, 2]], dtype=torch.int32),
                                epsilon=eps, delta=delta)
    assert int(out["num_accepted"][0]) == accepted
    # the emitted token after the kept node is its row's argmax (lowest id on ties)
    assert int(out["tokens"][0, accepted]) == 0
    assert int(out["near_ties"][0]) == 0


def test_limits():
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.full(V, 0.5), size=5)
    tl = _logits(p).unsqueeze(0)
    toks = torch.tensor([[0, 3, 5, 7, 1]], dtype=torch.int32)
    chain = [-1, 0, 1, 2, 3]
    # epsilon = 0: every token with mass passes -> the whole chain
    out = oracle.accept_typical(tl, chain, toks, epsilon=0.0, delta=1.0)
    assert int(out["num_accepted"][0]) == 4
    assert int(out["tokens"][0, 4]) == int(np.argmax(p[4]))
    # threshold 1 (epsilon 1, delta huge): nothing passes -> the root row's argmax
    out = oracle.accept_typical(tl, chain, toks, epsilon=1.0, delta=1e9)
    assert int(out["num_accepted"][0]) == 0
    assert int(out["tokens"][0, 0]) == int(np.argmax(p[0]))


@pytest.mark.parametrize("off,near", [(5e-7, 1), (-5e-7, 1), (2e-6, 0), (-2e-6, 0)])
def test_near_tie_window(off, near):
    """p(x) = 1/4 against delta / 4 with delta = 1 + 4 off (as float32): the decision is a
    near tie iff |p(x) - threshold| < 1e-6."""
    delta = float(np.float32(1.0 + 4.0 * off))
    thr = delta / 4.0
    tl = _logits([_uniform(4), _uniform(2)]).unsqueeze(0)
    out = oracle.accept_typical(tl, [-1, 0], torch.tensor([[0, 2]], dtype=torch.int32),
                                epsilon=0.9, delta=delta)
    assert int(out["near_ties"][0]) == near
    assert int(out["num_accepted"][0]) == (1 if 0.25 > thr else 0)


def test_near_tie_counts_only_on_accepted_paths():
    """Chain 0 -> 1 -> 2: node 2 sits 5e-7 below its threshold; it counts when node 1 is
    accepted, not when node 1 is rejected."""
    delta = float(np.float32(1.0 - 2e-6))  # threshold just under 1/4 for a uniform-4 row
    root = np.zeros(V)
    root[5], root[6] = 0.9, 0.1  # H = 0.325: threshold 0.722, far from 0.9 and from 0.1
    for node1_ok in (True, False):
        rows = [root, _uniform(4), _uniform(2)]
        toks = torch.tensor([[0, 5 if node1_ok else 6, 2]], dtype=torch.int32)
        out = oracle.accept_typical(_logits(rows).unsqueeze(0), [-1, 0, 1], toks, epsilon=0.9,
                                    delta=delta)
        assert int(out["near_ties"][0]) == (1 if node1_ok else 0)
        assert int(out["num_accepted"][0]) == (2 if node1_ok else 0)


def test_per_sequence_trees_and_tree_paths():
    """A tree: the deepest fully accepted node wins (ties: smallest row); per-sequence trees
    give each sequence's own result."""
    rng = np.random.default_rng(5)
    trees = [[-1, 0, 0, 1, 2], [-1, 0, 1, 1, 0]]
    B = 2
    p = rng.dirichlet(np.full(V, 0.3), size=(B, 5))
    tl = _logits(p)
    toks = torch.from_numpy(np.argmax(p, axis=-1).astype(np.int32))  # likely tokens
    # every node's token: the parent's argmax
    for b, t in enumerate(trees):
        for c in range(1, 5):
            toks[b, c] = int(np.argmax(p[b, t[c]]))
    per = oracle.accept_typical(tl, trees, toks, epsilon=0.0, delta=0.0)
    for b, t in enumerate(trees):
        one = oracle.accept_typical(tl[b:b + 1], t, toks[b:b + 1], epsilon=0.0, delta=0.0)
        Wb = one["path_nodes"].shape[1]
        assert torch.equal(per["path_nodes"][b, :Wb], one["path_nodes"][0])
        assert int(per["num_accepted"][b]) == 2  # depth 2 is reachable in both trees
    assert int(per["path_nodes"][0, 2]) == 3   # tree 0: nodes 3 and 4 at depth 2 -> row 3

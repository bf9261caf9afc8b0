"""The draft-length controller (host only): its closed form against the page's printed
example, its acceptance estimate against the rate that generated the histogram, its choice
against a hand-computed speedup table, and its smoothing and fallback rules."""
import numpy as np
import pytest

from conftest import read_golden
from speculative_decoding_verify_sv_gb300.gamma import GammaController, expected_emitted, speedup


def test_expected_emitted_matches_printed_example():
    alpha, gamma, emitted, accepted = (float(x) for x in read_golden("expected_tokens_closed_form.txt")[0])
    assert abs(expected_emitted(alpha, int(gamma)) - emitted) < 0.005
    assert abs(expected_emitted(alpha, int(gamma)) - 1.0 - accepted) < 0.005
    assert expected_emitted(0.5, 0) == 1.0 and expected_emitted(1.0, 3) == 4.0


def _rounds(alpha, gamma, B, rng):
    """Accepted counts of B sequences under a constant per-position acceptance rate."""
    acc = np.zeros(B, dtype=np.int64)
    alive = np.ones(B, dtype=bool)
    for _ in range(gamma):
        ok = alive & (rng.random(B) < alpha)
        acc += ok
        alive = ok
    return acc


@pytest.mark.parametrize("alpha,gamma", [(0.7, 5), (0.3, 3), (0.95, 8)])
def test_alpha_estimate_recovers_the_generating_rate(alpha, gamma):
    rng = np.random.default_rng(7)
    ctl = GammaController(gamma=gamma, gamma_max=8, decay=1.0)
    for _ in range(20):
        ctl.observe(_rounds(alpha, gamma, 2000, rng), gamma)
    assert abs(ctl.alpha - alpha) < 0.01


def test_best_gamma_against_a_hand_computed_table():
    # alpha = 0.8, draft cost 0.1 of a target step: speedups (1 - 0.8^(g+1)) / (0.2 (1 + 0.1 g))
    # g: 1 1.636, 2 2.033, 3 2.271, 4 2.401, 5 2.459, 6 2.470, 7 2.448, 8 2.405 -> 6
    ctl = GammaController(gamma=4, gamma_max=8, draft_cost=0.1, decay=1.0)
    ctl._acc, ctl._rej = 800.0, 200.0
    assert abs(ctl.alpha - 0.8) < 1e-12
    assert ctl.best() == 6
    assert abs(speedup(0.8, 6, 0.1) - 2.470) < 1e-3
    # free drafts and near-certain acceptance: the longest allowed
    ctl = GammaController(gamma=1, gamma_max=8, draft_cost=0.0, decay=1.0)
    ctl._acc, ctl._rej = 990.0, 10.0
    assert ctl.best() == 8
    # low acceptance and costly drafts: plain decoding (speedup 1.2 / 1.3 < 1 at g = 1)
    ctl = GammaController(gamma=1, gamma_max=8, draft_cost=0.3, decay=1.0)
    ctl._acc, ctl._rej = 200.0, 800.0
    assert ctl.best() == 0
    ctl = GammaController(gamma=1, gamma_max=8, draft_cost=0.3, decay=1.0, allow_fallback=False)
    ctl._acc, ctl._rej = 200.0, 800.0
    assert ctl.best() == 1


def test_one_step_per_update_towards_the_best():
    rng = np.random.default_rng(3)
    ctl = GammaController(gamma=1, gamma_max=8, draft_cost=0.1, decay=1.0)
    seen = [ctl.gamma]
    for _ in range(12):
        g = ctl.gamma
        seen.append(ctl.update(_rounds(0.8, g, 4000, rng), g))
    steps = np.diff(seen)
    assert set(np.unique(steps)).issubset({-1, 0, 1})
    assert seen[-1] in (5, 6, 7)  # the flat top of the table above
    # within the margin nothing moves
    ctl = GammaController(gamma=5, gamma_max=8, draft_cost=0.1, decay=1.0, margin=0.05)
    ctl._acc, ctl._rej = 800.0, 200.0
    assert ctl.update([], 0) == 5   # 2.470 at 6 is under 5 % above 2.459 at 5


def test_fallback_to_plain_decoding_and_probe():
    ctl = GammaController(gamma=2, gamma_max=8, draft_cost=0.3, decay=1.0, probe_every=4)
    rng = np.random.default_rng(5)
    for _ in range(10):
        g = ctl.gamma
        if g == 0:
            break
        ctl.update(_rounds(0.1, g, 1000, rng), g)
    assert ctl.gamma == 0
    for _ in range(3):
        assert ctl.update([], 0) == 0
    assert ctl.update([], 0) == 1   # the probe after probe_every rounds at 0
    with pytest.raises(ValueError):
        ctl.observe([3], 2)

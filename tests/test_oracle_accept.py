"""Pins of the oracle's token acceptance (CPU only).

The oracle is checked against what the pages and the mathematics fix: the published
Philox known-answer vectors and cuRAND's host Philox generator (library), the
expected-tokens closed form with its printed worked value, distribution preservation
(chi-square on the first emitted token and on the first two), degenerate cases,
greedy independence of the uniforms, closed-form ratios under temperature and top-k,
and the chain procedure against the tree formulation.
"""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from conftest import read_golden
from speculative_decoding_verify_sv_gb300 import workloads as wl

NEG_INF = float("-inf")


# ------------------------------------------------------------------- Philox

def test_philox_known_answers():
    """(P9) Published Philox4x32-10 known-answer vectors."""
    for r in read_golden("philox4x32_10_kat.txt"):
        v = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(v[0:4], v[4:6])
        assert [int(x) for x in out] == v[6:10]


def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if path and (os.path.exists(path) or not path.startswith("/")):
            try:
                return ctypes.CDLL(path)
            except OSError:
                pass
    return None


def test_philox_matches_curand_host_generator():
    """(P9) cuRAND's host Philox4x32-10 (a library run on the CPU): with offset 0 its
    i-th block of four words is philox(counter=(0, 0, i, 0), key=(seed_lo, seed_hi))
    (cuRAND keeps the element offset in counter words 2-3).  Our words must match."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:
        pytest.skip("cuRAND host generator unavailable")
    try:
        for seed in (0, 1234, 0x123456789ABCDEF):
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0
            n = 64
            buf = (ctypes.c_uint32 * n)()
            assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
            words = list(buf)
            key = [seed & 0xFFFFFFFF, seed >> 32]
            for i in range(n // 4):
                assert [int(x) for x in oracle.philox4x32_10([0, 0, i, 0], key)] == words[4 * i:4 * i + 4]
    finally:
        lib.curandDestroyGenerator(gen)


def test_uniform_mapping():
    """u = ((word >> 8) + 0.5) / 2^24 from words 0 and 1 of counter (c, b, round, domain)."""
    seed, rnd, b, c = 0xDEADBEEF12345678, 0x100000007, 3, 5
    w = oracle.philox4x32_10([c, b, rnd & 0xFFFFFFFF, rnd >> 32], [seed & 0xFFFFFFFF, seed >> 32])
    ua, us = oracle.uniforms(seed, rnd, b, c)
    assert ua == ((int(w[0]) >> 8) + 0.5) / 2 ** 24
    assert us == ((int(w[1]) >> 8) + 0.5) / 2 ** 24
    assert 0.0 < ua < 1.0 and 0.0 < us < 1.0


# ------------------------------------------------------------ constructions

def _log(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), NEG_INF)


def _chain_inputs(B, p_rows, q_rows, seed=0):
    """Fixed per-position target rows p_0..p_gamma (as float32 log-probs) and draft
    rows q_1..q_gamma (float32 probabilities) replicated over B sequences; drafts
    drawn from q by the drafter (numpy, seeded)."""
    p_rows = np.asarray(p_rows, dtype=np.float64)
    q_rows = np.asarray(q_rows, dtype=np.float64)
    gamma, V = q_rows.shape
    tl = torch.from_numpy(_log(p_rows).astype(np.float32)).unsqueeze(0).expand(B, gamma + 1, V).contiguous()
    q = torch.from_numpy(q_rows.astype(np.float32)).unsqueeze(0).expand(B, gamma, V).contiguous()
    rng = np.random.default_rng(seed)
    toks = np.empty((B, gamma), dtype=np.int32)
    for i in range(gamma):
        qi = q_rows[i] / q_rows[i].sum()
        toks[:, i] = rng.choice(V, size=B, p=qi)
    return tl, q, torch.from_numpy(toks)


def _alpha_rows(alpha, gamma, V):
    p = np.zeros((gamma + 1, V))
    p[:, 0], p[:, 1] = alpha, 1 - alpha
    q = np.zeros((gamma, V))
    q[:, 0] = 1.0
    return p, q


# ---------------------------------------------------------- closed form (P6)

def _emitted_moments(alpha, gamma):
    """Mean and variance of emitted tokens when each draft passes w.p. alpha."""
    probs = [alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma]
    vals = np.arange(gamma + 1) + 1
    mean = float(np.dot(probs, vals))
    var = float(np.dot(probs, vals ** 2) - mean ** 2)
    return mean, var


def test_closed_form_formula_matches_printed_value():
    (alpha, gamma, emitted, accepted), = [[float(x) for x in r] for r in read_golden("expected_tokens_closed_form.txt")]
    gamma = int(gamma)
    e = sum(alpha ** k for k in range(gamma + 1))
    assert abs(e - (1 - alpha ** (gamma + 1)) / (1 - alpha)) < 1e-12
    assert round(e, 2) == emitted
    assert round(sum(alpha ** k for k in range(1, gamma + 1)), 2) == accepted
    assert abs(_emitted_moments(alpha, gamma)[0] - e) < 1e-12


@pytest.mark.parametrize("construction", ["onehot", "overlap"])
def test_closed_form_expected_tokens(construction):
    """(P6) Constant acceptance alpha = 0.8, gamma = 4, 10^6 sequences: mean emitted
    3.3616 (printed ~3.36) and mean accepted 2.3616 (~2.36), within 4 sigma."""
    alpha, gamma, V, B = 0.8, 4, 16, 1_000_000
    if construction == "onehot":
        p, q = _alpha_rows(alpha, gamma, V)
    else:  # random p, q with sum(min(p, q)) = alpha: q on tokens 0..7, p = a*q + (1-a)*r
        rng = np.random.default_rng(7)
        q = np.zeros((gamma, V))
        q[:, :8] = rng.dirichlet(np.ones(8), size=gamma)
        r = np.zeros((gamma + 1, V))
        r[:, 8:] = rng.dirichlet(np.ones(8), size=gamma + 1)
        qe = np.vstack([q, q[-1:]])
        p = alpha * qe + (1 - alpha) * r
    tl, qq, toks = _chain_inputs(B, p, q, seed=1)
    out = oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, seed=99, round_=0)
    em = out["num_emitted"].double()
    mean, var = _emitted_moments(alpha, gamma)
    assert abs(mean - 3.3616) < 1e-9
    tol = 4 * math.sqrt(var / B)
    assert abs(em.mean().item() - mean) < tol
    assert abs(out["num_accepted"].double().mean().item() - (mean - 1)) < tol
    # reported near ties: |u - 0.8| < 1e-6 (~2e-6 per decision) and samples within
    # 1e-6 of a CDF boundary (~2e-6 / sum(w) per boundary side): tens per 10^6 rounds
    # (the word packs decision ties below bit 16 and sample ties above it)
    nt = out["near_ties"].to(torch.int64)
    assert int((nt & 0xFFFF).sum()) + int((nt >> 16).sum()) < 300


# ---------------------------------------------------------- chi-square (P5)

def _random_pq(gamma, V, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(V, 0.7), size=gamma + 1)
    q = rng.dirichlet(np.full(V, 0.7), size=gamma)
    return p, q


def test_chi_square_first_token():
    """(P5) The first emitted token is distributed as p_0 (V = 16, gamma = 4, 10^6)."""
    gamma, V, B = 4, 16, 1_000_000
    p, q = _random_pq(gamma, V, 2024)
    tl, qq, toks = _chain_inputs(B, p, q, seed=3)
    out = oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, seed=5, round_=1)
    first = out["tokens"][:, 0].numpy()
    counts = np.bincount(first, minlength=V)
    p0 = np.exp(_log(p[0]).astype(np.float32).astype(np.float64))
    p0 /= p0.sum()
    chi2, pval = stats.chisquare(counts, B * p0)
    assert pval > 1e-4, (chi2, pval)


def test_chi_square_first_two_tokens():
    """(P5) The first two output tokens are jointly p_0(x) p_1(y): within a round the
    second token comes from position 1; after a rejection at position 1 it comes from
    the next round, whose target rows start at p_1 (rows here do not depend on x)."""
    gamma, V, B = 4, 16, 1_000_000
    p, q = _random_pq(gamma, V, 77)
    tl, qq, toks = _chain_inputs(B, p, q, seed=4)
    r1 = oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, seed=8, round_=0)
    second = r1["tokens"][:, 1].clone()
    need = torch.nonzero(r1["num_emitted"] == 1).flatten()
    # next round for those sequences: targets p_1..p_gamma, p_gamma; drafts from q_2.., q_gamma
    p2 = np.vstack([p[1:], p[-1:]])
    q2 = np.vstack([q[1:], q[-1:]])
    tl2, qq2, toks2 = _chain_inputs(need.numel(), p2, q2, seed=6)
    r2 = oracle.accept_chain(oracle.EXACT, tl2, qq2, oracle.Q_PROBS_F32, toks2, seed=8, round_=1)
    second[need] = r2["tokens"][:, 0]
    x = r1["tokens"][:, 0].numpy().astype(np.int64)
    y = second.numpy().astype(np.int64)
    counts = np.bincount(x * V + y, minlength=V * V)
    pf = np.exp(_log(p).astype(np.float32).astype(np.float64))
    pf /= pf.sum(1, keepdims=True)
    expected = B * np.outer(pf[0], pf[1]).ravel()
    keep = expected > 0
    chi2, pval = stats.chisquare(counts[keep], expected[keep] * counts.sum() / expected[keep].sum())
    assert pval > 1e-4, (chi2, pval)


# -------------------------------------------------------- degenerate (P7, P8)

def test_p_equals_q_accepts_everything():
    """(P7) p = q (draft row i holds the same logits as target row i-1): every draft
    passes and the bonus is taken (gamma + 1 tokens), distributed as p_gamma."""
    gamma, V, B = 4, 16, 20000
    p, _ = _random_pq(gamma, V, 1)
    tl, _, toks = _chain_inputs(B, p, p[:gamma], seed=2)
    qlog = tl[:, :gamma].contiguous()
    out = oracle.accept_chain(oracle.EXACT, tl, qlog, oracle.Q_LOGITS, toks, seed=1, round_=0)
    assert torch.all(out["num_emitted"] == gamma + 1)
    assert torch.equal(out["tokens"][:, :gamma], toks)
    counts = np.bincount(out["tokens"][:, gamma].numpy(), minlength=V)
    pg = np.exp(_log(p[gamma]).astype(np.float32).astype(np.float64))
    assert stats.chisquare(counts, B * pg / pg.sum()).pvalue > 1e-4


def test_disjoint_supports_always_resample_from_p():
    """(P7) Disjoint supports: the first draft is rejected and the residual is p_0."""
    gamma, V, B = 4, 16, 50000
    rng = np.random.default_rng(11)
    q = np.zeros((gamma, V))
    q[:, :8] = rng.dirichlet(np.ones(8), size=gamma)
    p = np.zeros((gamma + 1, V))
    p[:, 8:] = rng.dirichlet(np.ones(8), size=gamma + 1)
    tl, qq, toks = _chain_inputs(B, p, q, seed=5)
    out = oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, seed=2, round_=3)
    assert torch.all(out["num_emitted"] == 1)
    first = out["tokens"][:, 0].numpy()
    assert np.all(first >= 8)
    p0 = np.exp(_log(p[0]).astype(np.float32).astype(np.float64))
    p0 /= p0.sum()
    assert stats.chisquare(np.bincount(first, minlength=V)[8:], B * p0[8:]).pvalue > 1e-4


def test_rejection_only_at_last_position():
    """(P7) p_i = q_{i+1} except the last position, whose supports are disjoint."""
    gamma, V, B = 4, 16, 20000
    rng = np.random.default_rng(12)
    q = np.zeros((gamma, V))
    q[:, :8] = rng.dirichlet(np.ones(8), size=gamma)
    p = np.zeros((gamma + 1, V))
    p[:gamma - 1] = q[:gamma - 1]
    p[gamma - 1, 8:] = rng.dirichlet(np.ones(8))
    p[gamma] = rng.dirichlet(np.ones(V))
    tl, qq, toks = _chain_inputs(B, p, q, seed=6)
    qlog = tl[:, :gamma].clone()
    qlog[:, gamma - 1] = torch.from_numpy(_log(q[gamma - 1]).astype(np.float32))
    out = oracle.accept_chain(oracle.EXACT, tl, qlog, oracle.Q_LOGITS, toks, seed=4, round_=0)
    assert torch.all(out["num_accepted"] == gamma - 1)
    assert torch.equal(out["tokens"][:, :gamma - 1], toks[:, :gamma - 1])
    assert torch.all(out["tokens"][:, gamma - 1] >= 8)


def test_greedy_is_argmax_chain_and_ignores_uniforms():
    """(P8) Greedy: accept while x_i = argmax of row i-1; emit that row's argmax
    (lowest id on ties); independent of seed and round."""
    B, gamma, V = 64, 5, 40
    g = torch.Generator().manual_seed(0)
    tl = torch.randint(-4, 5, (B, gamma + 1, V), generator=g).float()  # many ties
    am = torch.stack([torch.tensor([int(np.argmax(tl[b, i].numpy())) for i in range(gamma + 1)])
                      for b in range(B)])
    toks = am[:, :gamma].clone().int()
    cut = torch.randint(0, gamma + 1, (B,), generator=g)
    for b in range(B):
        if cut[b] < gamma:
            toks[b, cut[b]] = (am[b, cut[b]] + 1) % V
    o1 = oracle.accept_chain(oracle.GREEDY, tl, None, oracle.Q_LOGITS, toks, seed=1, round_=0)
    o2 = oracle.accept_chain(oracle.GREEDY, tl, None, oracle.Q_LOGITS, toks, seed=2, round_=9)
    for k in o1:
        assert torch.equal(o1[k], o2[k])
    for b in range(B):
        n = int(cut[b])
        assert int(o1["num_accepted"][b]) == n
        assert o1["tokens"][b, :n].tolist() == am[b, :n].tolist()
        assert int(o1["tokens"][b, n]) == int(am[b, n])


def test_all_argmax_drafts_give_bonus_argmax():
    """(P7) Greedy with every draft equal to the argmax: bonus = argmax of last row."""
    B, gamma, V = 8, 4, 100
    tl = torch.randn(B, gamma + 1, V, generator=torch.Generator().manual_seed(1))
    am = tl.argmax(-1).int()
    out = oracle.accept_chain(oracle.GREEDY, tl, None, oracle.Q_LOGITS, am[:, :gamma])
    assert torch.all(out["num_emitted"] == gamma + 1)
    assert torch.equal(out["tokens"], am)



@pytest.mark.parametrize("T", [1.0, 0.5])
def test_exact_with_top_1_is_greedy(T):
    """Exact sampling with top-k = 1 on both sides is greedy decoding: p and q are point
    masses at their argmaxes, so the drafter proposes q's argmax, the ratio p(x)/q(x) is 1 or
    0 (accepted iff x is p's argmax, for every uniform), and the residual [p - q]+ of a
    rejection, like the bonus, is p's argmax.  No decision or sample is a near tie."""
    B, gamma, V = 48, 4, 64
    g = torch.Generator().manual_seed(12)
    tl = torch.randn(B, gamma + 1, V, generator=g) * 3
    dl = torch.randn(B, gamma, V, generator=g) * 3
    # the draft row agrees with the target's argmax for a seeded number of positions
    keep = torch.randint(0, gamma + 1, (B,), generator=g)
    am = tl.argmax(-1)
    for b in range(B):
        for i in range(int(keep[b])):
            dl[b, i, am[b, i]] = dl[b, i].max() + 1.0
    toks = dl.argmax(-1).int()
    ex = oracle.accept_chain(oracle.EXACT, tl, dl, oracle.Q_LOGITS, toks, temperature=T, top_k=1,
                             seed=5, round_=3)
    gr = oracle.accept_chain(oracle.GREEDY, tl, None, oracle.Q_LOGITS, toks)
    for k in ("tokens", "num_emitted", "num_accepted"):
        assert torch.equal(ex[k], gr[k]), k
    assert int(ex["near_ties"].sum()) == 0
    assert sorted(set(ex["num_accepted"].tolist())) == list(range(gamma + 1))

# ------------------------------------------------- ratio and sampling formulas

def test_ratio_orientation_and_residual():
    """p = [.5,.25,.125,.125], q uniform: draft 0 (ratio 2) always passes; draft 2
    (ratio 1/2) passes iff u_acc < 1/2; the residual [p-q]+ is all on token 0."""
    p = np.array([0.5, 0.25, 0.125, 0.125])
    V, B = 4, 400
    tl = torch.from_numpy(np.log(p).astype(np.float32)).expand(B, 2, V).contiguous()
    q = torch.full((B, 1, V), 0.25)
    toks = torch.where(torch.arange(B) % 2 == 0, 0, 2).int().unsqueeze(1)
    out = oracle.accept_tree(oracle.EXACT, tl, q, oracle.Q_PROBS_F32, [-1, 0],
                             torch.cat([torch.zeros(B, 1, dtype=torch.int32), toks], 1),
                             seed=17, round_=2)
    for b in range(B):
        ua, us = oracle.uniforms(17, 2, b, 1)
        x = int(toks[b, 0])
        r = float(np.float32(p[x]) / 0.25) if x == 0 else 0.5
        assert abs(out["ratio"][b, 1].item() - r) < 1e-6
        acc = ua < out["ratio"][b, 1].item()
        assert int(out["num_accepted"][b]) == int(acc)
        if not acc:
            assert int(out["tokens"][b, 0]) == 0  # residual mass only on token 0


def test_temperature_and_top_k_ratio_closed_form():
    """Ratio p(x)/q(x) with y = z/T and top-k (ties keep the lower id), vs hand math."""
    V, T, k = 6, 0.7, 3
    zt = np.array([2.0, 1.0, 3.0, 1.0, -1.0, 0.5], dtype=np.float32)   # top-3: 2, 0, then 1 (tie 1/3 -> 1)
    zq = np.array([0.0, 2.0, 1.0, 1.0, 0.5, 1.0], dtype=np.float32)    # top-3: 1, then 2, 3 (tie 2/3/5 -> 2, 3)
    tl = torch.from_numpy(np.stack([zt, zt])).unsqueeze(0)
    ql = torch.from_numpy(zq).view(1, 1, V)
    def eff(z, keep):
        e = np.zeros(V)
        e[keep] = np.exp(z[keep].astype(np.float64) / T)
        return e / e.sum()
    pt, pq = eff(zt, [0, 1, 2]), eff(zq, [1, 2, 3])
    for x in range(V):
        out = oracle.accept_tree(oracle.EXACT, tl, ql, oracle.Q_LOGITS, [-1, 0],
                                 torch.tensor([[0, x]], dtype=torch.int32), temperature=T,
                                 top_k=k, seed=3)
        r = out["ratio"][0, 1].item()
        if pq[x] > 0:
            assert abs(r - pt[x] / pq[x]) < 1e-12 * max(1.0, pt[x] / pq[x])
            assert int(out["flags"][0]) == 0
        else:
            assert r == (math.inf if pt[x] > 0 else 0.0)
            assert int(out["flags"][0]) & 1


def test_top_p_nucleus_closed_form():
    """Top-p within top-k, on masses chosen so the nucleus is plain to see: the top-4
    distribution of the target row is (0.5, 0.25, 0.15, 0.10) (two entries outside the
    top 4); at top_p = 0.7 the first two stay (0.5 < 0.7 before the second, 0.75 >= 0.7
    before the third), so p' = (2/3, 1/3).  The q row's top-4 distribution is
    (0.45, 0.3, 0.15, 0.1): 0.45 and 0.3 stay (0.75 >= 0.7 before the third),
    q' = (0.6, 0.4).  The ratio p'(x)/q'(x) follows for every x (T = 1)."""
    V, k, top_p = 6, 4, 0.7
    pt = np.array([0.25, 0.001, 0.5, 0.15, 0.10, 0.002])   # top-4: 2, 0, 3, 4
    pq = np.array([0.3, 0.15, 0.45, 0.001, 0.002, 0.1])    # top-4: 2, 0, 1, 5
    zt, zq = np.log(pt), np.log(pq)
    tl = torch.from_numpy(np.stack([zt, zt])).unsqueeze(0)          # float64 rows
    ql = torch.from_numpy(zq).view(1, 1, V)
    p_eff = {2: 2 / 3, 0: 1 / 3}
    q_eff = {2: 0.6, 0: 0.4}
    for x in range(V):
        out = oracle.accept_tree(oracle.EXACT, tl.float(), ql.float(), oracle.Q_LOGITS,
                                 [-1, 0], torch.tensor([[0, x]], dtype=torch.int32),
                                 temperature=1.0, top_k=k, top_p=top_p, seed=3)
        r = out["ratio"][0, 1].item()
        px, qx = p_eff.get(x, 0.0), q_eff.get(x, 0.0)
        if qx > 0:
            assert abs(r - px / qx) < 1e-6, (x, r, px / qx)   # float32 logits of these masses
        else:
            assert r == (math.inf if px > 0 else 0.0)
    # top_p = 1 keeps the whole top-k set: the same as top-k alone
    toks = torch.tensor([[0, 3]], dtype=torch.int32)
    a1 = oracle.accept_tree(oracle.EXACT, tl.float(), ql.float(), oracle.Q_LOGITS, [-1, 0], toks,
                            top_k=k, top_p=1.0, seed=3)
    a2 = oracle.accept_tree(oracle.EXACT, tl.float(), ql.float(), oracle.Q_LOGITS, [-1, 0], toks,
                            top_k=k, seed=3)
    assert a1["ratio"][0, 1].item() == a2["ratio"][0, 1].item()


def test_chi_square_first_token_top_p():
    """(P5) with top-k 10 and top-p 0.8 on the target rows (q given as probabilities):
    the first emitted token follows the nucleus of p_0's top-10 distribution."""
    gamma, V, B, k, top_p = 4, 16, 400_000, 10, 0.8
    p, q = _random_pq(gamma, V, 31)
    tl, qq, toks = _chain_inputs(B, p, q, seed=13)
    out = oracle.accept_chain(oracle.EXACT, tl, qq, oracle.Q_PROBS_F32, toks, top_k=k,
                              top_p=top_p, seed=6, round_=2)
    first = out["tokens"][:, 0].numpy()
    counts = np.bincount(first, minlength=V)
    p0 = np.exp(_log(p[0]).astype(np.float32).astype(np.float64))
    order = np.argsort(-p0, kind="stable")[:k]
    w = p0[order] / p0[order].sum()
    before = np.cumsum(w) - w
    nucleus = order[before < top_p]
    expected = np.zeros(V)
    expected[nucleus] = p0[nucleus] / p0[nucleus].sum()
    assert counts[expected == 0].sum() == 0          # nothing outside the nucleus
    keep = expected > 0
    chi2, pval = stats.chisquare(counts[keep], B * expected[keep])
    assert pval > 1e-4, (chi2, pval)


def test_bonus_inverse_cdf_matches_searchsorted():
    """The bonus token is the smallest j with cumsum(p)_j > u * sum(p) (numpy search)."""
    V, B = 10, 300
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(V))
    z = np.log(p).astype(np.float32)
    tl = torch.from_numpy(z).view(1, 1, V).expand(B, 1, V).contiguous()
    out = oracle.accept_tree(oracle.EXACT, tl, None, oracle.Q_PROBS_F32, [-1],
                             torch.zeros((B, 1), dtype=torch.int32), seed=44, round_=5)
    pe = np.exp(z.astype(np.float64) - z.max())
    cdf = np.cumsum(pe / pe.sum())
    for b in range(B):
        _, us = oracle.uniforms(44, 5, b, 0)
        assert int(out["tokens"][b, 0]) == int(np.searchsorted(cdf, us * cdf[-1], side="right"))


# ------------------------------------------------------ chain == tree formulation

@pytest.mark.parametrize("mode", [oracle.GREEDY, oracle.EXACT])
@pytest.mark.parametrize("top_k,T", [(0, 1.0), (5, 0.7)])
def test_chain_procedure_equals_tree_formulation(mode, top_k, T):
    """The left-to-right chain procedure and the tree formulation on a chain tree give
    identical tokens, counts and near-tie reports."""
    B, gamma, V = 200, 5, 64
    lg = wl.chain_logits(B, gamma, V, sigma=2.0, draft_sigma=0.7, dtype=torch.bfloat16,
                         temperature=T, top_k=top_k, seed=31)
    ch = oracle.accept_chain(mode, lg["target_logits"], lg["draft_logits"], oracle.Q_LOGITS,
                             lg["draft_tokens"], temperature=T, top_k=top_k, seed=5, round_=7)
    nt = torch.zeros((B, gamma + 1), dtype=torch.int32)
    nt[:, 1:] = lg["draft_tokens"]
    tr = oracle.accept_tree(mode, lg["target_logits"], lg["draft_logits"], oracle.Q_LOGITS,
                            wl.chain_parent(gamma), nt, temperature=T, top_k=top_k, seed=5,
                            round_=7)
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties", "flags"):
        assert torch.equal(ch[k], tr[k]), k
    # every draft came from the drafter's own support: q(x) > 0
    assert int(tr["flags"].sum()) == 0
    pn = tr["path_nodes"]
    for b in range(B):
        n = int(tr["num_accepted"][b])
        assert pn[b, :n + 1].tolist() == list(range(n + 1))


def test_tree_path_is_deepest_accepted():
    """Tree acceptance picks the deepest fully accepted node (smallest row on ties),
    and emits that path's tokens then the final sample."""
    B = 300
    par = wl.TREE_T26
    lg = wl.medusa_logits(B, par, 50, sigma=2.0, seed=8, coverage=True, coverage_sigma=0.5)
    out = oracle.accept_tree(oracle.EXACT, lg["target_logits"], lg["draft_logits"],
                             oracle.Q_LOGITS, par, lg["node_tokens"], seed=3, round_=1)
    dep = wl.depths(par)
    acc = out["acc"]
    hist = np.bincount(out["num_accepted"].numpy(), minlength=5)
    assert hist[1:].sum() > 0  # the coverage variant accepts paths
    for b in range(B):
        ok = [True] + [False] * (len(par) - 1)
        for c in range(1, len(par)):
            ok[c] = ok[par[c]] and bool(acc[b, c])
        best = min((c for c in range(len(par)) if ok[c]), key=lambda c: (-dep[c], c))
        assert int(out["num_accepted"][b]) == dep[best]
        path = []
        a = best
        while a >= 0:
            path.append(a)
            a = par[a]
        path = path[::-1]
        assert out["path_nodes"][b, :len(path)].tolist() == path
        assert out["tokens"][b, :len(path) - 1].tolist() == [int(lg["node_tokens"][b, n]) for n in path[1:]]

"""GPU token acceptance vs the CPU oracle, through the C ABI.

Accepted lengths, paths and emitted token ids must be bit-identical on every sequence
that neither side reports as a decision near tie (|u - p/q| < 1e-6 for a decision that
matters, or a near top-p cut); a sequence with only a sample near tie (the final sample
within 1e-6 of a CDF boundary) is still compared on everything but its last token.
Near ties are counted and bounded.
"""
import math

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _compare(gpu, ref, keys, max_exempt_frac=0.01, max_sample_frac=None):
    """Exact agreement outside the near ties each side reports (see accept_parity)."""
    return compare(gpu, ref, keys, max_exempt_frac=max_exempt_frac,
                   max_sample_frac=max_sample_frac)


def _chain(mode, lg, q_kind=sv.Q_LOGITS, T=1.0, top_k=0, seed=3, rnd=1, q=None, top_p=1.0):
    dev = torch.device("cuda")
    tl = lg["target_logits"].to(dev)
    qq = (lg["draft_logits"] if q is None else q)
    qq = None if mode == sv.GREEDY and q is None else qq.to(dev)
    out = sv.sv_accept_chain(mode, tl, qq, q_kind, lg["draft_tokens"].to(dev), temperature=T,
                             top_k=top_k, seed=seed, round_=rnd, top_p=top_p)
    torch.cuda.synchronize()
    ref = oracle.accept_chain(mode, lg["target_logits"], None if qq is None else qq.cpu(), q_kind,
                              lg["draft_tokens"], temperature=T, top_k=top_k, seed=seed, round_=rnd,
                              top_p=top_p)
    return out, ref


@pytest.mark.parametrize("mode", [sv.GREEDY, sv.EXACT])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,top_k", [(1.0, 0), (0.7, 50)])
def test_chain(cuda_ok, mode, dtype, T, top_k):
    lg = wl.chain_logits(96, 5, 4000, sigma=3.0, draft_sigma=1.0, dtype=dtype, temperature=T,
                         top_k=top_k, seed=11)
    out, ref = _chain(mode, lg, T=T, top_k=top_k)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])
    assert sv.sv_read_device_status() == 0


def test_chain_q_as_probabilities(cuda_ok):
    lg = wl.chain_logits(64, 4, 1000, sigma=2.0, draft_sigma=0.5, dtype=torch.float32, seed=12)
    qp = wl.draft_probs(lg["draft_logits"])
    out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_PROBS_F32, q=qp)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])


def test_chain_large_vocab(cuda_ok):
    lg = wl.chain_logits(16, 4, 152064, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=13)
    out, ref = _chain(sv.EXACT, lg, seed=9, rnd=4)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])
    out, ref = _chain(sv.GREEDY, lg)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])


@pytest.mark.parametrize("parent", [wl.TREE_T26, wl.TREE_T64, wl.TREE_EXAMPLE7])
@pytest.mark.parametrize("mode", [sv.GREEDY, sv.EXACT])
def test_tree(cuda_ok, parent, mode):
    B = 64
    lg = wl.medusa_logits(B, parent, 2000, sigma=3.0, seed=14, coverage=True, coverage_sigma=0.7)
    dev = torch.device("cuda")
    q = lg["draft_logits"].to(dev) if mode == sv.EXACT else None
    out = sv.sv_accept_tree(mode, lg["target_logits"].to(dev), q, sv.Q_LOGITS, parent,
                            lg["node_tokens"].to(dev), seed=21, round_=2)
    torch.cuda.synchronize()
    ref = oracle.accept_tree(mode, lg["target_logits"], lg["draft_logits"] if q is not None else None,
                             oracle.Q_LOGITS, parent, lg["node_tokens"], seed=21, round_=2)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted", "path_nodes"])
    assert int(ref["num_accepted"].sum()) > 0  # paths do get accepted in this variant


@pytest.mark.parametrize("V,B", [(128256, 24), (270336, 4)])
def test_chain_large_vocab_top_k(cuda_ok, V, B):
    """Top-k 50 at T = 0.7 on long rows: the statistics remember each batch's maximum for
    rows up to 262,144 entries and re-read only the batches that can hold a kept entry
    (the second size has batches past that limit, which are always re-read); the final
    sample skips vectors below the k-th value."""
    lg = wl.chain_logits(B, 4, V, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16,
                         temperature=0.7, top_k=50, seed=16)
    for mode in (sv.EXACT, sv.GREEDY):
        out, ref = _chain(mode, lg, T=0.7, top_k=50, seed=5, rnd=2)
        _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])
    assert sv.sv_read_device_status() == 0


@pytest.mark.parametrize("dtype,V,B,q_probs", [
    (torch.bfloat16, 152064, 16, True),   # bf16 rows, f32 q probabilities (two q vectors per p vector)
    (torch.float32, 131072, 8, False),    # fp32 rows, q as logits
    (torch.float32, 131072, 8, True),
])
def test_select_ring_layouts(cuda_ok, dtype, V, B, q_probs):
    """Rows long enough that each select CTA's slice of the vocabulary streams through its
    shared-memory ring, for each stage layout the ring has."""
    lg = wl.chain_logits(B, 4, V, sigma=3.0, draft_sigma=1.0, dtype=dtype, seed=17)
    if q_probs:
        qp = wl.draft_probs(lg["draft_logits"])
        out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_PROBS_F32, q=qp, seed=8, rnd=5)
    else:
        out, ref = _chain(sv.EXACT, lg, seed=8, rnd=5)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.15)
    assert sv.sv_read_device_status() == 0


@pytest.mark.parametrize("V,B", [(4000, 96), (128256, 24)])
def test_chain_top_p(cuda_ok, V, B):
    """Top-k 50 then top-p 0.9 at T = 0.7 on p and q (the drafter samples within its own
    nucleus): tokens and counts equal the oracle's."""
    lg = wl.chain_logits(B, 5, V, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16,
                         temperature=0.7, top_k=50, top_p=0.9, seed=18)
    out, ref = _chain(sv.EXACT, lg, T=0.7, top_k=50, seed=6, rnd=3, top_p=0.9)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"])
    assert sv.sv_read_device_status() == 0


def test_tree_top_p(cuda_ok):
    B = 64
    par = wl.TREE_T26
    lg = wl.medusa_logits(B, par, 2000, sigma=3.0, seed=19, coverage=True, coverage_sigma=0.7)
    dev = torch.device("cuda")
    out = sv.sv_accept_tree(sv.EXACT, lg["target_logits"].to(dev), lg["draft_logits"].to(dev),
                            sv.Q_LOGITS, par, lg["node_tokens"].to(dev), top_k=20, top_p=0.8,
                            seed=23, round_=1)
    torch.cuda.synchronize()
    ref = oracle.accept_tree(oracle.EXACT, lg["target_logits"], lg["draft_logits"], oracle.Q_LOGITS,
                             par, lg["node_tokens"], top_k=20, top_p=0.8, seed=23, round_=1)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted", "path_nodes"], max_exempt_frac=0.05)
    # node tokens are the heads' ranked tokens: a nucleus narrower than the tree's caps
    # leaves some with q(x) = 0, which is reported (and read, which clears the word)
    assert sv.sv_read_device_status() & ~sv.SV_DEV_ZERO_DRAFT_PROB == 0


def test_top_p_after_tie_fallback(cuda_ok):
    """Every logit equal: the top-7 set is the 7 lowest ids (the counting path), and its
    nucleus at top_p = 0.5 is the 4 lowest (3/7 < 0.5 <= 4/7)."""
    B, gamma, V, k = 4, 3, 8192, 7
    tl = torch.zeros((B, gamma + 1, V), dtype=torch.bfloat16)
    ql = torch.zeros((B, gamma, V), dtype=torch.bfloat16)
    toks = torch.tensor([[0, 3, 2], [1, 2, 0], [3, 1, 1], [2, 0, 3]], dtype=torch.int32)
    lg = dict(target_logits=tl, draft_logits=ql, draft_tokens=toks)
    sv.sv_read_device_status()  # start from a clear status word
    out, ref = _chain(sv.EXACT, lg, T=1.0, top_k=k, seed=2, top_p=0.5)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=1.0)
    t = out["tokens"].cpu()
    assert torch.all(t[t >= 0] < 4)
    assert sv.sv_read_device_status() == 0


def test_top_k_tie_fallback(cuda_ok):
    """Every logit equal: more than 3072 entries tie at the threshold, so the kernel
    takes its counting path; the kept set is the k lowest ids."""
    B, gamma, V, k = 4, 3, 8192, 7
    tl = torch.zeros((B, gamma + 1, V), dtype=torch.bfloat16)
    ql = torch.zeros((B, gamma, V), dtype=torch.bfloat16)
    toks = torch.tensor([[0, 3, 6], [1, 7, 2], [6, 6, 9], [5, 4, 3]], dtype=torch.int32)
    lg = dict(target_logits=tl, draft_logits=ql, draft_tokens=toks)
    out, ref = _chain(sv.EXACT, lg, T=1.0, top_k=k, seed=2)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=1.0)
    assert torch.all(out["tokens"].cpu()[out["tokens"].cpu() >= 0] < 10)
    st = sv.sv_read_device_status()
    assert st & sv.SV_DEV_ZERO_DRAFT_PROB  # token 9 lies outside q's top-7


def test_bad_token_sets_status(cuda_ok):
    lg = wl.chain_logits(2, 2, 64, seed=15)
    lg["draft_tokens"][0, 0] = 64
    lg["draft_tokens"][1, 1] = -5
    out, ref = _chain(sv.EXACT, lg)
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_TOKEN
    assert int(out["num_accepted"][0]) == 0 and int(out["num_accepted"][1]) <= 1
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=1.0)


def _log(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -np.inf)


def test_chi_square_first_token_gpu(cuda_ok):
    """(P5) through the GPU: V = 16, gamma = 4, 10^6 sequences; also bit-equal to the oracle."""
    gamma, V, B = 4, 16, 1_000_000
    rng = np.random.default_rng(2024)
    p = rng.dirichlet(np.full(V, 0.7), size=gamma + 1)
    q = rng.dirichlet(np.full(V, 0.7), size=gamma)
    tl = torch.from_numpy(_log(p).astype(np.float32)).expand(B, gamma + 1, V).contiguous()
    qq = torch.from_numpy(q.astype(np.float32)).expand(B, gamma, V).contiguous()
    toks = np.empty((B, gamma), dtype=np.int32)
    for i in range(gamma):
        toks[:, i] = rng.choice(V, size=B, p=q[i] / q[i].sum())
    lg = dict(target_logits=tl, draft_logits=qq, draft_tokens=torch.from_numpy(toks))
    out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_PROBS_F32, q=qq, seed=5, rnd=1)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=1e-3)
    first = out["tokens"][:, 0].cpu().numpy()
    p0 = np.exp(_log(p[0]).astype(np.float32).astype(np.float64))
    assert stats.chisquare(np.bincount(first, minlength=V), B * p0 / p0.sum()).pvalue > 1e-4


def test_closed_form_gpu(cuda_ok):
    """(P6) through the GPU: alpha = 0.8, gamma = 4 -> mean emitted 3.3616, accepted 2.3616."""
    alpha, gamma, V, B = 0.8, 4, 16, 1_000_000
    p = np.zeros((gamma + 1, V))
    p[:, 0], p[:, 1] = alpha, 1 - alpha
    q = np.zeros((gamma, V))
    q[:, 0] = 1.0
    tl = torch.from_numpy(_log(p).astype(np.float32)).expand(B, gamma + 1, V).contiguous()
    qq = torch.from_numpy(q.astype(np.float32)).expand(B, gamma, V).contiguous()
    toks = torch.zeros((B, gamma), dtype=torch.int32)
    lg = dict(target_logits=tl, draft_logits=qq, draft_tokens=toks)
    out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_PROBS_F32, q=qq, seed=99, rnd=0)
    _compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=1e-3)
    probs = [alpha ** k * (1 - alpha) for k in range(gamma)] + [alpha ** gamma]
    vals = np.arange(gamma + 1) + 1
    mean = float(np.dot(probs, vals))
    sd = math.sqrt(float(np.dot(probs, vals ** 2)) - mean ** 2)
    em = out["num_emitted"].double().mean().item()
    assert abs(em - 3.3616) < 4 * sd / math.sqrt(B)
    assert abs(out["num_accepted"].double().mean().item() - 2.3616) < 4 * sd / math.sqrt(B)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_workloads(cuda_ok, cfg):
    """Each workload at full size: every sequence compared with the oracle, in both modes.
    With 128K-152K tokens many tokens carry less than 1e-6 of probability, and a sample
    that lands on one lies within 1e-6 of a CDF boundary by definition: such sequences
    are reported as near ties (about 1 in 12 at V = 152064)."""
    w = wl.make_workload(cfg, device="cuda")
    c = w["cfg"]
    modes = [sv.EXACT, sv.GREEDY]
    for mode in modes:
        if c["kind"] == "chain":
            out = sv.sv_accept_chain(mode, w["target_logits"], w["draft_logits"], sv.Q_LOGITS,
                                     w["draft_tokens"], temperature=c["temperature"],
                                     top_k=c["top_k"], seed=w["seed"], round_=0)
            torch.cuda.synchronize()
            ref = oracle.accept_chain(mode, w["target_logits"].cpu(), w["draft_logits"].cpu(),
                                      oracle.Q_LOGITS, w["draft_tokens"].cpu(),
                                      temperature=c["temperature"], top_k=c["top_k"],
                                      seed=w["seed"], round_=0)
            keys = ["tokens", "num_emitted", "num_accepted"]
        else:
            out = sv.sv_accept_tree(mode, w["target_logits"], w["draft_logits"], sv.Q_LOGITS,
                                    w["parent"], w["node_tokens"], temperature=c["temperature"],
                                    top_k=c["top_k"], seed=w["seed"], round_=0)
            torch.cuda.synchronize()
            ref = oracle.accept_tree(mode, w["target_logits"].cpu(), w["draft_logits"].cpu(),
                                     oracle.Q_LOGITS, w["parent"], w["node_tokens"].cpu(),
                                     temperature=c["temperature"], top_k=c["top_k"],
                                     seed=w["seed"], round_=0)
            keys = ["tokens", "num_emitted", "num_accepted", "path_nodes"]
        _compare(out, ref, keys, max_sample_frac=0.05 if c["V"] <= 32000 else 0.15)
    assert sv.sv_read_device_status() == 0

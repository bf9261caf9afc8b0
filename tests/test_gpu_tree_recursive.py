"""Exact tree acceptance with siblings tried in turn, on the GPU against the oracle: the
emitted tokens, counts and path must be identical except on sequences that either side
reports as a decision near tie; with only a sample near tie, everything but the last
token (bounded, as for the other acceptance tests)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl
from test_gpu_accept import _compare

pytestmark = pytest.mark.gpu

KEYS = ["tokens", "num_emitted", "num_accepted", "path_nodes"]


def _run(tl, q, q_kind, parent, toks, **kw):
    dev = torch.device("cuda")
    sv.sv_read_device_status()
    out = sv.sv_accept_tree_recursive(tl.to(dev), q.to(dev), q_kind, parent, toks.to(dev), **kw)
    torch.cuda.synchronize()
    ref = oracle.accept_tree_recursive(tl, q, q_kind, parent, toks, **kw)
    return out, ref


@pytest.mark.parametrize("dtype,T,top_k", [(torch.bfloat16, 1.0, 0), (torch.bfloat16, 0.7, 20),
                                           (torch.float32, 0.9, 0)])
def test_chain(cuda_ok, dtype, T, top_k):
    B, gamma, V = 64, 5, 4000
    lg = wl.chain_logits(B, gamma, V, sigma=3.0, draft_sigma=1.0, dtype=dtype, temperature=T,
                         top_k=top_k, seed=31)
    toks = torch.zeros((B, gamma + 1), dtype=torch.int32)
    toks[:, 1:] = lg["draft_tokens"]
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, wl.chain_parent(gamma),
                    toks, temperature=T, top_k=top_k, seed=5, round_=3)
    _compare(out, ref, KEYS)
    assert int(ref["num_accepted"].sum()) > 0
    assert sv.sv_read_device_status() == 0


def test_chain_large_vocab(cuda_ok):
    """152064-entry rows (the ragged-paged workload's vocabulary): the final sample's 149
    chunk sums are split five to a lane of the search."""
    B, gamma, V = 16, 4, 152064
    lg = wl.chain_logits(B, gamma, V, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=13)
    toks = torch.zeros((B, gamma + 1), dtype=torch.int32)
    toks[:, 1:] = lg["draft_tokens"]
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, wl.chain_parent(gamma),
                    toks, seed=9, round_=4)
    _compare(out, ref, KEYS, max_sample_frac=0.15)
    assert sv.sv_read_device_status() == 0


def test_tree_sixteen_cta_cluster(cuda_ok):
    """Eight sequences of a 26-node tree with 131072-entry rows: each sequence runs on a
    cluster of 16 CTAs (slices of 8192 entries), so the residual masses and the final
    sample's slice totals cross 16 CTAs."""
    B, parent, V = 8, wl.TREE_T26, 131072
    lg = wl.medusa_logits(B, parent, V, sigma=3.0, seed=41, coverage=True, coverage_sigma=0.7)
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, parent, lg["node_tokens"],
                    seed=21, round_=2)
    _compare(out, ref, KEYS, max_exempt_frac=0.25, max_sample_frac=0.5)
    assert sv.sv_read_device_status() == 0


@pytest.mark.parametrize("parent", [wl.TREE_T26, wl.TREE_T64, wl.TREE_EXAMPLE7])
def test_medusa_trees(cuda_ok, parent):
    B = 64
    lg = wl.medusa_logits(B, parent, 2000, sigma=3.0, seed=33, coverage=True, coverage_sigma=0.7)
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, parent,
                    lg["node_tokens"], seed=7, round_=1)
    _compare(out, ref, KEYS)
    assert int(ref["num_accepted"].sum()) > 0
    # siblings past the first are reached (rank order): some kept paths leave the first child
    pn = ref["path_nodes"][:, 1]
    assert int(((pn > 1) & (pn != -1)).sum()) > 0


def test_independent_sibling_drafts_q_probs(cuda_ok):
    """One level of m = 3 children drawn independently from q, q passed as probabilities:
    many sequences take the second and third sibling after residual updates."""
    V, B, m = 16, 4096, 3
    rng = np.random.default_rng(21)
    p = rng.dirichlet(np.full(V, 0.7))
    q = rng.dirichlet(np.full(V, 0.7))
    with np.errstate(divide="ignore"):
        lp = np.where(p > 0, np.log(p), -np.inf).astype(np.float32)
    tl = torch.from_numpy(lp).view(1, 1, V).expand(B, m + 1, V).contiguous()
    qq = torch.from_numpy(q.astype(np.float32)).view(1, 1, V).expand(B, 1, V).contiguous()
    toks = np.zeros((B, m + 1), dtype=np.int32)
    toks[:, 1:] = rng.choice(V, size=(B, m), p=q / q.sum())
    out, ref = _run(tl, qq, sv.Q_PROBS_F32, [-1] + [0] * m, torch.from_numpy(toks), seed=3,
                    round_=1)
    _compare(out, ref, KEYS)
    taken = ref["path_nodes"][:, 1]
    assert int((taken == 2).sum()) > 50 and int((taken == 3).sum()) > 50


def test_top_k_top_p_tree(cuda_ok):
    B, parent = 64, wl.TREE_T26
    lg = wl.medusa_logits(B, parent, 2000, sigma=3.0, seed=35, coverage=True, coverage_sigma=0.7)
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, parent,
                    lg["node_tokens"], top_k=20, top_p=0.8, seed=9, round_=2)
    _compare(out, ref, KEYS, max_exempt_frac=0.05)
    # ranked node tokens outside a narrow nucleus have q(x) = 0: reported, nothing else
    assert sv.sv_read_device_status() & ~sv.SV_DEV_ZERO_DRAFT_PROB == 0


def test_medusa_shape_large_vocab(cuda_ok):
    """The 64-node Medusa tree at V = 32000 (bf16), 8 sequences."""
    B, parent = 8, wl.TREE_T64
    lg = wl.medusa_logits(B, parent, 32000, sigma=3.0, seed=37, coverage=True, coverage_sigma=0.7)
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, parent,
                    lg["node_tokens"], seed=11, round_=4)
    _compare(out, ref, KEYS)


def test_bad_token_is_rejected_and_reported(cuda_ok):
    B, parent = 4, [-1, 0, 0, 1]
    lg = wl.medusa_logits(B, parent, 64, sigma=2.0, seed=39)
    toks = lg["node_tokens"].clone()
    toks[:, 1] = 64  # outside [0, V): rejected, so the second child decides
    out, ref = _run(lg["target_logits"], lg["draft_logits"], sv.Q_LOGITS, parent, toks, seed=1)
    _compare(out, ref, KEYS, max_exempt_frac=1.0)
    assert torch.all(out["path_nodes"][:, 1].cpu() != 1)
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_TOKEN


def test_siblings_with_small_residuals(cuda_ok):
    """q close to p (draft logits = target logits + N(0, 0.05)): a rejection leaves a
    residual of small mass (the total variation between p and q, a few percent), and the
    next siblings are decided against it.  The kernel forms each residual entry in float,
    so its near-tie windows widen with (1 + c) / n; outside them every output equals the
    oracle's, taken in double."""
    B, m, V = 2048, 4, 4000
    g = torch.Generator().manual_seed(41)
    z = torch.randn((B, 1, V), generator=g) * 3.0
    zq = z + torch.randn((B, 1, V), generator=g) * 0.05
    tl = torch.cat([z, torch.randn((B, m, V), generator=g) * 3.0], dim=1).to(torch.bfloat16)
    ql = zq.to(torch.bfloat16)
    qprob = torch.softmax(ql.float().double(), dim=-1)[:, 0]
    toks = torch.zeros((B, m + 1), dtype=torch.int32)
    toks[:, 1:] = torch.multinomial(qprob, m, replacement=True, generator=g).to(torch.int32)
    out, ref = _run(tl, ql, sv.Q_LOGITS, [-1] + [0] * m, toks, seed=13, round_=2)
    n_dec, n_smp = _compare(out, ref, KEYS, max_exempt_frac=0.02, max_sample_frac=0.05)
    taken = ref["path_nodes"][:, 1]
    # most first children pass; some sequences reach the later siblings through small
    # residuals
    assert int((taken == 1).sum()) > 0.8 * B
    assert int(((taken > 1) | (taken == -1)).sum()) > 20

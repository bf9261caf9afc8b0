"""Acceptance with more sequences than SMs and rows of 32K-64K entries against the CPU
oracle, through the C ABI.

With at least one sequence per SM the select kernel takes one CTA per sequence (no
cluster split of the final sample's pass), and rows this long stream through its
shared-memory ring.  These cases cover each weight form of the pass (q as logits, q as f32
probabilities, one-hot drafts, the bonus from p alone), both dtypes, greedy mode, shared
and per-sequence trees, the fused KV commit and repeatability.  The outputs must match the
oracle exactly outside the near ties either side reports.
"""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _chain(mode, lg, q_kind=sv.Q_LOGITS, q=None, T=1.0, seed=3, rnd=1):
    dev = torch.device("cuda")
    qq = lg["draft_logits"] if q is None else q
    if mode == sv.GREEDY or q_kind == sv.Q_DRAFT_ONEHOT:
        qq = None
    out = sv.sv_accept_chain(mode, lg["target_logits"].to(dev), None if qq is None else qq.to(dev),
                             q_kind, lg["draft_tokens"].to(dev), temperature=T, seed=seed, round_=rnd)
    torch.cuda.synchronize()
    ref = oracle.accept_chain(mode, lg["target_logits"], qq, q_kind, lg["draft_tokens"],
                              temperature=T, seed=seed, round_=rnd)
    return out, ref


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_large_batch_chain_bf16(cuda_ok, mode, T):
    B = _sms() + 37  # more sequences than SMs, not a multiple of anything
    lg = wl.chain_logits(B, 4, 40000, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16,
                         temperature=T, seed=61)
    launches0 = sv.sv_kernel_launches()
    out, ref = _chain(mode, lg, T=T, seed=7, rnd=2)
    assert sv.sv_kernel_launches() - launches0 == 2  # the statistics and select kernels
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


def test_large_batch_chain_f32_q_probabilities(cuda_ok):
    B = _sms() + 5
    lg = wl.chain_logits(B, 3, 32768, sigma=3.0, draft_sigma=1.0, dtype=torch.float32, seed=62)
    qp = wl.draft_probs(lg["draft_logits"])
    out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_PROBS_F32, q=qp, seed=5, rnd=3)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


def test_large_batch_chain_one_hot_drafts(cuda_ok):
    """Deterministic drafts: accepted iff u < p(x); after a rejection the token comes from p
    without the rejected draft."""
    B = _sms() + 9
    lg = wl.chain_logits(B, 4, 32768, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=63)
    out, ref = _chain(sv.EXACT, lg, q_kind=sv.Q_DRAFT_ONEHOT, seed=9, rnd=1)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


def test_large_batch_ragged_chains(cuda_ok):
    """Chains whose drafts end early (-1): the bonus of a sequence whose drafts all pass is
    drawn from p alone."""
    B = _sms() + 11
    lg = wl.chain_logits(B, 5, 32768, sigma=2.0, draft_sigma=0.3, dtype=torch.bfloat16, seed=64)
    toks = lg["draft_tokens"].clone()
    g = torch.Generator().manual_seed(5)
    cut = torch.randint(0, 6, (B,), generator=g)
    for b in range(B):
        toks[b, int(cut[b]):] = -1
    lg = dict(lg, draft_tokens=toks)
    out, ref = _chain(sv.EXACT, lg, seed=11, rnd=0)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_large_batch_tree(cuda_ok, mode):
    B, parent = _sms() + 3, wl.TREE_T26
    lg = wl.medusa_logits(B, parent, 32768, sigma=3.0, seed=65, coverage=True, coverage_sigma=0.7)
    dev = torch.device("cuda")
    q = lg["draft_logits"].to(dev) if mode == sv.EXACT else None
    out = sv.sv_accept_tree(mode, lg["target_logits"].to(dev), q, sv.Q_LOGITS, parent,
                            lg["node_tokens"].to(dev), seed=13, round_=4)
    torch.cuda.synchronize()
    ref = oracle.accept_tree(mode, lg["target_logits"], lg["draft_logits"] if q is not None else None,
                             oracle.Q_LOGITS, parent, lg["node_tokens"], seed=13, round_=4)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted", "path_nodes"], max_sample_frac=0.1)
    assert int(ref["num_accepted"].sum()) > 0
    assert sv.sv_read_device_status() == 0


def test_large_batch_per_sequence_trees(cuda_ok):
    """A different tree per sequence (a device parent array [B, N])."""
    B, N, V = _sms() + 2, 12, 32768
    trees = []
    for b in range(B):
        g = torch.Generator().manual_seed(200 + b)
        par = [-1]
        for i in range(1, N):
            par.append(int(torch.randint(0, i, (1,), generator=g)) if b % 3 else i - 1)
        trees.append(par)
    depth = max(max(wl.depths(t)) for t in trees)
    g = torch.Generator().manual_seed(66)
    tl = (torch.randn(B, N, V, generator=g) * 3.0).to(torch.bfloat16)
    q = (tl[:, :depth].float() + torch.randn(B, depth, V, generator=g)).to(torch.bfloat16)
    toks = torch.randint(0, V, (B, N), generator=g, dtype=torch.int32)
    # half the candidates are the target's most likely token of their parent's row
    for b in range(B):
        for i in range(1, N):
            if (b + i) % 2:
                toks[b, i] = int(tl[b, trees[b][i]].float().argmax())
    dev = torch.device("cuda")
    par = torch.tensor(trees, dtype=torch.int32, device=dev)
    out = sv.sv_accept_tree(sv.EXACT, tl.to(dev), q.to(dev), sv.Q_LOGITS, par, toks.to(dev), seed=6, round_=1)
    torch.cuda.synchronize()
    ref = oracle.accept_tree(oracle.EXACT, tl, q, oracle.Q_LOGITS, trees, toks, seed=6, round_=1)
    compare(out, ref, ["path_nodes", "tokens", "num_emitted", "num_accepted"], max_sample_frac=0.1)
    assert sv.sv_read_device_status() == 0


def test_large_batch_commit_matches_separate_calls(cuda_ok):
    """sv_accept_chain_commit (the commit fused into the select kernel): the same tokens as
    sv_accept_chain, and the kept path's K/V rows in the paged cache as sv_commit_kv writes
    them."""
    B, gamma, V, Hkv, D = _sms() + 21, 4, 32768, 2, 64
    lg = wl.chain_logits(B, gamma, V, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=67)
    dev = torch.device("cuda")
    att = wl.attention_inputs(B, gamma + 1, 2 * Hkv, Hkv, D, [100 + 7 * b for b in range(B)],
                              paged=True, extra=gamma + 1, seed=68, device=dev)
    def cache():
        return sv.KVCache(att["cache_k"].clone(), att["cache_v"].clone(), att["prefix_len"].clone(),
                          att["block_table"], 16)
    c1, c2 = cache(), cache()
    tl, qd, dt = lg["target_logits"].to(dev), lg["draft_logits"].to(dev), lg["draft_tokens"].to(dev)
    a = sv.sv_accept_chain_commit(sv.EXACT, tl, qd, sv.Q_LOGITS, dt, att["k_tree"], att["v_tree"], c1,
                                  seed=2, round_=3)
    b = sv.sv_accept_chain(sv.EXACT, tl, qd, sv.Q_LOGITS, dt, seed=2, round_=3)
    # a chain's kept path is nodes 0..num_accepted
    W = gamma + 1
    idx = torch.arange(W, dtype=torch.int32, device=dev).expand(B, W)
    pn = torch.where(idx <= b["num_accepted"].unsqueeze(1), idx, torch.full_like(idx, -1)).contiguous()
    sv.sv_commit_kv(att["k_tree"], att["v_tree"], pn, b["num_accepted"], c2)
    torch.cuda.synchronize()
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties"):
        assert torch.equal(a[k].cpu(), b[k].cpu()), k
    assert torch.equal(c1.prefix_len.cpu(), c2.prefix_len.cpu())
    assert torch.equal(c1.k.cpu(), c2.k.cpu()) and torch.equal(c1.v.cpu(), c2.v.cpu())
    assert sv.sv_read_device_status() == 0


def test_large_batch_repeatable(cuda_ok):
    """Three calls on the same inputs give bit-identical outputs (every sum has a fixed
    order, whatever order the CTAs run in)."""
    B = _sms() + 40
    lg = wl.chain_logits(B, 4, 65536, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=69)
    dev = torch.device("cuda")
    args = (lg["target_logits"].to(dev), lg["draft_logits"].to(dev), sv.Q_LOGITS, lg["draft_tokens"].to(dev))
    outs = [sv.sv_accept_chain(sv.EXACT, *args, seed=1, round_=1) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for k in ("tokens", "num_emitted", "num_accepted", "near_ties"):
            assert torch.equal(o[k].cpu(), outs[0][k].cpu()), k

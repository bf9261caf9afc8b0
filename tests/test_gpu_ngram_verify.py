"""Prompt-lookup drafts verified on the device end to end.

sv_ngram_draft proposes up to gamma copied tokens per sequence (-1 after them); the same
device buffers go straight into sv_accept_chain_commit with q_kind SV_Q_DRAFT_ONEHOT (the
drafts are copies, so q is a point mass at each: the jennyma11 blog, section "Prompt
Lookup / N-gram", sends them to the target's verification like any others).  Drafts,
acceptance and the committed cache are compared with the oracle's prompt lookup, chain
acceptance and commit on the same inputs.
"""
import math

import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl
from test_gpu_ngram import _histories

pytestmark = pytest.mark.gpu


def _target_logits(drafts, V, seed, agree=0.7, dtype=torch.bfloat16):
    """Target rows ~N(0, 2); where a draft exists, the target agrees with it with
    probability `agree`: its logit is raised by log(V) + 4, which gives it about 0.9 of the
    row's mass, so that accepted runs of several drafts occur."""
    B, gamma = drafts.shape
    g = torch.Generator().manual_seed(seed)
    tl = torch.randn((B, gamma + 1, V), generator=g) * 2.0
    boost = torch.rand((B, gamma), generator=g) < agree
    lift = math.log(V) + 4.0
    for i in range(gamma):
        d = drafts[:, i]
        sel = (d >= 0) & boost[:, i]
        tl[sel.nonzero().flatten(), i, d[sel].long()] += lift
    return tl.to(dtype)


@pytest.mark.parametrize("B,V,gamma,mode", [(128, 4096, 4, sv.EXACT), (128, 4096, 4, sv.GREEDY),
                                            (64, 152064, 5, sv.EXACT)])
def test_ngram_drafts_through_chain_verification(cuda_ok, B, V, gamma, mode):
    dev = torch.device("cuda")
    hist, lens = _histories(B, 1024, 40, seed=B + gamma)
    rd, rn = oracle.ngram_draft(hist, lens, 4, 1, gamma)
    assert int((rn > 0).sum()) > B // 4 and int((rn < gamma).sum()) > 0
    tl = _target_logits(rd, V, seed=3)
    inp = wl.attention_inputs(B, gamma + 1, 8, 2, 128, [int(x) for x in lens.clamp(min=1)],
                              paged=True, extra=gamma + 1, seed=4, device="cpu")
    cache = sv.KVCache(inp["cache_k"].to(dev), inp["cache_v"].to(dev), inp["prefix_len"].to(dev),
                       inp["block_table"].to(dev), 16)
    sv.sv_read_device_status()

    drafts, num = sv.sv_ngram_draft(hist.to(dev), lens.to(dev), 4, 1, gamma)
    out = sv.sv_accept_chain_commit(mode, tl.to(dev), None, sv.Q_DRAFT_ONEHOT, drafts,
                                    inp["k_tree"].to(dev), inp["v_tree"].to(dev), cache,
                                    temperature=1.0, seed=17, round_=2)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0  # -1 drafts are the end of a chain, not bad tokens

    assert torch.equal(drafts.cpu(), rd) and torch.equal(num.cpu(), rn)
    ref = oracle.accept_chain(mode, tl, None, oracle.Q_DRAFT_ONEHOT, rd, temperature=1.0,
                              seed=17, round_=2)
    # with 152064 entries most tokens carry less than 1e-6 of mass: many final samples
    # lie within 1e-6 of a CDF boundary (sample ties; the accepted drafts are compared)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=0.03,
            max_sample_frac=0.03 if V <= 4096 else 0.25)
    na = ref["num_accepted"]
    assert bool((na <= rn).all())            # never more than the proposed drafts
    assert int((na == rn).sum()) > 0 and int((na >= 2).sum()) > 0

    W = gamma + 1
    path = torch.arange(W, dtype=torch.int32).unsqueeze(0).expand(B, W).contiguous()
    ck, cv, pl = oracle.commit_kv(inp["k_tree"], inp["v_tree"], path, out["num_accepted"].cpu(),
                                  inp["cache_k"], inp["cache_v"], inp["prefix_len"],
                                  block_table=inp["block_table"], block_size=16)
    assert torch.equal(cache.prefix_len.cpu(), pl)
    assert torch.equal(cache.k.cpu(), ck) and torch.equal(cache.v.cpu(), cv)


def test_one_hot_chain_matches_oracle(cuda_ok):
    """Deterministic drafts without the n-gram step: random drafts, some cut short by -1."""
    B, gamma, V = 96, 4, 32000
    g = torch.Generator().manual_seed(23)
    drafts = torch.randint(0, V, (B, gamma), generator=g, dtype=torch.int32)
    cut = torch.randint(0, gamma + 1, (B,), generator=g)
    for b in range(B):
        drafts[b, int(cut[b]):] = -1
    tl = _target_logits(drafts, V, seed=5, agree=0.8)
    out = sv.sv_accept_chain(sv.EXACT, tl.cuda(), None, sv.Q_DRAFT_ONEHOT, drafts.cuda(), seed=3,
                             round_=9)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ref = oracle.accept_chain(oracle.EXACT, tl, None, oracle.Q_DRAFT_ONEHOT, drafts, seed=3,
                              round_=9)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=0.03,
            max_sample_frac=0.05)
    assert bool((ref["num_accepted"] <= cut.to(torch.int32)).all())

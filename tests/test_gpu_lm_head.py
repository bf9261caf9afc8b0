"""The LM-head projection on the tensor cores, alone and fused with the acceptance.

The projection ("推测解码技术详解", section "Medusa Heads"; lpnh.cn walkthrough, section 3.1:
a head is a Linear(H, V) from the hidden state to V logits) is compared with the oracle's
double-precision z = h W^T element by element.  The kernel accumulates in fp32 and stores
bf16, so each logit may differ from the exact value by half a bf16 ulp (the final
rounding) plus the fp32 accumulation error, bounded by Dm * 2^-23 * sum_k |h_k w_k|.  The
acceptance reads the stored logits, so its parity is bit-exact with the oracle run on those
stored bf16 logits (a one-ulp change of a logit may flip an integer decision, so the
acceptance is not compared on the exact logits).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(R, Dm, V, seed, sigma=3.0):
    """hidden ~N(0,1), weight ~N(0, sigma / sqrt(Dm)): logits about N(0, sigma)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn((R, Dm), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((V, Dm), generator=g, device="cuda") * (sigma / math.sqrt(Dm))).to(torch.bfloat16)
    return h, w


def _check_logits(z, h, w, rows=None):
    """Every listed row of z (bf16, device) against the oracle within the bound."""
    hc, wc = h.cpu(), w.cpu()
    if rows is not None:
        hc = hc[rows]
        z = z[rows]
    ref = oracle.lm_head(hc, wc)
    absdot = hc.double().abs() @ wc.double().abs().T
    Dm = h.shape[-1]
    ulp = torch.exp2(torch.floor(torch.log2(ref.abs().clamp_min(1e-30))) - 7)
    bound = 0.5 * ulp + Dm * 2.0 ** -23 * absdot
    err = (z.cpu().double() - ref).abs()
    bad = err > bound
    assert not bool(bad.any()), (f"{int(bad.sum())} logits outside the bound; worst excess "
                                 f"{float((err - bound).max()):.3e}")
    return ref


@pytest.mark.parametrize("R,Dm,V", [(200, 520, 4000), (128, 64, 256), (1, 4096, 2056)])
def test_projection_matches_oracle(cuda_ok, R, Dm, V):
    """Ragged row tile, ragged K block (520 = 8 x 64 + 8) and ragged vocabulary tile."""
    h, w = _inputs(R, Dm, V, seed=R + V)
    z = sv.sv_lm_head(h, w)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    _check_logits(z, h, w)


def test_projection_full_size_sampled_rows(cuda_ok):
    """The draft-chain workload's shapes: 384 target rows, hidden size 4096, 128256 tokens
    (403 GFLOP); six rows compared over the whole vocabulary."""
    R, Dm, V = 384, 4096, 128256
    h, w = _inputs(R, Dm, V, seed=9)
    z = sv.sv_lm_head(h, w)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    _check_logits(z, h, w, rows=[0, 127, 128, 200, 255, 383])


def _chain_case(B, gamma, Dm, V, seed, T, top_k):
    h, w = _inputs(B * (gamma + 1), Dm, V, seed)
    exact = oracle.lm_head(h.cpu(), w.cpu()).view(B, gamma + 1, V)
    g = torch.Generator().manual_seed(seed + 1)
    dl = (exact[:, :gamma] + torch.randn((B, gamma, V), generator=g, dtype=torch.float64)).to(torch.bfloat16)
    gc = torch.Generator().manual_seed(seed + 2)
    toks = torch.empty((B, gamma), dtype=torch.int32)
    for b in range(B):
        for i in range(gamma):
            toks[b, i] = wl._draft_sample(dl[b, i], T, top_k, gc)
    return h.view(B, gamma + 1, Dm), w, dl, toks


@pytest.mark.parametrize("mode,T,top_k", [(sv.EXACT, 1.0, 0), (sv.EXACT, 0.7, 50), (sv.GREEDY, 1.0, 0)])
def test_chain_acceptance_fused_with_projection(cuda_ok, mode, T, top_k):
    """Without top-k the target rows' statistics come from the projection's epilogue;
    with top-k the statistics kernel reads the stored rows."""
    B, gamma, Dm, V = 24, 5, 512, 32000
    h, w, dl, toks = _chain_case(B, gamma, Dm, V, seed=31, T=T, top_k=top_k)
    sv.sv_read_device_status()
    q = dl.cuda() if mode == sv.EXACT else None
    out = sv.sv_accept_chain_lmhead(mode, h, w, q, sv.Q_LOGITS, toks.cuda(), temperature=T,
                                    top_k=top_k, seed=7, round_=3)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    tl = out["target_logits"]
    _check_logits(tl.view(-1, V), h.view(-1, Dm), w)
    ref = oracle.accept_chain(mode, tl.cpu(), None if q is None else dl, oracle.Q_LOGITS, toks,
                              temperature=T, top_k=top_k, seed=7, round_=3)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_exempt_frac=0.02,
            max_sample_frac=0.05)
    # the same stored logits through the plain call give the same results
    plain = sv.sv_accept_chain(mode, tl, q, sv.Q_LOGITS, toks.cuda(), temperature=T, top_k=top_k,
                               seed=7, round_=3)
    torch.cuda.synchronize()
    dec = lambda x: (x.cpu().long() & 0xFFFF) == 0  # noqa: E731
    same = dec(out["near_ties"]) & dec(plain["near_ties"])
    for k in ("num_accepted", "num_emitted"):
        assert torch.equal(out[k].cpu()[same], plain[k].cpu()[same]), k


def test_tree_acceptance_fused_with_projection(cuda_ok):
    parent = wl.TREE_T26
    B, N, Dm, V = 16, len(parent), 256, 8000
    h, w = _inputs(B * N, Dm, V, seed=41)
    lg = wl.medusa_logits(B, parent, V, sigma=3.0, seed=42)
    dev = torch.device("cuda")
    out = sv.sv_accept_tree_lmhead(sv.EXACT, h.view(B, N, Dm), w, lg["draft_logits"].to(dev),
                                   sv.Q_LOGITS, parent, lg["node_tokens"].to(dev), seed=5, round_=1)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() & ~sv.SV_DEV_ZERO_DRAFT_PROB == 0
    tl = out["target_logits"]
    _check_logits(tl.view(-1, V), h, w)
    ref = oracle.accept_tree(oracle.EXACT, tl.cpu(), lg["draft_logits"], oracle.Q_LOGITS, parent,
                             lg["node_tokens"], seed=5, round_=1)
    compare(out, ref, ["path_nodes", "tokens", "num_emitted", "num_accepted"])


def test_chain_fused_full_size(cuda_ok):
    """The draft-chain workload's shapes (B = 64, gamma = 5, hidden 4096, V = 128256), T = 1
    without top-k (the epilogue's statistics), every sequence against the oracle on the
    stored logits; six rows of the projection over the whole vocabulary."""
    B, gamma, Dm, V = 64, 5, 4096, 128256
    h, w = _inputs(B * (gamma + 1), Dm, V, seed=51)
    g = torch.Generator(device="cuda").manual_seed(52)
    # draft rows: the projection of slightly perturbed hidden states (a draft model that
    # sees nearly the same context)
    hq = (h.float().view(B, gamma + 1, Dm)[:, :gamma] +
          0.3 * torch.randn((B, gamma, Dm), generator=g, device="cuda")).to(torch.bfloat16)
    dl = sv.sv_lm_head(hq, w)
    torch.cuda.synchronize()
    gc = torch.Generator().manual_seed(53)
    dlc = dl.cpu()
    toks = torch.empty((B, gamma), dtype=torch.int32)
    for b in range(B):
        for i in range(gamma):
            toks[b, i] = wl._draft_sample(dlc[b, i], 1.0, 0, gc)
    sv.sv_read_device_status()
    out = sv.sv_accept_chain_lmhead(sv.EXACT, h.view(B, gamma + 1, Dm), w, dl, sv.Q_LOGITS,
                                    toks.cuda(), seed=11, round_=0)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    tl = out["target_logits"]
    _check_logits(tl.view(-1, V), h, w, rows=[0, 5, 130, 255, 300, 383])
    ref = oracle.accept_chain(oracle.EXACT, tl.cpu(), dlc, oracle.Q_LOGITS, toks, seed=11, round_=0)
    compare(out, ref, ["tokens", "num_emitted", "num_accepted"], max_sample_frac=0.15)
    assert int(ref["num_accepted"].sum()) > 0

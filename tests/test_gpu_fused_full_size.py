"""The acceptance + KV commit call that the benchmark times, at the workloads' full sizes.

For each workload the fused call (sv_accept_chain_commit / sv_accept_tree_commit, with
the benchmark's arguments) is compared with the oracle on every sequence, repeated three
times from the same starting cache with bitwise-identical results, and its commit is
checked: the rows written are exactly the tree K/V rows of the kept path at positions
L_b .. L_b + accepted, nothing else in the cache changes, and prefix_len advances by
accepted + 1 (qwbw.cn sections 3.1.4 and 6.3).  On the ragged-paged workload (256
sequences of 152064-entry rows) this runs the ring variant of the select kernel with the
commit fused into it.
"""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cache(w):
    return sv.KVCache(w["cache_k"].clone(), w["cache_v"].clone(), w["prefix_len"].clone(),
                      None if w["block_table"] is None else w["block_table"].clone(),
                      w.get("block_size", 16))


def _expected_cache(w, path, num_accepted):
    """The cache after the commit by brute-force gather: row i of sequence b's kept path
    goes to position prefix_len[b] + i."""
    ek, ev = w["cache_k"].clone(), w["cache_v"].clone()
    pl = w["prefix_len"].cpu().tolist()
    pn = path.cpu()
    na = num_accepted.cpu().tolist()
    bs = w.get("block_size", 16)
    bt = None if w["block_table"] is None else w["block_table"].cpu()
    bi, ni, d0, d1 = [], [], [], []
    for b in range(len(pl)):
        for i in range(na[b] + 1):
            pos = pl[b] + i
            bi.append(b)
            ni.append(int(pn[b, i]))
            if bt is None:
                d0.append(b)
                d1.append(pos)
            else:
                d0.append(int(bt[b, pos // bs]))
                d1.append(pos % bs)
    dev = ek.device
    src = (torch.tensor(bi, device=dev), torch.tensor(ni, device=dev))
    dst = (torch.tensor(d0, device=dev), torch.tensor(d1, device=dev))
    ek[dst] = w["k_tree"][src]
    ev[dst] = w["v_tree"][src]
    new_pl = w["prefix_len"].cpu() + num_accepted.cpu() + 1
    return ek, ev, new_pl


@pytest.mark.parametrize("cfg,coverage", [(2, False), (2, True), (3, False), (4, False),
                                          (4, True), (5, False)])
def test_fused_call_full_size(cuda_ok, cfg, coverage):
    dev = torch.device("cuda")
    w = wl.make_workload(cfg, device=dev, coverage=coverage)
    c = w["cfg"]
    chain = c["kind"] == "chain"
    kw = dict(temperature=c["temperature"], top_k=c["top_k"], seed=w["seed"], round_=0)
    sv.sv_read_device_status()

    runs = []
    for _ in range(3):
        cb = _cache(w)
        if chain:
            r = sv.sv_accept_chain_commit(sv.EXACT, w["target_logits"], w["draft_logits"],
                                          sv.Q_LOGITS, w["draft_tokens"], w["k_tree"],
                                          w["v_tree"], cb, **kw)
        else:
            r = sv.sv_accept_tree_commit(sv.EXACT, w["target_logits"], w["draft_logits"],
                                         sv.Q_LOGITS, w["parent"], w["node_tokens"], w["k_tree"],
                                         w["v_tree"], cb, **kw)
        torch.cuda.synchronize()
        assert sv.sv_read_device_status() == 0
        runs.append((r, cb))

    # bitwise determinism over the three calls
    r0, c0 = runs[0]
    for r, cb in runs[1:]:
        for k in r0:
            assert torch.equal(r0[k], r[k]), k
        assert torch.equal(c0.prefix_len, cb.prefix_len)
        assert torch.equal(c0.k, cb.k) and torch.equal(c0.v, cb.v)
    del runs  # frees the two repeated caches (the first is kept in c0)

    # every sequence against the oracle
    if chain:
        ref = oracle.accept_chain(oracle.EXACT, w["target_logits"].cpu(), w["draft_logits"].cpu(),
                                  oracle.Q_LOGITS, w["draft_tokens"].cpu(), **kw)
        keys = ["tokens", "num_emitted", "num_accepted"]
    else:
        ref = oracle.accept_tree(oracle.EXACT, w["target_logits"].cpu(), w["draft_logits"].cpu(),
                                 oracle.Q_LOGITS, w["parent"], w["node_tokens"].cpu(), **kw)
        keys = ["tokens", "num_emitted", "num_accepted", "path_nodes"]
    compare(r0, ref, keys, max_exempt_frac=0.01,
            max_sample_frac=0.05 if c["V"] <= 32000 else 0.15)
    if coverage:
        assert int(r0["num_accepted"].sum()) > 0

    # the commit of the kernel's own kept path
    if chain:
        W = w["N"]
        path = torch.arange(W, dtype=torch.int32).unsqueeze(0).expand(c["B"], W)
    else:
        path = r0["path_nodes"]
    ek, ev, epl = _expected_cache(w, path, r0["num_accepted"])
    assert torch.equal(c0.prefix_len.cpu(), epl)
    assert torch.equal(c0.k, ek) and torch.equal(c0.v, ev)

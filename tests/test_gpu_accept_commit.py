"""The fused acceptance + commit calls against the two separate calls (bitwise), and the
commit they make against the oracle's commit of the same path."""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cache(w, dev):
    return sv.KVCache(w["cache_k"].clone(), w["cache_v"].clone(), w["prefix_len"].clone(),
                      None if w["block_table"] is None else w["block_table"].clone(),
                      w.get("block_size", 16))


@pytest.mark.parametrize("cfg,B,V,mode,coverage", [
    (2, 5, 4096, sv.EXACT, True),     # 64-node tree, paths accepted (coverage logits)
    (2, 3, 4096, sv.GREEDY, True),
    (3, 6, 4096, sv.EXACT, False),    # chain with top-k 50, T = 0.7
    (5, 12, 2048, sv.EXACT, False),   # chain over a paged cache
    (4, 2, 1024, sv.EXACT, True),     # 26-node tree, GQA 8
])
def test_fused_equals_separate_calls(cuda_ok, cfg, B, V, mode, coverage):
    dev = torch.device("cuda")
    w = wl.make_workload(cfg, device=dev, B=B, V=V, L=300, coverage=coverage)
    c = w["cfg"]
    chain = c["kind"] == "chain"
    toks = w["draft_tokens"] if chain else w["node_tokens"]
    q = w["draft_logits"] if mode == sv.EXACT else None
    kw = dict(temperature=c["temperature"], top_k=c["top_k"], seed=w["seed"], round_=3)

    ca = _cache(w, dev)  # separate calls
    if chain:
        ra = sv.sv_accept_chain(mode, w["target_logits"], q, sv.Q_LOGITS, toks, **kw)
        W = toks.shape[1] + 1
        path = torch.arange(W, dtype=torch.int32, device=dev).unsqueeze(0).expand(B, W).contiguous()
    else:
        ra = sv.sv_accept_tree(mode, w["target_logits"], q, sv.Q_LOGITS, w["parent"], toks, **kw)
        path = ra["path_nodes"]
    sv.sv_commit_kv(w["k_tree"], w["v_tree"], path, ra["num_accepted"], ca)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0

    cb = _cache(w, dev)  # fused
    if chain:
        rb = sv.sv_accept_chain_commit(mode, w["target_logits"], q, sv.Q_LOGITS, toks,
                                       w["k_tree"], w["v_tree"], cb, **kw)
    else:
        rb = sv.sv_accept_tree_commit(mode, w["target_logits"], q, sv.Q_LOGITS, w["parent"], toks,
                                      w["k_tree"], w["v_tree"], cb, **kw)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0

    for k in ("tokens", "num_emitted", "num_accepted", "near_ties"):
        assert torch.equal(ra[k], rb[k]), k
    if not chain:
        assert torch.equal(ra["path_nodes"], rb["path_nodes"])
    assert torch.equal(ca.prefix_len, cb.prefix_len)
    assert torch.equal(ca.k, cb.k) and torch.equal(ca.v, cb.v)
    if not chain and coverage and mode == sv.EXACT:
        assert int(rb["num_accepted"].sum()) > 0  # the commit moved more than the root

    # the committed cache equals the oracle's commit of the same path
    ck, cv, pl = oracle.commit_kv(w["k_tree"].cpu(), w["v_tree"].cpu(), path.cpu(),
                                  rb["num_accepted"].cpu(), w["cache_k"].cpu(), w["cache_v"].cpu(),
                                  w["prefix_len"].cpu(),
                                  block_table=None if w["block_table"] is None
                                  else w["block_table"].cpu(),
                                  block_size=w.get("block_size", 16))
    assert torch.equal(cb.prefix_len.cpu(), pl)
    assert torch.equal(cb.k.cpu(), ck) and torch.equal(cb.v.cpu(), cv)


def test_fused_full_size_bench_workload(cuda_ok):
    """The bench's default workload at full size: fused and separate calls agree."""
    dev = torch.device("cuda")
    w = wl.make_workload(2, device=dev)
    c = w["cfg"]
    kw = dict(temperature=c["temperature"], top_k=c["top_k"], seed=w["seed"], round_=0)
    ca, cb = _cache(w, dev), _cache(w, dev)
    ra = sv.sv_accept_tree(sv.EXACT, w["target_logits"], w["draft_logits"], sv.Q_LOGITS,
                           w["parent"], w["node_tokens"], **kw)
    sv.sv_commit_kv(w["k_tree"], w["v_tree"], ra["path_nodes"], ra["num_accepted"], ca)
    rb = sv.sv_accept_tree_commit(sv.EXACT, w["target_logits"], w["draft_logits"], sv.Q_LOGITS,
                                  w["parent"], w["node_tokens"], w["k_tree"], w["v_tree"], cb, **kw)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    for k in ("tokens", "num_emitted", "num_accepted", "near_ties", "path_nodes"):
        assert torch.equal(ra[k], rb[k]), k
    assert torch.equal(ca.prefix_len, cb.prefix_len)
    assert torch.equal(ca.k, cb.k) and torch.equal(ca.v, cb.v)

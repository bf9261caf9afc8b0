"""One tree per sequence (parent as a device array [B, N], parent_stride = N) on the GPU.

The tree-attention mask is per node ("推测解码技术详解", section "Tree Attention验证"; a
node's context is its own root path, lpnh.cn walkthrough section 3.2), so a batch whose
requests carry different trees (pruned per request, or built by a dynamic drafter) is
verified in one call.  Every output is compared with the oracle given the same trees
(attention: the oracle per sequence with its own tree; acceptance: the oracle's
per-sequence form, which keeps each sequence's index and so its uniforms).  A row that is not a BFS-ordered tree is reported
(SV_DEV_BAD_TREE) and its sequence keeps the root alone, without touching the others.
"""
import math

import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from accept_parity import compare
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N = 26


def _random_tree(n, max_depth, seed):
    g = torch.Generator().manual_seed(seed)
    par, dep = [-1], [0]
    for i in range(1, n):
        while True:
            a = int(torch.randint(0, i, (1,), generator=g))
            if dep[a] < max_depth:
                break
        par.append(a)
        dep.append(dep[a] + 1)
    return par


def _trees(B, max_depth=4):
    """B trees of N rows, each depth <= max_depth: the 26-node Medusa tree, the first 26
    rows of the 64-node one, the printed 7-node example with 19 more root children,
    random trees, and (when deep trees are allowed) a chain."""
    base = [list(wl.TREE_T26), list(wl.TREE_T64[:N]), list(wl.TREE_EXAMPLE7) + [0] * (N - 7)]
    if max_depth >= N - 1:
        base.append(wl.chain_parent(N - 1))
    out = []
    for b in range(B):
        out.append(base[b] if b < len(base) else _random_tree(N, max_depth, 100 + b))
    for t in out:
        assert oracle.check_tree(t) and len(t) == N
    return out


@pytest.mark.parametrize("Hq,Hkv,D,paged,dtype", [
    (16, 2, 128, False, torch.bfloat16),   # G = 8: two M tiles on the tensor-core kernel
    (2, 2, 128, True, torch.bfloat16),     # G = 1: 26 rows, row copies; 16-token pages
    (4, 4, 64, False, torch.bfloat16),
    (4, 2, 64, False, torch.float32),      # the fp32 kernel
])
def test_attention_per_sequence_trees(cuda_ok, Hq, Hkv, D, paged, dtype):
    B = 10
    trees = _trees(B, max_depth=N - 1)
    lens = [300 + 97 * b for b in range(B)]
    inp = wl.attention_inputs(B, N, Hq, Hkv, D, lens, dtype=dtype, paged=paged, extra=4, seed=8,
                              device="cpu")
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cache = sv.KVCache(g["cache_k"], g["cache_v"], g["prefix_len"], g["block_table"], 16)
    par = torch.tensor(trees, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(D)
    sv.sv_read_device_status()
    out = sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, par, scale)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    for b in range(B):
        ref = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                    inp["cache_v"], inp["prefix_len"], trees[b], scale,
                                    block_table=inp["block_table"], b_range=(b, b + 1))
        err = (out[b:b + 1].double().cpu() - ref).abs().max().item()
        assert err < tol, f"sequence {b}: max-abs error {err}"
    # the shared-tree call with sequence 0's tree agrees with the per-sequence call on it
    ws = sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, trees[0], scale)
    torch.cuda.synchronize()
    assert torch.equal(ws[0], out[0])


def _per_seq_logits(trees, V, seed, Dq=4):
    tl, ql, tk = [], [], []
    for b, t in enumerate(trees):
        lg = wl.medusa_logits(1, t, V, sigma=3.0, seed=seed + b, coverage=True, coverage_sigma=0.7)
        q = lg["draft_logits"]
        if q.shape[1] < Dq:
            q = torch.cat([q, torch.zeros((1, Dq - q.shape[1], V), dtype=q.dtype)], dim=1)
        tl.append(lg["target_logits"])
        ql.append(q)
        tk.append(lg["node_tokens"])
    return torch.cat(tl), torch.cat(ql), torch.cat(tk)


def _oracle_per_seq(fn, trees, tl, q, toks, **kw):
    """The oracle with the same per-sequence trees (one call, so that every sequence keeps
    its index, which keys its uniforms); outputs have N columns like the kernel's."""
    return fn(tl, q, trees, toks, **kw)


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_accept_per_sequence_trees(cuda_ok, mode):
    B, V = 40, 3000
    trees = _trees(B)
    tl, q, toks = _per_seq_logits(trees, V, seed=50)
    dev = torch.device("cuda")
    par = torch.tensor(trees, dtype=torch.int32, device=dev)
    qd = q.to(dev) if mode == sv.EXACT else None
    out = sv.sv_accept_tree(mode, tl.to(dev), qd, sv.Q_LOGITS, par, toks.to(dev), seed=4, round_=6)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ref = _oracle_per_seq(
        lambda t, qq, p, k, **kw: oracle.accept_tree(mode, t, qq, oracle.Q_LOGITS, p, k, **kw),
        trees, tl, q if mode == sv.EXACT else None, toks, seed=4, round_=6)
    compare(out, ref, ["path_nodes", "tokens", "num_emitted", "num_accepted"])
    assert int(ref["num_accepted"].sum()) > 0


def test_accept_commit_and_recursive_per_sequence_trees(cuda_ok):
    B, V = 24, 3000
    trees = _trees(B)
    tl, q, toks = _per_seq_logits(trees, V, seed=70)
    dev = torch.device("cuda")
    par = torch.tensor(trees, dtype=torch.int32, device=dev)
    # fused acceptance + commit: equal to the separate calls
    inp = wl.attention_inputs(B, N, 4, 2, 128, [200 + 13 * b for b in range(B)], paged=True,
                              extra=N, seed=3, device="cpu")
    def cache():
        return sv.KVCache(inp["cache_k"].to(dev), inp["cache_v"].to(dev), inp["prefix_len"].to(dev),
                          inp["block_table"].to(dev), 16)
    ca, cb = cache(), cache()
    ra = sv.sv_accept_tree(sv.EXACT, tl.to(dev), q.to(dev), sv.Q_LOGITS, par, toks.to(dev), seed=2)
    sv.sv_commit_kv(inp["k_tree"].to(dev), inp["v_tree"].to(dev), ra["path_nodes"], ra["num_accepted"], ca)
    rb = sv.sv_accept_tree_commit(sv.EXACT, tl.to(dev), q.to(dev), sv.Q_LOGITS, par, toks.to(dev),
                                  inp["k_tree"].to(dev), inp["v_tree"].to(dev), cb, seed=2)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    for k in ("path_nodes", "tokens", "num_emitted", "num_accepted", "near_ties"):
        assert torch.equal(ra[k], rb[k]), k
    assert torch.equal(ca.prefix_len, cb.prefix_len)
    assert torch.equal(ca.k, cb.k) and torch.equal(ca.v, cb.v)
    # siblings tried in turn, per sequence
    out = sv.sv_accept_tree_recursive(tl.to(dev), q.to(dev), sv.Q_LOGITS, par, toks.to(dev), seed=5,
                                      round_=1)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ref = _oracle_per_seq(
        lambda t, qq, p, k, **kw: oracle.accept_tree_recursive(t, qq, oracle.Q_LOGITS, p, k, **kw),
        trees, tl, q, toks, seed=5, round_=1)
    compare(out, ref, ["path_nodes", "tokens", "num_emitted", "num_accepted"])


def test_bad_tree_row_is_reported_and_contained(cuda_ok):
    B, V = 6, 512
    trees = _trees(B)
    tl, q, toks = _per_seq_logits(trees, V, seed=90)
    rows = torch.tensor(trees, dtype=torch.int32)
    rows[2, 5] = 9      # a parent after its child
    rows[4, 0] = 0      # a root that is not -1
    dev = torch.device("cuda")
    sv.sv_read_device_status()
    out = sv.sv_accept_tree(sv.EXACT, tl.to(dev), q.to(dev), sv.Q_LOGITS, rows.to(dev), toks.to(dev),
                            seed=1)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_TREE
    na = out["num_accepted"].cpu()
    assert int(na[2]) == 0 and int(na[4]) == 0
    pn = out["path_nodes"].cpu()
    assert int(pn[2, 0]) == 0 and bool((pn[2, 1:] == -1).all())
    ok = [0, 1, 3, 5]
    ref = _oracle_per_seq(
        lambda t, qq, p, k, **kw: oracle.accept_tree(oracle.EXACT, t, qq, oracle.Q_LOGITS, p, k, **kw),
        [trees[b] for b in ok], tl[ok], q[ok], toks[ok], seed=1)
    # the valid rows' results do not depend on the bad ones (sequence ids differ, so run
    # the same call on the valid rows alone and compare)
    out2 = sv.sv_accept_tree(sv.EXACT, tl[ok].to(dev), q[ok].to(dev), sv.Q_LOGITS,
                             rows[ok].contiguous().to(dev), toks[ok].to(dev), seed=1)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    compare(out2, ref, ["path_nodes", "tokens", "num_emitted", "num_accepted"])
    # attention with a bad row reports it too
    inp = wl.attention_inputs(B, N, 2, 2, 128, [64] * B, seed=1, device="cpu")
    cache = sv.KVCache(inp["cache_k"].to(dev), inp["cache_v"].to(dev), inp["prefix_len"].to(dev))
    sv.sv_tree_attention(inp["q"].to(dev), inp["k_tree"].to(dev), inp["v_tree"].to(dev), cache,
                         rows.to(dev), 1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_TREE

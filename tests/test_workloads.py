"""The seeded input recipe (CPU): the named candidate trees, the paged-cache layout, the
ragged prefix lengths, the drafter's samples and the workload shapes.  These generators
feed both the CUDA path's tests and the oracle's, so their structure is pinned here
independently of either."""
from collections import Counter

import pytest
import torch

from speculative_decoding_verify_sv_gb300 import workloads as wl


def _rank_tuples(parent):
    ranks = wl.child_ranks(parent)
    t = [()]
    for n in range(1, len(parent)):
        t.append(t[parent[n]] + (ranks[n],))
    return t


@pytest.mark.parametrize("name", ["TREE_EXAMPLE7", "TREE_T26", "TREE_T34", "TREE_T64"])
def test_named_trees_are_rank_closed_bfs_trees(name):
    """Every named tree lists parents before children in breadth-first order, and its nodes'
    rank tuples (the sibling rank at each depth of the root path) are closed: a node's parent
    is present, and so is its next-higher-ranked sibling (a Medusa tree keeps the best
    candidates of each head)."""
    par = getattr(wl, name)
    assert par[0] == -1 and all(0 <= par[n] < n for n in range(1, len(par)))
    T = _rank_tuples(par)
    assert len(set(T)) == len(T)
    S = set(T)
    for t in T[1:]:
        assert t[:-1] in S
        assert t[-1] == 0 or t[:-1] + (t[-1] - 1,) in S
    assert all(len(T[i]) <= len(T[i + 1]) for i in range(len(T) - 1))


def test_named_tree_sizes_and_caps():
    assert wl.TREE_T34 == wl.cartesian_tree([3, 2, 2, 1])
    full = wl.cartesian_tree([4, 3, 2, 1])
    assert len(full) == 1 + 4 + 12 + 24 + 24
    assert wl.TREE_T64 == full[:64]  # the last (lowest-ranked) leaf dropped
    assert len(wl.TREE_T26) == 26
    dep = wl.depths(wl.TREE_T26)
    assert max(dep) == 4 and [dep.count(k) for k in range(5)] == [1, 4, 7, 8, 6]
    kids = Counter(wl.TREE_T26[1:])
    assert all(c <= (4, 3, 2, 1)[dep[p]] for p, c in kids.items())
    # the tree-attention section's 7-node example: root A; B, C; D, E under B; F, G under C
    assert wl.depths(wl.TREE_EXAMPLE7) == [0, 1, 1, 2, 2, 2, 2]


@pytest.mark.parametrize("gamma", [1, 4, 63])
def test_chain_parent(gamma):
    par = wl.chain_parent(gamma)
    assert len(par) == gamma + 1 and wl.depths(par) == list(range(gamma + 1))
    assert wl.child_ranks(par) == [0] * (gamma + 1)


def test_ragged_prefix_lengths_are_seeded_and_in_range():
    cfg = wl.CONFIGS[5]
    a = wl.prefix_lengths(cfg, 256, seed=7)
    assert a == wl.prefix_lengths(cfg, 256, seed=7)
    assert a != wl.prefix_lengths(cfg, 256, seed=8)
    assert min(a) >= 512 and max(a) <= 8192 and len(set(a)) > 100
    assert wl.prefix_lengths(wl.CONFIGS[3], 4, seed=0) == [4096] * 4


def test_paged_cache_layout():
    """Each sequence owns just enough 16-token blocks for its prefix plus the commit room;
    the block ids of the batch are a permutation of the pool; unused entries are -1."""
    lens = [0, 5, 16, 17, 300]
    extra = 5
    inp = wl.attention_inputs(len(lens), 3, 4, 2, 64, lens, paged=True, extra=extra, seed=3)
    bt = inp["block_table"]
    need = [(L + extra + 15) // 16 for L in lens]
    assert bt.shape == (len(lens), max(need))
    used = []
    for b, n in enumerate(need):
        assert bool((bt[b, :n] >= 0).all()) and bool((bt[b, n:] == -1).all())
        used += bt[b, :n].tolist()
    assert sorted(used) == list(range(sum(need))) == list(range(inp["num_blocks"]))
    assert inp["cache_k"].shape == (sum(need), 16, 2, 64)
    assert used != sorted(used)  # shuffled, not in order


def test_contiguous_cache_room():
    inp = wl.attention_inputs(3, 6, 4, 2, 64, [10, 100, 33], extra=6, seed=1)
    assert inp["block_table"] is None
    assert inp["Lmax"] % 16 == 0 and inp["Lmax"] >= 100 + 6
    assert inp["cache_k"].shape == (3, inp["Lmax"], 2, 64)


def test_inputs_are_seeded():
    a = wl.attention_inputs(2, 3, 4, 2, 64, [20, 30], seed=5)
    b = wl.attention_inputs(2, 3, 4, 2, 64, [20, 30], seed=5)
    c = wl.attention_inputs(2, 3, 4, 2, 64, [20, 30], seed=6)
    for k in ("q", "k_tree", "v_tree", "cache_k", "cache_v"):
        assert torch.equal(a[k], b[k])
        assert not torch.equal(a[k], c[k])


def test_drafter_samples_from_its_own_top_k():
    """Chain drafts are the drafter's samples: within its top-k when top-k is set, its argmax
    at temperature 0, and draft row i is target row i plus the drafter's noise."""
    lg = wl.chain_logits(6, 4, 500, sigma=2.0, draft_sigma=1.0, dtype=torch.float32,
                         temperature=0.7, top_k=5, seed=4)
    dl, tok = lg["draft_logits"], lg["draft_tokens"]
    for b in range(6):
        for i in range(4):
            top = torch.topk(dl[b, i], 5).indices.tolist()
            assert int(tok[b, i]) in top
    g = wl.chain_logits(3, 2, 300, dtype=torch.float32, temperature=0.0, seed=9)
    assert torch.equal(g["draft_tokens"], g["draft_logits"].argmax(-1).to(torch.int32))
    resid = (lg["draft_logits"] - lg["target_logits"][:, :4]).flatten()
    assert 0.9 < float(resid.std()) < 1.1 and abs(float(resid.mean())) < 0.05


def test_medusa_node_tokens_follow_head_ranks():
    """A node with sibling rank i at depth d carries head d's rank-i token, so siblings carry
    distinct tokens."""
    par = wl.TREE_T26
    lg = wl.medusa_logits(3, par, 400, dtype=torch.float32, seed=2)
    dep, ranks = wl.depths(par), wl.child_ranks(par)
    heads, toks = lg["draft_logits"], lg["node_tokens"]
    assert heads.shape == (3, max(dep), 400) and toks.shape == (3, len(par))
    for b in range(3):
        order = [torch.sort(heads[b, d], descending=True, stable=True).indices for d in range(max(dep))]
        for n in range(1, len(par)):
            assert int(toks[b, n]) == int(order[dep[n] - 1][ranks[n]])
        for p in set(par[1:]):
            kids = [int(toks[b, n]) for n in range(1, len(par)) if par[n] == p]
            assert len(set(kids)) == len(kids)


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4, 5])
def test_workload_shapes(cfg_id):
    """Each workload at a reduced batch, vocabulary and prefix keeps its structure: the tree,
    the head layout, the dtype and the cache form."""
    cfg = wl.CONFIGS[cfg_id]
    L = (32, 80) if isinstance(cfg["L"], tuple) else 48
    w = wl.make_workload(cfg_id, B=2, V=256, L=L)
    par = wl.config_parent(cfg)
    N, Dmax = len(par), max(wl.depths(par))
    assert w["N"] == N and w["Dmax"] == Dmax
    assert w["q"].shape == (2, N, cfg["Hq"], cfg["D"]) and w["q"].dtype == cfg["dtype"]
    assert w["k_tree"].shape == (2, N, cfg["Hkv"], cfg["D"])
    assert w["target_logits"].shape == (2, N, 256) and w["target_logits"].dtype == cfg["dtype"]
    assert w["draft_logits"].shape == (2, (cfg["gamma"] if cfg["kind"] == "chain" else Dmax), 256)
    assert w["node_tokens"].shape == (2, N) and int(w["node_tokens"][:, 0].abs().sum()) == 0
    assert (w["block_table"] is not None) == cfg["paged"]
    if isinstance(L, tuple):
        assert all(L[0] <= int(x) <= L[1] for x in w["prefix_len"])
    else:
        assert w["prefix_len"].tolist() == [48, 48]

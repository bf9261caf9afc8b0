"""Pins of the oracle with one tree per sequence (CPU only).

A node's context is its own root path (lpnh.cn walkthrough, section 3.2; the mask of
"推测解码技术详解", section "Tree Attention验证"), so sequence b of a call whose trees
differ per sequence must give exactly what a call sharing sequence b's tree gives for
that sequence: same attention output, same decisions, path and tokens (the uniforms are
keyed by the sequence index, which is kept).  The shared-tree path itself is pinned by
the per-path brute force and the printed mask (test_oracle_attention, test_oracle_accept).
"""
import math

import numpy as np
import torch

import oracle
from speculative_decoding_verify_sv_gb300 import workloads as wl

N = 9
TREES = [
    [-1, 0, 0, 1, 1, 2, 2, 0, 3],   # the printed 7-node example with two more nodes
    [-1, 0, 1, 2, 3, 4, 5, 6, 7],   # a chain
    [-1, 0, 0, 0, 0, 0, 0, 0, 0],   # a star
    [-1, 0, 0, 1, 2, 2, 3, 5, 5],
]


def test_attention_per_sequence_equals_shared_tree_rows():
    B = len(TREES)
    inp = wl.attention_inputs(B, N, 4, 2, 32, [17, 40, 5, 23], dtype=torch.float32, seed=2)
    scale = 1.0 / math.sqrt(32)
    per = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], TREES, scale)
    for b, t in enumerate(TREES):
        shared = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                       inp["cache_v"], inp["prefix_len"], t, scale, b_range=(b, b + 1))
        assert torch.equal(per[b:b + 1], shared)
    # trees that differ give different outputs (the rows are really used)
    assert not torch.equal(per[1], oracle.tree_attention(
        inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"], inp["cache_v"], inp["prefix_len"],
        TREES[2], scale, b_range=(1, 2))[0])


def _logits(B, V, seed):
    g = torch.Generator().manual_seed(seed)
    tl = torch.randn((B, N, V), generator=g) * 2.0
    q = torch.randn((B, N - 1, V), generator=g) * 2.0
    toks = torch.randint(0, V, (B, N), generator=g, dtype=torch.int32)
    # make some decisions pass: a node's token is its parent row's argmax half the time
    for b, t in enumerate(TREES):
        for c in range(1, N):
            if (b + c) % 2 == 0:
                toks[b, c] = int(torch.argmax(tl[b, t[c]]))
    return tl, q, toks


def test_accept_per_sequence_equals_shared_tree_rows():
    B, V = len(TREES), 64
    tl, q, toks = _logits(B, V, 5)
    for mode in (oracle.EXACT, oracle.GREEDY):
        per = oracle.accept_tree(mode, tl, q, oracle.Q_LOGITS, TREES, toks, seed=3, round_=2)
        assert per["path_nodes"].shape == (B, N)
        for b, t in enumerate(TREES):
            shared = oracle.accept_tree(mode, tl, q, oracle.Q_LOGITS, t, toks, seed=3, round_=2)
            W = shared["path_nodes"].shape[1]
            for k in ("num_emitted", "num_accepted", "near_ties"):
                assert int(per[k][b]) == int(shared[k][b]), (mode, b, k)
            for k in ("path_nodes", "tokens"):
                assert torch.equal(per[k][b, :W], shared[k][b]), (mode, b, k)
                assert bool((per[k][b, W:] == -1).all())
            assert torch.equal(per["acc"][b], shared["acc"][b])
        if mode == oracle.GREEDY:
            assert int(per["num_accepted"].sum()) > 0


def test_recursive_per_sequence_equals_shared_tree_rows():
    B, V = len(TREES), 64
    tl, q, toks = _logits(B, V, 7)
    per = oracle.accept_tree_recursive(tl, q, oracle.Q_LOGITS, TREES, toks, seed=4, round_=1)
    for b, t in enumerate(TREES):
        shared = oracle.accept_tree_recursive(tl, q, oracle.Q_LOGITS, t, toks, seed=4, round_=1)
        W = shared["path_nodes"].shape[1]
        assert int(per["num_accepted"][b]) == int(shared["num_accepted"][b])
        assert torch.equal(per["tokens"][b, :W], shared["tokens"][b])
        assert torch.equal(per["path_nodes"][b, :W], shared["path_nodes"][b])


def test_a_bad_row_is_rejected():
    bad = [list(t) for t in TREES]
    bad[2][4] = 6  # a parent after its child
    B, V = len(TREES), 64
    tl, q, toks = _logits(B, V, 9)
    try:
        oracle.accept_tree(oracle.EXACT, tl, q, oracle.Q_LOGITS, bad, toks)
    except ValueError:
        pass
    else:
        raise AssertionError("a malformed tree row was accepted")

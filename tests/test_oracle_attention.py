"""Pins of the oracle's tree attention and tree structure (CPU only).

Each test checks the oracle against something other than itself: the mask printed
on the pages, torch's scaled_dot_product_attention as a library special case, or a
per-path brute force written as ordinary causal attention.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import read_golden
from speculative_decoding_verify_sv_gb300 import workloads as wl


def _sdpa_causal(q, k, v, scale, gqa):
    """Causal attention of the LAST rows q [Tq,H,D] over k, v [Tk,Hkv,D] (float64)."""
    Tq, Tk = q.shape[0], k.shape[0]
    qq = q.permute(1, 0, 2).unsqueeze(0)
    kk = k.permute(1, 0, 2).unsqueeze(0)
    vv = v.permute(1, 0, 2).unsqueeze(0)
    # query i sits at absolute position Tk - Tq + i
    mask = torch.ones((Tq, Tk), dtype=torch.bool).tril(diagonal=Tk - Tq)
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale,
                                         enable_gqa=gqa)
    return out[0].permute(1, 0, 2)


def test_mask_matches_printed_example():
    """(P1) The 7-node example's mask equals the printed matrix, and its bitmask rows
    are {1,3,5,11,19,37,69}."""
    rows = read_golden("tree_mask_example7.txt")
    printed = np.array([[int(x) for x in r] for r in rows], dtype=np.uint8)
    m = oracle.tree_mask(wl.TREE_EXAMPLE7)
    assert np.array_equal(m, printed)
    bits = [int(sum(int(m[n, j]) << j for j in range(7))) for n in range(7)]
    assert bits == [1, 3, 5, 11, 19, 37, 69]


def test_tree_validation():
    assert oracle.check_tree(wl.TREE_EXAMPLE7)
    assert oracle.check_tree(wl.TREE_T64) and len(wl.TREE_T64) == 64
    assert oracle.check_tree(wl.TREE_T34) and len(wl.TREE_T34) == 34
    assert oracle.check_tree(wl.TREE_T26) and len(wl.TREE_T26) == 26
    assert not oracle.check_tree([0, 0])
    assert not oracle.check_tree([-1, 1])
    assert not oracle.check_tree([-1, 0, 3, 1])


def test_tree_shapes_from_caps():
    """The literal Cartesian trees behind the Medusa workloads."""
    assert wl.cartesian_tree((3, 2, 2, 1)) == wl.TREE_T34
    assert wl.cartesian_tree((4, 3, 2, 1))[:64] == wl.TREE_T64
    dep = wl.depths(wl.TREE_T26)
    assert [dep.count(d) for d in range(5)] == [1, 4, 7, 8, 6]


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chain_equals_causal_attention(Hq, Hkv, dtype):
    """(P2) A chain tree is ordinary causal attention over [prefix; chain]."""
    B, gamma, D, L = 2, 5, 16, 37
    par = wl.chain_parent(gamma)
    N = len(par)
    inp = wl.attention_inputs(B, N, Hq, Hkv, D, [L, L - 9], dtype=dtype, seed=3)
    scale = 1.0 / math.sqrt(D)
    out = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], par, scale)
    for b in range(B):
        Lb = int(inp["prefix_len"][b])
        k = torch.cat([inp["cache_k"][b, :Lb], inp["k_tree"][b]]).double()
        v = torch.cat([inp["cache_v"][b, :Lb], inp["v_tree"][b]]).double()
        ref = _sdpa_causal(inp["q"][b].double(), k, v, scale, Hq != Hkv)
        torch.testing.assert_close(out[b], ref, rtol=1e-12, atol=1e-12)


def test_tree_equals_per_path_attention():
    """(P3) Each node's output is causal attention over [prefix; its root path]."""
    B, D, L, Hq, Hkv = 2, 8, 11, 4, 2
    par = wl.TREE_T26
    N = len(par)
    inp = wl.attention_inputs(B, N, Hq, Hkv, D, [L, 3], dtype=torch.float32, seed=5)
    scale = 0.37
    out = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], par, scale)
    for b in range(B):
        Lb = int(inp["prefix_len"][b])
        for n in range(N):
            path = []
            a = n
            while a >= 0:
                path.append(a)
                a = par[a]
            path = path[::-1]
            k = torch.cat([inp["cache_k"][b, :Lb], inp["k_tree"][b, path]]).double()
            v = torch.cat([inp["cache_v"][b, :Lb], inp["v_tree"][b, path]]).double()
            ref = _sdpa_causal(inp["q"][b, n:n + 1].double(), k, v, scale, True)
            torch.testing.assert_close(out[b, n], ref[0], rtol=1e-12, atol=1e-12)


def test_single_node_is_decode_attention():
    """(P4) N = 1 (root only) is plain decode attention over prefix + itself."""
    B, D, L, H = 3, 32, 50, 2
    inp = wl.attention_inputs(B, 1, H, H, D, [L, 1, 0], dtype=torch.float32, seed=9)
    scale = 1.0 / math.sqrt(D)
    out = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], [-1], scale)
    for b in range(B):
        Lb = int(inp["prefix_len"][b])
        k = torch.cat([inp["cache_k"][b, :Lb], inp["k_tree"][b]]).double()
        v = torch.cat([inp["cache_v"][b, :Lb], inp["v_tree"][b]]).double()
        for h in range(H):
            s = (k[:, h] @ inp["q"][b, 0, h].double()) * scale
            ref = torch.softmax(s, 0) @ v[:, h]
            torch.testing.assert_close(out[b, 0, h], ref, rtol=1e-12, atol=1e-12)


def test_paged_equals_contiguous():
    """The paged layout holds the same prefix rows: results are identical."""
    B, D, Hq, Hkv = 3, 16, 4, 2
    par = wl.TREE_EXAMPLE7
    N = len(par)
    lens = [40, 17, 33]
    pg = wl.attention_inputs(B, N, Hq, Hkv, D, lens, dtype=torch.bfloat16, paged=True,
                             block_size=16, seed=13)
    Lmax = 48
    ck = torch.zeros((B, Lmax, Hkv, D), dtype=torch.bfloat16)
    cv = torch.zeros_like(ck)
    for b in range(B):
        for pos in range(lens[b]):
            blk = int(pg["block_table"][b, pos // 16])
            ck[b, pos] = pg["cache_k"][blk, pos % 16]
            cv[b, pos] = pg["cache_v"][blk, pos % 16]
    a = oracle.tree_attention(pg["q"], pg["k_tree"], pg["v_tree"], pg["cache_k"], pg["cache_v"],
                              pg["prefix_len"], par, block_table=pg["block_table"], block_size=16)
    c = oracle.tree_attention(pg["q"], pg["k_tree"], pg["v_tree"], ck, cv, pg["prefix_len"], par)
    assert torch.equal(a, c)


def test_b_range_selects_rows():
    B, D, H = 4, 8, 2
    par = wl.chain_parent(2)
    inp = wl.attention_inputs(B, 3, H, H, D, [5, 6, 7, 8], dtype=torch.float32, seed=21)
    full = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                 inp["cache_v"], inp["prefix_len"], par)
    part = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                 inp["cache_v"], inp["prefix_len"], par, b_range=(1, 3))
    assert torch.equal(full[1:3], part)

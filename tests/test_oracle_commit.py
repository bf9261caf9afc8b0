"""Pins of the oracle's KV commit (CPU only).

The commit copies the tree K/V rows of the kept path (root first, then the accepted nodes in
depth order) to cache positions L_b .. L_b + accepted and advances prefix_len by accepted + 1
("MTP (Medusa)" article, sections 3.1.4 and 6.3; hncyxsy.com section 4.3).  It is checked
against a brute-force gather of the path rows on tiny caches, contiguous and paged with a
shuffled block table; every other position must be unchanged.  A second check ties it to the
tree attention (pinned on its own): after the commit, the last path node's tree attention over
the old prefix equals its attention with the committed rows as prefix.
"""
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _paths(parent, B, gen):
    """A random root path per sequence: (path_nodes [B, Dmax+1] padded with -1, accepted)."""
    N = len(parent)
    depth = [0] * N
    for i in range(1, N):
        depth[i] = depth[parent[i]] + 1
    W = max(depth) + 1
    pn = torch.full((B, W), -1, dtype=torch.int32)
    na = torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        a = int(torch.randint(0, N, (1,), generator=gen))
        chain = []
        while a >= 0:
            chain.append(a)
            a = parent[a]
        chain.reverse()
        pn[b, :len(chain)] = torch.tensor(chain, dtype=torch.int32)
        na[b] = len(chain) - 1
    return pn, na


def _brute(k_tree, v_tree, pn, na, ck, cv, pl, rowof):
    ck, cv, pl = ck.clone(), cv.clone(), pl.clone()
    for b in range(k_tree.shape[0]):
        L = int(pl[b])
        for i in range(int(na[b]) + 1):
            r = rowof(b, L + i)
            ck[r] = k_tree[b, int(pn[b, i])]
            cv[r] = v_tree[b, int(pn[b, i])]
        pl[b] = L + int(na[b]) + 1
    return ck, cv, pl


PARENT = [-1, 0, 0, 1, 1, 2, 2, 3, 5]  # depths 0,1,1,2,2,2,2,3,3


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_commit_contiguous_equals_brute_force(dtype):
    gen = torch.Generator().manual_seed(31)
    B, N, Hkv, D, Lmax = 5, len(PARENT), 2, 16, 24
    k_tree = torch.randn(B, N, Hkv, D, generator=gen).to(dtype)
    v_tree = torch.randn(B, N, Hkv, D, generator=gen).to(dtype)
    ck = torch.randn(B, Lmax, Hkv, D, generator=gen).to(dtype)
    cv = torch.randn(B, Lmax, Hkv, D, generator=gen).to(dtype)
    pl = torch.tensor([0, 3, 11, 19, 7], dtype=torch.int32)
    pn, na = _paths(PARENT, B, gen)
    got = oracle.commit_kv(k_tree, v_tree, pn, na, ck, cv, pl)
    flat_k, flat_v = ck.reshape(B * Lmax, Hkv, D), cv.reshape(B * Lmax, Hkv, D)
    ek, ev, epl = _brute(k_tree, v_tree, pn, na, flat_k, flat_v, pl, lambda b, p: b * Lmax + p)
    assert torch.equal(got[0].reshape(B * Lmax, Hkv, D), ek)
    assert torch.equal(got[1].reshape(B * Lmax, Hkv, D), ev)
    assert torch.equal(got[2], epl)
    # inputs untouched, and only the committed rows changed
    changed = (got[0] != ck).reshape(B, Lmax, -1).any(-1)
    for b in range(B):
        L, n = int(pl[b]), int(na[b]) + 1
        assert not changed[b, :L].any() and not changed[b, L + n:].any()


def test_commit_paged_equals_brute_force():
    gen = torch.Generator().manual_seed(32)
    B, N, Hkv, D, bs = 4, len(PARENT), 2, 8, 4
    max_blocks = 6
    num_blocks = B * max_blocks + 3
    perm = torch.randperm(num_blocks, generator=gen)[:B * max_blocks].to(torch.int32)
    bt = perm.reshape(B, max_blocks)
    k_tree = torch.randn(B, N, Hkv, D, generator=gen)
    v_tree = torch.randn(B, N, Hkv, D, generator=gen)
    ck = torch.randn(num_blocks, bs, Hkv, D, generator=gen)
    cv = torch.randn(num_blocks, bs, Hkv, D, generator=gen)
    pl = torch.tensor([2, 4, 13, 17], dtype=torch.int32)  # block boundaries crossed
    pn, na = _paths(PARENT, B, gen)
    got = oracle.commit_kv(k_tree, v_tree, pn, na, ck, cv, pl, block_table=bt, block_size=bs)
    rowof = lambda b, p: int(bt[b, p // bs]) * bs + p % bs
    fk, fv = ck.reshape(-1, Hkv, D), cv.reshape(-1, Hkv, D)
    ek, ev, epl = _brute(k_tree, v_tree, pn, na, fk, fv, pl, rowof)
    assert torch.equal(got[0].reshape(-1, Hkv, D), ek)
    assert torch.equal(got[1].reshape(-1, Hkv, D), ev)
    assert torch.equal(got[2], epl)


def test_commit_then_attention_over_the_committed_prefix():
    """Node a's tree attention over prefix L equals the attention of a's query, as the
    root of a one-node tree holding a's own K/V, over the committed prefix L + depth(a)
    (the path rows root .. parent(a) now in the cache)."""
    gen = torch.Generator().manual_seed(33)
    B, N, Hq, Hkv, D, Lmax = 3, len(PARENT), 4, 2, 16, 32
    q = torch.randn(B, N, Hq, D, generator=gen, dtype=torch.float64).float()
    k_tree = torch.randn(B, N, Hkv, D, generator=gen)
    v_tree = torch.randn(B, N, Hkv, D, generator=gen)
    ck = torch.randn(B, Lmax, Hkv, D, generator=gen)
    cv = torch.randn(B, Lmax, Hkv, D, generator=gen)
    pl = torch.tensor([5, 0, 17], dtype=torch.int32)
    pn, na = _paths(PARENT, B, gen)
    full = oracle.tree_attention(q, k_tree, v_tree, ck, cv, pl, PARENT)
    # commit root .. parent(a) (accepted = depth(a) - 1 rows after the root)
    na_m1 = na - 1
    keep = na >= 1
    nk, nv, npl = oracle.commit_kv(k_tree, v_tree, pn, torch.clamp(na_m1, min=0), ck, cv, pl)
    for b in range(B):
        a = int(pn[b, int(na[b])])
        if keep[b]:
            ckb, cvb, Lb = nk[b:b + 1], nv[b:b + 1], npl[b:b + 1]
        else:  # a is the root: nothing to commit
            ckb, cvb, Lb = ck[b:b + 1], cv[b:b + 1], pl[b:b + 1]
        one = oracle.tree_attention(q[b:b + 1, a:a + 1], k_tree[b:b + 1, a:a + 1],
                                    v_tree[b:b + 1, a:a + 1], ckb, cvb, Lb, [-1])
        assert torch.allclose(one[0, 0], full[b, a], rtol=0, atol=1e-12)

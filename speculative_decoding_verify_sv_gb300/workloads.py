"""Seeded synthetic inputs for the verify step.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.  It
holds no arithmetic of the verify method: it draws tensors from seeded torch
generators, builds the candidate-tree structures, and plays the *drafter* (which sits
upstream of verification): chain drafts are sampled from the draft distribution, and
Medusa node tokens are the per-depth ranked tokens of the head logits.

Workloads (sizes of the five verify workloads; logits "~N(0,s)" read as standard
deviation s):

  1 chain-f32      B=1,   gamma=4, V=1000,   Hq=Hkv=4,  D=64,  L=128,   fp32
  2 medusa-t64     B=8,   64-node tree, V=32000, Hq=Hkv=32, D=128, L=2048, bf16
  3 draft-chain    B=64,  gamma=5, V=128256, Hq=32/Hkv=8, D=128, L=4096, T=0.7, top-k 50
  4 long-tree      B=16,  26-node tree, V=32000, Hq=64/Hkv=8, D=128, L=32768
  5 ragged-paged   B=256, gamma=4, V=152064, Hq=32/Hkv=8, D=128, L~U{512..8192}, paged 16
"""
from __future__ import annotations

import math

import torch

# ------------------------------------------------------------------ trees

#: The 7-node example of the tree-attention section (root A; B, C; D, E under B; F, G under C).
TREE_EXAMPLE7 = [-1, 0, 0, 1, 1, 2, 2]

#: Literal Cartesian tree of per-depth caps (3, 2, 2, 1): 1+3+6+12+12 = 34 nodes.
TREE_T34 = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6, 7, 7, 8, 8, 9, 9,
            10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21]

#: Cartesian tree of caps (4, 3, 2, 1) (65 nodes) without its lowest-score leaf: 64 nodes.
TREE_T64 = [-1, 0, 0, 0, 0, 1, 1, 1, 2, 2, 2, 3, 3, 3, 4, 4, 4, 5, 5, 6, 6, 7, 7, 8, 8,
            9, 9, 10, 10, 11, 11, 12, 12, 13, 13, 14, 14, 15, 15, 16, 16, 17, 18, 19, 20,
            21, 22, 23, 24, 25, 26, 27, 28, 29, 30, 31, 32, 33, 34, 35, 36, 37, 38, 39]

#: 26-node Medusa-style tree (caps 4, 3, 2, 1; the 25 highest-score rank tuples).
TREE_T26 = [-1, 0, 0, 0, 0, 1, 1, 1, 2, 2, 3, 4, 5, 5, 6, 6, 7, 8, 8, 10, 12, 13, 14,
            16, 17, 19]


def chain_parent(gamma: int) -> list[int]:
    """A draft chain of gamma tokens as a tree: root, then one child per level."""
    return [-1] + list(range(gamma))


def cartesian_tree(caps) -> list[int]:
    """Parent array (BFS order) of the full tree with caps[d] children per depth-d node."""
    parent, level = [-1], [0]
    for cap in caps:
        nxt = []
        for p in level:
            for _ in range(cap):
                parent.append(p)
                nxt.append(len(parent) - 1)
        level = nxt
    return parent


def depths(parent) -> list[int]:
    d = []
    for p in parent:
        d.append(0 if p < 0 else d[p] + 1)
    return d


def child_ranks(parent) -> list[int]:
    """Rank of each node among its siblings (0 = first child), root 0."""
    seen: dict[int, int] = {}
    ranks = []
    for p in parent:
        if p < 0:
            ranks.append(0)
            continue
        ranks.append(seen.get(p, 0))
        seen[p] = ranks[-1] + 1
    return ranks


# ------------------------------------------------------------ generators

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, std, dtype, g, device, chunk_elems=1 << 28):
    """N(0, std) in dtype, drawn in float32 chunks (keeps peak memory low)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        tmp = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e] = tmp.to(dtype)
    return out


def attention_inputs(B, N, Hq, Hkv, D, prefix_lens, dtype=torch.bfloat16, paged=False,
                     block_size=16, extra=8, seed=0, device="cpu"):
    """Q [B,N,Hq,D], tree K/V [B,N,Hkv,D] and the prefix cache, all ~N(0,1).

    The cache has room for ``extra`` more positions per sequence (for the commit).
    Paged: a pool of fixed-size blocks; each sequence owns just enough blocks for
    L_b + extra positions, and the block table is a seeded random permutation of the
    pool (unused table entries are -1)."""
    g = _gen(device, seed)
    lens = torch.as_tensor(prefix_lens, dtype=torch.int32)
    assert lens.numel() == B
    q = _randn((B, N, Hq, D), 1.0, dtype, g, device)
    k_tree = _randn((B, N, Hkv, D), 1.0, dtype, g, device)
    v_tree = _randn((B, N, Hkv, D), 1.0, dtype, g, device)
    out = dict(q=q, k_tree=k_tree, v_tree=v_tree, prefix_len=lens.to(device))
    if not paged:
        Lmax = int(lens.max().item()) + extra
        Lmax = (Lmax + 15) // 16 * 16
        out["cache_k"] = _randn((B, Lmax, Hkv, D), 1.0, dtype, g, device)
        out["cache_v"] = _randn((B, Lmax, Hkv, D), 1.0, dtype, g, device)
        out["block_table"] = None
        out["Lmax"] = Lmax
    else:
        nblk = [(int(L) + extra + block_size - 1) // block_size for L in lens.tolist()]
        total = sum(nblk)
        perm = torch.randperm(total, generator=_gen("cpu", seed + 7)).to(torch.int32)
        max_blocks = max(nblk)
        bt = torch.full((B, max_blocks), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(nblk):
            bt[b, :n] = perm[off:off + n]
            off += n
        out["cache_k"] = _randn((total, block_size, Hkv, D), 1.0, dtype, g, device)
        out["cache_v"] = _randn((total, block_size, Hkv, D), 1.0, dtype, g, device)
        out["block_table"] = bt.to(device)
        out["block_size"] = block_size
        out["num_blocks"] = total
    return out


def _ranked_tokens(logits_row: torch.Tensor, k: int) -> torch.Tensor:
    """The k highest-logit token ids of one row, ties -> lower id (the drafter's top-k)."""
    order = torch.sort(logits_row.float(), descending=True, stable=True).indices
    return order[:k]


def _draft_sample(logits_row: torch.Tensor, T: float, top_k: int, g, top_p: float = 1.0) -> int:
    """The drafter's own sample from its row: Gumbel-max over the top_k highest logits
    (all tokens if top_k == 0), narrowed to their nucleus when top_p < 1 (the drafter
    samples only tokens its own distribution gives mass).  Sits upstream of
    verification."""
    z = logits_row.float().cpu()
    V = z.numel()
    if 0 < top_k < V:
        cand = _ranked_tokens(z, top_k)
        if top_p < 1.0 and T > 0:
            w = torch.softmax(z[cand].double() / T, dim=0)
            before = torch.cumsum(w, 0) - w
            cand = cand[before < top_p]
    else:
        cand = torch.arange(V)
    if T == 0:
        return int(cand[torch.argmax(z[cand])].item())
    u = torch.rand(cand.numel(), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    return int(cand[torch.argmax(z[cand].double() / T + gumbel)].item())


def chain_logits(B, gamma, V, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16,
                 temperature=1.0, top_k=0, seed=0, device="cpu", top_p=1.0):
    """Target logits [B,gamma+1,V] ~N(0,sigma); draft logits [B,gamma,V] with row i =
    target row i + N(0,draft_sigma) (the draft of token i+1 sees the same context as
    target row i); draft tokens [B,gamma] sampled by the drafter from its rows."""
    g = _gen(device, seed)
    tl = _randn((B, gamma + 1, V), sigma, torch.float32, g, device)
    noise = _randn((B, gamma, V), draft_sigma, torch.float32, g, device)
    dl = (tl[:, :gamma] + noise).to(dtype)
    tl = tl.to(dtype)
    gc = _gen("cpu", seed + 11)
    toks = torch.empty((B, gamma), dtype=torch.int32)
    dl_cpu = dl.float().cpu()
    for b in range(B):
        for i in range(gamma):
            toks[b, i] = _draft_sample(dl_cpu[b, i], temperature, top_k, gc, top_p)
    return dict(target_logits=tl, draft_logits=dl, draft_tokens=toks.to(device))


def medusa_logits(B, parent, V, sigma=3.0, dtype=torch.bfloat16, seed=0, device="cpu",
                  coverage=False, coverage_sigma=1.0):
    """Target logits [B,N,V] ~N(0,sigma); Medusa head logits [B,Dmax,V] ~N(0,sigma)
    (row d-1 = head d, which proposes depth-d tokens); node tokens [B,N]: the node with
    sibling rank i at depth d gets the rank-i token of head d (ties -> lower id).
    coverage=True makes target row n = head(depth n + 1) + N(0,coverage_sigma) so that
    paths get accepted (test variant)."""
    g = _gen(device, seed)
    N = len(parent)
    dep = depths(parent)
    Dmax = max(dep)
    ranks = child_ranks(parent)
    heads = _randn((B, Dmax, V), sigma, torch.float32, g, device)
    tl = _randn((B, N, V), sigma, torch.float32, g, device)
    if coverage:
        for n in range(N):
            if dep[n] < Dmax:
                tl[:, n] = heads[:, dep[n]] + coverage_sigma * tl[:, n] / sigma
    heads = heads.to(dtype)
    tl = tl.to(dtype)
    kmax = max(ranks) + 1
    hc = heads.float().cpu()
    toks = torch.zeros((B, N), dtype=torch.int32)
    for b in range(B):
        ranked = [_ranked_tokens(hc[b, d], kmax) for d in range(Dmax)]
        for n in range(1, N):
            toks[b, n] = ranked[dep[n] - 1][ranks[n]]
    return dict(target_logits=tl, draft_logits=heads, node_tokens=toks.to(device))


def draft_probs(draft_logits: torch.Tensor, temperature: float = 1.0) -> torch.Tensor:
    """The drafter's probabilities (float32) for callers that pass q as probabilities."""
    return torch.softmax(draft_logits.float() / temperature, dim=-1)


# --------------------------------------------------------------- workloads

CONFIGS = {
    1: dict(name="chain-f32", kind="chain", B=1, gamma=4, V=1000, Hq=4, Hkv=4, D=64, L=128,
            dtype=torch.float32, sigma=2.0, draft_sigma=0.5, temperature=1.0, top_k=0,
            mode="exact", paged=False),
    2: dict(name="medusa-t64", kind="tree", B=8, parent=TREE_T64, V=32000, Hq=32, Hkv=32,
            D=128, L=2048, dtype=torch.bfloat16, sigma=3.0, temperature=1.0, top_k=0,
            mode="exact", paged=False),
    3: dict(name="draft-chain", kind="chain", B=64, gamma=5, V=128256, Hq=32, Hkv=8, D=128,
            L=4096, dtype=torch.bfloat16, sigma=3.0, draft_sigma=1.0, temperature=0.7,
            top_k=50, mode="exact", paged=False),
    4: dict(name="long-tree", kind="tree", B=16, parent=TREE_T26, V=32000, Hq=64, Hkv=8,
            D=128, L=32768, dtype=torch.bfloat16, sigma=3.0, temperature=1.0, top_k=0,
            mode="exact", paged=False),
    5: dict(name="ragged-paged", kind="chain", B=256, gamma=4, V=152064, Hq=32, Hkv=8,
            D=128, L=(512, 8192), dtype=torch.bfloat16, sigma=3.0, draft_sigma=1.0,
            temperature=1.0, top_k=0, mode="exact", paged=True),
}


def config_parent(cfg: dict) -> list[int]:
    return chain_parent(cfg["gamma"]) if cfg["kind"] == "chain" else list(cfg["parent"])


def prefix_lengths(cfg: dict, B: int, seed: int) -> list[int]:
    L = cfg["L"]
    if isinstance(L, tuple):
        g = _gen("cpu", seed + 3)
        return torch.randint(L[0], L[1] + 1, (B,), generator=g).tolist()
    return [int(L)] * B


def make_workload(cfg_id: int, device="cpu", seed=None, B=None, V=None, L=None,
                  coverage=False, parent=None) -> dict:
    """All inputs of one verify step of workload ``cfg_id`` (optionally resized)."""
    cfg = dict(CONFIGS[cfg_id])
    if B is not None:
        cfg["B"] = B
    if V is not None:
        cfg["V"] = V
    if L is not None:
        cfg["L"] = L
    if parent is not None:
        cfg["kind"], cfg["parent"] = "tree", list(parent)
    seed = 1234 + cfg_id if seed is None else seed
    par = config_parent(cfg)
    N = len(par)
    Dmax = max(depths(par))
    lens = prefix_lengths(cfg, cfg["B"], seed)
    att = attention_inputs(cfg["B"], N, cfg["Hq"], cfg["Hkv"], cfg["D"], lens,
                           dtype=cfg["dtype"], paged=cfg["paged"], extra=Dmax + 1,
                           seed=seed, device=device)
    if cfg["kind"] == "chain":
        lg = chain_logits(cfg["B"], cfg["gamma"], cfg["V"], sigma=cfg["sigma"],
                          draft_sigma=cfg["draft_sigma"], dtype=cfg["dtype"],
                          temperature=cfg["temperature"], top_k=cfg["top_k"],
                          seed=seed + 100, device=device)
        node_tokens = torch.zeros((cfg["B"], N), dtype=torch.int32, device=device)
        node_tokens[:, 1:] = lg["draft_tokens"]
        lg["node_tokens"] = node_tokens
    else:
        lg = medusa_logits(cfg["B"], par, cfg["V"], sigma=cfg["sigma"], dtype=cfg["dtype"],
                           seed=seed + 100, device=device, coverage=coverage)
    return dict(cfg=cfg, parent=par, N=N, Dmax=Dmax, scale=1.0 / math.sqrt(cfg["D"]),
                seed=seed, **att, **lg)

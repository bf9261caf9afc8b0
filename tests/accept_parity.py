"""Comparison of acceptance outputs (GPU against the oracle) under the near-tie rule.

Both sides report near ties in one packed word per sequence:
  low 16 bits  -- decision ties: a decision with |u_acc - ratio| < 1e-6 whose parent lies
                  on an accepted path, a top-p cut within 1e-6 of top_p, or (sibling rule)
                  an empty residual handed to the next sibling.  Any of these can change
                  which nodes are accepted, so the whole sequence is exempt.
  high 16 bits -- sample ties: the final inverse-CDF sample within the window of a CDF
                  boundary, or its residual empty.  Only the last emitted token is in
                  doubt: the accepted length, the path and every accepted token are still
                  compared exactly.
"""
import torch

SAMPLE_TIE = 65536


def decision_ties(w: torch.Tensor) -> torch.Tensor:
    return w.to(torch.int64) & 0xFFFF


def sample_ties(w: torch.Tensor) -> torch.Tensor:
    return w.to(torch.int64) >> 16


def compare(gpu, ref, keys, max_exempt_frac=0.01, max_sample_frac=None):
    """Assert that `keys` agree exactly outside the reported near ties.

    max_exempt_frac bounds the sequences with a decision tie (on either side);
    max_sample_frac (default: the same) bounds those with only a sample tie.  Returns
    (decision-exempt count, sample-only count)."""
    g = {k: v.cpu() for k, v in gpu.items()}
    r = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in ref.items()}
    B = g["num_accepted"].shape[0]
    dec = (decision_ties(g["near_ties"]) > 0) | (decision_ties(r["near_ties"]) > 0)
    smp = ((sample_ties(g["near_ties"]) > 0) | (sample_ties(r["near_ties"]) > 0)) & ~dec
    keep = ~dec
    # counts and paths: exact on every sequence without a decision tie
    for k in keys:
        if k == "tokens":
            continue
        a, b = g[k][keep], r[k][keep]
        if not torch.equal(a, b):
            bad = torch.nonzero((g[k] != r[k]).reshape(B, -1).any(1) & keep).flatten()
            raise AssertionError(f"{k} differs on sequences {bad[:10].tolist()}: "
                                 f"gpu {g[k][bad[:3]].tolist()} oracle {r[k][bad[:3]].tolist()}")
    if "tokens" in keys:
        tg, tr = g["tokens"], r["tokens"]
        W = tg.shape[1]
        # the last emitted token sits at column num_accepted
        last = torch.zeros_like(tg, dtype=torch.bool)
        na = r["num_accepted"].to(torch.int64).clamp(0, W - 1)
        last[torch.arange(B), na] = True
        mask = keep.unsqueeze(1) & ~(smp.unsqueeze(1) & last)
        diff = (tg != tr) & mask
        if bool(diff.any()):
            bad = torch.nonzero(diff.any(1)).flatten()
            raise AssertionError(f"tokens differ on sequences {bad[:10].tolist()}: "
                                 f"gpu {tg[bad[:3]].tolist()} oracle {tr[bad[:3]].tolist()}")
    n_dec, n_smp = int(dec.sum()), int(smp.sum())
    assert n_dec <= max(2, max_exempt_frac * B), f"{n_dec} sequences with a decision near tie"
    lim = max_exempt_frac if max_sample_frac is None else max_sample_frac
    assert n_smp <= max(2, lim * B), f"{n_smp} sequences with a sample near tie"
    n_ex = n_dec + n_smp
    if n_ex >= 5:
        # the windows are worst-case bounds: most flagged sequences still agree exactly
        same = torch.ones(B, dtype=torch.bool)
        for k in keys:
            same &= (g[k] == r[k]).reshape(B, -1).all(1)
        flagged = dec | smp
        assert int(same[flagged].sum()) >= 0.8 * n_ex, "near-tie sequences mostly disagree"
    return n_dec, n_smp

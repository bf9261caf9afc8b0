"""GPU KV commit vs the oracle (bitwise), contiguous and paged, plus a brute-force gather."""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_commit_matches_oracle(cuda_ok, paged, dtype):
    par = wl.TREE_T26
    B, N, Hkv, D = 6, 26, 8, 128
    lens = [0, 15, 16, 17, 500, 31]
    inp = wl.attention_inputs(B, N, 4 * Hkv, Hkv, D, lens, dtype=dtype, paged=paged, extra=5,
                              seed=31)
    g = torch.Generator().manual_seed(5)
    dep = wl.depths(par)
    paths, nacc = torch.full((B, 5), -1, dtype=torch.int32), torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        leaf = int(torch.randint(0, N, (1,), generator=g))
        path = []
        a = leaf
        while a >= 0:
            path.append(a)
            a = par[a]
        path = path[::-1]
        paths[b, :len(path)] = torch.tensor(path, dtype=torch.int32)
        nacc[b] = dep[leaf]
    dev = torch.device("cuda")
    cache = sv.KVCache(inp["cache_k"].to(dev), inp["cache_v"].to(dev), inp["prefix_len"].to(dev),
                       None if inp["block_table"] is None else inp["block_table"].to(dev), 16)
    sv.sv_commit_kv(inp["k_tree"].to(dev), inp["v_tree"].to(dev), paths.to(dev), nacc.to(dev), cache)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    ck, cv, pl = oracle.commit_kv(inp["k_tree"], inp["v_tree"], paths, nacc, inp["cache_k"],
                                  inp["cache_v"], inp["prefix_len"], block_table=inp["block_table"])
    assert torch.equal(cache.prefix_len.cpu(), pl)
    assert torch.equal(cache.k.cpu(), ck)
    assert torch.equal(cache.v.cpu(), cv)
    # (P10) brute-force gather with tensor indexing: committed rows are the path rows
    for b in range(B):
        for i in range(int(nacc[b]) + 1):
            pos = lens[b] + i
            if inp["block_table"] is None:
                row_k = cache.k[b, pos]
            else:
                row_k = cache.k[int(inp["block_table"][b, pos // 16]), pos % 16]
            assert torch.equal(row_k.cpu(), inp["k_tree"][b, int(paths[b, i])])


def test_commit_bad_block_is_reported(cuda_ok):
    """The block table covers only positions 0..15; committing at 16 and 17 touches no
    memory, sets SV_DEV_BAD_BLOCK, and leaves the pool unchanged."""
    B, N, Hkv, D = 1, 2, 1, 8
    inp = wl.attention_inputs(B, N, 1, Hkv, D, [16], dtype=torch.bfloat16, paged=True, extra=0,
                              seed=3)
    assert inp["block_table"].shape == (1, 1)
    dev = torch.device("cuda")
    cache = sv.KVCache(inp["cache_k"].to(dev), inp["cache_v"].to(dev), inp["prefix_len"].to(dev),
                       inp["block_table"].to(dev), 16)
    paths = torch.tensor([[0, 1]], dtype=torch.int32, device=dev)
    nacc = torch.tensor([1], dtype=torch.int32, device=dev)
    before_k, before_v = cache.k.clone(), cache.v.clone()
    sv.sv_commit_kv(inp["k_tree"].to(dev), inp["v_tree"].to(dev), paths, nacc, cache)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_BLOCK
    assert torch.equal(cache.k, before_k) and torch.equal(cache.v, before_v)

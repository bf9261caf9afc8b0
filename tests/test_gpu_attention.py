"""GPU tree attention vs the CPU oracle (element by element), through the C ABI."""
import math

import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def _run(inp, parent, dtype, block_size=16):
    dev = torch.device("cuda")
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cache = sv.KVCache(g["cache_k"], g["cache_v"], g["prefix_len"], g["block_table"], block_size)
    D = g["q"].shape[-1]
    out = sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, parent, 1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    return out


def _check(inp, parent, dtype, b_range=None, block_size=16):
    out = _run(inp, parent, dtype, block_size)
    D = inp["q"].shape[-1]
    ref = oracle.tree_attention(inp["q"], inp["k_tree"], inp["v_tree"], inp["cache_k"],
                                inp["cache_v"], inp["prefix_len"], parent, 1.0 / math.sqrt(D),
                                block_table=inp["block_table"], block_size=block_size,
                                b_range=b_range)
    b0, b1 = b_range if b_range else (0, out.shape[0])
    err = (out[b0:b1].double().cpu() - ref).abs().max().item()
    assert err < TOL[dtype], err
    return out, err


@pytest.mark.parametrize("lens", [[0, 1, 63, 64, 65, 300, 1000, 129]])
def test_chain_gqa_ragged(cuda_ok, lens):
    par = wl.chain_parent(4)
    inp = wl.attention_inputs(len(lens), 5, 32, 8, 128, lens, dtype=torch.bfloat16, seed=1)
    _check(inp, par, torch.bfloat16)


def test_tree26_gqa64_multi_mtile(cuda_ok):
    """26 nodes x 8 group heads = 208 query rows: two 128-row M tiles per KV head."""
    par = wl.TREE_T26
    inp = wl.attention_inputs(3, 26, 64, 8, 128, [777, 0, 1500], dtype=torch.bfloat16, seed=2)
    _check(inp, par, torch.bfloat16)


def test_tree64_mha_long_prefix_splits(cuda_ok):
    """Few (b, head) pairs and a long prefix: the prefix is split and merged."""
    par = wl.TREE_T64
    Lmax_probe = 2048 + 8
    assert sv.sv_tree_attention_workspace_size(torch.bfloat16, 2, 64, 4, 4, 128, Lmax_probe) > 0
    inp = wl.attention_inputs(2, 64, 4, 4, 128, [2048, 1999], dtype=torch.bfloat16, seed=3)
    _check(inp, par, torch.bfloat16)


def test_paged_shuffled(cuda_ok):
    par = wl.chain_parent(4)
    lens = [512, 17, 0, 1024, 333, 800]
    inp = wl.attention_inputs(len(lens), 5, 32, 8, 128, lens, dtype=torch.bfloat16, paged=True,
                              seed=4)
    _check(inp, par, torch.bfloat16)


def test_head_dim_64_bf16(cuda_ok):
    par = wl.TREE_EXAMPLE7
    inp = wl.attention_inputs(2, 7, 8, 2, 64, [100, 250], dtype=torch.bfloat16, seed=5)
    _check(inp, par, torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128])
def test_fp32(cuda_ok, D):
    par = wl.chain_parent(4)
    inp = wl.attention_inputs(2, 5, 4, 4, D, [128, 37], dtype=torch.float32, seed=6)
    _check(inp, par, torch.float32)


def test_fp32_paged_tree(cuda_ok):
    par = wl.TREE_T26
    inp = wl.attention_inputs(2, 26, 4, 2, 64, [200, 45], dtype=torch.float32, paged=True, seed=7)
    _check(inp, par, torch.float32)


def test_root_only_is_decode(cuda_ok):
    inp = wl.attention_inputs(3, 1, 16, 4, 128, [0, 5, 700], dtype=torch.bfloat16, seed=8)
    _check(inp, [-1], torch.bfloat16)


def test_deterministic(cuda_ok):
    par = wl.TREE_T26
    inp = wl.attention_inputs(2, 26, 16, 4, 128, [900, 300], dtype=torch.bfloat16, seed=9)
    a = _run(inp, par, torch.bfloat16)
    b = _run(inp, par, torch.bfloat16)
    assert torch.equal(a, b)


def test_bad_prefix_sets_status(cuda_ok):
    """A prefix longer than the cache is clamped and reported, never trapped."""
    par = wl.chain_parent(1)
    inp = wl.attention_inputs(1, 2, 4, 4, 128, [10], dtype=torch.bfloat16, seed=10)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g["prefix_len"][0] = inp["Lmax"] + 100
    cache = sv.KVCache(g["cache_k"], g["cache_v"], g["prefix_len"])
    sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, par, 0.1)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_PREFIX
    assert sv.sv_read_device_status() == 0  # reading cleared it


@pytest.mark.parametrize("cfg,b_range", [(1, (0, 1)), (2, (0, 2)), (3, (5, 7)), (4, (3, 4)),
                                         (5, (100, 102))])
def test_full_size_workloads_sampled(cuda_ok, cfg, b_range):
    """Each workload at full size in the bench's launch configuration; the oracle
    recomputes a sample of sequences."""
    w = wl.make_workload(cfg, device="cuda")
    dtype = w["cfg"]["dtype"]
    cache = sv.KVCache(w["cache_k"], w["cache_v"], w["prefix_len"], w["block_table"],
                       w.get("block_size", 16))
    out = sv.sv_tree_attention(w["q"], w["k_tree"], w["v_tree"], cache, w["parent"], w["scale"])
    torch.cuda.synchronize()
    assert sv.sv_read_device_status() == 0
    b0, b1 = b_range
    sel = slice(b0, b1)
    if w["block_table"] is None:
        ck, cv = w["cache_k"][sel].cpu(), w["cache_v"][sel].cpu()
        bt = None
    else:
        ck, cv = w["cache_k"].cpu(), w["cache_v"].cpu()
        bt = w["block_table"][sel].cpu()
    ref = oracle.tree_attention(w["q"][sel].cpu(), w["k_tree"][sel].cpu(), w["v_tree"][sel].cpu(),
                                ck, cv, w["prefix_len"][sel].cpu(), w["parent"], w["scale"],
                                block_table=bt, block_size=w.get("block_size", 16))
    err = (out[sel].double().cpu() - ref).abs().max().item()
    assert err < TOL[dtype], err


def test_group_not_dividing_128_uses_general_path(cuda_ok):
    """GQA group of 3 heads: served by the mma.sync kernel."""
    par = wl.TREE_T26
    inp = wl.attention_inputs(2, 26, 12, 4, 128, [300, 1100], dtype=torch.bfloat16, seed=11)
    _check(inp, par, torch.bfloat16)


def test_rows_beyond_two_mma_tiles(cuda_ok):
    """64 nodes x 8 group heads = 512 rows: two groups of 256 rows per KV head."""
    par = wl.TREE_T64
    inp = wl.attention_inputs(2, 64, 16, 2, 128, [500, 77], dtype=torch.bfloat16, seed=12)
    _check(inp, par, torch.bfloat16)


def test_single_unit_cut_across_all_ctas(cuda_ok):
    """One (sequence, kv head) with a 32K prefix: every CTA holds a piece of it."""
    par = wl.chain_parent(3)
    inp = wl.attention_inputs(1, 4, 8, 1, 128, [32768], dtype=torch.bfloat16, seed=13)
    _check(inp, par, torch.bfloat16)


def test_fewer_tiles_than_ctas(cuda_ok):
    par = wl.chain_parent(1)
    inp = wl.attention_inputs(1, 2, 4, 1, 64, [10], dtype=torch.bfloat16, seed=14)
    _check(inp, par, torch.bfloat16)


def test_paged_block32_64_128_256(cuda_ok):
    par = wl.TREE_EXAMPLE7
    for bs in (32, 64, 128, 256):
        inp = wl.attention_inputs(3, 7, 16, 4, 128, [700, 33, 130], dtype=torch.bfloat16,
                                  paged=True, block_size=bs, seed=15 + bs)
        _check(inp, par, torch.bfloat16, block_size=bs)


def test_paged_block128_two_mma_tiles(cuda_ok):
    """Pages of 128 rows, one per 128-key tile, with two M tiles (208 rows)."""
    par = wl.TREE_T26
    inp = wl.attention_inputs(2, 26, 64, 8, 128, [600, 129], dtype=torch.bfloat16, paged=True,
                              block_size=128, seed=17)
    _check(inp, par, torch.bfloat16, block_size=128)


@pytest.mark.parametrize("D,paged,bs,lens", [(64, False, 16, [333, 1200, 128]),
                                          (128, True, 16, [600, 129, 1]),
                                          (64, True, 32, [257, 40, 1000])])
def test_two_mma_tiles_head_dim_and_pages(cuda_ok, D, paged, bs, lens):
    """Two M tiles (26 nodes x 8 group heads) with D = 64, and with pages shorter than a
    tile (16-row pages: one copy per page into the grouped layout at D = 128); ragged ends
    of the last tile (prefix lengths not multiples of 128)."""
    par = wl.TREE_T26
    inp = wl.attention_inputs(len(lens), 26, 64, 8, D, lens, dtype=torch.bfloat16, paged=paged,
                              block_size=bs, seed=31 + D + bs)
    _check(inp, par, torch.bfloat16, block_size=bs)


def test_two_mma_tiles_many_units_repeatable(cuda_ok):
    """More units than CTAs with two M tiles; three calls give identical outputs."""
    par = wl.TREE_T26
    inp = wl.attention_inputs(40, 26, 64, 8, 128, [64 * (i % 7) + 5 * i for i in range(40)],
                              dtype=torch.bfloat16, seed=37)
    out, _ = _check(inp, par, torch.bfloat16, b_range=(0, 6))
    for _ in range(2):
        assert torch.equal(_run(inp, par, torch.bfloat16), out)


def test_workspace_reused_across_calls_and_shapes(cuda_ok):
    """One zero-filled workspace serves a run of calls of different shapes; every call
    matches a call with a fresh workspace bit for bit."""
    cases = [(2, 26, 16, 4, 128, [900, 300], wl.TREE_T26, 21),
             (1, 4, 8, 1, 128, [32768], wl.chain_parent(3), 22),
             (3, 7, 16, 4, 128, [700, 33, 130], wl.TREE_EXAMPLE7, 23),
             (2, 64, 16, 2, 128, [500, 77], wl.TREE_T64, 24)]
    size = max(sv.sv_tree_attention_workspace_size(torch.bfloat16, B, N, Hq, Hkv, D, max(lens) + 8)
               for B, N, Hq, Hkv, D, lens, _, _ in cases)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        for B, N, Hq, Hkv, D, lens, par, seed in cases:
            inp = wl.attention_inputs(B, N, Hq, Hkv, D, lens, dtype=torch.bfloat16, seed=seed)
            g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
            cache = sv.KVCache(g["cache_k"], g["cache_v"], g["prefix_len"])
            out = sv.sv_tree_attention(g["q"], g["k_tree"], g["v_tree"], cache, par,
                                       1.0 / math.sqrt(D), workspace=ws)
            torch.cuda.synchronize()
            assert sv.sv_read_device_status() == 0
            assert torch.equal(out, _run(inp, par, torch.bfloat16))


def test_launch_counter_counts_kernels(cuda_ok):
    lib = sv.load_library()
    par = wl.chain_parent(4)
    inp = wl.attention_inputs(2, 5, 32, 8, 128, [100, 200], dtype=torch.bfloat16, seed=16)
    before = lib.sv_kernel_launches()
    _run(inp, par, torch.bfloat16)
    assert lib.sv_kernel_launches() - before >= 1

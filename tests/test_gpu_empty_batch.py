"""An empty batch (B = 0 sequences, R = 0 rows) through every entry point that launches
work: the call validates its other arguments, returns success, launches nothing and reads no
tensor (empty tensors may have NULL data pointers)."""
import pytest
import torch

import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _launches(fn):
    n0 = sv.sv_kernel_launches()
    out = fn()
    torch.cuda.synchronize()
    assert sv.sv_kernel_launches() == n0
    assert sv.sv_read_device_status() == 0
    return out


def test_empty_attention(cuda_ok):
    parent = wl.TREE_EXAMPLE7
    N, Hq, Hkv, D = len(parent), 8, 2, 128
    q = torch.empty((0, N, Hq, D), dtype=torch.bfloat16, device=DEV)
    kt = torch.empty((0, N, Hkv, D), dtype=torch.bfloat16, device=DEV)
    cache = sv.KVCache(torch.empty((0, 64, Hkv, D), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0, 64, Hkv, D), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0,), dtype=torch.int32, device=DEV))
    out = _launches(lambda: sv.sv_tree_attention(q, kt, kt.clone(), cache, parent, D ** -0.5))
    assert tuple(out.shape) == (0, N, Hq, D)


@pytest.mark.parametrize("mode", [sv.EXACT, sv.GREEDY])
def test_empty_acceptance(cuda_ok, mode):
    V, gamma = 1000, 4
    tl = torch.empty((0, gamma + 1, V), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((0, gamma, V), dtype=torch.bfloat16, device=DEV)
    dt = torch.empty((0, gamma), dtype=torch.int32, device=DEV)
    r = _launches(lambda: sv.sv_accept_chain(mode, tl, q, sv.Q_LOGITS, dt))
    assert r["tokens"].shape[0] == 0
    parent = wl.TREE_T26
    N = len(parent)
    tlt = torch.empty((0, N, V), dtype=torch.bfloat16, device=DEV)
    qt = torch.empty((0, max(wl.depths(parent)), V), dtype=torch.bfloat16, device=DEV)
    nt = torch.empty((0, N), dtype=torch.int32, device=DEV)
    r = _launches(lambda: sv.sv_accept_tree(mode, tlt, qt, sv.Q_LOGITS, parent, nt))
    assert r["path_nodes"].shape[0] == 0
    if mode == sv.EXACT:
        _launches(lambda: sv.sv_accept_tree_recursive(tlt, qt, sv.Q_LOGITS, parent, nt))
    _launches(lambda: sv.sv_accept_typical(tlt, parent, nt))


def test_empty_commit_and_fused_acceptance(cuda_ok):
    V, gamma, Hkv, D = 1000, 4, 2, 64
    kt = torch.empty((0, gamma + 1, Hkv, D), dtype=torch.bfloat16, device=DEV)
    cache = sv.KVCache(torch.empty((0, 64, Hkv, D), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0, 64, Hkv, D), dtype=torch.bfloat16, device=DEV),
                       torch.empty((0,), dtype=torch.int32, device=DEV))
    pn = torch.empty((0, gamma + 1), dtype=torch.int32, device=DEV)
    na = torch.empty((0,), dtype=torch.int32, device=DEV)
    _launches(lambda: sv.sv_commit_kv(kt, kt.clone(), pn, na, cache))
    tl = torch.empty((0, gamma + 1, V), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((0, gamma, V), dtype=torch.bfloat16, device=DEV)
    dt = torch.empty((0, gamma), dtype=torch.int32, device=DEV)
    _launches(lambda: sv.sv_accept_chain_commit(sv.EXACT, tl, q, sv.Q_LOGITS, dt, kt, kt.clone(), cache))


def test_empty_drafting_and_projection(cuda_ok):
    hist = torch.empty((0, 256), dtype=torch.int32, device=DEV)
    lens = torch.empty((0,), dtype=torch.int32, device=DEV)
    drafts, num = _launches(lambda: sv.sv_ngram_draft(hist, lens, max_ngram=3, min_ngram=1, gamma=4))
    assert drafts.shape[0] == 0 and num.shape[0] == 0
    h = torch.empty((0, 128), dtype=torch.bfloat16, device=DEV)
    w = torch.randn((1024, 128), device=DEV).to(torch.bfloat16)
    z = _launches(lambda: sv.sv_lm_head(h, w))
    assert tuple(z.shape) == (0, 1024)

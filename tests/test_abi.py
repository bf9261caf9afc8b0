"""The C ABI library loads, exports every symbol include/sv.h declares, and rejects bad
arguments on the host before any launch (CPU only; no compute call needs a GPU)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return sv.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "sv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sv_tree_attention", "sv_accept_chain", "sv_accept_tree", "sv_commit_kv",
              "sv_read_device_status", "sv_last_error", "sv_tree_attention_workspace_size",
              "sv_accept_workspace_size", "sv_tree_prepare", "sv_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    assert sv.sv_version().startswith("sv ")


def test_tree_prepare_matches_printed_mask(lib):
    anc, dep = sv.sv_tree_prepare([-1, 0, 0, 1, 1, 2, 2])
    assert anc == [1, 3, 5, 11, 19, 37, 69]
    assert dep == [0, 1, 1, 2, 2, 2, 2]


@pytest.mark.parametrize("parent", [[0], [-1, 1], [-1, 0, 3], [-1, -1]])
def test_invalid_trees_are_rejected(lib, parent):
    with pytest.raises(sv.SVError) as e:
        sv.sv_tree_prepare(parent)
    assert e.value.code == sv.SV_ERR_INVALID_ARG


def test_too_many_nodes_unsupported(lib):
    par = (ctypes.c_int32 * 65)(*([-1] + list(range(64))))
    assert lib.sv_tree_prepare(65, par, None, None) == sv.SV_ERR_UNSUPPORTED


def _cache(**kw):
    c = sv._KVCacheC()
    c.k = c.v = c.prefix_len = 16
    c.block_table = None
    c.Lmax = 128
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_attention_rejects_before_launch(lib):
    par = (ctypes.c_int32 * 1)(-1)
    P = ctypes.c_void_p(16)
    # head dim 96 is not compiled
    assert lib.sv_tree_attention(1, 1, 1, 4, 4, 96, P, P, P, _cache(), par, 0, 0.1, P, None, 0,
                                 None) == sv.SV_ERR_UNSUPPORTED
    # Hq not a multiple of Hkv
    assert lib.sv_tree_attention(1, 1, 1, 6, 4, 128, P, P, P, _cache(), par, 0, 0.1, P, None, 0,
                                 None) == sv.SV_ERR_INVALID_ARG
    # misaligned q
    assert lib.sv_tree_attention(1, 1, 1, 4, 4, 128, ctypes.c_void_p(18), P, P, _cache(), par, 0,
                                 0.1, P, None, 0, None) == sv.SV_ERR_INVALID_ARG
    # NaN scale
    assert lib.sv_tree_attention(1, 1, 1, 4, 4, 128, P, P, P, _cache(), par, 0, float("nan"), P,
                                 None, 0, None) == sv.SV_ERR_INVALID_ARG
    assert "scale" in lib.sv_last_error().decode()
    # missing workspace when the plan needs one (long prefix, small batch -> splits)
    need = lib.sv_tree_attention_workspace_size(1, 1, 1, 4, 4, 128, 32768)
    assert need > 0
    assert lib.sv_tree_attention(1, 1, 1, 4, 4, 128, P, P, P, _cache(Lmax=32768), par, 0, 0.1, P,
                                 None, 0, None) == sv.SV_ERR_WORKSPACE


def test_accept_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    par = (ctypes.c_int32 * 3)(-1, 0, 0)
    common = dict(seed=0, round=0)
    # V not a multiple of 8
    assert lib.sv_accept_chain(1, 1, 1, 4, 1001, P, P, 1, P, 1.0, 0, 1.0, 0, 0, P, P, P, P, P, 1 << 20,
                               None) == sv.SV_ERR_UNSUPPORTED
    # negative temperature, top_k too large
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, P, 1, P, -1.0, 0, 1.0, 0, 0, P, P, P, P, P, 1 << 20,
                               None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, P, 1, P, 1.0, 5000, 1.0, 0, 0, P, P, P, P, P,
                               1 << 20, None) == sv.SV_ERR_INVALID_ARG
    # exact mode needs q
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, None, 1, P, 1.0, 0, 1.0, 0, 0, P, P, P, P, P,
                               1 << 20, None) == sv.SV_ERR_INVALID_ARG
    # q rows must cover the tree depth
    assert lib.sv_accept_tree(1, 1, 1, 3, 1000, par, 0, P, P, P, 1, 0, 1.0, 0, 1.0, 0, 0, P, P, P, P, P,
                              P, 1 << 20, None) == sv.SV_ERR_INVALID_ARG
    # top_p outside (0, 1]; top_p < 1 without top-k in exact mode
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, P, 1, P, 1.0, 5, 0.0, 0, 0, P, P, P, P, P,
                               1 << 20, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, P, 1, P, 1.0, 5, 1.5, 0, 0, P, P, P, P, P,
                               1 << 20, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_accept_chain(1, 1, 1, 4, 1000, P, P, 1, P, 1.0, 0, 0.9, 0, 0, P, P, P, P, P,
                               1 << 20, None) == sv.SV_ERR_UNSUPPORTED
    # workspace too small
    need = lib.sv_accept_workspace_size(2, 3, 1000, 1)
    assert need > 0
    assert lib.sv_accept_tree(1, 1, 2, 3, 1000, par, 0, P, P, P, 1, 1, 1.0, 0, 1.0, 0, 0, P, P, P, P, P,
                              P, 16, None) == sv.SV_ERR_WORKSPACE
    del common


def test_commit_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    # rows must be whole 16-byte vectors: Hkv*D*2 = 6 bytes
    assert lib.sv_commit_kv(1, 1, 2, 1, 3, P, P, P, 2, P, _cache(), None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_commit_kv(1, 1, 2, 1, 8, P, P, None, 2, P, _cache(), None) == sv.SV_ERR_INVALID_ARG


def test_fused_accept_commit_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    par = (ctypes.c_int32 * 3)(-1, 0, 0)
    # a bad acceptance argument (V not a multiple of 8) is reported as by sv_accept_tree
    assert lib.sv_accept_tree_commit(1, 1, 1, 3, 1001, par, 0, P, P, P, 1, 2, 1.0, 0, 1.0, 0, 0,
                                     1, 4, 128, P, P, _cache(), P, P, P, P, P, P, 1 << 20,
                                     None) == sv.SV_ERR_UNSUPPORTED
    # a bad commit argument (missing tree V) is reported as by sv_commit_kv
    assert lib.sv_accept_tree_commit(1, 1, 1, 3, 1000, par, 0, P, P, P, 1, 2, 1.0, 0, 1.0, 0, 0,
                                     1, 4, 128, P, None, _cache(), P, P, P, P, P, P, 1 << 20,
                                     None) == sv.SV_ERR_INVALID_ARG
    assert "v_tree" in lib.sv_last_error().decode()
    # rows must be whole 16-byte vectors
    assert lib.sv_accept_chain_commit(1, 1, 1, 2, 1000, P, P, 1, P, 1.0, 0, 1.0, 0, 0,
                                      1, 1, 3, P, P, _cache(), P, P, P, P, P, 1 << 20,
                                      None) == sv.SV_ERR_UNSUPPORTED


def test_tree_recursive_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    par = (ctypes.c_int32 * 3)(-1, 0, 0)
    bad = (ctypes.c_int32 * 3)(-1, 2, 0)  # a parent after its child

    def call(parent=par, V=1000, q=P, Dq=1, T=1.0, top_k=0, top_p=1.0, ws=1 << 20):
        return lib.sv_accept_tree_recursive(1, 2, 3, V, parent, 0, P, P, q, 1, Dq, T, top_k, top_p,
                                            0, 0, P, P, P, P, P, P, ws, None)
    # greedy (temperature 0) has no sibling residuals: unsupported here
    assert call(T=0.0) == sv.SV_ERR_UNSUPPORTED
    assert "temperature" in lib.sv_last_error().decode()
    assert call(parent=bad) == sv.SV_ERR_INVALID_ARG
    assert call(V=1001) == sv.SV_ERR_UNSUPPORTED
    assert call(q=None) == sv.SV_ERR_INVALID_ARG
    assert call(Dq=0) == sv.SV_ERR_INVALID_ARG      # q rows must cover the tree depth
    assert call(top_p=0.9) == sv.SV_ERR_UNSUPPORTED  # top-p needs top-k
    assert call(ws=16) == sv.SV_ERR_WORKSPACE


def test_ngram_draft_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    # n-gram sizes out of order or past the maximum, gamma out of range, null pointers
    assert lib.sv_ngram_draft(2, 64, P, P, 1, 2, 4, P, P, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_ngram_draft(2, 64, P, P, 33, 1, 4, P, P, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_ngram_draft(2, 64, P, P, 3, 0, 4, P, P, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_ngram_draft(2, 64, P, P, 3, 1, 64, P, P, None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_ngram_draft(2, 64, None, P, 3, 1, 4, P, P, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_ngram_draft(2, 0, P, P, 3, 1, 4, P, P, None) == sv.SV_ERR_INVALID_ARG


def test_binding_requires_cuda_tensors(lib):
    import torch
    with pytest.raises(TypeError):
        sv.sv_accept_chain(sv.GREEDY, torch.zeros(1, 2, 8), None, sv.Q_LOGITS,
                           torch.zeros(1, 1, dtype=torch.int32))


def test_per_sequence_tree_argument_is_checked_before_launch(lib):
    """parent_stride: 0 = a host tree shared by the batch; >= N = one device row per
    sequence.  A stride between 1 and N-1, a NULL or misaligned row pointer are rejected."""
    P = ctypes.c_void_p(16)
    rows = ctypes.c_void_p(4096)  # a device address the host never reads
    def attn(parent, stride):
        return lib.sv_tree_attention(1, 2, 3, 4, 4, 128, P, P, P, _cache(), parent, stride, 0.1, P,
                                     P, 1 << 20, None)
    assert attn(rows, 2) == sv.SV_ERR_INVALID_ARG
    assert "parent_stride" in lib.sv_last_error().decode()
    assert attn(None, 3) == sv.SV_ERR_INVALID_ARG
    assert attn(ctypes.c_void_p(4098), 3) == sv.SV_ERR_INVALID_ARG

    def accept(parent, stride, Dq=2):
        return lib.sv_accept_tree(1, 1, 2, 3, 1000, parent, stride, P, P, P, 1, Dq, 1.0, 0, 1.0, 0,
                                  0, P, P, P, P, P, P, 1 << 20, None)
    assert accept(rows, -1) == sv.SV_ERR_INVALID_ARG
    assert accept(rows, 1) == sv.SV_ERR_INVALID_ARG
    assert accept(rows, 3, Dq=0) == sv.SV_ERR_INVALID_ARG  # exact mode needs q rows


def test_lm_head_rejects_before_launch(lib):
    P = ctypes.c_void_p(16)
    # hidden size not a multiple of 8, V not a multiple of 8, NULL or misaligned operands
    assert lib.sv_lm_head(4, 100, 1000, P, P, P, None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_lm_head(4, 128, 1001, P, P, P, None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_lm_head(4, 128, 1000, None, P, P, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_lm_head(4, 128, 1000, P, ctypes.c_void_p(24), P, None) == sv.SV_ERR_INVALID_ARG
    # the fused chain call checks the projection and the acceptance arguments, and its
    # workspace (statistics plus the projection's per-tile partials)
    need = lib.sv_accept_lmhead_workspace_size(2, 5, 1000, 4)
    assert need > lib.sv_accept_workspace_size(2, 5, 1000, 4)
    assert lib.sv_accept_chain_lmhead(1, 2, 4, 1000, 100, P, P, P, P, 1, P, 1.0, 0, 1.0, 0, 0,
                                      P, P, P, P, P, need, None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_accept_chain_lmhead(1, 2, 4, 1000, 128, P, P, P, P, 1, P, -1.0, 0, 1.0, 0, 0,
                                      P, P, P, P, P, need, None) == sv.SV_ERR_INVALID_ARG
    assert lib.sv_accept_chain_lmhead(1, 2, 4, 1000, 128, P, P, P, P, 1, P, 1.0, 0, 1.0, 0, 0,
                                      P, P, P, P, P, 16, None) == sv.SV_ERR_WORKSPACE
    par = (ctypes.c_int32 * 3)(-1, 0, 0)
    assert lib.sv_accept_tree_lmhead(1, 2, 3, 1000, 128, P, P, P, par, 0, P, P, 1, 0, 1.0, 0, 1.0,
                                     0, 0, P, P, P, P, P, P, need, None) == sv.SV_ERR_INVALID_ARG


def test_wait_limit_is_settable_and_restored(lib):
    default = sv.sv_get_wait_limit_ns()
    assert default == 2_000_000_000
    sv.sv_set_wait_limit_ns(1234)
    assert sv.sv_get_wait_limit_ns() == 1234
    sv.sv_set_wait_limit_ns(0)  # 0 restores the default
    assert sv.sv_get_wait_limit_ns() == default


def test_empty_batch_needs_no_device(lib):
    """B = 0 sequences (R = 0 rows for the projection): every entry point that launches work
    validates its other arguments and returns SV_OK with NULL tensors and no workspace,
    before any CUDA runtime call (this runs on a machine without a GPU)."""
    par = (ctypes.c_int32 * 3)(-1, 0, 0)
    E, G, BF, QL = sv.EXACT, sv.GREEDY, sv.SV_BF16, sv.Q_LOGITS
    empty_cache = _cache(k=None, v=None, prefix_len=None)
    calls = {
        "sv_tree_attention": lambda: lib.sv_tree_attention(BF, 0, 3, 8, 2, 128, None, None, None,
                                                           empty_cache, par, 0, 0.1, None, None, 0, None),
        "sv_accept_chain": lambda: lib.sv_accept_chain(E, BF, 0, 4, 1000, None, None, QL, None, 1.0, 0,
                                                       1.0, 0, 0, None, None, None, None, None, 0, None),
        "sv_accept_tree": lambda: lib.sv_accept_tree(E, BF, 0, 3, 1000, par, 0, None, None, None, QL, 1,
                                                     1.0, 0, 1.0, 0, 0, None, None, None, None, None,
                                                     None, 0, None),
        "sv_accept_tree_noalloc": lambda: lib.sv_accept_tree_noalloc(
            G, BF, 0, 3, 1000, par, 0, None, None, None, QL, 1, 1.0, 0, 1.0, 0, 0, None, None, None,
            None, None, None),
        "sv_accept_tree_recursive": lambda: lib.sv_accept_tree_recursive(
            BF, 0, 3, 1000, par, 0, None, None, None, QL, 1, 1.0, 0, 1.0, 0, 0, None, None, None, None,
            None, None, 0, None),
        "sv_accept_typical": lambda: lib.sv_accept_typical(BF, 0, 3, 1000, par, 0, None, None, 1.0, 0.3,
                                                           0.09, None, None, None, None, None, None, 0,
                                                           None),
        "sv_commit_kv": lambda: lib.sv_commit_kv(BF, 0, 3, 2, 128, None, None, None, 2, None,
                                                 empty_cache, None),
        "sv_accept_tree_commit": lambda: lib.sv_accept_tree_commit(
            E, BF, 0, 3, 1000, par, 0, None, None, None, QL, 1, 1.0, 0, 1.0, 0, 0, BF, 2, 128, None, None,
            empty_cache, None, None, None, None, None, None, 0, None),
        "sv_accept_chain_commit": lambda: lib.sv_accept_chain_commit(
            E, BF, 0, 4, 1000, None, None, QL, None, 1.0, 0, 1.0, 0, 0, BF, 2, 128, None, None,
            empty_cache, None, None, None, None, None, 0, None),
        "sv_ngram_draft": lambda: lib.sv_ngram_draft(0, 256, None, None, 3, 1, 4, None, None, None),
        "sv_lm_head": lambda: lib.sv_lm_head(0, 128, 1024, None, None, None, None),
        "sv_accept_chain_lmhead": lambda: lib.sv_accept_chain_lmhead(
            E, 0, 4, 1024, 128, None, None, None, None, QL, None, 1.0, 0, 1.0, 0, 0, None, None, None,
            None, None, 0, None),
        "sv_accept_tree_lmhead": lambda: lib.sv_accept_tree_lmhead(
            E, 0, 3, 1024, 128, None, None, None, par, 0, None, None, QL, 1, 1.0, 0, 1.0, 0, 0, None,
            None, None, None, None, None, 0, None),
    }
    for name, call in calls.items():
        assert call() == sv.SV_OK, (name, lib.sv_last_error().decode())
    # the other arguments are still checked: a bad V with B = 0 is refused
    assert lib.sv_accept_chain(E, BF, 0, 4, 1001, None, None, QL, None, 1.0, 0, 1.0, 0, 0, None, None,
                               None, None, None, 0, None) == sv.SV_ERR_UNSUPPORTED
    assert lib.sv_ngram_draft(0, 256, None, None, 3, 1, 0, None, None, None) == sv.SV_ERR_UNSUPPORTED

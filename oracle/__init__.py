"""CPU oracle for the speculative-decoding verify step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The product
path (``speculative_decoding_verify_sv_gb300``) never imports it and has no CPU
fallback.  The oracle shares no code with the CUDA path; inputs are torch CPU
tensors (or numpy arrays) holding the exact bits the GPU sees.

Every function follows oracle.c, whose header cites the page sections it restates.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
GREEDY, EXACT = 0, 1
Q_PROBS_F32, Q_LOGITS, Q_DRAFT_ONEHOT = 0, 1, 2
SAMPLE_TIE = 65536  # weight of a sample-class near tie in the packed near-tie word


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so (host code only)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            U64 = ctypes.c_uint64
            Dbl = ctypes.c_double
            lib.orc_philox4x32_10.argtypes = [P, P, P]
            lib.orc_uniforms.argtypes = [U64, U64, ctypes.c_uint32, I, I, P, P]
            lib.orc_check_tree.argtypes = [I, P]
            lib.orc_check_tree.restype = I
            lib.orc_tree_mask.argtypes = [I, P, P]
            lib.orc_tree_attention.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, I, I, I,
                                               P, I, Dbl, I, I, P]
            lib.orc_accept_tree.argtypes = [I, I, I, I, I, P, I, P, P, P, I, I, Dbl, I, Dbl, U64,
                                            U64, P, P, P, P, P, P, P, P]
            lib.orc_accept_tree.restype = I
            lib.orc_accept_chain.argtypes = [I, I, I, I, I, P, P, I, P, Dbl, I, Dbl, U64, U64,
                                             P, P, P, P, P]
            lib.orc_accept_chain.restype = I
            lib.orc_commit_kv.argtypes = [I, I, I, I, I, P, P, P, I, P, P, P, P, P, I, I, I]
            lib.orc_ngram_draft.argtypes = [I, I, P, P, I, I, I, P, P]
            lib.orc_accept_tree_recursive.argtypes = [I, I, I, I, P, I, P, P, P, I, I, Dbl, I,
                                                      Dbl, U64, U64, P, P, P, P, P, P]
            lib.orc_accept_tree_recursive.restype = I
            lib.orc_lm_head.argtypes = [I, I, I, P, I, P, I, P]
            lib.orc_accept_typical.argtypes = [I, I, I, I, P, I, P, P, Dbl, Dbl, Dbl, P, P, P, P, P,
                                               P]
            lib.orc_accept_typical.restype = I
            lib.orc_set_threads.argtypes = [I]
            lib.orc_get_threads.restype = I
            _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


# ----------------------------------------------------------------- marshalling

def _cpu(t):
    """A contiguous CPU tensor (keeps dtype and bits)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(t))
    return t.detach().to("cpu").contiguous()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float64:
        return F64  # logits computed by lm_head
    raise TypeError(f"oracle supports float32, bfloat16 and float64, got {t.dtype}")


def _i32(x):
    return _cpu(torch.as_tensor(x, dtype=torch.int32))


def _parents(parent, B):
    """(int32 tensor, stride, N, per-sequence?) of a tree argument: one parent list [N]
    shared by the batch, or [B, N] with sequence b's tree in row b."""
    par = _i32(parent)
    if par.dim() == 2:
        if par.shape[0] != B:
            raise ValueError(f"per-sequence parents must have B = {B} rows")
        return par, par.shape[1], par.shape[1], True
    return par, 0, par.numel(), False


# ------------------------------------------------------------------- Philox

def philox4x32_10(counter, key):
    """Raw Philox4x32-10 block: counter (4 x u32), key (2 x u32) -> 4 x u32."""
    c = np.asarray(counter, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(c.ctypes.data_as(ctypes.c_void_p), k.ctypes.data_as(ctypes.c_void_p),
                              out.ctypes.data_as(ctypes.c_void_p))
    return out


def uniforms(seed: int, round_: int, b: int, c: int, domain: int = 0):
    """(u_acc, u_smp) of sequence b, node c."""
    ua, us = ctypes.c_double(), ctypes.c_double()
    _load().orc_uniforms(seed, round_, domain, b, c, ctypes.byref(ua), ctypes.byref(us))
    return ua.value, us.value


# --------------------------------------------------------------------- trees

def check_tree(parent) -> bool:
    p = _i32(parent)
    return _load().orc_check_tree(p.numel(), _ptr(p)) == 0


def tree_mask(parent) -> np.ndarray:
    """[N,N] uint8: row n marks the nodes on n's root path."""
    p = _i32(parent)
    n = p.numel()
    m = np.zeros((n, n), dtype=np.uint8)
    _load().orc_tree_mask(n, _ptr(p), m.ctypes.data_as(ctypes.c_void_p))
    return m


# ----------------------------------------------------------------- attention

def tree_attention(q, k_tree, v_tree, cache_k, cache_v, prefix_len, parent, scale=None,
                   block_table=None, block_size=16, b_range=None) -> torch.Tensor:
    """Tree attention by definition; returns float64 [nb,N,Hq,D] for b in b_range.

    Contiguous cache [B,Lmax,Hkv,D] when block_table is None, else a paged pool
    [num_blocks,block_size,Hkv,D] addressed by block_table [B,max_blocks].  parent: one
    tree [N] for the batch, or [B,N] with one tree per sequence."""
    q, k_tree, v_tree = _cpu(q), _cpu(k_tree), _cpu(v_tree)
    cache_k, cache_v = _cpu(cache_k), _cpu(cache_v)
    dt = _dtype_code(q)
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    pl = _i32(prefix_len)
    par, pstride, _, _ = _parents(parent, B)
    if block_table is None:
        bt, max_blocks, Lmax = None, 0, cache_k.shape[1]
    else:
        bt = _i32(block_table)
        max_blocks, Lmax = bt.shape[1], 0
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    b0, b1 = (0, B) if b_range is None else b_range
    out = torch.zeros((b1 - b0, N, Hq, D), dtype=torch.float64)
    _load().orc_tree_attention(dt, B, N, Hq, Hkv, D, _ptr(q), _ptr(k_tree), _ptr(v_tree),
                               _ptr(cache_k), _ptr(cache_v), _ptr(pl), _ptr(bt), max_blocks,
                               block_size, Lmax, _ptr(par), pstride, float(scale), b0, b1, _ptr(out))
    return out


# ---------------------------------------------------------------- acceptance

def _q_args(q, q_kind):
    if q is None or q_kind == Q_DRAFT_ONEHOT:
        return None, 0
    q = _cpu(q)
    if q_kind == Q_PROBS_F32 and q.dtype != torch.float32:
        raise TypeError("q given as probabilities must be float32")
    return q, q.shape[1]


def accept_tree(mode, target_logits, q, q_kind, parent, node_tokens, temperature=1.0,
                top_k=0, seed=0, round_=0, top_p=1.0):
    """Tree acceptance; returns a dict of CPU tensors (see oracle.c).  top_p < 1 keeps
    the nucleus of the top-k distribution (needs 0 < top_k < V); top_p is taken as the
    float32 value the library's interface carries, so that both sides cut at the same
    threshold."""
    tl = _cpu(target_logits)
    dt = _dtype_code(tl)
    B, N, V = tl.shape
    par, pstride, _, per_seq = _parents(parent, B)
    toks = _i32(node_tokens)
    qq, Dq = _q_args(q, q_kind)
    W = N if per_seq else max(_depths(par.tolist())) + 1
    out = {
        "path_nodes": torch.full((B, W), -1, dtype=torch.int32),
        "tokens": torch.full((B, W), -1, dtype=torch.int32),
        "num_emitted": torch.zeros(B, dtype=torch.int32),
        "num_accepted": torch.zeros(B, dtype=torch.int32),
        "near_ties": torch.zeros(B, dtype=torch.int32),
        "acc": torch.zeros((B, N), dtype=torch.uint8),
        "ratio": torch.zeros((B, N), dtype=torch.float64),
        "flags": torch.zeros(B, dtype=torch.int32),
    }
    rc = _load().orc_accept_tree(
        mode, dt, B, N, V, _ptr(par), pstride, _ptr(toks), _ptr(tl), _ptr(qq), q_kind, Dq,
        float(temperature), int(top_k), float(np.float32(top_p)), int(seed), int(round_), _ptr(out["path_nodes"]),
        _ptr(out["tokens"]), _ptr(out["num_emitted"]), _ptr(out["num_accepted"]),
        _ptr(out["near_ties"]), _ptr(out["acc"]), _ptr(out["ratio"]), _ptr(out["flags"]))
    if rc != 0:
        raise ValueError(f"oracle accept_tree rejected its arguments (code {rc})")
    return out


def accept_chain(mode, target_logits, q, q_kind, draft_tokens, temperature=1.0, top_k=0,
                 seed=0, round_=0, top_p=1.0):
    """Chain acceptance as the left-to-right procedure; returns a dict of CPU tensors.
    top_p < 1 keeps the nucleus of the top-k distribution (needs 0 < top_k < V).  A draft
    of -1 ends a sequence's chain; q_kind Q_DRAFT_ONEHOT takes q = e_x at each draft (q
    may be None).  near_ties packs decision ties (low 16 bits) and sample ties (times
    SAMPLE_TIE)."""
    tl = _cpu(target_logits)
    dt = _dtype_code(tl)
    B, W, V = tl.shape
    gamma = W - 1
    toks = _i32(draft_tokens)
    qq, _ = _q_args(q, q_kind)
    out = {
        "tokens": torch.full((B, W), -1, dtype=torch.int32),
        "num_emitted": torch.zeros(B, dtype=torch.int32),
        "num_accepted": torch.zeros(B, dtype=torch.int32),
        "near_ties": torch.zeros(B, dtype=torch.int32),
        "flags": torch.zeros(B, dtype=torch.int32),
    }
    rc = _load().orc_accept_chain(mode, dt, B, gamma, V, _ptr(tl), _ptr(qq), q_kind, _ptr(toks),
                                  float(temperature), int(top_k), float(np.float32(top_p)), int(seed),
                                  int(round_), _ptr(out["tokens"]), _ptr(out["num_emitted"]),
                                  _ptr(out["num_accepted"]), _ptr(out["near_ties"]),
                                  _ptr(out["flags"]))
    if rc != 0:
        raise ValueError(f"oracle accept_chain rejected its arguments (code {rc})")
    return out


def _depths(parent):
    d = []
    for i, p in enumerate(parent):
        d.append(0 if p < 0 else d[p] + 1)
    return d


# ------------------------------------------------------------------- commit

def commit_kv(k_tree, v_tree, path_nodes, num_accepted, cache_k, cache_v, prefix_len,
              block_table=None, block_size=16):
    """Returns (cache_k, cache_v, prefix_len) after the commit; inputs are not modified."""
    k_tree, v_tree = _cpu(k_tree), _cpu(v_tree)
    ck, cv = _cpu(cache_k).clone(), _cpu(cache_v).clone()
    pl = _i32(prefix_len).clone()
    pn = _i32(path_nodes)
    na = _i32(num_accepted)
    dt = _dtype_code(k_tree)
    B, N, Hkv, D = k_tree.shape
    if block_table is None:
        bt, max_blocks, Lmax = None, 0, ck.shape[1]
    else:
        bt = _i32(block_table)
        max_blocks, Lmax = bt.shape[1], 0
    _load().orc_commit_kv(dt, B, N, Hkv, D, _ptr(k_tree), _ptr(v_tree), _ptr(pn), pn.shape[1],
                          _ptr(na), _ptr(ck), _ptr(cv), _ptr(pl), _ptr(bt), max_blocks,
                          block_size, Lmax)
    return ck, cv, pl


# ------------------------------------------------------------ n-gram drafts

def ngram_draft(history, length, max_n=3, min_n=1, gamma=4):
    """Prompt-lookup drafts (see oracle.c): returns (drafts [B,gamma] int32, num [B])."""
    h = _i32(history)
    ln = _i32(length)
    B, Lmax = h.shape
    drafts = torch.full((B, gamma), -1, dtype=torch.int32)
    num = torch.zeros(B, dtype=torch.int32)
    _load().orc_ngram_draft(B, Lmax, _ptr(h), _ptr(ln), int(max_n), int(min_n), int(gamma),
                            _ptr(drafts), _ptr(num))
    return drafts, num


def accept_tree_recursive(target_logits, q, q_kind, parent, node_tokens, temperature=1.0,
                          top_k=0, seed=0, round_=0, top_p=1.0):
    """Exact tree acceptance with siblings tried in rank order (see oracle.c); returns a
    dict of CPU tensors like accept_tree (no per-node decision outputs)."""
    tl = _cpu(target_logits)
    dt = _dtype_code(tl)
    B, N, V = tl.shape
    par, pstride, _, per_seq = _parents(parent, B)
    toks = _i32(node_tokens)
    qq, Dq = _q_args(q, q_kind)
    W = N if per_seq else max(_depths(par.tolist())) + 1
    out = {
        "path_nodes": torch.full((B, W), -1, dtype=torch.int32),
        "tokens": torch.full((B, W), -1, dtype=torch.int32),
        "num_emitted": torch.zeros(B, dtype=torch.int32),
        "num_accepted": torch.zeros(B, dtype=torch.int32),
        "near_ties": torch.zeros(B, dtype=torch.int32),
        "flags": torch.zeros(B, dtype=torch.int32),
    }
    rc = _load().orc_accept_tree_recursive(
        dt, B, N, V, _ptr(par), pstride, _ptr(toks), _ptr(tl), _ptr(qq), q_kind, Dq, float(temperature),
        int(top_k), float(np.float32(top_p)), int(seed), int(round_), _ptr(out["path_nodes"]),
        _ptr(out["tokens"]), _ptr(out["num_emitted"]), _ptr(out["num_accepted"]),
        _ptr(out["near_ties"]), _ptr(out["flags"]))
    if rc != 0:
        raise ValueError(f"oracle accept_tree_recursive rejected its arguments (code {rc})")
    return out


def accept_typical(target_logits, parent, node_tokens, temperature=1.0, epsilon=0.3,
                   delta=0.09):
    """Typical acceptance (see oracle.c, orc_accept_typical): node c is accepted iff
    p_parent(x_c) > min(epsilon, delta * exp(-H(p_parent))); the token after the kept path is
    the target's argmax.  parent [N] or [B, N]; returns a dict of CPU tensors, with the
    entropy (nats) of every row under "entropy"."""
    tl = _cpu(target_logits)
    dt = _dtype_code(tl)
    B, N, V = tl.shape
    par, pstride, _, per_seq = _parents(parent, B)
    toks = _i32(node_tokens)
    W = N if per_seq else max(_depths(par.tolist())) + 1
    out = {
        "path_nodes": torch.full((B, W), -1, dtype=torch.int32),
        "tokens": torch.full((B, W), -1, dtype=torch.int32),
        "num_emitted": torch.zeros(B, dtype=torch.int32),
        "num_accepted": torch.zeros(B, dtype=torch.int32),
        "near_ties": torch.zeros(B, dtype=torch.int32),
        "entropy": torch.zeros((B, N), dtype=torch.float64),
    }
    rc = _load().orc_accept_typical(
        dt, B, N, V, _ptr(par), pstride, _ptr(toks), _ptr(tl), float(temperature),
        float(np.float32(epsilon)), float(np.float32(delta)), _ptr(out["path_nodes"]),
        _ptr(out["tokens"]), _ptr(out["num_emitted"]), _ptr(out["num_accepted"]),
        _ptr(out["near_ties"]), _ptr(out["entropy"]))
    if rc != 0:
        raise ValueError(f"oracle accept_typical rejected its arguments (code {rc})")
    return out


def lm_head(hidden, weight):
    """Target logits from hidden states: z[..., v] = sum_k hidden[..., k] * weight[v, k] in
    double (see oracle.c, orc_lm_head).  hidden [..., Dm], weight [V, Dm], float32 or
    bfloat16; returns float64 [..., V], which accept_chain / accept_tree /
    accept_tree_recursive take as target logits."""
    h = _cpu(hidden)
    w = _cpu(weight)
    if h.dtype == torch.float64 or w.dtype == torch.float64:
        raise TypeError("hidden and weight are float32 or bfloat16")
    Dm = h.shape[-1]
    V = w.shape[0]
    if w.dim() != 2 or w.shape[1] != Dm:
        raise ValueError(f"weight must be [V, {Dm}], got {tuple(w.shape)}")
    rows = h.numel() // Dm if Dm > 0 else 0
    out = torch.zeros(tuple(h.shape[:-1]) + (V,), dtype=torch.float64)
    _load().orc_lm_head(rows, Dm, V, _ptr(h), _dtype_code(h), _ptr(w), _dtype_code(w), _ptr(out))
    return out

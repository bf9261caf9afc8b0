"""GB300-native verify step of speculative decoding: tree attention, token acceptance
and KV commit, as a C ABI (``include/sv.h``, ``libsv.so``) with this thin binding.

The binding only marshals arguments: it takes torch CUDA tensors, checks their
shapes/dtypes against the ABI's layouts, and passes raw pointers and the current
CUDA stream to ``libsv.so``.  Every step of the computation runs in the library's
kernels; there is no CPU fallback: if the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

__all__ = [
    "SVError", "KVCache", "library_path", "load_library", "sv_tree_attention",
    "sv_tree_attention_workspace_size", "sv_tree_attention_path", "sv_accept_chain", "sv_accept_tree",
    "sv_accept_workspace_size", "sv_accept_tree_noalloc", "sv_commit_kv", "sv_accept_tree_commit",
    "sv_accept_chain_commit", "sv_accept_tree_recursive", "sv_ngram_draft", "sv_tree_prepare", "sv_read_device_status",
    "sv_lm_head", "sv_accept_lmhead_workspace_size", "sv_accept_chain_lmhead", "sv_accept_tree_lmhead",
    "sv_accept_typical", "sv_set_wait_limit_ns", "sv_get_wait_limit_ns", "sv_inject_launch_failures",
    "sv_version", "sv_kernel_launches", "GREEDY", "EXACT", "Q_PROBS_F32", "Q_LOGITS", "Q_DRAFT_ONEHOT", "SV_MAX_TREE_NODES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libsv.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_WORKSPACE, SV_ERR_CUDA = 0, 1, 2, 3, 4
SV_F32, SV_BF16 = 0, 1
GREEDY, EXACT = 0, 1
Q_PROBS_F32, Q_LOGITS, Q_DRAFT_ONEHOT = 0, 1, 2  # q as probabilities, draft logits, one-hot drafts
SV_MAX_TREE_NODES = 64
SV_DEV_BAD_TOKEN, SV_DEV_BAD_BLOCK, SV_DEV_BAD_PREFIX, SV_DEV_ZERO_DRAFT_PROB = 1, 2, 4, 8
SV_DEV_TIMEOUT, SV_DEV_LAYOUT, SV_DEV_BAD_TREE = 0x10, 0x20, 0x40

_STATUS_NAMES = {1: "SV_ERR_INVALID_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_WORKSPACE",
                 4: "SV_ERR_CUDA"}


class SVError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


class _KVCacheC(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("Lmax", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libsv.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libsv.so is not built ({_LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
        lib.sv_tree_attention.argtypes = [I, I, I, I, I, I, P, P, P, _KVCacheC, P, I, F, P, P, SZ, P]
        lib.sv_tree_attention_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.sv_tree_attention_path.argtypes = [I, I, I, I, I, I]
        lib.sv_tree_attention_path.restype = I
        lib.sv_tree_attention_workspace_size.restype = SZ
        lib.sv_accept_chain.argtypes = [I, I, I, I, I, P, P, I, P, F, I, F, U64, U64, P, P, P, P, P,
                                        SZ, P]
        lib.sv_accept_tree.argtypes = [I, I, I, I, I, P, I, P, P, P, I, I, F, I, F, U64, U64, P, P, P, P,
                                       P, P, SZ, P]
        lib.sv_accept_tree_recursive.argtypes = [I, I, I, I, P, I, P, P, P, I, I, F, I, F, U64, U64,
                                                 P, P, P, P, P, P, SZ, P]
        lib.sv_accept_tree_noalloc.argtypes = [I, I, I, I, I, P, I, P, P, P, I, I, F, I, F, U64, U64, P,
                                               P, P, P, P, P]
        lib.sv_accept_workspace_size.argtypes = [I, I, I, I]
        lib.sv_accept_workspace_size.restype = SZ
        lib.sv_commit_kv.argtypes = [I, I, I, I, I, P, P, P, I, P, _KVCacheC, P]
        lib.sv_accept_tree_commit.argtypes = [I, I, I, I, I, P, I, P, P, P, I, I, F, I, F, U64, U64,
                                              I, I, I, P, P, _KVCacheC, P, P, P, P, P, P, SZ, P]
        lib.sv_accept_chain_commit.argtypes = [I, I, I, I, I, P, P, I, P, F, I, F, U64, U64,
                                               I, I, I, P, P, _KVCacheC, P, P, P, P, P, SZ, P]
        lib.sv_lm_head.argtypes = [I, I, I, P, P, P, P]
        lib.sv_set_wait_limit_ns.argtypes = [U64]
        lib.sv_set_wait_limit_ns.restype = None
        lib.sv_get_wait_limit_ns.restype = U64
        lib.sv_inject_launch_failures.argtypes = [I]
        lib.sv_inject_launch_failures.restype = None
        lib.sv_accept_typical.argtypes = [I, I, I, I, P, I, P, P, F, F, F, P, P, P, P, P, P, SZ, P]
        lib.sv_accept_lmhead_workspace_size.argtypes = [I, I, I, I]
        lib.sv_accept_lmhead_workspace_size.restype = SZ
        lib.sv_accept_chain_lmhead.argtypes = [I, I, I, I, I, P, P, P, P, I, P, F, I, F, U64, U64,
                                               P, P, P, P, P, SZ, P]
        lib.sv_accept_tree_lmhead.argtypes = [I, I, I, I, I, P, P, P, P, I, P, P, I, I, F, I, F,
                                              U64, U64, P, P, P, P, P, P, SZ, P]
        lib.sv_tree_prepare.argtypes = [I, P, P, P]
        lib.sv_read_device_status.argtypes = [P, P]
        lib.sv_ngram_draft.argtypes = [I, I, P, P, I, I, I, P, P, P]
        lib.sv_last_error.restype = ctypes.c_char_p
        lib.sv_version.restype = ctypes.c_char_p
        lib.sv_kernel_launches.restype = ctypes.c_uint64
        for fn in ("sv_tree_attention", "sv_accept_chain", "sv_accept_tree", "sv_commit_kv",
                   "sv_tree_prepare", "sv_read_device_status", "sv_accept_tree_noalloc",
                   "sv_accept_tree_commit", "sv_accept_chain_commit", "sv_ngram_draft",
                   "sv_accept_tree_recursive"):
            getattr(lib, fn).restype = ctypes.c_int32
        _lib = lib
        return lib


def _check(code: int):
    if code != SV_OK:
        raise SVError(code, load_library().sv_last_error().decode())


def sv_version() -> str:
    return load_library().sv_version().decode()


def sv_kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().sv_kernel_launches())


# ------------------------------------------------------------------ marshalling

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _parent_arr(parent: Sequence[int]):
    arr = (ctypes.c_int32 * len(parent))(*[int(x) for x in parent])
    return arr, len(parent)


def _tree_arg(parent, B: int, N: int):
    """The (pointer, parent_stride, output width) of a tree argument: a host sequence [N]
    shared by the batch (stride 0, width depth + 1), or a CUDA int32 tensor [B, S] (S >= N)
    with one tree per sequence (stride S, width N)."""
    if isinstance(parent, torch.Tensor) and parent.is_cuda:
        if parent.dtype != torch.int32 or parent.dim() != 2 or parent.shape[0] != B:
            raise ValueError(f"per-sequence parents must be a CUDA int32 tensor [B={B}, >= N]")
        if parent.stride(1) != 1 or parent.shape[1] < N or parent.stride(0) < N:
            raise ValueError(f"per-sequence parents need contiguous rows of at least N={N}")
        return ctypes.c_void_p(parent.data_ptr()), int(parent.stride(0)), N
    if isinstance(parent, torch.Tensor):
        parent = parent.tolist()
    par, n = _parent_arr(parent)
    if n != N:
        raise ValueError(f"parent has {n} entries, the tree has {N} rows")
    return par, 0, _tree_depth(parent) + 1


@dataclass
class KVCache:
    """KV prefix cache of one layer: contiguous k, v [B,Lmax,Hkv,D], or a paged pool
    [num_blocks,block_size,Hkv,D] with block_table [B,max_blocks]; prefix_len [B] int32."""
    k: torch.Tensor
    v: torch.Tensor
    prefix_len: torch.Tensor
    block_table: Optional[torch.Tensor] = None
    block_size: int = 16

    def c_struct(self) -> _KVCacheC:
        _dev(self.k, "cache.k")
        _dev(self.v, "cache.v", self.k.dtype, self.k.shape)
        _dev(self.prefix_len, "cache.prefix_len", torch.int32)
        c = _KVCacheC()
        c.k, c.v, c.prefix_len = self.k.data_ptr(), self.v.data_ptr(), self.prefix_len.data_ptr()
        if self.block_table is None:
            c.block_table = None
            c.Lmax = self.k.shape[1]
            c.block_size = c.max_blocks = c.num_blocks = 0
        else:
            _dev(self.block_table, "cache.block_table", torch.int32)
            c.block_table = self.block_table.data_ptr()
            c.Lmax = 0
            c.block_size = int(self.block_size)
            c.max_blocks = self.block_table.shape[1]
            c.num_blocks = self.k.shape[0]
        return c

    @property
    def max_prefix(self) -> int:
        if self.block_table is None:
            return self.k.shape[1]
        return self.block_table.shape[1] * int(self.block_size)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor], zero: bool = False):
    if nbytes == 0:
        return workspace, 0
    if workspace is None:
        workspace = (torch.zeros if zero else torch.empty)(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace has {workspace.numel()} bytes, need {nbytes}")
    return workspace, workspace.numel() * workspace.element_size()


# ------------------------------------------------------------------- attention

def sv_tree_attention_workspace_size(dtype, B, N, Hq, Hkv, D, max_prefix) -> int:
    dt = SV_BF16 if dtype == torch.bfloat16 else SV_F32
    return int(load_library().sv_tree_attention_workspace_size(dt, B, N, Hq, Hkv, D, max_prefix))


def sv_tree_attention_path(dtype, N, Hq, Hkv, D, block_size=0) -> int:
    """1: the tensor-core kernel serves these sizes; 0: the general kernel; -1: rejected."""
    dt = SV_BF16 if dtype == torch.bfloat16 else SV_F32
    return int(load_library().sv_tree_attention_path(dt, N, Hq, Hkv, D, block_size))


def sv_tree_attention(q, k_tree, v_tree, cache: KVCache, parent, scale, out=None,
                      workspace=None, stream=None) -> torch.Tensor:
    """Tree attention; q [B,N,Hq,D], k_tree/v_tree [B,N,Hkv,D]; returns out [B,N,Hq,D]."""
    lib = load_library()
    _dev(q, "q", (torch.bfloat16, torch.float32))
    B, N, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    _dev(k_tree, "k_tree", q.dtype, (B, N, Hkv, D))
    _dev(v_tree, "v_tree", q.dtype, (B, N, Hkv, D))
    if cache.k.dtype != q.dtype:
        raise TypeError("cache dtype differs from q")
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype, q.shape)
    cs = cache.c_struct()
    ws_need = sv_tree_attention_workspace_size(q.dtype, B, N, Hq, Hkv, D, cache.max_prefix)
    # a workspace passed in must have been zero-filled before its first use
    workspace, ws_bytes = _workspace(ws_need, q.device, workspace, zero=True)
    par, pstride, _ = _tree_arg(parent, B, N)
    _check(lib.sv_tree_attention(_dt(q), B, N, Hq, Hkv, D, _ptr(q), _ptr(k_tree), _ptr(v_tree),
                                 cs, par, pstride, float(scale), _ptr(out), _ptr(workspace), ws_bytes,
                                 _stream(stream)))
    return out


# ------------------------------------------------------------------ acceptance

def sv_accept_workspace_size(B, N, V, Dq) -> int:
    return int(load_library().sv_accept_workspace_size(B, N, V, Dq))


def _accept_outputs(B, W, device, outs):
    if outs is None:
        outs = {}
    i32 = dict(dtype=torch.int32, device=device)
    outs.setdefault("tokens", torch.empty((B, W), **i32))
    outs.setdefault("num_emitted", torch.empty(B, **i32))
    outs.setdefault("num_accepted", torch.empty(B, **i32))
    outs.setdefault("near_ties", torch.empty(B, **i32))
    return outs


def sv_accept_chain(mode, target_logits, q, q_kind, draft_tokens, temperature=1.0, top_k=0,
                    seed=0, round_=0, outs=None, workspace=None, stream=None, top_p=1.0) -> dict:
    """Chain acceptance; target_logits [B,gamma+1,V], q [B,gamma,V] (or None in greedy
    mode or with q_kind Q_DRAFT_ONEHOT), draft_tokens [B,gamma] int32 (-1 ends a sequence's
    drafts).  Returns dict of device tensors."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, W, V = target_logits.shape
    gamma = W - 1
    _dev(draft_tokens, "draft_tokens", torch.int32, (B, gamma))
    if q_kind == Q_DRAFT_ONEHOT:
        q = None  # one-hot drafts have no q rows
    if q is not None:
        if q_kind == Q_LOGITS:
            _dev(q, "q", target_logits.dtype, (B, gamma, V))
        else:
            _dev(q, "q", torch.float32, (B, gamma, V))
    outs = _accept_outputs(B, W, target_logits.device, outs)
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, W, V, gamma), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_chain(mode, _dt(target_logits), B, gamma, V, _ptr(target_logits), _ptr(q),
                               q_kind, _ptr(draft_tokens), float(temperature), int(top_k),
                               float(top_p), int(seed), int(round_), _ptr(outs["tokens"]),
                               _ptr(outs["num_emitted"]), _ptr(outs["num_accepted"]),
                               _ptr(outs["near_ties"]), _ptr(workspace), ws_bytes,
                               _stream(stream)))
    return outs


def _tree_depth(parent) -> int:
    d = []
    for p in parent:
        d.append(0 if p < 0 else d[p] + 1)
    return max(d)


def sv_accept_tree(mode, target_logits, q, q_kind, parent, node_tokens, temperature=1.0,
                   top_k=0, seed=0, round_=0, outs=None, workspace=None, stream=None, top_p=1.0) -> dict:
    """Tree acceptance; target_logits [B,N,V], q [B,Dq,V] (row d-1 = depth d),
    node_tokens [B,N] int32, parent (host sequence, BFS order).  Returns dict."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, N, V = target_logits.shape
    _dev(node_tokens, "node_tokens", torch.int32, (B, N))
    Dq = 0
    if q is not None:
        Dq = q.shape[1]
        if q_kind == Q_LOGITS:
            _dev(q, "q", target_logits.dtype, (B, Dq, V))
        else:
            _dev(q, "q", torch.float32, (B, Dq, V))
    par, pstride, W = _tree_arg(parent, B, N)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=target_logits.device))
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, N, V, Dq), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_tree(mode, _dt(target_logits), B, N, V, par, pstride, _ptr(node_tokens),
                              _ptr(target_logits), _ptr(q), q_kind, Dq, float(temperature),
                              int(top_k), float(top_p), int(seed), int(round_), _ptr(outs["path_nodes"]),
                              _ptr(outs["tokens"]), _ptr(outs["num_emitted"]),
                              _ptr(outs["num_accepted"]), _ptr(outs["near_ties"]),
                              _ptr(workspace), ws_bytes, _stream(stream)))
    return outs


def sv_accept_tree_recursive(target_logits, q, q_kind, parent, node_tokens, temperature=1.0,
                             top_k=0, top_p=1.0, seed=0, round_=0, outs=None, workspace=None,
                             stream=None) -> dict:
    """Exact tree acceptance with the siblings of a node tried in turn (the residual of a
    rejected child goes to the next); arguments and outputs as sv_accept_tree, exact mode
    only (temperature > 0)."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, N, V = target_logits.shape
    _dev(node_tokens, "node_tokens", torch.int32, (B, N))
    if q is None:
        raise ValueError("q is required (exact mode)")
    Dq = q.shape[1]
    _dev(q, "q", target_logits.dtype if q_kind == Q_LOGITS else torch.float32, (B, Dq, V))
    par, pstride, W = _tree_arg(parent, B, N)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=target_logits.device))
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, N, V, Dq), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_tree_recursive(_dt(target_logits), B, N, V, par, pstride, _ptr(node_tokens),
                                        _ptr(target_logits), _ptr(q), q_kind, Dq,
                                        float(temperature), int(top_k), float(top_p), int(seed),
                                        int(round_), _ptr(outs["path_nodes"]), _ptr(outs["tokens"]),
                                        _ptr(outs["num_emitted"]), _ptr(outs["num_accepted"]),
                                        _ptr(outs["near_ties"]), _ptr(workspace), ws_bytes,
                                        _stream(stream)))
    return outs


def sv_accept_tree_noalloc(mode, target_logits, q, q_kind, parent, node_tokens,
                           temperature=1.0, top_k=0, seed=0, round_=0, outs=None,
                           stream=None, top_p=1.0) -> dict:
    """sv_accept_tree without a workspace, for callers that cannot allocate device
    memory: the library keeps the per-row statistics in a fixed device array.  Calls
    that overlap on the GPU share that array and race; order them on one stream.  The
    output buffers are still the caller's (pass them in ``outs`` to avoid allocation)."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, N, V = target_logits.shape
    _dev(node_tokens, "node_tokens", torch.int32, (B, N))
    Dq = 0
    if q is not None:
        Dq = q.shape[1]
        _dev(q, "q", target_logits.dtype if q_kind == Q_LOGITS else torch.float32, (B, Dq, V))
    par, pstride, W = _tree_arg(parent, B, N)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=target_logits.device))
    _check(lib.sv_accept_tree_noalloc(mode, _dt(target_logits), B, N, V, par, pstride, _ptr(node_tokens),
                                      _ptr(target_logits), _ptr(q), q_kind, Dq, float(temperature),
                                      int(top_k), float(top_p), int(seed), int(round_), _ptr(outs["path_nodes"]),
                                      _ptr(outs["tokens"]), _ptr(outs["num_emitted"]),
                                      _ptr(outs["num_accepted"]), _ptr(outs["near_ties"]),
                                      _stream(stream)))
    return outs


# ---------------------------------------------------------------------- commit

def sv_commit_kv(k_tree, v_tree, path_nodes, num_accepted, cache: KVCache, stream=None) -> None:
    """Copy the accepted path's tree K/V into the cache and advance prefix_len."""
    lib = load_library()
    _dev(k_tree, "k_tree", (torch.bfloat16, torch.float32))
    B, N, Hkv, D = k_tree.shape
    _dev(v_tree, "v_tree", k_tree.dtype, k_tree.shape)
    _dev(path_nodes, "path_nodes", torch.int32)
    _dev(num_accepted, "num_accepted", torch.int32, (B,))
    if path_nodes.shape[0] != B:
        raise ValueError("path_nodes must have B rows")
    _check(lib.sv_commit_kv(_dt(k_tree), B, N, Hkv, D, _ptr(k_tree), _ptr(v_tree),
                            _ptr(path_nodes), path_nodes.shape[1], _ptr(num_accepted),
                            cache.c_struct(), _stream(stream)))


def _kv_args(k_tree, v_tree, cache: KVCache):
    _dev(k_tree, "k_tree", (torch.bfloat16, torch.float32))
    _dev(v_tree, "v_tree", k_tree.dtype, k_tree.shape)
    return _dt(k_tree), k_tree.shape[2], k_tree.shape[3], cache.c_struct()


def sv_accept_chain_commit(mode, target_logits, q, q_kind, draft_tokens, k_tree, v_tree,
                           cache: KVCache, temperature=1.0, top_k=0, seed=0, round_=0,
                           outs=None, workspace=None, stream=None, top_p=1.0) -> dict:
    """sv_accept_chain, then the commit of nodes 0..accepted of k_tree/v_tree
    [B,gamma+1,Hkv,D] into the cache, in the same launches."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, W, V = target_logits.shape
    gamma = W - 1
    _dev(draft_tokens, "draft_tokens", torch.int32, (B, gamma))
    if q_kind == Q_DRAFT_ONEHOT:
        q = None  # one-hot drafts have no q rows
    if q is not None:
        _dev(q, "q", target_logits.dtype if q_kind == Q_LOGITS else torch.float32, (B, gamma, V))
    if k_tree.shape[:2] != (B, W):
        raise ValueError("k_tree must be [B, gamma+1, Hkv, D]")
    kv_dt, Hkv, D, cs = _kv_args(k_tree, v_tree, cache)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, W, V, gamma), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_chain_commit(mode, _dt(target_logits), B, gamma, V, _ptr(target_logits),
                                      _ptr(q), q_kind, _ptr(draft_tokens), float(temperature),
                                      int(top_k), float(top_p), int(seed), int(round_), kv_dt, Hkv, D,
                                      _ptr(k_tree), _ptr(v_tree), cs, _ptr(outs["tokens"]),
                                      _ptr(outs["num_emitted"]), _ptr(outs["num_accepted"]),
                                      _ptr(outs["near_ties"]), _ptr(workspace), ws_bytes,
                                      _stream(stream)))
    return outs


def sv_accept_tree_commit(mode, target_logits, q, q_kind, parent, node_tokens, k_tree, v_tree,
                          cache: KVCache, temperature=1.0, top_k=0, seed=0, round_=0, outs=None,
                          workspace=None, stream=None, top_p=1.0) -> dict:
    """sv_accept_tree, then the commit of the kept path of k_tree/v_tree [B,N,Hkv,D] into
    the cache, in the same launches."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, N, V = target_logits.shape
    _dev(node_tokens, "node_tokens", torch.int32, (B, N))
    Dq = 0
    if q is not None:
        Dq = q.shape[1]
        _dev(q, "q", target_logits.dtype if q_kind == Q_LOGITS else torch.float32, (B, Dq, V))
    if k_tree.shape[:2] != (B, N):
        raise ValueError("k_tree must be [B, N, Hkv, D]")
    kv_dt, Hkv, D, cs = _kv_args(k_tree, v_tree, cache)
    par, pstride, W = _tree_arg(parent, B, N)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=target_logits.device))
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, N, V, Dq), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_tree_commit(mode, _dt(target_logits), B, N, V, par, pstride, _ptr(node_tokens),
                                     _ptr(target_logits), _ptr(q), q_kind, Dq, float(temperature),
                                     int(top_k), float(top_p), int(seed), int(round_), kv_dt, Hkv, D,
                                     _ptr(k_tree), _ptr(v_tree), cs, _ptr(outs["path_nodes"]),
                                     _ptr(outs["tokens"]), _ptr(outs["num_emitted"]),
                                     _ptr(outs["num_accepted"]), _ptr(outs["near_ties"]),
                                     _ptr(workspace), ws_bytes, _stream(stream)))
    return outs


# ------------------------------------------------------------------ tree, status

def sv_tree_prepare(parent):
    """(ancestor bitmasks, depths) of a tree; raises SVError if invalid."""
    lib = load_library()
    par, n = _parent_arr(parent)
    anc = (ctypes.c_uint64 * max(n, 1))()
    dep = (ctypes.c_int32 * max(n, 1))()
    _check(lib.sv_tree_prepare(n, par, anc, dep))
    return list(anc)[:n], list(dep)[:n]


def sv_read_device_status(stream=None) -> int:
    """Sticky device status bits (SV_DEV_*); reading clears them.  Synchronises."""
    lib = load_library()
    v = ctypes.c_uint32(0)
    _check(lib.sv_read_device_status(ctypes.byref(v), _stream(stream)))
    return int(v.value)


def sv_accept_typical(target_logits, parent, node_tokens, temperature=1.0, epsilon=0.3,
                      delta=0.09, outs=None, workspace=None, stream=None) -> dict:
    """Typical acceptance (the Medusa paper's rule): node c is accepted iff
    p_parent(x_c) > min(epsilon, delta * exp(-H(p_parent))); then the target's argmax at the
    kept node.  target_logits [B,N,V], node_tokens [B,N] int32, parent a host sequence [N]
    or a CUDA int32 tensor [B,N].  Returns dict of device tensors."""
    lib = load_library()
    _dev(target_logits, "target_logits", (torch.bfloat16, torch.float32))
    B, N, V = target_logits.shape
    _dev(node_tokens, "node_tokens", torch.int32, (B, N))
    par, pstride, W = _tree_arg(parent, B, N)
    outs = _accept_outputs(B, W, target_logits.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=target_logits.device))
    workspace, ws_bytes = _workspace(sv_accept_workspace_size(B, N, V, 0), target_logits.device,
                                     workspace)
    _check(lib.sv_accept_typical(_dt(target_logits), B, N, V, par, pstride, _ptr(node_tokens),
                                 _ptr(target_logits), float(temperature), float(epsilon),
                                 float(delta), _ptr(outs["path_nodes"]), _ptr(outs["tokens"]),
                                 _ptr(outs["num_emitted"]), _ptr(outs["num_accepted"]),
                                 _ptr(outs["near_ties"]), _ptr(workspace), ws_bytes,
                                 _stream(stream)))
    return outs


def sv_set_wait_limit_ns(ns: int) -> None:
    """Limit of the tensor-core attention kernel's waits for progress (0: the default 2 s)."""
    load_library().sv_set_wait_limit_ns(int(ns))


def sv_get_wait_limit_ns() -> int:
    return int(load_library().sv_get_wait_limit_ns())


def sv_inject_launch_failures(n: int) -> None:
    """Test hook: the library's next n launch requests fail (SV_ERR_CUDA) without
    launching; 0 clears."""
    load_library().sv_inject_launch_failures(int(n))


# ------------------------------------------------------------------- LM head

def sv_lm_head(hidden, weight, out=None, stream=None) -> torch.Tensor:
    """LM-head projection on the tensor cores: hidden [..., Dm] bf16, weight [V, Dm] bf16
    -> logits [..., V] bf16 (fp32 accumulation)."""
    lib = load_library()
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(weight, "weight", torch.bfloat16)
    Dm = hidden.shape[-1]
    V = weight.shape[0]
    if weight.dim() != 2 or weight.shape[1] != Dm:
        raise ValueError(f"weight must be [V, {Dm}]")
    R = hidden.numel() // Dm
    if out is None:
        out = torch.empty(tuple(hidden.shape[:-1]) + (V,), dtype=torch.bfloat16, device=hidden.device)
    _dev(out, "logits", torch.bfloat16, tuple(hidden.shape[:-1]) + (V,))
    _check(lib.sv_lm_head(R, Dm, V, _ptr(hidden), _ptr(weight), _ptr(out), _stream(stream)))
    return out


def sv_accept_lmhead_workspace_size(B, N, V, Dq) -> int:
    return int(load_library().sv_accept_lmhead_workspace_size(B, N, V, Dq))


def _lmhead_args(hidden, weight, B, N):
    _dev(hidden, "hidden", torch.bfloat16)
    _dev(weight, "weight", torch.bfloat16)
    if hidden.dim() != 3 or hidden.shape[:2] != (B, N):
        raise ValueError(f"hidden must be [B={B}, {N}, Dm]")
    Dm = hidden.shape[2]
    if weight.dim() != 2 or weight.shape[1] != Dm:
        raise ValueError(f"weight must be [V, {Dm}]")
    return Dm, weight.shape[0]


def sv_accept_chain_lmhead(mode, hidden, weight, q, q_kind, draft_tokens, temperature=1.0, top_k=0,
                           seed=0, round_=0, top_p=1.0, outs=None, logits=None, workspace=None,
                           stream=None) -> dict:
    """Chain acceptance fused with the LM-head projection of the target rows: hidden
    [B,gamma+1,Dm] bf16, weight [V,Dm] bf16; the target logits [B,gamma+1,V] (bf16) are
    returned under "target_logits" with the acceptance outputs."""
    lib = load_library()
    _dev(draft_tokens, "draft_tokens", torch.int32)
    B, gamma = draft_tokens.shape
    W = gamma + 1
    Dm, V = _lmhead_args(hidden, weight, B, W)
    if q_kind == Q_DRAFT_ONEHOT:
        q = None
    if q is not None:
        _dev(q, "q", torch.bfloat16 if q_kind == Q_LOGITS else torch.float32, (B, gamma, V))
    if logits is None:
        logits = torch.empty((B, W, V), dtype=torch.bfloat16, device=hidden.device)
    _dev(logits, "logits", torch.bfloat16, (B, W, V))
    outs = _accept_outputs(B, W, hidden.device, outs)
    workspace, ws_bytes = _workspace(sv_accept_lmhead_workspace_size(B, W, V, gamma), hidden.device,
                                     workspace)
    _check(lib.sv_accept_chain_lmhead(mode, B, gamma, V, Dm, _ptr(hidden), _ptr(weight), _ptr(logits),
                                      _ptr(q), q_kind, _ptr(draft_tokens), float(temperature),
                                      int(top_k), float(top_p), int(seed), int(round_),
                                      _ptr(outs["tokens"]), _ptr(outs["num_emitted"]),
                                      _ptr(outs["num_accepted"]), _ptr(outs["near_ties"]),
                                      _ptr(workspace), ws_bytes, _stream(stream)))
    outs["target_logits"] = logits
    return outs


def sv_accept_tree_lmhead(mode, hidden, weight, q, q_kind, parent, node_tokens, temperature=1.0,
                          top_k=0, seed=0, round_=0, top_p=1.0, outs=None, logits=None,
                          workspace=None, stream=None) -> dict:
    """Tree acceptance fused with the LM-head projection: hidden [B,N,Dm] bf16, weight
    [V,Dm] bf16; the target logits [B,N,V] bf16 are returned under "target_logits"."""
    lib = load_library()
    _dev(node_tokens, "node_tokens", torch.int32)
    B, N = node_tokens.shape
    Dm, V = _lmhead_args(hidden, weight, B, N)
    Dq = 0
    if q is not None:
        Dq = q.shape[1]
        _dev(q, "q", torch.bfloat16 if q_kind == Q_LOGITS else torch.float32, (B, Dq, V))
    par, pstride, W = _tree_arg(parent, B, N)
    if logits is None:
        logits = torch.empty((B, N, V), dtype=torch.bfloat16, device=hidden.device)
    _dev(logits, "logits", torch.bfloat16, (B, N, V))
    outs = _accept_outputs(B, W, hidden.device, outs)
    outs.setdefault("path_nodes", torch.empty((B, W), dtype=torch.int32, device=hidden.device))
    workspace, ws_bytes = _workspace(sv_accept_lmhead_workspace_size(B, N, V, Dq), hidden.device,
                                     workspace)
    _check(lib.sv_accept_tree_lmhead(mode, B, N, V, Dm, _ptr(hidden), _ptr(weight), _ptr(logits), par,
                                     pstride, _ptr(node_tokens), _ptr(q), q_kind, Dq,
                                     float(temperature), int(top_k), float(top_p), int(seed),
                                     int(round_), _ptr(outs["path_nodes"]), _ptr(outs["tokens"]),
                                     _ptr(outs["num_emitted"]), _ptr(outs["num_accepted"]),
                                     _ptr(outs["near_ties"]), _ptr(workspace), ws_bytes,
                                     _stream(stream)))
    outs["target_logits"] = logits
    return outs


def sv_ngram_draft(history, length, max_ngram=3, min_ngram=1, gamma=4, out=None,
                   stream=None):
    """Prompt-lookup drafts: history [B,Lmax] int32 and length [B] int32 (CUDA tensors).
    Returns (drafts [B,gamma] int32, -1 after the proposed tokens; num_drafts [B])."""
    lib = load_library()
    _dev(history, "history", torch.int32)
    if history.dim() != 2:
        raise ValueError("history must be [B, Lmax]")
    B, Lmax = history.shape
    _dev(length, "length", torch.int32, (B,))
    if out is None:
        drafts = torch.empty((B, gamma), dtype=torch.int32, device=history.device)
        num = torch.empty(B, dtype=torch.int32, device=history.device)
    else:
        drafts, num = out
        _dev(drafts, "drafts", torch.int32, (B, gamma))
        _dev(num, "num_drafts", torch.int32, (B,))
    _check(lib.sv_ngram_draft(B, Lmax, _ptr(history), _ptr(length), int(max_ngram),
                              int(min_ngram), int(gamma), _ptr(drafts), _ptr(num),
                              _stream(stream)))
    return drafts, num

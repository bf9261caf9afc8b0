"""One verify step through the C ABI: tree attention, acceptance, KV commit.

``VerifyStep`` owns the device workspaces and output buffers of one workload shape and
issues the ABI calls on one stream: attention, then acceptance with the commit of the
kept path fused into it (``accept_commit``; ``accept`` and ``commit`` are the separate
calls).  ``run_host`` is the end-to-end form: it
copies the step's inputs from (pinned) host tensors, runs the step, and copies the
accepted tokens back.  All arithmetic happens in libsv.so.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import (EXACT, GREEDY, Q_LOGITS, KVCache, sv_accept_chain, sv_accept_chain_commit,
               sv_accept_tree, sv_accept_tree_commit, sv_accept_workspace_size, sv_commit_kv,
               sv_tree_attention, sv_tree_attention_workspace_size)


# inputs of the attention call (the rest feed the acceptance)
_ATTN_INPUTS = ("q", "k_tree", "v_tree")


def _depths(parent):
    d = []
    for p in parent:
        d.append(0 if p < 0 else d[p] + 1)
    return d


class VerifyStep:
    """Buffers and calls of one verify step for a fixed batch shape.

    chain=True uses sv_accept_chain (parent must be a chain); otherwise sv_accept_tree.
    """

    def __init__(self, parent: Sequence[int], B: int, Hq: int, Hkv: int, D: int, V: int,
                 cache: KVCache, dtype=torch.bfloat16, mode=EXACT, q_kind=Q_LOGITS,
                 temperature: float = 1.0, top_k: int = 0, chain: bool = False,
                 device: Optional[torch.device] = None, top_p: float = 1.0):
        self.parent = list(parent)
        self.N = len(self.parent)
        self.Dmax = max(_depths(self.parent))
        self.B, self.Hq, self.Hkv, self.D, self.V = B, Hq, Hkv, D, V
        self.cache, self.dtype, self.mode, self.q_kind = cache, dtype, mode, q_kind
        self.temperature, self.top_k, self.chain = temperature, top_k, chain
        self.top_p = top_p
        self.device = device or cache.k.device
        self.scale = D ** -0.5
        ws = sv_tree_attention_workspace_size(dtype, B, self.N, Hq, Hkv, D, cache.max_prefix)
        # zero before first use: the kernel keeps completion words in it
        self.attn_ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=self.device)
        self.attn_splits = ws > 0
        Dq = self.Dmax
        self.acc_ws = torch.empty(sv_accept_workspace_size(B, self.N, V, Dq), dtype=torch.uint8,
                                  device=self.device)
        self.out = torch.empty((B, self.N, Hq, D), dtype=dtype, device=self.device)
        W = self.Dmax + 1
        # the outputs are views of one int32 buffer, tokens and counts first, so that the
        # end-to-end step reads them back with a single copy
        self._out_buf = torch.empty(2 * B * W + 3 * B, dtype=torch.int32, device=self.device)
        self._out_head = B * W + 3 * B  # tokens, num_emitted, num_accepted, near_ties
        o = self._out_buf
        self.outs = dict(tokens=o[:B * W].view(B, W), num_emitted=o[B * W:B * W + B],
                         num_accepted=o[B * W + B:B * W + 2 * B],
                         near_ties=o[B * W + 2 * B:B * W + 3 * B],
                         path_nodes=o[B * W + 3 * B:].view(B, W))
        if chain:
            pn = torch.arange(W, dtype=torch.int32, device=self.device)
            self.chain_path = pn.unsqueeze(0).expand(B, W).contiguous()

    def kernel_launches(self) -> int:
        """Kernels one step launches: attention, then the two acceptance kernels (the
        commit runs inside the second)."""
        return 1 + 2

    def attention(self, q, k_tree, v_tree, stream=None):
        return sv_tree_attention(q, k_tree, v_tree, self.cache, self.parent, self.scale,
                                 out=self.out, workspace=self.attn_ws, stream=stream)

    def accept(self, target_logits, q_draft, node_tokens, seed=0, round_=0, stream=None):
        if self.chain:
            toks = node_tokens[:, 1:] if node_tokens.shape[1] == self.N else node_tokens
            r = sv_accept_chain(self.mode, target_logits, q_draft, self.q_kind,
                                toks.contiguous() if not toks.is_contiguous() else toks,
                                temperature=self.temperature, top_k=self.top_k, top_p=self.top_p, seed=seed,
                                round_=round_, outs=self.outs, workspace=self.acc_ws,
                                stream=stream)
            # a chain's accepted path is nodes 0..num_accepted
            return r
        return sv_accept_tree(self.mode, target_logits, q_draft, self.q_kind, self.parent,
                              node_tokens, temperature=self.temperature, top_k=self.top_k, top_p=self.top_p,
                              seed=seed, round_=round_, outs=self.outs, workspace=self.acc_ws,
                              stream=stream)

    def commit(self, k_tree, v_tree, stream=None):
        path = self.chain_path if self.chain else self.outs["path_nodes"]
        sv_commit_kv(k_tree, v_tree, path, self.outs["num_accepted"], self.cache, stream=stream)

    def accept_commit(self, target_logits, q_draft, node_tokens, k_tree, v_tree, seed=0,
                      round_=0, stream=None):
        """Acceptance and the commit of the kept path in one call."""
        if self.chain:
            toks = node_tokens[:, 1:] if node_tokens.shape[1] == self.N else node_tokens
            return sv_accept_chain_commit(
                self.mode, target_logits, q_draft, self.q_kind,
                toks.contiguous() if not toks.is_contiguous() else toks, k_tree, v_tree,
                self.cache, temperature=self.temperature, top_k=self.top_k, top_p=self.top_p, seed=seed,
                round_=round_, outs=self.outs, workspace=self.acc_ws, stream=stream)
        return sv_accept_tree_commit(self.mode, target_logits, q_draft, self.q_kind, self.parent,
                                     node_tokens, k_tree, v_tree, self.cache,
                                     temperature=self.temperature, top_k=self.top_k, top_p=self.top_p, seed=seed,
                                     round_=round_, outs=self.outs, workspace=self.acc_ws,
                                     stream=stream)

    def run(self, q, k_tree, v_tree, target_logits, q_draft, node_tokens, seed=0, round_=0,
            stream=None):
        self.attention(q, k_tree, v_tree, stream)
        self.accept_commit(target_logits, q_draft, node_tokens, k_tree, v_tree, seed, round_,
                           stream)
        return self.out, self.outs

    # ------------------------------------------------------------ end to end

    def alloc_inputs(self, like: dict):
        """Device input buffers shaped like the host tensors in ``like``."""
        self.dev_in = {k: torch.empty_like(v, device=self.device) for k, v in like.items()}
        self._copy_stream = None
        B, W = self.B, self.Dmax + 1
        self._host_buf = torch.empty(self._out_head, dtype=torch.int32, pin_memory=True)
        h = self._host_buf
        self.host_out = dict(tokens=h[:B * W].view(B, W), num_emitted=h[B * W:B * W + B],
                             num_accepted=h[B * W + B:B * W + 2 * B],
                             near_ties=h[B * W + 2 * B:B * W + 3 * B])
        return self.dev_in

    def run_host(self, host_in: dict, seed=0, round_=0, stream=None):
        """H2D copies of the step inputs (pinned host tensors), the step, and the D2H
        copy of the emitted tokens and counts; returns the pinned host outputs.

        The attention's inputs are copied on the step's stream and the acceptance's (the
        logits, the node tokens) on a second stream at the same time, so that the logits'
        copy overlaps the attention; the acceptance waits for it.  The second stream first
        waits for everything already queued on the step's stream, which may still read
        these device buffers."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        d = self.dev_in
        if self._copy_stream is None:
            self._copy_stream = torch.cuda.Stream(self.device)
            self._copied = torch.cuda.Event()
        cs = self._copy_stream
        cs.wait_stream(s)
        with torch.cuda.stream(cs):
            for k, v in host_in.items():
                if k not in _ATTN_INPUTS:
                    d[k].copy_(v, non_blocking=True)
            self._copied.record(cs)
        with torch.cuda.stream(s):
            for k in _ATTN_INPUTS:
                d[k].copy_(host_in[k], non_blocking=True)
            self.attention(d["q"], d["k_tree"], d["v_tree"], s)
            s.wait_event(self._copied)
            self.accept_commit(d["target_logits"], d["draft_logits"], d["node_tokens"],
                               d["k_tree"], d["v_tree"], seed, round_, s)
            self._host_buf.copy_(self._out_buf[:self._out_head], non_blocking=True)
        return self.host_out

    def h2d_bytes(self, host_in: dict) -> int:
        return sum(v.numel() * v.element_size() for v in host_in.values())

    def d2h_bytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.host_out.values())

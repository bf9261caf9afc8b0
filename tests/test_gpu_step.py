"""The verify step through host buffers (VerifyStep.run_host: the attention's inputs and
the acceptance's inputs copied on two streams, the logits' copy overlapping the attention)
against the same step on device-resident inputs: the attention output, the emitted tokens
and counts and the committed cache must be identical, step after step."""
import pytest
import torch

import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl
from speculative_decoding_verify_sv_gb300.step import VerifyStep

pytestmark = pytest.mark.gpu


def _step(w, cache, chain):
    c = w["cfg"]
    return VerifyStep(w["parent"], c["B"], c["Hq"], c["Hkv"], c["D"], c["V"], cache,
                      dtype=c["dtype"], mode=sv.EXACT, q_kind=sv.Q_LOGITS,
                      temperature=c["temperature"], top_k=c["top_k"], chain=chain,
                      device=cache.k.device)


@pytest.mark.parametrize("cfg,B,V", [(2, 4, 4096), (3, 6, 4096), (5, 12, 2048)])
def test_host_step_equals_device_step(cuda_ok, cfg, B, V):
    dev = torch.device("cuda")
    w = wl.make_workload(cfg, device=dev, B=B, V=V, L=300, coverage=True)
    c = w["cfg"]
    chain = c["kind"] == "chain"
    toks = w["draft_tokens"] if chain else w["node_tokens"]
    bt = None if w["block_table"] is None else w["block_table"].clone()
    mk = lambda: sv.KVCache(w["cache_k"].clone(), w["cache_v"].clone(), w["prefix_len"].clone(),
                            bt, w.get("block_size", 16))
    ca, cb = mk(), mk()
    sa, sb = _step(w, ca, chain), _step(w, cb, chain)
    host = {k: w[k].cpu().pin_memory() for k in ("q", "k_tree", "v_tree", "target_logits",
                                                 "draft_logits")}
    host["node_tokens"] = toks.cpu().pin_memory()
    sb.alloc_inputs(host)
    for rnd in range(3):
        # the same prefix lengths every step, so that each step sees the same cache
        ca.prefix_len.copy_(w["prefix_len"])
        cb.prefix_len.copy_(w["prefix_len"])
        out_a, outs_a = sa.run(w["q"], w["k_tree"], w["v_tree"], w["target_logits"],
                               w["draft_logits"], toks, seed=w["seed"], round_=rnd)
        res_b = sb.run_host(host, seed=w["seed"], round_=rnd)
        torch.cuda.synchronize()
        assert torch.equal(out_a, sb.out)
        for k in ("tokens", "num_emitted", "num_accepted"):
            assert torch.equal(outs_a[k].cpu(), res_b[k]), k
        assert torch.equal(ca.prefix_len, cb.prefix_len)
        assert torch.equal(ca.k, cb.k) and torch.equal(ca.v, cb.v)
    assert sv.sv_read_device_status() == 0

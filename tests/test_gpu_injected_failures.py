"""Launch failures injected on the host (sv_inject_launch_failures), through the C ABI.

A call whose launch fails must report SV_ERR_CUDA with a message, launch nothing (the
library's kernel count does not move), leave its outputs and the KV cache untouched, and
leave the library usable: the next call gives the same results as a call that never saw a
failure.  No GPU fault is made: the failure is reported by the host in place of the launch.
"""
import pytest
import torch

import speculative_decoding_verify_sv_gb300 as sv
from speculative_decoding_verify_sv_gb300 import workloads as wl
from speculative_decoding_verify_sv_gb300.step import VerifyStep

pytestmark = pytest.mark.gpu


def _chain_inputs():
    lg = wl.chain_logits(8, 4, 4000, sigma=3.0, draft_sigma=1.0, dtype=torch.bfloat16, seed=81)
    dev = torch.device("cuda")
    return lg["target_logits"].to(dev), lg["draft_logits"].to(dev), lg["draft_tokens"].to(dev)


def test_failed_acceptance_launch_is_reported_and_harmless(cuda_ok):
    tl, q, dt = _chain_inputs()
    clean = sv.sv_accept_chain(sv.EXACT, tl, q, sv.Q_LOGITS, dt, seed=3, round_=1)
    torch.cuda.synchronize()
    outs = {k: torch.full_like(v, -7) for k, v in clean.items()}
    n0 = sv.sv_kernel_launches()
    sv.sv_inject_launch_failures(1)
    with pytest.raises(sv.SVError) as err:
        sv.sv_accept_chain(sv.EXACT, tl, q, sv.Q_LOGITS, dt, seed=3, round_=1, outs=outs)
    assert err.value.code == sv.SV_ERR_CUDA and "launch" in str(err.value)
    torch.cuda.synchronize()
    assert sv.sv_kernel_launches() == n0
    for v in outs.values():
        assert bool((v == -7).all())  # nothing was written
    # the injected failure was used up: the next call runs and matches the clean one
    again = sv.sv_accept_chain(sv.EXACT, tl, q, sv.Q_LOGITS, dt, seed=3, round_=1, outs=outs)
    torch.cuda.synchronize()
    for k in clean:
        assert torch.equal(again[k].cpu(), clean[k].cpu()), k
    assert sv.sv_kernel_launches() > n0
    assert sv.sv_read_device_status() == 0


def test_failed_step_leaves_the_cache_untouched(cuda_ok):
    """A verify step whose acceptance-and-commit launch fails (its attention ran) keeps the
    cache and prefix lengths as they were; the retried call commits as a clean step does."""
    w = wl.make_workload(2, device="cuda", B=4, V=4000, L=256)
    c = w["cfg"]

    def make_step():
        cache = sv.KVCache(w["cache_k"].clone(), w["cache_v"].clone(), w["prefix_len"].clone())
        step = VerifyStep(w["parent"], c["B"], c["Hq"], c["Hkv"], c["D"], c["V"], cache,
                          dtype=c["dtype"], mode=sv.EXACT, q_kind=sv.Q_LOGITS, device="cuda")
        return cache, step

    acc_args = (w["target_logits"], w["draft_logits"], w["node_tokens"], w["k_tree"], w["v_tree"], 5, 2)
    ref_cache, ref_step = make_step()
    ref_out, ref_res = ref_step.run(w["q"], w["k_tree"], w["v_tree"], w["target_logits"],
                                    w["draft_logits"], w["node_tokens"], seed=5, round_=2)
    torch.cuda.synchronize()

    cache, step = make_step()
    out = step.attention(w["q"], w["k_tree"], w["v_tree"])
    k0, v0, l0 = cache.k.clone(), cache.v.clone(), cache.prefix_len.clone()
    sv.sv_inject_launch_failures(1)
    with pytest.raises(sv.SVError) as err:
        step.accept_commit(*acc_args)
    assert err.value.code == sv.SV_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.equal(cache.prefix_len, l0)
    assert torch.equal(cache.k, k0) and torch.equal(cache.v, v0)
    res = step.accept_commit(*acc_args)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    for k in ("tokens", "num_emitted", "num_accepted", "path_nodes"):
        assert torch.equal(res[k].cpu(), ref_res[k].cpu()), k
    assert torch.equal(cache.prefix_len, ref_cache.prefix_len)
    assert torch.equal(cache.k, ref_cache.k) and torch.equal(cache.v, ref_cache.v)
    assert sv.sv_read_device_status() == 0


def test_injection_count_is_cleared_by_zero(cuda_ok):
    tl, q, dt = _chain_inputs()
    sv.sv_inject_launch_failures(3)
    sv.sv_inject_launch_failures(0)
    out = sv.sv_accept_chain(sv.EXACT, tl, q, sv.Q_LOGITS, dt, seed=1)
    torch.cuda.synchronize()
    assert int(out["num_emitted"].min()) >= 1

#!/usr/bin/env python
"""Verify-step benchmark: verified candidate tokens/s on one GB300 (per GPU replica).

A step is one pass of the whole hot path over one batch: tree attention (one layer),
token acceptance over the vocabulary, and the KV commit of the accepted path.
Default workload (the headline line): ragged-paged, the largest of the five -- B=256
chains of 4 drafts, GQA 32q/8kv x 128, prefixes U{512..8192} in a paged cache of
16-token blocks, vocab 152064, exact sampling at T=1.  The other four workloads follow
under "per_workload" (device-timed, fewer steps).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides; each step is timed with CUDA events on the
stream the kernels run on.  Between steps (outside the events) prefix_len is restored
and L2 is flushed by writing a buffer of twice its size, then reading another one of
that size (so that no dirty lines are left for the timed kernels to write back).  Each stage of the step
(attention; acceptance with the KV commit fused into it) is captured once into a CUDA
graph and replayed, so
that host launch overhead does not open gaps inside the timed windows (--eager times
the plain launches instead).  Under torchrun every rank
runs an independent replica (weak scaling, no collective on the data path); the
device time is the max over ranks.

--impl reference times the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "verified candidate tokens/s at 1 GB300; verify-step HBM GB/s vs peak"
ALL_CONFIGS = (1, 2, 3, 4, 5)
UNIT = "candidate tokens/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers

def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5,
                    help="workload id 1..5 (default 5, ragged-paged: the largest)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small profiling captures)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --config (no per_workload lines for the others)")
    ap.add_argument("--per-workload-steps", type=int, default=30)
    ap.add_argument("--mode", choices=["exact", "greedy"], default=None)
    ap.add_argument("--preheat-s", type=float, default=1.0,
                    help="untimed seconds of steps before warm-up (clock ramp)")
    ap.add_argument("--eager", action="store_true",
                    help="time plain launches instead of CUDA graph replays")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target duration of the oracle sample")
    return ap.parse_args()


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64,
                         device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled while the GPU works."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append(dict(sm=float(parts[0]), smax=float(parts[1]), util=float(parts[3]),
                                 hw=parts[4], hwt=parts[5], swt=parts[6], pcap=parts[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def committed_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    src = os.path.join(ROOT, "speculative_decoding_verify_sv_gb300", "csrc", kernel_file)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    for e in entries:
        if e.get("workload") == workload and e.get("source_sha") == sha:
            return e.get("dram_bytes_per_launch")
    return None


def attention_bytes(w, prefix_len=None) -> int:
    """Algorithmic bytes of one tree-attention launch: prefix K and V read once, tree
    Q/K/V read, O written.  prefix_len: the lengths the launch reads (default: the
    workload's, as generated)."""
    c = w["cfg"]
    es = 4 if c["dtype"] == torch.float32 else 2
    B, N, Hq, Hkv, D = c["B"], w["N"], c["Hq"], c["Hkv"], c["D"]
    lens = w["prefix_len"] if prefix_len is None else prefix_len
    prefix = int(lens.sum().item()) * Hkv * D * es * 2
    tree = B * N * (2 * Hq + 2 * Hkv) * D * es
    return prefix + tree


def accept_bytes(w) -> int:
    """Algorithmic bytes of acceptance: every target row and draft row read once."""
    c = w["cfg"]
    es = 4 if c["dtype"] == torch.float32 else 2
    B, N, V = c["B"], w["N"], c["V"]
    return B * (N + w["Dmax"]) * V * es


def attention_flops(w, prefix_len=None) -> int:
    """Algorithmic flops of one tree-attention launch: 4*D per (query row, attended key);
    a node attends to the prefix and to its root path (depth + 1 tree keys)."""
    from speculative_decoding_verify_sv_gb300 import workloads as wl
    c = w["cfg"]
    B, N, Hq, D = c["B"], w["N"], c["Hq"], c["D"]
    lens = w["prefix_len"] if prefix_len is None else prefix_len
    path_keys = sum(d + 1 for d in wl.depths(w["parent"]))
    keys = int(lens.sum().item()) * N * Hq + B * Hq * path_keys
    return 4 * keys * D


def workload_name(c, cfg_id) -> str:
    return f"{c['name']} (config {cfg_id})"


# ---------------------------------------------------------------- our arm

def time_workload(args, dist: Dist, cfg_id: int, K: int, warmup: int, preheat_s: float,
                  batch=None):
    """Time K verify steps of workload cfg_id on this rank's GPU (device time, CUDA events
    on the launch stream, L2 flushed between steps).  Returns the measurements and the
    objects the end-to-end leg reuses."""
    import speculative_decoding_verify_sv_gb300 as sv
    from speculative_decoding_verify_sv_gb300 import workloads as wl
    from speculative_decoding_verify_sv_gb300.step import VerifyStep

    dev = torch.device("cuda", dist.local_rank)
    w = wl.make_workload(cfg_id, device=dev, B=batch)
    c = w["cfg"]
    mode_name = args.mode or c["mode"]
    mode = sv.EXACT if mode_name == "exact" else sv.GREEDY
    chain = c["kind"] == "chain"
    cache = sv.KVCache(w["cache_k"], w["cache_v"], w["prefix_len"], w["block_table"],
                       w.get("block_size", 16))
    step = VerifyStep(w["parent"], c["B"], c["Hq"], c["Hkv"], c["D"], c["V"], cache,
                      dtype=c["dtype"], mode=mode, q_kind=sv.Q_LOGITS,
                      temperature=c["temperature"], top_k=c["top_k"], chain=chain, device=dev)
    toks = w["draft_tokens"] if chain else w["node_tokens"]
    # every step starts from these lengths (the commit advances them; prepare() restores)
    prefix0 = w["prefix_len"].clone()
    a_bytes = attention_bytes(w, prefix0)
    a_flops = attention_flops(w, prefix0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 1 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    emitted = torch.zeros(c["B"], dtype=torch.int64, device=dev)

    flush_read = torch.ones(flush.numel() // 4, dtype=torch.int32, device=dev)

    def prepare():
        cache.prefix_len.copy_(prefix0)
        flush.zero_()  # evicts the step's data from L2 ...
        torch.sum(flush_read)  # ... and reading another buffer evicts the dirty lines

    def device_step(i, ev=None):
        if ev:
            ev[0].record(stream)
        step.attention(w["q"], w["k_tree"], w["v_tree"], stream)
        if ev:
            ev[1].record(stream)
        step.accept_commit(w["target_logits"], w["draft_logits"], toks, w["k_tree"], w["v_tree"],
                           seed=w["seed"], round_=i, stream=stream)
        if ev:
            ev[2].record(stream)

    # pre-heat (clock ramp), then the warm-up steps
    sampler = ClockSampler(dev.index)
    sampler.start()
    t_end = time.perf_counter() + preheat_s
    i = 0
    while time.perf_counter() < t_end:
        prepare()
        device_step(i)
        i += 1
        if i % 20 == 0:
            torch.cuda.synchronize()
    for j in range(warmup):
        prepare()
        device_step(j)
    torch.cuda.synchronize()

    # one CUDA graph per stage; the acceptance round is fixed at capture (the work of a
    # step does not depend on it)
    graphs, launch_mode, per_step = None, "eager launches", None
    if not args.eager:
        try:
            n0 = sv.sv_kernel_launches()
            graphs = []
            for fn in (lambda st: step.attention(w["q"], w["k_tree"], w["v_tree"], st),
                       lambda st: step.accept_commit(w["target_logits"], w["draft_logits"], toks,
                                                     w["k_tree"], w["v_tree"], seed=w["seed"],
                                                     round_=0, stream=st)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, capture_error_mode="relaxed"):
                    fn(torch.cuda.current_stream())
                graphs.append(g)
            per_step = sv.sv_kernel_launches() - n0
            for _ in range(3):
                prepare()
                for g in graphs:
                    g.replay()
            torch.cuda.synchronize()
            launch_mode = "CUDA graph replay per stage (captured once)"
        except Exception as e:  # capture unsupported here: time the plain launches
            graphs = None
            launch_mode = f"eager launches (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()

    def timed_step(j, ev):
        if graphs is None:
            device_step(j, ev)
            return
        for k, g in enumerate(graphs):
            ev[k].record(stream)
            g.replay()
        ev[2].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    dist.barrier()
    torch.cuda.synchronize()
    launches0 = sv.sv_kernel_launches()
    t0 = time.perf_counter()
    for j in range(K):
        prepare()
        timed_step(j, evs[j])
        emitted.add_(step.outs["num_emitted"])
    torch.cuda.synchronize()
    dist.barrier()
    wall = time.perf_counter() - t0
    launches = sv.sv_kernel_launches() - launches0
    if graphs is not None:  # replays launch kernels without the host counter seeing them
        launches = per_step * K
    clocks = sampler.stop()
    status = sv.sv_read_device_status()

    tot = [e[0].elapsed_time(e[2]) for e in evs]
    att = [e[0].elapsed_time(e[1]) for e in evs]
    acc = [e[1].elapsed_time(e[2]) for e in evs]
    tc = sv.sv_tree_attention_path(c["dtype"], w["N"], c["Hq"], c["Hkv"], c["D"],
                                   w.get("block_size", 16) if c["paged"] else 0) == 1
    # every timed step verifies the same inputs with the same round: the last step's
    # accepted lengths and near-tie words are those of every step
    na = step.outs["num_accepted"].cpu().to(torch.int64)
    nt = step.outs["near_ties"].cpu().to(torch.int64) & 0xFFFFFFFF
    outcome = dict(
        accepted_length_histogram=torch.bincount(na.clamp(0, w["Dmax"]), minlength=w["Dmax"] + 1).tolist(),
        sequences_with_decision_near_ties=int(((nt & 0xFFFF) > 0).sum()),
        sequences_with_sample_near_ties=int(((nt >> 16) > 0).sum()))
    return dict(w=w, c=c, step=step, toks=toks, prepare=prepare, stream=stream, outcome=outcome,
                mode=mode, mode_name=mode_name, launch_mode=launch_mode, tot=tot, att=att,
                acc=acc, wall=wall, launches=launches, clocks=clocks, status=status,
                emitted=float(emitted.sum().item()), a_bytes=a_bytes, a_flops=a_flops,
                acc_bytes=accept_bytes(w), tc=tc, name=workload_name(c, cfg_id))


def _kernel_figures(r):
    """Mean attention and acceptance times (ms) of one run and their algorithmic GB/s."""
    a_ms = statistics.mean(r["att"])
    c_ms = statistics.mean(r["acc"])
    a_gbs = r["a_bytes"] / (a_ms / 1e3) / 1e9
    c_gbs = r["acc_bytes"] / (c_ms / 1e3) / 1e9
    return a_ms, c_ms, a_gbs, c_gbs


def per_workload_line(args, dist, cfg_id, K, peak):
    """Device-timed figures of one more workload (no end-to-end or CPU leg)."""
    r = time_workload(args, dist, cfg_id, K, max(3, min(args.warmup, 5)), 0.3)
    a_ms, c_ms, a_gbs, c_gbs = _kernel_figures(r)
    c = r["c"]
    cand = c["B"] * (r["w"]["N"] - 1)
    dev_ms = dist.max(sum(r["tot"]))
    out = {
        "workload": r["name"], "steps": K, "ms_per_step": dev_ms / K,
        "value": dist.sum(cand * K) / (dev_ms / 1e3), "unit": UNIT,
        "attention_us": 1e3 * a_ms, "attention_gbs": a_gbs, "attention_frac": a_gbs / peak,
        "attention_tflops": r["a_flops"] / (a_ms / 1e3) / 1e12,
        "attention_kernel": "attn_tc_kernel" if r["tc"] else "general (mma.sync / FFMA)",
        "accept_us": 1e3 * c_ms, "accept_gbs": c_gbs, "accept_frac": c_gbs / peak,
        "algorithmic_bytes": {"attention": r["a_bytes"], "accept": r["acc_bytes"]},
        "clocks": r["clocks"], "device_status": r["status"],
    }
    del r
    torch.cuda.empty_cache()
    return out


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def lm_head_line(args, dist, K):
    """The LM-head projection fused with the acceptance (draft-chain shapes: B = 64 chains
    of 5 drafts, hidden size 4096, V = 128256): the projection alone, projection then
    acceptance, and the fused call.  Inputs: hidden ~N(0,1), W ~N(0, 3/sqrt(4096)) (logits
    about N(0,3)), draft rows the projection of perturbed hidden states, random drafts."""
    import speculative_decoding_verify_sv_gb300 as sv
    dev = torch.device("cuda", dist.local_rank)
    B, gamma, Dm, V = 64, 5, 4096, 128256
    R = B * (gamma + 1)
    g = torch.Generator(device=dev).manual_seed(4321)
    h = torch.randn((R, Dm), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((V, Dm), generator=g, device=dev) * (3.0 / math.sqrt(Dm))).to(torch.bfloat16)
    hq = (h.float().view(B, gamma + 1, Dm)[:, :gamma]
          + 0.3 * torch.randn((B, gamma, Dm), generator=g, device=dev)).to(torch.bfloat16)
    dl = sv.sv_lm_head(hq, w)
    toks = torch.randint(0, V, (B, gamma), generator=g, device=dev, dtype=torch.int32)
    z = torch.empty((R, V), dtype=torch.bfloat16, device=dev)
    hv = h.view(B, gamma + 1, Dm)
    ws = torch.zeros(sv.sv_accept_lmhead_workspace_size(B, gamma + 1, V, gamma), dtype=torch.uint8,
                     device=dev)
    ws2 = torch.zeros(sv.sv_accept_workspace_size(B, gamma + 1, V, gamma), dtype=torch.uint8, device=dev)
    outs = sv.sv_accept_chain_lmhead(sv.EXACT, hv, w, dl, sv.Q_LOGITS, toks, workspace=ws)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(flush.numel() // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for a, b in evs:
            flush.zero_()
            torch.sum(flush_read)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)

    proj = timed(lambda: sv.sv_lm_head(h, w, out=z))
    unfused = timed(lambda: (sv.sv_lm_head(h, w, out=z),
                             sv.sv_accept_chain(sv.EXACT, z.view(B, gamma + 1, V), dl, sv.Q_LOGITS,
                                                toks, outs=outs, workspace=ws2)))
    fused = timed(lambda: sv.sv_accept_chain_lmhead(sv.EXACT, hv, w, dl, sv.Q_LOGITS, toks,
                                                    outs=outs, logits=outs["target_logits"],
                                                    workspace=ws))
    flops = 2.0 * R * V * Dm
    peak, kind = measured_bf16_tflops()
    tf = flops / (proj / 1e6) / 1e12
    return {
        "workload": "LM head + acceptance, draft-chain shapes (B=64, gamma=5, hidden 4096, V=128256)",
        "steps": K, "projection_us": proj, "projection_then_accept_us": unfused,
        "fused_us": fused, "candidates_per_s_fused": B * gamma / (fused / 1e6),
        "roofline": {"kernel": "lm_head_kernel (tcgen05 GEMM, statistics epilogue)",
                     "bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                     "frac": tf / peak, "peak_source": kind, "flops_per_launch": flops},
    }


def next_rows_lines(args, dist, K, peak):
    """The widened rows on synthetic inputs of the workloads' shapes, each timed with L2
    flushed before every call (median of K): bytes are the rows each call must read at
    least once, so GB/s is a lower bound of the achieved traffic.

    F2 sibling-recursive tree acceptance and F3 typical acceptance: the medusa-t64 shapes
    (B = 8, 64-node tree, V = 32000; target rows near the head rows, so paths get
    accepted).  F3 top-p: the draft-chain shapes (B = 64, gamma = 5, V = 128256, T = 0.7,
    top-k 50, top-p 0.9).  F4: prompt-lookup drafting over 256 histories of 8192 tokens,
    and exact verification of its deterministic drafts (no q rows) at the ragged-paged
    acceptance shapes (B = 256, gamma = 4, V = 152064)."""
    import speculative_decoding_verify_sv_gb300 as sv
    from speculative_decoding_verify_sv_gb300 import workloads as wl
    dev = torch.device("cuda", dist.local_rank)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(flush.numel() // 4, dtype=torch.int32, device=dev)

    def timed(fn):
        # the call is captured once into a CUDA graph (after warm-up calls), so that host
        # launch work opens no gap between the events
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for a, b in evs:
            flush.zero_()
            torch.sum(flush_read)
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return 1e3 * statistics.median(a.elapsed_time(b) for a, b in evs)

    def line(row, what, us, nbytes, extra=None):
        gbs = nbytes / (us / 1e6) / 1e9
        d = {"row": row, "workload": what, "us": us, "bytes": nbytes, "gbs": gbs,
             "frac_of_hbm": gbs / peak}
        d.update(extra or {})
        return d

    out = []
    # F2 and F3 typical: medusa-t64 shapes
    B, parent, V = 8, wl.TREE_T64, 32000
    N = len(parent)
    lg = wl.medusa_logits(B, parent, V, sigma=3.0, seed=77, coverage=True, coverage_sigma=0.7)
    tl, q, nt = lg["target_logits"].to(dev), lg["draft_logits"].to(dev), lg["node_tokens"].to(dev)
    Dq = q.shape[1]
    ws = torch.empty(sv.sv_accept_workspace_size(B, N, V, Dq), dtype=torch.uint8, device=dev)
    o_ind = sv.sv_accept_tree(sv.EXACT, tl, q, sv.Q_LOGITS, parent, nt, seed=3, workspace=ws)
    o_rec = sv.sv_accept_tree_recursive(tl, q, sv.Q_LOGITS, parent, nt, seed=3, workspace=ws)
    o_typ = sv.sv_accept_typical(tl, parent, nt, workspace=ws)
    t_ind = timed(lambda: sv.sv_accept_tree(sv.EXACT, tl, q, sv.Q_LOGITS, parent, nt, seed=3,
                                            outs=o_ind, workspace=ws))
    t_rec = timed(lambda: sv.sv_accept_tree_recursive(tl, q, sv.Q_LOGITS, parent, nt, seed=3,
                                                      outs=o_rec, workspace=ws))
    t_typ = timed(lambda: sv.sv_accept_typical(tl, parent, nt, outs=o_typ, workspace=ws))
    rows_b = B * (N + Dq) * V * tl.element_size()
    out.append(line("F2", "sibling-recursive tree acceptance, medusa-t64 shapes", t_rec, rows_b,
                    {"independent_rule_us": t_ind,
                     "mean_accepted": float(o_rec["num_accepted"].float().mean())}))
    out.append(line("F3", "typical acceptance, medusa-t64 shapes", t_typ, B * N * V * tl.element_size(),
                    {"mean_accepted": float(o_typ["num_accepted"].float().mean())}))
    del tl, q, nt, lg, ws
    # F3 top-p: draft-chain shapes
    B, gamma, V = 64, 5, 128256
    g = torch.Generator(device=dev).manual_seed(78)
    tl = (3.0 * torch.randn((B, gamma + 1, V), generator=g, device=dev)).to(torch.bfloat16)
    dl = (tl[:, :gamma].float() + torch.randn((B, gamma, V), generator=g, device=dev)).to(torch.bfloat16)
    toks = torch.argmax(dl.float(), dim=-1).to(torch.int32)
    ws = torch.empty(sv.sv_accept_workspace_size(B, gamma + 1, V, gamma), dtype=torch.uint8, device=dev)
    o = sv.sv_accept_chain(sv.EXACT, tl, dl, sv.Q_LOGITS, toks, temperature=0.7, top_k=50, top_p=0.9,
                           seed=5, workspace=ws)
    t_tp = timed(lambda: sv.sv_accept_chain(sv.EXACT, tl, dl, sv.Q_LOGITS, toks, temperature=0.7,
                                            top_k=50, top_p=0.9, seed=5, outs=o, workspace=ws))
    out.append(line("F3", "top-p 0.9 within top-k 50, T = 0.7, draft-chain shapes", t_tp,
                    B * (2 * gamma + 1) * V * 2))
    del tl, dl, toks, ws, o
    # F4: drafting over histories, then verifying the deterministic drafts
    B, L, gamma, V = 256, 8192, 4, 152064
    hist = torch.randint(0, 32000, (B, L), generator=g, device=dev, dtype=torch.int32)
    hist[:, L - 3:] = hist[:, 1000:1003]  # the last trigram occurs earlier: drafts exist
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    drafts, num = sv.sv_ngram_draft(hist, lens, max_ngram=3, min_ngram=1, gamma=gamma)
    t_ng = timed(lambda: sv.sv_ngram_draft(hist, lens, max_ngram=3, min_ngram=1, gamma=gamma,
                                           out=(drafts, num)))
    out.append(line("F4", "prompt-lookup drafts, 256 histories of 8192 tokens, n = 3..1", t_ng,
                    B * L * 4, {"mean_drafts": float(num.float().mean())}))
    tl = (3.0 * torch.randn((B, gamma + 1, V), generator=g, device=dev)).to(torch.bfloat16)
    ws = torch.empty(sv.sv_accept_workspace_size(B, gamma + 1, V, gamma), dtype=torch.uint8, device=dev)
    o = sv.sv_accept_chain(sv.EXACT, tl, None, sv.Q_DRAFT_ONEHOT, drafts, seed=6, workspace=ws)
    t_oh = timed(lambda: sv.sv_accept_chain(sv.EXACT, tl, None, sv.Q_DRAFT_ONEHOT, drafts, seed=6,
                                            outs=o, workspace=ws))
    out.append(line("F4", "exact verification of the drafts (q one-hot), ragged-paged acceptance shapes",
                    t_oh, B * (gamma + 1) * V * 2))
    del tl, ws, o, hist
    torch.cuda.empty_cache()
    return out


def run_ours(args, dist: Dist):
    import speculative_decoding_verify_sv_gb300 as sv  # noqa: F401 (fails loudly if missing)

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peaks()
    K = args.steps
    r = time_workload(args, dist, args.config, K, args.warmup, args.preheat_s, args.batch)
    w, c = r["w"], r["c"]
    dev_ms = dist.max(sum(r["tot"]))
    cand = c["B"] * (w["N"] - 1)
    units = dist.sum(cand * K)
    value = units / (dev_ms / 1e3)
    emitted_total = dist.sum(r["emitted"])
    a_ms, c_ms, achieved, c_gbs = _kernel_figures(r)
    kernel_file = "attention_tc.cu" if r["tc"] else "attention.cu"
    kernel_name = ("attn_tc_kernel (the one kernel of a sv_tree_attention call)" if r["tc"] else
                   "attn_mma_kernel / attn_f32_kernel + split merge")
    name = r["name"] if args.batch is None else f"{r['name']} with B={c['B']}"

    result = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": dist.world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": dev_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if c["dtype"] == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {
            "workload": name,
            "B": c["B"], "tree_nodes": w["N"], "candidates_per_step": cand,
            "Hq": c["Hq"], "Hkv": c["Hkv"], "D": c["D"], "V": c["V"],
            "prefix": c["L"] if not isinstance(c["L"], tuple) else f"U{{{c['L'][0]}..{c['L'][1]}}}",
            "paged": c["paged"], "mode": r["mode_name"], "temperature": c["temperature"],
            "top_k": c["top_k"], "l2": "flushed between steps: 2x L2 written, then another 2x L2 read, outside events",
            "timing": "CUDA events per step on the launch stream; sum over K steps",
            "launch": r["launch_mode"],
            "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "single GPU",
        },
        "roofline": {
            "kernel": kernel_name,
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes_per_launch": r["a_bytes"],
            "traffic": committed_traffic(kernel_file, name),
        },
        "roofline_accept": {
            "kernel": "accept_stats_kernel + accept_select_kernel (KV commit fused)",
            "bound": "hbm", "achieved": c_gbs, "peak": peak, "unit": "GB/s",
            "frac": c_gbs / peak, "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes_per_launch": r["acc_bytes"],
            "traffic": committed_traffic("accept.cu", name),
        },
        "breakdown_us": {
            "attention": 1e3 * a_ms, "accept_and_commit": 1e3 * c_ms,
            "accept_gbs": c_gbs,
            "attention_tflops": r["a_flops"] / (a_ms / 1e3) / 1e12,
        },
        "emitted_tokens_per_s": emitted_total / (dev_ms / 1e3),
        "mean_accepted": emitted_total / (c["B"] * K * dist.world) - 1.0,
        "outcome_per_step": dict(r["outcome"], note="sequences of one step (rank 0); every timed "
                                 "step verifies the same inputs with the same round"),
        "acceptance_rate": (emitted_total / (c["B"] * K * dist.world) - 1.0) / max(1, w["Dmax"]),
        "wall_s_timed_region": r["wall"],
        "gpu_launches": r["launches"],
        "device_status": r["status"],
        "clocks": r["clocks"],
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, dist, w, r["step"], r["prepare"], r["stream"], r["toks"],
                                cand)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, r["mode"])
    if not args.no_per_workload and args.batch is None:
        del r, w
        torch.cuda.empty_cache()
        K_pw = max(3, min(K, args.per_workload_steps))
        result["per_workload"] = [per_workload_line(args, dist, i, K_pw, peak)
                                  for i in sorted(ALL_CONFIGS) if i != args.config]
        result["lm_head"] = lm_head_line(args, dist, K_pw)
        result["next_rows"] = next_rows_lines(args, dist, K_pw, peak)
    return result


def run_e2e(args, dist, w, step, prepare, stream, toks, cand):
    """Same metric through the public step API with host inputs: every step copies its
    inputs from pinned host memory and reads the emitted tokens back."""
    host = {k: w[k].cpu().pin_memory() for k in ("q", "k_tree", "v_tree", "target_logits",
                                                 "draft_logits")}
    host["node_tokens"] = toks.cpu().pin_memory()
    step.alloc_inputs(host)
    for j in range(max(3, args.warmup)):
        prepare()
        step.run_host(host, seed=w["seed"], round_=j, stream=stream)
    torch.cuda.synchronize()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    dist.barrier()
    torch.cuda.synchronize()
    for j in range(K):
        prepare()
        evs[j][0].record(stream)
        step.run_host(host, seed=w["seed"], round_=j, stream=stream)
        evs[j][1].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms = dist.max(sum(a.elapsed_time(b) for a, b in evs))
    units = dist.sum(cand * K)
    return {"value": units / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": step.h2d_bytes(host),
            "d2h_bytes_per_step": step.d2h_bytes(), "ms_per_step": ms / K}


# ------------------------------------------------------------ CPU oracle

def _seq_on_host(w, b):
    """Sequence b's inputs on the host, with a cache of its own rows only: a contiguous
    cache row, or its blocks of a paged pool (in order, with a block table 0, 1, ...) with
    room for the commit."""
    sel = slice(b, b + 1)
    d = {k: w[k][sel].cpu() for k in ("q", "k_tree", "v_tree", "target_logits", "draft_logits",
                                      "prefix_len")}
    d["toks"] = (w["draft_tokens"] if "draft_tokens" in w and w["cfg"]["kind"] == "chain"
                 else w["node_tokens"])[sel].cpu()
    if w["block_table"] is None:
        d["cache_k"], d["cache_v"], d["bt"] = w["cache_k"][sel].cpu(), w["cache_v"][sel].cpu(), None
    else:
        bs = w.get("block_size", 16)
        nblk = min(w["block_table"].shape[1], (int(w["prefix_len"][b]) + w["N"] + bs - 1) // bs)
        ids = w["block_table"][b, :nblk].long()
        d["cache_k"], d["cache_v"] = w["cache_k"][ids].cpu(), w["cache_v"][ids].cpu()
        d["bt"] = torch.arange(nblk, dtype=torch.int32).unsqueeze(0)
    return d


def oracle_sample(w, budget_s: float, mode: int, b_limit=None):
    """Time the oracle on whole sequences (attention of every node and head, acceptance,
    commit) until the budget is spent, cycling over the workload's sequences (at most 64
    passes) when they take less; returns (candidates, seconds, sequence evaluations).
    Only the evaluated sequence's inputs are brought to the host, outside the timing."""
    import oracle
    c = w["cfg"]
    chain = c["kind"] == "chain"
    limit = 64 * c["B"] if b_limit is None else min(b_limit, c["B"])
    done, spent = 0, 0.0
    seqs = {}
    while done < limit and (done == 0 or spent < budget_s):
        b = done % c["B"]
        if b not in seqs:
            if len(seqs) >= 16:
                seqs.pop(next(iter(seqs)))
            seqs[b] = _seq_on_host(w, b)
        d = seqs[b]
        t0 = time.perf_counter()
        oracle.tree_attention(d["q"], d["k_tree"], d["v_tree"], d["cache_k"], d["cache_v"],
                              d["prefix_len"], w["parent"], w["scale"], block_table=d["bt"],
                              block_size=w.get("block_size", 16))
        if chain:
            r = oracle.accept_chain(mode, d["target_logits"], d["draft_logits"], oracle.Q_LOGITS,
                                    d["toks"], temperature=c["temperature"], top_k=c["top_k"],
                                    seed=w["seed"])
            W = d["toks"].shape[1] + 1
            path = torch.arange(W, dtype=torch.int32).unsqueeze(0)
        else:
            r = oracle.accept_tree(mode, d["target_logits"], d["draft_logits"], oracle.Q_LOGITS,
                                   w["parent"], d["toks"], temperature=c["temperature"],
                                   top_k=c["top_k"], seed=w["seed"])
            path = r["path_nodes"]
        oracle.commit_kv(d["k_tree"], d["v_tree"], path, r["num_accepted"], d["cache_k"],
                         d["cache_v"], d["prefix_len"], block_table=d["bt"],
                         block_size=w.get("block_size", 16))
        spent += time.perf_counter() - t0
        done += 1
    return done * (w["N"] - 1), spent, done


def cpu_baseline(w, budget_s, mode):
    import oracle
    cand, secs, seqs = oracle_sample(w, budget_s, mode)
    return {"value": cand / secs, "unit": UNIT, "cores": oracle.get_threads(), "kind": "oracle",
            "sample": f"{seqs} sequence evaluations ({min(seqs, w['cfg']['B'])} distinct of the "
                      f"workload's {w['cfg']['B']}: attention of every node and head over the full "
                      f"prefix, acceptance, commit), {secs:.1f} s"}


def run_reference(args, dist: Dist):
    """The oracle timed on the host cores on the same workload, metric and unit."""
    import oracle
    from speculative_decoding_verify_sv_gb300 import workloads as wl
    if dist.rank != 0:
        return None
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.make_workload(args.config, device=dev)
    c = w["cfg"]
    mode = oracle.EXACT if (args.mode or c["mode"]) == "exact" else oracle.GREEDY
    # each step: a bounded sample (one sequence), sized so the whole run stays short
    per_step_budget = max(0.5, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, mode, b_limit=1)
    cand, secs = 0, 0.0
    for _ in range(args.steps):
        cnd, s, _ = oracle_sample(w, per_step_budget, mode, b_limit=1)
        cand += cnd
        secs += s
    value = cand / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": f"{c['name']} (config {args.config})", "B": c["B"],
                   "tree_nodes": w["N"], "candidates_per_step": c["B"] * (w["N"] - 1)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.get_threads(),
                         "kind": "oracle",
                         "sample": "one sequence per step (attention of every node and head, "
                                   "acceptance, commit) of the workload"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.impl == "reference":
            res = run_reference(args, dist)
        else:
            res = run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()

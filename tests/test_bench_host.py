"""Host-side pieces of bench.py (CPU only): the algorithmic bytes and flops behind the
roofline figures against the per-workload figures worked out by hand from the shapes
(prefix K+V read once, tree Q/K/V read and O written, every target and q row read once),
and the rules that decide which stored ncu traffic and which peak a run may quote."""
import json
import os

import pytest
import torch

import bench
from speculative_decoding_verify_sv_gb300 import workloads as wl

# (attention bytes, acceptance bytes) per workload, multiplied out by hand:
#   1 chain-f32:   1*128*4*64*4*2 + 1*5*(4+4+4+4)*64*4 = 262,144 + 20,480;   1*(5+4)*1000*4
#   2 medusa-t64:  8*2048*32*128*2*2 + 8*64*(64+64)*128*2;  8*64*32000*2 + 8*4*32000*2
#   3 draft-chain: 64*4096*8*128*2*2 + 64*6*(64+16)*128*2;  64*6*128256*2 + 64*5*128256*2
#   4 long-tree:   16*32768*8*128*2*2 + 16*26*(128+16)*128*2; 16*26*32000*2 + 16*4*32000*2
HAND = {
    1: (282_624, 36_000),
    2: (285_212_672, 34_816_000),
    3: (1_081_606_144, 180_584_448),
    4: (2_162_819_072, 30_720_000),
}


def _shape_only(cfg_id):
    """The fields the byte formulas read, without allocating the workload's tensors."""
    cfg = wl.CONFIGS[cfg_id]
    parent = wl.config_parent(cfg)
    return dict(cfg=cfg, N=len(parent), Dmax=max(wl.depths(parent)), parent=parent,
                prefix_len=torch.tensor(wl.prefix_lengths(cfg, cfg["B"], seed=0)))


@pytest.mark.parametrize("cfg_id", sorted(HAND))
def test_algorithmic_bytes_match_hand_figures(cfg_id):
    w = _shape_only(cfg_id)
    attn, acc = HAND[cfg_id]
    assert bench.attention_bytes(w) == attn
    assert bench.accept_bytes(w) == acc


def test_ragged_paged_bytes_follow_the_seeded_lengths():
    w = _shape_only(5)
    lens = w["prefix_len"]
    assert lens.numel() == 256 and int(lens.min()) >= 512 and int(lens.max()) <= 8192
    # 4096 bytes of K and V per cached token (8 kv heads x 128 x bf16 x 2), plus the tree
    tree = 256 * 5 * (64 + 16) * 128 * 2
    assert bench.attention_bytes(w) == int(lens.sum()) * 4096 + tree
    # about 4.59e9 at the mean length of U{512..8192}
    assert abs(bench.attention_bytes(w) / 4.59e9 - 1.0) < 0.03
    assert bench.accept_bytes(w) == 700_710_912


def test_attention_flops_count_attended_keys():
    # 4 * D per (query row, key it attends): the prefix, then its root path.  The 64-node
    # tree has 1, 4, 12, 24, 23 nodes at depths 0..4: 1*1 + 4*2 + 12*3 + 24*4 + 23*5 = 256
    # tree keys per head and sequence (not the 64 x 64 block the tensor cores compute)
    w = _shape_only(2)
    assert bench.attention_flops(w) == 4 * 128 * (8 * 64 * 32 * 2048 + 8 * 32 * 256)
    assert abs(bench.attention_flops(w) / 17.2e9 - 1.0) < 0.01
    # a chain: node i sees i + 1 tree keys
    w = _shape_only(3)
    assert bench.attention_flops(w) == 4 * 128 * (64 * 6 * 32 * 4096 + 64 * 32 * 21)


def _fake_root(tmp_path, source_text, entry):
    csrc = tmp_path / "speculative_decoding_verify_sv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(source_text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps([entry]))
    return str(tmp_path)


def test_stored_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    import hashlib
    src = "__global__ void k() {}\n"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    root = _fake_root(tmp_path, src, dict(workload="w", source_sha=sha,
                                          dram_bytes_per_launch=1234))
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.committed_traffic("k.cu", "w") == 1234
    assert bench.committed_traffic("k.cu", "other workload") is None
    # the kernel changed since the capture: no traffic is quoted
    with open(os.path.join(root, "speculative_decoding_verify_sv_gb300", "csrc", "k.cu"), "a") as f:
        f.write("// edited\n")
    assert bench.committed_traffic("k.cu", "w") is None
    assert bench.committed_traffic("missing.cu", "w") is None


def test_peak_falls_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, kind = bench.measured_peaks()
    assert kind == "fallback" and peak == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6765.3}))
    assert bench.measured_peaks() == (6765.3, "measured")


class _FakeSmi:
    """Stands in for the nvidia-smi sampling process: returns fixed CSV rows."""

    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def kill(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clocks_are_read_from_samples_under_load():
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi(
        "1000, 2070, 100.0, 0, Not Active, Not Active, Not Active, Not Active\n"
        "2070, 2070, 900.0, 100, Not Active, Not Active, Not Active, Active\n"
        "2040, 2070, 910.0, 98, Not Active, Not Active, Not Active, Not Active\n"
        "not a sample\n")
    c = s.stop()
    # the idle sample (utilisation 0) is left out of the median and of the reasons
    assert c["sm_mhz"] == 2055.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 3 and c["samples_under_load"] == 2


def test_throttle_reasons_that_reject_a_run_are_reported():
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("1500, 2070, 1300.0, 100, Active, Not Active, Active, Not Active\n")
    c = s.stop()
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("")
    assert s.stop()["reasons"] == ["no samples"]
    s = bench.ClockSampler(0)  # nvidia-smi could not be started
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_attention_bytes_use_the_lengths_the_launch_reads():
    """The commit advances prefix_len after every step; the roofline counts the lengths
    each timed launch starts from (restored between steps), passed explicitly."""
    w = _shape_only(2)
    start = w["prefix_len"].clone()
    advanced = start + 5  # what prefix_len holds after a step that emitted 5 tokens
    w["prefix_len"] = advanced
    assert bench.attention_bytes(w, start) == HAND[2][0]
    assert bench.attention_bytes(w) == HAND[2][0] + 8 * 5 * 32 * 128 * 2 * 2
    assert bench.attention_flops(w, start) == 4 * 128 * (8 * 64 * 32 * 2048 + 8 * 32 * 256)

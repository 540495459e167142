"""Host-side logic of bench.py that the bench line depends on, checked on the CPU:
the effective FLOP count against the pairs the oracle actually weights, the
nominal pair count against its closed forms, the DRAM-traffic record's source-hash
rule, and the parsing of sampled nvidia-smi clock lines."""

import hashlib
import os
import shutil

import numpy as np
import pytest
import torch

import bench
from oracle import oracle
from transformer_scaled_dot_03_gb300 import inputs


@pytest.mark.parametrize("mask,n,m,lens", [
    ("none", 37, 53, None),
    ("causal", 40, 40, None),
    ("causal", 30, 70, None),        # bottom-right: row i sees keys j <= i + 40
    ("causal", 70, 30, None),        # rows 0..39 see no key
    ("key_padding", 33, 50, [50, 0, 17, 80]),
    ("causal_key_padding", 45, 45, [45, 10, 0]),
    ("causal_cache", 12, 60, [60, 12, 30, 5, 0]),
])
def test_effective_flops_counts_the_pairs_the_oracle_weights(mask, n, m, lens):
    B = len(lens) if lens else 2
    H, d = 2, 8
    x = inputs.make_inputs(B, H, n, m, d, d, mask, seed=900 + n + m, key_lengths=lens)
    w = inputs.Workload("t", B, H, n, m, d, d, mask, seed=0)
    _, _, W = oracle.attn_fwd(x.Q, x.K, x.V, x.mask, x.key_lengths, x.scale, weights=True)
    pairs = int(np.count_nonzero(W > 0))   # fp64 weights of visible keys do not underflow here
    assert bench.effective_flops(w, x) == pytest.approx(2.0 * (2 * d) * pairs, rel=0, abs=0)


def test_nominal_pairs_closed_forms():
    assert inputs.nominal_pairs(512, 512, "none") == 512 * 512
    assert inputs.nominal_pairs(1024, 1024, "causal") == 1024 * 1024 / 2
    assert inputs.nominal_pairs(100, 300, "causal") == 100 * 300 - 100 * 100 / 2
    assert inputs.nominal_pairs(300, 100, "causal_key_padding") == 100 * 100 / 2
    w = inputs.WORKLOADS["base_encoder_keypad"]
    assert w.flops() == 2.0 * w.B * w.H * (w.d_k + w.d_v) * w.n * w.m


def _source_hash(root):
    h = hashlib.sha256()
    for f in bench.KERNEL_SOURCES:
        h.update(open(os.path.join(root, f), "rb").read())
    return h.hexdigest()[:16]


def test_measured_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    # the committed record: reported for its workload while the sources hash to its value
    fields = {}
    for line in open(os.path.join(bench.ROOT, "profiles", "traffic.md"), encoding="utf-8"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    fresh = fields["kernel_source_sha256_16"] == _source_hash(bench.ROOT)
    got = bench.measured_traffic(fields["workload"])
    assert got == (int(fields["traffic_bytes_per_launch"]) if fresh else None)
    assert bench.measured_traffic("no_such_workload") is None
    # a copy of the tree whose record names another source hash reports nothing
    for f in bench.KERNEL_SOURCES:
        os.makedirs(tmp_path / os.path.dirname(f), exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, f), tmp_path / f)
    os.makedirs(tmp_path / "profiles")
    (tmp_path / "profiles" / "traffic.md").write_text(
        f"workload: base_encoder_keypad\nkernel_source_sha256_16: {'0' * 16}\ntraffic_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("base_encoder_keypad") is None
    (tmp_path / "profiles" / "traffic.md").write_text(
        f"workload: base_encoder_keypad\nkernel_source_sha256_16: {_source_hash(str(tmp_path))}\n"
        "traffic_bytes_per_launch: 123\n")
    assert bench.measured_traffic("base_encoder_keypad") == 123


def test_clock_summary_parses_sampled_lines():
    c = bench.Clocks(0)
    c.lines = [
        "2070, 2070, 410.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1995, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2055, 2070, 1388.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 0.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # unparsable: skipped
        "short line",
    ]
    s = c.summary()
    assert s == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c.lines = ["1500, 2070, 900.0, 0x28, Active, Not Active, Active, Not Active"]
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    c.lines = []
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

"""CPU pins for bench.py's accounting: the algorithmic flops and bytes the roofline
fractions are computed from, worked out by hand for the workloads' shapes, and the
rule that a committed DRAM-traffic figure is used only for the exact source it was
captured on."""

import hashlib
import json
import os

import numpy as np
import pytest

import bench
import oracle
from context_long_attention_lpt_gb300 import workloads as wl


def test_decode_accounting_by_hand():
    # 8 sequences x 32768 keys x 8 K/V heads x 128 x (K and V) x 2 bytes = 2^30 bytes;
    # one query per sequence sees every key: 8 x 32768 pairs per query head,
    # 4 x 128 x 32 flops per pair.
    w = wl.WORKLOADS["decode"]
    q_len, kv_len = [1] * 8, [32768] * 8
    costs = oracle.block_costs(q_len, kv_len, w.block_len, w.causal)
    acc = bench.workload_accounting(w, q_len, kv_len, np.asarray(costs), part_rows=128)
    assert acc["kv_bytes"] == 1073741824.0
    assert acc["flops"] == 4.0 * 128 * 32 * 8 * 32768
    assert acc["q_bytes"] == 8 * 32 * 128 * 2
    assert acc["part_bytes"] == 128 * 32 * 129 * 4
    assert acc["partial_bytes"] == acc["kv_bytes"] + acc["q_bytes"] + acc["part_bytes"]


def test_causal_tail_accounting_by_hand():
    # 512 queries after 131072 context keys: query t sees 131072 + t + 1 keys, so the
    # visible pairs are 512 x 131072 + (1 + ... + 512).
    w = wl.WORKLOADS["shortq"]
    q_len, kv_len = [512], [131072 + 512]
    costs = oracle.block_costs(q_len, kv_len, w.block_len, w.causal)
    acc = bench.workload_accounting(w, q_len, kv_len, np.asarray(costs), part_rows=0)
    pairs = 512 * 131072 + 512 * 513 // 2
    assert acc["flops"] == 4.0 * 128 * 32 * pairs
    assert acc["kv_bytes"] == (131072 + 512) * 8 * 128 * 2 * 2


def test_traffic_is_used_only_for_the_source_it_was_captured_on(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"source": "kernel.cu", "sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
             "bytes_per_launch": 123.0, "how": "test"}
    (prof / "dram_traffic.json").write_text(json.dumps({"k/w": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k", "w") == 123.0
    assert bench.traffic_for("k", "other") is None
    src.write_text("// kernel v2\n")  # any edit of the source voids the figure
    assert bench.traffic_for("k", "w") is None


@pytest.mark.parametrize("key", ["partial_decode/decode", "partial_tcgen05/shortq", "partial_tcgen05/largest",
                                 "partial_tcgen05/varlen"])
def test_committed_traffic_entries_are_well_formed(key):
    """Each committed figure names an existing kernel source, its hash and a byte count.
    (An edited source makes bench.py report null until the figure is captured again.)"""
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        e = json.load(f)[key]
    assert os.path.exists(os.path.join(bench.ROOT, e["source"]))
    assert len(e["sha256"]) == 64 and e["bytes_per_launch"] > 0


@pytest.mark.parametrize("name", ["tiny", "decode", "shortq", "varlen", "largest"])
def test_unit_pairs_equal_the_oracle_block_costs(name):
    """The closed form the CPU baseline and the reference arm count flops with equals the
    oracle's block costs summed over each sequence."""
    w = wl.WORKLOADS[name]
    q_len, kv_len = wl.lengths(w)
    for lq, lk in zip(q_len, kv_len):
        assert bench.unit_pairs(lq, lk, w.causal) == sum(oracle.block_costs([lq], [lk], w.block_len, w.causal))
    assert bench.unit_pairs(3, 10, True) == 8 + 9 + 10
    assert bench.unit_pairs(3, 10, False) == 30


def test_reference_arm_line_on_the_tiny_workload(capsys):
    """The reference arm (the oracle on the host) prints one JSON line with the contract's keys."""
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] in ("GB/s", "TFLOP/s")
    assert line["config"]["workload"] == "tiny" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_summary_keeps_only_the_timed_window(tmp_path):
    """Clock samples from before or after the timed region (an idle GPU) are left out."""
    import datetime
    import time

    p = tmp_path / "clk.csv"
    t = time.time()
    lines = []
    for dt, mhz, watts, cap in [(-0.2, 2070, 180, "Not Active"), (0.01, 1940, 1370, "Active"),
                                (0.03, 1950, 1365, "Active"), (0.3, 2070, 190, "Not Active")]:
        ts = datetime.datetime.fromtimestamp(t + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, {mhz}, 2070, {watts}, 0x4, Not Active, Not Active, Not Active, {cap}")
    p.write_text("\n".join(lines) + "\n")
    c = bench.ClockSampler("0", str(p))
    c.t0, c.t1 = t, t + 0.05
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 1945.0 and s["power_w_max"] == 1370.0
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"

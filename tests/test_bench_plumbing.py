"""The benchmark's host-side plumbing, on the CPU: workload names, the
row-count override, the reference arm's step sizing and the ncu traffic
record (its kernel, workload and size against the algorithmic bytes)."""
import json
import os

import pytest

import bench
from draft_token_markov_gb300 import workloads as W


def test_workload_names_match_the_workload_table():
    assert sorted(bench.WORKLOAD_NAMES) == sorted(W.BY_NAME)
    assert bench.DEFAULT_WORKLOAD == "deepseek"
    w = W.BY_NAME[bench.DEFAULT_WORKLOAD]
    assert (w.vocab, w.rank, w.rows, w.steps, w.live_rows) == (129280, 256, 8, 8, 6)


@pytest.mark.parametrize("rows", [1, 5, 8, 12, 64, 256])
def test_row_override_keeps_the_padding_rows_below_it(rows):
    w = W.with_rows(W.BY_NAME["batch"], rows)
    assert w.rows == rows
    assert all(b < rows for b in w.padding_rows)
    assert set(w.padding_rows) == {b for b in W.BY_NAME["batch"].padding_rows if b < rows}
    assert w.live_rows == rows - len(w.padding_rows)
    assert (w.vocab, w.rank, w.steps, w.mode) == (129280, 256, 8, W.INVCDF)


@pytest.mark.parametrize("steps,warmup", [(1, 0), (3, 3), (20, 3), (200, 20), (5000, 100)])
def test_reference_steps_stay_bounded(steps, warmup):
    s = bench.reference_step_seconds(steps, warmup)
    assert 0.05 <= s <= 8.0
    # the oracle time of the whole run stays near two minutes or less
    assert (steps + warmup) * s <= max(120.0 + 1e-9, (steps + warmup) * 0.05)


def test_traffic_record_describes_the_headline_kernel():
    with open(bench.TRAFFIC_FILE) as f:
        t = json.load(f)
    w = W.BY_NAME[bench.DEFAULT_WORKLOAD]
    assert t["workload"] == w.name
    assert t["kernel"].startswith("chain_tc_kernel<256, 0, 0>")
    assert t["dram_bytes_per_launch"] == t["dram_bytes_read"] + t["dram_bytes_write"]
    alg = W.algorithmic_bytes(w)
    # DRAM bytes of one launch: the head once plus base and cache, not re-reads
    assert 0.9 * alg <= t["dram_bytes_per_launch"] <= 1.1 * alg
    assert "--clock-control none" in t["command"]
    got = bench._traffic()
    assert got is None or got == t["dram_bytes_per_launch"]


def test_traffic_is_null_when_the_kernel_source_differs(tmp_path, monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        t = json.load(f)
    t["source_hash"] = "0" * 16
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(t))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench._traffic() is None

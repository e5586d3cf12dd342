"""Host logic of bench.py on CPU: which source file holds each workload's
dominant kernel, and the rule that a committed DRAM-traffic figure is
reported only while that source is unchanged since the counters were taken."""

import json
import os

import pytest

import bench
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "online_softmax_tiled_gb300", "csrc")


def _traffic():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_kernel_source_per_workload():
    expect = {
        "fwd_mha_n2048_d64": "fwd_tc64.cu",       # the persistent d = 64 forward
        "fwd_causal_n8192_d128": "fwd_tc.cu",
        "bwd_causal_n4096_d128": "bwd_tc.cu",
        "decode_gqa_l4096": "decode.cu",
        "decode_paged_gqa_l4096": "decode.cu",
        "decode_sparse_t8_i2048": "decode.cu",
    }
    for name, src in expect.items():
        assert bench.kernel_source(WORKLOADS[name]) == src, name
        assert os.path.exists(os.path.join(CSRC, src))


def test_traffic_entries_name_known_workloads():
    for name, entry in _traffic().items():
        assert name in WORKLOADS, name
        assert entry["dram_bytes_per_launch"] == entry["dram_read_bytes"] + entry["dram_write_bytes"]
        assert os.path.exists(os.path.join(ROOT, entry["capture"])), entry["capture"]


def test_traffic_is_dropped_once_the_source_changes(monkeypatch):
    w = WORKLOADS["fwd_mha_n2048_d64"]
    entry = _traffic()[w.name]
    monkeypatch.setattr(bench, "kernel_source_sha", lambda _w: entry["source_sha"])
    assert bench.profiled_traffic(w) == entry["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_sha", lambda _w: "0" * 16)
    assert bench.profiled_traffic(w) is None


@pytest.mark.parametrize("name", ["fwd_mha_n2048_d64", "fwd_causal_n8192_d128"])
def test_forward_traffic_reads_each_operand_once(name):
    """The committed counters of the forwards: DRAM reads equal the Q, K, V
    bytes to within 1 % (no re-reads), and the writes never exceed O."""
    w = WORKLOADS[name]
    entry = _traffic()[name]
    qkv = 2 * w.d * (w.B * w.Hq * w.Nq + 2 * w.B * w.Hkv * w.Nk)
    o = 2 * w.d * w.B * w.Hq * w.Nq
    assert abs(entry["dram_read_bytes"] - qkv) <= 0.01 * qkv
    assert entry["dram_write_bytes"] <= o

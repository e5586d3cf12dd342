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


def test_source_hash_covers_included_headers(tmp_path):
    """The hash that tags committed counters covers the kernel's .cu file and
    every local header it includes (directly or through another header), so
    a header change makes the counters stale."""
    files = bench.kernel_source_files(WORKLOADS["fwd_causal_n8192_d128"])
    names = [os.path.basename(p) for p in files]
    assert names[0] == "fwd_tc.cu"
    for hdr in ("common.cuh", "tc_ptx.cuh", "mask.cuh", "launchers.h", "attn.h"):
        assert hdr in names, hdr
    cu, hdr = tmp_path / "k.cu", tmp_path / "h.cuh"
    cu.write_text('#include "h.cuh"\n')
    hdr.write_text("int a;\n")
    assert [os.path.basename(p) for p in bench._local_includes(str(cu))] == ["h.cuh"]
    before = bench.hash_sources([str(cu), str(hdr)])
    hdr.write_text("int b;\n")
    assert bench.hash_sources([str(cu), str(hdr)]) != before


@pytest.mark.parametrize("name", ["fwd_mha_n2048_d64", "fwd_causal_n8192_d128"])
def test_forward_traffic_reads_each_operand_once(name):
    """The committed counters of the forwards: DRAM reads equal the Q, K, V
    bytes to within 1 % (no re-reads). Writes never exceed the bytes of O and
    LSE; they may fall short of them, because part of the output can still
    sit in L2 when the kernel ends, so there is no lower bound."""
    w = WORKLOADS[name]
    entry = _traffic()[name]
    qkv = 2 * w.d * (w.B * w.Hq * w.Nq + 2 * w.B * w.Hkv * w.Nk)
    o_lse = 2 * w.d * w.B * w.Hq * w.Nq + 4 * w.B * w.Hq * w.Nq
    assert abs(entry["dram_read_bytes"] - qkv) <= 0.01 * qkv
    assert entry["dram_write_bytes"] <= o_lse


def test_parity_tally_and_tolerances():
    """The bench's pre-timing check: errors per output, -inf rows on both
    sides count as equal, and the description's tolerances decide."""
    import numpy as np
    w = WORKLOADS["fwd_causal_n8192_d128"]
    got = {"o": np.array([[0.5, 0.25]]), "lse": np.array([-np.inf, 1.0])}
    t = bench.ParityTally(got)
    t.add("o", got["o"], np.array([[0.51, 0.25]]))
    t.add("lse", got["lse"], np.array([-np.inf, 1.0005]))
    rep = t.report()
    assert abs(rep["o"]["max_abs_err"] - 0.01) < 1e-12
    assert abs(rep["lse"]["max_abs_err"] - 0.0005) < 1e-12
    assert bench.parity_failures(w, rep) == []
    t.add("o", got["o"], np.array([[0.5, 0.3]]))        # 0.05 > 2e-2
    assert len(bench.parity_failures(w, t.report())) == 1
    wb = WORKLOADS["bwd_causal_n4096_d128"]
    tb = bench.ParityTally({"dq": np.ones(4)})
    tb.add("dq", np.ones(4), np.ones(4) * 1.06)          # 0.06 > 5e-2 * 1.06
    assert len(bench.parity_failures(wb, tb.report())) == 1

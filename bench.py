"""Benchmark of the tiled-attention hot path on GB300.

Default run (N=1): the long-context causal forward B=2, H=32, N=8192, d=128,
bf16 (the line's top-level value), followed in the same process by the
causal backward B=2, H=16, N=4096, d=128, the GQA split-KV decode (B=64,
Hq=32, Hkv=8, L=4096, 16 splits), the batched multi-head forward B=4,
H=16, N=2048, d=64, the forward and backward shapes with grouped-query heads
(4 query heads per KV head) and the paged GQA decode (16-token pages, ragged
lengths of mean 4096), each reported under ``workloads`` with its own
value, roofline, CPU baseline, end-to-end rate and clocks. ``--workload`` picks the
top-level workload and ``--extra`` the others (``--extra none``: only the
top-level one). A step is one pass of the workload's hot path through the C
ABI on inputs already resident in HBM; L2 is flushed (256 MiB write)
between timed steps unless the inputs exceed L2.

Before a workload is timed, one step's outputs are compared with the float64
oracle on the heads (or requests) that the CPU-baseline leg computes, at the
tolerances of the benchmark description; a mismatch ends the run with no
line. Prints ONE JSON line (rank 0). ``--impl reference`` times the float64
CPU oracle as the reference arm instead.

Multi-GPU: every rank runs an independent replica of the workload (the path
shards over batch and heads with no exchange), so value = N x units / max
over ranks of the timed region ("scaling": "weak").
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20


# ----------------------------------------------------------------- workload math

def make_workload_inputs(w):
    from workloads import make_doc_bounds, make_inputs, make_paged_inputs, make_sparse_inputs
    if w.kind == "decode_paged":
        return make_paged_inputs(w)
    if w.kind == "decode_sparse":
        return make_sparse_inputs(w)
    x = make_inputs(w)
    if w.doc_mean > 0:
        x["row_kv_start"], x["row_kv_end"] = make_doc_bounds(w.B, w.Nq, w.doc_mean, w.seed + 1)
    return x


def mask_spec(w, x):
    """The workload's mask as the oracle's dict (host arrays)."""
    spec = {"window_left": w.window_left, "window_right": w.window_right, "n_global": w.n_global}
    if "row_kv_start" in x:
        spec["row_kv_start"] = x["row_kv_start"].numpy()
        spec["row_kv_end"] = x["row_kv_end"].numpy()
    return spec


def visible_pairs(w, x):
    """Visible (query, key) pairs of one head, summed over the batch: each
    row sees [lo1, hi1] (window within its key range) and [lo2, hi2] (global
    keys within it)."""
    import numpy as np
    i = np.arange(w.Nq, dtype=np.int64)[None, :] + (w.Nk - w.Nq)
    s = np.zeros((w.B, w.Nq), dtype=np.int64)
    e = np.full((w.B, w.Nq), w.Nk, dtype=np.int64)
    if "row_kv_start" in x:
        s, e = x["row_kv_start"].numpy().astype(np.int64), x["row_kv_end"].numpy().astype(np.int64)
    lo1 = np.maximum(i - w.window_left if w.window_left >= 0 else 0, s)
    hi1 = np.minimum(i + w.window_right if w.window_right >= 0 else w.Nk - 1, e - 1)
    lo2, hi2 = s, np.minimum(w.n_global, e) - 1
    n1 = np.maximum(0, hi1 - lo1 + 1)
    n2 = np.maximum(0, hi2 - lo2 + 1)
    ov = np.maximum(0, np.minimum(hi1, hi2) - np.maximum(lo1, lo2) + 1)
    return int((n1 + n2 - ov).sum())


def paged_bytes(w, seq_lens):
    """Bytes a paged decode must move: each request's K and V rows once, its
    block-table entries, its length, q and o."""
    P = w.page_size
    keys = sum(int(n) for n in seq_lens)
    blocks = sum((int(n) + P - 1) // P for n in seq_lens)
    return (2 * w.Hkv * keys * w.d * 2 + 2 * len(seq_lens) * w.Hq * w.d * 2
            + 4 * (blocks + len(seq_lens)))


def sparse_bytes(w, counts):
    """Bytes a sparse-index decode must move: the K and V rows of every listed
    entry once per KV head, the list entries and counts, q and o (T tokens)."""
    n = sum(int(c) for c in counts)
    return (2 * w.Hkv * n * w.d * 2 + 2 * len(counts) * w.Hq * w.Nq * w.d * 2
            + 4 * (n + len(counts)))


def algorithmic_units(w, inputs=None):
    """(per-step units, unit name, bound) for a workload.

    FLOPs: 2 per multiply-add; the forward has two GEMMs (4·Nq·Nk·d per head,
    causal counts only the visible pairs), the backward five (2.5x the
    forward). Decode bytes: K and V read once plus q and o (paged decode:
    over each request's own length, plus its block-table entries)."""
    if w.kind == "decode_paged":
        return paged_bytes(w, inputs["seq_lens"].tolist()), "GB/s", "hbm"
    if w.kind == "decode_sparse":
        return sparse_bytes(w, inputs["counts"].tolist()), "GB/s", "hbm"
    if w.kind == "decode":
        bytes_ = 2 * w.B * w.Hkv * w.Nk * w.d * 2 + 2 * w.B * w.Hq * w.d * 2
        return bytes_, "GB/s", "hbm"
    if w.masked:
        flops = 4.0 * w.Hq * w.d * visible_pairs(w, inputs)
        return flops * (2.5 if w.kind == "bwd" else 1.0), "TFLOP/s", "tensor"
    if w.causal:
        shift = w.Nk - w.Nq
        pairs = sum(min(w.Nk, i + shift + 1) for i in range(w.Nq))
    else:
        pairs = w.Nq * w.Nk
    flops = 4.0 * w.B * w.Hq * w.d * pairs
    if w.kind == "bwd":
        flops *= 2.5
    return flops, "TFLOP/s", "tensor"


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the whole job's time is its slowest
    rank's); x itself on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float, unit: str) -> float:
    """Throughput of the whole job: every rank processed units_per_rank (weak
    scaling, independent replicas) in at most `seconds`."""
    return rate(world * units_per_rank, seconds, unit)


def rate(units, seconds, unit):
    return units / seconds / (1e12 if unit == "TFLOP/s" else 1e9)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 20 ms; the samples whose timestamps fall in
    the timed window (or, for a window shorter than the period, the ones
    next to it) give the reported clocks."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int):
        self.t_start = self.t_end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    @staticmethod
    def _ts(text):
        from datetime import datetime
        try:
            return datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            ts = self._ts(parts[0])
            if ts is not None:
                rows.append((ts, parts))
        if not rows:
            return None
        sel = [p for ts, p in rows if self.t_start <= ts <= self.t_end]
        if not sel:  # window shorter than the sampling period: nearest samples
            before = [p for ts, p in rows if ts < self.t_start][-1:]
            after = [p for ts, p in rows if ts > self.t_end][:1]
            sel = before + after
        num = lambda v: float(v) if v.replace(".", "", 1).isdigit() else None
        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        smax = [num(p[2]) for p in sel if num(p[2]) is not None]
        reasons = set()
        for p in sel:
            for name, val in zip(self.REASONS, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sel)}


# ----------------------------------------------------------------- CPU oracle

class ParityTally:
    """Largest |GPU - oracle| and |oracle| per output over the sampled units.
    Where both sides are -inf (a row with no visible key: LSE), the error is 0."""

    def __init__(self, outs):
        self.outs = outs          # name -> float64 host array of the GPU result, or None
        self.err = {}
        self.ref = {}

    def add(self, name, got, ref):
        import numpy as np
        if self.outs is None or name not in self.outs:
            return
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        both_inf = np.isneginf(got) & np.isneginf(ref)
        with np.errstate(invalid="ignore"):
            diff = np.where(both_inf, 0.0, np.abs(got - ref))
        fin = np.where(np.isfinite(ref), np.abs(ref), 0.0)
        e = float(np.max(diff)) if diff.size else 0.0
        r = float(np.max(fin)) if fin.size else 0.0
        if np.isnan(e):
            e = float("inf")
        self.err[name] = max(self.err.get(name, 0.0), e)
        self.ref[name] = max(self.ref.get(name, 0.0), r)

    def report(self):
        return {n: {"max_abs_err": self.err[n], "max_abs_ref": self.ref[n],
                    "rel": self.err[n] / self.ref[n] if self.ref[n] > 0 else None}
                for n in sorted(self.err)}


def parity_failures(w, report):
    """The outputs whose error exceeds the benchmark description's tolerance:
    float32 inputs max|err| <= 1e-5; bf16 O <= 2e-2, LSE <= 1e-3, gradients
    <= 5e-2 * max|ref|."""
    bad = []
    for name, r in report.items():
        if w.dtype == "f32":
            tol = 1e-5
        elif name == "lse":
            tol = 1e-3
        elif name in ("dq", "dk", "dv"):
            tol = 5e-2 * r["max_abs_ref"]
        else:
            tol = 2e-2
        if not r["max_abs_err"] <= tol:
            bad.append(f"{name}: max|err| {r['max_abs_err']:.3e} > {tol:.3e}")
    return bad


def cpu_oracle_sample(w, inputs, budget_s: float, gpu_outs=None):
    """Time the float64 oracle on whole (b, h) heads (decode: whole requests)
    of the workload until the budget is spent. When ``gpu_outs`` (name ->
    float64 host array of one GPU step's outputs) is given, every sampled
    unit is also compared with it. Returns (units processed, seconds,
    description, ParityTally)."""
    import numpy as np
    import torch

    import oracle
    from workloads import to_f64

    tally = ParityTally(gpu_outs)
    units_total, _, _ = algorithmic_units(w, inputs)
    t0 = time.perf_counter()
    done = 0
    if w.kind == "decode_sparse":
        cnt = inputs["counts"].numpy()
        idx = inputs["indices"].numpy()
        units = 0
        for b in range(w.B):
            o_r, l_r = oracle.decode_sparse(to_f64(inputs["q"][b:b + 1]),
                                            to_f64(inputs["k"][b:b + 1]),
                                            to_f64(inputs["v"][b:b + 1]), idx[b:b + 1],
                                            cnt[b:b + 1], w.scale)
            if gpu_outs is not None:
                tally.add("o", gpu_outs["o"][b:b + 1], o_r)
                tally.add("lse", gpu_outs["lse"][b:b + 1], l_r)
            units += sparse_bytes(w, cnt[b:b + 1].tolist())
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return units, time.perf_counter() - t0, f"{done} of {w.B} requests", tally
    if w.kind == "decode_paged":
        lens = inputs["seq_lens"].numpy()
        table = inputs["block_table"].numpy()
        kp, vp = inputs["k_pages"], inputs["v_pages"]
        units = 0
        for b in range(w.B):
            # only this request's pages are converted: the pool is shared
            pages = table[b, :(int(lens[b]) + w.page_size - 1) // w.page_size]
            idx = torch.as_tensor(pages.astype("int64"))
            k, v = to_f64(kp[idx]), to_f64(vp[idx])
            local = np.arange(len(pages), dtype=np.int32)[None, :]
            o_r, l_r = oracle.decode_paged(to_f64(inputs["q"][b:b + 1]), k, v, local,
                                           lens[b:b + 1], w.page_size, w.scale)
            if gpu_outs is not None:
                tally.add("o", gpu_outs["o"][b:b + 1], o_r)
                tally.add("lse", gpu_outs["lse"][b:b + 1], l_r)
            units += paged_bytes(w, lens[b:b + 1].tolist())
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return units, time.perf_counter() - t0, f"{done} of {w.B} requests", tally
    if w.kind == "decode":
        per_req = units_total / w.B
        for b in range(w.B):
            q = to_f64(inputs["q"][b:b + 1])
            k, v = to_f64(inputs["k"][b:b + 1]), to_f64(inputs["v"][b:b + 1])
            o_r, l_r = oracle.decode_splitkv(q, k, v, w.scale, w.num_splits)
            if gpu_outs is not None:
                tally.add("o", gpu_outs["o"][b:b + 1], o_r)
                tally.add("lse", gpu_outs["lse"][b:b + 1], l_r)
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return per_req * done, time.perf_counter() - t0, f"{done} of {w.B} requests", tally
    # Heads taken alternately from both ends of the (b, h) order, so that a
    # short budget still samples the first and the last batch entry and head.
    flat = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    heads = [flat[i // 2] if i % 2 == 0 else flat[-1 - i // 2] for i in range(len(flat))]
    per_head = units_total / len(heads)
    r = w.Hq // w.Hkv
    done_units = 0.0
    for b, h in heads:
        sl = lambda t, hh: to_f64(t[b:b + 1, hh:hh + 1])
        q, k, v = sl(inputs["q"], h), sl(inputs["k"], h // r), sl(inputs["v"], h // r)
        if w.kind == "bwd":
            if w.masked:
                ref = oracle.attention_bwd_masked(q, k, v, sl(inputs["do"], h), w.scale,
                                                  mask_spec(w, inputs))
            else:
                ref = oracle.attention_bwd(q, k, v, sl(inputs["do"], h), w.scale, w.causal)
            if gpu_outs is not None:
                tally.add("dq", gpu_outs["dq"][b:b + 1, h:h + 1], ref[0])
                if r == 1:  # with GQA a KV head's dK, dV sum over its group
                    tally.add("dk", gpu_outs["dk"][b:b + 1, h:h + 1], ref[1])
                    tally.add("dv", gpu_outs["dv"][b:b + 1, h:h + 1], ref[2])
            done_units += per_head
        elif w.masked:
            spec = mask_spec(w, inputs)
            xb = {}
            for key in ("row_kv_start", "row_kv_end"):
                if key in spec:
                    spec[key] = spec[key][b:b + 1]
                    xb[key] = inputs[key][b:b + 1]
            o_r, l_r = oracle.attention_fwd_masked(q, k, v, w.scale, spec)
            done_units += 4.0 * w.d * visible_pairs(
                dataclasses.replace(w, B=1), xb) if xb else units_total / len(heads)
        else:
            o_r, l_r = oracle.attention_fwd(q, k, v, w.scale, w.causal)
            done_units += per_head
        if w.kind == "fwd" and gpu_outs is not None:
            tally.add("o", gpu_outs["o"][b:b + 1, h:h + 1], o_r)
            tally.add("lse", gpu_outs["lse"][b:b + 1, h:h + 1], l_r)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done_units, time.perf_counter() - t0, f"{done} of {len(heads)} heads (b, h)", tally


def input_bytes(inputs):
    return sum(t.numel() * t.element_size() for t in inputs.values())


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------- reference arm

def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inputs = make_workload_inputs(w)
    units, unit, _ = algorithmic_units(w, inputs)
    budget = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inputs, budget / 4)
    done_units, secs = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        u, s, desc, _ = cpu_oracle_sample(w, inputs, budget)
        done_units += u
        secs += s
    value = rate(done_units, secs, unit)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, flushed=input_bytes(inputs) < L2_BYTES),
        "cpu_baseline": {"value": value, "unit": unit, "cores": host_cores(), "kind": "oracle",
                         "sample": f"per step {desc} of one batch, float64 NumPy"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


METRIC = "attn fwd/bwd TFLOP/s vs GB300 BF16 peak; split-KV decode GB/s vs HBM"


def workload_config(w, flushed: bool):
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk,
           "d": w.d, "causal": w.causal, "dtype": w.dtype}
    if w.kind in ("decode", "decode_paged", "decode_sparse"):
        cfg["num_splits"] = w.num_splits
    if w.kind == "decode_sparse":
        cfg["Nq"] = f"{w.Nq} query tokens per request"
        cfg["Nk"] = f"cache of {w.Nk} rows per request"
        cfg["n_index"] = f"{w.n_index} distinct rows listed per request, uniform, random order"
    if w.masked:
        cfg["mask"] = {"window_left": w.window_left, "window_right": w.window_right,
                       "n_global": w.n_global}
        if w.doc_mean:
            cfg["mask"]["documents"] = (f"packed, lengths uniform on [1, {2 * w.doc_mean - 1}], "
                                        "row key range = the row's document")
    if w.kind == "decode_paged":
        cfg["Nk"] = f"per-request lengths uniform on [1, {2 * w.Nk - 1}] (mean {w.Nk})"
        cfg["page_size"] = w.page_size
        cfg["pages"] = "pool handed out in a seeded random order"
    cfg["l2"] = ("flushed between timed steps (256 MiB write)" if flushed
                 else "inputs larger than L2 (129 MB); no flush")
    return cfg


# ----------------------------------------------------------------- GPU arm

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("hbm_gbs"), p.get("bf16_tflops"), p.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = {"fwd": "fwd_tc.cu", "bwd": "bwd_tc.cu", "decode": "decode.cu",
                  "decode_paged": "decode.cu", "decode_sparse": "decode.cu"}
FP32_FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def kernel_label(w):
    if w.kind == "fwd":
        return ("fwd_simt_kernel" if w.dtype == "f32" else
                "fwd_tc64_kernel (persistent)" if w.d == 64 else "fwd_tc_kernel") + \
            " (whole attn_fwd call, one launch)"
    if w.kind == "bwd":
        if w.dtype == "bf16" and w.d == 128:
            return "attn_bwd call (row-term preprocess + dK/dV key-tile pass + dQ query-tile pass)"
        return "attn_bwd call (row-term preprocess + main kernel + dQ convert)"
    if w.kind == "decode_paged":
        return "attn_decode_paged call (split kernel + merge kernel)"
    if w.kind == "decode_sparse":
        return "attn_decode_sparse call (split kernel + merge kernel)"
    return "attn_decode_splitkv call (split kernel + merge kernel)"


def kernel_source(w):
    """Source file of the workload's dominant kernel."""
    if w.kind == "fwd" and w.dtype == "bf16" and w.d == 64:
        return "fwd_tc64.cu"
    return KERNEL_SOURCES[w.kind]


def _local_includes(path):
    """Files named by the #include "..." lines of a source (csrc/ or include/)."""
    import re
    dirs = [os.path.dirname(path), os.path.join(ROOT, "include")]
    out = []
    with open(path, encoding="utf-8") as f:
        for name in re.findall(r'^\s*#\s*include\s+"([^"]+)"', f.read(), flags=re.M):
            for d in dirs:
                cand = os.path.join(d, name)
                if os.path.exists(cand):
                    out.append(os.path.normpath(cand))
                    break
    return out


def kernel_source_files(w):
    """The dominant kernel's .cu file and every local header it includes,
    directly or through other headers, in a fixed order."""
    root = os.path.join(ROOT, "online_softmax_tiled_gb300", "csrc", kernel_source(w))
    seen, todo = [], [root]
    while todo:
        p = todo.pop(0)
        if p in seen:
            continue
        seen.append(p)
        todo.extend(_local_includes(p))
    return [seen[0]] + sorted(seen[1:])


def hash_sources(paths):
    """Short hash over the names (relative to the repository) and contents of
    the given files, in order."""
    import hashlib
    h = hashlib.sha256()
    for path in paths:
        h.update(os.path.relpath(path, ROOT).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_source_sha(w):
    """Hash of the dominant kernel's source and of the headers it includes: a
    change to either makes committed counters stale."""
    return hash_sources(kernel_source_files(w))


def profiled_traffic(w):
    """Per-launch DRAM bytes (read + write) of the dominant kernel, from the
    committed ncu summary profiles/traffic.json; null when the kernel source
    changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get(w.name)
    if not entry or entry.get("source_sha") != kernel_source_sha(w):
        return None
    return entry.get("dram_bytes_per_launch")


def make_step(ost, w, x, dev, stream):
    """One step of the workload's hot path on device-resident inputs ``x``:
    returns (step callable, kernel launches per step, {output name: tensor})."""
    import torch
    if w.kind == "fwd":
        o = torch.empty_like(x["q"])
        lse = torch.empty(x["q"].shape[:-1], dtype=torch.float32, device=dev)
        if w.masked:
            amask = ost.make_mask(w.window_left, w.window_right, w.n_global,
                                  x.get("row_kv_start"), x.get("row_kv_end"))
            step = lambda: ost.attn_fwd_masked(x["q"], x["k"], x["v"], o, lse, w.scale, amask,
                                               stream)
        else:
            step = lambda: ost.attn_fwd(x["q"], x["k"], x["v"], o, lse, w.scale, w.causal,
                                        stream)
        return step, 1, {"o": o, "lse": lse}
    if w.kind == "bwd":
        amask = (ost.make_mask(w.window_left, w.window_right, w.n_global) if w.masked
                 else None)
        o, lse = ost.forward(x["q"], x["k"], x["v"], causal=w.causal, scale=w.scale, mask=amask)
        ws = torch.empty(ost.attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d,
                                                     w.torch_dtype),
                         dtype=torch.uint8, device=dev)
        dq, dk, dv = (torch.empty_like(x[n]) for n in ("q", "k", "v"))
        if w.masked:
            step = lambda: ost.attn_bwd_masked(x["q"], x["k"], x["v"], o, x["do"], lse, dq, dk,
                                               dv, w.scale, amask, ws, stream)
        else:
            step = lambda: ost.attn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, dq, dk, dv,
                                        w.scale, w.causal, ws, stream)
        return step, 3, {"dq": dq, "dk": dk, "dv": dv}
    rows = w.Hq * w.Nq if w.kind == "decode_sparse" else w.Hq
    ws = torch.empty(ost.attn_decode_workspace_size(w.B, rows, w.d, w.num_splits),
                     dtype=torch.uint8, device=dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:-1], dtype=torch.float32, device=dev)
    if w.kind == "decode_sparse":
        step = lambda: ost.attn_decode_sparse(x["q"], x["k"], x["v"], x["indices"], x["counts"],
                                              o, lse, w.scale, w.num_splits, ws, stream)
    elif w.kind == "decode_paged":
        step = lambda: ost.attn_decode_paged(x["q"], x["k_pages"], x["v_pages"],
                                             x["block_table"], x["seq_lens"], o, lse, w.scale,
                                             w.num_splits, ws, stream)
    else:
        step = lambda: ost.attn_decode_splitkv(x["q"], x["k"], x["v"], o, lse, w.scale,
                                               w.num_splits, ws, stream)
    return step, 2, {"o": o, "lse": lse}


class ParityError(RuntimeError):
    pass


def measure(args, w, ost, dev, world, rank, stream):
    """Warm up, check one step against the oracle (rank 0, the CPU-baseline
    leg), time ``args.steps`` steps and the end-to-end path; returns the
    workload's entry on rank 0 (None elsewhere)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    host = make_workload_inputs(w)
    x = {k: t.to(dev) for k, t in host.items()}
    units, unit, bound = algorithmic_units(w, host)
    in_bytes = sum(t.numel() * t.element_size() for t in host.values())
    flush = in_bytes < L2_BYTES
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    step, launches_per_step, out_map = make_step(ost, w, x, dev, stream)
    outs = tuple(out_map.values())

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        if flush:
            flush_buf.fill_(1)
        step()
    if ost.attn_sync_status(stream) != ost.ATTN_OK:
        raise RuntimeError(f"{w.name}: device error after the warm-up steps")

    if args.profile:
        # Short run for ncu: warm-up plus `steps` launches, nothing else.
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
        if ost.attn_sync_status(stream) != ost.ATTN_OK:
            raise RuntimeError(f"{w.name}: device error in the profiled steps")
        return None

    # --- the CPU-baseline leg: the oracle on a bounded sample of this step,
    # compared with the GPU's outputs of the same units before any timing
    cpu = None
    if rank == 0:
        from workloads import to_f64
        gpu_host = {n: to_f64(t) for n, t in out_map.items()}
        cpu_units, cpu_s, cpu_desc, tally = cpu_oracle_sample(w, host, args.cpu_budget,
                                                              gpu_outs=gpu_host)
        parity = tally.report()
        bad = parity_failures(w, parity)
        if bad:
            raise ParityError(f"{w.name}: GPU result differs from the oracle: " + "; ".join(bad))
        cpu = (cpu_units, cpu_s, cpu_desc, parity)
        del gpu_host

    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    # bring clocks up before the timed region
    t_end = time.time() + 0.5
    while time.time() < t_end:
        step()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    if sampler:
        sampler.mark_start()
    for i in range(args.steps):
        if flush:
            flush_buf.fill_(i & 0xff)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    if sampler:
        sampler.mark_end()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    if ost.attn_sync_status(stream) != ost.ATTN_OK:
        raise RuntimeError(f"{w.name}: device error in the timed steps")
    clocks = sampler.stop() if sampler else None

    # --- end to end through the public API: pinned host inputs in, results
    # out, every step. Two device buffer sets and three streams: step i's
    # inputs are copied in and step i-1's results copied out while the step
    # before computes, as a serving loop would overlap them.
    host_pinned = {k: t.pin_memory() for k, t in host.items()}
    x2 = {k: t.clone() for k, t in x.items()}
    step2, _, out_map2 = make_step(ost, w, x2, dev, stream)
    sets = [(x, step, outs), (x2, step2, tuple(out_map2.values()))]
    out_host = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host[0])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps_run(n):
        for i in range(n):
            b = i & 1
            xb, step_b, outs_b = sets[b]
            s_in.wait_event(comp_done[b])         # step i-2 has read these inputs
            with torch.cuda.stream(s_in):
                for k_, t in host_pinned.items():
                    xb[k_].copy_(t, non_blocking=True)
            in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            stream.wait_event(out_done[b])        # step i-2's results are out
            step_b()
            comp_done[b].record(stream)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                for dst, src in zip(out_host[b], outs_b):
                    dst.copy_(src, non_blocking=True)
            out_done[b].record(s_out)
        for b in range(2):
            stream.wait_event(out_done[b])

    e2e_steps_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(2, min(args.steps, 20))
    barrier()
    e_s.record(stream)
    s_in.wait_event(e_s)
    s_out.wait_event(e_s)
    e2e_steps_run(e2e_steps)
    e_e.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e_s.elapsed_time(e_e) / e2e_steps, dev)
    if ost.attn_sync_status(stream) != ost.ATTN_OK:
        raise RuntimeError(f"{w.name}: device error in the end-to-end steps")
    del x2, sets, step2, out_map2

    entry = None
    if rank == 0:
        ms_per_step = total_ms / args.steps
        hbm, tf_burst, _tf_sust, src = load_peaks()
        peak = hbm if bound == "hbm" else tf_burst
        peak_source = f"{src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops burst'})"
        if w.dtype == "f32":
            # float32 FFMA path: 152 SMs x 128 FMA lanes x 2 flops x 2.07 GHz max clock
            bound, peak, peak_source = "alu", FP32_FFMA_PEAK_TFLOPS, "derived (FFMA lanes x clock)"
        achieved = rate(units, ms_per_step / 1e3, unit)
        cpu_units, cpu_s, cpu_desc, parity = cpu
        entry = {
            "value": whole_job_rate(units * args.steps, world, total_ms / 1e3, unit),
            "unit": unit, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "dtype": w.dtype,
            "config": workload_config(w, flush),
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                         "unit": unit, "frac": achieved / peak,
                         "peak_source": peak_source,
                         "traffic": profiled_traffic(w),
                         "kernel": kernel_label(w)},
            "cpu_baseline": {"value": rate(cpu_units, cpu_s, unit), "unit": unit,
                             "cores": host_cores(), "kind": "oracle",
                             "sample": f"{cpu_desc} of one step, float64 NumPy, {cpu_s:.1f} s"},
            "parity": {"checked": f"{cpu_desc} of one warm-up step against the float64 oracle "
                                  "before timing",
                       "outputs": parity},
            "e2e": {"value": whole_job_rate(units, world, e2e_ms / 1e3, unit), "unit": unit,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
    del x, outs, out_map, step, host_pinned, out_host, flush_buf
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return entry


def run_gpu(args, w, extras):
    import torch
    import torch.distributed as dist

    import online_softmax_tiled_gb300 as ost

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    ost.lib()
    stream = torch.cuda.current_stream(dev)

    rc = 0
    try:
        main_entry = measure(args, w, ost, dev, world, rank, stream)
        extra_entries = {}
        for e in extras:
            extra_entries[e.name] = measure(args, e, ost, dev, world, rank, stream)
    except ParityError as err:
        print(str(err), file=sys.stderr)
        rc = 1
    if rc == 0 and rank == 0 and not args.profile:
        line = {"metric": METRIC, "value": main_entry["value"], "unit": main_entry["unit"],
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": main_entry["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic"}
        for key in ("config", "roofline", "cpu_baseline", "parity", "e2e", "gpu_launches",
                    "clocks"):
            line[key] = main_entry[key]
        if extra_entries:
            line["workloads"] = extra_entries
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return rc


DEFAULT_WORKLOAD = "fwd_causal_n8192_d128"
DEFAULT_EXTRA = ("bwd_causal_n4096_d128,decode_gqa_l4096,fwd_mha_n2048_d64,"
                 "fwd_gqa_causal_n8192_d128,bwd_gqa_causal_n4096_d128,decode_paged_gqa_l4096")


def main():
    from workloads import WORKLOADS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--extra", default=None,
                    help="comma-separated workloads timed after the top-level one and "
                         "reported under 'workloads' ('none': no others); default: "
                         f"{DEFAULT_EXTRA} when --workload is the default, else none")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of CPU oracle work for each cpu_baseline figure")
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up and timed launches, no JSON line (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    extra = args.extra
    if extra is None:
        extra = DEFAULT_EXTRA if args.workload == DEFAULT_WORKLOAD else "none"
    names = [n for n in extra.split(",") if n and n != "none" and n != w.name]
    for n in names:
        if n not in WORKLOADS:
            ap.error(f"unknown workload in --extra: {n}")
    return run_gpu(args, w, [WORKLOADS[n] for n in names])


if __name__ == "__main__":
    sys.exit(main())

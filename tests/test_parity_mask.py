"""GPU forward under general masks vs the float64 oracle.

Masks per the Flash Attention 2 post, section "Causal masking", option A:
sliding windows, attention sinks (global keys), prefix LM, documents packed
into one sequence, windows reaching right of the diagonal, Nq != Nk. The
tolerances are the benchmark description's: bf16 O <= 2e-2, LSE <= 1e-3;
float32 O and LSE <= 1e-5. Rows that see no key must give exactly O = 0 and
LSE = -inf.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, make_doc_bounds, make_inputs, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(ost, w, spec, rows=None):
    x = {k: t.to(DEV) for k, t in make_inputs(w).items()}
    rs = re = None
    if rows is not None:
        rs, re = rows[0].to(DEV), rows[1].to(DEV)
    mask = ost.make_mask(spec.get("window_left", -1), spec.get("window_right", -1),
                         spec.get("n_global", 0), rs, re)
    o, lse = ost.forward(x["q"], x["k"], x["v"], scale=w.scale, mask=mask)
    torch.cuda.synchronize()
    ospec = dict(spec)
    if rows is not None:
        ospec["row_kv_start"], ospec["row_kv_end"] = rows[0].numpy(), rows[1].numpy()
    o_ref, lse_ref = oracle.attention_fwd_masked(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                                 w.scale, ospec)
    return to_f64(o), to_f64(lse), o_ref, lse_ref


def _check(ost, w, spec, rows=None):
    o, lse, o_ref, lse_ref = _run(ost, w, spec, rows)
    tol_o, tol_l = (1e-5, 1e-5) if w.dtype == "f32" else (2e-2, 1e-3)
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(lse[empty])) and np.all(o[empty] == 0)
    assert not np.any(np.isneginf(lse[~empty]))
    assert np.max(np.abs(o - o_ref)) <= tol_o
    assert np.max(np.abs(lse[~empty] - lse_ref[~empty]), initial=0.0) <= tol_l
    return int(empty.sum())


SPECS = {
    "window100": {"window_left": 99, "window_right": 0},
    "sinks4_window64": {"window_left": 63, "window_right": 0, "n_global": 4},
    "prefix_lm77": {"window_left": -1, "window_right": 0, "n_global": 77},
    "local_both_sides": {"window_left": 40, "window_right": 25},
    "global_only_noncausal_window": {"window_left": 130, "window_right": 130, "n_global": 200},
}


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
@pytest.mark.parametrize("name", sorted(SPECS))
def test_window_and_global_masks(ost, dtype, d, name):
    w = Workload("mask", "fwd", 2, 4, 2, 530, 530, d, dtype, seed=d + len(name))
    _check(ost, w, SPECS[name])


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_document_masks(ost, dtype, d, causal):
    w = Workload("docs", "fwd", 2, 2, 1, 700, 700, d, dtype, seed=11 + int(causal))
    rows = make_doc_bounds(2, 700, 90, seed=5 + d)
    _check(ost, w, {"window_left": -1, "window_right": 0 if causal else -1}, rows)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("nq,nk,spec", [
    (600, 260, {"window_left": -1, "window_right": 0}),      # causal with Nq > Nk: empty rows
    (130, 700, {"window_left": 63, "window_right": 0}),      # decode-like suffix queries
    (257, 1000, {"window_left": 31, "window_right": 0, "n_global": 3}),
])
def test_unequal_lengths(ost, dtype, d, nq, nk, spec):
    w = Workload("ragged", "fwd", 1, 2, 2, nq, nk, d, dtype, seed=nq + nk)
    n_empty = _check(ost, w, spec)
    if nq > nk and spec.get("window_right") == 0:
        assert n_empty > 0


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_rows_without_keys_and_empty_tiles(ost, dtype, d):
    """Row ranges that are empty for whole 128-row query tiles: those tiles
    visit no key tile at all and still write O = 0, LSE = -inf."""
    N = 600
    start = torch.zeros((1, N), dtype=torch.int32)
    end = torch.full((1, N), N, dtype=torch.int32)
    end[0, 128:384] = 0                     # rows 128..383: nothing visible
    start[0, 450:] = 500                    # rows 450..: keys 500..599 only
    w = Workload("empty", "fwd", 1, 2, 1, N, N, d, dtype, seed=3)
    assert _check(ost, w, {"window_left": -1, "window_right": -1}, (start, end)) == 2 * 256


@pytest.mark.parametrize("d", [64, 128])
def test_causal_mask_equals_causal_call_bitwise(ost, d):
    w = Workload("causal", "fwd", 2, 4, 2, 700, 700, d, "bf16", seed=21)
    x = {k: t.to(DEV) for k, t in make_inputs(w).items()}
    o1, l1 = ost.forward(x["q"], x["k"], x["v"], causal=True, scale=w.scale)
    o2, l2 = ost.forward(x["q"], x["k"], x["v"], scale=w.scale, mask=ost.make_mask(-1, 0, 0))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

"""GPU backward vs the float64 oracle (JVP route), element by element.

Tolerance (from the benchmark description, written here): per gradient
tensor, max|err| <= 5e-2 * max|ref| for bf16 inputs with float32
accumulation; max|err| <= 1e-5 (absolute) for float32 inputs. The GPU takes O
and LSE from its own forward, as a training step would. Every assertion
message carries max|err| / max|ref|.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _grads(ost, w, scale=None):
    x = {k: t.to(DEV) for k, t in make_inputs(w).items()}
    scale = w.scale if scale is None else scale
    o, lse = ost.forward(x["q"], x["k"], x["v"], causal=w.causal, scale=scale)
    dq, dk, dv = ost.backward(x["q"], x["k"], x["v"], o, x["do"], lse, causal=w.causal,
                              scale=scale)
    torch.cuda.synchronize()
    return x, (dq, dk, dv), scale


def _check_grads(got, ref, dtype, where=""):
    """bf16: max|err| <= 5e-2 * max|ref| per gradient; float32: <= 1e-5."""
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g if isinstance(g, np.ndarray) else to_f64(g)
        err = float(np.max(np.abs(g - r)))
        mx = float(np.max(np.abs(r)))
        tol = 5e-2 * mx if dtype == "bf16" else 1e-5
        assert err <= tol, (name, where, f"max|err| {err:.3e}", f"max|ref| {mx:.3e}",
                            f"rel {err / mx if mx else float('nan'):.3e}", f"tol {tol:.3e}")


SMALL = [
    (1, 2, 2, 200, 200, 64, "bf16", True),
    (1, 2, 2, 300, 300, 128, "bf16", False),
    (1, 4, 2, 257, 257, 128, "bf16", True),      # GQA: dK, dV sum over the group
    (1, 2, 2, 130, 390, 64, "bf16", True),       # Nq < Nk
    (2, 2, 2, 64, 64, 128, "bf16", True),
    (1, 1, 1, 1, 77, 64, "bf16", False),
    (1, 2, 2, 100, 100, 64, "f32", True),
    (1, 4, 1, 90, 150, 128, "f32", False),
    # d = 128 bf16 runs the key-tile and query-tile passes: ragged tails on
    # both sides, Nq < Nk and Nq > Nk, one query row, GQA 8:1
    (1, 2, 2, 130, 390, 128, "bf16", True),
    (1, 8, 1, 200, 333, 128, "bf16", False),
    (1, 1, 1, 1, 300, 128, "bf16", True),
    (1, 2, 2, 513, 129, 128, "bf16", False),
    # more 128-row query tiles (176) than SMs: the persistent dQ pass runs
    # several tiles per CTA, taken from its work counter; GQA 4:1
    (2, 8, 2, 1400, 1400, 128, "bf16", True),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,causal", SMALL)
def test_small_shapes(ost, B, Hq, Hkv, Nq, Nk, d, dtype, causal):
    w = Workload("small", "bwd", B, Hq, Hkv, Nq, Nk, d, dtype, causal, seed=Nq * 7 + Nk)
    x, got, scale = _grads(ost, w)
    ref = oracle.attention_bwd(*(to_f64(x[n]) for n in ("q", "k", "v", "do")), scale, causal)
    _check_grads(got, ref, dtype)


def test_peaked_rows(ost):
    w = Workload("peaked", "bwd", 1, 2, 2, 256, 256, 128, "bf16", True, seed=21)
    x, got, scale = _grads(ost, w, scale=8.0 / np.sqrt(128))
    ref = oracle.attention_bwd(*(to_f64(x[n]) for n in ("q", "k", "v", "do")), scale, True)
    _check_grads(got, ref, "bf16", "peaked")


def test_causal_backward_workload_sampled_heads(ost):
    """B=2, H=16, N=4096, d=128 causal bf16 at full size; the oracle computes
    whole heads (dK, dV of a head need every query row of it): the two corner
    heads and two interior ones."""
    w = WORKLOADS["bwd_causal_n4096_d128"]
    x, got, scale = _grads(ost, w)
    for b, h in [(0, 0), (0, 7), (1, 9), (1, 15)]:
        sl = lambda t: to_f64(t[b:b + 1, h:h + 1])
        ref = oracle.attention_bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"]), scale, True)
        _check_grads([sl(g) for g in got], ref, "bf16", (b, h))


def test_gqa_backward_workload_sampled_kv_head(ost):
    """B=2, Hq=16, Hkv=4, N=4096, d=128 causal bf16: dK and dV of a KV head
    sum over its four query heads; the oracle computes one whole group (the
    four query heads and their KV head) at each end of the batch."""
    w = WORKLOADS["bwd_gqa_causal_n4096_d128"]
    x, got, scale = _grads(ost, w)
    for b, g in [(0, 0), (1, 3)]:
        hs = slice(4 * g, 4 * g + 4)
        qs = lambda t: to_f64(t[b:b + 1, hs])
        ks = lambda t: to_f64(t[b:b + 1, g:g + 1])
        ref = oracle.attention_bwd(qs(x["q"]), ks(x["k"]), ks(x["v"]), qs(x["do"]), scale, True)
        _check_grads([qs(got[0]), ks(got[1]), ks(got[2])], ref, "bf16", (b, g))

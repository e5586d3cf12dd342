"""The decode entry point that allocates nothing.

attn_decode_splitkv_noalloc serves callers that cannot allocate device
memory at decode time (memory partitioned up front, or a host program that
owns every allocation): its split partials live in a fixed array inside the
library instead of a caller workspace. Here it is called through the C ABI
twice in a row, on different inputs, and each result is compared with the
workspace entry point's result for the same inputs and with the float64
oracle, within the decode tolerance used by the other tests (O 2e-2, LSE
1e-3). This file is collected last so that a failure here cannot hide any
other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ATTN_ERR_WORKSPACE = -4


def _call_noalloc(ost, x, w):
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[:2], dtype=torch.float32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ost.lib().attn_decode_splitkv_noalloc(p(x["q"]), p(x["k"]), p(x["v"]), p(o), p(lse),
                                               w.B, w.Hq, w.Hkv, w.Nk, w.d, w.scale,
                                               w.num_splits, stream)
    return st, o, lse


def test_noalloc_decode_matches_workspace_decode_twice(ost):
    cases = [
        Workload("noalloc_a", "decode", 8, 16, 4, 1, 1000, 128, "bf16", num_splits=8, seed=31),
        Workload("noalloc_b", "decode", 3, 8, 2, 1, 333, 64, "bf16", num_splits=5, seed=32),
    ]
    for w in cases:  # two calls in a row on the shared array
        x = {k: t.to(DEV) for k, t in make_inputs(w).items()}
        o_ref, lse_ref = ost.decode(x["q"], x["k"], x["v"], w.num_splits, w.scale)
        st, o, lse = _call_noalloc(ost, x, w)
        assert st == 0, ost.attn_status_string(st)
        torch.cuda.synchronize()
        assert ost.attn_sync_status() == 0
        assert np.max(np.abs(to_f64(o) - to_f64(o_ref))) <= 2e-2
        assert np.max(np.abs(to_f64(lse) - to_f64(lse_ref))) <= 1e-3
        o64, lse64 = oracle.decode_splitkv(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                           w.scale, w.num_splits)
        assert np.max(np.abs(to_f64(o) - o64)) <= 2e-2
        assert np.max(np.abs(to_f64(lse) - lse64)) <= 1e-3


def test_noalloc_decode_rejects_oversized_partials(ost):
    # 64 x 64 x 64 (row, split) pairs of 130 floats = 136 MB > 24 MiB: rejected, nothing launched
    w = Workload("noalloc_big", "decode", 64, 64, 8, 1, 64, 128, "bf16", num_splits=64, seed=33)
    x = {k: torch.zeros(t.shape, dtype=t.dtype, device=DEV) for k, t in
         {"q": torch.empty(64, 64, 128, dtype=torch.bfloat16),
          "k": torch.empty(64, 8, 64, 128, dtype=torch.bfloat16),
          "v": torch.empty(64, 8, 64, 128, dtype=torch.bfloat16)}.items()}
    need = ost.attn_decode_workspace_size(w.B, w.Hq, w.d, w.num_splits)
    assert need > 24 * 1024 * 1024
    st, _, _ = _call_noalloc(ost, x, w)
    assert st == ATTN_ERR_WORKSPACE

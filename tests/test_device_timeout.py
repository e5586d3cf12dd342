"""A bounded device wait that runs out reaches the caller as a status.

Every wait inside the library's kernels is bounded; when one runs out the
kernel records a timeout in the device error word and returns, and
attn_sync_status reports ATTN_ERR_DEVICE_TIMEOUT. Here the library's
self-test kernel waits, with that same bounded wait, on a barrier nothing
arrives on (no bulk copy or tensor-core operation is in flight), so the
wait runs out after a short limit. The status must be the timeout, reading
it must clear it, and the context must stay usable: a decode right after
it runs and matches the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, make_inputs, to_f64

ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_DEVICE_TIMEOUT = -6


def test_selftest_rejects_limits_out_of_range():
    """Argument checks happen before any launch, so this needs no GPU."""
    import __graft_entry__
    __graft_entry__.build()
    import online_softmax_tiled_gb300 as ost
    for limit in (0, 1_000_001, 2**32 - 1):
        assert ost.lib().attn_selftest_bounded_wait(limit, None) == ATTN_ERR_INVALID_ARG


@pytest.mark.gpu
def test_wait_that_runs_out_reports_timeout_then_clean(ost):
    torch.cuda.synchronize()
    assert ost.attn_sync_status() == ost.ATTN_OK
    for limit_us in (1000, 20000):
        ost.attn_selftest_bounded_wait(limit_us)
        assert ost.attn_sync_status() == ATTN_ERR_DEVICE_TIMEOUT
        assert ost.attn_sync_status() == ost.ATTN_OK      # reading cleared the word
    # the context is intact: a real call runs and matches the oracle
    w = Workload("after_timeout", "decode", 2, 8, 2, 1, 300, 128, "bf16", num_splits=4, seed=61)
    x = {k: t.to("cuda:0") for k, t in make_inputs(w).items()}
    o, lse = ost.decode(x["q"], x["k"], x["v"], w.num_splits, w.scale)
    assert ost.attn_sync_status() == ost.ATTN_OK
    o_ref, lse_ref = oracle.decode_splitkv(to_f64(x["q"]), to_f64(x["k"]), to_f64(x["v"]),
                                           w.scale, w.num_splits)
    assert np.max(np.abs(to_f64(o) - o_ref)) <= 2e-2
    assert np.max(np.abs(to_f64(lse) - lse_ref)) <= 1e-3

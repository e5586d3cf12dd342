"""GPU paged, variable-length decode vs the float64 oracle.

The cache is a pool of fixed-size KV blocks reached through a per-request
block table (ML notes, KV-cache Q&A: block table as page table); each
request has its own length. Tolerance as for contiguous decode (benchmark
description): bf16 O max|err| <= 2e-2, LSE <= 1e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, Workload, make_inputs, make_paged_inputs, to_f64

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ATTN_ERR_DEVICE_INDEX = -7


def _to_dev(x):
    return {k: t.to(DEV) for k, t in x.items()}


def _run(ost, w, x):
    o, lse = ost.decode_paged(x["q"], x["k_pages"], x["v_pages"], x["block_table"],
                              x["seq_lens"], w.num_splits, w.scale)
    torch.cuda.synchronize()
    return o, lse


def _oracle(w, x):
    return oracle.decode_paged(to_f64(x["q"]), to_f64(x["k_pages"]), to_f64(x["v_pages"]),
                               x["block_table"].cpu().numpy(), x["seq_lens"].cpu().numpy(),
                               w.page_size, w.scale)


def _check(ost, w, seq_lens=None):
    x = _to_dev(make_paged_inputs(w, seq_lens))
    o, lse = _run(ost, w, x)
    o_ref, lse_ref = _oracle(w, x)
    got_o, got_lse = to_f64(o), to_f64(lse)
    err, mx = np.max(np.abs(got_o - o_ref)), np.max(np.abs(o_ref))
    msg = (f"max|err| {err:.3e}", f"max|ref| {mx:.3e}", f"rel {err / max(mx, 1e-30):.3e}")
    assert err <= 2e-2, msg
    assert err <= 1e-2 * mx, msg     # |O| is a few hundredths: a relative bound too
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(got_lse[empty])) and np.all(got_o[empty] == 0)
    assert np.max(np.abs(got_lse[~empty] - lse_ref[~empty]), initial=0.0) <= 1e-3


def test_paged_gqa_workload_full(ost):
    """B=64, Hq=32, Hkv=8, d=128, 16-token blocks, ragged lengths of mean
    4096, 16 splits: every output row."""
    _check(ost, WORKLOADS["decode_paged_gqa_l4096"])


def test_large_batch_long_chunks_at_their_boundaries(ost):
    """A batch large enough for the split grid to take chunks longer than
    capacity / num_splits (64 requests x 8 KV heads: 512-key chunks double
    to 1024 on a full device), with lengths on either side of the chunk
    boundaries, at the table's capacity, and empty: every output row."""
    w = Workload("paged_long_chunks", "decode_paged", 64, 32, 8, 1, 4096, 128, "bf16",
                 num_splits=16, seed=91, page_size=16)
    pattern = [1, 511, 512, 513, 1023, 1024, 1025, 2047, 2048, 4097, 8191, 8192, 0, 3000, 32, 33]
    _check(ost, w, [pattern[i % len(pattern)] for i in range(w.B)])


@pytest.mark.parametrize("B,Hq,Hkv,d,page,S,lens", [
    (4, 8, 2, 128, 32, 4, [0, 1, 31, 33]),         # an empty request, one key, ragged tails
    (3, 16, 2, 64, 16, 7, [300, 5, 1000]),         # group of 8, pages of 16 keys
    (2, 16, 2, 128, 16, 5, [777, 40]),             # group of 8 at d = 128 (a CTA pair)
    (2, 4, 4, 128, 64, 16, [2048, 100]),           # MHA; the short request leaves splits empty
    (2, 8, 1, 128, 48, 5, [777, 96]),              # stages straddle 48-key pages
    (2, 8, 2, 64, 1, 3, [70, 33]),                 # one key per page
    (1, 4, 2, 128, 16, 1, [4096]),                 # one split covers everything
    (5, 8, 4, 64, 128, 3, None),                   # drawn lengths, large pages
    (3, 8, 8, 128, 256, 2, [0, 0, 513]),           # two empty requests
])
def test_small_shapes(ost, B, Hq, Hkv, d, page, S, lens):
    w = Workload("paged", "decode_paged", B, Hq, Hkv, 1, 200, d, "bf16", num_splits=S,
                 seed=B * 100 + page + S, page_size=page)
    _check(ost, w, lens)


def test_identity_paging_equals_contiguous_decode_bitwise(ost):
    """A contiguous cache cut into 64-key pages in order, read through an
    identity block table with every length L, gives bit-for-bit the
    contiguous decode's result (same chunks: ceil(4096/16) = 256 keys)."""
    w = Workload("contig", "decode", 4, 16, 4, 1, 4096, 128, "bf16", num_splits=16, seed=41)
    x = _to_dev(make_inputs(w))
    o_ref, lse_ref = ost.decode(x["q"], x["k"], x["v"], w.num_splits, w.scale)
    P, n = 64, 4096 // 64

    def pages(t):  # [B, Hkv, L, d] -> [B * L/P, Hkv, P, d], request-major
        return t.view(w.B, w.Hkv, n, P, w.d).permute(0, 2, 1, 3, 4).reshape(-1, w.Hkv, P, w.d)

    table = torch.arange(w.B * n, dtype=torch.int32, device=DEV).view(w.B, n)
    lens = torch.full((w.B,), 4096, dtype=torch.int32, device=DEV)
    o, lse = ost.decode_paged(x["q"], pages(x["k"]).contiguous(), pages(x["v"]).contiguous(),
                              table, lens, w.num_splits, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_out_of_range_indices_are_flagged_not_read(ost):
    """A page index outside the pool and a length past the table are caught
    on the device: those requests read nothing (an empty request: O = 0,
    LSE = -inf for the bad length), the status says so, and the other
    requests are exact."""
    w = Workload("bad", "decode_paged", 4, 8, 2, 1, 200, 128, "bf16", num_splits=4, seed=7,
                 page_size=32)
    x = _to_dev(make_paged_inputs(w, [100, 200, 64, 150]))
    o_ref, lse_ref = _oracle(w, x)
    max_pages = x["block_table"].shape[1]
    x["block_table"][1, 2] = x["k_pages"].shape[0] + 5      # past the pool
    x["seq_lens"][3] = max_pages * w.page_size + 1           # past the table
    o, lse = _run(ost, w, x)
    assert ost.attn_sync_status() == ATTN_ERR_DEVICE_INDEX
    assert ost.attn_sync_status() == 0                        # reading clears it
    got_o, got_lse = to_f64(o), to_f64(lse)
    for b in (0, 2):
        assert np.max(np.abs(got_o[b] - o_ref[b])) <= 2e-2
        assert np.max(np.abs(got_lse[b] - lse_ref[b])) <= 1e-3
    assert np.all(got_o[3] == 0) and np.all(np.isneginf(got_lse[3]))

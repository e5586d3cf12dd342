"""Seeded synthetic workloads: shapes and input tensors.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__``. It
holds only shapes, seeds and random draws: none of the attention arithmetic
(that lives in the CUDA library and, separately, in the test oracle).

Recipe: one CPU ``torch.Generator`` seeded per workload; float32 N(0, 1)
draws in the order Q, K, V, then dO for a backward workload; each tensor is
then cast to the workload's dtype (bf16 by round-to-nearest-even). Both the
GPU path and the oracle see exactly these cast values.

Paged decode: per-request lengths uniform on [1, 2·Nk − 1] (mean Nk) unless
given; the pool holds exactly the pages the requests need plus a few spare
ones, drawn N(0, 1) as [num_pages, Hkv, page_size, d] for K then V, and the
pages are handed out to the requests in a random order (a seeded
permutation), so that logically consecutive blocks sit at scattered physical
addresses. Block-table entries past a request's last block are -1.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "fwd", "bwd" or "decode"
    B: int
    Hq: int
    Hkv: int
    Nq: int            # query rows per head (1 for decode)
    Nk: int            # key rows per head (KV length for decode)
    d: int
    dtype: str         # "f32" or "bf16"
    causal: bool = False
    num_splits: int = 1
    seed: int = 0
    page_size: int = 0  # paged decode only: tokens per KV block
    # general mask (forward): window around the diagonal (-1: unbounded),
    # keys visible to every row, packed documents of this mean length
    window_left: int = -1
    window_right: int = -1
    n_global: int = 0
    doc_mean: int = 0
    n_index: int = 0    # sparse-index decode: listed rows per request (Nq = tokens T)

    @property
    def masked(self) -> bool:
        return self.window_left >= 0 or self.n_global > 0 or self.doc_mean > 0 or (
            self.window_right >= 0 and not self.causal)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


# The five workloads of the benchmark description, by what they are.
WORKLOADS = {
    "fwd_f32_single_head": Workload("fwd_f32_single_head", "fwd", 1, 1, 1, 256, 256, 64, "f32"),
    "fwd_mha_n2048_d64": Workload("fwd_mha_n2048_d64", "fwd", 4, 16, 16, 2048, 2048, 64, "bf16"),
    "fwd_causal_n8192_d128": Workload("fwd_causal_n8192_d128", "fwd", 2, 32, 32, 8192, 8192, 128,
                                      "bf16", causal=True),
    "bwd_causal_n4096_d128": Workload("bwd_causal_n4096_d128", "bwd", 2, 16, 16, 4096, 4096, 128,
                                      "bf16", causal=True),
    "decode_gqa_l4096": Workload("decode_gqa_l4096", "decode", 64, 32, 8, 1, 4096, 128, "bf16",
                                 num_splits=16),
    # The long-context forward shape under a causal sliding window of 1024
    # keys, and causal within packed documents of mean length 1024.
    "fwd_swa_n8192_d128_w1024": Workload("fwd_swa_n8192_d128_w1024", "fwd", 2, 32, 32, 8192, 8192,
                                         128, "bf16", window_left=1023, window_right=0),
    "fwd_docs_n8192_d128": Workload("fwd_docs_n8192_d128", "fwd", 2, 32, 32, 8192, 8192, 128,
                                    "bf16", window_right=0, doc_mean=1024, seed=1),
    # The causal backward shape under a sliding window of 1024 keys.
    "bwd_swa_n4096_d128_w1024": Workload("bwd_swa_n4096_d128_w1024", "bwd", 2, 16, 16, 4096,
                                         4096, 128, "bf16", window_left=1023, window_right=0),
    # The long-context forward and the causal backward with grouped-query
    # heads: four query heads per KV head (8 KV heads of 32; 4 of 16).
    "fwd_gqa_causal_n8192_d128": Workload("fwd_gqa_causal_n8192_d128", "fwd", 2, 32, 8, 8192,
                                          8192, 128, "bf16", causal=True),
    "bwd_gqa_causal_n4096_d128": Workload("bwd_gqa_causal_n4096_d128", "bwd", 2, 16, 4, 4096,
                                          4096, 128, "bf16", causal=True),
    # Sparse-index decode as the ML notes' split-K kernel notes describe it:
    # T = 8 query tokens, 16 heads, 2048 listed rows per request, 32 splits;
    # 8 requests with caches of 16384 rows.
    "decode_sparse_t8_i2048": Workload("decode_sparse_t8_i2048", "decode_sparse", 8, 16, 16, 8,
                                       16384, 128, "bf16", num_splits=32, n_index=2048),
    # The GQA decode shape over a paged cache of 16-token blocks, with ragged
    # request lengths of mean 4096.
    "decode_paged_gqa_l4096": Workload("decode_paged_gqa_l4096", "decode_paged", 64, 32, 8, 1,
                                       4096, 128, "bf16", num_splits=16, page_size=16),
}


def make_inputs(w: Workload, *, Hkv: int | None = None, generator_seed: int | None = None):
    """Seeded CPU tensors for workload ``w``.

    fwd/bwd: q [B, Hq, Nq, d], k, v [B, Hkv, Nk, d] (+ do like q for bwd).
    decode:  q [B, Hq, d], k, v [B, Hkv, L, d].
    """
    g = torch.Generator().manual_seed(w.seed if generator_seed is None else generator_seed)
    hkv = w.Hkv if Hkv is None else Hkv
    if w.kind == "decode":
        q_shape = (w.B, w.Hq, w.d)
    else:
        q_shape = (w.B, w.Hq, w.Nq, w.d)
    kv_shape = (w.B, hkv, w.Nk, w.d)
    out = {
        "q": torch.randn(q_shape, generator=g, dtype=torch.float32),
        "k": torch.randn(kv_shape, generator=g, dtype=torch.float32),
        "v": torch.randn(kv_shape, generator=g, dtype=torch.float32),
    }
    if w.kind == "bwd":
        out["do"] = torch.randn(q_shape, generator=g, dtype=torch.float32)
    return {k: t.to(w.torch_dtype) for k, t in out.items()}


def make_paged_inputs(w: Workload, seq_lens=None, spare_pages: int = 3):
    """Seeded CPU tensors for a paged decode workload.

    q [B, Hq, d]; k_pages, v_pages [num_pages, Hkv, page_size, d];
    block_table [B, max_pages] int32 (-1 past each request's blocks);
    seq_lens [B] int32. ``seq_lens`` overrides the drawn lengths.
    """
    g = torch.Generator().manual_seed(w.seed)
    P = w.page_size
    if seq_lens is None:
        seq_lens = torch.randint(1, 2 * w.Nk, (w.B,), generator=g)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)
    blocks = [(int(n) + P - 1) // P for n in seq_lens]
    max_pages = max(1, max(blocks))
    num_pages = sum(blocks) + spare_pages
    q = torch.randn((w.B, w.Hq, w.d), generator=g, dtype=torch.float32)
    kp = torch.randn((num_pages, w.Hkv, P, w.d), generator=g, dtype=torch.float32)
    vp = torch.randn((num_pages, w.Hkv, P, w.d), generator=g, dtype=torch.float32)
    order = torch.randperm(num_pages, generator=g)
    table = torch.full((w.B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b, nb in enumerate(blocks):
        table[b, :nb] = order[nxt:nxt + nb].to(torch.int32)
        nxt += nb
    dt = w.torch_dtype
    return {"q": q.to(dt), "k_pages": kp.to(dt), "v_pages": vp.to(dt), "block_table": table,
            "seq_lens": seq_lens}


def make_sparse_inputs(w: Workload, counts=None):
    """Seeded CPU tensors for sparse-index decode: q [B, Hq, T, d]; k, v
    [B, Hkv, L, d] drawn N(0, 1); per request n_index distinct rows drawn
    uniformly from [0, L) in random order (indices [B, n_index] int32);
    counts [B] int32 (all n_index unless given)."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.Hq, w.Nq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.Nk, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Nk, w.d), generator=g, dtype=torch.float32)
    idx = torch.stack([torch.randperm(w.Nk, generator=g)[:w.n_index] for _ in range(w.B)])
    cnt = torch.full((w.B,), w.n_index) if counts is None else torch.as_tensor(counts)
    dt = w.torch_dtype
    return {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt), "indices": idx.to(torch.int32),
            "counts": cnt.to(torch.int32)}


def make_doc_bounds(B: int, N: int, mean_len: int, seed: int):
    """Documents packed back to back in each of B sequences of N tokens:
    lengths drawn uniformly from [1, 2·mean_len - 1] (the last one cut at N).
    Returns int32 CPU tensors row_kv_start, row_kv_end [B, N]: the key range
    [start, end) of each token's document."""
    g = torch.Generator().manual_seed(seed)
    start = torch.empty((B, N), dtype=torch.int32)
    end = torch.empty((B, N), dtype=torch.int32)
    for b in range(B):
        s = 0
        while s < N:
            n = int(torch.randint(1, 2 * mean_len, (1,), generator=g))
            e = min(N, s + n)
            start[b, s:e] = s
            end[b, s:e] = e
            s = e
    return start, end


def random_like_shape(shape, dtype: torch.dtype, seed: int, scale: float = 1.0):
    """N(0, scale²) draws of a given shape from a seeded CPU generator."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(dtype)


def to_f64(t: torch.Tensor):
    """Exact upcast of a CPU or GPU tensor to a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()

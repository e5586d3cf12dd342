"""ctypes binding of the C ABI in ``include/attn.h``.

Argument marshalling only: torch tensors supply device pointers, shapes and
the current CUDA stream; every step of the computation runs in the library's
CUDA kernels. If the library is missing the import fails loudly; there is no
fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH

ATTN_OK = 0
ATTN_F32 = 0
ATTN_BF16 = 1

_STATUS_NAMES = {
    0: "ATTN_OK", -1: "ATTN_ERR_INVALID_ARG", -2: "ATTN_ERR_UNSUPPORTED",
    -3: "ATTN_ERR_MISALIGNED", -4: "ATTN_ERR_WORKSPACE", -5: "ATTN_ERR_CUDA",
    -6: "ATTN_ERR_DEVICE_TIMEOUT", -7: "ATTN_ERR_DEVICE_INDEX",
}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS_NAMES.get(status, status)} "
                         f"({lib().attn_status_string(status).decode()})")


_LIB = None


class AttnMask(ctypes.Structure):
    """The C ``attn_mask``: window (left, right; -1 = unbounded), n_global
    keys visible to every row, optional per-row key ranges [B, Nq] int32."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("n_global", ctypes.c_int), ("row_kv_start", ctypes.c_void_p),
                ("row_kv_end", ctypes.c_void_p)]

_SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 +
                 [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_masked": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 +
                        [ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]),
    "attn_bwd_masked": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 +
                        [ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                         ctypes.c_size_t, ctypes.c_void_p]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 6),
    "attn_bwd_workspace_size_dt": (ctypes.c_size_t, [ctypes.c_int] * 7),
    "attn_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint, ctypes.c_void_p]),
    "attn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 +
                 [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_void_p]),
    "attn_decode_workspace_size": (ctypes.c_size_t, [ctypes.c_int] * 4),
    "attn_decode_splitkv": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 +
                            [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                             ctypes.c_void_p]),
    "attn_decode_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 7 +
                          [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                           ctypes.c_void_p]),
    "attn_decode_sparse": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 7 +
                           [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                            ctypes.c_void_p]),
    "attn_merge_partials": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 +
                            [ctypes.c_void_p]),
    "attn_decode_splitkv_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 +
                                    [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_sync_status": (ctypes.c_int, [ctypes.c_void_p]),
}


def lib() -> ctypes.CDLL:
    """Load the in-tree library (built by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built ({LIB_PATH} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


# ------------------------------------------------------------------ helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _device_contig(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on the GPU (device pointers)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _check(status: int, what: str):
    if status != ATTN_OK:
        raise AttnError(status, what)


# ------------------------------------------------ the C entry points by name

def attn_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None):
    """attn_fwd on torch tensors: q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d], o like q,
    lse [B,Hq,Nq] float32 or None."""
    _device_contig(q, k, v, o, lse)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                        float(scale), int(bool(causal)), _dt(q), _stream(stream))
    _check(st, "attn_fwd")


def make_mask(window_left=-1, window_right=-1, n_global=0, row_kv_start=None,
              row_kv_end=None) -> AttnMask:
    """An ``attn_mask``; the row ranges are int32 device tensors [B, Nq]
    kept alive by the caller for as long as the call runs."""
    for t in (row_kv_start, row_kv_end):
        if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous()):
            raise ValueError("row ranges must be contiguous int32 device tensors")
    return AttnMask(int(window_left), int(window_right), int(n_global),
                    None if row_kv_start is None else row_kv_start.data_ptr(),
                    None if row_kv_end is None else row_kv_end.data_ptr())


def attn_fwd_masked(q, k, v, o, lse, scale: float, mask, stream=None):
    """attn_fwd under an ``attn_mask`` (``make_mask``; None: no mask)."""
    _device_contig(q, k, v, o, lse)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    m = None if mask is None else ctypes.byref(mask)
    st = lib().attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq,
                               Nk, d, float(scale), m, _dt(q), _stream(stream))
    _check(st, "attn_fwd_masked")


def attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, d, dtype=None) -> int:
    """Workspace bytes of attn_bwd: for ``dtype`` (torch.float32 or
    torch.bfloat16) the exact need, else the largest over dtypes."""
    if dtype is None:
        return int(lib().attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, d))
    dt = ATTN_F32 if dtype == torch.float32 else ATTN_BF16 if dtype == torch.bfloat16 else None
    if dt is None:
        raise TypeError(f"unsupported dtype {dtype}: float32 or bfloat16")
    return int(lib().attn_bwd_workspace_size_dt(B, Hq, Hkv, Nq, Nk, d, dt))


def attn_bwd(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool, workspace,
             stream=None):
    _device_contig(q, k, v, o, do, lse, dq, dk, dv, workspace)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                        _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, d, float(scale),
                        int(bool(causal)), _dt(q), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "attn_bwd")


def attn_bwd_masked(q, k, v, o, do, lse, dq, dk, dv, scale: float, mask, workspace,
                    stream=None):
    """attn_bwd under an ``attn_mask`` (``make_mask``; None: no mask)."""
    _device_contig(q, k, v, o, do, lse, dq, dk, dv, workspace)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    m = None if mask is None else ctypes.byref(mask)
    st = lib().attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                               _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, d, float(scale), m, _dt(q),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(st, "attn_bwd_masked")


def attn_decode_workspace_size(B, Hq, d, num_splits) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, d, num_splits))


def attn_decode_splitkv(q, k_cache, v_cache, o, lse, scale: float, num_splits: int, workspace,
                        stream=None):
    """q [B,Hq,d], caches [B,Hkv,L,d] bf16; o [B,Hq,d] bf16; lse [B,Hq] or None."""
    _device_contig(q, k_cache, v_cache, o, lse, workspace)
    B, Hq, d = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    st = lib().attn_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B,
                                   Hq, Hkv, L, d, float(scale), int(num_splits), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "attn_decode_splitkv")


def attn_decode_splitkv_noalloc(q, k_cache, v_cache, o, lse, scale: float, num_splits: int,
                                stream=None):
    """Split-KV decode whose partials live in the library's fixed scratch array
    (no workspace argument): for callers that cannot allocate device memory
    when they decode. Same shapes and results as attn_decode_splitkv."""
    _device_contig(q, k_cache, v_cache, o, lse)
    B, Hq, d = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    st = lib().attn_decode_splitkv_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o),
                                           _ptr(lse), B, Hq, Hkv, L, d, float(scale),
                                           int(num_splits), _stream(stream))
    _check(st, "attn_decode_splitkv_noalloc")


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, scale: float,
                      num_splits: int, workspace, stream=None):
    """q [B,Hq,d] bf16; pages [num_pages,Hkv,page_size,d] bf16; block_table
    [B,max_pages] and seq_lens [B] int32 on the device; o [B,Hq,d] bf16;
    lse [B,Hq] float32 or None."""
    _device_contig(q, k_pages, v_pages, block_table, seq_lens, o, lse, workspace)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Hq, d = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    st = lib().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                 _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, num_pages,
                                 page_size, block_table.shape[1], d, float(scale),
                                 int(num_splits), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "attn_decode_paged")


def attn_decode_sparse(q, k_cache, v_cache, indices, counts, o, lse, scale: float,
                       num_splits: int, workspace, stream=None):
    """q [B,Hq,T,d] bf16; caches [B,Hkv,L,d] bf16; indices [B,max_idx] and
    counts [B] int32 on the device; o [B,Hq,T,d] bf16; lse [B,Hq,T] or None."""
    _device_contig(q, k_cache, v_cache, indices, counts, o, lse, workspace)
    if indices.dtype != torch.int32 or counts.dtype != torch.int32:
        raise TypeError("indices and counts must be int32")
    B, Hq, T, d = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    st = lib().attn_decode_sparse(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(indices),
                                  _ptr(counts), _ptr(o), _ptr(lse), B, Hq, Hkv, T, L,
                                  indices.shape[1], d, float(scale), int(num_splits),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(st, "attn_decode_sparse")


def attn_merge_partials(o_part, m_part, l_part, o, lse, stream=None):
    """o_part [rows,S,d], m_part/l_part [rows,S] float32 -> o [rows,d], lse [rows]."""
    _device_contig(o_part, m_part, l_part, o, lse)
    rows, S, d = o_part.shape
    st = lib().attn_merge_partials(_ptr(o_part), _ptr(m_part), _ptr(l_part), _ptr(o), _ptr(lse),
                                   rows, S, d, _dt(o), _stream(stream))
    _check(st, "attn_merge_partials")


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(status).decode()


def attn_sync_status(stream=None) -> int:
    return int(lib().attn_sync_status(_stream(stream)))


def attn_selftest_bounded_wait(limit_us: int, stream=None):
    """Launch the bounded-wait self-test (a wait that runs out after
    ``limit_us``); the next attn_sync_status reports the timeout."""
    _check(lib().attn_selftest_bounded_wait(int(limit_us), _stream(stream)),
           "attn_selftest_bounded_wait")


# ------------------------------------------- allocating conveniences (torch)

def forward(q, k, v, causal: bool = False, scale: float | None = None, with_lse: bool = True,
            stream=None, mask: AttnMask | None = None):
    """O, LSE = attention(q, k, v); outputs allocated by torch on q's device.
    ``mask`` (``make_mask``) replaces ``causal`` when given."""
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if with_lse else None
    if mask is not None:
        attn_fwd_masked(q, k, v, o, lse, scale, mask, stream)
    else:
        attn_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
             stream=None, mask: AttnMask | None = None):
    """dQ, dK, dV by recomputation from the forward's O and LSE (``mask``, the
    forward's mask, replaces ``causal`` when given)."""
    B, Hq, Nq, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    ws = torch.empty(attn_bwd_workspace_size(B, Hq, k.shape[1], Nq, k.shape[2], d, q.dtype),
                     dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if mask is not None:
        attn_bwd_masked(q, k, v, o, do, lse, dq, dk, dv, scale, mask, ws, stream)
    else:
        attn_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal, ws, stream)
    return dq, dk, dv


def decode(q, k_cache, v_cache, num_splits: int, scale: float | None = None, stream=None,
           workspace=None):
    """Split-KV decode: O [B,Hq,d] bf16 and LSE [B,Hq] float32."""
    B, Hq, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, Hq, d, num_splits),
                                dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    attn_decode_splitkv(q, k_cache, v_cache, o, lse, scale, num_splits, workspace, stream)
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, num_splits: int,
                 scale: float | None = None, stream=None, workspace=None):
    """Paged, variable-length split-KV decode: O [B,Hq,d] bf16, LSE [B,Hq] float32."""
    B, Hq, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, Hq, d, num_splits),
                                dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, scale, num_splits,
                      workspace, stream)
    return o, lse


def decode_sparse(q, k_cache, v_cache, indices, counts, num_splits: int,
                  scale: float | None = None, stream=None, workspace=None):
    """Sparse-index decode of T tokens per request: O [B,Hq,T,d] bf16, LSE [B,Hq,T]."""
    B, Hq, T, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, Hq * T, d, num_splits),
                                dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    attn_decode_sparse(q, k_cache, v_cache, indices, counts, o, lse, scale, num_splits, workspace,
                       stream)
    return o, lse

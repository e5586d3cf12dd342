"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, sizes workspaces as documented, and rejects bad arguments
before launching anything (these calls never reach a kernel)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import online_softmax_tiled_gb300 as ost
    return ost.lib()


def _declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    assert {"attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_decode_splitkv",
            "attn_decode_workspace_size", "attn_decode_paged", "attn_merge_partials",
            "attn_fwd_masked", "attn_bwd_masked", "attn_decode_sparse",
            "attn_status_string", "attn_sync_status"} <= names


def test_library_exports_every_declared_symbol(lib):
    from online_softmax_tiled_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # nothing else with the attn_ prefix leaks out of the library
    assert {n for n in exported if n.startswith("attn_")} == set(_declared_functions())


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        s = lib.attn_status_string(code)
        assert s and s != b"unknown status"
    assert lib.attn_status_string(42) == b"unknown status"


def _a256(x):
    return (x + 255) // 256 * 256


def test_workspace_sizes(lib):
    B, H, N, d = 2, 16, 4096, 128
    rows = B * H * N
    # row term, 256 bytes for the dQ pass's work counter, float32 dQ accumulator
    assert lib.attn_bwd_workspace_size(B, H, H, N, N, d) == \
        _a256(rows * 4) + 256 + _a256(rows * d * 4)
    B, Hq, d, S = 64, 32, 128, 16
    n = B * Hq * S
    assert lib.attn_decode_workspace_size(B, Hq, d, S) == _a256(n * d * 4) + 2 * _a256(n * 4)
    assert lib.attn_bwd_workspace_size(0, 1, 1, 1, 1, 64) == 0
    assert lib.attn_decode_workspace_size(1, 1, 64, 0) == 0
    # per dtype: bf16 at d = 128 writes dQ directly and needs only the row term
    B, H, N = 2, 16, 4096
    rows = B * H * N
    assert lib.attn_bwd_workspace_size_dt(B, H, H, N, N, 128, 1) == _a256(rows * 4) + 256
    for d, dt in ((64, 1), (128, 0), (64, 0)):
        assert lib.attn_bwd_workspace_size_dt(B, H, H, N, N, d, dt) == \
            lib.attn_bwd_workspace_size(B, H, H, N, N, d)
    assert lib.attn_bwd_workspace_size_dt(B, H, H, N, N, 128, 7) == 0
    assert lib.attn_bwd_workspace_size_dt(0, H, H, N, N, 128, 1) == 0


P = 1 << 20  # a 16-byte aligned stand-in address; never dereferenced on these paths


def _fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Nq=16, Nk=16, d=64, scale=0.125,
         causal=0, dt=1):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, dt, None)


@pytest.mark.parametrize("kwargs,expected", [
    (dict(d=96), UNSUPPORTED),
    (dict(d=32), UNSUPPORTED),
    (dict(Hq=3, Hkv=2), INVALID),
    (dict(causal=1, Nq=17, Nk=16), INVALID),
    (dict(causal=2), INVALID),
    (dict(q=None), INVALID),
    (dict(o=None), INVALID),
    (dict(B=0), INVALID),
    (dict(Nk=-1), INVALID),
    (dict(dt=7), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=0.0), INVALID),                 # the kernels take row maxima before scaling
    (dict(scale=-0.5), INVALID),
    (dict(scale=float("inf")), INVALID),
    (dict(q=P + 2), MISALIGNED),
    (dict(lse=P + 4), MISALIGNED),
])
def test_fwd_rejects_before_launch(lib, kwargs, expected):
    assert _fwd(lib, **kwargs) == expected


def test_bwd_rejects_before_launch(lib):
    args = [P] * 9 + [1, 2, 2, 16, 16, 64, 0.125, 1, 1]
    need = lib.attn_bwd_workspace_size(1, 2, 2, 16, 16, 64)
    assert lib.attn_bwd(*args, P, need - 1, None) == WORKSPACE
    assert lib.attn_bwd(*args, None, need, None) == WORKSPACE
    assert lib.attn_bwd(*args, P + 16, need, None) == MISALIGNED  # workspace wants 256-byte alignment
    bad = list(args)
    bad[5] = None  # lse
    assert lib.attn_bwd(*bad, P, need, None) == INVALID
    bad = list(args)
    bad[14] = 80   # d
    assert lib.attn_bwd(*bad, P, need, None) == UNSUPPORTED
    # bf16 at d = 128 checks the workspace against its own (smaller) need
    args128 = [P] * 9 + [1, 2, 2, 16, 16, 128, 0.125, 1, 1]
    need128 = lib.attn_bwd_workspace_size_dt(1, 2, 2, 16, 16, 128, 1)
    assert need128 < lib.attn_bwd_workspace_size(1, 2, 2, 16, 16, 128)
    assert lib.attn_bwd(*args128, P, need128 - 1, None) == WORKSPACE


def test_decode_rejects_before_launch(lib):
    def call(B=2, Hq=8, Hkv=2, L=100, d=128, S=4, ws=P, ws_bytes=None, q=P):
        need = lib.attn_decode_workspace_size(B, Hq, d, S) if ws_bytes is None else ws_bytes
        return lib.attn_decode_splitkv(q, P, P, P, P, B, Hq, Hkv, L, d, 0.1, S, ws, need, None)
    assert call(Hq=6, Hkv=4) == INVALID
    assert call(Hq=6, Hkv=2) == UNSUPPORTED      # group of 3
    assert call(Hq=32, Hkv=2) == UNSUPPORTED     # group of 16
    assert call(d=96) == UNSUPPORTED
    assert call(S=0) == INVALID
    assert call(L=0) == INVALID
    assert call(ws_bytes=100) == WORKSPACE
    assert call(q=P + 8) == MISALIGNED


def test_decode_paged_rejects_before_launch(lib):
    def call(B=2, Hq=8, Hkv=2, num_pages=16, page_size=64, max_pages=4, d=128, S=4, ws=P,
             ws_bytes=None, q=P, table=P, lens=P, kp=P):
        need = lib.attn_decode_workspace_size(B, Hq, d, S) if ws_bytes is None else ws_bytes
        return lib.attn_decode_paged(q, kp, P, table, lens, P, P, B, Hq, Hkv, num_pages,
                                     page_size, max_pages, d, 0.1, S, ws, need, None)
    assert call(page_size=0) == INVALID
    assert call(num_pages=0) == INVALID
    assert call(max_pages=0) == INVALID
    assert call(table=None) == INVALID
    assert call(lens=None) == INVALID
    assert call(Hq=6, Hkv=4) == INVALID
    assert call(Hq=32, Hkv=2) == UNSUPPORTED     # group of 16
    assert call(d=96) == UNSUPPORTED
    assert call(max_pages=1 << 20, page_size=2048) == UNSUPPORTED  # 2^31 key positions
    assert call(ws_bytes=100) == WORKSPACE
    assert call(kp=P + 8) == MISALIGNED
    assert call(table=P + 2) == MISALIGNED


def test_merge_rejects_before_launch(lib):
    assert lib.attn_merge_partials(P, P, P, P, P, 4, 2, 6, 1, None) == UNSUPPORTED
    assert lib.attn_merge_partials(P, P, P, P, P, 4, 2, 512, 1, None) == UNSUPPORTED
    assert lib.attn_merge_partials(P, P, P, P, P, 0, 2, 64, 1, None) == INVALID
    assert lib.attn_merge_partials(P, P, P, P, P, 4, 2, 64, 5, None) == INVALID
    assert lib.attn_merge_partials(None, P, P, P, P, 4, 2, 64, 1, None) == INVALID


def test_product_path_does_not_import_oracle():
    """The CUDA path and the oracle share no code: nothing in the package or
    the input generators imports the oracle."""
    imp = re.compile(r"^\s*(from|import)\s+oracle\b|importlib.*oracle", re.M)
    pkg = os.path.join(ROOT, "online_softmax_tiled_gb300")
    files = [os.path.join(ROOT, "workloads.py")]
    for dirpath, _, names in os.walk(pkg):
        files += [os.path.join(dirpath, f) for f in names if f.endswith(".py")]
    for f in files:
        assert not imp.search(open(f).read()), f


def test_fwd_masked_rejects_before_launch(lib):
    from online_softmax_tiled_gb300 import AttnMask

    def call(mask=None, scale=0.125, Nq=16, Nk=16, d=64, q=P):
        m = None if mask is None else ctypes.byref(mask)
        return lib.attn_fwd_masked(q, P, P, P, P, 1, 2, 2, Nq, Nk, d, scale, m, 1, None)
    half = AttnMask(-1, 0, 0, P, None)                  # only one of the two row-range arrays
    assert call(half) == INVALID
    assert call(AttnMask(-1, 0, 0, P + 2, P)) == MISALIGNED
    assert call(AttnMask(-1, 0, 0, None, None), scale=0.0) == INVALID
    assert call(AttnMask(3, 0, 0, None, None), d=96) == UNSUPPORTED
    assert call(q=None) == INVALID
    assert call(AttnMask(-1, 0, 0, None, None), q=P + 8) == MISALIGNED


def test_bwd_masked_rejects_before_launch(lib):
    from online_softmax_tiled_gb300 import AttnMask
    need = lib.attn_bwd_workspace_size(1, 2, 2, 16, 16, 64)

    def call(mask, Nq=16, d=64, dt=1, ws=P, ws_bytes=need, scale=0.125):
        m = None if mask is None else ctypes.byref(mask)
        return lib.attn_bwd_masked(*([P] * 9), 1, 2, 2, Nq, 16, d, scale, m, dt, ws, ws_bytes,
                                   None)
    assert call(AttnMask(-1, 0, 0, P, None)) == INVALID
    assert call(AttnMask(-1, 0, 0, P, P + 1)) == MISALIGNED
    assert call(AttnMask(7, 0, 0, None, None), ws_bytes=need - 1) == WORKSPACE
    assert call(AttnMask(7, 0, 0, None, None), scale=-1.0) == INVALID
    # a bf16 mask with global keys (or row ranges) lists at most 1024 query
    # tiles per key tile; a window alone takes its tiles from its bounds
    big = lib.attn_bwd_workspace_size(1, 2, 2, 70000, 16, 128)
    assert call(AttnMask(7, 0, 4, None, None), Nq=70000, d=128, ws_bytes=big) == UNSUPPORTED


def test_decode_sparse_rejects_before_launch(lib):
    def call(B=2, Hq=8, Hkv=2, T=4, L=100, n=50, d=128, S=4, ws=P, ws_bytes=None, idx=P):
        need = lib.attn_decode_workspace_size(B, Hq * T, d, S) if ws_bytes is None else ws_bytes
        return lib.attn_decode_sparse(P, P, P, idx, P, P, P, B, Hq, Hkv, T, L, n, d, 0.1, S, ws,
                                      need, None)
    assert call(T=0) == INVALID
    assert call(n=0) == INVALID
    assert call(idx=None) == INVALID
    assert call(Hq=6, Hkv=4) == INVALID
    assert call(Hq=32, Hkv=2) == UNSUPPORTED     # group of 16
    assert call(d=96) == UNSUPPORTED
    assert call(ws_bytes=lib.attn_decode_workspace_size(2, 8, 128, 4)) == WORKSPACE  # T ignored
    assert call(idx=P + 2) == MISALIGNED

"""GB300 (sm_103a) tiled exact softmax attention with the online-softmax
recurrence: forward with LSE, recomputing backward, split-KV decode and the
exact (o, m, l) merge, behind the C ABI of ``include/attn.h``.

The Python layer only marshals torch tensors into that ABI; the computation
runs in the library's CUDA kernels.
"""

from ._binding import (  # noqa: F401
    ATTN_BF16,
    ATTN_F32,
    ATTN_OK,
    AttnError,
    AttnMask,
    attn_bwd,
    attn_bwd_masked,
    attn_bwd_workspace_size,
    attn_selftest_bounded_wait,
    attn_decode_paged,
    attn_decode_sparse,
    attn_decode_splitkv,
    attn_decode_splitkv_noalloc,
    attn_decode_workspace_size,
    attn_fwd,
    attn_fwd_masked,
    attn_merge_partials,
    attn_status_string,
    attn_sync_status,
    backward,
    decode,
    decode_paged,
    decode_sparse,
    forward,
    lib,
    make_mask,
)
from ._build import LIB_PATH, build  # noqa: F401

"""Float64 CPU oracle for tiled exact softmax attention.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain statement of what the
CUDA path computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import it. The product
path (``online_softmax_tiled_gb300``) never imports it, and this package never
imports the product path: the two share no code.

Everything here works on NumPy float64 arrays. Inputs that arrive in bf16 or
fp32 are upcast exactly by the caller before they reach these functions.

Parity status of each function (what pins it is listed in ``attention.py``):
all functions are pinned; none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    NEG_INF,
    causal_allowed,
    scores,
    softmax_rows,
    logsumexp_rows,
    attention_probs,
    attention_fwd,
    attention_fwd_rows,
    softmax_jacobian,
    softmax_backward_jvp,
    attention_bwd,
    mask_allowed,
    attention_fwd_masked,
    attention_bwd_masked,
    tiled_forward,
    decode_split_partials,
    merge_partials,
    gather_paged,
    decode_paged,
    decode_sparse,
    decode_splitkv,
    default_scale,
)

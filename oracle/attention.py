"""Float64 reference for exact softmax attention, its backward, and split-KV decode.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline, never by the
product path.

Sources, by page and section:

* "Flash Attention 2" post (ahmadsaeedzaidi.github.io feed), §Standard
  Attention: S = Q Kᵀ, P = row-softmax(S), O = P V, every P row sums to 1.
  §Flash Attention 2, inner-loop steps 1-5 and the final safe normalisation:
  the tiled recurrence restated in ``tiled_forward``. §Worked Example: the
  N=6, d=2, B_r=B_c=2 numbers pinned in ``tests/golden/``. §Causal masking:
  the 0 / -inf mask added to the scores before the softmax.
* Softmax-backward note (shreyansh26.github.io feed), §The Softmax Derivative
  and §The Jacobian: J = diag(s) - s sᵀ, symmetric. §Backpropagating Through
  Softmax: the Jacobian-vector product s ∘ (g - rowsum(s ∘ g)); gradient rows
  sum to zero. §LogSoftmax Backward: logsumexp made stable by subtracting the
  row maximum.
* ML notes (haolingpu.github.io), attention Q&A: scores are divided by the
  square root of the head dimension (the ``scale`` argument); split-K notes:
  per-chunk (m, l, o) with l and o un-normalised, merged exactly on a common
  maximum, independent of chunk order.
* Attention-residuals kernel lab (manishklach.github.io), §Phase 2: a
  partition with no entries contributes exactly zero mass to the merge.
* ML notes, prefill/decode and the KV cache: a serving cache is kept in
  fixed-size blocks reached through a per-request block table
  (``gather_paged``, ``decode_paged``).
* ML notes, sparse-attention split-K kernel notes: T query tokens attend
  over an arbitrary scattered list of KV positions chosen upstream (by an
  indexer), gathered per tile; split-K partials merged exactly
  (``decode_sparse``).
* Flash Attention 2 post, §Causal masking, "Why": option A handles
  arbitrary masks (sliding window, document boundaries, prefix LM) as a
  0 / -inf term added to the scores before the online softmax
  (``mask_allowed``, ``attention_fwd_masked``, ``attention_bwd_masked``).

Readings where the pages are silent (each also listed in the design notes):

* ``scale`` multiplies Q Kᵀ before the softmax; the walkthrough omits it
  (scale = 1 there).
* LSE is the natural-log logsumexp of the *scaled* scores: LSE = m + ln(l).
* Causal alignment is bottom-right: key j is visible to query i iff
  j <= i + (Nk - Nq). At Nq = Nk this is the page's "key j <= query i".
* A row with no visible key has O = 0 and LSE = -inf; an empty split has
  m = -inf, l = 0, o = 0.
* GQA grouping is contiguous: query head h reads kv head h // (Hq // Hkv);
  dK and dV of a kv head sum over the query heads of its group.
* Split s of L keys into S splits covers [s*c, min((s+1)*c, L)), c = ceil(L/S).
* General masks: a window around each query's position on the key axis
  (bottom-right aligned, as for causal), OR the first ``n_global`` keys,
  AND, where given, a per-row key range [row_kv_start, row_kv_end) (the
  row's document). Causal is the window (unbounded left, 0 right).

Every function here is pinned by ``tests/test_oracle.py`` (worked example,
closed forms, invariants, finite differences, brute force); none is
"parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# Forward: the plain definition (Flash Attention 2 post, §Standard Attention)
# --------------------------------------------------------------------------

def causal_allowed(nq: int, nk: int, rows=None) -> np.ndarray:
    """Boolean visibility mask [len(rows), nk] for the causal case.

    Flash Attention 2 post, §Causal masking: future keys get -inf. Bottom-right
    alignment (key j visible to query i iff j <= i + nk - nq) is the reading
    for nq != nk; at nq == nk it is exactly the page's lower-triangular mask.
    """
    i = np.arange(nq) if rows is None else np.asarray(rows)
    j = np.arange(nk)
    return j[None, :] <= i[:, None] + (nk - nq)


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           nq_total: int | None = None, rows=None) -> np.ndarray:
    """Scaled, masked score matrix S = scale · q kᵀ for one head.

    q: [n, d] (all query rows, or the rows listed in ``rows``), k: [nk, d].
    Masked entries are -inf (Flash Attention 2 post, §Causal masking).
    """
    s = scale * (q @ k.T)
    if causal:
        nq = q.shape[0] if nq_total is None else nq_total
        s = np.where(causal_allowed(nq, k.shape[0], rows), s, NEG_INF)
    return s


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row-wise softmax with the row maximum subtracted first.

    Softmax-backward note, §Setup and §LogSoftmax Backward (stable form). A row
    whose entries are all -inf has no visible key and maps to a zero row.
    """
    m = s.max(axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    z = e.sum(axis=-1, keepdims=True)
    z_safe = np.where(z > 0, z, 1.0)
    return np.where(z > 0, e / z_safe, 0.0)


def logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """ln Σ_j exp(s_j), computed as m + ln Σ exp(s - m); -inf for empty rows."""
    m = s.max(axis=-1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    z = np.exp(s - m_safe[..., None]).sum(axis=-1)
    with np.errstate(divide="ignore"):
        return np.where(z > 0, m_safe + np.log(z), NEG_INF)


def _kv_head(h: int, hq: int, hkv: int) -> int:
    """Contiguous GQA grouping: query head h reads kv head h // (hq // hkv)."""
    return h // (hq // hkv)


def attention_probs(q: np.ndarray, k: np.ndarray, scale: float,
                    causal: bool = False) -> np.ndarray:
    """P = row-softmax(scale · q kᵀ) for one head (the N×N matrix the tiled
    method never materialises)."""
    return softmax_rows(scores(q, k, scale, causal))


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  causal: bool = False):
    """O = softmax(scale · Q Kᵀ) V and LSE, materialising S and P per head.

    q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d]. Returns O [B, Hq, Nq, d] and
    LSE [B, Hq, Nq], both float64.
    """
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = np.zeros((B, Hq, Nq, v.shape[-1]))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            s = scores(q[b, h], k[b, g], scale, causal)
            p = softmax_rows(s)
            o[b, h] = p @ v[b, g]
            lse[b, h] = logsumexp_rows(s)
    assert Nk == v.shape[2]
    return o, lse


def attention_fwd_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                       scale: float, causal: bool, b: int, h: int, rows):
    """O and LSE of the listed query rows of head (b, h) only.

    Each output row depends only on its own query row and on all keys
    (§Standard Attention), so a sample of rows can be checked at sizes where
    the full oracle would take too long.
    """
    Hq, Nq = q.shape[1], q.shape[2]
    g = _kv_head(h, Hq, k.shape[1])
    rows = np.asarray(rows)
    s = scores(q[b, h, rows], k[b, g], scale, causal, nq_total=Nq, rows=rows)
    return softmax_rows(s) @ v[b, g], logsumexp_rows(s)


# --------------------------------------------------------------------------
# General masks (Flash Attention 2 post, §Causal masking, option A)
# --------------------------------------------------------------------------

def mask_allowed(nq: int, nk: int, window_left: int = -1, window_right: int = -1,
                 n_global: int = 0, row_kv_start=None, row_kv_end=None) -> np.ndarray:
    """Boolean visibility [nq, nk] of one batch entry.

    Query row i sits at position i' = i + (nk - nq) of the key axis (the
    bottom-right alignment of the causal case). Key j is visible iff it lies
    in the row's window, i' - window_left <= j <= i' + window_right (a
    negative bound is absent), or j < n_global; and, when row bounds are
    given, row_kv_start[i] <= j < row_kv_end[i]. Causal is window (-1, 0);
    a sliding window of W keys is (W - 1, 0); attention sinks add n_global;
    prefix LM is causal with n_global = prefix length; documents packed in
    one sequence give each row its document's key range.
    """
    i = np.arange(nq)[:, None] + (nk - nq)
    j = np.arange(nk)[None, :]
    win = np.ones((nq, nk), dtype=bool)
    if window_left >= 0:
        win &= j >= i - window_left
    if window_right >= 0:
        win &= j <= i + window_right
    allowed = win | (j < n_global)
    if row_kv_start is not None:
        lo = np.asarray(row_kv_start)[:, None]
        hi = np.asarray(row_kv_end)[:, None]
        allowed &= (j >= lo) & (j < hi)
    return allowed


def _mask_of(mask, b: int, nq: int, nk: int) -> np.ndarray:
    """mask_allowed for batch entry b of a mask given as a dict (None: all keys)."""
    if mask is None:
        return np.ones((nq, nk), dtype=bool)
    rs, re = mask.get("row_kv_start"), mask.get("row_kv_end")
    return mask_allowed(nq, nk, mask.get("window_left", -1), mask.get("window_right", -1),
                        mask.get("n_global", 0), None if rs is None else rs[b],
                        None if re is None else re[b])


def attention_fwd_masked(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, mask):
    """O and LSE under a general mask: S = scale · Q Kᵀ + M with M = 0 where a
    key is visible and -inf elsewhere, then the plain softmax. A row with no
    visible key has O = 0 and LSE = -inf."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = np.zeros((B, Hq, Nq, v.shape[-1]))
    lse = np.zeros((B, Hq, Nq))
    for b in range(B):
        allowed = _mask_of(mask, b, Nq, Nk)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            s = np.where(allowed, scale * (q[b, h] @ k[b, g].T), NEG_INF)
            o[b, h] = softmax_rows(s) @ v[b, g]
            lse[b, h] = logsumexp_rows(s)
    return o, lse


def attention_bwd_masked(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                         scale: float, mask):
    """dQ, dK, dV under a general mask: P is zero on hidden keys, so the
    softmax Jacobian-vector product dS = P ∘ (dP - rowsum(P ∘ dP)) is zero
    there too; otherwise as ``attention_bwd``."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        allowed = _mask_of(mask, b, Nq, Nk)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            p = softmax_rows(np.where(allowed, scale * (q[b, h] @ k[b, g].T), NEG_INF))
            dp = do[b, h] @ v[b, g].T
            ds = softmax_backward_jvp(p, dp)
            dv[b, g] += p.T @ do[b, h]
            dq[b, h] = scale * (ds @ k[b, g])
            dk[b, g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


# --------------------------------------------------------------------------
# Backward (softmax-backward note; recomputation per Flash Attention 2 post)
# --------------------------------------------------------------------------

def softmax_jacobian(p_row: np.ndarray) -> np.ndarray:
    """J = diag(p) - p pᵀ for one softmax row (§The Jacobian)."""
    return np.diag(p_row) - np.outer(p_row, p_row)


def softmax_backward_jvp(p: np.ndarray, g: np.ndarray) -> np.ndarray:
    """dS = p ∘ (g - rowsum(p ∘ g)) (§Backpropagating Through Softmax)."""
    return p * (g - (p * g).sum(axis=-1, keepdims=True))


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                  scale: float, causal: bool = False, route: str = "jvp"):
    """Gradients dQ, dK, dV of L = Σ dO ∘ O for O = softmax(scale·Q Kᵀ) V.

    P is rebuilt from Q and K (nothing is saved from the forward). With
    dP = dO Vᵀ the chain rule gives dV = Pᵀ dO; the softmax step maps dP to
    dS by the Jacobian-vector product, either through the explicit Jacobian
    (``route="jacobian"``, one K×K matrix per row, for small N) or through the
    closed form (``route="jvp"``); then dQ = scale · dS K and
    dK = scale · dSᵀ Q. The row term is rowsum(P ∘ dP), computed here from P
    and dP as the note states (the GPU path uses the equal rowsum(dO ∘ O)).
    GQA: dK, dV of kv head g sum over the query heads that read it.
    """
    if route not in ("jvp", "jacobian"):
        raise ValueError(route)
    B, Hq, Nq, d = q.shape
    Hkv = k.shape[1]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            p = softmax_rows(scores(q[b, h], k[b, g], scale, causal))
            dp = do[b, h] @ v[b, g].T
            if route == "jvp":
                ds = softmax_backward_jvp(p, dp)
            else:
                ds = np.stack([softmax_jacobian(p[i]).T @ dp[i]
                               for i in range(Nq)]) if Nq else dp
            dv[b, g] += p.T @ do[b, h]
            dq[b, h] = scale * (ds @ k[b, g])
            dk[b, g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


# --------------------------------------------------------------------------
# The tiled online-softmax recurrence (self-check only)
# --------------------------------------------------------------------------

def _exp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """exp(a - b) with exp(-inf - (-inf)) taken as 0 (empty-so-far rows)."""
    with np.errstate(invalid="ignore"):
        x = a - b
    return np.where(np.isneginf(a), 0.0, np.exp(np.where(np.isnan(x), 0.0, x)))


def tiled_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  block_rows: int, block_cols: int, causal: bool = False,
                  trace=None):
    """One head, tile by tile, following the Flash Attention 2 post's inner
    loop (§Flash Attention 2, steps 1-5, then the safe normalisation).

    For query tile i and key/value tile j: S_ij = scale·Q_i K_jᵀ; local row max
    m_ij and P̃_ij = exp(S_ij - m_ij); local row sum l_ij; new running max
    m = max(m_old, m_ij); l = e^(m_old-m)·l_old + e^(m_ij-m)·l_ij;
    Õ = e^(m_old-m)·Õ_old + e^(m_ij-m)·(P̃_ij V_j). After the last tile
    O_i = Õ_i / l_i, and LSE = m + ln l. State starts at m = -inf, l = 0, Õ = 0
    (§Worked Example, Initialization).

    ``trace(i_tile, j_tile, state)`` is called after every inner step with the
    tile's S, m_ij and the running m, l, Õ (for the worked-example pins).
    Returns O [Nq, dv] and LSE [Nq].
    """
    nq, nk = q.shape[0], k.shape[0]
    o_all = np.zeros((nq, v.shape[1]))
    lse_all = np.zeros(nq)
    for ti, i0 in enumerate(range(0, nq, block_rows)):
        rows = np.arange(i0, min(i0 + block_rows, nq))
        qi = q[rows]
        m = np.full(len(rows), NEG_INF)
        l = np.zeros(len(rows))
        o_acc = np.zeros((len(rows), v.shape[1]))
        for tj, j0 in enumerate(range(0, nk, block_cols)):
            cols = np.arange(j0, min(j0 + block_cols, nk))
            s_ij = scale * (qi @ k[cols].T)
            if causal:
                vis = cols[None, :] <= rows[:, None] + (nk - nq)
                s_ij = np.where(vis, s_ij, NEG_INF)
            m_ij = s_ij.max(axis=1)
            p_ij = _exp_diff(s_ij, m_ij[:, None])
            l_ij = p_ij.sum(axis=1)
            m_new = np.maximum(m, m_ij)
            a_old = _exp_diff(m, m_new)
            a_new = _exp_diff(m_ij, m_new)
            l = a_old * l + a_new * l_ij
            o_acc = a_old[:, None] * o_acc + a_new[:, None] * (p_ij @ v[cols])
            m = m_new
            if trace is not None:
                trace(ti, tj, {"S": s_ij, "m_ij": m_ij, "m": m.copy(),
                               "l": l.copy(), "O": o_acc.copy()})
        l_safe = np.where(l > 0, l, 1.0)
        o_all[rows] = np.where(l[:, None] > 0, o_acc / l_safe[:, None], 0.0)
        with np.errstate(divide="ignore"):
            lse_all[rows] = np.where(l > 0, m + np.log(l_safe), NEG_INF)
    return o_all, lse_all


# --------------------------------------------------------------------------
# Split-KV decode and the exact (o, m, l) merge (ML notes, split-K notes)
# --------------------------------------------------------------------------

def decode_split_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                          scale: float, num_splits: int):
    """Per-split statistics for decode (query length 1).

    q: [B, Hq, d]; k, v: [B, Hkv, L, d]. Split s holds keys
    [s*c, min((s+1)*c, L)), c = ceil(L / num_splits). For each (b, h, s):
    m_s = max score, l_s = Σ exp(score - m_s), o_s = Σ exp(score - m_s) v
    (un-normalised, as the split-K notes define them). An empty split is
    (o, m, l) = (0, -inf, 0).
    Returns o_part [B, Hq, S, d], m_part [B, Hq, S], l_part [B, Hq, S].
    """
    B, Hq, d = q.shape
    Hkv, L = k.shape[1], k.shape[2]
    c = -(-L // num_splits)
    o_part = np.zeros((B, Hq, num_splits, v.shape[-1]))
    m_part = np.full((B, Hq, num_splits), NEG_INF)
    l_part = np.zeros((B, Hq, num_splits))
    for b in range(B):
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            for s in range(num_splits):
                lo, hi = s * c, min((s + 1) * c, L)
                if lo >= hi:
                    continue
                sc = scale * (k[b, g, lo:hi] @ q[b, h])
                m_s = sc.max()
                e = np.exp(sc - m_s)
                m_part[b, h, s] = m_s
                l_part[b, h, s] = e.sum()
                o_part[b, h, s] = e @ v[b, g, lo:hi]
    return o_part, m_part, l_part


def merge_partials(o_part: np.ndarray, m_part: np.ndarray, l_part: np.ndarray):
    """Exact merge over the last split axis: m = max_s m_s,
    l = Σ_s e^(m_s - m) l_s, O = Σ_s e^(m_s - m) o_s / l, LSE = m + ln l.

    ML notes (split-K): rescaling every chunk onto the common maximum makes the
    merge exact and order-independent. Attention-residuals lab, §Phase 2: a
    chunk with m_s = -inf carries zero mass. Rows with no mass at all give
    O = 0, LSE = -inf.
    """
    m = m_part.max(axis=-1)
    w = _exp_diff(m_part, m[..., None])
    l = (w * l_part).sum(axis=-1)
    o = (w[..., None] * o_part).sum(axis=-2)
    l_safe = np.where(l > 0, l, 1.0)
    out = np.where(l[..., None] > 0, o / l_safe[..., None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(l_safe), NEG_INF)
    return out, lse


def decode_splitkv(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   num_splits: int):
    """Decode output through the split-and-merge route: O [B, Hq, d],
    LSE [B, Hq]."""
    return merge_partials(*decode_split_partials(q, k, v, scale, num_splits))


def gather_paged(pages: np.ndarray, table_row: np.ndarray, length: int,
                 page_size: int) -> np.ndarray:
    """The logical cache [Hkv, length, d] of one request from a paged pool.

    ML notes (prefill/decode and the KV cache): the cache lives in
    fixed-size blocks and a per-request block table maps logical block
    t // page_size to a physical page; token t is row t % page_size of that
    page. pages: [num_pages, Hkv, page_size, d]; table_row: [max_pages].
    """
    t = np.arange(length)
    phys = table_row[t // page_size]
    return pages[phys, :, t % page_size, :].transpose(1, 0, 2)


def decode_paged(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                 block_table: np.ndarray, seq_lens: np.ndarray, page_size: int,
                 scale: float):
    """Query-length-1 attention of every request over its own tokens, read
    through its block table: O [B, Hq, d], LSE [B, Hq].

    Per request b and query head h (contiguous GQA grouping), over the
    request's seq_lens[b] tokens: S = scale · K q, P = softmax(S), O = P V,
    LSE = ln Σ exp(S). A request with no token has O = 0, LSE = -inf.
    """
    B, Hq, _ = q.shape
    Hkv = k_pages.shape[1]
    o = np.zeros((B, Hq, v_pages.shape[-1]))
    lse = np.full((B, Hq), NEG_INF)
    for b in range(B):
        length = int(seq_lens[b])
        if length == 0:
            continue
        k = gather_paged(k_pages, block_table[b], length, page_size)
        v = gather_paged(v_pages, block_table[b], length, page_size)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            sc = scale * (k[g] @ q[b, h])
            o[b, h] = softmax_rows(sc[None, :])[0] @ v[g]
            lse[b, h] = logsumexp_rows(sc[None, :])[0]
    return o, lse


def default_scale(d: int) -> float:
    """1/sqrt(d), the score scaling of the ML notes' attention Q&A."""
    return 1.0 / math.sqrt(d)


def decode_sparse(q: np.ndarray, k: np.ndarray, v: np.ndarray, indices: np.ndarray,
                  counts: np.ndarray, scale: float):
    """Attention of T query tokens per request over a scattered index list:
    O [B, Hq, T, d], LSE [B, Hq, T].

    ML notes, sparse-attention split-K notes: the kernel is given a list of
    KV positions per request (selected upstream) and attends over exactly
    those entries. Reading: one list per request, shared by its T tokens
    and all heads; entry e of request b is cache row indices[b, e] for
    e < counts[b]; a position listed twice counts twice (attention over the
    gathered list). q: [B, Hq, T, d]; k, v: [B, Hkv, L, d]. An empty list
    gives O = 0, LSE = -inf.
    """
    B, Hq, T, _ = q.shape
    Hkv = k.shape[1]
    o = np.zeros((B, Hq, T, v.shape[-1]))
    lse = np.full((B, Hq, T), NEG_INF)
    for b in range(B):
        n = int(counts[b])
        if n == 0:
            continue
        idx = np.asarray(indices[b, :n])
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            kk, vv = k[b, g, idx], v[b, g, idx]          # the gathered list
            s = scale * (q[b, h] @ kk.T)                 # [T, n]
            o[b, h] = softmax_rows(s) @ vv
            lse[b, h] = logsumexp_rows(s)
    return o, lse

"""Pins for the float64 oracle: what the pages and the mathematics fix.

Every check here is independent of the oracle's own formulas: the worked
example of the Flash Attention 2 post (transcribed under tests/golden/),
closed forms, invariants stated on the pages, library routines (SciPy),
pure-Python brute force, and central finite differences. The last block
plants mistakes in the oracle and checks that these pins catch them.
"""

import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import oracle.attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fa2_worked_example.txt")


# ---------------------------------------------------------------- helpers

def _parse_golden(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            out[key] = val
    return out


def _closed(term_list):
    """'c@e c@e ...' -> sum(c * e^e), evaluated in float64."""
    total = 0.0
    for t in term_list.split():
        c, e = t.split("@")
        total += float(c) * math.exp(float(e))
    return total


def _matrix(val):
    return np.array([[float(x) for x in row.split()] for row in val.split(";")])


def _closed_vector(val):
    return np.array([_closed(row) for row in val.split(";")])


def _closed_matrix(val):
    return np.array([[_closed(e) for e in row.split("|")] for row in val.split(";")])


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _brute_attention(q, k, v, scale, causal):
    """Pure-Python loops over one head: the definition, entry by entry."""
    nq, nk, dv = len(q), len(k), len(v[0])
    out, lse = [], []
    for i in range(nq):
        s = []
        for j in range(nk):
            if causal and j > i + (nk - nq):
                continue
            s.append((j, scale * sum(q[i][t] * k[j][t] for t in range(len(q[i])))))
        if not s:
            out.append([0.0] * dv)
            lse.append(-math.inf)
            continue
        mx = max(x for _, x in s)
        z = sum(math.exp(x - mx) for _, x in s)
        row = [sum(math.exp(x - mx) / z * v[j][c] for j, x in s) for c in range(dv)]
        out.append(row)
        lse.append(mx + math.log(z))
    return np.array(out), np.array(lse)


# ------------------------------------------------ worked example (golden)

def test_worked_example_inner_steps():
    g = _parse_golden(GOLDEN)
    q, kt, v = _matrix(g["Q"]), _matrix(g["KT"]), _matrix(g["V"])
    states = {}
    oracle.tiled_forward(q, kt.T, v, 1.0, 2, 2,
                         trace=lambda i, j, st: states.__setitem__((i, j), st))
    for j in range(3):
        st = states[(0, j)]
        tag = f"1_{j + 1}"
        np.testing.assert_array_equal(st["S"], _matrix(g[f"S_{tag}"]))
        np.testing.assert_array_equal(st["m_ij"], _matrix(g[f"m_local_{tag}"])[0])
        np.testing.assert_array_equal(st["m"], _matrix(g[f"m_run_{tag}"])[0])
        np.testing.assert_allclose(st["l"], _closed_vector(g[f"l_run_{tag}"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(st["O"], _closed_matrix(g[f"O_run_{tag}"]), rtol=0, atol=1e-14)


def test_worked_example_printed_decimals():
    g = _parse_golden(GOLDEN)
    q, kt, v = _matrix(g["Q"]), _matrix(g["KT"]), _matrix(g["V"])
    states = {}
    oracle.tiled_forward(q, kt.T, v, 1.0, 2, 2,
                         trace=lambda i, j, st: states.__setitem__((i, j), st))
    st = states[(0, 2)]
    np.testing.assert_allclose(st["l"], _matrix(g["l_run_1_3_printed"])[0], atol=5e-5)
    printed = _matrix(g["O_run_1_3_printed"])
    # Three printed entries agree to their 3 decimals; the [0,0] entry is the
    # page's slip (closed form 3.77253 vs printed 3.768).
    mask = np.ones_like(printed, dtype=bool)
    mask[0, 0] = False
    np.testing.assert_allclose(st["O"][mask], printed[mask], atol=5e-4)
    assert abs(st["O"][0, 0] - 3.772533) < 1e-6


def test_worked_example_tiled_equals_standard():
    g = _parse_golden(GOLDEN)
    q, kt, v = _matrix(g["Q"]), _matrix(g["KT"]), _matrix(g["V"])
    o_t, lse_t = oracle.tiled_forward(q, kt.T, v, 1.0, 2, 2)
    o_s, lse_s = oracle.attention_fwd(q[None, None], kt.T[None, None], v[None, None], 1.0)
    bound = float(g["tiled_vs_standard_max_abs"])
    assert np.max(np.abs(o_t - o_s[0, 0])) <= 4 * bound
    assert np.max(np.abs(lse_t - lse_s[0, 0])) <= 1e-14
    # O_1 = Õ_1 ⊘ l_1 (Step 6) with the closed forms of the last inner step
    o1 = _closed_matrix(g["O_run_1_3"]) / _closed_vector(g["l_run_1_3"])[:, None]
    np.testing.assert_allclose(o_s[0, 0, :2], o1, rtol=0, atol=1e-14)
    lse1 = _matrix(g["m_run_1_3"])[0] + np.log(_closed_vector(g["l_run_1_3"]))
    np.testing.assert_allclose(lse_s[0, 0, :2], lse1, rtol=0, atol=1e-14)


# -------------------------------------------------- forward invariants

@pytest.mark.parametrize("causal", [False, True])
def test_prob_rows_sum_to_one(causal):
    q, k = _rand((37, 16), 1), _rand((37, 16), 2)
    p = oracle.attention_probs(q, k, 0.25, causal)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert (p >= 0).all()
    if causal:
        assert (p[np.triu_indices(37, 1)] == 0).all()


def test_shift_invariance():
    s = _rand((9, 23), 3, 4.0)
    c = _rand((9, 1), 4, 30.0)
    np.testing.assert_allclose(oracle.softmax_rows(s + c), oracle.softmax_rows(s), atol=1e-15)
    np.testing.assert_allclose(oracle.logsumexp_rows(s + c), oracle.logsumexp_rows(s) + c[:, 0],
                               atol=1e-12)


def test_softmax_matches_scipy():
    q, k = _rand((40, 32), 5), _rand((50, 32), 6)
    s = 0.3 * q @ k.T
    np.testing.assert_allclose(oracle.softmax_rows(s), scipy.special.softmax(s, axis=1), atol=1e-15)
    np.testing.assert_allclose(oracle.logsumexp_rows(s), scipy.special.logsumexp(s, axis=1),
                               atol=1e-13)


@pytest.mark.parametrize("causal,nq,nk", [(False, 5, 7), (True, 6, 6), (True, 3, 8), (False, 1, 1)])
def test_brute_force_tiny(causal, nq, nk):
    q, k, v = _rand((nq, 3), 7), _rand((nk, 3), 8), _rand((nk, 2), 9)
    o_ref, lse_ref = _brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
    o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 0.7, causal)
    np.testing.assert_allclose(o[0, 0], o_ref, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], lse_ref, atol=1e-13)


def test_identical_keys_give_mean_of_v():
    k = np.tile(_rand((1, 8), 10), (12, 1))
    q, v = _rand((5, 8), 11), _rand((12, 4), 12)
    o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 0.5)
    np.testing.assert_allclose(o[0, 0], np.tile(v.mean(axis=0), (5, 1)), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], 0.5 * q @ k[0] + math.log(12), atol=1e-13)


def test_single_key():
    q, k, v = _rand((4, 6), 13), _rand((1, 6), 14), _rand((1, 6), 15)
    o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 0.9)
    np.testing.assert_allclose(o[0, 0], np.tile(v[0], (4, 1)), atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], 0.9 * q @ k[0], atol=1e-14)


def test_causal_first_row_and_offsets():
    q, k, v = _rand((6, 4), 16), _rand((6, 4), 17), _rand((6, 4), 18)
    o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], q[0] @ k[0], atol=1e-14)
    # bottom-right alignment: the last query row sees every key
    o_full, _ = oracle.attention_fwd(q[None, None, -1:], k[None, None], v[None, None], 1.0, False)
    np.testing.assert_allclose(o[0, 0, -1], o_full[0, 0, 0], atol=1e-15)


def test_large_scale_selects_argmax():
    q, k, v = _rand((7, 16), 19), _rand((11, 16), 20), _rand((11, 3), 21)
    o, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 200.0)
    np.testing.assert_allclose(o[0, 0], v[np.argmax(q @ k.T, axis=1)], atol=1e-6)


def test_gqa_equals_repeated_heads():
    B, Hq, Hkv, N, d = 2, 6, 2, 9, 5
    q, k, v = _rand((B, Hq, N, d), 22), _rand((B, Hkv, N, d), 23), _rand((B, Hkv, N, d), 24)
    o, lse = oracle.attention_fwd(q, k, v, 0.4, True)
    r = Hq // Hkv
    o2, lse2 = oracle.attention_fwd(q, np.repeat(k, r, axis=1), np.repeat(v, r, axis=1), 0.4, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_rows_subset_matches_full():
    B, H, N, d = 1, 2, 40, 8
    q, k, v = _rand((B, H, N, d), 25), _rand((B, H, N, d), 26), _rand((B, H, N, d), 27)
    o, lse = oracle.attention_fwd(q, k, v, 0.3, True)
    rows = [0, 5, 17, 39]
    o_r, lse_r = oracle.attention_fwd_rows(q, k, v, 0.3, True, 0, 1, rows)
    np.testing.assert_array_equal(o_r, o[0, 1, rows])
    np.testing.assert_array_equal(lse_r, lse[0, 1, rows])


@pytest.mark.parametrize("br,bc,nq,nk,causal", [
    (2, 2, 6, 6, False), (3, 5, 17, 23, False), (4, 4, 16, 16, True),
    (5, 3, 11, 19, True), (64, 64, 10, 10, False), (1, 7, 9, 30, True)])
def test_tiled_equals_full(br, bc, nq, nk, causal):
    q, k, v = _rand((nq, 8), 28, 2.0), _rand((nk, 8), 29, 2.0), _rand((nk, 6), 30)
    o_t, lse_t = oracle.tiled_forward(q, k, v, 0.8, br, bc, causal)
    o_s, lse_s = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 0.8, causal)
    np.testing.assert_allclose(o_t, o_s[0, 0], atol=1e-13)
    np.testing.assert_allclose(lse_t, lse_s[0, 0], atol=1e-13)


# -------------------------------------------------- backward pins

def _loss_grads_fd(q, k, v, g, scale, causal, h=1e-6):
    """Central differences of L = Σ g ∘ O(q, k, v) for every input entry."""
    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd(q_, k_, v_, scale, causal)
        return float((g * o).sum())
    grads = []
    for which in range(3):
        xs = [q.copy(), k.copy(), v.copy()]
        x = xs[which]
        gr = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = loss(*xs)
            x[idx] = x0 - h
            lm = loss(*xs)
            x[idx] = x0
            gr[idx] = (lp - lm) / (2 * h)
        grads.append(gr)
    return grads


def _fd_error(causal, hq=2, hkv=1, n=6, d=4, route="jvp"):
    rng_seed = 31 + hq + n + int(causal)
    q = _rand((1, hq, n, d), rng_seed)
    k = _rand((1, hkv, n, d), rng_seed + 1)
    v = _rand((1, hkv, n, d), rng_seed + 2)
    g = _rand((1, hq, n, d), rng_seed + 3)
    an = oracle.attention_bwd(q, k, v, g, 0.6, causal, route=route)
    fd = _loss_grads_fd(q, k, v, g, 0.6, causal)
    return max(np.max(np.abs(a - f)) for a, f in zip(an, fd))


@pytest.mark.parametrize("causal,hq,hkv,n", [(False, 1, 1, 5), (True, 2, 2, 7), (True, 4, 2, 6),
                                             (False, 3, 1, 4)])
def test_bwd_finite_differences(causal, hq, hkv, n):
    assert _fd_error(causal, hq, hkv, n) < 1e-7


def test_bwd_jacobian_route_equals_jvp_route():
    q, k, v, do = (_rand((2, 2, 33, 8), s) for s in (40, 41, 42, 43))
    for causal in (False, True):
        a = oracle.attention_bwd(q, k, v, do, 0.35, causal, route="jvp")
        b = oracle.attention_bwd(q, k, v, do, 0.35, causal, route="jacobian")
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, atol=1e-12)


def test_softmax_jacobian_symmetric_and_fd():
    s = _rand(9, 44, 2.0)
    p = oracle.softmax_rows(s[None])[0]
    j = oracle.softmax_jacobian(p)
    np.testing.assert_allclose(j, j.T, atol=0)
    h = 1e-6
    fd = np.stack([(oracle.softmax_rows((s + h * e)[None])[0] - oracle.softmax_rows((s - h * e)[None])[0])
                   / (2 * h) for e in np.eye(9)], axis=1)
    np.testing.assert_allclose(j, fd, atol=1e-9)


def test_softmax_backward_rows_sum_to_zero():
    p = oracle.softmax_rows(_rand((12, 20), 45, 3.0))
    ds = oracle.softmax_backward_jvp(p, _rand((12, 20), 46))
    np.testing.assert_allclose(ds.sum(axis=1), 0.0, atol=1e-15)


def test_row_term_two_ways():
    """rowsum(P ∘ dP) = rowsum(dO ∘ O): the row term the GPU computes from O."""
    q, k, v, do = (_rand((30, 8), s) for s in (47, 48, 49, 50))
    for causal in (False, True):
        p = oracle.attention_probs(q, k, 0.5, causal)
        o = p @ v
        dp = do @ v.T
        np.testing.assert_allclose((p * dp).sum(axis=1), (do * o).sum(axis=1), atol=1e-13)


def test_gqa_backward_sums_group():
    B, Hq, Hkv, N, d = 1, 4, 2, 7, 3
    q, do = _rand((B, Hq, N, d), 51), _rand((B, Hq, N, d), 52)
    k, v = _rand((B, Hkv, N, d), 53), _rand((B, Hkv, N, d), 54)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.5, True)
    r = Hq // Hkv
    dq2, dk2, dv2 = oracle.attention_bwd(q, np.repeat(k, r, 1), np.repeat(v, r, 1), do, 0.5, True)
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, r, N, d).sum(2), atol=1e-14)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, r, N, d).sum(2), atol=1e-14)


# -------------------------------------------------- decode / merge pins

def _decode_inputs(B=2, Hq=4, Hkv=2, L=37, d=8, seed=60):
    return _rand((B, Hq, d), seed), _rand((B, Hkv, L, d), seed + 1), _rand((B, Hkv, L, d), seed + 2)


@pytest.mark.parametrize("splits", [1, 2, 5, 16, 37, 50])
def test_decode_split_equals_attention(splits):
    q, k, v = _decode_inputs()
    o, lse = oracle.decode_splitkv(q, k, v, 0.3, splits)
    o_ref, lse_ref = oracle.attention_fwd(q[:, :, None], k, v, 0.3)
    np.testing.assert_allclose(o, o_ref[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse, lse_ref[:, :, 0], atol=1e-13)


def test_decode_partials_closed_form():
    q, k, v = _decode_inputs(B=1, Hq=1, Hkv=1, L=6, d=3)
    o_p, m_p, l_p = oracle.decode_split_partials(q, k, v, 1.0, 2)
    for s in range(2):
        sc = [sum(q[0, 0, t] * k[0, 0, j, t] for t in range(3)) for j in range(3 * s, 3 * s + 3)]
        mx = max(sc)
        assert m_p[0, 0, s] == pytest.approx(mx, abs=1e-14)
        assert l_p[0, 0, s] == pytest.approx(sum(math.exp(x - mx) for x in sc), abs=1e-14)
        want = [sum(math.exp(x - mx) * v[0, 0, 3 * s + j, c] for j, x in enumerate(sc)) for c in range(3)]
        np.testing.assert_allclose(o_p[0, 0, s], want, atol=1e-14)


def test_merge_order_independent_and_empty_split():
    q, k, v = _decode_inputs()
    o_p, m_p, l_p = oracle.decode_split_partials(q, k, v, 0.3, 8)
    o1, lse1 = oracle.merge_partials(o_p, m_p, l_p)
    perm = np.random.default_rng(0).permutation(8)
    o2, lse2 = oracle.merge_partials(o_p[:, :, perm], m_p[:, :, perm], l_p[:, :, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(lse1, lse2, atol=1e-13)
    # appending empty splits (m=-inf, l=0, o=0) leaves the result unchanged
    pad = lambda x, val: np.concatenate([x, np.full(x.shape[:2] + (3,) + x.shape[3:], val)], axis=2)
    o3, lse3 = oracle.merge_partials(pad(o_p, 0.0), pad(m_p, -np.inf), pad(l_p, 0.0))
    np.testing.assert_allclose(o3, o1, atol=1e-15)
    np.testing.assert_allclose(lse3, lse1, atol=1e-15)
    # all-empty rows: O = 0, LSE = -inf
    o4, lse4 = oracle.merge_partials(np.zeros((1, 2, 3)), np.full((1, 2), -np.inf), np.zeros((1, 2)))
    assert (o4 == 0).all() and np.isneginf(lse4).all()


def test_fully_masked_row_is_zero():
    # causal with Nq > Nk: the first rows see no key under bottom-right alignment
    q, k, v = _rand((5, 4), 70), _rand((3, 4), 71), _rand((3, 4), 72)
    o, lse = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0, True)
    assert (o[0, 0, :2] == 0).all() and np.isneginf(lse[0, 0, :2]).all()
    o_t, lse_t = oracle.tiled_forward(q, k, v, 1.0, 2, 2, True)
    np.testing.assert_allclose(o_t, o[0, 0], atol=1e-14)
    np.testing.assert_array_equal(np.isneginf(lse_t), np.isneginf(lse[0, 0]))


# ------------------------------------- planted mistakes must fail a pin

def test_planted_mistakes_are_caught(monkeypatch):
    """Each mutant below is a plausible slip; at least one pin must fail."""
    g = _parse_golden(GOLDEN)
    q, kt, v = _matrix(g["Q"]), _matrix(g["KT"]), _matrix(g["V"])

    def worked_example_error():
        o_s, _ = oracle.attention_fwd(q[None, None], kt.T[None, None], v[None, None], 1.0)
        o1 = _closed_matrix(g["O_run_1_3"]) / _closed_vector(g["l_run_1_3"])[:, None]
        return np.max(np.abs(o_s[0, 0, :2] - o1))

    def causal_brute_error():
        qq, kk, vv = _rand((6, 3), 80), _rand((6, 3), 81), _rand((6, 2), 82)
        o_ref, _ = _brute_attention(qq.tolist(), kk.tolist(), vv.tolist(), 1.0, True)
        o, _ = oracle.attention_fwd(qq[None, None], kk[None, None], vv[None, None], 1.0, True)
        return np.max(np.abs(o[0, 0] - o_ref))

    def gqa_error():
        qq, kk, vv = _rand((1, 4, 5, 3), 83), _rand((1, 2, 5, 3), 84), _rand((1, 2, 5, 3), 85)
        o, _ = oracle.attention_fwd(qq, kk, vv, 1.0)
        o2 = np.stack([_brute_attention(qq[0, h].tolist(), kk[0, h // 2].tolist(),
                                        vv[0, h // 2].tolist(), 1.0, False)[0] for h in range(4)])
        return np.max(np.abs(o[0] - o2))

    def merge_error():
        qq, kk, vv = _decode_inputs()
        o, _ = oracle.decode_splitkv(qq, kk, vv, 0.3, 5)
        o_ref, _ = _brute_attention([qq[0, 0].tolist()], kk[0, 0].tolist(), vv[0, 0].tolist(), 0.3, False)
        return np.max(np.abs(o[0, 0] - o_ref[0]))

    checks = [worked_example_error, causal_brute_error, gqa_error, merge_error,
              lambda: _fd_error(True, 2, 1, 5)]
    assert max(c() for c in checks) < 1e-7  # the real oracle passes every pin

    orig_jvp = oa.softmax_backward_jvp
    orig_allowed = oa.causal_allowed
    orig_softmax = oa.softmax_rows
    orig_exp_diff = oa._exp_diff
    mutants = {
        "dS without the row term": ("softmax_backward_jvp", lambda p, g_: p * g_),
        "dS with a flipped sign": ("softmax_backward_jvp", lambda p, g_: -orig_jvp(p, g_)),
        "causal mask off by one": ("causal_allowed",
                                   lambda nq, nk, rows=None: orig_allowed(nq, nk + 1, rows)[:, :nk]),
        "GQA grouping interleaved": ("_kv_head", lambda h, hq, hkv: h % hkv),
        "softmax over columns": ("softmax_rows", lambda s: orig_softmax(s.T).T if s.shape[0] == s.shape[1]
                                 else orig_softmax(s) * 0.5),
        "merge weight inverted": ("_exp_diff", lambda a, b: orig_exp_diff(b, a) if np.ndim(a) == 3
                                  else orig_exp_diff(a, b)),
    }
    for name, (attr, fn) in mutants.items():
        with monkeypatch.context() as mp:
            mp.setattr(oa, attr, fn)
            errs = []
            for c in checks:
                try:
                    errs.append(c())
                except Exception:  # a crash also counts as caught
                    errs.append(np.inf)
            assert max(errs) > 1e-6, f"pins missed the planted mistake: {name}"


# --------------------------------------------------------------------------
# Paged, variable-length decode
# --------------------------------------------------------------------------

def _paged_from_contiguous(k, page_size, rng):
    """Cut a contiguous cache [B, Hkv, L, d] into pages [P, Hkv, page_size, d]
    placed at random physical indices; returns (pages, block_table)."""
    B, Hkv, L, d = k.shape
    per = -(-L // page_size)
    perm = rng.permutation(B * per)
    pages = np.zeros((B * per, Hkv, page_size, d))
    table = np.zeros((B, per), dtype=np.int64)
    for b in range(B):
        for i in range(per):
            lo, hi = i * page_size, min((i + 1) * page_size, L)
            phys = perm[b * per + i]
            pages[phys, :, : hi - lo] = k[b, :, lo:hi]
            table[b, i] = phys
    return pages, table


def test_paged_decode_equals_attention_on_the_gathered_cache():
    rng = np.random.default_rng(11)
    B, Hq, Hkv, L, d, ps = 3, 4, 2, 70, 8, 16
    q = rng.standard_normal((B, Hq, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    kp, table = _paged_from_contiguous(k, ps, np.random.default_rng(1))
    vp, table_v = _paged_from_contiguous(v, ps, np.random.default_rng(1))
    assert np.array_equal(table, table_v)
    lens = np.array([70, 33, 16])
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, ps, 0.3)
    for b in range(B):
        ref_o, ref_lse = oracle.attention_fwd(q[b:b + 1, :, None, :], k[b:b + 1, :, :lens[b]],
                                              v[b:b + 1, :, :lens[b]], 0.3, False)
        np.testing.assert_allclose(o[b], ref_o[0, :, 0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse[0, :, 0], rtol=1e-12, atol=1e-12)


def test_paged_decode_independent_of_page_placement():
    rng = np.random.default_rng(12)
    B, Hq, Hkv, L, d, ps = 2, 2, 1, 50, 4, 8
    q = rng.standard_normal((B, Hq, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    lens = np.array([50, 21])
    outs = []
    for seed in (3, 4):
        kp, table = _paged_from_contiguous(k, ps, np.random.default_rng(seed))
        vp, _ = _paged_from_contiguous(v, ps, np.random.default_rng(seed))
        outs.append(oracle.decode_paged(q, kp, vp, table, lens, ps, 0.5))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def test_paged_decode_closed_forms():
    """Length 0: O = 0, LSE = -inf. Length 1: O = v_0, LSE = scale·k_0·q.
    Length 2: O = (e^s0 v0 + e^s1 v1) / (e^s0 + e^s1)."""
    rng = np.random.default_rng(13)
    Hkv, ps, d = 1, 4, 3
    pages = rng.standard_normal((3, Hkv, ps, d))
    vpages = rng.standard_normal((3, Hkv, ps, d))
    table = np.array([[2, 0], [1, 2], [0, 1]])
    q = rng.standard_normal((3, 1, d))
    o, lse = oracle.decode_paged(q, pages, vpages, table, np.array([0, 1, 2]), ps, 0.7)
    assert np.all(o[0] == 0) and lse[0, 0] == -np.inf
    k0, v0 = pages[1, 0, 0], vpages[1, 0, 0]
    np.testing.assert_allclose(o[1, 0], v0, rtol=1e-14)
    assert abs(lse[1, 0] - 0.7 * (k0 @ q[1, 0])) < 1e-14
    s0, s1 = 0.7 * (pages[0, 0, 0] @ q[2, 0]), 0.7 * (pages[0, 0, 1] @ q[2, 0])
    w0, w1 = np.exp(s0), np.exp(s1)
    np.testing.assert_allclose(o[2, 0], (w0 * vpages[0, 0, 0] + w1 * vpages[0, 0, 1]) / (w0 + w1),
                               rtol=1e-12)
    assert abs(lse[2, 0] - np.log(w0 + w1)) < 1e-12


# -------------------------------------------------- general masks (option A)

def _brute_masked(q, k, v, scale, visible):
    """Pure-Python loops over one head: each row's softmax over the keys the
    predicate visible(i, j) admits, built from index lists, not a mask matrix."""
    nq, nk, dv = len(q), len(k), len(v[0])
    out, lse = [], []
    for i in range(nq):
        s = [(j, scale * sum(q[i][t] * k[j][t] for t in range(len(q[i]))))
             for j in range(nk) if visible(i, j)]
        if not s:
            out.append([0.0] * dv)
            lse.append(-math.inf)
            continue
        mx = max(x for _, x in s)
        z = sum(math.exp(x - mx) for _, x in s)
        out.append([sum(math.exp(x - mx) / z * v[j][c] for j, x in s) for c in range(dv)])
        lse.append(mx + math.log(z))
    return np.array(out), np.array(lse)


def _mask_inputs(B=2, Hq=2, Hkv=1, nq=9, nk=9, d=4, seed=70):
    return (_rand((B, Hq, nq, d), seed), _rand((B, Hkv, nk, d), seed + 1),
            _rand((B, Hkv, nk, d), seed + 2), _rand((B, Hq, nq, d), seed + 3))


@pytest.mark.parametrize("nq,nk", [(9, 9), (5, 11)])
def test_mask_causal_and_full_specs_equal_the_pinned_paths(nq, nk):
    """Window (-1, 0) is the causal mask and (-1, -1) no mask at all: the
    general path reproduces the pinned causal / unmasked oracle exactly."""
    q, k, v, do = _mask_inputs(nq=nq, nk=nk)
    for spec, causal in (({"window_left": -1, "window_right": 0}, True),
                         ({"window_left": -1, "window_right": -1}, False), (None, False)):
        o_m, l_m = oracle.attention_fwd_masked(q, k, v, 0.7, spec)
        o_c, l_c = oracle.attention_fwd(q, k, v, 0.7, causal)
        assert np.array_equal(o_m, o_c) and np.array_equal(l_m, l_c)
        for a, b in zip(oracle.attention_bwd_masked(q, k, v, do, 0.7, spec),
                        oracle.attention_bwd(q, k, v, do, 0.7, causal)):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("wl,wr,ng,nq,nk", [(2, 0, 0, 8, 8), (3, 0, 2, 8, 10), (1, 2, 0, 7, 7),
                                            (-1, 1, 0, 6, 6), (2, -1, 3, 6, 9), (0, 0, 0, 5, 5)])
def test_window_and_global_keys_brute_force(wl, wr, ng, nq, nk):
    """Sliding windows, attention sinks (global keys), windows reaching right
    of the diagonal: the matrix-built mask agrees with per-row index lists."""
    q, k, v, _ = _mask_inputs(B=1, Hq=1, nq=nq, nk=nk, seed=80 + wl + 3 * wr + ng)
    spec = {"window_left": wl, "window_right": wr, "n_global": ng}
    o, lse = oracle.attention_fwd_masked(q, k, v, 0.9, spec)

    def visible(i, j):
        ip = i + nk - nq
        in_win = (wl < 0 or j >= ip - wl) and (wr < 0 or j <= ip + wr)
        return in_win or j < ng
    ob, lb = _brute_masked(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.9, visible)
    np.testing.assert_allclose(o[0, 0], ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], lb, rtol=0, atol=1e-12)


def _doc_bounds(lengths):
    """Per-row key range [start, end) of each row's document, for documents of
    the given lengths packed back to back (self-attention, nq = nk)."""
    starts, ends, s = [], [], 0
    for n in lengths:
        starts += [s] * n
        ends += [s + n] * n
        s += n
    return np.array(starts), np.array(ends)


@pytest.mark.parametrize("causal", [True, False])
def test_document_mask_is_attention_per_document(causal):
    """Packed documents: the masked result equals plain (causal) attention run
    on each document's slice alone."""
    lengths = [4, 1, 6, 3]
    n = sum(lengths)
    q, k, v, do = _mask_inputs(B=1, Hq=2, Hkv=1, nq=n, nk=n, seed=90 + int(causal))
    st, en = _doc_bounds(lengths)
    spec = {"window_left": -1, "window_right": 0 if causal else -1,
            "row_kv_start": st[None], "row_kv_end": en[None]}
    o, lse = oracle.attention_fwd_masked(q, k, v, 0.8, spec)
    grads = oracle.attention_bwd_masked(q, k, v, do, 0.8, spec)
    s = 0
    for ln in lengths:
        sl = slice(s, s + ln)
        o_d, l_d = oracle.attention_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.8, causal)
        np.testing.assert_allclose(o[:, :, sl], o_d, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, sl], l_d, rtol=0, atol=1e-13)
        g_d = oracle.attention_bwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], 0.8, causal)
        for a, b in zip(grads, g_d):
            np.testing.assert_allclose(a[:, :, sl], b, rtol=0, atol=1e-13)
        s += ln


def test_prefix_lm():
    """Causal with the first P keys global: rows inside the prefix attend to
    the whole prefix and nothing else; rows after it are ordinary causal rows."""
    n, P = 10, 4
    q, k, v, _ = _mask_inputs(B=1, Hq=1, nq=n, nk=n, seed=95)
    o, lse = oracle.attention_fwd_masked(q, k, v, 0.6,
                                         {"window_left": -1, "window_right": 0, "n_global": P})
    o_p, l_p = oracle.attention_fwd(q[:, :, :P], k[:, :, :P], v[:, :, :P], 0.6, False)
    o_c, l_c = oracle.attention_fwd(q, k, v, 0.6, True)
    np.testing.assert_allclose(o[:, :, :P], o_p, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[:, :, :P], l_p, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[:, :, P:], o_c[:, :, P:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[:, :, P:], l_c[:, :, P:], rtol=0, atol=1e-13)


def test_mask_rows_without_keys():
    """Rows whose key range is empty (or whose window lies past the keys) get
    O = 0, LSE = -inf and zero gradients; the other rows are unaffected."""
    q, k, v, do = _mask_inputs(B=1, Hq=1, nq=6, nk=6, seed=97)
    st = np.array([[0, 2, 3, 3, 0, 5]])
    en = np.array([[3, 2, 6, 3, 6, 6]])            # rows 1 and 3 empty
    spec = {"row_kv_start": st, "row_kv_end": en}
    o, lse = oracle.attention_fwd_masked(q, k, v, 0.7, spec)
    dq, dk, dv = oracle.attention_bwd_masked(q, k, v, do, 0.7, spec)
    for r in (1, 3):
        assert np.all(o[0, 0, r] == 0) and lse[0, 0, r] == -np.inf and np.all(dq[0, 0, r] == 0)
    ob, lb = _brute_masked(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.7,
                           lambda i, j: st[0, i] <= j < en[0, i])
    np.testing.assert_allclose(o[0, 0], ob, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(lse[0, 0]), np.isinf(lb))
    # a window entirely to the left of the keys: nothing visible anywhere
    o2, l2 = oracle.attention_fwd_masked(q, k, v, 0.7, {"window_left": 0, "window_right": 0,
                                                       "row_kv_start": st, "row_kv_end": st})
    assert np.all(o2 == 0) and np.all(l2 == -np.inf)


def _masked_fd_error(spec, n=6, hq=2, hkv=1, d=3, seed=99, h=1e-6):
    q, k, v, g = _mask_inputs(B=1, Hq=hq, Hkv=hkv, nq=n, nk=n, d=d, seed=seed)
    an = oracle.attention_bwd_masked(q, k, v, g, 0.6, spec)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd_masked(q_, k_, v_, 0.6, spec)
        return float((g * o).sum())
    err = 0.0
    for which, x in enumerate((q, k, v)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xs = [q.copy(), k.copy(), v.copy()]
            xs[which][idx] += h
            lp = loss(*xs)
            xs[which][idx] -= 2 * h
            lm = loss(*xs)
            err = max(err, abs((lp - lm) / (2 * h) - an[which][idx]))
    return err


@pytest.mark.parametrize("spec", [
    {"window_left": 1, "window_right": 0, "n_global": 1},
    {"window_left": -1, "window_right": 1},
    {"window_left": -1, "window_right": 0,
     "row_kv_start": np.array([[0, 0, 2, 2, 2, 5]]), "row_kv_end": np.array([[2, 2, 5, 5, 5, 6]])},
])
def test_masked_bwd_finite_differences(spec):
    assert _masked_fd_error(spec) < 1e-7


def test_planted_mask_mistakes_are_caught(monkeypatch):
    """Plausible slips in the mask builder: each makes a mask pin fail."""
    def window_error():
        nq, nk, wl, wr, ng = 6, 9, 2, 0, 2
        q, k, v, _ = _mask_inputs(B=1, Hq=1, nq=nq, nk=nk, seed=101)
        o, _ = oracle.attention_fwd_masked(q, k, v, 0.9, {"window_left": wl, "window_right": wr,
                                                          "n_global": ng})

        def visible(i, j):
            ip = i + nk - nq
            return (ip - wl <= j <= ip + wr) or j < ng
        ob, _ = _brute_masked(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.9, visible)
        return np.max(np.abs(o[0, 0] - ob))

    def document_error():
        lengths = [3, 4, 2]
        q, k, v, _ = _mask_inputs(B=1, Hq=1, nq=9, nk=9, seed=102)
        st, en = _doc_bounds(lengths)
        o, _ = oracle.attention_fwd_masked(q, k, v, 0.8, {"row_kv_start": st[None],
                                                          "row_kv_end": en[None]})
        o_d = [oracle.attention_fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], 0.8)[0]
               for a, b in ((0, 3), (3, 7), (7, 9))]
        return np.max(np.abs(o - np.concatenate(o_d, axis=2)))

    checks = [window_error, document_error]
    assert max(c() for c in checks) < 1e-9
    orig = oa.mask_allowed
    mutants = {
        "window one key wider": lambda nq, nk, wl=-1, wr=-1, ng=0, rs=None, re=None:
            orig(nq, nk, wl + 1 if wl >= 0 else wl, wr, ng, rs, re),
        "global keys dropped": lambda nq, nk, wl=-1, wr=-1, ng=0, rs=None, re=None:
            orig(nq, nk, wl, wr, 0, rs, re),
        "top-left alignment": lambda nq, nk, wl=-1, wr=-1, ng=0, rs=None, re=None:
            orig(nq, nq, wl, wr, ng, rs, re)[:, :nk] if nk <= nq else
            np.pad(orig(nq, nq, wl, wr, ng, rs, re), ((0, 0), (0, nk - nq))),
        "document end inclusive": lambda nq, nk, wl=-1, wr=-1, ng=0, rs=None, re=None:
            orig(nq, nk, wl, wr, ng, rs, None if re is None else np.asarray(re) + 1),
    }
    for name, fn in mutants.items():
        with monkeypatch.context() as mp:
            mp.setattr(oa, "mask_allowed", fn)
            errs = []
            for c in checks:
                try:
                    errs.append(c())
                except Exception:
                    errs.append(np.inf)
            assert max(errs) > 1e-6, f"pins missed the planted mistake: {name}"


# --------------------------------------------------------------------------
# Sparse-index decode (T query tokens over a scattered index list)
# --------------------------------------------------------------------------

def _sparse_inputs(B=2, Hq=4, Hkv=2, T=3, L=40, d=5, n=11, seed=120):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, T, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    idx = np.stack([rng.choice(L, size=n, replace=False) for _ in range(B)])
    return q, k, v, idx


def test_sparse_decode_brute_force():
    """Pure-Python loops over the listed rows of each (request, head, token)."""
    q, k, v, idx = _sparse_inputs()
    counts = np.array([11, 7])
    o, lse = oracle.decode_sparse(q, k, v, idx, counts, 0.8)
    for b in range(2):
        for h in range(4):
            g = h // 2
            rows = [int(j) for j in idx[b, :counts[b]]]
            for t in range(3):
                ob, lb = _brute_attention([q[b, h, t].tolist()], k[b, g, rows].tolist(),
                                          v[b, g, rows].tolist(), 0.8, False)
                np.testing.assert_allclose(o[b, h, t], ob[0], rtol=0, atol=1e-13)
                assert abs(lse[b, h, t] - lb[0]) < 1e-13


def test_sparse_decode_order_invariant_and_full_list_is_dense():
    """The list's order does not matter; listing every position once is
    ordinary (non-causal) attention over the whole cache."""
    q, k, v, idx = _sparse_inputs(n=40, L=40)
    counts = np.array([40, 40])
    o1, l1 = oracle.decode_sparse(q, k, v, idx, counts, 0.6)
    rng = np.random.default_rng(3)
    idx2 = np.stack([rng.permutation(r) for r in idx])
    o2, l2 = oracle.decode_sparse(q, k, v, idx2, counts, 0.6)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    o3, l3 = oracle.attention_fwd(q, k, v, 0.6, False)
    np.testing.assert_allclose(o1, o3, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l3, rtol=0, atol=1e-13)


def test_sparse_decode_closed_forms():
    """Empty list: O = 0, LSE = -inf. One entry: O = v_j, LSE = scale·q·k_j.
    A position listed twice weighs twice: O = (2 e^s0 v0 + e^s1 v1) / (2 e^s0 + e^s1)."""
    q, k, v, _ = _sparse_inputs(B=3, Hq=1, Hkv=1, T=1)
    idx = np.array([[5, 0, 0], [9, 0, 0], [4, 4, 7]])
    o, lse = oracle.decode_sparse(q, k, v, idx, np.array([0, 1, 3]), 0.7)
    assert np.all(o[0] == 0) and lse[0, 0, 0] == -np.inf
    np.testing.assert_allclose(o[1, 0, 0], v[1, 0, 9], rtol=1e-14)
    assert abs(lse[1, 0, 0] - 0.7 * (q[1, 0, 0] @ k[1, 0, 9])) < 1e-13
    s0, s1 = 0.7 * (q[2, 0, 0] @ k[2, 0, 4]), 0.7 * (q[2, 0, 0] @ k[2, 0, 7])
    w0, w1 = np.exp(s0), np.exp(s1)
    np.testing.assert_allclose(o[2, 0, 0], (2 * w0 * v[2, 0, 4] + w1 * v[2, 0, 7]) / (2 * w0 + w1),
                               rtol=1e-12)
    assert abs(lse[2, 0, 0] - np.log(2 * w0 + w1)) < 1e-12

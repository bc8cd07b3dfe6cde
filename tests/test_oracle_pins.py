"""Pins of the float64 oracle against what the pages fix.

Each test is built so that a plausible slip in the oracle (ratio inverted,
non-strict cut, residual replaced by p, wrong normaliser, temperature applied
the wrong way, argmax tie rule, reading padding) makes it fail.

Sources: "Speculative Decoding" (atonlee.tistory.com/330) ch.2-3; "Speculative
Decoding으로 LLM 추론 속도 높이기" (donmain.dev), section "품질은 rejection
sampling이 지킨다"; "Fast Inference from Transformers via Speculative Decoding"
notes, method details step 3; "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가",
section on why the output does not change.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _batch(p_rows, q_rows, tokens, r, u, T=1.0, dtype="f32"):
    """B sequences sharing the rows; tokens [B, g], r [B, g], u [B]."""
    p = np.asarray(p_rows, np.float64)
    q = np.asarray(q_rows, np.float64)
    g, V = q.shape
    tokens = np.asarray(tokens, np.int32).reshape(-1, g)
    B = tokens.shape[0]
    with np.errstate(divide="ignore"):
        tl = (np.log(p) * T).astype(np.float32)
        dl = (np.log(q) * T).astype(np.float32)
    target = np.broadcast_to(tl, (B, g + 1, V)).copy()
    draft = np.broadcast_to(dl, (B, g, V)).copy()
    uni = np.zeros((B, g + 1), np.float32)
    uni[:, :g] = np.asarray(r, np.float32).reshape(B, g)
    uni[:, g] = np.asarray(u, np.float32).reshape(B)
    return dict(target=target, draft=draft, dtype=dtype, tokens=tokens, num_draft=np.full(B, g, np.int32),
                uniforms=uni, temperature=np.full(B, T, np.float32))


def _run(oracle_mod, b, **kw):
    return oracle_mod.verify(b["target"], b["draft"], b["dtype"], b["tokens"], b["num_draft"], b["uniforms"],
                             b["temperature"], **kw)


def _grid(n):
    return (np.arange(n) + 0.5) / n


# ----------------------------------------------------------------------------
# worked example: q(x) = 0.4, p(x) = 0.1
# ----------------------------------------------------------------------------

def test_worked_example_accept_probability(oracle_mod):
    w = json.load(open(os.path.join(GOLD, "worked_numbers.json")))["accept_example"]
    p = [[w["p"], 0.6, 0.3], [1 / 3, 1 / 3, 1 / 3]]
    q = [[w["q"], 0.3, 0.3]]
    N = 4000
    r = _grid(N)
    b = _batch(p, q, np.zeros(N), r, np.full(N, 0.5))
    res = _run(oracle_mod, b)
    acc = (res.out_num_accepted == 1).mean()
    assert abs(acc - w["accept_probability"]) <= 1.0 / N
    # accepted exactly for r below p/q, rejected at and above it (strict test)
    assert np.all(res.out_num_accepted[r < 0.2499] == 1)
    assert np.all(res.out_num_accepted[r > 0.2501] == 0)
    # margins record |r - p/q|
    np.testing.assert_allclose(res.acc_margin[:, 0], np.abs(r.astype(np.float32) - 0.25), atol=1e-6)


def test_worked_example_output_law_is_p(oracle_mod):
    """Theorem on a grid: x ~ q (exact weights), r and u on fine midpoint grids."""
    w = json.load(open(os.path.join(GOLD, "worked_numbers.json")))["accept_example"]
    p0 = np.array([w["p"], 0.6, 0.3])
    q0 = np.array([w["q"], 0.3, 0.3])
    p = [p0, [1 / 3, 1 / 3, 1 / 3]]
    q = [q0]
    N = 300
    rr, uu = np.meshgrid(_grid(N), _grid(N), indexing="ij")
    law = np.zeros(3)
    accept_mass_x0 = 0.0
    for x in range(3):
        b = _batch(p, q, np.full(N * N, x), rr.ravel(), uu.ravel())
        res = _run(oracle_mod, b, diagnostics=False)
        y0 = res.out_tokens[:, 0]
        for j in range(3):
            law[j] += q0[x] * (y0 == j).mean()
        if x == 0:
            accept_mass_x0 = q0[0] * ((res.out_num_accepted == 1) & (y0 == 0)).mean()
    np.testing.assert_allclose(law, p0, atol=3.0 / N)
    assert accept_mass_x0 == pytest.approx(w["output_mass"], abs=1.0 / N)


def test_residual_support_and_inverse_cdf(oracle_mod):
    # p - q = (-0.3, 0.2, 0.1): on rejection the residual is (0, 2/3, 1/3)
    p = [[0.5, 0.3, 0.2], [0.25, 0.25, 0.5]]
    q = [[0.8, 0.1, 0.1]]
    N = 3000
    u = _grid(N)
    b = _batch(p, q, np.zeros(N), np.full(N, 0.9), u)  # r = 0.9 >= p/q = 0.625: reject
    res = _run(oracle_mod, b)
    assert np.all(res.out_num_accepted == 0)
    y = res.out_tokens[:, 0]
    assert set(np.unique(y)) == {1, 2}  # token 0 has zero residual weight
    # smallest j with u*S < C_j: token 1 below u = 2/3, token 2 above
    assert np.all(y[u < 2 / 3 - 1e-6] == 1) and np.all(y[u > 2 / 3 + 1e-6] == 2)
    np.testing.assert_allclose(res.resid_mass, 0.3, rtol=1e-6)
    assert np.all(res.out_tokens[:, 1] == -1)


def test_single_point_residual(oracle_mod):
    # worked example rows: a rejected x = 0 can only be replaced by token 1
    p = [[0.1, 0.6, 0.3], [1 / 3, 1 / 3, 1 / 3]]
    q = [[0.4, 0.3, 0.3]]
    N = 500
    b = _batch(p, q, np.zeros(N), np.full(N, 0.75), _grid(N))
    res = _run(oracle_mod, b)
    assert np.all(res.out_num_accepted == 0) and np.all(res.out_tokens[:, 0] == 1)


def test_bonus_token_law_when_all_accepted(oracle_mod):
    # q = p at every draft position: every draft passes; the bonus row is p_g
    rows = [[0.2, 0.3, 0.5], [0.6, 0.1, 0.3]]
    bonus = [0.1, 0.2, 0.3, 0.4]
    V = 4
    p = [r + [0.0] for r in rows] + [bonus]
    q = [r + [0.0] for r in rows]
    N = 4000
    u = _grid(N)
    rng = np.random.default_rng(3)
    b = _batch(p, q, np.stack([np.full(N, 2), np.full(N, 0)], 1), rng.random((N, 2)), u)
    res = _run(oracle_mod, b)
    assert np.all(res.out_num_accepted == 2)
    assert np.all(res.out_tokens[:, 0] == 2) and np.all(res.out_tokens[:, 1] == 0)
    freq = np.bincount(res.out_tokens[:, 2], minlength=V) / N
    np.testing.assert_allclose(freq, bonus, atol=2.0 / N)
    # the bonus sample follows the CDF of p_g in index order
    cdf = np.cumsum(bonus)
    expect = np.searchsorted(cdf, u, side="right")
    far = np.min(np.abs(u[:, None] - cdf[None, :]), axis=1) > 1e-6
    assert np.all(res.out_tokens[far, 2] == expect[far])


def test_cut_at_first_rejection(oracle_mod):
    # position 0 always rejects (p(x)=0), position 1 would accept: the round stops at 0
    p = [[0.0, 1.0], [0.5, 0.5], [0.5, 0.5]]
    q = [[1.0, 0.0], [0.5, 0.5]]
    b = _batch(p, q, [[0, 1]], [[0.1, 0.1]], [0.3])
    res = _run(oracle_mod, b)
    assert res.out_num_accepted[0] == 0
    assert list(res.out_tokens[0]) == [1, -1, -1]
    # k accepted then one replacement: accept, accept, reject
    p = [[0.5, 0.5]] * 3 + [[0.0, 1.0], [0.5, 0.5]]
    q = [[0.5, 0.5]] * 3 + [[1.0, 0.0]]
    b = _batch(p, q, [[0, 1, 0, 0]], [[0.3, 0.3, 0.3, 0.3]], [0.5])
    res = _run(oracle_mod, b)
    assert res.out_num_accepted[0] == 3
    assert list(res.out_tokens[0]) == [0, 1, 0, 1, -1]


def test_zero_q_draft_accepted_iff_p_positive(oracle_mod):
    p = [[0.5, 0.5, 0.0], [1.0, 0.0, 0.0]]
    q = [[1.0, 0.0, 0.0]]
    b = _batch(p, q, [[1]], [[0.999]], [0.5])
    res = _run(oracle_mod, b)
    assert res.out_num_accepted[0] == 1 and res.out_tokens[0, 0] == 1
    assert np.isinf(res.acc_margin[0, 0])


# ----------------------------------------------------------------------------
# greedy mode: accept iff draft == argmax p, emit argmax on rejection
# ----------------------------------------------------------------------------

def _greedy_case(rows, tokens, gmax=None, dtype="f32"):
    rows = np.asarray(rows, np.float32)
    g = len(tokens)
    gmax = g if gmax is None else gmax
    V = rows.shape[1]
    target = np.full((1, gmax + 1, V), np.inf, np.float32)
    target[0, : g + 1] = rows
    draft = np.full((1, gmax, V), np.nan, np.float32)  # never read when T = 0
    tok = np.full((1, gmax), -1, np.int32)
    tok[0, :g] = tokens
    return dict(target=target, draft=draft, dtype=dtype, tokens=tok, num_draft=np.array([g], np.int32),
                uniforms=np.full((1, gmax + 1), np.nan, np.float32), temperature=np.zeros(1, np.float32))


GREEDY_CASES = [
    # rows (g+1 of them), drafts, expected tokens, expected accepted
    ([[0, 3, 1, 3, -1, 2], [5, 5, 5, 5, 5, 5], [-np.inf, -np.inf, 7, 1, 7, 0]], [1, 0], [1, 0, 2], 2),
    ([[0, 3, 1, 3, -1, 2], [5, 5, 5, 5, 5, 5], [-np.inf, -np.inf, 7, 1, 7, 0]], [3, 0], [1, -1, -1], 0),
    ([[0, 3, 1, 3, -1, 2], [5, 5, 5, 5, 5, 5], [-np.inf, -np.inf, 7, 1, 7, 0]], [1, 4], [1, 0, -1], 1),
    ([[-np.inf] * 4], [], [0], 0),
    ([[1, 2, 3, 4], [4, 3, 2, 1]], [3], [3, 0], 1),
]


@pytest.mark.parametrize("rows,tokens,expect,n", GREEDY_CASES)
def test_greedy_golden(oracle_mod, rows, tokens, expect, n):
    res = _run(oracle_mod, _greedy_case(rows, tokens))
    assert list(res.out_tokens[0]) == expect
    assert res.out_num_accepted[0] == n
    assert res.seq_status[0] == 0


def test_greedy_equals_argmax_agreement_on_random_rows(oracle_mod):
    """Property: accepted prefix = longest prefix where draft == argmax."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        g = int(rng.integers(0, 5))
        rows = np.round(rng.normal(size=(g + 1, 7)) * 2) / 2
        am = [int(np.flatnonzero(r == r.max())[0]) for r in rows]
        tokens = [am[i] if rng.random() < 0.7 else int(rng.integers(0, 7)) for i in range(g)]
        res = _run(oracle_mod, _greedy_case(rows, tokens, gmax=4))
        n = 0
        while n < g and tokens[n] == am[n]:
            n += 1
        assert res.out_num_accepted[0] == n
        assert list(res.out_tokens[0, :n]) == tokens[:n] and res.out_tokens[0, n] == am[n]
        assert np.all(res.out_tokens[0, n + 1:] == -1)


# ----------------------------------------------------------------------------
# softmax at temperature T
# ----------------------------------------------------------------------------

def test_uniform_logits_give_one_over_V(oracle_mod):
    V, g = 1000, 2
    t = np.full((1, g + 1, V), 3.25, np.float32)
    d = np.full((1, g, V), -1.5, np.float32)
    res = oracle_mod.verify(t, d, "f32", np.array([[7, 999]], np.int32), np.array([g], np.int32),
                            np.full((1, g + 1), 0.5, np.float32), np.array([0.37], np.float32))
    np.testing.assert_allclose(res.p_hat[0], 1.0 / V, rtol=1e-13)
    np.testing.assert_allclose(res.q_hat[0], 1.0 / V, rtol=1e-13)
    T = float(np.float32(0.37))  # the oracle reads the float32 temperature
    np.testing.assert_allclose(res.logz_t[0], 3.25 / T + np.log(V), rtol=1e-13)
    np.testing.assert_allclose(res.logz_d[0], -1.5 / T + np.log(V), rtol=1e-13)
    assert res.out_num_accepted[0] == 2  # p == q everywhere: every draft passes


@pytest.mark.parametrize("T", [0.25, 0.7, 1.0, 3.0])
def test_softmax_values_match_library_softmax(oracle_mod, T):
    rng = np.random.default_rng(int(T * 100))
    V, g, B = 257, 3, 6
    t = rng.normal(0, 3, size=(B, g + 1, V)).astype(np.float32)
    d = (t[:, :g] + rng.normal(0, 1, size=(B, g, V))).astype(np.float32)
    tok = rng.integers(0, V, size=(B, g)).astype(np.int32)
    res = oracle_mod.verify(t, d, "f32", tok, np.full(B, g, np.int32), rng.random((B, g + 1)).astype(np.float32),
                            np.full(B, T, np.float32))
    T32 = float(np.float32(T))  # the oracle reads the float32 temperature
    t64, d64 = t.astype(np.float64) / T32, d.astype(np.float64) / T32
    for b in range(B):
        for i in range(g):
            assert res.p_hat[b, i] == pytest.approx(scipy.special.softmax(t64[b, i])[tok[b, i]], rel=1e-12)
            assert res.q_hat[b, i] == pytest.approx(scipy.special.softmax(d64[b, i])[tok[b, i]], rel=1e-12)
            assert res.logz_d[b, i] == pytest.approx(scipy.special.logsumexp(d64[b, i]), rel=1e-13)
        for i in range(g + 1):
            assert res.logz_t[b, i] == pytest.approx(scipy.special.logsumexp(t64[b, i]), rel=1e-13)


def test_temperature_divides_logits(oracle_mod):
    """logits l at T equal logits l/T at T = 1 (checks T divides, not multiplies)."""
    rng = np.random.default_rng(9)
    V, g, B = 64, 2, 4
    base = np.round(rng.normal(0, 2, size=(B, g + 1, V)) * 4) / 4  # exact in f32 after halving
    dbase = np.round(rng.normal(0, 2, size=(B, g, V)) * 4) / 4
    tok = rng.integers(0, V, size=(B, g)).astype(np.int32)
    u = rng.random((B, g + 1)).astype(np.float32)
    a = oracle_mod.verify(base.astype(np.float32), dbase.astype(np.float32), "f32", tok, np.full(B, g, np.int32), u,
                          np.full(B, 2.0, np.float32))
    b = oracle_mod.verify((base / 2).astype(np.float32), (dbase / 2).astype(np.float32), "f32", tok,
                          np.full(B, g, np.int32), u, np.full(B, 1.0, np.float32))
    np.testing.assert_allclose(a.p_hat, b.p_hat, rtol=1e-14)
    np.testing.assert_array_equal(a.out_tokens, b.out_tokens)
    # p_hat over every token of a row sums to one (normaliser)
    V2 = 37
    row = rng.normal(0, 2, size=V2).astype(np.float32)
    t = np.broadcast_to(row, (V2, 2, V2)).copy()
    d = np.broadcast_to(row[::-1].copy(), (V2, 1, V2)).copy()
    res = oracle_mod.verify(t, d, "f32", np.arange(V2, dtype=np.int32).reshape(V2, 1), np.ones(V2, np.int32),
                            np.full((V2, 2), 0.5, np.float32), np.full(V2, 0.8, np.float32))
    assert res.p_hat[:, 0].sum() == pytest.approx(1.0, abs=1e-14)
    assert res.q_hat[:, 0].sum() == pytest.approx(1.0, abs=1e-14)


def test_bf16_widening(oracle_mod):
    from speculative_decoding_verification_45_gb300 import workloads

    vals = np.array([1.0, -2.5, 3.140625, 0.0078125, -np.inf])
    bits = workloads.f64_to_bf16_bits(vals)
    V = vals.size
    t = np.broadcast_to(bits, (1, 2, V)).copy()
    d = np.broadcast_to(bits, (1, 1, V)).copy()
    res = oracle_mod.verify(t, d, "bf16", np.array([[2]], np.int32), np.array([1], np.int32),
                            np.full((1, 2), 0.5, np.float32), np.ones(1, np.float32))
    expect = np.exp(vals[2]) / np.exp(vals[:4]).sum()
    assert res.p_hat[0, 0] == pytest.approx(expect, rel=1e-14)


# ----------------------------------------------------------------------------
# edge cases and status bits
# ----------------------------------------------------------------------------

def test_zero_drafts_sample_from_p0(oracle_mod):
    p0 = np.array([0.05, 0.45, 0.5])
    N = 3000
    u = _grid(N)
    t = np.broadcast_to(np.log(p0).astype(np.float32), (N, 2, 3)).copy()
    d = np.full((N, 1, 3), np.nan, np.float32)
    res = oracle_mod.verify(t, d, "f32", np.full((N, 1), -1, np.int32), np.zeros(N, np.int32),
                            np.stack([np.full(N, np.nan), u], 1).astype(np.float32), np.ones(N, np.float32))
    assert np.all(res.out_num_accepted == 0) and np.all(res.seq_status == 0)
    freq = np.bincount(res.out_tokens[:, 0], minlength=3) / N
    np.testing.assert_allclose(freq, p0, atol=2.0 / N)
    assert np.all(res.out_tokens[:, 1] == -1)


def test_invalid_inputs_set_status_and_emit_minus_one(oracle_mod):
    V, g = 8, 2
    rng = np.random.default_rng(1)
    t = rng.normal(size=(5, g + 1, V)).astype(np.float32)
    d = rng.normal(size=(5, g, V)).astype(np.float32)
    tok = np.array([[1, 2], [1, 8], [1, 2], [1, 2], [3, 3]], np.int32)
    nd = np.array([2, 2, 2, 3, 2], np.int32)
    T = np.array([1.0, 1.0, -0.5, 1.0, 1.0], np.float32)
    t[4, 0, :] = -np.inf  # sampled row without a finite normaliser
    res = oracle_mod.verify(t, d, "f32", tok, nd, np.full((5, g + 1), 0.5, np.float32), T)
    assert list(res.seq_status) == [0, oracle_mod.STATUS_BAD_TOKEN, oracle_mod.STATUS_BAD_TEMPERATURE,
                                    oracle_mod.STATUS_BAD_NUM_DRAFT, oracle_mod.STATUS_BAD_LOGITS]
    for b in range(1, 5):
        assert np.all(res.out_tokens[b] == -1) and res.out_num_accepted[b] == 0
    for bad_t in [np.nan, np.inf, 1e-39]:
        r2 = oracle_mod.verify(t[:1], d[:1], "f32", tok[:1], nd[:1], np.full((1, g + 1), 0.5, np.float32),
                               np.array([bad_t], np.float32))
        assert r2.seq_status[0] == oracle_mod.STATUS_BAD_TEMPERATURE


def test_padding_is_never_read(oracle_mod):
    from speculative_decoding_verification_45_gb300 import workloads

    b = workloads.make_config(4, B=9)
    assert (b.num_draft < b.gmax).any()
    res = oracle_mod.verify_batch(b)
    assert np.all(res.seq_status == 0)
    for s in range(b.B):
        n = res.out_num_accepted[s]
        assert 0 <= n <= b.num_draft[s]
        assert np.all(res.out_tokens[s, n + 1:] == -1)
        assert np.all(res.out_tokens[s, :n] == b.tokens[s, :n])
        assert 0 <= res.out_tokens[s, n] < b.V


def test_results_do_not_depend_on_thread_count(oracle_mod):
    from speculative_decoding_verification_45_gb300 import workloads

    b = workloads.edge_batch("mixed", V=301, gamma=4, B=23)
    r1 = oracle_mod.verify_batch(b, nthreads=1)
    r5 = oracle_mod.verify_batch(b, nthreads=5)
    np.testing.assert_array_equal(r1.out_tokens, r5.out_tokens)
    np.testing.assert_array_equal(r1.out_num_accepted, r5.out_num_accepted)


def test_empty_batch(oracle_mod):
    res = oracle_mod.verify(np.zeros((0, 3, 4), np.float32), np.zeros((0, 2, 4), np.float32), "f32",
                            np.zeros((0, 2), np.int32), np.zeros(0, np.int32), np.zeros((0, 3), np.float32),
                            np.zeros(0, np.float32))
    assert res.out_tokens.shape == (0, 3)


# ----------------------------------------------------------------------------
# exact boundaries: rows whose softmax values are exact binary fractions
# ----------------------------------------------------------------------------

def test_strict_accept_test_at_exact_ratio(oracle_mod):
    """p(x) = 1/4, q(x) = 1/2 exactly: r = 1/2 sits on the threshold and must reject."""
    t = np.zeros((4, 2, 4), np.float32)                       # p uniform: 1/4 each
    d = np.full((4, 1, 4), -np.inf, np.float32)
    d[:, :, :2] = 0.0                                         # q = (1/2, 1/2, 0, 0)
    r = np.array([0.5, np.nextafter(np.float32(0.5), np.float32(0)), 0.0, 0.0], np.float32)
    tok = np.array([[0], [0], [0], [0]], np.int32)
    t[3, 0, 0] = -np.inf                                      # p(x) = 0 for the last copy
    res = oracle_mod.verify(t, d, "f32", tok, np.ones(4, np.int32), np.stack([r, np.full(4, 0.3)], 1)
                            .astype(np.float32), np.ones(4, np.float32))
    assert list(res.out_num_accepted) == [0, 1, 1, 0]        # p(x)=0 rejects even at r = 0


def test_inverse_cdf_at_exact_boundaries(oracle_mod):
    """Bonus row uniform over 4 ids: C = (1/4, 1/2, 3/4, 1); u on a boundary picks the next id."""
    u = np.array([0.0, 0.25, 0.5, 0.75, np.nextafter(np.float32(0.25), np.float32(0)),
                  np.nextafter(np.float32(1), np.float32(0))], np.float32)
    B = u.size
    t = np.zeros((B, 1, 4), np.float32)
    res = oracle_mod.verify(t, np.zeros((B, 0, 4), np.float32), "f32", np.zeros((B, 0), np.int32),
                            np.zeros(B, np.int32), u.reshape(B, 1), np.ones(B, np.float32))
    assert list(res.out_tokens[:, 0]) == [0, 1, 2, 3, 0, 3]


def test_uniform_columns_used(oracle_mod):
    """Accept draws come from columns i < g; the final sample from column gmax (not g)."""
    # g = 1 < gmax = 3; position 0 has p/q = 1/2 exactly
    t = np.full((1, 4, 4), np.inf, np.float32)
    t[0, :2] = 0.0
    d = np.full((1, 3, 4), np.inf, np.float32)
    d[0, 0] = -np.inf
    d[0, 0, :2] = 0.0
    uni = np.array([[0.9, 0.1, 0.1, 0.6]], np.float32)        # reject at 0 (0.9 >= 1/2)
    res = oracle_mod.verify(t, d, "f32", np.array([[1, -1, -1]], np.int32), np.array([1], np.int32), uni,
                            np.ones(1, np.float32))
    # residual = max(0, p - q) = (0, 0, 1/4, 1/4): u = 0.6 picks id 3, u = 0.1 would pick id 2
    assert res.out_num_accepted[0] == 0 and list(res.out_tokens[0]) == [3, -1, -1, -1]


def test_each_position_uses_its_own_uniform(oracle_mod):
    """Two positions with p/q = 1/2 exactly: r = (0.1, 0.9) accepts the first, rejects the second."""
    t = np.zeros((2, 3, 4), np.float32)                       # p uniform
    d = np.full((2, 2, 4), -np.inf, np.float32)
    d[:, :, :2] = 0.0                                         # q = (1/2, 1/2, 0, 0)
    uni = np.array([[0.1, 0.9, 0.5], [0.9, 0.1, 0.5]], np.float32)
    res = oracle_mod.verify(t, d, "f32", np.array([[0, 1], [0, 1]], np.int32), np.full(2, 2, np.int32), uni,
                            np.ones(2, np.float32))
    assert list(res.out_num_accepted) == [1, 0]


def test_bonus_row_normaliser(oracle_mod):
    """Rows with different shifts: the bonus sample's mass S is 1 (p of the bonus row)."""
    t = np.stack([np.log([0.5, 0.5, 1e-30, 1e-30]) + 3.0, np.log([0.1, 0.2, 0.3, 0.4]) - 5.0]).astype(np.float32)
    d = (np.log([[0.5, 0.5, 1e-30, 1e-30]]) + 7.0).astype(np.float32)
    res = oracle_mod.verify(t[None], d[None], "f32", np.array([[0]], np.int32), np.ones(1, np.int32),
                            np.array([[0.3, 0.5]], np.float32), np.ones(1, np.float32))
    assert res.out_num_accepted[0] == 1
    assert res.resid_mass[0] == pytest.approx(1.0, rel=1e-12)
    assert res.out_tokens[0, 1] == 2                          # C = (.1, .3, .6, 1): u = 0.5 -> id 2


# ----------------------------------------------------------------------------
# point-mass proposals (prompt lookup): q_i is 1 at the drafted id
# ----------------------------------------------------------------------------

def test_point_mass_accept_and_residual(oracle_mod):
    """p = (0.1, 0.6, 0.3), draft id 1: accepted iff r < 0.6; the residual is p
    without id 1, i.e. (0.25, 0, 0.75)."""
    N = 2000
    r, u = np.meshgrid(_grid(N // 40), _grid(40), indexing="ij")
    p = [[0.1, 0.6, 0.3], [1 / 3, 1 / 3, 1 / 3]]
    b = _batch(p, [[0.2, 0.2, 0.6]], np.full(r.size, 1), r.ravel(), u.ravel())
    res = oracle_mod.verify(b["target"], None, "f32", b["tokens"], b["num_draft"], b["uniforms"],
                            b["temperature"])
    acc = res.out_num_accepted == 1
    np.testing.assert_array_equal(acc, r.ravel() < 0.6 - 1e-6)
    rej = ~acc
    y = res.out_tokens[rej, 0]
    assert set(np.unique(y)) <= {0, 2}
    np.testing.assert_array_equal(y == 0, u.ravel()[rej] < 0.25)
    np.testing.assert_allclose(res.q_hat[:, 0], 1.0)
    assert np.all(np.isnan(res.logz_d))


def test_point_mass_output_law_is_p(oracle_mod):
    """Theorem with a deterministic proposal: the emitted token still follows p."""
    p0 = np.array([0.15, 0.45, 0.1, 0.3])
    N = 400
    rr, uu = np.meshgrid(_grid(N), _grid(N), indexing="ij")
    for x in range(4):
        b = _batch([p0, [0.25] * 4], [[0.25] * 4], np.full(N * N, x), rr.ravel(), uu.ravel())
        res = oracle_mod.verify(b["target"], None, "f32", b["tokens"], b["num_draft"], b["uniforms"],
                                b["temperature"], diagnostics=False)
        law = np.bincount(res.out_tokens[:, 0], minlength=4) / (N * N)
        np.testing.assert_allclose(law, p0, atol=3.0 / N)

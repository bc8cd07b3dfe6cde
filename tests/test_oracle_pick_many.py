"""Pins of oracle.pick_many, the oracle's final draw for many uniforms at once
(used by the draw-rate tests).  It must give exactly what oracle_verify gives as
the final token of a round for the same row and uniform: the bonus draw
(gamma_max = 0 rounds), the residual draw after a rejection at position 0, and
the point-mass residual; and the closed-form inverse CDF on a tiny row
("Speculative Decoding", ch.3: the draw from p or from norm(max(0, p - q)))."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads

LARGEST_BELOW_ONE = np.float32(np.nextafter(np.float32(1.0), np.float32(0.0)))


def _rows(n, V, seed, dtype):
    rng = np.random.default_rng(seed)
    t = rng.normal(0.0, 3.0, size=(n, 2, V))
    d = t[:, :1] + rng.normal(0.0, 0.7, size=(n, 1, V))
    if dtype == "bf16":
        return workloads.f64_to_bf16_bits(t), workloads.f64_to_bf16_bits(d)
    return t.astype(np.float32), d.astype(np.float32)


def test_tiny_row_closed_form(oracle_mod):
    # p = (0.1, 0.6, 0.3): u in [0, 0.1) -> 0, [0.1, 0.7) -> 1, [0.7, 1) -> 2
    logits = np.log(np.array([0.1, 0.6, 0.3], np.float64)).astype(np.float32)
    u = np.array([0.0, 0.05, 0.0999, 0.1001, 0.5, 0.6999, 0.7001, 0.95], np.float32)
    picks, margins, S = oracle_mod.pick_many(logits, "f32", 1.0, u)
    assert picks.tolist() == [0, 0, 0, 1, 1, 1, 2, 2]
    assert abs(S - 1.0) < 1e-12
    assert margins[2] == pytest.approx(1e-4, abs=1e-6) and margins[3] == pytest.approx(1e-4, abs=1e-6)


@pytest.mark.parametrize("dtype,V,T", [("f32", 37, 1.0), ("bf16", 1000, 0.7), ("bf16", 5000, 1.3)])
def test_bonus_draw_equals_a_round_with_no_drafts(oracle_mod, dtype, V, T):
    n, reps = 6, 40
    t, _ = _rows(n, V, 11, dtype)
    rng = np.random.default_rng(5)
    u = rng.random((n, reps), dtype=np.float32)
    for b in range(n):
        picks, margins, _ = oracle_mod.pick_many(t[b, 0], dtype, T, u[b])
        for k in range(reps):
            r = oracle_mod.verify(t[b:b + 1, :1], t[b:b + 1, :0], dtype, np.zeros((1, 0), np.int32),
                                  np.zeros(1, np.int32), u[b, k:k + 1][None, :], np.full(1, T, np.float32))
            assert r.out_tokens[0, 0] == picks[k]
            assert r.samp_margin[0] == pytest.approx(margins[k], rel=1e-12, abs=1e-15)


@pytest.mark.parametrize("point", [False, True])
def test_residual_draw_equals_a_round_rejected_at_position_zero(oracle_mod, point):
    dtype, V, T, n, reps = "bf16", 3000, 1.0, 4, 30
    t, d = _rows(n, V, 23, dtype)
    tf = workloads.bf16_bits_to_f64(t)
    df = workloads.bf16_bits_to_f64(d)
    rng = np.random.default_rng(9)
    for b in range(n):
        p = np.exp(tf[b, 0] - tf[b, 0].max())
        p /= p.sum()
        if point:
            x = int(np.argmax(p))  # u < p(x) fails for u just below 1
            picks, _, mass = oracle_mod.pick_many(t[b, 0], dtype, T, u_all := rng.random(reps, dtype=np.float32),
                                                  mode=oracle_mod.PICK_POINT, xn=x)
            assert mass == pytest.approx(1.0 - p[x], rel=1e-9)
        else:
            q = np.exp(df[b, 0] - df[b, 0].max())
            q /= q.sum()
            x = int(np.argmax(q - p))  # q(x) > p(x): rejected for u just below 1
            picks, _, mass = oracle_mod.pick_many(t[b, 0], dtype, T, u_all := rng.random(reps, dtype=np.float32),
                                                  mode=oracle_mod.PICK_RESIDUAL, draft_row=d[b, 0])
            assert mass == pytest.approx(np.maximum(p - q, 0).sum(), rel=1e-9)
        for k in range(reps):
            uni = np.array([[LARGEST_BELOW_ONE, u_all[k]]], np.float32)
            r = oracle_mod.verify(t[b:b + 1], None if point else d[b:b + 1], dtype, np.array([[x]], np.int32),
                                  np.ones(1, np.int32), uni, np.full(1, T, np.float32))
            assert r.out_num_accepted[0] == 0
            assert r.out_tokens[0, 0] == picks[k]

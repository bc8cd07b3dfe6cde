"""Monte-Carlo checks of the oracle's output law.

- chi-square of the oracle's outcomes against the brute-force law on tiny
  vocabularies (the law itself is pinned to the distribution-preservation
  theorem in test_enumerator.py);
- mean tokens per round on rows with an exact acceptance rate against
  E = (1 - a^(g+1)) / (1 - a) ("Speculative Decoding", atonlee.tistory.com/330,
  ch.4 table; "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가", section on the
  two numbers that set the gain).
"""
import numpy as np
import pytest

from oracle import analytic, enumerate_law
from speculative_decoding_verification_45_gb300 import workloads
from tests import law_checks


def _dirichlet_rows(seed, V, gamma, zero_frac=0.0):
    rng = np.random.default_rng(seed)

    def one():
        x = rng.dirichlet(np.ones(V))
        if zero_frac:
            m = rng.random(V) < zero_frac
            m[rng.integers(V)] = False
            x[m] = 0.0
            x /= x.sum()
        return x

    return np.array([one() for _ in range(gamma + 1)]), np.array([one() for _ in range(gamma)])


@pytest.mark.parametrize("V,gamma,zf,seed", [(3, 1, 0.0, 21), (4, 2, 0.0, 22), (4, 3, 0.25, 23), (6, 2, 0.0, 24)])
def test_oracle_outcomes_follow_enumerated_law(oracle_mod, V, gamma, zf, seed):
    p, q = _dirichlet_rows(seed, V, gamma, zf)
    # the float32 logits shift p and q by ~1e-7; take the law of the rows as stored
    batch = workloads.tiny_batch(p, q, N=200_000, seed=seed)
    p_st = np.exp(batch.target[0].astype(np.float64))
    q_st = np.exp(batch.draft[0].astype(np.float64))
    law = enumerate_law.outcome_law(p_st / p_st.sum(1, keepdims=True), q_st / q_st.sum(1, keepdims=True))
    res = oracle_mod.verify_batch(batch, diagnostics=False)
    keys = law_checks.outcome_keys(res.out_tokens, res.out_num_accepted)
    stat, pval, bins = law_checks.chi_square_vs_law(keys, law)
    assert pval > 1e-3, (stat, pval, bins)


@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.5, 2), (0.5, 7), (0.9, 7), (0.6, 10)])
def test_mean_tokens_per_round_matches_E(oracle_mod, alpha, gamma):
    p, q = workloads.alpha_rows(alpha, gamma)
    batch = workloads.tiny_batch(p, q, N=200_000, seed=int(alpha * 1000) + gamma)
    res = oracle_mod.verify_batch(batch, diagnostics=False)
    z = law_checks.mean_tokens_z(res.out_num_accepted, analytic.expected_tokens(alpha, gamma))
    assert abs(z) < 4.0, z


def test_worked_example_rates(oracle_mod):
    p, q = workloads.worked_example_rows()
    N = 400_000
    batch = workloads.tiny_batch(p, q, N=N, seed=77)
    res = oracle_mod.verify_batch(batch, diagnostics=False)
    drafted0 = batch.tokens[:, 0] == 0
    acc_rate = (res.out_num_accepted[drafted0] == 1).mean()
    se = np.sqrt(0.25 * 0.75 / drafted0.sum())
    assert abs(acc_rate - 0.25) < 5 * se
    freq0 = (res.out_tokens[:, 0] == 0).mean()
    assert abs(freq0 - 0.1) < 5 * np.sqrt(0.1 * 0.9 / N)

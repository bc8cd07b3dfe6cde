"""The brute-force outcome law, pinned to the distribution-preservation theorem.

The theorem ("Speculative Decoding", atonlee.tistory.com/330, ch.3; the "Fast
Inference from Transformers via Speculative Decoding" notes, proof sketch):
the token emitted at a position has law p at that position, whatever q is.
"""
import numpy as np
import pytest

from oracle import analytic, enumerate_law


def _rows(rng, V, gamma, zero_frac=0.0):
    def one():
        x = rng.dirichlet(np.ones(V))
        if zero_frac:
            m = rng.random(V) < zero_frac
            if m.all():
                m[0] = False
            x[m] = 0.0
            x /= x.sum()
        return x

    p = np.array([one() for _ in range(gamma + 1)])
    q = np.array([one() for _ in range(gamma)])
    return p, q


@pytest.mark.parametrize("V,gamma,zf,seed", [(3, 1, 0.0, 1), (4, 2, 0.0, 2), (5, 3, 0.0, 3), (4, 3, 0.3, 4),
                                             (6, 2, 0.4, 5), (2, 3, 0.0, 6)])
def test_theorem_every_emitted_token_has_law_p(V, gamma, zf, seed):
    rng = np.random.default_rng(seed)
    p, q = _rows(rng, V, gamma, zf)
    law = enumerate_law.outcome_law(p, q)
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    np.testing.assert_allclose(enumerate_law.marginal_first_token(law, V), p[0], atol=1e-12)
    for i in range(1, gamma + 1):
        np.testing.assert_allclose(enumerate_law.conditional_token(law, i, V), p[i], atol=1e-12)


def test_accepted_count_law_is_product_of_alphas():
    rng = np.random.default_rng(11)
    p, q = _rows(rng, 4, 3)
    law = enumerate_law.outcome_law(p, q)
    alphas = [analytic.acceptance_rate(p[i], q[i]) for i in range(3)]
    np.testing.assert_allclose(enumerate_law.accepted_count_law(law, 3), analytic.accepted_count_pmf(alphas),
                               atol=1e-12)


def test_worked_example_accept_path_mass():
    # q(x)=0.4, p(x)=0.1: the accept path emits x with probability 0.4 * 0.25 = 0.1
    p = [[0.1, 0.6, 0.3], [1 / 3, 1 / 3, 1 / 3]]
    q = [[0.4, 0.3, 0.3]]
    law = enumerate_law.outcome_law(p, q)
    accept_x = sum(pr for k, pr in law.items() if k[0] == 1 and k[1] == 0)
    assert accept_x == pytest.approx(0.1, abs=1e-15)
    # and no resample ever returns x, since max(0, p - q) is 0 there
    assert all(not (k[0] == 0 and k[1] == 0) for k in law)


def test_identical_rows_always_accept():
    p = [[0.2, 0.3, 0.5]] * 3
    law = enumerate_law.outcome_law(p, p[:2])
    assert enumerate_law.accepted_count_law(law, 2)[2] == pytest.approx(1.0)

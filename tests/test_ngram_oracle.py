"""The prompt-lookup proposer oracle and the draft-length rule, pinned by
hand-derived cases and by an independent search (Python's str.rfind)."""
import numpy as np
import pytest

from oracle import gamma_policy, ngram

CASES = [
    # context, min_n, max_n, gamma, expected proposal
    ([1, 2, 3, 4, 1, 2], 1, 3, 3, [3, 4, 1]),          # n=3 absent, n=2 at j=0
    ([5, 6, 7, 5, 6, 8, 5, 6], 1, 2, 3, [8, 5, 6]),     # most recent occurrence wins
    ([5, 6, 7, 5, 6, 8, 5, 6], 3, 4, 3, []),            # no match of length >= 3
    ([1, 2, 1], 1, 3, 3, [2, 1]),                       # proposal cut at the context end
    ([9, 9, 9, 9], 2, 2, 5, [9]),                       # overlapping occurrence allowed
    ([4, 7, 4, 7, 1, 4, 7], 1, 2, 2, [1, 4]),           # n=2 match at j=2 beats n=1 matches
    ([3], 1, 4, 2, []),                                 # nothing earlier
    ([1, 2, 3, 9, 2, 3, 1, 2, 3], 2, 3, 4, [9, 2, 3, 1]),  # n=3 at j=0 (longest wins over later n=2)
]


@pytest.mark.parametrize("ctx,mn,mx,k,expect", CASES)
def test_golden(ctx, mn, mx, k, expect):
    assert ngram.propose(ctx, mn, mx, k) == expect


def _rfind_proposal(ctx, mn, mx, k):
    """Same definition through string search: tokens as fixed-width fields."""
    enc = "".join(f"{t:06d}," for t in ctx)
    L = len(ctx)
    for n in range(mx, mn - 1, -1):
        if n < 1 or n >= L:
            continue
        suf = "".join(f"{t:06d}," for t in ctx[L - n:])
        pos = enc.rfind(suf, 0, (L - 1) * 7)  # an occurrence ending before the last token
        if pos >= 0:
            j = pos // 7
            return ctx[j + n:j + n + k]
    return []


def test_against_string_search():
    rng = np.random.default_rng(3)
    for _ in range(400):
        L = int(rng.integers(1, 60))
        ctx = list(rng.integers(0, 4, size=L))
        mn = int(rng.integers(1, 4))
        mx = mn + int(rng.integers(0, 4))
        k = int(rng.integers(1, 6))
        assert ngram.propose(ctx, mn, mx, k) == _rfind_proposal(ctx, mn, mx, k), (ctx, mn, mx, k)


def test_batch_padding():
    ctx = np.array([[1, 2, 1, 0, 0], [7, 8, 9, 7, 8]], np.int32)
    toks, num = ngram.propose_batch(ctx, [3, 5], 1, 2, 3)
    assert list(num) == [2, 3] and list(toks[0]) == [2, 1, -1] and list(toks[1]) == [9, 7, 8]


def test_gamma_rule():
    g, r, a = 4, 0, 0
    # two rejection rounds in a row lower gamma by one, twice -> 2
    for n in (1, 0, 2, 0):
        g, r, a = gamma_policy.step(g, r, a, g, n, 1, 8, down_after=2, up_after=3)
    assert g == 2
    # never below 1
    for _ in range(10):
        g, r, a = gamma_policy.step(g, r, a, g, 0, 1, 8, down_after=2, up_after=3)
    assert g == 1
    # three full-acceptance rounds raise it by one
    for _ in range(3):
        g, r, a = gamma_policy.step(g, r, a, g, g, 1, 8, down_after=2, up_after=3)
    assert g == 2
    # an interrupted streak does not count
    g, r, a = gamma_policy.step(g, r, a, g, g, 1, 8, 2, 3)
    g, r, a = gamma_policy.step(g, r, a, g, 0, 1, 8, 2, 3)
    g, r, a = gamma_policy.step(g, r, a, g, g, 1, 8, 2, 3)
    assert g == 2
    # no drafts: no change
    assert gamma_policy.step(5, 1, 1, 0, 0, 1, 8, 2, 3) == (5, 1, 1)


def test_vectorised_controller_matches_rule():
    from speculative_decoding_verification_45_gb300.policy import GammaController

    rng = np.random.default_rng(9)
    B, gmax = 64, 8
    ctl = GammaController(B, gmax, gamma_start=4, down_after=2, up_after=3)
    state = [(4, 0, 0)] * B
    for _ in range(200):
        g = np.minimum(ctl.gamma, rng.integers(0, gmax + 1, size=B))
        n = np.array([rng.integers(0, gi + 1) for gi in g])
        got = ctl.update(g, n)
        state = [gamma_policy.step(state[b][0], state[b][1], state[b][2], int(g[b]), int(n[b]), 1, gmax, 2, 3)
                 for b in range(B)]
        assert list(got) == [st[0] for st in state]

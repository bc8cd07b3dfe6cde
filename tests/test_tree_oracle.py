"""Pins of the tree-verification oracle (oracle_tree_verify) and of the tree
enumerator, on the CPU.

The rule (candidates are point masses, tried in index order against p without
the ids already rejected at that node) is the single-candidate rule of
"Speculative Decoding" (atonlee.tistory.com/330) ch.3 applied once per child;
the pins check what must follow from the pages and from mathematics:
  - the distribution-preservation theorem ([P1] ch.3): at every node reached,
    the next emitted token follows that node's target row (enumerator, exact);
  - a chain-shaped tree is the chain round with point-mass drafts, whose oracle
    is pinned in test_oracle_pins.py (exact equality);
  - exact acceptance fractions on uniform grids with binary-fraction rows;
  - greedy walks follow argmax children only and end on the argmax;
  - invalid trees are flagged.
"""
import itertools

import numpy as np
import pytest

from oracle import enumerate_law
from speculative_decoding_verification_45_gb300 import workloads
from tests import law_checks


def _random_tree(rng, N, V, dup=True):
    par = [-1] + [int(rng.integers(0, k)) for k in range(1, N)]
    tok = [-1] + [int(rng.integers(0, V)) for _ in range(1, N)]
    if not dup:  # distinct ids among siblings
        for k in range(N):
            kids = [c for c in range(1, N) if par[c] == k]
            ids = rng.permutation(V)[: len(kids)]
            for c, x in zip(kids, ids):
                tok[c] = int(x)
    return par, tok


def _dirichlet(rng, N, V, zero_frac=0.0):
    rows = rng.dirichlet(np.ones(V), size=N)
    if zero_frac:
        m = rng.random((N, V)) < zero_frac
        m[np.arange(N), rng.integers(0, V, N)] = False
        rows = np.where(m, 0.0, rows)
        rows /= rows.sum(1, keepdims=True)
    return rows


@pytest.mark.parametrize("seed", range(6))
def test_enumerated_tree_law_preserves_target(seed):
    """Theorem ([P1] ch.3, applied per child): the law sums to 1 and, at every
    node path of positive probability, the next emitted token follows that
    node's row exactly -- whatever the tree shape, duplicate sibling ids and
    zero probabilities."""
    rng = np.random.default_rng(100 + seed)
    V, N = int(rng.integers(2, 5)), int(rng.integers(2, 8))
    par, tok = _random_tree(rng, N, V, dup=True)
    p = _dirichlet(rng, N, V, zero_frac=0.3 if seed % 2 else 0.0)
    law = enumerate_law.tree_outcome_law(p, par, tok)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    # group by accepted node path; the next token after path (node_1..node_i) is
    # the token of node_{i+1} if one was accepted, else the final sample
    nxt = {}
    for key, pr in law.items():
        n = key[0]
        nodes, toks = key[1:1 + n], key[1 + n:]
        for i in range(n + 1):
            prefix = tuple(nodes[:i])
            d = nxt.setdefault(prefix, np.zeros(V))
            d[toks[i]] += pr
    for prefix, d in nxt.items():
        node = prefix[-1] if prefix else 0
        np.testing.assert_allclose(d / d.sum(), p[node], atol=1e-12)


def test_enumerator_chain_tree_equals_chain_law():
    """A chain-shaped tree is the chain round with point-mass drafts."""
    rng = np.random.default_rng(7)
    V, g = 3, 3
    p = _dirichlet(rng, g + 1, V)
    tok = [-1] + [int(x) for x in rng.integers(0, V, g)]
    law_t = enumerate_law.tree_emitted_law(enumerate_law.tree_outcome_law(p, [-1, 0, 1, 2], tok))
    q = np.zeros((g, V))
    q[np.arange(g), tok[1:]] = 1.0
    law_c = {}
    for key, pr in enumerate_law.outcome_law(p, q).items():
        toks = key[1:]
        law_c[toks] = law_c.get(toks, 0.0) + pr
    assert set(law_t) == set(law_c)
    for k in law_t:
        assert abs(law_t[k] - law_c[k]) < 1e-12


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_tree_equals_chain_oracle(oracle_mod, T):
    """Exact equality with the pinned chain oracle in point-mass mode: target row
    i = node i, draft x_i = candidate of node i+1, r_i = uniform of node i+1,
    final draw = uniform column 0."""
    rng = np.random.default_rng(11)
    B, g, V = 300, 5, 50
    tb = workloads.tree_batch(B, g + 1, V, dtype="f32", seed=5, shape="chain", temps=(T,), ragged=True, zipf=False)
    tb.temperature[:] = T
    ref_t = oracle_mod.tree_verify_batch(tb)
    gmax = g
    target = np.full((B, gmax + 1, V), np.inf, np.float32)
    tokens = np.full((B, gmax), -1, np.int32)
    uniforms = np.zeros((B, gmax + 1), np.float32)
    num_draft = (tb.num_nodes - 1).astype(np.int32)
    for b in range(B):
        n = int(tb.num_nodes[b])
        target[b, :n] = tb.target[b, :n]
        tokens[b, : n - 1] = tb.tokens[b, 1:n]
        uniforms[b, : n - 1] = tb.uniforms[b, 1:n]
        uniforms[b, gmax] = tb.uniforms[b, 0]
    ref_c = oracle_mod.verify(target, None, "f32", tokens, num_draft, uniforms, tb.temperature)
    np.testing.assert_array_equal(ref_t.out_num_accepted, ref_c.out_num_accepted)
    for b in range(B):
        n = int(ref_c.out_num_accepted[b])
        np.testing.assert_array_equal(ref_t.out_tokens[b, : n + 1], ref_c.out_tokens[b, : n + 1])
        np.testing.assert_array_equal(ref_t.out_path[b, :n], np.arange(1, n + 1))
        assert (ref_t.out_tokens[b, n + 1:] == -1).all() and (ref_t.out_path[b, n:] == -1).all()


def test_star_acceptance_fractions_exact(oracle_mod):
    """Root with children ids (1, 0) and p = (1/4, 1/2, 1/8, 1/8): on a midpoint
    grid of the two test uniforms child 1 passes for exactly 1/2 of the grid,
    child 2 for exactly 1/4 (u_2 * (1 - 1/2) < 1/4), and the rest falls through
    to p without {0, 1}: ids 2 and 3 each half of the u_0 grid."""
    p = np.array([[0.25, 0.5, 0.125, 0.125], [0.25] * 4, [0.25] * 4])
    K = 16
    grid = (np.arange(K) + 0.5) / K
    u1, u2, u0 = [a.ravel() for a in np.meshgrid(grid, grid, grid, indexing="ij")]
    cnt = u1.size
    tb = workloads.tree_tiny(p, [-1, 0, 0], [-1, 1, 0], cnt, seed=0)
    tb.uniforms[:] = np.stack([u0, u1, u2], axis=1).astype(np.float32)
    r = oracle_mod.tree_verify_batch(tb)
    first = r.out_tokens[:, 0]
    acc1 = (r.out_num_accepted == 1) & (r.out_path[:, 0] == 1)
    acc2 = (r.out_num_accepted == 1) & (r.out_path[:, 0] == 2)
    assert acc1.sum() * 2 == cnt and acc2.sum() * 4 == cnt
    fell = r.out_num_accepted == 0
    assert fell.sum() * 4 == cnt
    assert (first[fell] == 2).sum() * 2 == fell.sum() and (first[fell] == 3).sum() * 2 == fell.sum()
    assert set(np.unique(first[acc1])) == {1} and set(np.unique(first[acc2])) == {0}


def test_duplicate_sibling_ids_never_pass_twice(oracle_mod):
    """A repeated id among siblings has no mass left once rejected: the tree
    (1, 1, 0) under the root gives the same results as (1, 0)."""
    rng = np.random.default_rng(3)
    p = _dirichlet(rng, 4, 4)
    tb3 = workloads.tree_tiny(p, [-1, 0, 0, 0], [-1, 1, 1, 0], 20000, seed=9)
    tb2 = workloads.tree_tiny(p[[0, 1, 3]], [-1, 0, 0], [-1, 1, 0], 20000, seed=9)
    tb2.uniforms = tb3.uniforms[:, [0, 1, 3]].copy()
    r3, r2 = oracle_mod.tree_verify_batch(tb3), oracle_mod.tree_verify_batch(tb2)
    np.testing.assert_array_equal(r3.out_tokens[:, 0], r2.out_tokens[:, 0])
    assert not (r3.out_path[:, 0] == 2).any()


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_oracle_tree_outcomes_follow_enumerated_law(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    V, N = 4, 6
    par, tok = _random_tree(rng, N, V, dup=(seed == 33))
    p = _dirichlet(rng, N, V, zero_frac=0.2 if seed == 32 else 0.0)
    tb = workloads.tree_tiny(p, par, tok, 200_000, seed=seed)
    p_st = np.exp(tb.target[0].astype(np.float64))
    law = enumerate_law.tree_outcome_law(p_st / p_st.sum(1, keepdims=True), par, tok)
    r = oracle_mod.tree_verify_batch(tb)
    keys = law_checks.tree_outcome_keys(r.out_tokens, r.out_num_accepted, r.out_path)
    stat, pval, bins = law_checks.chi_square_vs_law(keys, law)
    assert pval > 1e-3, (stat, pval, bins)


def test_greedy_walk_follows_argmax_children(oracle_mod):
    tb = workloads.tree_batch(200, 12, 7, dtype="f32", seed=4, shape="random", temps=(0.0,), zipf=False, sigma=2.0)
    r = oracle_mod.tree_verify_batch(tb)
    V = tb.V
    for b in range(tb.B):
        nn, n = int(tb.num_nodes[b]), int(r.out_num_accepted[b])
        node = 0
        for i in range(n):
            c = int(r.out_path[b, i])
            am = int(np.argmax(tb.target[b, node]))
            assert tb.parent[b, c] == node and tb.tokens[b, c] == am == r.out_tokens[b, i]
            node = c
        am = int(np.argmax(tb.target[b, node]))
        assert r.out_tokens[b, n] == am
        kids = [c for c in range(1, nn) if tb.parent[b, c] == node]
        assert all(tb.tokens[b, c] != am for c in kids)
        assert 0 <= am < V


def test_invalid_trees_flagged(oracle_mod):
    tb = workloads.tree_batch(6, 8, 16, dtype="f32", seed=2, shape="random", temps=(1.0,), ragged=False, zipf=False)
    tb.parent[0, 3] = 3            # not an earlier node
    tb.tokens[1, 2] = 16           # id out of range
    tb.num_nodes[2] = 0            # no root
    tb.num_nodes[3] = 9            # more than N
    tb.temperature[4] = -1.0
    r = oracle_mod.tree_verify_batch(tb)
    assert list(r.seq_status[:5]) == [oracle_mod.STATUS_BAD_TREE, oracle_mod.STATUS_BAD_TOKEN,
                                      oracle_mod.STATUS_BAD_NUM_DRAFT, oracle_mod.STATUS_BAD_NUM_DRAFT,
                                      oracle_mod.STATUS_BAD_TEMPERATURE]
    assert (r.out_tokens[:5] == -1).all() and (r.out_num_accepted[:5] == 0).all() and (r.out_path[:5] == -1).all()
    assert r.seq_status[5] == 0 and r.out_tokens[5, 0] >= 0


def test_single_node_tree_samples_root_row(oracle_mod):
    """num_nodes = 1: no candidate; one token from the root row (bonus) on a u grid."""
    p = np.array([[0.5, 0.25, 0.125, 0.125]])
    K = 64
    tb = workloads.tree_tiny(p, [-1], [-1], K, seed=0)
    tb.uniforms[:, 0] = ((np.arange(K) + 0.5) / K).astype(np.float32)
    r = oracle_mod.tree_verify_batch(tb)
    assert (r.out_num_accepted == 0).all()
    counts = np.bincount(r.out_tokens[:, 0], minlength=4)
    np.testing.assert_array_equal(counts, (p[0] * K).astype(int))


def test_accept_test_is_strict_at_exact_boundaries(oracle_mod):
    """u equal to the threshold p(x)/(1 - p(R)) rejects (the printed test is the
    strict r < min(1, p/q)); the float just below accepts.  The root row is
    uniform over 4 ids (logits 0: p = 1/4 exactly); children carry ids 1, 0, 2,
    so child 1's threshold is 1/4 and child 3's, after ids 1 and 0 were
    rejected, is (1/4) / (1 - 1/2) = 1/2."""
    B4 = np.float32(0.25)
    b4 = np.nextafter(B4, np.float32(0.0))
    b2 = np.nextafter(np.float32(0.5), np.float32(0.0))
    cases = [  # (u_1, u_2, u_3) -> accepted node
        (B4, 0.9, 0.5, None), (b4, 0.9, 0.9, 1), (B4, 0.9, b2, 3), (0.3, 0.2, 0.9, 2)]
    N, V = 4, 4
    tb = workloads.tree_tiny(np.full((N, V), 0.25), [-1, 0, 0, 0], [-1, 1, 0, 2], len(cases), seed=0)
    tb.target[:] = 0.0
    for i, (u1, u2, u3, _) in enumerate(cases):
        tb.uniforms[i] = [0.3, u1, u2, u3]
    r = oracle_mod.tree_verify_batch(tb)
    for i, (_, _, _, want) in enumerate(cases):
        got = int(r.out_path[i, 0]) if r.out_num_accepted[i] else None
        assert got == want, (i, got, want)


def test_margins_recorded(oracle_mod):
    """acc_margin = |u_c - p(x_c)/(1 - p(R))| at every tested node (NaN at untested
    ones); samp_margin = distance of u_0 to the nearest CDF boundary of the pick.
    Uniform root row over 4 ids, children ids 1, 0, 2; u = (0.1, 0.3, 0.2, 0.9)."""
    tb = workloads.tree_tiny(np.full((4, 4), 0.25), [-1, 0, 0, 0], [-1, 1, 0, 2], 2, seed=0)
    tb.target[:] = 0.0
    tb.uniforms[0] = [0.1, 0.3, 0.2, 0.9]   # child 1 rejected (0.3 > 1/4), child 2 accepted (0.2 < 1/3)
    tb.uniforms[1] = [0.1, 0.3, 0.9, 0.9]   # all rejected: final from ids {3}, u_0 = 0.1
    r = oracle_mod.tree_verify_batch(tb)
    u = tb.uniforms.astype(np.float64)
    assert r.out_path[0, 0] == 2
    np.testing.assert_allclose(r.acc_margin[0, 1:3], [abs(u[0, 1] - 0.25), abs(u[0, 2] - 1.0 / 3)], rtol=1e-12)
    assert np.isnan(r.acc_margin[0, 3]) and np.isnan(r.acc_margin[0, 0])
    np.testing.assert_allclose(r.acc_margin[1, 1:4], [abs(u[1, 1] - 0.25), abs(u[1, 2] - 1.0 / 3),
                                                      abs(u[1, 3] - 0.5)], rtol=1e-12)
    assert r.out_num_accepted[1] == 0 and r.out_tokens[1, 0] == 3
    np.testing.assert_allclose(r.samp_margin[1], u[1, 0], rtol=1e-12)   # only id 3 left: CDF (0, 1]

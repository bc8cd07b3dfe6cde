"""Exact outcome law of one verification round by brute-force enumeration.

TEST INFRASTRUCTURE.  For tiny vocabularies and few drafts this walks every
random choice of a round in the pages' order and sums path probabilities:

  1. each draft token x_i is drawn from q_i ("Fast Inference from Transformers
     via Speculative Decoding" notes, method details, step 1);
  2. position i accepts x_i with probability min(1, p_i(x_i)/q_i(x_i)) and the
     round stops at the first rejection ("Speculative Decoding",
     atonlee.tistory.com/330, ch.2 and ch.3; the notes above, step 3);
  3. a rejection at i emits one token from norm(max(0, p_i - q_i)); if all
     gamma drafts pass, one bonus token is drawn from p_gamma (same sources).

The result maps outcomes (n, y_0, ..., y_n) -- n accepted drafts, then the
emitted tokens -- to their probability.  The rows are fixed per position (no
dependence on earlier tokens), which is also how the Monte-Carlo batches are
built.  Pure-Python loops: keep V**gamma small.
"""
from __future__ import annotations

import itertools

import numpy as np


def outcome_law(p_rows, q_rows) -> dict:
    p = np.asarray(p_rows, dtype=np.float64)
    q = np.asarray(q_rows, dtype=np.float64)
    gamma, V = q.shape
    assert p.shape == (gamma + 1, V)
    law: dict = {}

    def add(key, prob):
        if prob > 0.0:
            law[key] = law.get(key, 0.0) + prob

    for drafts in itertools.product(range(V), repeat=gamma):
        path = 1.0
        for i, x in enumerate(drafts):
            path *= q[i, x]
        if path == 0.0:
            continue
        alive = path  # probability of reaching position i with every earlier draft accepted
        stopped = False
        for i, x in enumerate(drafts):
            acc = 1.0 if p[i, x] >= q[i, x] else p[i, x] / q[i, x]
            rej = alive * (1.0 - acc)
            if rej > 0.0:
                resid = np.maximum(p[i] - q[i], 0.0)
                mass = resid.sum()
                for y in range(V):
                    if resid[y] > 0.0:
                        add((i,) + tuple(drafts[:i]) + (y,), rej * resid[y] / mass)
            alive *= acc
            if alive == 0.0:
                stopped = True
                break
        if not stopped:
            for y in range(V):
                add((gamma,) + tuple(drafts) + (y,), alive * p[gamma, y])
    return law


def marginal_first_token(law: dict, V: int) -> np.ndarray:
    """P(y_0 = j): the first emitted token, whatever the path."""
    out = np.zeros(V)
    for key, pr in law.items():
        out[key[1]] += pr
    return out


def conditional_token(law: dict, i: int, V: int) -> np.ndarray:
    """P(y_i = j | the round emits at least i+1 tokens), i.e. given n >= i."""
    out = np.zeros(V)
    for key, pr in law.items():
        n = key[0]
        if n >= i:
            out[key[1 + i]] += pr
    s = out.sum()
    return out / s if s > 0 else out


def accepted_count_law(law: dict, gamma: int) -> np.ndarray:
    out = np.zeros(gamma + 1)
    for key, pr in law.items():
        out[key[0]] += pr
    return out


def tree_outcome_law(p_rows, parent, tokens) -> dict:
    """Exact law of one tree round with deterministic (point-mass) candidates.

    p_rows[k] is the target distribution at node k (node 0 = root); node k >= 1
    carries tokens[k] under parent[k] < k.  At the current node the children
    are tried in index order; with R the ids already rejected there, child c
    passes with probability p(tok_c) / (1 - p(R)) (zero when tok_c is in R) --
    the single-candidate rule of "Speculative Decoding" (atonlee.tistory.com/
    330) ch.3 with q the point mass, applied to p without R.  When none passes
    (or the node is a leaf) one token is drawn from p without R, renormalised.
    Returns {(path nodes..., emitted token ids...): probability}, the key being
    (n, node_1..node_n, y_0..y_n) with n accepted nodes.
    """
    p = np.asarray(p_rows, dtype=np.float64)
    N, V = p.shape
    children = {k: [c for c in range(1, N) if parent[c] == k] for k in range(N)}
    law: dict = {}

    def add(key, prob):
        if prob > 0.0:
            law[key] = law.get(key, 0.0) + prob

    def walk(node, nodes, toks, prob):
        rejected = []
        alive = prob
        for c in children[node]:
            mass_left = 1.0 - sum(p[node, t] for t in set(rejected))
            pc = 0.0 if tokens[c] in rejected else p[node, tokens[c]]
            acc = pc / mass_left if mass_left > 0.0 else 0.0
            if acc > 0.0:
                walk(c, nodes + (c,), toks + (int(tokens[c]),), alive * acc)
            alive *= 1.0 - acc
            if tokens[c] not in rejected:
                rejected.append(int(tokens[c]))
            if alive <= 0.0:
                return
        w = p[node].copy()
        w[list(set(rejected))] = 0.0
        if w.sum() <= 0.0:
            w = p[node].copy()
        w /= w.sum()
        for y in range(V):
            add((len(nodes),) + nodes + toks + (y,), alive * w[y])

    walk(0, (), (), 1.0)
    return law


def tree_emitted_law(law: dict) -> dict:
    """{emitted token tuple: probability} of a tree round's law."""
    out: dict = {}
    for key, pr in law.items():
        n = key[0]
        toks = key[1 + n:]
        out[toks] = out.get(toks, 0.0) + pr
    return out

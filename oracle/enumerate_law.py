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

"""Closed forms about one speculative round (test infrastructure).

Sources (page title, section):
  [P1] "Speculative Decoding" (atonlee.tistory.com/330), ch.4: expected tokens
       per round E = (1 - a^(g+1)) / (1 - a) for acceptance rate a and g drafts,
       its tables for a in 0.5..0.9, and the speedup E / (g*c + 1) with c the
       cost of one draft step relative to one target step.
  [P2] "Speculative Decoding으로 LLM 추론 속도 높이기", section "품질은 rejection
       sampling이 지킨다": the same E and speedup with a worked example.
  [P3] "Fast Inference from Transformers via Speculative Decoding" notes, method
       details, expected accepted length: alpha = E_{x~q}[min(1, p(x)/q(x))].
  [P4] "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가", section on the two numbers
       that set the gain: E with k drafts and the speedup E / (1 + k c).

Reading: the pages call E both "tokens per round" and (in [P3]) "expected
accepted count"; the other pages count the correction/bonus token, so E here
is the mean of (accepted + 1).
"""
from __future__ import annotations

import numpy as np


def expected_tokens(alpha: float, gamma: int) -> float:
    """Mean tokens emitted by one round: sum_{k=0..gamma} alpha^k."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def expected_tokens_upper_bound(alpha: float) -> float:
    """Limit of expected_tokens as gamma grows: 1 / (1 - alpha)."""
    return 1.0 / (1.0 - alpha)


def speedup(alpha: float, gamma: int, c: float) -> float:
    """Wall-clock gain of one round over target-only decoding: E / (gamma * c + 1)."""
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def acceptance_rate(p: np.ndarray, q: np.ndarray) -> float:
    """alpha = E_{x~q}[min(1, p(x)/q(x))] = sum_x min(p(x), q(x))."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    return float(np.minimum(p, q).sum())


def accepted_count_pmf(alphas) -> np.ndarray:
    """Law of the accepted count n for per-position acceptance rates alphas[0..g-1].

    P(n = k) = prod_{i<k} alpha_i * (1 - alpha_k) for k < g, and prod of all for k = g.
    """
    a = np.asarray(alphas, dtype=np.float64)
    g = a.shape[0]
    out = np.empty(g + 1)
    run = 1.0
    for k in range(g):
        out[k] = run * (1.0 - a[k])
        run *= a[k]
    out[g] = run
    return out

"""Draft-length controller (test infrastructure: the rule written as plain loops).

Source: "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가" (ailab.paldyn.com),
checklist item 2: do not fix k; after rejections in a row lower k (down to 1)
to cut draft cost, and raise it again when acceptances keep coming.  "Speculative
Decoding" (atonlee.tistory.com/330) ch.4 and the notes on "Fast Inference from
Transformers via Speculative Decoding" (gamma's influence) say why: the best
gamma depends on the acceptance rate.

Reading: a round with a rejection (n < g) counts toward a rejection streak, a
round with every draft accepted (n == g, g > 0) toward an acceptance streak; any
round breaks the other streak.  After `down_after` rejection rounds in a row
gamma drops by one (not below gamma_min = 1) and the streak restarts; after
`up_after` full-acceptance rounds in a row gamma grows by one (not above
gamma_max) and the streak restarts.  A round with g == 0 changes nothing.
"""
from __future__ import annotations


def step(gamma: int, rej_run: int, acc_run: int, g: int, n: int, gamma_min: int, gamma_max: int,
         down_after: int, up_after: int):
    """One round of one sequence: returns (gamma, rej_run, acc_run)."""
    if g <= 0:
        return gamma, rej_run, acc_run
    if n < g:
        rej_run, acc_run = rej_run + 1, 0
        if rej_run >= down_after:
            gamma, rej_run = max(gamma_min, gamma - 1), 0
    else:
        acc_run, rej_run = acc_run + 1, 0
        if acc_run >= up_after:
            gamma, acc_run = min(gamma_max, gamma + 1), 0
    return gamma, rej_run, acc_run

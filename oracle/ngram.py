"""Prompt-lookup (n-gram) proposer, written as plain loops (test infrastructure).

Sources: "Speculative Decoding" (atonlee.tistory.com/330), ch.5 (prompt lookup:
no model; find the current suffix earlier in the context and use the tokens
that followed it as the draft); "Speculative Decoding으로 LLM 추론 속도 높이기"
(donmain.dev), section on turning it on in vLLM (the prompt_lookup_max /
prompt_lookup_min settings); "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가"
(ailab.paldyn.com), the draft-methods table and the n-gram paragraph (copy what
follows the same recent tokens found earlier; cost about zero).

Readings (the pages fix none of these details):
  - match lengths are tried from max_n down to min_n, so a longer match wins;
  - among the occurrences of that length the most recent one wins;
  - an occurrence is any earlier start j < L - n (overlap with the suffix is
    allowed); it is followed by at least one token because j + n <= L - 1;
  - the proposal is the min(gamma, L - (j + n)) tokens after the occurrence;
  - no occurrence of any length in [min_n, max_n]: no proposal (0 drafts).
"""
from __future__ import annotations


def propose(context, min_n: int, max_n: int, gamma: int) -> list:
    ctx = [int(t) for t in context]
    L = len(ctx)
    for n in range(max_n, min_n - 1, -1):
        if n < 1 or n >= L:
            continue
        suffix = ctx[L - n:]
        for j in range(L - n - 1, -1, -1):  # most recent first
            if ctx[j:j + n] == suffix:
                return ctx[j + n:j + n + gamma]
    return []


def propose_batch(contexts, lengths, min_n: int, max_n: int, gamma: int):
    """contexts [B, Lmax] (rows padded beyond lengths[b]); returns (tokens [B, gamma]
    with -1 padding, num_draft [B])."""
    import numpy as np

    B = len(lengths)
    tokens = np.full((B, gamma), -1, np.int32)
    num = np.zeros(B, np.int32)
    for b in range(B):
        prop = propose(contexts[b][: lengths[b]], min_n, max_n, gamma)
        tokens[b, : len(prop)] = prop
        num[b] = len(prop)
    return tokens, num

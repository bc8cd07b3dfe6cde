"""Host-side draft-length controller for a batch of sequences.

"투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가" (ailab.paldyn.com), checklist
item 2: do not fix the draft length k; after rejections in a row lower it (down
to 1) to save draft cost, and raise it again while acceptances continue.
"Speculative Decoding" (atonlee.tistory.com/330) ch.4 explains why: the best
length depends on the acceptance rate, so implementations adjust it.

Rule (one round of one sequence, g drafts, n accepted):
  n < g  -> rejection streak + 1, acceptance streak reset; after `down_after`
            rejection rounds in a row gamma -= 1 (floor gamma_min) and the
            streak restarts;
  n == g -> acceptance streak + 1, rejection streak reset; after `up_after`
            full-acceptance rounds in a row gamma += 1 (cap gamma_max) and the
            streak restarts;
  g == 0 -> no change.
Vectorised over the batch with numpy; the outputs of spec_verify
(num_draft, out_num_accepted) feed update().
"""
from __future__ import annotations

import numpy as np


class GammaController:
    def __init__(self, batch: int, gamma_max: int, gamma_start: int | None = None, gamma_min: int = 1,
                 down_after: int = 2, up_after: int = 2):
        if not (1 <= gamma_min <= gamma_max):
            raise ValueError("need 1 <= gamma_min <= gamma_max")
        start = gamma_max if gamma_start is None else gamma_start
        self.gamma_min, self.gamma_max = gamma_min, gamma_max
        self.down_after, self.up_after = down_after, up_after
        self.gamma = np.full(batch, min(max(start, gamma_min), gamma_max), np.int32)
        self.rej_run = np.zeros(batch, np.int32)
        self.acc_run = np.zeros(batch, np.int32)

    def update(self, num_draft, num_accepted) -> np.ndarray:
        g = np.asarray(num_draft, np.int32)
        n = np.asarray(num_accepted, np.int32)
        active = g > 0
        rej = active & (n < g)
        acc = active & (n >= g)
        self.rej_run = np.where(rej, self.rej_run + 1, np.where(acc, 0, self.rej_run))
        self.acc_run = np.where(acc, self.acc_run + 1, np.where(rej, 0, self.acc_run))
        down = rej & (self.rej_run >= self.down_after)
        up = acc & (self.acc_run >= self.up_after)
        self.gamma = np.where(down, np.maximum(self.gamma_min, self.gamma - 1), self.gamma)
        self.gamma = np.where(up, np.minimum(self.gamma_max, self.gamma + 1), self.gamma).astype(np.int32)
        self.rej_run = np.where(down, 0, self.rej_run).astype(np.int32)
        self.acc_run = np.where(up, 0, self.acc_run).astype(np.int32)
        return self.gamma.copy()

"""Monte-Carlo checks of the GPU path against what the pages fix:

- the worked example (draft 0.4, target 0.1: accepted with probability 0.25,
  emitted with probability 0.1) -- "Speculative Decoding으로 LLM 추론 속도
  높이기", section "품질은 rejection sampling이 지킨다";
- the output law on tiny vocabularies against the brute-force enumeration
  (chi-square), i.e. the distribution-preservation theorem of "Speculative
  Decoding" (atonlee.tistory.com/330) ch.3;
- mean tokens per round against E = (1 - a^(g+1))/(1 - a) (same page, ch.4;
  "투기적 디코딩 — 초안 모델을 무엇으로 세울 것인가").
"""
import json
import os

import numpy as np
import pytest

from oracle import analytic, enumerate_law
from speculative_decoding_verification_45_gb300 import workloads
from tests import law_checks
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def run(sv, batch, kernel=0):
    import torch

    toks, num = sv.verify(**sv.to_device(batch), kernel=kernel)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), num.cpu().numpy()


@gpu
def test_worked_example_monte_carlo(sv):
    w = json.load(open(os.path.join(GOLD, "worked_numbers.json")))["accept_example"]
    p, q = workloads.worked_example_rows()
    N = 1_000_000
    batch = workloads.tiny_batch(p, q, N=N, seed=2024)
    toks, num = run(sv, batch)
    drafted = batch.tokens[:, 0] == 0
    acc = (num[drafted] == 1).mean()
    se = np.sqrt(w["accept_probability"] * (1 - w["accept_probability"]) / drafted.sum())
    assert abs(acc - w["accept_probability"]) < 5 * se, acc
    emitted_by_accept = ((num == 1) & (toks[:, 0] == 0)).mean()
    se2 = np.sqrt(w["output_mass"] * (1 - w["output_mass"]) / N)
    assert abs(emitted_by_accept - w["output_mass"]) < 5 * se2
    freq0 = (toks[:, 0] == 0).mean()
    assert abs(freq0 - w["p"]) < 5 * se2


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("V,gamma,zf,seed", [(3, 1, 0.0, 31), (4, 2, 0.0, 32), (4, 3, 0.25, 33), (6, 2, 0.0, 34)])
def test_output_law_chi_square(sv, V, gamma, zf, seed, kernel):
    rng = np.random.default_rng(seed)

    def one():
        x = rng.dirichlet(np.ones(V))
        if zf:
            m = rng.random(V) < zf
            m[rng.integers(V)] = False
            x[m] = 0.0
            x /= x.sum()
        return x

    p = np.array([one() for _ in range(gamma + 1)])
    q = np.array([one() for _ in range(gamma)])
    batch = workloads.tiny_batch(p, q, N=1_000_000, seed=seed)
    p_st = np.exp(batch.target[0].astype(np.float64))
    q_st = np.exp(batch.draft[0].astype(np.float64))
    law = enumerate_law.outcome_law(p_st / p_st.sum(1, keepdims=True), q_st / q_st.sum(1, keepdims=True))
    toks, num = run(sv, batch, kernel)
    stat, pval, bins = law_checks.chi_square_vs_law(law_checks.outcome_keys(toks, num), law)
    assert pval > 1e-3, (stat, pval, bins)


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("alpha,gamma", [(0.8, 4), (0.5, 2), (0.5, 7), (0.9, 7), (0.7, 10)])
def test_mean_tokens_per_round(sv, alpha, gamma, kernel):
    p, q = workloads.alpha_rows(alpha, gamma)
    batch = workloads.tiny_batch(p, q, N=1_000_000, seed=int(alpha * 100) + gamma)
    _, num = run(sv, batch, kernel)
    z = law_checks.mean_tokens_z(num, analytic.expected_tokens(alpha, gamma))
    assert abs(z) < 4.0, z


@gpu
def test_greedy_is_argmax_agreement(sv):
    """T = 0 on random rows: accepted prefix = longest prefix with draft == argmax, then argmax."""
    rng = np.random.default_rng(8)
    B, g, V = 2000, 5, 37
    t = np.round(rng.normal(size=(B, g + 1, V)) * 2) / 2
    am = np.array([[int(np.flatnonzero(r == r.max())[0]) for r in seq] for seq in t])
    tokens = np.where(rng.random((B, g)) < 0.8, am[:, :g], rng.integers(0, V, size=(B, g))).astype(np.int32)
    batch = workloads.Batch(t.astype(np.float32), np.full((B, g, V), np.nan, np.float32), tokens,
                            np.full(B, g, np.int32), rng.random((B, g + 1)).astype(np.float32),
                            np.zeros(B, np.float32), "f32", "greedy-random")
    toks, num = run(sv, batch)
    for b in range(B):
        n = 0
        while n < g and tokens[b, n] == am[b, n]:
            n += 1
        assert num[b] == n
        assert list(toks[b, :n]) == list(tokens[b, :n]) and toks[b, n] == am[b, n]
        assert np.all(toks[b, n + 1:] == -1)


@gpu
def test_counters_and_accept_hist(sv, oracle_mod):
    """The optional counters and the accepted-count histogram agree with the
    accepted counts the call returns, on a ragged, mixed-temperature batch with
    an invalid sequence (which adds nothing), for both kernels."""
    import torch

    batch = workloads.make_config(4, B=40, seed=17)
    batch.num_draft[0] = -1                      # invalid: no counts
    ref = oracle_mod.verify_batch(batch, diagnostics=False)
    cnt = torch.zeros(3, dtype=torch.int64, device="cuda")
    hist = torch.zeros(sv.MAX_GAMMA + 1, dtype=torch.int64, device="cuda")
    for kernel in (0, 3):
        cnt.zero_()
        hist.zero_()
        toks, num = sv.verify(**sv.to_device(batch), kernel=kernel, counters=cnt, accept_hist=hist)
        torch.cuda.synchronize()
        valid = ref.seq_status == 0
        n = num.cpu().numpy()
        c = cnt.cpu().numpy()
        assert c[0] == int(batch.num_draft[valid].sum()) and c[1] == int(n[valid].sum()) and c[2] == valid.sum()
        np.testing.assert_array_equal(hist.cpu().numpy(), np.bincount(n[valid], minlength=sv.MAX_GAMMA + 1))

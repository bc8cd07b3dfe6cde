"""Prompt-lookup proposals and point-mass verification on the GPU.

- spec_ngram_propose equals the plain-loop oracle (oracle.ngram) exactly;
- spec_verify with draft_logits = NULL (q_i is 1 at the drafted id: a
  deterministic proposer, "Speculative Decoding" ch.5) equals the float64
  oracle's point-mass mode, and its output law is p (chi-square against the
  brute-force law with one-hot q);
- the acceptance counters match the outputs;
- proposer then verifier, end to end, equals the oracle pipeline.
"""
import numpy as np
import pytest

from oracle import enumerate_law, ngram
from speculative_decoding_verification_45_gb300 import workloads
from tests import law_checks, parity
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu


def _propose(sv, ctx, lens, mn, mx, gmax):
    import torch

    t, n = sv.ngram_propose(torch.from_numpy(ctx).cuda(), torch.from_numpy(lens).cuda(), mn, mx, gmax)
    torch.cuda.synchronize()
    return t.cpu().numpy(), n.cpu().numpy()


@gpu
@pytest.mark.parametrize("L,vocab,mn,mx,gmax", [(64, 4, 1, 3, 4), (1000, 20, 2, 4, 5), (4096, 50, 1, 8, 7),
                                                (3000, 1000, 3, 3, 16), (7, 3, 1, 64, 2),
                                                (20000, 40, 1, 6, 5)])
def test_proposals_match_oracle(sv, L, vocab, mn, mx, gmax):
    ctx, lens = workloads.ngram_contexts(48, L, vocab, seed=L + vocab)
    lens[:3] = [0, 1, 2]
    got_t, got_n = _propose(sv, ctx, lens, mn, mx, gmax)
    exp_t, exp_n = ngram.propose_batch(ctx, lens, mn, mx, gmax)
    np.testing.assert_array_equal(got_n, exp_n)
    np.testing.assert_array_equal(got_t, exp_t)


def _point_batch(cfg, B, seed):
    """Target rows of a workload with drafts proposed by lookup in a random context."""
    batch = workloads.make_config(cfg, B=B, seed=seed)
    rng = np.random.default_rng(seed)
    ctx, lens = workloads.ngram_contexts(batch.B, 2048, batch.V, seed=seed)
    # most proposals of a random-vocabulary context are id-copies: make them in range
    toks, num = ngram.propose_batch(ctx, lens, 1, 4, batch.gmax)
    for b in range(batch.B):
        g = int(batch.num_draft[b])
        k = min(g, int(num[b]))
        batch.tokens[b] = -1
        batch.tokens[b, :k] = toks[b, :k]
        batch.num_draft[b] = k
        if rng.random() < 0.5 and k > 0:  # half the time propose the target argmax (likely accepted)
            rows = workloads.logits_as_f64(batch.target[b, :k], batch.dtype)
            batch.tokens[b, :k] = np.argmax(rows, axis=1)
    return batch


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_point_mass_verify_parity(sv, oracle_mod, cfg, kernel):
    import torch

    batch = _point_batch(cfg, 48, 70 + cfg)
    ref = oracle_mod.verify_batch(batch, point=True)
    dev = sv.to_device(batch)
    counters = torch.zeros(3, dtype=torch.int64, device="cuda")
    toks, num = sv.verify(dev["target_logits"], None, dev["draft_tokens"], dev["num_draft"], dev["uniforms"],
                          dev["temperature"], kernel=kernel, counters=counters)
    torch.cuda.synchronize()
    toks, num = toks.cpu().numpy(), num.cpu().numpy()
    rep = parity.compare(batch, toks, num, ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    c = counters.cpu().numpy()
    assert c[0] == int(batch.num_draft.sum()) and c[1] == int(num.sum()) and c[2] == batch.B


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_point_mass_law_chi_square(sv, kernel):
    import torch

    rng = np.random.default_rng(5)
    V, gamma = 5, 3
    p = np.array([rng.dirichlet(np.ones(V)) for _ in range(gamma + 1)])
    drafts = [1, 3, 0]
    q = np.zeros((gamma, V))
    q[np.arange(gamma), drafts] = 1.0
    batch = workloads.tiny_batch(p, q, N=1_000_000, seed=9)
    p_st = np.exp(batch.target[0].astype(np.float64))
    law = enumerate_law.outcome_law(p_st / p_st.sum(1, keepdims=True), q)
    dev = sv.to_device(batch)
    toks, num = sv.verify(dev["target_logits"], None, dev["draft_tokens"], dev["num_draft"], dev["uniforms"],
                          dev["temperature"], kernel=kernel)
    torch.cuda.synchronize()
    stat, pval, bins = law_checks.chi_square_vs_law(law_checks.outcome_keys(toks.cpu().numpy(),
                                                                            num.cpu().numpy()), law)
    assert pval > 1e-3, (stat, pval, bins)


@gpu
def test_point_mode_equals_one_hot_draft_rows(sv, oracle_mod):
    """The oracle's point mode equals explicit one-hot draft rows (q = 1 at x)."""
    batch = _point_batch(3, 16, 33)
    ref_point = oracle_mod.verify_batch(batch, point=True)
    onehot = np.full(batch.draft.shape, workloads.f64_to_bf16_bits(np.array([-np.inf]))[0], np.uint16)
    zero = workloads.f64_to_bf16_bits(np.array([0.0]))[0]
    for b in range(batch.B):
        for i in range(int(batch.num_draft[b])):
            onehot[b, i, batch.tokens[b, i]] = zero
    batch.draft = onehot
    ref_rows = oracle_mod.verify_batch(batch)
    np.testing.assert_array_equal(ref_point.out_tokens, ref_rows.out_tokens)


@gpu
def test_lookup_then_verify_pipeline(sv, oracle_mod):
    import torch

    B, gmax, V = 32, 6, 4096
    ctx, lens = workloads.ngram_contexts(B, 3000, 400, seed=12)
    toks_t, num_t = sv.ngram_propose(torch.from_numpy(ctx).cuda(), torch.from_numpy(lens).cuda(), 2, 5, gmax)
    rng = np.random.default_rng(1)
    tl = workloads.f64_to_bf16_bits(rng.normal(0, 3, size=(B, gmax + 1, V)))
    temp = np.where(np.arange(B) % 2 == 0, 0.0, 0.8).astype(np.float32)
    uni = rng.random((B, gmax + 1)).astype(np.float32)
    t_dev = torch.from_numpy(tl.view(np.int16)).view(torch.bfloat16).cuda()
    out, num = sv.verify(t_dev, None, toks_t, num_t, torch.from_numpy(uni).cuda(), torch.from_numpy(temp).cuda())
    torch.cuda.synchronize()
    exp_t, exp_n = ngram.propose_batch(ctx, lens, 2, 5, gmax)
    np.testing.assert_array_equal(toks_t.cpu().numpy(), exp_t)
    batch = workloads.Batch(tl, np.zeros((B, gmax, V), np.uint16), exp_t, exp_n, uni, temp, "bf16", "pipeline")
    ref = oracle_mod.verify_batch(batch, point=True)
    rep = parity.compare(batch, out.cpu().numpy(), num.cpu().numpy(), ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]

"""Candidate-tree verification on the GPU (spec_tree_verify) against the float64
tree oracle: parity on Medusa-style, random, star and chain trees (ragged node
counts, sampled and greedy sequences, aligned and unaligned rows, full-size
vocabularies), equality with the chain kernel's point-mass mode on chain trees,
the output law on a tiny tree, invalid trees and counters."""
import numpy as np
import pytest

from oracle import enumerate_law
from speculative_decoding_verification_45_gb300 import workloads
from tests import law_checks, parity

gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_45_gb300 as m

    m.build()
    return m


def run_tree(sv, tb, **kw):
    import torch

    dev = sv.tree_to_device(tb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    toks, num, path = sv.tree_verify(**dev, status=status, **kw)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), num.cpu().numpy(), path.cpu().numpy(), int(status.cpu()[0])


@gpu
@pytest.mark.parametrize("shape,B,N,V,dtype", [
    ("medusa", 24, 64, 32000, "bf16"), ("random", 24, 40, 4099, "bf16"), ("star", 16, 33, 1024, "f32"),
    ("chain", 24, 17, 5000, "f32"), ("medusa", 8, 64, 128256, "bf16"), ("random", 8, 96, 151936, "bf16")])
def test_tree_parity(sv, oracle_mod, shape, B, N, V, dtype):
    seed = (sum(map(ord, shape)) * 7919 + N * 31 + V) % 1000  # fixed per case (str hashes vary by process)
    tb = workloads.tree_batch(B, N, V, dtype=dtype, seed=seed, shape=shape)
    ref = oracle_mod.tree_verify_batch(tb)
    toks, num, path, st = run_tree(sv, tb)
    rep = parity.compare_tree(tb, toks, num, path, ref)
    assert rep.mismatches_far == 0, (str(rep), rep.far_detail[:3])
    assert st == 0


@gpu
@pytest.mark.parametrize("seed", range(24))
def test_tree_random_sweep(sv, oracle_mod, seed):
    """Trees of random shape, size, vocabulary, dtype and temperature mix, at a
    cluster size from 1 to 16 (or the automatic one), against the oracle."""
    rng = np.random.default_rng(5000 + seed)
    shape = ("chain", "star", "random", "medusa")[seed % 4]
    B = int(rng.integers(1, 25))
    N = int(rng.integers(1, 97))
    V = int(rng.choice([int(rng.integers(2, 200)), int(rng.integers(200, 9000)), 32000, 4099]))
    dtype = "bf16" if rng.random() < 0.6 else "f32"
    temps = tuple(float(t) for t in rng.choice([0.0, 0.3, 0.7, 1.0, 2.0], size=int(rng.integers(1, 4))))
    C = (0, 1, 2, 3, 4, 8, 16)[seed % 7]
    tb = workloads.tree_batch(B, N, V, dtype=dtype, seed=6000 + seed, shape=shape, temps=temps,
                              ragged=bool(rng.random() < 0.7), zipf=bool(rng.random() < 0.5))
    ref = oracle_mod.tree_verify_batch(tb)
    toks, num, path, st = run_tree(sv, tb, cluster_size=C)
    rep = parity.compare_tree(tb, toks, num, path, ref)
    assert rep.mismatches_far == 0, (shape, B, N, V, dtype, temps, C, str(rep), rep.far_detail[:3])
    assert st == int(np.bitwise_or.reduce(ref.seq_status))


@gpu
@pytest.mark.parametrize("C", [1, 2, 3, 4, 8, 16])
def test_tree_cluster_sizes_agree(sv, oracle_mod, C):
    tb = workloads.tree_batch(12, 48, 32000, dtype="bf16", seed=41, shape="random")
    ref = oracle_mod.tree_verify_batch(tb)
    toks, num, path, _ = run_tree(sv, tb, cluster_size=C)
    rep = parity.compare_tree(tb, toks, num, path, ref)
    assert rep.mismatches_far == 0, (C, str(rep), rep.far_detail[:3])


@gpu
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_tree_equals_point_mass_verify(sv, T):
    """A chain-shaped tree is spec_verify with point-mass drafts: identical ids."""
    import torch

    B, g, V = 64, 6, 32000
    tb = workloads.tree_batch(B, g + 1, V, dtype="bf16", seed=8, shape="chain", temps=(T,))
    toks, num, path, _ = run_tree(sv, tb)
    target = np.full((B, g + 1, V), workloads.BF16_POS_INF, np.uint16)
    tokens = np.full((B, g), -1, np.int32)
    uniforms = np.zeros((B, g + 1), np.float32)
    for b in range(B):
        n = int(tb.num_nodes[b])
        target[b, :n] = tb.target[b, :n]
        tokens[b, : n - 1] = tb.tokens[b, 1:n]
        uniforms[b, : n - 1] = tb.uniforms[b, 1:n]
        uniforms[b, g] = tb.uniforms[b, 0]
    tt = torch.from_numpy(target.view(np.int16)).view(torch.bfloat16).cuda()
    ct, cn = sv.verify(tt, None, torch.from_numpy(tokens).cuda(), torch.from_numpy(tb.num_nodes - 1).cuda(),
                       torch.from_numpy(uniforms).cuda(), torch.from_numpy(tb.temperature).cuda())
    torch.cuda.synchronize()
    ct, cn = ct.cpu().numpy(), cn.cpu().numpy()
    np.testing.assert_array_equal(num, cn)
    for b in range(B):
        n = int(cn[b])
        np.testing.assert_array_equal(toks[b, : n + 1], ct[b, : n + 1])
        np.testing.assert_array_equal(path[b, :n], np.arange(1, n + 1))


@gpu
def test_tree_output_law_chi_square(sv):
    rng = np.random.default_rng(5)
    V, N = 4, 7
    par = [-1, 0, 0, 0, 1, 1, 2]
    tok = [-1, 2, 0, 2, 1, 3, 0]
    p = rng.dirichlet(np.ones(V), size=N)
    tb = workloads.tree_tiny(p, par, tok, 200_000, seed=12)
    p_st = np.exp(tb.target[0].astype(np.float64))
    law = enumerate_law.tree_outcome_law(p_st / p_st.sum(1, keepdims=True), par, tok)
    toks, num, path, _ = run_tree(sv, tb)
    keys = law_checks.tree_outcome_keys(toks, num, path)
    stat, pval, bins = law_checks.chi_square_vs_law(keys, law)
    assert pval > 1e-3, (stat, pval, bins)


@gpu
def test_tree_invalid_and_counters(sv, oracle_mod):
    import torch

    tb = workloads.tree_batch(8, 16, 2048, dtype="f32", seed=3, shape="random", ragged=False)
    tb.parent[0, 5] = 7
    tb.tokens[1, 3] = 2048
    tb.num_nodes[2] = 0
    tb.temperature[3] = float("nan")
    tb.temperature[4] = 1.0
    tb.target[4, 0] = np.nan   # the root row of a sampled sequence: no finite normaliser
    ref = oracle_mod.tree_verify_batch(tb)
    counters = torch.zeros(3, dtype=torch.int64, device="cuda")
    toks, num, path, st = run_tree(sv, tb, counters=counters)
    rep = parity.compare_tree(tb, toks, num, path, ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    assert st == int(np.bitwise_or.reduce(ref.seq_status))
    valid = ref.seq_status == 0
    c = counters.cpu().numpy()
    assert c[0] == int((tb.num_nodes[valid] - 1).sum()) and c[1] == int(num[valid].sum()) and c[2] == valid.sum()


@gpu
def test_tree_empty_batch_and_argument_checks(sv):
    import ctypes

    import torch

    lib = sv._native.load()
    assert lib.spec_tree_verify(None, None, None, None, None, None, None, None, None, 0, 4, 16, 0, None, None,
                                None) == 0
    tb = workloads.tree_batch(2, 4, 16, dtype="f32", seed=1, shape="chain")
    dev = sv.tree_to_device(tb)
    with pytest.raises(sv.SpecVerifyError):
        sv.tree_verify(**dev, cluster_size=17)
    torch.cuda.synchronize()

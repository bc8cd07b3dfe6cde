"""spec_sample: one token per row from softmax(logits / T) (or argmax at T = 0),
the round with no drafts -- draft-side sampling of a proposer and target-only
decoding ("Fast Inference from Transformers via Speculative Decoding" notes,
method details step 1).  The oracle is the float64 round with gamma_max = 0."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu


def _as_round(logits_rows, uniforms, temps, dtype):
    B, V = logits_rows.shape[0], logits_rows.shape[-1]
    return workloads.Batch(logits_rows.reshape(B, 1, V).copy(), logits_rows[:, :0].reshape(B, 0, V).copy(),
                           np.zeros((B, 0), np.int32), np.zeros(B, np.int32),
                           np.asarray(uniforms, np.float32).reshape(B, 1), np.asarray(temps, np.float32), dtype,
                           "sample")


def _run(sv, batch, kernel=0):
    import torch

    dev = sv.to_device(batch)
    out = sv.sample(dev["target_logits"][:, 0].contiguous(), dev["uniforms"][:, 0].contiguous(),
                    dev["temperature"], kernel=kernel)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@gpu
@pytest.mark.parametrize("kernel", [0, 2, 3])
@pytest.mark.parametrize("cfg", [3, 5])
def test_sample_matches_oracle(sv, oracle_mod, cfg, kernel):
    big = workloads.make_config(cfg, B=64)
    rng = np.random.default_rng(cfg)
    batch = _as_round(big.target[:, 0], rng.random(big.B).astype(np.float32), big.temperature, big.dtype)
    ref = oracle_mod.verify_batch(batch)
    got = _run(sv, batch, kernel)
    out = np.stack([got, np.zeros_like(got)], 1)[:, :1]
    rep = parity.compare(batch, out, np.zeros(batch.B, np.int32), ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]


@gpu
@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_sample_every_cluster_size_matches_oracle(sv, oracle_mod, cluster):
    """1024 rows of 128256 ids (half greedy): one CTA per row re-sweeps the
    owner's slice; clusters of 2 to 8 keep the chunk sums of pass 1.  Each
    launch shape agrees with the float64 oracle everywhere except within the
    tolerance of a CDF boundary, where the fp32 normaliser's rounding (it
    depends on how the row is split) may move the pick by one id."""
    import torch

    big = workloads.make_config(5)
    rows = np.concatenate([big.target[:, 0]] * 4)
    rng = np.random.default_rng(101)
    temps = np.where(np.arange(rows.shape[0]) % 2 == 1, 1.0, 0.0).astype(np.float32)
    batch = _as_round(rows, rng.random(rows.shape[0]).astype(np.float32), temps, big.dtype)
    ref = oracle_mod.verify_batch(batch)
    dev = sv.to_device(batch)
    got = sv.sample(dev["target_logits"][:, 0].contiguous(), dev["uniforms"][:, 0].contiguous(),
                    dev["temperature"], cluster_size=cluster)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    out = np.stack([got, np.zeros_like(got)], 1)[:, :1]
    rep = parity.compare(batch, out, np.zeros(batch.B, np.int32), ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    print(f"C={cluster}: {rep}")


@gpu
def test_sample_law_chi_square(sv):
    import scipy.stats

    p = np.array([0.05, 0.25, 0.0, 0.4, 0.3])
    N = 1_000_000
    with np.errstate(divide="ignore"):
        row = np.log(p).astype(np.float32)
    rng = np.random.default_rng(11)
    batch = _as_round(np.broadcast_to(row, (N, 5)).copy(), rng.random(N).astype(np.float32), np.ones(N), "f32")
    got = _run(sv, batch)
    counts = np.bincount(got, minlength=5)
    assert counts[2] == 0  # zero-probability id never drawn
    keep = p > 0
    stat, pval = scipy.stats.chisquare(counts[keep], p[keep] * N)
    assert pval > 1e-3, (counts, pval)


@gpu
def test_sample_greedy_ties_and_invalid(sv):
    rows = np.array([[1, 3, 3, 2], [0, 0, 0, 0], [-np.inf, 5, 1, 5], [1, 2, 3, 4]], np.float32)
    temps = np.array([0, 0, 0, -1.0], np.float32)
    batch = _as_round(rows, np.full(4, 0.5, np.float32), temps, "f32")
    got = _run(sv, batch)
    assert list(got) == [1, 0, 1, -1]


@gpu
@pytest.mark.parametrize("seed", range(200, 212))
def test_sample_random_rows(sv, oracle_mod, seed):
    """spec_sample on the first rows of random batches (workloads.random_batch:
    tiny to 70000 ids, bf16 or float32, mixed and invalid temperatures) at a
    cluster size from 1 to 16 or the automatic one, against the oracle."""
    import torch

    src = workloads.random_batch(seed)
    rng = np.random.default_rng(seed)
    temps = src.temperature.copy()
    batch = _as_round(src.target[:, 0], rng.random(src.B).astype(np.float32), temps, src.dtype)
    ref = oracle_mod.verify_batch(batch)
    dev = sv.to_device(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sv.sample(dev["target_logits"][:, 0].contiguous(), dev["uniforms"][:, 0].contiguous(),
                    dev["temperature"], status=status, cluster_size=(0, 1, 2, 4, 8, 16)[seed % 6])
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    out = np.stack([got, np.zeros_like(got)], 1)[:, :1]
    rep = parity.compare(batch, out, np.zeros(batch.B, np.int32), ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    assert int(status.item()) == int(np.bitwise_or.reduce(ref.seq_status))


@gpu
@pytest.mark.parametrize("mix", ["greedy", "sampled", "scattered", "invalid"])
def test_sample_row_order_matches_oracle(sv, oracle_mod, mix):
    """768 rows of 128256 ids fill more than one wave of clusters, so rows are
    handed out by cost, sampled rows first (they also draw from the row): one
    bin (every row greedy or every row sampled), the two kinds scattered over
    the batch at random, and some rows with an invalid temperature.  Each row's
    token must not depend on the order in which clusters took the rows."""
    import torch

    big = workloads.make_config(5)
    rows = np.concatenate([big.target[:, 0]] * 3)
    B = rows.shape[0]
    rng = np.random.default_rng(102)
    temps = {"greedy": np.zeros(B), "sampled": np.ones(B),
             "scattered": (rng.random(B) < 0.3).astype(np.float64),
             "invalid": np.where(rng.random(B) < 0.1, -1.0, (rng.random(B) < 0.5).astype(np.float64))}[mix]
    batch = _as_round(rows, rng.random(B).astype(np.float32), temps.astype(np.float32), big.dtype)
    ref = oracle_mod.verify_batch(batch)
    dev = sv.to_device(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sv.sample(dev["target_logits"][:, 0].contiguous(), dev["uniforms"][:, 0].contiguous(),
                    dev["temperature"], status=status)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    out = np.stack([got, np.zeros_like(got)], 1)[:, :1]
    rep = parity.compare(batch, out, np.zeros(batch.B, np.int32), ref)
    assert rep.mismatches_far == 0, rep.far_detail[:3]
    assert int(status.item()) == int(np.bitwise_or.reduce(ref.seq_status))

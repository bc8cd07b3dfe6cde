"""Parity on 48 seeded random batches (workloads.random_batch): random shapes
(tiny to 70000 ids, odd sizes, gamma_max 0 to 9, ragged drafts), bf16 and
float32, mixed temperatures and planted data problems; each run on one of the
kernels (full sweep, register loads, early exit), a cluster size from 1 to 16
(or the automatic one) and, for some seeds, point-mass proposals.  Tokens and
counts must be the float64 oracle's outside the parity tolerance, the status
bits exactly its, and the diagnostics of valid sequences within the softmax
tolerance."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu

KERNELS = (0, 2, 3)
CLUSTERS = (0, 0, 1, 2, 3, 5, 8, 16)


@gpu
@pytest.mark.parametrize("seed", range(48))
def test_random_batch_matches_oracle(sv, oracle_mod, seed):
    import torch

    batch = workloads.random_batch(seed)
    kernel = KERNELS[seed % 3]
    cluster = CLUSTERS[(seed // 3) % len(CLUSTERS)]
    point = seed % 5 == 4
    ref = oracle_mod.verify_batch(batch, point=point)
    dev = sv.to_device(batch)
    if point:
        dev["draft_logits"] = None
    d = sv.verify_debug(**dev, kernel=kernel, cluster_size=cluster)
    torch.cuda.synchronize()
    d = {k: v.cpu().numpy() for k, v in d.items()}
    rep = parity.compare(batch, d["out_tokens"], d["out_num_accepted"], ref, gpu_status=d["seq_status"])
    assert rep.mismatches_far == 0, (workloads.describe(batch), kernel, cluster, point, rep.far_detail[:3])
    assert int(d["status"][0]) == int(np.bitwise_or.reduce(ref.seq_status))
    # diagnostics are defined for valid sequences (a sequence with a data
    # problem may carry partial ones); early exit reports the rows it read
    ok = ref.seq_status == 0
    need = {}
    if kernel == 3:  # the rows read, every one of them
        need = {k: v[ok] for k, v in parity.read_masks(batch, d["out_num_accepted"], ok).items()}
    parity.softmax_close(d["p_hat"][ok], ref.p_hat[ok], need=need.get("p_hat"))
    parity.softmax_close(d["logz_t"][ok], ref.logz_t[ok], atol=1e-5, need=need.get("logz_t"))
    if not point:
        parity.softmax_close(d["q_hat"][ok], ref.q_hat[ok], need=need.get("q_hat"))
        parity.softmax_close(d["logz_d"][ok], ref.logz_d[ok], atol=1e-5, need=need.get("logz_d"))

"""GPU parity with the float64 oracle on the five workloads (full sizes, the
launch shape the benchmark times) and their diagnostics (softmax values within
rel 1e-5)."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity

gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_45_gb300 as m

    m.build()
    return m


def run_debug(sv, batch, kernel=0):
    import torch

    dev = sv.to_device(batch)
    d = sv.verify_debug(**dev, kernel=kernel)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in d.items()}


def check_batch(sv, oracle_mod, batch, diagnostics=True, kernel=0):
    d = run_debug(sv, batch, kernel)
    ref = oracle_mod.verify_batch(batch)
    rep = parity.compare(batch, d["out_tokens"], d["out_num_accepted"], ref, gpu_status=d["seq_status"])
    assert rep.mismatches_far == 0, (str(rep), rep.far_detail[:5])
    if diagnostics:
        # early exit: diagnostics for the rows read, and every one of those
        need = parity.read_masks(batch, d["out_num_accepted"]) if kernel == 3 else {}
        parity.softmax_close(d["p_hat"], ref.p_hat, need=need.get("p_hat"))
        parity.softmax_close(d["q_hat"], ref.q_hat, need=need.get("q_hat"))
        parity.softmax_close(d["logz_t"], ref.logz_t, atol=1e-5, need=need.get("logz_t"))
        parity.softmax_close(d["logz_d"], ref.logz_d, atol=1e-5, need=need.get("logz_d"))
    assert int(d["status"][0]) == int(np.bitwise_or.reduce(ref.seq_status)) if batch.B else True
    return rep, d, ref


@gpu
@pytest.mark.parametrize("cfg,greedy", [(1, False), (2, False), (2, True), (3, False), (4, False), (5, False)])
def test_config_parity(sv, oracle_mod, cfg, greedy):
    batch = workloads.make_config(cfg, greedy=greedy)
    rep, d, ref = check_batch(sv, oracle_mod, batch)
    print(f"cfg{cfg}{'-greedy' if greedy else ''}: {rep}")


@gpu
@pytest.mark.parametrize("cfg,greedy", [(1, False), (2, False), (2, True), (3, False), (4, False), (5, False)])
def test_config_parity_early_exit(sv, oracle_mod, cfg, greedy):
    """The row-ordered early-exit kernel: same outputs as the oracle (and the full sweep)."""
    batch = workloads.make_config(cfg, greedy=greedy)
    rep, d, ref = check_batch(sv, oracle_mod, batch, kernel=3)
    # no row after the cut was read: diagnostics stop at position n
    for b in range(batch.B):
        if batch.temperature[b] > 0:
            n = int(d["out_num_accepted"][b])
            assert np.all(np.isnan(d["logz_t"][b, n + 1:]))
    print(f"early cfg{cfg}{'-greedy' if greedy else ''}: {rep}")


@gpu
@pytest.mark.parametrize("cfg,seed", [(3, 11), (3, 12), (4, 13), (5, 14), (1, 15), (2, 16)])
def test_config_parity_more_seeds(sv, oracle_mod, cfg, seed):
    batch = workloads.make_config(cfg, seed=seed)
    rep, _, _ = check_batch(sv, oracle_mod, batch, diagnostics=False)
    print(f"cfg{cfg} seed {seed}: {rep}")


@gpu
def test_resid_mass_matches_oracle(sv, oracle_mod):
    batch = workloads.make_config(3)
    d = run_debug(sv, batch)
    ref = oracle_mod.verify_batch(batch)
    same_n = d["out_num_accepted"] == ref.out_num_accepted
    np.testing.assert_allclose(d["resid_mass"][same_n], ref.resid_mass[same_n], rtol=1e-5, atol=1e-7)


@gpu
@pytest.mark.parametrize("kernel", [2, 3])
def test_cluster_sizes_and_kernels_agree(sv, oracle_mod, kernel):
    """Both kernels (full sweep, early exit) at every cluster size give the
    oracle's result: the split of rows over CTAs is invisible."""
    import torch

    batch = workloads.make_config(4, B=12)
    ref = oracle_mod.verify_batch(batch)
    dev = sv.to_device(batch)
    for C in (1, 2, 4, 8, 16):
        toks, num = sv.verify(**dev, cluster_size=C, kernel=kernel)
        torch.cuda.synchronize()
        rep = parity.compare(batch, toks.cpu().numpy(), num.cpu().numpy(), ref)
        assert rep.mismatches_far == 0, (C, str(rep), rep.far_detail[:3])


@gpu
@pytest.mark.parametrize("cfg", [3, 5])
def test_register_kernel_parity(sv, oracle_mod, cfg):
    """The full sweep requested explicitly on the aligned workloads."""
    import torch

    batch = workloads.make_config(cfg, B=64 if cfg == 5 else None)
    ref = oracle_mod.verify_batch(batch)
    toks, num = sv.verify(**sv.to_device(batch), kernel=2)
    torch.cuda.synchronize()
    rep = parity.compare(batch, toks.cpu().numpy(), num.cpu().numpy(), ref)
    assert rep.mismatches_far == 0, (str(rep), rep.far_detail[:3])


@gpu
def test_deterministic_and_stream(sv):
    import torch

    batch = workloads.make_config(3, B=8)
    dev = sv.to_device(batch)
    a = [t.clone() for t in sv.verify(**dev)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = sv.verify(**dev, stream=s)
    s.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@gpu
@pytest.mark.parametrize("dtype,V,Cs", [("bf16", 32000, (2, 3, 4, 8, 16)), ("f32", 4096, (1, 2, 4)), ("f32", 1024, (1, 2)),
                                        ("f32", 8192, (1, 2))])
def test_narrow_slice_variants(sv, oracle_mod, dtype, V, Cs):
    """Slices of at most 8 (small grids), 4, 2 or 1 chunks per thread and row
    select the variants that read several rows per round trip.  At every such cluster size the
    results and diagnostics stay the oracle's, for draft rows and for point-mass
    proposals, with sampled and greedy sequences and ragged draft counts."""
    import torch

    batch = workloads.edge_batch("mixed", V=V, gamma=5, B=24, seed=77, dtype=dtype)
    ref = oracle_mod.verify_batch(batch)
    ref_point = oracle_mod.verify_batch(batch, point=True)
    dev = sv.to_device(batch)
    for C in Cs:
        d = sv.verify_debug(**dev, cluster_size=C, kernel=2)
        torch.cuda.synchronize()
        d = {k: v.cpu().numpy() for k, v in d.items()}
        rep = parity.compare(batch, d["out_tokens"], d["out_num_accepted"], ref, gpu_status=d["seq_status"])
        assert rep.mismatches_far == 0, (C, str(rep), rep.far_detail[:3])
        parity.softmax_close(d["p_hat"], ref.p_hat)
        parity.softmax_close(d["q_hat"], ref.q_hat)
        parity.softmax_close(d["logz_t"], ref.logz_t, atol=1e-5)
        parity.softmax_close(d["logz_d"], ref.logz_d, atol=1e-5)
        toks, num = sv.verify(dev["target_logits"], None, dev["draft_tokens"], dev["num_draft"], dev["uniforms"],
                              dev["temperature"], cluster_size=C, kernel=2)
        torch.cuda.synchronize()
        rep = parity.compare(batch, toks.cpu().numpy(), num.cpu().numpy(), ref_point)
        assert rep.mismatches_far == 0, (C, "point", str(rep), rep.far_detail[:3])


def _as_f32(batch):
    """The same workload with float32 logits (the bf16 values, exactly)."""
    import dataclasses

    if batch.dtype == "f32":
        return batch
    t = workloads.logits_as_f64(batch.target, "bf16").astype(np.float32)
    d = workloads.logits_as_f64(batch.draft, "bf16").astype(np.float32)
    return dataclasses.replace(batch, target=t, draft=d, dtype="f32", name=batch.name + "-f32")


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_fp32_full_vocabulary(sv, oracle_mod, kernel):
    """float32 logits at V=128256 (32064 chunks of four values per row: several
    batches per thread, the L2 prefetch of the next batch) and at V=151936 with
    ragged draft counts."""
    for cfg, B in ((3, 12), (4, 12)):
        check_batch(sv, oracle_mod, _as_f32(workloads.make_config(cfg, B=B)), kernel=kernel)

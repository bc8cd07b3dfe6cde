"""Edge cases on the GPU, each compared with the float64 oracle: no drafts,
rejection at the first position, every draft accepted (bonus), greedy ties,
-inf logits, vocabularies that are not a multiple of the 16-byte chunk (scalar
load path), float32 logits, gamma_max = 0, B = 0, rows that must never be read,
and per-sequence data errors (status bits, -1 tokens, no fault)."""
import numpy as np
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity
from tests.test_gpu_parity import check_batch, run_debug, sv  # noqa: F401

gpu = pytest.mark.gpu


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("kind", ["zero_draft", "reject_first", "accept_all", "greedy_ties", "neg_inf", "mixed"])
@pytest.mark.parametrize("V,dtype", [(1023, "bf16"), (50257, "bf16"), (4096, "bf16"), (1023, "f32"),
                                     (32000, "f32")])
def test_edge_kinds(sv, oracle_mod, kind, V, dtype, kernel):
    batch = workloads.edge_batch(kind, V=V, gamma=4, B=12, dtype=dtype)
    rep, d, ref = check_batch(sv, oracle_mod, batch, kernel=kernel)
    if kind == "reject_first":
        assert np.all(d["out_num_accepted"] == 0)
    if kind == "accept_all":
        assert np.all(d["out_num_accepted"] == 4)
    if kind == "greedy_ties":
        assert rep.mismatches_near == 0


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_large_gamma_and_tiny_vocab(sv, oracle_mod, kernel):
    for V in (1, 2, 7, 9, 300):
        for dtype in ("bf16", "f32"):
            batch = workloads.edge_batch("mixed", V=V, gamma=16, B=9, dtype=dtype, seed=V)
            check_batch(sv, oracle_mod, batch, kernel=kernel)


@gpu
def test_gamma_max_zero(sv, oracle_mod):
    batch = workloads.edge_batch("zero_draft", V=777, gamma=0, B=5)
    check_batch(sv, oracle_mod, batch)


@gpu
def test_empty_batch_is_noop(sv):
    import torch

    z = torch.zeros
    toks, num = sv.verify(z((0, 3, 8), dtype=torch.bfloat16, device="cuda"),
                          z((0, 2, 8), dtype=torch.bfloat16, device="cuda"),
                          z((0, 2), dtype=torch.int32, device="cuda"), z((0,), dtype=torch.int32, device="cuda"),
                          z((0, 3), device="cuda"), z((0,), device="cuda"))
    assert toks.shape == (0, 3) and num.shape == (0,)


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_unread_rows_are_never_read(sv, oracle_mod, kernel):
    """NaN in padding rows, in draft rows of greedy sequences and in draft rows
    after... would change results if read; rows are poisoned with NaN here."""
    batch = workloads.make_config(4, B=15)
    nan = np.uint16(0x7FC0)
    for b in range(batch.B):
        g = batch.num_draft[b]
        batch.target[b, g + 1:] = nan
        batch.draft[b, g:] = nan
        if batch.temperature[b] == 0:
            batch.draft[b] = nan
        batch.uniforms[b, g:batch.gmax] = np.nan
    check_batch(sv, oracle_mod, batch, diagnostics=False, kernel=kernel)


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_data_errors_set_status(sv, oracle_mod, kernel):
    batch = workloads.edge_batch("mixed", V=2048, gamma=3, B=12, seed=3)
    batch.num_draft[:] = 3
    batch.tokens[batch.tokens < 0] = 5
    batch.temperature[:] = 1.0
    batch.tokens[1, 0] = 2048          # out of range
    batch.tokens[2, 2] = -7            # out of range
    batch.num_draft[3] = 4             # > gamma_max
    batch.num_draft[4] = -1
    batch.temperature[5] = -1.0
    batch.temperature[6] = np.nan
    batch.temperature[7] = np.inf
    batch.temperature[8] = 1e-40       # positive subnormal
    tbits = workloads.f64_to_bf16_bits(np.full(2048, -np.inf))
    batch.target[9, 0] = tbits         # row without a finite normaliser
    batch.target[10, 1] = workloads.f64_to_bf16_bits(np.full(2048, np.inf))
    batch.tokens[11, 2] = 3            # valid
    rep, d, ref = check_batch(sv, oracle_mod, batch, diagnostics=False, kernel=kernel)
    assert list(d["seq_status"][:9]) == [0, 1, 1, 4, 4, 2, 2, 2, 2]
    assert d["seq_status"][9] == 8
    assert int(d["status"][0]) == 1 | 2 | 4 | 8 | int(d["seq_status"][10])


@gpu
def test_misaligned_logits_take_scalar_path(sv, oracle_mod):
    """Logit tensors offset by one element (not 16-byte aligned) are accepted."""
    import torch

    batch = workloads.edge_batch("mixed", V=4096, gamma=3, B=6)
    dev = sv.to_device(batch)
    big_t = torch.empty(dev["target_logits"].numel() + 1, dtype=torch.bfloat16, device="cuda")
    big_d = torch.empty(dev["draft_logits"].numel() + 1, dtype=torch.bfloat16, device="cuda")
    t = big_t[1:].view_as(dev["target_logits"]).copy_(dev["target_logits"])
    dd = big_d[1:].view_as(dev["draft_logits"]).copy_(dev["draft_logits"])
    assert t.data_ptr() % 16 != 0
    toks, num = sv.verify(t, dd, dev["draft_tokens"], dev["num_draft"], dev["uniforms"], dev["temperature"])
    ref = oracle_mod.verify_batch(batch)
    rep = parity.compare(batch, toks.cpu().numpy(), num.cpu().numpy(), ref)
    assert rep.mismatches_far == 0, rep.far_detail


@pytest.fixture(scope="module")
def max_vocab_batch():
    return workloads.edge_batch("mixed", V=1 << 24, gamma=1, B=2, dtype="bf16", seed=24)


@gpu
@pytest.mark.parametrize("kernel", [0, 3])
def test_maximum_vocabulary(sv, oracle_mod, max_vocab_batch, kernel):
    """V = SPEC_MAX_VOCAB (2^24): slices far larger than the shared-memory chunk
    sums (pass 2 rescans its tiles from global memory)."""
    check_batch(sv, oracle_mod, max_vocab_batch, kernel=kernel)


@gpu
def test_large_batch_many_ctas(sv, oracle_mod):
    """70000 sequences (more than the longest-first ordering handles, and a grid
    of 70000 clusters) of a tiny vocabulary."""
    batch = workloads.edge_batch("mixed", V=64, gamma=2, B=70000, dtype="f32", seed=70)
    check_batch(sv, oracle_mod, batch, diagnostics=False)

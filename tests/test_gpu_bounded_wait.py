"""The kernels' waits are bounded: a wait on an mbarrier that nothing completes
gives up after its limit, reports SPEC_STATUS_TIMEOUT through the status word
and returns, and the context stays usable (no fault, no hang)."""
import time

import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests import parity
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu


@gpu
def test_a_wait_that_cannot_finish_gives_up(sv, oracle_mod):
    import torch

    t0 = time.perf_counter()
    bits = sv.selftest_bounded_wait()
    elapsed = time.perf_counter() - t0
    assert bits == sv.STATUS_TIMEOUT
    assert elapsed < 5.0, elapsed  # the limit is 2^18 tries or 0.2 s
    # the context still works: a round on the ring kernel (the waits' user) and
    # on the default kernel afterwards give the oracle's answer
    batch = workloads.make_config(3, B=8)
    ref = oracle_mod.verify_batch(batch)
    for kernel in (sv.KERNEL_RING, sv.KERNEL_AUTO):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        toks, num = sv.verify(**sv.to_device(batch), kernel=kernel, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        rep = parity.compare(batch, toks.cpu().numpy(), num.cpu().numpy(), ref)
        assert rep.mismatches_far == 0, rep.far_detail[:3]

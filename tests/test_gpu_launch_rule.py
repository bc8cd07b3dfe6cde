"""The automatic launch choice on the five workloads (spec_verify_launch_shape,
which the call itself follows): the kernel that measured faster on GB300 in the
benchmark's per-config table (full sweep 2, early exit 3) and the cluster size
of the automatic rules.  A change of the rules shows here first."""
import pytest

from speculative_decoding_verification_45_gb300 import workloads
from tests.test_gpu_parity import sv  # noqa: F401

gpu = pytest.mark.gpu

# config -> (kernel, cluster size) on a 152-SM GB300
EXPECTED = {1: (3, 2), 2: (2, 8), 3: (2, 8), 4: (3, 10), 5: (3, 4)}


@gpu
@pytest.mark.parametrize("cfg", sorted(EXPECTED))
def test_automatic_kernel_and_cluster(sv, cfg):
    import torch

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected shapes are those of a 152-SM GB300")
    b = workloads.make_config(cfg)
    C, ctas, threads, kernel = sv.launch_shape(b.B, b.gmax, b.V, b.dtype)
    assert (kernel, C) == EXPECTED[cfg]
    assert ctas == b.B * C and threads == 256


@gpu
def test_sampler_cluster_for_long_rows(sv):
    import torch

    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected shapes are those of a 152-SM GB300")
    C, ctas, _, kernel = sv.launch_shape(256, 0, 128256, "bf16")
    assert (C, ctas, kernel) == (4, 1024, 2)  # rows of >= 4096 chunks: at least 4 CTAs each
    C, _, _, _ = sv.launch_shape(64, 0, 32000, "bf16")
    assert C == 4  # 4000 chunks: the one-wave rule alone (largest power of two with B*C <= 2*SMs)
    assert sv.launch_shape(1, 4, 128256, "bf16")[0] == 16  # one sequence, long rows: up to 16 CTAs
    assert sv.launch_shape(1, 5, 32000, "bf16")[0] == 8  # shorter rows stop at 8

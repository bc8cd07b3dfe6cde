"""The Python binding's argument checks, which run on the host before any
call into the library (no GPU needed): dtype, shape, contiguity, and host
inputs that are not page-locked."""
import pytest
import torch

import speculative_decoding_verification_45_gb300 as sv

CUDA0 = torch.device("cuda", 0)


def test_host_input_must_be_page_locked():
    with pytest.raises(ValueError, match="page-locked"):
        sv._check_input(torch.zeros(2, 3), "x", torch.float32, (2, 3), CUDA0)


@pytest.mark.parametrize("tensor,dtype,shape,exc,msg", [
    (torch.zeros(2, 3), torch.float32, (3, 2), ValueError, "expected shape"),
    (torch.zeros(3, 2).t(), torch.float32, (2, 3), ValueError, "contiguous"),
    (torch.zeros(2, 3, dtype=torch.int32), torch.float32, (2, 3), TypeError, "expected torch.float32"),
])
def test_dtype_shape_and_layout_are_checked(tensor, dtype, shape, exc, msg):
    with pytest.raises(exc, match=msg):
        sv._check_input(tensor, "x", dtype, shape, CUDA0)


def test_logits_dtype_must_be_bf16_or_f32():
    with pytest.raises(TypeError, match="bfloat16 or float32"):
        sv._dtype_code(torch.zeros(4, dtype=torch.float16))
    assert sv._dtype_code(torch.zeros(4, dtype=torch.bfloat16)) == sv.SPEC_BF16
    assert sv._dtype_code(torch.zeros(4)) == sv.SPEC_F32


def test_target_logits_must_be_three_dimensional():
    with pytest.raises(ValueError, match="gamma_max"):
        sv.verify(torch.zeros(4, 8), None, None, None, None, None)


def test_counter_tensors_are_checked():
    with pytest.raises(ValueError, match="64-bit"):
        sv._counter_ptr(torch.zeros(3, dtype=torch.int32), 3, "counters")


def test_empty_host_input_needs_no_page_locking():
    # gamma_max = 0 gives [B, 0, V] draft logits: nothing to read, nothing to pin
    sv._check_input(torch.zeros(3, 0, 5), "draft_logits", torch.float32, (3, 0, 5), CUDA0)

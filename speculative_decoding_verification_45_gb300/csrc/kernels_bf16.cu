// kernels_bf16.cu -- the verification kernels for bfloat16 logits and draft distributions.
// One translation unit per variant family so that nvcc builds them in parallel.

#include "spec_verify_kernels.cuh"

const void *specv::kernel_bf16(int kind) { return kernel_for_t<__nv_bfloat16, false>(kind); }

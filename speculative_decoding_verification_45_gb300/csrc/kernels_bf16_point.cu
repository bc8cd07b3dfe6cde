// kernels_bf16_point.cu -- the verification kernels for bfloat16 logits and point-mass proposals (no draft rows).
// One translation unit per variant family so that nvcc builds them in parallel.

#include "spec_verify_kernels.cuh"

const void *specv::kernel_bf16_point(int kind) { return kernel_for_t<__nv_bfloat16, true>(kind); }

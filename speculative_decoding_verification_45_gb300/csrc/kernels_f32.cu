// kernels_f32.cu -- the verification kernels for float32 logits and draft distributions.
// One translation unit per variant family so that nvcc builds them in parallel.

#include "spec_verify_kernels.cuh"

const void *specv::kernel_f32(int kind) { return kernel_for_t<float, false>(kind); }

// kernels_f32_point.cu -- the verification kernels for float32 logits and point-mass proposals (no draft rows).
// One translation unit per variant family so that nvcc builds them in parallel.

#include "spec_verify_kernels.cuh"

const void *specv::kernel_f32_point(int kind) { return kernel_for_t<float, true>(kind); }

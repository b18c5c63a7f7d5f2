// SwiGLU product of the BitTransformer feed-forward (BitNet 深度拆解 §3.1:
// down(silu(gate(h)) * up(h))): a = silu(y_gate) * y_up with
// silu(z) = z * sigmoid(z) = z / (1 + exp(-z)), formed in fp32 from the two
// BitLinear outputs.  The streaming decode kernel applies silu_mul in its
// epilogue; swiglu_kernel applies the same function to two finished outputs
// (the shapes that kernel does not take), so both give the same bits.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace bitnet {

// yg / (1 + exp(-yg)) * yu, each operation rounded to fp32 (expf of the CUDA
// math library; for very negative yg the exp overflows and the quotient is -0).
__device__ __forceinline__ float silu_mul(float yg, float yu) {
  return __fmul_rn(__fdiv_rn(yg, __fadd_rn(1.0f, expf(-yg))), yu);
}

// out[i] = silu_mul(yg[i], yu[i]) for i < n (grid-stride).
__global__ void __launch_bounds__(256) swiglu_kernel(const float *__restrict__ yg, const float *__restrict__ yu,
                                                      float *__restrict__ out, int64_t n) {
  pdl_wait_prior_grid();  // yg / yu come from the kernels before (launched with PDL)
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = silu_mul(yg[i], yu[i]);
}

}  // namespace bitnet

// Ternary matmul with group-wise weight scales, any shape (BitNet 深度拆解
// §4.3: every group of G consecutive weights of a row has its own scale; G = K
// is a per-channel scale), for the shapes the streaming decode kernel does
// not take (more than two tokens, G not a power of two up to 2048, K not a
// multiple of 64, long rows, unaligned pointers):
//   y[m, n] = fl(F * fl(s_m / 127)),  F = sum over g of acc_g * scale[n, g]
// in fp32 (fused multiply-add per group, groups in order), where acc_g is the
// exact integer product of group g.  One warp per output; the lanes split a
// group's K range, their integer sums are combined with shuffles.
#pragma once

#include "common.cuh"

namespace bitnet {

constexpr int kGroupedWarps = 8;

__global__ void __launch_bounds__(kGroupedWarps * 32)
    grouped_generic_kernel(const int8_t *__restrict__ xq, const float *__restrict__ scale,
                           const uint8_t *__restrict__ packed, const float *__restrict__ w_scale, int64_t M,
                           int64_t N, int64_t K, int64_t G, float *__restrict__ y, int32_t *__restrict__ acc_g) {
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t ng = K / G;
  const int64_t stride = (int64_t)gridDim.x * kGroupedWarps;
  for (int64_t o = (int64_t)blockIdx.x * kGroupedWarps + (threadIdx.x >> 5); o < M * N; o += stride) {
    const int64_t m = o / N, n = o % N;
    const int8_t *x = xq + m * K;
    float F = 0.0f;
    for (int64_t g = 0; g < ng; ++g) {
      int a = 0;
      for (int64_t k = g * G + lane; k < (g + 1) * G; k += 32) {
        const int64_t i = n * K + k;
        const int code = (packed[i >> 2] >> (2 * (i & 3))) & 3;
        a += (code - 1) * (int)x[k];
      }
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) a += __shfl_xor_sync(0xffffffffu, a, s);
      if (acc_g && lane == 0) acc_g[o * ng + g] = a;
      F = __fmaf_rn((float)a, __ldg(w_scale + n * ng + g), F);
    }
    if (lane == 0) y[o] = __fmul_rn(F, __fdiv_rn(__ldg(scale + m), 127.0f));
  }
}

}  // namespace bitnet

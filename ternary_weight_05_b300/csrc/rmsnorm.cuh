// RMSNorm in front of the per-token absmax quantisation (the BitLinear input
// of BitNet 深度拆解 §3.1: the block normalises h = RMSNorm(x) before the
// gate/up projections, in fp32 per §6.5), then the quantisation of §2.2 on h.
//
// Per token: S = sum_k x_k^2 in fp64 (each square is exact in fp64), the
// mean square ms = fl32(S / K), r = fl(1 / fl(sqrt(fl(ms + eps)))), and
// h_k = fl(fl(x_k * r) * g_k) (h_k = fl(x_k * r) without a weight).  Every
// fp32 step is the single IEEE operation named; only the order of the fp64
// sum is the kernel's own (a tree over the CTA), so S is within
// (K - 1) * 2^-53 * S of any other fp64 summation order.
#pragma once

#include "common.cuh"
#include "quant_act.cuh"

namespace bitnet {

__device__ __forceinline__ double block_sum_f64_256(double v, double *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red may still be read from a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double r = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) r += red[w];
  return r;
}

// The token's normalisation factor r (and its mean square) from a row of K
// elements (16-byte aligned, K % 8 == 0), one CTA of 256 threads per token.
template <typename T>
__device__ __forceinline__ float rms_factor(const T *row, int64_t K, float eps, double *red, float *ms_out) {
  double s = 0.0;
  for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += 256 * 8) {
    float v[8];
    load8(row + k, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) s = fma((double)v[i], (double)v[i], s);  // x^2 exact in fp64: one rounding
  }
  const double S = block_sum_f64_256(s, red);
  const float ms = __double2float_rn(__ddiv_rn(S, (double)K));
  if (ms_out) *ms_out = ms;
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// h = fl(fl(x * r) * g) for 8 elements (g == nullptr: h = fl(x * r)).
__device__ __forceinline__ void rms_apply8(float (&v)[8], float r, const float *g, int64_t k) {
  if (g) {
    const float4 g0 = *reinterpret_cast<const float4 *>(g + k), g1 = *reinterpret_cast<const float4 *>(g + k + 4);
    const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), gg[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], r);
  }
}

// RMSNorm + absmax int8 quantisation, one CTA per token.  Outputs: x_q and
// the absmax scale of h; optionally h itself (fp32) and the mean square.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_quant_kernel(const T *__restrict__ x, int64_t K,
                                                            const float *__restrict__ g, float eps,
                                                            int8_t *__restrict__ xq, float *__restrict__ scale,
                                                            float *__restrict__ h_out, float *__restrict__ ms_out) {
  __shared__ double redd[8];
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int64_t m = blockIdx.x;
  const T *row = x + m * K;
  const float r = rms_factor(row, K, eps, redd, (ms_out && threadIdx.x == 0) ? ms_out + m : nullptr);
  float amax = 0.0f;
  for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += 256 * 8) {
    float v[8];
    load8(row + k, v);
    rms_apply8(v, r, g, k);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = block_max_256(amax, red);
  const float s = amax < 1e-8f ? 1e-8f : amax;
  if (threadIdx.x == 0) scale[m] = s;
  const float c = quant_factor(s);
  for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += 256 * 8) {
    float v[8];
    load8(row + k, v);
    rms_apply8(v, r, g, k);
    if (h_out) {
      float4 *hp = reinterpret_cast<float4 *>(h_out + m * K + k);
      hp[0] = make_float4(v[0], v[1], v[2], v[3]);
      hp[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    *reinterpret_cast<uint2 *>(xq + m * K + k) = quantize8(v, s, c);
  }
}

}  // namespace bitnet

// Per-token absmax activation quantisation to int8.
//
// BitNet 深度拆解 §2.2 (absmax_quantize, bits = 8): the scale of token m is
// s = max(max_k |x[m,k]|, 1e-8) and q = clamp(round(x / s * 127), -127, 127),
// with round-half-even.  Every operation is the single IEEE fp32 operation
// the formula names (division first, then the multiply by 127).
//
// One CTA per token row.  When the row fits in registers (R vectors of 8
// elements per thread) it is read from memory once: absmax, block reduction,
// then quantisation from the registers.  Longer rows take two passes (the
// second hits L1/L2).
#pragma once

#include "common.cuh"

namespace bitnet {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ int8_t quantize_one(float v, float s) {
  const float r = __fmul_rn(__fdiv_rn(v, s), 127.0f);
  int q = __float2int_rn(r);
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  return static_cast<int8_t>(q);
}

// The factor c = fl(127 / s) of quantize_fast.
__device__ __forceinline__ float quant_factor(float s) { return __fdiv_rn(127.0f, s); }

// quantize_one for E elements of a token whose scale s bounds them all
// (|v| <= s), with c = quant_factor(s), mostly without a division.
// t = fl(v * c) and the exact r = fl(fl(v / s) * 127) are each within
// 127 (2^-23 + 2^-48) of 127 v / s (two roundings of relative size <= 2^-24
// on a value of magnitude <= 127; where a step underflows, an absolute error
// below 2^-140 instead), so |t - r| < 2^-14.  When t is
// farther than 2^-14 from every half-integer, t and r lie strictly between
// the same two half-integers and round to the same integer (no tie, no
// clamp needed: |r| <= 127).  t is rounded by adding 1.5 * 2^23, which under
// round-to-nearest-even leaves the nearest integer in the low mantissa bits
// (|t| < 2^22).  Elements within 2^-14 of a half-integer, and non-finite
// ones (the comparison fails for NaN), take quantize_one.
template <int E>
__device__ __forceinline__ void quantize_fast(const float (&v)[E], float s, float c, int8_t (&q)[E]) {
  constexpr float kMagic = 12582912.0f;         // 1.5 * 2^23
  constexpr float kEdge = 0.5f - 0.00006103515625f;  // 0.5 - 2^-14
  unsigned slow = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float t = __fmul_rn(v[e], c);
    const float a = __fadd_rn(t, kMagic);
    q[e] = static_cast<int8_t>(__float_as_int(a) - __float_as_int(kMagic));
    const float d = fabsf(__fsub_rn(t, __fsub_rn(a, kMagic)));
    if (!(d < kEdge)) slow |= 1u << e;
  }
  if (slow) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (slow & (1u << e)) q[e] = quantize_one(v[e], s);
  }
}

__device__ __forceinline__ float block_max_256(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

// 8 consecutive elements as fp32 (exact widening for bf16).
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0];
  const float4 b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Packs the int8 codes of 8 elements of a token (scale s, c = quant_factor(s))
// into two words.
__device__ __forceinline__ uint2 quantize8(const float (&v)[8], float s, float c) {
  int8_t q[8];
  quantize_fast(v, s, c, q);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) lo |= (uint32_t)(uint8_t)q[i] << (8 * i);
#pragma unroll
  for (int i = 0; i < 4; ++i) hi |= (uint32_t)(uint8_t)q[4 + i] << (8 * i);
  return make_uint2(lo, hi);
}

// VEC: the row start of x is 16-byte aligned, K is a multiple of 8 and the
// x_q row start is 8-byte aligned, so 8 elements move per access.
// R > 0 (VEC only): K <= kQuantThreads * 8 * R, the row is held in registers.
template <typename T, bool VEC, int R>
__global__ void __launch_bounds__(kQuantThreads) quant_act_kernel(const T *__restrict__ x, int64_t K,
                                                                  int8_t *__restrict__ xq,
                                                                  float *__restrict__ scale) {
  __shared__ float red[kQuantThreads / 32];
  // Let the next kernel launch (and prefetch its weights) right away; it
  // still waits for this grid to complete before reading x_q.
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int64_t m = blockIdx.x;
  const T *row = x + m * K;
  int8_t *qrow = xq + m * K;

  float amax = 0.0f;
  if (VEC && R > 0) {
    float v[R > 0 ? R : 1][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t k = ((int64_t)threadIdx.x + (int64_t)r * kQuantThreads) * 8;
      if (k < K) {
        load8(row + k, v[r]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[r][i] = 0.0f;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[r][i]));
    amax = block_max_256(amax, red);
    const float s = amax < 1e-8f ? 1e-8f : amax;
    const float c = quant_factor(s);
    if (threadIdx.x == 0) scale[m] = s;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t k = ((int64_t)threadIdx.x + (int64_t)r * kQuantThreads) * 8;
      if (k < K) *reinterpret_cast<uint2 *>(qrow + k) = quantize8(v[r], s, c);
    }
    return;
  }
  if (VEC) {
    for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += kQuantThreads * 8) {
      float v[8];
      load8(row + k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) amax = fmaxf(amax, fabsf(load_as_f32(row, k)));
  }
  amax = block_max_256(amax, red);
  const float s = amax < 1e-8f ? 1e-8f : amax;
  if (threadIdx.x == 0) scale[m] = s;

  if (VEC) {
    const float c = quant_factor(s);
    for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += kQuantThreads * 8) {
      float v[8];
      load8(row + k, v);
      *reinterpret_cast<uint2 *>(qrow + k) = quantize8(v, s, c);
    }
  } else {
    for (int64_t k = threadIdx.x; k < K; k += kQuantThreads) qrow[k] = quantize_one(load_as_f32(row, k), s);
  }
}

}  // namespace bitnet

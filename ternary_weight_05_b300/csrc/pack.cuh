// Offline weight preparation: absmean ternarisation, 2-bit packing, beta.
//
// BitNet 深度拆解 §2.2 (absmean_quantize): gamma = 1 / (alpha * mean|W| + eps),
// W_t = clamp(round(gamma * W), -1, 1), beta = mean|W_t|; §3.3 (pack_ternary):
// code = W_t + 1 in {0,1,2}, four codes per byte, the first in the low bits.
//
// mean|W| is reduced in fp64 in a fixed order so that the result is one
// defined number: the flattened matrix is cut into 4096-element chunks, each
// chunk is summed left to right by one thread, and one thread adds the chunk
// sums left to right.  All later steps are per element.
//
// Kernels, in stream order:
//   pack_chunk_sums  -> per-chunk fp64 sums into the workspace
//   pack_finalize    -> mean, gamma (device scalars), zero the nnz counter
//   pack_codes       -> packed bytes + nonzero count
//   pack_beta        -> beta = nnz / n
#pragma once

#include "common.cuh"

namespace bitnet {

constexpr int64_t kAbsChunk = 4096;
constexpr int kPackThreads = 256;

struct PackScratch {
  unsigned long long nnz;  // nonzero count
  float gamma;
  float mean;
  // followed (at offset 256) by ceil(n / 4096) chunk sums (double)
};
constexpr size_t kPackScratchHeader = 256;

template <typename T>
__global__ void __launch_bounds__(kPackThreads) pack_chunk_sums_kernel(const T *__restrict__ w, int64_t n,
                                                                       double *__restrict__ sums) {
  pdl_wait_prior_grid();  // W may come from the previous kernel (launched with PDL)
  const int64_t c = (int64_t)blockIdx.x * kPackThreads + threadIdx.x;
  const int64_t c0 = c * kAbsChunk;
  if (c0 >= n) return;
  const int64_t c1 = c0 + kAbsChunk < n ? c0 + kAbsChunk : n;
  double part = 0.0;
  for (int64_t i = c0; i < c1; ++i) part = __dadd_rn(part, (double)fabsf(load_as_f32(w, i)));
  sums[c] = part;
}

__global__ void pack_finalize_kernel(const double *__restrict__ sums, int64_t nchunks, int64_t n, float alpha,
                                     float eps, PackScratch *scr, float *absmean_out) {
  pdl_wait_prior_grid();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double total = 0.0;
  for (int64_t c = 0; c < nchunks; ++c) total = __dadd_rn(total, sums[c]);
  const float mean = __double2float_rn(__ddiv_rn(total, (double)n));
  float t = __fmul_rn(alpha, mean);
  t = __fadd_rn(t, eps);
  scr->gamma = __fdiv_rn(1.0f, t);
  scr->mean = mean;
  scr->nnz = 0ull;
  if (absmean_out) *absmean_out = mean;
}

__device__ __forceinline__ uint32_t ternary_code(float gamma, float w) {
  int q = __float2int_rn(__fmul_rn(gamma, w));  // NaN -> 0, +-inf saturate
  q = q > 1 ? 1 : (q < -1 ? -1 : q);
  return static_cast<uint32_t>(q + 1);
}

// Each thread packs 16 consecutive weights into one 32-bit word (4 bytes).
// The tail (n % 16 weights) is packed byte by byte by the first threads.
// WORD_STORE: `packed` is 4-byte aligned, so each thread stores one word.
template <typename T, bool WORD_STORE>
__global__ void __launch_bounds__(kPackThreads) pack_codes_kernel(const T *__restrict__ w, int64_t n,
                                                                  uint8_t *__restrict__ packed, PackScratch *scr) {
  pdl_wait_prior_grid();
  const float gamma = scr->gamma;
  const int64_t nwords = n / 16;
  unsigned cnt = 0;
  const int64_t stride = (int64_t)gridDim.x * kPackThreads;
  for (int64_t j = (int64_t)blockIdx.x * kPackThreads + threadIdx.x; j < nwords; j += stride) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t code = ternary_code(gamma, load_as_f32(w, j * 16 + e));
      cnt += code != 1u;
      word |= code << (2 * e);
    }
    if (WORD_STORE) {
      reinterpret_cast<uint32_t *>(packed)[j] = word;
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) packed[4 * j + b] = static_cast<uint8_t>(word >> (8 * b));
    }
  }
  // tail bytes: weights [16*nwords, n), padded with code 0 (n % 4 == 0 here)
  const int64_t tail0 = nwords * 4, nbytes = (n + 3) / 4;
  const int64_t t = (int64_t)blockIdx.x * kPackThreads + threadIdx.x;
  if (t < nbytes - tail0) {
    const int64_t b = tail0 + t;
    uint32_t byte = 0;
    for (int s = 0; s < 4; ++s) {
      const int64_t i = 4 * b + s;
      if (i < n) {
        const uint32_t code = ternary_code(gamma, load_as_f32(w, i));
        cnt += code != 1u;
        byte |= code << (2 * s);
      }
    }
    packed[b] = static_cast<uint8_t>(byte);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0 && cnt) atomicAdd(&scr->nnz, (unsigned long long)cnt);
}

// Group-wise scales (BitNet 深度拆解 §4.3: groups of group_size weights, each
// with its own gamma and beta; one group per row is the per-channel scale):
// group g of row n is W[n, gG .. gG + G - 1].  One thread per group does what
// the four kernels above do for a whole matrix, in the same order: the fp64
// sum of |w| in 4096-element chunks left to right, mean, gamma, the codes of
// the group (G / 4 bytes, G % 4 == 0) and beta_g = nnz_g / G.
template <typename T>
__global__ void __launch_bounds__(kPackThreads) pack_grouped_kernel(const T *__restrict__ w, int64_t groups,
                                                                    int64_t G, float alpha, float eps,
                                                                    uint8_t *__restrict__ packed,
                                                                    float *__restrict__ w_scale,
                                                                    float *__restrict__ absmean) {
  pdl_wait_prior_grid();
  const int64_t gi = (int64_t)blockIdx.x * kPackThreads + threadIdx.x;
  if (gi >= groups) return;
  const T *wg = w + gi * G;  // groups are consecutive in the row-major matrix
  double total = 0.0;
  for (int64_t c0 = 0; c0 < G; c0 += kAbsChunk) {
    const int64_t c1 = c0 + kAbsChunk < G ? c0 + kAbsChunk : G;
    double part = 0.0;
    for (int64_t i = c0; i < c1; ++i) part = __dadd_rn(part, (double)fabsf(load_as_f32(wg, i)));
    total = __dadd_rn(total, part);
  }
  const float mean = __double2float_rn(__ddiv_rn(total, (double)G));
  const float gamma = __fdiv_rn(1.0f, __fadd_rn(__fmul_rn(alpha, mean), eps));
  uint8_t *pg = packed + gi * (G / 4);
  int64_t nnz = 0;
  for (int64_t b = 0; b < G / 4; ++b) {
    uint32_t byte = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t code = ternary_code(gamma, load_as_f32(wg, 4 * b + s));
      nnz += code != 1u;
      byte |= code << (2 * s);
    }
    pg[b] = static_cast<uint8_t>(byte);
  }
  w_scale[gi] = __double2float_rn(__ddiv_rn((double)nnz, (double)G));
  if (absmean) absmean[gi] = mean;
}

__global__ void pack_beta_kernel(const PackScratch *scr, int64_t n, float *beta) {
  pdl_wait_prior_grid();
  if (threadIdx.x == 0 && blockIdx.x == 0) *beta = __double2float_rn(__ddiv_rn((double)scr->nnz, (double)n));
}

}  // namespace bitnet

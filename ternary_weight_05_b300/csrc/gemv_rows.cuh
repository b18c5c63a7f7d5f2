// Decode GEMV for one or two tokens: row-range partition, dp4a arithmetic.
//
// Same operation as gemv.cuh (BitNet 深度拆解 §3.1 integer-domain product,
// §1 ternary products, §2.3 dequantisation), organised for the latency- and
// bandwidth-critical decode case:
//   * CTA c owns a contiguous range of weight rows (in units of 8 rows, so the
//     ranges differ by at most 8 rows) and the whole K range.  Every output is
//     finished inside one CTA: no workspace, no cross-CTA atomics.
//   * A dedicated producer warp streams the CTA's rows with 2D TMA in stages of
//     64 rows x 512 K (8 KB, 128-byte swizzle); a partial last row group is
//     fetched with 8-row boxes so rows of the next CTA are not read.  The ring
//     is as deep as shared memory allows (up to 24 stages, 192 KB in flight
//     per SM): HBM latency under load is long, and the small stages of a
//     partial row group must not throttle the stream.  The first stages are
//     requested before waiting on the previous kernel.
//   * 16 compute warps: warp w takes the 16-byte column chunk w & 7 of the
//     stage and the 32-row half w >> 3; lane = row.  All lanes of a warp read
//     the same activation words (broadcast), so activation traffic from shared
//     memory is a quarter of the weight traffic.
//   * Fused form (XT = float or bf16): the CTA reads the activations x
//     itself and quantises them in its prologue, absmax per token then
//     clamp(rint(x / s * 127)) with the same fp32 operations as
//     quant_act_kernel (BitNet 深度拆解 §2.2), so the result is identical;
//     one kernel per BitLinear instead of two.  CTA 0 also writes x_q and s
//     when asked.
//   * A packed 32-bit word holds 16 weights; masking it with 0x03030303 << 2s
//     keeps field s of each byte scaled by 4^s, and dp4a against the bytes
//     x[4b + s] of the matching 16-K group gives 4^s * sum code * x exactly.
//     The four partial sums are shifted back and the per-token sum of x is
//     subtracted once: sum (code - 1) * x.
#pragma once

#include "common.cuh"
#include "quant_act.cuh"

namespace bitnet {

constexpr int kRowsComputeWarps = 16;
constexpr int kRowsThreads = (kRowsComputeWarps + 1) * 32;
constexpr int kRowsGroup = 64;                     // rows per stage
constexpr int kRowsStageBytes = kRowsGroup * 128;  // 8 KB
#ifndef BITNET_ROWS_MAX_STAGES
#define BITNET_ROWS_MAX_STAGES 24
#endif
constexpr int kRowsMaxStages = BITNET_ROWS_MAX_STAGES;
constexpr int kRowsBar = 1;
constexpr int kRowsXBudget = 96 * 1024;  // activation words in shared memory

struct GemvRowsParams {
  const int8_t *xq;        // int8 activations (XT = int8_t)
  const void *x;           // bf16 / fp32 activations (fused forms)
  int8_t *xq_out;          // fused forms, optional: x_q written by CTA 0
  float *scale_out;        // fused forms, optional: per-token absmax written by CTA 0
  const float *scale;
  const float *w_scale;
  float *y;
  int32_t *acc;
  int64_t N, K;
  int M;
  int NKB;    // K-blocks of 512
  int units;  // ceil(N / 8)
  int xrow;   // bytes per token of the activation words (NKB * 512)
  int NS;     // ring stages (<= kRowsMaxStages)
};

struct GemvRowsSmem {
  int ring, xbuf, xsum, red, fscale, bars, bytes;
};

__host__ __device__ inline GemvRowsSmem gemv_rows_smem_layout(int M, int xrow, int ns) {
  GemvRowsSmem L;
  L.ring = 0;
  L.xbuf = ns * kRowsStageBytes;
  L.xsum = L.xbuf + M * xrow;
  L.red = L.xsum + 16;
  L.fscale = L.red + 8 * kRowsGroup * M * 4;
  L.bars = L.fscale + 16;
  L.bytes = L.bars + 2 * ns * 8 + 16;
  return L;
}

__device__ __forceinline__ void rows_sync() { named_barrier_sync(kRowsBar, kRowsComputeWarps * 32); }

// Activation words for 16-K group q (zero beyond K): word s holds bytes
// x_q[16q + 4b + s], b = 0..3; returns sum of the 16 values.
__device__ __forceinline__ int rows_pack_group(const int8_t (&v)[16], uint8_t *dst) {
  uint32_t wv[4];
  int sum = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    wv[s] = (uint32_t)(uint8_t)v[s] | ((uint32_t)(uint8_t)v[4 + s] << 8) | ((uint32_t)(uint8_t)v[8 + s] << 16) |
            ((uint32_t)(uint8_t)v[12 + s] << 24);
    sum += v[s] + v[4 + s] + v[8 + s] + v[12 + s];
  }
  *reinterpret_cast<uint4 *>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  return sum;
}

// 16 consecutive activations as fp32 (fused forms; K % 16 == 0, 16-byte
// aligned rows: checked on the host).
__device__ __forceinline__ void rows_load16(const float *p, float (&v)[16]) {
  float a[8], b[8];
  load8(p, a);
  load8(p + 8, b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = a[i];
    v[8 + i] = b[i];
  }
}
__device__ __forceinline__ void rows_load16(const __nv_bfloat16 *p, float (&v)[16]) {
  float a[8], b[8];
  load8(p, a);
  load8(p + 8, b);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = a[i];
    v[8 + i] = b[i];
  }
}

template <int MT, typename XT>
__global__ void __launch_bounds__(kRowsThreads, 1)
    gemv_rows_kernel(const __grid_constant__ CUtensorMap map64, const __grid_constant__ CUtensorMap map8,
                     const GemvRowsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NS = p.NS;
  const GemvRowsSmem L = gemv_rows_smem_layout(MT, p.xrow, NS);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *empty = full + NS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NS);
  int32_t *xsum = reinterpret_cast<int32_t *>(smem + L.xsum);
  int32_t *red = reinterpret_cast<int32_t *>(smem + L.red);
  float *fscale = reinterpret_cast<float *>(smem + L.fscale);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = (int)((long long)p.units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)p.units * (blockIdx.x + 1) / gridDim.x);
  const int64_t R0 = (int64_t)u0 * 8;
  const int64_t R1 = min((int64_t)u1 * 8, p.N);
  const int ngroups = (int)((R1 - R0 + kRowsGroup - 1) / kRowsGroup);
  const int count = ngroups * p.NKB;

  // Dependents may launch now: they wait for this grid's completion before
  // reading anything it writes, and their weight prefetch can overlap it.
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRowsComputeWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kRowsComputeWarps) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      prefetch_tensormap(&map64);
      prefetch_tensormap(&map8);
      const uint64_t policy = l2_policy_evict_first();
      int grp = 0, kb = 0, issued = 0;
      for (int it = 0; it < count; ++it) {
        const int slot = it % NS;
        if (it >= NS && !mbar_wait(&empty[slot], (uint32_t)(((it / NS) - 1) & 1))) {
          raise_device_error(kDevErrTimeout);
          *abort_flag = 1;
        }
        if (*abort_flag) break;  // the compute warps walk the rest without waiting
        const int64_t r = R0 + (int64_t)grp * kRowsGroup;
        const int valid = (int)min((int64_t)kRowsGroup, R1 - r);
        uint8_t *dst = smem + L.ring + slot * kRowsStageBytes;
        if (valid == kRowsGroup) {
          mbar_arrive_expect_tx(&full[slot], kRowsStageBytes);
          tma_load_2d(dst, &map64, &full[slot], kb * 128, (int)r, policy);
        } else {
          const int boxes = (valid + 7) / 8;
          mbar_arrive_expect_tx(&full[slot], boxes * 8 * 128);
          for (int b = 0; b < boxes; ++b)
            tma_load_2d(dst + b * 8 * 128, &map8, &full[slot], kb * 128, (int)(r + 8 * b), policy);
        }
        ++issued;
        if (++kb == p.NKB) {
          kb = 0;
          ++grp;
        }
      }
      if (*abort_flag) {  // leave no copy in flight
        for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
          mbar_wait(&full[j % NS], (uint32_t)((j / NS) & 1));
      }
    }
    return;
  }

  // ---------------------------------------------------------- compute warps --
  pdl_wait_prior_grid();
  const int tid = threadIdx.x;
  // activation words: for 16-K group q, word s holds bytes x[16q + 4b + s]
  if (tid < MT) xsum[tid] = 0;
  if constexpr (std::is_same<XT, int8_t>::value) {
    if (tid < MT) fscale[tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), __ldg(p.scale + tid)), 127.0f);
  }
  rows_sync();
  if constexpr (!std::is_same<XT, int8_t>::value) {
    // fused absmax quantisation of x [MT, K] (bf16 or fp32)
    const XT *x = static_cast<const XT *>(p.x);
    const int groups = (int)(p.K / 16);
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) amax[m] = 0.0f;
    for (int i = tid; i < MT * groups; i += kRowsComputeWarps * 32) {
      const int m = i / groups, q = i % groups;
      float v[16];
      rows_load16(x + (int64_t)m * p.K + (int64_t)q * 16, v);
      float a = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) a = fmaxf(a, fabsf(v[e]));
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
        if (mm == m) amax[mm] = fmaxf(amax[mm], a);
    }
    float *redf = reinterpret_cast<float *>(red);  // [16 warps][MT], free until the main loop
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = amax[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (lane == 0) redf[warp * MT + m] = a;
    }
    rows_sync();
    float s[MT], cq[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = redf[m];
      for (int w = 1; w < kRowsComputeWarps; ++w) a = fmaxf(a, redf[w * MT + m]);
      s[m] = a < 1e-8f ? 1e-8f : a;
      cq[m] = quant_factor(s[m]);
    }
    if (tid < MT) {
      fscale[tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), s[tid]), 127.0f);
      if (blockIdx.x == 0 && p.scale_out) p.scale_out[tid] = s[tid];
    }
    const int groups_all = p.NKB * 32;  // zero groups pad K to the 512-K blocks
    int part[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m] = 0;
    for (int i = tid; i < MT * groups_all; i += kRowsComputeWarps * 32) {
      const int m = i / groups_all, q = i % groups_all;
      int8_t v[16];
      if (q < groups) {
        float f[16];
        rows_load16(x + (int64_t)m * p.K + (int64_t)q * 16, f);
        float sm = s[0], cm = cq[0];
#pragma unroll
        for (int mm = 1; mm < MT; ++mm)
          if (mm == m) {
            sm = s[mm];
            cm = cq[mm];
          }
        quantize_fast(f, sm, cm, v);
        if (blockIdx.x == 0 && p.xq_out) {
          int4 u;
          memcpy(&u, v, 16);
          *reinterpret_cast<int4 *>(p.xq_out + (int64_t)m * p.K + (int64_t)q * 16) = u;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0;
      }
      const int sum = rows_pack_group(v, smem + L.xbuf + (size_t)m * p.xrow + (size_t)q * 16);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
        if (mm == m) part[mm] += sum;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v = part[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && v) atomicAdd(&xsum[m], v);
    }
  } else {
    const int groups = p.NKB * 32;
    const bool vec = ((p.K & 15) == 0) && ((reinterpret_cast<uintptr_t>(p.xq) & 15) == 0);
    int part[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m] = 0;
    for (int i = tid; i < MT * groups; i += kRowsComputeWarps * 32) {
      const int m = i / groups, q = i % groups;
      const int64_t k0 = (int64_t)q * 16;
      int8_t v[16];
      const int8_t *src = p.xq + (int64_t)m * p.K + k0;
      if (vec && k0 + 16 <= p.K) {
        const int4 u = *reinterpret_cast<const int4 *>(src);
        memcpy(v, &u, 16);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = (k0 + e < p.K) ? src[e] : (int8_t)0;
      }
      const int sum = rows_pack_group(v, smem + L.xbuf + (size_t)m * p.xrow + (size_t)q * 16);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
        if (mm == m) part[mm] += sum;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v = part[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && v) atomicAdd(&xsum[m], v);
    }
  }
  rows_sync();

  const int kgrp = warp & 7, half = warp >> 3;
  const int row = half * 32 + lane;  // row within the stage
  const uint32_t wofs = row * 128 + (((kgrp ^ (row & 7)) & 7) << 4);
  const uint32_t ring = smem_u32(smem + L.ring);
  const uint32_t xs = smem_u32(smem + L.xbuf);
  int acc[MT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int s = 0; s < 4; ++s) acc[m][s] = 0;

  int grp = 0, kb = 0;
  for (int it = 0; it < count; ++it) {
    const int slot = it % NS;
    if (!*abort_flag && !mbar_wait(&full[slot], (uint32_t)((it / NS) & 1))) {
      raise_device_error(kDevErrTimeout);
      *abort_flag = 1;
    }
    const uint4 w = lds_u128(ring + slot * kRowsStageBytes + wofs);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const uint32_t xaddr = xs + (kb * 32 + kgrp * 4) * 16;
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t f0 = wv[u] & 0x03030303u, f1 = wv[u] & 0x0C0C0C0Cu;
      const uint32_t f2 = wv[u] & 0x30303030u, f3 = wv[u] & 0xC0C0C0C0u;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const uint4 xv = lds_u128(xaddr + m * p.xrow + u * 16);
        acc[m][0] = dp4a_u8s8(f0, xv.x, acc[m][0]);
        acc[m][1] = dp4a_u8s8(f1, xv.y, acc[m][1]);
        acc[m][2] = dp4a_u8s8(f2, xv.z, acc[m][2]);
        acc[m][3] = dp4a_u8s8(f3, xv.w, acc[m][3]);
      }
    }
    if (++kb == p.NKB) {
      // row group done: reduce the 8 column chunks, write the outputs
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        red[(kgrp * kRowsGroup + row) * MT + m] =
            acc[m][0] + (acc[m][1] >> 2) + (acc[m][2] >> 4) + (acc[m][3] >> 6);
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[m][s] = 0;
      }
      rows_sync();
      const int64_t rbase = R0 + (int64_t)grp * kRowsGroup;
      if (tid < kRowsGroup * MT) {
        const int r = tid % kRowsGroup, m = tid / kRowsGroup;
        const int64_t n = rbase + r;
        if (n < R1) {
          int32_t v = -xsum[m];
#pragma unroll
          for (int c = 0; c < 8; ++c) v += red[(c * kRowsGroup + r) * MT + m];
          if (p.acc) p.acc[(int64_t)m * p.N + n] = v;
          p.y[(int64_t)m * p.N + n] = __fmul_rn((float)v, fscale[m]);
        }
      }
      rows_sync();
      kb = 0;
      ++grp;
    }
  }
}

}  // namespace bitnet

// Decode-path W2A8 ternary GEMV: y[m, n] = (sum_k (code[n,k]-1) * x_q[m,k])
//                                            * (w_scale * s_m / 127)
//
// BitNet 深度拆解 §3.1 (the integer-domain product of W_ternary and X_q), §1 (a
// ternary weight turns the product into +x, 0 or -x), §2.3 (dequantisation by
// the product of the two scales); the decode GEMV of the microsoft-bitnet
// review §03.3 is the GPU kernel of this step.
//
// Structure (persistent, one CTA per SM):
//   * Thread 0 streams the packed weights with 2D TMA into a ring of 16 KB
//     stages (128 rows x 128 bytes = 128 rows x 512 K, 128-byte swizzle) with
//     an L2 evict-first policy; the first stages are requested before waiting
//     on the previous kernel (programmatic dependent launch).
//   * All 16 warps compute on each stage from shared memory.
//   * The work is the sequence of (slice, row tile, K-block) stages; every CTA
//     takes an equal contiguous range of it ("stream-K"), so all SMs move the
//     same number of weight bytes.  A row tile finished inside one CTA is
//     written directly; a row tile split between CTAs (or K slices) is summed
//     with exact int32 atomics in the workspace, and the CTA that completes the
//     last K-block writes the output and clears the workspace entries.
//
// The integer sum is formed as sum_k code*x - sum_k x (code = w + 1 in
// {0,1,2}), so the unsigned 2-bit codes feed the arithmetic directly.
//
// M <= 2: dp4a path.  Masking a packed word with 0x03030303 << 2s keeps field
//   s of each byte, scaled by 4^s; dp4a with the matching activation bytes
//   gives 4^s * sum code*x exactly; the four partial sums are shifted back.
// M >= 3: tensor-core path (mma.sync m16n8k16, f16 in, f32 accumulate).  A
//   2-bit field masked in place inside a 16-bit lane is an fp16 subnormal
//   (or, for bits 10-11, the smallest normals) equal to code * 4^i * 2^-24;
//   the activation for that K position is stored as x_q * 4^-i in fp16 (exact),
//   so every product is code*x*2^-24 and every partial sum is an integer
//   multiple of 2^-24 below 2^22 * 2^-24: fp32 accumulation is exact and
//   D * 2^24 is the exact integer sum.
#pragma once

#include "common.cuh"

namespace bitnet {

constexpr int kGemvConsumerWarps = 16;
constexpr int kGemvConsumers = kGemvConsumerWarps * 32;
constexpr int kGemvThreads = kGemvConsumers;
constexpr int kStageRows = 128;
constexpr int kStageRowBytes = 128;
constexpr int kStageBytes = kStageRows * kStageRowBytes;
constexpr int kStageK = kStageRowBytes * 4;  // 512 weights per stage row
constexpr int kGemvStages = 4;
constexpr int kGemvXBudget = 120 * 1024;  // shared memory for the activation slice
constexpr int kGemvConsumerBar = 1;       // named barrier id for the consumer warps

struct GemvParams {
  const uint8_t *packed;  // used by the generic path (the TMA path reads a tensor map)
  const int8_t *xq;
  const float *scale;
  const float *w_scale;
  float *y;
  int32_t *acc;
  int32_t *ws_partial;  // [NR * 128][M]
  unsigned *ws_ticket;  // [NR]
  int64_t N, K;
  int M;
  int NR;    // row tiles of 128 rows
  int NKB;   // K-blocks of 512
  int KBS;   // K-blocks per slice
  int S;     // slices
  int xrow;  // bytes per token row of the shared activation slice
  long long total;  // NR * NKB stages
};

// Shared-memory carve-up (offsets from a 1024-byte-aligned base).
struct GemvSmem {
  int ring, xbuf, xsum, red, fscale, bars, flags, bytes;
};

__host__ __device__ inline GemvSmem gemv_smem_layout(int M, int KBS, int xrow) {
  GemvSmem L;
  L.ring = 0;
  L.xbuf = kGemvStages * kStageBytes;
  L.xsum = L.xbuf + ((M * xrow + 15) / 16) * 16;
  L.red = L.xsum + ((M * KBS * 4 + 15) / 16) * 16;
  L.fscale = L.red + kStageRows * M * 4;
  L.bars = L.fscale + ((M * 4 + 15) / 16) * 16;
  L.flags = L.bars + 2 * kGemvStages * 8;
  L.bytes = L.flags + 16;
  return L;
}

struct StageCoord {
  int s, r, kbl, nk;
};

__device__ __forceinline__ StageCoord stage_coord(const GemvParams &p, long long g) {
  StageCoord c;
  const long long per_slice = (long long)p.NR * p.KBS;
  long long s = g / per_slice;
  if (s > p.S - 1) s = p.S - 1;
  const long long rem = g - s * per_slice;
  const int nk = min(p.KBS, p.NKB - (int)s * p.KBS);
  c.s = (int)s;
  c.nk = nk;
  c.r = (int)(rem / nk);
  c.kbl = (int)(rem % nk);
  return c;
}

// Next stage in (slice, row tile, K-block) order without dividing.
__device__ __forceinline__ void stage_advance(const GemvParams &p, StageCoord &c) {
  if (++c.kbl == c.nk) {
    c.kbl = 0;
    if (++c.r == p.NR) {
      c.r = 0;
      ++c.s;
      c.nk = min(p.KBS, p.NKB - c.s * p.KBS);
    }
  }
}

__device__ __forceinline__ void consumer_sync() { named_barrier_sync(kGemvConsumerBar, kGemvConsumers); }

// Activation-slice loader.  For slice s, K range [s*KBS*512, ...), writes the
// per-path layout of x_q into shared memory and the per-K-block sums of x_q.
//   HMMA: for each 16-K group, 8 half2 = (x[i]*sc_i, x[8+i]*sc_i), i = 0..7,
//         sc = {1, 4^-1, 4^-2, 4^-3, 4^-4, 4^-5, 1, 4^-1}.
//   DP4A: for each 16-K group, 4 words; word s holds bytes x[4b+s], b = 0..3.
template <bool HMMA>
__device__ void gemv_load_x_slice(const GemvParams &p, int s, uint8_t *xbuf, int32_t *xsum) {
  const int tid = threadIdx.x;
  const int nk = min(p.KBS, p.NKB - s * p.KBS);
  for (int i = tid; i < p.M * p.KBS; i += kGemvConsumers) xsum[i] = 0;
  consumer_sync();
  const int groups = nk * 32;
  const int64_t kbase = (int64_t)s * p.KBS * kStageK;
  const bool vec = ((p.K & 15) == 0) && ((reinterpret_cast<uintptr_t>(p.xq) & 15) == 0);
  for (int i = tid; i < p.M * groups; i += kGemvConsumers) {
    const int m = i / groups, q = i % groups;
    const int64_t k0 = kbase + (int64_t)q * 16;
    int8_t v[16];
    const int8_t *src = p.xq + (int64_t)m * p.K + k0;
    if (vec && k0 + 16 <= p.K) {
      const int4 u = *reinterpret_cast<const int4 *>(src);
      memcpy(v, &u, 16);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = (k0 + e < p.K) ? src[e] : (int8_t)0;
    }
    int sum = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) sum += v[e];
    if (HMMA) {
      uint32_t h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sh = (j < 6) ? 2 * j : 2 * (j - 6);
        const float sc = 1.0f / (float)(1 << sh);  // exact power of two
        const __half lo = __float2half_rn((float)v[j] * sc);
        const __half hi = __float2half_rn((float)v[8 + j] * sc);
        h[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
      }
      // xrow is 8 mod 128 (bank-conflict-free 8-byte fragment loads), so
      // the group is written with 8-byte stores.
      uint2 *dst = reinterpret_cast<uint2 *>(xbuf + (size_t)m * p.xrow + (size_t)q * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[j] = make_uint2(h[2 * j], h[2 * j + 1]);
    } else {
      uint32_t wv[4];
#pragma unroll
      for (int sl = 0; sl < 4; ++sl)
        wv[sl] = (uint32_t)(uint8_t)v[sl] | ((uint32_t)(uint8_t)v[4 + sl] << 8) |
                 ((uint32_t)(uint8_t)v[8 + sl] << 16) | ((uint32_t)(uint8_t)v[12 + sl] << 24);
      *reinterpret_cast<uint4 *>(xbuf + (size_t)m * p.xrow + (size_t)q * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
    atomicAdd(&xsum[m * p.KBS + q / 32], sum);
  }
  consumer_sync();
}

__device__ __forceinline__ void gemv_store_output(const GemvParams &p, const float *fscale, int64_t n, int m,
                                                  int32_t v) {
  if (p.acc) p.acc[(int64_t)m * p.N + n] = v;
  p.y[(int64_t)m * p.N + n] = __fmul_rn((float)v, fscale[m]);
}

// End of a segment (K-blocks [kb0, kb1] of slice s for row tile r): red holds
// sum code*x per (row, token).  Subtract the segment's sum of x, then either
// write the outputs (the segment is the whole K range) or add into the
// workspace; the CTA completing the row tile writes it.
__device__ void gemv_finish_segment(const GemvParams &p, int r, int s, int kb0, int kb1, int nk, int32_t *red,
                                    const int32_t *xsum, const float *fscale, volatile int *flag) {
  consumer_sync();
  const int tid = threadIdx.x;
  const bool whole = (p.S == 1) && kb0 == 0 && kb1 == nk - 1;
  const int entries = kStageRows * p.M;
  for (int i = tid; i < entries; i += kGemvConsumers) {
    const int row = i % kStageRows, m = i / kStageRows;
    int32_t xs = 0;
    for (int kb = kb0; kb <= kb1; ++kb) xs += xsum[m * p.KBS + kb];
    const int32_t v = red[row * p.M + m] - xs;
    red[row * p.M + m] = 0;
    const int64_t n = (int64_t)r * kStageRows + row;
    if (n >= p.N) continue;
    if (whole)
      gemv_store_output(p, fscale, n, m, v);
    else
      atomicAdd(&p.ws_partial[n * p.M + m], v);
  }
  if (whole) {
    consumer_sync();
    return;
  }
  __threadfence();
  consumer_sync();
  if (tid == 0) {
    const unsigned cnt = (unsigned)(kb1 - kb0 + 1);
    const unsigned old = atomicAdd(&p.ws_ticket[r], cnt);
    *flag = (old + cnt == (unsigned)p.NKB) ? 1 : 0;
  }
  consumer_sync();
  if (*flag) {
    __threadfence();
    for (int i = tid; i < entries; i += kGemvConsumers) {
      const int row = i % kStageRows, m = i / kStageRows;
      const int64_t n = (int64_t)r * kStageRows + row;
      if (n >= p.N) continue;
      const int32_t v = atomicExch(&p.ws_partial[n * p.M + m], 0);
      gemv_store_output(p, fscale, n, m, v);
    }
    if (tid == 0) atomicExch(&p.ws_ticket[r], 0u);
  }
  consumer_sync();
}

// Sum of v[0..7] over the 32 lanes; lane l ends with the total of v[(l>>2)&7].
__device__ __forceinline__ int warp_transpose_sum8(const int (&v)[8]) {
  const int lane = threadIdx.x & 31;
  int u[4];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int send = b4 ? v[i] : v[i + 4];
    const int keep = b4 ? v[i + 4] : v[i];
    u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  int w2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int send = b3 ? u[i] : u[i + 2];
    const int keep = b3 ? u[i + 2] : u[i];
    w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  int t;
  {
    const int send = b2 ? w2[0] : w2[1];
    const int keep = b2 ? w2[1] : w2[0];
    t = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  return t;
}

// ------------------------------------------------------------------------
// Compute policies.  Each consumes one 128 x 128-byte stage from shared
// memory and keeps per-thread partial sums; flush() adds them into red.

// M <= 2.  Warp w owns rows 8w..8w+7 of the stage; lane l owns packed word l
// (K positions 16l..16l+15 of the stage).
template <int MT>
struct Dp4aPolicy {
  static constexpr bool kHmma = false;
  int acc[8][MT][4];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[r][m][s] = 0;
  }

  __device__ __forceinline__ void compute(uint32_t stage, uint32_t xs, int xrow, int kbl, int M) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t w[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int row = warp * 8 + r;  // row & 7 == r
      w[r] = lds_u32(stage + row * kStageRowBytes + ((((lane >> 2) ^ r) & 7) << 4) + ((lane & 3) << 2));
    }
    uint4 xv[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) xv[m] = lds_u128(xs + m * xrow + (kbl * 32 + lane) * 16);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t f0 = w[r] & 0x03030303u, f1 = w[r] & 0x0C0C0C0Cu;
      const uint32_t f2 = w[r] & 0x30303030u, f3 = w[r] & 0xC0C0C0C0u;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        acc[r][m][0] = dp4a_u8s8(f0, xv[m].x, acc[r][m][0]);
        acc[r][m][1] = dp4a_u8s8(f1, xv[m].y, acc[r][m][1]);
        acc[r][m][2] = dp4a_u8s8(f2, xv[m].z, acc[r][m][2]);
        acc[r][m][3] = dp4a_u8s8(f3, xv[m].w, acc[r][m][3]);
      }
    }
  }

  __device__ __forceinline__ void flush(int32_t *red, int M) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        v[r] = acc[r][m][0] + (acc[r][m][1] >> 2) + (acc[r][m][2] >> 4) + (acc[r][m][3] >> 6);
      const int t = warp_transpose_sum8(v);
      if ((lane & 3) == 0 && m < M) {
        const int row = warp * 8 + (lane >> 2);
        atomicAdd(&red[row * M + m], t);
      }
    }
    reset();
  }
};

// M >= 3.  (RB row blocks of 16) x (WB 16-byte chunks) per warp, RB*WB = 4;
// 8/WB warps along K, 8/RB warp groups along rows.
template <int NT, int RB, int WB>
struct HmmaPolicy {
  static constexpr bool kHmma = true;
  static_assert(RB * WB == 4, "tile shape");
  float d[RB][NT][4];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[rb][nt][e] = 0.0f;
  }

  __device__ __forceinline__ void compute(uint32_t stage, uint32_t xs, int xrow, int kbl, int M) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    constexpr int KG = 8 / WB;
    const int kgrp = warp % KG, rgrp = warp / KG;
    uint32_t w0[RB][WB], w1[RB][WB];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      const int r0 = (rgrp * RB + rb) * 16 + g;  // r0 & 7 == g, (r0 + 8) & 7 == g
#pragma unroll
      for (int u = 0; u < WB; ++u) {
        const int ch = kgrp * WB + u;
        const uint32_t off = (((ch ^ g) & 7) << 4) + (t << 2);
        w0[rb][u] = lds_u32(stage + r0 * kStageRowBytes + off);
        w1[rb][u] = lds_u32(stage + (r0 + 8) * kStageRowBytes + off);
      }
    }
#pragma unroll
    for (int u = 0; u < WB; ++u) {
      const int q = kbl * 32 + (kgrp * WB + u) * 4 + t;  // 16-K group within the slice
      uint32_t hs0[RB], hs1[RB];
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        hs0[rb] = w0[rb][u] >> 12;
        hs1[rb] = w1[rb][u] >> 12;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = nt * 8 + g;
          if (tok < M) {
            const uint2 bv = lds_u64(xs + tok * xrow + q * 32 + j * 8);
            b0[nt] = bv.x;
            b1[nt] = bv.y;
          } else {
            b0[nt] = 0u;
            b1[nt] = 0u;
          }
        }
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          uint32_t a0, a1, a2, a3;
          if (j < 3) {
            const uint32_t m0 = 0x00030003u << (4 * j), m1 = 0x00030003u << (4 * j + 2);
            a0 = w0[rb][u] & m0;
            a1 = w1[rb][u] & m0;
            a2 = w0[rb][u] & m1;
            a3 = w1[rb][u] & m1;
          } else {
            a0 = hs0[rb] & 0x00030003u;
            a1 = hs1[rb] & 0x00030003u;
            a2 = hs0[rb] & 0x000C000Cu;
            a3 = hs1[rb] & 0x000C000Cu;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(d[rb][nt], a0, a1, a2, a3, b0[nt], b1[nt]);
        }
      }
    }
  }

  __device__ __forceinline__ void flush(int32_t *red, int M) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    constexpr int KG = 8 / WB;
    const int rgrp = warp / KG;
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = (rgrp * RB + rb) * 16 + g + ((e >> 1) << 3);
          const int tok = nt * 8 + 2 * t + (e & 1);
          if (tok < M) atomicAdd(&red[row * M + tok], __float2int_rn(d[rb][nt][e] * 16777216.0f));
        }
    reset();
  }
};

template <class Policy>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap wmap, const GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GemvSmem L = gemv_smem_layout(p.M, p.KBS, p.xrow);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
  uint64_t *empty = full + kGemvStages;
  volatile int *flags = reinterpret_cast<volatile int *>(smem + L.flags);  // [0] abort, [1] last-CTA
  int32_t *red = reinterpret_cast<int32_t *>(smem + L.red);
  int32_t *xsum = reinterpret_cast<int32_t *>(smem + L.xsum);
  float *fscale = reinterpret_cast<float *>(smem + L.fscale);

  const long long g0 = p.total * blockIdx.x / gridDim.x;
  const long long g1 = p.total * (blockIdx.x + 1) / gridDim.x;
  const int count = (int)(g1 - g0);
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < kGemvStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGemvConsumerWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < kStageRows * p.M; i += kGemvThreads) red[i] = 0;
  __syncthreads();

  // Thread 0 is also the TMA producer.  The weights do not depend on the
  // previous kernel, so the first stages are requested before waiting on it.
  uint64_t policy = 0;
  StageCoord pc = stage_coord(p, g0);  // producer position
  auto issue = [&](int j) {
    const int slot = j % kGemvStages;
    mbar_arrive_expect_tx(&full[slot], kStageBytes);
    tma_load_2d(smem + L.ring + slot * kStageBytes, &wmap, &full[slot], (pc.s * p.KBS + pc.kbl) * kStageRowBytes,
                pc.r * kStageRows, policy);
    stage_advance(p, pc);
  };
  int issued = 0;
  if (tid == 0) {
    prefetch_tensormap(&wmap);
    policy = l2_policy_evict_first();
    for (; issued < count && issued < kGemvStages; ++issued) issue(issued);
  }
  pdl_wait_prior_grid();
  if (tid < p.M) fscale[tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), __ldg(p.scale + tid)), 127.0f);

  Policy pol;
  pol.reset();
  const uint32_t ring = smem_u32(smem + L.ring);
  const uint32_t xs = smem_u32(smem + L.xbuf);
  int cur_s = -1, cur_r = -1, seg_kb0 = 0;
  StageCoord c = stage_coord(p, g0);
  for (int it = 0; it < count; ++it, stage_advance(p, c)) {
    if (c.s != cur_s) {
      gemv_load_x_slice<Policy::kHmma>(p, c.s, smem + L.xbuf, xsum);
      cur_s = c.s;
    }
    if (c.r != cur_r) {
      cur_r = c.r;
      seg_kb0 = c.kbl;
    }
    const int slot = it % kGemvStages;
    // After a timeout every thread keeps walking the same stages without
    // waiting, so all warps reach the same named barriers; the results are
    // then meaningless and the device error word says so.
    if (!flags[0] && !mbar_wait(&full[slot], (uint32_t)((it / kGemvStages) & 1))) {
      raise_device_error(kDevErrTimeout);
      flags[0] = 1;
    }
    pol.compute(ring + slot * kStageBytes, xs, p.xrow, c.kbl, p.M);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (tid == 0 && issued < count && !flags[0]) {
      // refill this slot once every warp has released stage `it`
      if (mbar_wait(&empty[slot], (uint32_t)((it / kGemvStages) & 1))) {
        issue(issued);
        ++issued;
      } else {
        raise_device_error(kDevErrTimeout);
        flags[0] = 1;
      }
    }
    if (c.kbl == c.nk - 1 || it == count - 1) {
      pol.flush(red, p.M);
      gemv_finish_segment(p, c.r, c.s, seg_kb0, c.kbl, c.nk, red, xsum, fscale, flags + 1);
      cur_r = -1;
    }
  }
  // Leave no bulk copy in flight (only possible after a timeout).
  if (tid == 0 && flags[0]) {
    for (int j = (issued > kGemvStages ? issued - kGemvStages : 0); j < issued; ++j)
      mbar_wait(&full[j % kGemvStages], (uint32_t)((j / kGemvStages) & 1));
  }
}

// ------------------------------------------------------------------------
// Generic path for shapes or pointers the TMA kernel does not take (K not a
// multiple of 64, K < 512, unaligned packed rows).  One warp per (row, token);
// lanes stride over the row's bytes.
__global__ void gemv_generic_kernel(const GemvParams p) {
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const uint8_t *packed = p.packed;
  const int lane = threadIdx.x & 31;
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int64_t kbytes = p.K / 4;
  for (long long item = wid; item < (long long)p.N * p.M; item += nwarps) {
    const int64_t n = item % p.N;
    const int m = (int)(item / p.N);
    const uint8_t *row = packed + n * kbytes;
    const int8_t *x = p.xq + (int64_t)m * p.K;
    int sum = 0;
    for (int64_t b = lane; b < kbytes; b += 32) {
      const unsigned byte = row[b];
#pragma unroll
      for (int s = 0; s < 4; ++s) sum += ((int)((byte >> (2 * s)) & 3u) - 1) * (int)x[4 * b + s];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const float f = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), __ldg(p.scale + m)), 127.0f);
      if (p.acc) p.acc[(int64_t)m * p.N + n] = sum;
      p.y[(int64_t)m * p.N + n] = __fmul_rn((float)sum, f);
    }
  }
}

}  // namespace bitnet

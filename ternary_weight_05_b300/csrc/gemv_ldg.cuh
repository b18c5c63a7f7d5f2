// Decode GEMV for one or two tokens streamed with plain coalesced loads.
//
// Same operation as the other GEMV kernels (BitNet 深度拆解 §3.1 integer-
// domain product, §1 ternary products, §2.3 dequantisation).  This is the
// decode kernel for rows of up to 8192 (one token) or 4096 (two tokens)
// weights, organised so that nothing serialises the weight stream:
//   * Every warp owns a contiguous range of whole rows, i.e. a contiguous
//     byte range of the packed matrix, and streams it through a private ring
//     of two 8 KB shared-memory stages with 1D bulk copies (cp.async.bulk):
//     up to 192 KB in flight per SM, no coupling between warps, no barrier
//     but the warp's own stage barriers.  The first stages are requested
//     before waiting on the previous kernel, since the weights do not depend
//     on it.  Lane l reads the 16-byte chunks l, l+32, ... of each row from
//     the stage (consecutive lanes, consecutive addresses: conflict-free).
//   * Because a lane always sees the same K chunks, its activation words live
//     in registers for the whole kernel: for 16-K group q, word s holds bytes
//     x_q[16q + 4b + s], b = 0..3, so masking a packed word with
//     0x03030303 << 2s and dp4a against word s gives 4^s * sum code * x
//     (2 integer operations per packed byte per token).
//   * A row's 32 lane sums are combined with warp shuffles; lane 0 subtracts
//     the token's sum of x_q and applies the fused dequantisation.
//   * Fused form (XT = float / bf16): the CTA quantises x itself in its
//     prologue (absmax, then clamp(rint(x / s * 127)), the operations of
//     quant_act_kernel), so one kernel runs the whole BitLinear.
#pragma once

#include "common.cuh"
#include "gemv_rows.cuh"
#include "quant_act.cuh"

namespace bitnet {

constexpr int kLdgWarps = 12;
constexpr int kLdgThreads = kLdgWarps * 32;
constexpr int kLdgStageBytes = 8192;  // per warp stage: whole rows, at most 8 KB
constexpr int kLdgStages = 2;         // stages per warp

struct GemvLdgParams {
  const uint8_t *packed;
  const int8_t *xq;   // int8 activations (XT = int8_t)
  const void *x;      // bf16 / fp32 activations (fused forms)
  int8_t *xq_out;     // fused forms, optional (CTA 0)
  float *scale_out;   // fused forms, optional (CTA 0)
  const float *scale;
  const float *w_scale;
  float *y;
  int32_t *acc;
  int64_t N, K;
  int M;
  int C;   // 16-byte chunks per packed row (K / 64)
  int SR;  // rows per stage (SR * K / 4 <= kLdgStageBytes)
};

// 1D bulk copy global -> shared, completing on `bar` (both addresses and the
// size multiples of 16 bytes), L2 evict-first: the weights are read once.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Shared memory: per-warp stage rings, activation words [MT][C * 64 bytes],
// per-token sums and output scales, the fused prologue's reduction scratch,
// then the stage barriers.
struct GemvLdgSmem {
  int ring, xw, xsum, fscale, redf, bars, bytes;
};
__host__ __device__ inline GemvLdgSmem gemv_ldg_smem_layout(int MT, int C) {
  GemvLdgSmem L;
  L.ring = 0;
  L.xw = kLdgWarps * kLdgStages * kLdgStageBytes;
  L.xsum = L.xw + MT * C * 64;
  L.fscale = L.xsum + 32;
  L.redf = L.fscale + 32;
  L.bars = L.redf + kLdgWarps * MT * 4 + 16;
  L.bytes = L.bars + kLdgWarps * kLdgStages * 8;
  return L;
}

template <int MT, int J, typename XT>
__global__ void __launch_bounds__(kLdgThreads, 1) gemv_ldg_kernel(const GemvLdgParams p) {
  extern __shared__ __align__(128) uint8_t lsm[];
  const GemvLdgSmem L = gemv_ldg_smem_layout(MT, p.C);
  uint8_t *xw = lsm + L.xw;                                     // [MT][C*64]
  int32_t *xsum = reinterpret_cast<int32_t *>(lsm + L.xsum);    // [MT]
  float *fscale = reinterpret_cast<float *>(lsm + L.fscale);    // [MT]
  float *redf = reinterpret_cast<float *>(lsm + L.redf);        // [warps][MT]
  uint64_t *bars = reinterpret_cast<uint64_t *>(lsm + L.bars);  // [warps][stages]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const long long gw = (long long)blockIdx.x * kLdgWarps + warp;
  const long long nw = (long long)gridDim.x * kLdgWarps;
  const int64_t r0 = (int64_t)(p.N * gw / nw), r1 = (int64_t)(p.N * (gw + 1) / nw);
  const int64_t rowb = p.K / 4;
  const int nst = (int)((r1 - r0 + p.SR - 1) / p.SR);  // this warp's stages
  uint8_t *ring = lsm + L.ring + (size_t)warp * kLdgStages * kLdgStageBytes;
  uint64_t *wbar = bars + warp * kLdgStages;
  pdl_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < kLdgWarps * kLdgStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The weights do not depend on the previous kernel: request the first
  // stages right away.
  uint64_t policy = 0;
  int issued = 0;  // stages requested (lane 0)
  auto issue = [&](int st) {
    ++issued;
    const int64_t ra = r0 + (int64_t)st * p.SR;
    const int64_t rbn = min(ra + p.SR, r1);
    const uint32_t bytes = (uint32_t)((rbn - ra) * rowb);
    uint64_t *bar = &wbar[st % kLdgStages];
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(ring + (st % kLdgStages) * kLdgStageBytes, p.packed + ra * rowb, bytes, bar, policy);
  };
  if (lane == 0) {
    policy = l2_policy_evict_first();
    for (int st = 0; st < nst && st < kLdgStages; ++st) issue(st);
  }

  pdl_wait_prior_grid();
  // ---------------------------------------------- activation words (smem) --
  if (tid < MT) xsum[tid] = 0;
  if constexpr (std::is_same<XT, int8_t>::value) {
    if (tid < MT) fscale[tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), __ldg(p.scale + tid)), 127.0f);
  }
  __syncthreads();
  const int groups = p.C * 4;  // 16-K groups per token
  {
    float s[MT];
    if constexpr (!std::is_same<XT, int8_t>::value) {
      const XT *x = static_cast<const XT *>(p.x);
      float amax[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) amax[m] = 0.0f;
      for (int i = tid; i < MT * groups; i += kLdgThreads) {
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
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a = amax[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0) redf[warp * MT + m] = a;
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a = redf[m];
        for (int ww = 1; ww < kLdgWarps; ++ww) a = fmaxf(a, redf[ww * MT + m]);
        s[m] = a < 1e-8f ? 1e-8f : a;
      }
      if (tid < MT) {
        fscale[tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale), s[tid]), 127.0f);
        if (blockIdx.x == 0 && p.scale_out) p.scale_out[tid] = s[tid];
      }
    }
    int part[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m] = 0;
    for (int i = tid; i < MT * groups; i += kLdgThreads) {
      const int m = i / groups, q = i % groups;
      int8_t v[16];
      if constexpr (std::is_same<XT, int8_t>::value) {
        const int4 u = *reinterpret_cast<const int4 *>(p.xq + (int64_t)m * p.K + (int64_t)q * 16);
        memcpy(v, &u, 16);
      } else {
        float f[16];
        rows_load16(static_cast<const XT *>(p.x) + (int64_t)m * p.K + (int64_t)q * 16, f);
        float sm = s[0];
#pragma unroll
        for (int mm = 1; mm < MT; ++mm)
          if (mm == m) sm = s[mm];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = quantize_one(f[e], sm);
        if (blockIdx.x == 0 && p.xq_out) {
          int4 u;
          memcpy(&u, v, 16);
          *reinterpret_cast<int4 *>(p.xq_out + (int64_t)m * p.K + (int64_t)q * 16) = u;
        }
      }
      const int sum = rows_pack_group(v, xw + (size_t)m * p.C * 64 + (size_t)q * 16);
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
  __syncthreads();

  // this lane's activation words, for chunks lane + 32 j
  uint32_t xr[MT][J][16];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lane + 32 * j;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c < p.C) v = *reinterpret_cast<const uint4 *>(xw + (size_t)m * p.C * 64 + (size_t)c * 64 + g * 16);
        xr[m][j][4 * g + 0] = v.x;
        xr[m][j][4 * g + 1] = v.y;
        xr[m][j][4 * g + 2] = v.z;
        xr[m][j][4 * g + 3] = v.w;
      }
    }
  int32_t xs[MT];
  float fs[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    xs[m] = xsum[m];
    fs[m] = fscale[m];
  }

  // ------------------------------------------------------------ main loop --
  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kLdgStages;
    if (ok && !mbar_wait(&wbar[slot], (uint32_t)((st / kLdgStages) & 1))) {
      raise_device_error(kDevErrTimeout);
      ok = false;  // keep walking (results undefined, the error word says so)
    }
    const uint8_t *stage = ring + slot * kLdgStageBytes;
    const int64_t ra = r0 + (int64_t)st * p.SR;
    const int nr = (int)(min(ra + p.SR, r1) - ra);
    for (int i = 0; i < nr; ++i) {
      const int64_t r = ra + i;
      int a[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int s = 0; s < 4; ++s) a[m][s] = 0;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = lane + 32 * j;
        uint4 wq = make_uint4(0u, 0u, 0u, 0u);
        if (c < p.C) wq = lds_u128(smem_u32(stage + (size_t)i * rowb + (size_t)c * 16));
        const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t f0 = wv[u] & 0x03030303u, f1 = wv[u] & 0x0C0C0C0Cu;
          const uint32_t f2 = wv[u] & 0x30303030u, f3 = wv[u] & 0xC0C0C0C0u;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            a[m][0] = dp4a_u8s8(f0, xr[m][j][4 * u + 0], a[m][0]);
            a[m][1] = dp4a_u8s8(f1, xr[m][j][4 * u + 1], a[m][1]);
            a[m][2] = dp4a_u8s8(f2, xr[m][j][4 * u + 2], a[m][2]);
            a[m][3] = dp4a_u8s8(f3, xr[m][j][4 * u + 3], a[m][3]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        int v = a[m][0] + (a[m][1] >> 2) + (a[m][2] >> 4) + (a[m][3] >> 6);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == m) {
          const int32_t o = v - xs[m];
          if (p.acc) p.acc[(int64_t)m * p.N + r] = o;
          p.y[(int64_t)m * p.N + r] = __fmul_rn((float)o, fs[m]);
        }
      }
    }
    // every lane's reads of this stage are done: refill it
    __syncwarp();
    if (lane == 0 && ok && st + kLdgStages < nst) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(st + kLdgStages);
    }
  }
  // After a timeout leave no bulk copy in flight (bounded waits on the
  // stages this lane requested last).
  if (!ok && lane == 0) {
    for (int st = (issued > kLdgStages ? issued - kLdgStages : 0); st < issued; ++st)
      mbar_wait(&wbar[st % kLdgStages], (uint32_t)((st / kLdgStages) & 1));
  }
}

}  // namespace bitnet

// Group-wise weight scales on the mma.sync tensor path (3..64 tokens).
//
// The product of BitNet 深度拆解 §4.3's group-wise form: every group of G
// consecutive weights of a row has its own scale, y[m, n] = (s_m / 127) *
// sum_g scale[n, g] * acc_g[m, n], acc_g = sum over the group of
// (code - 1) * x_q (exact int32).  Same units, ring and producer as
// gemv_mma_kernel, and the same exact fp16 encoding (a 2-bit field masked in
// place is code * 4^i * 2^-24; the prepared activations are x_q * 4^-i), so
// the fp32 accumulator of a group is exact: D * 2^24 - (sum of x_q over the
// group) is acc_g.
//   * Warp w takes the 16-row block w of a unit over all its K-blocks (the
//     groups, G <= 512 with G | 512, never straddle a 512-K unit, and a unit
//     is never split between CTAs), so a group's sum ends in one warp's
//     registers: at the group's last K-block the warp converts it, subtracts
//     the tokens' group sums of x_q (shared memory), optionally stores the
//     exact acc_g, and adds acc_g * scale[n, g] into an fp32 sum F with one
//     FMA (one rounding per group, in increasing g).
//   * At a segment end F goes to shared memory; a tile finished inside the
//     CTA writes y = fl(F * fl(s / 127)); a tile split between CTAs adds its
//     F into the workspace with fp32 atomics (the order of those few
//     additions is the hardware's; the tolerance of the group-scaled output
//     covers it) and the CTA that completes it (ticket) writes y.
#pragma once

#include "common.cuh"
#include "gemv_mma.cuh"

namespace bitnet {

struct GemvMmaGroups {
  const float *gscale;   // [N, NG] group scales
  const int32_t *xsumg;  // [M, NG] sum of x_q per token and group
  int32_t *acc_g;        // [M, N, NG] exact per-group products, or nullptr
  int G, NG, KBG;        // group size, groups per row, 64-K blocks per group
};

// Largest [M][NG] table of group sums kept in shared memory.
constexpr int kMmaGroupSumsBytes = 16384;

template <int NT8>
struct GemvMmaGroupedSmem {
  using B = GemvMmaSmem<NT8>;
  static constexpr int kTok = B::kTok, kBBytes = B::kBBytes, kBoxRows = B::kBoxRows, kStage = B::kStage;
  static constexpr int ring = 0;
  static constexpr int red = MmaCfg<NT8>::stages * kStage;  // F [tokens][kMmaRS] fp32
  static constexpr int toks = red + kTok * kMmaRS * 4;       // fscale [64]
  static constexpr int xsg = toks + 256;                     // [M][NG] int32
  static constexpr int bars = xsg + kMmaGroupSumsBytes;
  static constexpr int flags = bars + 2 * MmaCfg<NT8>::stages * 8;
  static constexpr int bytes = flags + 16;
};

template <int NT8>
__global__ void __launch_bounds__(kMmaThreads, MmaCfg<NT8>::ctas)
    gemv_mma_grouped_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                            const GemvMmaParams p, const GemvMmaGroups gp) {
  using L = GemvMmaGroupedSmem<NT8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *empty = full + MmaCfg<NT8>::stages;
  float *fsl = reinterpret_cast<float *>(smem + L::red);
  float *fscale_s = reinterpret_cast<float *>(smem + L::toks);
  int32_t *xsg_s = reinterpret_cast<int32_t *>(smem + L::xsg);
  volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flags);  // [0] abort, [1] last CTA

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const long long g0 = p.units * blockIdx.x / gridDim.x;
  const long long g1 = p.units * (blockIdx.x + 1) / gridDim.x;
  pdl_launch_dependents();
  if (tid == 0) {
    for (int i = 0; i < MmaCfg<NT8>::stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMmaWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kMmaWarps) {
    if (lane == 0)
      mma_producer<NT8, L::kStage, L::kBBytes, L::kBoxRows>(&wmap, &bmap, p, smem + L::ring, full, empty, flags, g0, g1);
    return;
  }

  // ---------------------------------------------------------- compute warps --
  pdl_wait_prior_grid();  // the token scales and group sums come from the prep kernel
  for (int i = tid; i < p.M; i += kMmaWarps * 32) fscale_s[i] = p.fscale[i];
  for (int i = tid; i < p.M * gp.NG; i += kMmaWarps * 32) xsg_s[i] = gp.xsumg[i];
  named_barrier_sync(kMmaBar, kMmaWarps * 32);
  const int64_t NRp = (int64_t)p.NRT * 128;
  float *ws_f = reinterpret_cast<float *>(p.ws_partial);  // split-tile sums F [tokens][NRp]
  const int g = lane >> 2, t = lane & 3;
  // With 64 tokens the running sums F live in the warp's rows of the slice
  // (registers hold the group accumulators d), else in registers.
  constexpr bool kFsmem = NT8 == 8;
  float d[NT8][4], F[NT8][kFsmem ? 1 : 4];
#pragma unroll
  for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      d[nt][e] = 0.0f;
      if (!kFsmem) F[nt][kFsmem ? 0 : e] = 0.0f;
    }

  int it = 0;  // units this CTA has taken (fewer than 2^31)
  long long u = g0;
  while (u < g1) {
    const int r = (int)(u / p.NCH);
    const int c0 = (int)(u % p.NCH);
    const long long tile_end = (long long)(r + 1) * p.NCH;
    const long long u_end = tile_end < g1 ? tile_end : g1;
    const int nch = (int)(u_end - u);
    const long long u_seg = u;  // unit u is chunk c0 + (u - u_seg) of tile r
    const int row0 = warp * 16 + g;                 // this lane's fragment rows: row0, row0 + 8
    const int64_t n0 = (int64_t)r * 128 + row0, n1 = n0 + 8;
    if constexpr (kFsmem) {  // this warp's rows of the slice hold F: start from zero
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) fsl[(nt * 8 + 2 * t + (e & 1)) * kMmaRS + row0 + ((e >> 1) << 3)] = 0.0f;
    }
    for (; u < u_end; ++u, ++it) {
      const int s = (int)(it % MmaCfg<NT8>::stages);
      if (!flags[0] && !mbar_wait(&full[s], (uint32_t)((it / MmaCfg<NT8>::stages) & 1))) {
        raise_device_error(kDevErrTimeout);
        flags[0] = 1;
      }
      const int c = c0 + (int)(u - u_seg);
      const uint32_t st = smem_u32(smem + L::ring + s * L::kStage);
      const int nkb = mma_chunk_kbs(p, c);
      float sc0 = 0.0f, sc1 = 0.0f;
#pragma unroll 1
      for (int k2 = 0; k2 < nkb; ++k2) {
        const int kb = c * 8 + k2, grp = kb / gp.KBG;
        if (kb % gp.KBG == 0) {  // the group's scales, ahead of its MMAs
          sc0 = n0 < p.N ? __ldg(gp.gscale + n0 * gp.NG + grp) : 0.0f;
          sc1 = n1 < p.N ? __ldg(gp.gscale + n1 * gp.NG + grp) : 0.0f;
        }
        const uint32_t off = (uint32_t)((((k2 ^ g) & 7) << 4) + (t << 2));
        const uint32_t w0 = lds_u32(st + row0 * 128 + off);
        const uint32_t w1 = lds_u32(st + (row0 + 8) * 128 + off);
        const uint32_t bst = st + 16384 + k2 * L::kTok * 128;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
          // one conflict-free 16-byte load per token tile holds the B
          // fragments of 16-K steps 2 jh and 2 jh + 1
          uint4 bq[NT8];
#pragma unroll
          for (int nt = 0; nt < NT8; ++nt) bq[nt] = mma_b_granule(bst, nt * 8 + g, t * 2 + jh);
#pragma unroll
          for (int jl = 0; jl < 2; ++jl) {
            uint32_t a0, a1, a2, a3;
            mma_a_frag(w0, w1, 2 * jh + jl, a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt)
              mma_f16_16816(d[nt], a0, a1, a2, a3, jl ? bq[nt].z : bq[nt].x, jl ? bq[nt].w : bq[nt].y);
          }
        }
        if ((kb + 1) % gp.KBG == 0) {  // the group is complete in d: fold it into F
#pragma unroll
          for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = nt * 8 + 2 * t + (e & 1);
              const int32_t ag = __float2int_rn(d[nt][e] * 16777216.0f) - (tok < p.M ? xsg_s[tok * gp.NG + grp] : 0);
              d[nt][e] = 0.0f;
              const int64_t n = (e >> 1) ? n1 : n0;
              if (tok < p.M && n < p.N) {
                if (gp.acc_g) gp.acc_g[((int64_t)tok * p.N + n) * gp.NG + grp] = ag;
                if constexpr (kFsmem) {
                  float *f = fsl + tok * kMmaRS + row0 + ((e >> 1) << 3);
                  *f = __fmaf_rn((float)ag, (e >> 1) ? sc1 : sc0, *f);
                } else {
                  F[nt][kFsmem ? 0 : e] = __fmaf_rn((float)ag, (e >> 1) ? sc1 : sc0, F[nt][kFsmem ? 0 : e]);
                }
              }
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------------------------- segment end --
    if constexpr (!kFsmem) {
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = row0 + ((e >> 1) << 3);
          const int tok = nt * 8 + 2 * t + (e & 1);
          if (tok < p.M) fsl[tok * kMmaRS + row] = F[nt][kFsmem ? 0 : e];
          F[nt][kFsmem ? 0 : e] = 0.0f;
        }
    }
    named_barrier_sync(kMmaBar, kMmaWarps * 32);
    const bool whole = (c0 == 0) && (nch == p.NCH);
    const int entries = 128 * p.M;
    if (whole) {
      for (int i = tid; i < entries; i += kMmaWarps * 32) {
        const int row = i & 127, tok = i >> 7;
        const int64_t n = (int64_t)r * 128 + row;
        if (n < p.N) p.y[(int64_t)tok * p.N + n] = __fmul_rn(fsl[tok * kMmaRS + row], fscale_s[tok]);
      }
    } else {
      for (int i = tid; i < entries; i += kMmaWarps * 32) {
        const int row = i & 127, tok = i >> 7;
        const int64_t n = (int64_t)r * 128 + row;
        const float v = fsl[tok * kMmaRS + row];
        if (n < p.N && v != 0.0f) atomicAdd(&ws_f[(int64_t)tok * NRp + n], v);
      }
      __threadfence();
      named_barrier_sync(kMmaBar, kMmaWarps * 32);
      if (tid == 0) {
        const unsigned old = atomicAdd(&p.ws_ticket[r], (unsigned)nch);
        flags[1] = (old + (unsigned)nch == (unsigned)p.NCH) ? 1 : 0;
      }
      named_barrier_sync(kMmaBar, kMmaWarps * 32);
      if (flags[1]) {
        __threadfence();
        constexpr int kU = 8;
        for (int i0 = tid; i0 < entries; i0 += kU * kMmaWarps * 32) {
          float v[kU];
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            const int i = i0 + k * kMmaWarps * 32;
            const int64_t n = (int64_t)r * 128 + (i & 127);
            v[k] = (i < entries && n < p.N) ? __ldcg(ws_f + (int64_t)(i >> 7) * NRp + n) : 0.0f;
          }
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            const int i = i0 + k * kMmaWarps * 32;
            const int64_t n = (int64_t)r * 128 + (i & 127);
            if (i < entries && n < p.N) {
              ws_f[(int64_t)(i >> 7) * NRp + n] = 0.0f;
              p.y[(int64_t)(i >> 7) * p.N + n] = __fmul_rn(v[k], fscale_s[i >> 7]);
            }
          }
        }
        if (tid == 0) atomicExch(&p.ws_ticket[r], 0u);
      }
    }
    named_barrier_sync(kMmaBar, kMmaWarps * 32);
  }
}

}  // namespace bitnet

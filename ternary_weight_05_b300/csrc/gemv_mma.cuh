// Decode-path W2A8 ternary GEMV for 3..64 tokens on the mma.sync tensor path.
//
// Same operation as the other GEMV kernels: y[m, n] = (sum_k (code[n,k]-1) *
// x_q[m,k]) * (w_scale * s_m / 127), the integer-domain product of BitNet
// 深度拆解 §3.1 (§1: a ternary weight turns each product into +x, 0 or -x)
// with the dequantisation of §2.3.
//
// A few tokens need 2 * M multiply-adds per weight: more than dp4a sustains
// at HBM speed for M > 2, while tcgen05 MMAs with N = 8..64 tokens cost far
// more per instruction than their arithmetic (measured: a tcgen05 form of
// this kernel was slower at every M up to 64).  mma.sync m16n8k16
// takes A (16 weight rows x 16 K) straight from registers, so decoding costs
// one AND per two weights and nothing else touches shared memory but the
// packed weights and the activations:
//   * A fragment: a 2-bit field masked in place inside a 16-bit lane is the
//     fp16 subnormal code * 4^i * 2^-24; B is the prepared activation matrix
//     (x_q * 4^-i in fp16, gemm_prep_kernel), so every product is
//     code * x * 2^-24 and fp32 accumulation is exact (D * 2^24 is the
//     integer sum of code * x; the per-token sum of x_q is subtracted once).
//   * Work units are (128-row tile, 512-K chunk) pairs; CTA c takes an equal
//     contiguous range of units (stream-K).  Each unit's 16 KB of packed
//     weights and its activation slice (prepared K-block-major, so the slice
//     is one box) arrive in one stage of a ring with two TMA copies (the cost
//     of a copy is per box, so boxes are few and large); 3 or 5 stages in
//     flight, weights requested before waiting on the previous kernel.
//   * Up to 16 tokens, warp w of the 8 compute warps takes the 64-K column w
//     of every unit for all 8 row blocks: its activation fragments are loaded
//     once per unit and reused 8 times, and the warps' exact int32 partial
//     sums are added in shared memory.  With 32 or 64 tokens the accumulators
//     of 8 row blocks would not fit in registers: warp w then takes row block
//     w over all K-blocks of the unit and owns its outputs alone.  At the end
//     of a row tile's segment each warp stores its exact int32 partial sums
//     into its own shared-memory slice [token][row]; the warps then add the
//     slices output by output, consecutive threads taking consecutive rows,
//     so that every global access below is coalesced.  A tile finished
//     inside the CTA is written directly; a tile split between CTAs is summed
//     with int32 atomics in the workspace and written by the CTA that
//     completes it (ticket), which re-zeroes the entries.  The per-token sums
//     and output scales are read into shared memory once per CTA.
// Every wait is bounded; on expiry the CTA records the error and walks out
// without waiting (outputs undefined, the device error word says so).
#pragma once

#include "common.cuh"

namespace bitnet {

constexpr int kMmaRows = 128;    // weight rows per tile
constexpr int kMmaChunkK = 512;  // K per work unit (one 128-byte column of packed rows)
constexpr int kMmaKB = 64;       // K per activation block (K-block-major layout)

struct GemvMmaParams {
  float *y;
  int32_t *acc;
  const int32_t *xsum;   // [M] sum of x_q per token
  const float *fscale;   // [M] w_scale * s_m / 127
  int32_t *ws_partial;   // [M][NRT * 128] (row fastest), zero on entry and exit
  unsigned *ws_ticket;   // [NRT], zero on entry and exit
  int64_t N, K;
  int M;
  int NRT;               // row tiles
  int NCH;               // 512-K chunks per row
  int NKB;               // 64-K blocks per row (K / 64)
  long long units;       // NRT * NCH
};

// Unit u = (row tile u / NCH, chunk u % NCH).  The K-blocks of chunk c are
// [8c, min(8c + 8, NKB)).
__device__ __forceinline__ int mma_chunk_kbs(const GemvMmaParams &p, int c) { return min(8, p.NKB - 8 * c); }

constexpr int kMmaWarps = 8;                 // compute warps (one 64-K column each)
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
// NT8 token tiles of 8.  CTAs per SM: two for 8 token rows (fits 96
// registers: measured 1.2x), else one.  Stages: as many as shared memory
// holds beside the reduction buffer.  WIDE (32 or 64 tokens): warp w owns row
// block w over all K-blocks of a unit (the accumulators of 8 row blocks would
// not fit in registers); otherwise warp w owns the 64-K column w of all 8 row
// blocks.
template <int NT8> struct MmaCfg {
  static constexpr int ctas = NT8 == 1 ? 2 : 1;
  static constexpr int stages = NT8 == 1 ? 3 : (NT8 == 2 ? 4 : (NT8 == 4 ? 3 : 2));
  static constexpr bool wide = NT8 >= 4;
  // partial-sum slices at a segment end: one per compute warp when the
  // warps split K (their sums are added), one shared slice when they split rows
  static constexpr int slices = wide ? 1 : 8;
};
constexpr int kMmaBar = 3;                   // named barrier of the compute warps
constexpr int kMmaRS = 132;                  // int32 per token row of a slice (128 rows + 4: no bank conflicts)

template <int NT8>
struct GemvMmaSmem {
  static constexpr int kTok = NT8 * 8;                  // token rows of the B box
  static constexpr int kBBytes = 8 * kTok * 128;        // activation slice of a unit
  static constexpr int kBoxRows = 8 * kTok < 256 ? 8 * kTok : 256;  // TMA box limit
  static constexpr int kStage = 16384 + kBBytes;
  static constexpr int ring = 0;
  static constexpr int red = MmaCfg<NT8>::stages * kStage;  // [slices][tokens][kMmaRS] int32
  static constexpr int toks = red + MmaCfg<NT8>::slices * kTok * kMmaRS * 4;  // xsum [64], fscale [64]
  static constexpr int bars = toks + 512;
  static constexpr int flags = bars + 2 * MmaCfg<NT8>::stages * 8;
  static constexpr int bytes = flags + 16;
};

// A fragment of 16-K step j (0..3) of a 64-K block from the packed words w0
// (row g) and w1 (row g + 8) of the lane: each 2-bit field masked in place
// inside a 16-bit lane is the fp16 value code * 4^i * 2^-24.
__device__ __forceinline__ void mma_a_frag(uint32_t w0, uint32_t w1, int j, uint32_t &a0, uint32_t &a1, uint32_t &a2,
                                           uint32_t &a3) {
  if (j < 3) {
    const uint32_t m0 = 0x00030003u << (4 * j), m1 = 0x00030003u << (4 * j + 2);
    a0 = w0 & m0;
    a1 = w1 & m0;
    a2 = w0 & m1;
    a3 = w1 & m1;
  } else {
    const uint32_t h0 = w0 >> 12, h1 = w1 >> 12;
    a0 = h0 & 0x00030003u;
    a1 = h1 & 0x00030003u;
    a2 = h0 & 0x000C000Cu;
    a3 = h1 & 0x000C000Cu;
  }
}

// The 16-byte granule ci of token row `tok` of an activation block (rows of
// 128 bytes, 128-byte swizzle): the B fragments (b0, b1) of 16-K steps
// 2 (ci % 2) and 2 (ci % 2) + 1 for the lanes with t = ci / 2.  Across a warp
// (g = token row % 8, t) the eight rows hit eight distinct granule columns.
__device__ __forceinline__ uint4 mma_b_granule(uint32_t bst, int tok, int ci) {
  return lds_u128(bst + tok * 128 + (((ci ^ (tok & 7)) & 7) << 4));
}

// The TMA producer of the tensor-core GEMV kernels (one thread): for every
// unit of the CTA's range, the 128 x 512-K packed-weight tile and the unit's
// activation slice into the next ring stage.  The weights are requested
// before waiting on the previous kernel (they do not depend on it).
template <int NT8, int kStage, int kBBytes, int kBoxRows>
__device__ __forceinline__ void mma_producer(const CUtensorMap *wmap, const CUtensorMap *bmap, const GemvMmaParams &p,
                                             uint8_t *ring, uint64_t *full, uint64_t *empty, volatile int *flags,
                                             long long g0, long long g1) {
  constexpr int kTok = NT8 * 8, S = MmaCfg<NT8>::stages;
  prefetch_tensormap(wmap);
  prefetch_tensormap(bmap);
  const uint64_t pol_w = l2_policy_evict_first(), pol_b = l2_policy_evict_last();
  int it = 0;  // units this CTA has taken (fewer than 2^31)
  bool waited = false;
  int r = (int)(g0 / p.NCH), c = (int)(g0 % p.NCH) - 1;  // unit g0 - 1: stepped below
  for (long long u = g0; u < g1; ++u, ++it) {
    const int s = it % S;
    if (it >= S && !mbar_wait(&empty[s], (uint32_t)(((it / S) - 1) & 1))) {
      raise_device_error(kDevErrTimeout);
      flags[0] = 1;
    }
    if (flags[0]) break;
    if (++c == p.NCH) {  // (tile, chunk) of unit u
      c = 0;
      ++r;
    }
    uint8_t *st = ring + s * kStage;
    mbar_arrive_expect_tx(&full[s], 16384 + kBBytes);
    tma_load_2d(st, wmap, &full[s], c * 128, r * 128, pol_w);
    if (!waited) {  // the activations come from the previous kernel
      pdl_wait_prior_grid();
      waited = true;
    }
    // the unit's 8 K-blocks x kTok token rows: one box, two for 64 tokens
    // (rows past K are zero-filled)
    for (int b = 0; b < 8 * kTok; b += kBoxRows) tma_load_2d(st + 16384 + b * 128, bmap, &full[s], 0, c * 8 * kTok + b, pol_b);
  }
  if (!waited) pdl_wait_prior_grid();
  if (flags[0]) {  // leave no copy in flight (bounded waits)
    for (int j = (it > S ? it - S : 0); j < it; ++j) mbar_wait(&full[j % S], (uint32_t)((j / S) & 1));
  }
}

template <int NT8>
__global__ void __launch_bounds__(kMmaThreads, MmaCfg<NT8>::ctas)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                    const GemvMmaParams p) {
  using L = GemvMmaSmem<NT8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *empty = full + MmaCfg<NT8>::stages;
  int32_t *red = reinterpret_cast<int32_t *>(smem + L::red);
  int32_t *xsum_s = reinterpret_cast<int32_t *>(smem + L::toks);
  float *fscale_s = reinterpret_cast<float *>(smem + L::toks + 256);
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
  pdl_wait_prior_grid();  // xsum / fscale come from the previous kernel
  for (int i = tid; i < p.M; i += kMmaWarps * 32) {
    xsum_s[i] = p.xsum[i];
    fscale_s[i] = p.fscale[i];
  }
  named_barrier_sync(kMmaBar, kMmaWarps * 32);
  const int64_t NRp = (int64_t)p.NRT * 128;  // rows of the split-tile partial sums [tokens][NRp]
  const int g = lane >> 2, t = lane & 3;
  constexpr bool kWide = MmaCfg<NT8>::wide;
  constexpr int RBN = kWide ? 1 : 8;  // row blocks in this warp's accumulators
  const int kb = warp;                // narrow: this warp's 64-K column of every unit
  float d[RBN][NT8][4];
#pragma unroll
  for (int rb = 0; rb < RBN; ++rb)
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) d[rb][nt][e] = 0.0f;

  int it = 0;  // units this CTA has taken (fewer than 2^31)
  long long u = g0;
  while (u < g1) {
    const int r = (int)(u / p.NCH);
    const int c0 = (int)(u % p.NCH);
    const long long tile_end = (long long)(r + 1) * p.NCH;
    const long long u_end = tile_end < g1 ? tile_end : g1;  // segment: units [u, u_end) of tile r
    const int nch = (int)(u_end - u);
    const long long u_seg = u;  // unit u is chunk c0 + (u - u_seg) of tile r
    for (; u < u_end; ++u, ++it) {
      const int s = (int)(it % MmaCfg<NT8>::stages);
      if (!flags[0] && !mbar_wait(&full[s], (uint32_t)((it / MmaCfg<NT8>::stages) & 1))) {
        raise_device_error(kDevErrTimeout);
        flags[0] = 1;
      }
      const int c = c0 + (int)(u - u_seg);
      if constexpr (kWide) {
        // row block `warp` over the unit's K-blocks
        const uint32_t st = smem_u32(smem + L::ring + s * L::kStage);
        const int r0 = warp * 16 + g;
        const int nkb = mma_chunk_kbs(p, c);
#pragma unroll 1
        for (int k2 = 0; k2 < nkb; ++k2) {
          const uint32_t off = (uint32_t)((((k2 ^ g) & 7) << 4) + (t << 2));
          const uint32_t w0 = lds_u32(st + r0 * 128 + off);
          const uint32_t w1 = lds_u32(st + (r0 + 8) * 128 + off);
          const uint32_t bst = st + 16384 + k2 * L::kTok * 128;
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            // the B fragments of j = 2 jh and 2 jh + 1 sit in one 16-byte
            // granule per token row: one conflict-free 16-byte load
            uint4 bq[NT8];
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) bq[nt] = mma_b_granule(bst, nt * 8 + g, t * 2 + jh);
#pragma unroll
            for (int jl = 0; jl < 2; ++jl) {
              const int j = 2 * jh + jl;
              uint32_t a0, a1, a2, a3;
              mma_a_frag(w0, w1, j, a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NT8; ++nt)
                mma_f16_16816(d[0][nt], a0, a1, a2, a3, jl ? bq[nt].z : bq[nt].x, jl ? bq[nt].w : bq[nt].y);
            }
          }
        }
      } else if (kb < mma_chunk_kbs(p, c)) {
        const uint32_t st = smem_u32(smem + L::ring + s * L::kStage);
        uint32_t w0[8], w1[8];
#pragma unroll
        for (int rb = 0; rb < 8; ++rb) {
          const int r0 = rb * 16 + g;  // r0 & 7 == g, (r0 + 8) & 7 == g
          const uint32_t off = (uint32_t)((((kb ^ g) & 7) << 4) + (t << 2));
          w0[rb] = lds_u32(st + r0 * 128 + off);
          w1[rb] = lds_u32(st + (r0 + 8) * 128 + off);
        }
        const uint32_t bst = st + 16384 + kb * L::kTok * 128;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
          uint4 bq[NT8];
#pragma unroll
          for (int nt = 0; nt < NT8; ++nt) bq[nt] = mma_b_granule(bst, nt * 8 + g, t * 2 + jh);
#pragma unroll
          for (int jl = 0; jl < 2; ++jl) {
            const int j = 2 * jh + jl;
#pragma unroll
            for (int rb = 0; rb < 8; ++rb) {
              uint32_t a0, a1, a2, a3;
              mma_a_frag(w0[rb], w1[rb], j, a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < NT8; ++nt)
                mma_f16_16816(d[rb][nt], a0, a1, a2, a3, jl ? bq[nt].z : bq[nt].x, jl ? bq[nt].w : bq[nt].y);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ------------------------------------------------------- segment end --
    // exact int32 partial sums into the warp's slice [token][row] (the
    // fragment layout makes these stores conflict-free); the compute warps
    // then add the slices per output, row by row, so that the outputs and
    // the split-tile partial sums are written with coalesced accesses
    {
      int32_t *sl = red + (kWide ? 0 : warp) * (L::kTok * kMmaRS);
#pragma unroll
      for (int rb = 0; rb < RBN; ++rb)
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = (kWide ? warp : rb) * 16 + g + ((e >> 1) << 3);
            const int tok = nt * 8 + 2 * t + (e & 1);
            const int v = __float2int_rn(d[rb][nt][e] * 16777216.0f);
            d[rb][nt][e] = 0.0f;
            if (tok < p.M) sl[tok * kMmaRS + row] = v;
          }
    }
    named_barrier_sync(kMmaBar, kMmaWarps * 32);
    const bool whole = (c0 == 0) && (nch == p.NCH);
    const int entries = 128 * p.M;
    auto total_of = [&](int row, int tok) {
      int v = 0;
#pragma unroll
      for (int sl = 0; sl < MmaCfg<NT8>::slices; ++sl) v += red[(sl * L::kTok + tok) * kMmaRS + row];
      return v;
    };
    auto write_out = [&](int64_t n, int tok, int32_t total) {
      const int32_t o = total - xsum_s[tok];
      if (p.acc) p.acc[(int64_t)tok * p.N + n] = o;
      p.y[(int64_t)tok * p.N + n] = __fmul_rn((float)o, fscale_s[tok]);
    };
    if (whole) {
      for (int i = tid; i < entries; i += kMmaWarps * 32) {
        const int row = i & 127, tok = i >> 7;
        const int64_t n = (int64_t)r * 128 + row;
        const int32_t v = total_of(row, tok);
        if (n < p.N) write_out(n, tok, v);
      }
    } else {
      for (int i = tid; i < entries; i += kMmaWarps * 32) {
        const int row = i & 127, tok = i >> 7;
        const int64_t n = (int64_t)r * 128 + row;
        const int32_t v = total_of(row, tok);
        if (n < p.N && v != 0) atomicAdd(&p.ws_partial[(int64_t)tok * NRp + n], v);
      }
      __threadfence();  // partial sums visible before the ticket
      named_barrier_sync(kMmaBar, kMmaWarps * 32);
      if (tid == 0) {
        const unsigned old = atomicAdd(&p.ws_ticket[r], (unsigned)nch);
        flags[1] = (old + (unsigned)nch == (unsigned)p.NCH) ? 1 : 0;
      }
      named_barrier_sync(kMmaBar, kMmaWarps * 32);
      if (flags[1]) {
        __threadfence();
        // eight independent loads in flight per thread, then their stores:
        // a load placed after a store that may alias would wait a whole L2
        // round trip per output
        constexpr int kU = 8;
        for (int i0 = tid; i0 < entries; i0 += kU * kMmaWarps * 32) {
          int32_t v[kU];
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            const int i = i0 + k * kMmaWarps * 32;
            const int64_t n = (int64_t)r * 128 + (i & 127);
            v[k] = (i < entries && n < p.N) ? __ldcg(p.ws_partial + (int64_t)(i >> 7) * NRp + n) : 0;
          }
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            const int i = i0 + k * kMmaWarps * 32;
            const int64_t n = (int64_t)r * 128 + (i & 127);
            if (i < entries && n < p.N) {
              p.ws_partial[(int64_t)(i >> 7) * NRp + n] = 0;  // leave the partial sums zero for the next call
              write_out(n, i >> 7, v[k]);
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

// Decode-path W2A8 ternary GEMV for 3..64 tokens on the tcgen05 tensor cores.
//
// Same operation as the other GEMV kernels: y[m, n] = (sum_k (code[n,k]-1) *
// x_q[m,k]) * (w_scale * s_m / 127), the integer-domain product of BitNet
// 深度拆解 §3.1 (§1: a ternary weight turns each product into +x, 0 or -x)
// with the dequantisation of §2.3.
//
// With a few tokens the work per weight is small but not negligible: 16
// tokens need about 2 * 16 multiply-adds per weight, more than the integer
// pipes (dp4a) or the legacy mma.sync path sustain at HBM speed on B300.  The
// tcgen05 tensor cores do it with room to spare, so the kernel stays bound by
// the packed-weight stream:
//   * D (128 weight rows x NT tokens, fp32 in TMEM) += A (128 rows x 16 K,
//     fp16 in TMEM) * B (NT tokens x 16 K, fp16 in shared memory), NT = 16, 32
//     or 64 (tokens beyond M are zero rows of B).
//   * A is decoded from the packed codes by four decoder warps and written to
//     TMEM with tcgen05.st (decoded weights never touch shared memory): a
//     2-bit field masked in place inside a 16-bit lane is the fp16 subnormal
//     code * 4^i * 2^-24.  B is the prepared activation matrix (x_q * 4^-i in
//     fp16, the K order of the decode; gemm_prep_kernel), so every product is
//     code * x * 2^-24 and fp32 accumulation is exact: D * 2^24 is the exact
//     integer sum of code * x.  The per-token sum of x_q is subtracted once,
//     when the output is written.
//   * Work units are (128-row tile, 512-K chunk) pairs.  CTA c takes an equal
//     contiguous range of units ("stream-K"), so every SM streams the same
//     number of weight bytes whatever the shape.  A row tile finished inside
//     one CTA is written directly; a tile split between CTAs is summed with
//     exact int32 atomics in the workspace, and the CTA completing its last
//     chunk (a ticket per tile) writes the outputs and re-zeroes the entries.
//   * Separate TMA producers for the weights (up to kTcWStages 16 KB stages in
//     flight, requested before waiting on the previous kernel) and for the
//     activations (L2-resident), so the weight stream never waits for the
//     tensor pipe.  Two accumulators let a segment's epilogue overlap the next
//     segment's MMAs.
// Warp roles: 0 weight producer, 1 TMEM owner + MMA issuer, 2 activation
// producer, 4-7 decoders (set 0), 8-11 epilogue, 12-15 ... further decoder
// sets; set d decodes the K-blocks c with c % kTcDecSets == d, so several
// blocks per TMEM lane quarter are in flight while a warp waits for its
// tcgen05.st to land.  Every wait is bounded; on expiry the
// CTA records the error, stops issuing, drains its copies and MMAs, frees
// TMEM and exits (outputs are then undefined and the device error word says
// so; the workspace must be re-zeroed).
#pragma once

#include "common.cuh"
#include "gemm.cuh"

namespace bitnet {

#ifndef BITNET_TC_DEC_SETS
#define BITNET_TC_DEC_SETS 1
#endif
constexpr int kTcDecSets = BITNET_TC_DEC_SETS;  // decoder warp sets of 4 warps
constexpr int kTcThreads = 384 + (kTcDecSets - 1) * 128;
// Two CTAs per SM (half the TMEM and shared memory each): two MMA issuers
// per SM measured 1.35x the throughput of one.
constexpr int kTcCtasPerSm = 2;
constexpr int kTcRows = 128;       // weight rows per tile (MMA M)
constexpr int kTcChunkK = 512;     // K per work unit (one 128-byte column of packed rows)
constexpr int kTcKB = 64;          // K per MMA step group (4 MMAs of K = 16)
constexpr int kTcWStages = 3;      // packed-weight stages (16 KB each)
constexpr int kTcStages = 4;       // activation stages in smem == A buffers in TMEM
constexpr int kTcTmemCols = 256;   // per CTA (two CTAs per SM)
constexpr int kTcACol = 128;       // A buffers: columns [128, 128 + 4 * 32)
constexpr int kTcEpiBar = 2;       // named barrier of the epilogue warps

struct GemvTcParams {
  float *y;
  int32_t *acc;
  const int32_t *xsum;   // [M] sum of x_q per token
  const float *fscale;   // [M] w_scale * s_m / 127
  int32_t *ws_partial;   // [NRT * 128][M], zero on entry and exit
  unsigned *ws_ticket;   // [NRT], zero on entry and exit
  int64_t N, K;
  int M;
  int NRT;               // row tiles
  int NCH;               // 512-K chunks per row
  int NKB;               // 64-K blocks per row (K / 64)
  long long units;       // NRT * NCH
};

template <int NT>
struct GemvTcSmem {
  static constexpr int kBStage = NT * 128;
  static constexpr int wstage = 0;
  static constexpr int bstage = kTcWStages * 16384;
  static constexpr int bars = bstage + kTcStages * kBStage;
  static constexpr int tmem_slot = bars + 512;
  static constexpr int flags = tmem_slot + 16;
  static constexpr int bytes = flags + 16;
};

// Unit u = (row tile u / NCH, chunk u % NCH).  The K-blocks of chunk c are
// [8c, min(8c + 8, NKB)).
__device__ __forceinline__ int tc_chunk_kbs(const GemvTcParams &p, int c) { return min(8, p.NKB - 8 * c); }

template <int NT>
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                   const GemvTcParams p) {
  using L = GemvTcSmem<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bfull = reinterpret_cast<uint64_t *>(smem + L::bars);  // [kTcStages] B TMA -> MMA
  uint64_t *kempty = bfull + kTcStages;                              // [kTcStages] MMA done -> B producer, decoders
  uint64_t *afull = kempty + kTcStages;                              // [kTcStages] decoders -> MMA
  uint64_t *wfull = afull + kTcStages;                               // [kTcWStages] W TMA -> decoders
  uint64_t *wempty = wfull + kTcWStages;                             // [kTcWStages] decoders -> W producer
  uint64_t *accfull = wempty + kTcWStages;                           // [2] MMA -> epilogue
  uint64_t *accempty = accfull + 2;                                  // [2] epilogue -> MMA
  uint64_t *drain = accempty + 2;                                    // [1] final MMA completion
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::tmem_slot);
  // [0] abort, [1] last CTA of a tile, [2] abort snapshot for the epilogue
  volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flags);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long g0 = p.units * blockIdx.x / gridDim.x;
  const long long g1 = p.units * (blockIdx.x + 1) / gridDim.x;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&afull[i], 4);
    }
    for (int i = 0; i < kTcWStages; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 4 * kTcDecSets);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], 4);
    }
    mbar_init(drain, 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTcTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (flags[0]) return;
    if (!mbar_wait(bar, parity)) {
      raise_device_error(kDevErrTimeout);
      flags[0] = 1;
    }
  };

  if (warp == 0) {
    // ---------------------------------------------------- weight producer --
    // The packed weights do not depend on earlier kernels: no PDL wait here.
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      const uint64_t pol = l2_policy_evict_first();
      long long wc = 0;
      for (long long u = g0; u < g1 && !flags[0]; ++u, ++wc) {
        const int ws = (int)(wc % kTcWStages);
        if (wc >= kTcWStages) wait(&wempty[ws], (uint32_t)(((wc / kTcWStages) - 1) & 1));
        if (flags[0]) break;
        const int r = (int)(u / p.NCH), c = (int)(u % p.NCH);
        mbar_arrive_expect_tx(&wfull[ws], 16384);
        tma_load_2d(smem + L::wstage + ws * 16384, &wmap, &wfull[ws], c * 128, r * kTcRows, pol);
      }
      if (flags[0]) {  // drain (bounded): every weight copy this thread may have in flight
        for (long long j = (wc > kTcWStages ? wc - kTcWStages : 0); j < wc; ++j)
          mbar_wait(&wfull[j % kTcWStages], (uint32_t)((j / kTcWStages) & 1));
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ activation producer --
    if (lane == 0) {
      prefetch_tensormap(&bmap);
      const uint64_t pol = l2_policy_evict_last();
      pdl_wait_prior_grid();  // the activations come from the previous kernel
      long long c_ = 0;
      for (long long u = g0; u < g1 && !flags[0]; ++u) {
        const int c = (int)(u % p.NCH);
        const int nkb = tc_chunk_kbs(p, c);
        for (int kb = 0; kb < nkb && !flags[0]; ++kb, ++c_) {
          const int s = (int)(c_ % kTcStages);
          if (c_ >= kTcStages) wait(&kempty[s], (uint32_t)(((c_ / kTcStages) - 1) & 1));
          if (flags[0]) break;
          mbar_arrive_expect_tx(&bfull[s], L::kBStage);
          tma_load_2d(smem + L::bstage + s * L::kBStage, &bmap, &bfull[s], (c * 8 + kb) * kTcKB, 0, pol);
        }
      }
      if (flags[0]) {
        for (long long j = (c_ > kTcStages ? c_ - kTcStages : 0); j < c_; ++j)
          mbar_wait(&bfull[j % kTcStages], (uint32_t)((j / kTcStages) & 1));
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = gemm_idesc(kTcRows, NT);
      const uint32_t bbase = smem_u32(smem + L::bstage);
      long long c_ = 0, seg = 0;
      bool first = true;
      for (long long u = g0; u < g1 && !flags[0]; ++u) {
        const int c = (int)(u % p.NCH);
        const int a = (int)(seg & 1);
        if (u == g0 || c == 0) {  // segment start
          if (seg >= 2) wait(&accempty[a], (uint32_t)(((seg >> 1) - 1) & 1));
          tc_fence_after();
          first = true;
        }
        const uint32_t d_tmem = tmem + (uint32_t)(a * NT);
        const int nkb = tc_chunk_kbs(p, c);
        for (int kb = 0; kb < nkb && !flags[0]; ++kb, ++c_) {
          const int s = (int)(c_ % kTcStages);
          const uint32_t par = (uint32_t)((c_ / kTcStages) & 1);
          wait(&bfull[s], par);
          wait(&afull[s], par);
          if (flags[0]) break;
          tc_fence_after();
          const uint64_t bdesc = smem_desc_sw128(bbase + s * L::kBStage);
          const uint32_t a_tmem = tmem + kTcACol + s * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ts(d_tmem, a_tmem + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, (first && kk == 0) ? 0u : 1u);
          first = false;
          tc_commit(&kempty[s]);
        }
        if (u == g1 - 1 || c == p.NCH - 1) {  // segment end
          tc_commit(&accfull[a]);
          ++seg;
        }
      }
      tc_commit(drain);  // completes once every MMA issued above has completed
      mbar_wait(drain, 0);
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // ---------------------------------------------------------- decoders --
    // tcgen05.st is warp-collective: the abort decision is made warp-uniform.
    const int dset = warp < 8 ? 0 : 1 + (warp - 12) / 4;
    const int quad = warp & 3, row = quad * 32 + lane;
    const uint32_t wbase = smem_u32(smem + L::wstage);
    long long c_ = 0, wc = 0;
    bool stop = false;
    for (long long u = g0; u < g1 && !stop; ++u, ++wc) {
      const int c = (int)(u % p.NCH);
      const int ws = (int)(wc % kTcWStages);
      wait(&wfull[ws], (uint32_t)((wc / kTcWStages) & 1));
      const int nkb = tc_chunk_kbs(p, c);
      for (int kb = 0; kb < nkb; ++kb, ++c_) {
        if ((int)(c_ % kTcDecSets) != dset) continue;  // another set decodes this block
        const int s = (int)(c_ % kTcStages);
        if (c_ >= kTcStages) wait(&kempty[s], (uint32_t)(((c_ / kTcStages) - 1) & 1));
        if (__any_sync(0xffffffffu, flags[0])) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint4 v = lds_u128(wbase + ws * 16384 + row * 128 + (((kb ^ (row & 7)) & 7) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t hs = w[q] >> 12;
#pragma unroll
          for (int i = 0; i < 6; ++i) h[8 * q + i] = w[q] & (0x00030003u << (2 * i));
          h[8 * q + 6] = hs & 0x00030003u;
          h[8 * q + 7] = hs & 0x000C000Cu;
        }
        tmem_st_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + kTcACol + s * 32, h);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[s]);
      }
      __syncwarp();
      if (lane == 0 && !stop) mbar_arrive(&wempty[ws]);
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------- epilogue --
    pdl_wait_prior_grid();  // xsum / fscale come from the previous kernel
    const int quad = warp & 3, row = quad * 32 + lane;
    const int etid = threadIdx.x - 8 * 32;  // 0..127
    long long seg = 0, u = g0;
    while (u < g1) {
      const int r = (int)(u / p.NCH);
      const int c0 = (int)(u % p.NCH);
      const long long tile_end = (long long)(r + 1) * p.NCH;
      const long long u_end = tile_end < g1 ? tile_end : g1;  // segment = units [u, u_end)
      const int nch = (int)(u_end - u);
      const bool whole = (c0 == 0) && (nch == p.NCH);
      const int a = (int)(seg & 1);
      wait(&accfull[a], (uint32_t)((seg >> 1) & 1));
      // The four epilogue warps share named barriers, so they take the abort
      // decision together, from one snapshot of the flag.
      named_barrier_sync(kTcEpiBar, 128);
      if (etid == 0) flags[2] = flags[0];
      named_barrier_sync(kTcEpiBar, 128);
      if (flags[2]) break;
      tc_fence_after();
      const int64_t n = (int64_t)r * kTcRows + row;
      // D * 2^24 is the exact integer sum of code * x over the segment.
#pragma unroll 1
      for (int cb = 0; cb < NT / 16 && cb * 16 < p.M; ++cb) {
        uint32_t t[16];
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * NT + cb * 16), t);
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = cb * 16 + j;
            if (tok < p.M) {
              const int32_t v = __float2int_rn(__uint_as_float(t[j]) * 16777216.0f);
              if (whole) {
                const int32_t o = v - __ldg(p.xsum + tok);
                if (p.acc) p.acc[(int64_t)tok * p.N + n] = o;
                p.y[(int64_t)tok * p.N + n] = __fmul_rn((float)o, __ldg(p.fscale + tok));
              } else if (v != 0) {
                atomicAdd(&p.ws_partial[n * p.M + tok], v);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[a]);
      if (!whole) {
        __threadfence();  // partial sums visible before the ticket
        named_barrier_sync(kTcEpiBar, 128);
        if (etid == 0) {
          const unsigned old = atomicAdd(&p.ws_ticket[r], (unsigned)nch);
          flags[1] = (old + (unsigned)nch == (unsigned)p.NCH) ? 1 : 0;
        }
        named_barrier_sync(kTcEpiBar, 128);
        if (flags[1]) {
          __threadfence();
          if (n < p.N) {
#pragma unroll 4
            for (int j = 0; j < p.M; ++j) {
              const int32_t o = atomicExch(&p.ws_partial[n * p.M + j], 0) - __ldg(p.xsum + j);
              if (p.acc) p.acc[(int64_t)j * p.N + n] = o;
              p.y[(int64_t)j * p.N + n] = __fmul_rn((float)o, __ldg(p.fscale + j));
            }
          }
          if (etid == 0) atomicExch(&p.ws_ticket[r], 0u);
        }
        named_barrier_sync(kTcEpiBar, 128);
      }
      u = u_end;
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace bitnet

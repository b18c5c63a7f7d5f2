// Decode GEMV for one or two tokens: warp-private bulk-copy streams.
//
// Same operation as the other GEMV kernels (BitNet 深度拆解 §3.1 integer-
// domain product, §1 ternary products, §2.3 dequantisation).  This is the
// decode kernel for rows of up to 8192 (one token) or 4096 (two tokens)
// weights, organised so that nothing serialises the weight stream:
//   * Every warp owns a contiguous range of whole rows, i.e. a contiguous
//     byte range of the packed matrix, and streams it through a private ring
//     of up to two 8 KB shared-memory stages (sized to the rows the warp
//     owns, so small matrices leave the SM's shared memory free) with 1D bulk
//     copies (cp.async.bulk): up to 192 KB in flight per SM, no coupling
//     between warps, no barrier but the warp's own stage barriers.  The first
//     stage is requested before waiting on the previous kernel, since the
//     weights do not depend on it, the others once the warp has read the
//     activations (a full ring ahead of those reads delays them).  Lane l
//     reads the 16-byte chunks l, l+32, ... of each row from the stage
//     (consecutive lanes, consecutive addresses: conflict-free).
//   * Because a lane always sees the same K chunks, its activation words live
//     in registers for the whole kernel: for 16-K group q, word s holds bytes
//     x_q[16q + 4b + s], b = 0..3, so masking a packed word with
//     0x03030303 << 2s and dp4a against word s gives 4^s * sum code * x
//     (2 integer operations per packed byte per token).
//   * The plain form takes the rows of a stage four at a time, with an
//     independent dp4a chain per row, and combines the four rows' 32 lane
//     sums in one transpose-reduce (6 shuffles instead of 20); the lane that
//     ends with a row's total subtracts token m's sum of x_q and applies the
//     fused dequantisation.  The other forms combine a row's lane sums with
//     five shuffles each.
//   * The activations are prefetched into L2 (one bulk prefetch) before the
//     weight stream is requested, so that the prologue's reads of x do not
//     queue behind the weights.
//   * Fused form (XT = float / bf16): the CTA quantises x itself in its
//     prologue (absmax, then clamp(rint(x / s * 127)), the operations of
//     quant_act_kernel, on 8-element halves of 16-K groups spread over all
//     threads), so one kernel runs the whole BitLinear.  The activation words
//     sit in shared memory in a lane-consecutive order before the lanes load
//     theirs.
//   * SwiGLU form (SW): the front half of the BitTransformer feed-forward of
//     BitNet 深度拆解 §3.1, silu(gate(h)) * up(h).  A stage holds gate rows
//     and the up rows of the same indices (two bulk copies); both sums are
//     formed together and lane m writes silu(y_gate) * y_up, each y exactly
//     as the GEMV epilogue forms it.
//   * Grouped form (GR): group-wise weight scales (BitNet 深度拆解 §4.3: each
//     group of G consecutive weights of a row has its own scale; G = K is a
//     per-channel scale).  A stage also carries its rows' scales (cp.async,
//     4 bytes each, by all lanes); the per-group Σ x_q come from the
//     prologue.  With P = G / 64 chunks per group and P <= 4 a lane owns
//     whole groups: its chunk slots hold the P chunks of groups lane,
//     lane + 32, ... (the order inside a group rotated per lane so that the
//     warp's 16-byte reads hit distinct bank groups), it sums a group in
//     registers and adds acc_g * scale_g into an fp32 partial.  For larger P
//     (G <= 2048) aligned runs of P lanes add their chunk sums by shuffles
//     and the run's first lane adds the term.  The warp then adds the
//     partials and lane m writes F * (s_m / 127).  With one group per row the
//     row sum is taken whole.
#pragma once

#include "common.cuh"
#include "gemv_rows.cuh"
#include "quant_act.cuh"
#include "swiglu.cuh"

namespace bitnet {

#ifndef BITNET_LDG_WARPS
#define BITNET_LDG_WARPS 12
#endif
constexpr int kLdgWarps = BITNET_LDG_WARPS;
constexpr int kLdgThreads = kLdgWarps * 32;
#ifndef BITNET_LDG_STAGE_BYTES
#define BITNET_LDG_STAGE_BYTES 8192
#endif
// Largest stage and ring per warp; a launch sizes its ring to the rows its
// warps own (p.RS bytes x p.NS stages), so that small matrices leave room on
// the SM for the next kernel's CTAs (programmatic dependent launch).
constexpr int kLdgStageBytes = BITNET_LDG_STAGE_BYTES;  // per warp stage: whole rows
#ifndef BITNET_LDG_RING_BYTES
#define BITNET_LDG_RING_BYTES 16384
#endif
constexpr int kLdgStages = BITNET_LDG_RING_BYTES / kLdgStageBytes;  // stages per warp ring
// Fused prologue: each thread keeps up to kLdgGroups 16-element activation
// groups in registers between the absmax and the quantisation (one read of
// x); the host only sends shapes with M * K / 16 <= kLdgGroups * kLdgThreads.
constexpr int kLdgGroups = 2;
// Rows of a stage the plain form reduces together (the transpose-reduce is
// written for four).
constexpr int kLdgBatch = 4;

constexpr int kLdgPlain = 0, kLdgSwiGLU = 1, kLdgGrouped = 2;  // kernel forms

struct GemvLdgParams {
  const uint8_t *packed;
  const int8_t *xq;   // int8 activations (XT = int8_t)
  const void *x;      // bf16 / fp32 activations (fused forms)
  int8_t *xq_out;     // fused forms, optional (CTA 0)
  float *scale_out;   // fused forms, optional (CTA 0)
  const float *scale;
  const float *w_scale;  // grouped form: [N, NG] group scales
  float *y;
  int32_t *acc;          // grouped form: [M, N, NG] per-group products
  const uint8_t *packed_up;  // SwiGLU form: the up rows (gate rows in `packed`)
  const float *w_scale_up;
  int32_t *acc_up;
  int64_t N, K;  // N: rows (SwiGLU: rows of each of gate and up)
  int M;
  int C;   // 16-byte chunks per packed row (K / 64)
  int SR;  // rows (SwiGLU: row pairs) per stage, SR * K / 4 (x2) <= kLdgStageBytes
  int RS;  // bytes per stage (SR rows, a multiple of 16)
  int NS;  // stages per warp (<= kLdgStages)
  int G, NG, P;  // grouped form: group size, groups per row, 16-byte chunks per group
  int GS, PS;    // log2 G and log2 P (G a power of two), or 31 / 0 with one group per row
  int LOCAL;     // grouped form, P <= 4: each lane owns whole groups (see gemv_ldg_kernel)
};

// 4-byte asynchronous copy global -> shared (per-thread completion groups).
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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
// the stage barriers, then (grouped form) per-group sums [MT][NG].
struct GemvLdgSmem {
  int ring, xw, xsum, fscale, redf, bars, xsumg, bytes;
};
__host__ __device__ inline GemvLdgSmem gemv_ldg_smem_layout(int MT, int C, int RS, int NS, int NG) {
  GemvLdgSmem L;
  L.ring = 0;
  L.xw = kLdgWarps * NS * RS;
  L.xsum = L.xw + MT * C * 64;
  L.fscale = L.xsum + 32;
  L.redf = L.fscale + 32;
  L.bars = (L.redf + kLdgWarps * MT * 4 + 16 + 15) & ~15;  // mbarriers: 8-byte aligned
  L.xsumg = L.bars + kLdgWarps * kLdgStages * 8;
  L.bytes = L.xsumg + MT * NG * 4;
  return L;
}

template <int MT, int J, typename XT, int FORM>
__global__ void __launch_bounds__(kLdgThreads, 1) gemv_ldg_kernel(const GemvLdgParams p) {
  constexpr bool SW = FORM == kLdgSwiGLU, GR = FORM == kLdgGrouped;
  extern __shared__ __align__(128) uint8_t lsm[];
  const GemvLdgSmem L = gemv_ldg_smem_layout(MT, p.C, p.RS, p.NS, GR ? p.NG : 0);
  const int NS = p.NS;
  int32_t *xsumg = reinterpret_cast<int32_t *>(lsm + L.xsumg);  // [MT][NG]
  uint8_t *xw = lsm + L.xw;                                     // [MT][C*64]
  int32_t *xsum = reinterpret_cast<int32_t *>(lsm + L.xsum);    // [MT]
  float *fscale = reinterpret_cast<float *>(lsm + L.fscale);    // [MT]
  float *redf = reinterpret_cast<float *>(lsm + L.redf);        // [warps][MT]
  uint64_t *bars = reinterpret_cast<uint64_t *>(lsm + L.bars);  // [warps][stages]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  // rows [N * gw / nw, N * (gw + 1) / nw) of the matrix, formed in 32-bit
  // arithmetic (N < 2^31, nw <= 2^16): N = qn * nw + rn, so N * gw / nw =
  // qn * gw + rn * gw / nw with rn * gw < nw^2 < 2^32
  const unsigned gw = blockIdx.x * kLdgWarps + warp, nw = gridDim.x * kLdgWarps;
  const unsigned qn = (unsigned)p.N / nw, rn = (unsigned)p.N % nw;
  const int64_t r0 = (int64_t)qn * gw + rn * gw / nw;
  const int64_t r1 = (int64_t)qn * (gw + 1) + rn * (gw + 1) / nw;
  const int64_t rowb = p.K / 4;
  const int nst = ((int)(r1 - r0) + p.SR - 1) / p.SR;  // this warp's stages
  // Stage st holds rows [stage_row(st), stage_row(st + 1)): the first stage
  // takes the remainder (1..SR rows), the others SR each, so that a warp
  // with one row more than its neighbours requests that row first instead
  // of waiting a whole round trip for it at the end of the launch.
  const int first_less = (int)(r1 - r0) - nst * p.SR;  // first stage's rows - SR (<= 0)
  auto stage_row = [&](int st) -> int64_t { return r0 + max(0, first_less + st * p.SR); };
  // ring slot of stage st and the parity of its use of that slot (NS is 1 or
  // 2: no division)
  static_assert(kLdgStages <= 2, "slot_of / use_of assume at most two stages per warp");
  auto slot_of = [&](int st) { return NS == 2 ? (st & 1) : 0; };
  auto use_of = [&](int st) { return (uint32_t)((NS == 2 ? st >> 1 : st) & 1); };
  uint8_t *ring = lsm + L.ring + (size_t)warp * NS * p.RS;
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
    const int64_t ra = stage_row(st);
    const int64_t rbn = stage_row(st + 1);
    const uint32_t bytes = (uint32_t)((rbn - ra) * rowb);
    uint64_t *bar = &wbar[slot_of(st)];
    uint8_t *dst = ring + slot_of(st) * p.RS;
    mbar_arrive_expect_tx(bar, SW ? 2 * bytes : bytes);
    bulk_load(dst, p.packed + ra * rowb, bytes, bar, policy);
    if (SW) bulk_load(dst + bytes, p.packed_up + ra * rowb, bytes, bar, policy);
  };
  // grouped form: every lane copies part of the stage's scales [rows][NG]
  // behind its packed rows, and commits one group per stage
  int issued_s = 0;
  auto issue_scales = [&](int st) {
    ++issued_s;
    const int64_t ra = stage_row(st);
    const int nr = (int)(stage_row(st + 1) - ra);
    float *dst = reinterpret_cast<float *>(ring + slot_of(st) * p.RS + (size_t)nr * rowb);
    const float *src = p.w_scale + ra * p.NG;
    for (int e = lane; e < nr * p.NG; e += 32) cp_async4(dst + e, src + e);
    cp_async_commit();
  };
  // The activations go to L2 ahead of the weight stream.  A prefetch is only
  // a hint (L2 stays coherent with the previous kernel's writes), so it may
  // be issued before waiting on that kernel; the reads of x come after.
  if (tid == 0) {
    const void *xs = std::is_same<XT, int8_t>::value ? static_cast<const void *>(p.xq) : p.x;
    const uint32_t xb = (uint32_t)((int64_t)p.M * p.K * sizeof(XT));
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(xs), "r"(xb) : "memory");
  }
  // Only the first stage goes out before the activations are read: a full
  // ring (192 KB per SM) ahead of them would hold their loads back by the
  // time it takes HBM to deliver it.  The other stages follow once this
  // warp's reads of x (x_q) have returned.
  if (lane == 0) {
    policy = l2_policy_evict_first();
    if (nst > 0) issue(0);
  }
  auto issue_rest = [&]() {
    if (lane == 0)
      for (int st = issued; st < nst && st < NS; ++st) issue(st);
  };
  if (GR)
    for (int st = 0; st < nst && st < NS; ++st) issue_scales(st);

  pdl_wait_prior_grid();
  // ---------------------------------------------- activation words (smem) --
  if (tid < MT) xsum[tid] = 0;
  if (GR)
    for (int i = tid; i < MT * p.NG; i += kLdgThreads) xsumg[i] = 0;
  if constexpr (std::is_same<XT, int8_t>::value) {
    if (tid < MT) {
      // grouped form: the token factor s / 127 (the weight scales are per group)
      fscale[tid] = GR ? __fdiv_rn(__ldg(p.scale + tid), 127.0f)
                       : __fdiv_rn(__fmul_rn(__ldg(p.w_scale), __ldg(p.scale + tid)), 127.0f);
      if (SW) fscale[MT + tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale_up), __ldg(p.scale + tid)), 127.0f);
    }
  }
  __syncthreads();
  const int groups = p.C * 4;  // 16-K groups per token
  // Activation words of 16-K group q = 4 c + u (chunk c): word s holds the
  // bytes x_q[16 q + 4 b + s], b = 0..3; the four words sit at granule
  // u * C + c of the token's area, so that the lanes' 16-byte reads of one u
  // (chunks lane + 32 j) are consecutive granules.
  auto xw_group = [&](int m, int q) { return xw + (size_t)m * p.C * 64 + ((size_t)(q & 3) * p.C + (q >> 2)) * 16; };
  {
    float s[MT], cq[MT];
    // fused forms: each thread quantises 8-element halves of 16-K groups
    // (up to kLdgGroups * 2 of them, kept in registers from the absmax on)
    float f[2 * kLdgGroups][8];
    if constexpr (!std::is_same<XT, int8_t>::value) {
      const XT *x = static_cast<const XT *>(p.x);
      float amax[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) amax[m] = 0.0f;
#pragma unroll
      for (int n = 0; n < 2 * kLdgGroups; ++n) {
        const int i = tid + n * kLdgThreads;
        if (i < MT * groups * 2) {
          const int m = MT == 1 ? 0 : i / (2 * groups), h = MT == 1 ? i : i % (2 * groups);
          load8(x + (int64_t)m * p.K + (int64_t)h * 8, f[n]);
          float a = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[n][e]));
#pragma unroll
          for (int mm = 0; mm < MT; ++mm)
            if (mm == m) amax[mm] = fmaxf(amax[mm], a);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a = amax[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0) redf[warp * MT + m] = a;
      }
      issue_rest();
      __syncthreads();
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a = redf[m];
        for (int ww = 1; ww < kLdgWarps; ++ww) a = fmaxf(a, redf[ww * MT + m]);
        s[m] = a < 1e-8f ? 1e-8f : a;
        cq[m] = quant_factor(s[m]);
      }
      if (tid < MT) {
        fscale[tid] = GR ? __fdiv_rn(s[tid], 127.0f) : __fdiv_rn(__fmul_rn(__ldg(p.w_scale), s[tid]), 127.0f);
        if (SW) fscale[MT + tid] = __fdiv_rn(__fmul_rn(__ldg(p.w_scale_up), s[tid]), 127.0f);
        if (blockIdx.x == 0 && p.scale_out) p.scale_out[tid] = s[tid];
      }
    }
    int part[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m] = 0;
    if constexpr (std::is_same<XT, int8_t>::value) {
      for (int i = tid; i < MT * groups; i += kLdgThreads) {
        const int m = MT == 1 ? 0 : i / groups, q = MT == 1 ? i : i % groups;
        int8_t v[16];
        const int4 u = *reinterpret_cast<const int4 *>(p.xq + (int64_t)m * p.K + (int64_t)q * 16);
        memcpy(v, &u, 16);
        const int sum = rows_pack_group(v, xw_group(m, q));
        if (GR && sum) atomicAdd(&xsumg[m * p.NG + ((q * 16) >> p.GS)], sum);
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
          if (mm == m) part[mm] += sum;
      }
      issue_rest();
    } else {
#pragma unroll
      for (int n = 0; n < 2 * kLdgGroups; ++n) {
        const int i = tid + n * kLdgThreads;
        if (i < MT * groups * 2) {
          const int m = MT == 1 ? 0 : i / (2 * groups), h = MT == 1 ? i : i % (2 * groups);
          const int q = h >> 1, half = h & 1;
          float sm = s[0], cm = cq[0];
#pragma unroll
          for (int mm = 1; mm < MT; ++mm)
            if (mm == m) {
              sm = s[mm];
              cm = cq[mm];
            }
          int8_t v[8];
          quantize_fast(f[n], sm, cm, v);
          int sum = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) sum += v[e];
          if (blockIdx.x == 0 && p.xq_out) {
            uint2 u;
            memcpy(&u, v, 8);
            *reinterpret_cast<uint2 *>(p.xq_out + (int64_t)m * p.K + (int64_t)h * 8) = u;
          }
          // this half holds b = 2 half, 2 half + 1 of the group: bytes 2 half
          // and 2 half + 1 of each of the four words
          uint16_t *w16 = reinterpret_cast<uint16_t *>(xw_group(m, q)) + half;
#pragma unroll
          for (int t = 0; t < 4; ++t) w16[2 * t] = (uint16_t)((uint8_t)v[t] | ((uint32_t)(uint8_t)v[4 + t] << 8));
          if (GR && sum) atomicAdd(&xsumg[m * p.NG + ((q * 16) >> p.GS)], sum);
#pragma unroll
          for (int mm = 0; mm < MT; ++mm)
            if (mm == m) part[mm] += sum;
        }
      }
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

  // the chunk of each of this lane's slots: lane + 32 j, or with lane-local
  // groups chunk P q + ((j % P + rot) % P) of group q = lane + 32 (j / P)
  const bool local = GR && p.LOCAL;
  int cj[J];
  {
    const int rot = local ? ((lane >> (3 - p.PS)) & (p.P - 1)) : 0;
#pragma unroll
    for (int j = 0; j < J; ++j)
      cj[j] = local ? p.P * (lane + 32 * (j >> p.PS)) + (((j & (p.P - 1)) + rot) & (p.P - 1)) : lane + 32 * j;
  }
  // this lane's activation words, for its chunks
  uint32_t xr[MT][J][16];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = cj[j];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c < p.C) v = *reinterpret_cast<const uint4 *>(xw_group(m, 4 * c + g));
        xr[m][j][4 * g + 0] = v.x;
        xr[m][j][4 * g + 1] = v.y;
        xr[m][j][4 * g + 2] = v.z;
        xr[m][j][4 * g + 3] = v.w;
      }
    }
  int32_t xs[MT];
  float fs[MT], fsu[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    xs[m] = xsum[m];
    fs[m] = fscale[m];
    fsu[m] = SW ? fscale[MT + m] : 0.0f;
  }

  // sum over the packed row at `row` (shared memory) of code * x, per token,
  // combined over the warp: every lane ends with the totals
  auto row_sums = [&](const uint8_t *row, int (&v)[MT]) {
    int a[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int s = 0; s < 4; ++s) a[m][s] = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lane + 32 * j;
      uint4 wq = make_uint4(0u, 0u, 0u, 0u);
      if (c < p.C) wq = lds_u128(smem_u32(row + (size_t)c * 16));
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
      int t = a[m][0] + (a[m][1] >> 2) + (a[m][2] >> 4) + (a[m][3] >> 6);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      v[m] = t;
    }
  };

  // Plain form: kLdgBatch rows of a stage at once (rows b .. b + 3 of the
  // stage at `stage`, those below nr), with independent dp4a chains per row,
  // then one transpose-reduce over the warp: the lanes trade halves of the
  // four row sums (xor 16, then xor 8) and finish with three butterfly
  // steps, 6 shuffles for four rows instead of 20.  Lane group g = lane / 8
  // ends with the totals of row b + g; lane 8 g + m writes token m's output.
  auto rows_batch = [&](const uint8_t *stage, int b, int nr, int64_t ra) {
    int a[kLdgBatch][MT][4];
#pragma unroll
    for (int r = 0; r < kLdgBatch; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int s = 0; s < 4; ++s) a[r][m][s] = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lane + 32 * j;
      // the four rows' chunks first (rows past the stage's end read as zero),
      // then each field of each word for all four rows in turn, so that
      // consecutive dp4a feed different accumulators
      uint32_t wv[kLdgBatch][4];
#pragma unroll
      for (int r = 0; r < kLdgBatch; ++r) {
        uint4 wq = make_uint4(0u, 0u, 0u, 0u);
        if (b + r < nr && c < p.C) wq = lds_u128(smem_u32(stage + (size_t)(b + r) * rowb + (size_t)c * 16));
        wv[r][0] = wq.x;
        wv[r][1] = wq.y;
        wv[r][2] = wq.z;
        wv[r][3] = wq.w;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int sf = 0; sf < 4; ++sf) {
          uint32_t f[kLdgBatch];
#pragma unroll
          for (int r = 0; r < kLdgBatch; ++r) f[r] = wv[r][u] & (0x03030303u << (2 * sf));
#pragma unroll
          for (int r = 0; r < kLdgBatch; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) a[r][m][sf] = dp4a_u8s8(f[r], xr[m][j][4 * u + sf], a[r][m][sf]);
        }
    }
    const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
    const int g = (lane >> 3) & 3;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int v[kLdgBatch];
#pragma unroll
      for (int r = 0; r < kLdgBatch; ++r) v[r] = a[r][m][0] + (a[r][m][1] >> 2) + (a[r][m][2] >> 4) + (a[r][m][3] >> 6);
      // xor 16: lanes 0-15 keep rows 0, 1; lanes 16-31 rows 2, 3
      int k0 = h16 ? v[2] : v[0], k1 = h16 ? v[3] : v[1];
      k0 += __shfl_xor_sync(0xffffffffu, h16 ? v[0] : v[2], 16);
      k1 += __shfl_xor_sync(0xffffffffu, h16 ? v[1] : v[3], 16);
      // xor 8: lanes with bit 3 clear keep the even row of their pair
      int k = h8 ? k1 : k0;
      k += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
      k += __shfl_xor_sync(0xffffffffu, k, 4);
      k += __shfl_xor_sync(0xffffffffu, k, 2);
      k += __shfl_xor_sync(0xffffffffu, k, 1);
      if ((lane & 7) == m && b + g < nr) {
        const int64_t r = ra + b + g;
        const int32_t o = k - xs[m];
        if (p.acc) p.acc[(int64_t)m * p.N + r] = o;
        p.y[(int64_t)m * p.N + r] = __fmul_rn((float)o, fs[m]);
      }
    }
  };

  // grouped form: the fp32 sum over the row's groups of acc_g * scale_g, per
  // token (every lane ends with the totals).  `sc` holds the row's NG scales;
  // with `accg` non-null the per-group products go to accg[(m * N + r) * NG + g].
  // per lane and chunk column j: its group, whether it leads the run of P
  // lanes, and the group's sum of x_q (constant over rows)
  int gj[J];
  int32_t xsg[MT][J];
  const bool lead = GR && (lane & (p.P - 1)) == 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    gj[j] = !GR ? 0 : (local ? lane + 32 * (j >> p.PS) : (lane + 32 * j) >> p.PS);
#pragma unroll
    for (int m = 0; m < MT; ++m) xsg[m][j] = (GR && gj[j] < p.NG) ? xsumg[m * p.NG + gj[j]] : 0;
  }
  auto row_grouped = [&](const uint8_t *row, const float *sc, int64_t r, float (&F)[MT]) {
    float f[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) f[m] = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lane + 32 * j;
      uint4 wq = make_uint4(0u, 0u, 0u, 0u);
      if (c < p.C) wq = lds_u128(smem_u32(row + (size_t)c * 16));
      const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
      int a[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int s = 0; s < 4; ++s) a[m][s] = 0;
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
      // this chunk's sum of code * x, then the run of P lanes of its group
      const int g = gj[j];
      const bool head = lead && c < p.C;
      const float w = head ? sc[g] : 0.0f;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        int t = a[m][0] + (a[m][1] >> 2) + (a[m][2] >> 4) + (a[m][3] >> 6);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
          if (o < p.P) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (head) {
          const int32_t ag = t - xsg[m][j];
          if (p.acc) p.acc[((int64_t)m * p.N + r) * p.NG + g] = ag;
          f[m] = __fmaf_rn((float)ag, w, f[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = f[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
      F[m] = v;
    }
  };

  // lane-local groups: the same sum with each group finished in registers
  auto row_local = [&](const uint8_t *row, const float *sc, int64_t r, float (&F)[MT]) {
    float f[MT];
    int a[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      f[m] = 0.0f;
#pragma unroll
      for (int s = 0; s < 4; ++s) a[m][s] = 0;
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = cj[j];
      uint4 wq = make_uint4(0u, 0u, 0u, 0u);
      if (c < p.C) wq = lds_u128(smem_u32(row + (size_t)c * 16));
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
      if ((j & (p.P - 1)) == p.P - 1) {  // the group's last chunk
        const int g = gj[j];
        if (g < p.NG) {
          const float w = sc[g];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int32_t ag = a[m][0] + (a[m][1] >> 2) + (a[m][2] >> 4) + (a[m][3] >> 6) - xsg[m][j];
            if (p.acc) p.acc[((int64_t)m * p.N + r) * p.NG + g] = ag;
            f[m] = __fmaf_rn((float)ag, w, f[m]);
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int s = 0; s < 4; ++s) a[m][s] = 0;
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = f[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
      F[m] = v;
    }
  };

  // ------------------------------------------------------------ main loop --
  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    const int slot = slot_of(st);
    if (ok && !mbar_wait(&wbar[slot], use_of(st))) {
      raise_device_error(kDevErrTimeout);
      ok = false;  // keep walking (results undefined, the error word says so)
    }
    const uint8_t *stage = ring + slot * p.RS;
    const int64_t ra = stage_row(st);
    const int nr = (int)(stage_row(st + 1) - ra);
    if (GR) {
      // this lane's scale copies of the stage are done; then everyone's
      if (issued_s > st + 1) cp_async_wait<1>();
      else cp_async_wait<0>();
      __syncwarp();
    }
    if constexpr (FORM == kLdgPlain) {
      for (int b = 0; b < nr; b += kLdgBatch) rows_batch(stage, b, nr, ra);
    } else
    for (int i = 0; i < nr; ++i) {
      const int64_t r = ra + i;
      if constexpr (GR) {
        const float *sc = reinterpret_cast<const float *>(stage + (size_t)nr * rowb) + (size_t)i * p.NG;
        if (p.NG == 1) {
          // one group per row: the whole-row sum, scaled once
          int v[MT];
          row_sums(stage + (size_t)i * rowb, v);
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (lane == m) {
              const int32_t ag = v[m] - xsumg[m];
              if (p.acc) p.acc[(int64_t)m * p.N + r] = ag;
              p.y[(int64_t)m * p.N + r] = __fmul_rn(__fmul_rn((float)ag, sc[0]), fs[m]);
            }
        } else {
          float F[MT];
          if (local) row_local(stage + (size_t)i * rowb, sc, r, F);
          else row_grouped(stage + (size_t)i * rowb, sc, r, F);
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (lane == m) p.y[(int64_t)m * p.N + r] = __fmul_rn(F[m], fs[m]);
        }
        continue;
      }
      int v[MT];
      row_sums(stage + (size_t)i * rowb, v);
      if constexpr (SW) {
        int vu[MT];
        row_sums(stage + (size_t)(nr + i) * rowb, vu);
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (lane == m) {
            const int32_t og = v[m] - xs[m], ou = vu[m] - xs[m];
            if (p.acc) p.acc[(int64_t)m * p.N + r] = og;
            if (p.acc_up) p.acc_up[(int64_t)m * p.N + r] = ou;
            p.y[(int64_t)m * p.N + r] = silu_mul(__fmul_rn((float)og, fs[m]), __fmul_rn((float)ou, fsu[m]));
          }
      } else {
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (lane == m) {
            const int32_t o = v[m] - xs[m];
            if (p.acc) p.acc[(int64_t)m * p.N + r] = o;
            p.y[(int64_t)m * p.N + r] = __fmul_rn((float)o, fs[m]);
          }
      }
    }
    // every lane's reads of this stage are done: refill it
    __syncwarp();
    if (lane == 0 && ok && st + NS < nst) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(st + NS);
    }
    if (GR && ok && st + NS < nst) issue_scales(st + NS);
  }
  // After a timeout leave no bulk copy in flight (bounded waits on the
  // stages this lane requested last).
  if (!ok && lane == 0) {
    for (int st = (issued > NS ? issued - NS : 0); st < issued; ++st)
      mbar_wait(&wbar[slot_of(st)], use_of(st));
  }
  if (GR) cp_async_wait<0>();
}

}  // namespace bitnet

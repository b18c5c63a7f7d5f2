// Prefill-path W2A8 ternary GEMM on the tcgen05 tensor cores.
//
// y[m, n] = (sum_k (code[n,k]-1) * x_q[m,k]) * (w_scale * s_m / 127): the
// integer-domain matmul of BitNet 深度拆解 §3.1 with the dequantisation of
// §2.3, for many tokens at once (the prefill counterpart of the decode GEMV).
//
// D (weight rows x tokens) = A (weight rows x K) * B (tokens x K)^T, one
// 128 x 128 tile per CTA iteration, kind::f16 MMA with fp32 accumulators in
// tensor memory:
//   * A comes from TMEM.  Decoder warps read the packed codes (TMA, 128-byte
//     swizzle) and turn each 2-bit field, masked in place inside a 16-bit
//     lane, into an fp16 subnormal code * 4^i * 2^-24; tcgen05.st writes them
//     straight into TMEM, so decoded weights never occupy shared memory.
//   * B is the activation matrix prepared once per call by gemm_prep_kernel:
//     x_q as fp16, scaled by 4^-i to match the weight encoding, in the same
//     K order as the decoded weights.  TMA loads 128 x 64 tiles with 128-byte
//     swizzle (the canonical K-major UMMA layout).
//   * Every product is code * x * 2^-24 and every partial sum an integer
//     multiple of 2^-24 below 2^22 * 2^-24, so fp32 accumulation is exact and
//     D * 2^24 - sum_k x_q is the exact integer accumulator.
//   * With 128-token tiles two accumulators (2 x 128 TMEM columns) let the
//     epilogue of one tile overlap the MMAs of the next; with the default
//     256-token tiles one accumulator of 256 columns fits beside the A
//     buffers, and the MMAs of the next tile wait for the epilogue.
//   * When the tiles leave a last wave less than half full, those tail tiles
//     are split by K across all CTAs (stream-K on the tail): after its whole
//     tiles each CTA takes an equal run of (tail tile, 64-K block) units; the
//     partial sums are added as exact int32 (D * 2^24) into the workspace,
//     and the epilogue warp whose ticket completes a 32-row x (tokens / 4)
//     block writes its outputs and re-zeroes the partials.
// Warp roles: 0 TMA producer, 1 TMEM owner + MMA issuer, 4-7 decoders (set
// 0), 8-11 epilogue, 12-15 ... further decoder sets.  Decoder set d takes
// the K-blocks c with c % kGemmDecSets == d, so several blocks are in
// flight per TMEM lane quarter while each warp waits for its tcgen05.st.  Every wait is bounded (kWaitLimitNs); on expiry the CTA
// records the error, stops issuing work, drains what it issued, frees TMEM
// and exits.
#pragma once

#include "common.cuh"
#include "quant_act.cuh"
#include "rmsnorm.cuh"

namespace bitnet {

#ifndef BITNET_GEMM_DEC_SETS
#define BITNET_GEMM_DEC_SETS 2
#endif
#ifndef BITNET_GEMM_STAGES
#define BITNET_GEMM_STAGES 4
#endif
constexpr int kGemmDecSets = BITNET_GEMM_DEC_SETS;  // decoder warp sets of 4 warps
// Epilogue: sets of four warps (one per TMEM lane quarter each), each set
// taking an equal share of the accumulator's 32-token column blocks.
#ifndef BITNET_GEMM_EPI_SETS
#define BITNET_GEMM_EPI_SETS 4
#endif
constexpr int kGemmEpiSets = BITNET_GEMM_EPI_SETS;
constexpr int kGemmEpiWarp2 = 12 + (kGemmDecSets - 1) * 4;  // first warp of epilogue set 1
constexpr int kGemmThreads = 384 + (kGemmDecSets - 1) * 128 + (kGemmEpiSets - 1) * 128;
constexpr int kGemmRows = 128;   // weight rows per tile (MMA M)
#ifndef BITNET_GEMM_TOK
#define BITNET_GEMM_TOK 256
#endif
constexpr int kGemmTok = BITNET_GEMM_TOK;  // tokens per tile (MMA N): 128 or 256
// Accumulator buffers in TMEM: two (the epilogue of one tile overlaps the
// MMAs of the next) when they fit beside the A buffers, else one.
constexpr int kGemmAccBufs = kGemmTok <= 128 ? 2 : 1;
constexpr int kGemmKB = 64;      // K per pipeline step (4 MMAs of K = 16)
constexpr int kGemmStages = BITNET_GEMM_STAGES;  // B stages in smem == A buffers in TMEM (<= 8)
static_assert(kGemmStages <= 8, "A buffers must fit beside the accumulators in TMEM");
constexpr int kGemmBStageBytes = kGemmTok * 128;
constexpr int kGemmWStages = 2;  // packed-weight stages (128 rows x 512 K)
constexpr int kGemmWStageBytes = kGemmRows * 128;
constexpr int kGemmTmemCols = 512;
constexpr int kGemmAccCol = 0;   // accumulators: columns [0, kGemmAccBufs * kGemmTok)
constexpr int kGemmACol = 256;   // A buffers: columns [256, 256 + stages * 32)

struct GemmParams {
  float *y;
  int32_t *acc;
  const int32_t *xsum;  // [M]
  const float *fscale;  // [M] = w_scale * s_m / 127
  int64_t M, N, K;
  int NRT, NTT, NKB;
  long long tiles;
  long long full_tiles;  // tiles [0, full_tiles) are taken whole, round robin
  int32_t *ws_part;      // split tail tiles: [tail][tokens][128 rows] int32, zero on entry and exit
  unsigned *ws_ticket;   // [tail][16] K-blocks done per epilogue block, zero on entry and exit
};

// One run of K-blocks [kb0, kb1) of tile t.
struct GemmSeg {
  long long t;
  int kb0, kb1;
};

// The segments of this CTA, in order: whole tiles blockIdx.x, + gridDim.x, ...
// below full_tiles; then its equal share of the (tail tile, K-block) units.
struct GemmSegIter {
  long long tf, u, u_end;
  __device__ explicit GemmSegIter(const GemmParams &p) {
    tf = blockIdx.x;
    const long long units = (p.tiles - p.full_tiles) * p.NKB;
    u = units * blockIdx.x / gridDim.x;
    u_end = units * (blockIdx.x + 1) / gridDim.x;
  }
  __device__ bool next(const GemmParams &p, GemmSeg &s) {
    if (tf < p.full_tiles) {
      s.t = tf;
      s.kb0 = 0;
      s.kb1 = p.NKB;
      tf += gridDim.x;
      return true;
    }
    if (u < u_end) {
      const long long tl = u / p.NKB;
      s.t = p.full_tiles + tl;
      s.kb0 = (int)(u % p.NKB);
      s.kb1 = (int)min((long long)p.NKB, s.kb0 + (u_end - u));
      u += s.kb1 - s.kb0;
      return true;
    }
    return false;
  }
};

struct GemmSmem {
  int bstage, wstage, bars, tmem_slot, flags, bytes;
};

// Barriers: 3 per B stage, 2 per weight stage, 4 accumulator, 1 drain.
constexpr int kGemmBarBytes = ((3 * kGemmStages + 2 * kGemmWStages + 5) * 8 + 15) / 16 * 16;

__host__ __device__ constexpr GemmSmem gemm_smem_layout() {
  return GemmSmem{0, kGemmStages * kGemmBStageBytes,
                  kGemmStages * kGemmBStageBytes + kGemmWStages * kGemmWStageBytes,
                  kGemmStages * kGemmBStageBytes + kGemmWStages * kGemmWStageBytes + kGemmBarBytes,
                  kGemmStages * kGemmBStageBytes + kGemmWStages * kGemmWStageBytes + kGemmBarBytes + 16,
                  kGemmStages * kGemmBStageBytes + kGemmWStages * kGemmWStageBytes + kGemmBarBytes + 32};
}

// ---------------------------------------------------------- tcgen05 PTX --

__device__ __forceinline__ void tmem_alloc(uint32_t *slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, fp32 accumulate.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (rows of 128 bytes), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: kind::f16, A = B = f16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t gemm_idesc(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// --------------------------------------------------------------- prep --

// One 16-K group of int8 activations in the B layout: element 2i+h of the
// group is x[8h + i] * 4^-e(i), e = {0,1,2,3,4,5,0,1}, as fp16 (exact: at most
// 7 significant bits, no smaller than 2^-10).  Returns the sum of the group.
__device__ __forceinline__ int prep_group(const int8_t (&v)[16], uint32_t *out) {
  uint32_t h[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = i < 6 ? i : i - 6;
    const float sc = 1.0f / (float)(1 << (2 * e));
    h[i] = (uint32_t)__half_as_ushort(__float2half_rn((float)v[i] * sc)) |
           ((uint32_t)__half_as_ushort(__float2half_rn((float)v[8 + i] * sc)) << 16);
    sum += v[i] + v[8 + i];
  }
  uint4 *dst = reinterpret_cast<uint4 *>(out);
  dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
  dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
  return sum;
}

// CTAs from `first` on zero `zero` (n16 16-byte words: the split-tile
// partial sums and tickets of the GEMV that follows), after the previous
// kernel, which may share the workspace, has finished.
__device__ __forceinline__ void prep_zero_tail(int64_t first, uint4 *zero, int64_t n16) {
  const int64_t cta = (int64_t)blockIdx.x - first, nct = (int64_t)gridDim.x - first;
  for (int64_t i = cta * 256 + threadIdx.x; i < n16; i += nct * 256) zero[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Where 16-K group q of token m goes in the prepared activations.  T == 0:
// row-major [M][K].  T > 0: K-block-major [K/64][T][64], T token rows per
// 64-K block (rows >= M are zero), so the 8 K-blocks of a 512-K chunk are
// one contiguous box of 8*T rows of 128 bytes.
__device__ __forceinline__ uint32_t *prep_out(uint32_t *xb, int64_t m, int64_t q, int64_t K, int T) {
  return T == 0 ? xb + m * (K / 2) + q * 8 : xb + ((q >> 2) * T + m) * 32 + (q & 3) * 8;
}

// Zero rows M..T-1 of the K-block-major layout (CTAs M..T-1 of a prep grid).
__device__ __forceinline__ void prep_zero_row(uint32_t *xb, int64_t m, int64_t K, int T) {
  for (int64_t q = threadIdx.x; q < K / 16; q += 256) {
    uint4 *dst = reinterpret_cast<uint4 *>(prep_out(xb, m, q, K, T));
    dst[0] = make_uint4(0u, 0u, 0u, 0u);
    dst[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Group sums for the group-scaled GEMV: with xsumg non-null the prep kernels
// also write xsumg[m][g] = sum of x_q over the token's group g of G weights
// (NG = K / G <= kPrepMaxGroups), and the output scale is s_m / 127 (the
// weight scales are per group and applied in the GEMV).
constexpr int kPrepMaxGroups = 1024;
struct PrepGroups {
  int32_t *xsumg;
  int G, NG;
};

// Adds a 16-K group's sum into the per-group bins (shared memory).
__device__ __forceinline__ void prep_bin(const PrepGroups &grp, int *bins, int64_t q, int sum) {
  if (grp.xsumg && sum) atomicAdd(&bins[(int)((q * 16) / grp.G)], sum);
}

// x_q int8 [M, K] -> fp16 B matrix [M, K] (per 16-K group, element 2i+h is
// x[16q + 8h + i] * 4^-e(i), e = {0,1,2,3,4,5,0,1}), per-token sum of x_q and
// the per-token output scale w_scale * s_m / 127.  One CTA per token (CTAs
// beyond M zero the GEMV's partial sums).
__global__ void __launch_bounds__(256) gemm_prep_kernel(const int8_t *__restrict__ xq, const float *__restrict__ scale,
                                                        const float *__restrict__ w_scale, int64_t K,
                                                        uint32_t *__restrict__ xb, int32_t *__restrict__ xsum,
                                                        float *__restrict__ fscale, int64_t M, uint4 *zero,
                                                        int64_t zero_n16, int T, const PrepGroups grp) {
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int64_t rows = M > T ? M : T;
  if ((int64_t)blockIdx.x >= rows) {
    prep_zero_tail(rows, zero, zero_n16);
    return;
  }
  if ((int64_t)blockIdx.x >= M) {
    prep_zero_row(xb, blockIdx.x, K, T);
    return;
  }
  __shared__ int red[8];
  __shared__ int bins[kPrepMaxGroups];
  if (grp.xsumg) {
    for (int i = threadIdx.x; i < grp.NG; i += 256) bins[i] = 0;
    __syncthreads();
  }
  const int64_t m = blockIdx.x;
  const int8_t *row = xq + m * K;
  int sum = 0;
  for (int64_t q = threadIdx.x; q < K / 16; q += 256) {
    const int4 u = *reinterpret_cast<const int4 *>(row + q * 16);
    int8_t v[16];
    memcpy(v, &u, 16);
    const int s16 = prep_group(v, prep_out(xb, m, q, K, T));
    prep_bin(grp, bins, q, s16);
    sum += s16;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < 8; ++w) t += red[w];
    xsum[m] = t;
    fscale[m] = grp.xsumg ? __fdiv_rn(__ldg(scale + m), 127.0f)
                          : __fdiv_rn(__fmul_rn(__ldg(w_scale), __ldg(scale + m)), 127.0f);
  }
  if (grp.xsumg)
    for (int i = threadIdx.x; i < grp.NG; i += 256) grp.xsumg[m * grp.NG + i] = bins[i];
}

// Fused BitLinear prologue for the tensor-core paths: per-token absmax
// quantisation of x (BitNet 深度拆解 §2.2, the same fp32 operations as
// quant_act_kernel) straight into the B layout, the per-token sum of x_q and
// the output scale.  Optionally also writes x_q and s.  One CTA per token;
// K % 16 == 0 and 16-byte aligned rows (checked on the host).
//
// With an RMSNorm (`norm` non-null: norm->g, norm->eps) the kernel first
// forms the token's normalisation factor r (rmsnorm.cuh) and quantises
// h = fl(fl(x * r) * g) instead of x.
struct PrepNorm {
  const float *g;  // [K] or nullptr (a weight of ones)
  float eps;
  float *ms_out;   // [M] mean squares, or nullptr
};

template <typename T>
__global__ void __launch_bounds__(256)
    fused_prep_kernel(const T *__restrict__ x, const float *__restrict__ w_scale, int64_t K,
                      uint32_t *__restrict__ xb, int32_t *__restrict__ xsum, float *__restrict__ fscale,
                      int8_t *__restrict__ xq_out, float *__restrict__ scale_out, int64_t M, uint4 *zero,
                      int64_t zero_n16, int TR, const PrepNorm norm, const PrepGroups grp) {
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int64_t rows = M > TR ? M : TR;
  if ((int64_t)blockIdx.x >= rows) {
    prep_zero_tail(rows, zero, zero_n16);
    return;
  }
  if ((int64_t)blockIdx.x >= M) {
    prep_zero_row(xb, blockIdx.x, K, TR);
    return;
  }
  __shared__ float redf[8];
  __shared__ int red[8];
  __shared__ double redd[8];
  __shared__ int bins[kPrepMaxGroups];
  if (grp.xsumg)
    for (int i = threadIdx.x; i < grp.NG; i += 256) bins[i] = 0;  // ordered by the reductions' barriers below
  const int64_t m = blockIdx.x;
  const T *row = x + m * K;
  const bool rms = norm.eps >= 0.0f;  // a negative eps marks "no RMSNorm"
  const float r =
      rms ? rms_factor(row, K, norm.eps, redd, (norm.ms_out && threadIdx.x == 0) ? norm.ms_out + m : nullptr) : 1.0f;
  float amax = 0.0f;
  for (int64_t k = (int64_t)threadIdx.x * 8; k < K; k += 256 * 8) {
    float v[8];
    load8(row + k, v);
    if (rms) rms_apply8(v, r, norm.g, k);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = block_max_256(amax, redf);
  const float s = amax < 1e-8f ? 1e-8f : amax;
  const float c = quant_factor(s);
  int sum = 0;
  for (int64_t q = threadIdx.x; q < K / 16; q += 256) {
    float f[8], g[8];
    load8(row + q * 16, f);
    load8(row + q * 16 + 8, g);
    if (rms) {
      rms_apply8(f, r, norm.g, q * 16);
      rms_apply8(g, r, norm.g, q * 16 + 8);
    }
    int8_t vf[8], vg[8], v[16];
    quantize_fast(f, s, c, vf);
    quantize_fast(g, s, c, vg);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = vf[i];
      v[8 + i] = vg[i];
    }
    if (xq_out) {
      int4 u;
      memcpy(&u, v, 16);
      *reinterpret_cast<int4 *>(xq_out + m * K + q * 16) = u;
    }
    const int s16 = prep_group(v, prep_out(xb, m, q, K, TR));
    prep_bin(grp, bins, q, s16);
    sum += s16;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < 8; ++w) t += red[w];
    xsum[m] = t;
    fscale[m] = grp.xsumg ? __fdiv_rn(s, 127.0f) : __fdiv_rn(__fmul_rn(__ldg(w_scale), s), 127.0f);
    if (scale_out) scale_out[m] = s;
  }
  if (grp.xsumg)
    for (int i = threadIdx.x; i < grp.NG; i += 256) grp.xsumg[m * grp.NG + i] = bins[i];
}

// --------------------------------------------------------------- main --

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr GemmSmem L = gemm_smem_layout();
  uint64_t *bfull = reinterpret_cast<uint64_t *>(smem + L.bars);  // [stages] TMA -> MMA
  uint64_t *kempty = bfull + kGemmStages;                            // [stages] MMA done -> producer, decoders
  uint64_t *afull = kempty + kGemmStages;                            // [stages] decoders -> MMA
  uint64_t *wfull = afull + kGemmStages;                             // [2] TMA -> decoders
  uint64_t *wempty = wfull + kGemmWStages;                           // [2] decoders -> producer
  uint64_t *accfull = wempty + kGemmWStages;                         // [2] MMA -> epilogue
  uint64_t *accempty = accfull + 2;                                  // [2] epilogue -> MMA
  uint64_t *drain = accempty + 2;                                    // [1] final MMA completion
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem_slot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flags);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGemmStages; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&afull[i], 4);
    }
    for (int i = 0; i < kGemmWStages; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 4 * kGemmDecSets);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], 4 * kGemmEpiSets);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kGemmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (*abort_flag) return;
    if (!mbar_wait(bar, parity)) {
      raise_device_error(kDevErrTimeout);
      *abort_flag = 1;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&bmap);
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_b = l2_policy_evict_last();
      long long c = 0, wc = 0;
      bool waited_prior = false;
      GemmSegIter it(p);
      GemmSeg sg;
      while (!*abort_flag && it.next(p, sg)) {
        const int rt = (int)(sg.t % p.NRT), tt = (int)(sg.t / p.NRT);
        for (int kb = sg.kb0; kb < sg.kb1 && !*abort_flag; ++kb, ++c) {
          if ((kb & 7) == 0 || kb == sg.kb0) {  // the 512-K weight block holding kb
            const int ws = (int)(wc % kGemmWStages);
            if (wc >= kGemmWStages) wait(&wempty[ws], (uint32_t)(((wc / kGemmWStages) - 1) & 1));
            if (*abort_flag) break;
            mbar_arrive_expect_tx(&wfull[ws], kGemmWStageBytes);
            tma_load_2d(smem + L.wstage + ws * kGemmWStageBytes, &wmap, &wfull[ws], (kb >> 3) * 128,
                        rt * kGemmRows, pol_w);
            ++wc;
          }
          if (!waited_prior) {  // activations come from the previous kernel
            pdl_wait_prior_grid();
            waited_prior = true;
          }
          const int s = (int)(c % kGemmStages);
          if (c >= kGemmStages) wait(&kempty[s], (uint32_t)(((c / kGemmStages) - 1) & 1));
          if (*abort_flag) break;
          mbar_arrive_expect_tx(&bfull[s], kGemmBStageBytes);
          tma_load_2d(smem + L.bstage + s * kGemmBStageBytes, &bmap, &bfull[s], kb * kGemmKB, tt * kGemmTok,
                      pol_b);
        }
      }
      if (!waited_prior) pdl_wait_prior_grid();
      if (*abort_flag) {
        // drain: wait (bounded) for every copy this thread may have in flight
        for (long long j = (c > kGemmStages ? c - kGemmStages : 0); j < c; ++j)
          mbar_wait(&bfull[j % kGemmStages], (uint32_t)((j / kGemmStages) & 1));
        for (long long j = (wc > kGemmWStages ? wc - kGemmWStages : 0); j < wc; ++j)
          mbar_wait(&wfull[j % kGemmWStages], (uint32_t)((j / kGemmWStages) & 1));
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      pdl_wait_prior_grid();
      const uint32_t idesc = gemm_idesc(kGemmRows, kGemmTok);
      const uint32_t bbase = smem_u32(smem + L.bstage);
      long long c = 0, tc = 0;
      GemmSegIter it(p);
      GemmSeg sg;
      for (; !*abort_flag && it.next(p, sg); ++tc) {
        const int a = (int)(tc % kGemmAccBufs);
        if (tc >= kGemmAccBufs) wait(&accempty[a], (uint32_t)(((tc / kGemmAccBufs) - 1) & 1));
        tc_fence_after();
        const uint32_t d_tmem = tmem + kGemmAccCol + a * kGemmTok;
        for (int kb = sg.kb0; kb < sg.kb1 && !*abort_flag; ++kb, ++c) {
          const int s = (int)(c % kGemmStages);
          const uint32_t par = (uint32_t)((c / kGemmStages) & 1);
          wait(&bfull[s], par);
          wait(&afull[s], par);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t bdesc = smem_desc_sw128(bbase + s * kGemmBStageBytes);
          const uint32_t a_tmem = tmem + kGemmACol + s * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ts(d_tmem, a_tmem + kk * 8, bdesc + (uint64_t)(kk * 2), idesc, (kb != sg.kb0) || kk != 0);
          tc_commit(&kempty[s]);
        }
        tc_commit(&accfull[a]);
      }
      // every MMA this thread issued has completed once `drain` flips
      tc_commit(drain);
      mbar_wait(drain, 0);
    }
  } else if ((warp >= 4 && warp < 8) || (warp >= 12 && warp < kGemmEpiWarp2)) {
    // ---------------------------------------------------------- decoders --
    // tcgen05.st is warp-collective: the abort decision is made warp-uniform.
    pdl_wait_prior_grid();
    const int dset = warp < 8 ? 0 : 1 + (warp - 12) / 4;
    const int quad = warp & 3, row = quad * 32 + lane;
    const uint32_t wbase = smem_u32(smem + L.wstage);
    long long c = 0, wc = 0;
    bool stop = false;
    GemmSegIter it(p);
    GemmSeg sg;
    while (!stop && it.next(p, sg)) {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++c) {
        const int ws = (int)(wc % kGemmWStages);
        if ((kb & 7) == 0 || kb == sg.kb0) wait(&wfull[ws], (uint32_t)((wc / kGemmWStages) & 1));
        const int chunk = kb & 7;
        const bool last_of_wstage = chunk == 7 || kb == sg.kb1 - 1;
        if ((int)(c % kGemmDecSets) != dset) {  // another set decodes this block
          if (__any_sync(0xffffffffu, *abort_flag)) {
            stop = true;
            break;
          }
          if (last_of_wstage) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[ws]);
            ++wc;
          }
          continue;
        }
        const int s = (int)(c % kGemmStages);
        if (c >= kGemmStages) wait(&kempty[s], (uint32_t)(((c / kGemmStages) - 1) & 1));
        if (__any_sync(0xffffffffu, *abort_flag)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint4 v = lds_u128(wbase + ws * kGemmWStageBytes + row * 128 + (((chunk ^ (row & 7)) & 7) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t hs = w[u] >> 12;
#pragma unroll
          for (int i = 0; i < 6; ++i) h[8 * u + i] = w[u] & (0x00030003u << (2 * i));
          h[8 * u + 6] = hs & 0x00030003u;
          h[8 * u + 7] = hs & 0x000C000Cu;
        }
        tmem_st_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + kGemmACol + s * 32, h);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[s]);
        if (last_of_wstage) {
          if (lane == 0) mbar_arrive(&wempty[ws]);
          ++wc;
        }
      }
    }
  } else if ((warp >= 8 && warp < 12) || warp >= kGemmEpiWarp2) {
    // ---------------------------------------------------------- epilogue --
    pdl_wait_prior_grid();
    const int quad = warp & 3, row = quad * 32 + lane;
    const int eset = warp < 12 ? 0 : 1 + (warp - kGemmEpiWarp2) / 4;  // which share of the columns
    const int cb_begin = eset * (kGemmTok / 32) / kGemmEpiSets, cb_end = (eset + 1) * (kGemmTok / 32) / kGemmEpiSets;
    long long tc = 0;
    GemmSegIter it(p);
    GemmSeg sg;
    for (; it.next(p, sg); ++tc) {
      const long long t = sg.t;
      const int rt = (int)(t % p.NRT), tt = (int)(t / p.NRT);
      const int a = (int)(tc % kGemmAccBufs);
      wait(&accfull[a], (uint32_t)((tc / kGemmAccBufs) & 1));
      if (__any_sync(0xffffffffu, *abort_flag)) break;  // tcgen05.ld is warp-collective
      tc_fence_after();
      const int64_t n = (int64_t)rt * kGemmRows + row;
      if (sg.kb0 != 0 || sg.kb1 != p.NKB) {
        // part of a split tail tile: add the exact partial sums (D * 2^24,
        // integers) into the workspace; the warp whose ticket completes this
        // block of 32 rows x (its token columns) writes the outputs
        const long long tl = t - p.full_tiles;
        int32_t *part = p.ws_part + (size_t)tl * kGemmTok * kGemmRows;  // [token column][row]
#pragma unroll 1
        for (int cb = cb_begin; cb < cb_end; ++cb) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + kGemmAccCol + a * kGemmTok + cb * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            atomicAdd(part + (size_t)(cb * 32 + j) * kGemmRows + row,
                      __float2int_rn(__uint_as_float(r[j]) * 16777216.0f));
        }
        __threadfence();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atomicAdd(p.ws_ticket + tl * 16 + eset * 4 + quad, (unsigned)(sg.kb1 - sg.kb0));
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + (unsigned)(sg.kb1 - sg.kb0) == (unsigned)p.NKB) {
          __threadfence();
#pragma unroll 1
          for (int cb = cb_begin; cb < cb_end; ++cb) {
            const int64_t tok0 = (int64_t)tt * kGemmTok + cb * 32;
            const int32_t xs_l = tok0 + lane < p.M ? __ldg(p.xsum + tok0 + lane) : 0;
            const float fs_l = tok0 + lane < p.M ? __ldg(p.fscale + tok0 + lane) : 0.0f;
            // all 32 partial sums in flight at once, then their stores (a
            // load after a store that may alias would wait a whole L2 round
            // trip per output)
#pragma unroll 1
            for (int j0 = 0; j0 < 32; j0 += 8) {
              int32_t total[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) total[j] = __ldcg(part + (size_t)(cb * 32 + j0 + j) * kGemmRows + row);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int32_t xs = __shfl_sync(0xffffffffu, xs_l, j0 + j);
                const float fs = __shfl_sync(0xffffffffu, fs_l, j0 + j);
                part[(size_t)(cb * 32 + j0 + j) * kGemmRows + row] = 0;
                const int64_t tok = tok0 + j0 + j;
                if (n < p.N && tok < p.M) {
                  const int32_t v = total[j] - xs;
                  if (p.acc) p.acc[tok * p.N + n] = v;
                  p.y[tok * p.N + n] = __fmul_rn((float)v, fs);
                }
              }
            }
          }
          if (lane == 0) p.ws_ticket[tl * 16 + eset * 4 + quad] = 0u;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[a]);
        continue;
      }
#pragma unroll 1
      for (int cb = cb_begin; cb < cb_end; ++cb) {
        // lane j fetches token tok0 + j's sum and scale (one coalesced load
        // each, issued before the TMEM load); the outputs take them by
        // shuffles, so no load waits behind an output store
        const int64_t tok0 = (int64_t)tt * kGemmTok + cb * 32;
        const int32_t xs_l = tok0 + lane < p.M ? __ldg(p.xsum + tok0 + lane) : 0;
        const float fs_l = tok0 + lane < p.M ? __ldg(p.fscale + tok0 + lane) : 0.0f;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + kGemmAccCol + a * kGemmTok + cb * 32, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          // shuffles by the whole warp (rows past N only skip the stores)
          const int32_t xs = __shfl_sync(0xffffffffu, xs_l, j);
          const float fs = __shfl_sync(0xffffffffu, fs_l, j);
          const int64_t tok = tok0 + j;
          if (n < p.N && tok < p.M) {
            const int32_t v = __float2int_rn(__uint_as_float(r[j]) * 16777216.0f) - xs;
            if (p.acc) p.acc[tok * p.N + n] = v;
            p.y[tok * p.N + n] = __fmul_rn((float)v, fs);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[a]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kGemmTmemCols);
  }
}

// ------------------------------------------------------------- host side --

inline size_t gemm_xb_bytes(int64_t M, int64_t K) { return (((size_t)M * (size_t)K * 2) + 1023) & ~(size_t)1023; }

// Whole tiles and stream-K tail: the tail is split when the last wave of
// whole tiles would be less than half full on `sms` CTAs.
struct GemmSplit {
  long long tiles, full_tiles, tail;
  size_t part_bytes;  // partial sums + tickets of the tail tiles
};
inline GemmSplit gemm_split(int64_t M, int64_t N, int sms) {
  GemmSplit s;
  s.tiles = (long long)((N + kGemmRows - 1) / kGemmRows) * ((M + kGemmTok - 1) / kGemmTok);
  const long long rem = s.tiles % sms;
  s.tail = (s.tiles > sms && rem > 0 && 2 * rem < sms) ? rem : 0;
  s.full_tiles = s.tiles - s.tail;
  s.part_bytes = (((size_t)s.tail * kGemmTok * kGemmRows * 4 + (size_t)s.tail * 16 * 4) + 255) & ~(size_t)255;
  return s;
}

// Workspace: prepared activations, per-token sums and scales, then the
// stream-K partials (sized for the 148 SMs of a B300).
inline size_t gemm_part_offset(int64_t M, int64_t K) {
  return gemm_xb_bytes(M, K) + (((size_t)M * 8 + 255) & ~(size_t)255) + 1024;
}
inline size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return gemm_part_offset(M, K) + gemm_split(M, N, 148).part_bytes;
}

}  // namespace bitnet

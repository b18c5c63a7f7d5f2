// C ABI of the BitNet b1.58 W2A8 library: argument validation, workspace
// layout, TMA descriptors and kernel launches.  The kernels live in the
// included .cuh files (one translation unit, so they share the device error
// word).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <cudaTypedefs.h>

#include "bitnet_w2a8.h"
#include "common.cuh"
#include "gemm.cuh"
#include "gemv.cuh"
#include "gemv_ldg.cuh"
#include "gemv_mma.cuh"
#include "gemv_mma_grouped.cuh"
#include "gemv_rows.cuh"
#include "grouped.cuh"
#include "pack.cuh"
#include "quant_act.cuh"
#include "rmsnorm.cuh"

using namespace bitnet;

// Scratch of bitnet_w2a8_gemv_static_scratch: a fixed array in the module
// (zero-initialised at load; every device that loads the library holds it).
static __device__ __align__(256) uint8_t g_gemv_static_scratch[BITNET_GEMV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
thread_local int t_pdl = 0;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Test hook (bitnet_test_inject_cuda_failures): pending injected failures of
// the device query, consumed one per query.
std::atomic<int> g_inject_cuda_failures{0};

// Every entry point that enqueues work calls this after validating its
// arguments and before any other CUDA call.
bitnet_status device_info(DeviceInfo **out) {
  for (int n = g_inject_cuda_failures.load(); n > 0; n = g_inject_cuda_failures.load())
    if (g_inject_cuda_failures.compare_exchange_weak(n, n - 1)) return BITNET_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BITNET_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.init) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return BITNET_ERR_CUDA;
    d.sms = prop.multiProcessorCount;
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.smem_optin = prop.sharedMemPerBlockOptin;
    d.init = true;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return BITNET_ERR_UNSUPPORTED;
  *out = &d;
  return BITNET_OK;
}

bitnet_status get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return BITNET_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return BITNET_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return BITNET_OK;
}

// Launches `kernel` with optional programmatic dependent launch.
template <typename... KArgs, typename... Args>
bitnet_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (t_pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? BITNET_OK : BITNET_ERR_CUDA;
}

// Dynamic shared memory already allowed per (device, kernel): the attribute
// is set once per kernel and device, and again only for a larger size.
std::unordered_map<const void *, size_t> g_smem_set[kMaxDevices];

template <typename K>
bitnet_status set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return BITNET_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BITNET_ERR_CUDA;
  const void *key = reinterpret_cast<const void *>(kernel);
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_smem_set[dev].find(key);
  if (it != g_smem_set[dev].end() && it->second >= bytes) return BITNET_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return BITNET_ERR_CUDA;
  g_smem_set[dev][key] = bytes;
  return BITNET_OK;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
constexpr int64_t kMaxElems = (int64_t)1 << 40;
// The tensor-core paths accumulate code * x (|.| <= 254 per term) in fp32 in
// units of 2^-24; the sum of a row stays an exact integer while 254 * K < 2^24.
constexpr int64_t kTensorMaxK = 65536;

bool shape_ok(int64_t N, int64_t K) { return N > 0 && K > 0 && K % 4 == 0 && N <= kMaxElems / K; }

// ------------------------------------------------------------------ GEMV --

struct GemvPlan {
  bool tma;
  int NR, NKB, KBS, S, xrow, grid;
  bool hmma;
  size_t smem;
  // Workspace: [partials | tickets] (must be zero on entry, left zero) at
  // offset 0 for every kernel, then the tensor-core path's prepared
  // activations, per-token sums and output scales (any contents).
  size_t ws_partial_bytes, ws_zero_bytes, ws_prep_xb, ws_prep_sums, ws_bytes;
};

// Token rows of the prepared activations of the mma.sync GEMV (2..64
// tokens: padded to 8, 16, 32 or 64, K-block-major); 0 for one token.
int gemv_mma_rows(int64_t M) {
  if (M < 2 || M > BITNET_GEMV_MAX_M) return 0;
  return M <= 8 ? 8 : (M <= 16 ? 16 : (M <= 32 ? 32 : 64));
}

GemvPlan plan_gemv(int64_t M, int64_t N, int64_t K, int sms) {
  GemvPlan pl = {};
  pl.NR = (int)cdiv(N, kStageRows);
  pl.NKB = (int)cdiv(K, kStageK);
  pl.hmma = M > 2;
  const int per_kb = pl.hmma ? 1024 : 512;  // activation bytes per token per K-block
  int kbs_max = (int)((kGemvXBudget / M - (pl.hmma ? 8 : 0)) / per_kb);
  kbs_max = std::max(1, kbs_max);
  pl.S = (int)cdiv(pl.NKB, kbs_max);
  pl.KBS = (int)cdiv(pl.NKB, pl.S);
  pl.xrow = pl.hmma ? pl.KBS * 1024 + 8 : pl.KBS * 512;
  const long long total = (long long)pl.NR * pl.NKB;
  pl.grid = (int)std::min<long long>(sms, total);
  pl.smem = gemv_smem_layout((int)M, pl.KBS, pl.xrow).bytes + 1024;
  pl.ws_partial_bytes = (size_t)pl.NR * kStageRows * M * 4;
  pl.ws_zero_bytes = ((pl.ws_partial_bytes + (size_t)pl.NR * 4) + 255) & ~(size_t)255;
  pl.ws_prep_xb = pl.ws_zero_bytes;
  pl.ws_prep_sums = pl.ws_prep_xb + gemm_xb_bytes(std::max<int64_t>(M, gemv_mma_rows(M)), K);
  pl.ws_bytes = pl.ws_prep_sums + (((size_t)M * 8 + 255) & ~(size_t)255) + 256;
  return pl;
}

template <class Policy>
bitnet_status launch_gemv_tma(const CUtensorMap &map, const GemvParams &p, const GemvPlan &pl,
                              cudaStream_t stream) {
  // the kernel adds split row tiles into zeroed partials and tickets
  if (cudaMemsetAsync(p.ws_partial, 0, pl.ws_zero_bytes, stream) != cudaSuccess) return BITNET_ERR_CUDA;
  auto k = gemv_tma_kernel<Policy>;
  if (set_smem(k, pl.smem) != BITNET_OK) return BITNET_ERR_CUDA;
  return launch(k, dim3(pl.grid), dim3(kGemvThreads), pl.smem, stream, map, p);
}

bitnet_status encode_packed_map(CUtensorMap *map, const uint8_t *packed, int64_t N, int64_t K, uint32_t box_x,
                                uint32_t box_y, CUtensorMapSwizzle swz) {
  if (get_encoder() != BITNET_OK) return BITNET_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 4), (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
  cuuint32_t box[2] = {box_x, box_y};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(packed), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BITNET_OK : BITNET_ERR_CUDA;
}

// Register-resident rows (one read of x) when the row has at most
// kQuantThreads * 8 * 8 elements; two passes otherwise.
template <typename T>
bitnet_status launch_quant(const T *x, bool vec, int64_t M, int64_t K, int8_t *x_q, float *scale,
                           cudaStream_t stream) {
  const dim3 grid((unsigned)M), block(kQuantThreads);
  const int64_t per = (int64_t)kQuantThreads * 8;
  if (!vec) return launch(quant_act_kernel<T, false, 0>, grid, block, 0, stream, x, K, x_q, scale);
  if (K <= per) return launch(quant_act_kernel<T, true, 1>, grid, block, 0, stream, x, K, x_q, scale);
  if (K <= 2 * per) return launch(quant_act_kernel<T, true, 2>, grid, block, 0, stream, x, K, x_q, scale);
  if (K <= 4 * per) return launch(quant_act_kernel<T, true, 4>, grid, block, 0, stream, x, K, x_q, scale);
  if (K <= 8 * per) return launch(quant_act_kernel<T, true, 8>, grid, block, 0, stream, x, K, x_q, scale);
  return launch(quant_act_kernel<T, true, 0>, grid, block, 0, stream, x, K, x_q, scale);
}

// Prep grid for the tensor-core GEMV: M token CTAs plus CTAs that zero the
// split-tile partials and tickets (32 KB each).
unsigned prep_grid(int64_t M, const GemvPlan &pl) {
  return (unsigned)(std::max<int64_t>(M, gemv_mma_rows(M)) +
                    std::min<int64_t>(148, cdiv((int64_t)pl.ws_zero_bytes, 32768)));
}

// The streaming-load kernel takes one or two tokens whose activation words
// fit in registers: 16-byte chunks per row <= 32 lanes x 4 (one token) or x 2.
int ldg_chunks_per_lane(int64_t M, int64_t K) { return (int)cdiv(K / 64, 32) * (M == 1 ? 1 : 2); }
bool ldg_ok(int64_t M, int64_t K, const void *packed) {
  return M <= 2 && K % 64 == 0 && aligned(packed, 16) && ldg_chunks_per_lane(M, K) <= 4 &&
         M * (K / 16) <= (int64_t)kLdgGroups * kLdgThreads && K / 4 <= kLdgStageBytes;
}

// Group sizes the streaming kernel takes: one group per row, or a power of
// two from 64 to 2048 weights (whole runs of 1..32 lanes).
bool ldg_group_ok(int64_t K, int64_t G) {
  return G == K || (G >= 64 && G <= 2048 && (G & (G - 1)) == 0 && K % G == 0);
}

// FORM kLdgSwiGLU: `packed`, `w_scale`, `acc` are the gate matrix's and
// packed_up, w_scale_up, acc_up the up matrix's (N rows each), y = silu(gate) * up.
// FORM kLdgGrouped: w_scale is [N, K / G] group scales, acc [M, N, K / G].
template <typename XT, int FORM = kLdgPlain>
bitnet_status launch_gemv_ldg(const int8_t *x_q, const float *scale, const void *x, int8_t *xq_out, float *scale_out,
                              int64_t M, const uint8_t *packed, const float *w_scale, int64_t N, int64_t K, float *y,
                              int32_t *acc, const DeviceInfo *d, cudaStream_t stream,
                              const uint8_t *packed_up = nullptr, const float *w_scale_up = nullptr,
                              int32_t *acc_up = nullptr, int64_t G = 0) {
  constexpr bool SW = FORM == kLdgSwiGLU, GR = FORM == kLdgGrouped;
  GemvLdgParams p = {};
  if (GR) {
    p.G = (int)G;
    p.NG = (int)(K / G);
    p.P = (int)(G / 64);
    // shifts for power-of-two groups; one group per row needs none (index 0)
    int gs = 0;
    while (((int64_t)1 << gs) < G) ++gs;
    p.GS = p.NG == 1 ? 31 : gs;
    p.PS = p.NG == 1 ? 0 : gs - 6;
  }
  int J = (int)cdiv(K / 64, 32);
  if (GR && p.NG > 1 && p.P <= 4) {
    // lane-local groups: P slots per group, groups lane, lane + 32, ...
    const int jl = p.P * (int)cdiv(p.NG, 32);
    if (jl <= (M == 1 ? 4 : 2)) {
      p.LOCAL = 1;
      J = jl;
    }
  }
  p.packed_up = packed_up;
  p.w_scale_up = w_scale_up;
  p.acc_up = acc_up;
  p.packed = packed;
  p.xq = x_q;
  p.x = x;
  p.xq_out = xq_out;
  p.scale_out = scale_out;
  p.scale = scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc = acc;
  p.N = N;
  p.K = K;
  p.M = (int)M;
  p.C = (int)(K / 64);
  const int grid = (int)std::min<int64_t>(d->sms, cdiv(N, kLdgWarps));
  // ring sized to the rows a warp owns: at most ceil(N / warps) rows
  // (SwiGLU: gate and up rows; grouped: the packed row and its scales)
  const int64_t rowb = (SW ? 2 : 1) * (K / 4) + (GR ? 4 * (K / G) : 0);
  const int64_t rpw = cdiv(N, (int64_t)grid * kLdgWarps);
  p.SR = (int)std::max<int64_t>(1, std::min<int64_t>(kLdgStageBytes / rowb, rpw));
  p.RS = (int)((p.SR * rowb + 15) & ~(int64_t)15);
  p.NS = (int)std::min<int64_t>(kLdgStages, cdiv(rpw, p.SR));
  const size_t smem = gemv_ldg_smem_layout((int)M, p.C, p.RS, p.NS, GR ? p.NG : 0).bytes + 128;
  auto run = [&](auto kernel) -> bitnet_status {
    if (set_smem(kernel, smem) != BITNET_OK) return BITNET_ERR_CUDA;
    return launch(kernel, dim3(grid), dim3(kLdgThreads), smem, stream, p);
  };
  if (M == 1) {
    switch (J) {
      case 1: return run(gemv_ldg_kernel<1, 1, XT, FORM>);
      case 2: return run(gemv_ldg_kernel<1, 2, XT, FORM>);
      case 3: return run(gemv_ldg_kernel<1, 3, XT, FORM>);
      default: return run(gemv_ldg_kernel<1, 4, XT, FORM>);
    }
  }
  return J == 1 ? run(gemv_ldg_kernel<2, 1, XT, FORM>) : run(gemv_ldg_kernel<2, 2, XT, FORM>);
}

// The row-range kernel takes one or two tokens whose activation words fit in
// shared memory beside the weight ring.
bool rows_ok(int64_t M, int64_t K) { return M <= 2 && M * cdiv(K, kStageK) * kStageK <= kRowsXBudget; }
// Two tokens whose rows are too long for the streaming kernel's registers
// (K > 4096) run on the tensor-core GEMV when the matrix is large: its fixed
// cost is higher (about 12 us against 6.5 us), its cost per byte lower
// (0.25 against 0.43 us per MB).  Measured: 28672 x 8192 takes 26.4 us
// against 31.8 us on the row-range kernel, 6912 x 6912 14.9 us against 11.6.
constexpr int64_t kTwoOnTcMinWeights = (int64_t)1 << 27;  // N * K, about 32 MB packed
bool two_on_tc(int64_t M, int64_t N, int64_t K, const void *packed) {
  return M == 2 && N * K >= kTwoOnTcMinWeights && !ldg_ok(M, K, packed) && K % 64 == 0 && K >= kStageK &&
         K <= kTensorMaxK && aligned(packed, 16);
}

// Row-range decode GEMV (M <= 2).  XT = int8_t: x_q and scale given;
// XT = float / bf16: fused form, x quantised in the kernel prologue (x_q and
// scale then optional outputs).
template <typename XT>
bitnet_status launch_gemv_rows(const int8_t *x_q, const float *scale, const void *x, int8_t *xq_out,
                               float *scale_out, int64_t M, const uint8_t *packed, const float *w_scale, int64_t N,
                               int64_t K, float *y, int32_t *acc, const DeviceInfo *d, cudaStream_t stream) {
  GemvRowsParams r = {};
  r.xq = x_q;
  r.x = x;
  r.xq_out = xq_out;
  r.scale_out = scale_out;
  r.scale = scale;
  r.w_scale = w_scale;
  r.y = y;
  r.acc = acc;
  r.N = N;
  r.K = K;
  r.M = (int)M;
  r.NKB = (int)cdiv(K, kStageK);
  r.units = (int)cdiv(N, 8);
  r.xrow = r.NKB * kStageK;
  {
    // as many 8 KB stages as shared memory holds beside the activations
    const size_t base = gemv_rows_smem_layout((int)M, r.xrow, 0).bytes + 1024;
    const size_t per = kRowsStageBytes + 16;
    const size_t avail = d->smem_optin > base ? d->smem_optin - base : 0;
    r.NS = (int)std::min<size_t>(kRowsMaxStages, avail / per);
    if (r.NS < 2) return BITNET_ERR_UNSUPPORTED;
  }
  CUtensorMap m64, m8;
  if (bitnet_status s = encode_packed_map(&m64, packed, N, K, 128, kRowsGroup, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  if (bitnet_status s = encode_packed_map(&m8, packed, N, K, 128, 8, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  const size_t smem = gemv_rows_smem_layout((int)M, r.xrow, r.NS).bytes + 1024;
  const int grid = std::min(d->sms, r.units);
  auto k = M == 1 ? gemv_rows_kernel<1, XT> : gemv_rows_kernel<2, XT>;
  if (set_smem(k, smem) != BITNET_OK) return BITNET_ERR_CUDA;
  return launch(k, dim3(grid), dim3(kRowsThreads), smem, stream, m64, m8, r);
}

// Decode GEMV on the tensor path (3 <= M <= 64): activation prep (fp16,
// K-block-major, 8/16/32/64 token rows), then the stream-K mma.sync kernel.
// With x_q == nullptr the prepared activations are already in the workspace
// (the fused BitLinear prologue wrote them).
// Group-scaled form of the tensor-core GEMV: the group scales [N, NG], the
// optional exact per-group products, and where the prep kernel writes the
// per-token group sums of x_q (in the workspace, after the GEMV's layout).
struct GroupedArgs {
  const float *gscale;
  int32_t *acc_g;
  int64_t G;
  int32_t *xsumg;
};

// Group sizes the grouped tensor-core GEMV takes: groups inside a 512-K
// unit (64, 128, 256, 512, or one group of up to 512 per row), at most
// kPrepMaxGroups groups, and a [64][NG] table of group sums in shared memory.
bool mma_group_ok(int64_t K, int64_t G) {
  if (G < 64 || K % G != 0 || 512 % G != 0) return false;
  const int64_t NG = K / G;
  return NG <= kPrepMaxGroups && 64 * NG * 4 <= kMmaGroupSumsBytes;
}

// Workspace of the grouped tensor-core path for tokens processed 64 at a
// time: the GEMV layout plus the group sums.
size_t grouped_tc_ws_bytes(int64_t M, int64_t N, int64_t K, int64_t G) {
  const int64_t Mc = std::min<int64_t>(M, BITNET_GEMV_MAX_M);
  return plan_gemv(Mc, N, K, 148).ws_bytes + (((size_t)Mc * (size_t)(K / G) * 4 + 255) & ~(size_t)255);
}

bitnet_status launch_gemv_mma(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                              const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc, void *workspace,
                              const GemvPlan &pl, const DeviceInfo *d, cudaStream_t stream,
                              const GroupedArgs *ga = nullptr) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint32_t *xb = reinterpret_cast<uint32_t *>(ws + pl.ws_prep_xb);
  int32_t *xsum = reinterpret_cast<int32_t *>(ws + pl.ws_prep_sums);
  float *fscale = reinterpret_cast<float *>(ws + pl.ws_prep_sums + (size_t)M * 4);
  const int NT = gemv_mma_rows(M);
  if (x_q) {
    const PrepGroups grp = ga ? PrepGroups{ga->xsumg, (int)ga->G, (int)(K / ga->G)} : PrepGroups{nullptr, 0, 0};
    bitnet_status st = launch(gemm_prep_kernel, dim3(prep_grid(M, pl)), dim3(256), 0, stream, x_q, scale, w_scale,
                              K, xb, xsum, fscale, M, static_cast<uint4 *>(workspace), (int64_t)(pl.ws_zero_bytes / 16),
                              NT, grp);
    if (st) return st;
  }
  CUtensorMap wmap, bmap;
  if (bitnet_status s = encode_packed_map(&wmap, packed, N, K, 128, kMmaRows, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  {
    // the activation slice of a unit: 8 K-blocks x NT token rows of 128 bytes,
    // one box (two for 64 tokens: a box is at most 256 rows)
    cuuint64_t dims[2] = {(cuuint64_t)kMmaKB, (cuuint64_t)(K / kMmaKB) * (cuuint64_t)NT};
    cuuint64_t strides[1] = {(cuuint64_t)kMmaKB * 2};
    cuuint32_t box[2] = {kMmaKB, (cuuint32_t)std::min(8 * NT, 256)};
    cuuint32_t estr[2] = {1, 1};
    if (g_encode(&bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xb, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return BITNET_ERR_CUDA;
  }
  GemvMmaParams p = {};
  p.y = y;
  p.acc = acc;
  p.xsum = xsum;
  p.fscale = fscale;
  p.ws_partial = reinterpret_cast<int32_t *>(ws);
  p.ws_ticket = reinterpret_cast<unsigned *>(ws + pl.ws_partial_bytes);
  p.N = N;
  p.K = K;
  p.M = (int)M;
  p.NRT = (int)cdiv(N, kMmaRows);
  p.NCH = (int)cdiv(K, kMmaChunkK);
  p.NKB = (int)(K / kMmaKB);
  p.units = (long long)p.NRT * p.NCH;
  auto run = [&](auto kernel, size_t smem, int ctas) -> bitnet_status {
    if (set_smem(kernel, smem) != BITNET_OK) return BITNET_ERR_CUDA;
    const int grid = (int)std::min<long long>((long long)d->sms * ctas, p.units);
    return launch(kernel, dim3(grid), dim3(kMmaThreads), smem, stream, wmap, bmap, p);
  };
  if (ga) {
    const GemvMmaGroups gp{ga->gscale, ga->xsumg, ga->acc_g, (int)ga->G, (int)(K / ga->G), (int)(ga->G / kMmaKB)};
    auto rung = [&](auto kernel, size_t smem, int ctas) -> bitnet_status {
      if (set_smem(kernel, smem) != BITNET_OK) return BITNET_ERR_CUDA;
      const int grid = (int)std::min<long long>((long long)d->sms * ctas, p.units);
      return launch(kernel, dim3(grid), dim3(kMmaThreads), smem, stream, wmap, bmap, p, gp);
    };
    switch (NT) {
      case 8: return rung(gemv_mma_grouped_kernel<1>, GemvMmaGroupedSmem<1>::bytes + 1024, MmaCfg<1>::ctas);
      case 16: return rung(gemv_mma_grouped_kernel<2>, GemvMmaGroupedSmem<2>::bytes + 1024, MmaCfg<2>::ctas);
      case 32: return rung(gemv_mma_grouped_kernel<4>, GemvMmaGroupedSmem<4>::bytes + 1024, MmaCfg<4>::ctas);
      default: return rung(gemv_mma_grouped_kernel<8>, GemvMmaGroupedSmem<8>::bytes + 1024, MmaCfg<8>::ctas);
    }
  }
  switch (NT) {
    case 8: return run(gemv_mma_kernel<1>, GemvMmaSmem<1>::bytes + 1024, MmaCfg<1>::ctas);
    case 16: return run(gemv_mma_kernel<2>, GemvMmaSmem<2>::bytes + 1024, MmaCfg<2>::ctas);
    case 32: return run(gemv_mma_kernel<4>, GemvMmaSmem<4>::bytes + 1024, MmaCfg<4>::ctas);
    default: return run(gemv_mma_kernel<8>, GemvMmaSmem<8>::bytes + 1024, MmaCfg<8>::ctas);
  }
}

bitnet_status check_gemm_args(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                              const float *w_scale, int64_t N, int64_t K, float *y, void *ws) {
  if (!x_q || !scale || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || !shape_ok(N, K) || M > kMaxElems / K || M > kMaxElems / N) return BITNET_ERR_SHAPE;
  if (!aligned(scale, 4) || !aligned(w_scale, 4) || !aligned(y, 4)) return BITNET_ERR_ALIGNMENT;
  if (!ws) return BITNET_ERR_WORKSPACE;
  return BITNET_OK;
}

// Device address of g_gemv_static_scratch per device, looked up once.
void *g_static_scratch_addr[kMaxDevices];

// Any non-null pointer: check_gemm_args only tests the workspace for null.
void *const g_static_scratch_dummy = reinterpret_cast<void *>(uintptr_t(256));

bitnet_status static_scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BITNET_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemv_static_scratch) != cudaSuccess || p == nullptr) return BITNET_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return BITNET_OK;
}

bitnet_status launch_gemm_tc(uint32_t *xb, int32_t *xsum, float *fscale, int64_t M, const uint8_t *packed, int64_t N,
                             int64_t K, float *y, int32_t *acc, const GemmSplit &sp, uint8_t *part,
                             const DeviceInfo *d, cudaStream_t stream);
bitnet_status bitlinear_tc(const void *x, bool bf, int64_t M, const uint8_t *packed, const float *w_scale, int64_t N,
                           int64_t K, float *y, int8_t *x_q, float *scale, int32_t *acc, void *workspace,
                           size_t workspace_bytes, const DeviceInfo *d, const PrepNorm &norm, cudaStream_t stream);

// Stream-K split of the GEMM's tail tiles when the workspace holds its
// partial sums (sized for 148 SMs), else whole tiles only.
GemmSplit gemm_plan_split(int64_t M, int64_t N, int64_t K, size_t ws_bytes, const DeviceInfo *d) {
  GemmSplit sp = gemm_split(M, N, d->sms);
  if (gemm_part_offset(M, K) + sp.part_bytes > ws_bytes) {
    sp.tail = 0;
    sp.full_tiles = sp.tiles;
    sp.part_bytes = 0;
  }
  return sp;
}

// Prep CTAs that zero the split tail's partial sums and tickets (32 KB each).
unsigned gemm_zero_ctas(const GemmSplit &sp) {
  return sp.part_bytes ? (unsigned)std::min<int64_t>(148, cdiv((int64_t)sp.part_bytes, 32768)) : 0u;
}

}  // namespace

extern "C" {

const char *bitnet_status_string(int status) {
  switch (status) {
    case BITNET_OK: return "BITNET_OK";
    case BITNET_ERR_INVALID_ARG: return "BITNET_ERR_INVALID_ARG";
    case BITNET_ERR_SHAPE: return "BITNET_ERR_SHAPE";
    case BITNET_ERR_ALIGNMENT: return "BITNET_ERR_ALIGNMENT";
    case BITNET_ERR_UNSUPPORTED: return "BITNET_ERR_UNSUPPORTED";
    case BITNET_ERR_CUDA: return "BITNET_ERR_CUDA";
    case BITNET_ERR_TIMEOUT: return "BITNET_ERR_TIMEOUT";
    case BITNET_ERR_WORKSPACE: return "BITNET_ERR_WORKSPACE";
    case BITNET_ERR_TOO_LARGE: return "BITNET_ERR_TOO_LARGE";
    default: return "BITNET_ERR_UNKNOWN";
  }
}

int bitnet_version(void) { return 100; }

int bitnet_test_inject_cuda_failures(int n) { return g_inject_cuda_failures.exchange(n > 0 ? n : 0); }

void bitnet_set_pdl(int enable) { t_pdl = enable ? 1 : 0; }

size_t bitnet_pack_workspace_bytes(int64_t N, int64_t K) {
  if (!shape_ok(N, K)) return 0;
  return kPackScratchHeader + (size_t)cdiv(N * K, kAbsChunk) * sizeof(double);
}

int bitnet_pack_weights(const void *W, int dtype, int64_t N, int64_t K, float alpha, float eps, uint8_t *packed,
                        float *beta, float *absmean, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (!W || !packed || !beta) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(eps)) return BITNET_ERR_INVALID_ARG;
  if (!shape_ok(N, K)) return BITNET_ERR_SHAPE;
  if (!aligned(W, dtype == BITNET_F32 ? 4 : 2) || !aligned(beta, 4) || !aligned(absmean, 4))
    return BITNET_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < bitnet_pack_workspace_bytes(N, K) || !aligned(workspace, 8))
    return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  const int64_t n = N * K;
  const int64_t nchunks = cdiv(n, kAbsChunk);
  PackScratch *scr = reinterpret_cast<PackScratch *>(workspace);
  double *sums = reinterpret_cast<double *>(reinterpret_cast<uint8_t *>(workspace) + kPackScratchHeader);
  const dim3 cgrid((unsigned)cdiv(nchunks, kPackThreads));
  const int64_t nwords = n / 16;
  const dim3 pgrid((unsigned)std::max<int64_t>(1, std::min<int64_t>(cdiv(nwords, kPackThreads), d->sms * 16)));
  const bool word_store = aligned(packed, 4);
  bitnet_status st;
  if (dtype == BITNET_F32) {
    const float *w = static_cast<const float *>(W);
    st = launch(pack_chunk_sums_kernel<float>, cgrid, dim3(kPackThreads), 0, stream, w, n, sums);
    if (!st) st = launch(pack_finalize_kernel, dim3(1), dim3(32), 0, stream, (const double *)sums, nchunks, n,
                         alpha, eps, scr, absmean);
    if (!st)
      st = word_store ? launch(pack_codes_kernel<float, true>, pgrid, dim3(kPackThreads), 0, stream, w, n, packed, scr)
                      : launch(pack_codes_kernel<float, false>, pgrid, dim3(kPackThreads), 0, stream, w, n, packed,
                               scr);
  } else {
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(W);
    st = launch(pack_chunk_sums_kernel<__nv_bfloat16>, cgrid, dim3(kPackThreads), 0, stream, w, n, sums);
    if (!st) st = launch(pack_finalize_kernel, dim3(1), dim3(32), 0, stream, (const double *)sums, nchunks, n,
                         alpha, eps, scr, absmean);
    if (!st)
      st = word_store ? launch(pack_codes_kernel<__nv_bfloat16, true>, pgrid, dim3(kPackThreads), 0, stream, w, n,
                               packed, scr)
                      : launch(pack_codes_kernel<__nv_bfloat16, false>, pgrid, dim3(kPackThreads), 0, stream, w, n,
                               packed, scr);
  }
  if (!st) st = launch(pack_beta_kernel, dim3(1), dim3(32), 0, stream, (const PackScratch *)scr, n, beta);
  return st;
}

int bitnet_quant_act(const void *x, int dtype, int64_t M, int64_t K, int8_t *x_q, float *scale,
                     cudaStream_t stream) {
  if (!x || !x_q || !scale) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || M > kMaxElems / K || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  if (!aligned(x, dtype == BITNET_F32 ? 4 : 2) || !aligned(scale, 4)) return BITNET_ERR_ALIGNMENT;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  const size_t esz = dtype == BITNET_F32 ? 4 : 2;
  const bool vec = aligned(x, 16) && ((K * (int64_t)esz) % 16 == 0) && (K % 8 == 0) && aligned(x_q, 8);
  if (dtype == BITNET_F32)
    return launch_quant(static_cast<const float *>(x), vec, M, K, x_q, scale, stream);
  return launch_quant(static_cast<const __nv_bfloat16 *>(x), vec, M, K, x_q, scale, stream);
}

size_t bitnet_gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || M > BITNET_GEMV_MAX_M || !shape_ok(N, K)) return 0;
  return plan_gemv(M, N, K, 148).ws_bytes;
}

int bitnet_w2a8_gemv(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                     const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  if (bitnet_status s = check_gemm_args(x_q, scale, M, packed, w_scale, N, K, y, workspace)) return s;
  if (!aligned(acc, 4)) return BITNET_ERR_ALIGNMENT;
  if (M > BITNET_GEMV_MAX_M) return BITNET_ERR_SHAPE;
  if (N > 0x7fffffff || K > 0x7fffffff) return BITNET_ERR_SHAPE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  GemvPlan pl = plan_gemv(M, N, K, d->sms);
  if (workspace_bytes < pl.ws_bytes || !aligned(workspace, 16)) return BITNET_ERR_WORKSPACE;

  GemvParams p = {};
  p.packed = packed;
  p.xq = x_q;
  p.scale = scale;
  p.w_scale = w_scale;
  p.y = y;
  p.acc = acc;
  p.ws_partial = static_cast<int32_t *>(workspace);
  p.ws_ticket = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(workspace) + pl.ws_partial_bytes);
  p.N = N;
  p.K = K;
  p.M = (int)M;
  p.NR = pl.NR;
  p.NKB = pl.NKB;
  p.KBS = pl.KBS;
  p.S = pl.S;
  p.xrow = pl.xrow;
  p.total = (long long)pl.NR * pl.NKB;

  const bool tma_ok = (K % 64 == 0) && K >= kStageK && aligned(packed, 16);
  if (!tma_ok) {
    const long long items = (long long)N * M;
    const int blocks = (int)std::min<long long>(cdiv(items, 8), (long long)d->sms * 16);
    return launch(gemv_generic_kernel, dim3(blocks), dim3(256), 0, stream, p);
  }
  if (ldg_ok(M, K, packed) && aligned(x_q, 16))  // one or two tokens, rows up to 8192 / 4096
    return launch_gemv_ldg<int8_t>(x_q, scale, nullptr, nullptr, nullptr, M, packed, w_scale, N, K, y, acc, d, stream);
  if (rows_ok(M, K) && !(two_on_tc(M, N, K, packed) && aligned(x_q, 16)))
    // one or two tokens: row-range kernel, whole K per CTA, no workspace use
    return launch_gemv_rows<int8_t>(x_q, scale, nullptr, nullptr, nullptr, M, packed, w_scale, N, K, y, acc, d,
                                    stream);
  if (M >= 2 && K <= kTensorMaxK && aligned(x_q, 16))
    return launch_gemv_mma(x_q, scale, M, packed, w_scale, N, K, y, acc, workspace, pl, d, stream);
  CUtensorMap map;
  if (bitnet_status s = encode_packed_map(&map, packed, N, K, kStageRowBytes, kStageRows,
                                          CU_TENSOR_MAP_SWIZZLE_128B))
    return s;
  switch (M) {
    case 1: return launch_gemv_tma<Dp4aPolicy<1>>(map, p, pl, stream);
    case 2: return launch_gemv_tma<Dp4aPolicy<2>>(map, p, pl, stream);
    default: break;
  }
  if (M <= 8) return launch_gemv_tma<HmmaPolicy<1, 4, 1>>(map, p, pl, stream);
  if (M <= 16) return launch_gemv_tma<HmmaPolicy<2, 4, 1>>(map, p, pl, stream);
  if (M <= 32) return launch_gemv_tma<HmmaPolicy<4, 2, 2>>(map, p, pl, stream);
  return launch_gemv_tma<HmmaPolicy<8, 1, 4>>(map, p, pl, stream);
}

size_t bitnet_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || !shape_ok(N, K) || M > kMaxElems / K) return 0;
  return gemm_workspace_bytes(M, N, K);
}

int bitnet_w2a8_gemm(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                     const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  if (bitnet_status s = check_gemm_args(x_q, scale, M, packed, w_scale, N, K, y, workspace)) return s;
  if (!aligned(acc, 4)) return BITNET_ERR_ALIGNMENT;
  if (N > 0x7fffffff || K > 0x7fffffff || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  if (workspace_bytes < gemm_workspace_bytes(M, N, K) || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;

  const bool tc_ok = (K % 64 == 0) && K >= 512 && K <= kTensorMaxK && aligned(packed, 16) && aligned(x_q, 16);
  if (!tc_ok) {
    GemvParams p = {};
    p.packed = packed;
    p.xq = x_q;
    p.scale = scale;
    p.w_scale = w_scale;
    p.y = y;
    p.acc = acc;
    p.N = N;
    p.K = K;
    p.M = (int)M;
    const long long items = (long long)N * M;
    const int blocks = (int)std::min<long long>(cdiv(items, 8), (long long)d->sms * 16);
    return launch(gemv_generic_kernel, dim3(blocks), dim3(256), 0, stream, p);
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint32_t *xb = reinterpret_cast<uint32_t *>(ws);
  int32_t *xsum = reinterpret_cast<int32_t *>(ws + gemm_xb_bytes(M, K));
  float *fscale = reinterpret_cast<float *>(ws + gemm_xb_bytes(M, K) + (size_t)M * 4);

  const GemmSplit sp = gemm_plan_split(M, N, K, workspace_bytes, d);
  uint8_t *part = ws + gemm_part_offset(M, K);
  bitnet_status st = launch(gemm_prep_kernel, dim3((unsigned)M + gemm_zero_ctas(sp)), dim3(256), 0, stream, x_q,
                            scale, w_scale, K, xb, xsum, fscale, M, reinterpret_cast<uint4 *>(part),
                            (int64_t)(sp.part_bytes / 16), 0, PrepGroups{nullptr, 0, 0});
  if (st) return st;
  return launch_gemm_tc(xb, xsum, fscale, M, packed, N, K, y, acc, sp, part, d, stream);
}

}  // extern "C"

namespace {

// Main prefill GEMM launch; the prepared activations are at xb (workspace).
bitnet_status launch_gemm_tc(uint32_t *xb, int32_t *xsum, float *fscale, int64_t M, const uint8_t *packed, int64_t N,
                             int64_t K, float *y, int32_t *acc, const GemmSplit &sp, uint8_t *part,
                             const DeviceInfo *d, cudaStream_t stream) {
  CUtensorMap wmap, bmap;
  if (bitnet_status s = encode_packed_map(&wmap, packed, N, K, 128, kGemmRows, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {kGemmKB, kGemmTok};
    cuuint32_t estr[2] = {1, 1};
    if (g_encode(&bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xb, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return BITNET_ERR_CUDA;
  }
  GemmParams p = {};
  p.y = y;
  p.acc = acc;
  p.xsum = xsum;
  p.fscale = fscale;
  p.M = M;
  p.N = N;
  p.K = K;
  p.NRT = (int)cdiv(N, kGemmRows);
  p.NTT = (int)cdiv(M, kGemmTok);
  p.NKB = (int)cdiv(K, kGemmKB);
  p.tiles = (long long)p.NRT * p.NTT;
  p.full_tiles = sp.tail ? sp.full_tiles : p.tiles;
  p.ws_part = sp.tail ? reinterpret_cast<int32_t *>(part) : nullptr;
  p.ws_ticket = sp.tail ? reinterpret_cast<unsigned *>(part + (size_t)sp.tail * kGemmTok * kGemmRows * 4) : nullptr;
  const size_t smem = gemm_smem_layout().bytes + 1024;
  if (set_smem(gemm_tc_kernel, smem) != BITNET_OK) return BITNET_ERR_CUDA;
  const int grid = (int)std::min<long long>(d->sms, p.tiles);
  return launch(gemm_tc_kernel, dim3(grid), dim3(kGemmThreads), smem, stream, wmap, bmap, p);
}

}  // namespace

extern "C" {

// Decode GEMV whose scratch is the file-scope array g_gemv_static_scratch instead of a
// caller workspace, for callers that cannot allocate device memory.  The
// array is part of the loaded module: each device that loads the library
// holds it until exit.  In host code `g_gemv_static_scratch` is only a
// host-side stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress, looked up once per device (with that device current)
// on the first call there.
int bitnet_w2a8_gemv_static_scratch(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                                    const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc,
                                    cudaStream_t stream) {
  // Validate everything bitnet_w2a8_gemv checks before the scratch address is
  // looked up, so that a rejected call makes no CUDA call at all.
  if (bitnet_status s = check_gemm_args(x_q, scale, M, packed, w_scale, N, K, y, g_static_scratch_dummy))
    return s;
  if (!aligned(acc, 4)) return BITNET_ERR_ALIGNMENT;
  if (M > BITNET_GEMV_MAX_M || N > 0x7fffffff || K > 0x7fffffff) return BITNET_ERR_SHAPE;
  const size_t need = bitnet_gemv_workspace_bytes(M, N, K);
  if (need == 0) return BITNET_ERR_SHAPE;
  if (need > BITNET_GEMV_STATIC_SCRATCH_BYTES) return BITNET_ERR_TOO_LARGE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  void *scratch = nullptr;
  if (bitnet_status s = static_scratch_address(&scratch)) return s;
  // The array keeps whatever the previous call left.  That is harmless: the
  // GEMV takes its workspace with any contents and zeroes, in stream order,
  // the part it accumulates into (the stream-K partial sums and tickets).
  return bitnet_w2a8_gemv(x_q, scale, M, packed, w_scale, N, K, y, acc, scratch, need, stream);
}

size_t bitnet_bitlinear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || !shape_ok(N, K) || M > kMaxElems / K || M > kMaxElems / N) return 0;
  const size_t base = M <= BITNET_GEMV_MAX_M ? plan_gemv(M, N, K, 148).ws_bytes : gemm_workspace_bytes(M, N, K);
  // + int8 activations and scales for the unfused fallback
  return base + (((size_t)M * (size_t)K + 255) & ~(size_t)255) + (((size_t)M * 4 + 255) & ~(size_t)255);
}

int bitnet_bitlinear(const void *x, int dtype, int64_t M, const uint8_t *packed, const float *w_scale, int64_t N,
                     int64_t K, float *y, int8_t *x_q, float *scale, int32_t *acc, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || !shape_ok(N, K) || M > kMaxElems / K || M > kMaxElems / N) return BITNET_ERR_SHAPE;
  if (N > 0x7fffffff || K > 0x7fffffff || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  const size_t esz = dtype == BITNET_F32 ? 4 : 2;
  if (!aligned(x, esz) || !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(scale, 4) || !aligned(acc, 4))
    return BITNET_ERR_ALIGNMENT;
  const size_t need = bitnet_bitlinear_workspace_bytes(M, N, K);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;

  const bool fused = aligned(x, 16) && (K % 64 == 0) && K >= kStageK && aligned(packed, 16) && aligned(x_q, 16);
  const bool bf = dtype == BITNET_BF16;
  if (fused && ldg_ok(M, K, packed)) {
    return bf ? launch_gemv_ldg<__nv_bfloat16>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N, K, y, acc, d,
                                               stream)
              : launch_gemv_ldg<float>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N, K, y, acc, d, stream);
  }
  if (fused && rows_ok(M, K) && !two_on_tc(M, N, K, packed)) {
    return bf ? launch_gemv_rows<__nv_bfloat16>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N, K, y, acc, d,
                                                stream)
              : launch_gemv_rows<float>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N, K, y, acc, d, stream);
  }
  if (fused && K <= kTensorMaxK)
    return bitlinear_tc(x, bf, M, packed, w_scale, N, K, y, x_q, scale, acc, workspace, workspace_bytes, d,
                        PrepNorm{nullptr, -1.0f, nullptr}, stream);
  // Unfused: quantise into the caller's buffers or the workspace tail, then
  // the GEMV / GEMM entry points.
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t base = M <= BITNET_GEMV_MAX_M ? plan_gemv(M, N, K, d->sms).ws_bytes : gemm_workspace_bytes(M, N, K);
  int8_t *xq_buf = x_q ? x_q : reinterpret_cast<int8_t *>(ws + base);
  float *s_buf = scale ? scale : reinterpret_cast<float *>(ws + base + (((size_t)M * (size_t)K + 255) & ~(size_t)255));
  if (int st = bitnet_quant_act(x, dtype, M, K, xq_buf, s_buf, stream)) return st;
  if (M <= BITNET_GEMV_MAX_M)
    return bitnet_w2a8_gemv(xq_buf, s_buf, M, packed, w_scale, N, K, y, acc, workspace, base, stream);
  return bitnet_w2a8_gemm(xq_buf, s_buf, M, packed, w_scale, N, K, y, acc, workspace, base, stream);
}

}  // extern "C"

namespace {

// The fused BitLinear on the tensor cores (M >= 3, and two tokens on a large
// matrix with long rows): one prep kernel
// quantises x (after an RMSNorm when norm.eps >= 0) straight into the
// operand layout, then the GEMV (M <= 64) or the GEMM.
bitnet_status bitlinear_tc(const void *x, bool bf, int64_t M, const uint8_t *packed, const float *w_scale, int64_t N,
                           int64_t K, float *y, int8_t *x_q, float *scale, int32_t *acc, void *workspace,
                           size_t workspace_bytes, const DeviceInfo *d, const PrepNorm &norm, cudaStream_t stream) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  {
    uint32_t *xb;
    int32_t *xsum;
    float *fscale;
    GemvPlan pl = {};
    if (M <= BITNET_GEMV_MAX_M) {
      pl = plan_gemv(M, N, K, d->sms);
      xb = reinterpret_cast<uint32_t *>(ws + pl.ws_prep_xb);
      xsum = reinterpret_cast<int32_t *>(ws + pl.ws_prep_sums);
    } else {
      xb = reinterpret_cast<uint32_t *>(ws);
      xsum = reinterpret_cast<int32_t *>(ws + gemm_xb_bytes(M, K));
    }
    fscale = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xsum) + (size_t)M * 4);
    const bool gemv = M <= BITNET_GEMV_MAX_M;
    const GemmSplit sp = gemv ? GemmSplit{} : gemm_plan_split(M, N, K, workspace_bytes, d);
    uint8_t *part = ws + gemm_part_offset(M, K);
    const dim3 pgrid = gemv ? dim3(prep_grid(M, pl)) : dim3((unsigned)M + gemm_zero_ctas(sp));
    uint4 *zero = gemv ? static_cast<uint4 *>(workspace) : reinterpret_cast<uint4 *>(part);
    const int64_t zero_n16 = gemv ? (int64_t)(pl.ws_zero_bytes / 16) : (int64_t)(sp.part_bytes / 16);
    const int trows = gemv ? gemv_mma_rows(M) : 0;
    bitnet_status st =
        bf ? launch(fused_prep_kernel<__nv_bfloat16>, pgrid, dim3(256), 0, stream,
                    static_cast<const __nv_bfloat16 *>(x), w_scale, K, xb, xsum, fscale, x_q, scale, M, zero, zero_n16,
                    trows, norm, PrepGroups{nullptr, 0, 0})
           : launch(fused_prep_kernel<float>, pgrid, dim3(256), 0, stream, static_cast<const float *>(x), w_scale, K,
                    xb, xsum, fscale, x_q, scale, M, zero, zero_n16, trows, norm, PrepGroups{nullptr, 0, 0});
    if (st) return st;
    if (M <= BITNET_GEMV_MAX_M)
      return launch_gemv_mma(nullptr, nullptr, M, packed, w_scale, N, K, y, acc, workspace, pl, d, stream);
    return launch_gemm_tc(xb, xsum, fscale, M, packed, N, K, y, acc, sp, part, d, stream);
  }
}

}  // namespace

extern "C" {

int bitnet_rmsnorm_quant_act(const void *x, int dtype, int64_t M, int64_t K, const float *g, float eps, int8_t *x_q,
                             float *scale, float *h, float *ms, cudaStream_t stream) {
  if (!x || !x_q || !scale) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.0f) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || K % 8 != 0 || M > kMaxElems / K || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(x_q, 8) || !aligned(scale, 4) || !aligned(h, 16) ||
      !aligned(ms, 4))
    return BITNET_ERR_ALIGNMENT;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  return dtype == BITNET_F32
             ? launch(rmsnorm_quant_kernel<float>, dim3((unsigned)M), dim3(256), 0, stream,
                      static_cast<const float *>(x), K, g, eps, x_q, scale, h, ms)
             : launch(rmsnorm_quant_kernel<__nv_bfloat16>, dim3((unsigned)M), dim3(256), 0, stream,
                      static_cast<const __nv_bfloat16 *>(x), K, g, eps, x_q, scale, h, ms);
}

int bitnet_bitlinear_rmsnorm(const void *x, int dtype, int64_t M, const float *g, float eps, const uint8_t *packed,
                             const float *w_scale, int64_t N, int64_t K, float *y, int8_t *x_q, float *scale,
                             float *ms, int32_t *acc, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.0f) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || !shape_ok(N, K) || K % 8 != 0 || M > kMaxElems / K || M > kMaxElems / N) return BITNET_ERR_SHAPE;
  if (N > 0x7fffffff || K > 0x7fffffff || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(g, 16) || !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(scale, 4) ||
      !aligned(ms, 4) || !aligned(acc, 4) || !aligned(x_q, 8))
    return BITNET_ERR_ALIGNMENT;
  const size_t need = bitnet_bitlinear_workspace_bytes(M, N, K);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  const bool bf = dtype == BITNET_BF16;
  // M >= 3 (and two tokens on a large matrix with long rows) on the tensor
  // cores: the RMSNorm, the quantisation and the
  // operand layout in one prep kernel, then the GEMV / GEMM
  if ((M >= 3 || two_on_tc(M, N, K, packed)) && K % 64 == 0 && K >= kStageK && K <= kTensorMaxK &&
      aligned(packed, 16) && aligned(x_q, 16))
    return bitlinear_tc(x, bf, M, packed, w_scale, N, K, y, x_q, scale, acc, workspace, workspace_bytes, d,
                        PrepNorm{g, eps, ms}, stream);
  // otherwise: RMSNorm + quantisation into int8 (the caller's buffers or the
  // workspace tail), then the GEMV / GEMM entry points
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t base = M <= BITNET_GEMV_MAX_M ? plan_gemv(M, N, K, d->sms).ws_bytes : gemm_workspace_bytes(M, N, K);
  int8_t *xq_buf = x_q ? x_q : reinterpret_cast<int8_t *>(ws + base);
  float *s_buf = scale ? scale : reinterpret_cast<float *>(ws + base + (((size_t)M * (size_t)K + 255) & ~(size_t)255));
  if (int st = bitnet_rmsnorm_quant_act(x, dtype, M, K, g, eps, xq_buf, s_buf, nullptr, ms, stream)) return st;
  if (M <= BITNET_GEMV_MAX_M)
    return bitnet_w2a8_gemv(xq_buf, s_buf, M, packed, w_scale, N, K, y, acc, workspace, base, stream);
  return bitnet_w2a8_gemm(xq_buf, s_buf, M, packed, w_scale, N, K, y, acc, workspace, base, stream);
}

size_t bitnet_bitlinear_swiglu_workspace_bytes(int64_t M, int64_t I, int64_t K) {
  const size_t base = bitnet_bitlinear_workspace_bytes(M, I, K);
  if (base == 0) return 0;
  // + y_gate and y_up for the unfused fallback
  return base + 2 * (((size_t)M * (size_t)I * 4 + 255) & ~(size_t)255);
}

int bitnet_bitlinear_swiglu(const void *x, int dtype, int64_t M, const uint8_t *packed_gate,
                            const float *w_scale_gate, const uint8_t *packed_up, const float *w_scale_up, int64_t I,
                            int64_t K, float *out, int8_t *x_q, float *scale, int32_t *acc_gate, int32_t *acc_up,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !packed_gate || !w_scale_gate || !packed_up || !w_scale_up || !out) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || !shape_ok(I, K) || M > kMaxElems / K || M > kMaxElems / I) return BITNET_ERR_SHAPE;
  if (I > 0x7fffffff || K > 0x7fffffff || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  const size_t esz = dtype == BITNET_F32 ? 4 : 2;
  if (!aligned(x, esz) || !aligned(w_scale_gate, 4) || !aligned(w_scale_up, 4) || !aligned(out, 4) ||
      !aligned(scale, 4) || !aligned(acc_gate, 4) || !aligned(acc_up, 4))
    return BITNET_ERR_ALIGNMENT;
  const size_t need = bitnet_bitlinear_swiglu_workspace_bytes(M, I, K);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;

  // One streaming kernel for one or two tokens: both matrices' rows in each
  // stage, silu(gate) * up in the epilogue.
  const bool fused = aligned(x, 16) && (K % 64 == 0) && K >= kStageK && aligned(packed_gate, 16) &&
                     aligned(packed_up, 16) && aligned(x_q, 16);
  if (fused && ldg_ok(M, K, packed_gate)) {
    return dtype == BITNET_BF16
               ? launch_gemv_ldg<__nv_bfloat16, kLdgSwiGLU>(nullptr, nullptr, x, x_q, scale, M, packed_gate, w_scale_gate,
                                                      I, K, out, acc_gate, d, stream, packed_up, w_scale_up, acc_up)
               : launch_gemv_ldg<float, kLdgSwiGLU>(nullptr, nullptr, x, x_q, scale, M, packed_gate, w_scale_gate, I, K,
                                              out, acc_gate, d, stream, packed_up, w_scale_up, acc_up);
  }
  // Otherwise: the gate BitLinear (quantising x), the up matrix on the same
  // int8 activations, then silu(gate) * up elementwise -- the same fp32
  // operations as the streaming kernel's epilogue.
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t base = bitnet_bitlinear_workspace_bytes(M, I, K);
  const size_t ybytes = ((size_t)M * (size_t)I * 4 + 255) & ~(size_t)255;
  float *yg = reinterpret_cast<float *>(ws + base);
  float *yu = reinterpret_cast<float *>(ws + base + ybytes);
  // the gate call's int8 activations and scales: the caller's buffers or the
  // tail of the gate call's own workspace (the part the gate call uses only
  // when it is given no buffers of its own)
  const size_t mm_ws = M <= BITNET_GEMV_MAX_M ? plan_gemv(M, I, K, d->sms).ws_bytes : gemm_workspace_bytes(M, I, K);
  int8_t *xq_buf = x_q ? x_q : reinterpret_cast<int8_t *>(ws + mm_ws);
  float *s_buf = scale ? scale : reinterpret_cast<float *>(ws + mm_ws + (((size_t)M * (size_t)K + 255) & ~(size_t)255));
  if (int st = bitnet_bitlinear(x, dtype, M, packed_gate, w_scale_gate, I, K, yg, xq_buf, s_buf, acc_gate, workspace,
                                base, stream))
    return st;
  const int st = M <= BITNET_GEMV_MAX_M
                     ? bitnet_w2a8_gemv(xq_buf, s_buf, M, packed_up, w_scale_up, I, K, yu, acc_up, workspace, mm_ws,
                                        stream)
                     : bitnet_w2a8_gemm(xq_buf, s_buf, M, packed_up, w_scale_up, I, K, yu, acc_up, workspace, mm_ws,
                                        stream);
  if (st) return st;
  const int64_t n = M * I;
  const unsigned grid = (unsigned)std::min<int64_t>((int64_t)d->sms * 8, cdiv(n, 256));
  return launch(swiglu_kernel, dim3(grid), dim3(256), 0, stream, (const float *)yg, (const float *)yu, out, n);
}

// ------------------------------------------------- group-wise weight scales --

namespace {
bool group_shape_ok(int64_t N, int64_t K, int64_t G) {
  return shape_ok(N, K) && G > 0 && G % 4 == 0 && K % G == 0 && K <= 0x7fffffff && N <= 0x7fffffff;
}

// The grouped tensor-core path's shape and alignment rules.
bool grouped_tc_ok(int64_t M, int64_t N, int64_t K, int64_t G, const void *packed, const void *x, const void *x_q) {
  (void)M;
  (void)N;
  return K % 64 == 0 && K >= kStageK && K <= kTensorMaxK && mma_group_ok(K, G) && aligned(packed, 16) &&
         aligned(x, 16) && aligned(x_q, 16);
}

// Group-scaled matmul on the tensor cores for M >= 3, 64 tokens at a time
// (chunks of equal size, each >= 3 tokens): per chunk the prep kernel (the
// fused one from bf16 / fp32 x, else from int8 x_q) writes the operand
// layout and the group sums, then the grouped GEMV.
bitnet_status grouped_tc(const void *x, bool bf, const int8_t *x_q_in, const float *scale_in, int64_t M,
                         const uint8_t *packed, const float *gscale, int64_t N, int64_t K, int64_t G, float *y,
                         int8_t *xq_out, float *scale_out, int32_t *acc_g, void *workspace, const DeviceInfo *d,
                         cudaStream_t stream) {
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const int64_t NG = K / G;
  const int64_t chunks = cdiv(M, BITNET_GEMV_MAX_M);
  for (int64_t c = 0; c < chunks; ++c) {
    const int64_t m0 = M * c / chunks, Mc = M * (c + 1) / chunks - m0;
    const GemvPlan pl = plan_gemv(Mc, N, K, d->sms);
    int32_t *xsumg = reinterpret_cast<int32_t *>(ws + pl.ws_bytes);
    const GroupedArgs ga{gscale, acc_g ? acc_g + m0 * N * NG : nullptr, G, xsumg};
    if (x_q_in) {
      if (bitnet_status st = launch_gemv_mma(x_q_in + m0 * K, scale_in + m0, Mc, packed, gscale, N, K, y + m0 * N,
                                             nullptr, workspace, pl, d, stream, &ga))
        return st;
      continue;
    }
    uint32_t *xb = reinterpret_cast<uint32_t *>(ws + pl.ws_prep_xb);
    int32_t *xsum = reinterpret_cast<int32_t *>(ws + pl.ws_prep_sums);
    float *fscale = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(xsum) + (size_t)Mc * 4);
    const PrepGroups grp{xsumg, (int)G, (int)NG};
    const PrepNorm nonorm{nullptr, -1.0f, nullptr};
    int8_t *xq_c = xq_out ? xq_out + m0 * K : nullptr;
    float *s_c = scale_out ? scale_out + m0 : nullptr;
    const dim3 pgrid(prep_grid(Mc, pl));
    bitnet_status st =
        bf ? launch(fused_prep_kernel<__nv_bfloat16>, pgrid, dim3(256), 0, stream,
                    static_cast<const __nv_bfloat16 *>(x) + m0 * K, gscale, K, xb, xsum, fscale, xq_c, s_c, Mc,
                    static_cast<uint4 *>(workspace), (int64_t)(pl.ws_zero_bytes / 16), gemv_mma_rows(Mc), nonorm, grp)
           : launch(fused_prep_kernel<float>, pgrid, dim3(256), 0, stream, static_cast<const float *>(x) + m0 * K,
                    gscale, K, xb, xsum, fscale, xq_c, s_c, Mc, static_cast<uint4 *>(workspace),
                    (int64_t)(pl.ws_zero_bytes / 16), gemv_mma_rows(Mc), nonorm, grp);
    if (st) return st;
    if (bitnet_status s2 = launch_gemv_mma(nullptr, nullptr, Mc, packed, gscale, N, K, y + m0 * N, nullptr, workspace,
                                           pl, d, stream, &ga))
      return s2;
  }
  return BITNET_OK;
}
}  // namespace

int bitnet_pack_weights_grouped(const void *W, int dtype, int64_t N, int64_t K, int64_t G, float alpha, float eps,
                                uint8_t *packed, float *w_scale, float *absmean, cudaStream_t stream) {
  if (!W || !packed || !w_scale) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(eps)) return BITNET_ERR_INVALID_ARG;
  if (!group_shape_ok(N, K, G)) return BITNET_ERR_SHAPE;
  if (!aligned(W, dtype == BITNET_F32 ? 4 : 2) || !aligned(w_scale, 4) || !aligned(absmean, 4))
    return BITNET_ERR_ALIGNMENT;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  const int64_t groups = N * (K / G);
  const dim3 grid((unsigned)cdiv(groups, kPackThreads));
  return dtype == BITNET_F32
             ? launch(pack_grouped_kernel<float>, grid, dim3(kPackThreads), 0, stream, static_cast<const float *>(W),
                      groups, G, alpha, eps, packed, w_scale, absmean)
             : launch(pack_grouped_kernel<__nv_bfloat16>, grid, dim3(kPackThreads), 0, stream,
                      static_cast<const __nv_bfloat16 *>(W), groups, G, alpha, eps, packed, w_scale, absmean);
}

int bitnet_w2a8_grouped(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                        const float *w_scale, int64_t N, int64_t K, int64_t G, float *y, int32_t *acc_g,
                        cudaStream_t stream) {
  if (!x_q || !scale || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || M > 0x7fffffff || !group_shape_ok(N, K, G) || M > kMaxElems / K || M > kMaxElems / N)
    return BITNET_ERR_SHAPE;
  if (!aligned(scale, 4) || !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(acc_g, 4))
    return BITNET_ERR_ALIGNMENT;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  if (ldg_ok(M, K, packed) && aligned(x_q, 16) && ldg_group_ok(K, G))
    return launch_gemv_ldg<int8_t, kLdgGrouped>(x_q, scale, nullptr, nullptr, nullptr, M, packed, w_scale, N, K, y,
                                                acc_g, d, stream, nullptr, nullptr, nullptr, G);
  const unsigned grid = (unsigned)std::min<int64_t>((int64_t)d->sms * 16, cdiv(M * N, kGroupedWarps));
  return launch(grouped_generic_kernel, dim3(grid), dim3(kGroupedWarps * 32), 0, stream, x_q, scale, packed, w_scale,
                M, N, K, G, y, acc_g);
}

size_t bitnet_bitlinear_grouped_workspace_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || M > kMaxElems / K) return 0;
  return (((size_t)M * (size_t)K + 255) & ~(size_t)255) + (((size_t)M * 4 + 255) & ~(size_t)255);
}

int bitnet_bitlinear_grouped(const void *x, int dtype, int64_t M, const uint8_t *packed, const float *w_scale,
                             int64_t N, int64_t K, int64_t G, float *y, int8_t *x_q, float *scale, int32_t *acc_g,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (dtype != BITNET_F32 && dtype != BITNET_BF16) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || M > 0x7fffffff || !group_shape_ok(N, K, G) || M > kMaxElems / K || M > kMaxElems / N)
    return BITNET_ERR_SHAPE;
  const size_t esz = dtype == BITNET_F32 ? 4 : 2;
  if (!aligned(x, esz) || !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(scale, 4) || !aligned(acc_g, 4))
    return BITNET_ERR_ALIGNMENT;
  const size_t need = bitnet_bitlinear_grouped_workspace_bytes(M, K);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  // one streaming kernel (quantisation in its prologue) for one or two tokens
  if (aligned(x, 16) && aligned(x_q, 16) && ldg_ok(M, K, packed) && ldg_group_ok(K, G)) {
    return dtype == BITNET_BF16
               ? launch_gemv_ldg<__nv_bfloat16, kLdgGrouped>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N,
                                                             K, y, acc_g, d, stream, nullptr, nullptr, nullptr, G)
               : launch_gemv_ldg<float, kLdgGrouped>(nullptr, nullptr, x, x_q, scale, M, packed, w_scale, N, K, y,
                                                     acc_g, d, stream, nullptr, nullptr, nullptr, G);
  }
  // three or more tokens on the tensor cores when the workspace holds that
  // path's layout: the fused prep kernel (quantisation, operand layout, group
  // sums) and the grouped GEMV, 64 tokens at a time
  if (M >= 3 && grouped_tc_ok(M, N, K, G, packed, x, x_q) && workspace_bytes >= grouped_tc_ws_bytes(M, N, K, G))
    return grouped_tc(x, dtype == BITNET_BF16, nullptr, nullptr, M, packed, w_scale, N, K, G, y, x_q, scale, acc_g,
                      workspace, d, stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int8_t *xq_buf = x_q ? x_q : reinterpret_cast<int8_t *>(ws);
  float *s_buf = scale ? scale : reinterpret_cast<float *>(ws + (((size_t)M * (size_t)K + 255) & ~(size_t)255));
  if (int st = bitnet_quant_act(x, dtype, M, K, xq_buf, s_buf, stream)) return st;
  return bitnet_w2a8_grouped(xq_buf, s_buf, M, packed, w_scale, N, K, G, y, acc_g, stream);
}

size_t bitnet_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t G) {
  if (M <= 0 || !group_shape_ok(N, K, G) || M > kMaxElems / K || M > kMaxElems / N) return 0;
  const size_t base = bitnet_bitlinear_grouped_workspace_bytes(M, K);
  if (M < 3 || !mma_group_ok(K, G) || K % 64 != 0 || K < kStageK || K > kTensorMaxK) return base;
  return std::max(base, grouped_tc_ws_bytes(M, N, K, G));
}

int bitnet_w2a8_grouped_ws(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                           const float *w_scale, int64_t N, int64_t K, int64_t G, float *y, int32_t *acc_g,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!x_q || !scale || !packed || !w_scale || !y) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || M > 0x7fffffff || !group_shape_ok(N, K, G) || M > kMaxElems / K || M > kMaxElems / N)
    return BITNET_ERR_SHAPE;
  if (!aligned(scale, 4) || !aligned(w_scale, 4) || !aligned(y, 4) || !aligned(acc_g, 4))
    return BITNET_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < bitnet_grouped_workspace_bytes(M, N, K, G) || !aligned(workspace, 256))
    return BITNET_ERR_WORKSPACE;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  if (M >= 3 && grouped_tc_ok(M, N, K, G, packed, x_q, x_q))
    return grouped_tc(nullptr, false, x_q, scale, M, packed, w_scale, N, K, G, y, nullptr, nullptr, acc_g, workspace, d,
                      stream);
  return bitnet_w2a8_grouped(x_q, scale, M, packed, w_scale, N, K, G, y, acc_g, stream);
}

// ------------------------------------------- training-time (fake-quant) BitLinear --

namespace {
size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }
}  // namespace

size_t bitnet_bitlinear_fake_quant_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const size_t pk = bitnet_pack_workspace_bytes(N, K);
  const size_t bl = bitnet_bitlinear_workspace_bytes(M, N, K);
  const size_t gr = bitnet_bitlinear_grouped_workspace_bytes(M, K);
  if (pk == 0 || bl == 0 || gr == 0) return 0;
  return round256((size_t)(N * K / 4)) + 256 + std::max(pk, std::max(bl, gr));
}

int bitnet_bitlinear_fake_quant(const void *W, int w_dtype, const void *x, int x_dtype, int64_t M, int64_t N,
                                int64_t K, float alpha, float eps, const float *weight_scale, float *y,
                                uint8_t *packed, float *beta, int8_t *x_q, float *scale, int32_t *acc,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!W || !x || !y) return BITNET_ERR_INVALID_ARG;
  if ((w_dtype != BITNET_F32 && w_dtype != BITNET_BF16) || (x_dtype != BITNET_F32 && x_dtype != BITNET_BF16))
    return BITNET_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(eps)) return BITNET_ERR_INVALID_ARG;
  if (M <= 0 || !shape_ok(N, K) || M > kMaxElems / K || M > kMaxElems / N) return BITNET_ERR_SHAPE;
  if (N > 0x7fffffff || K > 0x7fffffff || M > 0x7fffffff) return BITNET_ERR_SHAPE;
  if (!aligned(beta, 4) || !aligned(weight_scale, 4) || !aligned(y, 4)) return BITNET_ERR_ALIGNMENT;
  const size_t need = bitnet_bitlinear_fake_quant_workspace_bytes(M, N, K);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return BITNET_ERR_WORKSPACE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t pbytes = round256((size_t)(N * K / 4));
  uint8_t *pk = packed ? packed : ws;
  float *bt = beta ? beta : reinterpret_cast<float *>(ws + pbytes);
  float *am = reinterpret_cast<float *>(ws + pbytes + 128);
  uint8_t *tail = ws + pbytes + 256;
  const size_t tail_bytes = workspace_bytes - pbytes - 256;
  // the shadow weights, ternarised and packed for this call ([Deep-dive] §2.2, §3.3)
  if (int st = bitnet_pack_weights(W, w_dtype, N, K, alpha, eps, pk, bt, am, tail, tail_bytes, stream)) return st;
  // the forward on them: with a per-output weight_scale (the training module's
  // learned scale) as a one-group-per-row scale, else with beta
  if (weight_scale)
    return bitnet_bitlinear_grouped(x, x_dtype, M, pk, weight_scale, N, K, K, y, x_q, scale, acc, tail, tail_bytes,
                                    stream);
  return bitnet_bitlinear(x, x_dtype, M, pk, bt, N, K, y, x_q, scale, acc, tail, tail_bytes, stream);
}

int bitnet_selftest_wait_timeout(int64_t limit_ns, cudaStream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000) return BITNET_ERR_INVALID_ARG;
  DeviceInfo *d;
  if (bitnet_status s = device_info(&d)) return s;
  return launch(selftest_wait_kernel, dim3(1), dim3(32), 0, stream, (unsigned long long)limit_ns);
}

int bitnet_check_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BITNET_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return BITNET_ERR_CUDA;
  if (v == 0) return BITNET_OK;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return BITNET_ERR_CUDA;
  return BITNET_ERR_TIMEOUT;
}

}  // extern "C"

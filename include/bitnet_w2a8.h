/*
 * bitnet_w2a8.h -- C ABI of the BitNet b1.58 W2A8 ternary-matmul library for
 * NVIDIA B300 (sm_103a).
 *
 * The operations follow these pages (cited by title and section):
 *   [Deep-dive] "BitNet 深度拆解：当大模型被压到 1.58 bit——从三元权重、BitLinear
 *               到 bitnet.cpp 的端侧推理革命（2026）"
 *   [Review]    "BitNet 深度解析：1.58-bit 大模型如何跑向普通 CPU"
 *
 * Conventions shared by every call
 *   - Device pointers are CUDA device (or managed) memory owned by the caller;
 *     host pointers are named as such.  The library allocates no device
 *     memory: scratch space is passed in as a caller-owned workspace (the
 *     one exception is the fixed array of bitnet_w2a8_gemv_static_scratch,
 *     part of the loaded module, not a runtime allocation).
 *   - Every call validates its arguments on the host before enqueuing
 *     anything.  On a non-zero status nothing has been enqueued.
 *   - Calls are asynchronous and stream-ordered on `stream` (0 = legacy
 *     default stream).  All scalars the kernels consume (beta, scales) live in
 *     device memory, so calls chain without host synchronisation.
 *   - Kernels that wait on an on-chip barrier give up after ~1.5 s, set a
 *     device error word and return; bitnet_check_device_error() reports it.
 *   - Shapes are int64; every tensor is dense and row-major.
 *   - The library is thread-compatible: concurrent calls on different
 *     streams must use different workspaces.
 */
#ifndef BITNET_W2A8_H
#define BITNET_W2A8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
  BITNET_OK = 0,
  BITNET_ERR_INVALID_ARG = 1, /* null pointer, unknown dtype, non-finite alpha/eps */
  BITNET_ERR_SHAPE = 2,       /* M/N/K <= 0, K % 4 != 0, gemv M > 64, size overflow */
  BITNET_ERR_ALIGNMENT = 3,   /* a float/int32 pointer not aligned to its element size */
  BITNET_ERR_UNSUPPORTED = 4, /* no sm_103 device / kernel image for this device */
  BITNET_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  BITNET_ERR_TIMEOUT = 6,     /* a device-side bounded wait expired */
  BITNET_ERR_WORKSPACE = 7,   /* workspace null or smaller than required */
  BITNET_ERR_TOO_LARGE = 8    /* needs more scratch than the library's fixed array holds */
} bitnet_status;

/* Element type of floating-point inputs. */
typedef enum { BITNET_F32 = 0, BITNET_BF16 = 1 } bitnet_dtype;

/* Largest token count bitnet_w2a8_gemv accepts (decode path). */
#define BITNET_GEMV_MAX_M 64

/* Human-readable name of a status code (static storage, never NULL). */
const char *bitnet_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int bitnet_version(void);

/* Workspace bytes bitnet_pack_weights needs for an [N, K] matrix. */
size_t bitnet_pack_workspace_bytes(int64_t N, int64_t K);

/*
 * bitnet_pack_weights -- offline absmean ternarisation and 2-bit packing.
 * [Deep-dive] §2.2 (absmean_quantize), §2.3 (beta), §3.3 (pack_ternary).
 *
 *   W        device, [N, K] row-major, dtype BITNET_F32 or BITNET_BF16
 *            (bf16 is widened exactly to fp32 first).
 *   alpha,eps host scalars (the pages use 1 and 1e-8).
 *   packed   device, N*K/4 bytes out.  Element i = n*K + k of the flattened
 *            matrix is field i%4 (bits 2*(i%4)..+1) of byte i/4, holding code
 *            w+1 in {0,1,2}.  Row n occupies bytes [n*K/4, (n+1)*K/4).
 *   beta     device, 1 float out: mean(|W_ternary|) = (#nonzero)/(N*K).
 *   absmean  device, 1 float out (may be NULL): mean|W| as used for gamma.
 *   workspace device, >= bitnet_pack_workspace_bytes(N, K) bytes, any contents.
 *
 * Arithmetic: S = sum|w| in fp64 over 4096-element chunks of the flattened
 * matrix, each summed in order, chunk sums added in order; mean = (float)(S/n);
 * gamma = 1/(fl32(alpha*mean) + eps) in fp32; code = clamp(rint(fl32(gamma*w)),
 * -1, 1) + 1 with round-half-even (a NaN product gives code 1).
 * Errors: INVALID_ARG (null W/packed/beta, bad dtype, non-finite alpha or eps),
 * SHAPE (N, K <= 0, K % 4 != 0), ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_pack_weights(const void *W, int dtype, int64_t N, int64_t K, float alpha, float eps,
                        uint8_t *packed, float *beta, float *absmean, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/*
 * bitnet_quant_act -- per-token absmax quantisation of activations to int8.
 * [Deep-dive] §2.2 (absmax_quantize with bits = 8, qmax = 127).
 *
 *   x      device, [M, K] row-major, BITNET_F32 or BITNET_BF16.
 *   x_q    device, [M, K] int8 out: clamp(rint(fl32(fl32(x/s) * 127)), -127, 127).
 *   scale  device, [M] float out: s = max(max_k |x[m,k]|, fl32(1e-8)) (the
 *          absmax itself, not absmax/127).
 * Errors: INVALID_ARG, SHAPE (M, K <= 0), ALIGNMENT, UNSUPPORTED, CUDA.
 */
int bitnet_quant_act(const void *x, int dtype, int64_t M, int64_t K, int8_t *x_q, float *scale,
                     cudaStream_t stream);

/* Workspace bytes bitnet_w2a8_gemv needs (0 for shapes the call rejects). */
size_t bitnet_gemv_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * bitnet_w2a8_gemv -- decode-path ternary matmul with fused dequantisation.
 * [Deep-dive] §3.1 (integer-domain matmul of W_ternary and X_q), §1 (the
 * -1/0/+1 products), §2.3 (Y = acc * beta * act_scale); [Review] §03.3 (a W2A8
 * GEMV is the GPU decode kernel of this method).
 *
 *   x_q      device, [M, K] int8 (from bitnet_quant_act), 1 <= M <= 64.
 *   scale    device, [M] float: per-token absmax s_m.
 *   packed   device, [N, K/4] bytes in the bitnet_pack_weights format.
 *   w_scale  device, 1 float: the weight scale (beta, or absmean).
 *   y        device, [M, N] float out: y = acc * (w_scale * s_m / 127) in fp32.
 *   acc      device, [M, N] int32 out or NULL: acc = sum_k (code-1) * x_q,
 *            exact.
 *   workspace device, >= bitnet_gemv_workspace_bytes(M, N, K) bytes, 16-byte
 *            aligned, any contents: the call zeroes, in stream order, the
 *            part it accumulates into.
 * Packed codes equal to 3 never come out of bitnet_pack_weights; the GEMV
 * does not define a result for them.
 * Errors: INVALID_ARG, SHAPE (M outside 1..64, N, K <= 0, K % 4 != 0),
 * ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_w2a8_gemv(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                     const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes bitnet_w2a8_gemm needs. */
size_t bitnet_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * bitnet_w2a8_gemm -- prefill-path ternary matmul (same operation and
 * arguments as bitnet_w2a8_gemv, any M >= 1; tuned for M >= 256) on the
 * tcgen05 tensor cores with TMEM accumulators, 128 weight rows x 256 tokens
 * per tile.  When the tiles leave a last wave less than half full, those
 * tiles are split by K across all SMs and their exact int32 partial sums
 * meet in the workspace.  Same citations as the GEMV.
 *   workspace device, >= bitnet_gemm_workspace_bytes(M, N, K) bytes,
 *             256-byte aligned, any contents (the call prepares what it
 *             uses, in stream order; no state is kept between calls).
 * Shapes outside the tensor-core path (K % 64 != 0, K < 512, K > 65536,
 * unaligned pointers) run a plain CUDA-core kernel with the same results.
 * Errors: as bitnet_w2a8_gemv (any M >= 1).
 */
int bitnet_w2a8_gemm(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                     const float *w_scale, int64_t N, int64_t K, float *y, int32_t *acc,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes bitnet_bitlinear needs. */
size_t bitnet_bitlinear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * bitnet_bitlinear -- the whole BitLinear forward of [Deep-dive] §3.1 in one
 * call: per-token absmax int8 quantisation of x (§2.2), the ternary integer
 * product and the rescale y = acc * w_scale * s_m / 127 (§2.3).  The
 * quantisation is fused into the matmul's prologue ([Deep-dive] §5.3 names
 * this fusion as a key optimisation): for one or two tokens one kernel
 * (except two tokens with K > 4096 on a matrix of N * K >= 2^27 weights);
 * otherwise one kernel that quantises straight into the tensor-core operand
 * layout plus the GEMV (M <= 64) or GEMM kernel.  Results are bit-identical to
 * bitnet_quant_act followed by bitnet_w2a8_gemv / bitnet_w2a8_gemm.
 *
 *   x        device, [M, K] row-major, BITNET_F32 or BITNET_BF16.
 *   packed, w_scale, N, K, y, acc: as bitnet_w2a8_gemv.
 *   x_q      device, [M, K] int8 out, or NULL.
 *   scale    device, [M] float out (per-token absmax), or NULL.
 *   workspace device, >= bitnet_bitlinear_workspace_bytes(M, N, K) bytes,
 *            256-byte aligned, any contents.
 * Shapes the fused kernels do not take (K % 64 != 0, K < 512, unaligned
 * pointers) run quant_act and the matmul entry points in sequence.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_bitlinear(const void *x, int dtype, int64_t M, const uint8_t *packed, const float *w_scale,
                     int64_t N, int64_t K, float *y, int8_t *x_q, float *scale, int32_t *acc,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * bitnet_rmsnorm_quant_act -- RMSNorm, then the per-token absmax int8
 * quantisation of the normalised activations: the input side of a BitLinear
 * inside the BitTransformer block of [Deep-dive] §3.1 (the block applies an
 * RMSNorm before the gate/up projections, in fp32 per §6.5), followed by the
 * absmax quantisation of §2.2 applied to h instead of x.
 *
 * Per token m: S = sum_k x[m,k]^2 in fp64 (each square exact), ms =
 * fl32(S / K), r = fl(1 / fl(sqrt(fl(ms + eps)))), h[k] = fl(fl(x[m,k] * r)
 * * g[k]) (fl(x[m,k] * r) when g is NULL), then scale[m] = max(max_k |h|,
 * 1e-8) and x_q = clamp(rint(fl(fl(h / s) * 127)), -127, 127).  The fp64 sum
 * is a tree over the token's threads, so S may differ from another
 * summation order by at most (K - 1) * 2^-53 * S; ms can then be the
 * neighbouring fp32 value only when S / K lies that close to a rounding
 * boundary.
 *
 *   x        device, [M, K] row-major, BITNET_F32 or BITNET_BF16, 16-byte aligned.
 *   g        device, [K] float RMSNorm weight (16-byte aligned), or NULL for ones.
 *   eps      finite, >= 0 (nn.RMSNorm's fp32 default is 2^-23).
 *   x_q      device, [M, K] int8 out (8-byte aligned).
 *   scale    device, [M] float out: absmax of h.
 *   h        device, [M, K] float out (16-byte aligned), or NULL.
 *   ms       device, [M] float out: the mean squares, or NULL.
 * Errors: INVALID_ARG (null x / x_q / scale, dtype, eps), SHAPE (M, K <= 0,
 * K % 8 != 0), ALIGNMENT, UNSUPPORTED, CUDA.
 */
int bitnet_rmsnorm_quant_act(const void *x, int dtype, int64_t M, int64_t K, const float *g, float eps,
                             int8_t *x_q, float *scale, float *h, float *ms, cudaStream_t stream);

/*
 * bitnet_bitlinear_rmsnorm -- RMSNorm in front of the BitLinear forward:
 * y = BitLinear(h) with h = RMSNorm(x) formed as bitnet_rmsnorm_quant_act
 * forms it ([Deep-dive] §3.1, §5.3 fusion).  For M >= 3, and for two tokens
 * with K > 4096 and N * K >= 2^27 (K % 64 == 0, 512 <= K <= 65536), one
 * prep kernel computes the RMSNorm, the absmax
 * quantisation and the tensor-core operand layout, followed by the GEMV
 * (M <= 64) or GEMM kernel; otherwise bitnet_rmsnorm_quant_act runs first,
 * then the int8 GEMV / GEMM.  Results are bit-identical between the two
 * routes.
 *
 *   x, g, eps   as bitnet_rmsnorm_quant_act.
 *   packed, w_scale, N, K, y, acc: as bitnet_w2a8_gemv.
 *   x_q, scale  device outs (x_q 8-byte aligned), or NULL.
 *   ms          device, [M] float out (mean squares), or NULL.
 *   workspace   device, >= bitnet_bitlinear_workspace_bytes(M, N, K) bytes,
 *               256-byte aligned, any contents.
 * Errors: INVALID_ARG, SHAPE (also K % 8 != 0), ALIGNMENT, WORKSPACE,
 * UNSUPPORTED, CUDA.
 */
int bitnet_bitlinear_rmsnorm(const void *x, int dtype, int64_t M, const float *g, float eps,
                             const uint8_t *packed, const float *w_scale, int64_t N, int64_t K, float *y,
                             int8_t *x_q, float *scale, float *ms, int32_t *acc, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes bitnet_bitlinear_swiglu needs. */
size_t bitnet_bitlinear_swiglu_workspace_bytes(int64_t M, int64_t I, int64_t K);

/*
 * bitnet_bitlinear_swiglu -- the front half of the BitTransformer
 * feed-forward of [Deep-dive] §3.1, down(silu(gate(h)) * up(h)): two
 * BitLinears on the same activations and their SwiGLU product
 *   out[m, i] = silu(y_gate[m, i]) * y_up[m, i],  silu(z) = z / (1 + exp(-z)),
 * with y_gate, y_up formed exactly as bitnet_bitlinear forms y (x quantised
 * once) and the product in fp32: yg / (1 + expf(-yg)), then * yu, each
 * operation rounded to nearest.  The down projection is a plain
 * bitnet_bitlinear on `out` (BITNET_F32).
 *
 * For M <= 2 (K % 64 == 0, 512 <= K <= 8192 for one token, <= 4096 for two)
 * one kernel streams the rows of both matrices and applies the product in
 * its epilogue.  Other shapes run the gate BitLinear, the up matrix on the
 * same int8 activations and an elementwise kernel (same arithmetic, same
 * bits).  A fused gate+up matrix packed as [2I, K] (gate rows first) is
 * passed as packed_gate = base, packed_up = base + I * K / 4 with the same
 * w_scale for both.
 *
 *   x          device, [M, K] row-major, BITNET_F32 or BITNET_BF16.
 *   packed_gate, packed_up: device, [I, K / 4] packed codes each (as
 *              bitnet_pack_weights writes them).
 *   w_scale_gate, w_scale_up: device, one float each (beta of each matrix).
 *   out        device, [M, I] float.
 *   x_q, scale device, [M, K] int8 and [M] float outs, or NULL.
 *   acc_gate, acc_up: device, [M, I] int32 outs (the exact integer
 *              products), or NULL.
 *   workspace  device, >= bitnet_bitlinear_swiglu_workspace_bytes(M, I, K)
 *              bytes, 256-byte aligned, any contents.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_bitlinear_swiglu(const void *x, int dtype, int64_t M, const uint8_t *packed_gate,
                            const float *w_scale_gate, const uint8_t *packed_up,
                            const float *w_scale_up, int64_t I, int64_t K, float *out, int8_t *x_q,
                            float *scale, int32_t *acc_gate, int32_t *acc_up, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * Group-wise and per-channel weight scales ([Deep-dive] §4.3: in practice the
 * weights are cut into groups of group_size -- commonly 128 -- and every group
 * computes its own gamma and beta; one group per output row is the
 * per-channel scale of [Hands-on] §2.1).  A group is G consecutive weights of
 * one output row, W[n, g*G .. g*G + G - 1]; a row holds K / G groups.
 *
 * bitnet_pack_weights_grouped -- ternarises every group as bitnet_pack_weights
 * ternarises a whole matrix (mean|W_g| in fp64 over 4096-element chunks left
 * to right, gamma_g = 1 / (alpha * mean + eps) in fp32, codes
 * clamp(rint(gamma_g * w), -1, 1) + 1, beta_g = nnz_g / G).
 *   W        device, [N, K] row-major, BITNET_F32 or BITNET_BF16.
 *   G        group size: G % 4 == 0, K % G == 0 (G = K: per channel).
 *   packed   device, N * K / 4 bytes out, the same layout as bitnet_pack_weights.
 *   w_scale  device, [N, K / G] float out: beta per group.
 *   absmean  device, [N, K / G] float out (mean|W_g|), or NULL.
 * No workspace.  Errors: INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED, CUDA.
 */
int bitnet_pack_weights_grouped(const void *W, int dtype, int64_t N, int64_t K, int64_t G, float alpha,
                                float eps, uint8_t *packed, float *w_scale, float *absmean,
                                cudaStream_t stream);

/*
 * bitnet_w2a8_grouped -- the ternary matmul with group scales, any M:
 *   y[m, n] = fl(F * fl(s_m / 127)),  F = sum_g acc_g[m, n] * w_scale[n, g]
 * where acc_g is the exact int32 product of group g (sum over its K range of
 * (code - 1) * x_q) and F is formed in fp32 (one rounding per group term and
 * per addition; the order is the kernel's).  The error of y against the
 * exact value is at most (K / G + 8) * 2^-24 times
 * (s_m / 127) * sum_g |acc_g * w_scale[n, g]|.
 * One or two tokens (K % 64 == 0, K <= 8192 / 4096, G = K or a power of two
 * from 64 to 2048, x_q and packed 16-byte aligned) stream through one kernel
 * at HBM speed; other shapes use a plain one-warp-per-output kernel.
 *   x_q, scale, packed: as bitnet_w2a8_gemv.
 *   w_scale  device, [N, K / G] float (any values, e.g. beta or mean|W_g|).
 *   y        device, [M, N] float out.
 *   acc_g    device, [M, N, K / G] int32 out (per-group products), or NULL.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED, CUDA.
 */
int bitnet_w2a8_grouped(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                        const float *w_scale, int64_t N, int64_t K, int64_t G, float *y,
                        int32_t *acc_g, cudaStream_t stream);

/* Workspace bytes bitnet_bitlinear_grouped needs (its unfused fallback's
 * int8 activations and scales). */
size_t bitnet_bitlinear_grouped_workspace_bytes(int64_t M, int64_t K);

/*
 * bitnet_bitlinear_grouped -- the BitLinear forward with group scales:
 * per-token absmax quantisation of x (bitnet_quant_act's arithmetic), then
 * bitnet_w2a8_grouped.  For one or two tokens on the streaming kernel's
 * shapes the quantisation runs in that kernel's prologue (one kernel).
 *   x        device, [M, K], BITNET_F32 or BITNET_BF16.
 *   x_q, scale: device outs ([M, K] int8, [M] float), or NULL.
 *   workspace device, >= bitnet_bitlinear_grouped_workspace_bytes(M, K),
 *            256-byte aligned, any contents.  With at least
 *            bitnet_grouped_workspace_bytes(M, N, K, G) bytes, three or more
 *            tokens run on the tensor cores (as bitnet_w2a8_grouped_ws: one
 *            prep kernel quantises into the operand layout and forms the
 *            group sums, then the grouped GEMV, 64 tokens at a time).
 *   other arguments as bitnet_w2a8_grouped.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_bitlinear_grouped(const void *x, int dtype, int64_t M, const uint8_t *packed,
                             const float *w_scale, int64_t N, int64_t K, int64_t G, float *y,
                             int8_t *x_q, float *scale, int32_t *acc_g, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes of bitnet_w2a8_grouped_ws, and of bitnet_bitlinear_grouped
 * on its tensor-core path (0 for shapes the group calls reject). */
size_t bitnet_grouped_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t G);

/*
 * bitnet_w2a8_grouped_ws -- bitnet_w2a8_grouped (same operation, arguments
 * and error bound, [Deep-dive] §4.3 group-wise scales) with a workspace, so
 * that three or more tokens run on the tensor cores: G in {64, 128, 256,
 * 512} or a single group per row of at most 512 weights (K % G == 0, K % 64
 * == 0, 512 <= K <= 65536, at most 1024 groups per row and
 * 64 * (K / G) * 4 <= 16 KB), x_q and packed 16-byte aligned.  Per 64
 * tokens, a prep kernel writes the fp16 operand layout and each token's sum
 * of x_q per group, then the mma.sync GEMV accumulates each group exactly,
 * stores acc_g if asked and adds acc_g * w_scale[n, g] into F with one fp32
 * FMA per group.  Other shapes (and M <= 2) take bitnet_w2a8_grouped's
 * kernels.
 *   workspace device, >= bitnet_grouped_workspace_bytes(M, N, K, G) bytes,
 *             256-byte aligned, any contents.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_w2a8_grouped_ws(const int8_t *x_q, const float *scale, int64_t M, const uint8_t *packed,
                           const float *w_scale, int64_t N, int64_t K, int64_t G, float *y, int32_t *acc_g,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes bitnet_bitlinear_fake_quant needs. */
size_t bitnet_bitlinear_fake_quant_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * bitnet_bitlinear_fake_quant -- the training-time BitLinear forward of
 * [Deep-dive] §3.1: the fp32 (or bf16) shadow weights W are ternarised on
 * every call (bitnet_pack_weights: absmean, §2.2), x is absmax-quantised per
 * token, and the integer product is rescaled by s_m / 127 and by the
 * per-output weight_scale[n] (the module's learned scale) -- or by beta when
 * weight_scale is NULL.  The straight-through estimator of §2.4 only affects
 * the backward pass, which this library does not compute.
 * Results equal bitnet_pack_weights followed by bitnet_bitlinear (beta) or by
 * bitnet_bitlinear_grouped with G = K (weight_scale).
 *   W        device, [N, K] row-major, BITNET_F32 or BITNET_BF16.
 *   x        device, [M, K], BITNET_F32 or BITNET_BF16.
 *   alpha, eps: as bitnet_pack_weights.
 *   weight_scale device, [N] float, or NULL (beta).
 *   y        device, [M, N] float out.
 *   packed, beta: device outs (N * K / 4 bytes, one float), or NULL (then in
 *            the workspace).
 *   x_q, scale, acc: device outs as bitnet_bitlinear, or NULL.
 *   workspace device, >= bitnet_bitlinear_fake_quant_workspace_bytes(M, N, K),
 *            256-byte aligned, any contents.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
int bitnet_bitlinear_fake_quant(const void *W, int w_dtype, const void *x, int x_dtype, int64_t M,
                                int64_t N, int64_t K, float alpha, float eps,
                                const float *weight_scale, float *y, uint8_t *packed, float *beta,
                                int8_t *x_q, float *scale, int32_t *acc, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* Bytes of the fixed device array behind bitnet_w2a8_gemv_static_scratch. */
#define BITNET_GEMV_STATIC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * bitnet_w2a8_gemv_static_scratch -- bitnet_w2a8_gemv for callers that cannot
 * allocate device memory.  No page counterpart: this is a packaging variant of
 * the decode GEMV above, not a separate step of the method.
 *
 * Some callers may not call cudaMalloc at all: plugins whose host framework
 * owns every device allocation, runtimes that pre-plan a fixed memory budget,
 * or code that runs where an allocation could block or fail.  This entry
 * point takes the same arguments as bitnet_w2a8_gemv minus the workspace and
 * computes the same result (same kernels, same dispatch).  Its scratch is a
 * 4 MiB array compiled into the library (BITNET_GEMV_STATIC_SCRATCH_BYTES);
 * every GPU that loads the library holds that array until the process exits.
 * The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 *   - Limit: a shape whose bitnet_gemv_workspace_bytes(M, N, K) exceeds
 *     BITNET_GEMV_STATIC_SCRATCH_BYTES is rejected with BITNET_ERR_TOO_LARGE
 *     (nothing enqueued).  For example M=16 fits N up to ~65k rows, M=64 up
 *     to ~16k.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with that device current) and caches it.
 *     Make that first call outside any stream capture.
 *   - Sharing: every call, on every stream, uses the same array, and the
 *     array keeps the last call's contents.  Stale contents do not matter:
 *     like bitnet_w2a8_gemv with any workspace, the call zeroes, in stream
 *     order, the part it accumulates into (the streaming and row-range
 *     kernels, which take one token and most two-token shapes, do not touch
 *     the array at all).  Two calls that can overlap on the GPU
 *     (different streams, no ordering between them) race on the array and
 *     give wrong results.  Order them on one stream, or use
 *     bitnet_w2a8_gemv with separate workspaces.
 * Errors: as bitnet_w2a8_gemv, plus TOO_LARGE; WORKSPACE never occurs.
 */
int bitnet_w2a8_gemv_static_scratch(const int8_t *x_q, const float *scale, int64_t M,
                                    const uint8_t *packed, const float *w_scale, int64_t N,
                                    int64_t K, float *y, int32_t *acc, cudaStream_t stream);

/*
 * bitnet_selftest_wait_timeout -- exercises the failure path without a
 * fault: one kernel waits on an on-chip barrier that nothing completes,
 * gives up after limit_ns (1 us .. 1 s) of wall-clock time, records the
 * timeout in the device error word exactly as a stuck pipeline stage would,
 * and returns; the next bitnet_check_device_error reports
 * BITNET_ERR_TIMEOUT and the context stays usable.
 * Errors: INVALID_ARG (limit out of range), UNSUPPORTED, CUDA.
 */
int bitnet_selftest_wait_timeout(int64_t limit_ns, cudaStream_t stream);

/*
 * bitnet_test_inject_cuda_failures -- test hook for the host-side failure
 * path: the next n entry-point calls that get past argument validation fail
 * with BITNET_ERR_CUDA at their device query, before any other CUDA call
 * (nothing is enqueued), as a failing cudaGetDevice would make them.  n <= 0
 * clears the count.  Returns the count that was pending.
 */
int bitnet_test_inject_cuda_failures(int n);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns BITNET_OK, BITNET_ERR_TIMEOUT (a kernel's bounded
 * wait expired since the last check) or BITNET_ERR_CUDA.
 */
int bitnet_check_device_error(cudaStream_t stream);

/*
 * Enables (1) or disables (0) programmatic dependent launch for the kernels
 * this thread enqueues: a kernel may then start its weight prefetch while the
 * previous kernel in the stream is still running.  Off by default.
 */
void bitnet_set_pdl(int enable);

#ifdef __cplusplus
}
#endif

#endif /* BITNET_W2A8_H */

/*
 * bitnet_oracle.c -- plain, slow CPU oracle for the BitNet b1.58 W2A8 path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry point and the CPU-baseline leg of the benchmark may load or
 * call this file.  The CUDA library shares no code, header, table or helper
 * with it, and neither side includes the other.
 *
 * Sources (pages on the BitNet subject; cited by title and section):
 *   [Deep-dive]  "BitNet 深度拆解：当大模型被压到 1.58 bit——从三元权重、BitLinear
 *                 到 bitnet.cpp 的端侧推理革命（2026）"
 *   [devpress]   devpress.csdn.net BitNet post, section "三值量化：把乘法变成加减法"
 *   [Hands-on]   "1-bit推理框架bitnet.cpp实测：三元权重原理与本地部署"
 *
 * Every floating-point step is written as the one IEEE-754 operation it names
 * (build with -O2 -ffp-contract=off, no fast-math; x86-64 SSE arithmetic has
 * no excess precision).  Rounding to integer is rint() in the default
 * round-to-nearest-even mode, which is the rounding torch.round performs.
 *
 * Readings where the pages leave a step open (listed again in the design
 * notes of the repository):
 *   - mean|W| is summed in fp64 in a fixed order: chunks of 4096 consecutive
 *     row-major elements, each summed left to right, chunk sums added left to
 *     right; the mean is (float)(S / n).
 *   - eps is added after alpha*mean, in fp32, as the absmean listing writes it.
 *   - beta = mean(|W_ternary|) = nnz / n, formed in fp64 and rounded once.
 *   - the dequantised output divides by qmax = 127 (the BitLinear forward in
 *     [Deep-dive] section 3.1 multiplies by the raw absmax only).
 *   - a NaN product gamma*w ternarises to 0; NaN activations are unspecified.
 *
 * Pins: every function below is checked against values fixed by the pages or
 * by mathematics (worked examples, closed forms, invariants, brute force); see
 * tests/test_oracle_pins.py.  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_ABS_CHUNK 4096

/* bf16 is the upper half of an fp32 word, so widening is exact (activation
 * dtype, [Deep-dive] section 6.5: norms etc. stay fp32, only linear inputs
 * are quantised). */
void oracle_bf16_to_f32(const uint16_t *in, int64_t n, float *out) {
  for (int64_t i = 0; i < n; i++) {
    uint32_t bits = (uint32_t)in[i] << 16;
    memcpy(&out[i], &bits, sizeof bits);
  }
}

/* S = sum |w_i|, fp64, fixed order (reading of weight.abs().mean() in the
 * absmean listing, [Deep-dive] section 2.2). */
double oracle_abs_sum(const float *w, int64_t n) {
  double total = 0.0;
  for (int64_t c0 = 0; c0 < n; c0 += ORACLE_ABS_CHUNK) {
    int64_t c1 = c0 + ORACLE_ABS_CHUNK < n ? c0 + ORACLE_ABS_CHUNK : n;
    double part = 0.0;
    for (int64_t i = c0; i < c1; i++) part += fabs((double)w[i]);
    total += part;
  }
  return total;
}

/* mean|W| rounded to fp32 (the weight tensor is fp32). */
float oracle_absmean(const float *w, int64_t n) {
  if (n <= 0) return 0.0f;
  return (float)(oracle_abs_sum(w, n) / (double)n);
}

/* gamma = 1 / (alpha * mean|W| + eps), three fp32 operations in the order of
 * the absmean listing, [Deep-dive] section 2.2. */
float oracle_gamma(float mean, float alpha, float eps) {
  float t = alpha * mean;
  t = t + eps;
  return 1.0f / t;
}

/* W_ternary = clamp(round(gamma * w), -1, 1), [Deep-dive] section 2.2. */
int oracle_ternarize(float gamma, float w) {
  float p = gamma * w;
  if (isnan(p)) return 0;
  float r = rintf(p);
  if (r > 1.0f) r = 1.0f;
  if (r < -1.0f) r = -1.0f;
  return (int)r; /* -0.0 becomes 0 */
}

/* INT2 packing, [Deep-dive] section 3.3 (pack_ternary): code = w + 1 in
 * {0,1,2}; the flattened codes are grouped four to a byte, the first in the
 * lowest two bits; a ragged tail is padded with code 0. */
void oracle_pack_codes(const int8_t *q, int64_t n, uint8_t *packed) {
  int64_t nbytes = (n + 3) / 4;
  for (int64_t j = 0; j < nbytes; j++) {
    unsigned byte = 0;
    for (int s = 0; s < 4; s++) {
      int64_t i = 4 * j + s;
      unsigned code = i < n ? (unsigned)(q[i] + 1) : 0u;
      byte |= (code & 3u) << (2 * s);
    }
    packed[j] = (uint8_t)byte;
  }
}

/* Unpacking, [Deep-dive] section 3.3 (unpack_ternary): field s of byte j is
 * flat element 4j+s; value = code - 1 (a code 3, never produced, reads +2). */
void oracle_unpack_codes(const uint8_t *packed, int64_t n, int8_t *q) {
  for (int64_t i = 0; i < n; i++) {
    int code = (packed[i / 4] >> (2 * (i % 4))) & 3;
    q[i] = (int8_t)(code - 1);
  }
}

/* Offline weight preparation: absmean ternarisation, 2-bit packing and the
 * beta scale, [Deep-dive] sections 2.2, 2.3 and 3.3.  W is [N, K] row-major
 * fp32; packed receives ceil(N*K/4) bytes. */
void oracle_pack_weights(const float *W, int64_t N, int64_t K, float alpha, float eps,
                         uint8_t *packed, float *beta, float *absmean) {
  int64_t n = N * K;
  float mean = oracle_absmean(W, n);
  float gamma = oracle_gamma(mean, alpha, eps);
  int64_t nnz = 0;
  int64_t nbytes = (n + 3) / 4;
  for (int64_t j = 0; j < nbytes; j++) {
    int8_t q[4] = {0, 0, 0, 0};
    int64_t cnt = n - 4 * j < 4 ? n - 4 * j : 4;
    for (int64_t s = 0; s < cnt; s++) {
      q[s] = (int8_t)oracle_ternarize(gamma, W[4 * j + s]);
      if (q[s] != 0) nnz++;
    }
    oracle_pack_codes(q, cnt, &packed[j]);
  }
  *beta = (float)((double)nnz / (double)n);
  *absmean = mean;
}

/* Per-token absmax activation quantisation, [Deep-dive] section 2.2
 * (absmax_quantize, bits = 8): s = max(max_k |x|, 1e-8);
 * q = clamp(round(x / s * 127), -127, 127).  Divide first, then multiply. */
void oracle_quant_act(const float *x, int64_t M, int64_t K, int8_t *xq, float *scale) {
  const float qmax = 127.0f;
  for (int64_t m = 0; m < M; m++) {
    const float *row = x + m * K;
    float s = 0.0f;
    for (int64_t k = 0; k < K; k++) {
      float a = fabsf(row[k]);
      if (a > s) s = a;
    }
    if (s < 1e-8f) s = 1e-8f;
    scale[m] = s;
    for (int64_t k = 0; k < K; k++) {
      float v = row[k] / s;
      v = v * qmax;
      float r = rintf(v);
      if (r > qmax) r = qmax;
      if (r < -qmax) r = -qmax;
      xq[m * K + k] = (int8_t)r;
    }
  }
}

/* Integer contraction acc[m, n] = sum_k W_ternary[n, k] * x_q[m, k] over the
 * packed weights ("整数域矩阵乘", [Deep-dive] section 3.1; the -1/0/+1 product
 * identity of section 1), for output rows n in [n_begin, n_end).  Accumulated
 * in int64 and stored as int32 (|acc| <= 254 K). */
void oracle_contract(const int8_t *xq, const uint8_t *packed, int64_t M, int64_t N, int64_t K,
                     int64_t n_begin, int64_t n_end, int32_t *acc) {
  for (int64_t n = n_begin; n < n_end; n++) {
    for (int64_t m = 0; m < M; m++) {
      int64_t a = 0;
      for (int64_t k = 0; k < K; k++) {
        int64_t i = n * K + k;
        int w = ((packed[i / 4] >> (2 * (i % 4))) & 3) - 1;
        a += (int64_t)w * (int64_t)xq[m * K + k];
      }
      acc[m * N + n] = (int32_t)a;
    }
  }
}

/* Dequantisation Y = acc * beta * s_m / 127 ([Deep-dive] section 2.3, with
 * the activation scale read as absmax / qmax), computed in fp64 and rounded
 * once to fp32. */
void oracle_epilogue(const int32_t *acc, const float *scale, float w_scale, int64_t M, int64_t N,
                     float *y) {
  for (int64_t m = 0; m < M; m++)
    for (int64_t n = 0; n < N; n++)
      y[m * N + n] =
          (float)((double)acc[m * N + n] * (double)w_scale * (double)scale[m] / 127.0);
}

/* SwiGLU feed-forward product of the BitTransformer block ([Deep-dive]
 * section 3.1: down(F.silu(gate(h)) * up(h))): for the two BitLinear outputs
 * of the same activations, a = silu(y_gate) * y_up with silu(z) = z * sigmoid(z)
 * = z / (1 + exp(-z)).  The BitLinear outputs are taken exactly, in fp64, from
 * the integer accumulators (acc * w_scale * s_m / 127, not rounded to fp32),
 * and the product is returned in fp64: the reference value the fp32 GPU result
 * is compared with.  acc_gate / acc_up are [M, I]. */
void oracle_swiglu(const int32_t *acc_gate, const int32_t *acc_up, const float *scale, float w_scale_gate,
                   float w_scale_up, int64_t M, int64_t I, double *out) {
  for (int64_t m = 0; m < M; m++)
    for (int64_t i = 0; i < I; i++) {
      double yg = (double)acc_gate[m * I + i] * (double)w_scale_gate * (double)scale[m] / 127.0;
      double yu = (double)acc_up[m * I + i] * (double)w_scale_up * (double)scale[m] / 127.0;
      out[m * I + i] = yg / (1.0 + exp(-yg)) * yu;
    }
}

/* silu(z) in fp64, the same definition, for the pins. */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* Group-wise weight scales ([Deep-dive] section 4.3: in practice the weights
 * are cut into groups of group_size -- commonly 128 -- and every group gets
 * its own gamma and beta; one group per output row is the per-channel scale
 * of [Hands-on] section 2.1).  Reading: a group is G consecutive weights of
 * one output row, W[n, g*G .. g*G + G - 1] (G divides K, G % 4 == 0), so a
 * row holds K / G groups; each group is ternarised exactly as a whole matrix
 * is (oracle_pack_weights: mean|W_g| in the fixed fp64 order, gamma_g,
 * codes, beta_g = nnz_g / G).  The packed bytes keep the row-major layout of
 * the per-tensor format; w_scale[n * (K / G) + g] = beta_g and
 * absmean[n * (K / G) + g] = mean|W_g|. */
void oracle_pack_weights_grouped(const float *W, int64_t N, int64_t K, int64_t G, float alpha, float eps,
                                 uint8_t *packed, float *w_scale, float *absmean) {
  const int64_t ng = K / G;
  for (int64_t n = 0; n < N; n++)
    for (int64_t g = 0; g < ng; g++) {
      const int64_t off = n * K + g * G; /* a multiple of 4: the group's bytes start at off / 4 */
      oracle_pack_weights(W + off, 1, G, alpha, eps, packed + off / 4, &w_scale[n * ng + g], &absmean[n * ng + g]);
    }
}

/* Per-group integer products: acc_g[(m * N + n) * (K / G) + g] =
 * sum over k in group g of W_ternary[n, k] * x_q[m, k], rows n in
 * [n_begin, n_end). */
void oracle_contract_grouped(const int8_t *xq, const uint8_t *packed, int64_t M, int64_t N, int64_t K, int64_t G,
                             int64_t n_begin, int64_t n_end, int32_t *acc_g) {
  const int64_t ng = K / G;
  for (int64_t n = n_begin; n < n_end; n++)
    for (int64_t m = 0; m < M; m++)
      for (int64_t g = 0; g < ng; g++) {
        int64_t a = 0;
        for (int64_t k = g * G; k < (g + 1) * G; k++) {
          int64_t i = n * K + k;
          int w = ((packed[i / 4] >> (2 * (i % 4))) & 3) - 1;
          a += (int64_t)w * (int64_t)xq[m * K + k];
        }
        acc_g[(m * N + n) * ng + g] = (int32_t)a;
      }
}

/* Dequantisation with group scales: y[m, n] = (s_m / 127) * sum_g
 * w_scale[n, g] * acc_g[m, n, g], in fp64 (each product is exact; the sum
 * runs over g in order), returned unrounded.  cond[m, n] = (s_m / 127) *
 * sum_g |w_scale[n, g] * acc_g[m, n, g]| bounds what any summation order of
 * the terms can lose to rounding. */
void oracle_epilogue_grouped(const int32_t *acc_g, const float *scale, const float *w_scale, int64_t M, int64_t N,
                             int64_t ng, double *y, double *cond) {
  for (int64_t m = 0; m < M; m++)
    for (int64_t n = 0; n < N; n++) {
      double t = 0.0, c = 0.0;
      for (int64_t g = 0; g < ng; g++) {
        double p = (double)acc_g[(m * N + n) * ng + g] * (double)w_scale[n * ng + g];
        t += p;
        c += fabs(p);
      }
      y[m * N + n] = t * (double)scale[m] / 127.0;
      cond[m * N + n] = c * (double)scale[m] / 127.0;
    }
}

/* RMSNorm in front of a BitLinear (the feed-forward input of the
 * BitTransformer block, [Deep-dive] section 3.1: h = norm2(x), then gate(h)
 * and up(h); norms stay fp32, same section and section 6.5).  nn.RMSNorm
 * computes h_k = x_k / sqrt(mean_k(x_k^2) + eps) * g_k per token.  Readings:
 *   - the sum of squares S is formed in fp64, left to right (the square of an
 *     fp32 value is exact in fp64); ms = (float)(S / K);
 *   - t = ms + eps and the inverse rms r = 1 / sqrt(t) are three fp32 IEEE
 *     operations (add, sqrt, division), the division once per token;
 *   - h_k = (x_k * r) * g_k, two fp32 products; g = NULL means the module's
 *     initial weight, all ones, and the second product is skipped (x * 1).
 * The absmax quantisation of section 2.2 then runs on h. */
double oracle_sum_squares(const float *x, int64_t K) {
  double s = 0.0;
  for (int64_t k = 0; k < K; k++) s += (double)x[k] * (double)x[k];
  return s;
}

/* One token: h = (x * r) * g from a given mean square ms. */
void oracle_rmsnorm_apply(const float *x, const float *g, int64_t K, float ms, float eps, float *h, float *r_out) {
  float t = ms + eps;
  float rms = sqrtf(t);
  float r = 1.0f / rms;
  for (int64_t k = 0; k < K; k++) {
    float v = x[k] * r;
    h[k] = g ? v * g[k] : v;
  }
  if (r_out) *r_out = r;
}

/* x, h [M, K] row-major; g [K] or NULL; ms [M] receives each token's mean
 * square (fp32). */
void oracle_rmsnorm(const float *x, const float *g, int64_t M, int64_t K, float eps, float *h, float *ms) {
  for (int64_t m = 0; m < M; m++) {
    float msq = (float)(oracle_sum_squares(x + m * K, K) / (double)K);
    ms[m] = msq;
    oracle_rmsnorm_apply(x + m * K, g, K, msq, eps, h + m * K, 0);
  }
}

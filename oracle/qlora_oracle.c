/*
 * qlora_oracle.c -- plain, slow, obviously-correct CPU oracle for the QLoRA
 * NF4 linear-layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table generator or helper
 * with the CUDA library: every step below is written out from the method's
 * definition on the source pages, cited per function as
 *   <page title> -- <section>.
 * Page titles used below:
 *   [QLoRA-26]  "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化" (datawhale, ch. 26)
 *   [QLoRA-22]  "QLoRA and 4bit Quantization | QLoRA 与 4-bit NormalFloat 量化核心机制" (datawhale, ch. 22)
 *   [Gemma-9]   "第 09 期 | QLoRA 4-bit 量化微调：消费级显卡也能训" (agentupdate gemma lesson 9)
 *   [Finetune-4] "QLoRA 的三个核心技术" (gufacode finetune chapter 4)
 *
 * Precision rules (what the pages fix, and the readings taken where they do
 * not):
 *   - quantisation decisions are taken in IEEE binary32 (round to nearest
 *     even, no fused multiply-add, no fast math; build with -ffp-contract=off);
 *   - dequantised weights are bf16 values (compute dtype bf16, [Gemma-9]
 *     section 9.3) obtained by ONE round-to-nearest-even of a binary32
 *     product;
 *   - forward and backward contractions run in binary64 over inputs that are
 *     exactly representable (bf16 values widened to float).
 *
 * Parity pins: every function here is pinned by the not-gpu tests in
 * tests/test_oracle_*.py against values printed on the pages, closed forms,
 * invariants, brute force on tiny inputs and fp64 torch autograd.  The
 * conventions the pages leave open (double-quantisation group layout and
 * rounding, nibble order, tie-break) are pinned only by the conventions
 * stated here: "parity unpinned" by the pages for those three choices.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Codebook.  [QLoRA-26] Step 4 (create_nf4_lookup_table) and [QLoRA-22]
 * Step 4 print the same 16 decimal values; each entry is the binary32 value
 * nearest to the printed decimal (the C compiler converts literals with
 * correct rounding).  Index 7 is the exact zero. */
static const float ORACLE_NF4[16] = {
    -1.0f,  -0.696f, -0.525f, -0.395f, -0.284f, -0.185f, -0.091f, 0.0f,
    0.080f, 0.161f,  0.246f,  0.338f,  0.441f,  0.563f,  0.723f,  1.0f};

#define ORACLE_ZERO_INDEX 7

/* Quantile-formula codebook.  [QLoRA-26] Step 2 gives the construction
 *   q_i = Phi^-1(p_i),  p_i = (i - 0.5) / 16,  i = 1 .. 16
 * (garbled in the page's extraction), Phi the standard normal CDF.  The
 * page does not say how the quantiles are brought to [-1, 1], where the
 * normalised weights live; reading: divided by the largest, q_16, so that
 * the table runs from -1 to 1 like the printed one.  The quantiles are
 * symmetric (Phi^-1(1 - p) = -Phi^-1(p)); the upper half is computed and
 * mirrored, so the binary32 table is exactly symmetric, with no zero.
 * Phi^-1 here: bisection on Phi(x) = erfc(-x / sqrt 2) / 2 in binary64 until
 * the bracket stops shrinking (erfc from the C library). */
static double oracle_phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

double oracle_inv_normal(double p) {
  if (!(p > 0.0 && p < 1.0)) return NAN;
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 2000; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (mid <= lo || mid >= hi) break;
    if (oracle_phi(mid) < p)
      lo = mid;
    else
      hi = mid;
  }
  return 0.5 * (lo + hi);
}

static float ORACLE_NF4_QUANTILE[16];
static int oracle_quantile_ready = 0;

static void oracle_make_quantile_table(void) {
  if (oracle_quantile_ready) return;
  const double q16 = oracle_inv_normal(15.5 / 16.0);
  for (int i = 9; i <= 16; ++i) {
    const float c = (float)(oracle_inv_normal((i - 0.5) / 16.0) / q16);
    ORACLE_NF4_QUANTILE[i - 1] = c;
    ORACLE_NF4_QUANTILE[16 - i] = -c;
  }
  oracle_quantile_ready = 1;
}

/* Codebook 0: the printed table; 1: the quantile formula. */
static const float *oracle_table(int32_t codebook) {
  if (codebook == 1) {
    oracle_make_quantile_table();
    return ORACLE_NF4_QUANTILE;
  }
  return ORACLE_NF4;
}

void oracle_codebook_values(int32_t codebook, float out[16]) {
  const float *t = oracle_table(codebook);
  for (int k = 0; k < 16; ++k) out[k] = t[k];
}

void oracle_nf4_codebook(float out[16]) {
  for (int k = 0; k < 16; ++k) out[k] = ORACLE_NF4[k];
}

/* Nearest codepoint.  [QLoRA-26] Step 2: a normalised weight is mapped to
 * the closest entry of the table (0.20 -> 0.161).  Distances are binary32
 * |xn - c_k|; on an exact tie of the binary32 distances the lower index wins
 * (the pages are silent on ties). */
static int oracle_nearest_in(const float *table, float xn) {
  int best = 0;
  float bestd = fabsf(xn - table[0]);
  for (int k = 1; k < 16; ++k) {
    float d = fabsf(xn - table[k]);
    if (d < bestd) {
      bestd = d;
      best = k;
    }
  }
  return best;
}

int oracle_nearest_code(float xn) { return oracle_nearest_in(ORACLE_NF4, xn); }

int oracle_nearest_code_cb(int32_t codebook, float xn) {
  return oracle_nearest_in(oracle_table(codebook), xn);
}

/* Indices for `count` consecutive binary32 bit patterns starting at
 * `start_bits` (used to compare against an exhaustive device sweep). */
void oracle_nearest_codes_bits(uint32_t start_bits, int64_t count, uint8_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    uint32_t b = start_bits + (uint32_t)i;
    float f;
    memcpy(&f, &b, 4);
    out[i] = (uint8_t)oracle_nearest_code(f);
  }
}

/* Indices of the weights w with `count` consecutive binary32 bit patterns
 * starting at `start_bits`, in a block whose absolute maximum is `absmax`
 * (> 0): the quantiser's two steps for one element, the binary32 division
 * w / absmax ([Gemma-9] 9.2.1, "normalise to [-1, 1]") and the nearest
 * codepoint ([QLoRA-26] Step 2).  Used to compare against exhaustive device
 * sweeps of one block constant. */
void oracle_nearest_codes_scaled_bits(uint32_t start_bits, int64_t count, float absmax,
                                      uint8_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    uint32_t b = start_bits + (uint32_t)i;
    float w;
    memcpy(&w, &b, 4);
    volatile float xn = w / absmax;
    out[i] = (uint8_t)oracle_nearest_code(xn);
  }
}

/* binary32 -> bf16 bits, round to nearest, ties to even, on the bit
 * pattern.  NaN stays NaN (quiet bit set). */
uint16_t oracle_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

void oracle_bf16_rne_array(const float *in, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Status codes (oracle-local). */
#define ORACLE_OK 0
#define ORACLE_EINVAL 1

/* Blockwise NF4 quantisation with optional double quantisation.
 *
 *  [Gemma-9] 9.2.1: weights are split into blocks, each block is normalised
 *  to [-1, 1] by its absolute maximum, and each normalised value is stored as
 *  the 4-bit index of its nearest NF4 codepoint ([QLoRA-26] Step 2).
 *  [QLoRA-22] "engineering notes": 64 or 128 weights share one scale; blocks
 *  here are `block` consecutive weights of the row-major flattened matrix
 *  (cols % block == 0 keeps blocks inside one row).
 *  [QLoRA-22] Step 3/4 docstring: real QLoRA stores two 4-bit indices per
 *  uint8.  Reading (pages silent on order): element 2j in the HIGH nibble,
 *  element 2j+1 in the LOW nibble.
 *  [Gemma-9] 9.2.2 and [Finetune-4]: the per-block constants are themselves
 *  quantised to 8 bits (double quantisation).  Reading: `group` consecutive
 *  block constants share one binary32 scale s2 = max/127; each constant is
 *  stored as clamp(rint_even(a / s2), -127, 127) in int8.  group == 0 keeps
 *  the constants in binary32 (absmax_f32).
 *
 *  Steps per block b with weights w_i:
 *    a_b = max_i |w_i|                       (exact)
 *    xn_i = w_i / a_b                        (binary32 IEEE division)
 *    idx_i = nearest codepoint of xn_i       (oracle_nearest_code)
 *    a_b == 0  ->  idx_i = 7 (the zero codepoint of the printed table), no
 *                  division; with the quantile table (no zero) any index
 *                  dequantises to 0 there, and 7 is kept as the convention.
 *  `codebook` selects the table: 0 printed, 1 quantile formula.
 *  Steps per group g (group > 0):
 *    gmax = max_b a_b; s2 = gmax / 127 (binary32); code_b = clamp(rint(a_b/s2))
 *    gmax == 0 -> s2 = 0 and every code 0.
 *
 *  Returns the number of non-finite input weights (those blocks produce
 *  unspecified indices), or -1 on invalid arguments.
 */
int64_t oracle_quantize_nf4(const float *w, int64_t rows, int64_t cols, int32_t block,
                            int32_t group, uint8_t *packed, int8_t *absmax_code,
                            float *absmax_f32, float *scale2, uint8_t *idx_out,
                            int32_t codebook) {
  if (rows < 0 || cols < 0 || block <= 0 || (block & 1) || group < 0) return -1;
  if (codebook != 0 && codebook != 1) return -1;
  const float *table = oracle_table(codebook);
  if (cols % block) return -1;
  const int64_t n = rows * cols;
  const int64_t nblocks = n / block;
  float *a = (float *)malloc((size_t)(nblocks > 0 ? nblocks : 1) * sizeof(float));
  if (!a) return -1;
  int64_t nonfinite = 0;

#pragma omp parallel for schedule(static) reduction(+ : nonfinite)
  for (int64_t b = 0; b < nblocks; ++b) {
    const float *wb = w + b * block;
    float amax = 0.0f;
    for (int32_t i = 0; i < block; ++i) {
      float v = wb[i];
      if (!isfinite(v)) {
        nonfinite++;
        continue;
      }
      float m = fabsf(v);
      if (m > amax) amax = m;
    }
    a[b] = amax;
    for (int32_t i = 0; i < block; i += 2) {
      int q0, q1;
      if (amax == 0.0f) {
        q0 = q1 = ORACLE_ZERO_INDEX;
      } else {
        float xn0 = wb[i] / amax;
        float xn1 = wb[i + 1] / amax;
        q0 = oracle_nearest_in(table, xn0);
        q1 = oracle_nearest_in(table, xn1);
      }
      int64_t e = b * block + i;
      if (idx_out) {
        idx_out[e] = (uint8_t)q0;
        idx_out[e + 1] = (uint8_t)q1;
      }
      packed[e / 2] = (uint8_t)((q0 << 4) | q1);
    }
  }

  if (group == 0) {
    if (absmax_f32)
      for (int64_t b = 0; b < nblocks; ++b) absmax_f32[b] = a[b];
  } else {
    const int64_t ngroups = (nblocks + group - 1) / group;
    for (int64_t g = 0; g < ngroups; ++g) {
      int64_t b0 = g * group, b1 = b0 + group;
      if (b1 > nblocks) b1 = nblocks;
      float gmax = 0.0f;
      for (int64_t b = b0; b < b1; ++b)
        if (a[b] > gmax) gmax = a[b];
      float s2 = gmax / 127.0f;
      scale2[g] = s2;
      for (int64_t b = b0; b < b1; ++b) {
        float c = 0.0f;
        if (s2 != 0.0f) c = rintf(a[b] / s2);
        if (c > 127.0f) c = 127.0f;
        if (c < -127.0f) c = -127.0f;
        absmax_code[b] = (int8_t)c;
      }
    }
  }
  free(a);
  return nonfinite;
}

/* Dequantisation to bf16.  [QLoRA-26] Step 3 / Step 4 (TODO 1): the
 * approximate weight is the codepoint selected by the stored index times the
 * block's scale factor; [Gemma-9] 9.2.2 (mermaid): the 8-bit constants are
 * dequantised first, then used on the 4-bit weights; [Gemma-9] 9.3: compute
 * dtype bf16.
 *    a_hat = (float)code_b * s2_g            (binary32 product; DQ)
 *    a_hat = absmax_f32[b]                   (no DQ)
 *    w_hat = bf16_rne((float)c_idx * a_hat)  (binary32 product, one rounding)
 */
int oracle_dequant_bf16(const uint8_t *packed, const int8_t *absmax_code,
                        const float *absmax_f32, const float *scale2, int64_t rows,
                        int64_t cols, int32_t block, int32_t group, uint16_t *w_out,
                        int32_t codebook) {
  if (rows < 0 || cols < 0 || block <= 0 || (block & 1) || group < 0) return ORACLE_EINVAL;
  if (codebook != 0 && codebook != 1) return ORACLE_EINVAL;
  const float *table = oracle_table(codebook);
  if (cols % block) return ORACLE_EINVAL;
  const int64_t n = rows * cols;
  const int64_t nblocks = n / block;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    float ahat;
    if (group > 0)
      ahat = (float)absmax_code[b] * scale2[b / group];
    else
      ahat = absmax_f32[b];
    for (int32_t i = 0; i < block; ++i) {
      int64_t e = b * block + i;
      uint8_t byte = packed[e / 2];
      int q = (e & 1) ? (byte & 0x0f) : (byte >> 4);
      float prod = table[q] * ahat;
      w_out[e] = oracle_bf16_rne(prod);
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* LoRA dropout on the bypass input.  [QLoRA-26] Step 5 training config and
 * [Gemma-9] LoraConfig set lora_dropout = p: during training the LoRA
 * branch sees dropout(x) = x . keep / (1 - p) with keep ~ Bernoulli(1 - p)
 * per element, the base branch sees x.  The pages give no generator; the
 * reading taken: the counter-based Philox4x64-10 generator (Salmon et al.,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011) keyed by the
 * 64-bit seed (key = {seed, 0}), its 64-bit outputs in counter order
 * starting at counter 1 (output o: counter o / 4 + 1, word o % 4), two
 * 32-bit uniforms per output (element e of the row-major [M, K] input takes
 * output e / 2, low half for even e, high half for odd e), and
 * keep = (u >= round(p 2^32)). */
static void oracle_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2],
                                 uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
  uint64_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint64_t k[2] = {key_in[0], key_in[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += W0;
      k[1] += W1;
    }
    const unsigned __int128 p0 = (unsigned __int128)M0 * c[0];
    const unsigned __int128 p1 = (unsigned __int128)M1 * c[2];
    const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    const uint64_t n0 = hi1 ^ c[1] ^ k[0], n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* The o-th 64-bit output of the stream keyed by `seed`. */
uint64_t oracle_philox_stream(uint64_t seed, uint64_t o) {
  const uint64_t ctr[4] = {o / 4 + 1, 0, 0, 0};
  const uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  oracle_philox4x64_10(ctr, key, out);
  return out[o % 4];
}

/* keep[m * K + k] (0 or 1) of an [M, K] input for dropout probability p. */
void oracle_dropout_keep(uint64_t seed, double p, int64_t M, int64_t K, uint8_t *keep) {
  double t = floor(p * 4294967296.0 + 0.5);
  if (t > 4294967295.0) t = 4294967295.0;
  if (t < 0.0) t = 0.0;
  const uint64_t p32 = (uint64_t)t;
#pragma omp parallel for schedule(static)
  for (int64_t e2 = 0; e2 < (M * K + 1) / 2; ++e2) {
    const uint64_t v = oracle_philox_stream(seed, (uint64_t)e2);
    const uint64_t u0 = v & 0xffffffffull, u1 = v >> 32;
    keep[2 * e2] = u0 >= p32;
    if (2 * e2 + 1 < M * K) keep[2 * e2 + 1] = u1 >= p32;
  }
}

/* ------------------------------------------------------------------------ */
/* Forward.  [QLoRA-26] Step 3 (garbled formula, read as
 *   y = x W_hat^T + (x A^T) B^T * alpha / r )
 * and Step 4 (TODO 2: base output through F.linear with the dequantised
 * weight, LoRA increment through lora_A then lora_B then the scaling).  No
 * bias, no dropout.
 *   x: [M, K]   W_hat: [N, K]   A: [r, K]   B: [N, r]
 * All inputs are binary32 arrays holding bf16-exact values; every dot product
 * is accumulated in binary64 in ascending index order.
 * Only the rows listed in `rows` (nrows of them) are evaluated; outputs are
 * packed in that order: y is [nrows, N], t is [nrows, r] (t = x A^T).
 * With LoRA dropout (keep != NULL, [M, K] of 0/1, keep_scale = 1/(1 - p))
 * the LoRA branch takes dropout(x): t = keep_scale * (x . keep) A^T. */
void oracle_linear_fwd(const float *x, int64_t M, int64_t K, const float *w, int64_t N,
                       const float *A, const float *B, int32_t r, double alpha,
                       const int64_t *rows, int64_t nrows, double *y, double *t,
                       const uint8_t *keep, double keep_scale) {
  (void)M;
  const double s = alpha / (double)r;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const float *xm = x + rows[ri] * K;
    const uint8_t *km = keep ? keep + rows[ri] * K : NULL;
    double *tm = t + ri * r;
    for (int32_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        if (!km || km[k]) acc += (double)xm[k] * (double)A[j * K + k];
      tm[j] = km ? keep_scale * acc : acc;
    }
    for (int64_t n = 0; n < N; ++n) {
      const float *wn = w + n * K;
      double base = 0.0;
      for (int64_t k = 0; k < K; ++k) base += (double)xm[k] * (double)wn[k];
      double lora = 0.0;
      for (int32_t j = 0; j < r; ++j) lora += tm[j] * (double)B[n * r + j];
      y[ri * N + n] = base + s * lora;
    }
  }
}

/* Backward.  [QLoRA-26] Step 3 (gradients reach x, A and B; the NF4 state is
 * frozen) and Step 4 test "frozen base gradient contract"; [QLoRA-22] Step 1
 * item 4: the gradient also flows through the base weight (to x) but never
 * updates it.  With s = alpha / r and t = x A^T:
 *   u  = dY B                       [M, r]
 *   dX = dY W_hat + s * u A         [M, K]   (rows listed in `rows` only)
 *   dA = s * u^T x                  [r, K]
 *   dB = s * dY^T t                 [N, r]
 * Binary64 accumulation in ascending index order.  t_out and u_out are
 * [M, r] (all rows); dX is [nrows, K].
 * With LoRA dropout (keep != NULL, keep_scale = 1/(1 - p)): t is taken from
 * dropout(x) as in the forward, and the gradient of the LoRA branch with
 * respect to its input passes the same mask and scale:
 *   dX = dY W_hat + s * keep_scale * keep . (u A),   dA = s * keep_scale * u^T (x . keep). */
void oracle_linear_bwd(const float *x, const float *dY, int64_t M, int64_t K, int64_t N,
                       const float *w, const float *A, const float *B, int32_t r,
                       double alpha, const int64_t *rows, int64_t nrows, double *dX,
                       double *dA, double *dB, double *t_out, double *u_out,
                       const uint8_t *keep, double keep_scale) {
  const double s = alpha / (double)r;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float *xm = x + m * K;
    const float *gm = dY + m * N;
    const uint8_t *km = keep ? keep + m * K : NULL;
    for (int32_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        if (!km || km[k]) acc += (double)xm[k] * (double)A[j * K + k];
      t_out[m * r + j] = km ? keep_scale * acc : acc;
      double acc2 = 0.0;
      for (int64_t n = 0; n < N; ++n) acc2 += (double)gm[n] * (double)B[n * r + j];
      u_out[m * r + j] = acc2;
    }
  }
  /* dX: one row of dY at a time.  Each dX[m, k] is still one sum over n in
   * ascending order; the loops only run n outside k so that W_hat is read
   * row by row. */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const int64_t m = rows[ri];
    const float *gm = dY + m * N;
    const double *um = u_out + m * r;
    double *base = dX + ri * K;
    for (int64_t k = 0; k < K; ++k) base[k] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double g = (double)gm[n];
      const float *wn = w + n * K;
      for (int64_t k = 0; k < K; ++k) base[k] += g * (double)wn[k];
    }
    const uint8_t *km = keep ? keep + m * K : NULL;
    for (int64_t k = 0; k < K; ++k) {
      double lora = 0.0;
      for (int32_t j = 0; j < r; ++j) lora += um[j] * (double)A[j * K + k];
      if (km) lora = km[k] ? keep_scale * lora : 0.0;
      base[k] = base[k] + s * lora;
    }
  }
  /* dA[j, k] = s * sum_m u[m, j] x[m, k] and dB[n, j] = s * sum_m dY[m, n] t[m, j]:
   * each a sum over m in ascending order, kept in a binary64 accumulator per
   * element while the rows of x (of dY) are read one after another. */
  const int64_t kChunk = 256;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t k0 = 0; k0 < K; k0 += kChunk) {
    const int64_t k1 = k0 + kChunk < K ? k0 + kChunk : K;
    double *acc = (double *)calloc((size_t)(k1 - k0) * (size_t)r, sizeof(double));
    for (int64_t m = 0; m < M; ++m)
      for (int32_t j = 0; j < r; ++j) {
        const double uj = u_out[m * r + j];
        for (int64_t k = k0; k < k1; ++k)
          if (!keep || keep[m * K + k]) acc[j * (k1 - k0) + (k - k0)] += uj * (double)x[m * K + k];
      }
    const double sa = keep ? s * keep_scale : s;
    for (int32_t j = 0; j < r; ++j)
      for (int64_t k = k0; k < k1; ++k) dA[j * K + k] = sa * acc[j * (k1 - k0) + (k - k0)];
    free(acc);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t n0 = 0; n0 < N; n0 += kChunk) {
    const int64_t n1 = n0 + kChunk < N ? n0 + kChunk : N;
    double *acc = (double *)calloc((size_t)(n1 - n0) * (size_t)r, sizeof(double));
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = n0; n < n1; ++n) {
        const double g = (double)dY[m * N + n];
        for (int32_t j = 0; j < r; ++j) acc[(n - n0) * r + j] += g * t_out[m * r + j];
      }
    for (int64_t n = n0; n < n1; ++n)
      for (int32_t j = 0; j < r; ++j) dB[n * r + j] = s * acc[(n - n0) * r + j];
    free(acc);
  }
}

/* binary64 -> bf16 bits, round to nearest, ties to even: bf16 keeps 8
 * significant bits (the binary32 exponent range), so v = m 2^e with
 * m in [0.5, 1) is rounded as rint(m 2^8) 2^(e-8) (rint rounds half to even
 * in the default rounding mode); below 2^-126 the spacing is fixed at
 * 2^-133.  Finite inputs below 2^128 only. */
uint16_t oracle_bf16_rne_double(double v) {
  double q;
  if (v == 0.0) {
    q = v;
  } else if (fabs(v) < ldexp(1.0, -126)) {
    q = rint(ldexp(v, 133)) * ldexp(1.0, -133);
  } else {
    int e;
    frexp(v, &e);
    q = ldexp(rint(ldexp(v, 8 - e)), e - 8);
  }
  float f = (float)q; /* exact: q has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Adapter merge.  [QLoRA-26] Step 5 (conclusion: adapter merge and
 * deployment loading are what a trained adapter still has to pass) and
 * [Select-65] (a merged model as the delivered artifact).  Merging folds the
 * LoRA branch of the forward formula into the base weight:
 *   x W_hat^T + (x A^T) B^T alpha/r = x (W_hat + alpha/r B A)^T,
 * so the merged weight is W_hat + (alpha/r) B A, here in bf16 (the compute
 * dtype), rounded once from the binary64 sum (ascending j).
 *   w_hat [N, K], A [r, K], B [N, r]; exact (nullable) gets the binary64
 *   values before rounding, bits the bf16 patterns. */
void oracle_merge_bf16(const float *w_hat, int64_t N, int64_t K, const float *A, const float *B,
                       int32_t r, double alpha, double *exact, uint16_t *bits) {
  const double s = alpha / (double)r;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      double lora = 0.0;
      for (int32_t j = 0; j < r; ++j) lora += (double)B[n * r + j] * (double)A[j * K + k];
      const double v = (double)w_hat[n * K + k] + s * lora;
      if (exact) exact[n * K + k] = v;
      bits[n * K + k] = oracle_bf16_rne_double(v);
    }
  }
}

/* Storage accounting.  [QLoRA-26] Step 4 (qlora_trainable_state_ledger:
 * packed size (numel + 1) // 2 bytes) and [Finetune-4] (4.5 -> ~4.127 bits
 * per parameter): bytes of packed indices, block constants and second-level
 * scales for one matrix. */
int oracle_nf4_storage_bytes(int64_t rows, int64_t cols, int32_t block, int32_t group,
                             int64_t *packed_b, int64_t *const_b, int64_t *scale_b) {
  if (rows < 0 || cols < 0 || block <= 0 || group < 0) return ORACLE_EINVAL;
  const int64_t n = rows * cols;
  const int64_t nblocks = (n + block - 1) / block;
  *packed_b = (n + 1) / 2;
  if (group == 0) {
    *const_b = nblocks * 4; /* binary32 absmax per block */
    *scale_b = 0;
  } else {
    *const_b = nblocks * 1; /* int8 code per block */
    *scale_b = ((nblocks + group - 1) / group) * 4;
  }
  return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Thread count of the OpenMP loops above (timing only: every result is
 * independent of it, each output element being one sequential sum). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * CPU oracle for the MXFP8 publishing GEMM and its Lamport mailbox.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes, and the passage each step follows:
 *
 *  - MXFP8 operands (page "vllm.models.deepseek_v41.nvidia.specialized_decode.
 *    boundary.publishing_gemm", PublishingMxfp8Linear.__call__ and _compile:
 *    Float8E4M3FN elements, Float8E8M0FNU scales, sf_vec_size=32).  E4M3FN and
 *    E8M0FNU codes are decoded to exact doubles from the formats' definitions.
 *  - The product C[n, m] = sum_k W[n, k] x[m, k] (same page, module
 *    description, "GEMM structure"), accumulated in FP64 with k ascending, then
 *    rounded ONCE from the double to BF16, round-to-nearest-even.
 *  - The publish (same page, module description and publish_value): every
 *    output goes into mailbox[stage_state[0]][token][column] as BF16 with
 *    negative zero cleared (each 0x8000 half-word becomes 0x0000), packed so
 *    column c is the low half of a 32-bit word and c + 1 the high half; then
 *    stage_state[1] is set to that generation (epilog_warp, "hand the
 *    generation to the consumer").
 *  - The consume (page "vllm.models.deepseek_v41.nvidia.ops.cute_dsl.
 *    all_gather", module description steps 2 and 3, with one rank): read the
 *    generation stage_state[1], copy every slot of the m published rows to the
 *    output, store the sentinel word 0x80000000 back into each, and advance
 *    the next generation stage_state[0] to (g + 1) mod 3 with the arrival
 *    count stage_state[2] cleared.
 *
 * Parity of the GEMM is pinned by the tests against exact rational sums,
 * integer-valued closed forms and a library float64 matmul.  The one thing no
 * pin fixes is the tensor core's own FP32 summation order; the GPU path is
 * held to a tolerance there, not bit-exactness.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GENERATIONS 3
#define ORACLE_SENTINEL 0x80000000u

/* Status codes of the mailbox model. */
#define ORACLE_OK 0
#define ORACLE_ERR_ARGS 1
#define ORACLE_ERR_STATE 5
#define ORACLE_ERR_SENTINEL 4 /* a consume would poll forever: a word is still the sentinel */

/* E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities; exponent 15 with mantissa 7 is NaN; exponent 0 is subnormal
 * (mantissa / 8 * 2^-6). */
double oracle_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int exponent = (code >> 3) & 0xF;
  int mantissa = code & 0x7;
  double magnitude;
  if (exponent == 15 && mantissa == 7) return NAN;
  if (exponent == 0)
    magnitude = ldexp((double)mantissa / 8.0, -6);
  else
    magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
  return sign ? -magnitude : magnitude;
}

/* E8M0FNU: an unsigned biased exponent, value 2^(code - 127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* Round a double to BF16 (8 exponent bits, 7 stored mantissa bits), once,
 * round-to-nearest with ties to even, and return the 16 bits. */
uint16_t oracle_bf16_rne(double value) {
  if (isnan(value)) return 0x7FC0;
  int negative = signbit(value) ? 1 : 0;
  double magnitude = fabs(value);
  if (magnitude == 0.0) return (uint16_t)(negative << 15);
  if (isinf(magnitude)) return (uint16_t)((negative << 15) | 0x7F80);
  int e2;
  frexp(magnitude, &e2);           /* magnitude = f * 2^e2, f in [0.5, 1) */
  int exponent = e2 - 1;           /* floor(log2(magnitude)) */
  if (exponent < -126) exponent = -126; /* subnormals share the quantum 2^-133 */
  double quantum = ldexp(1.0, exponent - 7);
  double units = magnitude / quantum; /* exact: division by a power of two */
  double lower = floor(units);
  double fraction = units - lower;
  double rounded;
  if (fraction > 0.5)
    rounded = lower + 1.0;
  else if (fraction < 0.5)
    rounded = lower;
  else
    rounded = (fmod(lower, 2.0) == 0.0) ? lower : lower + 1.0;
  double result = rounded * quantum;
  if (result >= ldexp(1.0, 128)) return (uint16_t)((negative << 15) | 0x7F80);
  /* result is exactly representable in BF16, so also in binary32, whose top
   * 16 bits are then the BF16 encoding. */
  float as_float = (float)result;
  uint32_t bits;
  memcpy(&bits, &as_float, sizeof bits);
  return (uint16_t)((bits >> 16) | ((uint32_t)negative << 15));
}

/* The publish's sanitisation of one BF16 half-word: negative zero becomes
 * positive zero, so no packed 32-bit word can equal the sentinel. */
uint16_t oracle_clear_negative_zero(uint16_t half) {
  return half == 0x8000 ? (uint16_t)0x0000 : half;
}

/* One dot product sum_k W[n, k] x[t, k] in FP64, k ascending, each operand the
 * decoded element times its block's scale 2^(s - 127). */
double oracle_dot(int k, const uint8_t* w_row, const uint8_t* w_scale_row,
                  const uint8_t* x_row, const uint8_t* x_scale_row) {
  double sum = 0.0;
  for (int kk = 0; kk < k; ++kk) {
    double w = oracle_e4m3_value(w_row[kk]) * oracle_e8m0_value(w_scale_row[kk / 32]);
    double x = oracle_e4m3_value(x_row[kk]) * oracle_e8m0_value(x_scale_row[kk / 32]);
    sum += w * x;
  }
  return sum;
}

/* acc[t][n] = sum_k W[n, k] x[t, k] in FP64 for t < m, n < N.  Layouts:
 * W [N][K], W scales [N][K/32], x [m][K], x scales [m][K/32], all row-major
 * bytes.  Each row is decoded once, then the sums run k ascending. */
int oracle_gemm_fp64(int n, int k, int m, const uint8_t* w, const uint8_t* w_scale,
                     const uint8_t* x, const uint8_t* x_scale, double* acc) {
  if (n <= 0 || k <= 0 || m <= 0 || k % 32) return ORACLE_ERR_ARGS;
  int blocks = k / 32;
  double* xv = (double*)malloc(sizeof(double) * (size_t)m * (size_t)k);
  double* wv = (double*)malloc(sizeof(double) * (size_t)k);
  if (!xv || !wv) {
    free(xv);
    free(wv);
    return ORACLE_ERR_ARGS;
  }
  for (int t = 0; t < m; ++t)
    for (int kk = 0; kk < k; ++kk)
      xv[(size_t)t * k + kk] = oracle_e4m3_value(x[(size_t)t * k + kk]) *
                               oracle_e8m0_value(x_scale[(size_t)t * blocks + kk / 32]);
  for (int col = 0; col < n; ++col) {
    for (int kk = 0; kk < k; ++kk)
      wv[kk] = oracle_e4m3_value(w[(size_t)col * k + kk]) *
               oracle_e8m0_value(w_scale[(size_t)col * blocks + kk / 32]);
    for (int t = 0; t < m; ++t) {
      const double* xr = xv + (size_t)t * k;
      double sum = 0.0;
      for (int kk = 0; kk < k; ++kk) sum += wv[kk] * xr[kk];
      acc[(size_t)t * n + col] = sum;
    }
  }
  free(xv);
  free(wv);
  return ORACLE_OK;
}

/* C [m][N] as BF16 bits: the FP64 sums rounded once (C keeps negative zero;
 * only the mailbox copy is sanitised). */
int oracle_gemm_bf16(int n, int k, int m, const uint8_t* w, const uint8_t* w_scale,
                     const uint8_t* x, const uint8_t* x_scale, uint16_t* c) {
  double* acc = (double*)malloc(sizeof(double) * (size_t)m * (size_t)n);
  if (!acc) return ORACLE_ERR_ARGS;
  int status = oracle_gemm_fp64(n, k, m, w, w_scale, x, x_scale, acc);
  if (status == ORACLE_OK)
    for (size_t i = 0; i < (size_t)m * (size_t)n; ++i) c[i] = oracle_bf16_rne(acc[i]);
  free(acc);
  return status;
}

/* C = BF16(alpha * sum_k W x): the global scale of the gemm page's
 * epilog_warp (use_scale), applied to the FP64 sum before the one rounding. */
int oracle_gemm_bf16_scaled(int n, int k, int m, const uint8_t* w, const uint8_t* w_scale,
                            const uint8_t* x, const uint8_t* x_scale, float alpha, uint16_t* c) {
  double* acc = (double*)malloc(sizeof(double) * (size_t)m * (size_t)n);
  if (!acc) return ORACLE_ERR_ARGS;
  int status = oracle_gemm_fp64(n, k, m, w, w_scale, x, x_scale, acc);
  if (status == ORACLE_OK)
    for (size_t i = 0; i < (size_t)m * (size_t)n; ++i)
      c[i] = oracle_bf16_rne((double)alpha * acc[i]);
  free(acc);
  return status;
}

/* Selected outputs only: out[i] = BF16(sum_k W[cols[i], k] x[rows[i], k]).
 * Used to check full-size runs at sampled positions. */
int oracle_gemm_sample(int n, int k, int m, const uint8_t* w, const uint8_t* w_scale,
                       const uint8_t* x, const uint8_t* x_scale, int count,
                       const int32_t* rows, const int32_t* cols, uint16_t* out) {
  if (n <= 0 || k <= 0 || m <= 0 || k % 32) return ORACLE_ERR_ARGS;
  int blocks = k / 32;
  for (int i = 0; i < count; ++i) {
    int t = rows[i], col = cols[i];
    if (t < 0 || t >= m || col < 0 || col >= n) return ORACLE_ERR_ARGS;
    out[i] = oracle_bf16_rne(oracle_dot(k, w + (size_t)col * k, w_scale + (size_t)col * blocks,
                                        x + (size_t)t * k, x_scale + (size_t)t * blocks));
  }
  return ORACLE_OK;
}

/* Mailbox words: mailbox[g][t][w] for g < 3, t < capacity, w < N/2 (32-bit
 * words, word w holding columns 2w (low half) and 2w + 1 (high half)).
 * State words: [0] next generation, [1] active generation, [2] arrival count,
 * [3] error flags.  At rest every word is the sentinel and the state is zero. */
int oracle_mailbox_init(uint32_t* mailbox, int32_t* state, int capacity, int n) {
  if (capacity <= 0 || n <= 0 || n % 8) return ORACLE_ERR_ARGS;
  size_t words = (size_t)ORACLE_GENERATIONS * (size_t)capacity * (size_t)(n / 2);
  for (size_t i = 0; i < words; ++i) mailbox[i] = ORACLE_SENTINEL;
  for (int i = 0; i < 4; ++i) state[i] = 0;
  return ORACLE_OK;
}

/* The epilogue's publish of C [m][N] (BF16 bits) into generation state[0],
 * followed by state[1] = that generation. */
int oracle_publish(uint32_t* mailbox, int32_t* state, int capacity, int n, int m,
                   const uint16_t* c) {
  if (capacity <= 0 || n <= 0 || n % 8 || m <= 0 || m > capacity) return ORACLE_ERR_ARGS;
  int g = state[0];
  if (g < 0 || g >= ORACLE_GENERATIONS) return ORACLE_ERR_STATE;
  int half_n = n / 2;
  for (int t = 0; t < m; ++t)
    for (int w = 0; w < half_n; ++w) {
      uint32_t low = oracle_clear_negative_zero(c[(size_t)t * n + 2 * w]);
      uint32_t high = oracle_clear_negative_zero(c[(size_t)t * n + 2 * w + 1]);
      mailbox[((size_t)g * capacity + t) * half_n + w] = low | (high << 16);
    }
  state[1] = g;
  return ORACLE_OK;
}

/* The consumer: generation g = state[1]; copy the m rows out, reset them to
 * the sentinel, state[0] = (g + 1) mod 3, state[2] = 0.  A slot that still
 * holds a sentinel word would make the GPU consumer poll until its time
 * limit; the oracle reports that as ORACLE_ERR_SENTINEL (after doing the rest
 * of the call, as the bounded GPU poll does). */
int oracle_consume(uint32_t* mailbox, int32_t* state, int capacity, int n, int m,
                   uint16_t* out) {
  if (capacity <= 0 || n <= 0 || n % 8 || m <= 0 || m > capacity) return ORACLE_ERR_ARGS;
  int g = state[1];
  if (g < 0 || g >= ORACLE_GENERATIONS) return ORACLE_ERR_STATE;
  int half_n = n / 2;
  int status = ORACLE_OK;
  for (int t = 0; t < m; ++t)
    for (int w = 0; w < half_n; ++w) {
      size_t slot = ((size_t)g * capacity + t) * half_n + w;
      uint32_t word = mailbox[slot];
      if (word == ORACLE_SENTINEL) status = ORACLE_ERR_SENTINEL;
      out[(size_t)t * n + 2 * w] = (uint16_t)(word & 0xFFFF);
      out[(size_t)t * n + 2 * w + 1] = (uint16_t)(word >> 16);
      mailbox[slot] = ORACLE_SENTINEL;
    }
  state[0] = (g + 1) % ORACLE_GENERATIONS;
  state[2] = 0;
  return status;
}

/* One whole call of the path: GEMM, publish, consume.  C may be NULL. */
int oracle_chain(int n, int k, int m, const uint8_t* w, const uint8_t* w_scale,
                 const uint8_t* x, const uint8_t* x_scale, uint32_t* mailbox,
                 int32_t* state, int capacity, uint16_t* c, uint16_t* out) {
  uint16_t* local = c;
  if (!local) local = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)m * (size_t)n);
  if (!local) return ORACLE_ERR_ARGS;
  int status = oracle_gemm_bf16(n, k, m, w, w_scale, x, x_scale, local);
  if (status == ORACLE_OK) status = oracle_publish(mailbox, state, capacity, n, m, local);
  if (status == ORACLE_OK) status = oracle_consume(mailbox, state, capacity, n, m, out);
  if (!c) free(local);
  return status;
}

/* ------------------------------------------------------------------------
 * The Lamport all-gather with one rank (page "vllm.models.deepseek_v41.
 * nvidia.ops.cute_dsl.all_gather", module description steps 1-3 and
 * _AllGatherKernel.kernel), word by word.  Its own mailbox is
 * mailbox[generation][pack] = [3][capacity_words] 32-bit words; its state is
 * int32[2]: [0] the call's generation, [1] the arrival count.
 * ------------------------------------------------------------------------ */

int oracle_gather_init(uint32_t* mailbox, int32_t* state, int capacity_words) {
  if (capacity_words <= 0 || capacity_words % 4) return ORACLE_ERR_ARGS;
  for (size_t i = 0; i < (size_t)ORACLE_GENERATIONS * capacity_words; ++i)
    mailbox[i] = ORACLE_SENTINEL;
  state[0] = 0;
  state[1] = 0;
  return ORACLE_OK;
}

/* One call on `words` input words (a positive multiple of 4, at most the
 * capacity): (1) publish every word into this rank's slot of generation g,
 * a word equal to the sentinel going out as 0; (2) collect: read the slot, a
 * sentinel word there meaning the poll would not end (ORACLE_ERR_SENTINEL),
 * write the word to the output, store the sentinel back; (3) advance the
 * generation and clear the arrival count. */
int oracle_all_gather(uint32_t* mailbox, int32_t* state, int capacity_words, const uint32_t* in,
                      int words, uint32_t* out) {
  if (capacity_words <= 0 || capacity_words % 4 || words <= 0 || words % 4 ||
      words > capacity_words)
    return ORACLE_ERR_ARGS;
  int g = state[0];
  if (g < 0 || g >= ORACLE_GENERATIONS) return ORACLE_ERR_STATE;
  uint32_t* slot = mailbox + (size_t)g * capacity_words;
  for (int i = 0; i < words; ++i) slot[i] = in[i] == ORACLE_SENTINEL ? 0u : in[i];
  int status = ORACLE_OK;
  for (int i = 0; i < words; ++i) {
    if (slot[i] == ORACLE_SENTINEL) status = ORACLE_ERR_SENTINEL;
    out[i] = slot[i];
    slot[i] = ORACLE_SENTINEL;
  }
  state[0] = (g + 1) % ORACLE_GENERATIONS;
  state[1] = 0;
  return status;
}

/* ------------------------------------------------------------------------
 * The tagged-pair mailbox (page "vllm.models.deepseek_v41.amd.mono.common.
 * sync", Mailbox: every 32-bit value stored next to the launch's tag, a
 * consumer polls until all tags match, nothing is reset).  Pairs are
 * pairs[t][w] = (word, tag) for t < capacity, w < N/2, word w holding BF16
 * columns 2w (low half) and 2w + 1; tag 0 is the armed state, never live.
 * ------------------------------------------------------------------------ */

int oracle_tagged_init(uint32_t* pairs, int capacity, int n) {
  if (capacity <= 0 || n <= 0 || n % 8) return ORACLE_ERR_ARGS;
  memset(pairs, 0, sizeof(uint32_t) * 2 * (size_t)capacity * (size_t)(n / 2));
  return ORACLE_OK;
}

/* put: C [m][N] (BF16 bits, moved unchanged) with `tag`. */
int oracle_tagged_publish(uint32_t* pairs, int capacity, int n, int m, const uint16_t* c,
                          uint32_t tag) {
  if (capacity <= 0 || n <= 0 || n % 8 || m <= 0 || m > capacity || tag == 0)
    return ORACLE_ERR_ARGS;
  int half_n = n / 2;
  for (int t = 0; t < m; ++t)
    for (int w = 0; w < half_n; ++w) {
      size_t at = 2 * ((size_t)t * half_n + w);
      pairs[at] = (uint32_t)c[(size_t)t * n + 2 * w] | ((uint32_t)c[(size_t)t * n + 2 * w + 1] << 16);
      pairs[at + 1] = tag;
    }
  return ORACLE_OK;
}

/* poll: the value words of rows t < m once every tag equals `tag`; a stale
 * tag means the poll would not end (ORACLE_ERR_SENTINEL; the words are still
 * copied).  Nothing is reset. */
int oracle_tagged_consume(const uint32_t* pairs, int capacity, int n, int m, uint32_t tag,
                          uint16_t* out) {
  if (capacity <= 0 || n <= 0 || n % 8 || m <= 0 || m > capacity || tag == 0)
    return ORACLE_ERR_ARGS;
  int half_n = n / 2;
  int status = ORACLE_OK;
  for (int t = 0; t < m; ++t)
    for (int w = 0; w < half_n; ++w) {
      size_t at = 2 * ((size_t)t * half_n + w);
      if (pairs[at + 1] != tag) status = ORACLE_ERR_SENTINEL;
      out[(size_t)t * n + 2 * w] = (uint16_t)(pairs[at] & 0xFFFF);
      out[(size_t)t * n + 2 * w + 1] = (uint16_t)(pairs[at] >> 16);
    }
  return status;
}

/*
 * fp8_oracle.c -- plain, slow, obviously-correct CPU oracle for the FP8
 * quantize + scaled-GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Sources (page title, section):
 *   [P2] "What is FP8 inference on H100 (Transformer Engine)?" (aivaro.ru
 *        answers/458): s2 "Architecture" -- E4M3 = 4 exponent bits + 3 mantissa
 *        bits; s3 "How FP8 inference works", steps 2-6 and its pseudocode
 *        example fp8_gemm -- amax -> scale = amax/448 -> x/scale rounded to
 *        float8_e4m3fn -> matmul with FP32 accumulation -> result times
 *        scale_A*scale_B -> FP16; s5 "Impact on accuracy" -- E4M3 range
 *        -448..448; s8 "Limitations" -- scales are stored as float32.
 *   [P5] "FP8 chi tiet" (transformers fine-grained FP8 guide), opening
 *        bullets -- weights quantized per 2-D block weight_block_size=(128,128);
 *        activations quantized per token per group of 128 input channels.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R1 E4M3 is the "fn" variant: bias 7, no infinities, S.1111.111 = NaN.
 *   R2 the stored scale is the dequant factor s = fl32(amax / 448), an IEEE
 *      single-precision divide; quantization is fl32(x / s) (IEEE single
 *      divide, round-to-nearest) followed by an E4M3 rounding.
 *   R3 E4M3 rounding is round-to-nearest-even with saturation to +-448
 *      (|y| > 448 after rounding clamps to 448); the sign is kept, so a
 *      negative value that rounds to zero gives 0x80.
 *   R4 amax == 0 gives s = 1.0f.
 *   R5 groups run along K (input channels) per token; weight blocks are 128
 *      output rows x 128 input columns; a partial edge block in N uses only
 *      its valid rows.
 *   R6 the GEMM result R is computed in double from the decoded operands; it
 *      is the exact sum of products, scaled in double and left unrounded.
 *   R7 block-scaled mode: the partial sum over each 128-wide K block is
 *      multiplied by that block's activation-group scale and weight-block
 *      scale before the blocks are added (the only way both scale grids can
 *      act on one dot product).
 *   R8 static / delayed scaling ([P1] "Technical assignment: implement FP8
 *      inference on H100", stage 3 steps 1-2: a calibrated scale, or the
 *      Transformer Engine recipe DelayedScaling(margin=0, interval=4)): the
 *      quantizer step is the same E4M3(fl32(x / s)) with the given s (any
 *      |x / s| > 448 saturates); the next scale from a window of recorded
 *      amaxes is s = fl32(max / 448) (1 when the max is 0, as R4) times
 *      2^margin -- a larger margin leaves more headroom, as in the recipe,
 *      whose quantization multiplier is divided by 2^margin.
 *   R10 UE8M0 scales ([P5] "UE8M0 scale format": DeepSeek-V4-style
 *      checkpoints keep FP8 weight scales as packed float8_e8m0fnu, and the
 *      Blackwell DeepGEMM kernels take only such scales): a scale is a power
 *      of two 2^(c - 127) stored as its biased exponent byte c (c = 255 is
 *      NaN).  The quantizer first takes the FP32 scale of R2/R4,
 *      fl32(amax / 448), then rounds it UP to a power of two (so no element
 *      exceeds 448 by more than that FP32 rounding), clamped to 2^-127, the
 *      smallest UE8M0 value; x / s is then an exact power-of-two division.
 *   R11 E5M2 ([P2] s2: 5 exponent + 2 mantissa bits, the format named for
 *      gradients; [P3] s2 the same split): the IEEE-style layout, bias 15,
 *      S.11111.00 = infinity, S.11111.xx (xx != 0) = NaN, largest finite
 *      value 1.75 * 2^15 = 57344; encoding rounds to nearest even and, like
 *      the E4M3 path, saturates finite overflow (and infinities) to +-57344.
 *   R9 per-channel weight scaling ([P2] s5 "How to minimize the losses":
 *      per-tensor scaling, or per-channel scaling for weights): one unit per
 *      output channel, i.e. per row of W[N][K], quantized as in [P2] s3 steps
 *      2-4; the GEMM multiplies the exact dot product by the activation's
 *      per-tensor scale and the row's scale.
 *
 * Layouts: activations A[M][K] and weights W[N][K] are row-major with K
 * contiguous, given as raw 16-bit patterns (FP16 or BF16).  Token-group scales
 * are stored sa[g*M + m] (K/128 rows of M); weight-block scales are stored
 * sb[i*(K/128) + j] (ceil(N/128) rows of K/128).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---------------------------------------------------------------- threads */

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------- 16-bit float decoders */

static float f32_of_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t bits_of_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.  Every
 * binary16 value is exactly representable in binary32. */
float oracle_half_to_float(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int f = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return (float)(sign ? -v : v);
}

/* bfloat16 is by definition the upper 16 bits of a binary32 pattern. */
float oracle_bf16_to_float(uint16_t h) { return f32_of_bits((uint32_t)h << 16); }

static float in_to_float(uint16_t h, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_bf16_to_float(h) : oracle_half_to_float(h);
}

/* ------------------------------------------------------------ O1: decode */

/* E4M3 (fn): value = (-1)^s * (1 + m/8) * 2^(e-7) for e >= 1, the subnormal
 * (-1)^s * (m/8) * 2^-6 for e == 0, and NaN for e == 15 && m == 7 [P2 s2, R1].
 * Largest finite: e = 15, m = 6 -> 1.75 * 2^8 = 448 [P2 s3 step 3, s5]. */
double oracle_e4m3_decode(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* The same value as an exact integer count of 2^-9 units (|n| <= 229376).
 * Used only by the exact integer cross-check of the GEMM. */
int64_t oracle_e4m3_units(uint8_t b) {
  int s = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  int64_t n = (e == 0) ? (int64_t)m : ((int64_t)(8 + m) << (e - 1));
  return s ? -n : n;
}

/* ------------------------------------------------------------ O2: encode */

/* Round a binary32 value to E4M3 with round-to-nearest-even and saturation
 * [P2 s3 step 4, R1, R3].  Pure integer arithmetic on the binary32 bits:
 * the magnitude is an integer mantissa times a power of two, so the grid
 * point and the tie can be decided exactly. */
uint8_t oracle_e4m3_encode(float y) {
  uint32_t u = bits_of_f32(y);
  uint8_t sign = (uint8_t)((u >> 31) << 7);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7F); /* NaN stays NaN */
  if (a >= 0x43E80000u) return (uint8_t)(sign | 0x7E); /* |y| >= 464 (incl. inf): clamp */
  int ebits = (int)(a >> 23);
  if (ebits == 0) return sign; /* binary32 subnormal or zero: far below 2^-10 */
  /* |y| = mant * 2^(e - 23), mant in [2^23, 2^24) */
  uint64_t mant = (uint64_t)((a & 0x7FFFFFu) | 0x800000u);
  int e = ebits - 127;
  /* E4M3 binade exponent (subnormals share the quantum of binade -6) */
  int ee = e < -6 ? -6 : e;
  /* grid step is 2^(ee - 3); n = |y| / step = mant * 2^(e - 23 - ee + 3) */
  int shift = 20 + (ee - e); /* >= 20 */
  uint64_t n;
  if (shift >= 40) {
    n = 0; /* mant < 2^24 <= half the step: rounds to zero */
  } else {
    uint64_t q = mant >> shift;
    uint64_t rem = mant & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1;
    n = q;
  }
  /* value = n * 2^(ee - 3); n <= 16 */
  if (n == 0) return sign;
  if (n == 16) { /* carry into the next binade */
    n = 8;
    ee += 1;
  }
  int code;
  if (n < 8) {
    code = (int)n; /* only possible for ee == -6: E4M3 subnormal */
  } else {
    code = ((ee + 7) << 3) | (int)(n - 8);
  }
  if (code > 0x7E) code = 0x7E; /* 480 does not exist in E4M3 fn */
  return (uint8_t)(sign | code);
}

/* ----------------------------------------------------- E5M2 codec [R11] */

double oracle_e5m2_decode(uint8_t b) {
  int sign = b >> 7;
  int E = (b >> 2) & 31;
  int m = b & 3;
  double v;
  if (E == 31) {
    if (m != 0) return NAN;
    v = INFINITY;
  } else if (E == 0) {
    v = ldexp((double)m, -16); /* subnormal: m * 2^-2 * 2^-14 */
  } else {
    v = ldexp(1.0 + m / 4.0, E - 15);
  }
  return sign ? -v : v;
}

/* Round-to-nearest-even onto the E5M2 grid with saturation to +-57344; the
 * same exact integer method as the E4M3 encoder (grid step 2^(e - 2) in the
 * normal binades, 2^-16 below 2^-14). */
uint8_t oracle_e5m2_encode(float y) {
  uint32_t u = bits_of_f32(y);
  uint8_t sign = (uint8_t)((u >> 31) << 7);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint8_t)(sign | 0x7F); /* NaN */
  if (a >= 0x47700000u) return (uint8_t)(sign | 0x7B); /* |y| >= 61440 = (57344 + 65536) / 2, incl. inf */
  int ebits = (int)(a >> 23);
  if (ebits == 0) return sign; /* binary32 subnormal or zero: far below 2^-17 */
  uint64_t mant = (uint64_t)((a & 0x7FFFFFu) | 0x800000u);
  int e = ebits - 127;
  int ee = e < -14 ? -14 : e;
  int shift = 21 + (ee - e); /* |y| / 2^(ee - 2) = mant * 2^(e - 23 - ee + 2) */
  uint64_t n;
  if (shift >= 40) {
    n = 0;
  } else {
    uint64_t q = mant >> shift;
    uint64_t rem = mant & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1;
    n = q;
  }
  /* value = n * 2^(ee - 2); n <= 8 */
  if (n == 0) return sign;
  if (n == 8) { /* carry into the next binade */
    n = 4;
    ee += 1;
  }
  int code;
  if (n < 4) {
    code = (int)n; /* ee == -14: E5M2 subnormal */
  } else {
    code = ((ee + 15) << 2) | (int)(n - 4);
  }
  if (code > 0x7B) code = 0x7B; /* above 57344 only infinity remains: saturate */
  return (uint8_t)(sign | code);
}

void oracle_e5m2_encode_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_encode(y[i]);
}

/* --------------------------------------------------- O3: the quantizers */

static float scale_of_amax(float amax) {
  /* [P2 s3 step 3 and pseudocode]: scale = max|x| / 448, in FP32 [R2, R4] */
  if (amax == 0.0f) return 1.0f;
  return amax / 448.0f;
}

/* Per-tensor: one scale over all numel elements [P2 s3 steps 2-4]. */
void oracle_quantize_per_tensor(const uint16_t* x, int dtype, int64_t numel,
                                uint8_t* q, float* scale_out) {
  float amax = 0.0f;
  for (int64_t i = 0; i < numel; ++i) {
    float v = fabsf(in_to_float(x[i], dtype));
    if (v > amax) amax = v;
  }
  float s = scale_of_amax(amax);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < numel; ++i) {
    float t = in_to_float(x[i], dtype) / s;
    q[i] = oracle_e4m3_encode(t);
  }
  *scale_out = s;
}

/* Per token, per group of 128 input channels [P5 opening bullets, R5].
 * x: [M][K]; q: [M][K]; sa: [K/128][M]. K must be a multiple of 128. */
void oracle_quantize_token_group(const uint16_t* x, int dtype, int64_t M, int64_t K,
                                 uint8_t* q, float* sa) {
  int64_t G = K / 128;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      const uint16_t* row = x + m * K + g * 128;
      float amax = 0.0f;
      for (int k = 0; k < 128; ++k) {
        float v = fabsf(in_to_float(row[k], dtype));
        if (v > amax) amax = v;
      }
      float s = scale_of_amax(amax);
      for (int k = 0; k < 128; ++k) {
        float t = in_to_float(row[k], dtype) / s;
        q[m * K + g * 128 + k] = oracle_e4m3_encode(t);
      }
      sa[g * M + m] = s;
    }
  }
}

/* Per 128x128 weight block [P5 opening bullets, R5].
 * w: [N][K]; q: [N][K]; sb: [ceil(N/128)][K/128].  K % 128 == 0. */
void oracle_quantize_weight_block(const uint16_t* w, int dtype, int64_t N, int64_t K,
                                  uint8_t* q, float* sb) {
  int64_t NB = (N + 127) / 128;
  int64_t KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bi = 0; bi < NB; ++bi) {
    for (int64_t bj = 0; bj < KB; ++bj) {
      int64_t r0 = bi * 128;
      int64_t r1 = r0 + 128 < N ? r0 + 128 : N;
      float amax = 0.0f;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = bj * 128; c < bj * 128 + 128; ++c) {
          float v = fabsf(in_to_float(w[r * K + c], dtype));
          if (v > amax) amax = v;
        }
      float s = scale_of_amax(amax);
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = bj * 128; c < bj * 128 + 128; ++c) {
          float t = in_to_float(w[r * K + c], dtype) / s;
          q[r * K + c] = oracle_e4m3_encode(t);
        }
      sb[bi * KB + bj] = s;
    }
  }
}

/* Per output channel [R9]: one scale per row of W.
 * w: [N][K]; q: [N][K]; sb: [N]. */
void oracle_quantize_per_channel(const uint16_t* w, int dtype, int64_t N, int64_t K,
                                 uint8_t* q, float* sb) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    const uint16_t* row = w + n * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float v = fabsf(in_to_float(row[k], dtype));
      if (v > amax) amax = v;
    }
    float s = scale_of_amax(amax);
    for (int64_t k = 0; k < K; ++k) q[n * K + k] = oracle_e4m3_encode(in_to_float(row[k], dtype) / s);
    sb[n] = s;
  }
}

/* UE8M0 [R10]: the value of a scale code, and the code of the power-of-two
 * scale that a dynamic quantizer uses for a given amax. */
float oracle_ue8m0_decode(uint8_t c) {
  if (c == 0xFF) return f32_of_bits(0x7FC00000u);
  return ldexpf(1.0f, (int)c - 127);
}

uint8_t oracle_ue8m0_of_amax(float amax) {
  float s = scale_of_amax(amax);             /* fl32(amax / 448), 1 when amax == 0 */
  int e;
  float m = frexpf(s, &e);                   /* s = m * 2^e, m in [0.5, 1) */
  int k = (m == 0.5f) ? e - 1 : e;           /* the smallest k with 2^k >= s */
  if (k < -127) k = -127;
  return (uint8_t)(k + 127);
}

/* Token-group and weight-block quantizers with UE8M0 scales [R10]: as the
 * FP32-scale ones, with s replaced by its power-of-two round-up.  The scales
 * are returned as codes; their values are oracle_ue8m0_decode(code). */
void oracle_quantize_token_group_ue8m0(const uint16_t* x, int dtype, int64_t M, int64_t K,
                                       uint8_t* q, uint8_t* sa_code) {
  int64_t G = K / 128;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      const uint16_t* row = x + m * K + g * 128;
      float amax = 0.0f;
      for (int k = 0; k < 128; ++k) {
        float v = fabsf(in_to_float(row[k], dtype));
        if (v > amax) amax = v;
      }
      uint8_t c = oracle_ue8m0_of_amax(amax);
      float s = oracle_ue8m0_decode(c);
      for (int k = 0; k < 128; ++k) q[m * K + g * 128 + k] = oracle_e4m3_encode(in_to_float(row[k], dtype) / s);
      sa_code[g * M + m] = c;
    }
  }
}

void oracle_quantize_weight_block_ue8m0(const uint16_t* w, int dtype, int64_t N, int64_t K,
                                        uint8_t* q, uint8_t* sb_code) {
  int64_t NB = (N + 127) / 128;
  int64_t KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t bi = 0; bi < NB; ++bi) {
    for (int64_t bj = 0; bj < KB; ++bj) {
      int64_t r0 = bi * 128;
      int64_t r1 = r0 + 128 < N ? r0 + 128 : N;
      float amax = 0.0f;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = bj * 128; c < bj * 128 + 128; ++c) {
          float v = fabsf(in_to_float(w[r * K + c], dtype));
          if (v > amax) amax = v;
        }
      uint8_t code = oracle_ue8m0_of_amax(amax);
      float s = oracle_ue8m0_decode(code);
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = bj * 128; c < bj * 128 + 128; ++c)
          q[r * K + c] = oracle_e4m3_encode(in_to_float(w[r * K + c], dtype) / s);
      sb_code[bi * KB + bj] = code;
    }
  }
}

/* ------------------------------------------------------------ O4: GEMM */

static int64_t row_of(const int64_t* rows, int64_t i) { return rows ? rows[i] : i; }

/* dec[b] = oracle_e4m3_decode(b) for all 256 codes (a lookup of O1). */
static void decode_table(double* dec) {
  for (int b = 0; b < 256; ++b) dec[b] = oracle_e4m3_decode((uint8_t)b);
}

/* Per-tensor scaled GEMM [P2 s3 steps 5-6 and pseudocode, R6]:
 *   R[i][n] = (sum_k dec(qa[m][k]) * dec(qb[n][k])) * sa * sb,  m = rows[i].
 * qa: [M][K], qb: [N][K] (weight layout, so C = A * W^T).  R: [nrows][N].
 * rows == NULL means rows 0..nrows-1.  The inner sum is exact in double
 * (every product is a multiple of 2^-18 below 2^17.6, and K <= 2^16). */
void oracle_gemm_per_tensor(const uint8_t* qa, float sa, const uint8_t* qb, float sb,
                            int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                            double* R) {
  double dec[256];
  decode_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = row_of(rows, i);
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += dec[qa[m * K + k]] * dec[qb[n * K + k]];
      R[i * N + n] = acc * (double)sa * (double)sb;
    }
  }
}

/* Per-channel weight scales [R9]:
 *   R[i][n] = (sum_k dec(qa[m][k]) * dec(qb[n][k])) * sa * sb[n],  m = rows[i]. */
void oracle_gemm_per_channel(const uint8_t* qa, float sa, const uint8_t* qb, const float* sb,
                             int64_t N, int64_t K, const int64_t* rows, int64_t nrows, double* R) {
  double dec[256];
  decode_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = row_of(rows, i);
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += dec[qa[m * K + k]] * dec[qb[n * K + k]];
      R[i * N + n] = acc * (double)sa * (double)sb[n];
    }
  }
}

/* Block-scaled GEMM [P5 opening bullets for the block geometry, R6, R7]:
 *   R[i][n] = sum_kb sa[kb][m] * sb[n/128][kb] * (sum_{k in kb} dec*dec).
 * sa: [K/128][M_total], sb: [ceil(N/128)][K/128]. */
void oracle_gemm_block(const uint8_t* qa, const float* sa, int64_t M_total,
                       const uint8_t* qb, const float* sb, int64_t N, int64_t K,
                       const int64_t* rows, int64_t nrows, double* R) {
  int64_t KB = K / 128;
  double dec[256];
  decode_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = row_of(rows, i);
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t kb = 0; kb < KB; ++kb) {
        double part = 0.0;
        for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
          part += dec[qa[m * K + k]] * dec[qb[n * K + k]];
        acc += part * (double)sa[kb * M_total + m] * (double)sb[(n / 128) * KB + kb];
      }
      R[i * N + n] = acc;
    }
  }
}

/* Exact integer cross-check: sum over k in [k0, k1) of units(qa)*units(qb),
 * in units of 2^-18.  |sum| <= 2^36 * K stays far inside int64. */
void oracle_dot_units(const uint8_t* qa, const uint8_t* qb, int64_t M, int64_t N, int64_t K,
                      int64_t k0, int64_t k1, int64_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int64_t acc = 0;
      for (int64_t k = k0; k < k1; ++k)
        acc += oracle_e4m3_units(qa[m * K + k]) * oracle_e4m3_units(qb[n * K + k]);
      out[m * N + n] = acc;
    }
}

/* ---------------------------------------------------- array conveniences */

void oracle_e4m3_decode_array(const uint8_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}

void oracle_e4m3_encode_array(const float* y, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(y[i]);
}

void oracle_to_float_array(const uint16_t* x, int dtype, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = in_to_float(x[i], dtype);
}

/* The quantizer's elementwise step for a given scale: q = E4M3(fl32(x / s)).
 * It is also the whole static / delayed-scaling quantizer [R8], and serves
 * the exhaustive tests over all 16-bit inputs and many scales. */
void oracle_quantize_with_scale(const uint16_t* x, int dtype, int64_t n, float s, uint8_t* q) {
  for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(in_to_float(x[i], dtype) / s);
}

/* Delayed scaling [R8]: the next dequant factor from H recorded amaxes. */
float oracle_scale_from_history(const float* h, int64_t H, int margin) {
  float m = 0.0f;
  for (int64_t i = 0; i < H; ++i)
    if (h[i] > m) m = h[i];
  return ldexpf(scale_of_amax(m), margin);
}

/* Exact max|x| over n 16-bit inputs, as FP32. */
float oracle_amax(const uint16_t* x, int dtype, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = fabsf(in_to_float(x[i], dtype));
    if (v > m) m = v;
  }
  return m;
}

/* Many scales at once: q[j][i] = E4M3(fl32(x[i] / s[j])). */
void oracle_quantize_scales_grid(const uint16_t* x, int dtype, int64_t n, const float* s,
                                 int64_t ns, uint8_t* q) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < ns; ++j)
    for (int64_t i = 0; i < n; ++i)
      q[j * n + i] = oracle_e4m3_encode(in_to_float(x[i], dtype) / s[j]);
}

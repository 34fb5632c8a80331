/*
 * bitlinear_oracle.c -- plain, slow, single-threaded CPU definition of the
 * BitNet b1.58 BitLinear forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker for the
 * CUDA library: it is built and called by the test-suite, by the smoke check
 * and by the CPU-baseline leg of the benchmark, never by the library itself.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * What the method computes (BitLinear, "absmean" ternary weights, 8-bit
 * activations; anthology note-168 on arXiv 2402.17764, section "What it does";
 * yousumm.com transcript of the BitNet b1.58 2B4T video, the "ABS mean
 * quantizer" / "eight-bit numbers" paragraph):
 *
 *   gamma = mean(|W|)                                  (per weight matrix)
 *   W_q   = clip(round(W / (gamma + eps)), -1, +1)     (ternary weights)
 *   s     = 127 / max_k |x[m,k]|                       (per token m)
 *   x_q   = clip(round(x * s), -128, 127)              (int8 activations)
 *   acc   = W_q . x_q   in int32   (the product "only involves integer
 *           addition": anthology note-168, "The part that is a bet rather than
 *           a measurement")
 *   y     = acc * gamma / s
 *
 * Readings taken where the formulas leave a step open (each one is listed in
 * the design notes):
 *   R1  mean(|W|) is the exact real mean of the fp32 values, rounded once to
 *       fp32 with round-half-to-even.  It does not depend on summation order.
 *   R2  gamma + eps is one fp32 addition (RNE); W / (gamma+eps) is one IEEE
 *       fp32 division; round() is round-half-to-even.
 *   R3  packing: four codes per byte (four ternary weights in one byte,
 *       yousumm.com transcript); code = q + 1 in {0,1,2}; weight k of a row
 *       sits in byte k/4 at bits 2*(k%4) (least significant first); rows are
 *       contiguous, K/4 bytes each.  Code 3 is never written.
 *   R4  max|x| is clamped from below at 1e-5 before 127/max|x|, so an
 *       all-zero token gives x_q = 0 and y = 0 instead of inf/NaN.
 *   R5  x * s is one fp32 multiplication (RNE), then round-half-to-even.
 *   R6  dequant is t = fp32(gamma / s[m]) followed by y = fp32(fp32(acc) * t);
 *       fp32(acc) is exact because |acc| <= 127*K < 2^24.
 *   R9  the sub-layer norm ahead of a BitLinear is RMS normalisation with an
 *       optional per-channel gain, applied before the quantisation:
 *       x_n = fp32(fp32(x * g) / fp32(sqrt(fp32(mean(x^2) + eps)))), the
 *       mean of squares exact and rounded once (see the function).
 *   R10 squared ReLU on the output is fp32(max(y,0) * max(y,0)).
 *   R11 base-3 packing: five codes per byte as sum (q+1) * 3^i, least
 *       significant first, rows of ceil(K/5) bytes padded with 121 (zero
 *       codes) to a multiple of 16.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no fast-math (so every float
 * operation is a single IEEE-754 binary32 operation with RNE).  The same
 * source is also built with -fopenmp: the loops over independent outputs
 * (rows of the product, tokens, packed bytes) then run on several host
 * threads.  Every output is still computed by the same sequential code, so
 * both builds give identical results.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* R1: gamma = mean |W|, exact.                                              */
/* ------------------------------------------------------------------------ */

/* A fixed-point accumulator for exact sums of non-negative values.  For the
 * absmean one unit is 2^-149 (the smallest fp32 subnormal), so every finite
 * |w| is an integer number of units below 2^278 and 2^32 of them stay below
 * 2^310.  For the mean of squares (R9) one unit is 2^-298, every finite x^2
 * is below 2^554 units and 2^24 of them below 2^578.  640 bits hold both. */
#define ORC_LIMBS 20 /* 640 bits */

typedef struct {
  uint32_t limb[ORC_LIMBS]; /* little-endian limbs */
} orc_big;

static void orc_big_add_shifted(orc_big* a, uint32_t v, int bit_offset) {
  int li = bit_offset / 32;
  int sh = bit_offset % 32;
  uint64_t part = (uint64_t)v << sh; /* at most 24 + 31 = 55 bits */
  uint64_t carry = 0;
  for (int i = li; i < ORC_LIMBS; ++i) {
    uint64_t add = (i == li) ? (part & 0xffffffffu) : (i == li + 1) ? (part >> 32) : 0;
    uint64_t t = (uint64_t)a->limb[i] + add + carry;
    a->limb[i] = (uint32_t)t;
    carry = t >> 32;
    if (i > li + 1 && carry == 0) break;
  }
}

/* Decompose a finite fp32 magnitude into (integer significand, offset) with
 * |w| = sig * 2^(offset) units of 2^-149.  Returns 0 for non-finite input. */
static int orc_decompose(float w, uint32_t* sig, int* offset) {
  uint32_t u;
  memcpy(&u, &w, 4);
  u &= 0x7fffffffu;
  uint32_t e = u >> 23, f = u & 0x7fffffu;
  if (e == 255) return 0;
  if (e == 0) {
    *sig = f;      /* subnormal: f * 2^-149 */
    *offset = 0;
  } else {
    *sig = f | 0x800000u; /* (1.f) * 2^(e-127) = sig * 2^(e-150) = sig * 2^(e-1) units */
    *offset = (int)e - 1;
  }
  return 1;
}

static int orc_big_highest_bit(const orc_big* a) {
  for (int i = ORC_LIMBS - 1; i >= 0; --i)
    if (a->limb[i]) {
      int b = 31;
      while (!((a->limb[i] >> b) & 1u)) --b;
      return i * 32 + b;
    }
  return -1;
}

static uint32_t orc_big_bit(const orc_big* a, int b) { return (a->limb[b / 32] >> (b % 32)) & 1u; }

/* Round (Q + R/n) units of 2^unit_exp to the nearest fp32, ties to even.
 * The fp32 quantum is 2^(p-23) units for a top set bit p, never finer than
 * the subnormal quantum 2^-149, which is 2^(-149-unit_exp) units. */
static float orc_round_to_f32(const orc_big* Q, uint64_t R, uint64_t n, int unit_exp) {
  const int qmin = -149 - unit_exp; /* subnormal quantum, as a bit index of Q */
  int p = orc_big_highest_bit(Q);
  int ulp = (p - 23 > qmin) ? p - 23 : qmin; /* fp32 quantum, as a power of two in units */
  uint64_t M = 0;                      /* kept significand: bits [ulp, p] of Q */
  for (int b = p; b >= ulp; --b) M = (M << 1) | orc_big_bit(Q, b);
  /* compare the discarded part (bits below ulp, plus R/n) with half a quantum */
  int cmp; /* -1 below half, 0 exactly half, +1 above half */
  if (ulp == 0) {
    /* discarded part is R/n of one unit */
    unsigned __int128 twoR = (unsigned __int128)R * 2u;
    cmp = (twoR > n) ? 1 : (twoR == n ? 0 : -1);
  } else {
    int half_bit = orc_big_bit(Q, ulp - 1);
    int below_nonzero = (R != 0);
    for (int b = 0; b < ulp - 1 && !below_nonzero; ++b) below_nonzero = orc_big_bit(Q, b);
    if (!half_bit) cmp = -1;
    else cmp = below_nonzero ? 1 : 0;
  }
  if (cmp > 0 || (cmp == 0 && (M & 1u))) {
    M += 1;
    if (M == (1u << 24)) {
      M = 1u << 23;
      ulp += 1;
    }
  }
  uint32_t bits;
  if (M >= (1u << 23)) {
    /* value = M * 2^(ulp + unit_exp), M in [2^23, 2^24): biased exponent ulp + unit_exp + 150 */
    int biased = ulp + unit_exp + 150;
    if (biased >= 255) bits = 0x7f800000u;
    else bits = ((uint32_t)biased << 23) | (uint32_t)(M - (1u << 23));
  } else {
    bits = (uint32_t)M; /* subnormal: ulp == qmin, value = M * 2^-149 */
  }
  float out;
  memcpy(&out, &bits, 4);
  return out;
}

/* floor(S / n) into Q and the remainder, most significant limb first. */
static uint64_t orc_big_divide(const orc_big* S, uint64_t n, orc_big* Q) {
  memset(Q, 0, sizeof *Q);
  unsigned __int128 rem = 0;
  for (int i = ORC_LIMBS - 1; i >= 0; --i) {
    unsigned __int128 cur = (rem << 32) | S->limb[i];
    Q->limb[i] = (uint32_t)(cur / n);
    rem = cur % n;
  }
  return (uint64_t)rem;
}

/* gamma = mean(|W|) over n values, exact then rounded once (reading R1).
 * Returns NaN if any value is not finite.  n must be in [1, 2^32]. */
float oracle_absmean(const float* W, uint64_t n) {
  orc_big S;
  memset(&S, 0, sizeof S);
  for (uint64_t i = 0; i < n; ++i) {
    uint32_t sig;
    int off;
    if (!orc_decompose(W[i], &sig, &off)) return NAN;
    if (sig) orc_big_add_shifted(&S, sig, off);
  }
  orc_big Q;
  uint64_t rem = orc_big_divide(&S, n, &Q);
  return orc_round_to_f32(&Q, rem, n, -149);
}

/* ------------------------------------------------------------------------ */
/* R2: absmean ternarisation.                                                */
/* ------------------------------------------------------------------------ */

/* W_q[i] = clip(rint(W[i] / fp32(gamma + eps)), -1, 1). */
void oracle_ternarize(const float* W, uint64_t n, float gamma, float eps, int8_t* q) {
  float d = gamma + eps;
  for (uint64_t i = 0; i < n; ++i) {
    float r = rintf(W[i] / d);
    if (r > 1.0f) r = 1.0f;
    if (r < -1.0f) r = -1.0f;
    q[i] = (int8_t)r; /* -0.0f converts to 0 */
  }
}

/* ------------------------------------------------------------------------ */
/* R3: 2-bit packing, four weights per byte.                                 */
/* ------------------------------------------------------------------------ */

/* n must be a multiple of 4.  Writes n/4 bytes. */
void oracle_pack(const int8_t* q, uint64_t n, uint8_t* packed) {
  for (uint64_t i = 0; i < n / 4; ++i) {
    unsigned byte = 0;
    for (int j = 0; j < 4; ++j) byte |= (unsigned)(q[4 * i + j] + 1) << (2 * j);
    packed[i] = (uint8_t)byte;
  }
}

/* Inverse of oracle_pack.  Returns the number of code-3 fields seen (which
 * oracle_pack never writes); those decode to +2. */
uint64_t oracle_unpack(const uint8_t* packed, uint64_t n, int8_t* q) {
  uint64_t bad = 0;
#pragma omp parallel for reduction(+ : bad) schedule(static)
  for (uint64_t i = 0; i < n; ++i) {
    unsigned code = (packed[i / 4] >> (2 * (i % 4))) & 3u;
    if (code == 3) ++bad;
    q[i] = (int8_t)((int)code - 1);
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* R11: base-3 packing, five weights per byte (1.6 bits per weight).         */
/* The pages put the information in one ternary weight at log2(3) = 1.58    */
/* bits and the weights of the 2B model at about 0.4 GB, under 2 bits per    */
/* weight, without spelling the format out.  Reading: byte j of a row holds  */
/* the digits d_i = q[5j + i] + 1 (i = 0..4, least significant first) as     */
/* sum d_i * 3^i, a value in 0..242; positions at or past K take d = 1       */
/* (q = 0).  A row takes ceil(K / 5) bytes, padded to a multiple of 16 bytes */
/* with 121 (five zero codes).                                               */
/* ------------------------------------------------------------------------ */

int64_t oracle_tq5_row_bytes(int64_t K) {
  const int64_t used = (K + 4) / 5;
  return (used + 15) / 16 * 16;
}

void oracle_pack_tq5(const int8_t* q, int64_t N, int64_t K, uint8_t* out) {
  const int64_t pitch = oracle_tq5_row_bytes(K);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < pitch; ++j) {
      unsigned value = 0, weight = 1;
      for (int i = 0; i < 5; ++i) {
        const int64_t k = 5 * j + i;
        const unsigned digit = k < K ? (unsigned)(q[n * K + k] + 1) : 1u;
        value += digit * weight;
        weight *= 3u;
      }
      out[n * pitch + j] = (uint8_t)value;
    }
  }
}

/* Inverse of oracle_pack_tq5.  Returns the number of bytes above 242 (not a */
/* five-digit base-3 value; decoded as five zero codes) plus the number of   */
/* padding digits that are not zero codes.                                   */
uint64_t oracle_unpack_tq5(const uint8_t* in, int64_t N, int64_t K, int8_t* q) {
  const int64_t pitch = oracle_tq5_row_bytes(K);
  uint64_t bad = 0;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t j = 0; j < pitch; ++j) {
      unsigned value = in[n * pitch + j];
      if (value > 242u) {
        ++bad;
        value = 121u;
      }
      for (int i = 0; i < 5; ++i) {
        const unsigned digit = value % 3u;
        value /= 3u;
        const int64_t k = 5 * j + i;
        if (k < K) q[n * K + k] = (int8_t)((int)digit - 1);
        else if (digit != 1u) ++bad;
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ */
/* R4, R5: per-token absmax int8 activation quantisation.                    */
/* ------------------------------------------------------------------------ */

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
void oracle_bf16_to_f32(const uint16_t* x, uint64_t n, float* out) {
  for (uint64_t i = 0; i < n; ++i) {
    uint32_t u = (uint32_t)x[i] << 16;
    memcpy(&out[i], &u, 4);
  }
}

void oracle_quant_act(const float* X, int64_t M, int64_t K, float clamp_eps, int8_t* x_q, float* s) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float* row = X + m * K;
    float a = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float v = fabsf(row[k]);
      if (v > a) a = v;
    }
    if (a < clamp_eps) a = clamp_eps;
    float sm = 127.0f / a;
    s[m] = sm;
    for (int64_t k = 0; k < K; ++k) {
      float r = rintf(row[k] * sm);
      if (r > 127.0f) r = 127.0f;
      if (r < -128.0f) r = -128.0f;
      x_q[m * K + k] = (int8_t)r;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* R9: sub-layer RMS normalisation ahead of the activation quantisation.     */
/* The transcript says BitNet b1.58 2B4T adds a normalisation inside each    */
/* sub-layer (paragraph after the poker-chip analogy); its formula is not on */
/* the pages.  Reading, per token, in this order:                            */
/*   ms  = mean_k x[k]^2, the exact real mean of the squares of the fp32     */
/*         values, rounded once to fp32 (ties to even), as gamma in R1;      */
/*   r   = fp32 sqrt(fp32(ms + eps))  (IEEE square root), eps > 0;           */
/*   x_n = fp32(fp32(x[k] * g[k]) / r)  (one IEEE multiply, one division),   */
/*         g an optional per-channel gain (1 when absent);                   */
/* then x_n is quantised exactly as any activation row (R4, R5).             */
/* ------------------------------------------------------------------------ */

/* mean_k x[k]^2, exact then rounded once to fp32.  x = sig * 2^off units of
 * 2^-149, so x^2 = sig^2 * 2^(2 off) units of 2^-298; sig^2 < 2^48 is added
 * as two 32-bit halves.  Non-finite input gives NaN. */
float oracle_mean_sq(const float* x, int64_t K) {
  orc_big S;
  memset(&S, 0, sizeof S);
  for (int64_t k = 0; k < K; ++k) {
    uint32_t sig;
    int off;
    if (!orc_decompose(x[k], &sig, &off)) return NAN;
    const uint64_t sq = (uint64_t)sig * (uint64_t)sig;
    if ((uint32_t)sq) orc_big_add_shifted(&S, (uint32_t)sq, 2 * off);
    if ((uint32_t)(sq >> 32)) orc_big_add_shifted(&S, (uint32_t)(sq >> 32), 2 * off + 32);
  }
  orc_big Q;
  uint64_t rem = orc_big_divide(&S, (uint64_t)K, &Q);
  return orc_round_to_f32(&Q, rem, (uint64_t)K, -298);
}

void oracle_rmsnorm_quant_act(const float* X, int64_t M, int64_t K, const float* gain, float eps, float clamp_eps,
                              int8_t* x_q, float* s) {
  float* xn = (float*)malloc((size_t)K * sizeof(float));
  if (!xn) return;
  for (int64_t m = 0; m < M; ++m) {
    const float* row = X + m * K;
    const float ms = oracle_mean_sq(row, K);
    const float v = ms + eps;
    const float r = sqrtf(v);
    for (int64_t k = 0; k < K; ++k) {
      const float t = gain ? row[k] * gain[k] : row[k];
      xn[k] = t / r;
    }
    oracle_quant_act(xn, 1, K, clamp_eps, x_q + m * K, &s[m]);
  }
  free(xn);
}

/* R10: squared ReLU on the BitLinear output, the FFN activation that the    */
/* same transcript paragraph names: y' = fp32(max(y, 0) * max(y, 0)).        */
void oracle_relu2(float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    const float r = y[i] > 0.0f ? y[i] : 0.0f;
    y[i] = r * r;
  }
}

/* ------------------------------------------------------------------------ */
/* Integer product and R6 dequantisation.                                    */
/* ------------------------------------------------------------------------ */

/* acc[m,n] = sum_k q[n,k] * x_q[m,k]; q is [N,K] ternary, x_q is [M,K]. */
void oracle_matmul_int(const int8_t* q, const int8_t* x_q, int64_t M, int64_t N, int64_t K, int32_t* acc) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int64_t sum = 0;
      for (int64_t k = 0; k < K; ++k) sum += (int64_t)q[n * K + k] * (int64_t)x_q[m * K + k];
      acc[m * N + n] = (int32_t)sum;
    }
}

void oracle_dequant(const int32_t* acc, float gamma, const float* s, int64_t M, int64_t N, float* y) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    float t = gamma / s[m];
    for (int64_t n = 0; n < N; ++n) y[m * N + n] = (float)acc[m * N + n] * t;
  }
}

/* The forward pass from packed weights: unpack, integer product, dequant.
 * acc may be NULL.  Returns 0 on success, -1 on allocation failure, and the
 * (positive) count of code-3 fields if the packed weights hold any. */
int64_t oracle_forward(const uint8_t* packed, float gamma, const int8_t* x_q, const float* s, int64_t M, int64_t N,
                       int64_t K, float* y, int32_t* acc) {
  int8_t* q = (int8_t*)malloc((size_t)(N * K));
  int32_t* a = acc ? acc : (int32_t*)malloc((size_t)(M * N) * sizeof(int32_t));
  if (!q || !a) {
    free(q);
    if (!acc) free(a);
    return -1;
  }
  uint64_t bad = oracle_unpack(packed, (uint64_t)(N * K), q);
  oracle_matmul_int(q, x_q, M, N, K, a);
  oracle_dequant(a, gamma, s, M, N, y);
  free(q);
  if (!acc) free(a);
  return (int64_t)bad;
}

/* Host threads the loops above run on: 1 in the plain build. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

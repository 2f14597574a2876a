/*
 * fp4_oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see fp4_oracle.h).
 *
 * Sources, cited by page title and section:
 *   [P1] "perf(cuda): enable hardware NVFP4/MXFP4 conversion on Blackwell
 *        builds" (mlxcel #1934), Problem/Background: e2m1 conversion is
 *        round-to-nearest with satfinite (cvt.rn.satfinite.e2m1x2.f32); the
 *        same quantize template serves MXFP4 and NVFP4.
 *   [P2] "epic: NVIDIA Volta (sm_70) inference acceleration program #1536",
 *        Baseline / Diagnosis item 3: qmv over affine 4-bit group-64 weights.
 *   [P3] "mlx 0.30.7.3 -> 0.30.7.6", hunks qqmm.cpp (quantize_input, the
 *        M=1 route, W stored [N,K] "always transposed"), qqmm_utils.cu
 *        (compute_qqmm_pointers: alpha = amax_x*amax_w/(448*6)^2, beta = 0),
 *        qqmm_utils.h (get_padded_scale_dims / pad_and_swizzle_scales: 128x4
 *        tiles, zero padding, 16-byte aligned start) and quantized.cpp
 *        (fast::Quantize::eval_gpu: NVFP4 optional global scale).
 *   [P4] "mlx: opt-in dense GEMM for nvfp4 prefill ... - #287", the global
 *        scale representation comment: the checkpoint multiplier m versus
 *        MLX's m x 2688 form (Nvfp4MaxProduct = 448*6 = 2688).
 *
 * Readings where the pages are silent are frozen in the comments below; they
 * are the same readings the design document lists.
 */
#include "fp4_oracle.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define E2M1_MAX 6.0
#define E4M3_MAX 448.0
#define NVFP4_MAX_PRODUCT 2688.0f /* 448 * 6, [P4] */

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16                                                                      */
/* ------------------------------------------------------------------------ */

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

double orc_bf16_to_double(uint16_t b) { return (double)bf16_to_float(b); }

/* Round v to the nearest bf16 (8 significant bits, exponent range of fp32),
 * ties to even, overflow to infinity.  Done on the real value directly, so
 * there is exactly one rounding. */
uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  (void)frexp(a, &e);                /* a = m * 2^e, 0.5 <= m < 1 */
  int quantum = e - 8;               /* 8 significant bits */
  if (quantum < -133) quantum = -133; /* bf16 subnormal spacing 2^-133 */
  double n = rint(ldexp(a, -quantum)); /* default rounding mode: nearest-even */
  double r = ldexp(n, quantum);
  if (r >= 0x1p128) return sign | 0x7F80;
  float f = (float)r;                /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

uint16_t orc_bf16_from_float(float v) { return orc_bf16_from_double((double)v); }

/* ------------------------------------------------------------------------ */
/* scalar codecs                                                             */
/* ------------------------------------------------------------------------ */

/* e2m1 by its definition: exponent bias 1, one mantissa bit, exponent 0 is
 * subnormal (0 or 0.5).  Pinned against the eight magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6} and the maximum 6 stated in [P3]/[P4]. */
double orc_e2m1_decode(unsigned code) {
  unsigned e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return (code & 8u) ? -mag : mag;
}

/* Round-to-nearest, ties to the even code, satfinite [P1].  Brute force over
 * the eight magnitudes.  Reading where the pages are silent: the sign bit is
 * copied from v, so -0 and small negatives that round to zero give code 0x8.
 * NaN input is outside the contract. */
unsigned orc_e2m1_encode(float v) {
  double a = fabs((double)v);
  unsigned best = 0;
  if (a >= 6.0) { /* satfinite; also keeps huge |v| out of the distance test */
    best = 7;
  } else {
    double bestd = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
      double d = fabs(a - orc_e2m1_decode(c));
      if (d < bestd || (d == bestd && (c & 1u) == 0)) {
        best = c;
        bestd = d;
      }
    }
  }
  return best | (signbit(v) ? 8u : 0u);
}

/* E4M3 (OCP FP8): bias 7, three mantissa bits, exponent 0 subnormal, S.1111.111
 * is NaN, no infinity, largest finite 448 [P3 qqmm_utils.cu F8E4M3_MAX]. */
double orc_e4m3_decode(unsigned byte) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* Round-to-nearest-even with satfinite: the nearest finite E4M3 value (ties to
 * the even code), so everything above 448 gives 448.  Brute force. */
unsigned orc_e4m3_encode(float v) {
  double a = fabs((double)v);
  unsigned best = 0;
  if (a >= 448.0) { /* satfinite; also keeps huge |v| out of the distance test */
    best = 0x7E;
  } else {
    double bestd = INFINITY;
    for (unsigned c = 0; c <= 0x7E; ++c) {
      double d = fabs(a - orc_e4m3_decode(c));
      if (d < bestd || (d == bestd && (c & 1u) == 0)) {
        best = c;
        bestd = d;
      }
    }
  }
  return best | (signbit(v) ? 0x80u : 0u);
}

/* E8M0: 2^(byte-127); 0xFF is NaN. */
double orc_e8m0_decode(unsigned byte) {
  if ((byte & 0xFFu) == 0xFFu) return NAN;
  return ldexp(1.0, (int)(byte & 0xFFu) - 127);
}

/* ------------------------------------------------------------------------ */
/* global scale and alpha                                                    */
/* ------------------------------------------------------------------------ */

float orc_amax(const uint16_t* x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(bf16_to_float(x[i]));
    if (a > m) m = a;
  }
  return m;
}

/* Global scale in the multiplier form m = amax / 2688, the checkpoint form of
 * [P4]; MLX's form m*2688 is the tensor amax itself. One fp32 division. */
float orc_global_scale(const uint16_t* x, int64_t n) {
  float amax = orc_amax(x, n);
  return amax / NVFP4_MAX_PRODUCT;
}

/* [P3 qqmm_utils.cu compute_qqmm_pointers]: alpha = amax_x*amax_w/(448*6)^2,
 * evaluated as the hunk writes it: the two amaxes multiplied, then multiplied by
 * the fp32 constant 1/(448*6*448*6). */
float orc_alpha_from_amax(float amax_x, float amax_w) {
  const float inv = 1.0f / (448.0f * 6.0f * 448.0f * 6.0f);
  float p = amax_x * amax_w;
  return p * inv;
}

/* ------------------------------------------------------------------------ */
/* quantizers                                                                */
/* ------------------------------------------------------------------------ */

static void put_code(uint32_t* row, int64_t k, unsigned code) {
  row[k / 8] |= (uint32_t)(code & 15u) << (4 * (k % 8));
}

static unsigned get_code(const uint32_t* row, int64_t k) {
  return (row[k / 8] >> (4 * (k % 8))) & 15u;
}

/* NVFP4, one group of 16 (reading of [P1]/[P3]; the exact fp32 op order is
 * not printed on the pages and is frozen here):
 *   b = max|x_i|, p = fl(6*gs), s = (b == 0) ? 0 : fl(b/p), s8 = E4M3(s),
 *   d = fl(s8*gs), r = (d == 0) ? 0 : fl(1/d), q_i = e2m1(fl(x_i*r)).
 * gs = 1 when no global scale is given. */
void orc_nvfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols,
                        const float* global_scale, uint32_t* q, uint8_t* scales) {
  const float gs = global_scale ? *global_scale : 1.0f;
  const int64_t ng = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint32_t* qrow = q + r * (cols / 8);
    memset(qrow, 0, (size_t)(cols / 8) * 4);
    for (int64_t g = 0; g < ng; ++g) {
      float xf[16];
      float b = 0.0f;
      for (int i = 0; i < 16; ++i) {
        xf[i] = bf16_to_float(x[r * cols + g * 16 + i]);
        if (fabsf(xf[i]) > b) b = fabsf(xf[i]);
      }
      float p = 6.0f * gs;
      float s = (b == 0.0f) ? 0.0f : b / p;
      unsigned s8 = orc_e4m3_encode(s);
      float d = (float)orc_e4m3_decode(s8) * gs;
      float rcp = (d == 0.0f) ? 0.0f : 1.0f / d;
      for (int i = 0; i < 16; ++i) put_code(qrow, g * 16 + i, orc_e2m1_encode(xf[i] * rcp));
      scales[r * ng + g] = (uint8_t)s8;
    }
  }
}

/* MXFP4, one group of 32.  The pages name the format but not its scale rule;
 * the reading is the OCP MX v1.0 rule: shared exponent
 * se = clamp(floor(log2(amax)) - 2, -127, 127) (2 = largest exponent of e2m1),
 * byte = se + 127, q_i = e2m1(x_i * 2^-se) (an exact product).  An all-zero
 * group gets byte 0 and sign-only codes. */
void orc_mxfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols,
                        uint32_t* q, uint8_t* scales) {
  const int64_t ng = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint32_t* qrow = q + r * (cols / 8);
    memset(qrow, 0, (size_t)(cols / 8) * 4);
    for (int64_t g = 0; g < ng; ++g) {
      float xf[32];
      float b = 0.0f;
      for (int i = 0; i < 32; ++i) {
        xf[i] = bf16_to_float(x[r * cols + g * 32 + i]);
        if (fabsf(xf[i]) > b) b = fabsf(xf[i]);
      }
      int se;
      if (b == 0.0f) {
        se = -127;
      } else {
        int e;
        (void)frexpf(b, &e); /* b = m*2^e, 0.5 <= m < 1, so floor(log2 b) = e-1 */
        se = (e - 1) - 2;
        if (se < -127) se = -127;
        if (se > 127) se = 127;
      }
      float mul = ldexpf(1.0f, -se);
      for (int i = 0; i < 32; ++i) put_code(qrow, g * 32 + i, orc_e2m1_encode(xf[i] * mul));
      scales[r * ng + g] = (uint8_t)(se + 127);
    }
  }
}

/* ---- stochastic rounding ------------------------------------------------ */
/* The pages name a stochastic-rounding variant of fp_quantize (P1, the
 * USE_SR template parameter of the NVFP4/MXFP4 quantizer, which needs the
 * Blackwell converters) without stating its rule or its random numbers.  The
 * reading implemented here: block scales exactly as for round-to-nearest; each
 * element v = x * mul is rounded to one of the two e2m1 values around |v|
 * (lo <= |v| < hi), up with probability floor(2^24 (|v| - lo) / (hi - lo)) / 2^24,
 * decided by the top 24 bits of one 32-bit random word; |v| >= 6 gives 6; the
 * sign is kept.  The random word of element e (row-major index r*cols + c) is
 * word e % 4 of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC 2011) at the 128-bit counter
 * offset + floor(e / 4) (little-endian 32-bit words) under the key (low, high
 * 32 bits of seed).  Pinned by tests/test_oracle_sr.py. */

/* Philox4x32 with 10 rounds, written from the paper's definition: each round
 * multiplies words 0 and 2 by the two round multipliers (64-bit products split
 * into high and low halves), mixes the high halves with words 3 and 1 and the
 * round key, and bumps the key by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The random word of element e (see the contract above). */
uint32_t orc_sr_word(uint64_t seed, uint64_t offset, uint64_t e) {
  const uint64_t blk = offset + (e >> 2);
  const uint32_t carry = blk < offset ? 1u : 0u;
  const uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), carry, 0u};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[e & 3];
}

/* Stochastic e2m1 rounding of v with random word u (rule above).  The two
 * neighbours come from a scan of the value table; the probability fraction is
 * exact in double. */
unsigned orc_e2m1_encode_sr(float v, uint32_t u) {
  const double a = fabs((double)v);
  unsigned code;
  if (a >= 6.0) {
    code = 7;
  } else {
    unsigned lo = 0;
    for (unsigned c = 0; c < 8; ++c)
      if (orc_e2m1_decode(c) <= a) lo = c;  /* the table is increasing */
    const double vlo = orc_e2m1_decode(lo), vhi = orc_e2m1_decode(lo + 1);
    const double t = floor(ldexp((a - vlo) / (vhi - vlo), 24));
    code = ((double)(u >> 8) < t) ? lo + 1 : lo;
  }
  return code | (signbit(v) ? 8u : 0u);
}

void orc_nvfp4_quantize_sr(const uint16_t* x, int64_t rows, int64_t cols, const float* global_scale,
                           uint64_t seed, uint64_t offset, uint32_t* q, uint8_t* scales) {
  const float gs = global_scale ? *global_scale : 1.0f;
  const int64_t ng = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint32_t* qrow = q + r * (cols / 8);
    memset(qrow, 0, (size_t)(cols / 8) * 4);
    for (int64_t g = 0; g < ng; ++g) {
      float xf[16];
      float b = 0.0f;
      for (int i = 0; i < 16; ++i) {
        xf[i] = bf16_to_float(x[r * cols + g * 16 + i]);
        if (fabsf(xf[i]) > b) b = fabsf(xf[i]);
      }
      float p = 6.0f * gs;
      float s = (b == 0.0f) ? 0.0f : b / p;
      unsigned s8 = orc_e4m3_encode(s);
      float d = (float)orc_e4m3_decode(s8) * gs;
      float rcp = (d == 0.0f) ? 0.0f : 1.0f / d;
      for (int i = 0; i < 16; ++i) {
        const uint64_t e = (uint64_t)(r * cols + g * 16 + i);
        put_code(qrow, g * 16 + i, orc_e2m1_encode_sr(xf[i] * rcp, orc_sr_word(seed, offset, e)));
      }
      scales[r * ng + g] = (uint8_t)s8;
    }
  }
}

void orc_mxfp4_quantize_sr(const uint16_t* x, int64_t rows, int64_t cols, uint64_t seed, uint64_t offset,
                           uint32_t* q, uint8_t* scales) {
  const int64_t ng = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint32_t* qrow = q + r * (cols / 8);
    memset(qrow, 0, (size_t)(cols / 8) * 4);
    for (int64_t g = 0; g < ng; ++g) {
      float xf[32];
      float b = 0.0f;
      for (int i = 0; i < 32; ++i) {
        xf[i] = bf16_to_float(x[r * cols + g * 32 + i]);
        if (fabsf(xf[i]) > b) b = fabsf(xf[i]);
      }
      int se;
      if (b == 0.0f) {
        se = -127;
      } else {
        int e;
        (void)frexpf(b, &e);
        se = (e - 1) - 2;
        if (se < -127) se = -127;
        if (se > 127) se = 127;
      }
      float mul = ldexpf(1.0f, -se);
      for (int i = 0; i < 32; ++i) {
        const uint64_t el = (uint64_t)(r * cols + g * 32 + i);
        put_code(qrow, g * 32 + i, orc_e2m1_encode_sr(xf[i] * mul, orc_sr_word(seed, offset, el)));
      }
      scales[r * ng + g] = (uint8_t)(se + 127);
    }
  }
}

/* Affine 4-bit (test-data generator only; the pages give no rule):
 * per group lo = min, hi = max, scale = bf16(fl((hi-lo)/15)), bias = bf16(lo),
 * q = clamp(rint((w - bias)/scale), 0, 15), q = 0 when scale is 0. */
void orc_affine_quantize(const uint16_t* w, int64_t rows, int64_t cols, int group,
                         uint32_t* q, uint16_t* scales, uint16_t* biases) {
  const int64_t ng = cols / group;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    uint32_t* qrow = q + r * (cols / 8);
    memset(qrow, 0, (size_t)(cols / 8) * 4);
    for (int64_t g = 0; g < ng; ++g) {
      const uint16_t* src = w + r * cols + g * group;
      float lo = bf16_to_float(src[0]), hi = lo;
      for (int i = 1; i < group; ++i) {
        float v = bf16_to_float(src[i]);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      uint16_t sb = orc_bf16_from_float((hi - lo) / 15.0f);
      uint16_t bb = orc_bf16_from_float(lo);
      double s = orc_bf16_to_double(sb), bias = orc_bf16_to_double(bb);
      for (int i = 0; i < group; ++i) {
        double v = orc_bf16_to_double(src[i]);
        double qq = (s == 0.0) ? 0.0 : rint((v - bias) / s);
        if (qq < 0) qq = 0;
        if (qq > 15) qq = 15;
        put_code(qrow, g * group + i, (unsigned)qq);
      }
      scales[r * ng + g] = sb;
      biases[r * ng + g] = bb;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* scale tiles [P3 qqmm_utils.h]: rows padded to a multiple of 128, columns to */
/* a multiple of 4, padding bytes zero.  Inside a 128x4 tile (512 bytes) the    */
/* public cuBLAS block-scaling-factor layout the hunk points to puts (r, c) at  */
/* (r%32)*16 + (r/32)*4 + c; tiles are ordered row-tile major.                  */
/* ------------------------------------------------------------------------ */

int64_t orc_padded_rows(int64_t rows) { return ((rows + 127) / 128) * 128; }
int64_t orc_padded_cols(int64_t cols) { return ((cols + 3) / 4) * 4; }

int64_t orc_tiled_offset(int64_t r, int64_t c, int64_t padded_cols) {
  int64_t tile = (r / 128) * (padded_cols / 4) + c / 4;
  int64_t rr = r % 128;
  return tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
}

void orc_tile_scales(const uint8_t* linear, int64_t rows, int64_t cols, uint8_t* tiled) {
  int64_t rp = orc_padded_rows(rows), cp = orc_padded_cols(cols);
  memset(tiled, 0, (size_t)(rp * cp));
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) tiled[orc_tiled_offset(r, c, cp)] = linear[r * cols + c];
}

void orc_untile_scales(const uint8_t* tiled, int64_t rows, int64_t cols, uint8_t* linear) {
  int64_t cp = orc_padded_cols(cols);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) linear[r * cols + c] = tiled[orc_tiled_offset(r, c, cp)];
}

/* ------------------------------------------------------------------------ */
/* dequantize                                                                */
/* ------------------------------------------------------------------------ */

/* Exact value of element (r, k) in fp64.  NVFP4: code*E4M3(s)*gs; MXFP4:
 * code*2^(byte-127); affine: q*s + b.  Each is exact in fp64. */
static double deq_exact(const uint32_t* q, const void* scales, const uint16_t* biases,
                        int64_t r, int64_t k, int64_t cols, int mode, int group, double gs) {
  unsigned c = get_code(q + r * (cols / 8), k);
  int64_t si = r * (cols / group) + k / group;
  if (mode == 2) return orc_e2m1_decode(c) * orc_e4m3_decode(((const uint8_t*)scales)[si]) * gs;
  if (mode == 1) return orc_e2m1_decode(c) * orc_e8m0_decode(((const uint8_t*)scales)[si]);
  return (double)c * orc_bf16_to_double(((const uint16_t*)scales)[si]) +
         orc_bf16_to_double(biases[si]);
}

void orc_dequantize_f64(const uint32_t* q, const void* scales, const uint16_t* biases,
                        int64_t rows, int64_t cols, int mode, int group,
                        const float* global_scale, double* out) {
  double gs = global_scale ? (double)*global_scale : 1.0;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < cols; ++k)
      out[r * cols + k] = deq_exact(q, scales, biases, r, k, cols, mode, group, gs);
}

/* Output of the dequantize operation [P3 quantized.cpp fp_dequantize /
 * affine_dequantize]: the fp32 value, then RNE to bf16.  Reading: NVFP4 is
 * fl(fl(code*s8)*gs) (code*s8 is exact), MXFP4 fl(code*2^e) (exact unless it
 * overflows), affine fl(fl(q*s) + b) (q*s is exact). */
void orc_dequantize_bf16(const uint32_t* q, const void* scales, const uint16_t* biases,
                         int64_t rows, int64_t cols, int mode, int group,
                         const float* global_scale, uint16_t* out) {
  const float gs = global_scale ? *global_scale : 1.0f;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t k = 0; k < cols; ++k) {
      unsigned c = get_code(q + r * (cols / 8), k);
      int64_t si = r * (cols / group) + k / group;
      float v;
      if (mode == 2) {
        float cs = (float)orc_e2m1_decode(c) * (float)orc_e4m3_decode(((const uint8_t*)scales)[si]);
        v = cs * gs;
      } else if (mode == 1) {
        v = (float)orc_e2m1_decode(c) * (float)orc_e8m0_decode(((const uint8_t*)scales)[si]);
      } else {
        float qs = (float)c * bf16_to_float(((const uint16_t*)scales)[si]);
        v = qs + bf16_to_float(biases[si]);
      }
      out[r * cols + k] = orc_bf16_from_float(v);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* matmuls                                                                   */
/* ------------------------------------------------------------------------ */

/* qmv [P2 Diagnosis 3, P3 qqmm.cpp M=1 route]: y = x . deq(W)^T with W stored
 * [N, K]; accumulation in fp64; NVFP4 includes the weight global scale. */
void orc_qmv(const uint16_t* x, const uint32_t* w, const void* scales, const uint16_t* biases,
             const float* global_scale_w, int64_t N, int64_t K, int mode, int group,
             const int64_t* rows, int64_t nrows, double* y) {
  double gs = global_scale_w ? (double)*global_scale_w : 1.0;
  int64_t n_out = rows ? nrows : N;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < n_out; ++i) {
    int64_t n = rows ? rows[i] : i;
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
      acc += orc_bf16_to_double(x[k]) * deq_exact(w, scales, biases, n, k, K, mode, group, gs);
    y[i] = acc;
  }
}

/* qqmm [P3 qqmm.cpp / qqmm_utils.cu]: out = alpha * (Xq . Wq^T) over code*block
 * scale values (global scales live in alpha), W stored [N, K], beta = 0. */
void orc_qqmm(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
              float alpha, int64_t M, int64_t N, int64_t K, int mode,
              const int64_t* mrows, int64_t nm, const int64_t* ncols, int64_t nn, double* out) {
  const int group = (mode == 1) ? 32 : 16;
  int64_t om = mrows ? nm : M, on = ncols ? nn : N;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < om; ++i) {
    int64_t m = mrows ? mrows[i] : i;
    for (int64_t j = 0; j < on; ++j) {
      int64_t n = ncols ? ncols[j] : j;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += deq_exact(xq, sx, NULL, m, k, K, mode, group, 1.0) *
               deq_exact(wq, sw, NULL, n, k, K, mode, group, 1.0);
      out[i * on + j] = (double)alpha * acc;
    }
  }
}

/* qmm, the dense W4A16 GEMM ["mlx: opt-in dense GEMM for nvfp4 prefill ..." and
 * qmm_sm80 in "perf(cuda): enable hardware NVFP4/MXFP4 conversion on Blackwell
 * builds"]: out[i, n] = sum_k x[m_i, k] * deq(W)[n, k] in fp64 over the listed
 * rows m_i of x (NULL means all M rows), every column n; deq includes the NVFP4
 * weight global scale.  x is [M, K] bf16, W [N, K] packed. */
void orc_qmm(const uint16_t* x, int64_t M, const uint32_t* w, const void* scales, const uint16_t* biases,
             const float* global_scale_w, int64_t N, int64_t K, int mode, int group,
             const int64_t* rows, int64_t nrows, double* out) {
  const double gs = global_scale_w ? (double)*global_scale_w : 1.0;
  const int64_t om = rows ? nrows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < om; ++i) {
    const uint16_t* xr = x + (rows ? rows[i] : i) * K;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += orc_bf16_to_double(xr[k]) * deq_exact(w, scales, biases, n, k, K, mode, group, gs);
      out[i * N + n] = acc;
    }
  }
}

/* gather_qmm [P2 Diagnosis 1 and 5: gather_gemm / grouped GEMM for MoE]: each
 * routed row r multiplies activation row lhs[r] by expert rhs[r]'s weights. */
void orc_gather_qmm(const uint16_t* x, const int32_t* lhs, const int32_t* rhs, int64_t R,
                    const uint32_t* w, const void* scales, const uint16_t* biases,
                    int64_t E, int64_t N, int64_t K, int mode, int group,
                    const int64_t* rows, int64_t nrows, double* out) {
  (void)E;
  int64_t on = rows ? nrows : R;
  const int64_t wq_per_expert = N * (K / 8);
  const int64_t s_per_expert = N * (K / group);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < on; ++i) {
    int64_t r = rows ? rows[i] : i;
    const uint16_t* xr = x + (int64_t)lhs[r] * K;
    int64_t e = rhs[r];
    const uint32_t* we = w + e * wq_per_expert;
    const void* se = (mode == 0) ? (const void*)((const uint16_t*)scales + e * s_per_expert)
                                 : (const void*)((const uint8_t*)scales + e * s_per_expert);
    const uint16_t* be = biases ? biases + e * s_per_expert : NULL;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += orc_bf16_to_double(xr[k]) * deq_exact(we, se, be, n, k, K, mode, group, 1.0);
      out[i * N + n] = acc;
    }
  }
}

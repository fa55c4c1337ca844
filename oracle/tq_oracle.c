/*
 * tq_oracle.c -- plain CPU oracle for the ternary FWHT-128 linear layers.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
 * baseline leg of the benchmark; never by the product path.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Every function is the literal definition, one element at a time, in the
 * order the pages give.  Build with -O2 -ffp-contract=off so that no
 * multiply-add is fused behind our back (the fp32 results are compared bit
 * for bit).  Page names are explained in tq_oracle.h.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* ---------------------------------------------------------------- Hadamard */

/* [dpshk] sec. 2.1: entry (i, j) is -1 to the number of common set bits. */
int tqo_hadamard_entry(int i, int j) {
  unsigned v = (unsigned)(i & j);
  int ones = 0;
  while (v) { ones += (int)(v & 1u); v >>= 1; }
  return (ones & 1) ? -1 : 1;
}

/* [dpshk] sec. 2.1 / [mhpq] sec. 2.2: H_2n = [[H_n, H_n], [H_n, -H_n]]. */
void tqo_sylvester(int n, int8_t *h) {
  h[0] = 1;
  for (int m = 1; m < n; m *= 2) {
    /* h currently holds H_m in its top-left m x m corner (row stride n). */
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < m; ++j) {
        int8_t v = h[i * n + j];
        h[i * n + (j + m)] = v;
        h[(i + m) * n + j] = v;
        h[(i + m) * n + (j + m)] = (int8_t)(-v);
      }
  }
}

/* The normalisation 1/sqrt(n) for n = 128 ([dpshk] sec. 2.3; [zwxr] sec. 2.1,
 * normalised transform), rounded once to fp32. */
uint32_t tqo_norm_const_bits(void) {
  float c = (float)(1.0 / sqrt(128.0));
  return f32_to_bits(c);
}

/* [xxqk] sec. 2: log2(n) rounds of (a + b, a - b); the round with pair
 * distance h = 1 comes first and h = 64 last. */
void tqo_fwht128_f32(const float *in, float *out) {
  float v[128];
  for (int i = 0; i < 128; ++i) v[i] = in[i];
  for (int h = 1; h < 128; h *= 2) {
    for (int i = 0; i < 128; ++i) {
      if ((i & h) == 0) {
        float a = v[i];
        float b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
  float c = bits_to_f32(tqo_norm_const_bits());
  for (int i = 0; i < 128; ++i) out[i] = v[i] * c;
}

/* Dense matrix-vector form of the same rotation in fp64. */
void tqo_fwht128_f64(const double *in, double *out) {
  double tmp[128];
  double c = 1.0 / sqrt(128.0);
  for (int i = 0; i < 128; ++i) {
    double acc = 0.0;
    for (int j = 0; j < 128; ++j) acc += (double)tqo_hadamard_entry(i, j) * in[j];
    tmp[i] = acc * c;
  }
  for (int i = 0; i < 128; ++i) out[i] = tmp[i];
}

/* ------------------------------------------------------------ fp16 / bf16 */

/* IEEE 754 binary32 -> binary16, round to nearest, ties to even. */
uint16_t tqo_f32_to_f16(float f) {
  uint32_t x = f32_to_bits(f);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t bexp = (x >> 23) & 0xffu;
  uint32_t frac = x & 0x7fffffu;
  if (bexp == 0xffu) return (uint16_t)(sign | (frac ? 0x7e00u : 0x7c00u));
  if (bexp == 0) return sign; /* fp32 subnormals are far below half of 2^-24 */
  int e = (int)bexp - 127;    /* value = m * 2^(e - 23), m has 24 bits */
  uint32_t m = frac | 0x800000u;
  if (e >= -14) {
    /* normal binary16: keep 11 significant bits */
    uint32_t q = m >> 13, rem = m & 0x1fffu, half = 0x1000u;
    if (rem > half || (rem == half && (q & 1u))) q += 1;
    if (q == 0x800u) { q = 0x400u; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint32_t)((e + 15) << 10) | (q & 0x3ffu));
  }
  /* subnormal binary16: value in units of 2^-24 is m * 2^(e + 1) */
  int s = -(e + 1);
  if (s > 25) return sign;
  uint32_t q = m >> s, rem = m & ((1u << s) - 1u), half = 1u << (s - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  return (uint16_t)(sign | q); /* q == 0x400 becomes the smallest normal */
}

float tqo_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1fu;
  uint32_t frac = h & 0x3ffu;
  if (e == 0x1fu) return bits_to_f32(sign | 0x7f800000u | (frac << 13));
  if (e == 0) {
    /* zero or subnormal: frac * 2^-24, exact in fp32 */
    float v = (float)frac * 5.9604644775390625e-08f;
    return sign ? -v : v;
  }
  return bits_to_f32(sign | ((e - 15 + 127) << 23) | (frac << 13));
}

float tqo_bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------ quantiser */

/* [mhpq] sec. 1.1: scale = group mean of |w|; divide; round; clip to
 * {-1, 0, 1}.  [mhpq] sec. 1.3: one fp16 scale per 128 weights. */
uint16_t tqo_quantize_group(const float *wrot, int8_t *t) {
  float s[128];
  for (int i = 0; i < 128; ++i) s[i] = fabsf(wrot[i]);
  for (int h = 64; h >= 1; h /= 2)
    for (int i = 0; i < h; ++i) s[i] = s[i] + s[i + h];
  float mean = s[0] * 0.0078125f; /* * 2^-7 */
  uint16_t sbits = tqo_f32_to_f16(mean);
  float sc = tqo_f16_to_f32(sbits);
  for (int i = 0; i < 128; ++i) {
    if (sc == 0.0f) { t[i] = 0; continue; }
    float q = wrot[i] / sc;
    float r = nearbyintf(q); /* default rounding mode: ties to even */
    t[i] = (int8_t)(r > 1.0f ? 1 : (r < -1.0f ? -1 : (int)r));
  }
  return sbits;
}

static void load_group(const void *W, int wt, int64_t row, int64_t ldw, int64_t k0, float *dst) {
  if (wt == 0) {
    const float *w = (const float *)W + row * ldw + k0;
    for (int i = 0; i < 128; ++i) dst[i] = w[i];
  } else {
    const uint16_t *w = (const uint16_t *)W + row * ldw + k0;
    for (int i = 0; i < 128; ++i) dst[i] = tqo_bf16_to_f32(w[i]);
  }
}

void tqo_quantize_rows(const void *W, int wt, int64_t K, int64_t ldw,
                       const int64_t *rows, int64_t nrows, int8_t *T, uint16_t *S) {
  int64_t G = K / 128;
  float grp[128], rot[128];
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t n = rows ? rows[r] : r;
    for (int64_t g = 0; g < G; ++g) {
      load_group(W, wt, n, ldw, g * 128, grp);
      tqo_fwht128_f32(grp, rot);
      S[r * G + g] = tqo_quantize_group(rot, T + r * K + g * 128);
    }
  }
}

void tqo_quantize_matrix(const void *W, int wt, int64_t N, int64_t K, int64_t ldw,
                         int8_t *T, uint16_t *S) {
  tqo_quantize_rows(W, wt, K, ldw, 0, N, T, S);
}

/* ------------------------------------------------------------ packing */

/* [mhpq] sec. 3.1: two bits per weight, aligned and quick to decode. */
void tqo_pack2(const int8_t *T, int64_t N, int64_t K, uint8_t *codes, int64_t ld2) {
  for (int64_t n = 0; n < N; ++n) {
    uint8_t *row = codes + n * ld2;
    for (int64_t j = 0; j < ld2; ++j) row[j] = 0;
    for (int64_t k = 0; k < K; ++k) {
      unsigned code = (unsigned)(T[n * K + k] + 1);
      row[k / 4] = (uint8_t)(row[k / 4] | (code << (2 * (k % 4))));
    }
  }
}

void tqo_unpack2(const uint8_t *codes, int64_t ld2, int64_t N, int64_t K, int8_t *T) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      unsigned code = (codes[n * ld2 + k / 4] >> (2 * (k % 4))) & 3u;
      T[n * K + k] = (int8_t)((int)code - 1);
    }
}

int64_t tqo_ld3(int64_t K) {
  int64_t nb = (K + 4) / 5;
  return (nb + 15) / 16 * 16;
}

/* five base-3 digits per byte (3^5 = 243 <= 256), lowest K first */
void tqo_pack3(const int8_t *T, int64_t N, int64_t K, uint8_t *codes, int64_t ld3) {
  int64_t nb = (K + 4) / 5;
  for (int64_t n = 0; n < N; ++n) {
    uint8_t *row = codes + n * ld3;
    for (int64_t j = 0; j < ld3; ++j) row[j] = 0;
    for (int64_t j = 0; j < nb; ++j) {
      unsigned v = 0, p = 1;
      for (int i = 0; i < 5; ++i) {
        int64_t k = 5 * j + i;
        unsigned d = (k < K) ? (unsigned)(T[n * K + k] + 1) : 1u;
        v += d * p;
        p *= 3;
      }
      row[j] = (uint8_t)v;
    }
  }
}

void tqo_unpack3(const uint8_t *codes, int64_t ld3, int64_t N, int64_t K, int8_t *T) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      unsigned v = codes[n * ld3 + k / 5];
      for (int i = 0; i < (int)(k % 5); ++i) v /= 3;
      T[n * K + k] = (int8_t)((int)(v % 3) - 1);
    }
}

/* ------------------------------------------------------------ GEMV */

/* y = sum over groups of scale * (sum of t * x'), in fp64, where x' is the
 * activation rotated by the same block transform ([mhpq] sec. 2.3, rotation
 * absorbed on the activation side; [zwxr] activation-side Hadamard). */
void tqo_gemv_f64(const int8_t *T, const uint16_t *S, int64_t N, int64_t K,
                  const float *x, int64_t M, const int64_t *rows, int64_t nrows,
                  double *y) {
  int64_t G = K / 128;
  int64_t nout = rows ? nrows : N;
  double blk[128], rot[128];
  (void)N;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t r = 0; r < nout; ++r) y[m * nout + r] = 0.0;
    for (int64_t g = 0; g < G; ++g) {
      for (int i = 0; i < 128; ++i) blk[i] = (double)x[m * K + g * 128 + i];
      tqo_fwht128_f64(blk, rot);
      for (int64_t r = 0; r < nout; ++r) {
        const int8_t *t = T + r * K + g * 128;
        double part = 0.0;
        for (int i = 0; i < 128; ++i) part += (double)t[i] * rot[i];
        y[m * nout + r] += (double)tqo_f16_to_f32(S[r * G + g]) * part;
      }
    }
  }
}

/* ------------------------------------------- transform and group variants */

/* The block transform at sizes other than 128 (dpshk sec. 2.1 builds H for
 * any power of two; xxqk sec. 2.1/2.2 weigh block sizes against caches).
 * n-point staged butterflies in fp32, h = 1, 2, ..., n/2, then one multiply
 * by RN_fp32(1/sqrt(n)); n in {64, 128, 256}.  in and out may alias. */
uint32_t tqo_norm_const_bits_n(int n) {
  float c = (float)(1.0 / sqrt((double)n));
  return f32_to_bits(c);
}

void tqo_fwht_f32(int n, const float *in, float *out) {
  float v[256];
  for (int i = 0; i < n; ++i) v[i] = in[i];
  for (int h = 1; h < n; h *= 2) {
    for (int i = 0; i < n; ++i) {
      if ((i & h) == 0) {
        float a = v[i];
        float b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
  float c = bits_to_f32(tqo_norm_const_bits_n(n));
  for (int i = 0; i < n; ++i) out[i] = v[i] * c;
}

/* Dense fp64 form: out[i] = sum_j H[i][j] in[j] / sqrt(n). */
void tqo_fwht_f64(int n, const double *in, double *out) {
  double tmp[256];
  double c = 1.0 / sqrt((double)n);
  for (int i = 0; i < n; ++i) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += (double)tqo_hadamard_entry(i, j) * in[j];
    tmp[i] = acc * c;
  }
  for (int i = 0; i < n; ++i) out[i] = tmp[i];
}

/* absmean over a group of g in {128, 256} weights (mhpq sec. 1.4 tries group
 * 256: 16/256 = 0.0625 bit of scale per weight): halving tree s[i] += s[i+h]
 * for h = g/2 .. 1 in fp32, mean = sum * 2^-log2(g) (exact), fp16 RN scale,
 * IEEE division by the stored scale, round half to even, clamp; t = 0 when
 * the scale is 0. */
uint16_t tqo_quantize_group_n(int g, const float *wrot, int8_t *t) {
  float s[256] = {0.0f};
  for (int i = 0; i < g; ++i) s[i] = fabsf(wrot[i]);
  for (int h = g / 2; h >= 1; h /= 2)
    for (int i = 0; i < h; ++i) s[i] = s[i] + s[i + h];
  float inv = 1.0f / (float)g; /* 2^-7 or 2^-8, exact */
  float mean = s[0] * inv;
  uint16_t sbits = tqo_f32_to_f16(mean);
  float sc = tqo_f16_to_f32(sbits);
  for (int i = 0; i < g; ++i) {
    if (sc == 0.0f) { t[i] = 0; continue; }
    float q = wrot[i] / sc;
    float r = nearbyintf(q);
    t[i] = (int8_t)(r > 1.0f ? 1 : (r < -1.0f ? -1 : (int)r));
  }
  return sbits;
}

/* Quantise rows under a layout: FWHT block size `block` in {64, 128, 256},
 * scale group `group` in {128, 256}, and, when `residual` is set, the
 * residual two-pass form (xxqk sec. 3, residual calibrator: the difference
 * between the rotated weight and its ternary approximation is rotated once
 * more by the same block transform and ternarised with its own scale).
 *
 * Per row, in units of u = max(block, group) consecutive weights:
 *   w'  = FWHT_block of every block of the unit (fp32, as tqo_fwht_f32);
 *   s1, t1 per group of w' (tqo_quantize_group_n);
 *   residual: r = w' - s1 t1 (fp32; a zero trit dequantises to 0 whatever
 *   the scale), r' = FWHT_block of every block of r, s2, t2 per group of r'.
 * T is [nrows][Keff], Keff = K (2 K with residual): t1 in columns 0 .. K-1,
 * t2 in columns K .. 2K-1.  S is [nrows][Geff], Geff = K / group (twice that
 * with residual): the s1 first, then the s2. */
void tqo_quantize_layout_rows(const void *W, int wt, int64_t K, int64_t ldw, const int64_t *rows,
                              int64_t nrows, int block, int group, int residual, int8_t *T,
                              uint16_t *S) {
  int u = block > group ? block : group;
  int64_t G = K / group;
  int64_t Keff = residual ? 2 * K : K, Geff = residual ? 2 * G : G;
  float w[256], wr[256], r[256], rr[256];
  int8_t t1[256], t2[256];
  for (int64_t q = 0; q < nrows; ++q) {
    int64_t n = rows ? rows[q] : q;
    for (int64_t k0 = 0; k0 < K; k0 += u) {
      for (int i = 0; i < u; ++i) {
        if (wt == 0)
          w[i] = ((const float *)W)[n * ldw + k0 + i];
        else
          w[i] = tqo_bf16_to_f32(((const uint16_t *)W)[n * ldw + k0 + i]);
      }
      for (int b = 0; b < u; b += block) tqo_fwht_f32(block, w + b, wr + b);
      for (int g = 0; g < u; g += group) {
        uint16_t s1 = tqo_quantize_group_n(group, wr + g, t1 + g);
        S[q * Geff + (k0 + g) / group] = s1;
        float s1f = tqo_f16_to_f32(s1);
        for (int i = 0; i < group; ++i)
          r[g + i] = (t1[g + i] == 0) ? wr[g + i] : wr[g + i] - s1f * (float)t1[g + i];
      }
      for (int i = 0; i < u; ++i) T[q * Keff + k0 + i] = t1[i];
      if (!residual) continue;
      for (int b = 0; b < u; b += block) tqo_fwht_f32(block, r + b, rr + b);
      for (int g = 0; g < u; g += group)
        S[q * Geff + G + (k0 + g) / group] = tqo_quantize_group_n(group, rr + g, t2 + g);
      for (int i = 0; i < u; ++i) T[q * Keff + K + k0 + i] = t2[i];
    }
  }
}

/* y under a layout, fp64: the first pass meets x' = FWHT_block(x) (dense
 * fp64 form), the residual pass meets x'' = FWHT_block(x') -- the residual's
 * second rotation moved onto the activations (H is symmetric and, normalised,
 * its own inverse).  T [nrows][Keff], S [nrows][Geff] as produced above. */
void tqo_gemv_layout_f64(const int8_t *T, const uint16_t *S, int64_t K, const float *x, int64_t M,
                         int64_t nrows, int block, int group, int residual, double *y) {
  int64_t G = K / group;
  int64_t Keff = residual ? 2 * K : K, Geff = residual ? 2 * G : G;
  double *xr = (double *)malloc((size_t)K * sizeof(double));
  double *xrr = (double *)malloc((size_t)K * sizeof(double));
  double blk[256];
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t k0 = 0; k0 < K; k0 += block) {
      for (int i = 0; i < block; ++i) blk[i] = (double)x[m * K + k0 + i];
      tqo_fwht_f64(block, blk, xr + k0);
      tqo_fwht_f64(block, xr + k0, xrr + k0);
    }
    for (int64_t q = 0; q < nrows; ++q) {
      double acc = 0.0;
      for (int pass = 0; pass < (residual ? 2 : 1); ++pass) {
        const double *xa = pass == 0 ? xr : xrr;
        for (int64_t g = 0; g < G; ++g) {
          const int8_t *t = T + q * Keff + pass * K + g * group;
          double part = 0.0;
          for (int i = 0; i < group; ++i) part += (double)t[i] * xa[g * group + i];
          acc += (double)tqo_f16_to_f32(S[q * Geff + pass * G + g]) * part;
        }
      }
      y[m * nrows + q] = acc;
    }
  }
  free(xr);
  free(xrr);
}

/* ------------------------------------------------------------ 2:4 sparse */

/* kept positions (i0, i1) of pattern p, in the order (0,1) (0,2) (0,3)
 * (1,2) (1,3) (2,3) */
static const int kPat24[6][2] = {{0, 1}, {0, 2}, {0, 3}, {1, 2}, {1, 3}, {2, 3}};

/* [mhpq] sec. 1.2 (structured 2:4 sparsity, then ternarisation of what is
 * kept) with the absmean rule of sec. 1.1 on the kept weights. */
uint16_t tqo_quantize_group_24(const float *wrot, int8_t *t, uint8_t *keep) {
  float kept[64];
  int nk = 0;
  for (int j = 0; j < 32; ++j) {
    /* the two largest magnitudes of the quad; a tie goes to the lower index:
     * position i is kept when fewer than two others beat it */
    for (int i = 0; i < 4; ++i) {
      float a = fabsf(wrot[4 * j + i]);
      int beaten = 0;
      for (int o = 0; o < 4; ++o) {
        if (o == i) continue;
        float b = fabsf(wrot[4 * j + o]);
        if (b > a || (b == a && o < i)) ++beaten;
      }
      keep[4 * j + i] = (uint8_t)(beaten < 2);
      if (beaten < 2) kept[nk++] = fabsf(wrot[4 * j + i]);
    }
  }
  /* nk == 64: each quad keeps exactly two (a strict total order) */
  for (int h = 32; h >= 1; h /= 2)
    for (int i = 0; i < h; ++i) kept[i] = kept[i] + kept[i + h];
  float mean = kept[0] * 0.015625f; /* * 2^-6 */
  uint16_t sbits = tqo_f32_to_f16(mean);
  float sc = tqo_f16_to_f32(sbits);
  for (int i = 0; i < 128; ++i) {
    if (!keep[i] || sc == 0.0f) { t[i] = 0; continue; }
    float q = wrot[i] / sc;
    float r = nearbyintf(q);
    t[i] = (int8_t)(r > 1.0f ? 1 : (r < -1.0f ? -1 : (int)r));
  }
  return sbits;
}

void tqo_quantize_rows_24(const void *W, int wt, int64_t K, int64_t ldw, const int64_t *rows,
                          int64_t nrows, int8_t *T, uint8_t *KEEP, uint16_t *S) {
  int64_t G = K / 128;
  float grp[128], rot[128];
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t n = rows ? rows[r] : r;
    for (int64_t g = 0; g < G; ++g) {
      load_group(W, wt, n, ldw, g * 128, grp);
      tqo_fwht128_f32(grp, rot);
      S[r * G + g] = tqo_quantize_group_24(rot, T + r * K + g * 128, KEEP + r * K + g * 128);
    }
  }
}

int64_t tqo_ld24(int64_t K) { return K / 128 * 24; }

void tqo_pack24(const int8_t *T, const uint8_t *KEEP, int64_t N, int64_t K, uint8_t *codes,
                int64_t ld) {
  int64_t G = K / 128;
  for (int64_t n = 0; n < N; ++n) {
    uint8_t *row = codes + n * ld;
    for (int64_t b = 0; b < ld; ++b) row[b] = 0;
    for (int64_t g = 0; g < G; ++g) {
      uint8_t *grp = row + 24 * g;
      for (int j = 0; j < 32; ++j) {
        const int8_t *t = T + n * K + 128 * g + 4 * j;
        const uint8_t *kp = KEEP + n * K + 128 * g + 4 * j;
        int p = -1;
        for (int q = 0; q < 6; ++q)
          if (kp[kPat24[q][0]] && kp[kPat24[q][1]] &&
              kp[0] + kp[1] + kp[2] + kp[3] == 2)
            p = q;
        if (p < 0) p = 0; /* not a 2:4 quad: cannot be stored (callers pass valid masks) */
        unsigned c = (unsigned)(9 * p + 3 * (t[kPat24[p][0]] + 1) + (t[kPat24[p][1]] + 1));
        grp[j / 2] = (uint8_t)(grp[j / 2] | ((c & 15u) << (4 * (j % 2))));
        grp[16 + j / 4] = (uint8_t)(grp[16 + j / 4] | ((c >> 4) << (2 * (j % 4))));
      }
    }
  }
}

int64_t tqo_unpack24(const uint8_t *codes, int64_t ld, int64_t N, int64_t K, int8_t *T,
                     uint8_t *KEEP) {
  int64_t G = K / 128, bad = 0;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      const uint8_t *grp = codes + n * ld + 24 * g;
      for (int j = 0; j < 32; ++j) {
        unsigned c = ((grp[j / 2] >> (4 * (j % 2))) & 15u) | (((grp[16 + j / 4] >> (2 * (j % 4))) & 3u) << 4);
        int8_t *t = T + n * K + 128 * g + 4 * j;
        uint8_t *kp = KEEP + n * K + 128 * g + 4 * j;
        for (int i = 0; i < 4; ++i) { t[i] = 0; kp[i] = 0; }
        if (c >= 54) { ++bad; continue; }
        int p = (int)(c / 9), v = (int)(c % 9);
        kp[kPat24[p][0]] = 1;
        kp[kPat24[p][1]] = 1;
        t[kPat24[p][0]] = (int8_t)(v / 3 - 1);
        t[kPat24[p][1]] = (int8_t)(v % 3 - 1);
      }
    }
  return bad;
}

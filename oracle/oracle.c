/*
 * oracle.c — plain fp64 CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h).
 *
 * Built with -ffp-contract=off: every product and every sum is rounded on
 * its own, as the loops are written.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Value of a 16-bit binary floating-point pattern from its bit fields:
 * sign s, biased exponent E, fraction f; normal numbers are
 * (2^m + f) * 2^(E - bias - m), subnormals f * 2^(1 - bias - m). */
double or_decode_half(uint16_t bits, int32_t dtype) {
  const int m = (dtype == OR_BF16) ? 7 : 10;
  const int e = (dtype == OR_BF16) ? 8 : 5;
  const int bias = (1 << (e - 1)) - 1;
  const int s = (bits >> 15) & 1;
  const int E = (bits >> m) & ((1 << e) - 1);
  const int f = bits & ((1 << m) - 1);
  double mag;
  if (E == 0)
    mag = ldexp((double)f, 1 - bias - m);
  else if (E == (1 << e) - 1)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)((1 << m) + f), E - bias - m);
  return s ? -mag : mag;
}

/* Lookup of the decode above, filled once (65536 entries per format). */
static double g_lut[2][65536];
static int g_lut_ready = 0;

static void ensure_lut(void) {
  if (g_lut_ready) return;
  for (int dt = 0; dt < 2; ++dt)
    for (int b = 0; b < 65536; ++b) g_lut[dt][b] = or_decode_half((uint16_t)b, dt);
  g_lut_ready = 1;
}

#define W(dt, v) (g_lut[(dt)][(v)])

void or_set_threads(int32_t nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int32_t or_get_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}

void or_predict(int32_t d, int32_t n, int32_t r, int32_t dtype,
                const uint16_t* A, const uint16_t* Bm, const float* b1,
                const float* x, int32_t batch, double* u, double* logits) {
  ensure_lut();
  const int dt = (dtype == OR_BF16) ? 1 : 0;
  double* uu = (double*)malloc(sizeof(double) * (size_t)r);
  if (!uu) return;
  for (int32_t t = 0; t < batch; ++t) {
    const float* xt = x + (int64_t)t * d;
    /* stage 1: u = Bm x */
    for (int32_t k = 0; k < r; ++k) {
      double acc = 0.0;
      for (int32_t j = 0; j < d; ++j)
        acc += W(dt, Bm[(int64_t)k * d + j]) * (double)xt[j];
      uu[k] = acc;
      if (u) u[(int64_t)t * r + k] = acc;
    }
    /* stage 2: logit_i = A_i . u + b1_i */
    double* lt = logits + (int64_t)t * n;
#pragma omp parallel for schedule(static)
    for (int32_t i = 0; i < n; ++i) {
      double acc = 0.0;
      for (int32_t k = 0; k < r; ++k) acc += W(dt, A[(int64_t)i * r + k]) * uu[k];
      lt[i] = acc + (double)b1[i];
    }
  }
  free(uu);
}

int32_t or_compact(const double* logits, int32_t n, int32_t* idx) {
  int32_t c = 0;
  for (int32_t i = 0; i < n; ++i)
    if (logits[i] > 0.0) idx[c++] = i;
  return c;
}

int32_t or_union(const double* logits, int32_t n, int32_t batch,
                 int32_t* uidx, uint32_t* tok_mask) {
  int32_t c = 0;
  for (int32_t i = 0; i < n; ++i) {
    uint32_t mask = 0;
    for (int32_t t = 0; t < batch && t < 32; ++t)
      if (logits[(int64_t)t * n + i] > 0.0) mask |= (1u << t);
    if (mask) {
      uidx[c] = i;
      if (tok_mask) tok_mask[c] = mask;
      ++c;
    }
  }
  return c;
}

void or_hidden(int32_t d, int32_t dtype, int32_t gated, const uint16_t* W1,
               const float* b1, const float* x, const int32_t* idx,
               int32_t cnt, double* h) {
  ensure_lut();
  const int dt = (dtype == OR_BF16) ? 1 : 0;
  const int64_t stride = gated ? 2 * (int64_t)d : (int64_t)d;
#pragma omp parallel for schedule(static)
  for (int32_t p = 0; p < cnt; ++p) {
    const int64_t i = idx[p];
    const uint16_t* row = W1 + i * stride;
    double pre = 0.0;
    for (int32_t j = 0; j < d; ++j) pre += W(dt, row[j]) * (double)x[j];
    pre += (double)b1[i];
    double act = pre > 0.0 ? pre : 0.0; /* ReLU; ReLU(0) = 0 */
    if (gated) {
      const uint16_t* up = row + d;
      double v = 0.0;
      for (int32_t j = 0; j < d; ++j) v += W(dt, up[j]) * (double)x[j];
      act = act * v;
    }
    h[p] = act;
  }
}

void or_down(int32_t d, int32_t dtype, const uint16_t* W2, const float* b2,
             const int32_t* idx, int32_t cnt, const double* h, double* y) {
  ensure_lut();
  const int dt = (dtype == OR_BF16) ? 1 : 0;
  /* Each thread owns a block of output columns and sums over p in
   * ascending order, which is the column-wise definition read row-wise. */
  const int32_t CB = 64;
  const int32_t nb = (d + CB - 1) / CB;
#pragma omp parallel for schedule(static)
  for (int32_t b = 0; b < nb; ++b) {
    const int32_t j0 = b * CB, j1 = (j0 + CB < d) ? j0 + CB : d;
    double acc[64];
    for (int32_t j = j0; j < j1; ++j) acc[j - j0] = 0.0;
    for (int32_t p = 0; p < cnt; ++p) {
      const uint16_t* row = W2 + (int64_t)idx[p] * d;
      const double hp = h[p];
      for (int32_t j = j0; j < j1; ++j) acc[j - j0] += hp * W(dt, row[j]);
    }
    for (int32_t j = j0; j < j1; ++j) y[j] = acc[j - j0] + (b2 ? (double)b2[j] : 0.0);
  }
}

void or_sparse_ffn(int32_t d, int32_t dtype, int32_t gated,
                   const uint16_t* W1, const float* b1, const uint16_t* W2,
                   const float* b2, const float* x, const int32_t* idx,
                   int32_t cnt, double* y, double* h) {
  double* hh = h;
  if (!hh) hh = (double*)malloc(sizeof(double) * (size_t)(cnt > 0 ? cnt : 1));
  if (!hh) return;
  or_hidden(d, dtype, gated, W1, b1, x, idx, cnt, hh);
  or_down(d, dtype, W2, b2, idx, cnt, hh, y);
  if (!h) free(hh);
}

void or_dense_ffn(int32_t d, int32_t n, int32_t dtype, int32_t gated,
                  const uint16_t* W1, const float* b1, const uint16_t* W2,
                  const float* b2, const float* x, double* y) {
  int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  if (!all) return;
  for (int32_t i = 0; i < n; ++i) all[i] = i;
  or_sparse_ffn(d, dtype, gated, W1, b1, W2, b2, x, all, n, y, NULL);
  free(all);
}

int32_t or_layer_decode(int32_t d, int32_t n, int32_t r, int32_t dtype,
                        int32_t gated, const uint16_t* A, const uint16_t* Bm,
                        const float* b1, const uint16_t* W1,
                        const uint16_t* W2, const float* b2, const float* x,
                        double* logits, int32_t* idx, double* y,
                        float* x_next) {
  or_predict(d, n, r, dtype, A, Bm, b1, x, 1, NULL, logits);
  const int32_t cnt = or_compact(logits, n, idx);
  or_sparse_ffn(d, dtype, gated, W1, b1, W2, b2, x, idx, cnt, y, NULL);
  if (x_next)
    for (int32_t j = 0; j < d; ++j) x_next[j] = (float)((double)x[j] + y[j]);
  return cnt;
}

/* ------------------------------------------------------------ offline placement */
void or_profile_counts(const double* logits, int32_t n, int32_t batch,
                       uint32_t* counts) {
  for (int32_t t = 0; t < batch; ++t)
    for (int32_t i = 0; i < n; ++i)
      if (logits[(size_t)t * n + i] > 0.0) counts[i] += 1u;
}

typedef struct {
  uint32_t count;
  int32_t index;
} or_key;

/* more activations first; equal counts by ascending index */
static int or_key_cmp(const void* pa, const void* pb) {
  const or_key* a = (const or_key*)pa;
  const or_key* b = (const or_key*)pb;
  if (a->count != b->count) return a->count > b->count ? -1 : 1;
  return (a->index > b->index) - (a->index < b->index);
}

void or_hot_order(const uint32_t* counts, int32_t n, int32_t* perm) {
  or_key* k = (or_key*)malloc(sizeof(or_key) * (size_t)(n > 0 ? n : 1));
  if (!k) return;
  for (int32_t i = 0; i < n; ++i) {
    k[i].count = counts[i];
    k[i].index = i;
  }
  qsort(k, (size_t)n, sizeof(or_key), or_key_cmp);
  for (int32_t i = 0; i < n; ++i) perm[i] = k[i].index;
  free(k);
}

void or_permute_rows(const void* src, int32_t n, int32_t row_bytes,
                     const int32_t* perm, void* dst) {
  const unsigned char* s = (const unsigned char*)src;
  unsigned char* d = (unsigned char*)dst;
  for (int32_t k = 0; k < n; ++k)
    memcpy(d + (size_t)k * row_bytes, s + (size_t)perm[k] * row_bytes, (size_t)row_bytes);
}

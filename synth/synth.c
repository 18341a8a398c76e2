/*
 * synth.c — seeded synthetic workload generator (inputs only; see synth.h).
 *
 * Built with -ffp-contract=off so that every multiply and add is rounded on
 * its own, the same way on x86-64 and AArch64 hosts.
 */
#include "synth.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define SY_GAMMA 0x9e3779b97f4a7c15ULL

/* SplitMix64 output function (Steele, Lea & Flood 2014). */
uint64_t sy_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

uint64_t sy_stream_key(uint64_t seed, uint32_t tag, uint32_t layer) {
  uint64_t k = sy_mix64(seed + SY_GAMMA);
  uint64_t id = ((uint64_t)tag << 32) | (uint64_t)layer;
  return sy_mix64(k + (id + 1u) * SY_GAMMA);
}

/* Word k of the stream keyed by `key`: the SplitMix64 sequence started at
 * `key`, read at position k without stepping through 0..k-1. */
uint64_t sy_bits(uint64_t key, uint64_t k) {
  return sy_mix64(key + (k + 1u) * SY_GAMMA);
}

double sy_uniform(uint64_t key, uint64_t k) {
  /* top 53 bits, centred in their cell: never 0, never 1 */
  return ((double)(sy_bits(key, k) >> 11) + 0.5) * 0x1.0p-53;
}

static const double SY_TWO_PI = 6.283185307179586476925286766559;

/* Box–Muller: pair m = k/2 uses uniforms 2m and 2m+1; even k takes the
 * cosine branch, odd k the sine branch. */
double sy_normal(uint64_t key, uint64_t k) {
  uint64_t m = k >> 1;
  double u1 = sy_uniform(key, 2 * m), u2 = sy_uniform(key, 2 * m + 1);
  double rad = sqrt(-2.0 * log(u1));
  double th = SY_TWO_PI * u2;
  return (k & 1u) ? rad * sin(th) : rad * cos(th);
}

/* out[e] = scale * N(key, base + e), e in [0, count). Same values as
 * sy_normal, computed a pair at a time. */
static void fill_normal(uint64_t key, uint64_t base, int64_t count,
                        double scale, double* out) {
  int64_t e = 0;
  if (count <= 0) return;
  if (base & 1u) {
    out[0] = scale * sy_normal(key, base);
    e = 1;
  }
  for (; e + 1 < count; e += 2) {
    uint64_t m = (base + (uint64_t)e) >> 1;
    double u1 = sy_uniform(key, 2 * m), u2 = sy_uniform(key, 2 * m + 1);
    double rad = sqrt(-2.0 * log(u1));
    double th = SY_TWO_PI * u2;
    out[e] = scale * (rad * cos(th));
    out[e + 1] = scale * (rad * sin(th));
  }
  if (e < count) out[e] = scale * sy_normal(key, base + (uint64_t)e);
}

/* Round-to-nearest-even of |v| onto a binary format with `mbits` stored
 * mantissa bits and exponent bias `bias`, written from the bit-field
 * definition: find the unit in the last place q of the target binade (or
 * the subnormal unit), scale |v| by 2^-q exactly, round to an integer with
 * ties to even, and re-encode.  `emax_field` is the all-ones exponent. */
static uint16_t round_binary(double v, int mbits, int bias, int emax_field) {
  /* both formats are 16 bits wide: sign in bit 15 */
  const uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0u;
  const uint16_t inf = (uint16_t)((uint32_t)emax_field << mbits);
  if (isnan(v)) return (uint16_t)(inf | (1u << (mbits - 1)));
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | inf);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
  int q = (e - 1) - mbits;       /* ulp exponent in a's binade */
  int qmin = 1 - bias - mbits;   /* ulp of the subnormal range */
  if (q < qmin) q = qmin;
  double m = nearbyint(ldexp(a, -q)); /* exact scaling; RNE */
  uint64_t mant = (uint64_t)m;
  uint32_t out;
  if (q == qmin) {
    /* subnormal, or (mant == 2^mbits and above) the lowest normal binade:
     * with biased exponent 1 the bit pattern is the integer itself */
    out = (uint32_t)mant;
  } else {
    int E = q + mbits + bias;    /* biased exponent for mant in [2^m, 2^m+1] */
    if (mant == (1ull << (mbits + 1))) {
      mant >>= 1;
      E += 1;
    }
    if (E >= emax_field) return (uint16_t)(sign | inf);
    out = ((uint32_t)E << mbits) | (uint32_t)(mant - (1ull << mbits));
  }
  if (out >= inf) return (uint16_t)(sign | inf);
  return (uint16_t)(sign | out);
}

uint16_t sy_round_f16(double v) { return round_binary(v, 10, 15, 31); }
uint16_t sy_round_bf16(double v) { return round_binary(v, 7, 127, 255); }
uint16_t sy_round_half(double v, int32_t dtype) {
  return dtype == SY_BF16 ? sy_round_bf16(v) : sy_round_f16(v);
}

/* Standard normal CDF via the complementary error function. */
static double phi_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }
static double phi_pdf(double x) { return exp(-0.5 * x * x) / sqrt(SY_TWO_PI); }

double sy_probit(double p) {
  if (!(p > 0.0 && p < 1.0)) return NAN;
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (phi_cdf(mid) < p) lo = mid; else hi = mid;
  }
  double x = 0.5 * (lo + hi);
  for (int it = 0; it < 2; ++it) {
    double f = phi_pdf(x);
    if (f > 0.0) x -= (phi_cdf(x) - p) / f;
  }
  return x;
}

double sy_relu_m2(double q) {
  return (q * q + 1.0) * phi_cdf(q) + q * phi_pdf(q);
}

double sy_zipf_mean(int32_t n, double alpha, double c, double cap) {
  double s = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    double p = c * pow((double)(i + 1), -alpha);
    s += (p < cap) ? p : cap;
  }
  return s / (double)n;
}

double sy_zipf_calibrate(int32_t n, double alpha, double target, double cap) {
  if (!(target > 0.0 && target < cap) || n <= 0) return NAN;
  double lo = 0.0, hi = 1.0;
  while (sy_zipf_mean(n, alpha, hi, cap) < target) {
    hi *= 2.0;
    if (hi > 1e300) return NAN;
  }
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (sy_zipf_mean(n, alpha, mid, cap) < target) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

void sy_zipf_probs(int32_t n, double alpha, double c, double cap, double* p) {
  for (int32_t i = 0; i < n; ++i) {
    double v = c * pow((double)(i + 1), -alpha);
    p[i] = (v < cap) ? v : cap;
  }
}

int32_t sy_num_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}

#define SY_RB 4    /* W1 rows per inner block            */
#define SY_CB 256  /* W1 columns per inner block         */

int32_t sy_gen_layer(const sy_layer_spec* s, uint16_t* A, uint16_t* Bm,
                     float* b1, uint16_t* W1, uint16_t* W2, float* b2) {
  if (!s || s->d <= 0 || s->n <= 0 || s->r <= 0) return -1;
  if (s->dtype != SY_F16 && s->dtype != SY_BF16) return -1;
  const int64_t d = s->d, n = s->n, r = s->r;
  const int32_t dt = s->dtype;
  const uint64_t kA = sy_stream_key(s->seed, SY_TAG_A, (uint32_t)s->layer);
  const uint64_t kB = sy_stream_key(s->seed, SY_TAG_B, (uint32_t)s->layer);
  const uint64_t kN = sy_stream_key(s->seed, SY_TAG_NOISE, (uint32_t)s->layer);
  const uint64_t kW2 = sy_stream_key(s->seed, SY_TAG_W2, (uint32_t)s->layer);
  const uint64_t kU = sy_stream_key(s->seed, SY_TAG_UP, (uint32_t)s->layer);
  const double sr = 1.0 / sqrt((double)r), sd = 1.0 / sqrt((double)d),
               sn = 1.0 / sqrt((double)n);

  double* A64 = NULL;
  double* B64 = NULL;
  if (A || Bm || W1) {
    A64 = (double*)malloc(sizeof(double) * (size_t)(n * r));
    B64 = (double*)malloc(sizeof(double) * (size_t)(r * d));
    if (!A64 || !B64) {
      free(A64);
      free(B64);
      return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) fill_normal(kA, (uint64_t)(i * r), r, sr, A64 + i * r);
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < r; ++k) fill_normal(kB, (uint64_t)(k * d), d, sd, B64 + k * d);
    if (A)
      for (int64_t e = 0; e < n * r; ++e) A[e] = sy_round_half(A64[e], dt);
    if (Bm)
      for (int64_t e = 0; e < r * d; ++e) Bm[e] = sy_round_half(B64[e], dt);
  }

  if (b1) {
    double* p = (double*)malloc(sizeof(double) * (size_t)n);
    if (!p) {
      free(A64);
      free(B64);
      return -2;
    }
    sy_zipf_probs(s->n, s->alpha, s->zipf_c, s->p_cap, p);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) b1[i] = (float)(s->bias_scale * sy_probit(p[i]));
    free(p);
  }

  if (W1) {
    const int64_t rowstride = s->gated ? 2 * d : d;
    const int64_t nchunks = (n + 63) / 64;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      double acc[SY_RB][SY_CB];
      double nz[SY_CB];
      const int64_t i_lo = ch * 64, i_hi = (i_lo + 64 < n) ? i_lo + 64 : n;
      for (int64_t j0 = 0; j0 < d; j0 += SY_CB) {
        const int64_t cw = (j0 + SY_CB <= d) ? SY_CB : d - j0;
        for (int64_t i0 = i_lo; i0 < i_hi; i0 += SY_RB) {
          const int64_t rw = (i0 + SY_RB <= i_hi) ? SY_RB : i_hi - i0;
          for (int64_t ii = 0; ii < rw; ++ii)
            for (int64_t jj = 0; jj < cw; ++jj) acc[ii][jj] = 0.0;
          /* acc[i][j] = sum_k A64[i][k] * B64[k][j], k ascending */
          for (int64_t k = 0; k < r; ++k) {
            const double* brow = B64 + k * d + j0;
            for (int64_t ii = 0; ii < rw; ++ii) {
              const double a = A64[(i0 + ii) * r + k];
              for (int64_t jj = 0; jj < cw; ++jj) acc[ii][jj] += a * brow[jj];
            }
          }
          for (int64_t ii = 0; ii < rw; ++ii) {
            const int64_t i = i0 + ii;
            fill_normal(kN, (uint64_t)(i * d + j0), cw, sd, nz);
            uint16_t* dst = W1 + i * rowstride + j0;
            for (int64_t jj = 0; jj < cw; ++jj)
              dst[jj] = sy_round_half(acc[ii][jj] + s->noise * nz[jj], dt);
          }
        }
      }
      if (s->gated) {
        double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
        if (tmp) {
          for (int64_t i = i_lo; i < i_hi; ++i) {
            fill_normal(kU, (uint64_t)(i * d), d, sd, tmp);
            uint16_t* dst = W1 + i * rowstride + d;
            for (int64_t j = 0; j < d; ++j) dst[j] = sy_round_half(tmp[j], dt);
          }
          free(tmp);
        }
      }
    }
  }
  free(A64);
  free(B64);

  if (W2) {
#pragma omp parallel
    {
      double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(static)
      for (int64_t i = 0; i < n; ++i) {
        if (!tmp) continue;
        fill_normal(kW2, (uint64_t)(i * d), d, sn, tmp);
        for (int64_t j = 0; j < d; ++j) W2[i * d + j] = sy_round_half(tmp[j], dt);
      }
      free(tmp);
    }
  }
  if (b2)
    for (int64_t j = 0; j < d; ++j) b2[j] = 0.0f;
  return 0;
}

void sy_gen_x(uint64_t seed, int32_t step, int32_t batch, int32_t d, float* x) {
  const uint64_t key = sy_stream_key(seed, SY_TAG_X, (uint32_t)step);
  const int64_t tot = (int64_t)batch * d;
  double* tmp = (double*)malloc(sizeof(double) * (size_t)(tot > 0 ? tot : 1));
  if (!tmp) return;
  fill_normal(key, 0, tot, 1.0, tmp);
  for (int64_t e = 0; e < tot; ++e) x[e] = (float)tmp[e];
  free(tmp);
}

void sy_stack_plan(uint64_t seed, int32_t L, int32_t n, double a_lo,
                   double a_hi, double rho_hi, double rho_lo, double cap,
                   double* alpha, double* rho, double* c, double* scale) {
  const uint64_t key = sy_stream_key(seed, SY_TAG_ALPHA, 0);
  double* p = (double*)malloc(sizeof(double) * (size_t)n);
  double v = 1.0;
  for (int32_t l = 0; l < L; ++l) {
    double a = a_lo + (a_hi - a_lo) * sy_uniform(key, (uint64_t)l);
    double t = rho_hi - (rho_hi - rho_lo) * (a - a_lo) / (a_hi - a_lo);
    double cl = sy_zipf_calibrate(n, a, t, cap);
    alpha[l] = a;
    rho[l] = t;
    c[l] = cl;
    scale[l] = sqrt(v);
    if (p) {
      sy_zipf_probs(n, a, cl, cap, p);
      double g = 0.0;
      for (int32_t i = 0; i < n; ++i) g += sy_relu_m2(sy_probit(p[i]));
      v = v * (1.0 + g / (double)n);
    }
  }
  free(p);
}

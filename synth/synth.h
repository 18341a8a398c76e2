/*
 * synth.h — seeded synthetic workload generator for the activation-sparse
 * decode FFN (PowerInfer-style hot/cold neurons).
 *
 * This module makes INPUTS only: weight bytes, biases and decode-step
 * activations.  It holds none of the method's arithmetic (no predictor, no
 * compaction, no FFN); both the fp64 oracle and the CUDA library consume the
 * bytes it writes.  Everything is a pure function of (seed, tensor tag,
 * layer, element index), so any element can be regenerated on its own and
 * results do not depend on the thread count.
 *
 * Randomness: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used as a counter-based generator:
 * word k of a stream = mix(key + (k+1)*gamma).  Normals: Box–Muller on two
 * such uniforms.  Probit: bisection + Newton on Phi(x) = erfc(-x/sqrt2)/2.
 * Half-precision encodings: round-to-nearest-even from the IEEE-754
 * binary16 / bfloat16 bit-field definitions.
 *
 * Workload recipe (the pages give no formulas; this is the construction of
 * the seeded synthetic layers):
 *   A  (n x r) ~ N(0, 1/r),  Bm (r x d) ~ N(0, 1/d)          (predictor)
 *   W1 = round(A64 * Bm64 + noise * N(0, 1/d))               (up proj.)
 *   b1_i = bias_scale * probit(p_i),
 *   p_i = min(p_cap, zipf_c * (i+1)^-alpha)                  (hot-first)
 *   W2 (n x d) ~ N(0, 1/n), b2 = 0                           (down proj.)
 *   gated: W1 rows are [gate | up] per neuron; gate as W1 above, its bias
 *   b1; up ~ N(0, 1/d) with no bias.
 *   x ~ N(0, 1), rounded once to fp32, fresh per (seed, step, token).
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SY_F16 = 0, SY_BF16 = 1 };

/* Stream tags (one independent stream per tensor kind). */
enum {
  SY_TAG_A = 1,      /* predictor factor A, n x r            */
  SY_TAG_B = 2,      /* predictor factor Bm, r x d           */
  SY_TAG_NOISE = 3,  /* W1 (or W_gate) noise, n x d          */
  SY_TAG_W2 = 4,     /* down projection, n x d               */
  SY_TAG_UP = 5,     /* gated up projection, n x d           */
  SY_TAG_X = 6,      /* decode-step activations              */
  SY_TAG_ALPHA = 7,  /* per-layer Zipf exponent of a stack   */
  SY_TAG_PERM = 8    /* neuron shuffles (tests)              */
};

typedef struct {
  int32_t d, n, r;      /* model dim, FFN neurons, predictor rank           */
  int32_t dtype;        /* SY_F16 or SY_BF16                                */
  int32_t gated;        /* 0: ReLU FFN; 1: ReLU(gate) * up, rows [gate|up]  */
  int32_t layer;        /* layer index (selects streams)                    */
  uint64_t seed;
  double alpha;         /* Zipf exponent                                     */
  double zipf_c;        /* Zipf constant                                     */
  double p_cap;         /* probability cap (0.9)                             */
  double bias_scale;    /* scale of the probit biases (1 for one layer)      */
  double noise;         /* W1 noise amplitude (0.05)                         */
} sy_layer_spec;

/* --- counter-based random numbers --- */
uint64_t sy_mix64(uint64_t z);
uint64_t sy_stream_key(uint64_t seed, uint32_t tag, uint32_t layer);
uint64_t sy_bits(uint64_t key, uint64_t k);
double sy_uniform(uint64_t key, uint64_t k);  /* in (0, 1), 53-bit grid */
double sy_normal(uint64_t key, uint64_t k);   /* N(0, 1) */

/* --- encodings: round-to-nearest-even of a double --- */
uint16_t sy_round_f16(double v);
uint16_t sy_round_bf16(double v);
uint16_t sy_round_half(double v, int32_t dtype);

/* --- Zipf activation profile and probit biases --- */
double sy_probit(double p);
double sy_zipf_mean(int32_t n, double alpha, double c, double cap);
double sy_zipf_calibrate(int32_t n, double alpha, double target, double cap);
void sy_zipf_probs(int32_t n, double alpha, double c, double cap, double* p);

/* Second moment of ReLU(z) for z ~ N(q, 1): E[max(z,0)^2]. */
double sy_relu_m2(double q);

/* --- tensors --- */
/* Writes A [n][r], Bm [r][d] (half bytes), b1 [n] fp32, W1 [n][d] or gated
 * [n][2][d] (half bytes), W2 [n][d] (half bytes), b2 [d] fp32 (zeros).
 * Any output pointer may be NULL to skip that tensor (W1 needs the
 * unrounded factors, which are regenerated internally).  Returns 0 on
 * success, -1 on a bad spec, -2 on allocation failure. */
int32_t sy_gen_layer(const sy_layer_spec* s, uint16_t* A, uint16_t* Bm,
                     float* b1, uint16_t* W1, uint16_t* W2, float* b2);

/* x[t][j] for t in [0, batch), one decode step: fp32(N(0,1)). */
void sy_gen_x(uint64_t seed, int32_t step, int32_t batch, int32_t d, float* x);

/* Plan of a residual stack of L layers: per-layer Zipf exponent alpha_l ~
 * U[a_lo, a_hi] from the seed, density target rho_l falling linearly from
 * rho_hi (alpha = a_lo) to rho_lo (alpha = a_hi), calibrated Zipf constant
 * c_l, and bias scale s_l = sqrt(v_l), where v_l is the expected per-element
 * variance of the residual stream entering layer l under the recipe
 * (v_0 = 1, v_{l+1} = v_l * (1 + mean_i E[ReLU(N(q_i,1))^2]), q_i =
 * probit(p_i)).  Arrays have length L. */
void sy_stack_plan(uint64_t seed, int32_t L, int32_t n, double a_lo,
                   double a_hi, double rho_hi, double rho_lo, double cap,
                   double* alpha, double* rho, double* c, double* scale);

int32_t sy_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif

/*
 * oracle.h — plain fp64 CPU oracle of the activation-sparse decode FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline arm may load this library.  It shares no code,
 * header, table or constant with the CUDA library; the two meet only in the
 * weight and activation bytes that the seeded generator writes.
 *
 * What it computes is the plain definition of the method described on the
 * page "PowerInfer: Quick Massive Language Mannequin Serving with a
 * Client-grade GPU": an online predictor scores every FFN neuron, the engine
 * skips the neurons predicted inactive ("Online Section"), and the
 * neuron-aware operator computes only the rows / columns of the activated
 * neurons without converting the matrices to a dense or sparse format
 * ("Neuron Conscious Operator").  Neuron indices always refer to the
 * position of the neuron in the stored matrices ("Neuron Placement and
 * Administration": the neuron table maps a neuron to its matrix position).
 * The page does not print the predictor's form or the activation: here the
 * predictor is the low-rank linear scorer logits = A (Bm x) + b1, a neuron
 * is active iff its logit is > 0, the FFN activation is ReLU, and the down
 * projection W2 is stored with one row per neuron (its "column vectors").
 *
 * Precision: weights are decoded exactly from their binary16 / bfloat16 bit
 * fields; every product and sum is a double, accumulated in ascending index
 * order; there is no blocking or reordering beyond what the loops show.
 * Results do not depend on the OpenMP thread count: each output element is
 * computed by one thread in one fixed order.
 *
 * Layouts (row-major, one row per neuron):
 *   A [n][r], Bm [r][d], b1 [n] fp32, W1 [n][d] (gated: [n][2][d] = gate row
 *   then up row), W2 [n][d], b2 [d] fp32 or NULL, x [batch][d] fp32.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_F16 = 0, OR_BF16 = 1 };

/* Value of a binary16 (dtype 0) or bfloat16 (dtype 1) bit pattern. */
double or_decode_half(uint16_t bits, int32_t dtype);

/* Predictor: u[t] = Bm x[t] (u is [batch][r]); logits[t][i] = A_i . u[t]
 * + b1_i.  Either output may be NULL except logits. */
void or_predict(int32_t d, int32_t n, int32_t r, int32_t dtype,
                const uint16_t* A, const uint16_t* Bm, const float* b1,
                const float* x, int32_t batch, double* u, double* logits);

/* Compaction: idx = ascending {i : logits[i] > 0}; returns the count. */
int32_t or_compact(const double* logits, int32_t n, int32_t* idx);

/* Union over a batch: uidx = ascending {i : some token t has logit > 0},
 * tok_mask[k] bit t set iff token t is active at neuron uidx[k] (batch <=
 * 32).  Returns the union count. */
int32_t or_union(const double* logits, int32_t n, int32_t batch,
                 int32_t* uidx, uint32_t* tok_mask);

/* Activation of the listed neurons for one token:
 *   plain: h[p] = max(0, W1[idx[p]] . x + b1[idx[p]])
 *   gated: h[p] = max(0, Wg[idx[p]] . x + b1[idx[p]]) * (Wu[idx[p]] . x) */
void or_hidden(int32_t d, int32_t dtype, int32_t gated, const uint16_t* W1,
               const float* b1, const float* x, const int32_t* idx,
               int32_t cnt, double* h);

/* Down projection over the listed neurons for one token:
 *   y[j] = b2[j] + sum_p h[p] * W2[idx[p]][j]   (p ascending) */
void or_down(int32_t d, int32_t dtype, const uint16_t* W2, const float* b2,
             const int32_t* idx, int32_t cnt, const double* h, double* y);

/* Sparse FFN of one token over the listed neurons (or_hidden + or_down).
 * h may be NULL. */
void or_sparse_ffn(int32_t d, int32_t dtype, int32_t gated,
                   const uint16_t* W1, const float* b1, const uint16_t* W2,
                   const float* b2, const float* x, const int32_t* idx,
                   int32_t cnt, double* y, double* h);

/* Dense FFN of one token: the same over all n neurons. */
void or_dense_ffn(int32_t d, int32_t n, int32_t dtype, int32_t gated,
                  const uint16_t* W1, const float* b1, const uint16_t* W2,
                  const float* b2, const float* x, double* y);

/* One decode step of one layer for one token: predict, compact, sparse FFN.
 * logits [n], idx [n] (capacity n), y [d]; returns the active count.  If
 * x_next is not NULL it receives the residual stream fp32(x + y), rounded
 * once. */
int32_t or_layer_decode(int32_t d, int32_t n, int32_t r, int32_t dtype,
                        int32_t gated, const uint16_t* A, const uint16_t* Bm,
                        const float* b1, const uint16_t* W1,
                        const uint16_t* W2, const float* b2, const float* x,
                        double* logits, int32_t* idx, double* y,
                        float* x_next);

/* Offline profiling and neuron placement ("Offline Section": a profiler
 * records how often each neuron activates over sample inputs, and the
 * neurons are placed hot first; "Neuron Placement and Administration": the
 * neuron table maps a neuron's placed position to its original one).
 *   or_profile_counts: counts[i] += #{t < batch : logits[t][i] > 0}
 *     (logits [batch][n]).
 *   or_hot_order: perm[k] = the original neuron placed at position k: more
 *     activations first, equal counts in ascending original index.
 *   or_permute_rows: dst row k = src row perm[k], rows of row_bytes bytes. */
void or_profile_counts(const double* logits, int32_t n, int32_t batch,
                       uint32_t* counts);
void or_hot_order(const uint32_t* counts, int32_t n, int32_t* perm);
void or_permute_rows(const void* src, int32_t n, int32_t row_bytes,
                     const int32_t* perm, void* dst);

void or_set_threads(int32_t nthreads);
int32_t or_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif

// plan.cuh — density / batch-aware choice of the decode path (host code).
//
// The plan follows the planning step of "Efficient, VRAM-Constrained xLM
// Inference on Clients", section "Methodology, A. Pipelined Sharding": for a
// tier of tokens per step, a time estimator built on bytes moved and a
// profile of measured rates predicts the latency of each candidate plan and
// the cheapest one is kept.  Here the candidates are this library's decode
// paths, and the work they move follows "PowerInfer: Quick Massive Language
// Mannequin Serving with a Client-grade GPU", section "Online Section" (only
// predicted-active rows are read): a token reads the rows of its own active
// neurons; a batch on the union path reads every row active for at least one
// of its tokens once.
//
// Expected rows.  With p_i the probability that neuron i is active for a
// token (the offline profile's counts / tokens, or one density for all) and
// tokens independent, a token's expected active rows are sum_i p_i and the
// expected union of B tokens is sum_i (1 - (1 - p_i)^B).
//
// Time of a path = fixed + bytes / rate, with the fixed cost and the rate
// measured per path and batch tier (pi_cost_model; the built-in one was
// fitted to this GPU's sweep of the OPT-13B-shaped layer).
#pragma once

#include <cmath>
#include <cstdint>

#include "../../include/pi.h"

namespace pik {

// Expected active rows of one token and of the union of `batch` tokens.
inline void plan_expected_rows(const float* p, int n, float density, int batch, double* active,
                               double* uni) {
  double a = 0.0, u = 0.0;
  if (p) {
    for (int i = 0; i < n; ++i) {
      double q = p[i];
      q = q < 0.0 ? 0.0 : (q > 1.0 ? 1.0 : q);
      a += q;
      u += 1.0 - std::pow(1.0 - q, (double)batch);  // (1 - q)^B: no neuron active in any token
    }
  } else {
    double q = density;
    q = q < 0.0 ? 0.0 : (q > 1.0 ? 1.0 : q);
    a = q * n;
    u = (1.0 - std::pow(1.0 - q, (double)batch)) * n;
  }
  *active = a;
  *uni = u;
}

// Index of the batch tier of a cost model (tiers hold the largest batch
// they cover, ascending); the last tier for larger batches.
inline int plan_tier(const pi_cost_model& m, int batch) {
  for (int t = 0; t < PI_COST_TIERS; ++t)
    if (batch <= m.tier_max_batch[t]) return t;
  return PI_COST_TIERS - 1;
}

// Microseconds of moving `bytes` after a fixed cost of `fixed_us` at
// `gbs` GB/s.
inline double plan_time_us(double fixed_us, double bytes, double gbs) {
  return fixed_us + bytes / (gbs * 1e3);
}

}  // namespace pik

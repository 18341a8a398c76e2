// shard.cuh — neuron-sharded decode across G ranks (host code, one kernel).
//
// The FFN's neurons are independent until the down projection sums them:
// "PowerInfer: Quick Massive Language Mannequin Serving with a Client-grade
// GPU", section "Neuron Conscious Operator" (each active neuron adds its own
// column vector of the down projection), and "Neuron Placement and
// Administration" (a table maps the neurons a device holds to their places
// in the layer).  Rank g of G holds the neurons i = g, g + G, g + 2G, ... of
// the hot-first order (round robin keeps the hot prefix spread evenly) with
// a full copy of the predictor factor Bm, and decodes them with the ordinary
// calls into a partial output; one exchange of the G partial outputs
// (d floats per token, an all-gather) and their sum in rank order complete
// the layer.  Included at the end of pi_abi.cu.
#pragma once

#include <cuda_runtime.h>

#include "../../include/pi.h"

namespace pik {

// y[t][k] = residual[t][k] + sum_{g ascending} parts[g][t][k]  (fixed order).
__global__ void shard_reduce_kernel(const float4* parts, int G, long long count4,
                                    const float4* residual, float4* y) {
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < count4;
       k += (long long)gridDim.x * blockDim.x) {
    float4 s = residual ? residual[k] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < G; ++g) {
      const float4 v = parts[(long long)g * count4 + k];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    y[k] = s;
  }
}

// Rows of [0, n) that rank g of G holds: g, g + G, ...
inline int shard_rows(int n, int G, int g) { return g < n ? (n - 1 - g) / G + 1 : 0; }

}  // namespace pik

extern "C" {

pi_status pi_shard_desc(const pi_ffn_desc* desc, int32_t G, int32_t g, pi_ffn_desc* out) {
  if (!desc || !out) return PI_ERR_NULL;
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (G < 1 || G > 1024 || g < 0 || g >= G || g >= desc->n) return PI_ERR_SHAPE;
  pi_ffn_desc D = *desc;
  D.n = pik::shard_rows(desc->n, G, g);
  D.hot_prefix = pik::shard_rows(desc->hot_prefix, G, g);
  *out = D;
  return PI_OK;
}

pi_status pi_shard_layer(const pi_ffn_desc* desc, const pi_layer_weights* src, int32_t G,
                         int32_t g, const pi_layer_weights* dst, pi_stream stream) {
  pi_ffn_desc S;
  pi_status s = pi_shard_desc(desc, G, g, &S);
  if (s != PI_OK) return s;
  s = check_weights(*desc, src, true);
  if (s != PI_OK) return s;
  if (!dst) return PI_ERR_NULL;
  s = check_weights(S, dst, true);
  if (s != PI_OK) return s;
  if (dst->A == src->A || dst->b1 == src->b1 || dst->W1 == src->W1 ||
      (desc->layout == PI_LAYOUT_SPLIT && dst->W2 == src->W2))
    return PI_ERR_SHAPE;
  const pi_ffn_desc& D = *desc;
  const size_t rows = (size_t)S.n;
  const int m1 = D.gated ? 2 : 1;
  const size_t w1b = (size_t)(D.layout == PI_LAYOUT_PACKED ? m1 + 1 : m1) * D.d * 2;
  struct Job {
    const void* a;
    void* b;
    size_t row_bytes;
  } jobs[4] = {{src->A, const_cast<void*>(dst->A), (size_t)D.r * 2},
               {src->b1, const_cast<float*>(dst->b1), 4},
               {src->W1, const_cast<void*>(dst->W1), w1b},
               {src->W2, const_cast<void*>(dst->W2), (size_t)D.d * 2}};
  const int nj = D.layout == PI_LAYOUT_SPLIT ? 4 : 3;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  for (int j = 0; j < nj; ++j) {
    // row k of the shard = row g + k G of the layer: one strided copy
    const char* from = static_cast<const char*>(jobs[j].a) + (size_t)g * jobs[j].row_bytes;
    if (cudaMemcpy2DAsync(jobs[j].b, jobs[j].row_bytes, from, (size_t)G * jobs[j].row_bytes,
                          jobs[j].row_bytes, rows, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return PI_ERR_CUDA;
  }
  return PI_OK;
}

pi_status pi_shard_reduce(const float* parts, int32_t G, int32_t batch, int32_t d,
                          const float* residual, float* y, pi_stream stream) {
  if (!parts || !y) return PI_ERR_NULL;
  if (G < 1 || G > 1024 || batch < 1 || batch > pik::kMaxBatch || d < 8 || d > 8192 || (d & 7))
    return PI_ERR_SHAPE;
  const void* ps[] = {parts, residual, y};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  const long long c4 = (long long)batch * d / 4;
  const long long blocks = (c4 + 255) / 256;
  pik::shard_reduce_kernel<<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0,
                             reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float4*>(parts), G, c4, reinterpret_cast<const float4*>(residual),
      reinterpret_cast<float4*>(y));
  return cudaGetLastError() == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}

}  // extern "C"

// decoder.cuh — execution of a dispatch plan (host code, one small kernel).
//
// The plan (plan.cuh) follows the planning step of "Efficient,
// VRAM-Constrained xLM Inference on Clients", section "Methodology, A.
// Pipelined Sharding": per tier of tokens per step, the cheapest plan by a
// time estimator over measured rates.  pi_decode_planned runs the path a plan
// names; a pi_decoder keeps one plan and one captured CUDA graph per batch
// size, bound to fixed input / output buffers, so that a step of a given
// batch is one graph launch.  Included at the end of pi_abi.cu (it calls the
// entry points defined there).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pi.h"

namespace pik {

// y[k] += r[k] for k < count (float4 granularity; count % 4 == 0).
__global__ void add_residual_kernel(float4* y, const float4* r, long long count4) {
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < count4;
       k += (long long)gridDim.x * blockDim.x) {
    float4 a = y[k];
    const float4 b = r[k];
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
    y[k] = a;
  }
}

}  // namespace pik

struct pi_decoder {
  pi_ffn_desc desc;
  pi_layer_weights w;
  int allow_dense;
  pi_cost_model model;
  bool have_p;
  float density;
  float* p_active;  // host copy of the profile (n values) or nullptr
  const float* x;
  float* y;
  const float* residual;
  int32_t* dev_status;
  void* ws;
  size_t ws_bytes;
  int device;
  cudaStream_t cap;  // stream the graphs are captured on
  pi_plan plan[pik::kMaxBatch + 1];
  bool planned[pik::kMaxBatch + 1];
  cudaGraphExec_t graph[pik::kMaxBatch + 1];
  std::mutex mu;
};

extern "C" {

pi_status pi_decode_planned(const pi_ffn_desc* desc, const pi_layer_weights* w, int32_t path,
                            const float* x, int32_t batch, float* y, const float* residual,
                            int32_t* idx_out, int32_t* cnt_out, int32_t* dev_status, void* ws,
                            size_t ws_bytes, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > pik::kMaxBatch) return PI_ERR_SHAPE;
  const size_t d = (size_t)desc->d, n = (size_t)desc->n;
  switch (path) {
    case PI_PATH_FUSED:
      if (batch != 1) return PI_ERR_SHAPE;
      return pi_layer_decode(desc, w, x, 1, y, residual, idx_out, cnt_out, dev_status, ws,
                             ws_bytes, stream);
    case PI_PATH_PER_TOKEN:
      for (int t = 0; t < batch; ++t) {
        s = pi_layer_decode(desc, w, x + t * d, 1, y + t * d, residual ? residual + t * d : nullptr,
                            idx_out ? idx_out + t * n : nullptr, cnt_out ? cnt_out + t : nullptr,
                            dev_status, ws, ws_bytes, stream);
        if (s != PI_OK) return s;
      }
      return PI_OK;
    case PI_PATH_UNION:
      if (batch < 2 || desc->d % 128) return PI_ERR_SHAPE;
      return pi_layer_decode(desc, w, x, batch, y, residual, idx_out, cnt_out, dev_status, ws,
                             ws_bytes, stream);
    case PI_PATH_DENSE: {
      if (residual && !aligned16(residual)) return PI_ERR_ALIGN;
      s = pi_dense_ffn(desc, w, x, batch, y, ws, ws_bytes, stream);
      if (s != PI_OK || !residual) return s;
      const long long c4 = (long long)batch * desc->d / 4;
      pik::add_residual_kernel<<<(unsigned)((c4 + 255) / 256 < 1024 ? (c4 + 255) / 256 : 1024), 256,
                                 0, reinterpret_cast<cudaStream_t>(stream)>>>(
          reinterpret_cast<float4*>(y), reinterpret_cast<const float4*>(residual), c4);
      return cudaGetLastError() == cudaSuccess ? PI_OK : PI_ERR_CUDA;
    }
    default:
      return PI_ERR_SHAPE;
  }
}

pi_status pi_decoder_create(const pi_ffn_desc* desc, const pi_layer_weights* w,
                            const float* p_active, float density, int32_t allow_dense,
                            const pi_cost_model* model, const float* x, float* y,
                            const float* residual, int32_t* dev_status, void* ws, size_t ws_bytes,
                            pi_decoder** out) {
  if (!out) return PI_ERR_NULL;
  *out = nullptr;
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  s = check_weights(*desc, w, true);
  if (s != PI_OK) return s;
  if (!x || !y || !dev_status || !ws) return PI_ERR_NULL;
  const void* ps[] = {x, y, residual, dev_status, ws};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  if (ws_bytes < ws_layout(*desc, pik::kMaxBatch).total) return PI_ERR_WORKSPACE;
  pi_plan probe;
  s = pi_plan_dispatch(desc, 1, p_active, density, allow_dense, model, &probe);
  if (s != PI_OK) return s;
  pi_decoder* D = new pi_decoder();
  D->desc = *desc;
  D->w = *w;
  D->allow_dense = allow_dense;
  if (model) D->model = *model;
  else pi_default_cost_model(&D->model);
  D->have_p = p_active != nullptr;
  D->density = density;
  D->p_active = nullptr;
  if (p_active) {
    D->p_active = new float[(size_t)desc->n];
    for (int i = 0; i < desc->n; ++i) D->p_active[i] = p_active[i];
  }
  D->x = x;
  D->y = y;
  D->residual = residual;
  D->dev_status = dev_status;
  D->ws = ws;
  D->ws_bytes = ws_bytes;
  for (int b = 0; b <= pik::kMaxBatch; ++b) {
    D->planned[b] = false;
    D->graph[b] = nullptr;
  }
  if (cudaGetDevice(&D->device) != cudaSuccess ||
      cudaStreamCreateWithFlags(&D->cap, cudaStreamNonBlocking) != cudaSuccess) {
    delete[] D->p_active;
    delete D;
    return PI_ERR_CUDA;
  }
  *out = D;
  return PI_OK;
}

pi_status pi_decoder_plan(pi_decoder* D, int32_t batch, pi_plan* out) {
  if (!D || !out) return PI_ERR_NULL;
  if (batch < 1 || batch > pik::kMaxBatch) return PI_ERR_SHAPE;
  std::lock_guard<std::mutex> lk(D->mu);
  if (!D->planned[batch]) {
    pi_status s = pi_plan_dispatch(&D->desc, batch, D->p_active, D->density, D->allow_dense,
                                   &D->model, &D->plan[batch]);
    if (s != PI_OK) return s;
    D->planned[batch] = true;
  }
  *out = D->plan[batch];
  return PI_OK;
}

pi_status pi_decoder_run(pi_decoder* D, int32_t batch, pi_stream stream) {
  if (!D) return PI_ERR_NULL;
  pi_plan P;
  pi_status s = pi_decoder_plan(D, batch, &P);
  if (s != PI_OK) return s;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PI_ERR_CUDA;
  if (dev != D->device) return PI_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(D->mu);
  if (D->graph[batch]) {
    return cudaGraphLaunch(D->graph[batch], st) == cudaSuccess ? PI_OK : PI_ERR_CUDA;
  }
  // first step of this batch size: run it directly (this call's result;
  // also sets the kernels' launch attributes), then capture the same calls
  // into the graph that later steps replay
  s = pi_decode_planned(&D->desc, &D->w, P.path, D->x, batch, D->y, D->residual, nullptr,
                        nullptr, D->dev_status, D->ws, D->ws_bytes, stream);
  if (s != PI_OK) return s;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return PI_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return PI_OK;  // the caller is capturing: no graph of ours
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(D->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return PI_ERR_CUDA;
  const pi_status sc =
      pi_decode_planned(&D->desc, &D->w, P.path, D->x, batch, D->y, D->residual, nullptr, nullptr,
                        D->dev_status, D->ws, D->ws_bytes, reinterpret_cast<pi_stream>(D->cap));
  const cudaError_t ec = cudaStreamEndCapture(D->cap, &g);
  if (sc != PI_OK || ec != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return sc != PI_OK ? sc : PI_ERR_CUDA;
  }
  cudaGraphExec_t ge = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&ge, g, 0);
  cudaGraphDestroy(g);
  if (ei != cudaSuccess) return PI_ERR_CUDA;
  D->graph[batch] = ge;
  return PI_OK;
}

void pi_decoder_destroy(pi_decoder* D) {
  if (!D) return;
  for (int b = 0; b <= pik::kMaxBatch; ++b)
    if (D->graph[b]) cudaGraphExecDestroy(D->graph[b]);
  cudaStreamDestroy(D->cap);
  delete[] D->p_active;
  delete D;
}

}  // extern "C"

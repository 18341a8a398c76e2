// common.cuh — device helpers shared by the kernels of libpi (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pi.h"

namespace pik {

constexpr int kThreads = 512;             // block size of the persistent kernels
constexpr int kWarps = kThreads / 32;
constexpr int kPMax = 512;                // largest persistent grid supported
constexpr int kSMax = 8;                  // largest split of a predictor row
constexpr int kMaxBatch = 32;

// ------------------------------------------------------------------ loads
// 16-byte read-only load that does not allocate in L1 (weights streamed once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte read-only load through the non-coherent path.
__device__ __forceinline__ uint4 ld_nc(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Converts 8 packed 16-bit values (fp16 if DT == 0, bf16 if DT == 1).
template <int DT>
__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == 0) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    } else {
      // bfloat16 is the upper half of an fp32 pattern: widening is exact
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ sync
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void set_status(int* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

// Barrier state in the workspace: arrival counter and generation word on
// separate 128-byte lines.
struct GridBar {
  unsigned* count;
  unsigned* gen;
};

// Grid-wide barrier of `expected` blocks with a bounded wait.  Every block
// must call it the same number of times.  Returns false (and records
// PI_ERR_TIMEOUT) when the generation did not advance within limit_ns.
// Writes made by the block before the call are visible to every block after
// it (read them with ld.cg / __ldcg: L1 is not coherent across blocks).
__device__ __noinline__ bool grid_sync(GridBar bar, unsigned expected, int* status,
                                       uint64_t limit_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned g = ld_acquire(bar.gen);
    __threadfence();
    const unsigned prev = atomicAdd(bar.count, 1u);
    if (prev == expected - 1u) {
      atomicExch(bar.count, 0u);
      __threadfence();
      st_release(bar.gen, g + 1u);
    } else {
      const uint64_t t0 = global_ns();
      unsigned spins = 0;
      while (ld_acquire(bar.gen) == g) {
        if ((++spins & 63u) == 0u && global_ns() - t0 > limit_ns) {
          ok = 0;
          set_status(status, PI_ERR_TIMEOUT);
          break;
        }
        __nanosleep(20);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

}  // namespace pik

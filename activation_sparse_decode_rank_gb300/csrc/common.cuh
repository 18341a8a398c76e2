// common.cuh — device helpers shared by the kernels of libpi (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pi.h"

namespace pik {

constexpr int kThreads = 512;             // compute threads of a persistent block
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;     // + one producer warp issuing TMA copies
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

// Converts 8 packed 16-bit values (fp16 if DT == 0, bf16 if DT == 1) to four
// fp32 pairs (elements 2i, 2i + 1 in pair i).
template <int DT>
__device__ __forceinline__ void unpack4x2(const uint4& v, float2 f[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (DT == 0) {
      f[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    } else {
      f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
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

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barriers on one 64-bit arrival counter in the workspace.  Each
// barrier adds exactly one arrival per block, so at the start of a launch the
// counter is a multiple of the grid size P; a block reads it once
// (grid_base) and barrier k of the launch waits for base + k P arrivals.
// Arrival is a fire-and-forget reduction (no round trip); the wait is
// bounded by limit_ns and records PI_ERR_TIMEOUT when it runs out.  Writes
// made by the block before the call are visible to every block after it
// (read them with ld.cg / __ldcg: L1 is not coherent across blocks): the
// block's threads meet at __syncthreads first, and thread 0's release
// reduction is cumulative over the writes that meeting ordered before it, so
// no separate fence is needed.
__device__ __forceinline__ unsigned long long grid_base(const unsigned long long* ctr,
                                                        unsigned nblocks) {
  const unsigned long long v = ld_acquire64(ctr);
  return v - v % nblocks;
}

__device__ __noinline__ bool grid_sync(unsigned long long* ctr, unsigned long long target,
                                       int* status, uint64_t limit_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
    const uint64_t t0 = global_ns();
    unsigned spins = 0;
    while ((long long)(ld_acquire64(ctr) - target) < 0) {
      if ((++spins & 15u) == 0u && global_ns() - t0 > limit_ns) {
        ok = 0;
        set_status(status, PI_ERR_TIMEOUT);
        break;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// The two halves of grid_sync, for work between the block's arrival and
// its wait (work that no other block reads).  grid_arrive: every thread of
// the block calls it after its writes.  grid_wait: every thread calls it;
// thread 0 takes the bounded wait of grid_sync.
__device__ __forceinline__ void grid_arrive(unsigned long long* ctr) {
  __syncthreads();
  if (threadIdx.x == 0)
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
}
__device__ __noinline__ bool grid_wait(unsigned long long* ctr, unsigned long long target,
                                       int* status, uint64_t limit_ns) {
  __shared__ int s_okw;
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint64_t t0 = global_ns();
    unsigned spins = 0;
    while ((long long)(ld_acquire64(ctr) - target) < 0) {
      if ((++spins & 15u) == 0u && global_ns() - t0 > limit_ns) {
        ok = 0;
        set_status(status, PI_ERR_TIMEOUT);
        break;
      }
    }
    s_okw = ok;
  }
  __syncthreads();
  return s_okw != 0;
}

// ------------------------------------------------------------------ TMA bulk copies
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* m, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible (returns at once if the
// launch has no programmatic dependency), and let the next kernel launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// First statement of a kernel in a launch chain: wait for the previous
// kernel in the stream (its writes visible), then let the next kernel launch
// (its blocks wait at their own first statement).  Without a programmatic
// launch attribute both return at once.
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// Barrier among the kThreads compute threads only (the producer warp keeps
// running its own loop).
__device__ __forceinline__ void compute_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous (TMA) proxy.
// Invalidates an mbarrier so that its memory may be initialised again (no
// arrival or transaction may be pending on it).
__device__ __forceinline__ void mbar_inval(uint64_t* m) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(m)) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* m) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* m, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)),
               "r"(bytes)
               : "memory");
}

// L2 eviction priority for data read once (streamed weight rows).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// One-dimensional bulk copy global -> shared (TMA unit), completing on `m`,
// with the source lines marked evict-first in L2 (streamed once).
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, unsigned bytes, uint64_t* m) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(m)), "l"(l2_evict_first())
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Non-blocking test of the phase of parity `parity`.
__device__ __forceinline__ bool mbar_test(uint64_t* m, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(m)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Waits for the phase of parity `parity` of `m` to complete; gives up after
// limit_ns and returns false.  The common case (already complete) costs one
// non-blocking test.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, unsigned parity, uint64_t limit_ns) {
  if (mbar_test(m, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(m, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

// The same for a thread that only waits (the producer warp): sleeps between
// polls so that it takes no issue slots from the compute warps.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* m, unsigned parity, uint64_t limit_ns) {
  if (mbar_test(m, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(m, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// Transposing butterfly reduction of NV values (NV a power of two, <= 32)
// held by each lane of a warp: on return every lane holds the warp-wide sum
// of value index bfly_index<NV>(lane).  NV - 1 + log2(32 / NV) shuffles
// instead of 5 NV.
template <int NV>
__device__ __forceinline__ float warp_bfly_sum(float (&v)[NV]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = NV / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = (32 / NV) / 2; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

template <int NV>
__device__ __forceinline__ int bfly_index(int lane) {
  int vi = 0;
#pragma unroll
  for (int half = NV / 2, off = 16; half >= 1; half >>= 1, off >>= 1)
    if (lane & off) vi += half;
  return vi;
}

}  // namespace pik

// tcd.cuh — the batched FFN over every neuron (dense) on the fifth-generation
// tensor cores, operands staged by TMA tensor copies.
//
//   phase 1  H[i][t] = act(W1[i] . x_t + b1[i])        for all n neurons
//   phase 2  Y_b[t][c] = sum_{i in block b's range} H[i][t] W2[i][c]
//   phase 3  y[t][c] = b2[c] + sum_b Y_b[t][c] (b ascending) (+ residual)
//
// Both contractions are D (fp32, tensor memory) += A x B with the
// activations' high and low 16-bit parts stacked as A's rows (x = hi + lo,
// H = hi + lo: row t < bp holds token t's high part, bp + t its low part,
// so the two products land in separate accumulator lanes and are added in
// the epilogue) and the weights as B, both in shared memory.
// Shared-memory tiles use the 128-byte swizzle: rows of 64 16-bit elements
// (128 bytes), 8-row atoms of 1024 bytes, 16-byte chunk c of row r stored at
// chunk c ^ (r % 8) (the pattern follows the shared-memory address, so atoms
// are 1024-byte aligned); TMA writes that form and the matrix descriptors
// read it.
//   phase 1: A = x, K-major (M = 128 rows, 2 bp of them loaded; K = 64
//            columns per stage); B = the block's W1 rows, K-major (N = its
//            rows rounded up to 16, <= 256).
//   phase 2: A = H^T, K-major (M = 128 rows, 2 bp loaded; K = 64 neurons
//            per work item); B = the tile's columns of the W2 rows, read
//            N-major (N = 256 output columns, or 128).
// Roles: warp 0 issues the TMA copies, warp 1 the MMAs (and owns tensor
// memory), warps 2-5 read the accumulators back.  The weight boxes of the
// first stages are issued before the wait for the previous kernel (the
// weights are not written by it); x and H^T after.  Every wait is bounded;
// a block that gives up records PI_ERR_TIMEOUT, lets its copies and MMAs
// finish (bounded) and frees its tensor memory before it exits.
#pragma once

#include <cuda.h>

#include "tc.cuh"

namespace pik {

constexpr int kTdThreads = 192;
constexpr int kTdMaxStages = 12;
constexpr int kTdHalf = 128 * 128;  // bytes of one 128-row x 64-column half tile
constexpr int kTdMaxTiles = 256;    // column tiles of phase 2 (d <= 32768)

struct TdArgs {
  int d, n, batch, bp;
  int P;             // blocks of every phase
  int wrows;         // phase 1: most rows of a block (a multiple of 8, <= 256): the height
                     // of each weight tile's region in a stage
  int ncol1;         // phase 1: accumulator columns per weight tile (wrows rounded up to 16)
  int ns1, ns2;      // pipeline stages of phase 1 / phase 2
  int stage1, stage2;  // bytes per stage (multiples of 1024)
  int tcols1, tcols2;  // tensor-memory columns (powers of 2, >= 32)
  int hs;            // row stride of H^T
  int nct, nkb;      // phase 2: column tiles (d / nc2), neuron blocks of 64 (n / 64)
  int nc2;           // phase 2: columns per tile (256, or 128 where d % 256 != 0)
  int w2x;           // column of W2 within the W2 tensor's rows (packed records: m1 d)
  const float* b1;
  const float* b2;
  const float* residual;  // [batch][d] or NULL
  float* y;               // [batch][d]
  uint16_t* hT;           // H^T [2 bp][hs]: high parts, then low parts
  float* part;            // phase 2 partials [P][2][bp][nc2]
  int* status;
  unsigned long long limit_ns, drain_ns;
  // phase 2's partition, from the host: the first and last block with work
  // items in column tile ct, and each block's first column tile
  uint16_t tile_b0[kTdMaxTiles], tile_b1[kTdMaxTiles], first_tile[kPMax];
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
}

// 2D tiled tensor copy global -> shared, completing on `bar`; `pol` an L2
// cache policy.  The box and swizzle are the tensor map's.
__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar,
                                      uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major: sbo = the
// distance of 8-row groups (1024), lbo unused.  M-major: lbo = the distance
// of 64-element groups along M, sbo = that of 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of this family
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B of DT (f16 0 /
// bf16 1), A K-major or M-major, B K-major, M = 128, N = nn.
__device__ __forceinline__ uint32_t td_idesc(int dt, int nn, bool a_mmajor) {
  return (1u << 4) | ((uint32_t)dt << 7) | ((uint32_t)dt << 10) | ((a_mmajor ? 1u : 0u) << 15) |
         ((uint32_t)(nn >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void td_ld8(uint32_t (&r)[8], uint32_t taddr) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// The producer's copies after a give-up: the last copy issued into each
// stage (issue count `it`) lands before the block exits; bounded.
__device__ __forceinline__ void td_drain(uint64_t* full, int ns, int it, unsigned long long ns_limit,
                                         int* status) {
  for (int s = 0; s < ns && s < it; ++s) {
    const int k = s + ((it - 1 - s) / ns) * ns;  // last issue into stage s
    if (!mbar_wait_sleep(full + s, (unsigned)((k / ns) & 1), ns_limit))
      set_status(status, PI_ERR_TIMEOUT);
  }
}
// The MMA thread's operations after a give-up complete before tensor memory
// is freed; bounded.
__device__ __forceinline__ void td_mma_drain(uint64_t* fin, unsigned long long ns_limit,
                                             int* status) {
  tc_commit(fin);
  if (!mbar_wait_sleep(fin, 0u, ns_limit)) set_status(status, PI_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- phase 1
// Block b owns neurons [row0, row0 + rows), rows = 8 (g1 - g0) <= 256 (the
// 8-row groups split evenly).  D[j][i] = sum_k x2[j][k] W1[row0 + i][k]:
// A = x's high and low parts (M = 128 rows, of which the first 2 bp are
// loaded: rows t < bp the high parts, bp + t the low parts; the others
// give unused accumulator lanes), B = the block's weight rows (N = rows
// rounded up to 16, K-major), one accumulator chain of 4 MMAs per weight
// tile and stage.  Weight boxes of 128, 32 and 8 rows (three tensor maps
// over the W1 rows) cover the rows exactly.  Stage layout: x's region of
// 128 rows (16 KB), then NW weight regions of wrows rows (128 bytes each);
// the last B read may run up to 8 rows past its region (the guard after
// the last stage).  Epilogue: the warps owning accumulator lanes [0, 2 bp)
// copy them to shared memory (the stages, free by then), then all four
// add high and low parts, bias, activation, and store H^T.
template <int DT, bool GATED>
__global__ void __launch_bounds__(kTdThreads, 1)
    td_up_kernel(const __grid_constant__ TdArgs a, const __grid_constant__ CUtensorMap mw128,
                 const __grid_constant__ CUtensorMap mw32, const __grid_constant__ CUtensorMap mw8,
                 const __grid_constant__ CUtensorMap mx) {
  constexpr int NW = GATED ? 2 : 1;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  __shared__ __align__(8) uint64_t full[kTdMaxStages], empty[kTdMaxStages], accf, fin;
  __shared__ uint32_t s_taddr;
  __shared__ int s_bad, s_it;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ng = a.n >> 3;
  const int g0 = (int)((long long)blockIdx.x * ng / a.P);
  const int g1 = (int)((long long)(blockIdx.x + 1) * ng / a.P);
  const int row0 = 8 * g0, rows = 8 * (g1 - g0);
  const int nn = (rows + 15) & ~15;  // the MMA's N
  const int nkb = a.d >> 6;
  const int ns = a.ns1;
  const int bp2 = 2 * a.bp;
  const int nc = a.ncol1;  // accumulator columns per weight tile

  if (warp == 1) tmem_alloc(&s_taddr, (uint32_t)a.tcols1);
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full + s, 1u);
      mbar_init(empty + s, 1u);
    }
    mbar_init(&accf, 1u);
    mbar_init(&fin, 1u);
    fence_mbar_init();
    s_bad = 0;
    s_it = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = s_taddr;
  volatile int* vbad = &s_bad;

  // the weight boxes of the first stages: the weights are not written by
  // the kernels before this one, so they load while those finish
  const uint64_t pw = l2_evict_first(), px = l2_evict_last();
  const unsigned tx = (unsigned)(NW * rows * 128 + bp2 * 128);
  auto issue_w = [&](int it, int s) {
    unsigned char* st = sm + (size_t)s * a.stage1;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      unsigned char* wt = st + kTdHalf + (size_t)w * a.wrows * 128;
      const int xc = w * a.d + it * 64;
      int r = 0;
      while (r < rows) {
        const int rem = rows - r;
        const CUtensorMap* m = rem >= 128 ? &mw128 : (rem >= 32 ? &mw32 : &mw8);
        const int h = rem >= 128 ? 128 : (rem >= 32 ? 32 : 8);
        tma2d(wt + (size_t)r * 128, m, xc, row0 + r, full + s, pw);
        r += h;
      }
    }
  };
  const int npre = rows > 0 ? min(ns, nkb) : 0;
  if (tid == 0)
    for (int it = 0; it < npre; ++it) {
      mbar_expect_tx(full + it, tx);  // the stage's x box comes after the wait below
      issue_w(it, it);
    }
  pdl_enter();  // the previous kernel's results (x's high / low parts) are visible from here

  if (rows > 0) {
    if (warp == 0) {
      if (lane == 0) {  // TMA producer
        for (int it = 0; it < npre; ++it) tma2d(sm + (size_t)it * a.stage1, &mx, it * 64, 0, full + it, px);
        int it = npre;
        for (; it < nkb; ++it) {
          const int s = it % ns;
          if (it >= ns &&
              !mbar_wait_sleep(empty + s, (unsigned)(((it / ns) - 1) & 1), a.limit_ns)) {
            set_status(a.status, PI_ERR_TIMEOUT);
            *vbad = 1;
            break;
          }
          unsigned char* st = sm + (size_t)s * a.stage1;
          mbar_expect_tx(full + s, tx);
          tma2d(st, &mx, it * 64, 0, full + s, px);
          issue_w(it, s);
        }
        s_it = it;
      }
    } else if (warp == 1) {
      if (lane == 0) {  // MMA issuer
        const uint32_t idesc = td_idesc(DT, nn, false);
        bool ok = true;
        for (int it = 0; it < nkb; ++it) {
          const int s = it % ns;
          if (!mbar_wait(full + s, (unsigned)((it / ns) & 1), a.limit_ns)) {
            set_status(a.status, PI_ERR_TIMEOUT);
            *vbad = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sm + (size_t)s * a.stage1);
#pragma unroll
          for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)  // one chain per accumulator: consecutive MMAs
              tc_mma(taddr + (uint32_t)(w * nc), sw128_desc(sa + 32u * ks, 16u, 1024u),
                     sw128_desc(sa + (uint32_t)(kTdHalf + w * a.wrows * 128) + 32u * ks, 16u, 1024u),
                     idesc, (it > 0 || ks > 0) ? 1u : 0u);
          tc_commit(empty + s);  // the stage is free once these MMAs completed
        }
        if (ok) tc_commit(&accf);  // the accumulators are complete
      }
    } else {  // epilogue: warps 2..5, tensor-memory lane quarter warp % 4
      const int q = warp & 3;
      const int et = tid - 64;  // 0..127
      float* E = reinterpret_cast<float*>(sm);  // [NW][2 bp][nn + 4]
      const int ep = nn + 4;
      bool ok = mbar_wait(&accf, 0u, a.limit_ns);
      if (!ok) {
        set_status(a.status, PI_ERR_TIMEOUT);
        *vbad = 1;
      }
      tc_fence_after();
      if (ok && 32 * q < bp2) {
        const uint32_t lanebase = taddr + ((uint32_t)(q * 32) << 16);
        const int j = 32 * q + lane;  // accumulator row = x row
#pragma unroll
        for (int w = 0; w < NW; ++w)
          for (int c0 = 0; c0 < nn; c0 += 8) {
            uint32_t v[8];
            td_ld8(v, lanebase + (uint32_t)(w * nc + c0));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float* dst = E + ((size_t)w * bp2 + j) * ep + c0;
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = __uint_as_float(v[e]);
          }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
      if (ok) {
        for (int e = et; e < a.batch * rows; e += 128) {
          const int t = e / rows, i = e - t * rows;
          float hv = E[(size_t)t * ep + i] + E[(size_t)(a.bp + t) * ep + i] + __ldg(a.b1 + row0 + i);
          hv = hv > 0.f ? hv : 0.f;  // ReLU; ReLU(0) = 0
          if (GATED)
            hv *= E[((size_t)bp2 + t) * ep + i] + E[((size_t)bp2 + a.bp + t) * ep + i];
          uint16_t hh, hl;
          split16<DT>(hv, &hh, &hl);
          a.hT[(size_t)t * a.hs + row0 + i] = hh;
          a.hT[(size_t)(a.bp + t) * a.hs + row0 + i] = hl;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_bad) {  // block-uniform after the barrier
    if (tid == 0) td_drain(full, ns, s_it, a.drain_ns, a.status);
    if (tid == 32) td_mma_drain(&fin, a.drain_ns, a.status);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_free(taddr, (uint32_t)a.tcols1);
  }
}

// ---------------------------------------------------------------- phase 2
// Work items f = ct nkb + kb (column tile ct of nc2 = 256 or 128 outputs,
// block kb of 64 neurons) split evenly over the blocks: block b takes
// [b F / P, (b+1) F / P) and, as nct <= P, touches at most two column tiles
// (segments 0 and 1, accumulated in tensor-memory columns [seg nc2, seg nc2
// + nc2)).  D[j][c] = sum_i H2[j][i] W2[i][ct nc2 + c]: A = H^T's high and
// low parts (M = 128 rows, the first 2 bp loaded), B = the tile's columns
// of the block's W2 rows, N-major (nc2 / 64 boxes of 64 columns x 64 rows,
// lbo the distance of the boxes), one chain of four MMAs per item.  Stage
// layout: H^T's box region (16 KB), then the W2 boxes (8 KB each).
// Epilogue per segment: accumulator lanes t < bp hold the high parts' sums
// and bp + t the low parts' (batch <= 16: one warp, added by shuffle;
// batch 32: the low lanes' warp stages them in shared memory); the block
// writes its partial of the column tile.
__device__ __forceinline__ long long td_start(int b, long long F, int P) { return (long long)b * F / P; }

template <int DT>
__global__ void __launch_bounds__(kTdThreads, 1)
    td_down_kernel(const __grid_constant__ TdArgs a, const __grid_constant__ CUtensorMap mw2,
                   const __grid_constant__ CUtensorMap mh) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  __shared__ __align__(8) uint64_t full[kTdMaxStages], empty[kTdMaxStages], accf[2], fin;
  __shared__ uint32_t s_taddr;
  __shared__ int s_bad, s_it, s_efail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long F = (long long)a.nct * a.nkb;
  const int f0 = (int)td_start(blockIdx.x, F, a.P), f1 = (int)td_start(blockIdx.x + 1, F, a.P);
  const int ct0 = f0 / a.nkb;
  const int nseg = (f1 > f0) ? ((f1 - 1) / a.nkb - ct0 + 1) : 0;  // 1 or 2
  const int ns = a.ns2;
  const int bp2 = 2 * a.bp;
  const int nc2 = a.nc2, nbox = a.nc2 >> 6;
  constexpr int kW2Box = 64 * 128;  // 64 neuron rows x 64 columns
  float* X = reinterpret_cast<float*>(sm + (size_t)ns * a.stage2);  // [32][nc2 + 4] (batch 32)
  const int xp = nc2 + 4;

  if (warp == 1) tmem_alloc(&s_taddr, (uint32_t)a.tcols2);
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full + s, 1u);
      mbar_init(empty + s, 1u);
    }
    mbar_init(accf, 1u);
    mbar_init(accf + 1, 1u);
    mbar_init(&fin, 1u);
    fence_mbar_init();
    s_bad = 0;
    s_it = 0;
    s_efail = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = s_taddr;
  volatile int* vbad = &s_bad;

  // the W2 boxes of the first items: the weights are not written by the
  // kernels before this one, so they load while those finish
  const uint64_t pw = l2_evict_first(), ph = l2_evict_last();
  const unsigned tx = (unsigned)(nbox * kW2Box + bp2 * 128);
  const int npre = min(ns, f1 - f0);
  if (tid == 0)
    for (int it = 0; it < npre; ++it) {
      const int f = f0 + it, ct = f / a.nkb, kb = f - ct * a.nkb;
      unsigned char* st = sm + (size_t)it * a.stage2;
      mbar_expect_tx(full + it, tx);  // the item's H^T box comes after the wait below
      for (int g = 0; g < nbox; ++g)
        tma2d(st + kTdHalf + g * kW2Box, &mw2, a.w2x + ct * nc2 + 64 * g, kb * 64, full + it, pw);
    }
  pdl_enter();  // phase 1's H^T is visible from here

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      for (int it = 0; it < npre; ++it) {
        const int f = f0 + it, kb = f - (f / a.nkb) * a.nkb;
        tma2d(sm + (size_t)it * a.stage2, &mh, kb * 64, 0, full + it, ph);
      }
      int it = npre;
      for (int f = f0 + npre; f < f1; ++f, ++it) {
        const int s = it % ns;
        if (it >= ns && !mbar_wait_sleep(empty + s, (unsigned)(((it / ns) - 1) & 1), a.limit_ns)) {
          set_status(a.status, PI_ERR_TIMEOUT);
          *vbad = 1;
          break;
        }
        const int ct = f / a.nkb, kb = f - ct * a.nkb;
        unsigned char* st = sm + (size_t)s * a.stage2;
        mbar_expect_tx(full + s, tx);
        tma2d(st, &mh, kb * 64, 0, full + s, ph);
        for (int g = 0; g < nbox; ++g)
          tma2d(st + kTdHalf + g * kW2Box, &mw2, a.w2x + ct * nc2 + 64 * g, kb * 64, full + s, pw);
      }
      s_it = it;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      // A K-major, B N-major (transposed), M = 128, N = nc2
      const uint32_t idesc = td_idesc(DT, nc2, false) | (1u << 16);
      int it = 0;
      for (int f = f0; f < f1; ++f, ++it) {
        const int s = it % ns;
        if (!mbar_wait(full + s, (unsigned)((it / ns) & 1), a.limit_ns)) {
          set_status(a.status, PI_ERR_TIMEOUT);
          *vbad = 1;
          break;
        }
        tc_fence_after();
        const int ct = f / a.nkb;
        const int seg = ct - ct0;
        const bool first = (f == f0) || (f == ct * a.nkb);
        const uint32_t sa = smem_u32(sm + (size_t)s * a.stage2);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(taddr + (uint32_t)(seg * nc2), sw128_desc(sa + 32u * ks, 16u, 1024u),
                 sw128_desc(sa + (uint32_t)kTdHalf + 2048u * ks, (uint32_t)kW2Box, 1024u), idesc,
                 (!first || ks > 0) ? 1u : 0u);
        tc_commit(empty + s);
        if (f + 1 == f1 || (f + 1) % a.nkb == 0) tc_commit(accf + seg);  // segment complete
      }
    }
  } else {  // epilogue: warps 2..5; accumulator lanes 0..63 are warps 4 and 5's
    const int q = warp & 3;
    const uint32_t lanebase = taddr + ((uint32_t)(q * 32) << 16);
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait(accf + seg, 0u, a.limit_ns)) {
        set_status(a.status, PI_ERR_TIMEOUT);
        *vbad = 1;
        s_efail = 1;  // written by epilogue threads only, before the barrier
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (s_efail) break;  // uniform over the four epilogue warps
      tc_fence_after();
      const uint32_t col0 = (uint32_t)(seg * nc2);
      float* prow = a.part + ((size_t)blockIdx.x * 2 + seg) * a.bp * nc2;  // [bp][nc2]
      if (a.bp == 16) {
        if (q == 0) {  // lanes 0..15: high parts, 16..31: low parts
          for (int c0 = 0; c0 < nc2; c0 += 8) {
            uint32_t v[8];
            td_ld8(v, lanebase + col0 + (uint32_t)c0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = __uint_as_float(v[e]) + __shfl_down_sync(0xffffffffu, __uint_as_float(v[e]), 16);
            if (lane < a.batch) {
              float4* dst = reinterpret_cast<float4*>(prow + (size_t)lane * nc2 + c0);
              __stcg(dst, make_float4(o[0], o[1], o[2], o[3]));
              __stcg(dst + 1, make_float4(o[4], o[5], o[6], o[7]));
            }
          }
        }
      } else {  // bp == 32: warp 5 (lanes 32..63, low parts) stages, warp 4 adds
        if (q == 1) {
          for (int c0 = 0; c0 < nc2; c0 += 8) {
            uint32_t v[8];
            td_ld8(v, lanebase + col0 + (uint32_t)c0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            float* xr = X + (size_t)lane * xp + c0;
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[e] = __uint_as_float(v[e]);
          }
        }
        if (q < 2) asm volatile("bar.sync 2, 64;" ::: "memory");  // warps 4 and 5 only
        if (q == 0) {
          for (int c0 = 0; c0 < nc2; c0 += 8) {
            uint32_t v[8];
            td_ld8(v, lanebase + col0 + (uint32_t)c0);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const float* xr = X + (size_t)lane * xp + c0;
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(v[e]) + xr[e];
            if (lane < a.batch) {
              float4* dst = reinterpret_cast<float4*>(prow + (size_t)lane * nc2 + c0);
              __stcg(dst, make_float4(o[0], o[1], o[2], o[3]));
              __stcg(dst + 1, make_float4(o[4], o[5], o[6], o[7]));
            }
          }
        }
      }
      // X is read by warp 4 before warp 5 stages the next segment
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_bad) {
    if (tid == 0) td_drain(full, ns, s_it, a.drain_ns, a.status);
    if (tid == 32) td_mma_drain(&fin, a.drain_ns, a.status);
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_free(taddr, (uint32_t)a.tcols2);
  }
}

// ---------------------------------------------------------------- phase 3
// y[t][c] = b2[c] + the partials of the blocks with work items in column
// tile ct = c / nc2, in block order (the host's table), + residual.  Block j
// takes tile j % nct and its outputs e = (j / nct) 256 + thread, ...
__global__ void __launch_bounds__(256) td_sum_kernel(const __grid_constant__ TdArgs a) {
  pdl_enter();
  const int ct = blockIdx.x % a.nct, g = blockIdx.x / a.nct, ng = gridDim.x / a.nct;
  const int b0 = a.tile_b0[ct], b1 = a.tile_b1[ct];
  const int nc2 = a.nc2, q4 = nc2 >> 2, tot = a.batch * q4;  // four columns per thread
  for (int e = g * 256 + (int)threadIdx.x; e < tot; e += ng * 256) {
    const int t = e / q4, cl = 4 * (e - t * q4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int b = b0; b <= b1; ++b) {  // (unrolled: the partials' loads go out together)
      const float4 v = __ldcg(reinterpret_cast<const float4*>(
          a.part + (((size_t)b * 2 + (ct - a.first_tile[b])) * a.bp + t) * nc2 + cl));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    const int c = ct * nc2 + cl;
    if (a.b2) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(a.b2 + c));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    const size_t o = (size_t)t * a.d + c;
    if (a.residual) {
      const float4 v = *reinterpret_cast<const float4*>(a.residual + o);
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    *reinterpret_cast<float4*>(a.y + o) = s;
  }
}

}  // namespace pik

// tc.cuh — batched phase 1 on the fifth-generation tensor cores (tcgen05).
//
//   H[u][t] = mask_t(u) ? act(W1[U_u] . x_t + b1) : 0
//
// for a tile of 128 MH union positions (the MMA's M, in MH halves of 128)
// and all tokens (N = bp, 16 or 32).  Operands are staged by cp.async in
// shared memory in the tensor cores' K-major core-matrix layout (8 rows x
// 16 bytes per core matrix; core matrices adjacent in K are LBO = 128 bytes
// apart, 8-row groups SBO = 16 BK bytes apart for BK-column chunks).  One
// thread issues tcgen05.mma (kind::f16, fp32 accumulation in tensor memory)
// for each chunk and commits it to the chunk's stage mbarrier; a stage is
// refilled only after its MMAs completed.  x enters as its high and low
// 16-bit parts, both products accumulate in the same tensor-memory columns.
// The epilogue reads the accumulators back with tcgen05.ld: warp w takes
// lanes 32 (w % 4) .. + 31 (its lane quarter) and the column group w / 4.
#pragma once

#include "batched.cuh"

namespace pik {

constexpr int kTcStages = 4;  // pipeline depth
// columns per chunk: 128 for plain layers, 64 for gated ones (two weight tiles)
template <bool GATED>
__host__ __device__ constexpr int tc_bk() {
  return GATED ? 64 : 128;
}
// bytes of one stage: NW weight tiles of 128 MH rows, x high and low parts of bp rows
template <bool GATED, int MH>
__host__ __device__ constexpr int tc_stage_bytes(int bp) {
  return ((GATED ? 2 : 1) * 128 * MH + 2 * bp) * tc_bk<GATED>() * 2;
}

// K-major, no swizzle: core matrices adjacent in K are 128 bytes apart
// (LBO), 8-row groups sbo bytes apart (SBO: one row group's whole chunk)
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((128u >> 4) & 0x3FFF) << 16;  // LBO
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;   // SBO
  d |= (uint64_t)1 << 46;                       // descriptor version of this family
  return d;                                     // no swizzle, base offset 0
}

__device__ __forceinline__ void tc_mma(uint32_t dtm, uint64_t da, uint64_t db, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(dtm),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint64_t* mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(mbar))
      : "memory");
}

__device__ __forceinline__ void tc_ld4(uint32_t (&r)[4], uint32_t taddr) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}

template <int DT, bool GATED, int MH>
__global__ void __launch_bounds__(512, 1) bup_tc_kernel(const BatchArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint32_t s_taddr;
  __shared__ __align__(8) uint64_t s_mbar[kTcStages];
  __shared__ int s_bad;
  constexpr int NW = GATED ? 2 : 1;
  constexpr int S = kTcStages;
  constexpr int T = 128 * MH;  // union positions per tile
  constexpr int BK = tc_bk<GATED>();
  constexpr int PCS = BK / 8;               // 16-byte pieces (core-matrix columns) per row
  constexpr int kTcSBO = 8 * BK * 2;        // bytes of one 8-row group's chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bp = a.bp;
  const int U = a.dense ? a.n : __ldg(a.ucnt);
  const int lo_u = (int)((long long)blockIdx.x * U / a.P);
  const int hi_u = (int)((long long)(blockIdx.x + 1) * U / a.P);
  const int stage_bytes = tc_stage_bytes<GATED, MH>(bp);
  const int nchunks = a.d / BK;
  const size_t w1s = a.packed ? (size_t)a.rec : (GATED ? 2 * (size_t)a.d : (size_t)a.d);
  const uint32_t ncols = (uint32_t)a.tc_cols;  // tensor-memory columns: MH NW bp, power of 2 >= 32

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_taddr)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(s_mbar + s, 1u);
    fence_mbar_init();
    s_bad = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t taddr = s_taddr;
  // D f32, A and B of DT (f16 0 / bf16 1), both K-major, N = bp, M = 128
  const uint32_t idesc = (1u << 4) | ((uint32_t)DT << 7) | ((uint32_t)DT << 10) |
                         ((uint32_t)(bp >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  unsigned phase = 0u;  // bit s: parity of the next completion of stage s

  // waits for the MMAs of chunk c (stage c % S), bounded; a thread that
  // gives up records it in s_bad, read by all after the next barrier
  auto wait_chunk = [&](int c) {
    const int s = c % S;
    if (!s_bad && !mbar_wait(s_mbar + s, (phase >> s) & 1u, a.limit_ns)) {
      s_bad = 1;
      set_status(a.status, PI_ERR_TIMEOUT);
    }
    phase ^= 1u << s;
  };

  for (int t0 = lo_u; t0 < hi_u; t0 += T) {
    const int tn = min(T, hi_u - t0);
    auto issue = [&](int ch) {
      unsigned char* st = smem + (ch % S) * stage_bytes;
      const int k0 = ch * BK;
      for (int e = tid; e < NW * T * PCS; e += 512) {
        const int rw = e / PCS, pc = e - rw * PCS;
        const int w = rw / T, row = rw - w * T;
        unsigned char* dst = st + (size_t)w * (T / 8) * kTcSBO + (row >> 3) * kTcSBO + pc * 16 * 8 +
                             (row & 7) * 16;
        if (row < tn) {
          const int nid = a.dense ? t0 + row : __ldg(a.uidx + t0 + row);
          cp_async16(dst, a.W1 + (size_t)nid * w1s + (size_t)w * a.d + k0 + 8 * pc);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      unsigned char* xs = st + (size_t)NW * (T / 8) * kTcSBO;
      for (int e = tid; e < 2 * bp * PCS; e += 512) {
        const int rw = e / PCS, pc = e - rw * PCS;
        const int prt = rw / bp, t = rw - prt * bp;
        unsigned char* dst = xs + (size_t)prt * (bp / 8) * kTcSBO + (t >> 3) * kTcSBO + pc * 16 * 8 +
                             (t & 7) * 16;
        cp_async16(dst, (prt == 0 ? a.xhi : a.xlo) + (size_t)t * a.d + k0 + 8 * pc);
      }
    };
    for (int ch = 0; ch < S - 1; ++ch) {  // always S - 1 groups
      if (ch < nchunks) issue(ch);
      cp_async_commit();
    }
    for (int ch = 0; ch < nchunks; ++ch) {
      // chunk ch's copies landed (S - 1 groups went out ahead of it)
      asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncthreads();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (tid == 0 && !s_bad) {
        const unsigned char* st = smem + (ch % S) * stage_bytes;
        const uint32_t sa = smem_u32(st);
        const uint32_t sx = sa + (uint32_t)(NW * (T / 8) * kTcSBO);
        const uint32_t sxl = sx + (uint32_t)((bp / 8) * kTcSBO);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {  // 16 columns = two core matrices
          const uint32_t ko = (uint32_t)(ks * 2 * 128);
          const uint64_t dh = tc_desc(sx + ko, kTcSBO), dl = tc_desc(sxl + ko, kTcSBO);
#pragma unroll
          for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              const uint64_t dw =
                  tc_desc(sa + (uint32_t)(w * (T / 8) * kTcSBO + h * 16 * kTcSBO) + ko, kTcSBO);
              const uint32_t dtm = taddr + (uint32_t)((h * NW + w) * bp);  // columns of (h, w)
              tc_mma(dtm, dw, dh, idesc, (ch > 0 || ks > 0) ? 1u : 0u);
              tc_mma(dtm, dw, dl, idesc, 1u);
            }
        }
        tc_commit(s_mbar + ch % S);
      }
      // the previous chunk's MMAs ran while this chunk's copies were awaited;
      // once they are done, their stage takes chunk ch + S - 1
      if (ch >= 1) wait_chunk(ch - 1);
      if (ch + S - 1 < nchunks) issue(ch + S - 1);
      cp_async_commit();
    }
    wait_chunk(nchunks - 1);  // the tile's accumulators are complete
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // epilogue: bias, activation, the token's own mask bit, split, store H^T
    if (!s_bad) {  // block-uniform
      const int q = warp & 3, cg = warp >> 2;  // lane quarter, column group
      const int cw = bp / 4;                  // columns (tokens) per group: 4 or 8
#pragma unroll
      for (int h = 0; h < MH; ++h) {
        const int col = h * 128 + q * 32 + lane;  // position within the tile
        const bool valid = col < tn;
        const int pos = t0 + col;
        const int nid = valid ? (a.dense ? pos : __ldg(a.uidx + pos)) : 0;
        const float bias = valid ? __ldg(a.b1 + nid) : 0.f;
        const uint32_t tm = valid ? (a.dense ? 0xffffffffu : __ldg(a.tmask + pos)) : 0u;
        for (int c4 = 0; c4 < cw; c4 += 4) {
          const int tok0 = cg * cw + c4;
          uint32_t rg[4], ru[4];
          const uint32_t lanebase = taddr + ((uint32_t)(q * 32) << 16);
          tc_ld4(rg, lanebase + (uint32_t)((h * NW) * bp + tok0));
          if (GATED) tc_ld4(ru, lanebase + (uint32_t)((h * NW + 1) * bp + tok0));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = tok0 + i;
            if (valid && t < a.batch) {
              float hv = __uint_as_float(rg[i]) + bias;
              hv = hv > 0.f ? hv : 0.f;  // ReLU; ReLU(0) = 0
              if (GATED) hv *= __uint_as_float(ru[i]);
              if (!((tm >> t) & 1u)) hv = 0.f;  // token t skips this neuron
              uint16_t hh, hl;
              split16<DT>(hv, &hh, &hl);
              a.hhi[(size_t)t * a.hs + pos] = hh;
              a.hlo[(size_t)t * a.hs + pos] = hl;
            }
          }
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();  // accumulators read before the next tile overwrites them
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (s_bad) break;  // block-uniform
  }
  cp_async_wait_all();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

}  // namespace pik

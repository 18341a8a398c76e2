// kernels.cuh — CUDA kernels of libpi (sm_103a).
//
// Method: "PowerInfer: Quick Massive Language Mannequin Serving with a
// Client-grade GPU".  The online engine predicts the activated FFN neurons
// and skips the rest ("Online Section"); the neuron-aware operator reads only
// the activated neurons' rows of W1 and column vectors of W2 straight from
// the stored matrices ("Neuron Conscious Operator"); hot neurons sit first
// ("Offline Section"), so the hot block is a contiguous prefix that can be
// fetched before the mask is known.
#pragma once

#include "common.cuh"

namespace pik {

enum Mode { kFused = 0, kSparse = 1, kDense = 2 };

constexpr int kGroup = 4;        // neurons per round
constexpr int kMaxSlots = 16;    // TMA ring slots

struct FfnArgs {
  int d, n, r;
  int S;           // predictor row split (fused path)
  int P;           // grid size (all blocks co-resident)
  int hot;         // hot-prefix length
  int nch;         // d / 8: 16-byte column chunks of a row
  int rows_max;    // most neurons a block lists (own neurons, or list positions)
  int a_in_smem;   // fused: own predictor rows staged in shared memory (else read via L2)
  int a_stride;    // bytes between staged predictor rows (2 r + 16: conflict-free reads)
  int ns;          // ring slots (one neuron's W1 row(s) + W2 row each)
  int nh;          // fused: slots [0, nh) take the block's own hot neurons up front
  int grp;         // neurons per round: 1, 2 or kGroup, <= ns - nh
  int slot_bytes;
  int packed;      // PI_LAYOUT_PACKED: W1 holds [n][m d] per-neuron records
  // dynamic shared-memory offsets (bytes)
  int o_xs, o_us, o_As, o_b1s, o_flag, o_lst, o_lb, o_off, o_red, o_mbar, o_slots;  // o_off unused
  const uint16_t* A;
  const uint16_t* Bm;
  const float* b1;
  const uint16_t* W1;
  const uint16_t* W2;
  const float* b2;
  const float* x;
  const float* residual;
  float* y;
  const int* idx_in;
  const int* cnt_in;
  int cap;
  int* idx_out;
  int* cnt_out;
  int* status;
  unsigned long long* bar;  // grid barrier arrival counter
  float* upart;             // [r * S]
  int* loc_tot;             // [P] active count of each block's own neurons
  unsigned char* mask;      // [n] predicted mask (only when idx_out is wanted)
  float* part;              // [P][d]
  unsigned long long limit_ns;  // bound of every protocol wait (grid barriers, ring slots)
  unsigned long long drain_ns;  // bound of the wait for copies already issued to land
  int skip_issue;               // failure-path self-test only: 1 + the cold entry that the
                                // producer of every block leaves unissued (0: none)
};

// ------------------------------------------------------------ async copies
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(sdst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(void* sdst, const void* gsrc) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(sdst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (TMA unit; no completion to wait on).
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned long long bytes) {
  const char* c = static_cast<const char*>(p);
  while (bytes > 0) {
    const unsigned chunk = bytes > (1u << 20) ? (1u << 20) : (unsigned)bytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(chunk) : "memory");
    c += chunk;
    bytes -= chunk;
  }
}

__device__ __forceinline__ float dot8(const float f[8], const float x[8]) {
  float s = f[0] * x[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) s = fmaf(f[e], x[e], s);
  return s;
}

__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Arms ring slot `slot` with neuron `i`: its W1 row (gated: gate and up rows)
// and its W2 row, by bulk copies completing on the slot's "full" mbarrier.
// A slot holds [W1 part | W2 part], the byte layout of a packed record, so a
// packed layer needs one copy per neuron, a split one two.
template <bool GATED>
__device__ __forceinline__ void issue_neuron(const FfnArgs& a, unsigned char* slots, uint64_t* full,
                                             int slot, int i) {
  unsigned char* dst = slots + (size_t)slot * a.slot_bytes;
  mbar_expect_tx(full + slot, (unsigned)a.slot_bytes);
  if (a.packed) {
    bulk_g2s(dst, reinterpret_cast<const unsigned char*>(a.W1) + (size_t)i * a.slot_bytes,
             (unsigned)a.slot_bytes, full + slot);
  } else {
    const unsigned w1b = (GATED ? 4u : 2u) * (unsigned)a.d;
    const size_t rs = GATED ? 2 * (size_t)a.d : (size_t)a.d;
    bulk_g2s(dst, a.W1 + (size_t)i * rs, w1b, full + slot);
    bulk_g2s(dst + w1b, a.W2 + (size_t)i * a.d, 2u * (unsigned)a.d, full + slot);
  }
}

// Asks L2 to fetch neuron i's rows (no completion; used for hot neurons
// that do not fit the ring).
template <bool GATED>
__device__ __forceinline__ void prefetch_neuron(const FfnArgs& a, int i) {
  if (a.packed) {
    prefetch_l2(reinterpret_cast<const unsigned char*>(a.W1) + (size_t)i * a.slot_bytes,
                (unsigned long long)a.slot_bytes);
  } else {
    const size_t rs = GATED ? 2 * (size_t)a.d : (size_t)a.d;
    prefetch_l2(a.W1 + (size_t)i * rs, rs * 2);
    prefetch_l2(a.W2 + (size_t)i * a.d, (size_t)a.d * 2);
  }
}

// ------------------------------------------------------------ predictor (fused)
// Logits of this block's own neurons i = c + j P (j < rows); flag[j] =
// (logit > 0).  A row's r/8 sixteen-byte pieces go to lpr lanes (the next
// power of two), lane l holding piece l % lpr of u in registers for the whole
// pass; a warp covers 32 / lpr rows per load, four loads in flight per lane;
// each row's lpr partial dot products meet in a fixed xor tree.  Rows come
// from shared memory (staged) or through L2.
template <int DT>
__device__ __forceinline__ void own_logits(const FfnArgs& a, const unsigned char* As,
                                           const float* b1s, const float* us,
                                           unsigned char* flag, int rows) {
  const int rc = a.r >> 3;
  const bool in_smem = a.a_in_smem != 0;
  const int stride = a.a_stride, P = a.P, r = a.r;
  const uint16_t* Ag = a.A;
  const int c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int lpr = 1;
  while (lpr < rc) lpr <<= 1;  // <= 32 (r <= 256)
  const int rpw = 32 / lpr;     // rows per warp and load
  const int q = lane & (lpr - 1), sub = lane / lpr;
  const bool qok = q < rc;
  float u[8];
  if (qok) {
    load8(us + 8 * q, u);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = 0.f;
  }
  constexpr int RU = 4;          // rows per lane per pass
  const int step = kWarps * rpw;  // rows between a lane's consecutive loads
  for (int jb = warp * rpw; jb < rows; jb += step * RU) {  // warp-uniform bound
    uint4 v[RU];
#pragma unroll
    for (int t = 0; t < RU; ++t) {
      const int jr = jb + sub + t * step;
      v[t] = make_uint4(0u, 0u, 0u, 0u);
      if (qok && jr < rows) {
        if (in_smem)
          v[t] = *reinterpret_cast<const uint4*>(As + (size_t)jr * stride + 16 * q);
        else
          v[t] = ld_nc(Ag + ((size_t)c + (size_t)jr * P) * r + 8 * q);
      }
    }
    float acc[RU];
#pragma unroll
    for (int t = 0; t < RU; ++t) {
      float f[8];
      unpack8<DT>(v[t], f);
      acc[t] = dot8(f, u);
    }
    for (int o = lpr >> 1; o >= 1; o >>= 1)
#pragma unroll
      for (int t = 0; t < RU; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    if (q == 0) {
#pragma unroll
      for (int t = 0; t < RU; ++t) {
        const int jr = jb + sub + t * step;
        if (jr < rows) flag[jr] = (acc[t] + b1s[jr] > 0.f) ? 1 : 0;
      }
    }
  }
}

// ------------------------------------------------------------ FFN over a neuron list
// Row-gather GEMV + ReLU and row-axpy over the m neurons of lst (x: the
// token's d activations, in shared or global memory).  Rows reach
// shared memory by TMA bulk copies.  Entries [0, mh) are the block's own hot
// neurons, armed up front into slots (lst[k] - c) / P; the other entries
// cycle through slots [nh, ns), armed by the producer warp as soon as the
// compute warps release a slot ("empty" mbarrier, one arrival per compute
// warp).  Compute thread t owns the 16-byte column chunks t, t + kThreads,
// ... of every row and keeps x of those columns in registers.  Work goes in
// rounds of up to kGroup neurons:
//   A. each thread dots its chunks of the round's W1 rows with x (two fp32
//      FMA chains per value); one transposing butterfly per warp reduces all
//      of them; warp partials go to shared memory (double-buffered by round);
//   B. eight lanes of warp 0 add the kWarps partials in order, add the bias
//      and apply ReLU (times the up projection, gated);
//   C. each thread adds h_q times its chunks of the round's W2 rows.
// Every sum has a fixed order, so results are deterministic.  A round holds
// a.grp <= kGroup neurons; a.grp <= ns - nh (no round waits for a slot that
// only its own release would free), and a shallow ring takes smaller rounds
// so that copies stay in flight while a round is computed.  lb[k] is b1 of
// neuron lst[k]; red holds 2 x kGroup x NV x kWarps floats, hbuf 2 x kGroup.
// After the ring was abandoned (s_bad): the producer's last copy into each
// cold slot (iss[0]: slots with a copy, iss[1]: the parity of its phase)
// lands before the slots are re-armed or the block exits; bounded by
// drain_ns.  Not needed on the normal path, where the compute warps waited
// for every copy issued.
__device__ __forceinline__ void ring_drain(uint64_t* full, int nh, int nc, const unsigned* iss,
                                           unsigned long long drain_ns, int* status) {
  const unsigned issued = iss[0], par = iss[1];
  for (int q = 0; q < nc; ++q)
    if (((issued >> q) & 1u) && !mbar_wait_sleep(full + nh + q, (par >> q) & 1u, drain_ns))
      set_status(status, PI_ERR_TIMEOUT);
}

template <int DT, bool GATED, int NCH>
__device__ void ffn_ring(const FfnArgs& a, const float* xs, const int* lst, const float* lb, int m,
                         int mh, int nh, unsigned char* slots, uint64_t* full, uint64_t* empty,
                         float* red, float* hbuf, float (&yacc)[NCH][8], int* bad,
                         unsigned* iss) {
  constexpr int NV = GATED ? 2 : 1;
  constexpr int NR = kGroup * NV;  // values reduced per round
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  const int nc = a.ns - nh;
  const int mc = m - mh;
  // the arguments' fields used in the loops, in registers
  const int slot_bytes = a.slot_bytes, nch = a.nch, Pg = a.P, dd = a.d;
  const unsigned long long limit_ns = a.limit_ns;
  int* const status = a.status;
  volatile int* vbad = bad;
  if (warp == kWarps) {  // producer warp
    if (lane == 0) {
      // per cold slot: a copy was issued (bit set in `issued`) and the phase
      // parity of the latest one (bit of `par`)
      // entry kc goes to cold slot q = kc % nc in round kc / nc (parity rp),
      // both advanced by increments: this thread's loop paces the ring
      unsigned issued = 0u, par = 0u, rp = 0u;
      int q = 0;
      for (int kc = 0; kc < mc; ++kc) {
        // the slot's previous copy (round kc / nc - 1) was released
        // (compute warps that gave up release no slot: this wait then ends
        // at its own bound)
        if (kc >= nc && !mbar_wait_sleep(empty + nh + q, rp ^ 1u, a.limit_ns)) {
          set_status(a.status, PI_ERR_TIMEOUT);
          *vbad = 1;
          break;
        }
        if (kc + 1 != a.skip_issue) {  // self-test: that slot's phase never completes
          issue_neuron<GATED>(a, slots, full, nh + q, lst[mh + kc]);
          issued |= 1u << q;
          par = (par & ~(1u << q)) | (rp << q);
        }
        if (++q == nc) {
          q = 0;
          rp ^= 1u;
        }
      }
      // on the normal path the compute warps waited for every copy issued;
      // after a give-up, ring_drain waits for these before the block exits
      iss[0] = issued;
      iss[1] = par;
    }
    return;
  }
  __shared__ int s_stop[2];  // block-uniform decision to abandon the ring, per round buffer
  const unsigned w1b = (GATED ? 4u : 2u) * (unsigned)dd;
  float2 xr[NCH][4];  // x of the thread's columns, in pairs
  float2 y2[NCH][4];  // the thread's columns of the partial output
  bool colok[NCH];
  // x of the thread's columns: from shared memory, or (layer-sequence
  // kernel) from global memory written by other blocks before a grid-wide
  // wait, read through L2
  const bool xglob = __isGlobal(xs);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int cc = tid + j * kThreads;
    colok[j] = cc < nch;
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (colok[j]) {
      const float4* px = reinterpret_cast<const float4*>(xs + 8 * cc);
      if (xglob) {
        lo = __ldcg(px);
        hi = __ldcg(px + 1);
      } else {
        lo = px[0];
        hi = px[1];
      }
    }
    xr[j][0] = make_float2(lo.x, lo.y);
    xr[j][1] = make_float2(lo.z, lo.w);
    xr[j][2] = make_float2(hi.x, hi.y);
    xr[j][3] = make_float2(hi.z, hi.w);
#pragma unroll
    for (int e = 0; e < 4; ++e) y2[j][e] = make_float2(yacc[j][2 * e], yacc[j][2 * e + 1]);
  }
  int cslot = 0, cpar = 0;  // ring position of the next cold entry
  int buf = 0;
  const int grp = a.grp;
  for (int g0 = 0; g0 < m; g0 += grp) {
    const int kg = min(grp, m - g0);
    int sl[kGroup];
#pragma unroll
    for (int q = 0; q < kGroup; ++q) {
      sl[q] = 0;
      if (q < kg) {
        const int k = g0 + q;
        unsigned par = 0u;
        if (k < mh) {
          sl[q] = (lst[k] - c) / Pg;
        } else {
          sl[q] = nh + cslot;
          par = (unsigned)cpar;
          if (++cslot == nc) {
            cslot = 0;
            cpar ^= 1;
          }
        }
        if (!mbar_wait(full + sl[q], par, limit_ns)) {
          set_status(status, PI_ERR_TIMEOUT);
          *vbad = 1;
        }
      }
    }
    // A: partial dot products of the round (pairs of fp32 FMAs, two chains
    // per value), one transposing butterfly per warp, warp partials to
    // shared memory
    float pd[NR];
#pragma unroll
    for (int q = 0; q < kGroup; ++q) {
      float a0 = 0.f, a1 = 0.f, u0 = 0.f, u1 = 0.f;  // two chains per value
      if (q < kg) {
        const unsigned char* sp = slots + (size_t)sl[q] * slot_bytes;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (colok[j]) {
            const int cc = tid + j * kThreads;
            float2 f[4];
            unpack4x2<DT>(*reinterpret_cast<const uint4*>(sp + 16 * cc), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              a0 = fmaf(f[e].x, xr[j][e].x, a0);
              a1 = fmaf(f[e].y, xr[j][e].y, a1);
            }
            if (GATED) {
              unpack4x2<DT>(*reinterpret_cast<const uint4*>(sp + 2 * dd + 16 * cc), f);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                u0 = fmaf(f[e].x, xr[j][e].x, u0);
                u1 = fmaf(f[e].y, xr[j][e].y, u1);
              }
            }
          }
        }
      }
      pd[q * NV] = a0 + a1;
      if (GATED) pd[q * NV + NV - 1] = u0 + u1;
    }
    const float r = warp_bfly_sum<NR>(pd);
    float* rb = red + buf * (NR * kWarps);  // [value][warp]
    if ((lane & (32 / NR - 1)) == 0) rb[bfly_index<NR>(lane) * kWarps + warp] = r;
    // a wait of this round (or the producer) gave up: every compute warp
    // reads the one decision after the barrier and leaves the ring; the
    // slots are not released, so the producer issues nothing more
    compute_sync();
    // B: h of the round's neurons, eight lanes of warp 0 adding the kWarps
    // partials in order; every warp reads them after the second barrier
    float hq[kGroup];
    {
      float* hb = hbuf + buf * kGroup;
      if (warp == 0 && lane < kg) {
        float s0 = 0.f, s1 = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          s0 += rb[(lane * NV) * kWarps + w];
          if (GATED) s1 += rb[(lane * NV + NV - 1) * kWarps + w];
        }
        float h = s0 + lb[g0 + lane];
        h = h > 0.f ? h : 0.f;
        if (GATED) h *= s1;
        hb[lane] = h;
      }
      // a wait of this round (or the producer) gave up: every compute warp
      // reads the one decision after the barrier and leaves the ring; the
      // slots are not released, so the producer issues nothing more
      if (warp == 0 && lane == 0) s_stop[buf] = *vbad;
      compute_sync();
      if (s_stop[buf]) break;
#pragma unroll
      for (int q = 0; q < kGroup; ++q) hq[q] = hb[q];
    }
    // C: row-axpy of the round's W2 rows
#pragma unroll
    for (int q = 0; q < kGroup; ++q) {
      if (q < kg) {
        const float2 h2 = make_float2(hq[q], hq[q]);
        const unsigned char* sp = slots + (size_t)sl[q] * slot_bytes + w1b;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          if (colok[j]) {
            const int cc = tid + j * kThreads;
            float2 f[4];
            unpack4x2<DT>(*reinterpret_cast<const uint4*>(sp + 16 * cc), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              y2[j][e].x = fmaf(h2.x, f[e].x, y2[j][e].x);
              y2[j][e].y = fmaf(h2.y, f[e].y, y2[j][e].y);
            }
          }
        }
      }
    }
    // this warp is done with the round's slots: release the recycled ones
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < kGroup; ++q)
        if (q < kg && g0 + q >= mh) mbar_arrive(empty + sl[q]);
    }
    buf ^= 1;
  }
#pragma unroll
  for (int j = 0; j < NCH; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      yacc[j][2 * e] = y2[j][e].x;
      yacc[j][2 * e + 1] = y2[j][e].y;
    }
}

// Sums the P partial rows in a fixed order, adds b2 and the residual, writes
// y.  Block c owns a slice of the d/4 float4 columns, one column per compute
// warp at a time: lane l sums partials l, l + 32, l + 64, ... (all loads
// issued first), then the 32 lane sums meet in a fixed shuffle tree.
__device__ void final_reduce(const FfnArgs& a) {
  const int c = blockIdx.x, P = a.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D4 = a.d >> 2;
  const int j0 = (int)((long long)c * D4 / P), j1 = (int)((long long)(c + 1) * D4 / P);
  constexpr int PU = 6;  // loads in flight per lane (one batch up to 192 blocks)
  for (int j = j0 + warp; j < j1; j += kWarps) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < P; p0 += 32 * PU) {
      float4 v[PU];
#pragma unroll
      for (int u = 0; u < PU; ++u) {
        const int p = p0 + lane + 32 * u;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p < P) v[u] = __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)p * a.d) + j);
      }
#pragma unroll
      for (int u = 0; u < PU; ++u) {
        s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
      s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
      s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
      s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
    }
    if (lane == 0) {
      if (a.b2) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(a.b2) + j);
        s.x += b.x; s.y += b.y; s.z += b.z; s.w += b.w;
      }
      if (a.residual) {
        const float4 rr = __ldg(reinterpret_cast<const float4*>(a.residual) + j);
        s.x += rr.x; s.y += rr.y; s.z += rr.z; s.w += rr.w;
      }
      reinterpret_cast<float4*>(a.y)[j] = s;
    }
  }
}

// Ascending active list of the whole layer from the predicted mask: block c
// compacts mask[c n/P, (c+1) n/P), offset by the number of active neurons
// below its range.  Compute threads only.
__device__ void write_active_list(const FfnArgs& a, int* red_i) {
  const int c = blockIdx.x, P = a.P;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lo = (int)((long long)c * a.n / P), hi = (int)((long long)(c + 1) * a.n / P);
  int below = 0;
  const int lo16 = lo & ~15;
  for (int e = tid * 16; e < lo16; e += kThreads * 16) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(a.mask + e));
    below += __popc(v.x) + __popc(v.y) + __popc(v.z) + __popc(v.w);  // bytes are 0 or 1
  }
  if (tid < lo - lo16) below += __ldcg(a.mask + lo16 + tid);
  below = __reduce_add_sync(0xffffffffu, below);
  if (lane == 0) red_i[warp] = below;
  compute_sync();
  if (warp == 0) {
    int base = 0;
    for (int w = 0; w < kWarps; ++w) base += red_i[w];
    for (int b0 = lo; b0 < hi; b0 += 32) {
      const int i = b0 + lane;
      const bool f = (i < hi) && __ldcg(a.mask + i);
      const unsigned bal = __ballot_sync(0xffffffffu, f);
      if (f) a.idx_out[base + __popc(bal & ((1u << lane) - 1u))] = i;
      base += __popc(bal);
    }
  }
}

// ------------------------------------------------------------ persistent FFN kernel
// MODE kFused : predictor + mask + sparse FFN of one token (one launch).
//               Block c owns neurons c, c + P, c + 2P, ... (interleaving
//               spreads the hot prefix evenly), scores them and computes its
//               active ones; the rows of its first hot neurons were fetched
//               into shared memory before the mask was known.  Two grid-wide
//               waits: the predictor's u and the final split reduction.  The
//               per-block active counts vary, but with whole-neuron bulk
//               copies the chip's bandwidth, not one block, bounds the time.
// MODE kSparse: sparse FFN over a given active list (idx_in, cnt_in), split
//               evenly over the blocks.
// MODE kDense : FFN over all n neurons.
// kThreads compute threads + one producer warp per block; all P blocks
// must be co-resident (cooperative launch); every wait is bounded.
template <int DT, bool GATED, int NCH, int MODE>
__global__ void __launch_bounds__(kBlock, 1) ffn_kernel(const FfnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* xs = reinterpret_cast<float*>(smem + a.o_xs);
  int* lst = reinterpret_cast<int*>(smem + a.o_lst);
  float* lb = reinterpret_cast<float*>(smem + a.o_lb);
  float* red = reinterpret_cast<float*>(smem + a.o_red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.o_mbar);
  uint64_t* empty = full + kMaxSlots;
  unsigned char* slots = smem + a.o_slots;
  const int c = blockIdx.x, P = a.P;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool compute = tid < kThreads;
  __shared__ int s_m, s_mh, s_bad;
  __shared__ unsigned s_iss[2];  // the ring producer's issued slots and their phase parities
  __shared__ unsigned long long s_base;

  const int hot_own = (MODE == kFused && c < a.hot) ? (a.hot - 1 - c) / P + 1 : 0;
  const int nh = (MODE == kFused) ? a.nh : 0;
  const int nh_c = min(nh, hot_own);  // own hot neurons whose rows go to slots up front
  // Everything before pdl_wait() reads only weights: with programmatic
  // dependent launch it overlaps the end of the previous step, whose
  // outputs (x, the workspace) are not touched until after the wait.
  if (tid == 0) {
    for (int s = 0; s < a.ns; ++s) {
      mbar_init(full + s, 1u);
      mbar_init(empty + s, (unsigned)kWarps);
    }
    fence_mbar_init();
    // own hot neurons' rows go out first
    for (int j = 0; j < nh_c; ++j) issue_neuron<GATED>(a, slots, full, j, c + j * P);
    s_bad = 0;
  }
  int m = 0, mh = 0;

  if (MODE == kFused) {
    const int rows = (c < a.n) ? (a.n - 1 - c) / P + 1 : 0;  // own neurons
    unsigned char* As = smem + a.o_As;
    float* b1s = reinterpret_cast<float*>(smem + a.o_b1s);
    float* us = reinterpret_cast<float*>(smem + a.o_us);
    unsigned char* flag = smem + a.o_flag;
    const int units = a.r * a.S;
    const int seg = a.d / a.S;
    const int segc = seg >> 3;

    // 1. this block's first predictor-stage-1 units (Bm chunks)
    uint4 bw[2][2];
#pragma unroll
    for (int uu = 0; uu < 2; ++uu) {
      const int q = c + uu * P;
      const int k = q / a.S, s = q - k * a.S;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ch = tid + h * kThreads;
        bw[uu][h] = make_uint4(0u, 0u, 0u, 0u);
        if (compute && q < units && ch < segc)
          bw[uu][h] = ld_nc(a.Bm + (size_t)k * a.d + (size_t)s * seg + 8 * ch);
      }
    }
    // 3. more weights that do not depend on x: the own hot neurons beyond
    //    the slots towards L2, the own predictor rows and biases
    if (compute) {
      for (int j = nh_c + tid; j < hot_own; j += kThreads) prefetch_neuron<GATED>(a, c + j * P);
      const int rc = a.r >> 3;
      if (a.a_in_smem) {
        for (int e = tid; e < rows * rc; e += kThreads) {
          const int j = e / rc, q = e - j * rc;
          cp_async16(As + (size_t)j * a.a_stride + 16 * q,
                     a.A + ((size_t)c + (size_t)j * P) * a.r + 8 * q);
        }
      } else {
        for (int j = tid; j < rows; j += kThreads)
          prefetch_l2(a.A + ((size_t)c + (size_t)j * P) * a.r, (size_t)a.r * 2);
      }
      for (int j = tid; j < rows; j += kThreads) cp_async4(b1s + j, a.b1 + c + (size_t)j * P);
      cp_async_commit();
    }
    // 2. the previous step's outputs: x and the barrier state
    pdl_wait();
    if (tid == 0) s_base = grid_base(a.bar, (unsigned)P);
    for (int i = tid; i < (a.d >> 2); i += kBlock)
      reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(a.x) + i);
    __syncthreads();
    // 4. predictor stage 1: partial dot products of the units
    for (int q0 = c; q0 < units; q0 += 2 * P) {
      if (q0 != c) {
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
          const int q = q0 + uu * P;
          const int k = q / a.S, s = q - k * a.S;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ch = tid + h * kThreads;
            bw[uu][h] = make_uint4(0u, 0u, 0u, 0u);
            if (compute && q < units && ch < segc)
              bw[uu][h] = ld_nc(a.Bm + (size_t)k * a.d + (size_t)s * seg + 8 * ch);
          }
        }
      }
      float acc[2] = {0.f, 0.f};
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) {
        const int q = q0 + uu * P;
        const int s = q - (q / a.S) * a.S;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ch = tid + h * kThreads;
          if (compute && q < units && ch < segc) {
            float f[8], xv[8];
            unpack8<DT>(bw[uu][h], f);
            load8(xs + (size_t)s * seg + 8 * ch, xv);
            acc[uu] += dot8(f, xv);
          }
        }
      }
#pragma unroll
      for (int uu = 0; uu < 2; ++uu) acc[uu] = warp_sum(acc[uu]);
      if (compute && lane == 0) {
        red[warp * 2] = acc[0];
        red[warp * 2 + 1] = acc[1];
      }
      __syncthreads();
      if (tid < 2) {
        const int q = q0 + tid * P;
        if (q < units) {
          float sum = 0.f;
          for (int w = 0; w < kWarps; ++w) sum += red[w * 2 + tid];
          __stcg(a.upart + q, sum);
        }
      }
      __syncthreads();
    }
    if (!grid_sync(a.bar, s_base + (unsigned long long)P, a.status, a.limit_ns)) {
      cp_async_wait_all();
      if (tid == kThreads)
        for (int j = 0; j < nh_c; ++j) mbar_wait(full + j, 0u, a.drain_ns);
      __syncthreads();
      return;
    }
    // 5. u, logits of the own neurons, mask
    for (int k = tid; k < a.r; k += kBlock) {
      float sum = 0.f;
      for (int ss = 0; ss < a.S; ++ss) sum += __ldcg(a.upart + k * a.S + ss);
      us[k] = sum;
    }
    cp_async_wait_all();
    __syncthreads();
    if (compute) own_logits<DT>(a, As, b1s, us, flag, rows);
    __syncthreads();
    // 6. ordered list of the own active neurons (ballot + popc, one warp);
    //    the hot ones whose rows sit in slots come first
    if (warp == 0) {
      int cnt = 0, nhot = 0;
      for (int base = 0; base < rows; base += 32) {
        const int j = base + lane;
        const bool f = (j < rows) && flag[j];
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
        if (f) {
          lst[pos] = c + j * P;
          lb[pos] = b1s[j];
        }
        if (a.mask && j < rows) a.mask[(size_t)c + (size_t)j * P] = f ? 1 : 0;
        cnt += __popc(bal);
        nhot += __popc(__ballot_sync(0xffffffffu, f && j < nh_c));
      }
      if (lane == 0) {
        s_m = cnt;
        s_mh = nhot;
        __stcg(a.loc_tot + c, cnt);
      }
    }
    __syncthreads();
    m = s_m;
    mh = s_mh;
  } else {
    pdl_wait();
    if (tid == 0) s_base = grid_base(a.bar, (unsigned)P);
    for (int i = tid; i < (a.d >> 2); i += kBlock)
      reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(a.x) + i);
    int total;
    if (MODE == kSparse) {
      total = __ldg(a.cnt_in);
      if (total < 0 || total > a.cap || total > a.n) {
        if (c == 0 && tid == 0) set_status(a.status, PI_ERR_CAPACITY);
        return;  // uniform over the grid: no block reaches a grid-wide wait
      }
    } else {
      total = a.n;
    }
    const long long p0 = (long long)c * total / P, p1 = (long long)(c + 1) * total / P;
    m = (int)(p1 - p0);
    for (int k = tid; k < m; k += kBlock) {
      int v = (MODE == kSparse) ? __ldg(a.idx_in + p0 + k) : (int)(p0 + k);
      if ((unsigned)v >= (unsigned)a.n) {  // never read outside the matrices
        set_status(a.status, PI_ERR_INDEX);
        v = -1;
      }
      lst[k] = v;
    }
    __syncthreads();
    // drop rejected entries, keeping the order
    if (MODE == kSparse && warp == 0) {
      int w = 0;
      for (int base = 0; base < m; base += 32) {
        const int k = base + lane;
        const int v = (k < m) ? lst[k] : -1;
        const unsigned bal = __ballot_sync(0xffffffffu, v >= 0);
        __syncwarp();
        if (v >= 0) lst[w + __popc(bal & ((1u << lane) - 1u))] = v;
        __syncwarp();
        w += __popc(bal);
      }
      if (lane == 0) s_m = w;
    }
    __syncthreads();
    if (MODE == kSparse) m = s_m;
    for (int k = tid; k < m; k += kBlock) lb[k] = __ldg(a.b1 + lst[k]);
    __syncthreads();
  }

  float yacc[NCH][8];
#pragma unroll
  for (int j = 0; j < NCH; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) yacc[j][e] = 0.f;
  if (tid == kThreads) s_iss[0] = s_iss[1] = 0u;
  ffn_ring<DT, GATED, NCH>(a, xs, lst, lb, m, mh, nh, slots, full, empty, red,
                           red + 2 * kGroup * 2 * kWarps, yacc, &s_bad, s_iss);
  __syncthreads();
  if (s_bad && tid == kThreads) ring_drain(full, nh, a.ns - nh, s_iss, a.drain_ns, a.status);
  // speculative copies of own hot neurons that turned out inactive must land
  // before the block may exit
  if (MODE == kFused && tid == kThreads && mh < nh_c) {
    for (int j = 0; j < nh_c; ++j) {
      bool used = false;
      for (int k = 0; k < mh; ++k) used |= (lst[k] == c + j * P);
      if (!used && !mbar_wait(full + j, 0u, a.drain_ns)) set_status(a.status, PI_ERR_TIMEOUT);
    }
  }
  if (compute) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int cc = tid + j * kThreads;
      if (cc < a.nch) {
        float4* dst = reinterpret_cast<float4*>(a.part + (size_t)c * a.d + 8 * (size_t)cc);
        __stcg(dst, make_float4(yacc[j][0], yacc[j][1], yacc[j][2], yacc[j][3]));
        __stcg(dst + 1, make_float4(yacc[j][4], yacc[j][5], yacc[j][6], yacc[j][7]));
      }
    }
  }
  const unsigned long long nb = (MODE == kFused) ? 2ull : 1ull;
  if (!grid_sync(a.bar, s_base + nb * P, a.status, a.limit_ns)) return;
  pdl_trigger();  // no grid-wide wait is left: the next step may start launching
  if (!compute) return;
  final_reduce(a);
  if (MODE == kFused) {
    if (a.cnt_out && c == 0 && warp == 0) {
      int sum = 0;
      for (int b = lane; b < P; b += 32) sum += __ldcg(a.loc_tot + b);
      sum = __reduce_add_sync(0xffffffffu, sum);
      if (lane == 0) a.cnt_out[0] = sum;
    }
    if (a.idx_out) write_active_list(a, reinterpret_cast<int*>(red));
  }
}

// ------------------------------------------------------------ offline packing
// packed[i] = [W1 row(s) of i | W2 row of i], 16 bytes per thread-step.
__global__ void pack_kernel(const uint4* W1, const uint4* W2, uint4* packed, int n, int d8,
                            int m1) {
  const long long rec = (long long)(m1 + 1) * d8;
  const long long total = (long long)n * rec;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long i = e / rec, k = e - i * rec;
    packed[e] = (k < (long long)m1 * d8) ? W1[i * m1 * d8 + k] : W2[i * d8 + (k - (long long)m1 * d8)];
  }
}

// ------------------------------------------------------------ standalone predictor
// u[t][k] = Bm_k . x[t] for the tokens t < batch; one block per row k.
template <int DT, int TB>
__global__ void __launch_bounds__(256) predict_u_kernel(const uint16_t* Bm, const float* x, int d,
                                                        int r, int batch, float* u) {
  const int k = blockIdx.x;
  const uint16_t* row = Bm + (size_t)k * d;
  const int nch = d >> 3;
  float acc[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0.f;
  for (int ch = threadIdx.x; ch < nch; ch += 256) {
    float f[8];
    unpack8<DT>(ld_nc(row + 8 * ch), f);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      if (t < batch) {
        const float4 x0 = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * d + 8 * ch));
        const float4 x1 = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * d + 8 * ch + 4));
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        acc[t] += dot8(f, xv);
      }
    }
  }
  __shared__ float red[8][TB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0) red[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < TB && threadIdx.x < batch) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
    u[(size_t)threadIdx.x * r + k] = s;
  }
}

// logits[t][i] = A_i . u[t] + b1_i; each row read once for all tokens.
template <int DT, int TB>
__global__ void __launch_bounds__(256) predict_logits_kernel(const uint16_t* A, const float* b1,
                                                             const float* u, int n, int r,
                                                             int batch, float* logits) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* us = reinterpret_cast<float*>(smem);  // [batch][r]
  for (int e = threadIdx.x; e < batch * r; e += 256) us[e] = u[e];
  __syncthreads();
  const int rc = r >> 3;
  int G = 1;
  while (G < rc) G <<= 1;
  const int RPW = 32 / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / G, l = lane - g * G;
  const int rows_per_block = 8 * RPW * 4;
  const int i0 = blockIdx.x * rows_per_block;
  for (int base = i0 + warp * RPW; base < i0 + rows_per_block; base += 8 * RPW) {
    const int i = base + g;
    float f[8];
    const bool ok = (i < n) && (l < rc);
    if (ok) unpack8<DT>(ld_nc(A + (size_t)i * r + 8 * l), f);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      if (t < batch) {
        float acc = 0.f;
        if (ok) {
          const float4 u0 = *reinterpret_cast<const float4*>(us + t * r + 8 * l);
          const float4 u1 = *reinterpret_cast<const float4*>(us + t * r + 8 * l + 4);
          const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          acc = dot8(f, uv);
        }
        for (int o = G >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (i < n && l == 0) logits[(size_t)t * n + i] = acc + __ldg(b1 + i);
      }
    }
  }
}

// ------------------------------------------------------------ compaction
// Per token: idx[t][*] = ascending {i : logits[t][i] > 0}, cnt[t] = count.
// Each thread scans a contiguous segment; a block-wide exclusive scan of the
// segment counts gives the output offsets, so the list is ascending.
__global__ void __launch_bounds__(1024) compact_kernel(const float* logits, int n, int* idx,
                                                       int* cnt, int cap, int* status) {
  const int t = blockIdx.x;
  const float* lg = logits + (size_t)t * n;
  int* out = idx + (size_t)t * cap;
  const int per = (n + 1023) / 1024;
  const int b = min(n, (int)threadIdx.x * per), e = min(b + per, n);
  int c = 0;
  for (int i = b; i < e; ++i) c += (lg[i] > 0.f) ? 1 : 0;
  __shared__ int wsum[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    wsum[lane] = s - v;  // exclusive
  }
  __syncthreads();
  int pos = wsum[warp] + incl - c;
  for (int i = b; i < e; ++i) {
    if (lg[i] > 0.f) {
      if (pos < cap) out[pos] = i;
      ++pos;
    }
  }
  if (threadIdx.x == 1023) {
    cnt[t] = pos;
    if (pos > cap) set_status(status, PI_ERR_CAPACITY);
  }
}

// Union over the batch: uidx = ascending {i : some token active},
// tmask[k] = bitmask of the active tokens at uidx[k].
__global__ void __launch_bounds__(1024) union_kernel(const float* logits, int n, int batch,
                                                     int* uidx, int* ucnt, uint32_t* tmask) {
  __shared__ int wsum[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int out = 0;
  for (int base = 0; base < n; base += 1024) {
    const int i = base + threadIdx.x;
    uint32_t msk = 0;
    if (i < n)
      for (int t = 0; t < batch; ++t) msk |= (logits[(size_t)t * n + i] > 0.f ? 1u : 0u) << t;
    const bool f = msk != 0u;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    int pre = 0, tot = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = wsum[w];
      pre += (w < warp) ? v : 0;
      tot += v;
    }
    if (f) {
      const int pos = out + pre + __popc(bal & ((1u << lane) - 1u));
      uidx[pos] = i;
      tmask[pos] = msk;
    }
    out += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) *ucnt = out;
}

// ------------------------------------------------------------ grid-wide compaction
// The same lists as compact_kernel / union_kernel, computed by the whole
// grid: blocks of kCB neurons; series t < batch are the tokens' lists,
// series 32 the union.
//   pass 1: each block's count per series -> scr[s][b];
//   pass 2 (one block): exclusive prefix of every series over the blocks,
//           in place, totals -> scr[33 nb + s];
//   pass 3: each block writes its entries at its offsets (ascending order),
//           the last block the counts.
constexpr int kCB = 256;
constexpr int kCSeries = 33;

__device__ __forceinline__ uint32_t token_mask(const float* logits, int n, int batch, int i) {
  uint32_t m = 0u;
  if (i < n)
    for (int t = 0; t < batch; ++t) m |= (logits[(size_t)t * n + i] > 0.f ? 1u : 0u) << t;
  return m;
}

__global__ void __launch_bounds__(kCB) cu_count_kernel(const float* logits, int n, int batch,
                                                       int want_union, int* scr, int nb) {
  pdl_enter();
  __shared__ int wc[kCSeries][kCB / 32];
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t m = token_mask(logits, n, batch, b * kCB + tid);
  for (int t = 0; t < batch; ++t) {
    const unsigned bal = __ballot_sync(0xffffffffu, (m >> t) & 1u);
    if (lane == 0) wc[t][warp] = __popc(bal);
  }
  const unsigned bu = __ballot_sync(0xffffffffu, m != 0u);
  if (lane == 0) wc[32][warp] = __popc(bu);
  __syncthreads();
  if (tid < kCSeries && (tid < batch || (tid == 32 && want_union))) {
    int sum = 0;
    for (int w = 0; w < kCB / 32; ++w) sum += wc[tid][w];
    scr[(size_t)tid * nb + b] = sum;
  }
}

__global__ void __launch_bounds__(1024) cu_scan_kernel(int* scr, int nb, int batch, int want_union) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int s = warp; s < kCSeries; s += 32) {
    if (!(s < batch || (s == 32 && want_union))) continue;
    int* row = scr + (size_t)s * nb;
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const int v0 = (b < nb) ? row[b] : 0;
      int v = v0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (b < nb) row[b] = run + v - v0;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) scr[(size_t)kCSeries * nb + s] = run;
  }
}

// fused = 1: scr holds the raw per-block counts of cu_count_kernel (no
// cu_scan_kernel ran); every block sums the counts of the blocks before it
// itself (integer sums: any order gives the same offsets).  Meant for few
// blocks (the work is quadratic in nb).
__global__ void __launch_bounds__(kCB) cu_write_kernel(const float* logits, int n, int batch,
                                                       const int* scr, int nb, int* idx, int* cnt,
                                                       int cap, int* uidx, int* ucnt,
                                                       uint32_t* tmask, int* status, int fused) {
  pdl_enter();
  __shared__ int wc[kCSeries][kCB / 32];
  __shared__ unsigned wb[kCSeries][kCB / 32];
  __shared__ int boff[kCSeries], btot[kCSeries];
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = b * kCB + tid;
  const uint32_t m = token_mask(logits, n, batch, i);
  const bool want_union = uidx != nullptr;
  if (fused) {
    for (int s = warp; s < kCSeries; s += kCB / 32) {
      if (!(s < batch || (s == 32 && want_union))) continue;
      const int* row = scr + (size_t)s * nb;
      int before = 0, all = 0;
      for (int q = lane; q < nb; q += 32) {
        const int v = row[q];
        all += v;
        if (q < b) before += v;
      }
      before = __reduce_add_sync(0xffffffffu, before);
      all = __reduce_add_sync(0xffffffffu, all);
      if (lane == 0) {
        boff[s] = before;
        btot[s] = all;
      }
    }
  }
  for (int t = 0; t < batch; ++t) {
    const unsigned bal = __ballot_sync(0xffffffffu, (m >> t) & 1u);
    if (lane == 0) wb[t][warp] = bal;
  }
  const unsigned bu = __ballot_sync(0xffffffffu, m != 0u);
  if (lane == 0) wb[32][warp] = bu;
  __syncthreads();
  if (tid < kCSeries) {  // exclusive offsets of the warps, after the blocks before this one
    const bool on = tid < batch || (tid == 32 && want_union);
    int run = on ? (fused ? boff[tid] : scr[(size_t)tid * nb + b]) : 0;
    for (int w = 0; w < kCB / 32; ++w) {
      wc[tid][w] = run;
      run += __popc(wb[tid][w]);
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int t = 0; t < batch; ++t) {
    if ((m >> t) & 1u) {
      const int pos = wc[t][warp] + __popc(wb[t][warp] & lt);
      if (pos < cap) idx[(size_t)t * cap + pos] = i;
    }
  }
  if (want_union && m != 0u) {
    const int pos = wc[32][warp] + __popc(bu & lt);
    uidx[pos] = i;
    tmask[pos] = m;
  }
  if (b == nb - 1) {
    if (tid < batch) {
      const int tot = fused ? btot[tid] : scr[(size_t)kCSeries * nb + tid];
      cnt[tid] = tot;
      if (tot > cap) set_status(status, PI_ERR_CAPACITY);
    }
    if (tid == 32 && want_union) *ucnt = fused ? btot[32] : scr[(size_t)kCSeries * nb + 32];
  }
}

// ------------------------------------------------------------ offline placement
// "Offline Section": a profiler counts how often each neuron activates over
// sample inputs and the neurons are placed hot first; the placed layer's
// row k is the original row perm[k] ("Neuron Placement and Administration":
// perm is the neuron table).

// counts[i] += #{t < batch : logits[t][i] > 0}; one thread per neuron.
__global__ void profile_count_kernel(const float* logits, int n, int batch, unsigned* counts) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    unsigned c = 0u;
    for (int t = 0; t < batch; ++t) c += logits[(size_t)t * n + i] > 0.f ? 1u : 0u;
    counts[i] += c;
  }
}

// perm[rank(i)] = i, rank(i) = #{j : c_j > c_i} + #{j < i : c_j == c_i}:
// more activations first, equal counts in ascending index.  Each thread
// compares its count with every count (tiles staged in shared memory).
constexpr int kRankTile = 2048;
__global__ void __launch_bounds__(256) rank_kernel(const unsigned* counts, int n, int* perm) {
  __shared__ unsigned tile[kRankTile];
  const int i = blockIdx.x * 256 + threadIdx.x;
  const unsigned ci = i < n ? counts[i] : 0u;
  int rank = 0;
  for (int j0 = 0; j0 < n; j0 += kRankTile) {
    const int m = min(kRankTile, n - j0);
    __syncthreads();
    for (int e = threadIdx.x; e < m; e += 256) tile[e] = counts[j0 + e];
    __syncthreads();
    for (int jj = 0; jj < m; ++jj) {
      const unsigned cj = tile[jj];
      rank += (cj > ci || (cj == ci && j0 + jj < i)) ? 1 : 0;
    }
  }
  if (i < n) perm[rank] = i;
}

// dst row k = src row perm[k], rows of q16 sixteen-byte pieces.  An entry
// outside [0, n) is not followed: the row is left alone and PI_ERR_INDEX
// is recorded.
__global__ void gather_rows16_kernel(const uint4* src, uint4* dst, const int* perm, int n,
                                     long long q16, int* status) {
  const long long tot = (long long)n * q16;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
       e += (long long)gridDim.x * blockDim.x) {
    const long long k = e / q16, q = e - k * q16;
    const int pk = __ldg(perm + k);
    if ((unsigned)pk >= (unsigned)n) {
      if (q == 0) set_status(status, PI_ERR_INDEX);
      continue;
    }
    dst[e] = __ldg(src + (long long)pk * q16 + q);
  }
}
__global__ void gather_f32_kernel(const float* src, float* dst, const int* perm, int n,
                                  int* status) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n; k += gridDim.x * blockDim.x) {
    const int pk = __ldg(perm + k);
    if ((unsigned)pk >= (unsigned)n) {
      set_status(status, PI_ERR_INDEX);
      continue;
    }
    dst[k] = __ldg(src + pk);
  }
}

// Failure-path diagnostic: one grid-wide wait whose last arrival never
// comes (expected = grid + 1), so every block gives up after limit_ns.
__global__ void wait_timeout_kernel(unsigned long long* bar, int* status,
                                    unsigned long long limit_ns) {
  __shared__ unsigned long long s_base;
  if (threadIdx.x == 0) s_base = grid_base(bar, gridDim.x);
  __syncthreads();
  grid_sync(bar, s_base + gridDim.x + 1u, status, limit_ns);
}

}  // namespace pik

// seq.cuh — decode through a sequence of FFN layers in one persistent launch.
//
// Same method as the one-layer kernel (predictor, mask, hot-first row
// gather, row-axpy, fixed-order split reduction; "PowerInfer: Quick Massive
// Language Mannequin Serving with a Client-grade GPU", sections "Online
// Section" and "Neuron Conscious Operator"), run for J jobs in a row.  Job j
// uses layer table entry j % R; chained jobs form a residual stack
// (x_{j+1} = x_j + FFN_j(x_j)), independent jobs read their own x.
//
// Two grid-wide waits per job.  Block c owns the 8-column chunks
// [c nch / P, (c+1) nch / P) of the layer's d columns:
//   R  after the previous job's partial rows are complete: the block sums
//      its columns of the P partials (fixed order), adds b2 and the residual
//      and writes them (chained: its columns of the next x);
//   U  predictor stage 1 over its own columns only (split-K): a partial u
//      of r values per block, so no block needs the whole new x yet.  The
//      partials meet in 64-bit fixed-point accumulators (value x 2^32,
//      integer reductions in memory): integer addition is associative, so
//      u is the same whatever order the blocks arrive in (deterministic),
//      and it is exact up to the one rounding of each partial to 2^-32;
//   -- wait 1 --
//   L  full x and u, logits of the block's own neurons, their ordered
//      active list;
//      ring: the row-gather GEMV + ReLU and row-axpy of those neurons;
//   -- wait 2 -- (partial rows written)
// Between its arrival at wait 2 and the end of that wait, the block
// requests the next job's own hot neurons' rows (into ring slots) and Bm
// columns (into shared memory); the job's predictor rows and biases are
// requested in the same way at wait 1, and an independent job's x before
// U.  The transfers overlap the waits and delay no arrival.  Independent
// jobs also run the previous job's R beside their own U on other warps
// (when the warps suffice), and only the U warps make the block's arrival
// at wait 1; chained jobs run R, then U, which needs R's columns.
// With balancing on (large layers), the blocks publish their cold active
// neurons after the lists are built and, after one more grid-wide wait, each
// takes an equal share of them by global rank.
// A job reads its x only after every partial row of the previous job is
// complete (its wait 2): jobs never overlap in anything that depends on
// their inputs.
#pragma once

#include "kernels.cuh"

namespace pik {

constexpr int kSeqMaxLayers = 128;
constexpr int kSeqMaxQ = 8;  // most own 8-column chunks per block

struct SeqLayer {
  const uint16_t* A;
  const uint16_t* Bm;
  const float* b1;
  const uint16_t* W1;
  const uint16_t* W2;
  const float* b2;
  int hot;
  int r;  // this layer's predictor rank (<= the launch's f.r, which sizes the buffers)
};

struct SeqArgs {
  FfnArgs f;              // shape, grid, shared-memory plan, workspace (weights per job)
  int J, R, chain;
  const float* x;         // chained: [d]; else [J][d]
  float* y;               // [J][d] (chained: x_{j+1})
  int* cnt_out;           // [J] or NULL
  unsigned char* mask_out;  // [J][n] or NULL
  unsigned long long* uacc;  // [2][r] fixed-point u, 16 words (128 bytes) apart; zero at launch
  int bm_smem;            // stage the next job's own Bm columns in the last ring slot
  int a_slots;            // stage the next job's own predictor rows in ring slots [nh, ns - 1)
                          // (when they do not fit beside the ring)
  int balance;            // spread the cold active neurons evenly (one more grid-wide wait)
  int2* glist;            // [P][rows_max] published cold entries (neuron, b1 bits)
  int* gcnt;              // [P] published cold counts
  SeqLayer L[kSeqMaxLayers];
};

template <int DT, bool GATED, int NCH>
__global__ void __launch_bounds__(kBlock, 1) seq_kernel(const SeqArgs sa) {
  extern __shared__ __align__(128) unsigned char smem[];
  const FfnArgs& f = sa.f;
  int* lst = reinterpret_cast<int*>(smem + f.o_lst);
  float* lb = reinterpret_cast<float*>(smem + f.o_lb);
  float* red = reinterpret_cast<float*>(smem + f.o_red);
  float* xo = red + 2 * kGroup * 2 * kWarps + 2 * kGroup;  // own x columns (<= 64 floats)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + f.o_mbar);
  uint64_t* empty = full + kMaxSlots;
  unsigned char* slots = smem + f.o_slots;
  // own predictor rows: staged in the fixed region, or in idle ring slots
  unsigned char* As = sa.a_slots ? slots + (size_t)f.nh * f.slot_bytes : smem + f.o_As;
  float* b1s = reinterpret_cast<float*>(smem + f.o_b1s);
  float* us = reinterpret_cast<float*>(smem + f.o_us);
  unsigned char* flag = smem + f.o_flag;
  const int c = blockIdx.x, P = f.P;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool compute = tid < kThreads;
  __shared__ int s_m, s_mh, s_bad;
  __shared__ unsigned s_iss[2];  // the ring producer's issued slots and their phase parities
  __shared__ unsigned long long s_base;

  const int rows = (c < f.n) ? (f.n - 1 - c) / P + 1 : 0;  // own neurons c, c + P, ...
  const int q0 = (int)((long long)c * f.nch / P), q1 = (int)((long long)(c + 1) * f.nch / P);
  const int nq = q1 - q0;  // own 8-column chunks (<= kSeqMaxQ, checked by the host)

  unsigned char* bms = slots + (size_t)(f.ns - 1) * f.slot_bytes;  // staged Bm columns
  FfnArgs a = f;  // the current job's weights
  if (sa.a_slots) a.a_in_smem = 1;  // own_logits reads the staged rows
  int nh_c = 0;   // own hot neurons whose rows went to slots for the current job

  // The weights of job j that do not depend on its x.  prep_set points the
  // job's arguments at them; prep_issue requests the first of them: the
  // producer lane re-arms the ring barriers (no copy may be in flight) and
  // sends the own hot neurons' rows to their slots; compute threads
  // [t0, t0 + nt) stage the own Bm columns ([k][q], 16 bytes each, in the
  // last ring slot, a cold one) as one copy group, the own predictor rows
  // (a_slots: into the idle slots after the hot ones) as a second group,
  // and send the hot rows beyond the slots towards L2.
  bool armed = false;  // the ring barriers hold a previous job's state
  auto prep_set = [&](int j) {
    const SeqLayer& Lw = sa.L[j % sa.R];
    a.A = Lw.A;
    a.Bm = Lw.Bm;
    a.b1 = Lw.b1;
    a.W1 = Lw.W1;
    a.W2 = Lw.W2;
    a.b2 = Lw.b2;
    a.hot = Lw.hot;
    a.r = Lw.r;
    nh_c = min(f.nh, (c < a.hot) ? (a.hot - 1 - c) / P + 1 : 0);
  };
  auto prep_issue = [&](int t0, int nt) {
    if (tid == kThreads) {
      for (int s = 0; s < f.ns; ++s) {
        if (armed) {
          mbar_inval(full + s);
          mbar_inval(empty + s);
        }
        mbar_init(full + s, 1u);
        mbar_init(empty + s, (unsigned)kWarps);
      }
      fence_mbar_init();
      for (int k = 0; k < nh_c; ++k) issue_neuron<GATED>(a, slots, full, k, c + k * P);
    }
    armed = true;
    const int t = tid - t0;
    if (t >= 0 && t < nt) {
      const int hot_own = (c < a.hot) ? (a.hot - 1 - c) / P + 1 : 0;
      if (sa.bm_smem)
        for (int e = t; e < a.r * nq; e += nt) {
          const int k = e / nq, q = e - k * nq;
          cp_async16(bms + (size_t)e * 16, a.Bm + (size_t)k * f.d + 8 * (q0 + q));
        }
      cp_async_commit();
      if (sa.a_slots) {
        const int rc = a.r >> 3;
        for (int e = t; e < rows * rc; e += nt) {
          const int jj = e / rc, q = e - jj * rc;
          cp_async16(As + (size_t)jj * f.a_stride + 16 * q,
                     a.A + ((size_t)c + (size_t)jj * P) * a.r + 8 * q);
        }
      }
      cp_async_commit();
      for (int k = nh_c + t; k < hot_own; k += nt) prefetch_neuron<GATED>(a, c + k * P);
    }
  };

  // The job's predictor rows (staged, or towards L2) and biases: issued by
  // every compute thread once the block has arrived at the first grid-wide
  // wait (they are first read by the logits, after it), one copy group.
  auto rows_issue = [&]() {
    if (compute) {
      if (sa.a_slots) {
        // staged at the job's start (prep_issue)
      } else if (f.a_in_smem) {
        const int rc = a.r >> 3;
        for (int e = tid; e < rows * rc; e += kThreads) {
          const int jj = e / rc, q = e - jj * rc;
          cp_async16(As + (size_t)jj * f.a_stride + 16 * q,
                     a.A + ((size_t)c + (size_t)jj * P) * a.r + 8 * q);
        }
      } else {
        for (int jj = tid; jj < rows; jj += kThreads)
          prefetch_l2(a.A + ((size_t)c + (size_t)jj * P) * a.r, (size_t)a.r * 2);
      }
      for (int jj = tid; jj < rows; jj += kThreads) cp_async4(b1s + jj, a.b1 + c + (size_t)jj * P);
      cp_async_commit();
    }
  };
  // On a failed grid-wide wait: let this block's own copies land, then leave.
  auto bail = [&]() {
    cp_async_wait_all();
    if (tid == kThreads)
      for (int k = 0; k < nh_c; ++k) mbar_wait(full + k, 0u, f.drain_ns);
    __syncthreads();
  };

  // R of job jr: own columns of y_jr, one float4 column per compute warp
  // (warps below 2 nq): lane l sums partials l, l + 32, ... (loads issued
  // first), then a fixed shuffle tree; + b2 (+ the residual x_jr when
  // chained, and its columns become the next x's)
  auto reduce_cols = [&](int jr, const float* b2r) {
    if (warp < 2 * nq) {
      const int col4 = 2 * q0 + warp;
      const float4 bb = b2r ? __ldg(reinterpret_cast<const float4*>(b2r) + col4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      constexpr int PU = 6;  // loads in flight per lane (one batch up to 192 blocks)
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p0 = 0; p0 < P; p0 += 32 * PU) {
        float4 v[PU];
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const int p = p0 + lane + 32 * u;
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (p < P) v[u] = __ldcg(reinterpret_cast<const float4*>(f.part + (size_t)p * f.d) + col4);
        }
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          s.x += v[u].x;
          s.y += v[u].y;
          s.z += v[u].z;
          s.w += v[u].w;
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
        s.x += bb.x;
        s.y += bb.y;
        s.z += bb.z;
        s.w += bb.w;
        float4* xo4 = reinterpret_cast<float4*>(xo) + warp;
        if (sa.chain) {
          const float4 rr = *xo4;  // x_j at these columns
          s.x += rr.x;
          s.y += rr.y;
          s.z += rr.z;
          s.w += rr.w;
          *xo4 = s;  // x_{j+1}
        }
        reinterpret_cast<float4*>(sa.y + (size_t)jr * f.d)[col4] = s;
      }
    }
  };
  // Independent steps, when the warps suffice: job j - 1's column reduce
  // (warps below 2 nq) runs beside job j's stage 1 (the nU warps after
  // them), and those warps alone make the block's arrival at wait 1; the
  // reduce warps join before that wait ends.  Chained steps need the
  // reduce's columns for stage 1 and keep the two in sequence.
  const int nU = (f.r + 31) >> 5;
  const bool ov = !sa.chain && 2 * nq + nU <= kWarps;
  const int ub = ov ? 64 * nq : 0;  // first stage-1 thread
  const float* b2prev = nullptr;

  if (tid == 0) s_bad = 0;
  prep_set(0);
  prep_issue(0, kThreads);
  pdl_wait();
  if (tid == 0) s_base = grid_base(f.bar, (unsigned)P);
  unsigned long long nbar = 0;

  for (int j = 0; j < sa.J; ++j) {
    // own columns of this job's x: job 0 reads them here; later jobs find
    // them in xo (written by the previous job's R phase)
    if (j == 0 && tid < nq * 8) xo[tid] = __ldcg(sa.x + 8 * q0 + tid);
    cp_async_wait_group<1>();  // this job's staged Bm columns (its predictor rows may still land)
    __syncthreads();
    if (ov && j > 0) reduce_cols(j - 1, b2prev);
    // U: partial predictor stage 1 over the own columns, u_c[k] for k < r
    const int ut = tid - ub;  // k of this thread
    if (ut >= 0 && ut < a.r) {
      const uint16_t* row = a.Bm + (size_t)ut * f.d + 8 * q0;
      float acc = 0.f;
      for (int qb = 0; qb < nq; qb += 4) {  // batches of 4 pieces, loads first
        uint4 wv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (qb + t < nq)
            wv[t] = sa.bm_smem
                        ? *reinterpret_cast<const uint4*>(bms + ((size_t)ut * nq + qb + t) * 16)
                        : ld_nc(row + 8 * (qb + t));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (qb + t < nq) {
            float w[8], xv[8];
            unpack8<DT>(wv[t], w);
            load8(xo + 8 * (qb + t), xv);
            acc += dot8(w, xv);
          }
        }
      }
      if (!(fabsf(acc) < 8388608.f)) {  // |partial| >= 2^23, or NaN
        set_status(f.status, PI_ERR_RANGE);
        acc = 0.f;
      }
      const long long v = __double2ll_rn((double)acc * 4294967296.0);
      unsigned long long* dst = sa.uacc + ((size_t)(j & 1) * f.r + ut) * 16;
      asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(dst), "l"((unsigned long long)v)
                   : "memory");
    }
    ++nbar;
    if (ov) {  // the stage-1 warps meet, one of them arrives for the block
      if (ut >= 0 && ut < 32 * nU) {
        asm volatile("bar.sync 5, %0;" ::"r"(32 * nU) : "memory");
        if (ut == 0)
          asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(f.bar) : "memory");
      }
    } else {
      grid_arrive(f.bar);
    }
    rows_issue();
    if (!grid_wait(f.bar, s_base + nbar * P, f.status, f.limit_ns)) {
      bail();
      return;
    }
    // L: u, own logits and list
    if (tid < f.r) {
      // u[k] from its accumulator; block 0 clears the other buffer (last
      // read by the previous job, before this job's first wait) for the
      // next, over the largest rank of the launch
      if (tid < a.r) {
        const unsigned long long v = __ldcg(sa.uacc + ((size_t)(j & 1) * f.r + tid) * 16);
        us[tid] = (float)((double)(long long)v * 2.3283064365386963e-10);  // x 2^-32
      }
      if (c == 0) sa.uacc[((size_t)((j + 1) & 1) * f.r + tid) * 16] = 0ull;
    }
    cp_async_wait_all();  // this job's staged predictor rows and biases
    // the staging wrote ring slots through the generic proxy; the ring's
    // bulk copies (async proxy) write them again later
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (compute) own_logits<DT>(a, As, b1s, us, flag, rows);
    __syncthreads();
    {
      // ordered list of the own active neurons, all compute warps: warp w
      // takes 32-row chunks w, w + 16, ...; chunk counts, their exclusive
      // prefix (warp 0), then every warp writes its entries.  The hot ones
      // whose rows sit in slots (row < nh_c <= 16, chunk 0) come first.
      unsigned char* mrow = sa.mask_out ? sa.mask_out + (size_t)j * f.n : nullptr;
      int* ccnt = reinterpret_cast<int*>(red);  // chunk counts, then offsets
      const int nck = (rows + 31) >> 5;         // <= 256 (checked by the host)
      if (compute)
        for (int ch = warp; ch < nck; ch += kWarps) {
          const int jj = ch * 32 + lane;
          const unsigned bal = __ballot_sync(0xffffffffu, jj < rows && flag[jj]);
          if (lane == 0) ccnt[ch] = __popc(bal);
        }
      __syncthreads();
      if (warp == 0) {
        int run = 0;
        for (int b0 = 0; b0 < nck; b0 += 32) {
          const int b = b0 + lane;
          const int v0 = (b < nck) ? ccnt[b] : 0;
          int v = v0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
          }
          if (b < nck) ccnt[b] = run + v - v0;
          run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
          s_m = run;
          s_mh = 0;  // set below from chunk 0, if the block has rows
          __stcg(f.loc_tot + c, run);
        }
      }
      __syncthreads();
      if (compute)
        for (int ch = warp; ch < nck; ch += kWarps) {
          const int jj = ch * 32 + lane;
          const bool fl = jj < rows && flag[jj];
          const unsigned bal = __ballot_sync(0xffffffffu, fl);
          if (fl) {
            const int pos = ccnt[ch] + __popc(bal & ((1u << lane) - 1u));
            lst[pos] = c + jj * P;
            lb[pos] = b1s[jj];
          }
          if (mrow && jj < rows) mrow[(size_t)c + (size_t)jj * P] = fl ? 1 : 0;
          if (ch == 0) {
            const unsigned hb = __ballot_sync(0xffffffffu, fl && jj < nh_c);
            if (lane == 0) s_mh = __popc(hb);
          }
        }
    }
    __syncthreads();
    int m = s_m;
    const int mh = s_mh;
    if (sa.balance) {
      // Cold entries (those without a slot) are spread over the blocks by
      // their rank in the concatenation of all blocks' lists: block c takes
      // ranks c, c + P, ...  The split depends only on the lists, so the
      // per-block sums keep a fixed order.
      int2* gl = sa.glist + (size_t)c * f.rows_max;
      for (int e = tid; e < m - mh; e += kBlock)
        gl[e] = make_int2(lst[mh + e], __float_as_int(lb[mh + e]));
      if (tid == 0) __stcg(sa.gcnt + c, m - mh);
      ++nbar;
      if (!grid_sync(f.bar, s_base + nbar * P, f.status, f.limit_ns)) {
        bail();
        return;
      }
      int* pre = reinterpret_cast<int*>(red);  // [P + 1] exclusive prefix of the counts
      if (warp == 0) {
        int run = 0;
        for (int b0 = 0; b0 < P; b0 += 32) {
          const int b = b0 + lane;
          int v = (b < P) ? __ldcg(sa.gcnt + b) : 0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
          }
          if (b < P) pre[b + 1] = run + v;
          run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) pre[0] = 0;
      }
      __syncthreads();
      const int C = pre[P];
      const int mc = (C > c) ? (C - 1 - c) / P + 1 : 0;
      for (int t = tid; t < mc; t += kBlock) {
        const int k = c + t * P;
        int lo = 0, hi = P;  // pre[lo] <= k < pre[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (pre[mid] <= k) lo = mid;
          else hi = mid;
        }
        const int2 e = __ldcg(sa.glist + (size_t)lo * f.rows_max + (k - pre[lo]));
        lst[mh + t] = e.x;
        lb[mh + t] = __int_as_float(e.y);
      }
      __syncthreads();
      m = mh + mc;
    }
    float yacc[NCH][8];
#pragma unroll
    for (int q = 0; q < NCH; ++q)
#pragma unroll
      for (int e = 0; e < 8; ++e) yacc[q][e] = 0.f;
    // the job's whole x, read by the ring from global memory (a chained
    // job's x is complete only after the first grid-wide wait)
    const float* xg = sa.chain ? (j == 0 ? sa.x : sa.y + (size_t)(j - 1) * f.d)
                               : sa.x + (size_t)j * f.d;
    if (tid == kThreads) s_iss[0] = s_iss[1] = 0u;
    ffn_ring<DT, GATED, NCH>(a, xg, lst, lb, m, mh, f.nh, slots, full, empty, red,
                             red + 2 * kGroup * 2 * kWarps, yacc, &s_bad, s_iss);
    __syncthreads();
    // copies of own hot neurons that turned out inactive land before the
    // slots are re-armed
    if (tid == kThreads && mh < nh_c) {
      for (int k = 0; k < nh_c; ++k) {
        bool used = false;
        for (int e = 0; e < mh; ++e) used |= (lst[e] == c + k * P);
        if (!used && !mbar_wait(full + k, 0u, f.drain_ns)) set_status(f.status, PI_ERR_TIMEOUT);
      }
    }
    nh_c = 0;  // every slot copy of this job has landed
    __syncthreads();
    if (s_bad) {  // a ring wait gave up (block-uniform after the barrier)
      if (tid == kThreads) ring_drain(full, f.nh, f.ns - f.nh, s_iss, f.drain_ns, f.status);
      cp_async_wait_all();
      __syncthreads();
      return;
    }
    const float* b2j = a.b2;
    if (compute) {  // the partial rows go out first: wait 2 fences them
#pragma unroll
      for (int q = 0; q < NCH; ++q) {
        const int cc = tid + q * kThreads;
        if (cc < f.nch) {
          float4* dst = reinterpret_cast<float4*>(f.part + (size_t)c * f.d + 8 * (size_t)cc);
          __stcg(dst, make_float4(yacc[q][0], yacc[q][1], yacc[q][2], yacc[q][3]));
          __stcg(dst + 1, make_float4(yacc[q][4], yacc[q][5], yacc[q][6], yacc[q][7]));
        }
      }
    }
    ++nbar;
    grid_arrive(f.bar);
    // the next job's hot rows and Bm columns, requested while this block
    // waits (the ring is done and no slot copy is in flight)
    if (j + 1 < sa.J) {
      prep_set(j + 1);
      prep_issue(0, kThreads);
    }
    if (!grid_wait(f.bar, s_base + nbar * P, f.status, f.limit_ns)) {
      bail();
      return;
    }
    if (j + 1 == sa.J) pdl_trigger();  // no grid-wide wait is left
    if (!sa.chain && j + 1 < sa.J && tid < nq * 8)  // the next step's own columns
      xo[tid] = __ldcg(sa.x + (size_t)(j + 1) * f.d + 8 * q0 + tid);
    if (sa.cnt_out && c == 0 && warp == 0) {
      int sum = 0;
      for (int b = lane; b < P; b += 32) sum += __ldcg(f.loc_tot + b);
      sum = __reduce_add_sync(0xffffffffu, sum);
      if (lane == 0) sa.cnt_out[j] = sum;
    }
    if (!ov) reduce_cols(j, b2j);
    b2prev = b2j;
  }
  // independent steps: the last job's column reduce
  if (ov && warp < 2 * nq) reduce_cols(sa.J - 1, b2prev);
}

}  // namespace pik

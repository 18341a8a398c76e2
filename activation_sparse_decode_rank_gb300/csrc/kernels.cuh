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

struct FfnArgs {
  int d, n, r;
  int S;          // predictor row split (fused path)
  int P;          // grid size (all blocks co-resident)
  int hot;        // hot-prefix length (rows fetched into L2 up front)
  int nch;        // d / 8: 16-byte column chunks of a row
  int rows_max;   // ceil(n / P)
  // dynamic shared-memory offsets (bytes)
  int o_xs, o_us, o_As, o_b1s, o_flag, o_lst, o_off, o_wl, o_red;
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
  GridBar bar;
  float* upart;   // [r * S]
  int* loc_cnt;   // [P]
  int* loc_idx;   // [n]
  float* part;    // [P][d]
  unsigned long long limit_ns;
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

// ------------------------------------------------------------ predictor
// Stage 1 of the fused path: the r x S units (row k of Bm, column segment s)
// are spread over the grid; unit q's partial dot product goes to upart[q].
template <int DT>
__device__ void fused_u(const FfnArgs& a, const float* xs, float* red) {
  const int c = blockIdx.x;
  const int units = a.r * a.S;
  const int seg = a.d / a.S;
  const int segc = seg >> 3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q0 = c; q0 < units; q0 += 4 * a.P) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int uu = 0; uu < 4; ++uu) {
      const int q = q0 + uu * a.P;
      if (q < units) {
        const int k = q / a.S, s = q - k * a.S;
        const uint16_t* row = a.Bm + (size_t)k * a.d + (size_t)s * seg;
        const float* xp = xs + (size_t)s * seg;
        for (int ch = threadIdx.x; ch < segc; ch += kThreads) {
          float f[8], xv[8];
          unpack8<DT>(ld_nc(row + 8 * ch), f);
          const float4 x0 = *reinterpret_cast<const float4*>(xp + 8 * ch);
          const float4 x1 = *reinterpret_cast<const float4*>(xp + 8 * ch + 4);
          xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w;
          xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
          acc[uu] += dot8(f, xv);
        }
      }
    }
#pragma unroll
    for (int uu = 0; uu < 4; ++uu) acc[uu] = warp_sum(acc[uu]);
    if (lane == 0) {
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) red[warp * 4 + uu] = acc[uu];
    }
    __syncthreads();
    if (threadIdx.x < 4) {
      const int q = q0 + threadIdx.x * a.P;
      if (q < units) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[w * 4 + threadIdx.x];
        __stcg(a.upart + q, s);
      }
    }
    __syncthreads();
  }
}

// Stage 2 of the fused path: logits of this block's neuron slice from the
// A rows staged in shared memory; flag[row] = (logit > 0).
template <int DT>
__device__ void fused_logits(const FfnArgs& a, const uint16_t* As, const float* b1s,
                             const float* us, int* flag, int rows) {
  const int rc = a.r >> 3;
  int G = 1;
  while (G < rc) G <<= 1;
  const int RPW = 32 / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / G, l = lane - g * G;
  float uf[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) uf[e] = (l < rc) ? us[8 * l + e] : 0.f;
  for (int base = warp * RPW; base < rows; base += kWarps * RPW) {
    const int row = base + g;
    float acc = 0.f;
    if (row < rows && l < rc) {
      float f[8];
      unpack8<DT>(*reinterpret_cast<const uint4*>(As + (size_t)row * a.r + 8 * l), f);
      acc = dot8(f, uf);
    }
    for (int o = G >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (row < rows && l == 0) flag[row] = (acc + b1s[row] > 0.f) ? 1 : 0;
  }
}

// ------------------------------------------------------------ FFN rows
// Row-gather GEMV + ReLU and row-axpy over the m neurons listed in wl.
// Thread t owns the 16-byte column chunks t, t + kThreads, ... of every row;
// KC neurons are in flight at a time (all their W1 and W2 loads issued
// before any is used).  The per-neuron dot products are reduced across the
// block in a fixed order, so the result is deterministic.
template <int DT, bool GATED, int NCH, int KC>
__device__ void ffn_rows(const FfnArgs& a, const float* xs, const int* wl, int m, float* red,
                         float (&yacc)[NCH][8]) {
  constexpr int NV = GATED ? 2 : 1;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const size_t rs = GATED ? 2 * (size_t)a.d : (size_t)a.d;
  float xr[NCH][8];
  bool colok[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int cc = t + j * kThreads;
    colok[j] = cc < a.nch;
#pragma unroll
    for (int e = 0; e < 8; ++e) xr[j][e] = colok[j] ? xs[8 * cc + e] : 0.f;
  }
  int buf = 0;
  for (int base = 0; base < m; base += KC) {
    const int kc = min(KC, m - base);
    int nk[KC];
    float bk[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) nk[k] = (k < kc) ? wl[base + k] : -1;
#pragma unroll
    for (int k = 0; k < KC; ++k) bk[k] = (nk[k] >= 0) ? __ldg(a.b1 + nk[k]) : 0.f;
    uint4 w1[KC][NCH], wu[GATED ? KC : 1][NCH], w2[KC][NCH];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        w1[k][j] = z;
        w2[k][j] = z;
        if (GATED) wu[GATED ? k : 0][j] = z;
        if (nk[k] >= 0 && colok[j]) {
          const size_t col = 8 * (size_t)(t + j * kThreads);
          const size_t nrow = (size_t)nk[k];
          w1[k][j] = ld_stream(a.W1 + nrow * rs + col);
          if (GATED) wu[GATED ? k : 0][j] = ld_stream(a.W1 + nrow * rs + a.d + col);
          w2[k][j] = ld_stream(a.W2 + nrow * (size_t)a.d + col);
        }
      }
    }
    float pd[KC][NV];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        float f[8];
        unpack8<DT>(w1[k][j], f);
        s0 += dot8(f, xr[j]);
        if (GATED) {
          unpack8<DT>(wu[GATED ? k : 0][j], f);
          s1 += dot8(f, xr[j]);
        }
      }
      pd[k][0] = warp_sum(s0);
      if (GATED) pd[k][NV - 1] = warp_sum(s1);
    }
    float* rb = red + buf * (kWarps * KC * NV);
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < KC; ++k)
#pragma unroll
        for (int v = 0; v < NV; ++v) rb[(warp * KC + k) * NV + v] = pd[k][v];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      if (k < kc) {
        float s0 = 0.f, s1 = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          s0 += rb[(w * KC + k) * NV];
          if (GATED) s1 += rb[(w * KC + k) * NV + NV - 1];
        }
        float h = s0 + bk[k];
        h = h > 0.f ? h : 0.f;  // ReLU; ReLU(0) = 0
        if (GATED) h *= s1;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float f[8];
          unpack8<DT>(w2[k][j], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) yacc[j][e] = fmaf(h, f[e], yacc[j][e]);
        }
      }
    }
    buf ^= 1;
  }
}

// Sums the P partial rows in ascending block order (fixed split over
// threads), adds b2 and the residual, writes y.  Block c owns a slice of
// the d/4 float4 columns.
__device__ void final_reduce(const FfnArgs& a, float4* red4) {
  const int c = blockIdx.x, P = a.P;
  const int D4 = a.d >> 2;
  const int j0 = (int)((long long)c * D4 / P), j1 = (int)((long long)(c + 1) * D4 / P);
  constexpr int JB = 8, Q = kThreads / JB;
  const int jl = threadIdx.x % JB, q = threadIdx.x / JB;
  const int p0 = q * P / Q, p1 = (q + 1) * P / Q;
  for (int jb = j0; jb < j1; jb += JB) {
    const int j = jb + jl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < j1) {
      for (int p = p0; p < p1; ++p) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)p * a.d) + j);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    }
    red4[q * JB + jl] = acc;
    __syncthreads();
    if (q == 0 && j < j1) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int qq = 0; qq < Q; ++qq) {
        const float4 v = red4[qq * JB + jl];
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
      }
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
    __syncthreads();
  }
}

// ------------------------------------------------------------ persistent FFN kernel
// MODE kFused : predictor + compaction + sparse FFN of one token (one launch)
// MODE kSparse: sparse FFN over a given active list (idx_in, cnt_in)
// MODE kDense : FFN over all n neurons
// All P blocks must be co-resident (cooperative launch); the grid-wide waits
// are bounded by limit_ns.
template <int DT, bool GATED, int NCH, int KC, int MODE>
__global__ void __launch_bounds__(kThreads, 1) ffn_kernel(const FfnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* xs = reinterpret_cast<float*>(smem + a.o_xs);
  int* wl = reinterpret_cast<int*>(smem + a.o_wl);
  float* red = reinterpret_cast<float*>(smem + a.o_red);
  const int c = blockIdx.x, P = a.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int m = 0;

  if (MODE == kFused) {
    const int lo = (int)((long long)c * a.n / P), hi = (int)((long long)(c + 1) * a.n / P);
    const int rows = hi - lo;
    uint16_t* As = reinterpret_cast<uint16_t*>(smem + a.o_As);
    float* b1s = reinterpret_cast<float*>(smem + a.o_b1s);
    float* us = reinterpret_cast<float*>(smem + a.o_us);
    int* flag = reinterpret_cast<int*>(smem + a.o_flag);
    int* lst = reinterpret_cast<int*>(smem + a.o_lst);
    int* off = reinterpret_cast<int*>(smem + a.o_off);
    __shared__ int s_cnt;

    // The predictor's A rows and biases of this slice do not depend on x:
    // start fetching them now, behind stage 1.
    {
      const char* src = reinterpret_cast<const char*>(a.A + (size_t)lo * a.r);
      const int bytes = rows * a.r * 2;
      for (int o = threadIdx.x * 16; o < bytes; o += kThreads * 16)
        cp_async16(reinterpret_cast<char*>(As) + o, src + o);
      for (int i = threadIdx.x; i < rows; i += kThreads) cp_async4(b1s + i, a.b1 + lo + i);
      cp_async_commit();
    }
    // Hot block: bring this block's share of the hot rows of W1 and W2
    // towards the chip before the mask is known.
    if (a.hot > 0 && threadIdx.x == 0) {
      const int h0 = (int)((long long)c * a.hot / P), h1 = (int)((long long)(c + 1) * a.hot / P);
      if (h1 > h0) {
        const size_t rs = GATED ? 2 * (size_t)a.d : (size_t)a.d;
        prefetch_l2(a.W1 + (size_t)h0 * rs, (unsigned long long)(h1 - h0) * rs * 2);
        prefetch_l2(a.W2 + (size_t)h0 * a.d, (unsigned long long)(h1 - h0) * a.d * 2);
      }
    }
    for (int i = threadIdx.x; i < (a.d >> 2); i += kThreads)
      reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(a.x) + i);
    __syncthreads();

    fused_u<DT>(a, xs, red);
    if (!grid_sync(a.bar, (unsigned)P, a.status, a.limit_ns)) {
      cp_async_wait_all();
      return;
    }
    for (int k = threadIdx.x; k < a.r; k += kThreads) {
      float s = 0.f;
      for (int ss = 0; ss < a.S; ++ss) s += __ldcg(a.upart + k * a.S + ss);
      us[k] = s;
    }
    cp_async_wait_all();
    __syncthreads();
    fused_logits<DT>(a, As, b1s, us, flag, rows);
    __syncthreads();
    // ordered compaction of this slice: ballot + popc, one warp
    if (warp == 0) {
      int cnt = 0;
      for (int base = 0; base < rows; base += 32) {
        const int i = base + lane;
        const bool f = (i < rows) && flag[i];
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
        if (f) {
          lst[pos] = lo + i;
          __stcg(a.loc_idx + lo + pos, lo + i);
        }
        cnt += __popc(bal);
      }
      if (lane == 0) {
        s_cnt = cnt;
        __stcg(a.loc_cnt + c, cnt);
      }
    }
    if (!grid_sync(a.bar, (unsigned)P, a.status, a.limit_ns)) return;
    // exclusive scan of the P slice counts (one warp)
    if (warp == 0) {
      int run = 0;
      if (lane == 0) off[0] = 0;
      for (int base = 0; base < P; base += 32) {
        const int b = base + lane;
        int v = (b < P) ? __ldcg(a.loc_cnt + b) : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        if (b < P) off[b + 1] = run + incl;
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
    const int total = off[P];
    if (a.idx_out)
      for (int k = threadIdx.x; k < s_cnt; k += kThreads) a.idx_out[off[c] + k] = lst[k];
    if (a.cnt_out && c == 0 && threadIdx.x == 0) a.cnt_out[0] = total;
    // even split of the global active list over the grid
    const long long p0 = (long long)c * total / P, p1 = (long long)(c + 1) * total / P;
    m = (int)(p1 - p0);
    for (int k = threadIdx.x; k < m; k += kThreads) {
      const int p = (int)(p0 + k);
      int lo_b = 0, hi_b = P - 1;  // largest b with off[b] <= p
      while (lo_b < hi_b) {
        const int mid = (lo_b + hi_b + 1) >> 1;
        if (off[mid] <= p) lo_b = mid; else hi_b = mid - 1;
      }
      const int slo = (int)((long long)lo_b * a.n / P);
      wl[k] = __ldcg(a.loc_idx + slo + (p - off[lo_b]));
    }
  } else {
    for (int i = threadIdx.x; i < (a.d >> 2); i += kThreads)
      reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(a.x) + i);
    int total;
    if (MODE == kSparse) {
      total = __ldg(a.cnt_in);
      if (total < 0 || total > a.cap || total > a.n) {
        if (c == 0 && threadIdx.x == 0) set_status(a.status, PI_ERR_CAPACITY);
        return;  // uniform over the grid: no block reaches a grid-wide wait
      }
    } else {
      total = a.n;
    }
    const long long p0 = (long long)c * total / P, p1 = (long long)(c + 1) * total / P;
    m = (int)(p1 - p0);
    for (int k = threadIdx.x; k < m; k += kThreads) {
      int v = (MODE == kSparse) ? __ldg(a.idx_in + p0 + k) : (int)(p0 + k);
      if ((unsigned)v >= (unsigned)a.n) {  // never read outside the matrices
        set_status(a.status, PI_ERR_INDEX);
        v = -1;
      }
      wl[k] = v;
    }
  }
  __syncthreads();

  float yacc[NCH][8];
#pragma unroll
  for (int j = 0; j < NCH; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) yacc[j][e] = 0.f;
  ffn_rows<DT, GATED, NCH, KC>(a, xs, wl, m, red, yacc);

#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int cc = threadIdx.x + j * kThreads;
    if (cc < a.nch) {
      float4* dst = reinterpret_cast<float4*>(a.part + (size_t)c * a.d + 8 * (size_t)cc);
      __stcg(dst, make_float4(yacc[j][0], yacc[j][1], yacc[j][2], yacc[j][3]));
      __stcg(dst + 1, make_float4(yacc[j][4], yacc[j][5], yacc[j][6], yacc[j][7]));
    }
  }
  if (!grid_sync(a.bar, (unsigned)P, a.status, a.limit_ns)) return;
  final_reduce(a, reinterpret_cast<float4*>(red));
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
  extern __shared__ __align__(16) unsigned char smem[];
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

// Failure-path diagnostic: one grid-wide wait whose last arrival never
// comes (expected = grid + 1), so every block gives up after limit_ns.
__global__ void wait_timeout_kernel(GridBar bar, int* status, unsigned long long limit_ns) {
  grid_sync(bar, gridDim.x + 1u, status, limit_ns);
}

}  // namespace pik

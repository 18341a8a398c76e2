// batched.cuh — batched decode (2 <= batch <= 32) of the activation-sparse
// FFN on tensor cores.
//
// Every token keeps its own predicted mask; the union of the tokens' active
// neurons is read once and turned into a dense tile contraction:
//   phase 1  H[u][t] = mask_t(u) ? act(W1[U_u] . x_t + b1[U_u]) : 0
//            (act = ReLU, or ReLU(gate) * up), one tile of 64 union neurons
//            at a time, A = activations (tokens x d), B = W1 rows;
//   phase 2  Y_g[t][cols] = sum_{u in group g} H[u][t] W2[U_u][cols]
//            over 8 neuron groups x (P / 8) column slices;
//   phase 3  y[t] = b2 + sum_g Y_g[t] (g ascending) (+ residual).
// Tensor-core operands are 16-bit: x and H are split into a high and a low
// 16-bit part (x = hi + lo), so each product is taken twice and the sum keeps
// about 16 more bits than one rounding would.  mma.sync m16n8k16 with fp32
// accumulation; operands staged in shared memory by cp.async, fragments by
// ldmatrix (rows padded by 16 bytes: conflict-free).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace pik {

constexpr int kBT = 64;          // union neurons per phase-1 tile
constexpr int kBK = 128;         // columns per phase-1 chunk (256 for plain layers, d % 256 == 0)
constexpr int kBStages = 3;      // cp.async pipeline depth (measured: deeper was not faster)
constexpr int kBN2 = 64;         // union neurons per phase-2 chunk
constexpr int kGroups2 = 8;      // neuron groups of phase 2

struct BatchArgs {
  int d, n, batch, bp;        // bp: batch padded to 16 or 32 (rows of the A operand)
  int P;                      // phase-1 grid; phase-2 grid = kGroups2 * slices
  int slices, cw;             // phase-2 column slices and their width (multiple of 8)
  int packed;                 // PI_LAYOUT_PACKED
  int rec;                    // elements per packed record ((gated ? 3 : 2) d)
  const uint16_t* W1;
  const uint16_t* W2;
  const float* b1;
  const float* b2;
  const float* x;             // [batch][d]
  const float* residual;      // [batch][d] or NULL
  float* y;                   // [batch][d]
  const int* uidx;            // union neurons, ascending
  const int* ucnt;            // union count (device)
  int dense;                  // 1: all n neurons, every token (uidx / ucnt / tmask unused)
  int tc_cols;                // tensor-memory columns of the tcgen05 phase 1
  unsigned long long limit_ns;  // bound of every wait (tcgen05 phase 1)
  const uint32_t* tmask;      // token bitmask per union position
  uint16_t* xhi;              // [bp][d] activations, high and low 16-bit parts
  uint16_t* xlo;
  uint16_t* hhi;              // [bp][hs] H transposed (token-major), high / low parts
  uint16_t* hlo;
  int hs;                     // row stride of hhi / hlo (>= n + kBN2, multiple of 8)
  float* part;                // [kGroups2][bp][d]
  int* status;
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}

// D += A (16x16, row) * B (16x8, col), 16-bit inputs, fp32 accumulate.
template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  if (DT == 0)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// v = hi + lo with hi, lo 16-bit (lo = the rounding error of hi).
template <int DT>
__device__ __forceinline__ void split16(float v, uint16_t* hi, uint16_t* lo) {
  if (DT == 0) {
    const __half h = __float2half_rn(v);
    const __half l = __float2half_rn(v - __half2float(h));
    *hi = __half_as_ushort(h);
    *lo = __half_as_ushort(l);
  } else {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    *hi = __bfloat16_as_ushort(h);
    *lo = __bfloat16_as_ushort(l);
  }
}

// ---------------------------------------------------------------- batched predictor
// Stage 1 split over the columns: block c of G owns the 8-column chunks
// [c nch / G, (c+1) nch / G) and writes the partial u of every (token, k),
// part[c][t][k]; thread k keeps the batch's sums in registers, x's columns
// of the block are staged in shared memory.  With xhi non-NULL the block
// also writes the high / low 16-bit parts of its columns of x for the FFN
// phases ([bp][d], zero rows for padded tokens: the operand split of phase
// 0, done here while x is at hand).
template <int DT, int TB>
__global__ void __launch_bounds__(256) bpu_partial_kernel(const uint16_t* Bm, const float* x, int d,
                                                          int r, int batch, int G, float* part,
                                                          uint16_t* xhi, uint16_t* xlo, int bp) {
  extern __shared__ __align__(16) float xs[];  // [batch][w]
  const int c = blockIdx.x, tid = threadIdx.x, nch = d >> 3;
  const int q0 = (int)((long long)c * nch / G), q1 = (int)((long long)(c + 1) * nch / G);
  const int nq = q1 - q0, w = nq * 8;
  // the block's columns of Bm (weights, not written by the kernels before
  // this one) head for L2 while those finish; x after the wait
  for (int k = tid; k < r; k += 256) {
    const char* p0 = reinterpret_cast<const char*>(Bm + (size_t)k * d + 8 * q0);
    const char* p1 = p0 + 16 * nq;  // every address prefetched lies in [p0, p1)
    for (const char* p = p0; p < p1; p += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    if (nq > 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(p1 - 16));
  }
  pdl_enter();
  for (int e = tid; e < batch * w; e += 256) {
    const int t = e / w, j = e - t * w;
    xs[e] = x[(size_t)t * d + 8 * q0 + j];
  }
  __syncthreads();
  if (xhi) {
    for (int e = tid; e < bp * w; e += 256) {
      const int t = e / w, j = e - t * w;
      uint16_t hi = 0, lo = 0;
      if (t < batch) split16<DT>(xs[e], &hi, &lo);
      const size_t o = (size_t)t * d + 8 * q0 + j;
      xhi[o] = hi;
      xlo[o] = lo;
    }
  }
  for (int k = tid; k < r; k += 256) {
    float acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.f;
    const uint16_t* row = Bm + (size_t)k * d + 8 * q0;
    for (int q = 0; q < nq; ++q) {
      float f[8];
      unpack8<DT>(ld_nc(row + 8 * q), f);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        if (t < batch) {
          float xv[8];
          load8(xs + t * w + 8 * q, xv);
          acc[t] += dot8(f, xv);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TB; ++t)
      if (t < batch) part[((size_t)c * batch + t) * r + k] = acc[t];
  }
}

// u[t][k] = sum_c part[c][t][k], then its high / low 16-bit parts for the
// tensor cores ([bp][r]; zero rows for padded tokens).  Block = 32 outputs
// e = t r + k (consecutive, so every load of a warp is one 128-byte line);
// warp w sums c = w, w + 8, ...; the 8 warp sums are added in warp order.
template <int DT>
__global__ void __launch_bounds__(256) bpu_reduce_kernel(const float* part, int r, int batch, int bp,
                                                         int G, uint16_t* uhi, uint16_t* ulo) {
  pdl_enter();
  __shared__ float ws[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;  // t * r + k
  const int tot = batch * r;             // partials hold the real tokens only
  float s = 0.f;
  if (e < tot) {
#pragma unroll 4
    for (int c = warp; c < G; c += 8) s += part[(size_t)c * tot + e];
  }
  ws[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < bp * r) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += ws[w][lane];
    uint16_t hi, lo;
    split16<DT>(v, &hi, &lo);  // padded tokens (e >= tot): 0
    uhi[e] = hi;
    ulo[e] = lo;
  }
}

// logits[t][i] = A_i . u[t] + b1_i on the tensor cores: block = 64 neurons x
// all tokens, K = r.  A rows (the B operand, one neuron per row) and u's
// high / low parts (the A operand, one token per row) staged in shared
// memory with 16-byte row padding; warp w takes neurons 8w .. 8w + 7.
constexpr int kLT = 64;
template <int DT, int MT>
__global__ void __launch_bounds__(256) blogit_kernel(const uint16_t* A, const float* b1,
                                                     const uint16_t* uhi, const uint16_t* ulo, int n,
                                                     int r, int batch, int bp, float* logits) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rowb = 2 * r + 16;
  unsigned char* As = smem;               // [kLT][rowb]
  unsigned char* Us = smem + kLT * rowb;  // [2 bp][rowb]: high parts, then low parts
  const int i0 = blockIdx.x * kLT;
  const int tn = min(kLT, n - i0);
  const int pcs = r >> 3;
  // the A rows (weights, not written by the kernels before this one) load
  // while those finish; u after the wait
  for (int e = tid; e < kLT * pcs; e += 256) {
    const int row = e / pcs, pc = e - row * pcs;
    unsigned char* dst = As + (size_t)row * rowb + 16 * pc;
    if (row < tn) cp_async16(dst, A + (size_t)(i0 + row) * r + 8 * pc);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_enter();
  for (int e = tid; e < 2 * bp * pcs; e += 256) {
    const int rw = e / pcs, pc = e - rw * pcs;
    const int prt = rw / bp, t = rw - prt * bp;
    cp_async16(Us + (size_t)rw * rowb + 16 * pc, (prt == 0 ? uhi : ulo) + (size_t)t * r + 8 * pc);
  }
  cp_async_commit();
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  float acc[MT][4], accl[MT][4];  // products of the high / low parts (independent chains)
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[m][e] = accl[m][e] = 0.f;
  for (int ks = 0; ks < (r >> 4); ++ks) {
    uint32_t b[2];
    ldsm_x2(b, As + (size_t)(warp * 8 + (lane & 7)) * rowb + (ks * 16 + 8 * ((lane >> 3) & 1)) * 2);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      uint32_t ah[4], al[4];
      const int rr = m * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int cb = (ks * 16 + 8 * (lane >> 4)) * 2;
      ldsm_x4(ah, Us + (size_t)rr * rowb + cb);
      ldsm_x4(al, Us + (size_t)(bp + rr) * rowb + cb);
      mma16816<DT>(acc[m], ah, b);
      mma16816<DT>(accl[m], al, b);
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[m][e] += accl[m][e];
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = m * 16 + g + 8 * (e >> 1);
      const int col = warp * 8 + 2 * tq + (e & 1);
      if (t < batch && col < tn)
        logits[(size_t)t * n + i0 + col] = acc[m][e] + __ldg(b1 + i0 + col);
    }
}

// ---------------------------------------------------------------- phase 0
// xhi/xlo[t][j] = split(x[t][j]) for t < batch, 0 for padded rows.
template <int DT>
__global__ void bsplit_x_kernel(const BatchArgs a) {
  pdl_enter();
  const long long tot = (long long)a.bp * a.d;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / a.d);
    uint16_t hi = 0, lo = 0;
    if (t < a.batch) split16<DT>(a.x[e], &hi, &lo);
    a.xhi[e] = hi;
    a.xlo[e] = lo;
  }
}

// ---------------------------------------------------------------- phase 1
// Shared-memory layout of one pipeline stage: W1 rows [kBT][kBK] (gated:
// gate rows then up rows), then x high / low parts [bp][kBK]; rows padded by
// 16 bytes.
template <int BK>
__host__ __device__ constexpr int bup_row_bytes() {
  return BK * 2 + 16;  // bytes per staged row
}
template <bool GATED, int BK>
__host__ __device__ constexpr int bup_stage_bytes(int bp) {
  return ((GATED ? 2 : 1) * kBT + 2 * bp) * bup_row_bytes<BK>();
}

template <int DT, bool GATED, int MT, int BK>
__global__ void __launch_bounds__(512, 1) bup_kernel(const BatchArgs a) {
  pdl_enter();
  constexpr int kRowB = bup_row_bytes<BK>();
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = a.dense ? a.n : __ldg(a.ucnt);
  const int lo_u = (int)((long long)blockIdx.x * U / a.P);
  const int hi_u = (int)((long long)(blockIdx.x + 1) * U / a.P);
  const int stage_bytes = bup_stage_bytes<GATED, BK>(a.bp);
  constexpr int NW = GATED ? 2 : 1;
  const int ksteps = BK / 16;
  const int nchunks = a.d / BK;
  constexpr int S = kBStages;
  constexpr int CV = NW * MT * 2 * 4;  // accumulator values per lane
  // the k slices' partial sums [KQ - 1][NG][32][CV], in the stages (free
  // between a tile's last chunk and the next tile's first copies)
  float* comb = reinterpret_cast<float*>(smem);
  const size_t w1s = a.packed ? (size_t)a.rec : (GATED ? 2 * (size_t)a.d : (size_t)a.d);

  for (int t0 = lo_u; t0 < hi_u; t0 += kBT) {
    const int tn = min(kBT, hi_u - t0);
    // warp -> (n group ng of 16 rows: n tiles 2 ng and 2 ng + 1; k slice
    // kq: k-steps kq, kq + KQ, ...): NG groups cover the tile's rows, so a
    // tile with few rows (a sparse union) spreads its K over more warps;
    // every m tile: one x fragment feeds 2 NW products per part, the B
    // fragments of both n tiles come in one ldmatrix.x4
    const int lg = tn <= 16 ? 0 : (tn <= 32 ? 1 : 2);
    const int NG = 1 << lg, KQ = 16 >> lg;
    const int ng = warp & (NG - 1), kq = warp >> lg;
    // issue the cp.async loads of chunk ch into stage ch % S
    auto issue = [&](int ch) {
      unsigned char* st = smem + (ch % S) * stage_bytes;
      const int k0 = ch * BK;
      constexpr int CPR = BK / 8;  // 16-byte pieces per row
      for (int e = tid; e < NW * kBT * CPR; e += 512) {
        const int rw = e / CPR, pc = e - rw * CPR;
        const int w = rw / kBT, row = rw - w * kBT;
        unsigned char* dst = st + (size_t)rw * kRowB + 16 * pc;
        if (row < tn) {
          const int nid = a.dense ? t0 + row : __ldg(a.uidx + t0 + row);
          cp_async16(dst, a.W1 + (size_t)nid * w1s + (size_t)w * a.d + k0 + 8 * pc);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      unsigned char* xs_ = st + (size_t)NW * kBT * kRowB;
      for (int e = tid; e < 2 * a.bp * CPR; e += 512) {
        const int rw = e / CPR, pc = e - rw * CPR;
        const int part = rw / a.bp, t = rw - part * a.bp;
        const uint16_t* src = (part == 0 ? a.xhi : a.xlo) + (size_t)t * a.d + k0 + 8 * pc;
        cp_async16(xs_ + (size_t)rw * kRowB + 16 * pc, src);
      }
    };
    // products of the high / low parts (independent chains), [w][m][n tile][e]
    float acc[NW][MT][2][4], accl[NW][MT][2][4];
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[w][m][j][e] = accl[w][m][j][e] = 0.f;
    for (int ch = 0; ch < S - 1; ++ch) {  // always S - 1 groups
      if (ch < nchunks) issue(ch);
      cp_async_commit();
    }
    for (int ch = 0; ch < nchunks; ++ch) {
      if (ch + S - 1 < nchunks) issue(ch + S - 1);
      cp_async_commit();
      asm volatile("cp.async.wait_group %0;" ::"n"(kBStages - 1) : "memory");
      __syncthreads();
      const unsigned char* st = smem + (ch % S) * stage_bytes;
      const unsigned char* xs_ = st + (size_t)NW * kBT * kRowB;
      for (int ks = kq; ks < ksteps; ks += KQ) {
        uint32_t ah[MT][4], al[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          // A fragment rows: tokens m*16 .. +15, columns ks*16 .. +15
          const int r = m * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int cbyte = (ks * 16 + 8 * (lane >> 4)) * 2;
          ldsm_x4(ah[m], xs_ + (size_t)r * kRowB + cbyte);
          ldsm_x4(al[m], xs_ + (size_t)(a.bp + r) * kRowB + cbyte);
        }
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          // B fragments of n tiles 2 ng (b4[0..1]) and 2 ng + 1 (b4[2..3]):
          // neurons ng*16 .. +15 (rows), k = ks*16 .. +15
          uint32_t b4[4];
          const int r = w * kBT + ng * 16 + (lane & 7) + 8 * (lane >> 4);
          const int cbyte = (ks * 16 + 8 * ((lane >> 3) & 1)) * 2;
          ldsm_x4(b4, st + (size_t)r * kRowB + cbyte);
          const uint32_t b0[2] = {b4[0], b4[1]}, b1[2] = {b4[2], b4[3]};
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            mma16816<DT>(acc[w][m][0], ah[m], b0);
            mma16816<DT>(accl[w][m][0], al[m], b0);
            mma16816<DT>(acc[w][m][1], ah[m], b1);
            mma16816<DT>(accl[w][m][1], al[m], b1);
          }
        }
      }
      __syncthreads();
    }
    // high + low, then the KQ k slices meet in a fixed order (0, 1, ...)
    float v[CV];
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[((w * MT + m) * 2 + jn) * 4 + e] = acc[w][m][jn][e] + accl[w][m][jn][e];
    if (kq > 0) {
      float* cp = comb + ((size_t)((kq - 1) * NG + ng) * 32 + lane) * CV;
#pragma unroll
      for (int e = 0; e < CV; ++e) cp[e] = v[e];
    }
    __syncthreads();
    if (kq == 0) {
      for (int q = 1; q < KQ; ++q) {
        const float* cp = comb + ((size_t)((q - 1) * NG + ng) * 32 + lane) * CV;
#pragma unroll
        for (int e = 0; e < CV; ++e) v[e] += cp[e];
      }
      // epilogue: bias, activation, the token's own mask bit, split, store H^T
      const int g = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = m * 16 + g + 8 * (e >> 1);                 // token
            const int col = (2 * ng + jn) * 8 + 2 * tq + (e & 1);    // neuron within the tile
            if (col < tn && t < a.batch) {
              const int pos = t0 + col;
              const int nid = a.dense ? pos : __ldg(a.uidx + pos);
              float h = v[((0 * MT + m) * 2 + jn) * 4 + e] + __ldg(a.b1 + nid);
              h = h > 0.f ? h : 0.f;  // ReLU; ReLU(0) = 0
              if (GATED) h *= v[(((NW - 1) * MT + m) * 2 + jn) * 4 + e];
              if (!a.dense && !((__ldg(a.tmask + pos) >> t) & 1u)) h = 0.f;  // token t skips it
              uint16_t hh, hl;
              split16<DT>(h, &hh, &hl);
              a.hhi[(size_t)t * a.hs + pos] = hh;
              a.hlo[(size_t)t * a.hs + pos] = hl;
            }
          }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- phase 2
// Block (g, s): union positions of group g, columns [s cw, s cw + cw).
// Stage: W2 rows [kBN2][cw] then H^T high / low [bp][kBN2], rows padded.
__host__ __device__ inline int bdn_w2_row(int cw) { return cw * 2 + 16; }
constexpr int kHRowB = kBN2 * 2 + 16;
__host__ __device__ inline int bdn_stage_bytes(int cw, int bp) {
  return kBN2 * bdn_w2_row(cw) + 2 * bp * kHRowB;
}

template <int DT, int MT>
__global__ void __launch_bounds__(512, 1) bdown_kernel(const BatchArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x / a.slices, s = blockIdx.x - g * a.slices;
  const int U = a.dense ? a.n : __ldg(a.ucnt);
  // group boundaries on multiples of 8 positions: every 16-byte piece of an
  // H^T row starts 16-byte aligned; the last group ends at U
  const int lo_u = (int)((long long)g * U / kGroups2) & ~7;
  const int hi_u = (g == kGroups2 - 1) ? U : ((int)((long long)(g + 1) * U / kGroups2) & ~7);
  const int c0 = s * a.cw;
  const int cn = min(a.cw, a.d - c0);  // columns of this slice (multiple of 8)
  if (cn <= 0) return;
  const int NT = cn / 8;
  const int w2row = bdn_w2_row(a.cw);
  const int stage_bytes = bdn_stage_bytes(a.cw, a.bp);
  constexpr int S = kBStages;
  const size_t w2s = a.packed ? (size_t)a.rec : (size_t)a.d;  // W2 rows (packed: inside records)
  const uint16_t* w2base = a.W2;
  // warp w owns the n-tile pairs w and w + 16 (tiles 2p, 2p + 1 < NT), all
  // m tiles; one ldmatrix.x4.trans loads the B fragments of a pair
  constexpr int NPW = 2;
  // high / low part products (independent chains), [pair][tile][m][e]
  float acc[NPW][2][MT][4], accl[NPW][2][MT][4];
#pragma unroll
  for (int q = 0; q < NPW; ++q)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[q][j][m][e] = accl[q][j][m][e] = 0.f;
  const int nchunks = (hi_u - lo_u + kBN2 - 1) / kBN2;
  auto issue = [&](int ch) {
    unsigned char* st = smem + (ch % S) * stage_bytes;
    const int p0 = lo_u + ch * kBN2;
    const int cpr = cn / 8;  // 16-byte pieces per W2 row piece
    for (int e = tid; e < kBN2 * cpr; e += 512) {
      const int row = e / cpr, pc = e - row * cpr;
      unsigned char* dst = st + (size_t)row * w2row + 16 * pc;
      if (p0 + row < hi_u) {
        const int nid = a.dense ? p0 + row : __ldg(a.uidx + p0 + row);
        cp_async16(dst, w2base + (size_t)nid * w2s + c0 + 8 * pc);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    unsigned char* hs_ = st + (size_t)kBN2 * w2row;
    constexpr int HPR = kBN2 / 8;
    for (int e = tid; e < 2 * a.bp * HPR; e += 512) {
      const int rw = e / HPR, pc = e - rw * HPR;
      const int part = rw / a.bp, t = rw - part * a.bp;
      unsigned char* dst = hs_ + (size_t)rw * kHRowB + 16 * pc;
      const int q0 = p0 + 8 * pc;  // first position of the piece (multiple of 8)
      const uint16_t* src = (part == 0 ? a.hhi : a.hlo) + (size_t)t * a.hs + q0;
      if (q0 + 8 <= hi_u) {
        cp_async16(dst, src);
      } else if (q0 >= hi_u) {
        // past the group: never written by phase 1 for this call
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      } else {
        // the piece that holds the union end (last group only)
        uint16_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (q0 + i < hi_u) ? src[i] : (uint16_t)0;
        uint4 pk;
        pk.x = v[0] | ((uint32_t)v[1] << 16);
        pk.y = v[2] | ((uint32_t)v[3] << 16);
        pk.z = v[4] | ((uint32_t)v[5] << 16);
        pk.w = v[6] | ((uint32_t)v[7] << 16);
        *reinterpret_cast<uint4*>(dst) = pk;
      }
    }
  };
  for (int ch = 0; ch < S - 1; ++ch) {  // always S - 1 groups
    if (ch < nchunks) issue(ch);
    cp_async_commit();
  }
  for (int ch = 0; ch < nchunks; ++ch) {
    if (ch + S - 1 < nchunks) issue(ch + S - 1);
    cp_async_commit();
    asm volatile("cp.async.wait_group %0;" ::"n"(kBStages - 1) : "memory");
    __syncthreads();
    const unsigned char* st = smem + (ch % S) * stage_bytes;
    const unsigned char* hs_ = st + (size_t)kBN2 * w2row;
#pragma unroll
    for (int ks = 0; ks < kBN2 / 16; ++ks) {
      uint32_t ah[MT][4], al[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int r = m * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int cbyte = (ks * 16 + 8 * (lane >> 4)) * 2;
        ldsm_x4(ah[m], hs_ + (size_t)r * kHRowB + cbyte);
        ldsm_x4(al[m], hs_ + (size_t)(a.bp + r) * kHRowB + cbyte);
      }
#pragma unroll
      for (int q = 0; q < NPW; ++q) {
        const int pr = warp + 16 * q;
        if (2 * pr < NT) {
          // W2 stored [k = neuron][n = column]: transposed loads give the
          // (k pair, n) layout of the B operand; matrices 0/1: tile 2 pr,
          // 2/3: tile 2 pr + 1 (within the padded row even past NT)
          uint32_t b4[4];
          const int kr = ks * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(b4, st + (size_t)kr * w2row + (2 * pr + (lane >> 4)) * 16);
          const uint32_t b0[2] = {b4[0], b4[1]}, b1[2] = {b4[2], b4[3]};
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            mma16816<DT>(acc[q][0][m], ah[m], b0);
            mma16816<DT>(accl[q][0][m], al[m], b0);
            mma16816<DT>(acc[q][1][m], ah[m], b1);
            mma16816<DT>(accl[q][1][m], al[m], b1);
          }
        }
      }
    }
    __syncthreads();
  }
  // partial Y of group g, this slice
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int q = 0; q < NPW; ++q)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ntile = 2 * (warp + 16 * q) + j;
      if (ntile < NT) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = m * 16 + gq + 8 * (e >> 1);
            const int col = c0 + ntile * 8 + 2 * tq + (e & 1);
            a.part[((size_t)g * a.bp + t) * a.d + col] = acc[q][j][m][e] + accl[q][j][m][e];
          }
      }
    }
}

// ---------------------------------------------------------------- phase 3
__global__ void bsum_kernel(const BatchArgs a) {
  pdl_enter();
  const long long tot = (long long)a.batch * a.d;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
       e += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(e / a.d), j = (int)(e - (long long)t * a.d);
    float s = 0.f;
    for (int g = 0; g < kGroups2; ++g) s += a.part[((size_t)g * a.bp + t) * a.d + j];
    if (a.b2) s += a.b2[j];
    if (a.residual) s += a.residual[e];
    a.y[e] = s;
  }
}

}  // namespace pik

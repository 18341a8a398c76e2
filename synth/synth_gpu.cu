// synth_gpu.cu — the seeded workload generator of synth.c, on the GPU, for
// layers too large to generate on the host in reasonable time (the 48-layer
// OPT-30B-shaped stack).  Inputs only: none of the method's arithmetic.
//
// Same definitions as synth.c, element for element: SplitMix64 counter
// streams, Box–Muller normals, W1 = round(A64 Bm64 + noise N(0,1/d)) with the
// k-sum in ascending order, every multiply and add rounded on its own
// (__dmul_rn / __dadd_rn, as the host build with -ffp-contract=off), and the
// same round-to-nearest-even bit-field encoding.  The only possible
// difference from the host bytes comes from log / sin / cos, whose last-bit
// rounding may differ between libraries; tests bound how often that shows up
// after rounding to 16 bits.
#include <cuda_runtime.h>
#include <stdint.h>

#define SY_GAMMA 0x9e3779b97f4a7c15ULL

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ double uniform(uint64_t key, uint64_t k) {
  const uint64_t b = mix64(key + (k + 1u) * SY_GAMMA);
  return __dmul_rn(__dadd_rn((double)(b >> 11), 0.5), 0x1.0p-53);
}

__device__ __forceinline__ double normal(uint64_t key, uint64_t k) {
  const uint64_t m = k >> 1;
  const double u1 = uniform(key, 2 * m), u2 = uniform(key, 2 * m + 1);
  const double rad = __dsqrt_rn(__dmul_rn(-2.0, log(u1)));
  const double th = __dmul_rn(6.283185307179586476925286766559, u2);
  return (k & 1u) ? __dmul_rn(rad, sin(th)) : __dmul_rn(rad, cos(th));
}

// Round-to-nearest-even onto a 16-bit binary format (mbits stored mantissa
// bits, exponent bias `bias`, all-ones exponent emax), from the bit fields.
__device__ uint16_t round_binary(double v, int mbits, int bias, int emax) {
  const uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0u;
  const uint16_t inf = (uint16_t)((uint32_t)emax << mbits);
  if (isnan(v)) return (uint16_t)(inf | (1u << (mbits - 1)));
  const double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | inf);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);
  int q = (e - 1) - mbits;
  const int qmin = 1 - bias - mbits;
  if (q < qmin) q = qmin;
  const double m = rint(ldexp(a, -q));
  uint64_t mant = (uint64_t)m;
  uint32_t out;
  if (q == qmin) {
    out = (uint32_t)mant;
  } else {
    int E = q + mbits + bias;
    if (mant == (1ull << (mbits + 1))) {
      mant >>= 1;
      E += 1;
    }
    if (E >= emax) return (uint16_t)(sign | inf);
    out = ((uint32_t)E << mbits) | (uint32_t)(mant - (1ull << mbits));
  }
  if (out >= inf) return (uint16_t)(sign | inf);
  return (uint16_t)(sign | out);
}

__device__ __forceinline__ uint16_t round_half(double v, int dtype) {
  return dtype == 1 ? round_binary(v, 7, 127, 255) : round_binary(v, 10, 15, 31);
}

// out[e] = scale * N(key, base + e) in fp64
__global__ void normals_f64(uint64_t key, long long count, double scale, double* out) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < count;
       e += (long long)gridDim.x * blockDim.x)
    out[e] = __dmul_rn(scale, normal(key, (uint64_t)e));
}

// bits[e] = round(f64[e])
__global__ void round_f64(const double* in, long long count, int dtype, uint16_t* out) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < count;
       e += (long long)gridDim.x * blockDim.x)
    out[e] = round_half(in[e], dtype);
}

// bits[i][j] (row stride `stride`) = round(scale * N(key, i d + j))
__global__ void normal_rows(uint64_t key, int n, int d, double scale, int dtype, uint16_t* out,
                            long long stride) {
  const long long tot = (long long)n * d;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < tot;
       e += (long long)gridDim.x * blockDim.x) {
    const long long i = e / d, j = e - i * d;
    out[i * stride + j] = round_half(__dmul_rn(scale, normal(key, (uint64_t)e)), dtype);
  }
}

// W1[i][j] = round(sum_k A64[i][k] Bm64[k][j] (k ascending) + noise * (sd * N(kN, i d + j)))
// Tiles of 32 rows x 64 columns; A and Bm tiles staged in shared memory.
__global__ void __launch_bounds__(256) w1_kernel(const double* A64, const double* B64, int n, int d,
                                                 int r, uint64_t kN, double sd, double noise,
                                                 int dtype, uint16_t* W1, long long stride) {
  __shared__ double As[32][33];
  __shared__ double Bs[32][64];
  const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 64;
  const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;  // 64 columns x 4 row groups
  double acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.0;
  for (int k0 = 0; k0 < r; k0 += 32) {
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      const int ii = e / 32, kk = e % 32;
      As[ii][kk] = (i0 + ii < n && k0 + kk < r) ? A64[(long long)(i0 + ii) * r + k0 + kk] : 0.0;
    }
    for (int e = threadIdx.x; e < 32 * 64; e += 256) {
      const int kk = e / 64, jj = e % 64;
      Bs[kk][jj] = (k0 + kk < r && j0 + jj < d) ? B64[(long long)(k0 + kk) * d + j0 + jj] : 0.0;
    }
    __syncthreads();
    const int kmax = (r - k0) < 32 ? (r - k0) : 32;
    for (int kk = 0; kk < kmax; ++kk) {
      const double b = Bs[kk][tx];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = __dadd_rn(acc[q], __dmul_rn(As[ty * 8 + q][kk], b));
    }
    __syncthreads();
  }
  const int j = j0 + tx;
  if (j >= d) return;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = i0 + ty * 8 + q;
    if (i < n) {
      const double nz = __dmul_rn(sd, normal(kN, (uint64_t)((long long)i * d + j)));
      W1[(long long)i * stride + j] = round_half(__dadd_rn(acc[q], __dmul_rn(noise, nz)), dtype);
    }
  }
}

uint64_t host_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

uint64_t stream_key(uint64_t seed, uint32_t tag, uint32_t layer) {
  const uint64_t k = host_mix64(seed + SY_GAMMA);
  const uint64_t id = ((uint64_t)tag << 32) | (uint64_t)layer;
  return host_mix64(k + (id + 1u) * SY_GAMMA);
}

}  // namespace

extern "C" {

// Writes one layer's A [n][r], Bm [r][d], W1 [n][d] (gated [n][2][d]) and
// W2 [n][d] as 16-bit patterns into device buffers (b1 / b2 are made on the
// host: they are small).  A64 / B64 are caller-provided device scratch of
// n r and r d doubles.  Returns a cudaError_t value (0 = success).
int sy_gpu_gen_layer(int d, int n, int r, int dtype, int gated, int layer, uint64_t seed,
                     double noise, uint16_t* A, uint16_t* Bm, uint16_t* W1, uint16_t* W2,
                     double* A64, double* B64, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint64_t kA = stream_key(seed, 1, (uint32_t)layer), kB = stream_key(seed, 2, (uint32_t)layer);
  const uint64_t kN = stream_key(seed, 3, (uint32_t)layer), kW2 = stream_key(seed, 4, (uint32_t)layer);
  const uint64_t kU = stream_key(seed, 5, (uint32_t)layer);
  const double sr = 1.0 / sqrt((double)r), sd = 1.0 / sqrt((double)d), sn = 1.0 / sqrt((double)n);
  const int blocks = 152 * 8;
  normals_f64<<<blocks, 256, 0, st>>>(kA, (long long)n * r, sr, A64);
  normals_f64<<<blocks, 256, 0, st>>>(kB, (long long)r * d, sd, B64);
  round_f64<<<blocks, 256, 0, st>>>(A64, (long long)n * r, dtype, A);
  round_f64<<<blocks, 256, 0, st>>>(B64, (long long)r * d, dtype, Bm);
  const long long stride = gated ? 2LL * d : (long long)d;
  dim3 grid((unsigned)((d + 63) / 64), (unsigned)((n + 31) / 32));
  w1_kernel<<<grid, 256, 0, st>>>(A64, B64, n, d, r, kN, sd, noise, dtype, W1, stride);
  if (gated) normal_rows<<<blocks, 256, 0, st>>>(kU, n, d, sd, dtype, W1 + d, stride);
  normal_rows<<<blocks, 256, 0, st>>>(kW2, n, d, sn, dtype, W2, (long long)d);
  return (int)cudaGetLastError();
}

}  // extern "C"

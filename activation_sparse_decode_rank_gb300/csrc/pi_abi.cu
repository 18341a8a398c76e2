// pi_abi.cu — host side of the libpi C ABI (declared in include/pi.h):
// argument validation, workspace layout, launch configuration.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <utility>
#include <string>
#include <unordered_map>

#include "kernels.cuh"
#include "batched.cuh"
#include "seq.cuh"
#include "plan.cuh"
#include "tc.cuh"
#include "tcd.cuh"

using namespace pik;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte offsets of the workspace regions.
struct WsLayout {
  size_t ctrl, upart, loc_tot, mask, part, u, logits, total;
  size_t uacc;  // sequence kernel: 2 x r fixed-point accumulators, one 128-byte line each
  size_t glist, gcnt;  // sequence kernel: published cold entries and counts
  size_t cscr;         // grid-wide compaction counts (the last region: pi_compact finds it at
                       // the end of the workspace)
  // batched path (batch > 1)
  size_t bidx, bcnt, uidx, ucnt, tmask, xhi, xlo, hhi, hlo, bpart, ppart, uhi, ulo;
  int bp, hs;
};

int batch_pad(int batch) { return batch <= 16 ? 16 : 32; }
// counts of the grid-wide compaction: [kCSeries][blocks] + totals
size_t compact_scratch_bytes(int n) {
  const size_t nb = ((size_t)n + kCB - 1) / kCB;
  return round_up(sizeof(int) * (kCSeries * nb + kCSeries), 256);
}
int h_stride(int n) { return (int)round_up((size_t)n + kBN2, 64); }

WsLayout ws_layout(const pi_ffn_desc& D, int batch) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes > 0 ? bytes : 1, kAlign);
    return o;
  };
  L.ctrl = take(256);  // grid barrier arrival counter (64-bit)
  // predictor partials: r x kSMax (one-layer kernel) or r x P (sequence kernel)
  L.upart = take(sizeof(float) * (size_t)D.r * (kPMax > kSMax ? kPMax : kSMax));
  L.loc_tot = take(sizeof(int) * kPMax);
  L.mask = take((size_t)D.n);
  L.part = take(sizeof(float) * (size_t)kPMax * D.d);
  L.u = take(sizeof(float) * (size_t)batch * D.r);
  L.logits = take(sizeof(float) * (size_t)batch * D.n);
  L.uacc = take(2 * 128 * (size_t)D.r);
  L.glist = take(8 * ((size_t)D.n + kPMax));
  L.gcnt = take(sizeof(int) * kPMax);
  L.bp = batch_pad(batch);
  L.hs = h_stride(D.n);
  if (batch > 1) {
    L.bidx = take(sizeof(int) * (size_t)batch * D.n);
    L.bcnt = take(sizeof(int) * (size_t)batch);
    L.uidx = take(sizeof(int) * (size_t)D.n);
    L.ucnt = take(sizeof(int));
    L.tmask = take(sizeof(uint32_t) * (size_t)D.n);
    L.xhi = take(2 * (size_t)L.bp * D.d);
    L.xlo = take(2 * (size_t)L.bp * D.d);
    L.hhi = take(2 * (size_t)L.bp * L.hs);
    L.hlo = take(2 * (size_t)L.bp * L.hs);
    // phase-2 partials: [kGroups2][bp][d] (mma.sync phases) or [P][2][bp][256]
    // (tensor-memory phases of the dense FFN)
    const size_t pg = (size_t)kGroups2 * L.bp * D.d, pt = (size_t)kPMax * 2 * L.bp * 256;
    L.bpart = take(sizeof(float) * (pg > pt ? pg : pt));
    L.ppart = take(sizeof(float) * (size_t)kPMax * batch * D.r);  // predictor partials [G][batch][r]
    L.uhi = take(2 * (size_t)L.bp * D.r);
    L.ulo = take(2 * (size_t)L.bp * D.r);
  }
  L.cscr = take(compact_scratch_bytes(D.n));
  L.total = off;
  return L;
}

pi_status check_desc(const pi_ffn_desc* D) {
  if (!D) return PI_ERR_NULL;
  if (D->dtype != PI_F16 && D->dtype != PI_BF16) return PI_ERR_DTYPE;
  if (D->d < 8 || D->d > 8192 || (D->d & 7)) return PI_ERR_SHAPE;
  if (D->r < 8 || D->r > 256 || (D->r & 7)) return PI_ERR_SHAPE;
  if (D->n < 1 || D->n > (1 << 24)) return PI_ERR_SHAPE;
  if (D->gated != 0 && D->gated != 1) return PI_ERR_SHAPE;
  if (D->hot_prefix < 0 || D->hot_prefix > D->n) return PI_ERR_SHAPE;
  if (D->layout != PI_LAYOUT_SPLIT && D->layout != PI_LAYOUT_PACKED) return PI_ERR_SHAPE;
  return PI_OK;
}

pi_status check_weights(const pi_ffn_desc& D, const pi_layer_weights* w, bool need_pred) {
  if (!w) return PI_ERR_NULL;
  if (!w->b1 || !w->W1) return PI_ERR_NULL;
  if (D.layout == PI_LAYOUT_SPLIT && !w->W2) return PI_ERR_NULL;
  if (D.layout == PI_LAYOUT_PACKED && w->W2) return PI_ERR_SHAPE;
  if (need_pred && (!w->A || !w->Bm)) return PI_ERR_NULL;
  const void* ps[] = {w->A, w->Bm, w->b1, w->W1, w->W2, w->b2};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  return PI_OK;
}

struct DevInfo {
  int sms = 0;
  int smem_optin = 0;
};

std::mutex g_mu;
std::unordered_map<int, DevInfo> g_dev;
std::unordered_map<const void*, int> g_smem_set;  // kernel -> dynamic smem attribute set (per process)
unsigned long long g_limit_ns = 0;
int g_launch_mode = -1;  // 0: cooperative launch, 1: programmatic dependent launch

pi_status dev_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PI_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DevInfo di;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return PI_ERR_CUDA;
    it = g_dev.emplace(dev, di).first;
  }
  *out = it->second;
  return PI_OK;
}

unsigned long long wait_limit_ns() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_limit_ns == 0) {
    g_limit_ns = 1000000000ull;  // 1 s
    if (const char* e = std::getenv("PI_WAIT_LIMIT_NS")) {
      const unsigned long long v = std::strtoull(e, nullptr, 10);
      if (v >= 1000ull && v <= 10000000000ull) g_limit_ns = v;
    }
  }
  return g_limit_ns;
}

// Bounds of a persistent launch's waits: the protocol waits take the
// process-wide limit; the wait for copies already issued to land takes at
// least 2 s, so that no block leaves with a copy in flight.
void set_waits(FfnArgs& a) {
  a.limit_ns = wait_limit_ns();
  a.drain_ns = a.limit_ns > 2000000000ull ? a.limit_ns : 2000000000ull;
}

// How persistent grids are launched.  Default: programmatic dependent
// launch, which lets a step's weight prefetch overlap the end of the
// previous step in the same stream; every block is resident because the grid
// has one block per SM and a block fills an SM.  PI_LAUNCH=cooperative
// selects a cooperative launch instead (the driver then also checks
// co-residency, but consecutive steps do not overlap).
int launch_mode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_launch_mode < 0) {
    const char* e = std::getenv("PI_LAUNCH");
    g_launch_mode = (e && std::string(e) == "cooperative") ? 0 : 1;
  }
  return g_launch_mode;
}

// Launch of one kernel of a chain with programmatic dependent launch: the
// kernel may be scheduled while the previous kernel in the stream runs and
// waits for it at its first statement (pdl_enter), so the chain pays no
// launch gap between its kernels.  Returns the launch's CUDA error.
template <typename... KArgs, typename... Args>
cudaError_t launch_chain(void (*k)(KArgs...), unsigned grid, unsigned block, size_t smem,
                         cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

pi_status ensure_smem(const void* fn, int bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  int& cur = g_smem_set[fn];  // per process; the attribute applies to the current device
  if (bytes > cur) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return PI_ERR_CUDA;
    cur = bytes;
  }
  return PI_OK;
}

pi_status map_launch_error(cudaError_t e) {
  if (e == cudaSuccess) return PI_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) return PI_ERR_LAUNCH;
  return PI_ERR_CUDA;
}

using FfnFn = void (*)(const FfnArgs);

template <int MODE>
FfnFn pick_ffn(int dtype, int gated, bool wide) {
  if (dtype == PI_F16) {
    if (!gated) return wide ? ffn_kernel<0, false, 2, MODE> : ffn_kernel<0, false, 1, MODE>;
    return wide ? ffn_kernel<0, true, 2, MODE> : ffn_kernel<0, true, 1, MODE>;
  }
  if (!gated) return wide ? ffn_kernel<1, false, 2, MODE> : ffn_kernel<1, false, 1, MODE>;
  return wide ? ffn_kernel<1, true, 2, MODE> : ffn_kernel<1, true, 1, MODE>;
}

// Shared-memory layout of a persistent launch for a given predictor-row
// placement; returns the bytes before the ring slots (16-byte aligned).
int layout_fixed(const pi_ffn_desc& D, int mode, int P, int rows_max, int a_in_smem, FfnArgs& a,
                 bool no_xs = false) {
  int off = 0;
  auto take = [&](int bytes, int align) {
    off = (off + align - 1) / align * align;
    const int o = off;
    off += bytes;
    return o;
  };
  a.o_xs = no_xs ? 0 : take(4 * D.d, 16);  // the layer-sequence kernel reads x from global memory
  a.o_lst = take(4 * (rows_max + kMaxSlots), 16);
  a.o_lb = take(4 * (rows_max + kMaxSlots), 16);
  a.o_red = take(4 * (2 * kGroup * 2 * kWarps + 2 * kGroup + 64), 16);  // butterfly partials, h
  a.o_mbar = take(2 * 8 * kMaxSlots, 16);
  a.o_us = a.o_As = a.o_b1s = a.o_flag = a.o_off = 0;
  (void)P;
  if (mode == kFused) {
    a.o_us = take(4 * D.r, 16);
    a.o_b1s = take(4 * rows_max, 16);
    a.o_flag = take(rows_max, 16);
    if (a_in_smem) a.o_As = take(rows_max * (2 * D.r + 16), 16);
  }
  return (off + 127) / 128 * 128;
}

// Fills the shape fields, grid size and shared-memory plan of a persistent
// launch; returns the dynamic shared-memory bytes, or 0 if the shape does
// not fit.
int plan_ffn(const pi_ffn_desc& D, int mode, int P, int positions, int smem_limit, FfnArgs& a,
             bool no_xs = false) {
  a.d = D.d;
  a.n = D.n;
  a.r = D.r;
  a.P = P;
  a.hot = D.hot_prefix;
  a.nch = D.d / 8;
  a.rows_max = (positions + P - 1) / P;
  int S = 1;
  while (D.r * S < P && S < kSMax && (D.d / (2 * S)) % 8 == 0 && D.d / (2 * S) >= 256) S *= 2;
  a.S = S;
  a.slot_bytes = (D.gated ? 3 : 2) * D.d * 2;
  a.packed = D.layout == PI_LAYOUT_PACKED ? 1 : 0;
  a.a_stride = 2 * D.r + 16;
  auto slots_for = [&](int fixed) {
    const int ns = (smem_limit - fixed) / a.slot_bytes;
    return ns < kMaxSlots ? ns : kMaxSlots;
  };
  a.a_in_smem = 0;
  int fixed = layout_fixed(D, mode, P, a.rows_max, 0, a, no_xs);
  int ns = slots_for(fixed);
  if (mode == kFused) {
    FfnArgs t = a;
    const int fixed_s = layout_fixed(D, mode, P, a.rows_max, 1, t, no_xs);
    const int ns_s = slots_for(fixed_s);
    if (ns_s >= 10 || ns_s >= ns) {  // stage A only if the ring stays deep
      a = t;
      a.a_in_smem = 1;
      fixed = fixed_s;
      ns = ns_s;
    } else {
      layout_fixed(D, mode, P, a.rows_max, 0, a, no_xs);
    }
  }
  if (ns < 2) return 0;
  a.ns = ns;
  a.nh = 0;
  if (mode == kFused && D.hot_prefix > 0) {
    const int hot_per_block = (D.hot_prefix + P - 1) / P;
    const int cap = ns - 2 * kGroup > ns / 4 ? ns - 2 * kGroup : ns / 4;  // keep two rounds of cold slots
    a.nh = hot_per_block < cap ? hot_per_block : cap;
    if (a.nh < 0) a.nh = 0;
  }
  if (a.ns < 8) a.nh = 0;  // shallow ring: keep every slot for the active rows
  // rounds of up to kGroup neurons: larger rounds cost less per neuron (the
  // round's barriers and reductions are shared), as long as enough slots stay
  // in flight while a round is computed (measured on the OPT-30B shape with 7
  // cold slots: 3 neurons per round 31.2 us per layer, 4: 33.0, 2: 42)
  const int nc = a.ns - a.nh;
  a.grp = nc >= 10 ? kGroup : (nc >= 6 ? 3 : (nc >= 4 ? 2 : 1));
  a.o_slots = fixed;
  return fixed + ns * a.slot_bytes;
}

// limit_ns / skip_issue: the failure-path self-test's shorter protocol
// bound and unissued entry (0: the process-wide bound, none).
template <int MODE>
pi_status launch_ffn(const pi_ffn_desc& D, FfnArgs& a, int positions, cudaStream_t st,
                     unsigned long long limit_ns = 0, int skip_issue = 0) {
  DevInfo di;
  pi_status s = dev_info(&di);
  if (s != PI_OK) return s;
  const int P = di.sms < kPMax ? di.sms : kPMax;  // also <= kThreads (one scan lane per block)
  const bool wide = (D.d / 8) > kThreads;
  FfnFn fn = pick_ffn<MODE>(D.dtype, D.gated, wide);
  const int limit = di.smem_optin - 1024;  // static shared memory and margin
  const int smem = plan_ffn(D, MODE, P, positions, limit, a);
  if (smem == 0 || a.grp < 1) return PI_ERR_SHAPE;
  s = ensure_smem(reinterpret_cast<const void*>(fn), smem);
  if (s != PI_OK) return s;
  set_waits(a);
  if (limit_ns) a.limit_ns = limit_ns;
  a.skip_issue = skip_issue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (launch_mode() == 0) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    int per_sm = 0;  // the grid must fit at one block per SM
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBlock, (size_t)smem) !=
        cudaSuccess)
      return PI_ERR_CUDA;
    if (per_sm < 1) return PI_ERR_LAUNCH;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return map_launch_error(cudaLaunchKernelEx(&cfg, fn, a));
}

void bind_ws(FfnArgs& a, const WsLayout& L, void* ws) {
  char* b = static_cast<char*>(ws);
  a.bar = reinterpret_cast<unsigned long long*>(b + L.ctrl);
  a.upart = reinterpret_cast<float*>(b + L.upart);
  a.loc_tot = reinterpret_cast<int*>(b + L.loc_tot);
  a.mask = reinterpret_cast<unsigned char*>(b + L.mask);
  a.part = reinterpret_cast<float*>(b + L.part);
}

void bind_weights(FfnArgs& a, const pi_layer_weights& w) {
  a.A = static_cast<const uint16_t*>(w.A);
  a.Bm = static_cast<const uint16_t*>(w.Bm);
  a.b1 = w.b1;
  a.W1 = static_cast<const uint16_t*>(w.W1);
  a.W2 = static_cast<const uint16_t*>(w.W2);
  a.b2 = w.b2;
}

// ------------------------------------------------------------ tensor maps
// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the
// driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  }
  return g_encode;
}

// Map over a row-major matrix of 16-bit elements (rows x inner, row pitch
// `pitch` elements): boxes of 64 elements x box_rows rows, 128-byte swizzle,
// rows past the end read as zero.
bool make_map(CUtensorMap* m, const void* base, size_t inner, size_t rows, size_t pitch,
              unsigned box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// PI_BATCH_LEGACY=1 runs the dense batched FFN on the mma.sync phases
// instead of the tensor-memory ones (read once per process).
int g_batch_legacy = -1;
bool batch_legacy() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_batch_legacy < 0) {
    const char* e = std::getenv("PI_BATCH_LEGACY");
    g_batch_legacy = (e && std::atoi(e) != 0) ? 1 : 0;
  }
  return g_batch_legacy == 1;
}

// The dense batched FFN (all n neurons, every token) on the tcgen05 / TMA
// phases of tcd.cuh, x already split into its high / low parts.  Sets *used
// = false, launching nothing, where the shape does not fit them (d % 128,
// n % 64, more column tiles than blocks, more than 256 rows per block, a
// residual that is not 16-byte aligned) or PI_BATCH_LEGACY is set; the
// mma.sync phases run then.
pi_status launch_td(const pi_ffn_desc& D, const BatchArgs& a, const DevInfo& di, cudaStream_t st,
                    bool* used) {
  *used = false;
  if (batch_legacy()) return PI_OK;
  const int P = di.sms;
  const int NW = D.gated ? 2 : 1;
  if (D.d % 128 != 0 || D.n % 64 != 0) return PI_OK;
  const int nc2 = D.d % 256 == 0 ? 256 : 128;  // phase 2's columns per tile (the MMA's N)
  const int nct = D.d / nc2, nkb = D.n / 64;
  if (nct > P || nct > kTdMaxTiles || P > kPMax || (long long)nct * nkb < P) return PI_OK;
  // the high and low parts of x and of H^T are read as one [2 bp][...] box
  if (a.xlo != a.xhi + (size_t)a.bp * D.d || a.hlo != a.hhi + (size_t)a.bp * a.hs) return PI_OK;
  // the final sum moves four columns at a time (y, b2 and the weights are
  // checked for 16-byte alignment at the entry points)
  if (a.residual && !aligned16(a.residual)) return PI_OK;
  TdArgs t{};
  t.d = D.d;
  t.n = D.n;
  t.batch = a.batch;
  t.bp = a.bp;
  t.P = P;
  const int ng = D.n / 8;
  const int rmax = 8 * ((ng + P - 1) / P);  // most rows of a block
  if (rmax > 256) return PI_OK;              // one accumulator tile per block
  const int bp2 = 2 * a.bp;
  const int budget = di.smem_optin - 2048;  // static shared memory and the 1024-byte alignment
  t.wrows = rmax;
  t.ncol1 = (int)round_up((size_t)rmax, 16);
  t.stage1 = kTdHalf + NW * t.wrows * 128;
  // the last stage's last B read may run (ncol1 - wrows) rows past it
  const int guard1 = (int)round_up((size_t)(t.ncol1 - t.wrows) * 128, 1024);
  t.ns1 = std::min(kTdMaxStages, (budget - guard1) / t.stage1);
  t.nc2 = nc2;
  t.stage2 = kTdHalf + (nc2 / 64) * 64 * 128;
  // batch 32: the low parts' accumulator lanes staged in shared memory
  const int xst = a.bp == 32 ? (int)round_up((size_t)32 * (nc2 + 4) * sizeof(float), 1024) : 0;
  t.ns2 = std::min(kTdMaxStages, (budget - xst) / t.stage2);
  if (t.ns1 < 2 || t.ns2 < 2) return PI_OK;
  // the phase-1 epilogue's staging of the accumulators fits in the stages
  if ((size_t)NW * bp2 * (t.ncol1 + 4) * sizeof(float) > (size_t)t.ns1 * t.stage1) return PI_OK;
  auto pow2 = [](int v) {
    int p = 32;
    while (p < v) p <<= 1;
    return p;
  };
  t.tcols1 = pow2(NW * t.ncol1);
  t.tcols2 = pow2(2 * nc2);
  if (t.tcols1 > 512) return PI_OK;
  t.hs = a.hs;
  t.nct = nct;
  t.nkb = nkb;
  const size_t w1row = a.packed ? (size_t)a.rec : (size_t)NW * D.d;
  const size_t w2row = a.packed ? (size_t)a.rec : (size_t)D.d;
  t.w2x = a.packed ? NW * D.d : 0;
  t.b1 = a.b1;
  t.b2 = a.b2;
  t.residual = a.residual;
  t.y = a.y;
  t.hT = a.hhi;
  t.part = a.part;
  // phase 2's partition: block b takes work items [b F / P, (b+1) F / P)
  {
    const long long F = (long long)nct * nkb;
    for (int c = 0; c < nct; ++c) {
      t.tile_b0[c] = 0xffff;
      t.tile_b1[c] = 0;
    }
    for (int b = 0; b < P; ++b) {
      const long long s0 = (long long)b * F / P, s1 = (long long)(b + 1) * F / P;
      t.first_tile[b] = (uint16_t)(s0 / nkb);
      for (long long c = s0 / nkb; c <= (s1 - 1) / nkb; ++c) {
        if (t.tile_b0[c] == 0xffff) t.tile_b0[c] = (uint16_t)b;
        t.tile_b1[c] = (uint16_t)b;
      }
    }
  }
  t.status = a.status;
  t.limit_ns = wait_limit_ns();
  t.drain_ns = t.limit_ns > 2000000000ull ? t.limit_ns : 2000000000ull;
  CUtensorMap m128, m32, m8, mx, mw2, mh;
  const void* w2base = a.packed ? static_cast<const void*>(a.W1) : static_cast<const void*>(a.W2);
  if (!make_map(&m128, a.W1, w1row, D.n, w1row, 128) || !make_map(&m32, a.W1, w1row, D.n, w1row, 32) ||
      !make_map(&m8, a.W1, w1row, D.n, w1row, 8) ||
      !make_map(&mx, a.xhi, D.d, bp2, D.d, (unsigned)bp2) ||
      !make_map(&mw2, w2base, w2row, D.n, w2row, 64) ||
      !make_map(&mh, a.hhi, a.hs, bp2, a.hs, (unsigned)bp2))
    return PI_OK;
  *used = true;
  const bool bf = D.dtype == PI_BF16;
  using F1 = void (*)(const TdArgs, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                      const CUtensorMap);
  F1 f1 = bf ? (D.gated ? td_up_kernel<1, true> : td_up_kernel<1, false>)
             : (D.gated ? td_up_kernel<0, true> : td_up_kernel<0, false>);
  const int smem1 = t.ns1 * t.stage1 + guard1 + 1024;
  pi_status s = ensure_smem(reinterpret_cast<const void*>(f1), smem1);
  if (s != PI_OK) return s;
  if (launch_chain(f1, P, kTdThreads, smem1, st, t, m128, m32, m8, mx) != cudaSuccess)
    return PI_ERR_CUDA;
  using F2 = void (*)(const TdArgs, const CUtensorMap, const CUtensorMap);
  F2 f2 = bf ? td_down_kernel<1> : td_down_kernel<0>;
  const int smem2 = t.ns2 * t.stage2 + xst + 1024;
  s = ensure_smem(reinterpret_cast<const void*>(f2), smem2);
  if (s != PI_OK) return s;
  if (launch_chain(f2, P, kTdThreads, smem2, st, t, mw2, mh) != cudaSuccess) return PI_ERR_CUDA;
  const int g3 = std::max(1, std::min((a.batch * nc2 / 4 + 255) / 256, (4 * P + nct - 1) / nct));
  if (launch_chain(td_sum_kernel, nct * g3, 256, 0, st, t) != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

// ------------------------------------------------------------ batched path
// The three tensor-core phases of a batched sparse FFN over the union of the
// tokens' active neurons (uidx / ucnt / tmask in device memory).
// uidx == NULL: the dense batched FFN (all n neurons, every token).
pi_status launch_batched(const pi_ffn_desc& D, const pi_layer_weights& w, const float* x,
                         int batch, const int* uidx, const int* ucnt, const uint32_t* tmask,
                         float* y, const float* residual, const WsLayout& L, void* ws,
                         cudaStream_t st, int32_t* dev_status, bool x_split = false) {
  DevInfo di;
  pi_status s = dev_info(&di);
  if (s != PI_OK) return s;
  char* b = static_cast<char*>(ws);
  BatchArgs a{};
  a.d = D.d;
  a.n = D.n;
  a.batch = batch;
  a.bp = L.bp;
  a.P = di.sms;
  a.slices = di.sms / kGroups2 > 0 ? di.sms / kGroups2 : 1;
  a.cw = (int)round_up((size_t)((D.d + a.slices - 1) / a.slices), 16);  // whole n-tile pairs
  a.packed = D.layout == PI_LAYOUT_PACKED;
  a.rec = (D.gated ? 3 : 2) * D.d;
  a.W1 = static_cast<const uint16_t*>(w.W1);
  a.W2 = a.packed ? a.W1 + (size_t)(D.gated ? 2 : 1) * D.d : static_cast<const uint16_t*>(w.W2);
  a.b1 = w.b1;
  a.b2 = w.b2;
  a.x = x;
  a.residual = residual;
  a.y = y;
  a.uidx = uidx;
  a.ucnt = ucnt;
  a.tmask = tmask;
  a.dense = uidx == nullptr;
  a.xhi = reinterpret_cast<uint16_t*>(b + L.xhi);
  a.xlo = reinterpret_cast<uint16_t*>(b + L.xlo);
  a.hhi = reinterpret_cast<uint16_t*>(b + L.hhi);
  a.hlo = reinterpret_cast<uint16_t*>(b + L.hlo);
  a.hs = L.hs;
  a.part = reinterpret_cast<float*>(b + L.bpart);
  a.status = dev_status;  // may be NULL
  const bool bf = D.dtype == PI_BF16;
  const bool m2 = a.bp == 32;
  // phase 0: split x
  // (skipped when the batched predictor of this call already wrote them)
  if (!x_split &&
      launch_chain(bf ? bsplit_x_kernel<1> : bsplit_x_kernel<0>, di.sms * 4, 256, 0, st, a) !=
          cudaSuccess)
    return PI_ERR_CUDA;
  // the dense FFN on the tensor-memory phases where the shape allows
  if (a.dense) {
    bool used = false;
    s = launch_td(D, a, di, st, &used);
    if (s != PI_OK || used) return s;
  }
  // phase 1
  const int nw = D.gated ? 2 : 1;
  // plain layers take 256-column chunks when d allows (fewer pipeline steps
  // per byte); gated ones 128 (their stages would not fit three deep)
  const bool wide = !D.gated && D.d % 256 == 0;
  const int rowb = (wide ? 256 : 128) * 2 + 16;
  // (the k slices' partial sums reuse the stages: 15 x 32 x CV floats at
  // most, less than the three stages hold)
  const int smem1 = kBStages * ((nw * kBT + 2 * a.bp) * rowb);
  using Fn = void (*)(const BatchArgs);
  Fn f1;
  if (!bf) {
    if (!D.gated)
      f1 = wide ? (m2 ? bup_kernel<0, false, 2, 256> : bup_kernel<0, false, 1, 256>)
                : (m2 ? bup_kernel<0, false, 2, 128> : bup_kernel<0, false, 1, 128>);
    else f1 = m2 ? bup_kernel<0, true, 2, 128> : bup_kernel<0, true, 1, 128>;
  } else {
    if (!D.gated)
      f1 = wide ? (m2 ? bup_kernel<1, false, 2, 256> : bup_kernel<1, false, 1, 256>)
                : (m2 ? bup_kernel<1, false, 2, 128> : bup_kernel<1, false, 1, 128>);
    else f1 = m2 ? bup_kernel<1, true, 2, 128> : bup_kernel<1, true, 1, 128>;
  }
  int smem_launch = smem1;
  // tcgen05 phase 1 with PI_BATCH_TC=1 (measured slower than the mma.sync
  // kernel so far: one commit round trip per 64-128-column chunk)
  bool use_tc = false;
  if (const char* e = std::getenv("PI_BATCH_TC")) use_tc = std::atoi(e) != 0;
  if (use_tc) {
    const int mh = 1;  // 128-position tiles (measured faster than 256 with narrower chunks)
    int cols = mh * nw * a.bp, pw = 32;
    while (pw < cols) pw <<= 1;
    a.tc_cols = pw;
    const int stg = kTcStages * (D.gated ? tc_stage_bytes<true, 1>(a.bp)
                                         : tc_stage_bytes<false, 1>(a.bp));
    if (!bf) f1 = D.gated ? bup_tc_kernel<0, true, 1> : bup_tc_kernel<0, false, 1>;
    else f1 = D.gated ? bup_tc_kernel<1, true, 1> : bup_tc_kernel<1, false, 1>;
    smem_launch = stg;
    a.limit_ns = wait_limit_ns();
  }
  if (smem_launch + 1024 > di.smem_optin) return PI_ERR_SHAPE;
  s = ensure_smem(reinterpret_cast<const void*>(f1), smem_launch);
  if (s != PI_OK) return s;
  if (launch_chain(f1, a.P, 512, smem_launch, st, a) != cudaSuccess) return PI_ERR_CUDA;
  // phase 2
  const int smem2 = kBStages * bdn_stage_bytes(a.cw, a.bp);
  Fn f2 = bf ? (m2 ? bdown_kernel<1, 2> : bdown_kernel<1, 1>)
             : (m2 ? bdown_kernel<0, 2> : bdown_kernel<0, 1>);
  if (smem2 + 1024 > di.smem_optin || a.cw / 8 > 64) return PI_ERR_SHAPE;
  s = ensure_smem(reinterpret_cast<const void*>(f2), smem2);
  if (s != PI_OK) return s;
  if (launch_chain(f2, kGroups2 * a.slices, 512, smem2, st, a) != cudaSuccess) return PI_ERR_CUDA;
  // phase 3
  if (launch_chain(bsum_kernel, di.sms * 4, 256, 0, st, a) != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

// ------------------------------------------------------------ fixed scratch
// Scratch of pi_layer_decode_static: a fixed array in the device image
// instead of a caller workspace.  Zero at load; every call clears its
// barrier block before launching.
static __device__ __align__(256) unsigned char g_static_scratch[PI_STATIC_SCRATCH_BYTES];

std::unordered_map<int, void*> g_static_ptr;  // device -> address of g_static_scratch

// Device address of g_static_scratch on the current device, looked up once
// per device (host code only has a stand-in for the symbol).  The lookup
// is refused while `st` is being captured into a graph (the capture would
// be invalidated); later calls on the device only read the cached address.
pi_status static_scratch(void** out, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PI_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_static_ptr.find(dev);
  if (it == g_static_ptr.end()) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return PI_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return PI_ERR_CAPTURE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return PI_ERR_CUDA;
    it = g_static_ptr.emplace(dev, p).first;
  }
  *out = it->second;
  return PI_OK;
}

// Regions of the fused batch-1 kernel's scratch with exactly P partial rows:
// the barrier block, the predictor partials (r x kSMax), the per-block
// counts, the n-byte mask and the P x d partial outputs, each rounded up to
// 256 bytes.
WsLayout static_layout(const pi_ffn_desc& D, int P) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes > 0 ? bytes : 1, kAlign);
    return o;
  };
  L.ctrl = take(256);
  L.upart = take(sizeof(float) * (size_t)D.r * kSMax);
  L.loc_tot = take(sizeof(int) * (size_t)P);
  L.mask = take((size_t)D.n);
  L.part = take(sizeof(float) * (size_t)P * D.d);
  L.u = L.logits = 0;
  L.total = off;
  return L;
}

// Batch-1 sparse FFN over a caller's active list (the body of pi_sparse_ffn
// for batch 1, and of its failure-path self-test).
pi_status sparse_one(const pi_ffn_desc* desc, const pi_layer_weights* w, const float* x,
                     const int32_t* idx, const int32_t* cnt, int32_t cap, float* y,
                     int32_t* dev_status, void* ws, size_t ws_bytes, pi_stream stream,
                     unsigned long long limit_ns, int skip_issue) {
  if (!x || !y || !idx || !cnt || !dev_status || !ws) return PI_ERR_NULL;
  const void* ps[] = {x, y, idx, cnt, dev_status, ws};
  for (const void* p : ps)
    if (!aligned16(p)) return PI_ERR_ALIGN;
  if (cap < 0) return PI_ERR_SHAPE;
  const WsLayout L = ws_layout(*desc, 1);
  if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
  FfnArgs a{};
  bind_weights(a, *w);
  bind_ws(a, L, ws);
  a.x = x;
  a.residual = nullptr;
  a.y = y;
  a.idx_in = idx;
  a.cnt_in = cnt;
  a.cap = cap;
  a.status = dev_status;
  const int positions = cap < desc->n ? cap : desc->n;
  return launch_ffn<kSparse>(*desc, a, positions > 0 ? positions : 1,
                             reinterpret_cast<cudaStream_t>(stream), limit_ns, skip_issue);
}

}  // namespace

// ------------------------------------------------------------ layer sequence
using SeqFn = void (*)(const SeqArgs);
SeqFn pick_seq(int dtype, int gated, bool wide) {
  if (dtype == PI_F16) {
    if (!gated) return wide ? seq_kernel<0, false, 2> : seq_kernel<0, false, 1>;
    return wide ? seq_kernel<0, true, 2> : seq_kernel<0, true, 1>;
  }
  if (!gated) return wide ? seq_kernel<1, false, 2> : seq_kernel<1, false, 1>;
  return wide ? seq_kernel<1, true, 2> : seq_kernel<1, true, 1>;
}

extern "C" {

pi_status pi_layer_decode_static(const pi_ffn_desc* desc, const pi_layer_weights* w, const float* x,
                                 float* y, const float* residual, int32_t* idx_out,
                                 int32_t* cnt_out, int32_t* dev_status, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  s = check_weights(*desc, w, true);
  if (s != PI_OK) return s;
  if (!x || !y || !dev_status) return PI_ERR_NULL;
  const void* ps[] = {x, y, residual, idx_out, cnt_out, dev_status};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  // a shape too large even for a one-block grid is refused before any CUDA call
  if (static_layout(*desc, 1).total > PI_STATIC_SCRATCH_BYTES) return PI_ERR_WORKSPACE;
  DevInfo di;
  s = dev_info(&di);
  if (s != PI_OK) return s;
  const int P = di.sms < kPMax ? di.sms : kPMax;
  const WsLayout L = static_layout(*desc, P);
  if (L.total > PI_STATIC_SCRATCH_BYTES) return PI_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  s = static_scratch(&scratch, st);
  if (s != PI_OK) return s;
  if (cudaMemsetAsync(static_cast<char*>(scratch) + L.ctrl, 0, 256, st) != cudaSuccess)
    return PI_ERR_CUDA;
  FfnArgs a{};
  bind_weights(a, *w);
  bind_ws(a, L, scratch);
  a.x = x;
  a.residual = residual;
  a.y = y;
  a.idx_out = idx_out;
  a.cnt_out = cnt_out;
  a.status = dev_status;
  if (!a.idx_out) a.mask = nullptr;
  return launch_ffn<kFused>(*desc, a, desc->n, st);
}


size_t pi_workspace_size(const pi_ffn_desc* desc, int32_t batch) {
  if (check_desc(desc) != PI_OK) return 0;
  if (batch < 1 || batch > kMaxBatch) return 0;
  return ws_layout(*desc, batch).total;
}

void pi_default_cost_model(pi_cost_model* out) {
  if (!out) return;
  *out = pi_cost_model{};
  const int32_t tiers[PI_COST_TIERS] = {1, 4, 16, 32};
  // per tier (batch <= 1, 4, 16, 32): fixed microseconds and GB/s of a
  // least-squares fit to the measured sweep (five densities per batch)
  const double fused_fix = 15.4, fused_gbs = 4610.0;
  const double union_fix[PI_COST_TIERS] = {34.2, 34.2, 37.9, 51.5};
  const double union_gbs[PI_COST_TIERS] = {2574.0, 2574.0, 2424.0, 1912.0};
  // dense: the batch-1 kernel, then the tensor-memory phases (a fixed cost
  // for the operand split and the partial sum)
  const double dense_fix[PI_COST_TIERS] = {3.0, 8.0, 8.0, 8.0};
  const double dense_gbs[PI_COST_TIERS] = {5926.0, 5910.0, 5780.0, 5300.0};
  for (int t = 0; t < PI_COST_TIERS; ++t) {
    out->tier_max_batch[t] = tiers[t];
    out->fixed_us[PI_PATH_FUSED][t] = out->fixed_us[PI_PATH_PER_TOKEN][t] = fused_fix;
    out->gbs[PI_PATH_FUSED][t] = out->gbs[PI_PATH_PER_TOKEN][t] = fused_gbs;
    out->fixed_us[PI_PATH_UNION][t] = union_fix[t];
    out->gbs[PI_PATH_UNION][t] = union_gbs[t];
    out->fixed_us[PI_PATH_DENSE][t] = dense_fix[t];
    out->gbs[PI_PATH_DENSE][t] = dense_gbs[t];
  }
}

pi_status pi_plan_dispatch(const pi_ffn_desc* desc, int32_t batch, const float* p_active,
                           float density, int32_t allow_dense, const pi_cost_model* model,
                           pi_plan* out) {
  if (!desc || !out) return PI_ERR_NULL;
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > 32) return PI_ERR_SHAPE;
  if (!p_active && !(density >= 0.f && density <= 1.f)) return PI_ERR_SHAPE;
  pi_cost_model M;
  if (model) M = *model;
  else pi_default_cost_model(&M);
  for (int t = 0; t < PI_COST_TIERS; ++t) {
    if (t > 0 && M.tier_max_batch[t] < M.tier_max_batch[t - 1]) return PI_ERR_SHAPE;
    for (int k = 0; k < PI_PATHS; ++k)
      if (!(M.gbs[k][t] > 0.0)) return PI_ERR_SHAPE;
  }
  const pi_ffn_desc& D = *desc;
  double active = 0.0, uni = 0.0;
  plan_expected_rows(p_active, D.n, density, batch, &active, &uni);
  const double e = 2.0, m = D.gated ? 3.0 : 2.0;
  const double pred = (double)D.n * D.r * e + (double)D.r * D.d * e + 4.0 * D.n;
  const double row = m * D.d * e;
  const int t = plan_tier(M, batch);
  pi_plan P{};
  for (int k = 0; k < PI_PATHS; ++k) P.est_us[k] = P.bytes[k] = -1.0;
  P.active_rows = active;
  P.union_rows = uni;
  if (batch == 1) {
    P.bytes[PI_PATH_FUSED] = pred + active * row;
    P.est_us[PI_PATH_FUSED] = plan_time_us(M.fixed_us[PI_PATH_FUSED][0], P.bytes[PI_PATH_FUSED],
                                           M.gbs[PI_PATH_FUSED][0]);
  } else {
    const double one = pred + active * row;
    P.bytes[PI_PATH_PER_TOKEN] = batch * one;
    P.est_us[PI_PATH_PER_TOKEN] =
        batch * plan_time_us(M.fixed_us[PI_PATH_PER_TOKEN][0], one, M.gbs[PI_PATH_PER_TOKEN][0]);
    if (D.d % 128 == 0) {
      P.bytes[PI_PATH_UNION] = pred + uni * row;
      P.est_us[PI_PATH_UNION] = plan_time_us(M.fixed_us[PI_PATH_UNION][t], P.bytes[PI_PATH_UNION],
                                             M.gbs[PI_PATH_UNION][t]);
    }
  }
  if (allow_dense) {
    P.bytes[PI_PATH_DENSE] = (double)D.n * row;
    P.est_us[PI_PATH_DENSE] = plan_time_us(M.fixed_us[PI_PATH_DENSE][t], P.bytes[PI_PATH_DENSE],
                                           M.gbs[PI_PATH_DENSE][t]);
  }
  int best = -1;
  for (int k = 0; k < PI_PATHS; ++k)  // ties go to the lower path number
    if (P.est_us[k] >= 0.0 && (best < 0 || P.est_us[k] < P.est_us[best])) best = k;
  P.path = static_cast<pi_path>(best);
  *out = P;
  return PI_OK;
}

const char* pi_status_string(pi_status s) {
  switch (s) {
    case PI_OK: return "ok";
    case PI_ERR_NULL: return "a required pointer is NULL";
    case PI_ERR_SHAPE: return "a size or the batch is outside the supported range";
    case PI_ERR_DTYPE: return "dtype must be PI_F16 or PI_BF16";
    case PI_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case PI_ERR_WORKSPACE: return "workspace smaller than pi_workspace_size()";
    case PI_ERR_CAPACITY: return "more active neurons than the index list holds";
    case PI_ERR_LAUNCH: return "the persistent grid cannot be co-resident on this GPU";
    case PI_ERR_TIMEOUT: return "a bounded grid-wide wait ran out";
    case PI_ERR_CUDA: return "a CUDA runtime call failed";
    case PI_ERR_INDEX: return "an active-list entry is outside [0, n)";
    case PI_ERR_RANGE: return "a predictor partial sum is outside the fixed-point range";
    case PI_ERR_CAPTURE:
      return "a one-time setup of this call cannot run while the stream is being captured";
  }
  return "unknown status";
}

// pi_predict; with split_x (batched calls of pi_layer_decode) the batched
// stage 1 also writes x's operand parts for the FFN phases and *split is set.
pi_status predict_impl(const pi_ffn_desc* desc, const void* A, const void* Bm, const float* b1,
                       const float* x, int32_t batch, float* logits, void* ws, size_t ws_bytes,
                       pi_stream stream, bool split_x, bool* split) {
  if (split) *split = false;
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > kMaxBatch) return PI_ERR_SHAPE;
  if (!A || !Bm || !b1 || !x || !logits || !ws) return PI_ERR_NULL;
  const void* ps[] = {A, Bm, b1, x, logits, ws};
  for (const void* p : ps)
    if (!aligned16(p)) return PI_ERR_ALIGN;
  const WsLayout L = ws_layout(*desc, batch);
  if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
  const pi_ffn_desc& D = *desc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (batch > 1 && D.r % 16 == 0) {
    // column-split stage 1 + fixed-order reduction, stage 2 on the tensor cores
    DevInfo di;
    pi_status s = dev_info(&di);
    if (s != PI_OK) return s;
    char* b = static_cast<char*>(ws);
    float* part = reinterpret_cast<float*>(b + L.ppart);
    uint16_t* uhi = reinterpret_cast<uint16_t*>(b + L.uhi);
    uint16_t* ulo = reinterpret_cast<uint16_t*>(b + L.ulo);
    const int nch = D.d / 8;
    const int G = nch < di.sms ? nch : (di.sms < kPMax ? di.sms : kPMax);
    const int wmax = 8 * ((nch + G - 1) / G);
    const size_t smem1 = sizeof(float) * (size_t)batch * wmax;
    const bool bf = D.dtype == PI_BF16;
    const uint16_t* Bh = static_cast<const uint16_t*>(Bm);
    const bool tb8 = batch <= 8;
    auto fp = bf ? (tb8 ? bpu_partial_kernel<1, 8> : bpu_partial_kernel<1, 32>)
                 : (tb8 ? bpu_partial_kernel<0, 8> : bpu_partial_kernel<0, 32>);
    uint16_t* xhi = split_x ? reinterpret_cast<uint16_t*>(b + L.xhi) : nullptr;
    uint16_t* xlo = split_x ? reinterpret_cast<uint16_t*>(b + L.xlo) : nullptr;
    if (launch_chain(fp, G, 256, smem1, st, Bh, x, D.d, D.r, batch, G, part, xhi, xlo, L.bp) !=
        cudaSuccess)
      return PI_ERR_CUDA;
    if (split) *split = split_x;
    const int bp = L.bp;
    const unsigned gr = (unsigned)((bp * D.r + 31) / 32);
    if (launch_chain(bf ? bpu_reduce_kernel<1> : bpu_reduce_kernel<0>, gr, 256, 0, st,
                     (const float*)part, D.r, batch, bp, G, uhi, ulo) != cudaSuccess)
      return PI_ERR_CUDA;
    const int smem2 = (kLT + 2 * bp) * (2 * D.r + 16);
    using LFn = void (*)(const uint16_t*, const float*, const uint16_t*, const uint16_t*, int, int,
                         int, int, float*);
    LFn fl = bf ? (bp == 32 ? blogit_kernel<1, 2> : blogit_kernel<1, 1>)
                : (bp == 32 ? blogit_kernel<0, 2> : blogit_kernel<0, 1>);
    s = ensure_smem(reinterpret_cast<const void*>(fl), smem2);
    if (s != PI_OK) return s;
    if (launch_chain(fl, (unsigned)((D.n + kLT - 1) / kLT), 256, smem2, st,
                     static_cast<const uint16_t*>(A), b1, (const uint16_t*)uhi,
                     (const uint16_t*)ulo, D.n, D.r, batch, bp, logits) != cudaSuccess)
      return PI_ERR_CUDA;
    return PI_OK;
  }
  float* u = reinterpret_cast<float*>(static_cast<char*>(ws) + L.u);
  const uint16_t* Bh = static_cast<const uint16_t*>(Bm);
  const uint16_t* Ah = static_cast<const uint16_t*>(A);
  const int tb = batch == 1 ? 1 : (batch <= 8 ? 8 : 32);
  const bool bf = D.dtype == PI_BF16;
#define PI_U(DT, TB) predict_u_kernel<DT, TB><<<D.r, 256, 0, st>>>(Bh, x, D.d, D.r, batch, u)
  if (!bf) {
    if (tb == 1) PI_U(0, 1); else if (tb == 8) PI_U(0, 8); else PI_U(0, 32);
  } else {
    if (tb == 1) PI_U(1, 1); else if (tb == 8) PI_U(1, 8); else PI_U(1, 32);
  }
#undef PI_U
  if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  int rc = D.r / 8, G = 1;
  while (G < rc) G <<= 1;
  const int rows_per_block = 8 * (32 / G) * 4;
  const unsigned grid = (unsigned)((D.n + rows_per_block - 1) / rows_per_block);
  const size_t smem = sizeof(float) * (size_t)batch * D.r;
#define PI_L(DT, TB) \
  predict_logits_kernel<DT, TB><<<grid, 256, smem, st>>>(Ah, b1, u, D.n, D.r, batch, logits)
  if (!bf) {
    if (tb == 1) PI_L(0, 1); else if (tb == 8) PI_L(0, 8); else PI_L(0, 32);
  } else {
    if (tb == 1) PI_L(1, 1); else if (tb == 8) PI_L(1, 8); else PI_L(1, 32);
  }
#undef PI_L
  if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

pi_status pi_predict(const pi_ffn_desc* desc, const void* A, const void* Bm, const float* b1,
                     const float* x, int32_t batch, float* logits, void* ws, size_t ws_bytes,
                     pi_stream stream) {
  return predict_impl(desc, A, Bm, b1, x, batch, logits, ws, ws_bytes, stream, false, nullptr);
}

pi_status pi_compact(const float* logits, int32_t n, int32_t batch, int32_t* idx, int32_t* cnt,
                     int32_t cap, int32_t* union_idx, int32_t* union_cnt, uint32_t* tok_mask,
                     int32_t* dev_status, void* ws, size_t ws_bytes, pi_stream stream) {
  if (n < 1 || n > (1 << 24) || batch < 1 || batch > kMaxBatch || cap < 0) return PI_ERR_SHAPE;
  if (!logits || !idx || !cnt) return PI_ERR_NULL;
  if (cap < n && !dev_status) return PI_ERR_NULL;
  if (union_idx && (!union_cnt || !tok_mask)) return PI_ERR_NULL;
  const void* ps[] = {logits, idx, cnt, union_idx, union_cnt, tok_mask, dev_status};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t need = compact_scratch_bytes(n);
  if (ws && ws_bytes >= need) {
    // grid-wide: counts in the workspace's last region (see ws_layout)
    int* scr = reinterpret_cast<int*>(static_cast<char*>(ws) + ((ws_bytes - need) & ~(size_t)15));
    const int nb = (n + kCB - 1) / kCB;
    const int wu = union_idx ? 1 : 0;
    // up to 128 blocks the write kernel sums the counts before it itself
    const int fused = nb <= 128 ? 1 : 0;
    if (launch_chain(cu_count_kernel, nb, kCB, 0, st, logits, n, batch, wu, scr, nb) !=
            cudaSuccess ||
        (!fused &&
         launch_chain(cu_scan_kernel, 1, 1024, 0, st, scr, nb, batch, wu) != cudaSuccess) ||
        launch_chain(cu_write_kernel, nb, kCB, 0, st, logits, n, batch, (const int*)scr, nb, idx,
                     cnt, cap, union_idx, union_cnt, tok_mask, dev_status, fused) != cudaSuccess)
      return PI_ERR_CUDA;
    return PI_OK;
  }
  // without a workspace: one block per token, one block for the union
  compact_kernel<<<batch, 1024, 0, st>>>(logits, n, idx, cnt, cap, dev_status);
  if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  if (union_idx) {
    union_kernel<<<1, 1024, 0, st>>>(logits, n, batch, union_idx, union_cnt, tok_mask);
    if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  }
  return PI_OK;
}

pi_status pi_sparse_ffn(const pi_ffn_desc* desc, const pi_layer_weights* w, const float* x,
                        int32_t batch, const int32_t* idx, const int32_t* cnt, int32_t cap,
                        const int32_t* union_idx, const int32_t* union_cnt,
                        const uint32_t* tok_mask, float* y, int32_t* dev_status, void* ws,
                        size_t ws_bytes, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > kMaxBatch) return PI_ERR_SHAPE;
  s = check_weights(*desc, w, false);
  if (s != PI_OK) return s;
  if (batch > 1) {
    if (!x || !y || !union_idx || !union_cnt || !tok_mask || !ws) return PI_ERR_NULL;
    const void* pb[] = {x, y, union_idx, union_cnt, tok_mask, ws};
    for (const void* p : pb)
      if (!aligned16(p)) return PI_ERR_ALIGN;
    if (desc->d % kBK) return PI_ERR_SHAPE;  // the batched path tiles d by 128
    const WsLayout L = ws_layout(*desc, batch);
    if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
    (void)idx;
    (void)cnt;
    (void)cap;
    return launch_batched(*desc, *w, x, batch, union_idx, union_cnt, tok_mask, y, nullptr, L, ws,
                          reinterpret_cast<cudaStream_t>(stream), dev_status);
  }
  return sparse_one(desc, w, x, idx, cnt, cap, y, dev_status, ws, ws_bytes, stream, 0, 0);
}

pi_status pi_dense_ffn(const pi_ffn_desc* desc, const pi_layer_weights* w, const float* x,
                       int32_t batch, float* y, void* ws, size_t ws_bytes, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > kMaxBatch) return PI_ERR_SHAPE;
  s = check_weights(*desc, w, false);
  if (s != PI_OK) return s;
  if (!x || !y || !ws) return PI_ERR_NULL;
  const void* ps[] = {x, y, ws};
  for (const void* p : ps)
    if (!aligned16(p)) return PI_ERR_ALIGN;
  const WsLayout L = ws_layout(*desc, batch);
  if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
  if (batch > 1 && desc->d % kBK == 0)  // every row read once for all tokens, tensor cores
    return launch_batched(*desc, *w, x, batch, nullptr, nullptr, nullptr, y, nullptr, L, ws,
                          reinterpret_cast<cudaStream_t>(stream), nullptr);
  for (int t = 0; t < batch; ++t) {
    FfnArgs a{};
    bind_weights(a, *w);
    bind_ws(a, L, ws);
    a.x = x + (size_t)t * desc->d;
    a.residual = nullptr;
    a.y = y + (size_t)t * desc->d;
    a.status = nullptr;
    s = launch_ffn<kDense>(*desc, a, desc->n, reinterpret_cast<cudaStream_t>(stream));
    if (s != PI_OK) return s;
  }
  return PI_OK;
}

pi_status pi_layer_decode(const pi_ffn_desc* desc, const pi_layer_weights* w, const float* x,
                          int32_t batch, float* y, const float* residual, int32_t* idx_out,
                          int32_t* cnt_out, int32_t* dev_status, void* ws, size_t ws_bytes,
                          pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (batch < 1 || batch > kMaxBatch) return PI_ERR_SHAPE;
  s = check_weights(*desc, w, true);
  if (s != PI_OK) return s;
  if (!x || !y || !dev_status || !ws) return PI_ERR_NULL;
  const void* ps[] = {x, y, residual, dev_status, ws};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  // the active lists and counts are written element by element
  if ((reinterpret_cast<uintptr_t>(idx_out) | reinterpret_cast<uintptr_t>(cnt_out)) & 3u)
    return PI_ERR_ALIGN;
  const WsLayout L = ws_layout(*desc, batch);
  if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
  const size_t d = (size_t)desc->d, n = (size_t)desc->n;
  if (batch > 1 && desc->d % kBK == 0) {
    // batched: predictor over all tokens (A, Bm read once), per-token lists,
    // their union, then the tensor-core contraction over the union
    char* b = static_cast<char*>(ws);
    float* logits = reinterpret_cast<float*>(b + L.logits);
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(b + L.bidx);
    int32_t* cnt = cnt_out ? cnt_out : reinterpret_cast<int32_t*>(b + L.bcnt);
    int32_t* uidx = reinterpret_cast<int32_t*>(b + L.uidx);
    int32_t* ucnt = reinterpret_cast<int32_t*>(b + L.ucnt);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(b + L.tmask);
    bool split = false;  // the predictor also wrote x's operand parts
    s = predict_impl(desc, w->A, w->Bm, w->b1, x, batch, logits, ws, ws_bytes, stream, true,
                     &split);
    if (s != PI_OK) return s;
    s = pi_compact(logits, desc->n, batch, idx, cnt, desc->n, uidx, ucnt, tmask, dev_status, ws,
                   ws_bytes, stream);
    if (s != PI_OK) return s;
    return launch_batched(*desc, *w, x, batch, uidx, ucnt, tmask, y, residual, L, ws,
                          reinterpret_cast<cudaStream_t>(stream), dev_status, split);
  }
  for (int t = 0; t < batch; ++t) {
    FfnArgs a{};
    bind_weights(a, *w);
    bind_ws(a, L, ws);
    a.x = x + t * d;
    a.residual = residual ? residual + t * d : nullptr;
    a.y = y + t * d;
    a.idx_out = idx_out ? idx_out + t * n : nullptr;
    a.cnt_out = cnt_out ? cnt_out + t : nullptr;
    if (!a.idx_out) a.mask = nullptr;  // the mask is only kept to build idx_out
    a.status = dev_status;
    s = launch_ffn<kFused>(*desc, a, desc->n, reinterpret_cast<cudaStream_t>(stream));
    if (s != PI_OK) return s;
  }
  return PI_OK;
}

pi_status pi_decode_layers(const pi_ffn_desc* descs, const pi_layer_weights* layers, int32_t R,
                           int32_t J, const float* x, int32_t chain, float* y, int32_t* cnt_out,
                           uint8_t* mask_out, int32_t* dev_status, void* ws, size_t ws_bytes,
                           pi_stream stream) {
  if (!descs || !layers) return PI_ERR_NULL;
  if (R < 1 || R > kSeqMaxLayers || J < 1 || (chain != 0 && chain != 1)) return PI_ERR_SHAPE;
  pi_ffn_desc D = descs[0];
  int hot_max = 0, r_max = 0;
  for (int l = 0; l < R; ++l) {
    const pi_ffn_desc& E = descs[l];
    pi_status s = check_desc(&E);
    if (s != PI_OK) return s;
    if (E.d != D.d || E.n != D.n || E.dtype != D.dtype || E.gated != D.gated ||
        E.layout != D.layout)
      return PI_ERR_SHAPE;
    if (E.r > r_max) r_max = E.r;
    s = check_weights(E, &layers[l], true);
    if (s != PI_OK) return s;
    if (E.hot_prefix > hot_max) hot_max = E.hot_prefix;
  }
  if (!x || !y || !dev_status || !ws) return PI_ERR_NULL;
  const void* ps[] = {x, y, cnt_out, dev_status, ws};
  for (const void* p : ps)
    if (p && !aligned16(p)) return PI_ERR_ALIGN;
  D.r = r_max;  // buffers and shared memory for the largest rank; each job uses its own
  const WsLayout L = ws_layout(D, 1);
  if (ws_bytes < L.total) return PI_ERR_WORKSPACE;
  DevInfo di;
  pi_status s = dev_info(&di);
  if (s != PI_OK) return s;
  const int P = di.sms < kPMax ? di.sms : kPMax;
  if ((D.d / 8 + P - 1) / P > kSeqMaxQ) return PI_ERR_SHAPE;  // own columns per block
  if ((D.n + P - 1) / P > 32 * 256) return PI_ERR_SHAPE;      // own neurons per block
  D.hot_prefix = hot_max;
  const bool wide = (D.d / 8) > kThreads;
  SeqFn fn = pick_seq(D.dtype, D.gated, wide);
  FfnArgs a{};
  const int smem = plan_ffn(D, kFused, P, D.n, di.smem_optin - 1024, a, true);
  if (smem == 0 || a.grp < 1) return PI_ERR_SHAPE;
  s = ensure_smem(reinterpret_cast<const void*>(fn), smem);
  if (s != PI_OK) return s;
  bind_ws(a, L, ws);
  a.mask = nullptr;
  a.idx_out = nullptr;
  a.cnt_out = nullptr;
  a.status = dev_status;
  set_waits(a);
  SeqArgs sa{};
  sa.f = a;
  sa.J = J;
  sa.R = R;
  sa.chain = chain;
  sa.x = x;
  sa.y = y;
  sa.cnt_out = cnt_out;
  sa.mask_out = mask_out;
  sa.uacc = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + L.uacc);
  const int qmax = (D.d / 8 + P - 1) / P;
  sa.bm_smem = (a.nh < a.ns - 1 && D.r * qmax * 16 <= a.slot_bytes) ? 1 : 0;
  // predictor rows that do not fit beside the ring wait in its idle slots
  // (after the hot ones, before the Bm slot) between jobs
  sa.a_slots = (!a.a_in_smem && sa.bm_smem &&
                (long long)(a.ns - 1 - a.nh) * a.slot_bytes >= (long long)a.rows_max * a.a_stride)
                   ? 1 : 0;
  if (const char* e = std::getenv("PI_SEQ_A_SLOTS")) sa.a_slots = sa.a_slots && std::atoi(e) != 0;
  sa.glist = reinterpret_cast<int2*>(static_cast<char*>(ws) + L.glist);
  sa.gcnt = reinterpret_cast<int*>(static_cast<char*>(ws) + L.gcnt);
  sa.balance = 0;  // measured: no gain on the 48-layer stack (its extra wait costs the tail)
  if (const char* e = std::getenv("PI_SEQ_BALANCE")) sa.balance = std::atoi(e) != 0;

  for (int l = 0; l < R; ++l) {
    const pi_layer_weights& w = layers[l];
    SeqLayer& e = sa.L[l];
    e.A = static_cast<const uint16_t*>(w.A);
    e.Bm = static_cast<const uint16_t*>(w.Bm);
    e.b1 = w.b1;
    e.W1 = static_cast<const uint16_t*>(w.W1);
    e.W2 = static_cast<const uint16_t*>(w.W2);  // NULL when packed (records hold both)
    e.b2 = w.b2;
    e.hot = descs[l].hot_prefix;
    e.r = descs[l].r;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P);
  cfg.blockDim = dim3(kBlock);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (launch_mode() == 0) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kBlock, (size_t)smem) !=
        cudaSuccess)
      return PI_ERR_CUDA;
    if (per_sm < 1) return PI_ERR_LAUNCH;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the fixed-point u accumulators start at zero (the kernel keeps them so
  // between its jobs)
  if (cudaMemsetAsync(sa.uacc, 0, 2 * 128 * (size_t)D.r, cfg.stream) != cudaSuccess)
    return PI_ERR_CUDA;
  return map_launch_error(cudaLaunchKernelEx(&cfg, fn, sa));
}

pi_status pi_profile_counts(const float* logits, int32_t n, int32_t batch, uint32_t* counts,
                            pi_stream stream) {
  if (n < 1 || n > (1 << 24) || batch < 1 || batch > kMaxBatch) return PI_ERR_SHAPE;
  if (!logits || !counts) return PI_ERR_NULL;
  if (!aligned16(logits) || !aligned16(counts)) return PI_ERR_ALIGN;
  const unsigned grid = (unsigned)((n + 255) / 256);
  profile_count_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      logits, n, batch, reinterpret_cast<unsigned*>(counts));
  return cudaGetLastError() == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}

pi_status pi_hot_order(const uint32_t* counts, int32_t n, int32_t* perm, pi_stream stream) {
  if (n < 1 || n > (1 << 22)) return PI_ERR_SHAPE;
  if (!counts || !perm) return PI_ERR_NULL;
  if (!aligned16(counts) || !aligned16(perm)) return PI_ERR_ALIGN;
  rank_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const unsigned*>(counts), n, perm);
  return cudaGetLastError() == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}

pi_status pi_permute_neurons(const pi_ffn_desc* desc, const pi_layer_weights* src,
                             const int32_t* perm, const pi_layer_weights* dst,
                             int32_t* dev_status, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  if (!src || !dst || !perm || !dev_status) return PI_ERR_NULL;
  const pi_ffn_desc& D = *desc;
  s = check_weights(D, src, true);
  if (s != PI_OK) return s;
  s = check_weights(D, dst, true);
  if (s != PI_OK) return s;
  if (!aligned16(perm) || !aligned16(dev_status)) return PI_ERR_ALIGN;
  // out of place only: every permuted tensor gets a buffer of its own
  if (dst->A == src->A || dst->b1 == src->b1 || dst->W1 == src->W1 ||
      (D.layout == PI_LAYOUT_SPLIT && dst->W2 == src->W2))
    return PI_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int m1 = D.gated ? 2 : 1;
  const long long w1q = (D.layout == PI_LAYOUT_PACKED ? (long long)(m1 + 1) : m1) * D.d / 8;
  struct Job {
    const void* a;
    void* b;
    long long q16;
  } jobs[3] = {{src->A, const_cast<void*>(dst->A), D.r / 8},
               {src->W1, const_cast<void*>(dst->W1), w1q},
               {src->W2, const_cast<void*>(dst->W2), D.d / 8}};
  const int nj = D.layout == PI_LAYOUT_SPLIT ? 3 : 2;
  for (int j = 0; j < nj; ++j) {
    const long long tot = (long long)D.n * jobs[j].q16;
    const long long blocks = (tot + 255) / 256;
    gather_rows16_kernel<<<(unsigned)(blocks < 152 * 64 ? blocks : 152 * 64), 256, 0, st>>>(
        static_cast<const uint4*>(jobs[j].a), static_cast<uint4*>(jobs[j].b), perm, D.n,
        jobs[j].q16, dev_status);
  }
  gather_f32_kernel<<<(unsigned)((D.n + 255) / 256), 256, 0, st>>>(
      src->b1, const_cast<float*>(dst->b1), perm, D.n, dev_status);
  return cudaGetLastError() == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}

pi_status pi_pack_weights(const pi_ffn_desc* desc, const void* W1, const void* W2, void* packed,
                          pi_stream stream) {
  pi_ffn_desc D = desc ? *desc : pi_ffn_desc{};
  D.layout = PI_LAYOUT_SPLIT;
  pi_status s = check_desc(desc ? &D : nullptr);
  if (s != PI_OK) return s;
  if (!W1 || !W2 || !packed) return PI_ERR_NULL;
  if (!aligned16(W1) || !aligned16(W2) || !aligned16(packed)) return PI_ERR_ALIGN;
  const int m1 = D.gated ? 2 : 1, d8 = D.d / 8;
  const long long total = (long long)D.n * (m1 + 1) * d8;
  const unsigned grid = (unsigned)((total + 255) / 256 < 65535 * 8 ? (total + 255) / 256 : 65535 * 8);
  pack_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(W1), static_cast<const uint4*>(W2), static_cast<uint4*>(packed), D.n,
      d8, m1);
  if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

pi_status pi_selftest_ring_timeout(const pi_ffn_desc* desc, const pi_layer_weights* w,
                                   const float* x, const int32_t* idx, const int32_t* cnt,
                                   int32_t cap, float* y, int32_t* dev_status, void* ws,
                                   size_t ws_bytes, int64_t limit_ns, pi_stream stream) {
  pi_status s = check_desc(desc);
  if (s != PI_OK) return s;
  s = check_weights(*desc, w, false);
  if (s != PI_OK) return s;
  if (limit_ns < 1000 || limit_ns > 5000000000LL) return PI_ERR_SHAPE;
  return sparse_one(desc, w, x, idx, cnt, cap, y, dev_status, ws, ws_bytes, stream,
                    (unsigned long long)limit_ns, 1);
}

pi_status pi_selftest_wait_timeout(int32_t* dev_status, void* ws, size_t ws_bytes,
                                   int64_t limit_ns, pi_stream stream) {
  if (!dev_status || !ws) return PI_ERR_NULL;
  if (!aligned16(dev_status) || !aligned16(ws)) return PI_ERR_ALIGN;
  if (ws_bytes < 256) return PI_ERR_WORKSPACE;
  if (limit_ns < 1000 || limit_ns > 5000000000LL) return PI_ERR_SHAPE;
  wait_timeout_kernel<<<4, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long*>(ws), dev_status, (unsigned long long)limit_ns);
  if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
  return PI_OK;
}

}  // extern "C"

#include "decoder.cuh"
#include "shard.cuh"

// api.cu -- the C ABI declared in include/gbfuse.h (and the test and tuning
// hooks of include/gbfuse_debug.h): argument validation,
// TMA tensor-map encoding, kernel-family selection by shape, launch, and
// status codes.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/gbfuse.h"
#include "../../include/gbfuse_debug.h"
#include "internal.h"

namespace gbf {

// The device error word written by kernels that give up on a bounded wait.
__device__ unsigned g_gbf_error_word;

namespace {

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_inject{0};
std::atomic<int> g_force_splits{0};
std::atomic<int> g_force_path{0};
std::atomic<unsigned long long*> g_prof{nullptr};
std::atomic<size_t> g_prof_bytes{0};

constexpr int kMaxDevices = 64;

struct DevState {
  std::mutex mu;
  std::atomic<bool> ready{false};
  DeviceInfo info;
  unsigned* err = nullptr;
};
DevState g_dev[kMaxDevices];

std::mutex g_encode_mu;
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

// Current device, its properties and the address of its error word.  The
// lookup is made once per device; only a successful one is kept, so a call
// made before the device could answer (e.g. during a failed context set-up)
// does not disable the library on that device: the next call tries again.
gbf_status_t current_device(const DeviceInfo** info, unsigned** err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return GBF_ERR_NO_DEVICE;
  DevState& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int sms = 0, major = 0, minor = 0;
      void* p = nullptr;
      cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_gbf_error_word);
      if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();  // not sticky: leave no error behind for the caller
        return GBF_ERR_CUDA;
      }
      d.err = static_cast<unsigned*>(p);
      d.info.sms = sms;
      d.info.pairs = (major == 10 && minor == 3) ? max_active_pairs() : 0;
      if (d.info.pairs <= 0) d.info.pairs = sms / 2;
      d.info.quads = (major == 10 && minor == 3) ? max_active_quads() : 0;
      d.info.cc_major = major;
      d.info.cc_minor = minor;
      d.ready.store(true, std::memory_order_release);
    }
  }
  if (d.info.cc_major != 10 || d.info.cc_minor != 3) return GBF_ERR_NO_DEVICE;
  *info = &d.info;
  *err = d.err;
  return GBF_OK;
}

// The driver's tensor-map encoder (looked up until a lookup succeeds).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  PFN_cuTensorMapEncodeTiled_v12000 fn = g_encode.load(std::memory_order_acquire);
  if (fn) return fn;
  std::lock_guard<std::mutex> lock(g_encode_mu);
  fn = g_encode.load(std::memory_order_relaxed);
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && p) {
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    g_encode.store(fn, std::memory_order_release);
  } else {
    (void)cudaGetLastError();
  }
  return fn;
}

// Row-major 2-D tensor [outer][inner] with `row_bytes` between rows.
//
// Encoded maps are kept in a small per-thread cache keyed by every argument:
// a descriptor is a pure function of them, and a model calls the same layer
// shapes on the same buffers step after step, so an un-graphed call then
// skips the host-side encode.
struct TmapKey {
  const void* base;
  uint64_t inner, outer, row_bytes;
  uint32_t box_inner, box_outer;
  int dt, swz;
  bool operator==(const TmapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
           box_inner == o.box_inner && box_outer == o.box_outer && dt == o.dt && swz == o.swz;
  }
};
struct TmapEntry {
  CUtensorMap map;
  TmapKey key;
  bool valid;
};
constexpr int kTmapCacheSize = 32;
thread_local TmapEntry t_tmap_cache[kTmapCacheSize];
thread_local int t_tmap_next = 0;

bool tmap_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner,
             uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapSwizzle swz) {
  const TmapKey key{base, inner, outer, row_bytes, box_inner, box_outer, static_cast<int>(dt),
                    static_cast<int>(swz)};
  for (int i = 0; i < kTmapCacheSize; ++i) {
    const TmapEntry& e = t_tmap_cache[i];
    if (e.valid && e.key == key) {
      *m = e.map;
      return true;
    }
  }
  const PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  if (encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmapEntry& slot = t_tmap_cache[t_tmap_next];
  t_tmap_next = (t_tmap_next + 1) % kTmapCacheSize;
  slot.map = *m;
  slot.key = key;
  slot.valid = true;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

gbf_status_t check_common(int64_t M, int64_t N, int64_t K, int act) {
  if (M < 0 || N < 0 || K < 0) return GBF_ERR_INVALID_ARG;
  if (act < GBF_ACT_IDENTITY || act > GBF_ACT_GELU_TANH) return GBF_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GBF_ERR_UNSUPPORTED_SHAPE;
  if (N % 8 != 0 || K % 8 != 0) return GBF_ERR_UNSUPPORTED_SHAPE;
  return GBF_OK;
}

gbf_status_t check_ptrs(std::initializer_list<const void*> required,
                        std::initializer_list<const void*> optional) {
  for (const void* p : required) {
    if (!p) return GBF_ERR_INVALID_ARG;
    if (!aligned16(p)) return GBF_ERR_MISALIGNED;
  }
  for (const void* p : optional)
    if (p && !aligned16(p)) return GBF_ERR_MISALIGNED;
  return GBF_OK;
}

// Launch control; the wait-time counters are passed only when the
// registered buffer has room for every CTA of the launch.
KernelCtl make_ctl(unsigned* err, int64_t ctas) {
  unsigned long long* prof = g_prof.load();
  if (prof && static_cast<size_t>(ctas) * kProfSlots * 8 > g_prof_bytes.load()) prof = nullptr;
  return KernelCtl{err, static_cast<unsigned long long>(g_timeout_ns.load()), g_inject.load(),
                   prof};
}

int64_t plan_ctas(const GemmPlan& p) {
  if (p.path == kPathSwap || p.path == kPathW4)
    return static_cast<int64_t>(p.splits) * p.n_tiles * p.m_tiles;
  return p.grid;
}

gbf_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? GBF_OK : GBF_ERR_CUDA; }

EpiParams make_ep(const void* C, const void* bias, const void* residual, void* out, float alpha,
                  float beta, int act) {
  return EpiParams{static_cast<const __nv_bfloat16*>(C), static_cast<const __nv_bfloat16*>(bias),
                   static_cast<const __nv_bfloat16*>(residual), static_cast<__nv_bfloat16*>(out),
                   alpha, beta, act};
}

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

int choose_splits(int tiles, int num_kb, const DeviceInfo& dev) {
  const int slots = dev.sms * 2;  // the swapped kernels fit two CTAs per SM
  int s = tiles > 0 ? slots / tiles : 1;
  if (const int f = g_force_splits.load()) s = f;
  s = std::max(1, std::min(s, kMaxSplits));
  s = std::min(s, std::max(1, num_kb));
  return s;
}

// Dense GEMM (+ dual) launch after validation.  D rows of out.
gbf_status_t run_gemm(const void* A, const void* W, const void* W2, int layout, bool dual,
                      const EpiParams& ep, int64_t M, int64_t N, int64_t K,
                      const DeviceInfo& dev, unsigned* err, cudaStream_t stream) {
  if (M == 0 || N == 0) return GBF_OK;
  if (K == 0) {
    if (dual) {
      // act(0) * 0 + beta*C: a zero product through the GLU ending.
      EpiParams z = ep;
      z.alpha = 0.0f;
      z.act = GBF_ACT_IDENTITY;
      z.bias = nullptr;
      z.residual = nullptr;
      return cuda_status(launch_pointwise_epilogue(nullptr, z, M, N, dev.sms, stream));
    }
    return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev.sms, stream));
  }
  const bool kn = layout == GBF_B_KN;
  const GemmPlan plan = plan_gemm(M, N, K, dual, kn, dev);
  CUtensorMap tmA, tmW, tmW2;
  const uint32_t a_rows = plan.path == kPathSwap ? plan.mpad : kBM;
  const bool pair =
      plan.path == kPathPair || plan.path == kPathPairOne || plan.path == kPathPairSplit;
  if (!tmap_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, K * 2, kBK, a_rows,
               CU_TENSOR_MAP_SWIZZLE_128B))
    return GBF_ERR_CUDA;
  uint32_t w_rows = plan.path == kPathSwap ? 128
                    : pair                  ? (dual ? 128 : plan.bn / 2)
                                            : (dual ? 128 : kPersistBN);
  const void* ws[2] = {W, dual ? W2 : W};
  CUtensorMap* maps[2] = {&tmW, &tmW2};
  for (int i = 0; i < 2; ++i) {
    bool ok = kn ? tmap_2d(maps[i], ws[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, K, N * 2, 64, kBK,
                           CU_TENSOR_MAP_SWIZZLE_128B)
                 : tmap_2d(maps[i], ws[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, K * 2, kBK,
                           w_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return GBF_ERR_CUDA;
  }
  // the output for the TMA stores of the persistent kernels' epilogues
  CUtensorMap tmO{};
  if (plan.path != kPathSwap &&
      !tmap_2d(&tmO, ep.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, N * 2, 32, 32,
               CU_TENSOR_MAP_SWIZZLE_64B))
    return GBF_ERR_CUDA;
  if (pair) {
    return cuda_status(launch_gemm_pair(plan, kn, dual, tmA, tmW, tmW2, tmO, ep, static_cast<int>(M),
                                        static_cast<int>(N), static_cast<int>(K),
                                        make_ctl(err, plan_ctas(plan)), stream));
  }
  return cuda_status(launch_gemm(plan, kn, dual, tmA, tmW, tmW2, tmO, ep, static_cast<int>(M),
                                 static_cast<int>(N), static_cast<int>(K),
                                 make_ctl(err, plan_ctas(plan)), stream));
}

// Weight-only quantised GEMM launch after validation (fmt: WqFmt).
gbf_status_t run_w4(int fmt, const void* A, const uint8_t* Wq, const void* scales, int group,
                    const EpiParams& ep, int64_t M, int64_t N, int64_t K, const DeviceInfo& dev,
                    unsigned* err, cudaStream_t stream) {
  if (M == 0 || N == 0) return GBF_OK;
  if (K == 0) return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev.sms, stream));
  const GemmPlan plan = plan_w4a16(M, N, K, dev);
  CUtensorMap tmA, tmQ, tmS;
  const bool fp8 = fmt == kWqFp8;
  const bool nv = fmt == kWqNvfp4;
  const int64_t qcols = fp8 ? N : N / 2;  // weight bytes per k-row
  bool ok = tmap_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, K * 2, kBK, plan.mpad,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
            tmap_2d(&tmQ, Wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qcols, K, qcols, 256, kBK,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  ok = ok && (nv ? tmap_2d(&tmS, scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, N, K / 16, N, 256,
                           kBK / 16, CU_TENSOR_MAP_SWIZZLE_NONE)
                 : tmap_2d(&tmS, scales, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, K / group, N * 2,
                           256, 1, CU_TENSOR_MAP_SWIZZLE_NONE));
  if (!ok) return GBF_ERR_CUDA;
  return cuda_status(launch_wq_gemm(fmt, plan, tmA, tmQ, tmS, ep, static_cast<int>(M),
                                    static_cast<int>(N), static_cast<int>(K), group,
                                    make_ctl(err, plan_ctas(plan)), stream));
}

gbf_status_t check_w4(int64_t M, int64_t N, int64_t K, int group, int act) {
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (group <= 0) return GBF_ERR_INVALID_ARG;
  if (group % kBK != 0 || K % group != 0 || N % 32 != 0) return GBF_ERR_UNSUPPORTED_SHAPE;
  return GBF_OK;
}

// NVFP4: blocks of 16 along K; packed rows of N/2 bytes.
gbf_status_t check_nvfp4(int64_t M, int64_t N, int64_t K, int act) {
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (K % 16 != 0 || N % 32 != 0) return GBF_ERR_UNSUPPORTED_SHAPE;
  return GBF_OK;
}

}  // namespace

namespace {

// The CTA-pair kernel: pairs of 256-row M-tiles share each B tile (a unit of
// 512 x bn per pair of SMs), persistent over the units.  With one stream
// (single product only) a unit is one 256-row M-tile x 256 columns.
GemmPlan pair_plan(int64_t M, int64_t N, bool dual, bool kn, const DeviceInfo& dev,
                   int streams = 2) {
  GemmPlan p;
  p.path = kPathPair;
  p.m_tiles = ceil_div(M, 2 * kBM);
  p.n_tiles = ceil_div(N, dual ? 128 : kPersistBN);
  p.bn = 256;
  if (streams == 1 && !dual) {
    p.path = kPathPairOne;
    p.streams = 1;
    // 224-wide tiles for K-contiguous weights when they fill the rounds of
    // 256 x bn units better.  One stream's MMAs take about the same time
    // whatever their N, so the gain is only the fuller round (measured at
    // 1024 x 4096 x 4096: 1202 -> 1236 TFLOP/s); for B as [K][N] the wider
    // loads cost more than that (1536 x 8192 x 8192: 1587 -> 1500).
    auto eff1 = [&](int bn) {
      const int64_t tiles = static_cast<int64_t>(p.m_tiles) * ceil_div(N, bn);
      const int64_t rounds = (tiles + dev.pairs - 1) / dev.pairs;
      return static_cast<double>(M) * N / (static_cast<double>(rounds) * dev.pairs * 256 * bn);
    };
    if (!kn && eff1(224) > eff1(256) * 1.02) {
      p.bn = 224;
      p.n_tiles = ceil_div(N, 224);
    }
    p.grid = 2 * std::min(p.m_tiles * p.n_tiles, dev.pairs);
    // one tile per pair: the two accumulators need not alternate between
    // tiles, so two MMA streams share the tile's K blocks
    p.kpar = static_cast<int64_t>(p.m_tiles) * p.n_tiles <= dev.pairs;
    return p;
  }
  if (!dual) {
    // A 224-wide tile when it wastes less of the last round of tiles:
    // compare useful area / (rounds * pairs * tile area).
    // (a pair computes two M-tiles at a time: 512 x bn per round)
    auto eff = [&](int bn) {
      const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * ceil_div(N, bn);
      const int64_t rounds = (tiles + dev.pairs - 1) / dev.pairs;
      return static_cast<double>(M) * N / (static_cast<double>(rounds) * dev.pairs * 512 * bn);
    };
    if (eff(224) > eff(256) * 1.02) {
      p.bn = 224;
      p.n_tiles = ceil_div(N, 224);
    }
  }
  p.grid = 2 * std::min(((p.m_tiles + 1) / 2) * p.n_tiles, dev.pairs);
  return p;
}

// The one-SM persistent kernel: 128 x 256 tiles (128 x 128 of each product
// for the gate/up GEMM).  When the tiles fill at most half of the SMs, the
// single product runs in its split-K form instead: a cluster of two CTAs per
// tile, each over half of K (`split` true; needs enough K blocks to pay for
// the exchange of the partial sums).
GemmPlan persistent_plan(int64_t M, int64_t N, int64_t K, bool dual, bool split,
                         const DeviceInfo& dev) {
  GemmPlan p;
  p.path = kPathPersistent;
  p.m_tiles = ceil_div(M, kBM);
  p.n_tiles = ceil_div(N, dual ? 128 : kPersistBN);
  p.num_kb = ceil_div(K, kBK);
  p.grid = std::min(p.m_tiles * p.n_tiles, std::max(1, dev.sms));
  if (split && !dual && p.num_kb >= 2) {
    p.path = kPathPersistentSplit;
    p.splits = 2;
    p.grid = 2 * p.m_tiles * p.n_tiles;
  }
  return p;
}

// The one-stream pair kernel's split-K form: a cluster of two CTA pairs per
// 256 x 256 tile, pair kp over the K half kp, one tile per cluster.
GemmPlan pair_split_plan(int64_t M, int64_t N, int64_t K) {
  GemmPlan p;
  p.path = kPathPairSplit;
  p.streams = 1;
  p.bn = 256;
  p.m_tiles = ceil_div(M, 2 * kBM);
  p.n_tiles = ceil_div(N, 256);
  p.num_kb = ceil_div(K, kBK);
  p.splits = 2;
  p.grid = 4 * p.m_tiles * p.n_tiles;
  return p;
}

// Chosen only when every tile's cluster runs at once (one round) and K has
// enough blocks to pay for the exchange of the partial sums.
bool pair_split_fits(int64_t M, int64_t N, int64_t K, bool dual, const DeviceInfo& dev) {
  const int64_t tiles = static_cast<int64_t>(ceil_div(M, 2 * kBM)) * ceil_div(N, 256);
  return !dual && dev.quads > 0 && tiles <= dev.quads && ceil_div(K, kBK) >= 8;
}

bool split_pays(int64_t M, int64_t N, int64_t K, bool dual, const DeviceInfo& dev) {
  const int64_t tiles = static_cast<int64_t>(ceil_div(M, kBM)) * ceil_div(N, kPersistBN);
  return !dual && 2 * tiles <= dev.sms && ceil_div(K, kBK) >= 8;
}

// Relative time of a plan: rounds of units times the MMA area of a unit per
// SM, over the rate of one SM.  A pair unit is 512 x bn on two SMs; a
// persistent tile 128 x 256 on one SM, whose single MMA stream runs at
// about 0.8 of the rate of the pair kernel's two streams (measured: ~8.7
// against ~11 TFLOP/s per SM).
double plan_time(const GemmPlan& p, bool dual, const DeviceInfo& dev) {
  if (p.path == kPathPersistentSplit)  // one round, half of K per SM, plus the exchange
    return 0.55 * 128.0 * 256.0 / 0.8;
  if (p.path == kPathPairSplit)  // one round of pairs at one stream's rate, half of K
    return 0.55 * 256.0 * 256.0 / 2.0 / 0.9;
  if (p.path == kPathPair) {
    const int64_t units = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles;
    const int64_t rounds = (units + dev.pairs - 1) / dev.pairs;
    return static_cast<double>(rounds) * 512.0 * (dual ? 256 : p.bn) / 2.0;
  }
  if (p.path == kPathPairOne) {  // one MMA stream: about 0.9 of the two streams' rate
    // (a unit takes about as long at bn = 224 as at 256)
    const int64_t units = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    const int64_t rounds = (units + dev.pairs - 1) / dev.pairs;
    return static_cast<double>(rounds) * 256.0 * 256.0 / 2.0 / 0.9;
  }
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  const int64_t rounds = (tiles + std::max(1, dev.sms) - 1) / std::max(1, dev.sms);
  return static_cast<double>(rounds) * 128.0 * 256.0 / 0.8;
}

}  // namespace

int check_gemm_call(const void* A, const void* B, int b_layout, const void* C, const void* bias,
                    const void* residual, const void* out, int64_t M, int64_t N, int64_t K,
                    int act) {
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (b_layout != GBF_B_KN && b_layout != GBF_B_NK) return GBF_ERR_INVALID_ARG;
  return check_ptrs({A, B, out}, {C, bias, residual});
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, bool dual, bool kn, const DeviceInfo& dev) {
  GemmPlan p;
  if (M == 0 || N == 0 || K == 0) return p;
  if (M <= (dual ? kSwapDualMaxM : 128)) {
    p.num_kb = ceil_div(K, kBK);
    p.path = kPathSwap;
    p.mpad = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
    p.m_tiles = 1;
    p.n_tiles = ceil_div(N, kSwapBN);
    p.splits = choose_splits(p.n_tiles, p.num_kb, dev);
    return p;
  }
  // Above the swapped kernel's range: the kernel with the shorter estimated
  // time (the pair kernel's 512-row units leave most SMs idle when there are
  // few of them), unless a tuning hook forces one.
  const int force = g_force_path.load();
  if (force == kPathPersistentSplit && !dual) return persistent_plan(M, N, K, dual, true, dev);
  if (force == kPathPairSplit && !dual && ceil_div(K, kBK) >= 2) return pair_split_plan(M, N, K);
  if (force == kPathPersistent) return persistent_plan(M, N, K, dual, false, dev);
  GemmPlan pp = persistent_plan(M, N, K, dual, split_pays(M, N, K, dual, dev), dev);
  if (dev.pairs <= 0) return pp;
  GemmPlan qp = pair_plan(M, N, dual, kn, dev);
  qp.num_kb = pp.num_kb;
  if (force == kPathPair) return qp;
  GemmPlan best = plan_time(qp, dual, dev) < plan_time(pp, dual, dev) ? qp : pp;
  if (!dual) {
    GemmPlan op = pair_plan(M, N, dual, kn, dev, 1);
    op.num_kb = pp.num_kb;
    if (force == kPathPairOne) return op;
    if (plan_time(op, dual, dev) < plan_time(best, dual, dev)) best = op;
    if (pair_split_fits(M, N, K, dual, dev)) {
      const GemmPlan sp = pair_split_plan(M, N, K);
      if (plan_time(sp, dual, dev) < plan_time(best, dual, dev)) best = sp;
    }
  }
  return best;
}

GemmPlan plan_w4a16(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
  GemmPlan p;
  if (M == 0 || N == 0 || K == 0) return p;
  p.path = kPathW4;
  p.num_kb = ceil_div(K, kBK);
  p.mpad = M <= 16 ? 16 : 32;
  p.m_tiles = ceil_div(M, p.mpad);
  p.n_tiles = ceil_div(N, kW4BN);
  p.splits = choose_splits(p.n_tiles * p.m_tiles, p.num_kb, dev);
  return p;
}

}  // namespace gbf

using namespace gbf;

extern "C" {

gbf_status_t gemm_epilogue(const void* A, const void* B, int b_layout, const void* C,
                           const void* bias, const void* residual, void* out, int64_t M,
                           int64_t N, int64_t K, float alpha, float beta, int act,
                           void* workspace, size_t workspace_bytes, gbf_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (b_layout != GBF_B_KN && b_layout != GBF_B_NK) return GBF_ERR_INVALID_ARG;
  if ((st = check_ptrs({A, B, out}, {C, bias, residual})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  return run_gemm(A, B, nullptr, b_layout, false, make_ep(C, bias, residual, out, alpha, beta, act),
                  M, N, K, *dev, err, reinterpret_cast<cudaStream_t>(stream));
}

gbf_status_t swiglu_dual_gemm(const void* x, const void* w_gate, const void* w_up, int w_layout,
                              void* h, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                              const void* C, int act, void* workspace, size_t workspace_bytes,
                              gbf_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (w_layout != GBF_B_KN && w_layout != GBF_B_NK) return GBF_ERR_INVALID_ARG;
  if ((st = check_ptrs({x, w_gate, w_up, h}, {C})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  return run_gemm(x, w_gate, w_up, w_layout, true,
                  make_ep(C, nullptr, nullptr, h, alpha, beta, act), M, N, K, *dev, err,
                  reinterpret_cast<cudaStream_t>(stream));
}

gbf_status_t w4a16_gemm(const void* A, const uint8_t* Wq, const void* scales, int group_size,
                        const void* C, const void* bias, const void* residual, void* out,
                        int64_t M, int64_t N, int64_t K, float alpha, float beta, int act,
                        void* workspace, size_t workspace_bytes, gbf_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  gbf_status_t st = check_w4(M, N, K, group_size, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  return run_w4(kWqInt4, A, Wq, scales, group_size,
                make_ep(C, bias, residual, out, alpha, beta, act), M, N, K, *dev, err,
                reinterpret_cast<cudaStream_t>(stream));
}

gbf_status_t w8a16_fp8_gemm(const void* A, const uint8_t* Wq, const void* scales,
                            int group_size, const void* C, const void* bias,
                            const void* residual, void* out, int64_t M, int64_t N, int64_t K,
                            float alpha, float beta, int act, void* workspace,
                            size_t workspace_bytes, gbf_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  gbf_status_t st = check_w4(M, N, K, group_size, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  return run_w4(kWqFp8, A, Wq, scales, group_size,
                make_ep(C, bias, residual, out, alpha, beta, act), M, N, K, *dev, err,
                reinterpret_cast<cudaStream_t>(stream));
}

gbf_status_t w4a16_nvfp4_gemm(const void* A, const uint8_t* Wq, const uint8_t* scales,
                              const void* C, const void* bias, const void* residual, void* out,
                              int64_t M, int64_t N, int64_t K, float alpha, float beta, int act,
                              void* workspace, size_t workspace_bytes, gbf_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  gbf_status_t st = check_nvfp4(M, N, K, act);
  if (st != GBF_OK) return st;
  // the kernel carries the product scaled by 2^-19 and restores it through
  // alpha, which must leave room for that factor
  if (std::fabs(alpha) >= 0x1p100f && std::fabs(alpha) != INFINITY) return GBF_ERR_INVALID_ARG;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  return run_w4(kWqNvfp4, A, Wq, scales, 16, make_ep(C, bias, residual, out, alpha, beta, act),
                M, N, K, *dev, err, reinterpret_cast<cudaStream_t>(stream));
}

gbf_status_t swiglu_pointwise(const void* g, const void* u, const void* C, void* h, int64_t M,
                              int64_t N, float alpha, float beta, int act, gbf_stream_t stream) {
  gbf_status_t st = check_common(M, N, 8, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({g, u, h}, {C})) != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  return cuda_status(launch_swiglu_pointwise(
      static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(u),
      make_ep(C, nullptr, nullptr, h, alpha, beta, act), M, N, dev->sms,
      reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
gbf_status_t check_rms(const void* a, const void* x, const void* w, const void* norm,
                       const void* resid, int64_t M, int64_t N, float eps, bool need_resid) {
  if (M < 0 || N < 0 || !(eps >= 0.0f)) return GBF_ERR_INVALID_ARG;
  if (need_resid && !resid) return GBF_ERR_INVALID_ARG;
  gbf_status_t st = check_ptrs({a, x, w, norm}, {resid});
  if (st != GBF_OK) return st;
  if (N % 8 != 0 || N > kRmsMaxN || M > kMaxDim) return GBF_ERR_UNSUPPORTED_SHAPE;
  return GBF_OK;
}
}  // namespace

gbf_status_t add_rmsnorm(const void* a, const void* x, const void* weight, void* out_norm,
                         void* out_resid, int64_t M, int64_t N, float eps, gbf_stream_t stream) {
  gbf_status_t st = check_rms(a, x, weight, out_norm, out_resid, M, N, eps, false);
  if (st != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  return cuda_status(launch_add_rmsnorm(
      static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(x),
      static_cast<const __nv_bfloat16*>(weight), static_cast<__nv_bfloat16*>(out_norm),
      static_cast<__nv_bfloat16*>(out_resid), M, static_cast<int>(N), eps, dev->sms,
      reinterpret_cast<cudaStream_t>(stream)));
}

gbf_status_t add_rmsnorm_unfused(const void* a, const void* x, const void* weight,
                                 void* out_norm, void* out_resid, int64_t M, int64_t N,
                                 float eps, gbf_stream_t stream) {
  gbf_status_t st = check_rms(a, x, weight, out_norm, out_resid, M, N, eps, true);
  if (st != GBF_OK) return st;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // kernel 1: the residual add, bf16(a + x) written to out_resid
  const EpiParams add = make_ep(nullptr, nullptr, x, out_resid, 1.0f, 0.0f, GBF_ACT_IDENTITY);
  if ((st = cuda_status(launch_pointwise_epilogue(static_cast<const __nv_bfloat16*>(a), add, M,
                                                  N, dev->sms, s))) != GBF_OK)
    return st;
  // kernel 2: RMSNorm of the stored residual
  return cuda_status(launch_add_rmsnorm(static_cast<const __nv_bfloat16*>(out_resid), nullptr,
                                        static_cast<const __nv_bfloat16*>(weight),
                                        static_cast<__nv_bfloat16*>(out_norm), nullptr, M,
                                        static_cast<int>(N), eps, dev->sms, s));
}

size_t gbf_workspace_size(int op, int64_t M, int64_t N, int64_t K, int fused) {
  if (M < 0 || N < 0 || K < 0) return 0;
  if (op == GBF_OP_MLP) {
    const size_t h = align256(static_cast<size_t>(M * K) * 2);
    if (fused) return h;
    return 4 * h + align256(static_cast<size_t>(M * N) * 2);  // g, u (2h), h, D
  }
  if (fused) return 0;
  switch (op) {
    case GBF_OP_GEMM_EPILOGUE: return align256(static_cast<size_t>(M * N) * 2);
    case GBF_OP_SWIGLU: return 2 * align256(static_cast<size_t>(M * N) * 2);
    case GBF_OP_W4A16:
    case GBF_OP_W8A16_FP8:
    case GBF_OP_W4A16_NVFP4: return align256(static_cast<size_t>(K * N) * 2);
    default: return 0;
  }
}

namespace {
// MLP workspace sections (N = D, K = F): h first; the unfused chain adds
// g, u and the down GEMM's bf16 product.
size_t mlp_h_bytes(int64_t M, int64_t F) { return align256(static_cast<size_t>(M * F) * 2); }
}  // namespace

gbf_status_t gemm_epilogue_unfused(const void* A, const void* B, int b_layout, const void* C,
                                   const void* bias, const void* residual, void* out, int64_t M,
                                   int64_t N, int64_t K, float alpha, float beta, int act,
                                   void* workspace, size_t workspace_bytes, gbf_stream_t stream) {
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (b_layout != GBF_B_KN && b_layout != GBF_B_NK) return GBF_ERR_INVALID_ARG;
  if ((st = check_ptrs({A, B, out}, {C, bias, residual})) != GBF_OK) return st;
  const size_t need = gbf_workspace_size(GBF_OP_GEMM_EPILOGUE, M, N, K, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GBF_ERR_MISALIGNED;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const EpiParams ep = make_ep(C, bias, residual, out, alpha, beta, act);
  if (K == 0) return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev->sms, s));
  __nv_bfloat16* D = static_cast<__nv_bfloat16*>(workspace);
  st = run_gemm(A, B, nullptr, b_layout, false,
                make_ep(nullptr, nullptr, nullptr, D, 1.0f, 0.0f, GBF_ACT_IDENTITY), M, N, K,
                *dev, err, s);
  if (st != GBF_OK) return st;
  return cuda_status(launch_pointwise_epilogue(D, ep, M, N, dev->sms, s));
}

gbf_status_t swiglu_dual_gemm_unfused(const void* x, const void* w_gate, const void* w_up,
                                      int w_layout, void* h, int64_t M, int64_t N, int64_t K,
                                      float alpha, float beta, const void* C, int act,
                                      void* workspace, size_t workspace_bytes,
                                      gbf_stream_t stream) {
  gbf_status_t st = check_common(M, N, K, act);
  if (st != GBF_OK) return st;
  if (w_layout != GBF_B_KN && w_layout != GBF_B_NK) return GBF_ERR_INVALID_ARG;
  if ((st = check_ptrs({x, w_gate, w_up, h}, {C})) != GBF_OK) return st;
  const size_t need = gbf_workspace_size(GBF_OP_SWIGLU, M, N, K, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GBF_ERR_MISALIGNED;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  __nv_bfloat16* g = static_cast<__nv_bfloat16*>(workspace);
  __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) +
                                                      align256(static_cast<size_t>(M * N) * 2));
  const EpiParams plain_g = make_ep(nullptr, nullptr, nullptr, g, 1.0f, 0.0f, GBF_ACT_IDENTITY);
  const EpiParams plain_u = make_ep(nullptr, nullptr, nullptr, u, 1.0f, 0.0f, GBF_ACT_IDENTITY);
  if ((st = run_gemm(x, w_gate, nullptr, w_layout, false, plain_g, M, N, K, *dev, err, s)) !=
      GBF_OK)
    return st;
  if ((st = run_gemm(x, w_up, nullptr, w_layout, false, plain_u, M, N, K, *dev, err, s)) != GBF_OK)
    return st;
  return cuda_status(launch_swiglu_pointwise(
      g, u, make_ep(C, nullptr, nullptr, h, alpha, beta, act), M, N, dev->sms, s));
}

gbf_status_t w4a16_gemm_unfused(const void* A, const uint8_t* Wq, const void* scales,
                                int group_size, const void* C, const void* bias,
                                const void* residual, void* out, int64_t M, int64_t N, int64_t K,
                                float alpha, float beta, int act, void* workspace,
                                size_t workspace_bytes, gbf_stream_t stream) {
  gbf_status_t st = check_w4(M, N, K, group_size, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const size_t need = gbf_workspace_size(GBF_OP_W4A16, M, N, K, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GBF_ERR_MISALIGNED;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const EpiParams ep = make_ep(C, bias, residual, out, alpha, beta, act);
  if (K == 0) return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev->sms, s));
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(workspace);
  if ((st = cuda_status(launch_dequant_int4(Wq, static_cast<const __nv_bfloat16*>(scales),
                                            group_size, K, N, w, dev->sms, s))) != GBF_OK)
    return st;
  return run_gemm(A, w, nullptr, GBF_B_KN, false, ep, M, N, K, *dev, err, s);
}

gbf_status_t w8a16_fp8_gemm_unfused(const void* A, const uint8_t* Wq, const void* scales,
                                    int group_size, const void* C, const void* bias,
                                    const void* residual, void* out, int64_t M, int64_t N,
                                    int64_t K, float alpha, float beta, int act, void* workspace,
                                    size_t workspace_bytes, gbf_stream_t stream) {
  gbf_status_t st = check_w4(M, N, K, group_size, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const size_t need = gbf_workspace_size(GBF_OP_W8A16_FP8, M, N, K, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GBF_ERR_MISALIGNED;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const EpiParams ep = make_ep(C, bias, residual, out, alpha, beta, act);
  if (K == 0) return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev->sms, s));
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(workspace);
  if ((st = cuda_status(launch_dequant_fp8(Wq, static_cast<const __nv_bfloat16*>(scales),
                                           group_size, K, N, w, dev->sms, s))) != GBF_OK)
    return st;
  return run_gemm(A, w, nullptr, GBF_B_KN, false, ep, M, N, K, *dev, err, s);
}

gbf_status_t w4a16_nvfp4_gemm_unfused(const void* A, const uint8_t* Wq, const uint8_t* scales,
                                      const void* C, const void* bias, const void* residual,
                                      void* out, int64_t M, int64_t N, int64_t K, float alpha,
                                      float beta, int act, void* workspace,
                                      size_t workspace_bytes, gbf_stream_t stream) {
  gbf_status_t st = check_nvfp4(M, N, K, act);
  if (st != GBF_OK) return st;
  if ((st = check_ptrs({A, Wq, scales, out}, {C, bias, residual})) != GBF_OK) return st;
  const size_t need = gbf_workspace_size(GBF_OP_W4A16_NVFP4, M, N, K, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GBF_ERR_MISALIGNED;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || N == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const EpiParams ep = make_ep(C, bias, residual, out, alpha, beta, act);
  if (K == 0) return cuda_status(launch_pointwise_epilogue(nullptr, ep, M, N, dev->sms, s));
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(workspace);
  if ((st = cuda_status(launch_dequant_nvfp4(Wq, scales, K, N, w, dev->sms, s))) != GBF_OK)
    return st;
  return run_gemm(A, w, nullptr, GBF_B_KN, false, ep, M, N, K, *dev, err, s);
}

gbf_status_t mlp_swiglu_down(const void* x, const void* w_gate, const void* w_up,
                             const void* w_down, const void* residual, void* out, int64_t M,
                             int64_t D, int64_t F, void* workspace, size_t workspace_bytes,
                             gbf_stream_t stream) {
  gbf_status_t st = check_common(M, F, D, GBF_ACT_SILU);
  if (st != GBF_OK) return st;
  if ((st = check_common(M, D, F, GBF_ACT_IDENTITY)) != GBF_OK) return st;
  if ((st = check_ptrs({x, w_gate, w_up, w_down, out}, {residual, workspace})) != GBF_OK)
    return st;
  const size_t need = gbf_workspace_size(GBF_OP_MLP, M, D, F, 1);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  const DeviceInfo* dev;
  unsigned* err;
  if ((st = current_device(&dev, &err)) != GBF_OK) return st;
  if (M == 0 || D == 0) return GBF_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* h = workspace;
  if ((st = run_gemm(x, w_gate, w_up, GBF_B_NK, true,
                     make_ep(nullptr, nullptr, nullptr, h, 1.0f, 0.0f, GBF_ACT_SILU), M, F, D,
                     *dev, err, s)) != GBF_OK)
    return st;
  return run_gemm(h, w_down, nullptr, GBF_B_NK, false,
                  make_ep(nullptr, nullptr, residual, out, 1.0f, 0.0f, GBF_ACT_IDENTITY), M, D, F,
                  *dev, err, s);
}

gbf_status_t mlp_swiglu_down_unfused(const void* x, const void* w_gate, const void* w_up,
                                     const void* w_down, const void* residual, void* out,
                                     int64_t M, int64_t D, int64_t F, void* workspace,
                                     size_t workspace_bytes, gbf_stream_t stream) {
  gbf_status_t st = check_common(M, F, D, GBF_ACT_SILU);
  if (st != GBF_OK) return st;
  if ((st = check_common(M, D, F, GBF_ACT_IDENTITY)) != GBF_OK) return st;
  if ((st = check_ptrs({x, w_gate, w_up, w_down, out}, {residual, workspace})) != GBF_OK)
    return st;
  const size_t need = gbf_workspace_size(GBF_OP_MLP, M, D, F, 0);
  if (need && (!workspace || workspace_bytes < need)) return GBF_ERR_WORKSPACE;
  if (M == 0 || D == 0) return GBF_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t hb = mlp_h_bytes(M, F);
  // [g | u] (what swiglu_dual_gemm_unfused expects), then h, then the down GEMM's D
  uint8_t* gu = ws;
  uint8_t* h = ws + 2 * hb;
  uint8_t* d = ws + 3 * hb;
  if ((st = swiglu_dual_gemm_unfused(x, w_gate, w_up, GBF_B_NK, h, M, F, D, 1.0f, 0.0f, nullptr,
                                     GBF_ACT_SILU, gu, 2 * hb, stream)) != GBF_OK)
    return st;
  return gemm_epilogue_unfused(h, w_down, GBF_B_NK, nullptr, nullptr, residual, out, M, D, F,
                               1.0f, 0.0f, GBF_ACT_IDENTITY, d, need - 3 * hb, stream);
}

gbf_status_t gbf_check_device_error(gbf_stream_t stream) {
  const DeviceInfo* dev;
  unsigned* err;
  gbf_status_t st = current_device(&dev, &err);
  if (st != GBF_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GBF_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GBF_ERR_CUDA;
  if (word == 0) return GBF_OK;
  const unsigned zero = 0;
  if (cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return GBF_ERR_CUDA;
  return (word & 0xFFu) == GBF_ERR_TIMEOUT ? GBF_ERR_TIMEOUT : GBF_ERR_CUDA;
}

const char* gbf_status_string(gbf_status_t status) {
  switch (status) {
    case GBF_OK: return "ok";
    case GBF_ERR_INVALID_ARG: return "invalid argument";
    case GBF_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case GBF_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case GBF_ERR_WORKSPACE: return "workspace missing or too small";
    case GBF_ERR_CUDA: return "CUDA error";
    case GBF_ERR_TIMEOUT: return "kernel gave up on a bounded wait";
    case GBF_ERR_NO_DEVICE: return "no sm_103 device is current";
    default: return "unknown status";
  }
}

gbf_status_t gbf_set_wait_timeout_ns(uint64_t ns) {
  ns = std::max<uint64_t>(1000000ull, std::min<uint64_t>(ns, 60000000000ull));
  g_timeout_ns.store(ns);
  return GBF_OK;
}

gbf_status_t gbf_debug_inject_timeout(int on) {
  g_inject.store(on ? 1 : 0);
  return GBF_OK;
}

gbf_status_t gbf_debug_set_profile(void* counters, size_t bytes) {
  g_prof_bytes.store(counters ? bytes : 0);
  g_prof.store(static_cast<unsigned long long*>(counters));
  return GBF_OK;
}

gbf_status_t gbf_debug_force_splits(int splits) {
  if (splits < 0 || splits > kMaxSplits) return GBF_ERR_INVALID_ARG;
  g_force_splits.store(splits);
  return GBF_OK;
}

gbf_status_t gbf_debug_force_path(int path) {
  if (path != 0 && path != kPathPersistent && path != kPathPair && path != kPathPersistentSplit &&
      path != kPathPairOne && path != kPathPairSplit)
    return GBF_ERR_INVALID_ARG;
  g_force_path.store(path);
  return GBF_OK;
}

int gbf_kernel_path(int op, int64_t M, int64_t N, int64_t K, int b_layout, int* splits) {
  if (splits) *splits = 0;
  DeviceInfo dev;
  const DeviceInfo* d = nullptr;
  unsigned* err = nullptr;
  if (current_device(&d, &err) == GBF_OK) {
    dev = *d;
  } else {
    dev.sms = 152;  // a GB300 (the planner's answer for a machine without one)
    dev.pairs = 76;
    dev.quads = 36;
  }
  GemmPlan p;
  switch (op) {
    case GBF_OP_GEMM_EPILOGUE:
    case GBF_OP_SWIGLU:
      if (check_common(M, N, K, 0) != GBF_OK || (b_layout != GBF_B_KN && b_layout != GBF_B_NK))
        return -1;
      p = plan_gemm(M, N, K, op == GBF_OP_SWIGLU, b_layout == GBF_B_KN, dev);
      break;
    case GBF_OP_W4A16:
    case GBF_OP_W8A16_FP8:
      if (check_w4(M, N, K, 64, 0) != GBF_OK) return -1;
      p = plan_w4a16(M, N, K, dev);
      break;
    case GBF_OP_W4A16_NVFP4:
      if (check_nvfp4(M, N, K, 0) != GBF_OK) return -1;
      p = plan_w4a16(M, N, K, dev);
      break;
    default: return -1;
  }
  if (splits) *splits = p.splits;
  return p.path;
}

int gbf_version(void) { return 100; }

}  // extern "C"

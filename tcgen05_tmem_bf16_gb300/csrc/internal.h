// internal.h -- declarations shared by the library's translation units
// (kernel launchers and the C-ABI layer).  Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gbf {

// Pointwise ending of a product: act(alpha*acc + beta*C + bias) + residual.
struct EpiParams {
  const __nv_bfloat16* C;         // [M][N] or null
  const __nv_bfloat16* bias;      // [N] or null
  const __nv_bfloat16* residual;  // [M][N] or null (may alias out)
  __nv_bfloat16* out;             // [M][N]
  float alpha;
  float beta;
  int act;
};

// Per-launch control: the device error word, the wait limit and the
// test-only timeout injection.
struct KernelCtl {
  unsigned* err;
  unsigned long long timeout_ns;
  int inject;
  unsigned long long* prof;  // per-CTA wait-time counters (kProfSlots each) or null
};
constexpr int kProfSlots = 32;  // [2*site] cycles waited, [2*site+1] waits; [31] CTA cycles

// Kernel families (gbf_kernel_path codes).
enum Path {
  kPathNone = 0,
  kPathPersistent = 1,
  kPathSwap = 2,
  kPathW4 = 3,
  kPathPair = 4,
  kPathPersistentSplit = 5,  // the one-SM persistent kernel, K split over a CTA pair per tile
  kPathPairOne = 6,          // the CTA-pair kernel with one MMA stream (units of one M-tile)
  kPathPairSplit = 7,        // the one-stream CTA-pair kernel, K split over two pairs per tile
};

struct GemmPlan {
  int path = kPathNone;
  int mpad = 0;      // swapped kernels: MMA N (padded rows of A per tile)
  int splits = 1;    // swapped kernels: cluster split-K size
  int m_tiles = 0;
  int n_tiles = 0;
  int num_kb = 0;    // 64-wide K blocks
  int grid = 0;      // persistent kernels: CTAs
  int bn = 256;      // pair kernel: tile width (MMA N)
  int streams = 2;   // pair kernel: M-tiles (MMA streams) per unit of work
  bool kpar = false; // one-stream pair kernel: two MMA streams over alternate K blocks
};

struct DeviceInfo {
  int sms = 0;
  int pairs = 0;  // CTA pairs (clusters of two 1-SM CTAs) that fit at once
  int quads = 0;  // clusters of four 1-SM CTAs (two pairs) that fit at once
  int cc_major = 0;
  int cc_minor = 0;
};

// ---- argument checks (api.cu) -------------------------------------------------
// The status gemm_epilogue / gemm_epilogue_unfused return for these arguments
// before any workspace or device check (a GBF_* code; 0 = acceptable).
int check_gemm_call(const void* A, const void* B, int b_layout, const void* C, const void* bias,
                    const void* residual, const void* out, int64_t M, int64_t N, int64_t K,
                    int act);

// ---- planning (api.cu) -------------------------------------------------------
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, bool dual, bool kn, const DeviceInfo& dev);
GemmPlan plan_w4a16(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);

// ---- launchers ---------------------------------------------------------------
// Dense bf16 GEMM with fused ending (gemm_tc.cu).  tmA: activations [M][K];
// tmW / tmW2: weights (tmW2 = up weights of the dual GEMM); tmO: the output
// [M][N] in boxes of 32 x 32 with the 64-byte swizzle (used by the
// persistent kernel's TMA stores; the swapped kernel writes directly).
cudaError_t launch_gemm(const GemmPlan& plan, bool w_kn, bool dual, const CUtensorMap& tmA,
                        const CUtensorMap& tmW, const CUtensorMap& tmW2, const CUtensorMap& tmO,
                        const EpiParams& ep, int M, int N, int K, const KernelCtl& ctl,
                        cudaStream_t stream);

// The same on CTA pairs with tcgen05.mma.cta_group::2 (gemm_pair.cu).  tmO:
// the output [M][N] bf16 in boxes of 32 x 32 with the 64-byte swizzle (the
// epilogue writes it with TMA stores).
cudaError_t launch_gemm_pair(const GemmPlan& plan, bool w_kn, bool dual, const CUtensorMap& tmA,
                             const CUtensorMap& tmW, const CUtensorMap& tmW2,
                             const CUtensorMap& tmO, const EpiParams& ep, int M, int N, int K,
                             const KernelCtl& ctl, cudaStream_t stream);
int max_active_pairs();
int max_active_quads();

// Weight-only quantised GEMM (wq_gemm.cu).  tmA: activations; tmQ: the
// weight codes (int4, nvfp4: [K][N/2] bytes; fp8: [K][N]); tmS: scales
// (int4, fp8: bf16 [K/G][N]; nvfp4: E4M3 bytes [K/16][N]).
enum WqFmt { kWqInt4 = 0, kWqFp8 = 1, kWqNvfp4 = 2 };
cudaError_t launch_wq_gemm(int fmt, const GemmPlan& plan, const CUtensorMap& tmA,
                           const CUtensorMap& tmQ, const CUtensorMap& tmS, const EpiParams& ep,
                           int M, int N, int K, int group, const KernelCtl& ctl,
                           cudaStream_t stream);

// Pointwise kernels of the unfused compositions (pointwise.cu).  D == null
// means a zero product (used for K == 0).
cudaError_t launch_pointwise_epilogue(const __nv_bfloat16* D, const EpiParams& ep, int64_t M,
                                      int64_t N, int sms, cudaStream_t stream);
cudaError_t launch_swiglu_pointwise(const __nv_bfloat16* g, const __nv_bfloat16* u,
                                    const EpiParams& ep, int64_t M, int64_t N, int sms,
                                    cudaStream_t stream);
cudaError_t launch_dequant_int4(const uint8_t* Wq, const __nv_bfloat16* scales, int group,
                                int64_t K, int64_t N, __nv_bfloat16* w, int sms,
                                cudaStream_t stream);
// FP8 (bf16 group scales) and NVFP4 (E4M3 block scales) weights -> bf16 [K][N].
cudaError_t launch_dequant_fp8(const uint8_t* Wq, const __nv_bfloat16* scales, int group,
                               int64_t K, int64_t N, __nv_bfloat16* w, int sms,
                               cudaStream_t stream);
cudaError_t launch_dequant_nvfp4(const uint8_t* Wq, const uint8_t* scales, int64_t K, int64_t N,
                                 __nv_bfloat16* w, int sms, cudaStream_t stream);

// Fused residual add + RMSNorm (rmsnorm.cu).  x == null: no add (plain
// RMSNorm of a); resid == null: the residual is not written.  N <= 16384.
cudaError_t launch_add_rmsnorm(const __nv_bfloat16* a, const __nv_bfloat16* x,
                               const __nv_bfloat16* w, __nv_bfloat16* norm,
                               __nv_bfloat16* resid, int64_t M, int N, float eps, int sms,
                               cudaStream_t stream);
constexpr int kRmsMaxN = 16384;

// Tile geometry shared by the planner and the kernels.
constexpr int kBM = 128;        // MMA M: rows of TMEM / output tile height
constexpr int kBK = 64;         // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kPersistBN = 256; // persistent kernel: MMA N
constexpr int kSwapBN = 128;    // swapped kernel: output columns per tile (= MMA M)
constexpr int kSwapDualMaxM = 32;  // gate/up GEMM on the swapped kernel up to this M
constexpr int kW4BN = 512;      // W4A16 kernel: output columns per tile
constexpr int kMaxSplits = 8;   // portable cluster size limit

}  // namespace gbf

// gemm_tc.cu -- tcgen05/TMEM bf16 GEMM with the pointwise ending fused into
// the epilogue, for sm_103a.
//
// The ending act(alpha*acc + beta*C + bias) + residual is applied to each
// accumulator tile after it leaves tensor memory and before its one write
// to HBM ("Fusion and Epilogues", epilogue-fusion bullet; "Kernel fusion"
// guide, Concept).  The gate/up variant computes both products from the same
// x tile in one MMA and applies act(gate)*up in the epilogue ("Fusion
// Thinking", Pattern 2, level 2).
//
// Two kernels:
//  * gemm_persistent_kernel -- mid-size M (the planner picks it over the
//    CTA-pair kernel of gemm_pair.cu when it fills the SMs better).  One CTA
//    per SM walks output tiles
//    of 128 x 256 (dual: 128 x 128 from a 256-wide stacked [gate; up] B
//    tile).  Warp 0 issues TMA loads into a 4-stage shared-memory ring, warp 1
//    issues tcgen05.mma into one of two 256-column TMEM accumulators, warps
//    4-7 drain the other accumulator through the epilogue, so the ending of
//    tile t overlaps the main loop of tile t+1.
//  * gemm_swap_kernel -- small M (<= 128).  Computes out^T = W~^T * A^T so
//    that the weight tile fills the 128-row MMA and the few rows of A become
//    the MMA's N (16..128).  The K range is split across the CTAs of a thread
//    block cluster; the output rows are shared out among the ranks, each
//    rank receives the other ranks' partial sums of its rows in its shared
//    memory (bulk copies; for M = 128 it loads them through distributed
//    shared memory), sums them in rank order and applies the ending.  No
//    global scratch memory is used.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gbf {

constexpr int kUK = 16;  // K per tcgen05.mma, kind::f16

// ============================================================ shared pieces

// ============================================================ persistent kernel

constexpr int kPStages = 4;
constexpr int kPABytes = kBM * kBK * 2;             // 16 KB
constexpr int kPBBytes = kPersistBN * kBK * 2;      // 32 KB
constexpr int kPStageBytes = kPABytes + kPBBytes;   // 48 KB
constexpr int kPThreads = 384;  // warps 0-3 roles, warps 4-11 epilogue (two warpgroups)
// ring | barriers (1 KB) | output staging: 8 epilogue warps x 2 buffers of 2 KB
constexpr int kPBarBytes = 1024;
constexpr int kPSmem = 1024 + kPStages * kPStageBytes + kPBarBytes + 8 * 2 * kStageChunkBytes;
static_assert(kPSmem <= 227 * 1024, "shared memory per CTA");

struct PersistArgs {
  int M, N, K;
  int m_tiles, n_tiles, num_kb;
  EpiParams ep;
  KernelCtl ctl;
};

// Split-K form (SPLIT): a cluster of two CTAs computes one tile, each over
// half of the K range; each then parks the partial sums of the other CTA's
// half of the columns in its (now idle) stage memory as [column][row] fp32
// (64 KB), sends them to that CTA with bulk copies, and applies the ending
// to its own 128 columns as rank 0's partial + rank 1's partial.
constexpr int kPSplitHalf = kPersistBN / 2;                     // columns each rank finishes
constexpr int kPSplitBytes = kPSplitHalf * kBM * 4;             // 64 KB of fp32 partials
static_assert(2 * kPSplitBytes <= kPStages * kPStageBytes, "partials fit in the ring");

template <bool W_KN, bool DUAL, bool SPLIT>
__global__ void __launch_bounds__(kPThreads, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmW2,
                           const __grid_constant__ CUtensorMap tmO, const PersistArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPStages * kPStageBytes);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* recvb = done + 1;  // split-K: the peer's partial sums have landed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recvb + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  uint8_t* staging = smem + kPStages * kPStageBytes + kPBarBytes;  // 1024-aligned
  static_assert(!(SPLIT && DUAL), "split-K form for the single product only");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // split-K: rank r of the cluster takes k blocks [kb0, kb1) of its cluster's tile
  const uint32_t rank = SPLIT ? (cluster_ctarank() & 1u) : 0u;
  const int tile0 = SPLIT ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = SPLIT ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int kb0 = SPLIT ? static_cast<int>((static_cast<int64_t>(rank) * a.num_kb) / 2) : 0;
  const int kb1 =
      SPLIT ? static_cast<int>((static_cast<int64_t>(rank + 1) * a.num_kb) / 2) : a.num_kb;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);  // one arrive per epilogue warp
    }
    mbar_init(done, 1);
    if (SPLIT) {
      mbar_init(recvb, 1);
      mbar_arrive_expect_tx(recvb, kPSplitBytes);  // the peer's 128 x 128 partials
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    if (DUAL) tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (SPLIT) cluster_sync_all();  // both CTAs' barriers exist before any copy between them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const WaitCtl ctl{a.ctl.err, a.ctl.timeout_ns, abort_flag, prof_slots(a.ctl.prof)};
  const long long t_start = clock64();
  const int num_tiles = a.m_tiles * a.n_tiles;
  const int out_bn = DUAL ? 128 : 256;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t fills[kPStages];
#pragma unroll
      for (int i = 0; i < kPStages; ++i) fills[i] = 0;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = tile0; t < num_tiles && ok; t += tile_step) {
        int mb, nb;
        tile_coords(t, a.m_tiles, a.n_tiles, mb, nb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(&empty[s], ph ^ 1, ctl, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + s * kPStageBytes;
          uint8_t* sb = sa + kPABytes;
          mbar_arrive_expect_tx(&full[s], kPStageBytes);
          tma_load_2d(sa, &tmA, &full[s], kb * kBK, mb * kBM);
          if constexpr (W_KN) {
            // B[K][N]: four 64-column blocks of 64 k-rows (MN-major operand).
            if constexpr (DUAL) {
              for (int j = 0; j < 2; ++j) {
                tma_load_2d(sb + j * 8192, &tmW, &full[s], nb * 128 + 64 * j, kb * kBK);
                tma_load_2d(sb + (2 + j) * 8192, &tmW2, &full[s], nb * 128 + 64 * j, kb * kBK);
              }
            } else {
              for (int j = 0; j < 4; ++j)
                tma_load_2d(sb + j * 8192, &tmW, &full[s], nb * 256 + 64 * j, kb * kBK);
            }
          } else {
            // W[N][K]: rows of 64 k (K-major operand); dual stacks gate over up.
            if constexpr (DUAL) {
              tma_load_2d(sb, &tmW, &full[s], kb * kBK, nb * 128);
              tma_load_2d(sb + 128 * 128, &tmW2, &full[s], kb * kBK, nb * 128);
            } else {
              tma_load_2d(sb, &tmW, &full[s], kb * kBK, nb * 256);
            }
          }
          fills[s]++;
          if (++s == kPStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int i = 0; i < kPStages; ++i)
        if (fills[i]) wait_bar(&full[i], (fills[i] - 1) & 1, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kPersistBN, false, W_KN);
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int t = tile0; t < num_tiles && ok; t += tile_step, ++local) {
        const int buf = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!wait_bar(&tempty[buf], aph ^ 1, ctl, kSiteMmaAccEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * 256;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bar(&full[s], ph, ctl, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(stages + s * kPStageBytes);
          const uint32_t b0 = a0 + kPABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = W_KN ? sdesc_sw128(b0 + k * 2048, 8192, 1024)
                                     : sdesc_sw128(b0 + k * 32, 16, 1024);
            mma_ss(d, ad, bd, idesc, (kb > kb0 || k != 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          if (++s == kPStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if (!(a.ctl.inject && local == 0)) mma_commit(&tfull[buf]);
      }
      mma_commit(done);
      wait_bar(done, 0, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (!SPLIT && warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // Warps 4-7 and 8-11 read the same TMEM lanes (warp % 4 selects the lane
    // quarter); the first warpgroup takes the left half of the tile's
    // columns, the second the right half.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const uint64_t pol = l2_evict_first_policy();
    constexpr int kChunks = (DUAL ? 128 : 256) / 32;
    constexpr int kMine = kChunks / 2;
    uint8_t* my_staging = staging + (warp - 4) * 2 * kStageChunkBytes;
    int flip = 0;
    int local = 0;
    for (int t = tile0; t < num_tiles; t += tile_step, ++local) {
      int mb, nb;
      tile_coords(t, a.m_tiles, a.n_tiles, mb, nb);
      const int buf = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      const int64_t row = static_cast<int64_t>(mb) * kBM + q * 32 + lane;
      RowLoads L;
      epi_row_prefetch(L, row, nb * out_bn + half * kMine * 32, a.M, a.N, a.ep, pol);
      if (!wait_bar(&tfull[buf], aph, ctl, kSiteEpiAccFull)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * 256 + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < kMine; ++cc) {
        const int c = half * kMine + cc;
        const int col0 = nb * out_bn + c * 32;
        uint32_t acc[32], up[32];
        tmem_ld32(tb + c * 32, acc);
        if constexpr (DUAL) tmem_ld32(tb + 128 + c * 32, up);
        tmem_wait_ld();
        if (cc == kMine - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        const RowLoads cur = L;
        if (cc + 1 < kMine) epi_row_prefetch(L, row, col0 + 32, a.M, a.N, a.ep, pol);
        uint32_t w[16];
        switch (a.ep.act) {
          case kActRelu: epi_row32_pack<kActRelu, DUAL>(acc, up, cur, a.ep, w); break;
          case kActSilu: epi_row32_pack<kActSilu, DUAL>(acc, up, cur, a.ep, w); break;
          case kActGeluTanh: epi_row32_pack<kActGeluTanh, DUAL>(acc, up, cur, a.ep, w); break;
          default: epi_row32_pack<kActIdentity, DUAL>(acc, up, cur, a.ep, w); break;
        }
        store_chunk32(my_staging, flip, w, &tmO, row - lane, col0, a.M, a.N, pol);
      }
    }
    // every staged chunk written to global memory before the CTA may exit
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  if constexpr (SPLIT) {
    // ------------------------------------------------------------ split-K exchange + ending
    // (one tile per cluster: the launch has two CTAs per tile)
    const bool epi = warp >= 4;
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;      // warpgroup: chunks 2*half, 2*half + 1 of a half-tile
    const int rl = q * 32 + lane;          // row within the tile = TMEM lane
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);  // accumulator 0
    float* park = reinterpret_cast<float*>(stages);                 // [column][row], 64 KB
    float* recv = reinterpret_cast<float*>(stages + kPSplitBytes);  // the peer's, same layout
    const int t = tile0;
    int mb = 0, nb = 0;
    if (t < num_tiles) tile_coords(t, a.m_tiles, a.n_tiles, mb, nb);
    const uint64_t pol = l2_evict_first_policy();
    const int64_t row = static_cast<int64_t>(mb) * kBM + rl;
    const int mine = static_cast<int>(rank) * kPSplitHalf;       // first column this rank finishes
    const int theirs = kPSplitHalf - mine;                       // the peer's first column
    if (epi) {
      wait_bar(&tfull[0], 0, ctl, kSiteEpiAccFull);
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        uint32_t v[32];
        tmem_ld32(tb + theirs + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) park[(c * 32 + j) * kBM + rl] = __uint_as_float(v[j]);
      }
      fence_proxy_async_smem();  // the bulk copies read what these threads wrote
    }
    cluster_sync_all();  // both ranks parked
    if (threadIdx.x == 128) {
      const uint32_t peer = rank ^ 1u;
      constexpr int kPiece = kPSplitBytes / 4;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        bulk_copy_to_peer(mapa_shared(smem_u32(stages + kPSplitBytes + i * kPiece), peer),
                          smem_u32(stages + i * kPiece), kPiece,
                          mapa_shared(smem_u32(recvb), peer));
    }
    if (epi) {
      uint8_t* my_staging = staging + (warp - 4) * 2 * kStageChunkBytes;
      int flip = 0;
      // not cut short by the abort flag: the peer sends whatever its state
      wait_bar(recvb, 0, ctl, kSiteEpiAccFull, /*honor_abort=*/false);
      RowLoads L;
      epi_row_prefetch(L, row, nb * 256 + mine + 2 * half * 32, a.M, a.N, a.ep, pol);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        const int col0 = nb * 256 + mine + c * 32;
        uint32_t own[32], sum[32];
        tmem_ld32(tb + mine + c * 32, own);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float o = __uint_as_float(own[j]);
          const float p = recv[(c * 32 + j) * kBM + rl];
          // rank 0's partial first, in both ranks
          sum[j] = __float_as_uint(rank == 0 ? o + p : p + o);
        }
        const RowLoads cur = L;
        if (cc == 0) epi_row_prefetch(L, row, col0 + 32, a.M, a.N, a.ep, pol);
        uint32_t w[16];
        switch (a.ep.act) {
          case kActRelu: epi_row32_pack<kActRelu, false>(sum, sum, cur, a.ep, w); break;
          case kActSilu: epi_row32_pack<kActSilu, false>(sum, sum, cur, a.ep, w); break;
          case kActGeluTanh: epi_row32_pack<kActGeluTanh, false>(sum, sum, cur, a.ep, w); break;
          default: epi_row32_pack<kActIdentity, false>(sum, sum, cur, a.ep, w); break;
        }
        if (t < num_tiles) store_chunk32(my_staging, flip, w, &tmO, row - lane, col0, a.M, a.N, pol);
      }
      if (lane == 0) bulk_wait<0>();
      __syncwarp();
    }
    // no rank leaves while copies into or out of its shared memory may be in flight
    cluster_sync_all();
  }

  if (ctl.prof && threadIdx.x == 0) atomicAdd(&ctl.prof[31], static_cast<unsigned long long>(clock64() - t_start));
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ============================================================ swapped small-M kernel

// Sum of the NACC accumulators (spaced MPAD columns apart) for 16 columns of
// this thread's lane, accumulator 0 first.
template <int NACC, int MPAD>
__device__ __forceinline__ void acc_sum16(uint32_t taddr, float (&out)[16]) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
#pragma unroll
  for (int a = 1; a < NACC; ++a) {
    tmem_ld16(taddr + a * MPAD, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] += __uint_as_float(r[j]);
  }
}

constexpr int kSwapIssuers = 2;  // MMA issuing threads of the swapped kernel
// Weight k blocks prefetched into L2 before the wait for the previous kernel
// (same box: M = 1 / 16 / 128 sweeps 24.2 / 24.4 / 34.6 -> 23.7 / 24.0 /
// 33.9 us with 4; 8 and 16 gained less or lost).
constexpr int kSwapL2Prefetch = 4;

template <int MPAD, bool DUAL = false>
struct SwapCfg {
  // weight tile: 128 rows x 64 k (16 KB); the gate/up GEMM stages the gate
  // and the up tile of the same 128 output columns (32 KB)
  static constexpr int kWTile = kSwapBN * kBK * 2;
  static constexpr int kWBytes = (DUAL ? 2 : 1) * kWTile;
  static constexpr int kXBytes = MPAD * kBK * 2;             // activation tile
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kStages = DUAL ? 3 : (MPAD <= 32 ? 5 : (MPAD <= 64 ? 4 : 3));
  // Consecutive 16-deep K steps go to kAcc accumulators in turn: with a
  // narrow MMA (N = MPAD) the time per MMA is set by the accumulator's
  // read-after-write chain, not by its arithmetic, so independent chains
  // multiply the MMA rate; the epilogue sums them in a fixed order.  The
  // gate/up GEMM keeps kAcc gate and kAcc up accumulators.
  static constexpr int kAcc = MPAD <= 32 ? 4 : 2;
  static constexpr int kProducts = DUAL ? 2 : 1;
  static constexpr int kCols = kProducts * kAcc * MPAD;
  static constexpr uint32_t kTmemCols = kCols <= 64 ? 64 : (kCols <= 128 ? 128 : 256);
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
  // Split-K exchange by pushing (see the kernel's epilogue): the partial, as
  // kQuads 4-row groups of every product, plus the largest receive area
  // (S * ceil(kQuads / S) < kQuads + kMaxSplits groups) must fit in the
  // stage memory; otherwise the ranks pull through distributed shared memory.
  static constexpr int kQuads = MPAD / 4;
  static constexpr int kQuadBytes = kProducts * 128 * 16;
  static constexpr bool kPush =
      (2 * kQuads + kMaxSplits) * kQuadBytes <= kStages * kStageBytes;
  static_assert(kCols <= 256, "TMEM budget of two CTAs per SM");
  static_assert(!DUAL || kSmem <= 113 * 1024, "two CTAs per SM");
  static_assert(kStages * kStageBytes >= kProducts * 128 * MPAD * 4, "reduction buffer must fit");
};

struct SwapArgs {
  int M, N, K;
  int num_kb;
  int splits;
  EpiParams ep;
  KernelCtl ctl;
};

// GLU ending of one output column for R consecutive rows (swapped gate/up
// GEMM): h = act(alpha*g) * (alpha*u) + beta*C.
template <int ACT, int R>
__device__ __forceinline__ void epi_col_glu(const float (&g)[R], const float (&u)[R],
                                            const ColLoads<R>& L, int64_t m0, int n, int M,
                                            int N, const EpiParams& e, uint64_t pol) {
  if (n >= N) return;
  const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int64_t m = m0 + j;
    if (m < M)
      st_stream_u16(e.out + m * N + n,
                    f_to_bf16bits(fmaf(beta, L.c[j],
                                       act_apply<ACT>(e.alpha * g[j]) * (e.alpha * u[j]))),
                    pol);
  }
}

template <int MPAD, bool W_KN, bool DUAL>
__global__ void __launch_bounds__(256, 2)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmW2, const SwapArgs a) {
  using Cfg = SwapCfg<MPAD, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* dfull = empty + Cfg::kStages;
  uint64_t* done = dfull + 1;
  uint64_t* recvb = done + 1;  // split-K partials pushed here by the other ranks
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recvb + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.splits;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int nb = blockIdx.y;
  const int mb = blockIdx.z;
  const int kb0 = static_cast<int>((static_cast<int64_t>(rank) * a.num_kb) / S);
  const int kb1 = static_cast<int>((static_cast<int64_t>(rank + 1) * a.num_kb) / S);

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kSwapIssuers);
    }
    mbar_init(dfull, kSwapIssuers);
    mbar_init(done, kSwapIssuers);
    if (Cfg::kPush && S > 1) {
      // expects the other S - 1 ranks' copies of this rank's 4-row groups
      const int r = static_cast<int>(rank);
      const int nq = ((r + 1) * Cfg::kQuads) / S - (r * Cfg::kQuads) / S;
      mbar_init(recvb, 1);
      mbar_arrive_expect_tx(recvb, static_cast<uint32_t>((S - 1) * nq * Cfg::kQuadBytes));
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    if constexpr (DUAL) tma_prefetch_desc(&tmW2);
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const WaitCtl ctl{a.ctl.err, a.ctl.timeout_ns, abort_flag, prof_slots(a.ctl.prof)};
  const long long t_start = clock64();

  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t fills[Cfg::kStages];
#pragma unroll
      for (int i = 0; i < Cfg::kStages; ++i) fills[i] = 0;
      // weight tiles of k block kb into stage s (read-only inputs, read once:
      // evict-first, so that the ending's operands pulled into L2 stay)
      const uint64_t wpol = policy_evict_first();
      auto load_w = [&](int s, int kb) {
        uint8_t* sw = stages + s * Cfg::kStageBytes;
#pragma unroll
        for (int w = 0; w < Cfg::kProducts; ++w) {
          const CUtensorMap* map = w == 0 ? &tmW : &tmW2;
          uint8_t* dst = sw + w * Cfg::kWTile;
          if constexpr (W_KN) {
            tma_load_2d_hint(dst, map, &full[s], nb * kSwapBN, kb * kBK, wpol);
            tma_load_2d_hint(dst + 8192, map, &full[s], nb * kSwapBN + 64, kb * kBK, wpol);
          } else {
            tma_load_2d_hint(dst, map, &full[s], kb * kBK, nb * kSwapBN, wpol);
          }
        }
      };
      auto load_x = [&](int s, int kb) {
        tma_load_2d(stages + s * Cfg::kStageBytes + Cfg::kWBytes, &tmA, &full[s], kb * kBK,
                    mb * MPAD);
      };
      // Nothing is read before the previous kernel in the stream has
      // completed: any input, weights included, may be its output.  While it
      // finishes, the first stages' weight tiles are only prefetched into L2
      // (which a later write would update), so the ring fills from L2 once
      // the wait returns.
      for (int kb = kb0; kb < kb1 && kb < kb0 + kSwapL2Prefetch; ++kb) {
#pragma unroll
        for (int w = 0; w < Cfg::kProducts; ++w) {
          const CUtensorMap* map = w == 0 ? &tmW : &tmW2;
          if constexpr (W_KN) {
            tma_prefetch_l2_2d(map, nb * kSwapBN, kb * kBK);
            tma_prefetch_l2_2d(map, nb * kSwapBN + 64, kb * kBK);
          } else {
            tma_prefetch_l2_2d(map, kb * kBK, nb * kSwapBN);
          }
        }
      }
      griddep_wait();
      int s = 0;
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&empty[s], ph ^ 1, ctl, kSiteProducerEmpty)) break;
        mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        load_w(s, kb);
        load_x(s, kb);
        fills[s]++;
        if (++s == Cfg::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      for (int i = 0; i < Cfg::kStages; ++i)
        if (fills[i]) wait_bar(&full[i], (fills[i] - 1) & 1, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // Two MMA issuers: warp 1 issues K steps 0-1 and warp 3 K steps 2-3 of
    // every stage (the MMAs of one thread complete one after another, those
    // of two threads overlap).  K step k goes to accumulator k*kAcc/4, so each
    // accumulator has one writer.
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, MPAD, W_KN, false);
      constexpr int kSteps = kBK / kUK;              // 4
      constexpr int kPer = kSteps / kSwapIssuers;    // K steps per issuer and stage
      const int k0 = warp == 1 ? 0 : kPer;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&full[s], ph, ctl, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w0 = smem_u32(stages + s * Cfg::kStageBytes);
        const uint32_t x0 = w0 + Cfg::kWBytes;
#pragma unroll
        for (int k = k0; k < k0 + kPer; ++k) {
          const uint64_t ad = W_KN ? sdesc_sw128(w0 + k * 2048, 8192, 1024)
                                   : sdesc_sw128(w0 + k * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(x0 + k * 32, 16, 1024);
          const int acc = k * Cfg::kAcc / kSteps;
          const uint32_t accum = (kb > kb0 || (k % (kSteps / Cfg::kAcc)) != 0) ? 1u : 0u;
          mma_ss(tmem_base + acc * MPAD, ad, bd, idesc, accum);
          if constexpr (DUAL) {
            const uint32_t w1 = w0 + Cfg::kWTile;
            const uint64_t ad2 = W_KN ? sdesc_sw128(w1 + k * 2048, 8192, 1024)
                                      : sdesc_sw128(w1 + k * 32, 16, 1024);
            mma_ss(tmem_base + (Cfg::kAcc + acc) * MPAD, ad2, bd, idesc, accum);
          }
        }
        mma_commit(&empty[s]);
        if (++s == Cfg::kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (ok && !a.ctl.inject) mma_commit(dfull);
      mma_commit(done);
      wait_bar(done, 0, ctl, kSiteDrain, false);
    }
    __syncwarp();
  }

  // ---- epilogue warps: partial sums, cluster reduction, ending
  // With split-K every rank parks its fp32 partial in its own shared memory.
  // Push exchange (when it fits): the output rows are shared out among the
  // ranks as 4-row groups, each rank copies every other rank's groups to
  // that rank with one bulk copy, and each rank sums its own groups over
  // ranks 0..S-1 in that order (deterministic) from local shared memory.
  // Otherwise the 16-row chunks go to the ranks round-robin (chunk c to rank
  // c % S) and all eight warps of each rank pull the other partials of its
  // chunks through distributed shared memory, again summing in rank order.
  const bool epi = warp >= 4;
  const int q = warp & 3;
  const int tid = threadIdx.x - 128;  // 0..127 for the epilogue warps = TMEM lane
  const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  float4* red = reinterpret_cast<float4*>(stages);
  constexpr int kChunks = MPAD / 16;
  bool have = false;
  const uint64_t pol = l2_evict_first_policy();
  const int n = nb * kSwapBN + tid;
  // The ending's C and residual rows [r0, r0 + nr) of this warp's 32
  // columns are pulled into L2 as soon as the previous kernel has finished,
  // so that their loads after the main loop hit L2 (one 64-byte segment per
  // row and operand; lane j takes rows j, j + 32, ...).
  auto l2_rows = [&](int r0, int nr) {
    const int n0 = nb * kSwapBN + q * 32;
    if (n0 >= a.N) return;
    for (int j = lane; j < nr; j += 32) {
      const int64_t m = static_cast<int64_t>(mb) * MPAD + r0 + j;
      if (m >= a.M) break;
      if (a.ep.C) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.ep.C + m * a.N + n0));
      if (a.ep.residual)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.ep.residual + m * a.N + n0));
    }
  };
  bool pushed = false;
  if constexpr (Cfg::kPush) {
    if (S > 1) {
      pushed = true;
      constexpr int kP = Cfg::kProducts;
      const int r = static_cast<int>(rank);
      const int qa = (r * Cfg::kQuads) / S;  // this rank's 4-row groups [qa, qa + nq)
      const int nq = ((r + 1) * Cfg::kQuads) / S - qa;
      uint8_t* recv = stages + Cfg::kQuads * Cfg::kQuadBytes;  // [sender][group][product][lane]
      ColLoads<4> L4;
      if (epi) griddep_wait();  // the ending reads C, bias, residual and writes out
      if (epi) l2_rows(4 * qa, 4 * nq);
      if (epi && nq > 0)
        col_prefetch<4>(L4, static_cast<int64_t>(mb) * MPAD + 4 * qa, n, a.M, a.N, a.ep, pol);
      if (epi) {
        have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
        tc_fence_after();
        // park: red[(group * kP + product) * 128 + lane] = rows 4 group .. +3
#pragma unroll 1
        for (int c = 0; c < kP * kChunks; ++c) {
          float v[16];
          acc_sum16<Cfg::kAcc, MPAD>(tb + (c / kChunks) * Cfg::kAcc * MPAD + (c % kChunks) * 16,
                                     v);
#pragma unroll
          for (int w = 0; w < 4; ++w)
            red[(((c % kChunks) * 4 + w) * kP + c / kChunks) * 128 + tid] =
                make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
        }
        fence_proxy_async_smem();  // the bulk copies read what these threads wrote
      }
      cluster_sync_all();  // every rank parked, every receive barrier armed
      if (threadIdx.x == 128) {
        for (int i = 1; i < S; ++i) {
          const int p = (r + i) % S;
          const int pa = (p * Cfg::kQuads) / S;
          const int pn = ((p + 1) * Cfg::kQuads) / S - pa;
          if (pn > 0)
            bulk_copy_to_peer(
                mapa_shared(smem_u32(recv + r * pn * Cfg::kQuadBytes), static_cast<uint32_t>(p)),
                smem_u32(stages + pa * Cfg::kQuadBytes), static_cast<uint32_t>(pn * Cfg::kQuadBytes),
                mapa_shared(smem_u32(recvb), static_cast<uint32_t>(p)));
        }
      }
      if (epi && nq > 0) {
        // Not cut short by the abort flag: every peer issues its copies after
        // the cluster barrier above whatever its state, so this wait ends
        // (bounded by the timeout) and the final barrier then follows them.
        wait_bar(recvb, 0, ctl, kSiteEpiAccFull, /*honor_abort=*/false);
        const float4* in = reinterpret_cast<const float4*>(recv);
#pragma unroll 1
        for (int g = qa; g < qa + nq; ++g) {
          const int i = g - qa;
          if (g != qa)
            col_prefetch<4>(L4, static_cast<int64_t>(mb) * MPAD + 4 * g, n, a.M, a.N, a.ep, pol);
          float v[kP][4];
#pragma unroll
          for (int pr = 0; pr < kP; ++pr) {
            float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int p = 0; p < S; ++p) {
              const float4 f = p == r ? red[(g * kP + pr) * 128 + tid]
                                      : in[((p * nq + i) * kP + pr) * 128 + tid];
              if (p == 0) {
                t = f;
              } else {
                t.x += f.x;
                t.y += f.y;
                t.z += f.z;
                t.w += f.w;
              }
            }
            v[pr][0] = t.x;
            v[pr][1] = t.y;
            v[pr][2] = t.z;
            v[pr][3] = t.w;
          }
          const int64_t m0 = static_cast<int64_t>(mb) * MPAD + 4 * g;
          if constexpr (DUAL) {
            switch (a.ep.act) {
              case kActRelu: epi_col_glu<kActRelu, 4>(v[0], v[kP - 1], L4, m0, n, a.M, a.N, a.ep, pol); break;
              case kActSilu: epi_col_glu<kActSilu, 4>(v[0], v[kP - 1], L4, m0, n, a.M, a.N, a.ep, pol); break;
              case kActGeluTanh:
                epi_col_glu<kActGeluTanh, 4>(v[0], v[kP - 1], L4, m0, n, a.M, a.N, a.ep, pol);
                break;
              default: epi_col_glu<kActIdentity, 4>(v[0], v[kP - 1], L4, m0, n, a.M, a.N, a.ep, pol); break;
            }
          } else {
            switch (a.ep.act) {
              case kActRelu: epi_col<kActRelu, 4>(v[0], L4, m0, n, a.M, a.N, a.ep, pol); break;
              case kActSilu: epi_col<kActSilu, 4>(v[0], L4, m0, n, a.M, a.N, a.ep, pol); break;
              case kActGeluTanh: epi_col<kActGeluTanh, 4>(v[0], L4, m0, n, a.M, a.N, a.ep, pol); break;
              default: epi_col<kActIdentity, 4>(v[0], L4, m0, n, a.M, a.N, a.ep, pol); break;
            }
          }
        }
      }
      // No rank leaves while copies from or into its shared memory may be in
      // flight: every copy has completed on its receiver's barrier, which the
      // receiver waited for before arriving.  The arrival is relaxed, so it
      // does not first wait for this thread's stores of the ending.
      cluster_sync_relaxed_arrive();
    }
  }
  if constexpr (!Cfg::kPush) {
    if (S > 1) {
      // Pull exchange (the single product at M > 64): 16-row chunks go to the
      // ranks round-robin (chunk c to rank c % S).  After the park and a
      // cluster barrier all eight warps of the rank reduce its chunks, two
      // threads per column (rows 16c .. 16c+7 and 16c+8 .. 16c+15), loading
      // the other ranks' partials through distributed shared memory and
      // summing in rank order 0..S-1.
      static_assert(!DUAL, "the gate/up GEMM always pushes");
      pushed = true;
      const int h = threadIdx.x >> 7;    // row half of each chunk
      const int col = threadIdx.x & 127;  // column of the tile
      const int ncol = nb * kSwapBN + col;
      const int r = static_cast<int>(rank);
      ColLoads<8> L8;
      griddep_wait();  // every thread: the ending reads C, bias, residual and writes out
      if (epi)
        for (int c = r; c < kChunks; c += S) l2_rows(16 * c, 16);
      if (r < kChunks)  // this rank's first chunk: operands early
        col_prefetch<8>(L8, static_cast<int64_t>(mb) * MPAD + r * 16 + 8 * h, ncol, a.M, a.N,
                        a.ep, pol);
      if (epi) {
        have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
        tc_fence_after();
        // park: red[(chunk * 4 + v) * 128 + lane] = rows 16 chunk + 4v .. +3
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          float v[16];
          acc_sum16<Cfg::kAcc, MPAD>(tb + c * 16, v);
#pragma unroll
          for (int w = 0; w < 4; ++w)
            red[(c * 4 + w) * 128 + tid] =
                make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
        }
      }
      // every rank parked (the other warps only wrote registers: their loads
      // of the first chunk's operands stay in flight across the barrier)
      if (epi) cluster_sync_all();
      else cluster_sync_relaxed_arrive();
#pragma unroll 1
      for (int c = r; c < kChunks; c += S) {
        if (c != r)
          col_prefetch<8>(L8, static_cast<int64_t>(mb) * MPAD + c * 16 + 8 * h, ncol, a.M, a.N,
                          a.ep, pol);
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.0f;
        for (int p = 0; p < S; ++p) {
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            float4* src = &red[(c * 4 + 2 * h + w) * 128 + col];
            const float4 f = p == r ? *src
                                    : ld_dsmem_f4(mapa_shared(smem_u32(src),
                                                              static_cast<uint32_t>(p)));
            v[4 * w] += f.x;
            v[4 * w + 1] += f.y;
            v[4 * w + 2] += f.z;
            v[4 * w + 3] += f.w;
          }
        }
        const int64_t m0 = static_cast<int64_t>(mb) * MPAD + c * 16 + 8 * h;
        switch (a.ep.act) {
          case kActRelu: epi_col<kActRelu, 8>(v, L8, m0, ncol, a.M, a.N, a.ep, pol); break;
          case kActSilu: epi_col<kActSilu, 8>(v, L8, m0, ncol, a.M, a.N, a.ep, pol); break;
          case kActGeluTanh: epi_col<kActGeluTanh, 8>(v, L8, m0, ncol, a.M, a.N, a.ep, pol); break;
          default: epi_col<kActIdentity, 8>(v, L8, m0, ncol, a.M, a.N, a.ep, pol); break;
        }
      }
      // No rank leaves while another may still read its shared memory: every
      // remote load's value has been used before its thread arrives.  The
      // arrival is relaxed, so it does not first wait for the ending's stores.
      cluster_sync_relaxed_arrive();
    }
  }
  if (!pushed) {  // S == 1: the accumulator straight from tensor memory
    ColLoads<16> L;
    if (epi) griddep_wait();  // the ending reads C, bias, residual and writes out
    if (epi) l2_rows(0, MPAD);
    if (epi)  // the first chunk's operands early
      col_prefetch<16>(L, static_cast<int64_t>(mb) * MPAD, n, a.M, a.N, a.ep, pol);
    if (epi) {
      have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        if (c != 0)
          col_prefetch<16>(L, static_cast<int64_t>(mb) * MPAD + c * 16, n, a.M, a.N, a.ep, pol);
        float v[Cfg::kProducts][16];
#pragma unroll
        for (int pr = 0; pr < Cfg::kProducts; ++pr) {
          float rr[16];
          acc_sum16<Cfg::kAcc, MPAD>(tb + pr * Cfg::kAcc * MPAD + c * 16, rr);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[pr][j] = have ? rr[j] : 0.0f;
        }
        const int64_t m0 = static_cast<int64_t>(mb) * MPAD + c * 16;
        if constexpr (DUAL) {
          switch (a.ep.act) {
            case kActRelu: epi_col_glu<kActRelu, 16>(v[0], v[1], L, m0, n, a.M, a.N, a.ep, pol); break;
            case kActSilu: epi_col_glu<kActSilu, 16>(v[0], v[1], L, m0, n, a.M, a.N, a.ep, pol); break;
            case kActGeluTanh:
              epi_col_glu<kActGeluTanh, 16>(v[0], v[1], L, m0, n, a.M, a.N, a.ep, pol);
              break;
            default: epi_col_glu<kActIdentity, 16>(v[0], v[1], L, m0, n, a.M, a.N, a.ep, pol); break;
          }
        } else {
          switch (a.ep.act) {
            case kActRelu: epi_col<kActRelu, 16>(v[0], L, m0, n, a.M, a.N, a.ep, pol); break;
            case kActSilu: epi_col<kActSilu, 16>(v[0], L, m0, n, a.M, a.N, a.ep, pol); break;
            case kActGeluTanh: epi_col<kActGeluTanh, 16>(v[0], L, m0, n, a.M, a.N, a.ep, pol); break;
            default: epi_col<kActIdentity, 16>(v[0], L, m0, n, a.M, a.N, a.ep, pol); break;
          }
        }
      }
    }
  }

  if (ctl.prof && threadIdx.x == 0) atomicAdd(&ctl.prof[31], static_cast<unsigned long long>(clock64() - t_start));
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ============================================================ host launchers

namespace {

// cudaFuncSetAttribute once per kernel instantiation and device.
template <typename K>
cudaError_t ensure_smem_attr(K kernel, int bytes, std::atomic<uint64_t>& mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <bool W_KN, bool DUAL>
cudaError_t run_persistent(const GemmPlan& p, const CUtensorMap& tmA, const CUtensorMap& tmW,
                           const CUtensorMap& tmW2, const CUtensorMap& tmO,
                           const PersistArgs& args, cudaStream_t stream) {
  static std::atomic<uint64_t> mask{0};
  auto kernel = gemm_persistent_kernel<W_KN, DUAL, false>;
  cudaError_t e = ensure_smem_attr(kernel, kPSmem, mask);
  if (e != cudaSuccess) return e;
  kernel<<<p.grid, kPThreads, kPSmem, stream>>>(tmA, tmW, tmW2, tmO, args);
  return cudaGetLastError();
}

// Split-K form: clusters of two CTAs, one cluster per tile.
template <bool W_KN>
cudaError_t run_persistent_split(const GemmPlan& p, const CUtensorMap& tmA,
                                 const CUtensorMap& tmW, const CUtensorMap& tmO,
                                 const PersistArgs& args, cudaStream_t stream) {
  static std::atomic<uint64_t> mask{0};
  auto kernel = gemm_persistent_kernel<W_KN, false, true>;
  cudaError_t e = ensure_smem_attr(kernel, kPSmem, mask);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid, 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmW, tmW, tmO, args);
}

template <int MPAD, bool W_KN, bool DUAL>
cudaError_t run_swap(const GemmPlan& p, const CUtensorMap& tmA, const CUtensorMap& tmW,
                     const CUtensorMap& tmW2, const SwapArgs& args, cudaStream_t stream) {
  static std::atomic<uint64_t> mask{0};
  auto kernel = gemm_swap_kernel<MPAD, W_KN, DUAL>;
  using Cfg = SwapCfg<MPAD, DUAL>;
  cudaError_t e = ensure_smem_attr(kernel, Cfg::kSmem, mask);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_tiles, p.m_tiles);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel in the stream finishes (it waits
  // with griddepcontrol.wait before touching anything that kernel writes)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmW, tmW2, args);
}

template <bool W_KN>
cudaError_t run_swap_mpad(const GemmPlan& p, bool dual, const CUtensorMap& tmA,
                          const CUtensorMap& tmW, const CUtensorMap& tmW2, const SwapArgs& args,
                          cudaStream_t stream) {
  if (dual) {
    switch (p.mpad) {
      case 16: return run_swap<16, W_KN, true>(p, tmA, tmW, tmW2, args, stream);
      case 32: return run_swap<32, W_KN, true>(p, tmA, tmW, tmW2, args, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.mpad) {
    case 16: return run_swap<16, W_KN, false>(p, tmA, tmW, tmW, args, stream);
    case 32: return run_swap<32, W_KN, false>(p, tmA, tmW, tmW, args, stream);
    case 64: return run_swap<64, W_KN, false>(p, tmA, tmW, tmW, args, stream);
    case 128: return run_swap<128, W_KN, false>(p, tmA, tmW, tmW, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(const GemmPlan& plan, bool w_kn, bool dual, const CUtensorMap& tmA,
                        const CUtensorMap& tmW, const CUtensorMap& tmW2, const CUtensorMap& tmO,
                        const EpiParams& ep, int M, int N, int K, const KernelCtl& ctl,
                        cudaStream_t stream) {
  if (plan.path == kPathPersistentSplit && !dual) {
    PersistArgs args{M, N, K, plan.m_tiles, plan.n_tiles, plan.num_kb, ep, ctl};
    return w_kn ? run_persistent_split<true>(plan, tmA, tmW, tmO, args, stream)
                : run_persistent_split<false>(plan, tmA, tmW, tmO, args, stream);
  }
  if (plan.path == kPathPersistent) {
    PersistArgs args{M, N, K, plan.m_tiles, plan.n_tiles, plan.num_kb, ep, ctl};
    if (w_kn)
      return dual ? run_persistent<true, true>(plan, tmA, tmW, tmW2, tmO, args, stream)
                  : run_persistent<true, false>(plan, tmA, tmW, tmW2, tmO, args, stream);
    return dual ? run_persistent<false, true>(plan, tmA, tmW, tmW2, tmO, args, stream)
                : run_persistent<false, false>(plan, tmA, tmW, tmW2, tmO, args, stream);
  }
  if (plan.path == kPathSwap) {
    SwapArgs args{M, N, K, plan.num_kb, plan.splits, ep, ctl};
    return w_kn ? run_swap_mpad<true>(plan, dual, tmA, tmW, tmW2, args, stream)
                : run_swap_mpad<false>(plan, dual, tmA, tmW, tmW2, args, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gbf

// gemm_pair.cu -- the persistent GEMM + fused ending on CTA pairs
// (tcgen05.mma.cta_group::2), for large M.
//
// Same ending and same results as gemm_persistent_kernel ("Fusion and
// Epilogues", epilogue-fusion bullet; "Fusion Thinking", Pattern 2 level 2 for
// the gate/up variant), computed on 256 x 256 tiles by two CTAs of a cluster
// running on two SMs:
//   * each CTA loads its own 128 rows of A and its own half (128 rows of the
//     N dimension) of the B tile into its shared memory -- for the gate/up
//     GEMM the even CTA loads the gate rows and the odd CTA the up rows, so
//     the accumulator's columns 0-127 are the gate product and 128-255 the
//     up product, exactly as in the single-CTA kernel;
//   * the even CTA issues one tcgen05.mma.cta_group::2 (M=256, N=256, K=16)
//     per step, which reads both CTAs' shared memory and writes rows 0-127 of
//     the accumulator into its own tensor memory and rows 128-255 into the
//     peer's;
//   * both CTAs' TMA loads complete on the even CTA's "full" barrier, and the
//     even CTA's commits arrive on both CTAs' "empty" and "accumulator full"
//     barriers (multicast); the odd CTA's epilogue warps report a drained
//     accumulator on the even CTA's barrier.
// Per SM this halves the shared-memory fill of the B operand compared with a
// 128 x 256 tile on one SM (32 KB instead of 48 KB per 64-deep K step for the
// same number of MMA cycles), which is what limits the single-CTA kernel.
//
// Two streams per pair.  The tcgen05.mma instructions of one issuing thread
// complete one after another, about 150 cycles each on this part whatever
// their N, which caps one stream of 256 x BN x 16 MMAs at 112-128 cycles of
// tensor work per 150.  So the pair runs two MMA streams, one per
// accumulator (TMEM columns 256i .. 256i+BN), issued by two threads of the
// even CTA.  They compute the two M-tiles of an M-tile pair with the same B
// tile: each ring stage holds both A tiles and the shared B tile, so a k
// step moves 2 x 16 KB of A and one B half per CTA for two tiles' MMAs
// (23 KB per tile instead of 30-32 KB).  The two epilogue warpgroups drain
// the accumulators in tile order (stream 0's, then stream 1's), each taking
// half of the tile's columns, with the C / residual rows of a tile pulled
// into L2 before its accumulator is ready.
//
// Forms for shapes with few tiles (template flags, chosen by the planner):
//   * one stream (STREAMS = 1): units of one 256-row M-tile, the single MMA
//     stream alternating between the two accumulators so that a tile's
//     ending overlaps the next tile's main loop;
//   * two K streams (KPAR, one stream per unit and one unit per pair): both
//     issuers on the one tile, the even and the odd K blocks into the two
//     accumulators, which the ending adds;
//   * split K (SPLIT): clusters of four CTAs, two pairs per tile, pair kp
//     over the K half kp; each CTA then finishes half of its rows' columns
//     after pushing the other half of its partial to the CTA with the same
//     rows in the other pair.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gbf {


// Raster group of M-tile pairs: the ~152 tiles in flight then span about 16
// M-tiles x 9 N-tiles, whose A and B panels (K = 8192: 64 + 40 MB) stay in L2.
constexpr int kQGroup = 8;
constexpr int kQABytes = kBM * kBK * 2;        // 16 KB: this CTA's 128 rows of A
constexpr int kQThreads = 384;                 // warps 0-3 roles, 4-11 epilogue
constexpr int kQTileM = 2 * kBM;               // 256 rows per pair tile
constexpr int kQSplitHalf = 128;               // split-K: columns each K half finishes
constexpr int kQSplitBytes = kQSplitHalf * kBM * 4;  // 64 KB: the other half's partial

// Tile width BN (MMA N) of the pair: 256, or 224 when that fills the last
// round of tiles better (the planner picks it for K-contiguous weights).
// Each CTA holds BN/2 rows of the B tile.
//
// STREAMS: M-tiles of 256 rows per unit of work.  Two (the default): a unit
// is an M-tile pair whose two tiles share each B tile and are computed by two
// MMA streams into the two accumulators.  One: a unit is one M-tile, a
// single MMA stream alternates between the two accumulators so that the
// ending of a tile overlaps the main loop of the next; twice as many units
// of half the size, for shapes whose M-tile pairs are fewer than the SM pairs.
template <int BN, int STREAMS = 2>
struct PairCfg {
  static constexpr int kStreams = STREAMS;
  // B region of a stage: room for 128 rows / columns of 64 k (16 KB); a
  // 224-wide tile fills 112 of them (K-major rows), or two 64-column boxes of
  // which the MMA reads the first 112 columns (N-major B[K][N])
  static constexpr int kBBytes = 128 * kBK * 2;
  static constexpr int kStageBytes = STREAMS * kQABytes + kBBytes;  // A0 (| A1) | B
  static constexpr int kStages = STREAMS == 2 ? 4 : 6;
  // ring | barriers (1 KB) | output staging: 8 epilogue warps x 2 buffers of 2 KB
  static constexpr int kBarBytes = 1024;
  static constexpr int kStagingBytes = 8 * 2 * kStageChunkBytes;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kStagingBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
  static constexpr int kChunks = BN / 32;             // 32-column epilogue chunks
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(BN % 32 == 0 && BN <= 256, "tile width");
  static_assert(STREAMS == 1 || STREAMS == 2, "one or two streams");
};

struct PairArgs {
  int M, N, K;
  int m_tiles, n_tiles, num_kb;
  EpiParams ep;
  KernelCtl ctl;
};

// v[j] += the fp32 accumulator column j of this thread's lane at taddr
// (32 columns, read 16 at a time to keep registers free).
__device__ __forceinline__ void add_acc32(uint32_t taddr, uint32_t (&v)[32]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t o[16];
    tmem_ld16(taddr + 16 * h, o);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[16 * h + j] = __float_as_uint(__uint_as_float(v[16 * h + j]) + __uint_as_float(o[j]));
  }
}

// Let in-flight copies land before an aborted CTA exits (bounded: ~2 ms).
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
}

template <bool W_KN, bool DUAL, int BN, int STREAMS, bool SPLIT, bool KPAR>
__global__ void __launch_bounds__(kQThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmO,
                     const PairArgs a) {
  using Cfg = PairCfg<BN, STREAMS>;
  constexpr int kQStages = Cfg::kStages;
  constexpr int kQStreams = Cfg::kStreams;
  // bytes the TMA engine writes into one CTA's stage
  constexpr int kLoadBytes =
      kQStreams * kQABytes + (W_KN ? 2 * 64 * kBK * 2 : (BN / 2) * kBK * 2);
  static_assert(!DUAL || BN == 256, "narrow tiles only for the single product");
  static_assert(!SPLIT || (!DUAL && BN == 256 && STREAMS == 1), "split-K: one stream, 256 wide");
  static_assert(!KPAR || (!DUAL && STREAMS == 1 && !SPLIT), "two K streams: one M-tile per unit");
  // MMA issuing threads: two streams of M-tiles, or (KPAR) two streams over
  // the alternate K blocks of the same tile, one accumulator each
  constexpr int kIssuers = (STREAMS == 2 || KPAR) ? 2 : 1;
  static_assert(!SPLIT || kQStages * Cfg::kStageBytes >= 2 * kQSplitBytes, "park + receive");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQStages * Cfg::kStageBytes);
  uint64_t* empty = full + kQStages;
  uint64_t* tfull = empty + kQStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint64_t* recvb = done + 1;  // split-K: the other K half's partial pushed here
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recvb + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  uint8_t* staging = smem + kQStages * Cfg::kStageBytes + Cfg::kBarBytes;  // 1024-aligned

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs are the cluster ranks {2i, 2i+1}; the split-K form runs two
  // pairs per cluster of four, pair kp over the K half kp of the same tile.
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = crank & 1u;
  const uint32_t lead = crank & ~1u;  // cluster rank of this pair's even CTA
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);
  const bool leader = rank == 0;
  const int kp = SPLIT ? static_cast<int>(crank >> 1) : 0;
  const int pair = SPLIT ? static_cast<int>(blockIdx.x >> 2) : static_cast<int>(blockIdx.x >> 1);
  const int npairs = SPLIT ? static_cast<int>(gridDim.x >> 2) : static_cast<int>(gridDim.x >> 1);
  const int kb_begin = SPLIT ? (kp * a.num_kb) / 2 : 0;
  const int kb_end = SPLIT ? ((kp + 1) * a.num_kb) / 2 : a.num_kb;
  // KPAR: K block kb_begin + i goes to stream i % 2; the second stream (and
  // its accumulator) takes part only when there are two blocks or more
  const bool two_k = KPAR && kb_end - kb_begin >= 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kQStreams);  // both issuers' commits
    }
    for (int i = 0; i < 2; ++i) {  // the two accumulators
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 16);  // 8 epilogue warps in each CTA of the pair
    }
    mbar_init(done, (KPAR && !two_k) ? 1 : kIssuers);
    if (SPLIT) {
      mbar_init(recvb, 1);
      mbar_arrive_expect_tx(recvb, kQSplitBytes);  // the other K half's 128 x 128 partial
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    if (DUAL) tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_holder, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const WaitCtl ctl{a.ctl.err, a.ctl.timeout_ns, abort_flag, prof_slots(a.ctl.prof)};
  const long long t_start = clock64();
  // units: STREAMS M-tiles (the last unit's second tile may be empty) x one N-tile
  const int m_pairs = (a.m_tiles + kQStreams - 1) / kQStreams;
  const int num_super = m_pairs * a.n_tiles;
  const int out_bn = DUAL ? 128 : BN;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t fills[kQStages];
#pragma unroll
      for (int i = 0; i < kQStages; ++i) fills[i] = 0;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // Nothing is read before the previous kernel in the stream has
      // completed: any input, weights included, may be its output.
      griddep_wait();
      for (int t = pair; t < num_super && ok; t += npairs) {
        int mp, nb;
        tile_coords(t, m_pairs, a.n_tiles, mp, nb, kQGroup);
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (!wait_bar(&empty[s], ph ^ 1, ctl, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + s * Cfg::kStageBytes;
          uint8_t* sb = sa + kQStreams * kQABytes;
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), lead);
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * kLoadBytes);
#pragma unroll
          for (int i = 0; i < kQStreams; ++i)  // rows past M read as zeros
            tma_load_2d_pair(sa + i * kQABytes, &tmA, bar, kb * kBK,
                             (kQStreams * mp + i) * kQTileM + static_cast<int>(rank) * kBM);
          const CUtensorMap* wmap = (DUAL && rank) ? &tmW2 : &tmW;
          const int n0 = DUAL ? nb * 128 : nb * BN + static_cast<int>(rank) * (BN / 2);
          if constexpr (W_KN) {
            tma_load_2d_pair(sb, wmap, bar, n0, kb * kBK);
            tma_load_2d_pair(sb + 8192, wmap, bar, n0 + 64, kb * kBK);
          } else {
            tma_load_2d_pair(sb, wmap, bar, kb * kBK, n0);
          }
          fills[s]++;
          if (++s == kQStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (ok) {
        // Every copy is consumed before the MMAs report the stage empty.
        for (int i = 0; i < kQStages; ++i)
          if (fills[i]) wait_bar(&empty[i], (fills[i] - 1) & 1, ctl, kSiteDrain, false);
      } else {
        settle_after_abort();
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // The pair's tiles in order l = 0, 1, ...: tile l is M-tile l % STREAMS
    // of unit l / STREAMS, accumulated in accumulator l & 1.  With two streams
    // warp 1 lane 0 issues the even tiles and warp 2 lane 0 the odd ones from
    // the same stages (each stream keeps its accumulator); with one stream
    // warp 1 issues every tile, alternating accumulators.  With two K
    // streams (KPAR) both issue every tile, warp 1 lane 0 its even and warp 2
    // lane 0 its odd K blocks, each into its own accumulator, and the ending
    // adds the two.  Warp 2 also allocates and frees the tensor memory,
    // outside this loop.
    const int st = warp - 1;
    if (lane == 0 && leader && st < kIssuers && (!KPAR || st == 0 || two_k)) {
      constexpr uint32_t idesc = idesc_bf16(kQTileM, BN, false, W_KN);
      int s = 0;
      uint32_t ph = 0;
      int l = st;
      bool ok = true;
      for (int t = pair, u = 0; t < num_super && ok; t += npairs, l += kQStreams, ++u) {
        const int acc = KPAR ? st : (l & 1);
        const uint32_t d = tmem_base + acc * 256;
        // uses of this accumulator so far: KPAR one per unit, else every other tile
        const int use = KPAR ? u : (l >> 1);
        if (!wait_bar(&tempty[acc], (use & 1) ^ 1, ctl, kSiteMmaAccEmpty)) break;
        tc_fence_after();
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (KPAR && ((kb - kb_begin) & 1) != st) {  // the other stream's block
            if (++s == kQStages) {
              s = 0;
              ph ^= 1;
            }
            continue;
          }
          if (!wait_bar(&full[s], ph, ctl, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s0 = smem_u32(stages + s * Cfg::kStageBytes);
          const uint32_t a0 = s0 + (KPAR ? 0 : st) * kQABytes;  // this stream's M-tile
          const uint32_t b0 = s0 + kQStreams * kQABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = W_KN ? sdesc_sw128(b0 + k * 2048, 8192, 1024)
                                     : sdesc_sw128(b0 + k * 32, 16, 1024);
            // the stream's first K step overwrites the accumulator
            mma_ss_pair(d, ad, bd, idesc, (kb != kb_begin + (KPAR ? st : 0) || k != 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[s], pair_mask);
          if (++s == kQStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if (!(a.ctl.inject && l == 0 && u == 0)) mma_commit_pair(&tfull[acc], pair_mask);
      }
      mma_commit_pair(done, static_cast<uint16_t>(1u << lead));
      wait_bar(done, 0, ctl, kSiteDrain, false);
    }
    __syncwarp();
  } else if (warp >= 4 && !SPLIT) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // the pair's tiles in order: local tile l belongs to stream l % 2
    griddep_wait();  // the ending reads C, bias, residual and writes out
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const uint64_t pol = l2_evict_first_policy();
    constexpr int kChunks = DUAL ? 4 : Cfg::kChunks;
    constexpr int kFirst = (kChunks + 1) / 2;  // chunks of warpgroup 0; the rest go to 1
    const int c_begin = half == 0 ? 0 : kFirst;
    const int c_end = half == 0 ? kFirst : kChunks;
    const uint32_t tempty_leader[2] = {mapa_shared(smem_u32(&tempty[0]), lead),
                                       mapa_shared(smem_u32(&tempty[1]), lead)};
    uint8_t* my_staging = staging + (warp - 4) * 2 * kStageChunkBytes;
    int flip = 0;
    // tile l of the pair: unit pair + (l / STREAMS) * npairs, M-tile l % STREAMS
    // of it, in accumulator l & 1 (use (l >> 1) of that accumulator)
    // (KPAR: tile l in both accumulators, use l of each, summed here)
    for (int local = 0; pair + (local / kQStreams) * npairs < num_super; ++local) {
      const int st = KPAR ? 0 : (local & 1);  // accumulator
      int mp, nb;
      tile_coords(pair + (local / kQStreams) * npairs, m_pairs, a.n_tiles, mp, nb, kQGroup);
      const int mb = kQStreams * mp + local % kQStreams;
      const uint32_t aph = KPAR ? (local & 1) : ((local >> 1) & 1);
      const int64_t row =
          static_cast<int64_t>(mb) * kQTileM + static_cast<int>(rank) * kBM + q * 32 + lane;
      epi_row_l2_prefetch(row, nb * out_bn + c_begin * 32, nb * out_bn + c_end * 32, a.M, a.N,
                          a.ep);
      RowLoads L;
      epi_row_prefetch(L, row, nb * out_bn + c_begin * 32, a.M, a.N, a.ep, pol);
      if (!wait_bar(&tfull[st], aph, ctl, kSiteEpiAccFull)) break;
      if (two_k && !wait_bar(&tfull[1], aph, ctl, kSiteEpiAccFull)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + st * 256 + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = c_begin; c < c_end; ++c) {
        const int col0 = nb * out_bn + c * 32;
        uint32_t acc[32], up[32];
        tmem_ld32(tb + c * 32, acc);
        if constexpr (DUAL) tmem_ld32(tb + 128 + c * 32, up);
        tmem_wait_ld();
        if constexpr (KPAR) {
          if (two_k) add_acc32(tb + 256 + c * 32, acc);  // the odd K blocks' accumulator
        }
        if (c == c_end - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(&tempty[st]);
            else mbar_arrive_cluster(tempty_leader[st]);
            if (two_k) {
              if (leader) mbar_arrive(&tempty[1]);
              else mbar_arrive_cluster(tempty_leader[1]);
            }
          }
        }
        const RowLoads cur = L;
        if (c + 1 < c_end) epi_row_prefetch(L, row, col0 + 32, a.M, a.N, a.ep, pol);
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
    // One tile per cluster.  The CTA of K half kp finishes columns
    // [128 kp, 128 kp + 128) of its 128 rows: it parks the other 128 columns
    // of its partial as [column][row] fp32 in its idle ring (consecutive
    // lanes on consecutive words), one thread pushes them with four 16 KB
    // bulk copies to the CTA holding the same rows in the other pair
    // (cluster rank crank ^ 2), and each CTA adds the copy it received to its
    // own columns, K half 0's partial first in both (the result does not
    // depend on which CTA finishes which columns).
    const bool epi = warp >= 4;
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;  // warpgroup: chunks 2*half, 2*half + 1 of the 128 columns
    const int rl = q * 32 + lane;      // row within the CTA's 128 = TMEM lane
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);  // accumulator 0
    float* park = reinterpret_cast<float*>(stages);
    const float* recv = reinterpret_cast<const float*>(stages + kQSplitBytes);
    const bool have_tile = pair < num_super;
    int mp = 0, nb = 0;
    if (have_tile) tile_coords(pair, m_pairs, a.n_tiles, mp, nb, kQGroup);
    const uint64_t pol = l2_evict_first_policy();
    const int64_t row =
        static_cast<int64_t>(mp) * kQTileM + static_cast<int>(rank) * kBM + rl;
    const int mine = kp * kQSplitHalf;         // first column this CTA finishes
    const int theirs = kQSplitHalf - mine;     // the counterpart's first column
    if (epi) {
      griddep_wait();  // the ending reads C, bias, residual and writes out
      if (have_tile)
        epi_row_l2_prefetch(row, nb * 256 + mine + half * 64, nb * 256 + mine + half * 64 + 64,
                            a.M, a.N, a.ep);
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
    cluster_sync_all();  // every CTA of the cluster parked, every receive barrier armed
    if (threadIdx.x == 128) {
      const uint32_t peer = crank ^ 2u;
      constexpr int kPiece = kQSplitBytes / 4;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        bulk_copy_to_peer(mapa_shared(smem_u32(stages + kQSplitBytes + i * kPiece), peer),
                          smem_u32(stages + i * kPiece), kPiece,
                          mapa_shared(smem_u32(recvb), peer));
    }
    if (epi) {
      uint8_t* my_staging = staging + (warp - 4) * 2 * kStageChunkBytes;
      int flip = 0;
      // not cut short by the abort flag: the counterpart sends whatever its state
      wait_bar(recvb, 0, ctl, kSiteEpiAccFull, /*honor_abort=*/false);
      RowLoads L;
      epi_row_prefetch(L, row, nb * 256 + mine + 2 * half * 32, a.M, a.N, a.ep, pol);
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        const int col0 = nb * 256 + mine + c * 32;
        uint32_t sum[32];  // this CTA's partial, then the total
        tmem_ld32(tb + mine + c * 32, sum);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float o = __uint_as_float(sum[j]);
          const float p = recv[(c * 32 + j) * kBM + rl];
          sum[j] = __float_as_uint(kp == 0 ? o + p : p + o);
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
        if (have_tile) store_chunk32(my_staging, flip, w, &tmO, row - lane, col0, a.M, a.N, pol);
      }
      // every staged chunk written to global memory before the CTA may exit
      if (lane == 0) bulk_wait<0>();
      __syncwarp();
    }
  }

  if (ctl.prof && threadIdx.x == 0) atomicAdd(&ctl.prof[31], static_cast<unsigned long long>(clock64() - t_start));
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal it or read its memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

namespace {

template <bool W_KN, bool DUAL, int BN, int STREAMS = 2, bool SPLIT = false, bool KPAR = false>
cudaError_t run_pair(const GemmPlan& p, const CUtensorMap& tmA, const CUtensorMap& tmW,
                     const CUtensorMap& tmW2, const CUtensorMap& tmO, const PairArgs& args,
                     cudaStream_t stream) {
  static std::atomic<uint64_t> mask{0};
  auto kernel = gemm_pair_kernel<W_KN, DUAL, BN, STREAMS, SPLIT, KPAR>;
  constexpr int kQSmem = PairCfg<BN, STREAMS>::kSmem;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
    if (e != cudaSuccess) return e;
    mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid, 1, 1);
  cfg.blockDim = dim3(kQThreads, 1, 1);
  cfg.dynamicSmemBytes = kQSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SPLIT ? 4 : 2;  // split-K: two pairs per tile
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel in the stream finishes (it waits
  // with griddepcontrol.wait before touching anything that kernel writes)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmW, tmW2, tmO, args);
}

}  // namespace

namespace {

// Clusters of `size` 1-SM CTAs of the pair kernel that fit on the device at once.
int max_active_clusters(int size) {
  cudaLaunchConfig_t cfg = {};
  constexpr int kQSmem = PairCfg<256>::kSmem;
  cfg.gridDim = dim3(size, 1, 1);
  cfg.blockDim = dim3(kQThreads, 1, 1);
  cfg.dynamicSmemBytes = kQSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kernel = gemm_pair_kernel<false, false, 256, 2, false, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int max_active_pairs() { return max_active_clusters(2); }
int max_active_quads() { return max_active_clusters(4); }

cudaError_t launch_gemm_pair(const GemmPlan& plan, bool w_kn, bool dual, const CUtensorMap& tmA,
                             const CUtensorMap& tmW, const CUtensorMap& tmW2,
                             const CUtensorMap& tmO, const EpiParams& ep, int M, int N, int K,
                             const KernelCtl& ctl, cudaStream_t stream) {
  PairArgs args{M, N, K, plan.m_tiles, plan.n_tiles, plan.num_kb, ep, ctl};
  if (plan.path == kPathPairSplit)  // split-K: clusters of two pairs, one tile each
    return w_kn ? run_pair<true, false, 256, 1, true>(plan, tmA, tmW, tmW2, tmO, args, stream)
                : run_pair<false, false, 256, 1, true>(plan, tmA, tmW, tmW2, tmO, args, stream);
  if (plan.streams == 1 && !dual && plan.kpar)  // one tile per pair: two K streams
    return w_kn ? run_pair<true, false, 256, 1, false, true>(plan, tmA, tmW, tmW2, tmO, args,
                                                             stream)
           : plan.bn == 224
               ? run_pair<false, false, 224, 1, false, true>(plan, tmA, tmW, tmW2, tmO, args,
                                                             stream)
               : run_pair<false, false, 256, 1, false, true>(plan, tmA, tmW, tmW2, tmO, args,
                                                             stream);
  if (plan.streams == 1 && !dual)  // one stream: units of one 256-row M-tile
    return w_kn ? run_pair<true, false, 256, 1>(plan, tmA, tmW, tmW2, tmO, args, stream)
           : plan.bn == 224
               ? run_pair<false, false, 224, 1>(plan, tmA, tmW, tmW2, tmO, args, stream)
               : run_pair<false, false, 256, 1>(plan, tmA, tmW, tmW2, tmO, args, stream);
  if (w_kn)
    return dual              ? run_pair<true, true, 256>(plan, tmA, tmW, tmW2, tmO, args, stream)
           : plan.bn == 224 ? run_pair<true, false, 224>(plan, tmA, tmW, tmW2, tmO, args, stream)
                            : run_pair<true, false, 256>(plan, tmA, tmW, tmW2, tmO, args, stream);
  if (dual) return run_pair<false, true, 256>(plan, tmA, tmW, tmW2, tmO, args, stream);
  return plan.bn == 224 ? run_pair<false, false, 224>(plan, tmA, tmW, tmW2, tmO, args, stream)
                        : run_pair<false, false, 256>(plan, tmA, tmW, tmW2, tmO, args, stream);
}

}  // namespace gbf

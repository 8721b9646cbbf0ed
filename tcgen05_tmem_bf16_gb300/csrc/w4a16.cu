// w4a16.cu -- weight-only int4 GEMM with on-chip dequantisation, sm_103a.
//
// The kernel streams the packed int4 weights and their group scales into
// shared memory with TMA, dequantises them on-chip to bf16, and feeds them to
// the tensor cores; the bf16 weight matrix never exists in HBM ("Fusion
// Thinking", Pattern 3, Dequant + GEMM: load INT4 weights + scales directly,
// unpack the high and low nibbles, w = (q - 8) * s, accumulate a . w).
//
// GB300 design.  out^T = W~^T * A^T: the weights are the MMA's A operand
// (128 rows = output columns) and the few activation rows are its N.  The
// dequantised A operand is written straight into TENSOR MEMORY with
// tcgen05.st and consumed by tcgen05.mma from there, so the 2-byte weights
// never make a round trip through shared memory: per weight, shared memory
// carries only the half byte the TMA engine wrote and the transform threads
// read once.
//
// Tile: 256 output columns.  Transform thread t (0..127, warps 4-7) owns
// packed byte column t: output columns n0+2t (high nibble) and n0+2t+1 (low
// nibble).  The even columns form one 128-row A operand (TMEM region E) and
// the odd columns another (region O), so every thread writes only its own
// TMEM lane, and the epilogue stores column pairs as one bf16x2.  Each
// 64-deep K block is two MMAs per 16-deep step (E and O).
//
// Dequantisation of a nibble q, exact as the definition wants:
//   bits 0x4300 | q  is the bf16 value 128 + q;
//   (128 + q) - 136 = q - 8 exactly (small integers);
//   (q - 8) * s with one bf16 multiply = bf16_rne((q - 8) * s).
//
// K is split across a thread-block cluster; partial sums meet in the
// rank-0 CTA through distributed shared memory, which applies the ending.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gbf {

constexpr int kW4Threads = 256;
constexpr int kW4ABytes = kBK * (kW4BN / 2);  // packed tile: 64 rows x 128 bytes = 8 KB
static_assert(kW4ABytes == 8192, "packed tile size");
constexpr int kW4TStages = 2;                     // TMEM A-operand stages

template <int MPAD>
struct W4Cfg {
  static constexpr int kXBytes = MPAD * kBK * 2;                 // activations, SW128
  static constexpr int kScaleBytes = 1024;                       // 256 bf16 + pad
  static constexpr int kStageBytes = kW4ABytes + kXBytes + kScaleBytes;
  static constexpr int kStages = MPAD <= 32 ? 8 : 6;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 256;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColDE = 0;
  static constexpr uint32_t kColDO = MPAD;
  static constexpr uint32_t kColA = 2 * MPAD;  // A stage j: E at +64j, O at +64j+32
  static_assert(kColA + 64 * kW4TStages <= kTmemCols, "TMEM budget");
  static_assert(kStages * kStageBytes >= 128 * 2 * MPAD * 4, "reduction buffer must fit");
};

struct W4Args {
  int M, N, K;
  int num_kb;
  int splits;
  EpiParams ep;
  KernelCtl ctl;
};

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ __nv_bfloat162 bits_bf2(uint32_t u) {
  return *reinterpret_cast<__nv_bfloat162*>(&u);
}

// Epilogue of output columns (n, n+1) for 16 rows m0..m0+15: operand loads
// first (independent, overlapping), then math and bf16x2 stores.
template <int ACT>
__device__ __forceinline__ void epi_pair16(const float (&ve)[16], const float (&vo)[16],
                                           int64_t m0, int n, int M, int N,
                                           const EpiParams& e) {
  if (n >= N) return;
  float b0 = 0.0f, b1 = 0.0f;
  if (e.bias) {
    const uint32_t b = *reinterpret_cast<const uint32_t*>(e.bias + n);
    b0 = bf16lo(b);
    b1 = bf16hi(b);
  }
  uint32_t c[16], r[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t m = m0 + j;
    const bool ok = m < M;
    const int64_t off = m * N + n;
    c[j] = (ok && e.C) ? *reinterpret_cast<const uint32_t*>(e.C + off) : 0u;
    r[j] = (ok && e.residual) ? *reinterpret_cast<const uint32_t*>(e.residual + off) : 0u;
  }
  const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int64_t m = m0 + j;
    if (m >= M) break;
    const float x0 = act_apply<ACT>(fmaf(beta, bf16lo(c[j]), e.alpha * ve[j]) + b0) + bf16lo(r[j]);
    const float x1 = act_apply<ACT>(fmaf(beta, bf16hi(c[j]), e.alpha * vo[j]) + b1) + bf16hi(r[j]);
    *reinterpret_cast<uint32_t*>(e.out + m * N + n) = pack_bf16x2(x0, x1);
  }
}

template <int MPAD>
__global__ void __launch_bounds__(kW4Threads, 2)
    w4a16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmS, const W4Args a, int group) {
  using Cfg = W4Cfg<MPAD>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment by pointer arithmetic on the shared array (keeps the
  // shared address space for the compiler).
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kStages * Cfg::kStageBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* afull = empty + Cfg::kStages;
  uint64_t* aempty = afull + kW4TStages;
  uint64_t* dfull = aempty + kW4TStages;
  uint64_t* done = dfull + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
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
      mbar_init(&empty[i], 4 + 1);  // 4 transform warps + the MMA commit
    }
    for (int i = 0; i < kW4TStages; ++i) {
      mbar_init(&afull[i], 4);
      mbar_init(&aempty[i], 1);
    }
    mbar_init(dfull, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 2) {
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const WaitCtl ctl{a.ctl.err, a.ctl.timeout_ns, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t stream_policy = policy_evict_first();
      uint32_t fills[Cfg::kStages];
#pragma unroll
      for (int i = 0; i < Cfg::kStages; ++i) fills[i] = 0;
      int s = 0;
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&empty[s], ph ^ 1, ctl, kSiteProducerEmpty)) break;
        uint8_t* sq = stages + s * Cfg::kStageBytes;
        uint8_t* sx = sq + kW4ABytes;
        uint8_t* ss = sx + Cfg::kXBytes;
        mbar_arrive_expect_tx(&full[s], kW4ABytes + Cfg::kXBytes + kW4BN * 2);
        tma_load_2d_hint(sq, &tmQ, &full[s], nb * (kW4BN / 2), kb * kBK, stream_policy);
        tma_load_2d(sx, &tmA, &full[s], kb * kBK, mb * MPAD);
        tma_load_2d(ss, &tmS, &full[s], nb * kW4BN, (kb * kBK) / group);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, MPAD, false, false);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        const int i = kb - kb0;
        const int j = i % kW4TStages;
        const uint32_t tph = (i / kW4TStages) & 1;
        if (!wait_bar(&afull[j], tph, ctl, kSiteMmaOperand) ||
            !wait_bar(&full[s], ph, ctl, kSiteMmaFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t x0 = smem_u32(stages + s * Cfg::kStageBytes + kW4ABytes);
        const uint32_t aE = tmem_base + Cfg::kColA + 64 * j;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t bd = sdesc_sw128(x0 + k * 32, 16, 1024);
          const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
          mma_ts(tmem_base + Cfg::kColDE, aE + k * 8, bd, idesc, accum);
          mma_ts(tmem_base + Cfg::kColDO, aE + 32 + k * 8, bd, idesc, accum);
        }
        mma_commit(&aempty[j]);
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
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dequantise into TMEM
    const int t = threadIdx.x - 128;      // packed byte column = TMEM lane
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const __nv_bfloat162 c136 = __floats2bfloat162_rn(136.0f, 136.0f);
    int s = 0;
    uint32_t ph = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      const int i = kb - kb0;
      const int j = i % kW4TStages;
      const uint32_t tph = (i / kW4TStages) & 1;
      if (!wait_bar(&full[s], ph, ctl, kSiteXformFull)) break;
      if (!wait_bar(&aempty[j], tph ^ 1, ctl, kSiteXformEmpty)) break;
      tc_fence_after();
      const uint8_t* sq = stages + s * Cfg::kStageBytes;
      const uint32_t sc = *reinterpret_cast<const uint32_t*>(sq + kW4ABytes + Cfg::kXBytes + 4 * t);
      const __nv_bfloat162 sE = bits_bf2(__byte_perm(sc, 0, 0x1010));
      const __nv_bfloat162 sO = bits_bf2(__byte_perm(sc, 0, 0x3232));
      uint32_t e[32], o[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const uint32_t b0 = sq[(2 * r) * 128 + t];
        const uint32_t b1 = sq[(2 * r + 1) * 128 + t];
        const uint32_t p = __byte_perm(b0, b1, 0x0400);  // byte0 = row 2r, byte2 = row 2r+1
        const uint32_t lo = (p & 0x000F000Fu) | 0x43004300u;
        const uint32_t hi = ((p >> 4) & 0x000F000Fu) | 0x43004300u;
        o[r] = bf2_bits(__hmul2(__hsub2(bits_bf2(lo), c136), sO));
        e[r] = bf2_bits(__hmul2(__hsub2(bits_bf2(hi), c136), sE));
      }
      const uint32_t aE = tmem_base + lane_off + Cfg::kColA + 64 * j;
      tmem_st16(aE, *reinterpret_cast<const uint32_t(*)[16]>(&e[0]));
      tmem_st16(aE + 16, *reinterpret_cast<const uint32_t(*)[16]>(&e[16]));
      tmem_st16(aE + 32, *reinterpret_cast<const uint32_t(*)[16]>(&o[0]));
      tmem_st16(aE + 48, *reinterpret_cast<const uint32_t(*)[16]>(&o[16]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[j]);
        mbar_arrive(&empty[s]);
      }
      if (++s == Cfg::kStages) {
        s = 0;
        ph ^= 1;
      }
    }
  }

  // ---- epilogue (warps 4-7): cluster reduction of the partial sums, ending.
  // Every rank parks its partial in its own shared memory; 16-row chunks are
  // shared out among the ranks (chunk c to rank c % S) and summed over ranks
  // 0..S-1 in order through distributed shared memory.
  const bool epi = warp >= 4;
  const int q = warp & 3;
  const int tid = threadIdx.x - 128;
  const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  float4* red = reinterpret_cast<float4*>(stages);
  constexpr int kChunks = MPAD / 16;  // per region
  bool have = false;
  if (epi) {
    have = wait_bar(dfull, 0, ctl, kSiteEpiAccFull);
    tc_fence_after();
    if (S > 1) {
#pragma unroll 1
      for (int c = 0; c < 2 * kChunks; ++c) {
        const uint32_t col = (c < kChunks ? Cfg::kColDE : Cfg::kColDO) + (c % kChunks) * 16;
        uint32_t r[16];
        tmem_ld16(tb + col, r);
        tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          red[(c * 4 + v) * 128 + tid] =
              make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                          __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
    }
  }
  if (S > 1) cluster_sync_all();
  if (epi) {
    const int n = nb * kW4BN + 2 * tid;
#pragma unroll 1
    for (int c = static_cast<int>(rank); c < kChunks; c += S) {
      float ve[16], vo[16];
      if (S == 1) {
        uint32_t re[16], ro[16];
        tmem_ld16(tb + Cfg::kColDE + c * 16, re);
        tmem_ld16(tb + Cfg::kColDO + c * 16, ro);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          ve[jj] = have ? __uint_as_float(re[jj]) : 0.0f;
          vo[jj] = have ? __uint_as_float(ro[jj]) : 0.0f;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) ve[jj] = vo[jj] = 0.0f;
        for (int p = 0; p < S; ++p) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float4 fe, fo;
            float4* pe = &red[(c * 4 + w) * 128 + tid];
            float4* po = &red[((kChunks + c) * 4 + w) * 128 + tid];
            if (p == static_cast<int>(rank)) {
              fe = *pe;
              fo = *po;
            } else {
              fe = ld_dsmem_f4(mapa_shared(smem_u32(pe), static_cast<uint32_t>(p)));
              fo = ld_dsmem_f4(mapa_shared(smem_u32(po), static_cast<uint32_t>(p)));
            }
            ve[4 * w] += fe.x; ve[4 * w + 1] += fe.y; ve[4 * w + 2] += fe.z; ve[4 * w + 3] += fe.w;
            vo[4 * w] += fo.x; vo[4 * w + 1] += fo.y; vo[4 * w + 2] += fo.z; vo[4 * w + 3] += fo.w;
          }
        }
      }
      const int64_t m0 = static_cast<int64_t>(mb) * MPAD + c * 16;
      switch (a.ep.act) {
        case kActRelu: epi_pair16<kActRelu>(ve, vo, m0, n, a.M, a.N, a.ep); break;
        case kActSilu: epi_pair16<kActSilu>(ve, vo, m0, n, a.M, a.N, a.ep); break;
        case kActGeluTanh: epi_pair16<kActGeluTanh>(ve, vo, m0, n, a.M, a.N, a.ep); break;
        default: epi_pair16<kActIdentity>(ve, vo, m0, n, a.M, a.N, a.ep); break;
      }
    }
  }
  if (S > 1) cluster_sync_all();

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

namespace {

template <int MPAD>
cudaError_t run_w4(const GemmPlan& p, const CUtensorMap& tmA, const CUtensorMap& tmQ,
                   const CUtensorMap& tmS, const W4Args& args, int group, cudaStream_t stream) {
  static std::atomic<uint64_t> mask{0};
  auto kernel = w4a16_kernel<MPAD>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             W4Cfg<MPAD>::kSmem);
    if (e != cudaSuccess) return e;
    mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_tiles, p.m_tiles);
  cfg.blockDim = dim3(kW4Threads, 1, 1);
  cfg.dynamicSmemBytes = W4Cfg<MPAD>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmQ, tmS, args, group);
}

}  // namespace

cudaError_t launch_w4a16(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmQ,
                         const CUtensorMap& tmS, const EpiParams& ep, int M, int N, int K,
                         int group, const KernelCtl& ctl, cudaStream_t stream) {
  W4Args args{M, N, K, plan.num_kb, plan.splits, ep, ctl};
  switch (plan.mpad) {
    case 16: return run_w4<16>(plan, tmA, tmQ, tmS, args, group, stream);
    case 32: return run_w4<32>(plan, tmA, tmQ, tmS, args, group, stream);
    case 64: return run_w4<64>(plan, tmA, tmQ, tmS, args, group, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gbf

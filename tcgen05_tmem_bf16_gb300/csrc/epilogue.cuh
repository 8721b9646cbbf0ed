// epilogue.cuh -- the fused ending shared by the dense GEMM kernels: operand
// prefetch, act(alpha*acc + beta*C + bias) + residual in fp32, bf16 stores;
// plus the persistent kernels' tile raster.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gbf {

// Round a pointer into dynamic shared memory up to 1024 bytes with pointer
// arithmetic on the shared array itself, so the compiler keeps the shared
// address space (ld/st.shared instead of generic accesses).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Pull the C and residual segments [col0, col1) of one row into L2 ahead of
// their loads (one prefetch per 128-byte line), so that an epilogue that
// starts as soon as an accumulator is ready does not wait on HBM latency.
__device__ __forceinline__ void epi_row_l2_prefetch(int64_t row, int col0, int col1, int M,
                                                    int N, const EpiParams& e) {
  if (row >= M) return;
  if (col1 > N) col1 = N;
  for (int col = col0; col < col1; col += 64) {
    const int64_t off = row * N + col;
    if (e.C) asm volatile("prefetch.global.L2 [%0];" ::"l"(e.C + off));
    if (e.residual) asm volatile("prefetch.global.L2 [%0];" ::"l"(e.residual + off));
  }
}

// Operands of the ending for 32 consecutive columns of one row, loaded
// before the accumulator is read from TMEM so that their latency overlaps.
struct RowLoads {
  uint4 c[4];
  uint4 b[4];
  uint4 r[4];
};

__device__ __forceinline__ void epi_row_prefetch(RowLoads& L, int64_t row, int col0, int M,
                                                 int N, const EpiParams& e, uint64_t pol) {
  const bool rok = row < M;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int col = col0 + v * 8;
    const bool ok = rok && col < N;
    const int64_t off = row * N + col;
    const uint4 z = make_uint4(0, 0, 0, 0);
    L.c[v] = (ok && e.C) ? ld_stream_u4(e.C + off, pol) : z;
    L.b[v] = (ok && e.bias) ? ldg_u4(e.bias + col) : z;
    L.r[v] = (ok && e.residual) ? ld_stream_u4(e.residual + off, pol) : z;  // may alias out
  }
}

// Epilogue of 32 consecutive output columns of one row (persistent kernel).
// `acc` holds fp32 bit patterns; for the dual GEMM `up` holds the up
// product and the result is act(alpha*g) * (alpha*u) + beta*C.
template <int ACT, bool DUAL>
__device__ __forceinline__ void epi_row32(const uint32_t (&acc)[32], const uint32_t (&up)[32],
                                          const RowLoads& L, int64_t row, int col0, int N,
                                          const EpiParams& e, uint64_t pol) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int col = col0 + v * 8;
    if (col >= N) break;
    const int64_t off = row * N + col;
    float x[8];
    if constexpr (DUAL) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = act_apply<ACT>(e.alpha * __uint_as_float(acc[v * 8 + i])) *
               (e.alpha * __uint_as_float(up[v * 8 + i]));
      if (e.C) {
        float c[8];
        unpack8(L.c[v], c);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = fmaf(e.beta, c[i], x[i]);
      }
    } else {
      float c[8], b[8], r[8];
      unpack8(L.c[v], c);
      unpack8(L.b[v], b);
      unpack8(L.r[v], r);
      const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = act_apply<ACT>(fmaf(beta, c[i], e.alpha * __uint_as_float(acc[v * 8 + i])) + b[i]) +
               r[i];
    }
    st_stream_u4(e.out + off, pack8(x), pol);
  }
}

// The ending of 32 consecutive output columns of one row, packed as 16
// bf16x2 words (column pairs), for the staged store below.  Columns past N
// see zero operands; the store does not write them.
template <int ACT, bool DUAL>
__device__ __forceinline__ void epi_row32_pack(const uint32_t (&acc)[32], const uint32_t (&up)[32],
                                               const RowLoads& L, const EpiParams& e,
                                               uint32_t (&w)[16]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float x[8];
    if constexpr (DUAL) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = act_apply<ACT>(e.alpha * __uint_as_float(acc[v * 8 + i])) *
               (e.alpha * __uint_as_float(up[v * 8 + i]));
      if (e.C) {
        float c[8];
        unpack8(L.c[v], c);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = fmaf(e.beta, c[i], x[i]);
      }
    } else {
      float c[8], b[8], r[8];
      unpack8(L.c[v], c);
      unpack8(L.b[v], b);
      unpack8(L.r[v], r);
      const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = act_apply<ACT>(fmaf(beta, c[i], e.alpha * __uint_as_float(acc[v * 8 + i])) + b[i]) +
               r[i];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) w[v * 4 + i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
  }
}

// Coalesced output through shared memory: each epilogue warp owns two 2 KB
// staging buffers; one buffer holds a 32-row x 32-column bf16 chunk, rows of
// 64 bytes in the tensor map's 64-byte swizzle (16-byte unit u of row r at
// u ^ ((r >> 1) & 3)), so a quarter-warp's 16-byte stores fall on distinct
// banks.  Lane 0 writes the chunk to global memory with one TMA store, which
// covers whole rows of 64 bytes instead of 32 separate 16-byte pieces.
constexpr int kStageChunkBytes = 32 * 64;

__device__ __forceinline__ void stage_row32(uint8_t* buf, int r, const uint32_t (&w)[16]) {
  const uint32_t base = smem_u32(buf) + static_cast<uint32_t>(r) * 64u;
  const uint32_t sw = static_cast<uint32_t>((r >> 1) & 3);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + ((u ^ sw) << 4)),
                 "r"(w[4 * u]), "r"(w[4 * u + 1]), "r"(w[4 * u + 2]), "r"(w[4 * u + 3])
                 : "memory");
}

// One warp's chunk (rows row0 .. row0+31, columns col0 .. col0+31) from the
// thread-per-row registers `w` to global memory through staging buffer
// `bufs[*flip]`.  The buffer's previous store (two chunks earlier) must have
// finished reading it first.
__device__ __forceinline__ void store_chunk32(uint8_t* bufs, int& flip, const uint32_t (&w)[16],
                                              const CUtensorMap* out_map, int64_t row0,
                                              int col0, int M, int N, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  uint8_t* buf = bufs + flip * kStageChunkBytes;
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
  stage_row32(buf, lane, w);
  fence_proxy_async_smem();  // the generic-proxy writes before the async-proxy read
  __syncwarp();
  if (lane == 0) {
    if (row0 < M && col0 < N) tma_store_2d(out_map, buf, col0, static_cast<int32_t>(row0), pol);
    bulk_commit();
  }
  flip ^= 1;
}

// Persistent tile raster: groups of `group` M-tiles (kGroupM by default);
// inside a group the N-tile index varies slowest, so the CTAs working at the
// same time share weight panels (and activation panels) in L2.
constexpr int kGroupM = 16;

__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int& mb, int& nb,
                                            int group = kGroupM) {
  const int per_group = group * n_tiles;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gm = min(group, m_tiles - first_m);
  const int local = t - g * per_group;
  nb = local / gm;
  mb = first_m + local % gm;
}

// Epilogue of one output column n for R consecutive rows m0..m0+R-1 (the
// swapped kernels): the operands are fetched first (col_prefetch, which can
// run before the accumulator is ready), then the math and the stores.
template <int R = 16>
struct ColLoads {
  float c[R];
  float r[R];
  float b;
};

template <int R>
__device__ __forceinline__ void col_prefetch(ColLoads<R>& L, int64_t m0, int n, int M, int N,
                                             const EpiParams& e, uint64_t pol) {
  const bool nok = n < N;
  L.b = (nok && e.bias) ? __bfloat162float(e.bias[n]) : 0.0f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int64_t m = m0 + j;
    const bool ok = nok && m < M;
    const int64_t off = m * N + n;
    L.c[j] = (ok && e.C) ? bf16bits_to_f(ld_stream_u16(e.C + off, pol)) : 0.0f;
    L.r[j] = (ok && e.residual) ? bf16bits_to_f(ld_stream_u16(e.residual + off, pol)) : 0.0f;
  }
}

template <int ACT, int R>
__device__ __forceinline__ void epi_col(const float (&v)[R], const ColLoads<R>& L, int64_t m0,
                                        int n, int M, int N, const EpiParams& e, uint64_t pol) {
  if (n >= N) return;
  const float beta = e.C ? e.beta : 0.0f;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int64_t m = m0 + j;
    if (m < M)
      st_stream_u16(e.out + m * N + n,
                    f_to_bf16bits(act_apply<ACT>(fmaf(beta, L.c[j], e.alpha * v[j]) + L.b) +
                                  L.r[j]),
                    pol);
  }
}

}  // namespace gbf

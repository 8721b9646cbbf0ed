// rmsnorm.cu -- fused residual add + RMSNorm, and its unfused composition.
//
// Per row m: r = a + x (fp32), out_resid = bf16(r) (the residual stream for
// the next block), out_norm = bf16(r * rsqrt(mean(r^2) + eps) * w) -- one
// pass over the row that reads a and x once and writes both results once
// ("Fusion Thinking", Pattern 1, Fused RMSNorm + residual).  The unfused
// composition is a residual-add kernel that writes bf16(r) followed by an
// RMSNorm kernel that reads it back (x = x + a; rmsnorm(x)).
//
// HBM-bound.  One CTA of 256 threads per row (grid-stride over rows); each
// thread holds R 16-byte vectors of the row in registers between the sum of
// squares and the scaling, so the row is read from HBM once, and loads its
// vectors of the CTA's next row before reducing the current one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace gbf {

namespace {

constexpr int kRmsThreads = 256;

template <int R>
__global__ void __launch_bounds__(kRmsThreads)
    add_rmsnorm_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ x,
                       const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ out_norm,
                       __nv_bfloat16* __restrict__ out_resid, int64_t M, int N, float eps) {
  __shared__ float partial[kRmsThreads / 32];
  const uint64_t pol = l2_evict_first_policy();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The loads of a CTA's next row are issued before the current row's
  // reduction, so each CTA keeps two rows of a and x in flight (R <= 4; wider
  // rows keep one, for registers).
  constexpr bool kAhead = R <= 4;
  uint4 ca[R], cx[R];  // this thread's vectors of the current row of a and x
  auto load_row = [&](int64_t row, uint4 (&ra)[R], uint4 (&rx)[R]) {
#pragma unroll
    for (int v = 0; v < R; ++v) {
      const int col = (threadIdx.x + v * kRmsThreads) * 8;
      if (col < N) {
        ra[v] = ld_stream_u4(a + row * N + col, pol);
        rx[v] = x ? ld_stream_u4(x + row * N + col, pol) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  if (kAhead && static_cast<int64_t>(blockIdx.x) < M) load_row(blockIdx.x, ca, cx);
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const int64_t base = row * N;
    uint4 na[R], nx[R];
    if (kAhead) {
      if (row + gridDim.x < M) load_row(row + gridDim.x, na, nx);
    } else {
      load_row(row, ca, cx);
    }
    float r[R][8];
    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < R; ++v) {
      const int col = (threadIdx.x + v * kRmsThreads) * 8;
      if (col < N) {
        float av[8], xv[8];
        unpack8(ca[v], av);
        unpack8(cx[v], xv);  // zeros without x: bf16 0x0000 is +0
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          r[v][i] = av[i] + xv[i];
          ss = fmaf(r[v][i], r[v][i], ss);
        }
        if (out_resid) st_stream_u4(out_resid + base + col, pack8(r[v]), pol);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) r[v][i] = 0.0f;
      }
    }
    // block sum of squares
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) partial[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < kRmsThreads / 32; ++i) tot += partial[i];
    __syncthreads();  // partial[] is reused by the next row
    const float rrms = rsqrtf(tot / static_cast<float>(N) + eps);
#pragma unroll
    for (int v = 0; v < R; ++v) {
      const int col = (threadIdx.x + v * kRmsThreads) * 8;
      if (col < N) {
        float wv[8], n[8];
        unpack8(ldg_u4(w + col), wv);
#pragma unroll
        for (int i = 0; i < 8; ++i) n[i] = r[v][i] * rrms * wv[i];
        st_stream_u4(out_norm + base + col, pack8(n), pol);
      }
    }
    if (kAhead) {
#pragma unroll
      for (int v = 0; v < R; ++v) {
        ca[v] = na[v];
        cx[v] = nx[v];
      }
    }
  }
}

// One wave of CTAs: as many per SM as fit (from the kernel's registers), so
// that every CTA's next row is in flight while it reduces the current one
// (4096 x 4096: 8 per SM 23.9 us, the 4 that fit 23.3 us, 3 or 6 24.6 us).
template <int R>
cudaError_t run_rms(const __nv_bfloat16* a, const __nv_bfloat16* x, const __nv_bfloat16* w,
                    __nv_bfloat16* norm, __nv_bfloat16* resid, int64_t M, int N, float eps,
                    int sms, cudaStream_t stream) {
  static std::atomic<int> per_sm{0};
  int fit = per_sm.load(std::memory_order_relaxed);
  if (fit <= 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, add_rmsnorm_kernel<R>, kRmsThreads,
                                                      0) != cudaSuccess ||
        fit <= 0) {
      (void)cudaGetLastError();
      fit = 4;
    } else {
      per_sm.store(fit, std::memory_order_relaxed);
    }
  }
  const int64_t cap = static_cast<int64_t>(sms) * fit;
  const int grid = static_cast<int>(M < cap ? M : cap);
  add_rmsnorm_kernel<R><<<grid, kRmsThreads, 0, stream>>>(a, x, w, norm, resid, M, N, eps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_add_rmsnorm(const __nv_bfloat16* a, const __nv_bfloat16* x,
                               const __nv_bfloat16* w, __nv_bfloat16* norm,
                               __nv_bfloat16* resid, int64_t M, int N, float eps, int sms,
                               cudaStream_t stream) {
  const int vecs = (N / 8 + kRmsThreads - 1) / kRmsThreads;  // 16-byte vectors per thread
  if (vecs <= 1) return run_rms<1>(a, x, w, norm, resid, M, N, eps, sms, stream);
  if (vecs <= 2) return run_rms<2>(a, x, w, norm, resid, M, N, eps, sms, stream);
  if (vecs <= 4) return run_rms<4>(a, x, w, norm, resid, M, N, eps, sms, stream);
  if (vecs <= 8) return run_rms<8>(a, x, w, norm, resid, M, N, eps, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gbf

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
// squares and the scaling, so the row is read from HBM once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const int64_t base = row * N;
    float r[R][8];
    float ss = 0.0f;
#pragma unroll
    for (int v = 0; v < R; ++v) {
      const int col = (threadIdx.x + v * kRmsThreads) * 8;
      if (col < N) {
        float av[8], xv[8];
        unpack8(ld_stream_u4(a + base + col, pol), av);
        if (x) {
          unpack8(ld_stream_u4(x + base + col, pol), xv);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[i] = 0.0f;
        }
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
  }
}

template <int R>
cudaError_t run_rms(const __nv_bfloat16* a, const __nv_bfloat16* x, const __nv_bfloat16* w,
                    __nv_bfloat16* norm, __nv_bfloat16* resid, int64_t M, int N, float eps,
                    int sms, cudaStream_t stream) {
  const int64_t cap = static_cast<int64_t>(sms) * 8;
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

// pointwise.cu -- the second kernels of the unfused reference compositions.
//
// Unfused, a product is written to HBM in bf16 and a separate kernel reads it
// back, applies the ending and writes the result again ("kernel fusion"
// wiki, the activation-after-matmul case; "Fusion Thinking", Pattern 2
// un-fused silu(gate)*up, and Pattern 3 un-fused dequantize-then-GEMM).  These
// kernels are that second pass.  They are HBM-bound: each thread moves
// 16-byte vectors, the grid is a multiple of the SM count and strides over the
// tensor.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace gbf {

namespace {

constexpr int kPwThreads = 256;

int pw_grid(int64_t vectors, int sms) {
  const int64_t want = (vectors + kPwThreads - 1) / kPwThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

// out = bf16(act(alpha*D + beta*C + bias) + residual); D == null -> 0.
template <int ACT>
__global__ void __launch_bounds__(kPwThreads)
    pointwise_epilogue_kernel(const __nv_bfloat16* __restrict__ D, const EpiParams e, int64_t M,
                              int64_t N) {
  const int64_t nvec = M * N / 8;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t off = v * 8;
    const int64_t col = off % N;
    float x[8];
    if (D) {
      unpack8(ldg_u4(D + off), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] *= e.alpha;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = 0.0f;
    }
    if (e.C) {
      float c[8];
      unpack8(ldg_u4(e.C + off), c);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = fmaf(e.beta, c[i], x[i]);
    }
    if (e.bias) {
      float b[8];
      unpack8(ldg_u4(e.bias + col), b);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] += b[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = act_apply<ACT>(x[i]);
    if (e.residual) {
      float r[8];
      unpack8(ld_u4(e.residual + off), r);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] += r[i];
    }
    st_u4(e.out + off, pack8(x));
  }
}

// h = bf16(act(alpha*g) * (alpha*u) + beta*C), g and u read as bf16.
template <int ACT>
__global__ void __launch_bounds__(kPwThreads)
    swiglu_pointwise_kernel(const __nv_bfloat16* __restrict__ g,
                            const __nv_bfloat16* __restrict__ u, const EpiParams e, int64_t M,
                            int64_t N) {
  const int64_t nvec = M * N / 8;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t off = v * 8;
    float gv[8], uv[8], x[8];
    unpack8(ldg_u4(g + off), gv);
    unpack8(ldg_u4(u + off), uv);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = act_apply<ACT>(e.alpha * gv[i]) * (e.alpha * uv[i]);
    if (e.C) {
      float c[8];
      unpack8(ldg_u4(e.C + off), c);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = fmaf(e.beta, c[i], x[i]);
    }
    st_u4(e.out + off, pack8(x));
  }
}

// w[k][n] = bf16((q - 8) * s[k/G][n]); byte j of row k holds column 2j in the
// high nibble, 2j+1 in the low nibble.  One thread: 4 bytes -> 8 columns.
// (q - 8) has 4 significant bits and s 8, so the fp32 product is exact and
// the conversion rounds it once.
__global__ void __launch_bounds__(kPwThreads)
    dequant_int4_kernel(const uint8_t* __restrict__ Wq, const __nv_bfloat16* __restrict__ s,
                        int group, int64_t K, int64_t N, __nv_bfloat16* __restrict__ w) {
  const int64_t words_per_row = N / 8;
  const int64_t nwords = K * words_per_row;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nwords;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = v / words_per_row;
    const int64_t n0 = (v % words_per_row) * 8;
    const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(Wq + k * (N / 2) + n0 / 2));
    float sc[8];
    unpack8(ldg_u4(s + (k / group) * N + n0), sc);
    float x[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (word >> (8 * b)) & 0xFFu;
      x[2 * b] = static_cast<float>(static_cast<int>(byte >> 4) - 8) * sc[2 * b];
      x[2 * b + 1] = static_cast<float>(static_cast<int>(byte & 0xFu) - 8) * sc[2 * b + 1];
    }
    st_u4(w + k * N + n0, pack8(x));
  }
}

// E4M3 byte -> float, exact: the sign and the 7 magnitude bits placed in a
// binary32 with the code's exponent field in the low exponent bits give the
// value times 2^-120 (subnormal codes land on binary32 subnormals with the
// same factor); one exact multiply by 2^120 restores it.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  const uint32_t bits = ((b & 0x80u) << 24) | ((b & 0x7Fu) << 20);
  return __uint_as_float(bits) * 0x1p120f;
}

// E2M1 code (low 4 bits) -> float, exact, the same way with factor 2^-126.
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
  const uint32_t bits = ((c & 0x8u) << 28) | ((c & 0x7u) << 22);
  return __uint_as_float(bits) * 0x1p126f;
}

// w[k][n] = bf16(e4m3(q[k][n]) * s[k/G][n]); the product is exact in fp32
// (4 x 8 significant bits), so packing rounds once.
__global__ void __launch_bounds__(kPwThreads)
    dequant_fp8_kernel(const uint8_t* __restrict__ Wq, const __nv_bfloat16* __restrict__ s,
                       int group, int64_t K, int64_t N, __nv_bfloat16* __restrict__ w) {
  const int64_t vecs_per_row = N / 8;
  const int64_t nvec = K * vecs_per_row;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = v / vecs_per_row;
    const int64_t n0 = (v % vecs_per_row) * 8;
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(Wq + k * N + n0));
    float sc[8];
    unpack8(ldg_u4(s + (k / group) * N + n0), sc);
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = e4m3_to_float((q.x >> (8 * i)) & 0xFFu) * sc[i];
      x[4 + i] = e4m3_to_float((q.y >> (8 * i)) & 0xFFu) * sc[4 + i];
    }
    st_u4(w + k * N + n0, pack8(x));
  }
}

// w[k][n] = e2m1(q[k][n]) * e4m3(S[k/16][n]), exact (at most 6 significant
// bits); codes packed two per byte along N, column 2j in the high nibble.
__global__ void __launch_bounds__(kPwThreads)
    dequant_nvfp4_kernel(const uint8_t* __restrict__ Wq, const uint8_t* __restrict__ S,
                         int64_t K, int64_t N, __nv_bfloat16* __restrict__ w) {
  const int64_t vecs_per_row = N / 8;
  const int64_t nvec = K * vecs_per_row;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < nvec;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = v / vecs_per_row;
    const int64_t n0 = (v % vecs_per_row) * 8;
    const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(Wq + k * (N / 2) + n0 / 2));
    const uint2 sb = __ldg(reinterpret_cast<const uint2*>(S + (k / 16) * N + n0));
    float x[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (word >> (8 * b)) & 0xFFu;
      const uint32_t sw = b < 2 ? sb.x : sb.y;
      const int sh = 16 * (b & 1);
      x[2 * b] = e2m1_to_float(byte >> 4) * e4m3_to_float((sw >> sh) & 0xFFu);
      x[2 * b + 1] = e2m1_to_float(byte & 0xFu) * e4m3_to_float((sw >> (sh + 8)) & 0xFFu);
    }
    st_u4(w + k * N + n0, pack8(x));
  }
}

cudaError_t launch_dequant_fp8(const uint8_t* Wq, const __nv_bfloat16* scales, int group,
                               int64_t K, int64_t N, __nv_bfloat16* w, int sms,
                               cudaStream_t stream) {
  dequant_fp8_kernel<<<pw_grid(K * N / 8, sms), kPwThreads, 0, stream>>>(Wq, scales, group, K,
                                                                          N, w);
  return cudaGetLastError();
}

cudaError_t launch_dequant_nvfp4(const uint8_t* Wq, const uint8_t* scales, int64_t K, int64_t N,
                                 __nv_bfloat16* w, int sms, cudaStream_t stream) {
  dequant_nvfp4_kernel<<<pw_grid(K * N / 8, sms), kPwThreads, 0, stream>>>(Wq, scales, K, N, w);
  return cudaGetLastError();
}

cudaError_t launch_pointwise_epilogue(const __nv_bfloat16* D, const EpiParams& ep, int64_t M,
                                      int64_t N, int sms, cudaStream_t stream) {
  const int grid = pw_grid(M * N / 8, sms);
  switch (ep.act) {
    case kActRelu:
      pointwise_epilogue_kernel<kActRelu><<<grid, kPwThreads, 0, stream>>>(D, ep, M, N);
      break;
    case kActSilu:
      pointwise_epilogue_kernel<kActSilu><<<grid, kPwThreads, 0, stream>>>(D, ep, M, N);
      break;
    case kActGeluTanh:
      pointwise_epilogue_kernel<kActGeluTanh><<<grid, kPwThreads, 0, stream>>>(D, ep, M, N);
      break;
    default:
      pointwise_epilogue_kernel<kActIdentity><<<grid, kPwThreads, 0, stream>>>(D, ep, M, N);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_swiglu_pointwise(const __nv_bfloat16* g, const __nv_bfloat16* u,
                                    const EpiParams& ep, int64_t M, int64_t N, int sms,
                                    cudaStream_t stream) {
  const int grid = pw_grid(M * N / 8, sms);
  switch (ep.act) {
    case kActRelu:
      swiglu_pointwise_kernel<kActRelu><<<grid, kPwThreads, 0, stream>>>(g, u, ep, M, N);
      break;
    case kActSilu:
      swiglu_pointwise_kernel<kActSilu><<<grid, kPwThreads, 0, stream>>>(g, u, ep, M, N);
      break;
    case kActGeluTanh:
      swiglu_pointwise_kernel<kActGeluTanh><<<grid, kPwThreads, 0, stream>>>(g, u, ep, M, N);
      break;
    default:
      swiglu_pointwise_kernel<kActIdentity><<<grid, kPwThreads, 0, stream>>>(g, u, ep, M, N);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_int4(const uint8_t* Wq, const __nv_bfloat16* scales, int group,
                                int64_t K, int64_t N, __nv_bfloat16* w, int sms,
                                cudaStream_t stream) {
  const int grid = pw_grid(K * N / 8, sms);
  dequant_int4_kernel<<<grid, kPwThreads, 0, stream>>>(Wq, scales, group, K, N, w);
  return cudaGetLastError();
}

}  // namespace gbf

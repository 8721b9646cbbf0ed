// common.cuh -- device-side pieces shared by the kernels: bounded waits that
// record a timeout instead of hanging, the fused epilogue arithmetic, and
// bf16 packing helpers.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace gbf {

// Status values written to the device error word (low byte); bits 8..15 say
// where the wait gave up.  Must agree with gbfuse.h.
constexpr unsigned kDevErrTimeout = 6;

enum WaitSite : unsigned {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteEpiAccFull = 4,
  kSiteDrain = 5,
  kSiteXformFull = 6,
  kSiteXformEmpty = 7,
  kSiteMmaOperand = 8,
};

// Per-launch control shared by every role of a CTA.
struct WaitCtl {
  unsigned* err;          // device error word (global)
  uint64_t timeout_ns;    // limit of one wait
  volatile int* abort;    // shared flag: some role of this CTA gave up
  unsigned long long* prof = nullptr;  // this CTA's wait counters, or null
};

// Wait-time profiling (off unless a buffer is registered): lane 0 of each
// waiting warp adds the cycles it spent in a wait to its site's counter.
__device__ __forceinline__ unsigned long long* prof_slots(unsigned long long* prof) {
  if (!prof) return nullptr;
  const unsigned bid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  return prof + static_cast<size_t>(bid) * 32;
}

// Wait until phase `parity` of `bar` has completed, for at most
// ctl.timeout_ns.  On expiry, records the site in the error word, raises the
// CTA's abort flag and returns false.  With honor_abort, returns false as
// soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait_bar_impl(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                              unsigned site, bool honor_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  // The clock and the abort flag are checked every 64 polls only, so that a
  // waiting warp spends its issue slots on try_wait (which suspends the warp
  // for a while) rather than on bookkeeping.
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (honor_abort && *ctl.abort) return false;
      if (globaltimer_ns() - t0 > ctl.timeout_ns) {
        atomicCAS(ctl.err, 0u, kDevErrTimeout | (site << 8));
        *ctl.abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                         unsigned site, bool honor_abort = true) {
  if (!ctl.prof) return wait_bar_impl(bar, parity, ctl, site, honor_abort);
  const long long c0 = clock64();
  const bool ok = wait_bar_impl(bar, parity, ctl, site, honor_abort);
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&ctl.prof[2 * site], static_cast<unsigned long long>(clock64() - c0));
    atomicAdd(&ctl.prof[2 * site + 1], 1ull);
  }
  return ok;
}

// ---------------------------------------------------------------- epilogue math

enum { kActIdentity = 0, kActRelu = 1, kActSilu = 2, kActGeluTanh = 3 };

// Activations in fp32.  SiLU(v) = v * sigmoid(v).  tanh-GELU uses the exact
// identity 0.5 v (1 + tanh z) = v * sigmoid(2 z), z = sqrt(2/pi)(v + 0.044715 v^3),
// which stays accurate where 1 + tanh z cancels (large negative v).
template <int ACT>
__device__ __forceinline__ float act_apply(float v) {
  if constexpr (ACT == kActRelu) {
    return fmaxf(v, 0.0f);
  } else if constexpr (ACT == kActSilu) {
    // approximate reciprocal (a few ulp of fp32, far below bf16's rounding);
    // 1/inf = 0 keeps large negative v at -0
    return v * __fdividef(1.0f, 1.0f + __expf(-v));
  } else if constexpr (ACT == kActGeluTanh) {
    const float z = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
    return v * __fdividef(1.0f, 1.0f + __expf(-2.0f * z));
  } else {
    return v;
  }
}

// ---------------------------------------------------------------- bf16 helpers

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x);
  f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z);
  f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint4 ldg_u4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 ld_u4(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void st_u4(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Streaming accesses of the ending's operands and results: they are touched
// once, so they are marked evict-first in L2 and do not push the GEMM's
// operand panels out.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_stream_u4(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_stream_u4(void* ptr, const uint4& v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint16_t ld_stream_u16(const void* ptr, uint64_t pol) {
  uint16_t v;
  asm volatile("ld.global.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_stream_u16(void* ptr, uint16_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u16 [%0], %1, %2;" ::"l"(ptr), "h"(v), "l"(pol)
               : "memory");
}
__device__ __forceinline__ float bf16bits_to_f(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f_to_bf16bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float ld_bf16f(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

}  // namespace gbf

// noalloc.cu -- gemm_epilogue_unfused_noalloc: the unfused GEMM + pointwise
// composition with its bf16 intermediate held in a scratch array that is
// built into the library, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not
// allowed -- a plugin or callback inside a host framework that owns all
// device memory, a process under a memory policy that forbids new device
// allocations after start-up, or a caller that has no allocator of its own.
// Such a caller still passes its inputs and output, but cannot hand over a
// workspace.
//
// The scratch is a file-scope __device__ array of kNoAllocMaxElems bf16
// elements (8 MiB).  Every GPU that loads this library holds it until the
// process exits.  In host code its name is only a host-side stand-in, so the
// device address is looked up with cudaGetSymbolAddress once per device, on
// the first call made while that device is current; that first call should
// therefore come before any stream capture.  A lookup that fails is not
// remembered: the call returns GBF_ERR_CUDA and the next call tries again.
//
// All calls share the one array and it keeps the last call's contents.
// Nothing in it has to start at zero: the GEMM writes every element of the
// M x N intermediate before the pointwise pass reads it.  Calls whose work
// overlaps on the GPU (different streams, or several host threads) race on
// the array and must be serialised by the caller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/gbfuse.h"
#include "internal.h"

namespace {

constexpr int64_t kNoAllocMaxElems = int64_t(1) << 22;  // 4,194,304 bf16 = 8 MiB
constexpr size_t kNoAllocBytes = static_cast<size_t>(kNoAllocMaxElems) * 2;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) __nv_bfloat16 g_noalloc_scratch[kNoAllocMaxElems];

struct ScratchSlot {
  std::mutex mu;
  std::atomic<void*> ptr{nullptr};
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the scratch array on the current device (null on failure).
void* scratch_address(int dev) {
  ScratchSlot& slot = g_slots[dev];
  void* p = slot.ptr.load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(slot.mu);
  p = slot.ptr.load(std::memory_order_relaxed);
  if (p) return p;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();  // not sticky: leave no error behind for the caller
    return nullptr;
  }
  slot.ptr.store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" gbf_status_t gemm_epilogue_unfused_noalloc(
    const void* A, const void* B, int b_layout, const void* C, const void* bias,
    const void* residual, void* out, int64_t M, int64_t N, int64_t K, float alpha, float beta,
    int act, gbf_stream_t stream) {
  // the same argument checks, in the same order, as the workspace entry point;
  // the size limit takes the place of its workspace check
  const gbf_status_t st = gbf::check_gemm_call(A, B, b_layout, C, bias, residual, out, M, N, K, act);
  if (st != GBF_OK) return st;
  if (M != 0 && N > kNoAllocMaxElems / M) return GBF_ERR_WORKSPACE;  // M*N beyond the array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return GBF_ERR_NO_DEVICE;
  void* scratch = scratch_address(dev);
  if (!scratch) return GBF_ERR_CUDA;
  return gemm_epilogue_unfused(A, B, b_layout, C, bias, residual, out, M, N, K, alpha, beta, act,
                               scratch, kNoAllocBytes, stream);
}

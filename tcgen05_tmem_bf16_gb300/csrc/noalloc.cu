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
// therefore come before any stream capture.
//
// All calls share the one array and it keeps the last call's contents.
// Nothing in it has to start at zero: the GEMM writes every element of the
// M x N intermediate before the pointwise pass reads it.  Calls whose work
// overlaps on the GPU (different streams, or several host threads) race on
// the array and must be serialised by the caller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gbfuse.h"

namespace {

constexpr int64_t kNoAllocMaxElems = int64_t(1) << 22;  // 4,194,304 bf16 = 8 MiB
constexpr size_t kNoAllocBytes = static_cast<size_t>(kNoAllocMaxElems) * 2;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) __nv_bfloat16 g_noalloc_scratch[kNoAllocMaxElems];

struct ScratchSlot {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t status = cudaSuccess;
};
ScratchSlot g_slots[kMaxDevices];

}  // namespace

extern "C" gbf_status_t gemm_epilogue_unfused_noalloc(
    const void* A, const void* B, int b_layout, const void* C, const void* bias,
    const void* residual, void* out, int64_t M, int64_t N, int64_t K, float alpha, float beta,
    int act, gbf_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return GBF_ERR_INVALID_ARG;
  if (M != 0 && N > kNoAllocMaxElems / M) return GBF_ERR_WORKSPACE;  // M*N beyond the array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return GBF_ERR_NO_DEVICE;
  ScratchSlot& slot = g_slots[dev];
  std::call_once(slot.once, [&slot]() {
    slot.status = cudaGetSymbolAddress(&slot.ptr, g_noalloc_scratch);
  });
  if (slot.status != cudaSuccess || slot.ptr == nullptr) return GBF_ERR_CUDA;
  return gemm_epilogue_unfused(A, B, b_layout, C, bias, residual, out, M, N, K, alpha, beta, act,
                               slot.ptr, kNoAllocBytes, stream);
}

// lmhead_argmax_verify_noalloc: the LM-head verify step with the library's own scratch in place
// of a caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is one file-scope __device__ array (512 bytes, the size of the verify workspace);
// every device that loads the library holds its own copy.  Its address is looked up once per
// device with cudaGetSymbolAddress.  Every call clears the scratch on the caller's stream and
// then hands it to lmhead_argmax_verify_path with the library's default kernel choice, so the
// validation, the kernel and the rounding are exactly those of lmhead_argmax_verify (the
// kernel leaves the scratch zeroed again).  Nothing here allocates.
#include <atomic>

#include "common.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

constexpr size_t kNoallocScratchBytes = 512;
static_assert(sizeof(LmheadWorkspace) <= kNoallocScratchBytes, "verify workspace exceeds the scratch");

static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of the scratch per device; two host threads making their first call on one
// device at once both store the same value.
std::atomic<void*> g_scratch_ptr[kMaxDevices];

}  // namespace
}  // namespace lowbit

using namespace lowbit;

extern "C" lowbit_status lmhead_argmax_verify_noalloc(const uint16_t* H, const void* packed_head,
                                                      int M, int N, int K, const int32_t* draft,
                                                      int32_t* argmax, int32_t* n_accept,
                                                      int32_t* bonus, void* stream) {
  // Shapes the workspace entry point accepts but whose workspace would not fit the scratch.
  if (lmhead_workspace_bytes(M, N, K) > kNoallocScratchBytes) return LOWBIT_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LOWBIT_ERR_CUDA;
  void* scratch = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!scratch) {  // first call on this device: find the scratch
    if (cudaGetSymbolAddress(&scratch, g_lmhead_scratch) != cudaSuccess || !scratch) return LOWBIT_ERR_CUDA;
    g_scratch_ptr[dev].store(scratch, std::memory_order_relaxed);
  }
  // The workspace entry point's own validation, before anything is enqueued.
  const lowbit_status st = check_lmhead_args(H, packed_head, M, N, K, draft, argmax, n_accept, bonus,
                                             scratch, kNoallocScratchBytes);
  if (st != LOWBIT_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel leaves the scratch zeroed, but a call that failed on the device may not have.
  if (cudaMemsetAsync(scratch, 0, kNoallocScratchBytes, s) != cudaSuccess) return LOWBIT_ERR_CUDA;
  return lmhead_argmax_verify_path(H, packed_head, M, N, K, draft, argmax, n_accept, bonus, scratch,
                                   kNoallocScratchBytes, 0, stream);
}

// lmhead_argmax_verify_noalloc: the LM-head verify step with the library's own scratch in place
// of a caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is one file-scope __device__ array per device (512 bytes, the size of the verify
// workspace).  Its address is looked up once per device with cudaGetSymbolAddress; every call
// clears it on the caller's stream and then runs the same tensor-core kernel as
// lmhead_argmax_verify, which leaves it zeroed again.  Nothing here allocates.
#include "common.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

constexpr size_t kNoallocScratchBytes = 512;
static_assert(sizeof(LmheadWorkspace) <= kNoallocScratchBytes, "verify workspace exceeds the scratch");

static __device__ __align__(256) unsigned char g_lmhead_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

inline bool is_aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace lowbit

using namespace lowbit;

extern "C" lowbit_status lmhead_argmax_verify_noalloc(const uint16_t* H, const void* packed_head,
                                                      int M, int N, int K, const int32_t* draft,
                                                      int32_t* argmax, int32_t* n_accept,
                                                      int32_t* bonus, void* stream) {
  if (!H || !packed_head || !draft || !argmax || !n_accept || !bonus) return LOWBIT_ERR_INVALID_ARG;
  if (K <= 0 || K % kGroup != 0 || K > 65536 || N < 1 || M < 2 || M > 32) return LOWBIT_ERR_SHAPE;
  const size_t need = lmhead_workspace_bytes(M, N, K);
  if (need == 0 || need > kNoallocScratchBytes) return LOWBIT_ERR_WORKSPACE;
  if (!is_aligned16(H) || !is_aligned16(packed_head)) return LOWBIT_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LOWBIT_ERR_CUDA;
  if (!g_scratch_ptr[dev]) {  // first call on this device: find the scratch
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_scratch) != cudaSuccess || !p) return LOWBIT_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel leaves the scratch zeroed, but a call that failed on the device may not have.
  if (cudaMemsetAsync(g_scratch_ptr[dev], 0, need, s) != cudaSuccess) return LOWBIT_ERR_CUDA;
  const cudaError_t e = launch_lmhead_tc(H, static_cast<const uint8_t*>(packed_head), M, N, K, draft,
                                         argmax, n_accept, bonus, g_scratch_ptr[dev], err, s);
  return e == cudaSuccess ? LOWBIT_OK : LOWBIT_ERR_CUDA;
}

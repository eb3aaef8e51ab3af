// A row-sharded LM head for verification across GPUs (small-vocabulary MTP study, section 3.3:
// drafts are verified against the full vocabulary; DFlash summary, section 4.1: greedy prefix
// acceptance).  Each GPU holds a contiguous slice of the vocabulary's rows, scores its slice
// (lmhead_argmax_partial, the verify kernel with a per-shard epilogue) and emits one 64-bit key
// per token: the logit's order-preserving bits and the row's global index, so that the larger
// key is the larger logit and, among equal logits, the lower row.  After the caller has
// gathered every shard's keys (one all-gather of W * M * 8 bytes), lmhead_accept_keys takes the
// maximum key per token -- the full head's argmax with the lowest index on ties -- and applies
// the prefix rule, identically on every GPU.
#include "common.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

__global__ void accept_keys_kernel(const unsigned long long* __restrict__ keys, int W, int M,
                                   const int32_t* __restrict__ draft, int32_t* __restrict__ argmax,
                                   int32_t* __restrict__ n_accept, int32_t* __restrict__ bonus) {
  __shared__ int win[32];
  const int m = threadIdx.x;
  if (m < M) {
    unsigned long long best = 0ull;
    for (int w = 0; w < W; ++w) {
      const unsigned long long k = keys[(size_t)w * M + m];
      best = k > best ? k : best;
    }
    win[m] = argmax_key_row(best);
    argmax[m] = win[m];
  }
  __syncthreads();
  if (m == 0) {
    int n = 0;
    while (n < M - 1 && draft[n] == win[n]) ++n;
    *n_accept = n;
    *bonus = win[n];
  }
}

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace lowbit

using namespace lowbit;

extern "C" {

lowbit_status lmhead_argmax_partial(const uint16_t* H, const void* packed_shard, int M, int N, int K,
                                    int row_offset, uint64_t* keys_out, void* workspace,
                                    size_t ws_bytes, void* stream) {
  if (!H || !packed_shard || !keys_out || row_offset < 0) return LOWBIT_ERR_INVALID_ARG;
  if (K <= 0 || K % kGroup != 0 || K > 65536 || N < 1 || M < 1 || M > 32) return LOWBIT_ERR_SHAPE;
  if ((long long)row_offset + N > 0x7FFFFFFFLL) return LOWBIT_ERR_SHAPE;
  if (!workspace || ws_bytes < lmhead_workspace_bytes(2, N, K)) return LOWBIT_ERR_WORKSPACE;
  if (!aligned(H, 16) || !aligned(packed_shard, 16) || !aligned(workspace, 16) || !aligned(keys_out, 8))
    return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed_shard);
  GemvProblem p = {H, pk, nullptr, N, K, 0, 1, 0, 0};
  p.early = allocation_covers(pk, kHeaderBytes + int4_payload_bytes(N, K)) ? 1 : 0;
  const cudaError_t e =
      launch_lmhead_keys_mma(p, M, static_cast<LmheadWorkspace*>(workspace), row_offset,
                             reinterpret_cast<unsigned long long*>(keys_out), err,
                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LOWBIT_OK : LOWBIT_ERR_CUDA;
}

lowbit_status lmhead_accept_keys(const uint64_t* keys, int W, int M, const int32_t* draft,
                                 int32_t* argmax, int32_t* n_accept, int32_t* bonus, void* stream) {
  if (!keys || !draft || !argmax || !n_accept || !bonus || W < 1) return LOWBIT_ERR_INVALID_ARG;
  if (M < 2 || M > 32) return LOWBIT_ERR_SHAPE;
  if (!aligned(keys, 8)) return LOWBIT_ERR_ALIGN;
  accept_keys_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const unsigned long long*>(keys), W, M, draft, argmax, n_accept, bonus);
  return cudaGetLastError() == cudaSuccess ? LOWBIT_OK : LOWBIT_ERR_CUDA;
}

}  // extern "C"

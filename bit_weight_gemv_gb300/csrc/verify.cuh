// Vocabulary argmax and greedy prefix acceptance, fused into the LM-head multiply.
//
// Small-vocabulary MTP study, section 3.3: drafts are verified against the full vocabulary,
// so outputs stay exact.  DFlash summary, section 4.1: a step accepts tau in [1, gamma+1]
// tokens; section 6 item 2: the drafter conditions on the last target-verified ("bonus")
// token.  Efficient-Qwen report, section 2.2: the target verifies the drafts in parallel.
//
// Reduction scheme (no spin-waits): each CTA reduces its rows to one (logit, row) key per
// token and folds it into a 64-bit atomicMax; the last CTA to finish (an atomic counter)
// reads the winners, applies the prefix rule and zeroes the workspace for the next call.
#pragma once

#include "common.cuh"

namespace lowbit {

struct LmheadWorkspace {
  unsigned long long keys[32];  // per token: order-preserving logit bits << 32 | ~row
  // CTAs that have folded in their keys (bits 0..30); bit 31 is set by any CTA whose logits
  // are incomplete (a wait gave up), before it counts itself.
  unsigned int counter;
  unsigned int pad[63];
};
static_assert(sizeof(LmheadWorkspace) == 512, "workspace layout");
constexpr unsigned int kFailedBit = 0x80000000u;

// Called once per CTA (thread 0): counts this CTA; returns whether it is the last one, and in
// *failed whether any CTA (this one included) reported incomplete logits.  A failing CTA's
// OR precedes its own increment on the same word, so the last increment sees every flag.
__device__ __forceinline__ bool finish_count(LmheadWorkspace* ws, bool my_failed, int* failed) {
  const unsigned int total = gridDim.x * gridDim.y * gridDim.z;
  if (my_failed) atomicOr(&ws->counter, kFailedBit);
  const unsigned int old = atomicAdd(&ws->counter, 1u);
  *failed = my_failed || (old & kFailedBit) != 0u;
  return (old & ~kFailedBit) + 1u == total;
}

// Larger key <=> larger logit; among equal logits, the lower row index wins.
__device__ __forceinline__ unsigned long long argmax_key(float v, int n) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

__device__ __forceinline__ int argmax_key_row(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, k, o);
    k = other > k ? other : k;
  }
  return k;
}

// Called by every thread of every CTA once the CTA's atomicMax calls have been issued.
// The last CTA writes argmax[0..M), n_accept, bonus and resets the workspace.
__device__ __forceinline__ void lmhead_finish(LmheadWorkspace* ws, int M,
                                              const int32_t* __restrict__ draft,
                                              int32_t* __restrict__ argmax,
                                              int32_t* __restrict__ n_accept,
                                              int32_t* __restrict__ bonus, bool my_failed = false) {
  __shared__ int is_last;
  __shared__ int win[32];
  __shared__ int failed_s;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = finish_count(ws, my_failed, &failed_s);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // A failed call writes no output; either way the workspace is left zeroed.
  const bool failed = failed_s != 0;
  if (threadIdx.x < M) {
    const int a = argmax_key_row(atomicExch(&ws->keys[threadIdx.x], 0ull));
    win[threadIdx.x] = a;
    if (!failed) argmax[threadIdx.x] = a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!failed) {
      int n = 0;
      while (n < M - 1 && draft[n] == win[n]) ++n;
      *n_accept = n;
      *bonus = win[n];
    }
    atomicExch(&ws->counter, 0u);
  }
}

// The finish of one shard of a row-sharded LM head: the last CTA writes the shard's best key
// per token (logit bits and global row, as argmax_key) to keys_out and resets the workspace;
// a failed call writes nothing.  Merging the shards' keys with a maximum gives the full head's
// argmax, lowest row on ties (lmhead_accept_keys).
__device__ __forceinline__ void keys_finish(LmheadWorkspace* ws, int M,
                                            unsigned long long* __restrict__ keys_out,
                                            bool my_failed = false) {
  __shared__ int is_last_k;
  __shared__ int failed_k;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last_k = finish_count(ws, my_failed, &failed_k);
  __syncthreads();
  if (!is_last_k) return;
  __threadfence();
  if (threadIdx.x < M) {
    const unsigned long long k = atomicExch(&ws->keys[threadIdx.x], 0ull);
    if (!failed_k) keys_out[threadIdx.x] = k;
  }
  __syncthreads();
  if (threadIdx.x == 0) atomicExch(&ws->counter, 0u);
}

// The draft head's finish (small-vocabulary MTP study, section 3.3: a trimmed head's rows are
// mapped back to full-vocabulary ids): the last CTA writes ids[t] = id_map[winner] (the
// winning row itself when id_map is null) and resets the workspace.
__device__ __forceinline__ void draft_finish(LmheadWorkspace* ws, int M,
                                             const int32_t* __restrict__ id_map,
                                             int32_t* __restrict__ ids, bool my_failed = false) {
  __shared__ int is_last_d;
  __shared__ int failed_d;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last_d = finish_count(ws, my_failed, &failed_d);
  __syncthreads();
  if (!is_last_d) return;
  __threadfence();
  if (threadIdx.x < M) {
    const int row = argmax_key_row(atomicExch(&ws->keys[threadIdx.x], 0ull));
    if (!failed_d) ids[threadIdx.x] = id_map ? id_map[row] : row;  // a failed call writes nothing
  }
  __syncthreads();
  if (threadIdx.x == 0) atomicExch(&ws->counter, 0u);
}

}  // namespace lowbit

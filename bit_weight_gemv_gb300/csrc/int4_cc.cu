// INT4 weight-only multiply on the CUDA cores for several tokens (M >= 2), and the
// CUDA-core variant of the fused LM-head argmax.  (M = 1 is the streaming kernel.)
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} q[n][k] * x[m][k]
// (Efficient-Qwen report, section 2.1: W = s (.) W_q with frozen symmetric per-group scales,
// group 128, W4A16 serving.)
//
// Work split: one CTA per 32 weight rows (a quarter of a 128-row layout tile); its warps split
// the K/128 groups; lane r of every warp owns weight row 32*cta + r.  A warp's load of one
// 32-input chunk is one contiguous 512-byte segment of the tile's block (16 bytes per lane),
// so every weight byte is read once with fully coalesced 128-bit loads.  Dequantisation happens in registers: a nibble ORed
// into bf16 128.0 is the exact value 128 + u (u = q + 8), multiplied with the bf16
// activation by a mixed-precision fma into fp32.  Per group the bias is removed with the
// group's activation sum:  sum (128+u) x - 136 sum x = sum q x.  Warp partial sums are
// reduced through shared memory and each output is rounded once to bf16.
#include "common.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// The K dimension is walked in segments of SEG groups whose activations [M][SEG*128] are
// staged in shared memory; within a segment the warps split the groups.  Each lane keeps
// MT fp32 partial sums (one per token) for its row.
template <int MT>
struct SegCfg {
  static constexpr int kSeg = (MT <= 4) ? 16 : (MT <= 8 ? 8 : (MT <= 16 ? 8 : 4));
};

// With ARGMAX the logits are not stored: each token's best (logit, row) of the tile is folded
// into the workspace and the last CTA applies greedy prefix acceptance (verify.cuh).
template <int MT, bool ARGMAX>
__global__ void __launch_bounds__(kThreads)
int4_gemm_cc_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, int M,
                    int N, int K, uint16_t* __restrict__ Y, int* __restrict__ err,
                    LmheadWorkspace* __restrict__ ws, const int32_t* __restrict__ draft,
                    int32_t* __restrict__ argmax, int32_t* __restrict__ n_accept,
                    int32_t* __restrict__ bonus) {
  constexpr int SEG = SegCfg<MT>::kSeg;
  __shared__ __align__(16) uint16_t xs[MT * SEG * kGroup];
  __shared__ float gsum[MT * SEG];
  __shared__ float red[kWarps * 32 * (MT < 8 ? MT : 8)];
  __shared__ int ok;
  const int G = K / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;  // 32-row unit: layout tile blockIdx.x / 4, quarter blockIdx.x % 4

  if (threadIdx.x == 0)
    ok = header_matches(reinterpret_cast<const PackedHeader*>(packed), kFormatInt4, 0, N, K);
  __syncthreads();
  if (!ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, LOWBIT_ERR_INVALID_ARG);
    return;
  }
  const int rit = (tile & 3) * 32 + lane;
  const uint8_t* tbase = packed + kHeaderBytes + (size_t)(tile >> 2) * G * kInt4Block;

  float total[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) total[t] = 0.f;

  for (int s0 = 0; s0 < G; s0 += SEG) {
    const int sg = min(SEG, G - s0);
    __syncthreads();
    // stage X[:, 128*s0 .. 128*(s0+sg)) for the live tokens (zero rows beyond M)
    const int vec_per_row = sg * kGroup / 8;
    for (int i = threadIdx.x; i < MT * vec_per_row; i += kThreads) {
      const int t = i / vec_per_row, v = i % vec_per_row;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (t < M) val = __ldg(reinterpret_cast<const uint4*>(X + (size_t)t * K + (size_t)s0 * kGroup) + v);
      reinterpret_cast<uint4*>(xs + t * SEG * kGroup)[v] = val;
    }
    __syncthreads();
    for (int i = warp; i < MT * sg; i += kWarps) {
      const int t = i / sg, g = i % sg;
      const uint2 v = reinterpret_cast<const uint2*>(xs + t * SEG * kGroup + g * kGroup)[lane];
      float s = bf16_bits_to_float(v.x & 0xFFFF) + bf16_bits_to_float(v.x >> 16) +
                bf16_bits_to_float(v.y & 0xFFFF) + bf16_bits_to_float(v.y >> 16);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
      if (lane == 0) gsum[t * SEG + g] = s;
    }
    __syncthreads();
    for (int gl = warp; gl < sg; gl += kWarps) {
      const int g = s0 + gl;
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = ld_stream(reinterpret_cast<const uint4*>(tbase + (size_t)g * kInt4Block +
                                                        j * (kRowTile * 16) + rit * 16));
      const float sc = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(
          tbase + (size_t)g * kInt4Block + kInt4ScaleOff + rit * 2)));
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w4[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t q0 = int4_pair_biased<0>(w4[i]), q1 = int4_pair_biased<1>(w4[i]);
          const uint32_t q2 = int4_pair_biased<2>(w4[i]), q3 = int4_pair_biased<3>(w4[i]);
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const uint4 xp = *reinterpret_cast<const uint4*>(
                xs + t * SEG * kGroup + gl * kGroup + 32 * j + 8 * i);
            float lo = 0.f, hi = 0.f;
            fma_bf16x2_f32(lo, hi, q0, xp.x);
            fma_bf16x2_f32(lo, hi, q1, xp.y);
            fma_bf16x2_f32(lo, hi, q2, xp.z);
            fma_bf16x2_f32(lo, hi, q3, xp.w);
            acc[t] += lo + hi;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t)
        total[t] = fmaf(sc, acc[t] - 136.f * gsum[t * SEG + gl], total[t]);
    }
  }
  // Cross-warp reduction, 8 tokens at a time through shared memory.
  constexpr int TB = MT < 8 ? MT : 8;
  const int n = tile * 32 + lane;
#pragma unroll
  for (int t0 = 0; t0 < MT; t0 += TB) {
    __syncthreads();
#pragma unroll
    for (int t = 0; t < TB; ++t) red[(t * kWarps + warp) * 32 + lane] = total[t0 + t];
    __syncthreads();
    for (int t = warp; t < TB; t += kWarps) {
      float y = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) y += red[(t * kWarps + w) * 32 + lane];
      if constexpr (ARGMAX) {
        const int tt = t0 + t;
        unsigned long long key = (n < N && tt < M) ? argmax_key(y, n) : 0ull;
        key = warp_max_u64(key);
        if (lane == 0 && tt < M) atomicMax(&ws->keys[tt], key);
      } else {
        if (n < N && t0 + t < M) Y[(size_t)(t0 + t) * N + n] = float_to_bf16_bits(y);
      }
    }
  }
  if constexpr (ARGMAX) lmhead_finish(ws, M, draft, argmax, n_accept, bonus);
}

template <int MT, bool ARGMAX = false>
cudaError_t launch_mt(const uint16_t* X, const uint8_t* packed, int M, int N, int K, uint16_t* Y,
                      int* err, cudaStream_t s, LmheadWorkspace* ws = nullptr,
                      const int32_t* draft = nullptr, int32_t* argmax = nullptr,
                      int32_t* n_accept = nullptr, int32_t* bonus = nullptr) {
  int4_gemm_cc_kernel<MT, ARGMAX><<<(unsigned)row_tiles(N) * 4, kThreads, 0, s>>>(
      X, packed, M, N, K, Y, err, ws, draft, argmax, n_accept, bonus);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_int4_gemm_cc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                                uint16_t* Y, int* err, cudaStream_t s) {
  if (M <= 2) return launch_mt<2>(X, packed, M, N, K, Y, err, s);
  if (M <= 4) return launch_mt<4>(X, packed, M, N, K, Y, err, s);
  if (M <= 8) return launch_mt<8>(X, packed, M, N, K, Y, err, s);
  if (M <= 16) return launch_mt<16>(X, packed, M, N, K, Y, err, s);
  return launch_mt<32>(X, packed, M, N, K, Y, err, s);
}

cudaError_t launch_lmhead_cc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                             const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                             int32_t* bonus, void* wsp, int* err, cudaStream_t s) {
  LmheadWorkspace* ws = reinterpret_cast<LmheadWorkspace*>(wsp);
  if (M <= 2) return launch_mt<2, true>(H, packed, M, N, K, nullptr, err, s, ws, draft, argmax, n_accept, bonus);
  if (M <= 4) return launch_mt<4, true>(H, packed, M, N, K, nullptr, err, s, ws, draft, argmax, n_accept, bonus);
  if (M <= 8) return launch_mt<8, true>(H, packed, M, N, K, nullptr, err, s, ws, draft, argmax, n_accept, bonus);
  if (M <= 16) return launch_mt<16, true>(H, packed, M, N, K, nullptr, err, s, ws, draft, argmax, n_accept, bonus);
  return launch_mt<32, true>(H, packed, M, N, K, nullptr, err, s, ws, draft, argmax, n_accept, bonus);
}

}  // namespace lowbit

// INT4 weight-only multiply on the CUDA cores.
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
#include "ptx.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// ---------------------------------------------------------------------------------- M = 1
// Streaming GEMV.  CTA = 32 weight rows (one quarter of a 128-row tile) x a K range; its 4 warps
// split the range's groups and a thread-block cluster along K splits it further when there are
// too few row quarters to fill the GPU (partial sums meet in distributed shared memory).
//
// Dequantisation is exact fp32 arithmetic with packed (f32x2) instructions: a nibble at bit
// 4i of a code word, ORed into the fp32 pattern of 2^23, is 2^23 + u * 16^i; subtracting
// 2^23 + 8 * 16^i leaves q * 16^i, and the activation is pre-scaled by 16^-i in shared memory
// (a power of two, exact), so each fma adds q * x exactly before its single rounding.  Five
// of the eight nibbles of a word sit at bits 0..19 and need no shift; the other three are
// read from the word shifted right by 12.
constexpr int kGemvWarps = 4;
constexpr int kGemvThreads = kGemvWarps * 32;

__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  return ((uint64_t)hi << 32) | lo;
}
// Consumption order of the 8 inputs of a word (k offsets within the 8) and their 16^i scales.
__device__ __constant__ int kGemvKoff[8] = {0, 2, 4, 6, 1, 3, 5, 7};
__device__ __constant__ float kGemvInvScale[8] = {1.f, 1.f / 16, 1.f / 256, 1.f / 4096,
                                                  1.f / 65536, 1.f / 256, 1.f / 4096, 1.f / 65536};

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Accumulate one 8-input word into four f32x2 accumulators; xp points at its 8 scaled inputs.
__device__ __forceinline__ void gemv_word(uint32_t w, const float4* xp, uint64_t (&acc)[4]) {
  constexpr uint32_t M = 0x4B000000u;  // 2^23
  const uint32_t w2 = w >> 12;
  const uint32_t v0 = (w & 0x0000Fu) | M, v1 = (w & 0x000F0u) | M;
  const uint32_t v2 = (w & 0x00F00u) | M, v3 = (w & 0x0F000u) | M;
  const uint32_t v4 = (w & 0xF0000u) | M, v5 = (w2 & 0x00F00u) | M;
  const uint32_t v6 = (w2 & 0x0F000u) | M, v7 = (w2 & 0xF0000u) | M;
  // -(2^23 + 8 * scale) for scales (1, 16), (256, 4096), (65536, 256), (4096, 65536)
  constexpr uint64_t B01 = ((uint64_t)0xCB000080u << 32) | 0xCB000008u;
  constexpr uint64_t B23 = ((uint64_t)0xCB008000u << 32) | 0xCB000800u;
  constexpr uint64_t B45 = ((uint64_t)0xCB000800u << 32) | 0xCB080000u;
  constexpr uint64_t B67 = ((uint64_t)0xCB080000u << 32) | 0xCB008000u;
  const float4 xa = xp[0], xb = xp[1];
  acc[0] = f32x2_fma(f32x2_add(pack2(v0, v1), B01), pack2(__float_as_uint(xa.x), __float_as_uint(xa.y)), acc[0]);
  acc[1] = f32x2_fma(f32x2_add(pack2(v2, v3), B23), pack2(__float_as_uint(xa.z), __float_as_uint(xa.w)), acc[1]);
  acc[2] = f32x2_fma(f32x2_add(pack2(v4, v5), B45), pack2(__float_as_uint(xb.x), __float_as_uint(xb.y)), acc[2]);
  acc[3] = f32x2_fma(f32x2_add(pack2(v6, v7), B67), pack2(__float_as_uint(xb.z), __float_as_uint(xb.w)), acc[3]);
}

__global__ void __launch_bounds__(kGemvThreads)
int4_gemv_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, int N, int K,
                 int groups_per_rank, uint16_t* __restrict__ Y, int* __restrict__ err) {
  extern __shared__ __align__(16) float xs[];  // scaled inputs of this CTA's K range
  __shared__ float red[kGemvWarps][32];
  __shared__ int ok;
  const int G = K / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x, ks = gridDim.x, qt = blockIdx.y;  // 32-row quarter tile
  const int g0 = min(G, rank * groups_per_rank), g1 = min(G, g0 + groups_per_rank);

  if (threadIdx.x == 0) {
    ok = header_matches(reinterpret_cast<const PackedHeader*>(packed), kFormatInt4, 0, N, K);
    grid_launch();
  }
  __syncthreads();
  const bool hdr_ok = ok != 0;
  if (!hdr_ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    record_error(err, LOWBIT_ERR_INVALID_ARG);

  const int rit = (qt & 3) * 32 + lane;
  const uint8_t* tbase = packed + kHeaderBytes + (size_t)(qt >> 2) * G * kInt4Block;
  auto codes_at = [&](int g, int c) {
    return reinterpret_cast<const uint4*>(tbase + (size_t)g * kInt4Block + c * (kRowTile * 16) + rit * 16);
  };
  auto scale_at = [&](int g) {
    return reinterpret_cast<const uint16_t*>(tbase + (size_t)g * kInt4Block + kInt4ScaleOff + rit * 2);
  };

  float total = 0.f;
  if (hdr_ok) {
    // Weights do not depend on the previous kernel: fetch the first group before waiting.
    int g = g0 + warp;
    uint4 cur[4];
    uint16_t cur_s = 0;
    if (g < g1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) cur[j] = ld_stream(codes_at(g, j));
      cur_s = __ldg(scale_at(g));
    }
    grid_wait();
    // Stage the scaled inputs of groups g0..g1 in consumption order.
    const int nk = (g1 - g0) * kGroup;
    const uint16_t* xg = X + (size_t)g0 * kGroup;
    for (int i = threadIdx.x; i < nk; i += kGemvThreads) {
      const int blk = i >> 3, j = i & 7;
      xs[i] = bf16_bits_to_float(xg[blk * 8 + kGemvKoff[j]]) * kGemvInvScale[j];
    }
    __syncthreads();
    for (; g < g1; g += kGemvWarps) {
      uint4 nxt[4];
      uint16_t nxt_s = 0;
      if (g + kGemvWarps < g1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) nxt[j] = ld_stream(codes_at(g + kGemvWarps, j));
        nxt_s = __ldg(scale_at(g + kGemvWarps));
      }
      uint64_t acc[4] = {0, 0, 0, 0};
      const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)(g - g0) * kGroup);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gemv_word(cur[j].x, xp + 8 * j + 0, acc);
        gemv_word(cur[j].y, xp + 8 * j + 2, acc);
        gemv_word(cur[j].z, xp + 8 * j + 4, acc);
        gemv_word(cur[j].w, xp + 8 * j + 6, acc);
      }
      float sum = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a)
        sum += __uint_as_float((uint32_t)acc[a]) + __uint_as_float((uint32_t)(acc[a] >> 32));
      total = fmaf(half_bits_to_float(cur_s), sum, total);
#pragma unroll
      for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
      cur_s = nxt_s;
    }
  } else {
    grid_wait();
  }
  red[warp][lane] = total;
  __syncthreads();
  float* part = xs;  // the CTA's partial sums for its 32 rows (reuses the input staging)
  if (warp == 0) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) y += red[w][lane];
    part[lane] = y;
  }
  if (ks > 1) {
    ptx::cluster_sync();
    if (hdr_ok && rank == 0 && warp == 0) {
      float y = 0.f;
      const uint32_t la = ptx::smem_addr(&part[lane]);
      for (int r = 0; r < ks; ++r) y += ptx::ld_dsmem_f32(la, r);
      const int n = qt * 32 + lane;
      if (n < N) Y[n] = float_to_bf16_bits(y);
    }
    ptx::cluster_sync();
  } else if (hdr_ok && warp == 0) {
    __syncwarp();
    const int n = qt * 32 + lane;
    if (n < N) Y[n] = float_to_bf16_bits(part[lane]);
  }
}

// ---------------------------------------------------------------------------- M tokens
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

cudaError_t launch_int4_gemv(const uint16_t* X, const uint8_t* packed, int N, int K, uint16_t* Y,
                             int* err, cudaStream_t s) {
  const int G = K / kGroup, NQ = row_tiles(N) * 4;
  int nsm = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  // Split K over a cluster until the grid holds about four CTAs per SM, keeping at least
  // eight groups per CTA (two per warp).
  int ks = 1;
  while (ks < 8 && NQ * ks < 4 * nsm && G / (ks * 2) >= 8) ks *= 2;
  // The staged inputs of a CTA's K range (4 bytes per input) must fit in shared memory.
  while (ks < 8 && (size_t)((G + ks - 1) / ks) * kGroup * sizeof(float) > 160 * 1024) ks *= 2;
  const int gpr = (G + ks - 1) / ks;
  const size_t smem = (size_t)gpr * kGroup * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(int4_gemv_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ks, (unsigned)NQ, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem < 128 ? 128 : smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)ks;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, int4_gemv_kernel, X, packed, N, K, gpr, Y, err);
}

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

// Binary-plane (ShiftAdd) weight multiply on the CUDA cores.
//
//   y[m][n] = sum_p sum_g alpha[p][n][g] * sum_{k in g} b[p][n][k] * x[m][k],  b in {-1,+1}
// (ShiftAddQwen README, introduction and "Method": a mat-vec is a sign-select-and-add per
// plane plus one scale per group).
//
// The SA instantiation reads the deployed ShiftAdd format (ShiftAddQwen README, "Format"): one
// block per (tile, super-block of 256 inputs), alpha = d * a with a u8 code a per (plane, group
// of G inputs) and one fp16 d per (row, super-block); its units of 128 inputs are the halves
// of a super-block.
//
// Same work split as the INT4 CUDA-core kernel: one CTA per 32 rows (a quarter of a 128-row
// layout tile), warps split the groups of a K segment, lane r owns row 32*cta + r and reads its
// 16 bytes of signs per (group, plane) as part of one contiguous 512-byte warp load.  The sign select is an XOR
// of the plane bit into the sign bit of the bf16 activation pair; the selected values are
// added into fp32 and scaled once per (plane, group).
#include "common.cuh"

namespace lowbit {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int MT>
struct BpSeg {
  static constexpr int kSeg = (MT <= 4) ? 16 : (MT <= 16 ? 8 : 4);
};

template <int MT, bool SA>
__global__ void __launch_bounds__(kThreads)
binplane_cc_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ packed, int P,
                   int GS, int M, int N, int K, uint16_t* __restrict__ Y, int* __restrict__ err) {
  constexpr int SEG = BpSeg<MT>::kSeg;
  __shared__ __align__(16) uint16_t xs[MT * SEG * kGroup];
  __shared__ float red[kWarps * 32 * (MT < 8 ? MT : 8)];
  __shared__ int ok;
  const int G = K / kGroup;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;  // 32-row unit: layout tile blockIdx.x / 4, quarter blockIdx.x % 4

  if (threadIdx.x == 0) {
    const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(packed);
    ok = SA ? header_matches_sa(hp, P, GS, N, K) : header_matches(hp, kFormatBinplane, P, N, K);
  }
  __syncthreads();
  if (!ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, LOWBIT_ERR_INVALID_ARG);
    return;
  }
  const int rit = (tile & 3) * 32 + lane;
  // units of 128 inputs; SA: unit g is half g % 2 of super-block g / 2
  const uint32_t BB = SA ? sa_block(P, GS) : binplane_block(P);
  const uint8_t* tbase = packed + kHeaderBytes + (size_t)(tile >> 2) * (SA ? G / 2 : G) * BB;

  float total[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) total[t] = 0.f;

  for (int s0 = 0; s0 < G; s0 += SEG) {
    const int sg = min(SEG, G - s0);
    __syncthreads();
    const int vec_per_row = sg * kGroup / 8;
    for (int i = threadIdx.x; i < MT * vec_per_row; i += kThreads) {
      const int t = i / vec_per_row, v = i % vec_per_row;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (t < M) val = __ldg(reinterpret_cast<const uint4*>(X + (size_t)t * K + (size_t)s0 * kGroup) + v);
      reinterpret_cast<uint4*>(xs + t * SEG * kGroup)[v] = val;
    }
    __syncthreads();
    for (int gl = warp; gl < sg; gl += kWarps) {
      const int g = s0 + gl;
      const uint8_t* blk = tbase + (size_t)(SA ? g / 2 : g) * BB;
      const int h = g & 1;
      float dsa = 0.f;
      if (SA) dsa = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(blk + sa_d_off(P, GS) + rit * 2)));
      for (int p = 0; p < P; ++p) {
        float a, a23;  // scale of words 0-1 and of words 2-3 of this unit
        uint4 wv;
        if (SA) {
          wv = ld_stream(reinterpret_cast<const uint4*>(blk + (p * 2 + h) * (kRowTile * 16) + rit * 16));
          const int GJ = kSuper / GS;
          const int g01 = GS == 64 ? 2 * h : (GS == 128 ? h : 0), g23 = GS == 64 ? 2 * h + 1 : g01;
          const uint8_t* ap = blk + sa_code_off(P) + (size_t)p * GJ * kRowTile + rit;
          a = dsa * (float)__ldg(ap + g01 * kRowTile);
          a23 = dsa * (float)__ldg(ap + g23 * kRowTile);
        } else {
          wv = ld_stream(reinterpret_cast<const uint4*>(blk + p * (kRowTile * 16) + rit * 16));
          a = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(
              blk + binplane_alpha_off(P) + (p * kRowTile + rit) * 2)));
          a23 = a;
        }
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (SA && j == 2 && GS == 64) {  // words 2-3 carry the next group's code
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              total[t] = fmaf(a, acc[t], total[t]);
              acc[t] = 0.f;
            }
            a = a23;
          }
          const uint32_t nw = ~w4[j];
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            uint32_t m[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 4 * i4 + e;       // pair i: inputs k0 + 2i (low) and k0 + 2i + 1 (high)
              m[e] = (nw << (15 - i)) & 0x80008000u;  // sign flip where the plane bit is 0
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              const uint4 xp = *reinterpret_cast<const uint4*>(
                  xs + t * SEG * kGroup + gl * kGroup + 32 * j + 8 * i4);
              float lo = 0.f, hi = 0.f;
              fma_bf16x2_f32(lo, hi, xp.x ^ m[0], 0x3F803F80u);
              fma_bf16x2_f32(lo, hi, xp.y ^ m[1], 0x3F803F80u);
              fma_bf16x2_f32(lo, hi, xp.z ^ m[2], 0x3F803F80u);
              fma_bf16x2_f32(lo, hi, xp.w ^ m[3], 0x3F803F80u);
              acc[t] += lo + hi;
            }
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) total[t] = fmaf(a, acc[t], total[t]);
      }
    }
  }
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
      if (n < N && t0 + t < M) Y[(size_t)(t0 + t) * N + n] = float_to_bf16_bits(y);
    }
  }
}

template <int MT, bool SA = false>
cudaError_t launch_bp(const uint16_t* X, const uint8_t* packed, int P, int GS, int M, int N, int K,
                      uint16_t* Y, int* err, cudaStream_t s) {
  binplane_cc_kernel<MT, SA><<<(unsigned)row_tiles(N) * 4, kThreads, 0, s>>>(X, packed, P, GS, M, N,
                                                                             K, Y, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_binplane_cc(const uint16_t* X, const uint8_t* packed, int P, int M, int N,
                               int K, uint16_t* Y, int* err, cudaStream_t s) {
  if (M <= 1) return launch_bp<1>(X, packed, P, 0, M, N, K, Y, err, s);
  if (M <= 2) return launch_bp<2>(X, packed, P, 0, M, N, K, Y, err, s);
  if (M <= 4) return launch_bp<4>(X, packed, P, 0, M, N, K, Y, err, s);
  if (M <= 8) return launch_bp<8>(X, packed, P, 0, M, N, K, Y, err, s);
  if (M <= 16) return launch_bp<16>(X, packed, P, 0, M, N, K, Y, err, s);
  return launch_bp<32>(X, packed, P, 0, M, N, K, Y, err, s);
}

cudaError_t launch_sa_cc(const uint16_t* X, const uint8_t* packed, int P, int G, int M, int N,
                         int K, uint16_t* Y, int* err, cudaStream_t s) {
  if (M <= 1) return launch_bp<1, true>(X, packed, P, G, M, N, K, Y, err, s);
  if (M <= 2) return launch_bp<2, true>(X, packed, P, G, M, N, K, Y, err, s);
  if (M <= 4) return launch_bp<4, true>(X, packed, P, G, M, N, K, Y, err, s);
  if (M <= 8) return launch_bp<8, true>(X, packed, P, G, M, N, K, Y, err, s);
  if (M <= 16) return launch_bp<16, true>(X, packed, P, G, M, N, K, Y, err, s);
  return launch_bp<32, true>(X, packed, P, G, M, N, K, Y, err, s);
}

}  // namespace lowbit

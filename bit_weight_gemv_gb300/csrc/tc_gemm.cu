// Tensor-core (tcgen05) weight-only multiply for M <= 32 activation rows: the skinny GEMM that
// verifies a 16-token draft block (Efficient-Qwen report, section 2.2 and 3.2: block size 16;
// DFlash summary, section 4.1), its INT4 and binary-plane weight formats (Efficient-Qwen
// report, section 2.1; ShiftAddQwen README, "Method"/"Format"), and the LM-head variant that
// folds the vocabulary argmax into the epilogue (small-vocabulary MTP study, section 3.3).
//
// Roles of one CTA (320 threads) working on 128 weight rows x a range of K groups:
//   warp 8 (one lane): producer -- per group, bulk-copies the packed codes/scales of the
//       block's four 32-row tiles and TMA-loads the activation tile X[0:16|32][128 inputs]
//       (128-byte swizzle, rows past M zero-filled) into a 6-stage shared-memory ring.
//   warps 0-7: dequantise -- thread (row r, half h) turns its row's 64 inputs of a unit into
//       bf16 and writes them straight into tensor memory (the MMA's A operand), then later
//       reads that unit's fp32 accumulator column block and applies the per-(row, group)
//       scale in fp32.
//   warp 9 (one lane): issues 8 tcgen05.mma (M=128, N=16|32, K=16) per unit into a
//       double-buffered TMEM accumulator and commits completion to mbarriers.
// A "unit" is one group of 128 inputs (INT4) or one (group, plane) pair (binary planes).
//
// Exactness of the operands:
//   INT4: a nibble ORed into bf16 128.0 is exactly 128 + u (u = q + 8); the group's
//     accumulator D = sum (128+u) x, so sum q x = D - 136 * sum x.
//   Binary planes: plane bit i of a 32-input word, ORed into bit j of bf16 1.0, is exactly
//     1 + beta * 2^(j-7) (beta in {0,1}); the activation of that input is pre-scaled by
//     2^(7-j) in shared memory, so D = sum x' + sum beta x and
//     sum b x = 2 (D - sum x') - sum x  (b = 2 beta - 1).
// Split-K (when there are too few 128-row blocks to fill the GPU) uses a thread-block
// cluster along K; the partial sums are reduced through distributed shared memory.
#include "common.cuh"
#include "ptx.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

using namespace ptx;

constexpr int kBlockRows = 128;
constexpr int kDqWarps = 8;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kStages = 6;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColA = 0;    // A[2]: 64 columns each (128 bf16 inputs)
constexpr uint32_t kColD = 128;  // D[2]: 32 columns each
constexpr int kFmtInt4 = 0, kFmtBinplane = 1;
constexpr int kEpiStore = 0, kEpiArgmax = 1;
constexpr uint32_t kBarDq = 1;

struct TcArgs {
  const uint8_t* packed;
  uint16_t* Y;
  int M, N, K, P;
  int groups_per_rank;
  int* err;
  LmheadWorkspace* ws;
  const int32_t* draft;
  int32_t* argmax;
  int32_t* n_accept;
  int32_t* bonus;
};

template <int FMT, int NMMA>
struct TcLayout {
  static constexpr uint32_t kAtom = NMMA * 128;  // one 64-input swizzle atom of the X tile
  static constexpr uint32_t kX = 2 * kAtom;      // X tile for one group of 128 inputs
  __host__ __device__ static uint32_t codes(int P) { return FMT == kFmtInt4 ? 4 * 2048 : 4 * P * 512; }
  __host__ __device__ static uint32_t scales(int P) { return FMT == kFmtInt4 ? 4 * 64 : 4 * P * 64; }
  __host__ __device__ static uint32_t stage(int P) {
    return (kX + codes(P) + scales(P) + 1023u) / 1024u * 1024u;
  }
  static constexpr uint32_t kCtrl = 1024;
  __host__ static size_t smem(int P) { return 1024 + (size_t)kStages * stage(P) + kCtrl; }
};

// j(i): the mantissa bit that carries pair i of a 32-input plane word (see binary planes).
__device__ __forceinline__ int bp_bit(int i) { return i < 7 ? i : (i < 14 ? i - 7 : i - 14); }

__device__ __forceinline__ void dequant_int4_chunk(const uint4 c, uint32_t (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[4 * i + 0] = int4_pair_biased<0>(w[i]);
    v[4 * i + 1] = int4_pair_biased<1>(w[i]);
    v[4 * i + 2] = int4_pair_biased<2>(w[i]);
    v[4 * i + 3] = int4_pair_biased<3>(w[i]);
  }
}

__device__ __forceinline__ void dequant_bp_word(uint32_t w, uint32_t (&v)[16]) {
  const uint32_t w7 = w >> 7, w14 = w >> 14;
#pragma unroll
  for (int j = 0; j < 7; ++j) {
    v[j] = (w & (0x00010001u << j)) | 0x3F803F80u;
    v[7 + j] = (w7 & (0x00010001u << j)) | 0x3F803F80u;
  }
  v[14] = (w14 & 0x00010001u) | 0x3F803F80u;
  v[15] = (w14 & 0x00020002u) | 0x3F803F80u;
}

template <int FMT, int NMMA, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
tc_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const TcArgs args) {
  using L = TcLayout<FMT, NMMA>;
  constexpr int TOK = NMMA / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int P = (FMT == kFmtInt4) ? 1 : args.P;
  const uint32_t SB = L::stage(P);
  uint8_t* ctrl = smem + kStages * SB;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kStages;
  uint64_t* aready = empty + kStages;
  uint64_t* mmadone = aready + 2;
  uint64_t* mmafinal = mmadone + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mmafinal + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] header ok, [1] abort
  float* xsum = reinterpret_cast<float*>(ctrl + 256);                    // [3][32] sum x
  float* xsum2 = xsum + 96;                                              // [3][32] sum x'

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x, ks = gridDim.x, rb = blockIdx.y;
  const int N = args.N, K = args.K, G = K / kGroup, C = K / 32, NT = row_tiles(N);
  const int g0 = min(G, rank * args.groups_per_rank);
  const int g1 = min(G, g0 + args.groups_per_rank);
  const int ngroups = g1 - g0;
  const int nunits = ngroups * P;

  if (threadIdx.x == 0) {
    flags[0] = header_matches(reinterpret_cast<const PackedHeader*>(args.packed),
                              FMT == kFmtInt4 ? kFormatInt4 : kFormatBinplane,
                              FMT == kFmtInt4 ? 0 : P, N, K);
    flags[1] = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&aready[a]), kDqThreads);
      mbar_init(smem_addr(&mmadone[a]), 1);
    }
    mbar_init(smem_addr(mmafinal), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool hdr_ok = flags[0] != 0;
  if (!hdr_ok && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    record_error(args.err, LOWBIT_ERR_INVALID_ARG);

  const uint8_t* codes_g = args.packed + kHeaderBytes;
  const uint8_t* scales_g =
      codes_g + (FMT == kFmtInt4 ? int4_codes_bytes(N, K) : binplane_codes_bytes(P, N, K));
  auto stage_x = [&](int s) { return smem + (size_t)s * SB; };
  auto stage_codes = [&](int s) { return smem + (size_t)s * SB + L::kX; };
  auto stage_scales = [&](int s) { return smem + (size_t)s * SB + L::kX + L::codes(P); };
  auto fail = [&]() {
    if (!flags[1]) {
      flags[1] = 1;
      record_error(args.err, LOWBIT_ERR_TIMEOUT);
    }
  };

  float acc[TOK];
#pragma unroll
  for (int j = 0; j < TOK; ++j) acc[j] = 0.f;
  const int q = warp & 3, h = (warp >> 2) & 1;
  const int tok0 = h * TOK;
  const bool epi_active = tok0 < args.M;

  if (hdr_ok && warp == kProducerWarp) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ngroups; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(smem_addr(&empty[s]), ((i / kStages) - 1) & 1)) {
          fail();
          break;
        }
        if (flags[1]) break;
        const int g = g0 + i;
        uint32_t bytes = L::kX;
        for (int qq = 0; qq < 4; ++qq)
          if (rb * 4 + qq < NT) bytes += (L::codes(P) + L::scales(P)) / 4;
        const uint32_t fb = smem_addr(&full[s]);
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_2d(smem_addr(stage_x(s)), &xmap, g * kGroup, 0, fb);
        tma_load_2d(smem_addr(stage_x(s)) + L::kAtom, &xmap, g * kGroup + 64, 0, fb);
        for (int qq = 0; qq < 4; ++qq) {
          const size_t t = (size_t)rb * 4 + qq;
          if ((int)t >= NT) break;
          if (FMT == kFmtInt4) {
            bulk_g2s(smem_addr(stage_codes(s)) + qq * 2048, codes_g + (t * C + 4 * g) * 512, 2048, fb);
            bulk_g2s(smem_addr(stage_scales(s)) + qq * 64, scales_g + (t * G + g) * 64, 64, fb);
          } else {
            bulk_g2s(smem_addr(stage_codes(s)) + qq * P * 512, codes_g + (t * G + g) * P * 512,
                     P * 512, fb);
            bulk_g2s(smem_addr(stage_scales(s)) + qq * P * 64, scales_g + (t * G + g) * P * 64,
                     P * 64, fb);
          }
        }
        issued = i + 1;
      }
      // No copy may still be in flight when the CTA exits.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(smem_addr(&full[i % kStages]), (i / kStages) & 1, 200000000LL);
    }
  } else if (hdr_ok && warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kBlockRows, NMMA);
      for (int u = 0; u < nunits; ++u) {
        const int i = u / P, p = u % P, s = i % kStages, a = u & 1;
        if (!mbar_wait(smem_addr(&aready[a]), (u >> 1) & 1)) {
          fail();
          break;
        }
        if (flags[1]) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + kColD + a * 32;
        const uint32_t a_tmem = tmem + kColA + a * 64;
        const uint32_t xs = smem_addr(stage_x(s));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(xs + (kk >> 2) * L::kAtom + (kk & 3) * 32);
          umma_ts(d_tmem, a_tmem + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_addr(&mmadone[a]));
        if (p == P - 1) umma_commit(smem_addr(&empty[s]));
      }
      umma_commit(smem_addr(mmafinal));
      mbar_wait(smem_addr(mmafinal), 0, 200000000LL);
    }
  } else if (hdr_ok && warp < kDqWarps) {
    const int r = q * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    auto wait_or_fail = [&](uint32_t bar, uint32_t parity) {
      if (flags[1]) return;
      if (!mbar_wait(bar, parity)) fail();
    };
    auto epilogue = [&](int v, float sc) {
      const int a = v & 1, iv = v / P;
      wait_or_fail(smem_addr(&mmadone[a]), (v >> 1) & 1);
      tc_fence_after();
      if (epi_active) {
        uint32_t d[TOK];
        if constexpr (TOK == 8) tmem_ld8(tlane + kColD + a * 32 + tok0, d);
        else tmem_ld16(tlane + kColD + a * 32 + tok0, d);
        tmem_ld_wait();
        const float* xs = xsum + (iv % 3) * 32 + tok0;
        if constexpr (FMT == kFmtInt4) {
#pragma unroll
          for (int j = 0; j < TOK; ++j) acc[j] = fmaf(sc, __uint_as_float(d[j]) - 136.f * xs[j], acc[j]);
        } else {
          const float* xs2 = xsum2 + (iv % 3) * 32 + tok0;
#pragma unroll
          for (int j = 0; j < TOK; ++j)
            acc[j] = fmaf(sc, 2.f * (__uint_as_float(d[j]) - xs2[j]) - xs[j], acc[j]);
        }
      }
    };
    float sc_prev = 0.f;
    for (int u = 0; u < nunits; ++u) {
      const int i = u / P, p = u % P, s = i % kStages, a = u & 1;
      if (p == 0) {
        wait_or_fail(smem_addr(&full[s]), (i / kStages) & 1);
        // Per-token activation sums of this group (and the pre-scaled binary-plane copy).
        const int buf = i % 3;
#pragma unroll
        for (int rep = 0; rep < NMMA / 16; ++rep) {
          const int ci = threadIdx.x + kDqThreads * rep;
          const int t = ci >> 4, lc = ci & 15, at = lc >> 3, c = lc & 7;
          uint8_t* px = stage_x(s) + at * L::kAtom + t * 128 + ((c ^ (t & 7)) << 4);
          uint4 xv = *reinterpret_cast<uint4*>(px);
          uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          float s1 = 0.f, s2 = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_bits_to_float(xw[e] & 0xFFFF), hi = bf16_bits_to_float(xw[e] >> 16);
            s1 += lo + hi;
            if constexpr (FMT == kFmtBinplane) {
              const int pi = 4 * (c & 3) + e;               // pair index inside the 32-input word
              const float f = (float)(1 << (7 - bp_bit(pi)));
              s2 += (lo + hi) * f;
              // multiply both bf16 halves by 2^(7-j): exact for normal values
              __nv_bfloat162 x2 = *reinterpret_cast<__nv_bfloat162*>(&xw[e]);
              x2 = __hmul2(x2, __floats2bfloat162_rn(f, f));
              xw[e] = *reinterpret_cast<uint32_t*>(&x2);
            }
          }
          if constexpr (FMT == kFmtBinplane) *reinterpret_cast<uint4*>(px) = make_uint4(xw[0], xw[1], xw[2], xw[3]);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) {
            s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, o);
            if constexpr (FMT == kFmtBinplane) s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
          }
          if ((lane & 15) == 0) {
            xsum[buf * 32 + t] = s1;
            if constexpr (FMT == kFmtBinplane) xsum2[buf * 32 + t] = s2;
          }
        }
        if constexpr (FMT == kFmtBinplane) fence_proxy_async_smem();
        named_barrier(kBarDq, kDqThreads);
      }
      // Dequantise this thread's 64 inputs of unit u into TMEM columns of A[a].
      float sc;
      uint32_t v[16];
      const uint32_t acol = tlane + kColA + a * 64 + 32 * h;
      if constexpr (FMT == kFmtInt4) {
        const uint8_t* cs = stage_codes(s) + q * 2048 + lane * 16;
        const uint4 c0 = *reinterpret_cast<const uint4*>(cs + (2 * h) * 512);
        const uint4 c1 = *reinterpret_cast<const uint4*>(cs + (2 * h + 1) * 512);
        sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(stage_scales(s) + q * 64 + lane * 2));
        dequant_int4_chunk(c0, v);
        tmem_st16(acol, v);
        dequant_int4_chunk(c1, v);
        tmem_st16(acol + 16, v);
      } else {
        const uint8_t* cs = stage_codes(s) + (q * P + p) * 512 + lane * 16 + h * 8;
        const uint2 wv = *reinterpret_cast<const uint2*>(cs);
        sc = half_bits_to_float(
            *reinterpret_cast<const uint16_t*>(stage_scales(s) + (q * P + p) * 64 + lane * 2));
        dequant_bp_word(wv.x, v);
        tmem_st16(acol, v);
        dequant_bp_word(wv.y, v);
        tmem_st16(acol + 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_addr(&aready[a]));
      if (u >= 1) epilogue(u - 1, sc_prev);
      sc_prev = sc;
      (void)r;
    }
    if (nunits > 0) epilogue(nunits - 1, sc_prev);
  }

  // ------------------------------------------------------------------ reduction + output
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [NMMA][128], reuses the stage ring
  if (hdr_ok && warp < kDqWarps && epi_active) {
    const int r = q * 32 + lane;
#pragma unroll
    for (int j = 0; j < TOK; ++j) red[(tok0 + j) * kBlockRows + r] = acc[j];
  }
  if (ks > 1) cluster_sync();
  else __syncthreads();
  if (hdr_ok) {
    const int rows = kBlockRows / ks, r0 = rank * rows;
    auto reduced = [&](int t, int rr) {
      float v = 0.f;
      if (ks == 1) return red[t * kBlockRows + rr];
      const uint32_t la = smem_addr(&red[t * kBlockRows + rr]);
      for (int qq = 0; qq < ks; ++qq) v += ld_dsmem_f32(la, qq);
      return v;
    };
    if constexpr (EPI == kEpiStore) {
      for (int idx = threadIdx.x; idx < args.M * rows; idx += kThreads) {
        const int t = idx / rows, rr = r0 + idx % rows;
        const int n = rb * kBlockRows + rr;
        const float v = reduced(t, rr);
        if (n < N) args.Y[(size_t)t * N + n] = float_to_bf16_bits(v);
      }
    } else {
      for (int t = warp; t < args.M; t += kThreads / 32) {
        unsigned long long best = 0ull;
        for (int rr = r0 + lane; rr < r0 + rows; rr += 32) {
          const int n = rb * kBlockRows + rr;
          const float v = reduced(t, rr);
          if (n < N) {
            const unsigned long long key = argmax_key(v, n);
            best = key > best ? key : best;
          }
        }
        best = warp_max_u64(best);
        if (lane == 0 && best) atomicMax(&args.ws->keys[t], best);
      }
    }
  }
  if (ks > 1) cluster_sync();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (EPI == kEpiArgmax) {
    if (hdr_ok) lmhead_finish(args.ws, args.M, args.draft, args.argmax, args.n_accept, args.bonus);
  }
}

// ------------------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

template <int FMT, int NMMA, int EPI>
cudaError_t launch_tc(const uint16_t* X, TcArgs args, cudaStream_t stream) {
  using L = TcLayout<FMT, NMMA>;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)args.K, (cuuint64_t)args.M};
  cuuint64_t strides[1] = {(cuuint64_t)args.K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)NMMA};
  cuuint32_t estr[2] = {1, 1};
  if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int RB = (args.N + kBlockRows - 1) / kBlockRows, G = args.K / kGroup;
  const int target = 2 * sm_count();
  int ks = 1;
  while (ks < 8 && RB * ks * 2 <= target && ks * 2 <= G) ks *= 2;
  args.groups_per_rank = (G + ks - 1) / ks;
  const int P = FMT == kFmtInt4 ? 1 : args.P;
  // At least 80 KB of shared memory per CTA keeps at most two CTAs on an SM, so the two
  // 256-column TMEM allocations always fit and tcgen05.alloc never has to wait.
  const size_t smem = L::smem(P) > 80 * 1024 ? L::smem(P) : 80 * 1024;
  auto kern = tc_gemm_kernel<FMT, NMMA, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ks, (unsigned)RB, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (ks > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, map, args);
}

TcArgs base_args(const uint8_t* packed, int P, int M, int N, int K, int* err) {
  TcArgs a = {};
  a.packed = packed;
  a.M = M;
  a.N = N;
  a.K = K;
  a.P = P;
  a.err = err;
  return a;
}

}  // namespace

cudaError_t launch_int4_gemm_tc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                                uint16_t* Y, int* err, cudaStream_t s) {
  TcArgs a = base_args(packed, 1, M, N, K, err);
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtInt4, 16, kEpiStore>(X, a, s)
                 : launch_tc<kFmtInt4, 32, kEpiStore>(X, a, s);
}

cudaError_t launch_binplane_tc(const uint16_t* X, const uint8_t* packed, int P, int M, int N,
                               int K, uint16_t* Y, int* err, cudaStream_t s) {
  TcArgs a = base_args(packed, P, M, N, K, err);
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtBinplane, 16, kEpiStore>(X, a, s)
                 : launch_tc<kFmtBinplane, 32, kEpiStore>(X, a, s);
}

cudaError_t launch_lmhead_tc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                             const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                             int32_t* bonus, void* ws, int* err, cudaStream_t s) {
  TcArgs a = base_args(packed, 1, M, N, K, err);
  a.ws = reinterpret_cast<LmheadWorkspace*>(ws);
  a.draft = draft;
  a.argmax = argmax;
  a.n_accept = n_accept;
  a.bonus = bonus;
  return M <= 16 ? launch_tc<kFmtInt4, 16, kEpiArgmax>(H, a, s)
                 : launch_tc<kFmtInt4, 32, kEpiArgmax>(H, a, s);
}

}  // namespace lowbit

// Tensor-core (tcgen05) weight-only multiply for M <= 32 activation rows: the skinny GEMM that
// verifies a 16-token draft block (Efficient-Qwen report, section 2.2 and 3.2: block size 16;
// DFlash summary, section 4.1), for INT4 and binary-plane weights (Efficient-Qwen report,
// section 2.1; ShiftAddQwen README, "Method"/"Format"), plus the LM-head variant whose
// epilogue folds in the vocabulary argmax (small-vocabulary MTP study, section 3.3).
//
// A CTA (352 threads) owns a K range and a sequence of 128-row blocks ("items"; more than one
// when the grid is persistent).  Roles:
//   warp 8, lane 0 -- producer: per group, ONE bulk copy of the packed (128 rows x 128 inputs)
//       block (codes and scales are contiguous in the layout) and two TMA loads (one per
//       64-input swizzle atom) of the activation tile X[0:16|32][128 inputs] (128-byte
//       swizzle, rows past M zero-filled) into a shared-memory ring.  The first weight blocks are fetched before waiting for
//       the previous kernel in the stream (programmatic dependent launch).
//   warps 0-7 -- dequantise: thread (row r, half h) writes its row's 64 inputs of a unit as
//       bf16 straight into tensor memory (the MMA's A operand); NB units later it reads that
//       unit's fp32 accumulator columns back and applies the per-(row, group) scale in fp32.
//   warp 9, lane 0 -- MMA: 8 x tcgen05.mma (M=128, N=16|32, K=16) per unit into one of NB
//       TMEM accumulators; completion is committed to mbarriers.
//   warp 10 (binary planes only) -- pre-scales each staged activation tile in place.
// A unit is one group of 128 inputs (INT4) or one (group, plane) pair (binary planes).  NB
// (3 for N=16, 2 for N=32) units are in flight between dequantisation and epilogue.
//
// Exactness of the operands (all bf16 arithmetic below is exact):
//   INT4: a nibble ORed into bf16 128.0 is 128 + u (u = q + 8); subtracting 136 leaves q, so a
//     group's accumulator is D = sum q x and the epilogue adds s * D.
//   sa format (ShiftAddQwen README, "Format": alpha = d * a, u8 code a per plane and group of G
//     inputs, one fp16 d per 256 inputs): a thread's 64 inputs share one code a (G >= 64), so
//     it writes +-a (exact in bf16) by XORing the sign into the bf16 pair (a, a); a unit is
//     one (half of a 256-input super-block, plane) and the epilogue adds d * D.
//   Binary planes: the plane bit of pair i of a 32-input word, ORed into mantissa bit j(i) in
//     1..6 of bf16 1.0, gives 1 + beta * 2^(j-7) (beta in {0,1}); subtracting 1 + 2^(j-8)
//     leaves b * 2^(j-8) with b = 2 beta - 1 in {-1, +1}.  The activation of that input is
//     pre-scaled by 2^(8-j) in shared memory, so D = sum b x and the epilogue adds alpha * D.
// When there are too few 128-row blocks to fill the GPU, K is split across a thread-block
// cluster and the partial sums are reduced through distributed shared memory.
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
constexpr int kXWarp = 10;
constexpr int kThreads = 352;
constexpr uint32_t kTmemCols = 256;
constexpr int kFmtInt4 = 0, kFmtBinplane = 1, kFmtSa = 2, kFmtNvfp4 = 3;
constexpr int kEpiStore = 0, kEpiArgmax = 1;

struct TcArgs {
  const uint8_t* packed;
  const uint16_t* X;
  uint16_t* Y;
  int M, N, K, P;
  int GS;            // sa format: inputs per scale code (64, 128, 256)
  int groups_per_rank;  // blocks (groups of 128 inputs; sa: super-blocks of 256) per K rank
  int ks;            // CTAs splitting one row block's groups (divides the cluster size)
  int cl_begin;      // first cluster of this matrix
  int ncl;           // clusters of this matrix (they walk its row blocks with stride ncl * C / ks)
  int* err;
  LmheadWorkspace* ws;
  const int32_t* draft;
  int32_t* argmax;       // ARGMAX epilogue: per-token winners (draft head: the mapped ids)
  const int32_t* id_map; // draft head: full-vocabulary id of each row (may be null)
  int32_t* n_accept;
  int32_t* bonus;
};

// One launch: up to kMaxGemvProblems matrices sharing M, each with its activation tensor map.
// A cluster of `cluster` CTAs holds cluster / ks row blocks of one matrix.
struct TcBatch {
  CUtensorMap maps[kMaxGemvProblems];
  TcArgs p[kMaxGemvProblems];
  int count;
  int cluster;
  int stages;  // sa format: ring stages (its blocks vary with P and G)
};

template <int FMT, int NMMA>
struct TcLayout {
  static constexpr int kStages = NMMA <= 16 ? 6 : 5;   // sa: chosen per launch (TcBatch::stages)
  static constexpr int NB = NMMA <= 16 ? 3 : 2;        // A/D buffers in tensor memory
  static constexpr uint32_t kColA = 0;                  // A[NB]: 64 columns each
  static constexpr uint32_t kColD = 64 * NB;            // D[NB]: NMMA columns each
  static_assert(64 * NB + NMMA * NB <= (int)kTmemCols, "tensor memory budget");
  static constexpr int KIN = FMT == kFmtSa ? kSuper : kGroup;  // inputs per block
  static constexpr uint32_t kAtom = NMMA * 128;  // one 64-input swizzle atom of the X tile
  static constexpr uint32_t kX = (KIN / 64) * kAtom;  // X tile for one block
  __host__ __device__ static uint32_t block(int P, int GS) {
    return FMT == kFmtInt4 ? kInt4Block
         : FMT == kFmtNvfp4 ? kNvfp4Block
         : (FMT == kFmtSa ? sa_block(P, GS) : binplane_block(P));
  }
  __host__ __device__ static uint32_t stage(int P, int GS) {
    return (kX + block(P, GS) + 1023u) / 1024u * 1024u;
  }
  static constexpr uint32_t kCtrl = 1024;
  static constexpr uint32_t kLut = FMT == kFmtNvfp4 ? 256 * 4 : 0;  // NVFP4 code-byte table
  __host__ static size_t smem(int P, int GS, int S) {
    return 1024 + (size_t)S * stage(P, GS) + kCtrl + kLut;
  }
};

// j(i): the mantissa bit (1..6) that carries pair i of a 32-input plane word.  Pairs 0-5 are
// read from the word shifted left by 1, pairs 6-11 from it shifted right by 5, pairs 12-15
// from it shifted right by 11.
__host__ __device__ __forceinline__ int bp_bit(int i) { return i < 6 ? i + 1 : (i < 12 ? i - 5 : i - 11); }

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void dequant_int4_chunk(const uint4 c, uint32_t (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  constexpr uint32_t k136 = 0x43084308u;  // bf16 pair (136, 136)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[4 * i + 0] = bf16x2_sub(int4_pair_biased<0>(w[i]), k136);
    v[4 * i + 1] = bf16x2_sub(int4_pair_biased<1>(w[i]), k136);
    v[4 * i + 2] = bf16x2_sub(int4_pair_biased<2>(w[i]), k136);
    v[4 * i + 3] = bf16x2_sub(int4_pair_biased<3>(w[i]), k136);
  }
}

__device__ __forceinline__ void dequant_bp_word(uint32_t w, uint32_t (&v)[16]) {
  const uint32_t wl = w << 1, w5 = w >> 5, w11 = w >> 11;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = bp_bit(i);
    const uint32_t src = i < 6 ? wl : (i < 12 ? w5 : w11);
    // bf16 pair of 1 + 2^(j-8): exponent of 1.0 with mantissa bit j-1 set
    const uint32_t c = (0x3F80u | (1u << (j - 1))) * 0x00010001u;
    v[i] = bf16x2_sub((src & (0x00010001u << j)) | 0x3F803F80u, c);
  }
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// sa: the bf16 pair (a, a) with the signs of inputs 2i, 2i+1 of word w taken from bits i and
// 16 + i (bit set = +1, so the sign bit is set where the plane bit is 0).
__device__ __forceinline__ void dequant_sa_word(uint32_t w, uint32_t apair, uint32_t (&v)[16]) {
  const uint32_t nw = ~w;
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = apair ^ ((nw << (15 - i)) & 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// NVFP4: E2M1 code (0..15) -> bf16 bits, from the fields (sign, two exponent bits with bias
// 1, one mantissa bit); every value has at most 2 significant bits, so bf16 holds it exactly.
__device__ __forceinline__ uint32_t e2m1_bf16(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float mag = e == 0 ? 0.5f * (float)m : __uint_as_float((126u + e) << 23 | m << 22);
  return (__float_as_uint(mag) >> 16) | ((c & 8u) << 12);
}
// E4M3 byte -> bf16 pair (b, b): sign, four exponent bits with bias 7, three mantissa bits;
// exponent 0 is subnormal, 0x7F / 0xFF NaN.  At most 4 significant bits: exact in bf16.
__device__ __forceinline__ uint32_t e4m3_bf16x2(uint32_t b) {
  float v = (b & 0x78u) ? __uint_as_float(((b & 0x7Fu) << 20) + (120u << 23)) : (float)(b & 7u) * 0x1p-9f;
  if ((b & 0x7Fu) == 0x7Fu) v = __uint_as_float(0x7FC00000u);
  const uint32_t h = (__float_as_uint(v) >> 16) | ((b & 0x80u) << 8);
  return h | (h << 16);
}
// One 16-byte NVFP4 chunk (32 inputs, code byte j = inputs 2j and 2j+1) -> 16 bf16 pairs
// w = e2m1 * e4m3 (exact: at most 6 significant bits); bytes 0-7 take scale pair sa, 8-15 sb.
__device__ __forceinline__ void dequant_nvfp4_chunk(const uint4 c, uint32_t sa, uint32_t sb,
                                                    const uint32_t* lut, uint32_t (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = bf16x2_mul(lut[(w[j >> 2] >> (8 * (j & 3))) & 0xFFu], j < 8 ? sa : sb);
}

// Where unit u of a CTA's walk stands: unit ub of its block (plane p, sa half hb), the block's
// stage s and that stage's phase parity, the TMEM buffer a and that buffer's phase parity.
// Advanced one unit at a time: recomputing these with runtime divisions (by the units per
// block, the groups, the ring depth) cost the MMA-issuing thread about a hundred
// instructions per unit of eight MMAs.
struct UnitPos {
  int ub = 0, p = 0, hb = 0, s = 0, a = 0;
  uint32_t sph = 0u, aph = 0u;
  __device__ __forceinline__ void next(int UB, int P, int S, int NB) {
    if (++a == NB) {
      a = 0;
      aph ^= 1u;
    }
    if (++p == P) {
      p = 0;
      ++hb;
    }
    if (++ub == UB) {
      ub = p = hb = 0;
      if (++s == S) {
        s = 0;
        sph ^= 1u;
      }
    }
  }
};

template <int FMT, int NMMA, int EPI>
__global__ void __launch_bounds__(kThreads, 2)
tc_gemm_kernel(const __grid_constant__ TcBatch batch) {
  using L = TcLayout<FMT, NMMA>;
  const int S = FMT == kFmtSa ? batch.stages : L::kStages;
  constexpr int TOK = NMMA / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int C = batch.cluster;
  const int lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);  // cluster, rank in it
  int pi = 0;
  for (int i = 1; i < batch.count; ++i)
    if (cid >= batch.p[i].cl_begin) pi = i;
  const TcArgs& args = batch.p[pi];
  const CUtensorMap* xmap = &batch.maps[pi];
  const int P = (FMT == kFmtInt4 || FMT == kFmtNvfp4) ? 1 : args.P, GS = args.GS;
  const uint32_t SB = L::stage(P, GS), BB = L::block(P, GS);
  const int UB = FMT == kFmtSa ? 2 * P : P;  // MMA units per block: (half, plane) for sa
  constexpr int NB = L::NB;
  uint8_t* ctrl = smem + (size_t)S * SB;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + S;
  uint64_t* xready = empty + S;
  uint64_t* aready = xready + S;        // [NB]
  uint64_t* mmadone = aready + NB;      // [NB]
  uint64_t* mmafinal = mmadone + NB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mmafinal + 1);
  // [0] header ok, [1] abort, [2] NVFP4 tensor scale (fp32 bits, from the header)
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* lut = reinterpret_cast<uint32_t*>(ctrl + L::kCtrl);  // NVFP4: code byte -> bf16 pair

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = args.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);
  const int N = args.N, K = args.K, G = K / L::KIN, RB = row_tiles(N);
  const int tile0 = ((cid - args.cl_begin) << (lc - lk)) + (crank >> lk);  // first row block
  const int tstride = args.ncl << (lc - lk);                               // row-block stride
  const int g0 = min(G, rank * args.groups_per_rank);
  const int g1 = min(G, g0 + args.groups_per_rank);
  const int ngroups = g1 - g0;
  const int upi = ngroups * UB;  // units per item
  const int nitems = tile0 < RB ? (RB - tile0 + tstride - 1) / tstride : 0;
  const int total_groups = nitems * ngroups;
  const int total_units = nitems * upi;

  if (threadIdx.x == 0) {
    const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(args.packed);
    flags[0] = FMT == kFmtSa ? header_matches_sa(hp, P, GS, N, K)
             : FMT == kFmtNvfp4 ? header_matches(hp, kFormatNvfp4, 0, N, K)
             : header_matches(hp, FMT == kFmtInt4 ? kFormatInt4 : kFormatBinplane,
                              FMT == kFmtInt4 ? 0 : P, N, K);
    flags[1] = 0;
    if (FMT == kFmtNvfp4 && flags[0]) flags[2] = (int)__ldg(reinterpret_cast<const uint32_t*>(hp) + 14);
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      // dequant warps, MMA commit and (binary planes) the X warp release a stage
      mbar_init(smem_addr(&empty[s]), kDqWarps + 1 + (FMT == kFmtBinplane ? 1 : 0));
      mbar_init(smem_addr(&xready[s]), 1);
    }
    for (int a = 0; a < NB; ++a) {
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
  if (FMT == kFmtNvfp4 && threadIdx.x < 256)  // byte j: inputs (2j, 2j+1) -> bf16 pair
    lut[threadIdx.x] = e2m1_bf16(threadIdx.x & 15u) | (e2m1_bf16(threadIdx.x >> 4) << 16);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) grid_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  const bool hdr_ok = flags[0] != 0;
  if (!hdr_ok && threadIdx.x == 0 && rank == 0 && tile0 == 0)
    record_error(args.err, LOWBIT_ERR_INVALID_ARG);

  const uint8_t* payload = args.packed + kHeaderBytes;
  auto stage_x = [&](int s) { return smem + (size_t)s * SB; };
  auto stage_blk = [&](int s) { return smem + (size_t)s * SB + L::kX; };
  auto fail = [&]() {
    if (!flags[1]) {
      flags[1] = 1;
      record_error(args.err, LOWBIT_ERR_TIMEOUT);
    }
  };
  auto item_rb = [&](int it) { return tile0 + it * tstride; };

  float acc[TOK];
#pragma unroll
  for (int j = 0; j < TOK; ++j) acc[j] = 0.f;
  const int q = warp & 3, h = (warp >> 2) & 1;
  const int tok0 = h * TOK;
  const bool epi_active = tok0 < args.M;
  const int r = q * 32 + lane;  // row inside the 128-row block (dequant warps)

  if (hdr_ok && warp == kProducerWarp) {
    if (lane == 0) {
      // block gi = it * ngroups + (g - g0) in stage s, walked in order
      auto issue_block = [&](int s, int it, int g) {
        bulk_g2s(smem_addr(stage_blk(s)), payload + ((size_t)item_rb(it) * G + g) * BB, BB,
                 smem_addr(&full[s]));
      };
      auto issue_x = [&](int s, int g) {
#pragma unroll
        for (int at = 0; at < L::KIN / 64; ++at)
          tma_load_2d(smem_addr(stage_x(s)) + at * L::kAtom, xmap, g * L::KIN + 64 * at, 0,
                      smem_addr(&full[s]));
      };
      const int pre = min(S, total_groups);
      int it = 0, g = g0;  // item and group of the next block
      for (int gi = 0; gi < pre; ++gi) {
        mbar_arrive_expect_tx(smem_addr(&full[gi]), L::kX + BB);
        issue_block(gi, it, g);
        if (++g == g1) {
          g = g0;
          ++it;
        }
      }
      grid_dependency_wait();  // activations come from the previous kernel in the stream
      for (int gi = 0, gx = g0; gi < pre; ++gi) {
        issue_x(gi, gx);
        if (++gx == g1) gx = g0;
      }
      int issued = pre;
      int s = pre % S;
      uint32_t ph = (uint32_t)(pre / S) & 1u;  // phase parity of block gi in stage s
      for (int gi = pre; gi < total_groups; ++gi) {
        if (!mbar_wait(smem_addr(&empty[s]), ph ^ 1u)) {
          fail();
          break;
        }
        if (flags[1]) break;
        mbar_arrive_expect_tx(smem_addr(&full[s]), L::kX + BB);
        issue_block(s, it, g);
        issue_x(s, g);
        issued = gi + 1;
        if (++g == g1) {
          g = g0;
          ++it;
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // No copy may still be in flight when the CTA exits.
      for (int gi = max(0, issued - S); gi < issued; ++gi)
        mbar_wait(smem_addr(&full[gi % S]), (gi / S) & 1, 200000000LL);
    }
  } else if (hdr_ok && warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kBlockRows, NMMA);
      UnitPos up;
      for (int u = 0; u < total_units; ++u, up.next(UB, P, S, NB)) {
        const int ub = up.ub, p = up.p, a = up.a, s = up.s;
        if (!mbar_wait(smem_addr(&aready[a]), up.aph)) {
          fail();
          break;
        }
        if (FMT == kFmtBinplane && p == 0 && !mbar_wait(smem_addr(&xready[s]), up.sph)) {
          fail();
          break;
        }
        if (flags[1]) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + L::kColD + a * NMMA;
        const uint32_t a_tmem = tmem + L::kColA + a * 64;
        const uint32_t xs = smem_addr(stage_x(s)) + (FMT == kFmtSa ? up.hb * 2 * L::kAtom : 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(xs + (kk >> 2) * L::kAtom + (kk & 3) * 32);
          umma_ts(d_tmem, a_tmem + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_addr(&mmadone[a]));
        if (ub == UB - 1) umma_commit(smem_addr(&empty[s]));
      }
      umma_commit(smem_addr(mmafinal));
      mbar_wait(smem_addr(mmafinal), 0, 200000000LL);
    }
  } else if (hdr_ok && warp == kXWarp) {
    if constexpr (FMT == kFmtBinplane) {
      // Pre-scale each staged activation tile in place: input k of pair i = (k % 32) / 2 is
      // multiplied by 2^(8 - j(i)) (exact for normal bf16 values).
      int s = 0;
      uint32_t ph = 0u;
      for (int gi = 0; gi < total_groups; ++gi, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
        if (flags[1] || !mbar_wait(smem_addr(&full[s]), ph)) {
          fail();
          break;
        }
        for (int ci = lane; ci < NMMA * 16; ci += 32) {
          const int t = ci >> 4, lc = ci & 15, at = lc >> 3, c = lc & 7;
          uint4* px = reinterpret_cast<uint4*>(stage_x(s) + at * L::kAtom + t * 128 + ((c ^ (t & 7)) << 4));
          uint4 xv = *px;
          uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float f = (float)(1 << (8 - bp_bit(4 * (c & 3) + e)));
            __nv_bfloat162 x2 = *reinterpret_cast<__nv_bfloat162*>(&xw[e]);
            x2 = __hmul2(x2, __floats2bfloat162_rn(f, f));
            xw[e] = *reinterpret_cast<uint32_t*>(&x2);
          }
          *px = make_uint4(xw[0], xw[1], xw[2], xw[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&xready[s]));
          mbar_arrive(smem_addr(&empty[s]));
        }
      }
    }
  } else if (hdr_ok && warp < kDqWarps) {
    grid_dependency_wait();

    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    auto wait_or_fail = [&](uint32_t bar, uint32_t parity) {
      if (flags[1]) return;
      if (!mbar_wait(bar, parity)) fail();
    };
    auto output_item = [&](int it) {
      const int n = item_rb(it) * kBlockRows + r;
      if constexpr (EPI == kEpiStore) {
        if (ks == 1) {
#pragma unroll
          for (int j = 0; j < TOK; ++j)
            if (tok0 + j < args.M && n < N) args.Y[(size_t)(tok0 + j) * N + n] = float_to_bf16_bits(acc[j]);
        }
      } else {
        if (ks == 1 && epi_active) {
#pragma unroll
          for (int j = 0; j < TOK; ++j) {
            unsigned long long key = (n < N) ? argmax_key(acc[j], n) : 0ull;
            key = warp_max_u64(key);
            if (lane == 0 && tok0 + j < args.M && key) atomicMax(&args.ws->keys[tok0 + j], key);
          }
        }
      }
    };
    // unit v's results: TMEM buffer a with phase parity aph; `last` = the item's last unit
    auto epilogue = [&](int a, uint32_t aph, bool last, int vit, float sc) {
      wait_or_fail(smem_addr(&mmadone[a]), aph);
      tc_fence_after();
      if (epi_active) {
        uint32_t d[TOK];
        if constexpr (TOK == 8) tmem_ld8(tlane + L::kColD + a * NMMA + tok0, d);
        else tmem_ld16(tlane + L::kColD + a * NMMA + tok0, d);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < TOK; ++j) acc[j] = fmaf(sc, __uint_as_float(d[j]), acc[j]);
      }
      if (last) {  // last unit of an item: its outputs are complete
        if (ks == 1) {
          output_item(vit);
#pragma unroll
          for (int j = 0; j < TOK; ++j) acc[j] = 0.f;
        }
      }
    };
    // Unit u's epilogue runs NB iterations after its dequantisation, just before the
    // dequantisation of unit u + NB that reuses its A and D buffers.
    float scq[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) scq[b] = 0.f;
    UnitPos up;
    int vlu = 0, vit = 0;  // unit-in-item and item of the next epilogue's unit
    auto next_v = [&]() {
      if (++vlu == upi) {
        vlu = 0;
        ++vit;
      }
    };
    for (int u = 0; u < total_units; ++u, up.next(UB, P, S, NB)) {
      const int ub = up.ub, p = up.p, a = up.a, s = up.s;
      if (u >= NB) {  // unit u - NB used buffer a one phase earlier
        float scv = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b == a) scv = scq[b];
        epilogue(a, up.aph ^ 1u, vlu == upi - 1, vit, scv);
        next_v();
      }
      if (ub == 0) wait_or_fail(smem_addr(&full[s]), up.sph);
      // Dequantise this thread's 64 inputs of unit u into TMEM columns of A[a].
      float sc;
      uint32_t v[16];
      const uint32_t acol = tlane + L::kColA + a * 64 + 32 * h;
      const uint8_t* blk = stage_blk(s);
      if constexpr (FMT == kFmtInt4) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(blk + (2 * h) * 2048 + r * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(blk + (2 * h + 1) * 2048 + r * 16);
        sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(blk + kInt4ScaleOff + r * 2));
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        dequant_int4_chunk(c0, v);
        tmem_st16(acol, v);
        dequant_int4_chunk(c1, v);
        tmem_st16(acol + 16, v);
      } else if constexpr (FMT == kFmtNvfp4) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(blk + (2 * h) * 2048 + r * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(blk + (2 * h + 1) * 2048 + r * 16);
        // scales of the thread's four runs of 16 inputs (runs 4h .. 4h+3 of the group)
        uint32_t sp[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sp[j] = e4m3_bf16x2(blk[kNvfp4ScaleOff + (4 * h + j) * kBlockRows + r]);
        sc = __int_as_float(flags[2]);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        dequant_nvfp4_chunk(c0, sp[0], sp[1], lut, v);
        tmem_st16(acol, v);
        dequant_nvfp4_chunk(c1, sp[2], sp[3], lut, v);
        tmem_st16(acol + 16, v);
      } else if constexpr (FMT == kFmtSa) {
        // unit (half hb, plane p); this thread's inputs 128hb + 64h .. +63 share code group
        // (128hb + 64h) / GS of the super-block (G a power of two: shifts)
        const int hb = up.hb, lg = 31 - __clz(GS), gj = kSuper >> lg;
        const uint2 wv = *reinterpret_cast<const uint2*>(blk + (p * 2 + hb) * 2048 + r * 16 + h * 8);
        const int gl = (128 * hb + 64 * h) >> lg;
        const uint32_t ab = __float_as_uint((float)blk[sa_code_off(P) + (p * gj + gl) * kBlockRows + r]) >> 16;
        sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(blk + sa_code_off(P) + P * gj * kBlockRows + r * 2));
        if (ub == UB - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        }
        dequant_sa_word(wv.x, ab * 0x00010001u, v);
        tmem_st16(acol, v);
        dequant_sa_word(wv.y, ab * 0x00010001u, v);
        tmem_st16(acol + 16, v);
      } else {
        const uint2 wv = *reinterpret_cast<const uint2*>(blk + p * 2048 + r * 16 + h * 8);
        sc = half_bits_to_float(
            *reinterpret_cast<const uint16_t*>(blk + binplane_alpha_off(P) + (p * kBlockRows + r) * 2));
        if (p == P - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        }
        dequant_bp_word(wv.x, v);
        tmem_st16(acol, v);
        dequant_bp_word(wv.y, v);
        tmem_st16(acol + 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_addr(&aready[a]));
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b == a) scq[b] = sc;
    }
    for (int v = max(0, total_units - NB); v < total_units; ++v) {  // the last NB units
      const int a = v % NB;
      float scv = 0.f;
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b == a) scv = scq[b];
      epilogue(a, (uint32_t)(v / NB) & 1u, vlu == upi - 1, vit, scv);
      next_v();
    }
  }

  // ------------------------------------------------------------------ split-K reduction
  grid_dependency_wait();  // every thread that writes outputs has waited for the previous grid
  __syncthreads();
  if (C > 1) {  // every CTA of the cluster takes part in both cluster barriers
    // With ks > 1 a CTA has one item; every rank's partial sums go through shared memory
    // (the stage ring is free now) and each rank reduces a slice of the rows across the
    // ks CTAs of its row block.
    float* red = reinterpret_cast<float*>(smem);  // [NMMA][128]
    if (ks > 1 && hdr_ok && warp < kDqWarps && epi_active) {
#pragma unroll
      for (int j = 0; j < TOK; ++j) red[(tok0 + j) * kBlockRows + r] = acc[j];
    }
    cluster_sync();
    if (ks > 1 && hdr_ok && nitems > 0) {
      const int rows = kBlockRows / ks, r0 = rank * rows, rb = tile0, base = crank - rank;
      auto reduced = [&](int t, int rr) {
        const uint32_t la = smem_addr(&red[t * kBlockRows + rr]);
        float v = 0.f;
        for (int qq = 0; qq < ks; ++qq) v += ld_dsmem_f32(la, (uint32_t)(base + qq));
        return v;
      };
      if constexpr (EPI == kEpiStore) {
        for (int idx = threadIdx.x; idx < args.M * rows; idx += kThreads) {
          const int t = idx / rows, rr = r0 + idx % rows, n = rb * kBlockRows + rr;
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
    cluster_sync();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (EPI == kEpiArgmax) {
    if (hdr_ok) {
      if (args.n_accept) lmhead_finish(args.ws, args.M, args.draft, args.argmax, args.n_accept, args.bonus);
      else draft_finish(args.ws, args.M, args.id_map, args.argmax);
    }
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
cudaError_t launch_tc_batch(const TcArgs* probs, int count, cudaStream_t stream) {
  using L = TcLayout<FMT, NMMA>;
  if (count < 1 || count > kMaxGemvProblems) return cudaErrorInvalidValue;
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  TcBatch batch = {};
  const int slots = 2 * sm_count();  // at most two CTAs per SM (tensor memory, shared memory)
  int ks[kMaxGemvProblems];
  if (count == 1) {
    // Split K across a cluster only when the row blocks alone cannot fill the GPU.
    const int RB = row_tiles(probs[0].N), G = probs[0].K / L::KIN;
    int k = 1;
    while (k < 8 && RB * k * 2 <= slots && k * 2 <= G) k *= 2;
    ks[0] = k;
  } else {
    // Several matrices: each takes the smallest power-of-two K split whose CTAs hold at most
    // the launch's groups per slot (so tall-K matrices do not become the long pole).
    long long units = 0;
    for (int i = 0; i < count; ++i) units += (long long)row_tiles(probs[i].N) * (probs[i].K / L::KIN);
    long long target = (units + slots - 1) / slots;
    if (target < 4) target = 4;
    for (int i = 0; i < count; ++i) {
      const int G = probs[i].K / L::KIN;
      int k = 1;
      while (k < 8 && k * 2 <= G && (G + k - 1) / k > target) k *= 2;
      ks[i] = k;
    }
  }
  int C = 1;
  for (int i = 0; i < count; ++i) C = ks[i] > C ? ks[i] : C;
  int order[kMaxGemvProblems];
  for (int i = 0; i < count; ++i) order[i] = i;
  auto per_cta = [&](int i) { return (probs[i].K / L::KIN + ks[i] - 1) / ks[i]; };
  for (int i = 1; i < count; ++i)  // stable insertion sort: most groups per CTA first
    for (int j = i; j > 0 && per_cta(order[j]) > per_cta(order[j - 1]); --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  long long clusters = 0;
  for (int i = 0; i < count; ++i) {
    const int o = order[i];
    TcArgs a = probs[o];
    const int RB = row_tiles(a.N), G = a.K / L::KIN, tpc = C / ks[o];
    a.ks = ks[o];
    a.groups_per_rank = (G + ks[o] - 1) / ks[o];
    a.cl_begin = (int)clusters;
    // A single matrix with no K split runs persistent (at most `slots` CTAs walking its row
    // blocks); otherwise every row block gets its own CTAs.
    a.ncl = (count == 1 && C == 1) ? (RB < slots ? RB : slots) : (RB + tpc - 1) / tpc;
    clusters += a.ncl;
    batch.p[i] = a;
    // X [M][K] bf16; one box = one 64-input swizzle atom for NMMA rows (rows >= M read as 0).
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)NMMA};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&batch.maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.X), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (clusters * C > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  batch.count = count;
  batch.cluster = C;
  const int P = (FMT == kFmtInt4 || FMT == kFmtNvfp4) ? 1 : probs[0].P, GS = probs[0].GS;
  // sa blocks grow with P and G: as many stages (2..6) as keep two CTAs on an SM.
  int S = L::kStages;
  if (FMT == kFmtSa) {
    S = (int)((110 * 1024 - 2048) / L::stage(P, GS));
    S = S < 2 ? 2 : (S > 6 ? 6 : S);
  }
  batch.stages = S;
  // At least 80 KB of shared memory per CTA keeps at most two CTAs on an SM, so their two
  // 256-column TMEM allocations always fit and tcgen05.alloc never has to wait.
  const size_t smem = L::smem(P, GS, S) > 80 * 1024 ? L::smem(P, GS, S) : 80 * 1024;
  auto kern = tc_gemm_kernel<FMT, NMMA, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, batch);
}

template <int FMT, int NMMA, int EPI>
cudaError_t launch_tc(TcArgs args, cudaStream_t stream) {
  return launch_tc_batch<FMT, NMMA, EPI>(&args, 1, stream);
}

TcArgs base_args(const uint16_t* X, const uint8_t* packed, int P, int M, int N, int K, int* err) {
  TcArgs a = {};
  a.packed = packed;
  a.X = X;
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
  TcArgs a = base_args(X, packed, 1, M, N, K, err);
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtInt4, 16, kEpiStore>(a, s)
                 : launch_tc<kFmtInt4, 32, kEpiStore>(a, s);
}

cudaError_t launch_int4_tc_grouped(const GemvProblem* probs, int count, int M, int* err,
                                   cudaStream_t s) {
  if (count < 1 || count > kMaxGemvProblems) return cudaErrorInvalidValue;
  TcArgs a[kMaxGemvProblems];
  for (int i = 0; i < count; ++i) {
    a[i] = base_args(probs[i].X, probs[i].packed, 1, M, probs[i].N, probs[i].K, err);
    a[i].Y = probs[i].Y;
  }
  return M <= 16 ? launch_tc_batch<kFmtInt4, 16, kEpiStore>(a, count, s)
                 : launch_tc_batch<kFmtInt4, 32, kEpiStore>(a, count, s);
}

cudaError_t launch_binplane_tc(const uint16_t* X, const uint8_t* packed, int P, int M, int N,
                               int K, uint16_t* Y, int* err, cudaStream_t s) {
  TcArgs a = base_args(X, packed, P, M, N, K, err);
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtBinplane, 16, kEpiStore>(a, s)
                 : launch_tc<kFmtBinplane, 32, kEpiStore>(a, s);
}

cudaError_t launch_sa_tc(const uint16_t* X, const uint8_t* packed, int P, int G, int M, int N,
                         int K, uint16_t* Y, int* err, cudaStream_t s) {
  TcArgs a = base_args(X, packed, P, M, N, K, err);
  a.GS = G;
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtSa, 16, kEpiStore>(a, s) : launch_tc<kFmtSa, 32, kEpiStore>(a, s);
}

cudaError_t launch_nvfp4_tc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                            uint16_t* Y, int* err, cudaStream_t s) {
  TcArgs a = base_args(X, packed, 1, M, N, K, err);
  a.Y = Y;
  return M <= 16 ? launch_tc<kFmtNvfp4, 16, kEpiStore>(a, s) : launch_tc<kFmtNvfp4, 32, kEpiStore>(a, s);
}

cudaError_t launch_draft_argmax_tc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                                   const int32_t* id_map, int32_t* ids, void* ws, int* err,
                                   cudaStream_t s) {
  TcArgs a = base_args(H, packed, 1, M, N, K, err);
  a.ws = reinterpret_cast<LmheadWorkspace*>(ws);
  a.id_map = id_map;
  a.argmax = ids;
  return M <= 16 ? launch_tc<kFmtNvfp4, 16, kEpiArgmax>(a, s) : launch_tc<kFmtNvfp4, 32, kEpiArgmax>(a, s);
}

cudaError_t launch_lmhead_tc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                             const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                             int32_t* bonus, void* ws, int* err, cudaStream_t s) {
  TcArgs a = base_args(H, packed, 1, M, N, K, err);
  a.ws = reinterpret_cast<LmheadWorkspace*>(ws);
  a.draft = draft;
  a.argmax = argmax;
  a.n_accept = n_accept;
  a.bonus = bonus;
  return M <= 16 ? launch_tc<kFmtInt4, 16, kEpiArgmax>(a, s)
                 : launch_tc<kFmtInt4, 32, kEpiArgmax>(a, s);
}

}  // namespace lowbit

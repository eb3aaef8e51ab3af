// Streaming INT4 mat-vec (M = 1) over one or several weight matrices in a single launch.
//
//   y[n] = sum_g s[n][g] * sum_{k in g} q[n][k] * x[k]
// (Efficient-Qwen report, section 2.1: W = s (.) W_q with frozen symmetric per-group scales,
// group 128, served as W4A16; at one token per step the cost is streaming the packed weights
// once.)
//
// Work unit: one 128-row layout tile x a contiguous range of its groups.  The blocks of that
// range are adjacent in the packed payload, so a producer lane moves each (tile, group) block
// with one bulk copy into a ring of shared-memory stages.  The weights never depend on the
// preceding kernel, so the first ring's worth is requested before the programmatic-dependency
// wait and streams in while the previous kernel is still finishing; the activations of each
// group (256 bytes) follow into the same stage once that wait returns.
//
// Schedule: every matrix gets its own split of K (ks CTAs per tile) so that no CTA holds much
// more than a handful of blocks, whatever the matrix's K; a thread-block cluster of C CTAs
// (C = the largest ks) holds C / ks tiles of one matrix, and each tile's partial sums meet in
// distributed shared memory.  Clusters of the matrices with the most blocks per CTA come
// first in the grid, so the longest CTAs start in the first wave.
//
// Arithmetic: a converter warp turns each half group's 64 bf16 activations into int16 with
// one power-of-two scale 2^sh, chosen so that the largest magnitude lands in [2^14, 2^15):
// every activation within 2^7 of the half group's largest keeps all 8 of its significant
// bits, smaller ones are rounded to a multiple of 2^-sh (at most 2^-15 of that largest).  A
// code word's 8 nibbles u = q + 8 are split into two words of 4 unsigned bytes with two
// masks, and the integer dot-product instruction (two 16-bit x 8-bit products added into 32
// bits) sums u * X exactly; 8 * sum X is removed per half group in integers, the half group's
// integer (below 2^24 in magnitude, so exact in fp32) is scaled by s * 2^-sh in fp32, and each
// output is rounded once to bf16.  A half group holding a non-finite activation makes its
// rows NaN.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "ptx.cuh"
#include "verify.cuh"

namespace lowbit {
namespace {

constexpr int kCWarps = 8;                          // compute warps: 4 row quarters x 2 K halves
constexpr int kConvWarp = kCWarps + 1;              // after the producer warp
// Activation converters of the INT4 kernel: at one row, two (even and odd blocks) measured
// faster than one; with two or four rows, one.
template <int MT> __host__ __device__ constexpr int conv_warps() { return MT == 1 ? 2 : 1; }
template <int MT> __host__ __device__ constexpr int stream_threads() { return (kCWarps + 1 + conv_warps<MT>()) * 32; }
constexpr uint32_t kXBytes = kGroup * 2;            // one group's bf16 activations
constexpr int kMaxStages = 6;
// Dynamic shared memory per CTA (ring + reduction slots).  The INT4 kernel's budget was swept on
// the decode layer (36, 44, 53, 62 KB: 44 best, by 6% on the four-launch step); the plane
// kernels keep four CTAs per SM with 53 KB.
constexpr size_t kInt4SmemBudget = 44 * 1024;
constexpr size_t kSmemBudget = 53 * 1024;
constexpr int kResidentPerSm = 4;  // CTAs per SM that the budget allows
// Blocks per CTA the K split aims for: long streams amortise each CTA's fixed costs (start,
// first-copy latency, exchange) once a matrix fills the GPU several times over; small
// matrices are split further by the schedule's occupancy rule.
constexpr int kInt4TargetBlocks = 32;
constexpr int kMaxSplit = 16;      // cluster sizes above 8 need the non-portable opt-in

// The first cache line holds what every CTA reads first (to find its matrix); each matrix's
// fields sit in their own 64-byte line after it.
struct StreamArgs {
  int count;
  int stages;
  int cluster;  // C
  int m;        // activation rows (INT4 kernel; 1 for the plane kernels)
  int stall;    // test-only stall setting (lowbit_debug_inject_stall); 0 in normal use
  int row_offset;  // sharded LM head: global vocabulary row of this shard's row 0
  int cl_begin[kMaxGemvProblems];  // copy of p[i].cluster_begin
  int* err;
  LmheadWorkspace* ws;     // NVFP4 draft head: argmax keys and CTA counter
  const int32_t* id_map;   // NVFP4 draft head: full-vocabulary id per row (may be null)
  int32_t* ids;            // draft head: mapped ids out; LM-head verify: argmax out
  const int32_t* draft;    // LM-head verify: draft tokens (M - 1)
  int32_t* n_accept;       // LM-head verify: accepted prefix length out
  int32_t* bonus;          // LM-head verify: the target's token after the prefix out
  unsigned long long* keys_out;  // sharded LM head: the shard's best key per token out
  GemvProblem p[kMaxGemvProblems];
};

// Wait limits in SM clock cycles.  Every wait gives up after kWaitLimit (about a second at the
// boost clock).  Under the test-only stall setting a launch's compute warps first wait on an
// mbarrier that nothing arrives on, give up after kStallLimit (about a millisecond) and skip
// their blocks; the producer then issues only its first ring of copies (and still waits for
// them before it exits) and the warps that prepare stages handle only those, so no other wait
// can run out.  The loops themselves are those of normal operation.
constexpr long long kWaitLimit = 2000000000LL;
constexpr long long kStallLimit = 2000000LL;

// The compute warps' check under the stall setting: true when the warp must skip its blocks.
__device__ __forceinline__ bool stalled_out(const StreamArgs& a, uint32_t never_bar, int* err,
                                            int& gave_up, int lane) {
  if (!a.stall) return false;
  const bool ok = ptx::mbar_wait(never_bar, 0u, kStallLimit);  // nothing arrives: times out
  if (!__all_sync(0xFFFFFFFFu, ok) && lane == 0) {
    record_error(err, LOWBIT_ERR_TIMEOUT);
    gave_up = 1;
  }
  return true;
}

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Stage and phase parity of block b in a ring of S stages, advanced one block at a time (a
// runtime division per block would cost more than the rest of a block's bookkeeping).
struct RingPos {
  int s;
  uint32_t ph;
  __device__ __forceinline__ void next(int S) {
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Two-way dot product: c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or with bytes 2 and 3
// (hi); a's halves signed, b's bytes unsigned.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Activation converter shared by the INT4 and NVFP4 kernels: the 128 bf16 activations of a
// stage (lane l holds inputs 4l..4l+3 in `raw`) to int16 with one power-of-two scale per run
// of 64 (lanes 0..15 and 16..31); returns the four int16 values (low 16 bits) and the run's
// 2^-sh (NaN when the run holds a non-finite value).
struct Converted {
  uint32_t i0, i1, i2, i3;
  float down;
};
__device__ __forceinline__ Converted convert_run64(uint2 raw, int lane) {
  const uint32_t mag = max(max(raw.x & 0x7FFFu, (raw.x >> 16) & 0x7FFFu),
                           max(raw.y & 0x7FFFu, (raw.y >> 16) & 0x7FFFu));
  // |x| bits order as |x|
  const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, lane < 16 ? mag : 0u);
  const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, lane < 16 ? 0u : mag);
  const uint32_t mmax = lane < 16 ? mlo : mhi;
  const int e = max((int)(mmax >> 7), 1);  // biased exponent of the run's max |x|
  const int sh = min(141 - e, 126);        // max |x| * 2^sh < 2^15
  const float up = __int_as_float((127 + sh) << 23);
  Converted c;
  c.down = mmax >= 0x7F80u ? __int_as_float(0x7FC00000) : __int_as_float((127 - sh) << 23);
  // x * 2^sh is exact; adding 1.5 * 2^23 rounds it to an integer (nearest, even on ties) and
  // leaves that integer's two's complement in the low 16 bits.
  constexpr float kRound = 12582912.f;
  c.i0 = __float_as_uint(fmaf(__uint_as_float(raw.x << 16), up, kRound)) & 0xFFFFu;
  c.i1 = __float_as_uint(fmaf(__uint_as_float(raw.x & 0xFFFF0000u), up, kRound)) & 0xFFFFu;
  c.i2 = __float_as_uint(fmaf(__uint_as_float(raw.y << 16), up, kRound)) & 0xFFFFu;
  c.i3 = __float_as_uint(fmaf(__uint_as_float(raw.y & 0xFFFF0000u), up, kRound)) & 0xFFFFu;
  return c;
}

// MT: activation rows the kernel is built for (1, 2 or 4); a.m <= MT rows are present.  Each
// unpacked code word serves every row, so the bytes streamed per output stay those of M = 1.
template <int MT>
__global__ void __launch_bounds__(stream_threads<MT>())
int4_stream_kernel(const __grid_constant__ StreamArgs a) {
  constexpr uint32_t STG = kInt4Block + MT * kXBytes;  // stage: block, then MT activation rows
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t xready[kMaxStages];  // the stage's int16 activations are set
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ __align__(8) uint64_t redbar;  // rank 0 of a split tile: partials have arrived
  __shared__ __align__(8) uint64_t never;   // nothing arrives on it (test-only stall setting)
  // Per stage: the int16 activations, one uint4 per code word j holding the 16-bit pairs
  // (X[8j], X[8j+4]), (X[8j+1], X[8j+5]), (X[8j+2], X[8j+6]), (X[8j+3], X[8j+7]) -- the
  // order in which the two byte words of code word j meet them -- and, for inputs 0..63 and
  // 64..127, (2^-sh of the first, of the second, sum X of the first, of the second).
  __shared__ __align__(16) uint4 xq[kMaxStages][MT][kGroup / 8];
  __shared__ __align__(16) float4 xmeta[kMaxStages][MT];
  __shared__ float red[kCWarps][MT][32];
  __shared__ float part[MT][kRowTile];
  __shared__ int ok;
  __shared__ int gave_up;  // some wait of this CTA timed out

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster, lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);  // cluster, rank in it
  int pi = 0;
  for (int i = 1; i < a.count; ++i)
    if (cid >= a.cl_begin[i]) pi = i;
  const GemvProblem& pr = a.p[pi];
  const int ks = pr.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);  // this CTA's share of its tile's groups
  const int tile = ((cid - pr.cluster_begin) << (lc - lk)) + (crank >> lk);
  const int G = pr.K / kGroup;
  const bool live = tile < row_tiles(pr.N);  // the last cluster of a matrix may be partly idle
  const int g0 = (rank * G) >> lk, g1 = ((rank + 1) * G) >> lk;
  const int nb = live ? g1 - g0 : 0;
  const int S = a.stages, M = MT == 1 ? 1 : a.m;

  if (threadIdx.x == 0) {
    // With `early`, the header is checked in parallel with the first copies (it then gates
    // only the outputs); otherwise it is checked before anything else is read.
    ok = live && (pr.early || header_matches(reinterpret_cast<const PackedHeader*>(pr.packed),
                                             kFormatInt4, 0, pr.N, pr.K));
    gave_up = 0;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&xready[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kCWarps);
    }
    // rank 0 of a split tile receives one arrival per row from each other rank
    ptx::mbar_init(ptx::smem_addr(&redbar), (uint32_t)(kRowTile * (ks > 1 ? ks - 1 : 1)));
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_mbar_init();
  }
  if (warp < kCWarps) {
#pragma unroll
    for (int m = 0; m < MT; ++m) red[warp][m][lane] = 0.f;
  }
  __syncthreads();
  // Half of a cluster barrier: its wait, just before the partial sums are exchanged, finds
  // every CTA's barriers initialised (and returns at once, as all arrived long before).
  if (C > 1) ptx::cluster_arrive();
  if (threadIdx.x == 0) grid_launch();  // dependents may begin their own weight prefetch
  const bool hdr_ok = ok != 0;  // with `early`: only "this CTA has work"; see out_ok below
  // A compute warp checks the header (it would only be waiting for its first stage); the
  // producer warp must not wait on this load before issuing its copies.
  if (pr.early && live && threadIdx.x == 0 &&
      !header_matches(reinterpret_cast<const PackedHeader*>(pr.packed), kFormatInt4, 0, pr.N, pr.K))
    ok = 0;  // read after the epilogue's barrier

  if (warp == kCWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && hdr_ok) {
      const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * kInt4Block;
      const uint16_t* xsrc = pr.X + (size_t)g0 * kGroup;
      const uint32_t tx = kInt4Block + (uint32_t)M * kXBytes;
      // activation row m of block b -> its slot in the stage
      auto copy_x = [&](int b, int s, uint32_t bar) {
        for (int m = 0; m < M; ++m)
          ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * STG + kInt4Block + m * kXBytes),
                        xsrc + (size_t)m * pr.K + (size_t)b * kGroup, kXBytes, bar);
      };
      const int pre = min(nb, S);
      for (int b = 0; b < pre; ++b) {
        const uint32_t bar = ptx::smem_addr(&full[b]);
        ptx::mbar_arrive_expect_tx(bar, tx);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * STG), wsrc + (size_t)b * kInt4Block,
                      kInt4Block, bar);
      }
      grid_wait();  // the activations may be the previous kernel's output
      for (int b = 0; b < pre; ++b) copy_x(b, b, ptx::smem_addr(&full[b]));
      int issued = pre;
      const int nbi = a.stall ? pre : nb;  // read once: the waits below clobber memory
      RingPos rp{pre % S, (uint32_t)(pre / S) & 1u};
      for (int b = pre; b < nbi; ++b, rp.next(S)) {
        const int s = rp.s;
        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), rp.ph ^ 1u)) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
          break;
        }
        const uint32_t bar = ptx::smem_addr(&full[s]);
        ptx::mbar_arrive_expect_tx(bar, tx);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * STG), wsrc + (size_t)b * kInt4Block,
                      kInt4Block, bar);
        copy_x(b, s, bar);
        issued = b + 1;
      }
      // Copies still in flight must land before the CTA may exit.
      for (int b = max(0, issued - S); b < issued; ++b)
        ptx::mbar_wait(ptx::smem_addr(&full[b % S]), (b / S) & 1);
    }
    __syncwarp();
  } else if (warp >= kConvWarp) {
    // ---------------------------------------------------------------- activation converters
    // Converter c owns the stages s with s % conv_warps == c: a block's conversion is a chain
    // of dependent reductions and shuffles, so two warps double the rate a CTA can convert
    // at.  Owning whole stages keeps each stage's phases in order for its one converter (a
    // parity wait can never meet a phase two behind), whatever the stage count.
    if (hdr_ok) {
      RingPos rp{0, 0u};
      const int nbs = a.stall ? min(nb, S) : nb;  // read once: the waits below clobber memory
      for (int b = 0; b < nbs; ++b, rp.next(S)) {
        const int s = rp.s;
        if (s % conv_warps<MT>() != warp - kConvWarp) continue;
        const bool landed = ptx::mbar_wait(ptx::smem_addr(&full[s]), rp.ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
          if (lane == 0) {
            record_error(a.err, LOWBIT_ERR_TIMEOUT);
            gave_up = 1;
          }
          break;
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {  // rows are independent: unrolled, their chains interleave
        if (m >= M) break;
        // lane l holds inputs 4l..4l+3 (code word l/2, nibbles 4(l&1)..4(l&1)+3)
        const uint2 raw =
            reinterpret_cast<const uint2*>(ring + (size_t)s * STG + kInt4Block + m * kXBytes)[lane];
        // lanes 0..15 hold inputs 0..63, lanes 16..31 inputs 64..127
        const Converted cv = convert_run64(raw, lane);
        const uint32_t i0 = cv.i0, i1 = cv.i1, i2 = cv.i2, i3 = cv.i3;
        const float down = cv.down;
        const int mine = (int)(int16_t)i0 + (int)(int16_t)i1 + (int)(int16_t)i2 + (int)(int16_t)i3;
        const int sum_lo = __reduce_add_sync(0xFFFFFFFFu, lane < 16 ? mine : 0);
        const int sum_hi = __reduce_add_sync(0xFFFFFFFFu, lane < 16 ? 0 : mine);
        const uint32_t p01 = i0 | (i1 << 16), p23 = i2 | (i3 << 16);
        const uint32_t o01 = __shfl_xor_sync(0xFFFFFFFFu, p01, 1);  // the word's other half
        const uint32_t o23 = __shfl_xor_sync(0xFFFFFFFFu, p23, 1);
        if ((lane & 1) == 0)
          xq[s][m][lane >> 1] = make_uint4(__byte_perm(p01, o01, 0x5410), __byte_perm(p01, o01, 0x7632),
                                        __byte_perm(p23, o23, 0x5410), __byte_perm(p23, o23, 0x7632));
        float* meta = reinterpret_cast<float*>(&xmeta[s][m]);
        if ((lane & 15) == 0) {
          meta[lane >> 4] = down;
          meta[2 + (lane >> 4)] = __int_as_float(lane < 16 ? sum_lo : sum_hi);
        }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&xready[s]));
      }
    }
  } else if (warp < kCWarps && hdr_ok) {
    // ---------------------------------------------------------------- compute
    const int q = warp & 3, h = warp >> 2;  // rows 32q..32q+31, inputs 64h..64h+63 of each group
    const int row = 32 * q + lane;
    float total[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) total[m] = 0.f;
    RingPos rp{0, 0u};
    const int nbc = stalled_out(a, ptx::smem_addr(&never), a.err, gave_up, lane) ? 0 : nb;
    for (int b = 0; b < nbc; ++b, rp.next(S)) {
      const int s = rp.s;
      const bool ready = ptx::mbar_wait(ptx::smem_addr(&xready[s]), rp.ph);
      if (!__all_sync(0xFFFFFFFFu, ready)) {  // warp-uniform exit keeps the warp converged
        if (lane == 0) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
        }
        break;
      }
      const uint8_t* st = ring + (size_t)s * STG;
      const uint4 c0 = *reinterpret_cast<const uint4*>(st + (2 * h) * (kRowTile * 16) + row * 16);
      const uint4 c1 = *reinterpret_cast<const uint4*>(st + (2 * h + 1) * (kRowTile * 16) + row * 16);
      const float sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + kInt4ScaleOff + row * 2));
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // nibble e of a word sits at bits 4(e/2) + 16(e%2): the masked word holds nibbles
        // (0, 4, 1, 5) in its bytes, the shifted one (2, 6, 3, 7)
        const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const uint4 x = xq[s][m][8 * h + i];
            acc[m][0] = dp2a_lo(x.x, lo, acc[m][0]);
            acc[m][1] = dp2a_hi(x.y, lo, acc[m][1]);
            acc[m][2] = dp2a_lo(x.z, hi, acc[m][2]);
            acc[m][3] = dp2a_hi(x.w, hi, acc[m][3]);
          }
        }
      }
      float4 meta[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < M) meta[m] = xmeta[s][m];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < M) {
          const int v = (acc[m][0] + acc[m][1]) + (acc[m][2] + acc[m][3]) -
                        8 * __float_as_int(h ? meta[m].w : meta[m].z);
          total[m] = fmaf(sc * (h ? meta[m].y : meta[m].x), (float)v, total[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) red[warp][m][lane] = total[m];
  }

  // -------------------------------------------------------------------- reduction + store
  __syncthreads();
  // header verified (before or alongside the copies) and every wait of this CTA completed
  const bool out_ok = ok != 0 && !gave_up;
  if (!out_ok && live && threadIdx.x == 0 && rank == 0 && tile == 0)
    record_error(a.err, LOWBIT_ERR_INVALID_ARG);
  if (threadIdx.x < kRowTile) {
    const int q = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int m = 0; m < MT; ++m) part[m][threadIdx.x] = red[q][m][l] + red[q + 4][m][l];
  }
  const int n = tile * kRowTile + (int)threadIdx.x;
  if (C > 1) ptx::cluster_wait();
  if (ks > 1) {
    // Ranks 1..ks-1 push their partial sums into rank 0's slots (one float per row and
    // activation row; each row's values followed by a remote arrival) and leave; rank 0 waits
    // for them, adds them in rank order and stores.
    float* slots = reinterpret_cast<float*>(ring + (size_t)S * STG);  // [ks-1][MT][128]
    const uint32_t owner = (uint32_t)(crank - rank);                 // rank 0's CTA
    if (live && threadIdx.x < kRowTile) {
      if (rank != 0) {
        // A CTA that gave up on a wait stays out of rank 0's shared memory: rank 0 may have
        // stopped waiting for it and exited.
        if (gave_up) return;
        for (int m = 0; m < M; ++m) {
          const uint32_t la = ptx::smem_addr(&slots[((rank - 1) * MT + m) * kRowTile + threadIdx.x]);
          ptx::st_dsmem_f32(ptx::map_to_rank(la, owner), part[m][threadIdx.x]);
        }
        ptx::mbar_arrive_remote(ptx::map_to_rank(ptx::smem_addr(&redbar), owner));
      } else {
        // Under the stall setting every live CTA gives up and pushes nothing, so the short
        // limit cannot end this wait before a push that is still coming.
        const bool got = ptx::mbar_wait_cluster(ptx::smem_addr(&redbar), 0, a.stall ? kStallLimit : kWaitLimit);
        if (!got) record_error(a.err, LOWBIT_ERR_TIMEOUT);
        grid_wait();
        for (int m = 0; m < M; ++m) {
          float y = part[m][threadIdx.x];
          for (int r = 1; r < ks; ++r) y += slots[((r - 1) * MT + m) * kRowTile + threadIdx.x];
          if (got && out_ok && n < pr.N) pr.Y[(size_t)m * pr.N + n] = float_to_bf16_bits(y);
        }
      }
    }
  } else {
    __syncthreads();
    if (out_ok && threadIdx.x < kRowTile) {
      grid_wait();
      if (n < pr.N)
        for (int m = 0; m < M; ++m) pr.Y[(size_t)m * pr.N + n] = float_to_bf16_bits(part[m][threadIdx.x]);
    }
  }
}

// ------------------------------------------------------------------------------ binary planes
// y[n] = sum_p sum_g alpha[p][n][g] * sum_{k in g} b[p][n][k] x[k],  b in {-1, +1}
// (ShiftAddQwen README, "Method": per plane a sign-select-and-add, then one scale per group).
//
// Same stream, schedule and reduction as the INT4 kernel; a stage holds one (tile, group)
// block of P sign planes plus alphas and the group's 256 bytes of activations.  The
// sign-select-and-add runs as table lookups: for each set of 4 inputs that one nibble of a
// sign word covers, a helper warp tabulates the 16 signed sums +-x0 +-x1 +-x2 +-x3 once per
// stage (2 KB per group, shared by every row and plane); a row then adds one table entry per
// nibble, so each 4 weights of a plane cost one shared-memory load and one add.
constexpr int kLutWarp = kCWarps + 1;
constexpr int kLutWarps = 2;  // table builders, each owning alternate ring stages
constexpr int kBpThreads = (kCWarps + 1 + kLutWarps) * 32;  // compute, producer, table warps
constexpr uint32_t kLutBytes = 32 * 16 * sizeof(float);  // 32 nibble sets x 16 sums
constexpr int kBpTargetBlocks = 5;
constexpr int kSaTargetBlocks = 3;  // blocks of 256 inputs
// sa stages are up to 41 KB (8 planes, G = 64): two of them and the split-K slots may exceed
// the four-per-SM budget, so the sa kernel may use up to this much.
constexpr size_t kSaSmemMax = 96 * 1024;


// acc += sum over the 8 nibbles of one sign word of the tabulated signed sums; `tab` points
// at the word's 8 tables of 16 floats (nibble n: inputs of pair slots 4n..4n+3).  The sa
// kernel's form (the shared-address form below measured 3% slower there, 6% faster for the
// binary planes).
__device__ __forceinline__ void lut_word(uint32_t w, const float* tab, float (&acc)[2]) {
#pragma unroll
  for (int n = 0; n < 8; ++n) acc[n & 1] += tab[16 * n + ((w >> (4 * n)) & 0xFu)];
}
// One table entry: the float at shared address a + OFF.
template <int OFF>
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(v) : "r"(a), "n"(OFF));
  return v;
}
// acc += sum over the 8 nibbles of one sign word of the tabulated signed sums; `tab` is the
// shared address of the word's 8 tables of 16 floats (nibble n: inputs of pair slots
// 4n..4n+3), 64-byte aligned, so that a nibble's byte offset (4 x nibble, at most 60) can be
// ORed into it: a shift, a masked OR, the load (table n at an immediate 64n) and the add.
__device__ __forceinline__ void lut_word(uint32_t w, uint32_t tab, float (&acc)[2]) {
  acc[0] += lds_f32<0>(ptx::and_or(w << 2, 0x3Cu, tab));
  acc[1] += lds_f32<64>(ptx::and_or(w >> 2, 0x3Cu, tab));
  acc[0] += lds_f32<128>(ptx::and_or(w >> 6, 0x3Cu, tab));
  acc[1] += lds_f32<192>(ptx::and_or(w >> 10, 0x3Cu, tab));
  acc[0] += lds_f32<256>(ptx::and_or(w >> 14, 0x3Cu, tab));
  acc[1] += lds_f32<320>(ptx::and_or(w >> 18, 0x3Cu, tab));
  acc[0] += lds_f32<384>(ptx::and_or(w >> 22, 0x3Cu, tab));
  acc[1] += lds_f32<448>(ptx::and_or(w >> 26, 0x3Cu, tab));
}

// Body of both plane kernels.  SA = false: fp16-alpha planes, one block per (tile, group of
// 128 inputs).  SA = true: the deployed format, one block per (tile, super-block of 256 inputs)
// with u8 codes a per (plane, group of G) and one fp16 d per row (alpha = d * a).
template <bool SA>
__device__ __forceinline__ void plane_stream_body(const StreamArgs& a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t tabready[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ __align__(8) uint64_t redbar;
  __shared__ __align__(8) uint64_t never;  // nothing arrives on it (test-only stall setting)
  __shared__ float red[kCWarps][32];
  __shared__ float part[kRowTile];
  __shared__ int ok;
  __shared__ int gave_up;  // some wait of this CTA timed out

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster, lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);
  int pi = 0;
  for (int i = 1; i < a.count; ++i)
    if (cid >= a.cl_begin[i]) pi = i;
  const GemvProblem& pr = a.p[pi];
  const int ks = pr.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);
  const int tile = ((cid - pr.cluster_begin) << (lc - lk)) + (crank >> lk);
  constexpr int KIN = SA ? kSuper : kGroup;  // inputs per block
  constexpr uint32_t XB = KIN * 2, LUT = (KIN / 4) * 16 * sizeof(float);  // activations, tables
  const int G = pr.K / KIN, P = pr.P, GS = pr.G;
  const bool live = tile < row_tiles(pr.N);
  const int g0 = (rank * G) >> lk, g1 = ((rank + 1) * G) >> lk;
  const int nb = live ? g1 - g0 : 0;
  const int S = a.stages;
  const uint32_t BB = SA ? sa_block(P, GS) : binplane_block(P), SB = BB + XB + LUT;
  auto header_ok = [&]() {
    const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(pr.packed);
    return SA ? header_matches_sa(hp, P, GS, pr.N, pr.K) : header_matches(hp, kFormatBinplane, P, pr.N, pr.K);
  };

  if (threadIdx.x == 0) {
    // the table lookups OR byte offsets into 64-byte aligned table addresses
    ok = live && (pr.early || header_ok()) && (ptx::smem_addr(smem) & 63u) == 0u;
    gave_up = 0;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&tabready[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kCWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&redbar), (uint32_t)(kRowTile * (ks > 1 ? ks - 1 : 1)));
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_mbar_init();
  }
  if (warp < kCWarps) red[warp][lane] = 0.f;
  __syncthreads();
  if (C > 1) ptx::cluster_arrive();
  if (threadIdx.x == 0) grid_launch();
  const bool hdr_ok = ok != 0;
  if (pr.early && live && threadIdx.x == 0 && !header_ok()) ok = 0;

  // stage s: block | activations (2 bytes per input) | tables (16 floats per 4 inputs)
  auto stage = [&](int s) { return smem + (size_t)s * SB; };
  if (warp == kCWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && hdr_ok) {
      const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * BB;
      const uint16_t* xsrc = pr.X + (size_t)g0 * KIN;
      const int pre = min(nb, S);
      for (int b = 0; b < pre; ++b) {
        const uint32_t bar = ptx::smem_addr(&full[b]);
        ptx::mbar_arrive_expect_tx(bar, BB + XB);
        ptx::bulk_g2s(ptx::smem_addr(stage(b)), wsrc + (size_t)b * BB, BB, bar);
      }
      grid_wait();
      for (int b = 0; b < pre; ++b)
        ptx::bulk_g2s(ptx::smem_addr(stage(b) + BB), xsrc + (size_t)b * KIN, XB,
                      ptx::smem_addr(&full[b]));
      int issued = pre;
      const int nbi = a.stall ? pre : nb;  // read once: the waits below clobber memory
      RingPos rp{pre % S, (uint32_t)(pre / S) & 1u};
      for (int b = pre; b < nbi; ++b, rp.next(S)) {
        const int s = rp.s;
        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), rp.ph ^ 1u)) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
          break;
        }
        const uint32_t bar = ptx::smem_addr(&full[s]);
        ptx::mbar_arrive_expect_tx(bar, BB + XB);
        ptx::bulk_g2s(ptx::smem_addr(stage(s)), wsrc + (size_t)b * BB, BB, bar);
        ptx::bulk_g2s(ptx::smem_addr(stage(s) + BB), xsrc + (size_t)b * KIN, XB, bar);
        issued = b + 1;
      }
      for (int b = max(0, issued - S); b < issued; ++b)
        ptx::mbar_wait(ptx::smem_addr(&full[b % S]), (b / S) & 1);
    }
    __syncwarp();
  } else if (warp >= kLutWarp) {
    // ---------------------------------------------------------------- tables
    // Nibble set c = 8w + n of a block (w = 32-input word, n = nibble): inputs k0 + {0, 2, 4, 6}
    // with k0 = 32w + 8n (n < 4, even inputs) or 32w + 8(n - 4) + 1 (n >= 4, odd inputs).
    // Lane l tabulates sets l, l + 32, ... (one per 128 inputs of the block).
    if (hdr_ok) {
      RingPos rp{0, 0u};
      const int nbs = a.stall ? min(nb, S) : nb;  // read once: the waits below clobber memory
      for (int b = 0; b < nbs; ++b, rp.next(S)) {
        const int s = rp.s;
        if (s % kLutWarps != warp - kLutWarp) continue;  // this warp's stages only
        const bool landed = ptx::mbar_wait(ptx::smem_addr(&full[s]), rp.ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
          if (lane == 0) {
            record_error(a.err, LOWBIT_ERR_TIMEOUT);
            gave_up = 1;
          }
          break;
        }
        const uint16_t* xr = reinterpret_cast<const uint16_t*>(stage(s) + BB);
#pragma unroll
        for (int half = 0; half < KIN / kGroup; ++half) {
          const int c = lane + 32 * half, w = c >> 3, n = c & 7;
          const int k0 = 32 * w + (n < 4 ? 8 * n : 8 * (n - 4) + 1);
          const float x0 = bf16_bits_to_float(xr[k0]), x1 = bf16_bits_to_float(xr[k0 + 2]);
          const float x2 = bf16_bits_to_float(xr[k0 + 4]), x3 = bf16_bits_to_float(xr[k0 + 6]);
          float e[16];
          e[0] = -((x0 + x1) + (x2 + x3));  // every sign -1
          const float d0 = 2.f * x0, d1 = 2.f * x1, d2 = 2.f * x2, d3 = 2.f * x3;
#pragma unroll
          for (int m = 1; m < 16; ++m) {  // set bit j of m flips input j to +1
            const int low = m & -m;
            const float d = low == 1 ? d0 : (low == 2 ? d1 : (low == 4 ? d2 : d3));
            e[m] = e[m & (m - 1)] + d;
          }
          float4* t = reinterpret_cast<float4*>(stage(s) + BB + XB) + 4 * c;
          t[0] = make_float4(e[0], e[1], e[2], e[3]);
          t[1] = make_float4(e[4], e[5], e[6], e[7]);
          t[2] = make_float4(e[8], e[9], e[10], e[11]);
          t[3] = make_float4(e[12], e[13], e[14], e[15]);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&tabready[s]));
      }
    }
  } else if (hdr_ok) {
    // ---------------------------------------------------------------- compute
    // Warp (q, h): rows 32q..32q+31, sign words 2h and 2h+1 (inputs 64h..64h+63) of each plane.
    const int q = warp & 3, h = warp >> 2;
    const int row = 32 * q + lane;
    float total = 0.f;
    RingPos rp{0, 0u};
    const int nbc = stalled_out(a, ptx::smem_addr(&never), a.err, gave_up, lane) ? 0 : nb;
    for (int b = 0; b < nbc; ++b, rp.next(S)) {
      const int s = rp.s;
      const bool ready = ptx::mbar_wait(ptx::smem_addr(&tabready[s]), rp.ph);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        if (lane == 0) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
        }
        break;
      }
      const uint8_t* st = stage(s);
      if constexpr (!SA) {
        // inputs 64h..64h+63: sign words 2h, 2h+1 of each plane, nibble sets 16h..16h+15
        const uint32_t tab = ptx::smem_addr(st + BB + XB) + 16 * 16 * 4 * h;
        for (int p = 0; p < P; ++p) {
          const uint2 sw = *reinterpret_cast<const uint2*>(st + p * (kRowTile * 16) + row * 16 + h * 8);
          const float al = half_bits_to_float(
              *reinterpret_cast<const uint16_t*>(st + binplane_alpha_off(P) + (p * kRowTile + row) * 2));
          float acc[2] = {0.f, 0.f};
          lut_word(sw.x, tab, acc);
          lut_word(sw.y, tab + 8 * 64, acc);
          total = fmaf(al, acc[0] + acc[1], total);
        }
      } else {
        // inputs 128h..128h+127: sign words 4h..4h+3 of each plane (the 16 bytes of half h),
        // nibble sets 32h..32h+31; code group of word w is (128h + 32w) / G.
        const float* tab = reinterpret_cast<const float*>(st + BB + XB) + 32 * 16 * h;
        const uint8_t* codes = st + sa_code_off(P) + row;
        const int GJ = kSuper >> (31 - __clz(GS));  // code groups per block (G a power of two)
        float sb = 0.f;  // sum_p sum_g a[p][g] * (sum of the selected activations of group g)
        for (int p = 0; p < P; ++p) {
          const uint4 sw = *reinterpret_cast<const uint4*>(st + (p * 2 + h) * (kRowTile * 16) + row * 16);
          const uint8_t* ap = codes + p * GJ * kRowTile;
          float acc[2] = {0.f, 0.f};
          lut_word(sw.x, tab, acc);
          lut_word(sw.y, tab + 8 * 16, acc);
          if (GS == 64) {  // words 0-1 and 2-3 of the half carry different codes
            sb = fmaf((float)ap[(2 * h) * kRowTile], acc[0] + acc[1], sb);
            acc[0] = acc[1] = 0.f;
          }
          lut_word(sw.z, tab + 16 * 16, acc);
          lut_word(sw.w, tab + 24 * 16, acc);
          const int gl = GS == 64 ? 2 * h + 1 : (GS == 128 ? h : 0);
          sb = fmaf((float)ap[gl * kRowTile], acc[0] + acc[1], sb);
        }
        const uint32_t doff = sa_code_off(P) + (uint32_t)(P * GJ) * kRowTile;  // d of the rows
        total = fmaf(half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + doff + row * 2)), sb, total);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
    }
    red[warp][lane] = total;
  }

  // -------------------------------------------------------------------- reduction + store
  __syncthreads();
  const bool out_ok = ok != 0 && !gave_up;  // header verified, every wait completed
  if (!out_ok && live && threadIdx.x == 0 && rank == 0 && tile == 0)
    record_error(a.err, LOWBIT_ERR_INVALID_ARG);
  if (threadIdx.x < kRowTile) {
    const int q = threadIdx.x >> 5, l = threadIdx.x & 31;
    part[threadIdx.x] = red[q][l] + red[q + 4][l];
  }
  const int n = tile * kRowTile + (int)threadIdx.x;
  if (C > 1) ptx::cluster_wait();
  if (ks > 1) {
    float* slots = reinterpret_cast<float*>(smem + (size_t)S * SB);  // [ks-1][128]
    const uint32_t owner = (uint32_t)(crank - rank);
    if (live && threadIdx.x < kRowTile) {
      if (rank != 0) {
        // A CTA that gave up on a wait stays out of rank 0's shared memory: rank 0 may have
        // stopped waiting for it and exited.
        if (gave_up) return;
        const uint32_t la = ptx::smem_addr(&slots[(rank - 1) * kRowTile + threadIdx.x]);
        ptx::st_dsmem_f32(ptx::map_to_rank(la, owner), part[threadIdx.x]);
        ptx::mbar_arrive_remote(ptx::map_to_rank(ptx::smem_addr(&redbar), owner));
      } else {
        // under the stall setting no push can still be coming (see the INT4 kernel)
        const bool got = ptx::mbar_wait_cluster(ptx::smem_addr(&redbar), 0, a.stall ? kStallLimit : kWaitLimit);
        if (!got) record_error(a.err, LOWBIT_ERR_TIMEOUT);
        float y = part[threadIdx.x];
        for (int r = 1; r < ks; ++r) y += slots[(r - 1) * kRowTile + threadIdx.x];
        grid_wait();
        if (got && out_ok && n < pr.N) pr.Y[n] = float_to_bf16_bits(y);
      }
    }
  } else {
    __syncthreads();
    if (out_ok && threadIdx.x < kRowTile) {
      grid_wait();
      if (n < pr.N) pr.Y[n] = float_to_bf16_bits(part[threadIdx.x]);
    }
  }
}

__global__ void __launch_bounds__(kBpThreads)
bp_stream_kernel(const __grid_constant__ StreamArgs a) {
  plane_stream_body<false>(a);
}

// The deployed ShiftAdd format at M = 1 (ShiftAddQwen README, "Format": alpha = d * a).
__global__ void __launch_bounds__(kBpThreads)
sa_stream_kernel(const __grid_constant__ StreamArgs a) {
  plane_stream_body<true>(a);
}

// ------------------------------------------------------------------------------ NVFP4, M = 1
// The trimmed draft head of the small-vocabulary MTP study (section 3.3) at one token: NVFP4
// weights (E2M1 codes, an E4M3 scale per 16 inputs, an fp32 tensor scale g) streamed as the
// INT4 kernel streams its blocks, against the same int16 activations.
//
// Decoding without tables: each code is taken as u = 2 * e2m1 + 12 in 0..24, found by two byte
// permutes per four codes.  One permute selects from the eight u of the positive codes, whose
// bytes are all below 0x80, so a code with its sign bit set -- which prmt reads as "replicate
// the byte's sign" -- yields 0; the other permute does the same for the negative codes with
// the sign bits flipped; their OR is u.  The integer dot product of a run of 16 is then
// sum x * u - 12 * sum x, exact, and the run is scaled by its E4M3 scale in fp32.
constexpr uint32_t kNvStage = kNvfp4Block + kXBytes;
constexpr uint32_t kUPosLo = 0x0F0E0D0Cu, kUPosHi = 0x18141210u;  // 12 + {0,1,2,3 | 4,6,8,12}
constexpr uint32_t kUNegLo = 0x090A0B0Cu, kUNegHi = 0x00040608u;  // 12 - {0,1,2,3 | 4,6,8,12}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// E4M3 byte -> its value times 2^-120, exactly: the byte's exponent and mantissa fields placed
// in a float's bit positions give a float with exponent e - 127 (e >= 1) or the subnormal
// m * 2^-129 (e = 0); 0x7F / 0xFF are NaN.
__device__ __forceinline__ float e4m3_down120(uint32_t b) {
  const uint32_t bits = ((b << 24) & 0x80000000u) | ((b & 0x7Fu) << 20);
  return (b & 0x7Fu) == 0x7Fu ? __uint_as_float(0x7FC00000u) : __uint_as_float(bits);
}

template <int EPI>
__global__ void __launch_bounds__(stream_threads<1>())
nvfp4_stream_kernel(const __grid_constant__ StreamArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t xready[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ __align__(8) uint64_t redbar;
  __shared__ __align__(8) uint64_t never;  // nothing arrives on it (test-only stall setting)
  __shared__ __align__(16) uint32_t xq[kMaxStages][kGroup / 2];  // int16 pairs (X[2i], X[2i+1])
  __shared__ float xdown[kMaxStages][2];                          // 2^-sh of inputs 0..63, 64..127
  __shared__ __align__(16) int xsum[kMaxStages][kGroup / 16];      // sum X of each run of 16
  __shared__ float red[kCWarps][32];
  __shared__ float part[kRowTile];
  __shared__ int ok;
  __shared__ int gave_up;
  __shared__ int tile_got;   // rank 0 of a split tile: every peer's partial sums arrived
  __shared__ int hdr_valid;  // the whole grid agrees on it: every CTA reads the same header
  __shared__ float gscale;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster, lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);
  const GemvProblem& pr = a.p[0];  // one matrix per launch
  const int ks = pr.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);
  const int tile = ((cid - pr.cluster_begin) << (lc - lk)) + (crank >> lk);
  const int G = pr.K / kGroup;
  const bool live = tile < row_tiles(pr.N);
  const int g0 = (rank * G) >> lk, g1 = ((rank + 1) * G) >> lk;
  const int nb = live ? g1 - g0 : 0;
  const int S = a.stages;
  const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(pr.packed);

  if (threadIdx.x == 0) {
    ok = live && (pr.early || header_matches(hp, kFormatNvfp4, 0, pr.N, pr.K));
    gave_up = 0;
    tile_got = 1;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&xready[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kCWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&redbar), (uint32_t)(kRowTile * (ks > 1 ? ks - 1 : 1)));
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_mbar_init();
  }
  if (warp < kCWarps) red[warp][lane] = 0.f;
  __syncthreads();
  if (C > 1) ptx::cluster_arrive();
  if (threadIdx.x == 0) grid_launch();
  const bool hdr_ok = ok != 0;
  if (threadIdx.x == 0) {
    // every CTA, live or not, checks the header: the argmax epilogue's CTA count depends on it
    hdr_valid = header_matches(hp, kFormatNvfp4, 0, pr.N, pr.K);
    if (!hdr_valid) ok = 0;
    gscale = __uint_as_float(__ldg(reinterpret_cast<const uint32_t*>(hp) + 14));
  }

  if (warp == kCWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && hdr_ok) {
      const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * kNvfp4Block;
      const uint16_t* xsrc = pr.X + (size_t)g0 * kGroup;
      const int pre = min(nb, S);
      for (int b = 0; b < pre; ++b) {
        const uint32_t bar = ptx::smem_addr(&full[b]);
        ptx::mbar_arrive_expect_tx(bar, kNvStage);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * kNvStage), wsrc + (size_t)b * kNvfp4Block,
                      kNvfp4Block, bar);
      }
      grid_wait();  // the activations may be the previous kernel's output
      for (int b = 0; b < pre; ++b)
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * kNvStage + kNvfp4Block), xsrc + (size_t)b * kGroup,
                      kXBytes, ptx::smem_addr(&full[b]));
      int issued = pre;
      const int nbi = a.stall ? pre : nb;  // read once: the waits below clobber memory
      RingPos rp{pre % S, (uint32_t)(pre / S) & 1u};
      for (int b = pre; b < nbi; ++b, rp.next(S)) {
        const int s = rp.s;
        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), rp.ph ^ 1u)) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
          break;
        }
        const uint32_t bar = ptx::smem_addr(&full[s]);
        ptx::mbar_arrive_expect_tx(bar, kNvStage);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * kNvStage), wsrc + (size_t)b * kNvfp4Block,
                      kNvfp4Block, bar);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * kNvStage + kNvfp4Block),
                      xsrc + (size_t)b * kGroup, kXBytes, bar);
        issued = b + 1;
      }
      for (int b = max(0, issued - S); b < issued; ++b)
        ptx::mbar_wait(ptx::smem_addr(&full[b % S]), (b / S) & 1);
    }
    __syncwarp();
  } else if (warp >= kConvWarp) {
    // ---------------------------------------------------------------- activation converters
    // converter c owns the stages s with s % 2 == c (each stage's phases met in order)
    if (hdr_ok) {
      RingPos rp{0, 0u};
      const int nbs = a.stall ? min(nb, S) : nb;  // read once: the waits below clobber memory
      for (int b = 0; b < nbs; ++b, rp.next(S)) {
        const int s = rp.s;
        if (s % conv_warps<1>() != warp - kConvWarp) continue;
        const bool landed = ptx::mbar_wait(ptx::smem_addr(&full[s]), rp.ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
          if (lane == 0) {
            record_error(a.err, LOWBIT_ERR_TIMEOUT);
            gave_up = 1;
          }
          break;
        }
        const uint2 raw = reinterpret_cast<const uint2*>(ring + (size_t)s * kNvStage + kNvfp4Block)[lane];
        const Converted cv = convert_run64(raw, lane);
        reinterpret_cast<uint2*>(xq[s])[lane] = make_uint2(cv.i0 | (cv.i1 << 16), cv.i2 | (cv.i3 << 16));
        int sum = (int)(int16_t)cv.i0 + (int)(int16_t)cv.i1 + (int)(int16_t)cv.i2 + (int)(int16_t)cv.i3;
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        if ((lane & 3) == 0) xsum[s][lane >> 2] = sum;
        if ((lane & 15) == 0) xdown[s][lane >> 4] = cv.down;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&xready[s]));
      }
    }
  } else if (warp < kCWarps && hdr_ok) {
    // ---------------------------------------------------------------- compute
    // Warp (q, h): rows 32q..32q+31, inputs 64h..64h+63 (chunks 2h, 2h+1; scale runs 4h..4h+3)
    const int q = warp & 3, h = warp >> 2;
    const int row = 32 * q + lane;
    float total = 0.f;
    RingPos rp{0, 0u};
    const int nbc = stalled_out(a, ptx::smem_addr(&never), a.err, gave_up, lane) ? 0 : nb;
    for (int b = 0; b < nbc; ++b, rp.next(S)) {
      const int s = rp.s;
      const bool ready = ptx::mbar_wait(ptx::smem_addr(&xready[s]), rp.ph);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        if (lane == 0) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
        }
        break;
      }
      const uint8_t* st = ring + (size_t)s * kNvStage;
      const uint4 c0 = *reinterpret_cast<const uint4*>(st + (2 * h) * (kRowTile * 16) + row * 16);
      const uint4 c1 = *reinterpret_cast<const uint4*>(st + (2 * h + 1) * (kRowTile * 16) + row * 16);
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint4* xw = reinterpret_cast<const uint4*>(xq[s]) + 8 * h;  // 4 pairs per code word
      const int4 sx = *reinterpret_cast<const int4*>(&xsum[s][4 * h]);
      const int sxs[4] = {sx.x, sx.y, sx.z, sx.w};
      float sub = 0.f;  // sum over the four runs of 16: e4m3 * 2^-120 * (integer dot product)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int acc0 = -12 * sxs[j], acc1 = 0;
#pragma unroll
        for (int i = 2 * j; i < 2 * j + 2; ++i) {
          const uint32_t wf = w[i] ^ 0x88888888u;
          const uint32_t lo = prmt(kUPosLo, kUPosHi, w[i]) | prmt(kUNegLo, kUNegHi, wf);
          const uint32_t hi = prmt(kUPosLo, kUPosHi, w[i] >> 16) | prmt(kUNegLo, kUNegHi, wf >> 16);
          const uint4 x = xw[i];
          acc0 = dp2a_lo(x.x, lo, acc0);
          acc1 = dp2a_hi(x.y, lo, acc1);
          acc0 = dp2a_lo(x.z, hi, acc0);
          acc1 = dp2a_hi(x.w, hi, acc1);
        }
        sub = fmaf(e4m3_down120(st[kNvfp4ScaleOff + (4 * h + j) * kRowTile + row]), (float)(acc0 + acc1), sub);
      }
      const float down = xdown[s][h];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
      total = fmaf(0.5f * down, sub * 0x1p120f, total);  // u - 12 is 2 * e2m1
    }
    red[warp][lane] = total;
  }

  // -------------------------------------------------------------------- reduction + output
  __syncthreads();
  const bool out_ok = ok != 0 && !gave_up;  // header verified, every wait completed
  if (!out_ok && live && threadIdx.x == 0 && rank == 0 && tile == 0)
    record_error(a.err, LOWBIT_ERR_INVALID_ARG);
  if (threadIdx.x < kRowTile) {
    const int q = threadIdx.x >> 5, l = threadIdx.x & 31;
    part[threadIdx.x] = red[q][l] + red[q + 4][l];
  }
  const int n = tile * kRowTile + (int)threadIdx.x;
  if (C > 1) ptx::cluster_wait();
  bool have = false;  // this thread holds row n's complete sum in y
  float y = 0.f;
  if (ks > 1) {
    float* slots = reinterpret_cast<float*>(ring + (size_t)S * kNvStage);  // [ks-1][128]
    const uint32_t owner = (uint32_t)(crank - rank);
    if (live && threadIdx.x < kRowTile) {
      if (rank != 0) {
        // a CTA that gave up on a wait stays out of rank 0's shared memory
        if (!gave_up) {
          const uint32_t la = ptx::smem_addr(&slots[(rank - 1) * kRowTile + threadIdx.x]);
          ptx::st_dsmem_f32(ptx::map_to_rank(la, owner), part[threadIdx.x]);
          ptx::mbar_arrive_remote(ptx::map_to_rank(ptx::smem_addr(&redbar), owner));
        }
      } else {
        // under the stall setting no push can still be coming (see the INT4 kernel)
        const bool got = ptx::mbar_wait_cluster(ptx::smem_addr(&redbar), 0, a.stall ? kStallLimit : kWaitLimit);
        if (!got) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          tile_got = 0;
        }
        y = part[threadIdx.x];
        for (int r = 1; r < ks; ++r) y += slots[(r - 1) * kRowTile + threadIdx.x];
        have = got && out_ok && n < pr.N;
      }
    }
  } else {
    __syncthreads();
    if (threadIdx.x < kRowTile) {
      y = part[threadIdx.x];
      have = out_ok && n < pr.N;
    }
  }
  y *= gscale;
  if constexpr (EPI == 0) {
    if (have) {
      grid_wait();
      pr.Y[n] = float_to_bf16_bits(y);
    }
  } else {
    if (hdr_valid) {
      grid_wait();  // the previous call on this workspace has reset it
      if (warp < kRowTile / 32) {  // warps 0..3 hold the tile's rows
        unsigned long long key = have ? argmax_key(y, n) : 0ull;
        key = warp_max_u64(key);
        if (lane == 0 && key) atomicMax(&a.ws->keys[0], key);
      }
      // a live tile whose sums are incomplete (a wait gave up here or in a peer) fails the call
      __syncthreads();
      draft_finish(a.ws, 1, a.id_map, a.ids, live && (gave_up || (ks > 1 && rank == 0 && !tile_got)));
    }
  }
}

// ------------------------------------------------------------------------------ Q8, M = 1
// The trimmed draft head in 8 bits (small-vocabulary MTP study, section 3.3, the Q8 arm of its
// table; w = d * q, int8 q, one fp16 d per 32 inputs) streamed as the INT4 kernel streams its
// blocks, against the same int16 activations.  Each code word holds four signed bytes in input
// order, so two integer dot products (16-bit x signed 8-bit, two products added into 32 bits)
// take a word against the two activation pairs it meets; a run of 32 inputs (below 2^27 in
// magnitude, so its fp32 value is within 2^-24 of exact) is scaled by its d in fp32.
constexpr uint32_t kQ8Stage = kQ8Block + kXBytes;

__device__ __forceinline__ int dp2a_lo_s8(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_s8(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int EPI>
__global__ void __launch_bounds__(stream_threads<1>())
q8_stream_kernel(const __grid_constant__ StreamArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t xready[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ __align__(8) uint64_t redbar;
  __shared__ __align__(8) uint64_t never;  // nothing arrives on it (test-only stall setting)
  __shared__ __align__(16) uint32_t xq[kMaxStages][kGroup / 2];  // int16 pairs (X[2i], X[2i+1])
  __shared__ float xdown[kMaxStages][2];                          // 2^-sh of inputs 0..63, 64..127
  __shared__ float red[kCWarps][32];
  __shared__ float part[kRowTile];
  __shared__ int ok;
  __shared__ int gave_up;
  __shared__ int tile_got;   // rank 0 of a split tile: every peer's partial sums arrived
  __shared__ int hdr_valid;  // the whole grid agrees on it: every CTA reads the same header

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster, lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);
  const GemvProblem& pr = a.p[0];  // one matrix per launch
  const int ks = pr.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);
  const int tile = ((cid - pr.cluster_begin) << (lc - lk)) + (crank >> lk);
  const int G = pr.K / kGroup;
  const bool live = tile < row_tiles(pr.N);
  const int g0 = (rank * G) >> lk, g1 = ((rank + 1) * G) >> lk;
  const int nb = live ? g1 - g0 : 0;
  const int S = a.stages;
  const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(pr.packed);

  if (threadIdx.x == 0) {
    ok = live && (pr.early || header_matches(hp, kFormatQ8, 0, pr.N, pr.K));
    gave_up = 0;
    tile_got = 1;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&xready[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kCWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&redbar), (uint32_t)(kRowTile * (ks > 1 ? ks - 1 : 1)));
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_mbar_init();
  }
  if (warp < kCWarps) red[warp][lane] = 0.f;
  __syncthreads();
  if (C > 1) ptx::cluster_arrive();
  if (threadIdx.x == 0) grid_launch();
  const bool hdr_ok = ok != 0;
  if (threadIdx.x == 0) {
    // every CTA, live or not, checks the header: the argmax epilogue's CTA count depends on it
    hdr_valid = header_matches(hp, kFormatQ8, 0, pr.N, pr.K);
    if (!hdr_valid) ok = 0;
  }

  if (warp == kCWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && hdr_ok) {
      const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * kQ8Block;
      const uint16_t* xsrc = pr.X + (size_t)g0 * kGroup;
      const int pre = min(nb, S);
      for (int b = 0; b < pre; ++b) {
        const uint32_t bar = ptx::smem_addr(&full[b]);
        ptx::mbar_arrive_expect_tx(bar, kQ8Stage);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * kQ8Stage), wsrc + (size_t)b * kQ8Block,
                      kQ8Block, bar);
      }
      grid_wait();  // the activations may be the previous kernel's output
      for (int b = 0; b < pre; ++b)
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * kQ8Stage + kQ8Block), xsrc + (size_t)b * kGroup,
                      kXBytes, ptx::smem_addr(&full[b]));
      int issued = pre;
      const int nbi = a.stall ? pre : nb;  // read once: the waits below clobber memory
      RingPos rp{pre % S, (uint32_t)(pre / S) & 1u};
      for (int b = pre; b < nbi; ++b, rp.next(S)) {
        const int s = rp.s;
        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), rp.ph ^ 1u)) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
          break;
        }
        const uint32_t bar = ptx::smem_addr(&full[s]);
        ptx::mbar_arrive_expect_tx(bar, kQ8Stage);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * kQ8Stage), wsrc + (size_t)b * kQ8Block,
                      kQ8Block, bar);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * kQ8Stage + kQ8Block),
                      xsrc + (size_t)b * kGroup, kXBytes, bar);
        issued = b + 1;
      }
      for (int b = max(0, issued - S); b < issued; ++b)
        ptx::mbar_wait(ptx::smem_addr(&full[b % S]), (b / S) & 1);
    }
    __syncwarp();
  } else if (warp >= kConvWarp) {
    // ---------------------------------------------------------------- activation converters
    // converter c owns the stages s with s % 2 == c (each stage's phases met in order)
    if (hdr_ok) {
      RingPos rp{0, 0u};
      const int nbs = a.stall ? min(nb, S) : nb;  // read once: the waits below clobber memory
      for (int b = 0; b < nbs; ++b, rp.next(S)) {
        const int s = rp.s;
        if (s % conv_warps<1>() != warp - kConvWarp) continue;
        const bool landed = ptx::mbar_wait(ptx::smem_addr(&full[s]), rp.ph);
        if (!__all_sync(0xFFFFFFFFu, landed)) {
          if (lane == 0) {
            record_error(a.err, LOWBIT_ERR_TIMEOUT);
            gave_up = 1;
          }
          break;
        }
        const uint2 raw = reinterpret_cast<const uint2*>(ring + (size_t)s * kQ8Stage + kQ8Block)[lane];
        const Converted cv = convert_run64(raw, lane);
        reinterpret_cast<uint2*>(xq[s])[lane] = make_uint2(cv.i0 | (cv.i1 << 16), cv.i2 | (cv.i3 << 16));
        if ((lane & 15) == 0) xdown[s][lane >> 4] = cv.down;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&xready[s]));
      }
    }
  } else if (warp < kCWarps && hdr_ok) {
    // ---------------------------------------------------------------- compute
    // Warp (q, h): rows 32q..32q+31, inputs 64h..64h+63 (chunks 4h..4h+3; scale runs 2h, 2h+1)
    const int q = warp & 3, h = warp >> 2;
    const int row = 32 * q + lane;
    float total = 0.f;
    RingPos rp{0, 0u};
    const int nbc = stalled_out(a, ptx::smem_addr(&never), a.err, gave_up, lane) ? 0 : nb;
    for (int b = 0; b < nbc; ++b, rp.next(S)) {
      const int s = rp.s;
      const bool ready = ptx::mbar_wait(ptx::smem_addr(&xready[s]), rp.ph);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        if (lane == 0) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
        }
        break;
      }
      const uint8_t* st = ring + (size_t)s * kQ8Stage;
      const uint2* xw = reinterpret_cast<const uint2*>(xq[s]) + 16 * h;  // pairs of 4 inputs
      float sub = 0.f;  // sum over the two runs of 32: d * (integer dot product)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(st + (4 * h + 2 * j) * (kRowTile * 16) + row * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(st + (4 * h + 2 * j + 1) * (kRowTile * 16) + row * 16);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        int acc0 = 0, acc1 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // word i: inputs 64h + 32j + 4i .. +3
          const uint2 x = xw[8 * j + i];
          acc0 = dp2a_lo_s8(x.x, w[i], acc0);
          acc1 = dp2a_hi_s8(x.y, w[i], acc1);
        }
        const float d = half_bits_to_float(
            *reinterpret_cast<const uint16_t*>(st + kQ8ScaleOff + (2 * h + j) * (kRowTile * 2) + row * 2));
        sub = fmaf(d, (float)(acc0 + acc1), sub);
      }
      const float down = xdown[s][h];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
      total = fmaf(down, sub, total);
    }
    red[warp][lane] = total;
  }

  // -------------------------------------------------------------------- reduction + output
  __syncthreads();
  const bool out_ok = ok != 0 && !gave_up;  // header verified, every wait completed
  if (!out_ok && live && threadIdx.x == 0 && rank == 0 && tile == 0)
    record_error(a.err, LOWBIT_ERR_INVALID_ARG);
  if (threadIdx.x < kRowTile) {
    const int q = threadIdx.x >> 5, l = threadIdx.x & 31;
    part[threadIdx.x] = red[q][l] + red[q + 4][l];
  }
  const int n = tile * kRowTile + (int)threadIdx.x;
  if (C > 1) ptx::cluster_wait();
  bool have = false;  // this thread holds row n's complete sum in y
  float y = 0.f;
  if (ks > 1) {
    float* slots = reinterpret_cast<float*>(ring + (size_t)S * kQ8Stage);  // [ks-1][128]
    const uint32_t owner = (uint32_t)(crank - rank);
    if (live && threadIdx.x < kRowTile) {
      if (rank != 0) {
        // a CTA that gave up on a wait stays out of rank 0's shared memory
        if (!gave_up) {
          const uint32_t la = ptx::smem_addr(&slots[(rank - 1) * kRowTile + threadIdx.x]);
          ptx::st_dsmem_f32(ptx::map_to_rank(la, owner), part[threadIdx.x]);
          ptx::mbar_arrive_remote(ptx::map_to_rank(ptx::smem_addr(&redbar), owner));
        }
      } else {
        // under the stall setting no push can still be coming (see the INT4 kernel)
        const bool got = ptx::mbar_wait_cluster(ptx::smem_addr(&redbar), 0, a.stall ? kStallLimit : kWaitLimit);
        if (!got) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          tile_got = 0;
        }
        y = part[threadIdx.x];
        for (int r = 1; r < ks; ++r) y += slots[(r - 1) * kRowTile + threadIdx.x];
        have = got && out_ok && n < pr.N;
      }
    }
  } else {
    __syncthreads();
    if (threadIdx.x < kRowTile) {
      y = part[threadIdx.x];
      have = out_ok && n < pr.N;
    }
  }
  if constexpr (EPI == 0) {
    if (have) {
      grid_wait();
      pr.Y[n] = float_to_bf16_bits(y);
    }
  } else {
    if (hdr_valid) {
      grid_wait();  // the previous call on this workspace has reset it
      if (warp < kRowTile / 32) {  // warps 0..3 hold the tile's rows
        unsigned long long key = have ? argmax_key(y, n) : 0ull;
        key = warp_max_u64(key);
        if (lane == 0 && key) atomicMax(&a.ws->keys[0], key);
      }
      // a live tile whose sums are incomplete (a wait gave up here or in a peer) fails the call
      __syncthreads();
      draft_finish(a.ws, 1, a.id_map, a.ids, live && (gave_up || (ks > 1 && rank == 0 && !tile_got)));
    }
  }
}

// ------------------------------------------------------------------------------ warp MMA, M <= 32
// The verify block (Efficient-Qwen report, section 2.2: the target checks a block of drafts
// in one pass; block size 16) on the warp-level tensor-core MMA: mma.sync m16n8k16, bf16
// operands, fp32 accumulation.  At this width a 16 x 8 output tile wastes no tensor work,
// while a 128-row tcgen05 MMA with N = 16 issues as slowly as one with N = 64, which caps a
// weight-streaming GEMM built on it near half of the HBM bandwidth.
//
// Same stream and schedule as the INT4 mat-vec.  A stage holds one (tile, group) block and
// the group's activations of every row: two TMA tile loads of 64 inputs x MT rows with the
// 128-byte swizzle (rows M..MT-1 zero-filled), so that the eight row addresses of an
// ldmatrix fall in distinct banks; a copy per row would cost the copy engine more than the
// block itself.  Compute warp w owns rows 16w..16w+15 of the tile: per 16
// inputs lane (g, t) unpacks pair t of two code words of rows 16w+g and 16w+g+8 -- exactly
// the A fragment of the MMA -- to exact bf16 q (the nibble ORed into bf16 128.0, minus 136),
// loads the activations' B fragments with ldmatrix and issues one MMA per 8 activation rows.
// After a group's 128 inputs it adds s * D to fp32 totals held in registers.
constexpr int kMmaInt4 = 0, kMmaPlanes = 1, kMmaSa = 2, kMmaQ8 = 3;  // weight formats of the warp-MMA kernels
// Inputs per block: a group of 128 (INT4, binary planes) or an sa super-block of 256.
__host__ __device__ constexpr int mma_kin(int fmt) { return fmt == kMmaSa ? kSuper : kGroup; }
// Stage layout: the block, then the activation tile (kin inputs x MT rows, 64-input swizzle
// atoms) at the next 1024-byte boundary.
__host__ __device__ constexpr uint32_t mma_block_bytes(int fmt, int P, int GS) {
  return fmt == kMmaInt4 ? kInt4Block
       : fmt == kMmaQ8 ? kQ8Block
       : fmt == kMmaPlanes ? (uint32_t)P * (kRowTile * 16 + kRowTile * 2)
       : (uint32_t)P * 2 * kRowTile * 16 + (uint32_t)P * (kSuper / GS) * kRowTile + kRowTile * 2;
}
__host__ __device__ constexpr uint32_t mma_x_off(int fmt, int P, int GS) {
  return (mma_block_bytes(fmt, P, GS) + 1023u) / 1024u * 1024u;
}
__host__ __device__ constexpr uint32_t mma_stage_bytes(int fmt, int P, int GS, int MT) {
  return mma_x_off(fmt, P, GS) + (uint32_t)MT * 2 * mma_kin(fmt);
}
// A pair of binary-plane signs -> the bf16 pair (+-1, +-1): bits 15 - sh and 31 - sh of w
// (set = +1) shifted onto the sign bits and XORed into bf16 (-1.0, -1.0), as one written-out
// logic op with immediate constants: the compiler's lowering of the expression took about
// twice the logic ops (with the written-out op binary planes at M=16 ran 11% faster and the
// sa format 9%).
__device__ __forceinline__ uint32_t pm1_pair_lop(uint32_t w, int sh) {
  uint32_t d;  // (x & mask) ^ bf16(-1.0, -1.0)
  asm("lop3.b32 %0, %1, 0x80008000, 0xBF80BF80, 0x6A;" : "=r"(d) : "r"(w << sh));
  return d;
}
constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;  // compute warps, producer
// Occupancy is what hides the fragment unpacking's latency: about 55 KB of shared memory per
// CTA keeps four CTAs (MT = 16; three for MT = 32, by registers) on an SM.
template <int MT> __host__ __device__ constexpr int mma_resident() { return MT == 16 ? 4 : 3; }
constexpr size_t kMmaSmemBudget = 56 * 1024;
// sa super-blocks with many planes need larger stages: two of them, fewer CTAs per SM
constexpr size_t kMmaSmemBudgetMax = 110 * 1024;

// Activations of every matrix of a launch as TMA tensor maps ([M][K] bf16, boxes of 64 inputs
// x MT rows); the maps precede the arguments shared with the other streaming kernels.
struct MmaArgs {
  CUtensorMap xmap[kMaxGemvProblems];
  StreamArgs s;
};
// Epilogues: bf16 outputs; the LM-head argmax + acceptance; one shard of a row-sharded LM head
// (the shard's best key per token); the draft head's id-mapped argmax.
constexpr int kEpiStore = 0, kEpiVerify = 1, kEpiKeys = 2, kEpiDraft = 3;

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t bf16x2_sub_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// The nibbles at bits 0..3 and 16..19 of a code word (inputs k and k+1) -> the bf16 pair
// (q[k], q[k+1]) exactly: 128 + u in bf16, minus 136.
__device__ __forceinline__ uint32_t q_pair(uint32_t w) {
  uint32_t u;  // one logic op: (w & mask) | bf16(128.0, 128.0); written out, since the
               // compiler's own lowering of this expression before the subtraction cost the
               // 248,320-row LM head 15% of its time
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(u) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
  return bf16x2_sub_rn(u, 0x43084308u);
}
// Two int8 codes (two's complement bytes of `w`) -> the exact bf16 pair (q, q').  One
// permute puts the two code bytes under the bf16 exponent byte 0x43; with bit 7 masked off a
// half is 128 + (q mod 128), and the byte's bit 7 (the code's sign) turns the subtrahend
// bf16 128.0 into 256.0, so one bf16 subtraction leaves q exactly: four ops per pair.
// sel: byte b of w to half 0, byte b + 1 to half 1, 0x43 above each.
__device__ __forceinline__ uint32_t q8_pair(uint32_t w, uint32_t sel) {
  uint32_t r, v, s;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(0x43434343u), "r"(sel));
  asm("lop3.b32 %0, %1, 0xFF7FFF7F, 0, 0xC0;" : "=r"(v) : "r"(r));      // r & mask
  asm("lop3.b32 %0, %1, 0x00800080, 0x43004300, 0xEA;" : "=r"(s) : "r"(r));  // (r & m) | c
  return bf16x2_sub_rn(v, s);
}

template <int FMT, int MT, int EPI>
__device__ __forceinline__ void mma_body(const MmaArgs& A) {
  constexpr int NT = MT / 8;  // MMA output tiles of 8 activation rows
  const StreamArgs& a = A.s;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned tiles
  uint8_t* ring = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ __align__(8) uint64_t empty[kMaxStages];
  __shared__ __align__(8) uint64_t never;  // nothing arrives on it (test-only stall setting)
  __shared__ int ok;
  __shared__ int gave_up;
  __shared__ int hdr_valid;  // the same in every CTA: they all read the one header
  __shared__ unsigned long long kmax[MT];  // verify: this CTA's best key per activation row
  __shared__ uint32_t peer_gave_up[kMaxSplit];  // written by the split-K peers of this tile
  // Totals [MT][128], written once every stage has been consumed: they reuse the ring (the
  // launcher allocates at least MT * 512 bytes).  After a timed-out wait a late copy may still
  // land there; the outputs are wrong then anyway and the error word says so.
  float (*part)[kRowTile] = reinterpret_cast<float (*)[kRowTile]>(ring);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.cluster, lc = __ffs(C) - 1;  // C and every ks are powers of two
  const int cid = (int)blockIdx.x >> lc, crank = (int)blockIdx.x & (C - 1);
  int pi = 0;
  for (int i = 1; i < a.count; ++i)
    if (cid >= a.cl_begin[i]) pi = i;
  const GemvProblem& pr = a.p[pi];
  const int ks = pr.ks, lk = __ffs(ks) - 1, rank = crank & (ks - 1);
  const int tile = ((cid - pr.cluster_begin) << (lc - lk)) + (crank >> lk);
  constexpr int KIN = mma_kin(FMT), NATOM = KIN / 64;
  const int G = pr.K / KIN;  // blocks along K
  const bool live = tile < row_tiles(pr.N);
  const int g0 = (rank * G) >> lk, g1 = ((rank + 1) * G) >> lk;
  const int nb = live ? g1 - g0 : 0;
  const int S = a.stages, M = a.m;
  const PackedHeader* hp = reinterpret_cast<const PackedHeader*>(pr.packed);
  const int P = FMT == kMmaInt4 ? 0 : pr.P, GS = FMT == kMmaSa ? pr.G : 0;
  const uint32_t BB = mma_block_bytes(FMT, P, GS), XOFF = mma_x_off(FMT, P, GS);
  const uint32_t STG = mma_stage_bytes(FMT, P, GS, MT);  // block, then the activation atoms
  auto header_ok = [&]() {
    return FMT == kMmaSa ? header_matches_sa(hp, P, GS, pr.N, pr.K)
                         : header_matches(hp, FMT == kMmaInt4 ? kFormatInt4
                                                : FMT == kMmaQ8 ? kFormatQ8 : kFormatBinplane,
                                          P, pr.N, pr.K);
  };

  if (threadIdx.x < MT) kmax[threadIdx.x] = 0ull;
  if (threadIdx.x == 0) {
    ok = live && (pr.early || header_ok());
    gave_up = 0;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&empty[s]), kMmaWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&never), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) grid_launch();
  const bool hdr_ok = ok != 0;  // with `early`: only "this CTA has work"; see out_ok below
  if (threadIdx.x == 32) {  // a compute warp checks the header; the producer does not wait on it
    const bool hv = header_ok();
    hdr_valid = hv;
    if (!hv) ok = 0;
  }

  if (a.stall) {
    // ---------------------------------------------------------------- test-only stall setting
    // The producer issues the first ring of copies and waits for them; the compute warps wait
    // on a barrier nothing arrives on, give up and leave their totals unwritten.  Kept apart
    // from the roles below so that normal operation runs exactly their code.
    if (warp == kMmaWarps) {
      if (hdr_ok && lane == 0) {
        const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * BB;
        const uint32_t tx = BB + MT * 2 * KIN;
        const int pre = min(nb, S);
        for (int b = 0; b < pre; ++b) {
          const uint32_t bar = ptx::smem_addr(&full[b]);
          ptx::mbar_arrive_expect_tx(bar, tx);
          ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * STG), wsrc + (size_t)b * BB, BB, bar);
        }
        grid_wait();
        for (int b = 0; b < pre; ++b) {
          const uint32_t dst = ptx::smem_addr(ring + (size_t)b * STG + XOFF);
#pragma unroll
          for (int at = 0; at < NATOM; ++at)
            ptx::tma_load_2d(dst + at * MT * 128, &A.xmap[pi], (g0 + b) * KIN + 64 * at, 0,
                             ptx::smem_addr(&full[b]));
        }
        for (int b = 0; b < pre; ++b) ptx::mbar_wait(ptx::smem_addr(&full[b]), 0u);
      }
      __syncwarp();
    } else if (hdr_ok) {
      stalled_out(a, ptx::smem_addr(&never), a.err, gave_up, lane);
    }
  } else if (warp == kMmaWarps) {
    // ---------------------------------------------------------------- producer
    if (hdr_ok && lane == 0) {
      const uint8_t* wsrc = pr.packed + kHeaderBytes + ((size_t)tile * G + g0) * BB;
      const CUtensorMap* xmap = &A.xmap[pi];
      const uint32_t tx = BB + MT * 2 * KIN;  // zero-filled rows count as copied
      auto copy_x = [&](int b, int s, uint32_t bar) {
        const uint32_t dst = ptx::smem_addr(ring + (size_t)s * STG + XOFF);
#pragma unroll
        for (int at = 0; at < NATOM; ++at)
          ptx::tma_load_2d(dst + at * MT * 128, xmap, (g0 + b) * KIN + 64 * at, 0, bar);
      };
      const int pre = min(nb, S);
      for (int b = 0; b < pre; ++b) {
        const uint32_t bar = ptx::smem_addr(&full[b]);
        ptx::mbar_arrive_expect_tx(bar, tx);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)b * STG), wsrc + (size_t)b * BB, BB, bar);
      }
      grid_wait();  // the activations may be the previous kernel's output
      for (int b = 0; b < pre; ++b) copy_x(b, b, ptx::smem_addr(&full[b]));
      int issued = pre;
      RingPos rp{pre % S, (uint32_t)(pre / S) & 1u};
      for (int b = pre; b < nb; ++b, rp.next(S)) {
        const int s = rp.s;
        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), rp.ph ^ 1u)) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
          break;
        }
        const uint32_t bar = ptx::smem_addr(&full[s]);
        ptx::mbar_arrive_expect_tx(bar, tx);
        ptx::bulk_g2s(ptx::smem_addr(ring + (size_t)s * STG), wsrc + (size_t)b * BB, BB, bar);
        copy_x(b, s, bar);
        issued = b + 1;
      }
      // copies still in flight must land before the CTA may exit
      for (int b = max(0, issued - S); b < issued; ++b)
        ptx::mbar_wait(ptx::smem_addr(&full[b % S]), (b / S) & 1);
    }
    __syncwarp();
  } else if (hdr_ok) {
    // ---------------------------------------------------------------- compute
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * warp + g;  // rows r0 and r0 + 8 of the tile
    // ldmatrix row of this lane: matrix lane/8 takes activation rows +8 and inputs +8.  In a
    // swizzled atom, 16-byte chunk c of row n sits at chunk c ^ (n % 8); the chunks a step
    // reads are 2 * (step % 4) + (inputs +8), so xsw[i] is the lane's address for step i % 4.
    const int xn = (lane & 7) + ((lane >> 4) << 3), xu = ((lane >> 3) & 1) ^ (lane & 7);
    uint32_t xsw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xsw[i] = (uint32_t)(xn * 128 + (((2 * i) ^ xu) << 4));
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    RingPos rp{0, 0u};
    for (int b = 0; b < nb; ++b, rp.next(S)) {
      const int s = rp.s;
      const bool landed = ptx::mbar_wait(ptx::smem_addr(&full[s]), rp.ph);
      if (!__all_sync(0xFFFFFFFFu, landed)) {
        if (lane == 0) {
          record_error(a.err, LOWBIT_ERR_TIMEOUT);
          gave_up = 1;
        }
        break;
      }
      const uint8_t* st = ring + (size_t)s * STG;
      const uint32_t xs = ptx::smem_addr(st + XOFF);
      if constexpr (FMT == kMmaInt4) {
        float d[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 32-input chunks
          const uint4 w0 = *reinterpret_cast<const uint4*>(st + c * (kRowTile * 16) + r0 * 16);
          const uint4 w1 = *reinterpret_cast<const uint4*>(st + c * (kRowTile * 16) + (r0 + 8) * 16);
          // word i holds inputs 8i..8i+7 of the chunk; pair t of it (inputs 8i+2t, 8i+2t+1) is
          // this lane's share, shifted down to nibble 0
          const uint32_t u0[4] = {w0.x >> (4 * t), w0.y >> (4 * t), w0.z >> (4 * t), w0.w >> (4 * t)};
          const uint32_t u1[4] = {w1.x >> (4 * t), w1.y >> (4 * t), w1.z >> (4 * t), w1.w >> (4 * t)};
#pragma unroll
          for (int j = 0; j < 2; ++j) {  // 16-input steps
            const uint32_t a0 = q_pair(u0[2 * j]), a1 = q_pair(u1[2 * j]);
            const uint32_t a2 = q_pair(u0[2 * j + 1]), a3 = q_pair(u1[2 * j + 1]);
#pragma unroll
            for (int hh = 0; hh < MT / 16; ++hh) {
              uint32_t b0, b1, b2, b3;
              // step 2c + j: atom c / 2, chunks 4 (c % 2) + 2j (+1)
              ldsm_x4(xs + xsw[(2 * c + j) & 3] + (c >> 1) * (MT * 128) + hh * 16 * 128, b0, b1, b2, b3);
              mma_16816(d[2 * hh], a0, a1, a2, a3, b0, b1);
              mma_16816(d[2 * hh + 1], a0, a1, a2, a3, b2, b3);
            }
          }
        }
        const float s0 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + kInt4ScaleOff + r0 * 2));
        const float s1 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + kInt4ScaleOff + (r0 + 8) * 2));
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          acc[i][0] = fmaf(s0, d[i][0], acc[i][0]);
          acc[i][1] = fmaf(s0, d[i][1], acc[i][1]);
          acc[i][2] = fmaf(s1, d[i][2], acc[i][2]);
          acc[i][3] = fmaf(s1, d[i][3], acc[i][3]);
        }
      } else if constexpr (FMT == kMmaQ8) {
        // Q8 (int8 codes, fp16 d per run of 32 inputs): step ss is 16-input chunk ss; this
        // lane's A share is bytes 2(t&1), 2(t&1)+1 of words t>>1 and 2 + (t>>1) of the chunk
        // in rows r0 and r0 + 8.  The MMA sums of a run's two steps are scaled by its d.
        const uint32_t b0 = (uint32_t)(2 * (t & 1));
        const uint32_t sel = b0 | 0x4040u | ((b0 + 1u) << 8);  // code, 0x43, next code, 0x43
        float d[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
        for (int ss = 0; ss < 8; ++ss) {
          const uint8_t* cp = st + ss * (kRowTile * 16) + 4 * (t >> 1);
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(cp + r0 * 16);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(cp + (r0 + 8) * 16);
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(cp + r0 * 16 + 8);
          const uint32_t w3 = *reinterpret_cast<const uint32_t*>(cp + (r0 + 8) * 16 + 8);
          const uint32_t a0 = q8_pair(w0, sel), a1 = q8_pair(w1, sel);
          const uint32_t a2 = q8_pair(w2, sel), a3 = q8_pair(w3, sel);
#pragma unroll
          for (int hh = 0; hh < MT / 16; ++hh) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(xs + xsw[ss & 3] + (ss >> 2) * (MT * 128) + hh * 16 * 128, b0, b1, b2, b3);
            mma_16816(d[2 * hh], a0, a1, a2, a3, b0, b1);
            mma_16816(d[2 * hh + 1], a0, a1, a2, a3, b2, b3);
          }
          if (ss & 1) {  // the run's second step: fold d * D into the totals
            const uint8_t* sp = st + kQ8ScaleOff + (ss >> 1) * (kRowTile * 2);
            const float s0 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(sp + r0 * 2));
            const float s1 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(sp + (r0 + 8) * 2));
#pragma unroll
            for (int i = 0; i < NT; ++i) {
              acc[i][0] = fmaf(s0, d[i][0], acc[i][0]);
              acc[i][1] = fmaf(s0, d[i][1], acc[i][1]);
              acc[i][2] = fmaf(s1, d[i][2], acc[i][2]);
              acc[i][3] = fmaf(s1, d[i][3], acc[i][3]);
              d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
      } else if constexpr (FMT == kMmaPlanes) {
        // Binary planes: word w of a plane row covers inputs 32w..32w+31, bit i the sign of
        // 32w + 2i and bit 16 + i that of 32w + 2i + 1.  Step s's A fragment takes pairs
        // i = 8 (s % 2) + t and i + 4 of word s / 2.
        for (int p = 0; p < P; ++p) {
          float d[NT][4];
#pragma unroll
          for (int i = 0; i < NT; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
          for (int hw = 0; hw < 2; ++hw) {  // words 2hw, 2hw + 1 (fewer live registers)
            const uint2 w0 = *reinterpret_cast<const uint2*>(st + p * (kRowTile * 16) + r0 * 16 + 8 * hw);
            const uint2 w1 = *reinterpret_cast<const uint2*>(st + p * (kRowTile * 16) + (r0 + 8) * 16 + 8 * hw);
            const uint32_t W0[2] = {w0.x, w0.y}, W1[2] = {w1.x, w1.y};
#pragma unroll
            for (int sq = 0; sq < 4; ++sq) {
              const int ss = 4 * hw + sq;
              const int sh = 15 - 8 * (ss & 1) - t;  // bit i to bit 15
              const uint32_t a0 = pm1_pair_lop(W0[sq >> 1], sh), a1 = pm1_pair_lop(W1[sq >> 1], sh);
              const uint32_t a2 = pm1_pair_lop(W0[sq >> 1], sh - 4), a3 = pm1_pair_lop(W1[sq >> 1], sh - 4);
#pragma unroll
              for (int hh = 0; hh < MT / 16; ++hh) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(xs + xsw[ss & 3] + (ss >> 2) * (MT * 128) + hh * 16 * 128, b0, b1, b2, b3);
                mma_16816(d[2 * hh], a0, a1, a2, a3, b0, b1);
                mma_16816(d[2 * hh + 1], a0, a1, a2, a3, b2, b3);
              }
            }
          }
          const uint8_t* al = st + binplane_alpha_off(P) + p * (kRowTile * 2);
          const float s0 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(al + r0 * 2));
          const float s1 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(al + (r0 + 8) * 2));
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            acc[i][0] = fmaf(s0, d[i][0], acc[i][0]);
            acc[i][1] = fmaf(s0, d[i][1], acc[i][1]);
            acc[i][2] = fmaf(s1, d[i][2], acc[i][2]);
            acc[i][3] = fmaf(s1, d[i][3], acc[i][3]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
      } else {
        // sa format (ShiftAddQwen README, "Format"): a super-block of 256 inputs, per plane two
        // halves of 128 laid out as a binary plane; alpha = d * a with one u8 code a per plane
        // and group of GS inputs, so the MMA sums of every GS / 16 steps are folded with
        // d * a (exact in fp32: 8 x 11 significant bits).
        // G is 64, 128 or 256: code-group arithmetic by shifts (a runtime division per fold
        // cost as much as the fold itself)
        const int lg = 31 - __clz(GS), lfk = lg - 4, fk = 1 << lfk;  // steps per code group
        const int gj = kSuper >> lg;                                  // code groups per block
        const uint32_t doff = sa_code_off(P) + (uint32_t)(P * gj) * kRowTile;
        const float d0 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + doff + r0 * 2));
        const float d1 = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + doff + (r0 + 8) * 2));
        for (int p = 0; p < P; ++p) {
          float d[NT][4];
#pragma unroll
          for (int i = 0; i < NT; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(st + (p * 2 + hb) * (kRowTile * 16) + r0 * 16);
            const uint4 w1 = *reinterpret_cast<const uint4*>(st + (p * 2 + hb) * (kRowTile * 16) + (r0 + 8) * 16);
            const uint32_t W0[4] = {w0.x, w0.y, w0.z, w0.w}, W1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ss = 0; ss < 8; ++ss) {
              const int kk = 8 * hb + ss;  // step within the super-block
              const int sh = 15 - 8 * (ss & 1) - t;
              const uint32_t a0 = pm1_pair_lop(W0[ss >> 1], sh), a1 = pm1_pair_lop(W1[ss >> 1], sh);
              const uint32_t a2 = pm1_pair_lop(W0[ss >> 1], sh - 4), a3 = pm1_pair_lop(W1[ss >> 1], sh - 4);
#pragma unroll
              for (int hh = 0; hh < MT / 16; ++hh) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(xs + xsw[kk & 3] + (kk >> 2) * (MT * 128) + hh * 16 * 128, b0, b1, b2, b3);
                mma_16816(d[2 * hh], a0, a1, a2, a3, b0, b1);
                mma_16816(d[2 * hh + 1], a0, a1, a2, a3, b2, b3);
              }
              if ((kk & (fk - 1)) == fk - 1) {  // the code group's last step
                const uint8_t* cd = st + sa_code_off(P) + (p * gj + (kk >> lfk)) * kRowTile;
                const float s0 = d0 * (float)cd[r0], s1 = d1 * (float)cd[r0 + 8];
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                  acc[i][0] = fmaf(s0, d[i][0], acc[i][0]);
                  acc[i][1] = fmaf(s0, d[i][1], acc[i][1]);
                  acc[i][2] = fmaf(s1, d[i][2], acc[i][2]);
                  acc[i][3] = fmaf(s1, d[i][3], acc[i][3]);
                  d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty[s]));
      }
    }
    // every warp has read its last stage before any total lands on the ring
    ptx::named_barrier(1, kMmaWarps * 32);
    // D element (row g | g + 8, column 2t | 2t + 1) of tile i: weight row r0 | r0 + 8,
    // activation row 8i + 2t | 8i + 2t + 1
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      part[8 * i + 2 * t][r0] = acc[i][0];
      part[8 * i + 2 * t + 1][r0] = acc[i][1];
      part[8 * i + 2 * t][r0 + 8] = acc[i][2];
      part[8 * i + 2 * t + 1][r0 + 8] = acc[i][3];
    }
  }

  // -------------------------------------------------------------------- reduction + output
  // The ks CTAs of a split tile reduce through distributed shared memory: rank r reads rows
  // r*128/ks .. (r+1)*128/ks - 1 of every peer's totals and finishes them.  Both cluster
  // barriers are reached by every CTA (its own waits are bounded), the second one keeping
  // each CTA's totals alive until its peers have read them.
  __syncthreads();
  const bool out_ok = ok != 0;
  if (!out_ok && live && threadIdx.x == 0 && rank == 0 && tile == 0)
    record_error(a.err, LOWBIT_ERR_INVALID_ARG);
  const bool owner_thread = threadIdx.x < kMmaWarps * 32;
  // The tile's totals are complete only if no CTA sharing it gave up on a wait: before the
  // cluster barrier, thread q stores this CTA's flag into split-K peer q's shared memory (the
  // barrier's release orders the stores); after it, each warp reads the ks flags it received.
  if (ks > 1 && threadIdx.x < (unsigned)ks)
    ptx::st_dsmem_u32(ptx::map_to_rank(ptx::smem_addr(&peer_gave_up[rank]),
                                       (uint32_t)(crank - rank + (int)threadIdx.x)),
                      (uint32_t)gave_up);
  if (C > 1) ptx::cluster_sync();
  const bool verify = EPI != kEpiStore && hdr_valid;
  bool tile_done = !gave_up;
  if (ks > 1) tile_done = !__any_sync(0xFFFFFFFFu, lane < ks && peer_gave_up[lane] != 0u);
  if (live && out_ok && tile_done && owner_thread) {
    grid_wait();  // outputs and the verify workspace belong to the previous kernel until now
    const int lr = 7 - lk, rows = kRowTile >> lk, rbase = rank * rows;
    const uint32_t base = (uint32_t)(crank - rank);  // rank 0 of this tile
    const int row0 = a.row_offset;  // read once: the loop's cluster loads clobber memory
    for (int i0 = 0; i0 < rows * MT; i0 += kMmaWarps * 32) {  // the same trip count in every lane
      const int idx = i0 + (int)threadIdx.x;
      const int m = idx >> lr, row = rbase + (idx & (rows - 1));
      const int n = tile * kRowTile + row;
      const bool in = idx < rows * MT && m < M && n < pr.N;
      float y = 0.f;
      if (in) {
        if (ks == 1) {
          y = part[m][row];
        } else {
          const uint32_t la = ptx::smem_addr(&part[m][row]);
          for (int q = 0; q < ks; ++q) y += ptx::ld_dsmem_f32(la, base + (uint32_t)q);
        }
      }
      if constexpr (EPI == kEpiStore) {
        if (in) pr.Y[(size_t)m * pr.N + n] = float_to_bf16_bits(y);
      } else {
        unsigned long long key = in ? argmax_key(y, n + row0) : 0ull;
        if (rows >= 32) {  // a warp's 32 values share one activation row
          key = warp_max_u64(key);
          if (lane == 0 && key) atomicMax(&kmax[min(m, MT - 1)], key);
        } else if (key) {
          atomicMax(&kmax[m], key);
        }
      }
    }
  }
  if (C > 1) ptx::cluster_sync();
  if (verify) {
    // one global atomic per activation row and CTA
    __syncthreads();
    grid_wait();
    if (threadIdx.x < M && kmax[threadIdx.x]) atomicMax(&a.ws->keys[threadIdx.x], kmax[threadIdx.x]);
    // a live tile whose totals are incomplete fails the call: nothing is written
    if constexpr (EPI == kEpiKeys)
      keys_finish(a.ws, M, a.keys_out, live && !tile_done);
    else if constexpr (EPI == kEpiDraft)
      draft_finish(a.ws, M, a.id_map, a.ids, live && !tile_done);
    else
      lmhead_finish(a.ws, M, a.draft, a.ids, a.n_accept, a.bonus, live && !tile_done);
  }
}

template <int MT, int EPI>
__global__ void __launch_bounds__(kMmaThreads, mma_resident<MT>())
int4_mma_kernel(const __grid_constant__ MmaArgs A) {
  mma_body<kMmaInt4, MT, EPI>(A);
}

// The same for binary planes (ShiftAddQwen README, "Method"): one MMA set per plane on exact
// +-1 fragments, alpha per (plane, row, group) applied in fp32.
template <int MT>
__global__ void __launch_bounds__(kMmaThreads, mma_resident<MT>())
bp_mma_kernel(const __grid_constant__ MmaArgs A) {
  mma_body<kMmaPlanes, MT, kEpiStore>(A);
}

// And for Q8 weights (the 8-bit draft head): bf16 outputs or the id-mapped argmax.
template <int MT, int EPI>
__global__ void __launch_bounds__(kMmaThreads, mma_resident<MT>())
q8_mma_kernel(const __grid_constant__ MmaArgs A) {
  mma_body<kMmaQ8, MT, EPI>(A);
}

// And for the deployed sa format: super-blocks of 256 inputs, alpha = d * a per code group.
template <int MT>
__global__ void __launch_bounds__(kMmaThreads, mma_resident<MT>())
sa_mma_kernel(const __grid_constant__ MmaArgs A) {
  mma_body<kMmaSa, MT, kEpiStore>(A);
}

int sm_count() {
  int dev = 0, nsm = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  return nsm;
}


// Schedule shared by the streaming kernels (blocks of `kin` inputs): ks per matrix aims at
// `target` blocks per
// CTA, then all splits are doubled while the doubled grid still fits the SMs' resident
// capacity (small launches).  Matrices are ordered by blocks per CTA, longest first.  Fills `a` and returns
// the cluster size C, the number of clusters, the largest blocks-per-CTA and the largest ks.
struct Schedule {
  int C, maxnb, kmax;
  long long clusters;
};

// Every split ks, and so the cluster size C, is a power of two (doubled from 1): the kernels
// place a CTA with shifts and masks.
bool make_schedule(const GemvProblem* probs, int count, int kin, int target, int max_split,
                   StreamArgs& a, Schedule& out, int resident_per_sm = kResidentPerSm) {
  static_assert((kMaxSplit & (kMaxSplit - 1)) == 0 && kRowTile == 128, "shift-based placement");
  const int nsm = sm_count();
  int ks[kMaxGemvProblems];
  long long ctas = 0;
  for (int i = 0; i < count; ++i) {
    const int G = probs[i].K / kin;
    int k = 1;
    while (k < max_split && k * 2 <= G && (G + k - 1) / k > target) k *= 2;
    ks[i] = k;
    ctas += (long long)row_tiles(probs[i].N) * k;
  }
  // Double every split while the doubled grid still fits the SMs' resident capacity: more
  // concurrent streams, each with fewer blocks.
  const long long resident = (long long)resident_per_sm * nsm;
  for (bool grew = true; grew;) {
    grew = false;
    long long next = 0;
    for (int i = 0; i < count; ++i) {
      const bool can = ks[i] < max_split && ks[i] * 2 <= probs[i].K / kin;
      next += (long long)row_tiles(probs[i].N) * ks[i] * (can ? 2 : 1);
    }
    if (next == ctas || next > resident) break;
    for (int i = 0; i < count; ++i)
      if (ks[i] < max_split && ks[i] * 2 <= probs[i].K / kin) ks[i] *= 2;
    ctas = next;
    grew = true;
  }
  int C = 1;
  for (int i = 0; i < count; ++i) C = ks[i] > C ? ks[i] : C;
  int order[kMaxGemvProblems];
  for (int i = 0; i < count; ++i) order[i] = i;
  auto per_cta = [&](int i) { return (probs[i].K / kin + ks[i] - 1) / ks[i]; };
  for (int i = 1; i < count; ++i)  // stable insertion sort: most blocks per CTA first
    for (int j = i; j > 0 && per_cta(order[j]) > per_cta(order[j - 1]); --j) {
      const int t = order[j];
      order[j] = order[j - 1];
      order[j - 1] = t;
    }
  long long clusters = 0;
  int maxnb = 1, kmax = 1;
  for (int i = 0; i < count; ++i) {
    const int o = order[i];
    a.p[i] = probs[o];
    a.p[i].ks = ks[o];
    a.p[i].cluster_begin = (int)clusters;
    a.cl_begin[i] = (int)clusters;
    const int tpc = C / ks[o];
    clusters += (row_tiles(probs[o].N) + tpc - 1) / tpc;
    maxnb = per_cta(o) > maxnb ? per_cta(o) : maxnb;
    kmax = ks[o] > kmax ? ks[o] : kmax;
  }
  if (clusters * C > 0x7FFFFFFFLL) return false;
  a.count = count;
  a.cluster = C;
  out.C = C;
  out.clusters = clusters;
  out.maxnb = maxnb;
  out.kmax = kmax;
  return true;
}

// Kernel attributes a launch may need: dynamic shared memory beyond the default (48 KB
// minus the kernel's static shared memory) and clusters above 8 CTAs.  An attribute holds
// for every later launch on the device, so each kernel asks once per device, for the whole
// per-CTA budget.
constexpr int kMaxDevices = 64;
struct OptIns {
  std::atomic<unsigned char> done[kMaxDevices];
};
OptIns g_int4_optins[3], g_bp_optins, g_sa_optins, g_nv_optins[2], g_q8_optins[2],
    g_mma_optins[14];  // one per kernel built

template <typename Kernel>
cudaError_t opt_in(Kernel kern, OptIns& o, size_t budget) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDevices && o.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && dev < kMaxDevices) o.done[dev].store(1, std::memory_order_release);
  return e;
}

template <typename Kernel, typename Args>
cudaError_t launch_streaming(Kernel kern, OptIns& o, size_t budget, const Args& a,
                             const Schedule& sc, size_t smem, int threads, cudaStream_t s) {
  if (smem > budget) return cudaErrorInvalidValue;
  cudaError_t e = opt_in(kern, o, budget);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sc.clusters * sc.C), 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (sc.C > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)sc.C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

namespace {

template <int MT>
cudaError_t launch_int4_stream_mt(const GemvProblem* probs, int count, int M, int* err,
                                  cudaStream_t s) {
  constexpr uint32_t stage = kInt4Block + MT * kXBytes;
  // Shared memory a row beyond the first adds to the kernel's static part (converted
  // activations, reduction buffers): the ring's budget shrinks by as much.  The split-K slots
  // grow with the rows; the ring keeps what they leave (at least two stages).
  constexpr size_t budget = kInt4SmemBudget - (size_t)(MT - 1) * 3200;
  StreamArgs a = {};
  Schedule sc;
  if (!make_schedule(probs, count, kGroup, kInt4TargetBlocks, kMaxSplit, a, sc))
    return cudaErrorInvalidValue;
  a.err = err;
  a.m = M;
  a.stall = debug_stall();
  // ring, then the partial-sum slots rank 0 of a split tile receives
  const size_t slots = (size_t)(sc.kmax - 1) * MT * kRowTile * sizeof(float);
  int S = slots < budget ? (int)((budget - slots) / stage) : 0;
  S = S > kMaxStages ? kMaxStages : (S < 2 ? 2 : S);
  S -= S % conv_warps<MT>();
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  const size_t smem = (size_t)a.stages * stage + slots;  // at most 2 * 9472 + 30720 bytes
  return launch_streaming(int4_stream_kernel<MT>, g_int4_optins[MT == 1 ? 0 : (MT == 2 ? 1 : 2)],
                          kSmemBudget, a, sc, smem, stream_threads<MT>(), s);
}

}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 x_map_encoder() {
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

template <int FMT, int MT, int EPI>
cudaError_t launch_mma_mt(const GemvProblem* probs, int count, int M, LmheadWorkspace* ws,
                          const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                          int32_t* bonus, int* err, cudaStream_t s,
                          unsigned long long* keys_out = nullptr, int row_offset = 0,
                          const int32_t* id_map = nullptr) {
  const int P = FMT == kMmaInt4 ? 0 : probs[0].P, GS = FMT == kMmaSa ? probs[0].G : 0;
  for (int i = 1; i < count; ++i)  // one stage size per launch
    if (FMT != kMmaInt4 && (probs[i].P != P || probs[i].G != probs[0].G)) return cudaErrorInvalidValue;
  const uint32_t stage = mma_stage_bytes(FMT, P, GS, MT);
  auto encode = x_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  MmaArgs A = {};
  StreamArgs& a = A.s;
  Schedule sc;
  if (!make_schedule(probs, count, mma_kin(FMT), FMT == kMmaSa ? kInt4TargetBlocks / 2 : kInt4TargetBlocks,
                     kMaxSplit, a, sc, mma_resident<MT>()))
    return cudaErrorInvalidValue;
  a.err = err;
  a.m = M;
  a.ws = ws;
  a.draft = draft;
  a.ids = argmax;
  a.n_accept = n_accept;
  a.bonus = bonus;
  a.keys_out = keys_out;
  a.row_offset = row_offset;
  a.id_map = id_map;
  a.stall = debug_stall();
  for (int i = 0; i < a.count; ++i) {
    // X [M][K] bf16 as matrix i's activations (in schedule order); rows >= M read as zero
    cuuint64_t dims[2] = {(cuuint64_t)a.p[i].K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)a.p[i].K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)MT};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&A.xmap[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.p[i].X),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const size_t budget = FMT == kMmaSa ? kMmaSmemBudgetMax : kMmaSmemBudget;
  int S = (int)((kMmaSmemBudget - 1024) / stage);  // aims at four CTAs per SM
  S = S > kMaxStages ? kMaxStages : (S < 2 ? 2 : S);
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  // the totals [MT][128] reuse the ring; 1 KB of slack aligns the ring
  const size_t smem = std::max((size_t)a.stages * stage, (size_t)MT * kRowTile * sizeof(float)) + 1024;
  if (smem > budget) return cudaErrorInvalidValue;
  if constexpr (FMT == kMmaInt4) {
    constexpr int slot_i = (MT == 16 ? 0 : 1) + (EPI == kEpiKeys ? 8 : 2 * EPI);
    return launch_streaming(int4_mma_kernel<MT, EPI>, g_mma_optins[slot_i], budget, A, sc, smem,
                            kMmaThreads, s);
  } else if constexpr (FMT == kMmaQ8) {
    constexpr int slot_q = 10 + (MT == 16 ? 0 : 1) + (EPI == kEpiDraft ? 2 : 0);
    return launch_streaming(q8_mma_kernel<MT, EPI>, g_mma_optins[slot_q], budget, A, sc, smem,
                            kMmaThreads, s);
  } else if constexpr (FMT == kMmaPlanes) {
    return launch_streaming(bp_mma_kernel<MT>, g_mma_optins[MT == 16 ? 4 : 5], budget, A, sc,
                            smem, kMmaThreads, s);
  } else {
    return launch_streaming(sa_mma_kernel<MT>, g_mma_optins[MT == 16 ? 6 : 7], budget, A, sc,
                            smem, kMmaThreads, s);
  }
}

}  // namespace

cudaError_t launch_int4_mma(const GemvProblem* probs, int count, int M, int* err, cudaStream_t s) {
  if (count < 1 || count > kMaxGemvProblems || M < 1 || M > 32) return cudaErrorInvalidValue;
  if (M <= 16)
    return launch_mma_mt<kMmaInt4, 16, kEpiStore>(probs, count, M, nullptr, nullptr, nullptr,
                                                  nullptr, nullptr, err, s);
  return launch_mma_mt<kMmaInt4, 32, kEpiStore>(probs, count, M, nullptr, nullptr, nullptr,
                                                nullptr, nullptr, err, s);
}

cudaError_t launch_sa_mma(const GemvProblem& prob, int M, int* err, cudaStream_t s) {
  if (M < 1 || M > 32 || prob.P < 1 || prob.P > 8) return cudaErrorInvalidValue;
  if (prob.G != 64 && prob.G != 128 && prob.G != 256) return cudaErrorInvalidValue;
  if (M <= 16)
    return launch_mma_mt<kMmaSa, 16, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                                nullptr, err, s);
  return launch_mma_mt<kMmaSa, 32, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                              nullptr, err, s);
}

cudaError_t launch_bp_mma(const GemvProblem& prob, int M, int* err, cudaStream_t s) {
  if (M < 1 || M > 32 || prob.P < 1 || prob.P > 8) return cudaErrorInvalidValue;
  if (M <= 16)
    return launch_mma_mt<kMmaPlanes, 16, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                                    nullptr, err, s);
  return launch_mma_mt<kMmaPlanes, 32, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                                  nullptr, err, s);
}

cudaError_t launch_lmhead_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws,
                              const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                              int32_t* bonus, int* err, cudaStream_t s) {
  if (M < 1 || M > 32) return cudaErrorInvalidValue;
  if (M <= 16)
    return launch_mma_mt<kMmaInt4, 16, kEpiVerify>(&prob, 1, M, ws, draft, argmax, n_accept, bonus,
                                                   err, s);
  return launch_mma_mt<kMmaInt4, 32, kEpiVerify>(&prob, 1, M, ws, draft, argmax, n_accept, bonus,
                                                 err, s);
}

cudaError_t launch_lmhead_keys_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws, int row_offset,
                                   unsigned long long* keys_out, int* err, cudaStream_t s) {
  if (M < 1 || M > 32) return cudaErrorInvalidValue;
  if (M <= 16)
    return launch_mma_mt<kMmaInt4, 16, kEpiKeys>(&prob, 1, M, ws, nullptr, nullptr, nullptr, nullptr,
                                                 err, s, keys_out, row_offset);
  return launch_mma_mt<kMmaInt4, 32, kEpiKeys>(&prob, 1, M, ws, nullptr, nullptr, nullptr, nullptr,
                                               err, s, keys_out, row_offset);
}

cudaError_t launch_q8_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws, const int32_t* id_map,
                          int32_t* ids, int* err, cudaStream_t s) {
  if (M < 1 || M > 32) return cudaErrorInvalidValue;
  if (!ws) {
    if (M <= 16)
      return launch_mma_mt<kMmaQ8, 16, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                                  nullptr, err, s);
    return launch_mma_mt<kMmaQ8, 32, kEpiStore>(&prob, 1, M, nullptr, nullptr, nullptr, nullptr,
                                                nullptr, err, s);
  }
  if (M <= 16)
    return launch_mma_mt<kMmaQ8, 16, kEpiDraft>(&prob, 1, M, ws, nullptr, ids, nullptr, nullptr, err,
                                                s, nullptr, 0, id_map);
  return launch_mma_mt<kMmaQ8, 32, kEpiDraft>(&prob, 1, M, ws, nullptr, ids, nullptr, nullptr, err, s,
                                              nullptr, 0, id_map);
}

cudaError_t launch_q8_stream(const GemvProblem& prob, LmheadWorkspace* ws, const int32_t* id_map,
                             int32_t* ids, int* err, cudaStream_t s) {
  StreamArgs a = {};
  Schedule sc;
  if (!make_schedule(&prob, 1, kGroup, kInt4TargetBlocks, kMaxSplit, a, sc)) return cudaErrorInvalidValue;
  a.err = err;
  a.m = 1;
  a.stall = debug_stall();
  a.ws = ws;
  a.id_map = id_map;
  a.ids = ids;
  const size_t slots = (size_t)(sc.kmax - 1) * kRowTile * sizeof(float);
  int S = slots < kInt4SmemBudget ? (int)((kInt4SmemBudget - slots) / kQ8Stage) : 0;
  S = S > kMaxStages ? kMaxStages : (S < 2 ? 2 : S);
  S -= S % conv_warps<1>();
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  const size_t smem = (size_t)a.stages * kQ8Stage + slots;
  if (ws) return launch_streaming(q8_stream_kernel<1>, g_q8_optins[1], kSmemBudget, a, sc, smem,
                                  stream_threads<1>(), s);
  return launch_streaming(q8_stream_kernel<0>, g_q8_optins[0], kSmemBudget, a, sc, smem,
                          stream_threads<1>(), s);
}

cudaError_t launch_int4_stream(const GemvProblem* probs, int count, int M, int* err, cudaStream_t s) {
  if (count < 1 || count > kMaxGemvProblems || M < 1 || M > kStreamMaxRows) return cudaErrorInvalidValue;
  if (M == 1) return launch_int4_stream_mt<1>(probs, count, M, err, s);
  if (M == 2) return launch_int4_stream_mt<2>(probs, count, M, err, s);
  return launch_int4_stream_mt<4>(probs, count, M, err, s);
}

cudaError_t launch_bp_stream(const GemvProblem* probs, int count, int* err, cudaStream_t s) {
  if (count < 1 || count > kMaxGemvProblems) return cudaErrorInvalidValue;
  StreamArgs a = {};
  Schedule sc;
  if (!make_schedule(probs, count, kGroup, kBpTargetBlocks, kMaxSplit, a, sc))
    return cudaErrorInvalidValue;
  int pmax = 1;
  for (int i = 0; i < count; ++i) pmax = probs[i].P > pmax ? probs[i].P : pmax;
  const size_t stage = binplane_block(pmax) + kXBytes + kLutBytes;
  const size_t slots = (size_t)(sc.kmax - 1) * kRowTile * sizeof(float);
  int S = (int)((kSmemBudget - slots) / stage);
  S = S < 2 ? 2 : (S > kMaxStages ? kMaxStages : S);
  S -= S % kLutWarps;  // the table warps share the stages evenly
  a.err = err;
  a.stall = debug_stall();
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  const size_t smem = (size_t)a.stages * stage + slots;
  return launch_streaming(bp_stream_kernel, g_bp_optins, kSmemBudget, a, sc, smem, kBpThreads, s);
}

cudaError_t launch_nvfp4_stream(const GemvProblem& prob, LmheadWorkspace* ws, const int32_t* id_map,
                                int32_t* ids, int* err, cudaStream_t s) {
  StreamArgs a = {};
  Schedule sc;
  if (!make_schedule(&prob, 1, kGroup, kInt4TargetBlocks, kMaxSplit, a, sc)) return cudaErrorInvalidValue;
  a.err = err;
  a.m = 1;
  a.stall = debug_stall();
  a.ws = ws;
  a.id_map = id_map;
  a.ids = ids;
  const size_t slots = (size_t)(sc.kmax - 1) * kRowTile * sizeof(float);
  int S = slots < kInt4SmemBudget ? (int)((kInt4SmemBudget - slots) / kNvStage) : 0;
  S = S > kMaxStages ? kMaxStages : (S < 2 ? 2 : S);
  S -= S % conv_warps<1>();
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  const size_t smem = (size_t)a.stages * kNvStage + slots;
  if (ws) return launch_streaming(nvfp4_stream_kernel<1>, g_nv_optins[1], kSmemBudget, a, sc, smem,
                                  stream_threads<1>(), s);
  return launch_streaming(nvfp4_stream_kernel<0>, g_nv_optins[0], kSmemBudget, a, sc, smem,
                          stream_threads<1>(), s);
}

cudaError_t launch_sa_stream(const GemvProblem* probs, int count, int* err, cudaStream_t s) {
  if (count < 1 || count > kMaxGemvProblems) return cudaErrorInvalidValue;
  StreamArgs a = {};
  Schedule sc;
  if (!make_schedule(probs, count, kSuper, kSaTargetBlocks, kMaxSplit, a, sc))
    return cudaErrorInvalidValue;
  size_t stage = 0;  // largest stage of the launch: block + activations + tables
  for (int i = 0; i < count; ++i) {
    const size_t st = sa_block(probs[i].P, probs[i].G) + kSuper * 2 + (kSuper / 4) * 16 * sizeof(float);
    stage = st > stage ? st : stage;
  }
  const size_t slots = (size_t)(sc.kmax - 1) * kRowTile * sizeof(float);
  int S = (int)((kSmemBudget > slots ? kSmemBudget - slots : 0) / stage);
  S = S < 2 ? 2 : (S > kMaxStages ? kMaxStages : S);
  S -= S % kLutWarps;  // the table warps share the stages evenly
  a.err = err;
  a.stall = debug_stall();
  a.stages = sc.maxnb < S ? sc.maxnb : S;
  const size_t smem = (size_t)a.stages * stage + slots;
  return launch_streaming(sa_stream_kernel, g_sa_optins, kSaSmemMax, a, sc, smem, kBpThreads, s);
}

}  // namespace lowbit

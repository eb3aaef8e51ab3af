// Internal definitions shared by the CUDA translation units of liblowbit.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lowbit.h"

namespace lowbit {

// ------------------------------------------------------------------ packed layout
constexpr uint32_t kMagic = 0x3242574Cu;  // "LWB2"
constexpr uint32_t kFormatInt4 = 1;
constexpr uint32_t kFormatBinplane = 2;
constexpr uint32_t kFormatSa = 3;
constexpr uint32_t kFormatNvfp4 = 4;
constexpr uint32_t kFormatQ8 = 5;
constexpr uint32_t kVersion = 2;
constexpr int kHeaderBytes = 128;
constexpr int kGroup = 128;    // inputs per quantisation group
constexpr int kRowTile = 128;  // weight rows per layout tile

struct PackedHeader {
  uint32_t magic, format, version, N, K, P, group, row_tile;
  uint64_t payload_offset, payload_bytes, block_bytes, reserved;
};
static_assert(sizeof(PackedHeader) == 64, "header layout");

__host__ __device__ inline int row_tiles(int N) { return (N + kRowTile - 1) / kRowTile; }

// The payload is one contiguous block per (128-row tile t, group g) at (t*(K/128) + g) * block.
// INT4 block: codes [4 chunks][128 rows][16 B] then scales [128 rows] fp16 = 8448 bytes.
constexpr uint32_t kInt4Block = 4 * kRowTile * 16 + kRowTile * 2;
constexpr uint32_t kInt4ScaleOff = 4 * kRowTile * 16;
// Binary-plane block: signs [P][128 rows][16 B] then alphas [P][128 rows] fp16.
__host__ __device__ inline uint32_t binplane_block(int P) { return (uint32_t)P * (kRowTile * 16 + kRowTile * 2); }
__host__ __device__ inline uint32_t binplane_alpha_off(int P) { return (uint32_t)P * kRowTile * 16; }

__host__ __device__ inline uint64_t int4_payload_bytes(int N, int K) {
  return (uint64_t)row_tiles(N) * (uint64_t)(K / kGroup) * kInt4Block;
}
__host__ __device__ inline uint64_t binplane_payload_bytes(int P, int N, int K) {
  return (uint64_t)row_tiles(N) * (uint64_t)(K / kGroup) * binplane_block(P);
}

// NVFP4: one block per (128-row tile, group of 128 inputs): the canonical code bytes (two E2M1
// codes per byte, low nibble = even input) [4 chunks][128 rows][16 B], then the E4M3 scales
// [8 per group][128 rows]; the fp32 tensor scale sits in the header's last u64 field.
constexpr uint32_t kNvfp4Block = 4 * kRowTile * 16 + 8 * kRowTile;
constexpr uint32_t kNvfp4ScaleOff = 4 * kRowTile * 16;
__host__ __device__ inline uint64_t nvfp4_payload_bytes(int N, int K) {
  return (uint64_t)row_tiles(N) * (uint64_t)(K / kGroup) * kNvfp4Block;
}

// Q8 (int8 codes, one fp16 scale per 32 inputs): one block per (128-row tile, group of 128
// inputs): the codes [8 chunks of 16 inputs][128 rows][16 B], then the scales [4 runs of 32
// inputs][128 rows] fp16.
constexpr uint32_t kQ8Block = 8 * kRowTile * 16 + 4 * kRowTile * 2;
constexpr uint32_t kQ8ScaleOff = 8 * kRowTile * 16;
__host__ __device__ inline uint64_t q8_payload_bytes(int N, int K) {
  return (uint64_t)row_tiles(N) * (uint64_t)(K / kGroup) * kQ8Block;
}

// The deployed ShiftAdd format: one block per (128-row tile, super-block of 256 inputs) holding
// signs [P][2 halves][128 rows][16 B], u8 scale codes [P][256/G groups][128 rows] and the
// rows' fp16 d [128].  G (inputs per scale code) is 64, 128 or 256.
constexpr int kSuper = 256;
__host__ __device__ inline uint32_t sa_code_off(int P) { return (uint32_t)P * 2 * kRowTile * 16; }
__host__ __device__ inline uint32_t sa_d_off(int P, int G) {
  return sa_code_off(P) + (uint32_t)P * (kSuper / G) * kRowTile;
}
__host__ __device__ inline uint32_t sa_block(int P, int G) { return sa_d_off(P, G) + kRowTile * 2; }
__host__ __device__ inline uint64_t sa_payload_bytes(int P, int G, int N, int K) {
  return (uint64_t)row_tiles(N) * (uint64_t)(K / kSuper) * sa_block(P, G);
}

// Kernel-side header check.  Returns true when the buffer holds (format, P, N, K).
__device__ __forceinline__ bool header_matches(const PackedHeader* h, uint32_t format, int P,
                                               int N, int K) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(h));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(h) + 1);
  return a.x == kMagic && a.y == format && a.z == kVersion && a.w == (uint32_t)N &&
         b.x == (uint32_t)K && b.y == (uint32_t)P;
}

// The same for the sa format, whose header also records the scale-code group G.
__device__ __forceinline__ bool header_matches_sa(const PackedHeader* h, int P, int G, int N, int K) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(h));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(h) + 1);
  return a.x == kMagic && a.y == kFormatSa && a.z == kVersion && a.w == (uint32_t)N &&
         b.x == (uint32_t)K && b.y == (uint32_t)P && b.z == (uint32_t)G;
}

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ small device helpers

// Streaming 16-byte load: weights are read once, so skip L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc_lo += lo(a) * lo(b), acc_hi += hi(a) * hi(b): bf16 x bf16 products added into fp32
// accumulators with one rounding each (sm_100+ mixed-precision fma).
__device__ __forceinline__ void fma_bf16x2_f32(float& acc_lo, float& acc_hi, uint32_t a,
                                               uint32_t b) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(a), "r"(b));
}

// INT4 nibble pair -> bf16x2 of (128 + u_even, 128 + u_odd): the nibbles sit at bits
// [4p, 4p+4) and [16+4p, 16+4p+4) of `word`; ORing a nibble into the low mantissa bits of
// bf16 128.0 (0x4300) gives 128 + u exactly.
template <int P>
__device__ __forceinline__ uint32_t int4_pair_biased(uint32_t word) {
  return ((word >> (4 * P)) & 0x000F000Fu) | 0x43004300u;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}
// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------------ launchers (host side)

// Host-side validation shared by the LM-head verify entry points (lmhead_argmax_verify and its
// variants): LOWBIT_OK or the status the call returns without enqueueing anything.
lowbit_status check_lmhead_args(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                const int32_t* draft, const int32_t* argmax, const int32_t* n_accept,
                                const int32_t* bonus, const void* workspace, size_t ws_bytes);

int* device_error_word();  // address of the current device's error word (nullptr on failure)

// The test-only stall setting (lowbit_debug_inject_stall): nonzero makes the streaming and
// warp-MMA launches that follow give up on their data waits.
int debug_stall();

// True when [p, p + bytes) lies inside one device allocation (driver range query); false when
// it does not or when the query is unavailable.
bool allocation_covers(const void* p, size_t bytes);

// One matrix of a streaming mat-vec launch (M = 1).  The launcher fills in the schedule.
// 64-byte aligned: a kernel reads one problem's fields from one cache line of its parameters.
struct alignas(64) GemvProblem {
  const uint16_t* X;       // [M][K] bf16
  const uint8_t* packed;   // header + INT4 payload for (N, K)
  uint16_t* Y;             // [M][N] bf16
  int N, K;
  int cluster_begin;       // first cluster of this matrix
  int ks;                  // CTAs that split one tile's groups (divides the cluster size)
  int early;               // 1: the payload is known to lie inside packed's allocation, so
                           //    weight copies may start before the header has been checked
  int P;                   // binary planes per weight (0 for INT4)
  int G;                   // sa format: inputs per scale code (64, 128 or 256)
};
constexpr int kMaxGemvProblems = 8;

cudaError_t launch_pack_int4(const int8_t* codes, const uint16_t* scales, int N, int K,
                             uint8_t* packed, cudaStream_t s);
cudaError_t launch_pack_binplane(const uint8_t* bits, const uint16_t* alpha, int P, int N, int K,
                                 uint8_t* packed, cudaStream_t s);
// INT4 streaming mat-vec for 1 <= M <= kStreamMaxRows activation rows (X [M][K], Y [M][N]).
// The library's default uses it up to kStreamDefaultRows rows (measured: at M = 2 it beats the
// tensor-core GEMM, at M = 4 it does not); path 1 reaches it up to kStreamMaxRows.
constexpr int kStreamMaxRows = 4;
constexpr int kStreamDefaultRows = 2;
cudaError_t launch_int4_stream(const GemvProblem* probs, int count, int M, int* err, cudaStream_t s);
// M = 1..32 on the warp-level tensor-core MMA (streaming skeleton): Y of every problem, or
// the LM-head verify epilogue (one problem; workspace as lmhead_argmax_verify).
cudaError_t launch_int4_mma(const GemvProblem* probs, int count, int M, int* err, cudaStream_t s);
// Binary planes (one matrix, P planes) on the same warp-level MMA kernel, 1 <= M <= 32.
cudaError_t launch_bp_mma(const GemvProblem& prob, int M, int* err, cudaStream_t s);
// The sa format (one matrix: P planes, code group G) on the same kernel, 1 <= M <= 32.
cudaError_t launch_sa_mma(const GemvProblem& prob, int M, int* err, cudaStream_t s);
struct LmheadWorkspace;
cudaError_t launch_lmhead_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws,
                              const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                              int32_t* bonus, int* err, cudaStream_t s);
// One shard of a row-sharded INT4 LM head (rows row_offset .. row_offset + N - 1 of the full
// vocabulary): keys_out[m] = the shard's best (logit, global row) key of token m.
cudaError_t launch_lmhead_keys_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws, int row_offset,
                                   unsigned long long* keys_out, int* err, cudaStream_t s);
// Binary-plane counterpart (M = 1); every problem carries its plane count P (1..8).
cudaError_t launch_bp_stream(const GemvProblem* probs, int count, int* err, cudaStream_t s);
// sa-format counterpart (M = 1); every problem carries P (1..8) and G (64, 128, 256).
cudaError_t launch_sa_stream(const GemvProblem* probs, int count, int* err, cudaStream_t s);
cudaError_t launch_pack_sa(const uint8_t* bits, const uint8_t* codes, const uint16_t* d, int P,
                           int G, int N, int K, uint8_t* packed, cudaStream_t s);
cudaError_t launch_sa_cc(const uint16_t* X, const uint8_t* packed, int P, int G, int M, int N,
                         int K, uint16_t* Y, int* err, cudaStream_t s);
struct LmheadWorkspace;
// NVFP4 at M = 1 (one matrix): bf16 logits into prob.Y when ws is null, else the draft head's
// id-mapped argmax (ids[0], workspace as lmhead_argmax_verify).
cudaError_t launch_nvfp4_stream(const GemvProblem& prob, LmheadWorkspace* ws, const int32_t* id_map,
                                int32_t* ids, int* err, cudaStream_t s);
cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int N, int K,
                             uint8_t* packed, cudaStream_t s);
cudaError_t launch_pack_q8(const int8_t* codes, const uint16_t* scales, int N, int K,
                           uint8_t* packed, cudaStream_t s);
// Q8 at M = 1 (one matrix): bf16 logits into prob.Y when ws is null, else the draft head's
// id-mapped argmax (ids[0], workspace as lmhead_argmax_verify).
cudaError_t launch_q8_stream(const GemvProblem& prob, LmheadWorkspace* ws, const int32_t* id_map,
                             int32_t* ids, int* err, cudaStream_t s);
// Q8 at 1 <= M <= 32 on the warp-level MMA: bf16 outputs into prob.Y when ws is null, else the
// id-mapped argmax of every row (ids[0..M)).
cudaError_t launch_q8_mma(const GemvProblem& prob, int M, LmheadWorkspace* ws, const int32_t* id_map,
                          int32_t* ids, int* err, cudaStream_t s);
cudaError_t launch_nvfp4_tc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                            uint16_t* Y, int* err, cudaStream_t s);
// Draft head: ids[m] = id_map[argmax_n logit[m][n]] (the row when id_map is null).
cudaError_t launch_draft_argmax_tc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                                   const int32_t* id_map, int32_t* ids, void* ws, int* err,
                                   cudaStream_t s);
cudaError_t launch_sa_tc(const uint16_t* X, const uint8_t* packed, int P, int G, int M, int N,
                         int K, uint16_t* Y, int* err, cudaStream_t s);
// Several INT4 multiplies with a common M >= 2 in one tensor-core launch (X, Y are [M][K], [M][N]).
cudaError_t launch_int4_tc_grouped(const GemvProblem* probs, int count, int M, int* err,
                                   cudaStream_t s);
cudaError_t launch_int4_gemm_cc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                                uint16_t* Y, int* err, cudaStream_t s);
cudaError_t launch_binplane_cc(const uint16_t* X, const uint8_t* packed, int P, int M, int N,
                               int K, uint16_t* Y, int* err, cudaStream_t s);
cudaError_t launch_int4_gemm_tc(const uint16_t* X, const uint8_t* packed, int M, int N, int K,
                                uint16_t* Y, int* err, cudaStream_t s);
cudaError_t launch_binplane_tc(const uint16_t* X, const uint8_t* packed, int P, int M, int N,
                               int K, uint16_t* Y, int* err, cudaStream_t s);
cudaError_t launch_lmhead_tc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                             const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                             int32_t* bonus, void* ws, int* err, cudaStream_t s);
cudaError_t launch_lmhead_cc(const uint16_t* H, const uint8_t* packed, int M, int N, int K,
                             const int32_t* draft, int32_t* argmax, int32_t* n_accept,
                             int32_t* bonus, void* ws, int* err, cudaStream_t s);

}  // namespace lowbit

// Offline repack kernels: canonical INT4 codes / binary sign planes / the deployed ShiftAdd
// format (sign planes with u8 scale codes and one fp16 d per 256 inputs) -> kernel layout.
//
// Efficient-Qwen report, section 2.1: INT4 codes under frozen symmetric per-group scales
// (group 128), served as W4A16.  ShiftAddQwen README, "Format" and "Layout": sign planes
// with per-group scales, written with bit-exact packing checks.  The layouts themselves are
// this library's (see include/lowbit.h): every (128-row tile, group of 128 inputs) is one
// contiguous block holding the tile's codes (rows side by side, so a warp's 16-byte-per-lane
// load of 32 rows is one 512-byte segment) followed by its scales, so a kernel can stage a
// whole block with a single bulk copy.
#include <string.h>

#include "common.cuh"

namespace lowbit {
namespace {

__device__ void write_header(uint8_t* packed, uint32_t format, int P, int N, int K, int group,
                             uint64_t payload_bytes, uint64_t block_bytes, uint64_t reserved) {
  PackedHeader h;
  h.magic = kMagic;
  h.format = format;
  h.version = kVersion;
  h.N = (uint32_t)N;
  h.K = (uint32_t)K;
  h.P = (uint32_t)P;
  h.group = (uint32_t)group;
  h.row_tile = kRowTile;
  h.payload_offset = kHeaderBytes;
  h.payload_bytes = payload_bytes;
  h.block_bytes = block_bytes;
  h.reserved = reserved;
  uint4* dst = reinterpret_cast<uint4*>(packed);
  const uint4* src = reinterpret_cast<const uint4*>(&h);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = src[i];
#pragma unroll
  for (int i = 4; i < kHeaderBytes / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
}

// One thread per 16-byte code unit (tile t, group g, chunk c, row r): 32 codes of row n,
// k = 128g + 32c .. +31, stored at block(t, g) + c*2048 + r*16.
__global__ void pack_int4_codes(const int8_t* __restrict__ codes, int N, int K,
                                uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int c4 = (int)(rest % 4);
  rest /= 4;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  const int c = 4 * g + c4;  // 32-input chunk index within the row
  uint32_t w[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};  // q = 0 padding
  if (n < N) {
    const uint4* src = reinterpret_cast<const uint4*>(codes + n * (long long)K + 32LL * c);
    uint4 v0 = src[0], v1 = src[1];
    const uint32_t b[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {  // k = 32c + 8i + e, e = 2p + o
        const uint32_t byte = (b[(8 * i + e) / 4] >> (8 * ((8 * i + e) % 4))) & 0xFFu;
        const uint32_t nib = (byte + 8u) & 0xFu;  // q + 8 (int8 two's complement)
        const int p = e >> 1, o = e & 1;
        word |= nib << (4 * p + 16 * o);
      }
      w[i] = word;
    }
  }
  uint8_t* dst = payload + (size_t)(t * G + g) * kInt4Block + (size_t)c4 * kRowTile * 16 + r * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// One thread per (tile, group, row) scale, stored at block(t, g) + 8192 + r*2.
__global__ void pack_int4_scales(const uint16_t* __restrict__ scales, int N, int K,
                                 uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  const long long tg = u / kRowTile;
  const int g = (int)(tg % G);
  const long long t = tg / G;
  const long long n = t * kRowTile + r;
  *reinterpret_cast<uint16_t*>(payload + (size_t)tg * kInt4Block + kInt4ScaleOff + r * 2) =
      (n < N) ? scales[n * G + g] : (uint16_t)0;
}

__global__ void pack_header(uint8_t* packed, uint32_t format, int P, int N, int K, int group,
                            unsigned long long payload_bytes, unsigned long long block_bytes,
                            unsigned long long reserved = 0) {
  if (threadIdx.x == 0 && blockIdx.x == 0)
    write_header(packed, format, P, N, K, group, payload_bytes, block_bytes, reserved);
}

// Even bits of a 32-bit word to its low half-word, odd bits to its high half-word.
__device__ __forceinline__ uint32_t split_even_odd(uint32_t x) {
  uint32_t e = x & 0x55555555u, o = (x >> 1) & 0x55555555u;
  e = (e | (e >> 1)) & 0x33333333u;  o = (o | (o >> 1)) & 0x33333333u;
  e = (e | (e >> 2)) & 0x0F0F0F0Fu;  o = (o | (o >> 2)) & 0x0F0F0F0Fu;
  e = (e | (e >> 4)) & 0x00FF00FFu;  o = (o | (o >> 4)) & 0x00FF00FFu;
  e = (e | (e >> 8)) & 0x0000FFFFu;  o = (o | (o >> 8)) & 0x0000FFFFu;
  return e | (o << 16);
}

// One thread per 16-byte unit (tile t, group g, plane p, row r) at block(t, g) + p*2048 + r*16.
__global__ void pack_binplane_codes(const uint8_t* __restrict__ bits, int P, int N, int K,
                                    uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int p = (int)(rest % P);
  rest /= P;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  uint4 v = make_uint4(0, 0, 0, 0);  // padding rows: all signs -1
  if (n < N) {
    const uint4 c = *reinterpret_cast<const uint4*>(bits + ((long long)p * N + n) * (K / 8) +
                                                    16LL * g);
    v = make_uint4(split_even_odd(c.x), split_even_odd(c.y), split_even_odd(c.z),
                   split_even_odd(c.w));
  }
  uint8_t* dst = payload + (size_t)(t * G + g) * binplane_block(P) + (size_t)p * kRowTile * 16 + r * 16;
  *reinterpret_cast<uint4*>(dst) = v;
}

// One thread per (tile, group, plane, row) scale at block(t, g) + 2048P + (p*128 + r)*2.
__global__ void pack_binplane_alpha(const uint16_t* __restrict__ alpha, int P, int N, int K,
                                    uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int p = (int)(rest % P);
  rest /= P;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  uint8_t* dst = payload + (size_t)(t * G + g) * binplane_block(P) + binplane_alpha_off(P) +
                 ((size_t)p * kRowTile + r) * 2;
  *reinterpret_cast<uint16_t*>(dst) = (n < N) ? alpha[((long long)p * N + n) * G + g] : (uint16_t)0;
}

// ---- sa format (ShiftAddQwen README, "Format"): block (t, j) per tile and super-block of 256.

// One thread per 16-byte unit (tile t, super-block j, plane p, half h, row r): the 128 signs of
// k = 256j + 128h .. +127, at block(t, j) + p*4096 + h*2048 + r*16, in the binary-plane word
// order (even inputs in the low half-word, odd inputs in the high half-word).
__global__ void pack_sa_signs(const uint8_t* __restrict__ bits, int P, int G, int N, int K,
                              uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int J = K / kSuper;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int h = (int)(rest % 2);
  rest /= 2;
  const int p = (int)(rest % P);
  rest /= P;
  const int j = (int)(rest % J);
  const long long t = rest / J;
  const long long n = t * kRowTile + r;
  uint4 v = make_uint4(0, 0, 0, 0);  // padding rows: all signs -1 (their d is 0)
  if (n < N) {
    const uint4 c = *reinterpret_cast<const uint4*>(bits + ((long long)p * N + n) * (K / 8) +
                                                    32LL * j + 16 * h);
    v = make_uint4(split_even_odd(c.x), split_even_odd(c.y), split_even_odd(c.z),
                   split_even_odd(c.w));
  }
  uint8_t* dst = payload + (size_t)(t * J + j) * sa_block(P, G) + ((size_t)p * 2 + h) * kRowTile * 16 +
                 r * 16;
  *reinterpret_cast<uint4*>(dst) = v;
}

// One thread per scale code (tile t, super-block j, plane p, group gl of the super-block, row r)
// at block(t, j) + 4096P + (p*(256/G) + gl)*128 + r.
__global__ void pack_sa_codes(const uint8_t* __restrict__ codes, int P, int G, int N, int K,
                              uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int J = K / kSuper, GJ = kSuper / G;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int gl = (int)(rest % GJ);
  rest /= GJ;
  const int p = (int)(rest % P);
  rest /= P;
  const int j = (int)(rest % J);
  const long long t = rest / J;
  const long long n = t * kRowTile + r;
  payload[(size_t)(t * J + j) * sa_block(P, G) + sa_code_off(P) + ((size_t)p * GJ + gl) * kRowTile + r] =
      (n < N) ? codes[((long long)p * N + n) * (K / G) + (long long)j * GJ + gl] : (uint8_t)0;
}

// One thread per (tile t, super-block j, row r) fp16 d at block(t, j) + sa_d_off + r*2.
__global__ void pack_sa_d(const uint16_t* __restrict__ d, int P, int G, int N, int K,
                          uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int J = K / kSuper;
  const int r = (int)(u % kRowTile);
  const long long tj = u / kRowTile;
  const long long n = (tj / J) * kRowTile + r;
  *reinterpret_cast<uint16_t*>(payload + (size_t)tj * sa_block(P, G) + sa_d_off(P, G) + r * 2) =
      (n < N) ? d[n * J + tj % J] : (uint16_t)0;
}

// ---- NVFP4 (E2M1 codes, an E4M3 scale per 16 inputs, an fp32 tensor scale).

// One thread per 16-byte unit (tile t, group g, chunk c, row r): the canonical code bytes of
// k = 128g + 32c .. +31 copied to block(t, g) + c*2048 + r*16.
__global__ void pack_nvfp4_codes(const uint8_t* __restrict__ codes, int N, int K,
                                 uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int c = (int)(rest % 4);
  rest /= 4;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  uint4 v = make_uint4(0, 0, 0, 0);  // padding rows: code 0 (+0)
  if (n < N) v = *reinterpret_cast<const uint4*>(codes + n * (long long)(K / 2) + 64LL * g + 16 * c);
  *reinterpret_cast<uint4*>(payload + (size_t)(t * G + g) * kNvfp4Block + (size_t)c * kRowTile * 16 +
                            r * 16) = v;
}

// One thread per scale byte (tile t, group g, sub-group j, row r) at block(t, g) + 8192 + j*128 + r.
__global__ void pack_nvfp4_scales(const uint8_t* __restrict__ scales, int N, int K,
                                  uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int j = (int)(rest % 8);
  rest /= 8;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  payload[(size_t)(t * G + g) * kNvfp4Block + kNvfp4ScaleOff + j * kRowTile + r] =
      (n < N) ? scales[n * (long long)(K / 16) + 8 * g + j] : (uint8_t)0;
}

// Q8: one thread per 16-byte code unit (tile t, group g, chunk c of 16 inputs, row r): the 16
// code bytes of row n, k = 128g + 16c .. +15, at block(t, g) + c*2048 + r*16.
__global__ void pack_q8_codes(const int8_t* __restrict__ codes, int N, int K,
                              uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int c = (int)(rest % 8);
  rest /= 8;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  uint4 v = make_uint4(0, 0, 0, 0);  // padding rows: code 0
  if (n < N) v = *reinterpret_cast<const uint4*>(codes + n * (long long)K + 128LL * g + 16 * c);
  *reinterpret_cast<uint4*>(payload + (size_t)(t * G + g) * kQ8Block + (size_t)c * kRowTile * 16 +
                            r * 16) = v;
}

// Q8: one thread per scale (tile t, group g, run j of 32 inputs, row r) at
// block(t, g) + 16384 + j*256 + r*2.
__global__ void pack_q8_scales(const uint16_t* __restrict__ scales, int N, int K,
                               uint8_t* __restrict__ payload, long long units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const int G = K / kGroup;
  const int r = (int)(u % kRowTile);
  long long rest = u / kRowTile;
  const int j = (int)(rest % 4);
  rest /= 4;
  const int g = (int)(rest % G);
  const long long t = rest / G;
  const long long n = t * kRowTile + r;
  *reinterpret_cast<uint16_t*>(payload + (size_t)(t * G + g) * kQ8Block + kQ8ScaleOff +
                               j * kRowTile * 2 + r * 2) =
      (n < N) ? scales[n * (long long)(K / 32) + 4 * g + j] : (uint16_t)0;
}

// Launched last by every pack call: the multiplies read their weights before their
// programmatic-dependency wait, so the kernel right before one must not be a weight writer.
__global__ void pack_done() {}

inline unsigned blocks_for(long long units, int threads) {
  return (unsigned)((units + threads - 1) / threads);
}

}  // namespace

cudaError_t launch_pack_int4(const int8_t* codes, const uint16_t* scales, int N, int K,
                             uint8_t* packed, cudaStream_t s) {
  const long long blocks = (long long)row_tiles(N) * (K / kGroup);
  const long long cu = blocks * 4 * kRowTile, su = blocks * kRowTile;
  pack_header<<<1, 32, 0, s>>>(packed, kFormatInt4, 0, N, K, kGroup, int4_payload_bytes(N, K),
                               kInt4Block);
  pack_int4_codes<<<blocks_for(cu, 256), 256, 0, s>>>(codes, N, K, packed + kHeaderBytes, cu);
  pack_int4_scales<<<blocks_for(su, 256), 256, 0, s>>>(scales, N, K, packed + kHeaderBytes, su);
  pack_done<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack_binplane(const uint8_t* bits, const uint16_t* alpha, int P, int N, int K,
                                 uint8_t* packed, cudaStream_t s) {
  const long long units = (long long)row_tiles(N) * (K / kGroup) * P * kRowTile;
  pack_header<<<1, 32, 0, s>>>(packed, kFormatBinplane, P, N, K, kGroup,
                               binplane_payload_bytes(P, N, K), binplane_block(P));
  pack_binplane_codes<<<blocks_for(units, 256), 256, 0, s>>>(bits, P, N, K, packed + kHeaderBytes, units);
  pack_binplane_alpha<<<blocks_for(units, 256), 256, 0, s>>>(alpha, P, N, K, packed + kHeaderBytes, units);
  pack_done<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack_sa(const uint8_t* bits, const uint8_t* codes, const uint16_t* d, int P,
                           int G, int N, int K, uint8_t* packed, cudaStream_t s) {
  const long long tj = (long long)row_tiles(N) * (K / kSuper);
  const long long su = tj * P * 2 * kRowTile, cu = tj * P * (kSuper / G) * kRowTile, du = tj * kRowTile;
  pack_header<<<1, 32, 0, s>>>(packed, kFormatSa, P, N, K, G, sa_payload_bytes(P, G, N, K),
                               sa_block(P, G));
  pack_sa_signs<<<blocks_for(su, 256), 256, 0, s>>>(bits, P, G, N, K, packed + kHeaderBytes, su);
  pack_sa_codes<<<blocks_for(cu, 256), 256, 0, s>>>(codes, P, G, N, K, packed + kHeaderBytes, cu);
  pack_sa_d<<<blocks_for(du, 256), 256, 0, s>>>(d, P, G, N, K, packed + kHeaderBytes, du);
  pack_done<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack_q8(const int8_t* codes, const uint16_t* scales, int N, int K,
                           uint8_t* packed, cudaStream_t s) {
  const long long blocks = (long long)row_tiles(N) * (K / kGroup);
  const long long cu = blocks * 8 * kRowTile, su = blocks * 4 * kRowTile;
  pack_header<<<1, 32, 0, s>>>(packed, kFormatQ8, 0, N, K, kGroup, q8_payload_bytes(N, K), kQ8Block);
  pack_q8_codes<<<blocks_for(cu, 256), 256, 0, s>>>(codes, N, K, packed + kHeaderBytes, cu);
  pack_q8_scales<<<blocks_for(su, 256), 256, 0, s>>>(scales, N, K, packed + kHeaderBytes, su);
  pack_done<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int N, int K,
                             uint8_t* packed, cudaStream_t s) {
  const long long blocks = (long long)row_tiles(N) * (K / kGroup);
  const long long cu = blocks * 4 * kRowTile, su = blocks * 8 * kRowTile;
  uint32_t gbits;
  memcpy(&gbits, &g, sizeof(gbits));
  pack_header<<<1, 32, 0, s>>>(packed, kFormatNvfp4, 0, N, K, kGroup, nvfp4_payload_bytes(N, K),
                               kNvfp4Block, gbits);
  pack_nvfp4_codes<<<blocks_for(cu, 256), 256, 0, s>>>(codes, N, K, packed + kHeaderBytes, cu);
  pack_nvfp4_scales<<<blocks_for(su, 256), 256, 0, s>>>(scales, N, K, packed + kHeaderBytes, su);
  pack_done<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

}  // namespace lowbit

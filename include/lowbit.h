/*
 * lowbit.h -- C ABI of liblowbit.so: weight-only low-bit GEMV/GEMM for speculative decoding
 * on GB300 (sm_103a).
 *
 * The library multiplies bf16 activation rows X[M][K] (M = 1 for plain decoding, M = 16 for
 * verifying a 16-token draft block) by a weight matrix W[N][K] stored in one of two low-bit
 * formats, and can fuse the vocabulary argmax and greedy draft acceptance into the LM-head
 * multiply.  Y = X * W^T is bf16 [M][N], accumulated in fp32.
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless the comment says otherwise.  bf16 and fp16 arrays
 *     are passed as uint16_t bit patterns.  Arrays are dense and row-major.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *     call only enqueues work on `stream` and returns; results are ready when the stream is.
 *   - The caller owns and allocates all memory; the library never allocates device memory.
 *   - Arguments are validated on the host before anything is enqueued; on error nothing is
 *     enqueued and no output is touched.  A CUDA launch error returns LOWBIT_ERR_CUDA.
 *   - K must be a multiple of 128 (the quantisation group).  N >= 1 is arbitrary.
 *   - Packed weight buffers start with a 128-byte header (magic, format, N, K, P).  Kernels
 *     check it against the call's arguments; on a mismatch they write no output and record
 *     LOWBIT_ERR_INVALID_ARG in a per-device error word that lowbit_device_error() returns.
 *     The M = 1 kernels may start reading weights before the header has been checked, but
 *     only when the host has verified that the payload the arguments describe lies inside
 *     the device allocation that contains `packed`; otherwise nothing but the header is read
 *     on a mismatch.  lowbit_validate_packed() checks a header synchronously.
 *   - Multiplies are launched with programmatic dependent launch: they request their packed
 *     weights (header included) before waiting for the preceding kernel on the stream, and
 *     read activations / write outputs only after that wait.  So the kernel immediately
 *     before a multiply on the same stream must not write that multiply's packed buffer.
 *     lowbit_pack_int4, lowbit_pack_binplane and lowbit_pack_sa end with an empty kernel,
 *     which makes "pack, then multiply" on one stream safe.
 *   - No C++ exception crosses this interface.
 */
#ifndef LOWBIT_H
#define LOWBIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lowbit_status {
  LOWBIT_OK = 0,
  LOWBIT_ERR_INVALID_ARG = 1, /* null pointer, negative size, wrong packed header */
  LOWBIT_ERR_SHAPE = 2,       /* K % 128 != 0, M outside 1..32, P outside 1..8, N < 1 */
  LOWBIT_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  LOWBIT_ERR_WORKSPACE = 4,   /* workspace missing or smaller than lmhead_workspace_bytes() */
  LOWBIT_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait gave up (recorded on the device) */
  LOWBIT_ERR_CUDA = 6         /* a CUDA runtime call or launch failed */
} lowbit_status;

/* Short English description of a status code (static string, never NULL). */
const char* lowbit_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int lowbit_version(void);

/* ------------------------------------------------------------------------------------------
 * Sizes (host-only, no CUDA call).  Return 0 for invalid shapes.
 */

/* Bytes of a packed INT4 buffer: 128-byte header + ceil(N/128)*128 rows of K/2 code bytes and
 * K/64 scale bytes.  For N a multiple of 128 the payload is exactly N*K/2 + N*K/64 bytes. */
size_t lowbit_int4_packed_bytes(int N, int K);

/* Bytes of a packed binary-plane buffer: header + ceil(N/128)*128 rows of P*K/8 sign bytes and
 * P*K/64 plane-scale bytes. */
size_t lowbit_binplane_packed_bytes(int P, int N, int K);

/* Bytes of a packed buffer of the deployed ShiftAdd format (lowbit_pack_sa): header +
 * ceil(N/128)*128 rows of P*K/8 sign bytes, P*K/G code bytes and K/128 bytes of d.  0 unless
 * K % 256 == 0, 1 <= P <= 8 and G is 64, 128 or 256. */
size_t lowbit_sa_packed_bytes(int P, int G, int N, int K);

/* Bytes of a packed NVFP4 buffer (lowbit_pack_nvfp4): header + ceil(N/128)*128 rows of K/2
 * code bytes and K/16 scale bytes. */
size_t lowbit_nvfp4_packed_bytes(int N, int K);

/* Bytes of a packed Q8 buffer (lowbit_pack_q8): header + ceil(N/128)*128 rows of K code bytes
 * and K/16 scale bytes (one fp16 per 32 inputs). */
size_t lowbit_q8_packed_bytes(int N, int K);

/* Bytes of the workspace lmhead_argmax_verify() needs (independent of N and K). */
size_t lmhead_workspace_bytes(int M, int N, int K);

/* ------------------------------------------------------------------------------------------
 * Offline repack (Efficient-Qwen report, section 2.1: codes rounded onto the INT4 grid under
 * frozen symmetric per-group scales, served as W4A16; ShiftAddQwen README, "Format" and
 * "Layout": binary planes with per-group scales and bit-exact packing).
 */

/* Repack canonical INT4 weights into the kernel layout.
 *   codes  : int8 [N][K], values in [-8, 7] (q of w = s*q); 16-byte aligned.  Values outside
 *            the range are out of contract: they are stored modulo 16.
 *   scales : fp16 [N][K/128], one symmetric scale per row and group of 128 inputs.
 *   packed : lowbit_int4_packed_bytes(N, K) bytes, 16-byte aligned; fully overwritten.
 * Layout of `packed` (little-endian): the header (magic 0x3242574C, format 1, version 2), then
 * rows in tiles of 128 (padding rows hold q = 0, scale 0).  Tile t and group g (inputs
 * 128g..128g+127) own one contiguous 8448-byte block at 128 + (t*(K/128) + g)*8448: for chunk
 * c = 0..3 and row r = n % 128 the 16 bytes at c*2048 + r*16 are four u32 words, word i
 * holding k = 128g + 32c + 8i + 2p + o (p = 0..3, o = 0..1) as the nibble q + 8 at bit
 * 4p + 16o; the fp16 scale s[n][g] sits at 8192 + r*2. */
lowbit_status lowbit_pack_int4(const int8_t* codes, const uint16_t* scales, int N, int K,
                               void* packed, void* stream);

/* Repack canonical binary planes (w = sum_p alpha_p * b_p, b in {-1,+1}).
 *   signbits : uint8 [P][N][K/8]; bit j (LSB first) of byte i is input k = 8i + j; 1 = +1.
 *   alpha    : fp16 [P][N][K/128], one scale per plane, row and group of 128 inputs.
 *   packed   : lowbit_binplane_packed_bytes(P, N, K) bytes, 16-byte aligned.
 * Layout: header (format 2), then tiles of 128 rows; tile t and group g own one contiguous
 * block of 2304*P bytes at 128 + (t*(K/128) + g)*2304*P: for plane p and row r = n % 128 the
 * 16 bytes at p*2048 + r*16 hold the 128 signs of k = 128g.. as four u32 words, word w
 * covering k0 = 128g + 32w with bit i = sign of k0 + 2i and bit 16 + i = sign of k0 + 2i + 1;
 * alpha[p][n][g] (fp16) sits at 2048*P + (p*128 + r)*2. */
lowbit_status lowbit_pack_binplane(const uint8_t* signbits, const uint16_t* alpha, int P, int N,
                                   int K, void* packed, void* stream);

/* Repack the deployed ShiftAdd format (ShiftAddQwen README, "Format": per super-block of 256
 * weights along the input dimension, Q sign planes, one u8 scale code per plane and group of G
 * weights, one fp16 scale d; alpha = d * a), so that
 *   w[n][k] = d[n][k/256] * sum_p a[p][n][k/G] * b[p][n][k],   b in {-1, +1}.
 *   signbits : uint8 [P][N][K/8], 16-byte aligned; bit j (LSB first) of byte i is input 8i + j;
 *              1 = +1.
 *   codes    : uint8 [P][N][K/G], the scale codes a (any alignment).
 *   d        : fp16 [N][K/256] (2-byte aligned).
 *   packed   : lowbit_sa_packed_bytes(P, G, N, K) bytes, 16-byte aligned; fully overwritten.
 *   1 <= P <= 8, G in {64, 128, 256}, K % 256 == 0 (else LOWBIT_ERR_SHAPE).
 * Layout: header (format 3, group field = G), then tiles of 128 rows; tile t and super-block
 * j (inputs 256j..256j+255) own one contiguous block of B = 4096P + 128P(256/G) + 256 bytes at
 * 128 + (t*(K/256) + j)*B: for plane p, half h and row r = n % 128 the 16 bytes at
 * p*4096 + h*2048 + r*16 hold the signs of k = 256j + 128h.. as four u32 words (word w covers
 * k0 = 256j + 128h + 32w: bit i = sign of k0 + 2i, bit 16 + i = sign of k0 + 2i + 1); the code
 * a[p][n][g] sits at 4096P + (p*(256/G) + g - j*(256/G))*128 + r, and d[n][j] (fp16) at
 * 4096P + 128P(256/G) + r*2.  Padding rows hold zero signs, codes and d. */
lowbit_status lowbit_pack_sa(const uint8_t* signbits, const uint8_t* codes, const uint16_t* d,
                             int P, int G, int N, int K, void* packed, void* stream);

/* Repack NVFP4 weights, the draft-head format of the small-vocabulary MTP study (section 3.3:
 * trim the head to the most used 32,768 tokens, quantise to NVFP4):
 *   w[n][k] = g * e4m3(scales[n][k/16]) * e2m1(code of k in row n).
 *   codes  : uint8 [N][K/2], 16-byte aligned; byte i holds inputs 2i (low nibble) and 2i + 1
 *            as 4-bit E2M1 codes (sign, two exponent bits with bias 1, one mantissa bit).
 *   scales : uint8 [N][K/16], E4M3 bytes (sign, four exponent bits with bias 7, three mantissa
 *            bits; 0x7F / 0xFF are NaN).       g : the fp32 tensor scale.
 *   packed : lowbit_nvfp4_packed_bytes(N, K) bytes, 16-byte aligned; fully overwritten.
 * Layout: header (format 4, the fp32 bits of g at byte 56), then per (tile t of 128 rows, group
 * j of 128 inputs) one block of 9216 bytes at 128 + (t*(K/128) + j)*9216: for chunk c = 0..3 and
 * row r the 16 code bytes of inputs 128j + 32c .. +31 at c*2048 + r*16, then the scale byte of
 * inputs 128j + 16i .. +15 at 8192 + i*128 + r (i = 0..7). */
lowbit_status lowbit_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int N, int K,
                                void* packed, void* stream);

/* Repack Q8 weights, the 8-bit arm of the small-vocabulary MTP study's trimmed draft head
 * (section 3.3; read as the llama.cpp Q8_0 recipe the ShiftAddQwen README names):
 *   w[n][k] = d[n][k/32] * q[n][k].
 *   codes  : int8 [N][K] (two's complement, the full range -128..127), 16-byte aligned.
 *   scales : fp16 [N][K/32], 2-byte aligned.
 *   packed : lowbit_q8_packed_bytes(N, K) bytes, 16-byte aligned; fully overwritten.
 * Layout: header (format 5), then per (tile t of 128 rows, group g of 128 inputs) one block of
 * 17408 bytes at 128 + (t*(K/128) + g)*17408: for chunk c = 0..7 and row r the 16 code bytes of
 * inputs 128g + 16c .. +15 at c*2048 + r*16, then d[n][4g + j] (fp16) at 16384 + j*256 + r*2
 * (j = 0..3).  Padding rows hold code 0 and scale 0. */
lowbit_status lowbit_pack_q8(const int8_t* codes, const uint16_t* scales, int N, int K, void* packed,
                             void* stream);

/* Synchronous check (copies the 128-byte header to the host after synchronising `stream`)
 * that `packed` holds format `format` (1 = INT4, 2 = binary planes, 3 = sa, 4 = NVFP4, 5 = Q8)
 * with these N, K and, for formats 2 and 3, P (pass 0 for the others).  For the sa format the
 * header's code group G is only checked to be 64, 128 or 256.
 * Returns LOWBIT_OK or LOWBIT_ERR_INVALID_ARG. */
lowbit_status lowbit_validate_packed(const void* packed, int format, int P, int N, int K,
                                     void* stream);

/* ------------------------------------------------------------------------------------------
 * Multiplies.
 */

/* Y = X * W^T for symmetric per-group INT4 weights (Efficient-Qwen report, section 2.1):
 *   y[m][n] = sum_g s[n][g] * sum_{k in g} q[n][k] * x[m][k], fp32 accumulation across
 *   groups, each output rounded once to bf16 (nearest, ties to even).
 *   X : bf16 [M][K], 16-byte aligned.   packed : from lowbit_pack_int4(N, K).
 *   Y : bf16 [M][N], written in full.   1 <= M <= 32.
 * M <= 2 runs the streaming kernel (path 1 also at M = 3, 4): each run of 64 activations of a
 * row is held as int16 times one power of two (exact for every activation within a factor 2^7
 * of the run's largest, otherwise rounded to a multiple of 2^-15 of that largest) and the
 * products within a run are summed exactly in integers; a non-finite activation makes every
 * output of its row NaN.
 * M >= 3 runs the skinny GEMM on the warp-level tensor-core MMA (exact bf16 q times the bf16
 * activations, fp32 accumulation within a group, then s times the group's sum added in fp32). */
lowbit_status lowbit_gemm_int4(const uint16_t* X, const void* packed, int M, int N, int K,
                               uint16_t* Y, void* stream);

/* One multiply of a grouped call: the arguments of lowbit_gemm_int4 other than M. */
typedef struct lowbit_gemm_desc {
  const uint16_t* X;    /* bf16 [M][K], device, 16-byte aligned */
  const void* packed;   /* from lowbit_pack_int4(N, K), device, 16-byte aligned */
  uint16_t* Y;          /* bf16 [M][N], device */
  int N;
  int K;
} lowbit_gemm_desc;

/* Several independent INT4 multiplies with a common M (for example the q, k and v projections
 * of a decoder layer, which read the same activations), each with the contract and rounding
 * of lowbit_gemm_int4.  They share ONE launch (the streaming kernel at M <= 2, the warp-MMA
 * GEMM above), so the launch, pipeline fill and drain are paid once for the group instead of
 * once per matrix.
 *   descs : HOST array of `count` descriptors, 1 <= count <= 8; read during the call only.
 *   The multiplies must be independent: no Y may overlap any X, packed buffer or other Y of
 *   the group.  Every descriptor is validated before anything is enqueued. */
lowbit_status lowbit_gemm_int4_grouped(const lowbit_gemm_desc* descs, int count, int M,
                                       void* stream);
/* The same with the kernel family forced: `path` as lowbit_gemm_int4_path (1: the streaming
 * kernel, M <= 4, else LOWBIT_ERR_SHAPE). */
lowbit_status lowbit_gemm_int4_grouped_path(const lowbit_gemm_desc* descs, int count, int M,
                                            int path, void* stream);

/* Y = X * W^T for binary-plane weights (ShiftAddQwen README, "Method" and "Format"):
 *   y[m][n] = sum_p sum_g alpha[p][n][g] * sum_{k in g} b[p][n][k] * x[m][k].
 *   Shapes and rounding as lowbit_gemm_int4; packed from lowbit_pack_binplane(P, N, K).
 *   M = 1 runs the table-driven streaming kernel; M >= 2 the warp-level MMA on exact +-1
 *   bf16 fragments, one MMA set per plane, alpha applied per (plane, group) in fp32. */
lowbit_status lowbit_gemm_binplane(const uint16_t* X, const void* packed, int P, int M, int N,
                                   int K, uint16_t* Y, void* stream);

/* Y = X * W^T for the deployed ShiftAdd format (ShiftAddQwen README, "Format"):
 *   y[m][n] = sum_j d[n][j] * sum_p sum_{g in j} a[p][n][g] * sum_{k in g} b[p][n][k] * x[m][k],
 *   fp32 accumulation, each output rounded once to bf16.  X, Y as lowbit_gemm_int4,
 *   1 <= M <= 32; packed from lowbit_pack_sa(P, G, N, K); K % 256 == 0.  M = 1 runs the
 *   streaming mat-vec (per plane a table-driven sign-select-and-add, one scale per group);
 *   M >= 2 runs the warp-level MMA on exact +-1 fragments, each code group's sums scaled by
 *   d * a in fp32 (path 2: the tcgen05 GEMM, weights written as +-a in bf16).
 *   The header (format 3, P, N, K, G) is checked on the device as for the other formats. */
lowbit_status lowbit_gemm_sa(const uint16_t* X, const void* packed, int P, int G, int M, int N,
                             int K, uint16_t* Y, void* stream);

/* Y = X * W^T for NVFP4 weights (packed by lowbit_pack_nvfp4), 1 <= M <= 32, g applied in fp32
 * per output, each output rounded once to bf16.  M = 1 runs the streaming mat-vec (int16
 * activations, as the INT4 kernel); M >= 2 the tensor cores (each weight written to tensor
 * memory as the exact bf16 of e2m1 * e4m3).  (The draft step itself needs only the argmax:
 * lowbit_draft_argmax, which chooses its kernel the same way.) */
lowbit_status lowbit_gemm_nvfp4(const uint16_t* X, const void* packed, int M, int N, int K,
                                uint16_t* Y, void* stream);

/* Y = X * W^T for Q8 weights (lowbit_pack_q8), 1 <= M <= 32, fp32 accumulation, each output
 * rounded once to bf16.  M = 1 streams the weights (activations held as int16 per run of 64 as
 * in lowbit_gemm_int4; integer dot products against the signed codes, each run of 32 scaled
 * by its d in fp32); M >= 2 runs the warp-level MMA (each code written exactly as bf16, the
 * MMA sums of every 32 inputs scaled by d in fp32).  path: 0 the library's choice, 1 the
 * streaming kernel (M = 1 only, else LOWBIT_ERR_SHAPE), 3 the warp-level MMA. */
lowbit_status lowbit_gemm_q8(const uint16_t* X, const void* packed, int M, int N, int K, uint16_t* Y,
                             void* stream);
lowbit_status lowbit_gemm_q8_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                  uint16_t* Y, int path, void* stream);

/* The draft step of a trimmed Q8 head: as lowbit_draft_argmax (ids[m] = id_map[argmax], fp32
 * logits never rounded, lowest row on ties, the same workspace rules), for a head packed by
 * lowbit_pack_q8.  M = 1 streams; M >= 2 runs the warp-level MMA. */
lowbit_status lowbit_draft_argmax_q8(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                     const int32_t* id_map, int32_t* ids, void* workspace,
                                     size_t ws_bytes, void* stream);

/* Draft step of a trimmed NVFP4 head (small-vocabulary MTP study, section 3.3: the draft head
 * keeps the 32,768 most used rows of the vocabulary; its winners are mapped back to the full
 * vocabulary before verification):
 *   H      : bf16 [M][K] hidden rows, 1 <= M <= 32.   packed_head : from lowbit_pack_nvfp4.
 *   id_map : int32 [N], the full-vocabulary id of each head row, or NULL (ids are rows).
 *   ids    : int32 [M] out: id_map[argmax_n logit[m][n]], argmax over fp32 logits (never
 *            rounded), lowest row on ties.  Logits are not written anywhere.
 *   workspace : as lmhead_argmax_verify (lmhead_workspace_bytes, zero-filled once, left zero;
 *            calls sharing one must not overlap). */
lowbit_status lowbit_draft_argmax(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                  const int32_t* id_map, int32_t* ids, void* workspace,
                                  size_t ws_bytes, void* stream);

/* LM-head verify step (small-vocabulary MTP study, section 3.3: full-vocabulary verification;
 * DFlash summary, section 4.1: tau in [1, gamma + 1]; Efficient-Qwen report, section 2.2).
 *   H        : bf16 [M][K] hidden rows of one verify block, 2 <= M <= 32 (M - 1 drafts).
 *   packed_head : INT4 head from lowbit_pack_int4(N, K), N = vocabulary rows.
 *   draft    : int32 [M-1] draft token ids for positions 1..M-1 of the block.
 *   argmax   : int32 [M] out: a[m] = argmax_n logit[m][n] over fp32 logits (never rounded),
 *              lowest index on ties.  Logits are not written anywhere.
 *   n_accept : int32 [1] out: n = largest j <= M-1 with draft[i] == a[i] for all i < j.
 *   bonus    : int32 [1] out: a[n], the target's token after the accepted prefix.
 *   workspace: lmhead_workspace_bytes(M, N, K) bytes, 16-byte aligned, ZERO-FILLED ONCE
 *              before first use; every call leaves it zero again.  Calls that share a
 *              workspace must not overlap on the GPU.  After a failed call, re-zero it. */
lowbit_status lmhead_argmax_verify(const uint16_t* H, const void* packed_head, int M, int N,
                                   int K, const int32_t* draft, int32_t* argmax,
                                   int32_t* n_accept, int32_t* bonus, void* workspace,
                                   size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Row-sharded LM head: verification with the vocabulary split across GPUs (small-vocabulary MTP
 * study, section 3.3: drafts are verified against the full vocabulary; DFlash summary, section
 * 4.1: greedy prefix acceptance).  Each GPU holds a contiguous slice of the head's rows, packed
 * on its own with lowbit_pack_int4; the only exchange is W * M 64-bit keys.
 *
 *   1. On every GPU: lmhead_argmax_partial on its slice -> keys_out[M].
 *   2. The caller all-gathers the keys of all W GPUs into keys[W][M] (shard order is free).
 *   3. On every GPU: lmhead_accept_keys(keys, W, ...) -> the same argmax, n_accept and bonus
 *      as lmhead_argmax_verify on the whole head (argmax over fp32 logits, lowest row on ties).
 *
 * Key of a token: (order-preserving bits of its best fp32 logit in the slice) << 32 |
 * (0xFFFFFFFF - global row), so that a larger key is a larger logit and, between equal logits,
 * the lower row; the maximum over slices is the full head's winner.
 */

/* Step 1.  packed_shard: lowbit_pack_int4 of rows row_offset .. row_offset + N - 1 of the head
 * (N rows, K inputs); H: bf16 [M][K], 1 <= M <= 32; row_offset >= 0 and row_offset + N < 2^31.
 *   keys_out : uint64 [M] out, 8-byte aligned (device).
 *   workspace: as lmhead_argmax_verify (lmhead_workspace_bytes(2, N, K), zero once, left zero).
 * Runs the default verify kernel (warp-level MMA); logits are never written. */
lowbit_status lmhead_argmax_partial(const uint16_t* H, const void* packed_shard, int M, int N, int K,
                                    int row_offset, uint64_t* keys_out, void* workspace,
                                    size_t ws_bytes, void* stream);

/* Step 3.  keys: uint64 [W][M] (device, 8-byte aligned), every shard's keys_out; draft: int32
 * [M-1]; argmax: int32 [M] out; n_accept, bonus: int32 [1] out, as lmhead_argmax_verify.
 * 2 <= M <= 32, W >= 1.  One small kernel. */
lowbit_status lmhead_accept_keys(const uint64_t* keys, int W, int M, const int32_t* draft,
                                 int32_t* argmax, int32_t* n_accept, int32_t* bonus, void* stream);

/* ------------------------------------------------------------------------------------------
 * For callers that cannot allocate device memory.
 */

/* lmhead_argmax_verify without the `workspace` argument.  The method has no counterpart to this
 * function: it is a library convenience for callers that own no device allocator and so cannot
 * provide the 512-byte workspace -- for example a plugin whose device memory is planned ahead
 * of time by its host engine, or a C caller that links only this library and the CUDA runtime
 * and must not allocate on its serving path.
 *   Arguments, shapes, results and rounding are those of lmhead_argmax_verify.
 *   Scratch: the library holds one 512-byte scratch per device in place of `workspace`.  The
 *     first call on a device looks up its address (cudaGetSymbolAddress); make that first call
 *     before any stream capture on that device.  Nothing is allocated or freed, ever.
 *   Zeroing: the scratch must be zero when the kernel starts; every call clears it on `stream`
 *     itself (cudaMemsetAsync) before the kernel, so the caller never has to.
 *   Limit: shapes whose workspace (lmhead_workspace_bytes) would exceed 512 bytes return
 *     LOWBIT_ERR_WORKSPACE; every shape lmhead_argmax_verify accepts fits today.
 *   Concurrency: all calls on one device share the one scratch, so two calls that may run at
 *     the same time (for example on two streams with no ordering between them) race and give
 *     wrong results.  Order such calls, or use lmhead_argmax_verify with one workspace each. */
lowbit_status lmhead_argmax_verify_noalloc(const uint16_t* H, const void* packed_head, int M,
                                           int N, int K, const int32_t* draft, int32_t* argmax,
                                           int32_t* n_accept, int32_t* bonus, void* stream);

/* ------------------------------------------------------------------------------------------
 * Kernel-family selection (diagnostics and testing).  Same contract as the functions above,
 * plus `path`: 0 = the library's choice; 1 = the CUDA-core kernels (INT4: the streaming
 * kernel up to M = 4, integer dot products on block-scaled int16 activations, and a
 * row-per-lane bf16 kernel above; planes: the table-driven streaming kernel at M = 1 and a
 * sign-XOR kernel above; LM head: the row-per-lane kernel); 2 = the tcgen05 kernels
 * (dequantisation into tensor memory, tcgen05 MMA with fp32 accumulation); 3 (INT4, binary planes,
 * the sa format and the LM head, any M) = the warp-level MMA kernels (mma.sync m16n8k16 on bf16 fragments
 * unpacked in registers; binary planes too).  The library's choice for M >= 3 INT4, for binary
 * planes and the sa format at M >= 2 and for the LM head is 3:
 * with 16 activation rows a 128-row tcgen05 MMA issues as slowly as with 64, and the
 * weight stream then outruns it.  Other values: INVALID_ARG.
 */
lowbit_status lowbit_gemm_int4_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                    uint16_t* Y, int path, void* stream);
lowbit_status lowbit_gemm_binplane_path(const uint16_t* X, const void* packed, int P, int M,
                                        int N, int K, uint16_t* Y, int path, void* stream);
lowbit_status lmhead_argmax_verify_path(const uint16_t* H, const void* packed_head, int M, int N,
                                        int K, const int32_t* draft, int32_t* argmax,
                                        int32_t* n_accept, int32_t* bonus, void* workspace,
                                        size_t ws_bytes, int path, void* stream);
/* path 1 at M >= 2: CUDA-core kernel (sign select by XOR into the activation's sign bit). */
lowbit_status lowbit_gemm_sa_path(const uint16_t* X, const void* packed, int P, int G, int M,
                                  int N, int K, uint16_t* Y, int path, void* stream);
/* NVFP4: path 1 = the streaming mat-vec (M = 1 only; M > 1 returns LOWBIT_ERR_SHAPE), which
 * reads each code byte through a table of the two codes' 2 * e2m1 values and takes integer dot
 * products with block-scaled int16 activations, each run of 16 scaled by its e4m3 scale in
 * fp32; path 2 = the tensor-core kernel.  The library's choice is path 1 at M = 1. */
lowbit_status lowbit_gemm_nvfp4_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                     uint16_t* Y, int path, void* stream);
lowbit_status lowbit_draft_argmax_path(const uint16_t* H, const void* packed_head, int M, int N,
                                       int K, const int32_t* id_map, int32_t* ids,
                                       void* workspace, size_t ws_bytes, int path, void* stream);

/* ------------------------------------------------------------------------------------------
 * Device-side error word.
 */

/* Testing only: with `on` nonzero, every later launch of the streaming and warp-MMA kernels
 * (the library's default kernels, path 1 at M = 1 and path 3) has its compute warps wait for
 * data on a barrier that nothing arrives on, so that its bounded waits give up: each data
 * wait then ends after about a millisecond instead of about a second.  Such a call writes no
 * output (Y, argmax, n_accept, bonus, ids keep their previous contents), leaves the LM-head
 * workspace zeroed, and records LOWBIT_ERR_TIMEOUT in the device error word.  A CTA still
 * waits for its own copies in flight before it exits.  The tcgen05 and CUDA-core kernels are
 * not affected.  The setting is process-wide; pass 0 to restore normal operation. */
lowbit_status lowbit_debug_inject_stall(int on);

/* Synchronises `stream`, then returns (in *status_out) and clears the current device's
 * error word: LOWBIT_OK, LOWBIT_ERR_INVALID_ARG (a kernel found a packed header that did not
 * match its arguments) or LOWBIT_ERR_TIMEOUT (a bounded wait gave up).  The function's own
 * return value reports failures of the query itself. */
lowbit_status lowbit_device_error(void* stream, int* status_out);

#ifdef __cplusplus
}
#endif

#endif /* LOWBIT_H */

// extern "C" entry points of liblowbit.so: host-side validation, then kernel dispatch.
// Declarations and the full contract are in include/lowbit.h.
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace lowbit {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxK = 65536;

// One error word per device (see lowbit_device_error).
__device__ int g_device_error;
std::atomic<int> g_debug_stall{0};
// Device address of the error word per device; concurrent first calls on one device both
// store the same value.
std::atomic<int*> g_err_ptr[kMaxDevices];

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline lowbit_status check_shape(int M, int N, int K, int Mmax) {
  if (K <= 0 || K % kGroup != 0 || K > kMaxK) return LOWBIT_ERR_SHAPE;
  if (N < 1) return LOWBIT_ERR_SHAPE;
  if (M < 1 || M > Mmax) return LOWBIT_ERR_SHAPE;
  return LOWBIT_OK;
}

// The sa format: K a multiple of the 256-input super-block, 1..8 planes, G in {64, 128, 256}.
inline lowbit_status check_sa(int P, int G, int M, int N, int K) {
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (K % kSuper != 0 || P < 1 || P > 8 || (G != 64 && G != 128 && G != 256)) return LOWBIT_ERR_SHAPE;
  return LOWBIT_OK;
}

inline lowbit_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LOWBIT_OK : LOWBIT_ERR_CUDA; }

}  // namespace

int debug_stall() { return g_debug_stall.load(std::memory_order_relaxed); }

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* w = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    w = static_cast<int*>(p);
    g_err_ptr[dev].store(w, std::memory_order_relaxed);
  }
  return w;
}

bool allocation_covers(const void* p, size_t bytes) {
  // looked up once, on the first call (a function-local static initialises exactly once even
  // when several host threads make that call together)
  static const PFN_cuPointerGetAttribute_v4000 get_attr = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &fn, 4000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuPointerGetAttribute_v4000>(nullptr);
    return reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(fn);
  }();
  if (!get_attr || !p) return false;
  CUdeviceptr start = 0;
  size_t size = 0;
  const CUdeviceptr dp = (CUdeviceptr)(uintptr_t)p;
  if (get_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS) return false;
  if (get_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS) return false;
  return dp >= start && bytes <= size && dp - start <= size - bytes;
}

lowbit_status check_lmhead_args(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                const int32_t* draft, const int32_t* argmax, const int32_t* n_accept,
                                const int32_t* bonus, const void* workspace, size_t ws_bytes) {
  if (!H || !packed_head || !draft || !argmax || !n_accept || !bonus) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (M < 2) return LOWBIT_ERR_SHAPE;
  if (!workspace || ws_bytes < lmhead_workspace_bytes(M, N, K)) return LOWBIT_ERR_WORKSPACE;
  if (!aligned16(H) || !aligned16(packed_head) || !aligned16(workspace)) return LOWBIT_ERR_ALIGN;
  return LOWBIT_OK;
}

}  // namespace lowbit

using namespace lowbit;

extern "C" {

const char* lowbit_status_string(int status) {
  switch (status) {
    case LOWBIT_OK: return "ok";
    case LOWBIT_ERR_INVALID_ARG: return "invalid argument";
    case LOWBIT_ERR_SHAPE: return "unsupported shape";
    case LOWBIT_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LOWBIT_ERR_WORKSPACE: return "workspace missing or too small";
    case LOWBIT_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    case LOWBIT_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int lowbit_version(void) { return 100; }

size_t lowbit_int4_packed_bytes(int N, int K) {
  if (check_shape(1, N, K, 1) != LOWBIT_OK) return 0;
  return kHeaderBytes + int4_payload_bytes(N, K);
}

size_t lowbit_binplane_packed_bytes(int P, int N, int K) {
  if (check_shape(1, N, K, 1) != LOWBIT_OK || P < 1 || P > 8) return 0;
  return kHeaderBytes + binplane_payload_bytes(P, N, K);
}

size_t lowbit_sa_packed_bytes(int P, int G, int N, int K) {
  if (check_sa(P, G, 1, N, K) != LOWBIT_OK) return 0;
  return kHeaderBytes + sa_payload_bytes(P, G, N, K);
}

size_t lowbit_nvfp4_packed_bytes(int N, int K) {
  if (check_shape(1, N, K, 1) != LOWBIT_OK) return 0;
  return kHeaderBytes + nvfp4_payload_bytes(N, K);
}

size_t lowbit_q8_packed_bytes(int N, int K) {
  if (check_shape(1, N, K, 1) != LOWBIT_OK) return 0;
  return kHeaderBytes + q8_payload_bytes(N, K);
}

size_t lmhead_workspace_bytes(int M, int N, int K) {
  if (M < 2 || M > 32 || N < 1 || K <= 0 || K % kGroup != 0) return 0;
  return 512;
}

lowbit_status lowbit_pack_int4(const int8_t* codes, const uint16_t* scales, int N, int K,
                               void* packed, void* stream) {
  if (!codes || !scales || !packed) return LOWBIT_ERR_INVALID_ARG;
  lowbit_status st = check_shape(1, N, K, 1);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(codes) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  return from_cuda(launch_pack_int4(codes, scales, N, K, static_cast<uint8_t*>(packed),
                                    static_cast<cudaStream_t>(stream)));
}

lowbit_status lowbit_pack_binplane(const uint8_t* signbits, const uint16_t* alpha, int P, int N,
                                   int K, void* packed, void* stream) {
  if (!signbits || !alpha || !packed) return LOWBIT_ERR_INVALID_ARG;
  lowbit_status st = check_shape(1, N, K, 1);
  if (st != LOWBIT_OK) return st;
  if (P < 1 || P > 8) return LOWBIT_ERR_SHAPE;
  if (!aligned16(signbits) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  return from_cuda(launch_pack_binplane(signbits, alpha, P, N, K, static_cast<uint8_t*>(packed),
                                        static_cast<cudaStream_t>(stream)));
}

lowbit_status lowbit_pack_sa(const uint8_t* signbits, const uint8_t* codes, const uint16_t* d,
                             int P, int G, int N, int K, void* packed, void* stream) {
  if (!signbits || !codes || !d || !packed) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_sa(P, G, 1, N, K);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(signbits) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  return from_cuda(launch_pack_sa(signbits, codes, d, P, G, N, K, static_cast<uint8_t*>(packed),
                                  static_cast<cudaStream_t>(stream)));
}

lowbit_status lowbit_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, float g, int N, int K,
                                void* packed, void* stream) {
  if (!codes || !scales || !packed) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(1, N, K, 1);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(codes) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  return from_cuda(launch_pack_nvfp4(codes, scales, g, N, K, static_cast<uint8_t*>(packed),
                                     static_cast<cudaStream_t>(stream)));
}

lowbit_status lowbit_pack_q8(const int8_t* codes, const uint16_t* scales, int N, int K, void* packed,
                             void* stream) {
  if (!codes || !scales || !packed) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(1, N, K, 1);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(codes) || !aligned16(packed) || ((uintptr_t)scales & 1u)) return LOWBIT_ERR_ALIGN;
  return from_cuda(launch_pack_q8(codes, scales, N, K, static_cast<uint8_t*>(packed),
                                  static_cast<cudaStream_t>(stream)));
}

lowbit_status lowbit_gemm_q8(const uint16_t* X, const void* packed, int M, int N, int K, uint16_t* Y,
                             void* stream) {
  return lowbit_gemm_q8_path(X, packed, M, N, K, Y, 0, stream);
}

lowbit_status lowbit_gemm_q8_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                  uint16_t* Y, int path, void* stream) {
  if (!X || !packed || !Y || (path != 0 && path != 1 && path != 3)) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (path == 1 && M != 1) return LOWBIT_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, 0, 0};
  p.early = allocation_covers(pk, kHeaderBytes + q8_payload_bytes(N, K)) ? 1 : 0;
  if (path == 0) path = M == 1 ? 1 : 3;
  if (path == 1) return from_cuda(launch_q8_stream(p, nullptr, nullptr, nullptr, err, s));
  return from_cuda(launch_q8_mma(p, M, nullptr, nullptr, nullptr, err, s));
}

lowbit_status lowbit_draft_argmax_q8(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                     const int32_t* id_map, int32_t* ids, void* workspace,
                                     size_t ws_bytes, void* stream) {
  if (!H || !packed_head || !ids) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (!workspace || ws_bytes < lmhead_workspace_bytes(2, N, K)) return LOWBIT_ERR_WORKSPACE;
  if (!aligned16(H) || !aligned16(packed_head) || !aligned16(workspace)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed_head);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemvProblem p = {H, pk, nullptr, N, K, 0, 1, 0, 0, 0};
  p.early = allocation_covers(pk, kHeaderBytes + q8_payload_bytes(N, K)) ? 1 : 0;
  LmheadWorkspace* ws = static_cast<LmheadWorkspace*>(workspace);
  if (M == 1) return from_cuda(launch_q8_stream(p, ws, id_map, ids, err, s));
  return from_cuda(launch_q8_mma(p, M, ws, id_map, ids, err, s));
}

lowbit_status lowbit_validate_packed(const void* packed, int format, int P, int N, int K,
                                     void* stream) {
  if (!packed) return LOWBIT_ERR_INVALID_ARG;
  PackedHeader h;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LOWBIT_ERR_CUDA;
  if (cudaMemcpy(&h, packed, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return LOWBIT_ERR_CUDA;
  // INT4, NVFP4 and Q8 headers record no plane count; the sa header records its code group G,
  // which this call does not take, so any supported G is accepted there.
  const bool planes = format == (int)kFormatBinplane || format == (int)kFormatSa;
  const uint32_t want_p = planes ? (uint32_t)P : 0u;
  const bool group_ok = format == (int)kFormatSa
                            ? (h.group == 64u || h.group == 128u || h.group == 256u)
                            : h.group == (uint32_t)kGroup;
  const bool ok = h.magic == kMagic && h.format == (uint32_t)format && h.version == kVersion &&
                  h.N == (uint32_t)N && h.K == (uint32_t)K && h.P == want_p && group_ok &&
                  h.row_tile == (uint32_t)kRowTile;
  return ok ? LOWBIT_OK : LOWBIT_ERR_INVALID_ARG;
}

lowbit_status lowbit_gemm_int4(const uint16_t* X, const void* packed, int M, int N, int K,
                               uint16_t* Y, void* stream) {
  return lowbit_gemm_int4_path(X, packed, M, N, K, Y, 0, stream);
}

lowbit_status lowbit_gemm_int4_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                    uint16_t* Y, int path, void* stream) {
  if (!X || !packed || !Y || path < 0 || path > 3) return LOWBIT_ERR_INVALID_ARG;
  lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(X) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = (M <= kStreamDefaultRows) ? 1 : 3;
  if (path == 3) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, 0};
    p.early = allocation_covers(pk, kHeaderBytes + int4_payload_bytes(N, K)) ? 1 : 0;
    return from_cuda(launch_int4_mma(&p, 1, M, err, s));
  }
  if (path == 1 && M <= kStreamMaxRows) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, 0};
    p.early = allocation_covers(pk, kHeaderBytes + int4_payload_bytes(N, K)) ? 1 : 0;
    return from_cuda(launch_int4_stream(&p, 1, M, err, s));
  }
  if (path == 1) return from_cuda(launch_int4_gemm_cc(X, pk, M, N, K, Y, err, s));
  return from_cuda(launch_int4_gemm_tc(X, pk, M, N, K, Y, err, s));
}

lowbit_status lowbit_gemm_int4_grouped(const lowbit_gemm_desc* descs, int count, int M,
                                       void* stream) {
  return lowbit_gemm_int4_grouped_path(descs, count, M, 0, stream);
}

lowbit_status lowbit_gemm_int4_grouped_path(const lowbit_gemm_desc* descs, int count, int M,
                                            int path, void* stream) {
  if (!descs || count < 1 || count > kMaxGemvProblems || path < 0 || path > 3)
    return LOWBIT_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const lowbit_gemm_desc& d = descs[i];
    if (!d.X || !d.packed || !d.Y) return LOWBIT_ERR_INVALID_ARG;
    lowbit_status st = check_shape(M, d.N, d.K, 32);
    if (st != LOWBIT_OK) return st;
    if (!aligned16(d.X) || !aligned16(d.packed)) return LOWBIT_ERR_ALIGN;
  }
  if (path == 1 && M > kStreamMaxRows) return LOWBIT_ERR_SHAPE;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = M <= kStreamDefaultRows ? 1 : 3;
  GemvProblem p[kMaxGemvProblems];
  for (int i = 0; i < count; ++i) {
    p[i] = GemvProblem{descs[i].X, static_cast<const uint8_t*>(descs[i].packed), descs[i].Y,
                       descs[i].N, descs[i].K, 0, 1, 0, 0};
    p[i].early = allocation_covers(descs[i].packed,
                                   kHeaderBytes + int4_payload_bytes(descs[i].N, descs[i].K)) ? 1 : 0;
  }
  if (path == 1) return from_cuda(launch_int4_stream(p, count, M, err, s));
  if (path == 3) return from_cuda(launch_int4_mma(p, count, M, err, s));
  for (int i = 0; i < count; ++i) p[i].early = 0;
  return from_cuda(launch_int4_tc_grouped(p, count, M, err, s));
}


lowbit_status lowbit_gemm_binplane(const uint16_t* X, const void* packed, int P, int M, int N,
                                   int K, uint16_t* Y, void* stream) {
  return lowbit_gemm_binplane_path(X, packed, P, M, N, K, Y, 0, stream);
}

lowbit_status lowbit_gemm_binplane_path(const uint16_t* X, const void* packed, int P, int M,
                                        int N, int K, uint16_t* Y, int path, void* stream) {
  if (!X || !packed || !Y || path < 0 || path > 3) return LOWBIT_ERR_INVALID_ARG;
  lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (P < 1 || P > 8) return LOWBIT_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = (M == 1) ? 1 : 3;
  if (path == 1 && M == 1) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, P};
    p.early = allocation_covers(pk, kHeaderBytes + binplane_payload_bytes(P, N, K)) ? 1 : 0;
    return from_cuda(launch_bp_stream(&p, 1, err, s));
  }
  if (path == 3) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, P};
    p.early = allocation_covers(pk, kHeaderBytes + binplane_payload_bytes(P, N, K)) ? 1 : 0;
    return from_cuda(launch_bp_mma(p, M, err, s));
  }
  if (path == 1) return from_cuda(launch_binplane_cc(X, pk, P, M, N, K, Y, err, s));
  return from_cuda(launch_binplane_tc(X, pk, P, M, N, K, Y, err, s));
}

lowbit_status lowbit_gemm_sa(const uint16_t* X, const void* packed, int P, int G, int M, int N,
                             int K, uint16_t* Y, void* stream) {
  return lowbit_gemm_sa_path(X, packed, P, G, M, N, K, Y, 0, stream);
}

lowbit_status lowbit_gemm_sa_path(const uint16_t* X, const void* packed, int P, int G, int M,
                                  int N, int K, uint16_t* Y, int path, void* stream) {
  if (!X || !packed || !Y || path < 0 || path > 3) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_sa(P, G, M, N, K);
  if (st != LOWBIT_OK) return st;
  if (!aligned16(X) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = (M == 1) ? 1 : 3;
  if (path == 1 && M == 1) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, P, G};
    p.early = allocation_covers(pk, kHeaderBytes + sa_payload_bytes(P, G, N, K)) ? 1 : 0;
    return from_cuda(launch_sa_stream(&p, 1, err, s));
  }
  if (path == 3) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, P, G};
    p.early = allocation_covers(pk, kHeaderBytes + sa_payload_bytes(P, G, N, K)) ? 1 : 0;
    return from_cuda(launch_sa_mma(p, M, err, s));
  }
  if (path == 1) return from_cuda(launch_sa_cc(X, pk, P, G, M, N, K, Y, err, s));
  return from_cuda(launch_sa_tc(X, pk, P, G, M, N, K, Y, err, s));
}

lowbit_status lowbit_gemm_nvfp4(const uint16_t* X, const void* packed, int M, int N, int K,
                                uint16_t* Y, void* stream) {
  return lowbit_gemm_nvfp4_path(X, packed, M, N, K, Y, 0, stream);
}

lowbit_status lowbit_gemm_nvfp4_path(const uint16_t* X, const void* packed, int M, int N, int K,
                                     uint16_t* Y, int path, void* stream) {
  if (!X || !packed || !Y || path < 0 || path > 2) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (path == 1 && M != 1) return LOWBIT_ERR_SHAPE;
  if (!aligned16(X) || !aligned16(packed)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = M == 1 ? 1 : 2;
  if (path == 1) {
    GemvProblem p = {X, pk, Y, N, K, 0, 1, 0, 0, 0};
    p.early = allocation_covers(pk, kHeaderBytes + nvfp4_payload_bytes(N, K)) ? 1 : 0;
    return from_cuda(launch_nvfp4_stream(p, nullptr, nullptr, nullptr, err, s));
  }
  return from_cuda(launch_nvfp4_tc(X, pk, M, N, K, Y, err, s));
}

lowbit_status lowbit_draft_argmax(const uint16_t* H, const void* packed_head, int M, int N, int K,
                                  const int32_t* id_map, int32_t* ids, void* workspace,
                                  size_t ws_bytes, void* stream) {
  return lowbit_draft_argmax_path(H, packed_head, M, N, K, id_map, ids, workspace, ws_bytes, 0,
                                  stream);
}

lowbit_status lowbit_draft_argmax_path(const uint16_t* H, const void* packed_head, int M, int N,
                                       int K, const int32_t* id_map, int32_t* ids,
                                       void* workspace, size_t ws_bytes, int path, void* stream) {
  if (!H || !packed_head || !ids || path < 0 || path > 2) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_shape(M, N, K, 32);
  if (st != LOWBIT_OK) return st;
  if (path == 1 && M != 1) return LOWBIT_ERR_SHAPE;
  if (!workspace || ws_bytes < lmhead_workspace_bytes(2, N, K)) return LOWBIT_ERR_WORKSPACE;
  if (!aligned16(H) || !aligned16(packed_head) || !aligned16(workspace)) return LOWBIT_ERR_ALIGN;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed_head);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = M == 1 ? 1 : 2;
  if (path == 1) {
    GemvProblem p = {H, pk, nullptr, N, K, 0, 1, 0, 0, 0};
    p.early = allocation_covers(pk, kHeaderBytes + nvfp4_payload_bytes(N, K)) ? 1 : 0;
    return from_cuda(launch_nvfp4_stream(p, static_cast<LmheadWorkspace*>(workspace), id_map, ids,
                                         err, s));
  }
  return from_cuda(launch_draft_argmax_tc(H, pk, M, N, K, id_map, ids, workspace, err, s));
}

lowbit_status lmhead_argmax_verify(const uint16_t* H, const void* packed_head, int M, int N,
                                   int K, const int32_t* draft, int32_t* argmax,
                                   int32_t* n_accept, int32_t* bonus, void* workspace,
                                   size_t ws_bytes, void* stream) {
  return lmhead_argmax_verify_path(H, packed_head, M, N, K, draft, argmax, n_accept, bonus,
                                   workspace, ws_bytes, 0, stream);
}

lowbit_status lmhead_argmax_verify_path(const uint16_t* H, const void* packed_head, int M, int N,
                                        int K, const int32_t* draft, int32_t* argmax,
                                        int32_t* n_accept, int32_t* bonus, void* workspace,
                                        size_t ws_bytes, int path, void* stream) {
  if (path < 0 || path > 3) return LOWBIT_ERR_INVALID_ARG;
  const lowbit_status st = check_lmhead_args(H, packed_head, M, N, K, draft, argmax, n_accept,
                                             bonus, workspace, ws_bytes);
  if (st != LOWBIT_OK) return st;
  int* err = device_error_word();
  if (!err) return LOWBIT_ERR_CUDA;
  const uint8_t* pk = static_cast<const uint8_t*>(packed_head);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (path == 0) path = 3;
  if (path == 1)
    return from_cuda(launch_lmhead_cc(H, pk, M, N, K, draft, argmax, n_accept, bonus, workspace,
                                      err, s));
  if (path == 3) {
    GemvProblem p = {H, pk, nullptr, N, K, 0, 1, 0, 0};
    p.early = allocation_covers(pk, kHeaderBytes + int4_payload_bytes(N, K)) ? 1 : 0;
    return from_cuda(launch_lmhead_mma(p, M, static_cast<LmheadWorkspace*>(workspace), draft,
                                       argmax, n_accept, bonus, err, s));
  }
  return from_cuda(launch_lmhead_tc(H, pk, M, N, K, draft, argmax, n_accept, bonus, workspace,
                                    err, s));
}

lowbit_status lowbit_debug_inject_stall(int on) {
  g_debug_stall.store(on ? 1 : 0, std::memory_order_relaxed);
  return LOWBIT_OK;
}

lowbit_status lowbit_device_error(void* stream, int* status_out) {
  if (!status_out) return LOWBIT_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LOWBIT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return LOWBIT_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return LOWBIT_ERR_CUDA;
  *status_out = v;
  return LOWBIT_OK;
}

}  // extern "C"

// Host side of the C ABI declared in attn_jvp.h: argument validation,
// bulk-tensor-copy descriptors, per-device scratch, kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <map>
#include <utility>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_jvp.h"
#include "attn_bwd_kernel.cuh"
#include "attn_plan.h"

static_assert(attn::kPlanBM == attn::kBM && attn::kPlanBN == attn::kBN,
              "the work list is planned with the kernel's tile sizes");

// The kernels are instantiated once, in the attn_inst_*.cu files; these
// declarations keep this file from instantiating its own copies.
#define ATTN_FWD_DECL(DQ, DVV, JVP, BM, F16) \
  extern template cudaError_t launch_attn<DQ, DVV, JVP, BM, F16>(const KernelParams&, int, cudaStream_t);
// every bias mode, both element types
#define ATTN_FWD_DECL_ALL(DQ, DVV, JVP)                                                   \
  ATTN_FWD_DECL(DQ, DVV, JVP, kNoBias, false) ATTN_FWD_DECL(DQ, DVV, JVP, kNoBias, true)       \
  ATTN_FWD_DECL(DQ, DVV, JVP, kBiasRing, false) ATTN_FWD_DECL(DQ, DVV, JVP, kBiasRing, true)   \
  ATTN_FWD_DECL(DQ, DVV, JVP, kBiasGlobal, false) ATTN_FWD_DECL(DQ, DVV, JVP, kBiasGlobal, true)
// no bias ring (its plan does not fit shared memory)
#define ATTN_FWD_DECL_NORING(DQ, DVV, JVP)                                              \
  ATTN_FWD_DECL(DQ, DVV, JVP, kNoBias, false) ATTN_FWD_DECL(DQ, DVV, JVP, kNoBias, true)       \
  ATTN_FWD_DECL(DQ, DVV, JVP, kBiasGlobal, false) ATTN_FWD_DECL(DQ, DVV, JVP, kBiasGlobal, true)
namespace attn {
ATTN_FWD_DECL_ALL(64, 64, true)
ATTN_FWD_DECL_ALL(64, 128, true)
ATTN_FWD_DECL_ALL(128, 64, true)
ATTN_FWD_DECL_ALL(128, 128, true)
ATTN_FWD_DECL_NORING(256, 64, true)
ATTN_FWD_DECL_NORING(256, 128, true)
ATTN_FWD_DECL_ALL(64, 64, false)
ATTN_FWD_DECL_ALL(64, 128, false)
ATTN_FWD_DECL_ALL(128, 64, false)
ATTN_FWD_DECL_ALL(128, 128, false)
ATTN_FWD_DECL_ALL(256, 64, false)
ATTN_FWD_DECL_ALL(256, 128, false)
ATTN_FWD_DECL_ALL(64, 256, false)
ATTN_FWD_DECL_ALL(128, 256, false)
ATTN_FWD_DECL_ALL(256, 256, false)
extern template cudaError_t launch_attn<64, 64, false, kNoBias, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn<64, 64, true, kNoBias, false, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn<64, 64, false, kNoBias, false, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn<64, 64, true, kNoBias, true, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn<64, 64, false, kNoBias, true, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn<128, 128, false, kNoBias, false, true>(const KernelParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, false, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, false, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, false, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, false, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, true, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, true, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, true, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 64, true, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, false, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, false, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, false, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, false, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, true, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, true, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, true, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<64, 128, true, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, false, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, false, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, false, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, false, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, true, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, true, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, true, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 64, true, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, false, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, false, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, false, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, false, true, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, true, false, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, true, false, true>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, true, true, false>(const BwdParams&, int, cudaStream_t);
extern template cudaError_t launch_attn_bwd<128, 128, true, true, true>(const BwdParams&, int, cudaStream_t);
}

namespace {

// One instantiation; a bias ring whose plan does not fit shared memory
// (Dqk = 256 with tangents) reads the bias per thread instead.
template <int DQ, int DVK, bool JVP, int BMODE, bool F16>
cudaError_t launch_fitting(const attn::KernelParams& kp, int grid, cudaStream_t cs) {
  if constexpr (BMODE == attn::kBiasRing && !attn::Plan<DQ, DVK, JVP, attn::kBiasRing>::FITS)
    return attn::launch_attn<DQ, DVK, JVP, attn::kBiasGlobal, F16>(kp, grid, cs);
  else
    return attn::launch_attn<DQ, DVK, JVP, BMODE, F16>(kp, grid, cs);
}

// The kernel instantiation for the kernel head dims (kq, kv), each 64, 128
// or 256 (16 and 32 run as 64; with tangents kv = 256 runs as two column
// slices of kv = 128), tangents, bias / mask mode and element type.
template <bool JVP, int BMODE, bool F16>
cudaError_t dispatch_dims(int kq, int kv, const attn::KernelParams& kp, int grid, cudaStream_t cs) {
  switch (kq * 1000 + kv) {
    case 64064: return launch_fitting<64, 64, JVP, BMODE, F16>(kp, grid, cs);
    case 64128: return launch_fitting<64, 128, JVP, BMODE, F16>(kp, grid, cs);
    case 128064: return launch_fitting<128, 64, JVP, BMODE, F16>(kp, grid, cs);
    case 128128: return launch_fitting<128, 128, JVP, BMODE, F16>(kp, grid, cs);
    case 256064: return launch_fitting<256, 64, JVP, BMODE, F16>(kp, grid, cs);
    case 256128: return launch_fitting<256, 128, JVP, BMODE, F16>(kp, grid, cs);
    case 64256:
      if constexpr (!JVP) return launch_fitting<64, 256, false, BMODE, F16>(kp, grid, cs);
      break;
    case 128256:
      if constexpr (!JVP) return launch_fitting<128, 256, false, BMODE, F16>(kp, grid, cs);
      break;
    case 256256:
      if constexpr (!JVP) return launch_fitting<256, 256, false, BMODE, F16>(kp, grid, cs);
      break;
  }
  return cudaErrorInvalidValue;
}

template <bool JVP, bool F16>
cudaError_t dispatch_mode(int kq, int kv, int mode, const attn::KernelParams& kp, int grid, cudaStream_t cs) {
  switch (mode) {
    case attn::kNoBias: return dispatch_dims<JVP, attn::kNoBias, F16>(kq, kv, kp, grid, cs);
    case attn::kBiasRing: return dispatch_dims<JVP, attn::kBiasRing, F16>(kq, kv, kp, grid, cs);
    case attn::kBiasGlobal: return dispatch_dims<JVP, attn::kBiasGlobal, F16>(kq, kv, kp, grid, cs);
  }
  return cudaErrorInvalidValue;
}

// The lean ping-pong kernel: head dims <= 64, no bias or mask, dense,
// non-causal, N a positive multiple of the 64-key tile.
cudaError_t dispatch_lean(bool jvp, bool f16, const attn::KernelParams& kp, int grid, cudaStream_t cs) {
  using namespace attn;
  if (f16)
    return jvp ? launch_attn<64, 64, true, kNoBias, true, false, true>(kp, grid, cs)
               : launch_attn<64, 64, false, kNoBias, true, false, true>(kp, grid, cs);
  return jvp ? launch_attn<64, 64, true, kNoBias, false, false, true>(kp, grid, cs)
             : launch_attn<64, 64, false, kNoBias, false, false, true>(kp, grid, cs);
}

cudaError_t dispatch_attn(int kq, int kv, bool jvp, int mode, bool f16, const attn::KernelParams& kp, int grid,
                          cudaStream_t cs) {
  if (f16)
    return jvp ? dispatch_mode<true, true>(kq, kv, mode, kp, grid, cs)
               : dispatch_mode<false, true>(kq, kv, mode, kp, grid, cs);
  return jvp ? dispatch_mode<true, false>(kq, kv, mode, kp, grid, cs)
             : dispatch_mode<false, false>(kq, kv, mode, kp, grid, cs);
}

constexpr int kMaxDevices = 64;

// Per-device scratch: word 0 = device error word.
struct DeviceState {
  int* scratch = nullptr;
  int num_sms = 0;
};

// Jagged work lists live in one buffer per (device, stream): word 0 = list
// length, bytes [256, 256 + capacity * 8) = the list.  Calls on one stream
// are ordered, so they can share it; calls on different streams never do.
constexpr int kListOffsetBytes = 256;
constexpr int kListCapacity = attn::kPlanListBytes / static_cast<int>(sizeof(int2));

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_skip_first_load{0};

attn_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.scratch == nullptr) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    int* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(p, 0, 256) != cudaSuccess) {
      cudaFree(p);
      return ATTN_ERR_CUDA;
    }
    d.scratch = p;
    d.num_sms = sms;
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &d;
  return ATTN_OK;
}

std::mutex g_list_mu;
std::map<std::pair<int, cudaStream_t>, int*> g_lists;

// The work-list buffer of (current device, stream), allocated on first use
// and kept until the process exits.
attn_status stream_list(cudaStream_t stream, int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_list_mu);
  int*& buf = g_lists[std::make_pair(dev, stream)];
  if (buf == nullptr) {
    void* p = nullptr;
    if (cudaMalloc(&p, kListOffsetBytes + attn::kPlanListBytes) != cudaSuccess) return ATTN_ERR_CUDA;
    buf = static_cast<int*>(p);
  }
  *out = buf;
  return ATTN_OK;
}

// 3-D view [z][rows][d] (d innermost) of bf16 (f16 = false) or fp16
// elements, box 64 x box_rows x 1, 128-byte swizzle; rows past `rows` and
// columns past `d` read as zeros.
bool encode_map(CUtensorMap* m, const void* base, uint64_t d, uint64_t rows, uint64_t z,
                uint32_t box_rows, bool f16) {
  cuuint64_t dims[3] = {d, rows, z};
  cuuint64_t strides[2] = {d * 2, d * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D view [z][rows][inner] of bytes (e5m2 elements), box box_inner x
// box_rows x 1 with the given swizzle; out-of-range elements read as zeros.
bool encode_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t z,
                   uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  cuuint64_t dims[3] = {inner, rows, z};
  cuuint64_t strides[2] = {inner, inner * rows};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D fp32 view of the bias [b][h][m][n] (n innermost), box 32 x 128 x 1 x
// 1, 128-byte swizzle, keys / rows past the end read as zeros.  A broadcast
// (stride 0) head or batch dimension becomes a size-1 dimension.  Returns
// false (the kernel then reads the bias per thread) when the layout does not
// fit a tensor map: key stride other than 1, a row / head / batch stride
// that is not a multiple of 4 elements, a broadcast query-row dimension, or
// a base that is not 16-byte aligned.
bool encode_bias_map(CUtensorMap* m, const float* base, const int64_t* st, uint64_t B, uint64_t H,
                     uint64_t M, uint64_t N, int* bcast_h, int* bcast_b) {
  if (base == nullptr || !aligned16(base) || st[3] != 1 || st[2] <= 0 || N == 0 || M == 0)
    return false;
  for (int i = 0; i < 3; ++i)
    if (st[i] < 0 || (st[i] % 4) != 0) return false;
  *bcast_h = st[1] == 0 ? 1 : 0;
  *bcast_b = st[0] == 0 ? 1 : 0;
  cuuint64_t dims[4] = {N, M, *bcast_h ? 1 : H, *bcast_b ? 1 : B};
  // strides of size-1 dimensions are never stepped; give them the extent
  // of the dimension below
  const uint64_t s2 = static_cast<uint64_t>(st[2]) * 4;
  const uint64_t s1 = *bcast_h ? s2 * M : static_cast<uint64_t>(st[1]) * 4;
  const uint64_t s0 = *bcast_b ? s1 * dims[2] : static_cast<uint64_t>(st[0]) * 4;
  cuuint64_t strides[3] = {s2, s1, s0};
  cuuint32_t box[4] = {32, static_cast<cuuint32_t>(attn::kBM), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

attn_status run(const attn_shape* s, const void* q, const void* k, const void* v, const void* tq,
                const void* tk, const void* tv, const int32_t* offsets, const attn_bias* bias,
                int causal, float sm_scale, void* o, void* to, float* lse, void* stream,
                bool jvp, const DeviceState* fixed = nullptr, bool f16 = false) {
  if (s == nullptr) return ATTN_ERR_INVALID_ARG;
  const bool jagged = offsets != nullptr;
  if (s->B < 0 || s->H < 0 || s->Dqk < 0 || s->Dv < 0) return ATTN_ERR_INVALID_ARG;
  auto dim_ok = [](int d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; };
  if (!dim_ok(s->Dqk) || !dim_ok(s->Dv)) return ATTN_ERR_UNSUPPORTED;
  // kernel head dims: 16 and 32 run zero-padded to 64 (the tensor maps keep
  // the true dims and their 64-column boxes read zeros past them).  With
  // tangents, Dv = 256 runs as two column slices of 128: O and tO of 256
  // columns each would take all 512 tensor-memory columns, leaving none for
  // the scores, so each slice is its own work unit.
  const int kq = s->Dqk < 64 ? 64 : s->Dqk;
  int kv = s->Dv < 64 ? 64 : s->Dv;
  int n_vh = 1;  // (the kernels with tangents and kv = 128 read it)
  if (jvp && kv == 256) {
    kv = 128;
    n_vh = 2;
  }
  if (!std::isnan(sm_scale) && !(sm_scale > 0.f && std::isfinite(sm_scale)))
    return ATTN_ERR_INVALID_ARG;
  const bool has_bias = bias != nullptr && (bias->bias != nullptr || bias->mask != nullptr);
  int64_t work_rows = 0;
  if (jagged) {
    if (s->T < 0 || s->T > 0x7fffffffLL || s->max_seq_len < 0) return ATTN_ERR_INVALID_ARG;
    if (has_bias) return ATTN_ERR_UNSUPPORTED;  // bias / mask are dense-only
    work_rows = (s->B > 0 && s->H > 0) ? s->T : 0;
  } else {
    if (s->M < 0 || s->N < 0) return ATTN_ERR_INVALID_ARG;
    if (causal && s->M != s->N) return ATTN_ERR_INVALID_ARG;
    work_rows = static_cast<int64_t>(s->B) * s->H * s->M;
    if (static_cast<int64_t>(s->B) * s->H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  }
  if (work_rows == 0) return ATTN_OK;  // nothing to compute or write
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  const bool have_keys = jagged ? true : s->N > 0;
  if (have_keys && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (jvp) {
    if (tq == nullptr || to == nullptr) return ATTN_ERR_INVALID_ARG;
    if (have_keys && (tk == nullptr || tv == nullptr)) return ATTN_ERR_INVALID_ARG;
  }
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  if (have_keys && (!aligned16(k) || !aligned16(v))) return ATTN_ERR_MISALIGNED;
  if (jvp && (!aligned16(tq) || !aligned16(to))) return ATTN_ERR_MISALIGNED;
  if (jvp && have_keys && (!aligned16(tk) || !aligned16(tv))) return ATTN_ERR_MISALIGNED;
  if (has_bias && bias->bias != nullptr && (reinterpret_cast<uintptr_t>(bias->bias) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;

  DeviceState* ds = nullptr;
  DeviceState fixed_state;
  if (fixed != nullptr) {
    fixed_state = *fixed;
    ds = &fixed_state;
  } else {
    attn_status st = device_state(&ds);
    if (st != ATTN_OK) return st;
  }

  attn::KernelParams kp;
  std::memset(&kp, 0, sizeof(kp));
  const float scale = std::isnan(sm_scale) ? 1.0f / std::sqrt(static_cast<float>(s->Dqk)) : sm_scale;
  kp.B = s->B;
  kp.H = s->H;
  kp.n_vh = n_vh;
  kp.jagged = jagged ? 1 : 0;
  kp.causal = causal ? 1 : 0;
  kp.sm_scale = scale;
  kp.scale_log2 = scale * attn::kLog2e;
  kp.offsets = offsets;
  kp.o = static_cast<uint16_t*>(o);
  kp.to = static_cast<uint16_t*>(to);
  kp.lse = lse;
  kp.dv_out = s->Dv;
  kp.err = ds->scratch;
  kp.timeout_ns = g_timeout_ns.load();
  kp.skip_first_load = g_skip_first_load.load();
  if (has_bias) {
    kp.bias = bias->bias;
    kp.mask = bias->mask;
    for (int i = 0; i < 4; ++i) {
      kp.bias_stride[i] = bias->bias_stride[i];
      kp.mask_stride[i] = bias->mask_stride[i];
    }
    if (kp.bias != nullptr && !jagged)
      kp.bias_tma = encode_bias_map(&kp.tm_bias, kp.bias, bias->bias_stride, s->B, s->H, s->M, s->N,
                                    &kp.bias_bcast_h, &kp.bias_bcast_b)
                        ? 1
                        : 0;
  }
  const uint64_t dqk = s->Dqk, dvv = s->Dv;
  bool ok = true;
  if (jagged) {
    kp.M = kp.N = s->max_seq_len;
    kp.T = s->T;
    kp.max_seq_len = s->max_seq_len;
    kp.n_mt = (s->max_seq_len + attn::kBM - 1) / attn::kBM;
    const uint64_t T = static_cast<uint64_t>(s->T), H = static_cast<uint64_t>(s->H);
    ok = ok && encode_map(&kp.tm_q, q, dqk, T, H, attn::kBM, f16);
    ok = ok && encode_map(&kp.tm_k, k, dqk, T, H, attn::kBN, f16);
    ok = ok && encode_map(&kp.tm_v, v, dvv, T, H, attn::kBN, f16);
    if (jvp) {
      ok = ok && encode_map(&kp.tm_tq, tq, dqk, T, H, attn::kBM, f16);
      ok = ok && encode_map(&kp.tm_tk, tk, dqk, T, H, attn::kBN, f16);
      ok = ok && encode_map(&kp.tm_tv, tv, dvv, T, H, attn::kBN, f16);
    }
  } else {
    kp.M = s->M;
    kp.N = s->N;
    kp.n_mt = (s->M + attn::kBM - 1) / attn::kBM;
    const uint64_t BH = static_cast<uint64_t>(s->B) * s->H;
    const uint64_t M = s->M;
    // With no keys no key tile is ever loaded; the maps only need to be valid.
    const uint64_t N = s->N > 0 ? static_cast<uint64_t>(s->N) : M;
    const void* kb = s->N > 0 ? k : q;
    const void* vb = s->N > 0 ? v : q;
    const uint64_t dvk = s->N > 0 ? dvv : dqk;
    ok = ok && encode_map(&kp.tm_q, q, dqk, M, BH, attn::kBM, f16);
    ok = ok && encode_map(&kp.tm_k, kb, dqk, N, BH, attn::kBN, f16);
    ok = ok && encode_map(&kp.tm_v, vb, dvk, N, BH, attn::kBN, f16);
    if (jvp) {
      const void* tkb = s->N > 0 ? tk : tq;
      const void* tvb = s->N > 0 ? tv : tq;
      ok = ok && encode_map(&kp.tm_tq, tq, dqk, M, BH, attn::kBM, f16);
      ok = ok && encode_map(&kp.tm_tk, tkb, dqk, N, BH, attn::kBN, f16);
      ok = ok && encode_map(&kp.tm_tv, tvb, dvk, N, BH, attn::kBN, f16);
    }
  }
  if (!ok) return ATTN_ERR_CUDA;
  const int64_t units = static_cast<int64_t>(s->B) * s->H * kp.n_mt * n_vh;
  if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  kp.num_units = static_cast<int>(units);
  int grid = static_cast<int>(units < ds->num_sms ? units : ds->num_sms);
  if (grid < 1) grid = 1;  // the jagged tail fill still runs

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // A caller-fixed scratch is shared by every call: its error word must
  // start each launch at zero.
  if (fixed != nullptr && cudaMemsetAsync(ds->scratch, 0, sizeof(int), cs) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // Jagged: order the (sequence, query tile) pairs by cost on the device
  // (the offsets live there) so the kernel can balance them.
  // (The allocation-free entry point keeps the slot order.)
  if (jagged && fixed == nullptr && attn::plan_jagged_supported(s->max_seq_len)) {
    int* lbuf = nullptr;
    const attn_status ls = stream_list(cs, &lbuf);
    if (ls != ATTN_OK) return ls;
    int2* list = reinterpret_cast<int2*>(reinterpret_cast<char*>(lbuf) + kListOffsetBytes);
    if (attn::launch_plan_jagged(offsets, s->B, s->max_seq_len, causal ? 1 : 0, list, lbuf,
                                 kListCapacity, cs) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_launches.fetch_add(1);
    kp.unit_list = list;
    kp.unit_count = lbuf;
  }
  // Dense with a key mask that does not depend on the query row: the key
  // length of each (b, h) up to its last attended key, computed on the
  // device (the mask lives there), so that trailing key tiles that every
  // row masks are not visited.  (The allocation-free entry point, which has
  // no buffer for it, visits every key tile.)
  if (!jagged && kp.mask != nullptr && kp.mask_stride[2] == 0 && fixed == nullptr && s->N > 0 &&
      static_cast<int64_t>(s->B) * s->H <= (kListOffsetBytes + attn::kPlanListBytes) / static_cast<int>(sizeof(int))) {
    int* lbuf = nullptr;
    const attn_status ls = stream_list(cs, &lbuf);
    if (ls != ATTN_OK) return ls;
    if (attn::launch_plan_keylen(kp.mask, kp.mask_stride, s->B, s->H, s->N, lbuf, cs) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_launches.fetch_add(1);
    kp.keylen = lbuf;
  }
  cudaError_t e = cudaErrorInvalidValue;
  // bias through the shared-memory ring when a tensor map describes it,
  // else per-thread loads; a mask alone also takes the ring mode
  const int mode = (kp.bias == nullptr && kp.mask == nullptr) ? attn::kNoBias
                   : (kp.bias != nullptr && kp.bias_tma == 0) ? attn::kBiasGlobal
                                                               : attn::kBiasRing;
  const bool lean = !jagged && !causal && mode == attn::kNoBias && kq == 64 && kv == 64 && n_vh == 1 &&
                    s->N > 0 && s->N % attn::kBN == 0 && kp.keylen == nullptr && kp.unit_list == nullptr;
  e = lean ? dispatch_lean(jvp, f16, kp, grid, cs) : dispatch_attn(kq, kv, jvp, mode, f16, kp, grid, cs);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1);
  return ATTN_OK;
}

// ------------------------------------------------------------ e5m2 forward
attn_status run_f8(const attn_shape* s, const void* q, const void* k, const void* vt, int causal,
                   float sm_scale, void* o, float* lse, void* stream) {
  if (s == nullptr) return ATTN_ERR_INVALID_ARG;
  if (s->B < 0 || s->H < 0 || s->M < 0 || s->N < 0 || s->Dqk < 0 || s->Dv < 0) return ATTN_ERR_INVALID_ARG;
  if (!((s->Dqk == 64 && s->Dv == 64) || (s->Dqk == 128 && s->Dv == 128))) return ATTN_ERR_UNSUPPORTED;
  if (!std::isnan(sm_scale) && !(sm_scale > 0.f && std::isfinite(sm_scale))) return ATTN_ERR_INVALID_ARG;
  if (causal && s->M != s->N) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->B) * s->H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(s->B) * s->H;
  if (BH == 0 || s->M == 0) return ATTN_OK;  // nothing to write
  // V^T rows are N bytes apart: bulk tensor copies need a multiple of 16
  if (s->N % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  if (q == nullptr || o == nullptr || lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (s->N > 0 && (k == nullptr || vt == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  if (s->N > 0 && (!aligned16(k) || !aligned16(vt))) return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;

  attn::KernelParams kp;
  std::memset(&kp, 0, sizeof(kp));
  const float scale = std::isnan(sm_scale) ? 1.0f / std::sqrt(static_cast<float>(s->Dqk)) : sm_scale;
  kp.B = s->B;
  kp.H = s->H;
  kp.M = s->M;
  kp.N = s->N;
  kp.causal = causal ? 1 : 0;
  kp.sm_scale = scale;
  kp.scale_log2 = scale * attn::kLog2e;
  kp.n_vh = 1;
  kp.o = static_cast<uint16_t*>(o);  // e5m2 bytes; the kernel addresses them as such
  kp.lse = lse;
  kp.dv_out = s->Dv;
  kp.err = ds->scratch;
  kp.timeout_ns = g_timeout_ns.load();
  kp.n_mt = (s->M + attn::kBM - 1) / attn::kBM;
  const uint64_t D = static_cast<uint64_t>(s->Dqk), Z = static_cast<uint64_t>(BH);
  const uint64_t M = s->M;
  const uint64_t N = s->N > 0 ? static_cast<uint64_t>(s->N) : 16;  // no keys: valid, never read
  const void* kb = s->N > 0 ? k : q;
  const void* vb = s->N > 0 ? vt : q;
  // Q, K: one 128-byte swizzled chunk per row (zeros past D); V^T: rows of
  // 64 keys with 64-byte swizzle, Dv rows per box
  bool ok = encode_map_u8(&kp.tm_q, q, D, M, Z, 128, attn::kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_map_u8(&kp.tm_k, kb, D, s->N > 0 ? N : M, Z, 128, attn::kBN, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_map_u8(&kp.tm_v, vb, s->N > 0 ? N : D, s->N > 0 ? D : M, Z, 64,
                           static_cast<uint32_t>(s->Dv), CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return ATTN_ERR_CUDA;
  const int64_t units = BH * kp.n_mt;
  if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  kp.num_units = static_cast<int>(units);
  const int grid = static_cast<int>(units < ds->num_sms ? units : ds->num_sms);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = s->Dqk == 64
                            ? attn::launch_attn<64, 64, false, attn::kNoBias, false, true>(kp, grid, cs)
                            : attn::launch_attn<128, 128, false, attn::kNoBias, false, true>(kp, grid, cs);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1);
  return ATTN_OK;
}

// ------------------------------------------------------------- backward
// Jagged backward: tokens of sequence b past its first min(len, max_seq_len)
// attend nothing and are attended by nothing, so their dQ, dK, dV are zero.
// One block per sequence; rows are d 16-bit elements (d a multiple of 8).
// A NULL output is left alone (each gradient pass zeroes its own).
__global__ void attn_bwd_zero_tail_kernel(const int* offsets, int H, long long T, int max_seq_len,
                                          uint16_t* dq, uint16_t* dk, uint16_t* dv, int dqk, int dv_) {
  const int b = blockIdx.x;
  const int begin = offsets[b], end = offsets[b + 1];
  const int first = begin + max(0, min(end - begin, max_seq_len));
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  // one pass per row width: dq / dk rows are dqk wide, dv rows dv_ wide
  for (int pass = 0; pass < 2; ++pass) {
    const int d = pass == 0 ? dqk : dv_;
    uint16_t* a = pass == 0 ? dq : dv;
    uint16_t* c = pass == 0 ? dk : nullptr;
    if (a == nullptr && c == nullptr) continue;
    const int chunks = d / 8;  // 16-byte chunks per row
    const long long per_head = static_cast<long long>(end - first) * chunks;
    for (long long i = threadIdx.x; i < per_head * H; i += blockDim.x) {
      const long long h = i / per_head, rem = i % per_head;
      const long long row = h * T + first + rem / chunks;
      const long long off = row * d + (rem % chunks) * 8;
      if (a != nullptr) *reinterpret_cast<uint4*>(a + off) = z;
      if (c != nullptr) *reinterpret_cast<uint4*>(c + off) = z;
    }
  }
}

// One pass of the dQ kernel (kv = false) or of the dK / dV kernel; key
// bit 1 for Dqk = 128, bit 0 for Dv = 128 (else 64).
template <bool KV, bool F16, bool BM>
cudaError_t dispatch_bwd_dims(int key, const attn::BwdParams& bp, int grid, cudaStream_t cs) {
  switch (key) {
    case 0: return attn::launch_attn_bwd<64, 64, KV, F16, BM>(bp, grid, cs);
    case 1: return attn::launch_attn_bwd<64, 128, KV, F16, BM>(bp, grid, cs);
    case 2: return attn::launch_attn_bwd<128, 64, KV, F16, BM>(bp, grid, cs);
    case 3: return attn::launch_attn_bwd<128, 128, KV, F16, BM>(bp, grid, cs);
  }
  return cudaErrorInvalidValue;
}

template <bool BM>
cudaError_t dispatch_bwd_bm(int key, bool kv, bool f16, const attn::BwdParams& bp, int grid, cudaStream_t cs) {
  if (f16)
    return kv ? dispatch_bwd_dims<true, true, BM>(key, bp, grid, cs) : dispatch_bwd_dims<false, true, BM>(key, bp, grid, cs);
  return kv ? dispatch_bwd_dims<true, false, BM>(key, bp, grid, cs) : dispatch_bwd_dims<false, false, BM>(key, bp, grid, cs);
}

// bm: the launch has a bias and / or a mask
cudaError_t dispatch_bwd(int key, bool kv, bool f16, bool bm, const attn::BwdParams& bp, int grid, cudaStream_t cs) {
  return bm ? dispatch_bwd_bm<true>(key, kv, f16, bp, grid, cs) : dispatch_bwd_bm<false>(key, kv, f16, bp, grid, cs);
}

attn_status run_bwd(const attn_shape* s, const void* q, const void* k, const void* v, const void* o,
                    const void* dout, const float* lse, const int32_t* offsets, const attn_bias* bias,
                    int causal, float sm_scale, void* dq, void* dk, void* dv, float* delta,
                    void* stream, bool f16, unsigned stages) {
  if (s == nullptr) return ATTN_ERR_INVALID_ARG;
  if (stages == 0 || (stages & ~static_cast<unsigned>(ATTN_BWD_ALL)) != 0) return ATTN_ERR_INVALID_ARG;
  const bool jagged = offsets != nullptr;
  if (s->B < 0 || s->H < 0 || s->Dqk < 0 || s->Dv < 0) return ATTN_ERR_INVALID_ARG;
  if (!jagged && (s->M < 0 || s->N < 0)) return ATTN_ERR_INVALID_ARG;
  if (jagged && (s->T < 0 || s->T > 0x7fffffffLL || s->max_seq_len < 0)) return ATTN_ERR_INVALID_ARG;
  const bool has_bias = bias != nullptr && (bias->bias != nullptr || bias->mask != nullptr);
  if (has_bias && jagged) return ATTN_ERR_UNSUPPORTED;  // bias / mask are dense-only
  auto dim_ok = [](int d) { return d == 16 || d == 32 || d == 64 || d == 128; };
  if (!dim_ok(s->Dqk) || !dim_ok(s->Dv)) return ATTN_ERR_UNSUPPORTED;
  if (!std::isnan(sm_scale) && !(sm_scale > 0.f && std::isfinite(sm_scale)))
    return ATTN_ERR_INVALID_ARG;
  if (!jagged && causal && s->M != s->N) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->B) * s->H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = static_cast<int64_t>(s->B) * s->H;
  // rows of the query side and of the key side (jagged: the packed tokens)
  const int64_t n_q = jagged ? s->T : s->M, n_k = jagged ? s->T : s->N;
  if (BH == 0 || (n_q == 0 && n_k == 0)) return ATTN_OK;  // nothing to write
  const bool rows_q = n_q > 0, rows_k = n_k > 0;
  if (rows_q && (q == nullptr || o == nullptr || dout == nullptr || lse == nullptr || dq == nullptr ||
                 delta == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (rows_k && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr))
    return ATTN_ERR_INVALID_ARG;
  for (const void* p : {q, o, dout, static_cast<const void*>(lse), static_cast<const void*>(dq),
                        static_cast<const void*>(delta)})
    if (rows_q && !aligned16(p)) return ATTN_ERR_MISALIGNED;
  for (const void* p : {k, v, static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (rows_k && !aligned16(p)) return ATTN_ERR_MISALIGNED;
  if (has_bias && bias->bias != nullptr && (reinterpret_cast<uintptr_t>(bias->bias) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;

  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const float scale = std::isnan(sm_scale) ? 1.0f / std::sqrt(static_cast<float>(s->Dqk)) : sm_scale;
  // 16 and 32 run zero-padded in the 64-wide kernels
  const int key = (s->Dqk == 128 ? 2 : 0) + (s->Dv == 128 ? 1 : 0);
  const uint64_t dqk = static_cast<uint64_t>(s->Dqk), dv_ = static_cast<uint64_t>(s->Dv),
                 M = static_cast<uint64_t>(n_q), N = static_cast<uint64_t>(n_k);
  // tensor-map z: b * H + h dense, h jagged (rows are the packed tokens)
  const uint64_t Z = jagged ? static_cast<uint64_t>(s->H) : static_cast<uint64_t>(BH);

  // Delta = rowsum(dO o O)
  if (rows_q && (stages & ATTN_BWD_DELTA)) {
    const long long rows = (jagged ? static_cast<long long>(s->H) : static_cast<long long>(BH)) * n_q;
    const long long want = (rows + 31) / 32;  // 8 warps x 4 rows per 256-thread block
    const int blocks = static_cast<int>(want < 16LL * ds->num_sms ? want : 16LL * ds->num_sms);
    if (f16)
      attn::attn_bwd_delta_kernel<true><<<blocks, 256, 0, cs>>>(
          static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), delta, rows, s->Dv);
    else
      attn::attn_bwd_delta_kernel<false><<<blocks, 256, 0, cs>>>(
          static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), delta, rows, s->Dv);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  // jagged: gradients of the tokens past each sequence's max_seq_len
  if (jagged && s->B > 0 && (stages & (ATTN_BWD_DQ | ATTN_BWD_DKDV))) {
    const bool zq = (stages & ATTN_BWD_DQ) != 0, zkv = (stages & ATTN_BWD_DKDV) != 0;
    attn_bwd_zero_tail_kernel<<<s->B, 256, 0, cs>>>(
        offsets, s->H, s->T, s->max_seq_len, zq ? static_cast<uint16_t*>(dq) : nullptr,
        zkv ? static_cast<uint16_t*>(dk) : nullptr, zkv ? static_cast<uint16_t*>(dv) : nullptr, s->Dqk,
        s->Dv);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  for (int pass = 0; pass < 2; ++pass) {
    const bool kv = pass == 1;
    const int64_t rows = kv ? n_k : n_q;
    if (rows == 0 || !(stages & (kv ? ATTN_BWD_DKDV : ATTN_BWD_DQ))) continue;
    attn::BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    bp.B = s->B;
    bp.H = s->H;
    bp.M = jagged ? s->max_seq_len : s->M;
    bp.N = jagged ? s->max_seq_len : s->N;
    bp.causal = causal ? 1 : 0;
    bp.jagged = jagged ? 1 : 0;
    bp.offsets = offsets;
    bp.T = jagged ? s->T : 0;
    bp.max_seq_len = s->max_seq_len;
    bp.n_rt = static_cast<int>(((jagged ? s->max_seq_len : rows) + attn::kBM - 1) / attn::kBM);
    bp.scale_log2 = scale * attn::kLog2e;
    bp.sm_scale = scale;
    bp.lse = lse;
    bp.delta = delta;
    bp.out1 = static_cast<uint16_t*>(kv ? dk : dq);
    bp.out2 = static_cast<uint16_t*>(kv ? dv : nullptr);
    bp.d_qk = s->Dqk;
    bp.d_v = s->Dv;
    if (has_bias) {
      bp.bias = bias->bias;
      bp.mask = bias->mask;
      for (int i = 0; i < 4; ++i) {
        bp.bias_stride[i] = bias->bias_stride[i];
        bp.mask_stride[i] = bias->mask_stride[i];
      }
    }
    bp.err = ds->scratch;
    bp.timeout_ns = g_timeout_ns.load();
    // the streamed side has no rows: its maps are never used, only valid
    const bool other = kv ? rows_q : rows_k;
    const uint64_t Ro = other ? (kv ? M : N) : static_cast<uint64_t>(rows);
    if (bp.n_rt == 0) continue;  // jagged with max_seq_len = 0: nothing attends
    const void* r1 = kv ? k : q;
    const void* r2 = kv ? v : dout;
    const void* t1 = other ? (kv ? q : k) : r1;
    const void* t2 = other ? (kv ? dout : v) : r2;
    // R1 / T1 (q or k) are Dqk wide, R2 / T2 (do or v) Dv wide
    bool ok = encode_map(&bp.tm_r1, r1, dqk, rows, Z, attn::kBM, f16);
    ok = ok && encode_map(&bp.tm_r2, r2, dv_, rows, Z, attn::kBM, f16);
    ok = ok && encode_map(&bp.tm_t1, t1, dqk, Ro, Z, 64, f16);
    ok = ok && encode_map(&bp.tm_t2, t2, dv_, Ro, Z, 64, f16);
    if (!ok) return ATTN_ERR_CUDA;
    const int64_t units = BH * bp.n_rt;
    if (units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    bp.num_units = static_cast<int>(units);
    // Jagged: order this pass's (sequence, row tile) pairs by cost on the
    // device (the offsets live there) so the kernel can balance them; the
    // dK / dV pass counts query tiles per key tile.  (The second pass's
    // planning kernel runs after the first pass's kernel has read the list.)
    if (jagged && attn::plan_jagged_supported(s->max_seq_len)) {
      int* lbuf = nullptr;
      const attn_status ls = stream_list(cs, &lbuf);
      if (ls != ATTN_OK) return ls;
      int2* list = reinterpret_cast<int2*>(reinterpret_cast<char*>(lbuf) + kListOffsetBytes);
      if (attn::launch_plan_jagged(offsets, s->B, s->max_seq_len, causal ? 1 : 0, list, lbuf, kListCapacity,
                                   cs, kv ? 1 : 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
      g_launches.fetch_add(1);
      bp.unit_list = list;
      bp.unit_count = lbuf;
    }
    const int grid = static_cast<int>(units < ds->num_sms ? units : ds->num_sms);
    if (dispatch_bwd(key, kv, f16, has_bias, bp, grid, cs) != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  return ATTN_OK;
}

// ------------------------------------------------ allocation-free variant
// Callers that may not allocate device memory (an embedding framework
// that owns every allocation, a graph-building runtime that forbids
// cudaMalloc while recording, a real-time path with a frozen memory budget)
// use attn_fwd_jvp_noalloc.  Its only scratch -- the kernel's error word --
// lives in this fixed device array instead of a cudaMalloc'd buffer.  Every
// device that loads the library holds the array until the process exits.
constexpr int kNoAllocScratchWords = 64;  // 256 bytes; the kernel uses word 0
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchWords];

// Scratch words one forward + JVP launch needs: the error word, whatever
// the problem size.
constexpr int kScratchWordsPerLaunch = 1;

std::mutex g_noalloc_mu;
DeviceState g_noalloc_dev[kMaxDevices];  // scratch = device address of the array

// Per-device set-up, run on the first call on a device with that device
// current: the array's device address (host code only sees a stand-in
// symbol), the SM count and the descriptor-encoding entry point.  Nothing
// here allocates.
attn_status noalloc_state(DeviceState* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  DeviceState& d = g_noalloc_dev[dev];
  if (d.scratch == nullptr) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ATTN_ERR_CUDA;
    d.num_sms = sms;
    d.scratch = static_cast<int*>(ptr);
  }
  {
    std::lock_guard<std::mutex> lk2(g_mu);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  *out = d;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd_jvp(const attn_shape* shape, const void* q, const void* k, const void* v,
                         const void* tq, const void* tk, const void* tv, const int32_t* offsets,
                         const attn_bias* bias, int causal, float sm_scale, void* o, void* to,
                         float* lse, void* stream) {
  return run(shape, q, k, v, tq, tk, tv, offsets, bias, causal, sm_scale, o, to, lse, stream,
             true);
}

attn_status attn_fwd(const attn_shape* shape, const void* q, const void* k, const void* v,
                     const int32_t* offsets, const attn_bias* bias, int causal, float sm_scale,
                     void* o, float* lse, void* stream) {
  return run(shape, q, k, v, nullptr, nullptr, nullptr, offsets, bias, causal, sm_scale, o,
             nullptr, lse, stream, false);
}

attn_status attn_fwd_jvp_f16(const attn_shape* shape, const void* q, const void* k, const void* v,
                             const void* tq, const void* tk, const void* tv, const int32_t* offsets,
                             const attn_bias* bias, int causal, float sm_scale, void* o, void* to,
                             float* lse, void* stream) {
  return run(shape, q, k, v, tq, tk, tv, offsets, bias, causal, sm_scale, o, to, lse, stream,
             true, nullptr, true);
}

attn_status attn_fwd_f16(const attn_shape* shape, const void* q, const void* k, const void* v,
                         const int32_t* offsets, const attn_bias* bias, int causal, float sm_scale,
                         void* o, float* lse, void* stream) {
  return run(shape, q, k, v, nullptr, nullptr, nullptr, offsets, bias, causal, sm_scale, o,
             nullptr, lse, stream, false, nullptr, true);
}

attn_status attn_bwd(const attn_shape* shape, const void* q, const void* k, const void* v,
                     const void* o, const void* dout, const float* lse, const int32_t* offsets,
                     const attn_bias* bias, int causal, float sm_scale, void* dq, void* dk, void* dv,
                     float* delta, void* stream) {
  return run_bwd(shape, q, k, v, o, dout, lse, offsets, bias, causal, sm_scale, dq, dk, dv, delta,
                 stream, false, ATTN_BWD_ALL);
}

attn_status attn_bwd_stages(const attn_shape* shape, const void* q, const void* k, const void* v,
                            const void* o, const void* dout, const float* lse, const int32_t* offsets,
                            const attn_bias* bias, int causal, float sm_scale, void* dq, void* dk,
                            void* dv, float* delta, int f16, unsigned stages, void* stream) {
  return run_bwd(shape, q, k, v, o, dout, lse, offsets, bias, causal, sm_scale, dq, dk, dv, delta,
                 stream, f16 != 0, stages);
}

attn_status attn_bwd_f16(const attn_shape* shape, const void* q, const void* k, const void* v,
                         const void* o, const void* dout, const float* lse, const int32_t* offsets,
                         const attn_bias* bias, int causal, float sm_scale, void* dq, void* dk,
                         void* dv, float* delta, void* stream) {
  return run_bwd(shape, q, k, v, o, dout, lse, offsets, bias, causal, sm_scale, dq, dk, dv, delta,
                 stream, true, ATTN_BWD_ALL);
}

attn_status attn_fwd_f8(const attn_shape* shape, const void* q, const void* k, const void* vt,
                        int causal, float sm_scale, void* o, float* lse, void* stream) {
  return run_f8(shape, q, k, vt, causal, sm_scale, o, lse, stream);
}

attn_status attn_sync_check(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  // The error words that exist on this device: the per-device scratch of
  // the allocating entry points and the fixed array of the allocation-free
  // one, each only once a call has set it up.  Nothing here allocates.
  int* words[2];
  {
    std::lock_guard<std::mutex> lk(g_mu);
    words[0] = g_dev[dev].scratch;
  }
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    words[1] = g_noalloc_dev[dev].scratch;
  }
  bool timed_out = false;
  for (int* w : words) {
    if (w == nullptr) continue;
    int word = 0;
    if (cudaMemcpy(&word, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (word != 0) {
      if (cudaMemset(w, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
      timed_out = true;
    }
  }
  return timed_out ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED:
      return "unsupported configuration for this entry point (head dims, bias / mask with jagged inputs, "
             "FP8 key count; attn_jvp.h lists each entry point's supported set)";
    case ATTN_ERR_MISALIGNED: return "a device pointer is not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA error (no device, launch failure or driver entry point missing)";
    case ATTN_ERR_TIMEOUT: return "a device pipeline wait ran out of time; outputs are undefined";
  }
  return "unknown status";
}

attn_status attn_fwd_jvp_noalloc(const attn_shape* shape, const void* q, const void* k,
                                 const void* v, const void* tq, const void* tk, const void* tv,
                                 const int32_t* offsets, const attn_bias* bias, int causal,
                                 float sm_scale, void* o, void* to, float* lse, void* stream) {
  static_assert(kScratchWordsPerLaunch <= kNoAllocScratchWords,
                "the fixed scratch array is smaller than one launch needs");
  if (kScratchWordsPerLaunch > kNoAllocScratchWords) return ATTN_ERR_UNSUPPORTED;
  DeviceState fixed;
  if (shape != nullptr) {
    attn_status st = noalloc_state(&fixed);
    if (st != ATTN_OK) return st;
  }
  return run(shape, q, k, v, tq, tk, tv, offsets, bias, causal, sm_scale, o, to, lse, stream, true,
             shape != nullptr ? &fixed : nullptr);
}

uint64_t attn_launch_count(void) { return g_launches.load(); }

void attn_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns);
}

void attn_debug_skip_first_load(int enable) { g_skip_first_load.store(enable ? 1 : 0); }

}  // extern "C"

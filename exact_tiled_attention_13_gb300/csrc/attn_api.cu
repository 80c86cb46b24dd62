// Host side of the C ABI declared in include/attn.h: argument validation, TMA
// descriptor encoding, kernel dispatch, and the device watchdog word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_fwd_kernel.cuh"

namespace eta {

// Instantiated in the attn_inst_*.cu translation units.
#define ETA_DECLARE_C(D, DV, C)                                                          \
  extern template cudaError_t launch_attn<D, DV, C, BIAS_NONE>(const LaunchArgs &);         \
  extern template cudaError_t launch_attn<D, DV, C, BIAS_DENSE_TMA>(const LaunchArgs &);    \
  extern template cudaError_t launch_attn<D, DV, C, BIAS_DENSE_DIRECT>(const LaunchArgs &); \
  extern template cudaError_t launch_attn<D, DV, C, BIAS_KEY>(const LaunchArgs &);
#define ETA_DECLARE(D, DV) ETA_DECLARE_C(D, DV, false) ETA_DECLARE_C(D, DV, true)
ETA_DECLARE(64, 64)
ETA_DECLARE(64, 128)
ETA_DECLARE(128, 64)
ETA_DECLARE(128, 128)
#undef ETA_DECLARE
#undef ETA_DECLARE_C

namespace {

__device__ unsigned int g_watchdog = 0;

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_fault{FAULT_NONE};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 supported, -1 unsupported
  unsigned int *watchdog = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int device_pointer_ok(const void *ptr, int dev) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_INVALID_ARG;
  }
  if (attr.type == cudaMemoryTypeManaged) return ATTN_OK;
  if (attr.type == cudaMemoryTypeDevice && attr.device == dev) return ATTN_OK;
  return ATTN_ERR_INVALID_ARG;
}

// Current device: supported (compute capability 10.3) and its watchdog address.
int current_device(int *dev_out, unsigned int **watchdog) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) ? ATTN_ERR_NO_DEVICE
                                                                         : ATTN_ERR_CUDA;
  }
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceInfo &info = g_devices[dev];
  if (info.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      info.checked = -1;
    } else {
      void *addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_watchdog) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      info.watchdog = static_cast<unsigned int *>(addr);
      info.checked = 1;
    }
  }
  if (info.checked < 0) return ATTN_ERR_UNSUPPORTED_DEVICE;
  *dev_out = dev;
  *watchdog = info.watchdog;
  return ATTN_OK;
}

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  return g_encode ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D tiled map over a row-major [dim2][dim1][dim0] tensor, 128-byte swizzle.
int encode_3d(CUtensorMap *map, CUtensorMapDataType type, size_t elem, const void *ptr,
              uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0, uint32_t box1) {
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {dim0 * elem, dim0 * dim1 * elem};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, type, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, int DV, bool C>
cudaError_t dispatch_bias(int bias, const LaunchArgs &a) {
  switch (bias) {
    case BIAS_DENSE_TMA: return launch_attn<D, DV, C, BIAS_DENSE_TMA>(a);
    case BIAS_DENSE_DIRECT: return launch_attn<D, DV, C, BIAS_DENSE_DIRECT>(a);
    case BIAS_KEY: return launch_attn<D, DV, C, BIAS_KEY>(a);
    default: return launch_attn<D, DV, C, BIAS_NONE>(a);
  }
}
template <int D, int DV>
cudaError_t dispatch(bool causal, int bias, const LaunchArgs &a) {
  return causal ? dispatch_bias<D, DV, true>(bias, a) : dispatch_bias<D, DV, false>(bias, a);
}

}  // namespace
}  // namespace eta

using namespace eta;

extern "C" int attn_version(void) { return 100; }

extern "C" const char *attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument (pointer, alignment, overlap, size, mode or scale)";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head width (d and d_v must be 64 or 128)";
    case ATTN_ERR_NO_DEVICE: return "no CUDA device or driver available";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
    case ATTN_ERR_LAUNCH: return "kernel launch rejected by the CUDA runtime";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out (watchdog tripped)";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    default: return "unknown error code";
  }
}

extern "C" unsigned long long attn_set_wait_timeout_ns(unsigned long long ns) {
  return g_timeout_ns.exchange(ns == 0 ? kDefaultTimeoutNs : ns);
}

extern "C" int attn_set_fault_injection(int fault) {
  if (fault != FAULT_NONE && fault != FAULT_SKIP_FIRST_K) return ATTN_ERR_INVALID_ARG;
  g_fault.store(fault);
  return ATTN_OK;
}

extern "C" int attn_fwd_ex(const void *Q, const void *K, const void *V, int mode, const float *C,
                           const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                           void *O, int out_dtype, float *LSE, void *stream) {
  // ---- arguments (no CUDA call before these pass)
  if (mode & ~(ATTN_MASK_CAUSAL | ATTN_BIAS_DENSE | ATTN_BIAS_KEY)) return ATTN_ERR_INVALID_ARG;
  const bool causal = (mode & ATTN_MASK_CAUSAL) != 0;
  const bool dense = (mode & ATTN_BIAS_DENSE) != 0;
  const bool key = (mode & ATTN_BIAS_KEY) != 0;
  if (dense && key) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (BH < 1 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || (d_v != 64 && d_v != 128)) return ATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return ATTN_OK;  // empty buffers may be null
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;  // every row would lack an allowed key
  if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
  if (dense != (C != nullptr) || key != (ckey != nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
      (C && !aligned(C, 16)) || (ckey && !aligned(ckey, 4)) || (LSE && !aligned(LSE, 4)))
    return ATTN_ERR_INVALID_ARG;

  const size_t qrows = static_cast<size_t>(BH) * static_cast<size_t>(Nq);
  const size_t krows = static_cast<size_t>(BH) * static_cast<size_t>(Nk);
  const size_t o_bytes = qrows * d_v * (out_dtype == ATTN_OUT_F32 ? 4 : 2);
  const size_t lse_bytes = LSE ? qrows * 4 : 0;
  const void *ins[5] = {Q, K, V, C, ckey};
  const size_t in_bytes[5] = {qrows * d * 2, krows * d * 2, krows * d_v * 2,
                              C ? qrows * static_cast<size_t>(Nk) * 4 : 0, ckey ? krows * 4 : 0};
  for (int i = 0; i < 5; ++i) {
    if (ranges_overlap(O, o_bytes, ins[i], in_bytes[i]) || ranges_overlap(LSE, lse_bytes, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  }
  if (ranges_overlap(O, o_bytes, LSE, lse_bytes)) return ATTN_ERR_INVALID_ARG;

  // ---- device
  int dev = -1;
  unsigned int *watchdog = nullptr;
  int rc = current_device(&dev, &watchdog);
  if (rc != ATTN_OK) return rc;
  const void *ptrs[7] = {Q, K, V, O, C, ckey, LSE};
  for (const void *ptr : ptrs)
    if (ptr && device_pointer_ok(ptr, dev) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  if ((rc = get_encoder()) != ATTN_OK) return rc;

  LaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  const uint64_t nq = static_cast<uint64_t>(Nq), nk = static_cast<uint64_t>(Nk),
                 bh = static_cast<uint64_t>(BH);
  if (encode_3d(&a.tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Q, d, nq, bh, SW_CHUNK, BM) != ATTN_OK ||
      encode_3d(&a.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, d, nk, bh, SW_CHUNK, BN) != ATTN_OK ||
      encode_3d(&a.tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, d_v, nk, bh, SW_CHUNK, BN) != ATTN_OK)
    return ATTN_ERR_CUDA;
  // The dense bias goes through TMA when its rows are 16-byte multiples; otherwise the
  // softmax warps read it directly.
  int bias = BIAS_NONE;
  if (dense) bias = (Nk % 4 == 0) ? BIAS_DENSE_TMA : BIAS_DENSE_DIRECT;
  if (key) bias = BIAS_KEY;
  if (bias == BIAS_DENSE_TMA &&
      encode_3d(&a.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, nk, nq, bh, CCHUNK, BM) != ATTN_OK)
    return ATTN_ERR_CUDA;

  const int nq_tiles = (Nq + BM - 1) / BM;
  const int nqc = q_tiles_per_cta(bias);
  a.p.BH = BH;
  a.p.Nq = Nq;
  a.p.Nk = Nk;
  a.p.nq_tiles = nq_tiles;
  a.p.nkv_tiles = (Nk + BN - 1) / BN;
  a.p.causal_off = Nk - Nq;
  a.p.ctas_per_head = (nq_tiles + nqc - 1) / nqc;
  a.p.scale_log2 = scale * LOG2E;
  a.p.out_f32 = out_dtype == ATTN_OUT_F32 ? 1 : 0;
  a.p.O = O;
  a.p.LSE = LSE;
  a.p.C = C;
  a.p.ckey = ckey;
  a.p.status = watchdog;
  a.p.timeout_ns = g_timeout_ns.load();
  a.p.fault = g_fault.load();
  a.stream = static_cast<cudaStream_t>(stream);
  if (static_cast<uint64_t>(BH) * a.p.ctas_per_head > 0x7FFFFFFFull) return ATTN_ERR_INVALID_ARG;

  cudaError_t e;
  if (d == 64 && d_v == 64) e = dispatch<64, 64>(causal, bias, a);
  else if (d == 64) e = dispatch<64, 128>(causal, bias, a);
  else if (d_v == 64) e = dispatch<128, 64>(causal, bias, a);
  else e = dispatch<128, 128>(causal, bias, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

extern "C" int attn_fwd(const void *Q, const void *K, const void *V, int mode, const float *C,
                        int BH, int N, int d, int d_v, float scale, void *O, int out_dtype,
                        float *LSE, void *stream) {
  if (mode & ATTN_BIAS_KEY) return ATTN_ERR_INVALID_ARG;  // the per-key vector needs attn_fwd_ex
  return attn_fwd_ex(Q, K, V, mode, C, nullptr, BH, N, N, d, d_v, scale, O, out_dtype, LSE, stream);
}

extern "C" int attn_device_status(void *stream, unsigned int *detail) {
  if (detail) *detail = 0;
  int dev = -1;
  unsigned int *watchdog = nullptr;
  int rc = current_device(&dev, &watchdog);
  if (rc != ATTN_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  unsigned int word = 0;
  if (cudaMemcpy(&word, watchdog, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (detail) *detail = word;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(watchdog, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    return ATTN_ERR_DEVICE_TIMEOUT;
  }
  return ATTN_OK;
}

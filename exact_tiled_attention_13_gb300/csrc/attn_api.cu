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
#include "attn_merge_kernel.cuh"
#include "attn_bwd_kernel.cuh"

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
// CTA-pair forward kernels (attn_pair_inst.cu, attn_pair_dense_inst.cu, attn_pair_key_inst.cu).
template <int D, int DV, bool CAUSAL, int BIAS>
cudaError_t launch_attn_pair(const LaunchArgs &);
#define ETA_DECLARE_PAIR(D, C)                                                          \
  extern template cudaError_t launch_attn_pair<D, 128, C, BIAS_NONE>(const LaunchArgs &); \
  extern template cudaError_t launch_attn_pair<D, 128, C, BIAS_DENSE_TMA>(const LaunchArgs &);
ETA_DECLARE_PAIR(64, false)
ETA_DECLARE_PAIR(64, true)
ETA_DECLARE_PAIR(128, false)
ETA_DECLARE_PAIR(128, true)
#undef ETA_DECLARE_PAIR
extern template cudaError_t launch_attn_pair<64, 128, false, BIAS_KEY>(const LaunchArgs &);
extern template cudaError_t launch_attn_pair<64, 128, true, BIAS_KEY>(const LaunchArgs &);
#define ETA_DECLARE_BWD_C(D, DV, C)                                                       \
  extern template cudaError_t launch_bwd<D, DV, C, BWD_BIAS_NONE>(const BwdLaunchArgs &);  \
  extern template cudaError_t launch_bwd<D, DV, C, BWD_BIAS_DENSE>(const BwdLaunchArgs &); \
  extern template cudaError_t launch_bwd<D, DV, C, BWD_BIAS_KEY>(const BwdLaunchArgs &);
#define ETA_DECLARE_BWD(D, DV) ETA_DECLARE_BWD_C(D, DV, false) ETA_DECLARE_BWD_C(D, DV, true)
ETA_DECLARE_BWD(64, 64)
ETA_DECLARE_BWD(64, 128)
ETA_DECLARE_BWD(128, 64)
ETA_DECLARE_BWD(128, 128)
#undef ETA_DECLARE_BWD
#undef ETA_DECLARE_BWD_C

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
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

// The context current on this thread, or null; *known is false when the driver entry point
// could not be found (then nothing is known about the thread's binding).
CUcontext thread_context(bool *known) {
  std::call_once(g_ctx_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  *known = g_ctx_current != nullptr && g_ctx_current(&ctx) == CUDA_SUCCESS;
  return *known ? ctx : nullptr;
}

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
  // Make the device's primary context current on this thread: a thread that has not yet
  // made a runtime call that binds it (a framework's worker thread, say) would otherwise
  // have no context for the driver calls that encode the tensor maps. Done once per thread
  // and device, and again whenever the thread has been left with no current context (a
  // context popped or destroyed through the driver API since).
  thread_local int bound_dev = -1;
  bool known = false;
  if (bound_dev != dev || (thread_context(&known) == nullptr && known)) {
    if (cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    bound_dev = dev;
  }
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

template <int D, int DV, bool C>
cudaError_t dispatch_bwd_bias(int bias, const BwdLaunchArgs &a) {
  switch (bias) {
    case BWD_BIAS_DENSE: return launch_bwd<D, DV, C, BWD_BIAS_DENSE>(a);
    case BWD_BIAS_KEY: return launch_bwd<D, DV, C, BWD_BIAS_KEY>(a);
    default: return launch_bwd<D, DV, C, BWD_BIAS_NONE>(a);
  }
}
template <int D, int DV>
cudaError_t dispatch_bwd(bool causal, int bias, const BwdLaunchArgs &a) {
  return causal ? dispatch_bwd_bias<D, DV, true>(bias, a) : dispatch_bwd_bias<D, DV, false>(bias, a);
}

}  // namespace
}  // namespace eta

using namespace eta;

extern "C" int attn_version(void) { return ATTN_ABI_VERSION; }

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
    case ATTN_ERR_SCRATCH_LIMIT:
      return "the split plan needs more scratch than the library's fixed array (ATTN_STATIC_SCRATCH_BYTES)";
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

namespace eta {
namespace {

// One forward problem as the entry points receive it.
struct Problem {
  const void *Q, *K, *V;
  int mode;
  const float *C, *ckey;
  int BH, Nq, Nk, d, d_v;
  float scale;
  void *O;
  int out_dtype;
  float *LSE;
  void *stream;
  bool causal() const { return (mode & ATTN_MASK_CAUSAL) != 0; }
  bool dense() const { return (mode & ATTN_BIAS_DENSE) != 0; }
  bool shared() const { return (mode & ATTN_BIAS_SHARED) != 0; }
  size_t c_bytes() const {
    return C ? static_cast<size_t>(shared() ? 1 : BH) * Nq * static_cast<size_t>(Nk) * 4 : 0;
  }
  bool key() const { return (mode & ATTN_BIAS_KEY) != 0; }
  int bias() const {
    if (dense()) return (Nk % 4 == 0) ? BIAS_DENSE_TMA : BIAS_DENSE_DIRECT;
    return key() ? BIAS_KEY : BIAS_NONE;
  }
  int nkv_tiles() const { return (Nk + BN - 1) / BN; }
  int ctas_per_head() const {
    const int nqc = q_tiles_per_cta(bias(), d_v);
    return ((Nq + BM - 1) / BM + nqc - 1) / nqc;
  }
  size_t o_bytes() const {
    return static_cast<size_t>(BH) * Nq * d_v * (out_dtype == ATTN_OUT_F32 ? 4 : 2);
  }
  size_t lse_bytes() const { return LSE ? static_cast<size_t>(BH) * Nq * 4 : 0; }
};

constexpr int kEmpty = 1;  // check_shape: a valid call with nothing to do

// Checks of mode, sizes and scale (no pointer is looked at).
int check_shape(int mode, int BH, int Nq, int Nk, int d, int d_v, int out_dtype, float scale) {
  if (mode & ~(ATTN_MASK_CAUSAL | ATTN_BIAS_DENSE | ATTN_BIAS_KEY | ATTN_BIAS_SHARED)) return ATTN_ERR_INVALID_ARG;
  if ((mode & ATTN_BIAS_DENSE) && (mode & ATTN_BIAS_KEY)) return ATTN_ERR_INVALID_ARG;
  if ((mode & ATTN_BIAS_SHARED) && !(mode & ATTN_BIAS_DENSE)) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (BH < 1 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || (d_v != 64 && d_v != 128)) return ATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return kEmpty;                // empty buffers may be null
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;  // every row would lack an allowed key
  return ATTN_OK;
}

// Pointer checks that need no CUDA call: presence, alignment, overlaps.
int check_pointers(const Problem &a) {
  if (!a.Q || !a.K || !a.V || !a.O) return ATTN_ERR_INVALID_ARG;
  if (a.dense() != (a.C != nullptr) || a.key() != (a.ckey != nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(a.Q, 16) || !aligned(a.K, 16) || !aligned(a.V, 16) || !aligned(a.O, 16) ||
      (a.C && !aligned(a.C, 16)) || (a.ckey && !aligned(a.ckey, 4)) || (a.LSE && !aligned(a.LSE, 4)))
    return ATTN_ERR_INVALID_ARG;
  const size_t qrows = static_cast<size_t>(a.BH) * static_cast<size_t>(a.Nq);
  const size_t krows = static_cast<size_t>(a.BH) * static_cast<size_t>(a.Nk);
  const void *ins[5] = {a.Q, a.K, a.V, a.C, a.ckey};
  const size_t in_bytes[5] = {qrows * a.d * 2, krows * a.d * 2, krows * a.d_v * 2, a.c_bytes(),
                              a.ckey ? krows * 4 : 0};
  for (int i = 0; i < 5; ++i) {
    if (ranges_overlap(a.O, a.o_bytes(), ins[i], in_bytes[i]) ||
        ranges_overlap(a.LSE, a.lse_bytes(), ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  }
  if (ranges_overlap(a.O, a.o_bytes(), a.LSE, a.lse_bytes())) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Heads per scheduling group: as many as keep their K and V (bf16) within about 48 MB, a
// good part of the 126 MB L2 (see unit_of_block in the kernels).
int head_group(int BH, int Nk, int d, int d_v) {
  const double per_head = static_cast<double>(Nk) * (d + d_v) * 2.0;
  const double g = 48.0 * 1024 * 1024 / (per_head > 1.0 ? per_head : 1.0);
  return g >= BH ? BH : (g < 1.0 ? 1 : static_cast<int>(g));
}

// The persistent CTA-pair kernel (attn_fwd_pair_kernel.cuh) serves problems with 128 value
// columns in one key range without a bias term (causal or not), with a dense bias read
// through TMA (there attn_fwd_kernel holds one query tile per CTA and its chain
// softmax -> P V -> next S is exposed), and at d = 64 with a per-key bias, which it folds
// into the score product. Everything else goes to attn_fwd_kernel. Measured on 16 heads of
// N = 16384 without a mask, the pair kernel is 4 % faster with scores x 4 and 8 % with plain
// scores, although a tile that moves a row's exponent reference there waits for the
// previous P V before rescaling o. A per-key bias added by the pair kernel's softmax (as the
// dense bias is) made it slower than attn_fwd_kernel (73.5 against 60.4 us on 8 heads of
// N = 4096, d = 64): the add and the row maximum it then needs lengthen the hand-off of the
// reference between its warpgroups; folded into the product, the softmax is the unbiased one.
bool use_pair_kernel(const Problem &a, int n_splits) {
  if (a.d_v != 128 || n_splits != 1) return false;
  const int bias = a.bias();
  return bias == BIAS_DENSE_TMA || bias == BIAS_NONE || (bias == BIAS_KEY && a.d == 64);
}

template <int D, bool C>
cudaError_t dispatch_pair(int bias, const LaunchArgs &a) {
  if constexpr (D == 64)
    if (bias == BIAS_KEY) return launch_attn_pair<D, 128, C, BIAS_KEY>(a);
  return bias == BIAS_DENSE_TMA ? launch_attn_pair<D, 128, C, BIAS_DENSE_TMA>(a)
                                : launch_attn_pair<D, 128, C, BIAS_NONE>(a);
}

// Launches the attention kernel. With n_splits > 1 each CTA covers `split_tiles` K/V
// tiles of its head and writes fp32 partials to O_dst / LSE_dst instead of O / LSE.
int launch_forward(const Problem &a, unsigned int *watchdog, int n_splits, int split_tiles,
                   void *O_dst, float *LSE_dst, int out_f32) {
  int rc;
  if ((rc = get_encoder()) != ATTN_OK) return rc;
  LaunchArgs la;
  std::memset(&la, 0, sizeof(la));
  const uint64_t nq = static_cast<uint64_t>(a.Nq), nk = static_cast<uint64_t>(a.Nk),
                 bh = static_cast<uint64_t>(a.BH);
  if (encode_3d(&la.tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.Q, a.d, nq, bh, SW_CHUNK, BM) != ATTN_OK ||
      encode_3d(&la.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.d, nk, bh, SW_CHUNK, BN) != ATTN_OK ||
      encode_3d(&la.tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.V, a.d_v, nk, bh, SW_CHUNK, BN) != ATTN_OK)
    return ATTN_ERR_CUDA;
  // The dense bias goes through TMA when its rows are 16-byte multiples; otherwise the
  // softmax warps read it directly.
  const int bias = a.bias();
  if (bias == BIAS_DENSE_TMA &&
      encode_3d(&la.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.C, nk, nq, a.shared() ? 1 : bh, CCHUNK, BM) != ATTN_OK)
    return ATTN_ERR_CUDA;

  la.p.BH = a.BH;
  la.p.Nq = a.Nq;
  la.p.Nk = a.Nk;
  la.p.nq_tiles = (a.Nq + BM - 1) / BM;
  la.p.nkv_tiles = a.nkv_tiles();
  la.p.causal_off = a.Nk - a.Nq;
  la.p.ctas_per_head = a.ctas_per_head();
  la.p.n_splits = n_splits;
  la.p.split_tiles = split_tiles;
  la.p.head_group = head_group(a.BH, a.Nk, a.d, a.d_v);
  la.p.scale_log2 = a.scale * LOG2E;
  la.p.out_f32 = out_f32;
  la.p.O = O_dst;
  la.p.LSE = LSE_dst;
  la.p.C = a.C;
  la.p.c_shared = a.shared() ? 1 : 0;
  la.p.ckey = a.ckey;
  la.p.status = watchdog;
  la.p.timeout_ns = g_timeout_ns.load();
  la.p.fault = g_fault.load();
  la.stream = static_cast<cudaStream_t>(a.stream);
  if (static_cast<uint64_t>(a.BH) * la.p.ctas_per_head * n_splits > 0x3FFFFFFFull)
    return ATTN_ERR_INVALID_ARG;

  cudaError_t e;
  const bool causal = a.causal();
  if (use_pair_kernel(a, n_splits)) {
    // CTA pairs: each CTA copies 64 keys of every K tile (one 64 x 64 box per 128-byte span).
    if (encode_3d(&la.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.K, a.d, nk, bh, SW_CHUNK, BN / 2) != ATTN_OK)
      return ATTN_ERR_CUDA;
    // Its epilogue stores O with TMA, 32 rows x 128 bytes per box.
    const int rc_o = out_f32 ? encode_3d(&la.tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, O_dst, a.d_v, nq, bh, 32, 32)
                             : encode_3d(&la.tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, O_dst, a.d_v, nq, bh, 64, 32);
    if (rc_o != ATTN_OK) return ATTN_ERR_CUDA;
    // Units of 256 query rows (a query tile in each CTA of the pair), whatever the bias.
    la.p.ctas_per_head = (la.p.nq_tiles + 1) / 2;
    if (a.d == 64) e = causal ? dispatch_pair<64, true>(bias, la) : dispatch_pair<64, false>(bias, la);
    else e = causal ? dispatch_pair<128, true>(bias, la) : dispatch_pair<128, false>(bias, la);
  } else if (a.d == 64 && a.d_v == 64) e = dispatch<64, 64>(causal, bias, la);
  else if (a.d == 64) e = dispatch<64, 128>(causal, bias, la);
  else if (a.d_v == 64) e = dispatch<128, 64>(causal, bias, la);
  else e = dispatch<128, 128>(causal, bias, la);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

constexpr int kMaxSplits = 1024;


// Number of key ranges for a split launch and the K/V tiles of each. A request of
// n_splits ranges is rounded to whole tiles: split_tiles = ceil(nkv / n_splits), and
// only ceil(nkv / split_tiles) ranges are non-empty. n_splits == 0 chooses the count
// for `sms` multiprocessors: the one that minimises waves x tiles per range, plus a
// small charge per range for writing and merging its partials.
void split_plan(const Problem &a, int n_splits, int sms, int *splits, int *split_tiles) {
  const int nkv = a.nkv_tiles();
  if (n_splits <= 0) {
    const long long base = static_cast<long long>(a.BH) * a.ctas_per_head();
    int best = 1;
    double best_cost = 1e300;
    for (int s = 1; s <= nkv && s <= kMaxSplits; ++s) {
      const int chunk = (nkv + s - 1) / s;
      const int eff = (nkv + chunk - 1) / chunk;
      if (eff != s) continue;  // the same ranges as a smaller request
      const long long waves = (base * eff + sms - 1) / sms;
      const double cost = static_cast<double>(waves) * chunk + 0.125 * eff;
      if (cost < best_cost) {
        best_cost = cost;
        best = s;
      }
    }
    n_splits = best;
  }
  if (n_splits > nkv) n_splits = nkv;
  *split_tiles = (nkv + n_splits - 1) / n_splits;
  *splits = (nkv + *split_tiles - 1) / *split_tiles;
}

unsigned long long split_workspace_bytes(const Problem &a, int splits) {
  if (splits <= 1) return 0;
  return static_cast<unsigned long long>(splits) * a.BH * a.Nq * (a.d_v + 1) * 4ull;
}

int sm_count(int dev, int *sms) {
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace
}  // namespace eta

extern "C" int attn_fwd_ex(const void *Q, const void *K, const void *V, int mode, const float *C,
                           const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                           void *O, int out_dtype, float *LSE, void *stream) {
  // ---- arguments (no CUDA call before these pass)
  int rc = check_shape(mode, BH, Nq, Nk, d, d_v, out_dtype, scale);
  if (rc == kEmpty) return ATTN_OK;
  if (rc != ATTN_OK) return rc;
  const Problem a{Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, O, out_dtype, LSE, stream};
  if ((rc = check_pointers(a)) != ATTN_OK) return rc;

  // ---- device
  int dev = -1;
  unsigned int *watchdog = nullptr;
  if ((rc = current_device(&dev, &watchdog)) != ATTN_OK) return rc;
  const void *ptrs[7] = {Q, K, V, O, C, ckey, LSE};
  for (const void *ptr : ptrs)
    if (ptr && device_pointer_ok(ptr, dev) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  return launch_forward(a, watchdog, 1, a.nkv_tiles(), O, LSE, out_dtype == ATTN_OUT_F32 ? 1 : 0);
}

extern "C" int attn_fwd_splitkv_plan(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                     int n_splits, int *splits, unsigned long long *workspace_bytes) {
  if (splits) *splits = 0;
  if (workspace_bytes) *workspace_bytes = 0;
  if (!splits || !workspace_bytes || n_splits < 0) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(mode, BH, Nq, Nk, d, d_v, ATTN_OUT_F32, 1.0f);
  if (rc == kEmpty) {
    *splits = 1;
    return ATTN_OK;
  }
  if (rc != ATTN_OK) return rc;
  const Problem a{nullptr, nullptr, nullptr, mode, nullptr, nullptr, BH, Nq, Nk, d, d_v,
                  1.0f, nullptr, ATTN_OUT_F32, nullptr, nullptr};
  int sms = 0;
  if (n_splits == 0) {
    int dev = -1;
    unsigned int *watchdog = nullptr;
    if ((rc = current_device(&dev, &watchdog)) != ATTN_OK) return rc;
    if ((rc = sm_count(dev, &sms)) != ATTN_OK) return rc;
  }
  int tiles = 0;
  split_plan(a, n_splits, sms, splits, &tiles);
  *workspace_bytes = split_workspace_bytes(a, *splits);
  return ATTN_OK;
}

extern "C" int attn_fwd_splitkv(const void *Q, const void *K, const void *V, int mode,
                                const float *C, const float *ckey, int BH, int Nq, int Nk, int d,
                                int d_v, float scale, int n_splits, void *workspace,
                                unsigned long long workspace_bytes, void *O, int out_dtype,
                                float *LSE, void *stream) {
  // ---- arguments (no CUDA call before these pass)
  if (n_splits < 0) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(mode, BH, Nq, Nk, d, d_v, out_dtype, scale);
  if (rc == kEmpty) return ATTN_OK;
  if (rc != ATTN_OK) return rc;
  const Problem a{Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, O, out_dtype, LSE, stream};
  if ((rc = check_pointers(a)) != ATTN_OK) return rc;

  // ---- device and plan
  int dev = -1;
  unsigned int *watchdog = nullptr;
  if ((rc = current_device(&dev, &watchdog)) != ATTN_OK) return rc;
  int sms = 0;
  if (n_splits == 0 && (rc = sm_count(dev, &sms)) != ATTN_OK) return rc;
  int splits = 1, tiles = 0;
  split_plan(a, n_splits, sms, &splits, &tiles);
  const unsigned long long need = split_workspace_bytes(a, splits);
  if (splits > 1) {
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    const void *bufs[7] = {Q, K, V, C, ckey, O, LSE};
    const size_t qrows = static_cast<size_t>(BH) * Nq, krows = static_cast<size_t>(BH) * Nk;
    const size_t sizes[7] = {qrows * d * 2, krows * d * 2, krows * d_v * 2, a.c_bytes(),
                             ckey ? krows * 4 : 0, a.o_bytes(), a.lse_bytes()};
    for (int i = 0; i < 7; ++i)
      if (ranges_overlap(workspace, need, bufs[i], sizes[i])) return ATTN_ERR_INVALID_ARG;
  }
  const void *ptrs[8] = {Q, K, V, O, C, ckey, LSE, splits > 1 ? workspace : nullptr};
  for (const void *ptr : ptrs)
    if (ptr && device_pointer_ok(ptr, dev) != ATTN_OK) return ATTN_ERR_INVALID_ARG;

  const int out_f32 = out_dtype == ATTN_OUT_F32 ? 1 : 0;
  if (splits == 1) return launch_forward(a, watchdog, 1, a.nkv_tiles(), O, LSE, out_f32);

  // Partials: O_part [splits][BH][Nq][d_v] fp32, then L_part [splits][BH][Nq] fp32.
  float *O_part = static_cast<float *>(workspace);
  float *L_part = O_part + static_cast<size_t>(splits) * BH * Nq * d_v;
  if ((rc = launch_forward(a, watchdog, splits, tiles, O_part, L_part, 1)) != ATTN_OK) return rc;
  const long long rows = static_cast<long long>(BH) * Nq;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d_v == 64 ? launch_merge<64>(O_part, L_part, splits, rows, O, out_f32, LSE, st)
                                  : launch_merge<128>(O_part, L_part, splits, rows, O, out_f32, LSE, st);
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

// ------------------------------------------------------------------ backward pass
namespace eta {
namespace {
unsigned long long bwd_workspace_bytes(int BH, int Nq) {
  const unsigned long long nqp = static_cast<unsigned long long>((Nq + BM - 1) / BM) * BM;
  return 2ull * static_cast<unsigned long long>(BH) * nqp * 4ull;
}
}  // namespace
}  // namespace eta

extern "C" int attn_bwd_workspace_bytes(int BH, int Nq, unsigned long long *bytes) {
  if (bytes) *bytes = 0;
  if (!bytes || BH < 1 || Nq < 0) return ATTN_ERR_INVALID_ARG;
  *bytes = bwd_workspace_bytes(BH, Nq);
  return ATTN_OK;
}

extern "C" int attn_bwd(const void *Q, const void *K, const void *V, const void *O, int o_dtype,
                        const void *dO, const float *LSE, int mode, const float *C,
                        const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                        float *dQ, float *dK, float *dV, void *workspace,
                        unsigned long long workspace_bytes, void *stream) {
  // ---- arguments (no CUDA call before these pass)
  int rc = check_shape(mode, BH, Nq, Nk, d, d_v, o_dtype, scale);
  if (rc < 0) return rc;
  if (Nk == 0) return Nq == 0 ? ATTN_OK : ATTN_ERR_INVALID_ARG;
  const bool no_queries = Nq == 0;
  const size_t qrows = static_cast<size_t>(BH) * static_cast<size_t>(Nq);
  const size_t krows = static_cast<size_t>(BH) * static_cast<size_t>(Nk);
  const unsigned long long need = bwd_workspace_bytes(BH, Nq);
  if (!K || !V || !dK || !dV) return ATTN_ERR_INVALID_ARG;
  if (!no_queries && (!Q || !O || !dO || !LSE || !dQ || !workspace || workspace_bytes < need))
    return ATTN_ERR_INVALID_ARG;
  const bool dense = (mode & ATTN_BIAS_DENSE) != 0, key = (mode & ATTN_BIAS_KEY) != 0;
  if (dense != (C != nullptr) || key != (ckey != nullptr)) return ATTN_ERR_INVALID_ARG;
  const void *a16[9] = {Q, K, V, O, dO, C, dQ, dK, dV};
  for (const void *ptr : a16)
    if (ptr && !aligned(ptr, 16)) return ATTN_ERR_INVALID_ARG;
  if ((LSE && !aligned(LSE, 4)) || (ckey && !aligned(ckey, 4)) || (workspace && !aligned(workspace, 16)))
    return ATTN_ERR_INVALID_ARG;
  // Outputs (dQ, dK, dV, workspace) overlap no input and no other output.
  const void *ins[8] = {Q, K, V, O, dO, LSE, C, ckey};
  const size_t c_rows = (mode & ATTN_BIAS_SHARED) ? static_cast<size_t>(Nq) : qrows;
  const size_t in_bytes[8] = {qrows * d * 2, krows * d * 2, krows * d_v * 2,
                              qrows * d_v * (o_dtype == ATTN_OUT_F32 ? 4 : 2), qrows * d_v * 2,
                              qrows * 4, C ? c_rows * static_cast<size_t>(Nk) * 4 : 0,
                              ckey ? krows * 4 : 0};
  const void *outs[4] = {dQ, dK, dV, no_queries ? nullptr : workspace};
  const size_t out_bytes[4] = {qrows * d * 4, krows * d * 4, krows * d_v * 4, need};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 8; ++i)
      if (ranges_overlap(outs[o], out_bytes[o], ins[i], in_bytes[i])) return ATTN_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 4; ++o2)
      if (ranges_overlap(outs[o], out_bytes[o], outs[o2], out_bytes[o2])) return ATTN_ERR_INVALID_ARG;
  }

  // ---- device
  int dev = -1;
  unsigned int *watchdog = nullptr;
  if ((rc = current_device(&dev, &watchdog)) != ATTN_OK) return rc;
  const void *ptrs[12] = {Q, K, V, O, dO, LSE, C, ckey, dQ, dK, dV, no_queries ? nullptr : workspace};
  for (const void *ptr : ptrs)
    if (ptr && device_pointer_ok(ptr, dev) != ATTN_OK) return ATTN_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (no_queries) {  // no query sees any key: the key and value gradients are zero
    if (cudaMemsetAsync(dK, 0, krows * d * 4, st) != cudaSuccess ||
        cudaMemsetAsync(dV, 0, krows * d_v * 4, st) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
  }
  if ((rc = get_encoder()) != ATTN_OK) return rc;

  BwdLaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  const uint64_t nq = static_cast<uint64_t>(Nq), nk = static_cast<uint64_t>(Nk),
                 bh = static_cast<uint64_t>(BH);
  if (encode_3d(&a.tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Q, d, nq, bh, SW_CHUNK, BM) != ATTN_OK ||
      encode_3d(&a.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, d, nk, bh, SW_CHUNK, BN) != ATTN_OK ||
      encode_3d(&a.tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, d_v, nk, bh, SW_CHUNK, BN) != ATTN_OK ||
      encode_3d(&a.tmdO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dO, d_v, nq, bh, SW_CHUNK, BM) != ATTN_OK)
    return ATTN_ERR_CUDA;
  const int nq_tiles = (Nq + BM - 1) / BM;
  BwdParams &pp = a.p;
  pp.BH = BH;
  pp.Nq = Nq;
  pp.Nk = Nk;
  pp.nq_tiles = nq_tiles;
  pp.nkv_tiles = (Nk + BN - 1) / BN;
  pp.causal_off = Nk - Nq;
  pp.nqp = nq_tiles * BM;
  pp.head_group = head_group(BH, Nq + Nk, d, d_v);
  pp.scale_log2 = scale * LOG2E;
  pp.scale = scale;
  float *Lp = static_cast<float *>(workspace);
  float *Dd = Lp + static_cast<size_t>(BH) * pp.nqp;
  pp.Lp = Lp;
  pp.Dd = Dd;
  pp.C = C;
  pp.c_shared = (mode & ATTN_BIAS_SHARED) ? 1 : 0;
  pp.ckey = ckey;
  pp.dQ = dQ;
  pp.dK = dK;
  pp.dV = dV;
  pp.status = watchdog;
  pp.timeout_ns = g_timeout_ns.load();
  a.stream = st;
  if (static_cast<uint64_t>(BH) * (pp.nkv_tiles > nq_tiles ? pp.nkv_tiles : nq_tiles) > 0x7FFFFFFFull)
    return ATTN_ERR_INVALID_ARG;

  const int out_f32 = o_dtype == ATTN_OUT_F32 ? 1 : 0;
  const uint16_t *dO16 = static_cast<const uint16_t *>(dO);
  cudaError_t e = d_v == 64 ? launch_bwd_prep<64>(O, out_f32, dO16, LSE, BH, Nq, pp.nqp, Lp, Dd, st)
                            : launch_bwd_prep<128>(O, out_f32, dO16, LSE, BH, Nq, pp.nqp, Lp, Dd, st);
  if (e == cudaSuccess) {
    const bool causal = (mode & ATTN_MASK_CAUSAL) != 0;
    const int bias = dense ? BWD_BIAS_DENSE : (key ? BWD_BIAS_KEY : BWD_BIAS_NONE);
    if (d == 64 && d_v == 64) e = dispatch_bwd<64, 64>(causal, bias, a);
    else if (d == 64) e = dispatch_bwd<64, 128>(causal, bias, a);
    else if (d_v == 64) e = dispatch_bwd<128, 64>(causal, bias, a);
    else e = dispatch_bwd<128, 128>(causal, bias, a);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

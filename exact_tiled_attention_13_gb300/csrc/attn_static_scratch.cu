// attn_fwd_splitkv_static: the split forward pass for callers that cannot allocate
// device memory. Its partials live in a fixed array of this translation unit instead of
// a caller-provided workspace; everything else is attn_fwd_splitkv.
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"

namespace {

constexpr unsigned long long kScratchBytes = ATTN_STATIC_SCRATCH_BYTES;

// One copy per device (a __device__ variable exists once in every device's instance of
// the module). Nothing in it has to start at zero: every partial the merge kernel reads
// is written earlier in the same call by the attention kernel.
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_scratch on the current device, looked up once per device and kept for
// the life of the process (a cudaDeviceReset unloads the module and invalidates it; the
// header tells callers not to reset a device the library is still used on).
int scratch_on_current_device(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) ? ATTN_ERR_NO_DEVICE
                                                                         : ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  // The library holds device code for compute capability 10.3 only: on any other device the
  // symbol lookup would fail, so report the unsupported device the way every entry point does.
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ready[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(static_cast<void **>(&ptr), g_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_splitkv_static(const void *Q, const void *K, const void *V, int mode,
                                       const float *C, const float *ckey, int BH, int Nq, int Nk,
                                       int d, int d_v, float scale, int n_splits, void *O,
                                       int out_dtype, float *LSE, void *stream) {
  int splits = 0;
  unsigned long long need = 0;
  int rc = attn_fwd_splitkv_plan(mode, BH, Nq, Nk, d, d_v, n_splits, &splits, &need);
  if (rc != ATTN_OK) return rc;
  if (need > kScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  if (need > 0 && (rc = scratch_on_current_device(&scratch)) != ATTN_OK) return rc;
  return attn_fwd_splitkv(Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale, n_splits, scratch,
                          need > 0 ? kScratchBytes : 0, O, out_dtype, LSE, stream);
}

// Backward-pass kernel instances for d = 128, d_v = 128.
#include "attn_bwd_kernel.cuh"

namespace eta {
#define ETA_BWD_INST(C)                                                    \
  template cudaError_t launch_bwd<128, 128, C, BWD_BIAS_NONE>(const BwdLaunchArgs &);  \
  template cudaError_t launch_bwd<128, 128, C, BWD_BIAS_DENSE>(const BwdLaunchArgs &); \
  template cudaError_t launch_bwd<128, 128, C, BWD_BIAS_KEY>(const BwdLaunchArgs &);
ETA_BWD_INST(false)
ETA_BWD_INST(true)
#undef ETA_BWD_INST
}  // namespace eta

// Backward-pass kernel instances for d = 64, d_v = 64.
#include "attn_bwd_kernel.cuh"

namespace eta {
#define ETA_BWD_INST(C)                                                    \
  template cudaError_t launch_bwd<64, 64, C, BWD_BIAS_NONE>(const BwdLaunchArgs &);  \
  template cudaError_t launch_bwd<64, 64, C, BWD_BIAS_DENSE>(const BwdLaunchArgs &); \
  template cudaError_t launch_bwd<64, 64, C, BWD_BIAS_KEY>(const BwdLaunchArgs &);
ETA_BWD_INST(false)
ETA_BWD_INST(true)
#undef ETA_BWD_INST
}  // namespace eta

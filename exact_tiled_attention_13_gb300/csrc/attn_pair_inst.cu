// Kernel instances of the CTA-pair forward pass without a bias term (d_v = 128): d = 64 and
// 128, with and without the causal mask.
#include "attn_fwd_pair_kernel.cuh"

namespace eta {
template cudaError_t launch_attn_pair<64, 128, false, BIAS_NONE>(const LaunchArgs &);
template cudaError_t launch_attn_pair<64, 128, true, BIAS_NONE>(const LaunchArgs &);
template cudaError_t launch_attn_pair<128, 128, false, BIAS_NONE>(const LaunchArgs &);
template cudaError_t launch_attn_pair<128, 128, true, BIAS_NONE>(const LaunchArgs &);
}  // namespace eta

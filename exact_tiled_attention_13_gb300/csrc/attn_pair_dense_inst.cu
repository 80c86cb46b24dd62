// Kernel instances of the CTA-pair forward pass with a dense bias read through TMA
// (d_v = 128): d = 64 and 128, with and without the causal mask.
#include "attn_fwd_pair_kernel.cuh"

namespace eta {
template cudaError_t launch_attn_pair<64, 128, false, BIAS_DENSE_TMA>(const LaunchArgs &);
template cudaError_t launch_attn_pair<64, 128, true, BIAS_DENSE_TMA>(const LaunchArgs &);
template cudaError_t launch_attn_pair<128, 128, false, BIAS_DENSE_TMA>(const LaunchArgs &);
template cudaError_t launch_attn_pair<128, 128, true, BIAS_DENSE_TMA>(const LaunchArgs &);
}  // namespace eta

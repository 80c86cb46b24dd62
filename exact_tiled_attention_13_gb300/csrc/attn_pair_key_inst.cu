// Kernel instances of the CTA-pair forward pass with a per-key bias folded into the score
// product (d = 64, d_v = 128), with and without the causal mask.
#include "attn_fwd_pair_kernel.cuh"

namespace eta {
template cudaError_t launch_attn_pair<64, 128, false, BIAS_KEY>(const LaunchArgs &);
template cudaError_t launch_attn_pair<64, 128, true, BIAS_KEY>(const LaunchArgs &);
}  // namespace eta

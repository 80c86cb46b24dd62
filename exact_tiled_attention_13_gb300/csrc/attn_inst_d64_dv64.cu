// Kernel instances for d = 64, d_v = 64 (one translation unit per head-width pair so
// the instances compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace eta {
template cudaError_t launch_attn<64, 64, MODE_NONE, false>(const LaunchArgs &);
template cudaError_t launch_attn<64, 64, MODE_CAUSAL, false>(const LaunchArgs &);
template cudaError_t launch_attn<64, 64, MODE_DENSE, true>(const LaunchArgs &);
template cudaError_t launch_attn<64, 64, MODE_DENSE, false>(const LaunchArgs &);
}  // namespace eta

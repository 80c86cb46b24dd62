// Kernel instances for d = 128, d_v = 128 (one translation unit per head-width pair so
// the instances compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace eta {
template cudaError_t launch_attn<128, 128, MODE_NONE, false>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, MODE_CAUSAL, false>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, MODE_DENSE, true>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, MODE_DENSE, false>(const LaunchArgs &);
}  // namespace eta

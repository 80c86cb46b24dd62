// Kernel instances for d = 128, d_v = 128: with and without the causal mask, for each bias
// source (one translation unit per head-width pair so the instances compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace eta {
template cudaError_t launch_attn<128, 128, false, BIAS_NONE>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, false, BIAS_DENSE_TMA>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, false, BIAS_DENSE_DIRECT>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, false, BIAS_KEY>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, true, BIAS_NONE>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, true, BIAS_DENSE_TMA>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, true, BIAS_DENSE_DIRECT>(const LaunchArgs &);
template cudaError_t launch_attn<128, 128, true, BIAS_KEY>(const LaunchArgs &);
}  // namespace eta

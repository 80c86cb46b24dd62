// Merge of the per-key-range partial results of a split forward pass.
//
// A split launch runs the attention kernel once per range of K/V tiles and stores, for
// every query row and range s, the normalised partial output O_s = o_s / l_s (fp32) and
// its log-sum-exp LSE_s = m_s + ln l_s (-inf when the range holds no allowed key). The
// pages combine two partial softmax states by rescaling both to the larger maximum
// ("AI Infra ch. 5", section 5.4, the blockwise-softmax statistics (m, l); "Compilers
// and kernels", section "FlashAttention rewrites the algorithm around IO": the same
// alpha rescaling). Written with LSE instead of (m, l), for ranges s = 0 .. S-1:
//
//     M = max_s LSE_s,  w_s = exp(LSE_s - M),  O = sum_s w_s O_s / sum_s w_s,
//     LSE = M + ln sum_s w_s,
//
// since l_s exp(m_s - M) = exp(LSE_s - M). The sum runs over s in increasing order in
// one lane per output element, so the result is deterministic (no atomics). A row
// whose every range is empty gets O = 0 and LSE = -inf.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace eta {

// One warp per query row; lane i holds columns [i*VEC, i*VEC + VEC) of the row (VEC = DV/32
// consecutive floats, one vector load per range), so a row's partials are read as whole
// 16-byte (DV = 128) or 8-byte (DV = 64) pieces. The ranges' LSE values are spread over the
// lanes (range s on lane s mod 32): each weight is computed once and passed on by shuffle.
// The per-element sums still run over s in increasing order. The merge is a few loads per
// lane and bound by memory latency, so a lane issues the loads of a whole batch of up to 32
// ranges before it uses the first.
// O_part: [S][rows][DV] fp32; L_part: [S][rows] fp32; O: [rows][DV] (fp32 or bf16);
// LSE: [rows] or null.
template <int DV>
__global__ void __launch_bounds__(128)
    attn_merge_kernel(const float *__restrict__ O_part, const float *__restrict__ L_part,
                      int n_splits, long long rows, void *O, int out_f32, float *LSE) {
  static_assert(DV == 64 || DV == 128, "d_v of the merge");
  constexpr int VEC = DV / 32;
  constexpr int UNROLL = 32;
  using vec_t = typename std::conditional<VEC == 4, float4, float2>::type;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  grid_dep_wait();  // the attention kernel's partials
  if (threadIdx.x == 0) grid_dep_launch();
  if (row >= rows) return;

  float M = -INFINITY;
  for (int s0 = 0; s0 < n_splits; s0 += 32)
    if (s0 + lane < n_splits) M = fmaxf(M, __ldg(L_part + (s0 + lane) * rows + row));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));

  float acc[VEC] = {};
  float wsum = 0.0f;
  if (M != -INFINITY) {
    const vec_t *src = reinterpret_cast<const vec_t *>(O_part) + row * (DV / VEC) + lane;
    const long long range_stride = rows * (DV / VEC);
    for (int s0 = 0; s0 < n_splits; s0 += 32) {
      // Weight of range s0 + lane (0 past the last range; exp(-inf) = 0 for an empty one).
      const float wl = s0 + lane < n_splits ? expf(__ldg(L_part + (s0 + lane) * rows + row) - M) : 0.0f;
      const int n = n_splits - s0 < 32 ? n_splits - s0 : 32;
      for (int k0 = 0; k0 < n; k0 += UNROLL) {
        vec_t v[UNROLL];
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          const int s = s0 + (k0 + k < n ? k0 + k : n - 1);  // clamped: weight 0 below
          v[k] = __ldg(src + s * range_stride);
        }
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          const float wk = __shfl_sync(0xFFFFFFFFu, wl, (k0 + k) & 31);
          const float w = k0 + k < n ? wk : 0.0f;
          const float *x = reinterpret_cast<const float *>(&v[k]);
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[j] = fmaf(w, x[j], acc[j]);
          wsum += w;
        }
      }
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  if (out_f32) {
    vec_t r;
    float *x = reinterpret_cast<float *>(&r);
#pragma unroll
    for (int j = 0; j < VEC; ++j) x[j] = acc[j] * inv;
    reinterpret_cast<vec_t *>(O)[row * (DV / VEC) + lane] = r;
  } else {
    uint32_t packed[VEC / 2];
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j) packed[j] = pack_bf16(acc[2 * j] * inv, acc[2 * j + 1] * inv);
    uint16_t *dst = static_cast<uint16_t *>(O) + row * DV + lane * VEC;
    if constexpr (VEC == 4)
      *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    else
      *reinterpret_cast<uint32_t *>(dst) = packed[0];
  }
  if (LSE != nullptr && lane == 0) LSE[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

template <int DV>
cudaError_t launch_merge(const float *O_part, const float *L_part, int n_splits, long long rows,
                         void *O, int out_f32, float *LSE, cudaStream_t stream) {
  constexpr int kRowsPerBlock = 4;  // one warp per row
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(attn_merge_kernel<DV>, dim3(static_cast<unsigned>(blocks)),
                                   dim3(32 * kRowsPerBlock), 0, stream, O_part, L_part, n_splits, rows, O,
                                   out_f32, LSE);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace eta

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
// one thread per output element, so the result is deterministic (no atomics). A row
// whose every range is empty gets O = 0 and LSE = -inf.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"

namespace eta {

constexpr int MERGE_ROWS_PER_BLOCK = 8;  // one warp per query row

// O_part: [S][rows][DV] fp32; L_part: [S][rows] fp32; O: [rows][DV] (fp32 or bf16);
// LSE: [rows] or null.
template <int DV>
__global__ void __launch_bounds__(32 * MERGE_ROWS_PER_BLOCK)
    attn_merge_kernel(const float *__restrict__ O_part, const float *__restrict__ L_part,
                      int n_splits, long long rows, void *O, int out_f32, float *LSE) {
  constexpr int W = DV / 32;  // columns per lane: 4 (d_v = 128) or 2 (d_v = 64)
  const long long row = static_cast<long long>(blockIdx.x) * MERGE_ROWS_PER_BLOCK + threadIdx.x / 32;
  if (row >= rows) return;
  const int lane = threadIdx.x % 32;

  // The ranges' loads are independent: batches of 8 are issued before any is used, so
  // the kernel is not a chain of memory round trips.
  float M = -INFINITY;
#pragma unroll 8
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, __ldg(L_part + s * rows + row));

  float acc[W];
#pragma unroll
  for (int c = 0; c < W; ++c) acc[c] = 0.0f;
  float wsum = 0.0f;
  if (M != -INFINITY) {
    constexpr int B = 8;
    for (int s0 = 0; s0 < n_splits; s0 += B) {
      float w[B], v[B][W];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int s = s0 + k < n_splits ? s0 + k : n_splits - 1;  // clamped: weight 0 below
        w[k] = __ldg(L_part + s * rows + row);
        const float *src = O_part + (s * rows + row) * DV + lane * W;
        if constexpr (W == 4) {
          const float4 t = __ldg(reinterpret_cast<const float4 *>(src));
          v[k][0] = t.x, v[k][1] = t.y, v[k][2] = t.z, v[k][3] = t.w;
        } else {
          const float2 t = __ldg(reinterpret_cast<const float2 *>(src));
          v[k][0] = t.x, v[k][1] = t.y;
        }
      }
      // In increasing range order, as the sums are defined.
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const float wk = s0 + k < n_splits ? expf(w[k] - M) : 0.0f;  // 0 for an empty range
#pragma unroll
        for (int c = 0; c < W; ++c) acc[c] = fmaf(wk, v[k][c], acc[c]);
        wsum += wk;
      }
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int c = 0; c < W; ++c) acc[c] *= inv;

  if (out_f32) {
    float *dst = static_cast<float *>(O) + row * DV + lane * W;
    if constexpr (W == 4)
      *reinterpret_cast<float4 *>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else
      *reinterpret_cast<float2 *>(dst) = make_float2(acc[0], acc[1]);
  } else {
    uint16_t *dst = static_cast<uint16_t *>(O) + row * DV + lane * W;
    if constexpr (W == 4)
      *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
    else
      *reinterpret_cast<uint32_t *>(dst) = pack_bf16(acc[0], acc[1]);
  }
  if (LSE != nullptr && lane == 0) LSE[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

template <int DV>
cudaError_t launch_merge(const float *O_part, const float *L_part, int n_splits, long long rows,
                         void *O, int out_f32, float *LSE, cudaStream_t stream) {
  const long long blocks = (rows + MERGE_ROWS_PER_BLOCK - 1) / MERGE_ROWS_PER_BLOCK;
  attn_merge_kernel<DV><<<static_cast<unsigned>(blocks), 32 * MERGE_ROWS_PER_BLOCK, 0, stream>>>(
      O_part, L_part, n_splits, rows, O, out_f32, LSE);
  return cudaGetLastError();
}

}  // namespace eta

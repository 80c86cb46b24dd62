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

// One thread per output element: a block of d_v threads per query row, so that every
// (range, element) load of the whole grid can be in flight at once (the work is a few
// loads per thread; it is bound by memory latency, not by bandwidth or arithmetic).
// O_part: [S][rows][DV] fp32; L_part: [S][rows] fp32; O: [rows][DV] (fp32 or bf16);
// LSE: [rows] or null.
template <int DV>
__global__ void __launch_bounds__(DV)
    attn_merge_kernel(const float *__restrict__ O_part, const float *__restrict__ L_part,
                      int n_splits, long long rows, void *O, int out_f32, float *LSE) {
  const long long row = blockIdx.x;
  const int col = threadIdx.x;
  grid_dep_wait();  // the attention kernel's partials
  if (col == 0) grid_dep_launch();

  // The ranges' loads are independent and issued in batches of 32, so for up to 32
  // ranges each pass is one memory round trip (the partials usually come from DRAM).
  constexpr int B = 32;
  float M = -INFINITY;
  for (int s0 = 0; s0 < n_splits; s0 += B) {
    float w[B];
#pragma unroll
    for (int k = 0; k < B; ++k) w[k] = __ldg(L_part + (s0 + k < n_splits ? s0 + k : s0) * rows + row);
#pragma unroll
    for (int k = 0; k < B; ++k) M = fmaxf(M, w[k]);  // the clamped repeats change nothing
  }

  float acc = 0.0f, wsum = 0.0f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n_splits; s0 += B) {
      float w[B], v[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int s = s0 + k < n_splits ? s0 + k : n_splits - 1;  // clamped: weight 0 below
        w[k] = __ldg(L_part + s * rows + row);
        v[k] = __ldg(O_part + (s * rows + row) * DV + col);
      }
      // In increasing range order, as the sums are defined.
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const float wk = s0 + k < n_splits ? expf(w[k] - M) : 0.0f;  // 0 for an empty range
        acc = fmaf(wk, v[k], acc);
        wsum += wk;
      }
    }
  }
  const float r = wsum > 0.0f ? acc * (1.0f / wsum) : 0.0f;
  if (out_f32) {
    static_cast<float *>(O)[row * DV + col] = r;
  } else {
    // Pairs of neighbouring columns are packed by the even thread of each pair.
    const float hi = __shfl_down_sync(0xFFFFFFFFu, r, 1);
    if ((col & 1) == 0)
      *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(O) + row * DV + col) = pack_bf16(r, hi);
  }
  if (LSE != nullptr && col == 0) LSE[row] = wsum > 0.0f ? M + logf(wsum) : -INFINITY;
}

template <int DV>
cudaError_t launch_merge(const float *O_part, const float *L_part, int n_splits, long long rows,
                         void *O, int out_f32, float *LSE, cudaStream_t stream) {
  if (rows > 0x7FFFFFFFll) return cudaErrorInvalidValue;  // one block per row
  const cudaError_t e = launch_pdl(attn_merge_kernel<DV>, dim3(static_cast<unsigned>(rows)), dim3(DV), 0, stream,
                                   O_part, L_part, n_splits, rows, O, out_f32, LSE);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace eta

// Exact attention forward pass, tile by tile, for sm_103a.
//
// The recurrence is the one in "Compilers and kernels", section "FlashAttention
// rewrites the algorithm around IO": for each query row, over key/value blocks B_t,
//   b_t = max_{j in B_t} S_ij, m_t = max(m_{t-1}, b_t), alpha_t = exp(m_{t-1} - m_t),
//   l_t = alpha_t l_{t-1} + sum exp(S_ij - m_t), o_t = alpha_t o_{t-1} + sum exp(S_ij - m_t) v_j,
// and finally O_i = o_T / l_T. Blocks are 128-key tiles; a key the mask forbids gets
// S_ij = -inf and contributes exp(-inf) = 0, which is the same as leaving it out of
// the partition. Exponentials are evaluated as 2^x on log2(e)-scaled scores.
//
// One CTA owns NQ query tiles of 128 rows of one head (NQ = 2 without a dense bias,
// so one tile's softmax overlaps the other tile's matrix products; NQ = 1 with a
// dense bias, whose time is the bias bytes). Warp roles:
//   softmax warpgroup q (warps 4q..4q+3): thread = query row = tensor-memory lane.
//     Reads its row of S from tensor memory, masks, takes the tile max, the new
//     running max and alpha, writes P as bf16 back over S, rescales its row of o by
//     alpha when some alpha in the warp differs from 1, and at the end writes O and LSE.
//   MMA warp: issues S_q = Q_q K_t^T (A and B from shared memory) and o_q += P_q V_t
//     (A = P from tensor memory, B = V from shared memory) with tcgen05.mma; fp32
//     accumulators stay in tensor memory.
//   load warp: TMA copies of Q once and K_t, V_t into rings of shared-memory slots
//     guarded by full/empty mbarrier pairs (AI Infra ch. 5, Fig. 5-5: producer
//     copies, consumer computes, one full and one empty barrier per slot).
//   bias load warp (dense bias only): TMA copies of 128 x 32 fp32 bias chunks.
// Causal tiles above the diagonal are never loaded or multiplied; tiles are visited
// from the diagonal down so each row meets an allowed key in its first tile.
//
// Every mbarrier wait is bounded in time. A wait that runs out records where it
// stopped in a device status word, sets a shared abort flag that ends every other
// wait of the CTA, and the CTA drains its copies and MMAs and frees tensor memory
// before it returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace eta {

enum { MODE_NONE = 0, MODE_CAUSAL = 1, MODE_DENSE = 2 };

constexpr int BM = 128;     // query rows per Q tile (= tensor-memory lanes)
constexpr int BN = 128;     // keys per K/V tile
constexpr int CCHUNK = 32;  // bias columns per dense-bias chunk (128 bytes of fp32)
constexpr int CCHUNK_BYTES = BM * CCHUNK * 4;
constexpr int SW_CHUNK = 64;                 // bf16 columns per 128-byte swizzle span
constexpr int SW_CHUNK_BYTES = 128 * 128;    // one 128-row x 128-byte box
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

struct KernelParams {
  int BH;
  int N;
  int num_tiles;      // ceil(N / 128): number of Q tiles and of K/V tiles per head
  int ctas_per_head;  // ceil(num_tiles / NQ)
  float scale_log2;   // scale * log2(e)
  int out_f32;        // O element type: 1 fp32, 0 bf16
  void *O;
  float *LSE;
  const float *C;           // dense bias, read directly when it cannot go through TMA
  unsigned int *status;     // watchdog word (device memory)
  unsigned long long timeout_ns;
};

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

template <int D, int DV, int MODE, bool C_TMA>
struct Cfg {
  static_assert(D == 64 || D == 128, "d must be 64 or 128");
  static_assert(DV == 64 || DV == 128, "d_v must be 64 or 128");
  static constexpr bool DENSE = MODE == MODE_DENSE;
  static constexpr bool C_RING = DENSE && C_TMA;
  static constexpr int NQ = DENSE ? 1 : 2;
  static constexpr int Q_TILE = BM * D * 2;
  static constexpr int K_TILE = BN * D * 2;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int BUDGET = 224 * 1024;
  static constexpr int KV_PAIRS = cmin(4, (BUDGET - NQ * Q_TILE) / (K_TILE + V_TILE));
  static constexpr int KS = DENSE ? 2 : cmin(4, KV_PAIRS + ((BUDGET - NQ * Q_TILE - KV_PAIRS * (K_TILE + V_TILE)) >= K_TILE ? 1 : 0));
  static constexpr int VS = DENSE ? 2 : KV_PAIRS;
  static constexpr int CS = C_RING ? cmin(8, (BUDGET - NQ * Q_TILE - KS * K_TILE - VS * V_TILE) / CCHUNK_BYTES) : 0;
  static_assert(KS >= 2 && VS >= 2, "need at least two K and two V slots");
  static_assert(!C_RING || CS >= 4, "need at least one bias tile in flight");

  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQ * Q_TILE;
  static constexpr int V_OFF = K_OFF + KS * K_TILE;
  static constexpr int C_OFF = V_OFF + VS * V_TILE;
  static constexpr int BAR_OFF = C_OFF + CS * CCHUNK_BYTES;
  // barrier indices
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + KS;
  static constexpr int B_VFULL = B_KEMPTY + KS;
  static constexpr int B_VEMPTY = B_VFULL + VS;
  static constexpr int B_CFULL = B_VEMPTY + VS;
  static constexpr int B_CEMPTY = B_CFULL + CS;
  static constexpr int B_SFULL = B_CEMPTY + CS;
  static constexpr int B_PFULL = B_SFULL + NQ;
  static constexpr int B_OFULL = B_PFULL + NQ;
  static constexpr int B_DRAIN = B_OFULL + NQ;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr int TMEMPTR_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int ABORT_OFF = TMEMPTR_OFF + 4;
  static constexpr int SMEM_USED = ABORT_OFF + 4;
  static constexpr int SMEM_TOTAL = SMEM_USED + 1024;  // room to align the base to 1024 B
  static_assert(SMEM_TOTAL <= 232448, "shared memory over the sm_103a per-CTA limit");

  static constexpr int MMA_WARP = 4 * NQ;
  static constexpr int LOAD_WARP = 4 * NQ + 1;
  static constexpr int CLOAD_WARP = 4 * NQ + 2;
  static constexpr int NUM_WARPS = 4 * NQ + 2 + (C_RING ? 1 : 0);
  static constexpr int THREADS = 32 * NUM_WARPS;
  // tensor memory: S_q at columns [q*128, q*128+128), o_q after all S tiles
  static constexpr int S_COL = 0;
  static constexpr int O_COL = NQ * BN;
  static constexpr int TMEM_COLS = pow2_at_least(NQ * (BN + DV));
  static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");

  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, true);
};

// Watchdog codes: bit 31 set, role in bits 24-27, barrier index in bits 8-23.
enum { ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_CLOAD = 4, ROLE_DRAIN = 5 };

struct Watchdog {
  volatile int *abort_flag;
  unsigned int *status;
  unsigned long long timeout_ns;

  __device__ void trip(int role, int bar) {
    *abort_flag = 1;
    atomicCAS(status, 0u, 0x80000000u | (static_cast<unsigned>(role) << 24) |
                              (static_cast<unsigned>(bar & 0xFFFF) << 8));
  }

  // Bounded wait of one thread; false on timeout or when another role aborted.
  __device__ bool wait1(uint32_t bar_addr, uint32_t parity, int role, int bar, bool drain) {
    if (mbar_try_wait(bar_addr, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
      if (mbar_try_wait(bar_addr, parity)) return true;
      if ((spin & 15u) == 0) {
        if (!drain && *abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) {
          trip(drain ? ROLE_DRAIN : role, bar);
          return false;
        }
      }
    }
  }

  // Whole-warp bounded wait: every lane observes the barrier; the result is uniform.
  __device__ bool wait(uint32_t bar_addr, uint32_t parity, int role, int bar) {
    const bool ok = wait1(bar_addr, parity, role, bar, false);
    return __all_sync(0xFFFFFFFFu, ok);
  }
  __device__ bool drain(uint32_t bar_addr, uint32_t parity, int bar) {
    const bool ok = wait1(bar_addr, parity, ROLE_DRAIN, bar, true);
    return __all_sync(0xFFFFFFFFu, ok);
  }
};

// Per-CTA schedule: which query tiles it owns and which K/V tiles each one visits.
// Iteration `it` visits K/V tile j = hi_max - it; query tile q takes part in
// iterations [first_it[q], n_it), i.e. K/V tiles hi_q down to 0.
template <int NQ, int MODE>
struct Schedule {
  int bh, cta_q, n_exist, hi_max, n_it;
  int first_it[NQ];

  __device__ Schedule(const KernelParams &p) {
    bh = blockIdx.x / p.ctas_per_head;
    // Within a head, the CTA with the most causal work starts first.
    cta_q = p.ctas_per_head - 1 - static_cast<int>(blockIdx.x % p.ctas_per_head);
    n_exist = cmin(NQ, p.num_tiles - cta_q * NQ);
    hi_max = (MODE == MODE_CAUSAL) ? cta_q * NQ + n_exist - 1 : p.num_tiles - 1;
    n_it = hi_max + 1;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int hi_q = (MODE == MODE_CAUSAL) ? cta_q * NQ + q : p.num_tiles - 1;
      first_it[q] = (q < n_exist) ? hi_max - hi_q : n_it;  // n_it: never active
    }
  }
  __device__ int q_tile(int q) const { return cta_q * NQ + q; }
};

template <int D, int DV, int MODE, bool C_TMA>
__global__ void __launch_bounds__(Cfg<D, DV, MODE, C_TMA>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmC,
                    const KernelParams p) {
  using CF = Cfg<D, DV, MODE, C_TMA>;
  constexpr int NQ = CF::NQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + CF::BAR_OFF;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + CF::TMEMPTR_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::ABORT_OFF);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const Schedule<NQ, MODE> sch(p);
  Watchdog wd{abort_flag, p.status, p.timeout_ns};

  // ------------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    mbar_init(BAR(CF::B_QFULL), 1);
    for (int s = 0; s < CF::KS; ++s) {
      mbar_init(BAR(CF::B_KFULL + s), 1);
      mbar_init(BAR(CF::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < CF::VS; ++s) {
      mbar_init(BAR(CF::B_VFULL + s), 1);
      mbar_init(BAR(CF::B_VEMPTY + s), 1);
    }
    for (int s = 0; s < CF::CS; ++s) {
      mbar_init(BAR(CF::B_CFULL + s), 1);
      mbar_init(BAR(CF::B_CEMPTY + s), 4);  // one arrival per softmax warp
    }
    for (int q = 0; q < NQ; ++q) {
      mbar_init(BAR(CF::B_SFULL + q), 1);
      mbar_init(BAR(CF::B_PFULL + q), 4);  // one arrival per softmax warp
      mbar_init(BAR(CF::B_OFULL + q), 1);
    }
    mbar_init(BAR(CF::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == CF::MMA_WARP) {
    tmem_alloc(smem_u32(tmem_ptr), CF::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp < 4 * NQ) {
    // ================================================================ softmax
    const int q = warp / 4;
    const int row = threadIdx.x % BM;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const uint32_t t_s = tmem + lane_off + CF::S_COL + q * BN;
    const uint32_t t_o = tmem + lane_off + CF::O_COL + q * DV;
    const int qt = sch.q_tile(q);
    const int q_row = qt * BM + row;
    const bool exists = q < sch.n_exist;
    const float sl2 = p.scale_log2;
    float m2 = -INFINITY;  // running max m_t, in log2(e)-scaled units
    float l = 0.0f;        // running sum l_t
    uint32_t s_phase = 0;
    bool ok = true;
    int cpos = 0;  // dense-bias ring position
    if (exists) {
      for (int it = sch.first_it[q]; it < sch.n_it; ++it) {
        const int j = sch.hi_max - it;
        ok = wd.wait(BAR(CF::B_SFULL + q), s_phase, ROLE_SOFTMAX, CF::B_SFULL + q);
        s_phase ^= 1;
        if (!ok) break;
        tc_fence_after();

        // Row of S (raw Q K^T) for this thread's query, 128 keys.
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(t_s + 0, r0);
        tmem_ld32(t_s + 32, r1);
        tmem_ld32(t_s + 64, r2);
        tmem_ld32(t_s + 96, r3);
        tmem_wait_ld(r0);
        tmem_wait_ld(r1);
        tmem_wait_ld(r2);
        tmem_wait_ld(r3);
        float x[BN];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]);
          x[32 + c] = __uint_as_float(r1[c]);
          x[64 + c] = __uint_as_float(r2[c]);
          x[96 + c] = __uint_as_float(r3[c]);
        }

        if constexpr (CF::DENSE) {
          // x = (scale * S + C) * log2(e): the bias joins after the scaling, unscaled.
          if constexpr (C_TMA) {
#pragma unroll
            for (int cc = 0; cc < BN / CCHUNK; ++cc) {
              const int slot = cpos % CF::CS;
              const uint32_t par = (cpos / CF::CS) & 1;
              ok = wd.wait(BAR(CF::B_CFULL + slot), par, ROLE_SOFTMAX, CF::B_CFULL + slot);
              if (!ok) break;
              const uint8_t *chunk = smem + CF::C_OFF + slot * CCHUNK_BYTES + row * 128;
#pragma unroll
              for (int u = 0; u < CCHUNK / 4; ++u) {
                const float4 cv =
                    *reinterpret_cast<const float4 *>(chunk + ((u ^ (row & 7)) << 4));
                const int c = cc * CCHUNK + 4 * u;
                x[c + 0] = fmaf(x[c + 0], sl2, cv.x * LOG2E);
                x[c + 1] = fmaf(x[c + 1], sl2, cv.y * LOG2E);
                x[c + 2] = fmaf(x[c + 2], sl2, cv.z * LOG2E);
                x[c + 3] = fmaf(x[c + 3], sl2, cv.w * LOG2E);
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(BAR(CF::B_CEMPTY + slot));
              ++cpos;
            }
            if (!ok) break;
          } else {
            const bool row_ok = q_row < p.N;
            const float *crow = p.C + (static_cast<size_t>(sch.bh) * p.N + (row_ok ? q_row : 0)) *
                                          static_cast<size_t>(p.N);
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const int kv = j * BN + c;
              const float cv = (row_ok && kv < p.N) ? __ldg(crow + kv) : 0.0f;
              x[c] = fmaf(x[c], sl2, cv * LOG2E);
            }
          }
        }

        // Forbidden keys: above the causal diagonal, and past the end of the sequence.
        const bool diag = (MODE == MODE_CAUSAL) && (j == qt);
        const bool tail = (j == p.num_tiles - 1) && (p.N % BN != 0);
        if (diag || tail) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int kv = j * BN + c;
            if ((diag && kv > q_row) || kv >= p.N) x[c] = -INFINITY;
          }
        }

        // b_t and m_t = max(m_{t-1}, b_t)
        float b = x[0];
#pragma unroll
        for (int c = 1; c + 1 < BN; c += 2) b = fmax3(b, x[c], x[c + 1]);
        b = fmaxf(b, x[BN - 1]);
        const float m_new = CF::DENSE ? fmaxf(m2, b) : fmaxf(m2, b * sl2);
        // No allowed key seen yet: every p is 0 and alpha is irrelevant; use 0 as reference.
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = ex2_approx(m2 - m_use);  // alpha_t = exp(m_{t-1} - m_t)

        // p_ij = exp(S_ij - m_t) as bf16 into tensor memory over S; l_t accumulates fp32 p.
        uint32_t pk0[32], pk1[32];
        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k0 = 2 * c, k1 = 2 * c + 1;
          const float p0 = CF::DENSE ? ex2_approx(x[k0] - m_use) : ex2_approx(fmaf(x[k0], sl2, -m_use));
          const float p1 = CF::DENSE ? ex2_approx(x[k1] - m_use) : ex2_approx(fmaf(x[k1], sl2, -m_use));
          rs0 += p0;
          rs1 += p1;
          pk0[c] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k0 = 64 + 2 * c, k1 = 64 + 2 * c + 1;
          const float p0 = CF::DENSE ? ex2_approx(x[k0] - m_use) : ex2_approx(fmaf(x[k0], sl2, -m_use));
          const float p1 = CF::DENSE ? ex2_approx(x[k1] - m_use) : ex2_approx(fmaf(x[k1], sl2, -m_use));
          rs0 += p0;
          rs1 += p1;
          pk1[c] = pack_bf16(p0, p1);
        }
        l = alpha * l + (rs0 + rs1);
        tmem_st32(t_s + 0, pk0);
        tmem_st32(t_s + 32, pk1);
        tmem_wait_st();

        // o_t = alpha_t o_{t-1}: the previous P V has completed (the S tile just read was
        // committed after it). Skipped when alpha is 1 for every row of the warp.
        if (it > sch.first_it[q] && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * cc, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(t_o + 32 * cc, o);
          }
          tmem_wait_st();
        }
        m2 = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(CF::B_PFULL + q));
      }

      // ------------------------------------------------ epilogue: O = o_T / l_T, LSE
      if (ok) ok = wd.wait(BAR(CF::B_OFULL + q), 0, ROLE_SOFTMAX, CF::B_OFULL + q);
      if (ok) {
        tc_fence_after();
        const bool row_ok = q_row < p.N;
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;  // no allowed key: O = 0
        const size_t orow = (static_cast<size_t>(sch.bh) * p.N + (row_ok ? q_row : 0)) * DV;
#pragma unroll
        for (int cc = 0; cc < DV / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(t_o + 32 * cc, o);
          tmem_wait_ld(o);
          if (row_ok) {
            if (p.out_f32) {
              float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.O) + orow + 32 * cc);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv_l,
                                     __uint_as_float(o[4 * v + 1]) * inv_l,
                                     __uint_as_float(o[4 * v + 2]) * inv_l,
                                     __uint_as_float(o[4 * v + 3]) * inv_l);
            } else {
              uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.O) + orow + 32 * cc);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
                w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
                w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
                w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
                dst[v] = w;
              }
            }
          }
        }
        if (row_ok && p.LSE != nullptr) {
          // LSE_i = m_i + ln l_i, from the log2-scaled running max.
          p.LSE[static_cast<size_t>(sch.bh) * p.N + q_row] =
              (l > 0.0f) ? (m2 + lg2_approx(l)) * LN2 : -INFINITY;
        }
      }
    }
  } else if (warp == CF::MMA_WARP) {
    // ================================================================ MMA issue
    uint32_t p_phase[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) p_phase[q] = 0;
    bool ok = wd.wait(BAR(CF::B_QFULL), 0, ROLE_MMA, CF::B_QFULL);
    tc_fence_after();

    auto issue_s = [&](int q, int kslot) {
      const uint32_t a0 = sbase + CF::Q_OFF + q * CF::Q_TILE;
      const uint32_t b0 = sbase + CF::K_OFF + kslot * CF::K_TILE;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (ks / 4) * SW_CHUNK_BYTES + (ks % 4) * 32;
        mma_ss(tmem + CF::S_COL + q * BN, smem_desc(a0 + off, 16, 1024),
               smem_desc(b0 + off, 16, 1024), CF::IDESC_S, ks > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int q, int vslot, bool accumulate) {
      const uint32_t b0 = sbase + CF::V_OFF + vslot * CF::V_TILE;
#pragma unroll
      for (int ks = 0; ks < BN / 16; ++ks) {
        mma_ts(tmem + CF::O_COL + q * DV, tmem + CF::S_COL + q * BN + ks * 8,
               smem_desc(b0 + ks * 16 * 128, SW_CHUNK_BYTES, 1024), CF::IDESC_PV,
               (ks > 0 || accumulate) ? 1u : 0u);
      }
    };

    for (int it = 0; ok && it < sch.n_it; ++it) {
      const int kslot = it % CF::KS;
      const int vprev = (it + CF::VS - 1) % CF::VS;
      ok = wd.wait(BAR(CF::B_KFULL + kslot), (it / CF::KS) & 1, ROLE_MMA, CF::B_KFULL + kslot);
      if (ok && it > 0)
        ok = wd.wait(BAR(CF::B_VFULL + vprev), ((it - 1) / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vprev);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (it < sch.first_it[q]) continue;
        if (it > sch.first_it[q]) {
          // o_q += P_q V_{it-1}, once the softmax has written P and rescaled o.
          ok = wd.wait(BAR(CF::B_PFULL + q), p_phase[q], ROLE_MMA, CF::B_PFULL + q);
          p_phase[q] ^= 1;
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) issue_pv(q, vprev, it - 1 > sch.first_it[q]);
          __syncwarp();
        }
        if (lane == 0) {
          issue_s(q, kslot);  // S_q = Q_q K_it^T
          mma_commit(BAR(CF::B_SFULL + q));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(BAR(CF::B_KEMPTY + kslot));
        if (it > 0) mma_commit(BAR(CF::B_VEMPTY + vprev));
      }
      __syncwarp();
    }
    if (ok) {
      const int last = sch.n_it - 1;
      const int vslot = last % CF::VS;
      ok = wd.wait(BAR(CF::B_VFULL + vslot), (last / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vslot);
      if (ok) tc_fence_after();
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (!ok || sch.first_it[q] >= sch.n_it) continue;
        ok = wd.wait(BAR(CF::B_PFULL + q), p_phase[q], ROLE_MMA, CF::B_PFULL + q);
        p_phase[q] ^= 1;
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          issue_pv(q, vslot, last > sch.first_it[q]);
          mma_commit(BAR(CF::B_OFULL + q));
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(BAR(CF::B_VEMPTY + vslot));
      __syncwarp();
    }
    // Nothing may still be in flight on the tensor cores when tensor memory is freed.
    if (lane == 0) mma_commit(BAR(CF::B_DRAIN));
    __syncwarp();
    wd.drain(BAR(CF::B_DRAIN), 0, CF::B_DRAIN);
  } else if (warp == CF::LOAD_WARP) {
    // ================================================================ TMA: Q, K, V
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(BAR(CF::B_QFULL), sch.n_exist * CF::Q_TILE);
      for (int q = 0; q < sch.n_exist; ++q)
        for (int kc = 0; kc < D / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::Q_OFF + q * CF::Q_TILE + kc * SW_CHUNK_BYTES, &tmQ, kc * SW_CHUNK,
                      sch.q_tile(q) * BM, sch.bh, BAR(CF::B_QFULL));
    }
    __syncwarp();
    bool ok = true;
    int k_issued = 0, v_issued = 0;
    for (int it = 0; it < sch.n_it; ++it) {
      const int j = sch.hi_max - it;
      const int ks = it % CF::KS;
      ok = wd.wait(BAR(CF::B_KEMPTY + ks), ((it / CF::KS) & 1) ^ 1, ROLE_LOAD, CF::B_KEMPTY + ks);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(CF::B_KFULL + ks), CF::K_TILE);
        for (int kc = 0; kc < D / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::K_OFF + ks * CF::K_TILE + kc * SW_CHUNK_BYTES, &tmK, kc * SW_CHUNK,
                      j * BN, sch.bh, BAR(CF::B_KFULL + ks));
      }
      __syncwarp();
      ++k_issued;
      const int vs = it % CF::VS;
      ok = wd.wait(BAR(CF::B_VEMPTY + vs), ((it / CF::VS) & 1) ^ 1, ROLE_LOAD, CF::B_VEMPTY + vs);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(CF::B_VFULL + vs), CF::V_TILE);
        for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::V_OFF + vs * CF::V_TILE + kc * SW_CHUNK_BYTES, &tmV, kc * SW_CHUNK,
                      j * BN, sch.bh, BAR(CF::B_VFULL + vs));
      }
      __syncwarp();
      ++v_issued;
    }
    // Wait for the last copy into each slot to land before the CTA may exit.
    wd.drain(BAR(CF::B_QFULL), 0, CF::B_QFULL);
    for (int s = 0; s < CF::KS && s < k_issued; ++s) {
      const int last = s + ((k_issued - 1 - s) / CF::KS) * CF::KS;
      wd.drain(BAR(CF::B_KFULL + s), (last / CF::KS) & 1, CF::B_KFULL + s);
    }
    for (int s = 0; s < CF::VS && s < v_issued; ++s) {
      const int last = s + ((v_issued - 1 - s) / CF::VS) * CF::VS;
      wd.drain(BAR(CF::B_VFULL + s), (last / CF::VS) & 1, CF::B_VFULL + s);
    }
  } else if (CF::C_RING && warp == CF::CLOAD_WARP) {
    // ================================================================ TMA: dense bias
    if (lane == 0) tma_prefetch_desc(&tmC);
    int issued = 0;
    for (int it = 0; it < sch.n_it; ++it) {
      const int j = sch.hi_max - it;
      bool ok = true;
      for (int cc = 0; cc < BN / CCHUNK; ++cc) {
        const int pos = issued;
        const int slot = pos % CF::CS;
        ok = wd.wait(BAR(CF::B_CEMPTY + slot), ((pos / CF::CS) & 1) ^ 1, ROLE_CLOAD,
                     CF::B_CEMPTY + slot);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(BAR(CF::B_CFULL + slot), CCHUNK_BYTES);
          tma_load_3d(sbase + CF::C_OFF + slot * CCHUNK_BYTES, &tmC, j * BN + cc * CCHUNK,
                      sch.q_tile(0) * BM, sch.bh, BAR(CF::B_CFULL + slot));
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) break;
    }
    for (int s = 0; s < CF::CS && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / CF::CS) * CF::CS;
      wd.drain(BAR(CF::B_CFULL + s), (last / CF::CS) & 1, CF::B_CFULL + s);
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == CF::MMA_WARP) tmem_dealloc(tmem, CF::TMEM_COLS);
}

// ---------------------------------------------------------------------- host side
struct LaunchArgs {
  CUtensorMap tmQ, tmK, tmV, tmC;
  KernelParams p;
  cudaStream_t stream;
};

// Number of query tiles one CTA owns for a given mode (the host sizes the grid with it).
constexpr int q_tiles_per_cta(int mode) { return mode == MODE_DENSE ? 1 : 2; }

template <int D, int DV, int MODE, bool C_TMA>
cudaError_t launch_attn(const LaunchArgs &a) {
  using CF = Cfg<D, DV, MODE, C_TMA>;
  auto kern = attn_fwd_kernel<D, DV, MODE, C_TMA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.ctas_per_head);
  kern<<<grid, CF::THREADS, CF::SMEM_TOTAL, a.stream>>>(a.tmQ, a.tmK, a.tmV, a.tmC, a.p);
  return cudaGetLastError();
}

}  // namespace eta

// Exact attention forward pass on CTA pairs, for sm_103a: no bias term, a dense bias read
// through TMA, or (d = 64) a per-key bias, with or without the causal mask, d = 64 or 128,
// d_v = 128.
//
// The recurrence is the one in "Compilers and kernels", section "FlashAttention rewrites
// the algorithm around IO" (b_t, m_t, alpha_t, l_t, o_t, O_i = o_T / l_T), evaluated over
// 128-key tiles as in attn_fwd_kernel.cuh. What differs is how the work is laid on the
// chip.
//
// A cluster of two CTAs on two SMs owns 256 query rows of one head at a time (a unit), 128
// in each CTA. The tensor-core products are the pair's (.cta_group::2, M = 256): S = Q K^T
// with each CTA's Q rows in its own shared memory and the K tile split between the two (64
// keys each), and o += P V with each CTA's P in its own tensor memory and the V tile split
// by columns (64 value columns each). So each SM stages and streams half of every K and V
// tile: half the shared-memory operand traffic and half the L2 traffic per SM of one CTA
// doing all 128 keys, at the same tensor rate.
//
// One query tile per CTA leaves room in tensor memory (512 columns) for two S buffers, two
// P buffers (bf16) and o. An S buffer is released as soon as the softmax has loaded it, so
// S(t+1) and S(t+2) are computed while the softmax of S(t) runs, and the chain softmax -> P
// -> P V -> next S no longer serialises the tensor cores (the products of one query tile
// depend on its softmax only through P).
//
// The grid is persistent: one cluster per pair of SMs, each taking units in a fixed order
// (longest first, alternating direction every round of clusters, so the long units spread
// evenly). Rings, buffers and barrier phases run on across units: the next unit's Q is
// loaded into the second Q buffer, and its first S products and softmax tiles run while the
// current unit's epilogue runs; its first P V waits only for the epilogue to have read o.
//
// With a dense bias each CTA streams its own 128 rows of C: four 128 x 32 fp32 chunks per
// key tile through two TMA rings, one per softmax warpgroup (each consumed in order by its
// warpgroup alone), filled by two lanes of the V copy warp; the rings take the room of the
// deeper K/V rings and of the second Q buffer.
//
// A per-key bias c_j is not added by the softmax (that add and the row maximum it then
// needs would lengthen the hand-off between the warpgroups) but folded into the S product:
// each K slot holds a second 128-byte atom whose logical columns 0 and 1 are c_j / scale as
// bf16 high and low parts for this CTA's 64 keys, written by the Q/K copy warp, and a
// constant tile of ones is the query side of one more 16-wide step of the contraction.
//
// Warp roles (16 warps in each CTA):
//   softmax, warps 0-7: two warpgroups that take the key tiles in turn (tiles are numbered
//     across units; even tiles in the first warpgroup, odd ones in the second); thread =
//     query row = tensor-memory lane, a whole row of 128 keys per tile. The two warpgroups
//     run out of phase, so one's exponentials overlap the other's loads and maxima. The
//     recurrence couples consecutive tiles only through the exponent reference: each warp
//     passes the reference it settled on to the other warpgroup's warp of the same rows (a
//     word per row in shared memory and an mbarrier), and keeps its own share of l; the
//     shares are brought to the final reference and added by the epilogue warps. The
//     warpgroup whose tile moves the reference rescales o (all 128 columns of its rows) once
//     the previous P V has completed.
//   epilogue, warps 12-15: per unit, O = o / l and LSE; o is released to the next unit's
//     first P V as soon as it is in registers (all 128 columns packed to bf16 first for bf16
//     output), while the softmax warps are already on that unit; each warp stages its 32 rows
//     in the unit's idle Q buffer one 32 x 128-byte box at a time and stores them with TMA.
//   MMA, warps 8 (S products) and 11 (P V products) of the even CTA: issue the pair's
//     products; each commit signals the mbarrier at the same offset in both CTAs
//     (multicast). S(t) waits for the softmax to have loaded S(t-2) from its buffer.
//   Q/K load (warp 9) and V load (warp 10, lane 0; lanes 1-2 the bias rings) of both CTAs:
//     TMA copies of this CTA's halves; completion is signalled on the even CTA's full
//     barriers, whose expected byte count covers both halves, so an MMA warp waits once per
//     tile. With a per-key bias the whole Q/K warp runs its loop and writes each K slot's
//     bias columns; each CTA's writers add one arrival to the even CTA's K-full barrier.
// Every wait is an mbarrier wait bounded in time, as in attn_fwd_kernel.cuh (no named
// barriers: a warp that gave up cannot leave another waiting forever).
#pragma once

#include "attn_fwd_kernel.cuh"

namespace eta {

template <int D, int DV, bool CAUSAL, int BIAS>
struct PairCfg {
  static_assert(D == 64 || D == 128, "d must be 64 or 128");
  static_assert(DV == 128, "the pair kernel splits 128 value columns in two 128-byte halves");
  static_assert(BIAS == BIAS_NONE || BIAS == BIAS_DENSE_TMA || BIAS == BIAS_KEY, "bias kind");
  static constexpr bool DENSE = BIAS == BIAS_DENSE_TMA;  // [Nq][Nk] bias rows through a TMA ring
  // A per-key bias c_j rides in the S product: one more 16-wide step of the contraction
  // with ones on the query side and c_j / scale on the key side (bf16 high and low parts),
  // so S holds q k + c / scale and the softmax takes the path without a bias.
  static constexpr bool KEYB = BIAS == BIAS_KEY;
  static_assert(!KEYB || D == 64, "the key-bias columns take a second 128-byte atom of each K slot (d = 64)");
  static constexpr bool BIASED = DENSE;  // the softmax adds a bias to scale S itself
  static constexpr int Q_TILE = BM * D * 2;       // this CTA's 128 query rows
  static constexpr int STAGE = 4 * 32 * 128;      // epilogue stage: one 32-row x 128-byte box per epilogue warp
  static constexpr int Q_BUF = Q_TILE > STAGE ? Q_TILE : STAGE;
  static constexpr int KH_ROWS = BN / 2;          // keys of a K tile held by one CTA
  static constexpr int KH_BOX = KH_ROWS * 128;    // one 64-row x 128-byte box
  static constexpr int KH_TILE = KH_ROWS * D * 2;  // bytes of one CTA's K copy
  // K slot: the K columns in D / 64 atoms of 64 rows x 128 bytes, then, with a per-key bias,
  // one atom whose logical columns 0 and 1 hold the bias parts (8-15 zero, 16-63 unused).
  static constexpr int KH_SLOT = KH_TILE + (KEYB ? KH_BOX : 0);
  static constexpr int VH_COLS = DV / 2;          // value columns held by one CTA
  static constexpr int VH_TILE = BN * VH_COLS * 2;
  static constexpr int NS = 2;                    // S buffers (and P buffers) in tensor memory
  // The dense bias stream takes the room of the deeper K/V rings and of the second Q buffer
  // (a unit's Q copy then waits for the previous unit's epilogue, which stages through it).
  static constexpr int KS = DENSE ? 2 : 4;
  static constexpr int VS = DENSE ? 3 : 4;
  static constexpr int NQB = DENSE ? 1 : 2;       // Q buffers: unit k uses buffer k % NQB
  static_assert(VS >= 3, "the softmax tells P(t) V apart by the phase of its V slot");
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQB * Q_BUF;
  static constexpr int V_OFF = K_OFF + KS * KH_SLOT;
  static constexpr int RX_OFF = V_OFF + VS * VH_TILE;  // references passed on, 2 x 128 fp32
  static constexpr int LX_OFF = RX_OFF + 2 * BM * 4;    // per unit % 2: [m, l, l'][2 warpgroups][128 rows]
  static constexpr int C_OFF = (LX_OFF + 2 * 3 * 2 * BM * 4 + 1023) / 1024 * 1024;  // dense bias rings (128-byte swizzle)
  static constexpr int BAR_RESERVE = 1024;               // barriers, tensor-memory address, abort flag
  // Two dense-bias rings of RS chunks, one per softmax warpgroup, each consumed in order by
  // its warpgroup only (a ring shared by both could let one warpgroup wait on a slot whose
  // previous fill has not landed yet, and a parity wait cannot tell those phases apart).
  static constexpr int RS = DENSE ? cmin(4, (232448 - 1024 - BAR_RESERVE - C_OFF) / (2 * CCHUNK_BYTES)) : 0;
  static constexpr int CS = 2 * RS;
  static_assert(!DENSE || RS >= 2, "need two bias chunks in flight per warpgroup");
  // With a per-key bias: the query side of the bias step, 128 rows whose logical columns 0
  // and 1 are 1 (8-15 zero), in the 128-byte swizzle of the other operands.
  static constexpr int ONES_OFF = C_OFF;
  static constexpr int ONES_BYTES = KEYB ? BM * 128 : 0;
  static constexpr int BAR_OFF = C_OFF + CS * CCHUNK_BYTES + ONES_BYTES;
  static constexpr int B_QFULL = 0;               // 2: Q of the unit in buffer 0 / 1 landed (both CTAs)
  static constexpr int B_QEMPTY = B_QFULL + 2;    // 2: buffer read by its unit's last S and used by its epilogue (5)
  static constexpr int B_KFULL = B_QEMPTY + 2;    // KS: K halves landed (and, with a per-key bias, both CTAs' bias columns)
  static constexpr int B_KEMPTY = B_KFULL + KS;
  static constexpr int B_VFULL = B_KEMPTY + KS;
  static constexpr int B_VEMPTY = B_VFULL + VS;   // P(t) V done (V slot free, P buffer free, o holds P(t) V)
  static constexpr int B_SFULL = B_VEMPTY + VS;   // S(t) computed (both CTAs)
  static constexpr int B_SEMPTY = B_SFULL + NS;   // S(t) loaded by the 4 softmax warps of each CTA (even CTA)
  static constexpr int B_PFULL = B_SEMPTY + NS;   // P(t) written by the 4 softmax warps of each CTA (even CTA)
  static constexpr int B_OFULL = B_PFULL + NS;    // a unit's last P V done
  static constexpr int B_OEMPTY = B_OFULL + 1;    // o read by the unit's epilogue, 4 warps x 2 CTAs (even CTA)
  static constexpr int B_DRAIN = B_OEMPTY + 1;    // products of the S issuer drained
  static constexpr int B_DRAIN2 = B_DRAIN + 1;    // products of the P V issuer drained
  static constexpr int B_HREF = B_DRAIN2 + 1;     // 8: reference passed on by warpgroup g, warp q (4 g + q)
  static constexpr int B_LDONE = B_HREF + 8;      // 2: a unit's (m, l, l') per row written by the 8 softmax warps
  static constexpr int B_LEMPTY = B_LDONE + 2;    // 2: read by the 4 epilogue warps
  static constexpr int B_CFULL = B_LEMPTY + 2;    // CS: a 128 x 32 bias chunk landed
  static constexpr int B_CEMPTY = B_CFULL + CS;   // CS: read by the tile's 4 softmax warps
  static constexpr int NUM_BARS = B_CEMPTY + CS;
  static_assert(NUM_BARS * 8 + 8 <= BAR_RESERVE, "barrier region");
  static constexpr int TMEMPTR_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int ABORT_OFF = TMEMPTR_OFF + 4;
  static constexpr int SMEM_USED = ABORT_OFF + 4;
  // At least 120 KB so one CTA holds an SM (it allocates all of the SM's tensor memory).
  static constexpr int SMEM_TOTAL = SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
  static_assert(SMEM_TOTAL <= 232448, "shared memory over the sm_103a per-CTA limit");

  static constexpr int MMA_WARP = 8;    // issues the S products
  static constexpr int LOAD_WARP = 9;   // Q and K
  static constexpr int VLOAD_WARP = 10; // V
  static constexpr int PV_WARP = 11;    // issues the P V products
  static constexpr int EPI_WARP0 = 12;  // warps 12-15: epilogue
  static constexpr int NUM_WARPS = 16;
  static constexpr int THREADS = 32 * NUM_WARPS;
  static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;
  static constexpr int REGS_SOFTMAX = 176;
  static constexpr int REGS_CTRL = 80;
  static constexpr int REGS_EPI = 80;
  static constexpr int REGS_NEEDED = 128 * (2 * REGS_SOFTMAX + REGS_CTRL + REGS_EPI);
  static_assert(REGS_NEEDED <= THREADS * LAUNCH_REGS,
                "register split exceeds the registers the block is launched with");
  // Tensor memory: S(t) in buffer t % 2, P(t) (bf16 pairs, 64 columns) in its own buffer
  // t % 2, then o. An S buffer is free once the softmax has loaded it, a P buffer once the
  // P V product that read it has completed.
  static constexpr int P_COL = NS * BN;
  static constexpr int O_COL = P_COL + NS * (BN / 2);
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + DV <= TMEM_COLS, "tensor memory holds 512 columns");

  static constexpr uint32_t IDESC_S = idesc_bf16_f32(2 * BM, BN, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(2 * BM, DV, true);
};

// One unit: query rows [256 pt, 256 pt + 256) of head bh, this CTA's 128 of them in query
// tile qt; K/V tiles hi_max down to 0 (the pair's last row decides hi_max, so the even
// CTA's rows may meet a last tile that is wholly above their causal limit: its scores are
// all masked and its P is 0).
template <bool CAUSAL>
struct PairSchedule {
  int bh, pt, qt, hi_max, n_it;
  __device__ PairSchedule(const KernelParams &p, unsigned unit, unsigned rank) {
    int r;
    unit_of_block(unit, p.BH, p.ctas_per_head, p.head_group, &bh, &r);
    pt = p.ctas_per_head - 1 - r;  // longest first
    qt = 2 * pt + static_cast<int>(rank);
    const int top = p.nkv_tiles - 1;
    if (CAUSAL) {
      const int last_row = cmin(2 * pt * BM + 2 * BM - 1, p.Nq - 1);
      hi_max = cmin(floor_div(last_row + p.causal_off, BN), top);
    } else {
      hi_max = top;
    }
    n_it = hi_max >= 0 ? hi_max + 1 : 0;
  }
};

// The k-th unit of cluster c among C: the units in grid order (longest first), taken a round
// of C at a time, each round in the opposite direction to the one before. Returns a value
// >= the number of units when cluster c has no k-th unit.
__device__ __forceinline__ unsigned pair_unit(int k, unsigned c, unsigned C) {
  return static_cast<unsigned>(k) * C + ((k & 1) ? (C - 1 - c) : c);
}

// An assignment of units to clusters computed on the host: cluster c takes the units
// unit[start[c]] .. unit[start[c + 1] - 1], in that order. Built by longest processing time
// first over the grid order (each unit, in order, to the cluster with the least work so far,
// a unit's work counted as its key tiles plus two for its start and end): the grid order
// keeps the heads that share K/V in L2 close in time, and the alternating rounds of
// pair_unit leave the busiest cluster up to 6 % above the mean where a group of heads ends
// and the next one starts again with long units. It is used only where units average at
// least 16 key tiles: on short units the start and end of each unit, which the count above
// models only roughly, weigh more, and the alternating rounds measured faster there (N =
// 2048 causal: 68.3 against 70.1 us; N = 8192 causal: 0.708 against 0.697 ms). With n = 0
// the units go by pair_unit.
struct PairPlan {
  static constexpr int MAX_CLUSTERS = 128;
  static constexpr int MAX_UNITS = 12288;
  int n;
  uint16_t start[MAX_CLUSTERS + 1];
  uint16_t unit[MAX_UNITS];
};

__device__ __forceinline__ unsigned plan_unit(const PairPlan &plan, int k, unsigned c, unsigned C,
                                              unsigned n_units) {
  if (plan.n == 0) return pair_unit(k, c, C);
  const int i = plan.start[c] + k;
  return i < plan.start[c + 1] ? plan.unit[i] : n_units;
}

// Waits (bounded) about 20 us: after an abort, copies already issued by this CTA that
// signal the other CTA's barriers cannot be observed here; give them time to land.
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < 20000ull) {
  }
}

template <int D, int DV, bool CAUSAL, int BIAS>
__global__ void __launch_bounds__(PairCfg<D, DV, CAUSAL, BIAS>::THREADS, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmC,
                         const __grid_constant__ CUtensorMap tmO, const __grid_constant__ KernelParams p,
                         const __grid_constant__ PairPlan plan) {
  using CF = PairCfg<D, DV, CAUSAL, BIAS>;
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
  const uint32_t rank = pair::cluster_rank();
  const bool leader = rank == 0;
  // The even CTA's copy of a barrier (the one the MMA warps wait on).
  auto LBAR = [&](int i) -> uint32_t { return pair::map_shared(BAR(i), 0); };
  const unsigned cl = blockIdx.x >> 1, n_cl = gridDim.x >> 1;
  const unsigned n_units = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.ctas_per_head);
  Watchdog wd{sbase + CF::ABORT_OFF, p};
#ifdef ETA_PHASE_TRACE
  int trace_n = 0;
#endif

  // ------------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      if (q >= CF::NQB) break;
      mbar_init(BAR(CF::B_QFULL + q), 1);
      mbar_init(BAR(CF::B_QEMPTY + q), 1 + 4);  // the last S's commit and this CTA's 4 epilogue warps
    }
    for (int s = 0; s < CF::KS; ++s) {
      mbar_init(BAR(CF::B_KFULL + s), CF::KEYB ? 3 : 1);  // + each CTA's bias-column writer
      mbar_init(BAR(CF::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < CF::VS; ++s) {
      mbar_init(BAR(CF::B_VFULL + s), 1);
      mbar_init(BAR(CF::B_VEMPTY + s), 1);
    }
    for (int b = 0; b < CF::NS; ++b) {
      mbar_init(BAR(CF::B_SFULL + b), 1);
      mbar_init(BAR(CF::B_SEMPTY + b), 8);  // one arrival per softmax warp of the tile, both CTAs
      mbar_init(BAR(CF::B_PFULL + b), 8);
    }
    mbar_init(BAR(CF::B_OFULL), 1);
    mbar_init(BAR(CF::B_OEMPTY), 8);  // every epilogue warp of both CTAs
    mbar_init(BAR(CF::B_DRAIN), 1);
    mbar_init(BAR(CF::B_DRAIN2), 1);
    for (int h = 0; h < 8; ++h) mbar_init(BAR(CF::B_HREF + h), 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(BAR(CF::B_LDONE + q), 8);
      mbar_init(BAR(CF::B_LEMPTY + q), 4);
    }
    for (int s = 0; s < CF::CS; ++s) {
      mbar_init(BAR(CF::B_CFULL + s), 1);
      mbar_init(BAR(CF::B_CEMPTY + s), 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if constexpr (CF::KEYB) {
    // Logical 16-byte unit u of row r sits at unit u ^ (r % 8) of the row (128-byte swizzle).
    // The ones tile: unit 0 = bf16 (1, 1, 0, ...), unit 1 = 0. Each K slot's bias atom:
    // unit 1 = 0 here, unit 0 written for every tile.
    for (int r = threadIdx.x; r < BM; r += CF::THREADS) {
      uint8_t *row_p = smem + CF::ONES_OFF + r * 128;
      *reinterpret_cast<uint4 *>(row_p + ((r & 7) << 4)) = make_uint4(0x3F803F80u, 0u, 0u, 0u);
      *reinterpret_cast<uint4 *>(row_p + ((1 ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = threadIdx.x; i < CF::KS * CF::KH_ROWS; i += CF::THREADS) {
      const int r = i % CF::KH_ROWS;
      uint8_t *row_p = smem + CF::K_OFF + (i / CF::KH_ROWS) * CF::KH_SLOT + CF::KH_TILE + r * 128;
      *reinterpret_cast<uint4 *>(row_p + ((1 ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  // The other CTA signals this CTA's barriers, so both CTAs initialise theirs first; and
  // the pair's tensor-memory allocation is one collective instruction of a warp in each
  // CTA, issued once both are known to be running.
  pair::cluster_sync();
  if (warp == CF::MMA_WARP) {
    pair::tmem_alloc(smem_u32(tmem_ptr), CF::TMEM_COLS);
    pair::tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  grid_dep_wait();
  if (threadIdx.x == 0) grid_dep_launch();

  if (warp < CF::MMA_WARP) {
    // ================================================================ softmax
    regs_increase<CF::REGS_SOFTMAX>();
    const int wg = warp / 4;  // this warpgroup takes the tiles t with t % 2 == wg
    const int wq = warp % 4;  // tensor-memory lanes [32 wq, 32 wq + 32)
    const int row = 32 * wq + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t t_o = tmem + lane_off + CF::O_COL;
    const uint32_t t_s = tmem + lane_off + wg * BN;                 // S(t) for t % 2 == wg
    const uint32_t t_p = tmem + lane_off + CF::P_COL + wg * (BN / 2);  // P(t) for t % 2 == wg
    float *rx = reinterpret_cast<float *>(smem + CF::RX_OFF);  // [2 warpgroups][128 rows]
    float *lx = reinterpret_cast<float *>(smem + CF::LX_OFF);  // [unit % 2][m, l, l'][2 warpgroups][128]
    const int h_mine = CF::B_HREF + 4 * wg + wq;
    const int h_other = CF::B_HREF + 4 * (wg ^ 1) + wq;
    const float sl2 = p.scale_log2;
    // x is raw S without a bias (exponents x scale log2 e) and scale S + C with one
    // (exponents x log2 e).
    const float scale = sl2 * LN2;
    const float xs = CF::BIASED ? LOG2E : sl2;
    bool ok = true;
    int g0 = 0;  // global number of this unit's first tile

    for (int k = 0; ok; ++k) {
      const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
      if (unit >= n_units) break;
      const PairSchedule<CAUSAL> sch(p, unit, rank);
      const int q_row = sch.qt * BM + row;
      int j_mask = CAUSAL ? floor_div(sch.qt * BM + p.causal_off + 1, BN) : INT_MAX;
      if (p.Nk % BN != 0) j_mask = cmin(j_mask, p.nkv_tiles - 1);
      const int lim = CAUSAL ? cmin(q_row + p.causal_off, p.Nk - 1) : p.Nk - 1;
      float m_prev = -INFINITY;  // reference of this warpgroup's previous tile, log2(e)-scaled
      float l = 0.0f;            // this warpgroup's share of l (fp32 p, for LSE), relative to m_prev
      float lr = 0.0f;           // the same with each tile's largest p as rounded (for O)

      for (int t = g0 + ((wg - g0) & 1); t < g0 + sch.n_it; t += 2) {
        const int j = sch.hi_max - (t - g0);
        ok = wd.wait(BAR(CF::B_SFULL + wg), (t >> 1) & 1, ROLE_SOFTMAX, CF::B_SFULL + wg);
        if (!ok) break;
        tc_fence_after();
        ETA_TRACE(1);
        // The loads return each 32-key quarter's maximum with the values.
        uint32_t r0[32], r1[32], r2[32], r3[32];
        float mx0 = tmem_ld32_max(t_s + 0, r0);
        float mx1 = tmem_ld32_max(t_s + 32, r1);
        float mx2 = tmem_ld32_max(t_s + 64, r2);
        float mx3 = tmem_ld32_max(t_s + 96, r3);
        tmem_wait_ld_max(r0, mx0);
        tmem_wait_ld_max(r1, mx1);
        tmem_wait_ld_max(r2, mx2);
        tmem_wait_ld_max(r3, mx3);
        // S(t) is in registers: its buffer may take S(t + 2).
        tc_fence_before();
        __syncwarp();
        if (leader) mbar_arrive_elect(BAR(CF::B_SEMPTY + wg));
        else pair::mbar_arrive_cluster_elect(LBAR(CF::B_SEMPTY + wg));
        float x[BN];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(r0[c]);
          x[32 + c] = __uint_as_float(r1[c]);
          x[64 + c] = __uint_as_float(r2[c]);
          x[96 + c] = __uint_as_float(r3[c]);
        }
        if constexpr (CF::DENSE) {
          // x = scale S + C: this row's 32 biases of each chunk, 16-byte unit u of row r at
          // u ^ r % 8 (the copy's 128-byte swizzle), so the reads have no bank conflicts.
#pragma unroll
          for (int cc = 0; cc < BN / CCHUNK; ++cc) {
            const int cpos = (BN / CCHUNK) * (t >> 1) + cc;  // position in this warpgroup's ring
            const int slot = wg * CF::RS + cpos % CF::RS;
            ok = wd.wait(BAR(CF::B_CFULL + slot), (cpos / CF::RS) & 1, ROLE_SOFTMAX, CF::B_CFULL + slot);
            if (!ok) break;
            const uint8_t *chunk = smem + CF::C_OFF + slot * CCHUNK_BYTES + row * 128;
#pragma unroll
            for (int u = 0; u < CCHUNK / 4; ++u) {
              const float4 cv = *reinterpret_cast<const float4 *>(chunk + ((u ^ (row & 7)) << 4));
              const int c = cc * CCHUNK + 4 * u;
              fma2(x[c + 0], x[c + 1], x[c + 0], x[c + 1], scale, scale, cv.x, cv.y);
              fma2(x[c + 2], x[c + 3], x[c + 2], x[c + 3], scale, scale, cv.z, cv.w);
            }
            __syncwarp();
            mbar_arrive_elect(BAR(CF::B_CEMPTY + slot));
          }
          if (!ok) break;
        }
        // bt: the tile's row maximum of x (raw S without a bias, scale S + C with one).
        float bt;
        if (j >= j_mask) {  // the causal diagonal or the ragged last tile: mask, then the maximum
          const int lim_j = lim - j * BN;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c > lim_j) x[c] = -INFINITY;
          bt = row_max128(x);
        } else if constexpr (CF::BIASED) {
          bt = row_max128(x);
        } else {
          bt = fmaxf(fmax3(mx0, mx1, mx2), mx3);
        }
        ETA_TRACE(2);
        // The reference after tile t - 1 (from the other warpgroup; none at a unit's first
        // tile), then this tile's: moved to b_t only when b_t exceeds it by more than
        // RESCALE_TAU (log2 units), as in attn_fwd_kernel.cuh. It is passed on at once: the
        // other warpgroup's next tile waits for it, and nothing else. Every tile but the very
        // first waits for its predecessor's, so the phases of the two barriers stay in step.
        float m_in = -INFINITY;
        if (t > 0) {
          ok = wd.wait(BAR(h_other), ((t - 1) >> 1) & 1, ROLE_SOFTMAX, h_other);
          if (!ok) break;
          if (t > g0) m_in = rx[(wg ^ 1) * BM + row];
        }
        const float bs = bt * xs;
        const bool move = bs > m_in + RESCALE_TAU;  // also the first allowed key (m_in = -inf)
        const float m_new = move ? bs : m_in;
        rx[wg * BM + row] = m_new;
        __syncwarp();
        mbar_arrive_elect(BAR(h_mine));
        ETA_TRACE(3);
        // No allowed key seen yet: every p is 0; use 0 as reference.
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        // P buffer wg was last read by P(t-2) V. (VS >= 3: P(t-2-VS) V completed before this
        // warpgroup's previous tile, P(t-2+VS) V needs a later P of its own.)
        if (t >= CF::NS) {
          const int pv = t - CF::NS;
          ok = wd.wait(BAR(CF::B_VEMPTY + pv % CF::VS), (pv / CF::VS) & 1, ROLE_SOFTMAX, CF::B_VEMPTY + pv % CF::VS);
          if (!ok) break;
          tc_fence_after();
        }
        // p_ij = 2^(x scale log2e - m) as bf16 into the P buffer, 32 keys at a time; the row
        // sum runs alongside in four independent packed chains.
        const float neg_m = -m_use;
        float s[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) s[c] = 0.0f;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint32_t pk[16];
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const int c = 32 * qq + 2 * c2;
            float a0, a1;
            fma2(a0, a1, x[c], x[c + 1], xs, xs, neg_m, neg_m);
            const float p0 = ex2_approx(a0);
            const float p1 = ex2_approx(a1);
            const int e = 2 * (c2 & 3);
            add2(s[e], s[e + 1], s[e], s[e + 1], p0, p1);
            pk[c2] = pack_bf16(p0, p1);
          }
          tmem_st16(t_p + 16 * qq, pk);
        }
        if (__any_sync(0xFFFFFFFFu, move && m_in != -INFINITY)) {
          // o (after P(t-1) V) is relative to m_in: o_t = alpha_t o_{t-1} needs that product
          // complete, which the wait here overlaps with the exponentials above; P(t) V, which
          // adds to o, waits for this tile's arrival below. Rows that saw no allowed key yet
          // have o = 0. (VS >= 3: P(t-1-VS) V completed before P(t-2) V, waited above;
          // P(t-1+VS) V needs a later P of this warpgroup.)
          const int pv = t - 1;
          ok = wd.wait(BAR(CF::B_VEMPTY + pv % CF::VS), (pv / CF::VS) & 1, ROLE_SOFTMAX, CF::B_VEMPTY + pv % CF::VS);
          if (!ok) break;
          tc_fence_after();
          const float alpha_o = move ? ex2_approx(m_in - m_use) : 1.0f;
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * cc, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float f0, f1;
              mul2(f0, f1, __uint_as_float(o[c]), __uint_as_float(o[c + 1]), alpha_o, alpha_o);
              o[c] = __float_as_uint(f0);
              o[c + 1] = __float_as_uint(f1);
            }
            tmem_st32(t_o + 32 * cc, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (leader) mbar_arrive_elect(BAR(CF::B_PFULL + wg));
        else pair::mbar_arrive_cluster_elect(LBAR(CF::B_PFULL + wg));
        ETA_TRACE(4);

        add2(s[0], s[1], s[0], s[1], s[2], s[3]);
        add2(s[4], s[5], s[4], s[5], s[6], s[7]);
        add2(s[0], s[1], s[0], s[1], s[4], s[5]);
        const float tile_sum = s[0] + s[1];
        // The tile's largest p as rounded to bf16 joins O's denominator (see
        // attn_fwd_kernel.cuh); this warpgroup's shares move from m_prev to the new reference.
        const float pmax = ex2_approx(fmaf(bt, xs, neg_m));
        const float corr = __uint_as_float(pack_bf16(pmax, pmax) << 16) - pmax;
        const float alpha = ex2_approx(m_prev - m_use);  // 1 when the reference stayed; 0 from -inf
        l = fmaf(alpha, l, tile_sum);
        lr = fmaf(alpha, lr, tile_sum + corr);
        m_prev = m_new;
        ETA_TRACE(5);
      }
      if (!ok) break;

      // The unit's row statistics go to the epilogue warps, which bring both warpgroups'
      // shares of l to the final reference (the larger of the two: the reference only
      // moves up) while these warps go on with the next unit.
      if (k >= 2) {
        ok = wd.wait(BAR(CF::B_LEMPTY + (k & 1)), ((k >> 1) & 1) ^ 1, ROLE_SOFTMAX, CF::B_LEMPTY + (k & 1));
        if (!ok) break;
      }
      float *lxk = lx + (k & 1) * (3 * 2 * BM);
      lxk[(0 * 2 + wg) * BM + row] = m_prev;
      lxk[(1 * 2 + wg) * BM + row] = l;
      lxk[(2 * 2 + wg) * BM + row] = lr;
      __syncwarp();
      mbar_arrive_elect(BAR(CF::B_LDONE + (k & 1)));
      ETA_TRACE(45);
      g0 += sch.n_it;
    }
  } else if (warp >= CF::EPI_WARP0) {
    // ================================================================ epilogue
    // O = o_T / l_T and LSE for each unit, in unit order: the rows of lanes [32 e, 32 e + 32).
    regs_decrease<CF::REGS_EPI>();
    const int e = warp - CF::EPI_WARP0;
    const int row = 32 * e + lane;
    const uint32_t t_o = tmem + (static_cast<uint32_t>(32 * e) << 16) + CF::O_COL;
    const float *lx = reinterpret_cast<const float *>(smem + CF::LX_OFF);
    bool ok = true;
    int n_o = 0;  // units so far whose o was written (phases of B_OFULL / B_OEMPTY)
    for (int k = 0; ok; ++k) {
      const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
      if (unit >= n_units) break;
      const PairSchedule<CAUSAL> sch(p, unit, rank);
      const int q_row = sch.qt * BM + row;
      ok = wd.wait(BAR(CF::B_LDONE + (k & 1)), (k >> 1) & 1, ROLE_SOFTMAX, CF::B_LDONE + (k & 1));
      if (!ok) break;
      ETA_TRACE(41);
      const float *lxk = lx + (k & 1) * (3 * 2 * BM);
      const float m0 = lxk[(0 * 2 + 0) * BM + row], m1 = lxk[(0 * 2 + 1) * BM + row];
      const float l0 = lxk[(1 * 2 + 0) * BM + row], l1 = lxk[(1 * 2 + 1) * BM + row];
      const float lr0 = lxk[(2 * 2 + 0) * BM + row], lr1 = lxk[(2 * 2 + 1) * BM + row];
      __syncwarp();
      mbar_arrive_elect(BAR(CF::B_LEMPTY + (k & 1)));
      const float m_last = fmaxf(m0, m1);
      const float m_use = (m_last == -INFINITY) ? 0.0f : m_last;
      const float f0 = ex2_approx(m0 - m_use), f1 = ex2_approx(m1 - m_use);  // 0 for a share of -inf
      const float l_row = fmaf(l0, f0, l1 * f1);
      const float lr_row = fmaf(lr0, f0, lr1 * f1);
      const float inv_l = (lr_row > 0.0f) ? 1.0f / lr_row : 0.0f;  // no allowed key: O = 0
      const int row0 = q_row - lane;
      const size_t obase = (static_cast<size_t>(sch.bh) * p.Nq + row0) * DV;
      const int esz = p.out_f32 ? 4 : 2;
      if (sch.n_it == 0) {
        // A unit whose rows see no key: O = 0, written directly (its Q copy, which no product
        // waited for, may still be landing in the buffer the others stage through).
        if (q_row < p.Nq) {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.O) + (obase + static_cast<size_t>(lane) * DV) * esz);
          for (int v = 0; v < DV * esz / 16; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
      } else {
        ok = wd.wait(BAR(CF::B_OFULL), n_o & 1, ROLE_SOFTMAX, CF::B_OFULL);
        if (!ok) break;
        tc_fence_after();
        ETA_TRACE(42);
        // The unit's Q buffer is idle once its last S completed (and is reloaded only after
        // this epilogue releases it): each warp stages its 32 rows there one box of 32 rows x
        // 128 bytes at a time, in the tensor map's 128-byte swizzle (16-byte unit u of row r
        // at u ^ r % 8, so the writes have no bank conflicts), and one lane stores it with
        // TMA; rows past Nq are clipped by the copy.
        const uint32_t stage = sbase + CF::Q_OFF + (k % CF::NQB) * CF::Q_BUF + e * (32 * 128);
        auto put = [&](int u, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
          st_shared_v4(stage + lane * 128 + ((u ^ (lane & 7)) << 4), a0, a1, a2, a3);
        };
        auto store_box = [&](int x) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmO, stage, x, row0, sch.bh);
            bulk_commit();
          }
          __syncwarp();
        };
        // The previous box has been read out of the stage.
        auto stage_free = [&]() {
          if (lane == 0) bulk_wait_read();
          __syncwarp();
        };
        // o / l for 32 columns, in place.
        auto load_o = [&](int col, uint32_t (&o)[32]) {
          tmem_ld32(t_o + col, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float f0, f1;
            mul2(f0, f1, __uint_as_float(o[c]), __uint_as_float(o[c + 1]), inv_l, inv_l);
            o[c] = __float_as_uint(f0);
            o[c + 1] = __float_as_uint(f1);
          }
        };
        // Once o is in registers, the next unit's first P V may overwrite it.
        auto release_o = [&]() {
          tc_fence_before();
          __syncwarp();
          if (leader) mbar_arrive_elect(BAR(CF::B_OEMPTY));
          else pair::mbar_arrive_cluster_elect(LBAR(CF::B_OEMPTY));
          ETA_TRACE(43);
        };
        if (p.out_f32) {
          // Four boxes of 32 fp32 columns; each column block is loaded while the previous
          // box is still being read out of the stage.
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t f[32];
            load_o(32 * h, f);
            if (h == 3) release_o();
            if (h > 0) stage_free();
#pragma unroll
            for (int v = 0; v < 8; ++v) put(v, f[4 * v + 0], f[4 * v + 1], f[4 * v + 2], f[4 * v + 3]);
            store_box(32 * h);
          }
        } else {
          // All 128 columns as bf16 pairs in registers first, so o is released early; then
          // two boxes of 64 columns.
          uint32_t bv[64];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t f[32];
            load_o(32 * h, f);
#pragma unroll
            for (int c = 0; c < 16; ++c) bv[16 * h + c] = pack_bf16(__uint_as_float(f[2 * c]), __uint_as_float(f[2 * c + 1]));
          }
          release_o();
#pragma unroll
          for (int box = 0; box < 2; ++box) {
            if (box > 0) stage_free();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              put(v, bv[32 * box + 4 * v + 0], bv[32 * box + 4 * v + 1], bv[32 * box + 4 * v + 2], bv[32 * box + 4 * v + 3]);
            store_box(64 * box);
          }
        }
        stage_free();
        ++n_o;
      }
      // LSE_i = m_i + ln l_i, from the log2-scaled reference.
      if (q_row < p.Nq && p.LSE != nullptr)
        p.LSE[static_cast<size_t>(sch.bh) * p.Nq + q_row] =
            (l_row > 0.0f) ? (m_last + lg2_approx(l_row)) * LN2 : -INFINITY;
      // The stage's generic writes come before the next TMA copy into this Q buffer.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      mbar_arrive_elect(BAR(CF::B_QEMPTY + k % CF::NQB));
      ETA_TRACE(44);
    }
  } else {
    regs_decrease<CF::REGS_CTRL>();
    if ((warp == CF::MMA_WARP || warp == CF::PV_WARP) && leader) {
      // ============================================================== MMA issue (even CTA)
      // Two issuing warps, one for the S products and one for the P V products. The tensor
      // cores take few instructions ahead, so an issuing thread blocks on every product;
      // with one issuer, its waits and commits between products left the pipe idle. Each
      // commit covers the products of its own thread.
      const uint16_t both = 3;
      const bool s_role = warp == CF::MMA_WARP;
      const int drain_bar = s_role ? CF::B_DRAIN : CF::B_DRAIN2;
      bool ok = true;
      int g0 = 0, n_o = 0;
      for (int k = 0; ok; ++k) {
        const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
        if (unit >= n_units) break;
        const PairSchedule<CAUSAL> sch(p, unit, rank);
        const int qb = k % CF::NQB;
        if (s_role) {
          ok = wd.wait(BAR(CF::B_QFULL + qb), (k / CF::NQB) & 1, ROLE_MMA, CF::B_QFULL + qb);
          if (ok) tc_fence_after();
          for (int i = 0; ok && i < sch.n_it; ++i) {
            const int t = g0 + i;
            const int kslot = t % CF::KS;
            const int b = t & 1;
            ok = wd.wait(BAR(CF::B_KFULL + kslot), (t / CF::KS) & 1, ROLE_MMA, CF::B_KFULL + kslot);
            // Buffer b is free once both CTAs' softmax warps have loaded S(t - 2).
            if (ok && t >= CF::NS)
              ok = wd.wait(BAR(CF::B_SEMPTY + b), ((t >> 1) & 1) ^ 1, ROLE_MMA, CF::B_SEMPTY + b);
            if (!ok) break;
            ETA_TRACE(24);
            tc_fence_after();
            const uint64_t a_desc = smem_desc(sbase + CF::Q_OFF + qb * CF::Q_BUF, 16, 1024);
            const uint64_t b_desc = smem_desc(sbase + CF::K_OFF + kslot * CF::KH_SLOT, 16, 1024);
            const uint32_t d_tmem = tmem + b * BN;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t a_off = ((ks / 4) * SW_CHUNK_BYTES + (ks % 4) * 32) >> 4;
              const uint32_t b_off = ((ks / 4) * CF::KH_BOX + (ks % 4) * 32) >> 4;
              pair::mma_ss_elect(d_tmem, a_desc + a_off, b_desc + b_off, CF::IDESC_S, ks > 0 ? 1u : 0u);
            }
            if constexpr (CF::KEYB)  // S += ones x (c / scale): the bias step
              pair::mma_ss_elect(d_tmem, smem_desc(sbase + CF::ONES_OFF, 16, 1024), b_desc + (CF::KH_TILE >> 4),
                                 CF::IDESC_S, 1u);
            ETA_TRACE(25);
            pair::mma_commit_multicast_elect(BAR(CF::B_SFULL + b), both);
            pair::mma_commit_multicast_elect(BAR(CF::B_KEMPTY + kslot), both);
          }
          // The unit's Q buffer is no longer read (its epilogue then stages O there).
          if (ok) pair::mma_commit_multicast_elect(BAR(CF::B_QEMPTY + qb), both);
        } else {
          for (int i = 0; ok && i < sch.n_it; ++i) {
            const int t = g0 + i;
            const int b = t & 1;
            const int vslot = t % CF::VS;
            // V and o are usually ready long before P: P, the wait on the critical path, is
            // taken last so that the product is issued as soon as P arrives.
            ETA_TRACE(20);
            ok = wd.wait(BAR(CF::B_VFULL + vslot), (t / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vslot);
            // The unit's first product overwrites o: the previous unit's epilogue has read it.
            if (ok && i == 0 && n_o > 0)
              ok = wd.wait(BAR(CF::B_OEMPTY), (n_o - 1) & 1, ROLE_MMA, CF::B_OEMPTY);
            ETA_TRACE(21);
            if (ok) ok = wd.wait(BAR(CF::B_PFULL + b), (t >> 1) & 1, ROLE_MMA, CF::B_PFULL + b);
            if (!ok) break;
            ETA_TRACE(22);
            tc_fence_after();
            const uint64_t b_desc = smem_desc(sbase + CF::V_OFF + vslot * CF::VH_TILE, SW_CHUNK_BYTES, 1024);
            const uint32_t a_tmem = tmem + CF::P_COL + b * (BN / 2);
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
              pair::mma_ts_elect(tmem + CF::O_COL, a_tmem + 8 * ks, b_desc + ((ks * 16 * 128) >> 4), CF::IDESC_PV,
                                 (i > 0 || ks > 0) ? 1u : 0u);
            ETA_TRACE(23);
            pair::mma_commit_multicast_elect(BAR(CF::B_VEMPTY + vslot), both);
          }
          if (ok && sch.n_it > 0) {
            pair::mma_commit_multicast_elect(BAR(CF::B_OFULL), both);
            ++n_o;
          }
        }
        g0 += sch.n_it;
      }
      // Nothing may still be in flight on the tensor cores when tensor memory is freed.
      pair::mma_commit_multicast_elect(BAR(drain_bar), 1);
      wd.drain(BAR(drain_bar), 0, drain_bar);
    } else if (warp == CF::LOAD_WARP && (lane == 0 || CF::KEYB)) {
      // ============================================================== TMA: Q, K halves
      // Lane 0 issues the copies. With a per-key bias the whole warp runs the loop and also
      // writes the bias columns of each K slot, two of this CTA's 64 keys a lane: v =
      // c_j / scale as bf16 parts hi = bf16(v) and lo = bf16(v - hi) (v - hi is exact in
      // fp32), so hi + lo carries v to about 2^-17 relative; c_j = -inf gives (-inf, 0),
      // which the product turns into S = -inf (1 x -inf, never 0 x inf); keys past Nk get 0
      // (their scores are masked). A tile's values are loaded as soon as the previous tile's
      // columns are out, so the load overlaps the wait for the slot.
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
      }
      auto wait_slot = [&](int b, uint32_t parity) -> bool {
        return CF::KEYB ? wd.wait(BAR(b), parity, ROLE_LOAD, b) : wd.wait1(BAR(b), parity, ROLE_LOAD, b, false);
      };
      const float inv_scale = 1.0f / (p.scale_log2 * LN2);
      const int r0 = 2 * lane;
      bool ok = true;
      int g0 = 0;
      for (int k = 0; ok; ++k) {
        const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
        if (unit >= n_units) break;
        const PairSchedule<CAUSAL> sch(p, unit, rank);
        const int qb = k % CF::NQB;
        // Q buffer qb was last used by unit k - NQB (its last S and its epilogue).
        ok = wait_slot(CF::B_QEMPTY + qb, ((k / CF::NQB) & 1) ^ 1);
        if (!ok) break;
        if (lane == 0) {
          if (leader) mbar_arrive_expect_tx(BAR(CF::B_QFULL + qb), 2 * CF::Q_TILE);
          for (int kc = 0; kc < D / SW_CHUNK; ++kc)
            pair::tma_load_3d(sbase + CF::Q_OFF + qb * CF::Q_BUF + kc * SW_CHUNK_BYTES, &tmQ, kc * SW_CHUNK,
                              sch.qt * BM, sch.bh, LBAR(CF::B_QFULL + qb));
        }
        const float *ck = CF::KEYB ? p.ckey + static_cast<size_t>(sch.bh) * p.Nk : nullptr;
        auto load_bias = [&](int i, float &c0, float &c1) {
          const int key = (sch.hi_max - i) * BN + CF::KH_ROWS * static_cast<int>(rank) + r0;
          c0 = key < p.Nk ? __ldg(ck + key) : 0.0f;
          c1 = key + 1 < p.Nk ? __ldg(ck + key + 1) : 0.0f;
        };
        float c0 = 0.0f, c1 = 0.0f;
        if (CF::KEYB && sch.n_it > 0) load_bias(0, c0, c1);
        for (int i = 0; i < sch.n_it; ++i) {
          const int t = g0 + i;
          const int j = sch.hi_max - i;
          const int ks = t % CF::KS;
          ok = wait_slot(CF::B_KEMPTY + ks, ((t / CF::KS) & 1) ^ 1);
          if (!ok) break;
          // Test hook: the first K copy is never issued, so the S product's wait runs out.
          if (lane == 0 && !(p.fault == FAULT_SKIP_FIRST_K && t == 0)) {
            if (leader) mbar_arrive_expect_tx(BAR(CF::B_KFULL + ks), 2 * CF::KH_TILE);
            for (int kc = 0; kc < D / SW_CHUNK; ++kc)
              pair::tma_load_3d(sbase + CF::K_OFF + ks * CF::KH_SLOT + kc * CF::KH_BOX, &tmK, kc * SW_CHUNK,
                                j * BN + CF::KH_ROWS * static_cast<int>(rank), sch.bh, LBAR(CF::B_KFULL + ks));
          }
          if constexpr (CF::KEYB) {
            uint8_t *atom = smem + CF::K_OFF + ks * CF::KH_SLOT + CF::KH_TILE;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = r0 + e;
              const float v = (e == 0 ? c0 : c1) * inv_scale;
              const float hi = __uint_as_float(pack_bf16(0.0f, v) & 0xFFFF0000u);
              const float lo = isinf(v) ? 0.0f : v - hi;
              *reinterpret_cast<uint4 *>(atom + r * 128 + ((r & 7) << 4)) = make_uint4(pack_bf16(hi, lo), 0u, 0u, 0u);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) pair::mbar_arrive_cluster(LBAR(CF::B_KFULL + ks));
            if (i + 1 < sch.n_it) load_bias(i + 1, c0, c1);
          }
        }
        g0 += sch.n_it;
      }
      if (wd.aborted()) settle_after_abort();
    } else if (warp == CF::VLOAD_WARP && (lane == 0 || (CF::DENSE && lane <= 2))) {
      // ============================================================== TMA: V halves (lane 0)
      // and, with a dense bias, lane 1 + w filling warpgroup w's bias ring: three threads of
      // one warp, each waiting only on its own ring, so neither stream holds up the others.
      bool ok = true;
      int g0 = 0;
      if (lane == 0) {
        tma_prefetch_desc(&tmV);
        for (int k = 0; ok; ++k) {
          const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
          if (unit >= n_units) break;
          const PairSchedule<CAUSAL> sch(p, unit, rank);
          for (int i = 0; i < sch.n_it; ++i) {
            const int t = g0 + i;
            const int j = sch.hi_max - i;
            const int vs = t % CF::VS;
            ok = wd.wait1(BAR(CF::B_VEMPTY + vs), ((t / CF::VS) & 1) ^ 1, ROLE_LOAD, CF::B_VEMPTY + vs, false);
            if (!ok) break;
            if (leader) mbar_arrive_expect_tx(BAR(CF::B_VFULL + vs), 2 * CF::VH_TILE);
            pair::tma_load_3d(sbase + CF::V_OFF + vs * CF::VH_TILE, &tmV, CF::VH_COLS * static_cast<int>(rank),
                              j * BN, sch.bh, LBAR(CF::B_VFULL + vs));
          }
          g0 += sch.n_it;
        }
      } else if constexpr (CF::DENSE) {
        // This CTA's 128 bias rows of each of warpgroup w's tiles, as four 128 x 32 chunks
        // (columns past Nk and rows past Nq arrive as zeros and are masked or not stored).
        const int w = lane - 1;
        if (w == 0) tma_prefetch_desc(&tmC);
        for (int k = 0; ok; ++k) {
          const unsigned unit = plan_unit(plan, k, cl, n_cl, n_units);
          if (unit >= n_units) break;
          const PairSchedule<CAUSAL> sch(p, unit, rank);
          for (int i = 0; ok && i < sch.n_it; ++i) {
            const int t = g0 + i;
            if ((t & 1) != w) continue;
            const int j = sch.hi_max - i;
            for (int cc = 0; cc < BN / CCHUNK; ++cc) {
              const int cpos = (BN / CCHUNK) * (t >> 1) + cc;
              const int slot = w * CF::RS + cpos % CF::RS;
              ok = wd.wait1(BAR(CF::B_CEMPTY + slot), ((cpos / CF::RS) & 1) ^ 1, ROLE_CLOAD, CF::B_CEMPTY + slot, false);
              if (!ok) break;
              mbar_arrive_expect_tx(BAR(CF::B_CFULL + slot), CCHUNK_BYTES);
              tma_load_3d(sbase + CF::C_OFF + slot * CCHUNK_BYTES, &tmC, j * BN + cc * CCHUNK, sch.qt * BM,
                          p.c_shared ? 0 : sch.bh, BAR(CF::B_CFULL + slot));
            }
          }
          g0 += sch.n_it;
        }
      }
      if (wd.aborted()) settle_after_abort();
    }
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  // Neither CTA releases its tensor or shared memory while the pair's products may still
  // read them: the even CTA's MMA warps have drained their products before they get here.
  tc_fence_before();
  __syncthreads();
  pair::cluster_sync();
  tc_fence_after();
  if (warp == CF::MMA_WARP) pair::tmem_dealloc(tmem, CF::TMEM_COLS);
}

// Clusters that can be resident at once for an instance (looked up once per device).
template <int D, int DV, bool CAUSAL, int BIAS>
int pair_max_clusters(int dev) {
  using CF = PairCfg<D, DV, CAUSAL, BIAS>;
  static int cached[64] = {0};
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(CF::THREADS);
  cfg.dynamicSmemBytes = CF::SMEM_TOTAL;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_fwd_pair_kernel<D, DV, CAUSAL, BIAS>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

// Host copies of the grid order (unit_of_block) and of a unit's key tile count (PairSchedule).
inline int host_floor_div(int a, int b) { return a >= 0 ? a / b : -((b - 1 - a) / b); }
inline int pair_unit_tiles(const KernelParams &p, unsigned b, bool causal) {
  const unsigned per_group = static_cast<unsigned>(p.head_group) * static_cast<unsigned>(p.ctas_per_head);
  const int gi = static_cast<int>(b / per_group);
  const int g0 = gi * p.head_group;
  const int gl = p.BH - g0 < p.head_group ? p.BH - g0 : p.head_group;
  const int rem = static_cast<int>(b - static_cast<unsigned>(gi) * per_group);
  const int r = rem / gl;
  const int pt = p.ctas_per_head - 1 - r;
  const int top = p.nkv_tiles - 1;
  int hi_max = top;
  if (causal) {
    const int last_row = cmin(2 * pt * BM + 2 * BM - 1, p.Nq - 1);
    hi_max = cmin(host_floor_div(last_row + p.causal_off, BN), top);
  }
  return hi_max >= 0 ? hi_max + 1 : 0;
}

// Builds the assignment of PairPlan for n_cl clusters (n = 0 when the units do not fit the
// table). The last plan built is kept per calling thread, keyed by what it depends on.
inline const PairPlan &pair_plan(const KernelParams &p, bool causal, unsigned n_cl) {
  struct Cache {
    PairPlan plan;
    long long key[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  };
  static thread_local Cache cache;
  const long long key[9] = {p.BH, p.Nq, p.Nk, p.nkv_tiles, p.causal_off, p.ctas_per_head, p.head_group,
                            causal ? 1 : 0, static_cast<long long>(n_cl)};
  bool same = true;
  for (int i = 0; i < 9; ++i) same = same && cache.key[i] == key[i];
  if (same) return cache.plan;
  PairPlan &plan = cache.plan;
  const long long n_units = static_cast<long long>(p.BH) * p.ctas_per_head;
  plan.n = 0;
  long long total_tiles = 0;
  for (long long b = 0; b < n_units && n_units <= PairPlan::MAX_UNITS; ++b)
    total_tiles += pair_unit_tiles(p, static_cast<unsigned>(b), causal);
  const bool long_units = total_tiles >= 16 * n_units;
  if (long_units && n_units <= PairPlan::MAX_UNITS && n_cl >= 1 && n_cl <= PairPlan::MAX_CLUSTERS) {
    // Each unit, in grid order, to the cluster with the least work so far (lowest index on a
    // tie); then the clusters' lists are laid end to end.
    static thread_local int owner[PairPlan::MAX_UNITS];
    long long load[PairPlan::MAX_CLUSTERS];
    int count[PairPlan::MAX_CLUSTERS];
    for (unsigned c = 0; c < n_cl; ++c) load[c] = 0, count[c] = 0;
    for (long long b = 0; b < n_units; ++b) {
      unsigned best = 0;
      for (unsigned c = 1; c < n_cl; ++c)
        if (load[c] < load[best]) best = c;
      const int tiles = pair_unit_tiles(p, static_cast<unsigned>(b), causal);
      load[best] += tiles > 0 ? tiles + 2 : 1;
      owner[b] = static_cast<int>(best);
      ++count[best];
    }
    plan.start[0] = 0;
    for (unsigned c = 0; c < n_cl; ++c) plan.start[c + 1] = static_cast<uint16_t>(plan.start[c] + count[c]);
    int fill[PairPlan::MAX_CLUSTERS];
    for (unsigned c = 0; c < n_cl; ++c) fill[c] = plan.start[c];
    for (long long b = 0; b < n_units; ++b) plan.unit[fill[owner[b]]++] = static_cast<uint16_t>(b);
    plan.n = static_cast<int>(n_units);
  }
  for (int i = 0; i < 9; ++i) cache.key[i] = key[i];
  return plan;
}

// Launches the persistent pair kernel: min(units, resident clusters) clusters of 2 CTAs.
template <int D, int DV, bool CAUSAL, int BIAS>
cudaError_t launch_attn_pair(const LaunchArgs &a) {
  using CF = PairCfg<D, DV, CAUSAL, BIAS>;
  auto kern = attn_fwd_pair_kernel<D, DV, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs * CF::THREADS < CF::REGS_NEEDED) return cudaErrorLaunchOutOfResources;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int resident = pair_max_clusters<D, DV, CAUSAL, BIAS>(dev);
  if (resident < 1) return cudaErrorLaunchOutOfResources;
  const unsigned units = static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.ctas_per_head);
  const unsigned clusters = units < static_cast<unsigned>(resident) ? units : static_cast<unsigned>(resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(CF::THREADS);
  cfg.dynamicSmemBytes = CF::SMEM_TOTAL;
  cfg.stream = a.stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  const PairPlan &plan = pair_plan(a.p, CAUSAL, clusters);
  e = cudaLaunchKernelEx(&cfg, kern, a.tmQ, a.tmK, a.tmV, a.tmC, a.tmO, a.p, plan);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace eta

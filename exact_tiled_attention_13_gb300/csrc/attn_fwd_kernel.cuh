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
// dense bias, whose time is the bias bytes, and for d_v = 128 without a bias, where
// this kernel runs only split launches: those cover a few query tiles, and the 32 KB
// of the second Q slot deepen the K/V rings instead). With one query tile, tensor memory
// holds two S buffers that the key tiles take in turn: S(t) is computed ahead of
// P(t-1) V, while the softmax still works on tile t-1. Warp roles (12 or 8 warps):
//   softmax warpgroup q (warps 4q..4q+3): thread = query row = tensor-memory lane.
//     Reads its row of S from tensor memory, masks, takes the tile max b_t, the new
//     exponent reference and alpha_t, writes P as bf16 back over S, rescales its row of o
//     in tensor memory when the reference moves (rarely: see RESCALE_TAU), accumulates
//     l_t, and at the end writes O = o/l (staged through its idle Q tile so the stores
//     write whole 128-byte row segments) and LSE.
//   control warpgroup, one thread per copy role:
//     MMA (whole warp, one elected lane issues): S_q = Q_q K_t^T (A and B from shared
//       memory) and o_q += P_q V_t (A = P from tensor memory, B = V from shared memory)
//       with tcgen05.mma; fp32 accumulators stay in tensor memory.
//     Q/K load, V load: TMA copies of Q once and of K_t, V_t into rings of shared-memory
//       slots guarded by full/empty mbarrier pairs (AI Infra ch. 5, Fig. 5-5: producer
//       copies, consumer computes, one full and one empty barrier per slot).
//     bias load: TMA copies of 128 x 32 fp32 dense-bias chunks, or the whole warp copying
//       each K/V tile's 128 per-key biases (scaled by log2(e)) into a small ring.
//   After its last K copy the Q/K warp prefetches into L2 the Q tiles of the block one
//   SM count ahead, the one the hardware is likely to start next on a freed SM.
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

#include <climits>
#include <cstdint>

#include "ptx.cuh"

namespace eta {

// Bias source of a kernel instance (the causal mask is a separate template flag).
enum { BIAS_NONE = 0, BIAS_DENSE_TMA = 1, BIAS_DENSE_DIRECT = 2, BIAS_KEY = 3 };

// Phase trace (diagnostics only; compiled in with -DETA_PHASE_TRACE): lane 0 of every
// warp of the first ETA_TRACE_CTAS CTAs appends (clock64 << 8 | event) records.
#ifdef ETA_PHASE_TRACE
constexpr int ETA_TRACE_CTAS = 8;
constexpr int ETA_TRACE_WARPS = 16;
constexpr int ETA_TRACE_EVENTS = 1024;
__device__ unsigned long long g_eta_trace[ETA_TRACE_CTAS][ETA_TRACE_WARPS][ETA_TRACE_EVENTS];
#define ETA_TRACE(ev)                                                                        \
  do {                                                                                       \
    const unsigned long long eta_t = (static_cast<unsigned long long>(clock64()) << 8) | (ev); \
    if (blockIdx.x < ETA_TRACE_CTAS && threadIdx.x / 32 < ETA_TRACE_WARPS && (threadIdx.x % 32) == 0 && \
        trace_n < ETA_TRACE_EVENTS)                                                          \
      g_eta_trace[blockIdx.x][threadIdx.x / 32][trace_n] = eta_t;                            \
    ++trace_n;                                                                               \
  } while (0)
#else
#define ETA_TRACE(ev) \
  do {                \
  } while (0)
#endif

constexpr int BM = 128;     // query rows per Q tile (= tensor-memory lanes)
constexpr int BN = 128;     // keys per K/V tile
constexpr int CCHUNK = 32;  // bias columns per dense-bias chunk (128 bytes of fp32)
constexpr int CCHUNK_BYTES = BM * CCHUNK * 4;
constexpr int SW_CHUNK = 64;                 // bf16 columns per 128-byte swizzle span
constexpr int SW_CHUNK_BYTES = 128 * 128;    // one 128-row x 128-byte box
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
// Softmax reference moves only for a tile max this far above it (log2 units): p <= 256.
constexpr float RESCALE_TAU = 8.0f;

struct KernelParams {
  int BH;
  int Nq, Nk;         // queries and keys per head
  int nq_tiles;       // ceil(Nq / 128)
  int nkv_tiles;      // ceil(Nk / 128)
  int causal_off;     // Nk - Nq: query i may see keys j <= i + causal_off
  int ctas_per_head;  // ceil(nq_tiles / NQ)
  int n_splits;       // key ranges per head (1: the whole key sequence)
  int split_tiles;    // K/V tiles per key range
  int head_group;     // heads per scheduling group (see unit_of_block)
  float scale_log2;   // scale * log2(e)
  int out_f32;        // O element type: 1 fp32, 0 bf16
  void *O;    // with n_splits > 1: fp32 partial outputs [n_splits][BH][Nq][d_v]
  float *LSE; // with n_splits > 1: partial LSE [n_splits][BH][Nq]
  const float *C;           // dense bias [BH][Nq][Nk], read directly when it cannot go through TMA
  int c_shared;             // 1: C is one [Nq][Nk] array for every head (head index 0)
  const float *ckey;        // per-key bias [BH][Nk]
  unsigned int *status;     // watchdog word (device memory)
  unsigned long long timeout_ns;
  int fault;                // test hook: FAULT_SKIP_FIRST_K makes a wait run out
};

// Test hook values (KernelParams::fault).
enum { FAULT_NONE = 0, FAULT_SKIP_FIRST_K = 1 };

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

template <int D, int DV, bool CAUSAL, int BIAS>
struct Cfg {
  static_assert(D == 64 || D == 128, "d must be 64 or 128");
  static_assert(DV == 64 || DV == 128, "d_v must be 64 or 128");
  static constexpr bool DENSE = BIAS == BIAS_DENSE_TMA || BIAS == BIAS_DENSE_DIRECT;
  static constexpr bool C_RING = BIAS == BIAS_DENSE_TMA;
  static constexpr bool KEY = BIAS == BIAS_KEY;
  static constexpr bool BIASED = DENSE || KEY;  // scores carry an additive bias
  static constexpr int NQ = (DENSE || (BIAS == BIAS_NONE && DV == 128)) ? 1 : 2;
  static constexpr int Q_TILE = BM * D * 2;
  static constexpr int K_TILE = BN * D * 2;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int KB = KEY ? 4 : 0;  // per-key bias ring: 128 fp32 per K/V tile
  static constexpr int BUDGET = 224 * 1024 - KB * BN * 4;
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
  static constexpr int KB_OFF = C_OFF + CS * CCHUNK_BYTES;
  static constexpr int BAR_OFF = KB_OFF + KB * BN * 4;
  // barrier indices
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + KS;
  static constexpr int B_VFULL = B_KEMPTY + KS;
  static constexpr int B_VEMPTY = B_VFULL + VS;
  static constexpr int B_CFULL = B_VEMPTY + VS;
  static constexpr int B_CEMPTY = B_CFULL + CS;
  static constexpr int B_KBFULL = B_CEMPTY + CS;
  static constexpr int B_KBEMPTY = B_KBFULL + KB;
  // S buffers in tensor memory: one per query tile, or two with one query tile, so that
  // S(t + 1) is computed while the softmax works on S(t).
  static constexpr bool DBUF = NQ == 1;
  static constexpr int NSB = DBUF ? 2 : NQ;
  static constexpr int B_SFULL = B_KBEMPTY + KB;  // S buffer ready (with two query tiles: and the previous P_q V done)
  static constexpr int B_PFULL = B_SFULL + NSB;   // P written over S buffer b and o rescaled
  static constexpr int B_OFULL = B_PFULL + NSB;   // last P_q V done
  static constexpr int B_DRAIN = B_OFULL + NQ;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr int TMEMPTR_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int ABORT_OFF = TMEMPTR_OFF + 4;
  static constexpr int SMEM_USED = ABORT_OFF + 4;
  // Room to align the base to 1024 B, and at least 120 KB so that one CTA holds an SM:
  // the CTA allocates most of the SM's tensor memory, and a second resident CTA would
  // block in tcgen05.alloc.
  static constexpr int SMEM_TOTAL = SMEM_USED + 1024 > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
  static_assert(SMEM_TOTAL <= 232448, "shared memory over the sm_103a per-CTA limit");

  // Warpgroups: NQ softmax warpgroups and one control warpgroup (MMA warp, Q/K load
  // warp, V load warp, bias load warp).
  static constexpr int CTRL_WARP0 = 4 * NQ;
  static constexpr int MMA_WARP = CTRL_WARP0;
  static constexpr int LOAD_WARP = CTRL_WARP0 + 1;   // Q and K
  static constexpr int VLOAD_WARP = CTRL_WARP0 + 2;  // V
  static constexpr int CLOAD_WARP = CTRL_WARP0 + 3;  // dense or per-key bias
  static constexpr int NUM_WARPS = 4 * NQ + 4;
  static constexpr int THREADS = 32 * NUM_WARPS;
  // Register budgets per warpgroup (setmaxnreg, two query tiles only): the softmax
  // warpgroups keep a whole row of S and the packed P in registers; the control
  // warpgroup needs few. setmaxnreg redistributes the registers the block was launched
  // with (THREADS x LAUNCH_REGS = 384 x 168 = 64512), so the budgets must add up to at
  // most that: 128 * (2 * 216 + 72) = 64512. A larger sum would never be granted.
  static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;
  static constexpr bool SPLIT_REGS = NQ == 2;
  static constexpr int REGS_SOFTMAX = 216;
  static constexpr int REGS_CTRL = 72;
  static constexpr int REGS_NEEDED = SPLIT_REGS ? 128 * (NQ * REGS_SOFTMAX + REGS_CTRL) : 0;
  static_assert(!SPLIT_REGS || REGS_NEEDED <= THREADS * LAUNCH_REGS,
                "register split exceeds the registers the block is launched with");
  static_assert(!SPLIT_REGS || (REGS_SOFTMAX >= LAUNCH_REGS && REGS_CTRL <= LAUNCH_REGS),
                "softmax warpgroups grow, the control warpgroup shrinks");
  // tensor memory: S buffer b at columns [b*128, b*128+128), o_q after all S buffers
  static constexpr int S_COL = 0;
  static constexpr int O_COL = NSB * BN;
  static constexpr int TMEM_COLS = pow2_at_least(NSB * BN + NQ * DV);
  static_assert(TMEM_COLS <= 512, "tensor memory holds 512 columns");

  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, true);
};

// Watchdog codes: bit 31 set, role in bits 24-27, barrier index in bits 8-23.
enum { ROLE_SOFTMAX = 1, ROLE_MMA = 2, ROLE_LOAD = 3, ROLE_CLOAD = 4, ROLE_DRAIN = 5 };

template <class Params>
struct WatchdogT {
  // The abort flag lives in shared memory; the status word and the timeout are read from
  // the kernel parameters only on the slow path, so the common case holds one register.
  uint32_t abort_addr;
  const Params &p;

  __device__ bool aborted() const {
    int v;
    asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(abort_addr) : "memory");
    return v != 0;
  }
  __device__ void trip(int role, int bar) {
    asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort_addr), "r"(1) : "memory");
    atomicCAS(p.status, 0u, 0x80000000u | (static_cast<unsigned>(role) << 24) |
                                (static_cast<unsigned>(bar & 0xFFFF) << 8));
  }

  // Bounded wait of one thread; false on timeout or when another role aborted.
  __device__ bool wait1(uint32_t bar_addr, uint32_t parity, int role, int bar, bool drain) {
    if (mbar_try_wait(bar_addr, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
      if (mbar_try_wait(bar_addr, parity)) return true;
      if ((spin & 15u) == 0) {
        if (!drain && aborted()) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
          trip(drain ? ROLE_DRAIN : role, bar);
          return false;
        }
      }
    }
  }

  // Whole-warp bounded wait: every lane observes the barrier; the result is uniform.
  // The common case (phase already complete) is one try_wait and one vote.
  __device__ bool wait(uint32_t bar_addr, uint32_t parity, int role, int bar) {
    if (__all_sync(0xFFFFFFFFu, mbar_try_wait(bar_addr, parity))) return true;
    const bool ok = wait1(bar_addr, parity, role, bar, false);
    return __all_sync(0xFFFFFFFFu, ok);
  }
  __device__ bool drain(uint32_t bar_addr, uint32_t parity, int bar) {
    const bool ok = wait1(bar_addr, parity, ROLE_DRAIN, bar, true);
    return __all_sync(0xFFFFFFFFu, ok);
  }
};

using Watchdog = WatchdogT<KernelParams>;

// Grid order. Each head has U work units, unit r = 0 holding the most work (for a causal
// mask, the query tiles that see the most keys). Heads are taken in groups of G whose
// K/V fit in L2 together; within a group the blocks go by unit rank first and head
// second, so every head's largest unit starts before any head's smaller ones (longest
// first) and the blocks that share a head's K/V still run close in time. Block b maps
// to head *bh and rank *r.
__device__ __forceinline__ void unit_of_block(unsigned b, int BH, int U, int G, int *bh, int *r) {
  const unsigned per_group = static_cast<unsigned>(G) * static_cast<unsigned>(U);
  const int gi = static_cast<int>(b / per_group);
  const int g0 = gi * G;
  const int gl = BH - g0 < G ? BH - g0 : G;
  const int rem = static_cast<int>(b - static_cast<unsigned>(gi) * per_group);
  *r = rem / gl;
  *bh = g0 + rem % gl;
}

// Per-CTA schedule: which query tiles it owns and which K/V tiles each one visits.
// Iteration `it` visits K/V tile j = hi_max - it; query tile q takes part in
// iterations [first_it(q), n_it), i.e. K/V tiles hi(q) down to 0. With a causal mask
// a query tile's last K/V tile is the one holding the last key its last row may see;
// a query tile whose rows may see no key at all (Nq > Nk) takes part in none.
__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((b - 1 - a) / b); }

template <int NQ, bool CAUSAL>
struct Schedule {
  static_assert(NQ == 1 || NQ == 2, "one or two query tiles per CTA");
  int bh, cta_q, n_exist, hi_max, n_it;
  int first0, first1;  // first_it of query tiles 0 and 1

  __device__ explicit Schedule(const KernelParams &p, unsigned unit) {
    // A head's units: key range, then query tiles from the last (most causal work) down.
    int r;
    unit_of_block(unit, p.BH, p.ctas_per_head * p.n_splits, p.head_group, &bh, &r);
    const int split = r / p.ctas_per_head;
    cta_q = p.ctas_per_head - 1 - r % p.ctas_per_head;
    n_exist = cmin(NQ, p.nq_tiles - cta_q * NQ);
    const int lo = split * p.split_tiles;  // this CTA's K/V tiles: lo .. top
    const int top = cmin(lo + p.split_tiles, p.nkv_tiles) - 1;
    const int hi0 = hi(p, 0, top);
    const int hi1 = NQ == 2 ? hi(p, 1, top) : lo - 1;
    hi_max = n_exist == 2 ? hi1 : hi0;  // hi grows with the query tile
    n_it = hi_max >= lo ? hi_max - lo + 1 : 0;
    if (CAUSAL) {
      first0 = hi0 >= lo ? hi_max - hi0 : n_it;
      first1 = (n_exist == 2 && hi1 >= lo) ? hi_max - hi1 : n_it;
    } else {  // every query tile visits the whole range (n_it is 0 for an empty range)
      first0 = 0;
      first1 = n_exist == 2 ? 0 : n_it;
    }
  }
  __device__ int q_tile(int q) const { return cta_q * NQ + q; }
  // Last K/V tile query tile q visits, at most `top` (below the range's first: none).
  __device__ int hi(const KernelParams &p, int q, int top) const {
    if (!CAUSAL) return top;
    const int last_row = cmin(q_tile(q) * BM + BM - 1, p.Nq - 1);
    return cmin(floor_div(last_row + p.causal_off, BN), top);
  }
  // First iteration query tile q takes part in; n_it when it takes part in none.
  __device__ int first_it(int q) const { return q == 0 ? first0 : first1; }
};

// Row maximum of 128 values with eight independent three-input max chains.
__device__ __forceinline__ float row_max128(const float (&x)[BN]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
  for (int c = 16; c < BN; c += 16) {
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], x[c + 2 * k], x[c + 2 * k + 1]);
  }
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(fmax3(m[3], m[4], m[5]), m[6], m[7]));
}

template <int D, int DV, bool CAUSAL, int BIAS>
__global__ void __launch_bounds__(Cfg<D, DV, CAUSAL, BIAS>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ KernelParams p) {
  using CF = Cfg<D, DV, CAUSAL, BIAS>;
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
#ifdef ETA_PHASE_TRACE
  int trace_n = 0;
#endif
  ETA_TRACE(90);
  const Schedule<NQ, CAUSAL> sch(p, blockIdx.x);
  Watchdog wd{sbase + CF::ABORT_OFF, p};

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
    if constexpr (CF::KEY) {
      // Every softmax warpgroup that visits any K/V tile releases every slot once.
      int consumers = 0;
      for (int q = 0; q < NQ; ++q) consumers += sch.first_it(q) < sch.n_it ? 4 : 0;
      for (int s = 0; s < CF::KB; ++s) {
        mbar_init(BAR(CF::B_KBFULL + s), 1);
        mbar_init(BAR(CF::B_KBEMPTY + s), consumers > 0 ? consumers : 1);
      }
    }
    for (int b = 0; b < CF::NSB; ++b) {
      mbar_init(BAR(CF::B_SFULL + b), 1);
      mbar_init(BAR(CF::B_PFULL + b), 4);  // one arrival per softmax warp
    }
    for (int q = 0; q < NQ; ++q) mbar_init(BAR(CF::B_OFULL + q), 1);
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
  // Set-up done: now wait for the previous kernel on the stream (programmatic launch) before
  // any global memory is touched, and let the next one start launching.
  grid_dep_wait();
  if (threadIdx.x == 0) grid_dep_launch();

  if (warp < CF::CTRL_WARP0) {
    // ================================================================ softmax
    if constexpr (CF::SPLIT_REGS) regs_increase<CF::REGS_SOFTMAX>();
    const int q = warp / 4;
    const int row = threadIdx.x % BM;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const uint32_t t_s = tmem + lane_off + CF::S_COL + q * BN;
    const uint32_t t_o = tmem + lane_off + CF::O_COL + q * DV;
    const int qt = sch.q_tile(q);
    const int q_row = qt * BM + row;
    const bool exists = q < sch.n_exist;
    const bool has_keys = sch.first_it(q) < sch.n_it;  // some K/V tile is visible to this tile
    const float sl2 = p.scale_log2;
    float m2 = -INFINITY;  // running max m_t, in log2(e)-scaled units
    float l = 0.0f;        // running sum l_t of the fp32 p (for LSE)
    float lr = 0.0f;       // l_t with each tile's largest p as rounded to bf16 (for O)
    uint32_t s_phase = 0;
    bool ok = true;
    int cpos = 0;  // dense-bias ring position
    if constexpr (CF::KEY) {
      // Per-key bias slots of iterations this query tile skips are released at once.
      if (has_keys)
        for (int it = 0; it < sch.first_it(q); ++it) {
          __syncwarp();
          mbar_arrive_elect(BAR(CF::B_KBEMPTY + it % CF::KB));
        }
    }
    // Tiles j >= j_mask need an elementwise mask: those that reach past the causal limit
    // of the tile's first row, and the last tile when Nk is not a multiple of 128. lim is
    // the last key this row may see (the causal limit i + (Nk - Nq), or the last key).
    int j_mask = CAUSAL ? floor_div(qt * BM + p.causal_off + 1, BN) : INT_MAX;
    if (p.Nk % BN != 0) j_mask = cmin(j_mask, p.nkv_tiles - 1);
    const int lim = CAUSAL ? cmin(q_row + p.causal_off, p.Nk - 1) : p.Nk - 1;
    if (exists && has_keys) {
      for (int it = sch.first_it(q); it < sch.n_it; ++it) {
        const int j = sch.hi_max - it;
        // This tile's S buffer: the query tile's own, or (one query tile) buffer it % 2.
        const int sb = CF::DBUF ? (it & 1) : q;
        const uint32_t t_sb = CF::DBUF ? t_s + static_cast<uint32_t>((it & 1) * BN) : t_s;
        ok = wd.wait(BAR(CF::B_SFULL + sb), CF::DBUF ? static_cast<uint32_t>((it >> 1) & 1) : s_phase,
                     ROLE_SOFTMAX, CF::B_SFULL + sb);
        s_phase ^= 1;
        if (!ok) break;
        tc_fence_after();
        ETA_TRACE(1);

        // Row of S (raw Q K^T) for this thread's query, 128 keys.
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(t_sb + 0, r0);
        tmem_ld32(t_sb + 32, r1);
        tmem_ld32(t_sb + 64, r2);
        tmem_ld32(t_sb + 96, r3);
        tmem_wait_ld(r0);
        tmem_wait_ld(r1);
        tmem_wait_ld(r2);
        tmem_wait_ld(r3);
        ETA_TRACE(2);
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
          if constexpr (CF::C_RING) {
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
                float b0, b1, b2, b3;
                mul2(b0, b1, cv.x, cv.y, LOG2E, LOG2E);
                mul2(b2, b3, cv.z, cv.w, LOG2E, LOG2E);
                fma2(x[c + 0], x[c + 1], x[c + 0], x[c + 1], sl2, sl2, b0, b1);
                fma2(x[c + 2], x[c + 3], x[c + 2], x[c + 3], sl2, sl2, b2, b3);
              }
              __syncwarp();
              mbar_arrive_elect(BAR(CF::B_CEMPTY + slot));
              ++cpos;
            }
            if (!ok) break;
          } else {
            const bool row_ok = q_row < p.Nq;
            const int c_bh = p.c_shared ? 0 : sch.bh;
            const float *crow = p.C + (static_cast<size_t>(c_bh) * p.Nq + (row_ok ? q_row : 0)) *
                                          static_cast<size_t>(p.Nk);
#pragma unroll
            for (int c = 0; c < BN; ++c) {
              const int kv = j * BN + c;
              const float cv = (row_ok && kv < p.Nk) ? __ldg(crow + kv) : 0.0f;
              x[c] = fmaf(x[c], sl2, cv * LOG2E);
            }
          }
        }
        if constexpr (CF::KEY) {
          // x = (scale * S + c_j) * log2(e), c_j the same for every row: broadcast reads.
          const int slot = it % CF::KB;
          ok = wd.wait(BAR(CF::B_KBFULL + slot), (it / CF::KB) & 1, ROLE_SOFTMAX, CF::B_KBFULL + slot);
          if (!ok) break;
          const float4 *kb = reinterpret_cast<const float4 *>(smem + CF::KB_OFF + slot * BN * 4);
#pragma unroll
          for (int u = 0; u < BN / 4; ++u) {
            const float4 cv = kb[u];  // c_j log2(e), stored so by the bias copy
            fma2(x[4 * u + 0], x[4 * u + 1], x[4 * u + 0], x[4 * u + 1], sl2, sl2, cv.x, cv.y);
            fma2(x[4 * u + 2], x[4 * u + 3], x[4 * u + 2], x[4 * u + 3], sl2, sl2, cv.z, cv.w);
          }
          __syncwarp();
          mbar_arrive_elect(BAR(CF::B_KBEMPTY + slot));
        }

        // Forbidden keys: past the causal limit, and past the end of the keys.
        if (j >= j_mask) {
          const int lim_j = lim - j * BN;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c > lim_j) x[c] = -INFINITY;
        }

        // b_t, then the exponent reference m_t. The recurrence's m_t = max(m_{t-1}, b_t)
        // may be replaced by any reference that is used consistently for p, l and o: the
        // final o_T / l_T is the same function. The reference moves to b_t only when b_t
        // exceeds it by more than RESCALE_TAU (log2 units), so p <= 2^RESCALE_TAU stays
        // far inside bf16 and fp32 range, and o needs rescaling (alpha_t != 1) only then.
        const float b = row_max128(x);
        const float bs = CF::BIASED ? b : b * sl2;  // b_t in log2 units
        const bool move = bs > m2 + RESCALE_TAU;    // also the first allowed key (m2 = -inf)
        const float m_new = move ? bs : m2;
        // No allowed key seen yet: every p is 0; use 0 as reference.
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = move ? ex2_approx(m2 - m_use) : 1.0f;
        if (__any_sync(0xFFFFFFFFu, move) && it > sch.first_it(q)) {
          // o_t = alpha_t o_{t-1} once the previous P V has completed: with two query tiles
          // the S tile just read was committed after it; with two S buffers S(it) is issued
          // before P(it-1) V, so wait for that product's commit on its V slot. (Every
          // earlier P V completed before S(it), so the slot's phases cannot be confused.)
          // Rare once a row has seen its largest scores. On a query tile's first K/V tile
          // o holds no result yet (the first P V overwrites it).
          if constexpr (CF::DBUF) {
            const int pv = it - 1;
            ok = wd.wait(BAR(CF::B_VEMPTY + pv % CF::VS), (pv / CF::VS) & 1, ROLE_SOFTMAX, CF::B_VEMPTY + pv % CF::VS);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(t_o + 32 * cc, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float f0, f1;
              mul2(f0, f1, __uint_as_float(o[c]), __uint_as_float(o[c + 1]), alpha, alpha);
              o[c] = __float_as_uint(f0);
              o[c + 1] = __float_as_uint(f1);
            }
            tmem_st32(t_o + 32 * cc, o);
          }
        }

        // p_ij = exp(S_ij - m_t) as bf16 into tensor memory over S, 32 keys at a time;
        // the row sum runs alongside in four independent packed chains.
        const float neg_m = -m_use;
        float s[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) s[k] = 0.0f;
        uint32_t pk[32];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const int c = 32 * qq + 2 * c2;
            float a0, a1;
            if constexpr (CF::BIASED) {
              add2(a0, a1, x[c], x[c + 1], neg_m, neg_m);
            } else {
              fma2(a0, a1, x[c], x[c + 1], sl2, sl2, neg_m, neg_m);
            }
            const float p0 = ex2_approx(a0);
            const float p1 = ex2_approx(a1);
            const int k = 2 * (c2 & 3);
            add2(s[k], s[k + 1], s[k], s[k + 1], p0, p1);
            pk[16 * (qq & 1) + c2] = pack_bf16(p0, p1);
          }
          if (qq & 1) tmem_st32(t_sb + 32 * (qq / 2), pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        mbar_arrive_elect(BAR(CF::B_PFULL + sb));
        ETA_TRACE(4);

        // l_t = alpha_t l_{t-1} + sum_j p_ij.
        add2(s[0], s[1], s[0], s[1], s[2], s[3]);
        add2(s[4], s[5], s[4], s[5], s[6], s[7]);
        add2(s[0], s[1], s[0], s[1], s[4], s[5]);
        // The tile's largest p, computed as in the loop, and its bf16 rounding: under a
        // stale reference it need not be exactly 1, so the denominator of O takes it as
        // rounded, like the P that multiplies V (a row dominated by one key then gets
        // that key's v to fp32 accuracy). The other p round as they would with the
        // eager reference; LSE keeps the fp32 sum.
        float pmax;
        if constexpr (CF::BIASED) {
          pmax = ex2_approx(b + neg_m);
        } else {
          pmax = ex2_approx(fmaf(b, sl2, neg_m));
        }
        const float pmax_r = __uint_as_float(pack_bf16(pmax, pmax) << 16);
        const float tile_sum = s[0] + s[1];
        l = fmaf(alpha, l, tile_sum);
        lr = fmaf(alpha, lr, tile_sum + (pmax_r - pmax));
        ETA_TRACE(5);
        m2 = m_new;
      }

    }
    // ------------------------------------------------ epilogue: O = o_T / l_T, LSE
    // A query tile that may see no key (Nq > Nk with a causal mask) has no o: its rows
    // get the defined result of a row without an allowed key, O = 0 and LSE = -inf.
    if (exists && ok) {
      if (has_keys) ok = wd.wait(BAR(CF::B_OFULL + q), 0, ROLE_SOFTMAX, CF::B_OFULL + q);
      ETA_TRACE(6);
      if (ok) {
        if (has_keys) tc_fence_after();
        const bool row_ok = q_row < p.Nq;
        const float inv_l = (lr > 0.0f) ? 1.0f / lr : 0.0f;  // no allowed key: O = 0
        // Key range `split` of a split launch writes its own slice of the partials.
        int ubh, ur;
        unit_of_block(blockIdx.x, p.BH, p.ctas_per_head * p.n_splits, p.head_group, &ubh, &ur);
        const int split = ur / p.ctas_per_head;
        const size_t lrow = (static_cast<size_t>(split) * p.BH + sch.bh) * p.Nq + (row_ok ? q_row : 0);
        const size_t orow = lrow * DV;
        if (has_keys && !CF::DENSE) {
          // This warpgroup's Q tile is idle now (its last product has completed): each warp
          // stages 32 rows x 128 bytes of O there at a time, in 16-byte units placed at
          // (unit ^ row % 8) so that neither side of the stage has bank conflicts, and
          // stores them as whole 128-byte row segments, four rows per instruction.
          static_assert(CF::Q_TILE / 4 >= 32 * 128, "a warp's stage is 32 rows of 128 bytes");
          uint8_t *stage = smem + CF::Q_OFF + q * CF::Q_TILE + (warp % 4) * (CF::Q_TILE / 4);
          uint4 *srow = reinterpret_cast<uint4 *>(stage + lane * 128);
          const int row0 = q_row - lane;  // the warp's first query row
          const int rows_ok = p.Nq - row0 < 32 ? (p.Nq - row0 > 0 ? p.Nq - row0 : 0) : 32;
          const size_t obase = ((static_cast<size_t>(split) * p.BH + sch.bh) * p.Nq + row0) * DV;
          const int sub = lane % 8;
          // All eight shared loads go before the global stores, which the compiler could not
          // otherwise move them past.
          auto store_stage = [&](uint8_t *g0, int row_bytes) {
            __syncwarp();
            uint4 val[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 4 * i + lane / 8;
              val[i] = *reinterpret_cast<const uint4 *>(stage + rr * 128 + 16 * (sub ^ (rr & 7)));
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 4 * i + lane / 8;
              if (rr < rows_ok)
                *reinterpret_cast<uint4 *>(g0 + static_cast<size_t>(rr) * row_bytes + 16 * sub) = val[i];
            }
          };
          if (p.out_f32) {
#pragma unroll 1
            for (int cc = 0; cc < DV / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(t_o + 32 * cc, o);
              tmem_wait_ld(o);
              float f[32];
#pragma unroll
              for (int c = 0; c < 32; c += 2)
                mul2(f[c], f[c + 1], __uint_as_float(o[c]), __uint_as_float(o[c + 1]), inv_l, inv_l);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                srow[v ^ (lane & 7)] = make_uint4(__float_as_uint(f[4 * v + 0]), __float_as_uint(f[4 * v + 1]),
                                                  __float_as_uint(f[4 * v + 2]), __float_as_uint(f[4 * v + 3]));
              store_stage(reinterpret_cast<uint8_t *>(static_cast<float *>(p.O) + obase + 32 * cc), DV * 4);
            }
          } else {
#pragma unroll 1
            for (int cc = 0; cc < DV / 64; ++cc) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                tmem_ld32(t_o + 64 * cc + 32 * h, o);
                tmem_wait_ld(o);
                float f[32];
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                  mul2(f[c], f[c + 1], __uint_as_float(o[c]), __uint_as_float(o[c + 1]), inv_l, inv_l);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  srow[(4 * h + v) ^ (lane & 7)] =
                      make_uint4(pack_bf16(f[8 * v + 0], f[8 * v + 1]), pack_bf16(f[8 * v + 2], f[8 * v + 3]),
                                 pack_bf16(f[8 * v + 4], f[8 * v + 5]), pack_bf16(f[8 * v + 6], f[8 * v + 7]));
              }
              store_stage(reinterpret_cast<uint8_t *>(static_cast<uint16_t *>(p.O) + obase + 64 * cc), DV * 2);
            }
          }
        } else {
          // Direct stores, one row per lane: for a tile that sees no key (O = 0; its Q copy
          // may still be landing, so nothing is staged) and for the dense-bias kernel, whose
          // single softmax warpgroup measured slower with the staged stores. Every lane runs
          // the tensor-memory loads (warp-collective); only the stores depend on the row.
#pragma unroll
          for (int cc = 0; cc < DV / 32; ++cc) {
            uint32_t o[32];
            if (has_keys) {
              tmem_ld32(t_o + 32 * cc, o);
              tmem_wait_ld(o);
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = 0u;
            }
            float f[32];
#pragma unroll
            for (int c = 0; c < 32; c += 2)
              mul2(f[c], f[c + 1], __uint_as_float(o[c]), __uint_as_float(o[c + 1]), inv_l, inv_l);
            if (row_ok) {
              if (p.out_f32) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.O) + orow + 32 * cc);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v] = make_float4(f[4 * v + 0], f[4 * v + 1], f[4 * v + 2], f[4 * v + 3]);
              } else {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.O) + orow + 32 * cc);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  dst[v] = make_uint4(pack_bf16(f[8 * v + 0], f[8 * v + 1]), pack_bf16(f[8 * v + 2], f[8 * v + 3]),
                                      pack_bf16(f[8 * v + 4], f[8 * v + 5]), pack_bf16(f[8 * v + 6], f[8 * v + 7]));
              }
            }
          }
        }
        if (row_ok && p.LSE != nullptr) {
          // LSE_i = m_i + ln l_i, from the log2-scaled running max.
          p.LSE[lrow] =
              (l > 0.0f) ? (m2 + lg2_approx(l)) * LN2 : -INFINITY;
        }
        ETA_TRACE(92);
      }
    }
  } else {
    // Control warpgroup. The MMA role runs on the whole warp with one elected lane issuing
    // each instruction; each copy role runs on lane 0 alone while the other lanes wait at
    // the warp barrier below.
    if constexpr (CF::SPLIT_REGS) regs_decrease<CF::REGS_CTRL>();
    if (warp == CF::MMA_WARP) {
      // ============================================================== MMA issue
      // The whole warp runs this loop; each MMA and commit is issued by one elected lane.
      uint32_t p_phase[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) p_phase[q] = 0;
      bool ok = wd.wait(BAR(CF::B_QFULL), 0, ROLE_MMA, CF::B_QFULL);
      tc_fence_after();

      // The descriptors' address field holds (address >> 4) in 14 bits; shared-memory
      // addresses stay below 2^18, so adding (offset >> 4) to a descriptor never carries.
      auto issue_s = [&](int q, int kslot, int b) {  // S buffer b = Q_q K^T
        const uint64_t a_desc = smem_desc(sbase + CF::Q_OFF + q * CF::Q_TILE, 16, 1024);
        const uint64_t b_desc = smem_desc(sbase + CF::K_OFF + kslot * CF::K_TILE, 16, 1024);
        const uint32_t d_tmem = tmem + CF::S_COL + b * BN;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks / 4) * SW_CHUNK_BYTES + (ks % 4) * 32) >> 4;
          mma_ss_elect(d_tmem, a_desc + off, b_desc + off, CF::IDESC_S, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int q, int vslot, bool accumulate, int b) {  // o_q += P (S buffer b) V
        const uint64_t b_desc =
            smem_desc(sbase + CF::V_OFF + vslot * CF::V_TILE, SW_CHUNK_BYTES, 1024);
        const uint32_t d_tmem = tmem + CF::O_COL + q * DV;
        const uint32_t a_tmem = tmem + CF::S_COL + b * BN;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_ts_elect(d_tmem, a_tmem + ks * 8, b_desc + ((ks * 16 * 128) >> 4), CF::IDESC_PV,
                       (ks > 0 || accumulate) ? 1u : 0u);
      };
      // P_q written and o_q rescaled (one barrier) before o_q += P_q V.
      auto wait_pv_inputs = [&](int q) -> bool {
        const bool r = wd.wait(BAR(CF::B_PFULL + q), p_phase[q], ROLE_MMA, CF::B_PFULL + q);
        p_phase[q] ^= 1;
        return r;
      };

      if constexpr (CF::DBUF) {
        // One query tile, two S buffers: S(it) goes to buffer it % 2 as soon as K(it) has
        // landed, ahead of P(it-1) V, whose P the softmax may still be writing. S(it)
        // overwrites P(it-2), which P(it-2) V, issued before it, has read.
        for (int it = 0; ok && it < sch.n_it; ++it) {
          const int kslot = it % CF::KS;
          ok = wd.wait(BAR(CF::B_KFULL + kslot), (it / CF::KS) & 1, ROLE_MMA, CF::B_KFULL + kslot);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, kslot, it & 1);  // S buffer it % 2 = Q K_it^T
          mma_commit_elect(BAR(CF::B_SFULL + (it & 1)));
          mma_commit_elect(BAR(CF::B_KEMPTY + kslot));
          if (it > 0) {
            const int pv = it - 1, vslot = pv % CF::VS;
            ok = wd.wait(BAR(CF::B_VFULL + vslot), (pv / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vslot);
            if (ok) ok = wd.wait(BAR(CF::B_PFULL + (pv & 1)), (pv >> 1) & 1, ROLE_MMA, CF::B_PFULL + (pv & 1));
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, vslot, pv > 0, pv & 1);  // o += P_{it-1} V_{it-1}
            mma_commit_elect(BAR(CF::B_VEMPTY + vslot));
          }
        }
        if (ok && sch.n_it > 0) {
          const int pv = sch.n_it - 1, vslot = pv % CF::VS;
          ok = wd.wait(BAR(CF::B_VFULL + vslot), (pv / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vslot);
          if (ok) ok = wd.wait(BAR(CF::B_PFULL + (pv & 1)), (pv >> 1) & 1, ROLE_MMA, CF::B_PFULL + (pv & 1));
          if (ok) {
            tc_fence_after();
            issue_pv(0, vslot, pv > 0, pv & 1);
            mma_commit_elect(BAR(CF::B_OFULL));
            mma_commit_elect(BAR(CF::B_VEMPTY + vslot));
          }
        }
      } else {
        for (int it = 0; ok && it < sch.n_it; ++it) {
          const int kslot = it % CF::KS;
          const int vprev = (it + CF::VS - 1) % CF::VS;
          ok = wd.wait(BAR(CF::B_KFULL + kslot), (it / CF::KS) & 1, ROLE_MMA, CF::B_KFULL + kslot);
          ETA_TRACE(20);
          if (ok && it > 0)
            ok = wd.wait(BAR(CF::B_VFULL + vprev), ((it - 1) / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vprev);
          if (!ok) break;
          tc_fence_after();
  #pragma unroll
          for (int q = 0; q < NQ; ++q) {
            if (it < sch.first_it(q)) continue;
            ETA_TRACE(21);
            if (it > sch.first_it(q)) {
              ok = wait_pv_inputs(q);
              if (!ok) break;
              ETA_TRACE(22 + q);
              tc_fence_after();
              issue_pv(q, vprev, it - 1 > sch.first_it(q), q);  // o_q += P_q V_{it-1}
            }
            issue_s(q, kslot, q);  // S_q = Q_q K_it^T
            mma_commit_elect(BAR(CF::B_SFULL + q));
            ETA_TRACE(24 + q);
          }
          if (!ok) break;
          mma_commit_elect(BAR(CF::B_KEMPTY + kslot));
          if (it > 0) mma_commit_elect(BAR(CF::B_VEMPTY + vprev));
        }
        if (ok && sch.n_it > 0) {
          const int last = sch.n_it - 1;
          const int vslot = last % CF::VS;
          ok = wd.wait(BAR(CF::B_VFULL + vslot), (last / CF::VS) & 1, ROLE_MMA, CF::B_VFULL + vslot);
          if (ok) tc_fence_after();
  #pragma unroll
          for (int q = 0; q < NQ; ++q) {
            if (!ok || sch.first_it(q) >= sch.n_it) continue;
            ok = wait_pv_inputs(q);
            if (!ok) break;
            tc_fence_after();
            issue_pv(q, vslot, last > sch.first_it(q), q);
            mma_commit_elect(BAR(CF::B_OFULL + q));
          }
          if (ok) mma_commit_elect(BAR(CF::B_VEMPTY + vslot));
        }
      }
      // Nothing may still be in flight on the tensor cores when tensor memory is freed.
      mma_commit_elect(BAR(CF::B_DRAIN));
      wd.drain(BAR(CF::B_DRAIN), 0, CF::B_DRAIN);
    } else if (warp == CF::LOAD_WARP && lane == 0) {
      // ============================================================== TMA: Q, K
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(BAR(CF::B_QFULL), sch.n_exist * CF::Q_TILE);
      for (int q = 0; q < sch.n_exist; ++q)
        for (int kc = 0; kc < D / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::Q_OFF + q * CF::Q_TILE + kc * SW_CHUNK_BYTES, &tmQ,
                      kc * SW_CHUNK, sch.q_tile(q) * BM, sch.bh, BAR(CF::B_QFULL));
      // K runs ahead on its own ring; V has its own producer so neither blocks the other.
      // last[s] is the last iteration whose copy was issued into slot s (-1: none).
      int last[CF::KS];
      for (int s = 0; s < CF::KS; ++s) last[s] = -1;
      for (int it = 0; it < sch.n_it; ++it) {
        const int j = sch.hi_max - it;
        const int ks = it % CF::KS;
        const bool ok =
            wd.wait1(BAR(CF::B_KEMPTY + ks), ((it / CF::KS) & 1) ^ 1, ROLE_LOAD, CF::B_KEMPTY + ks, false);
        ETA_TRACE(30);
        if (!ok) break;
        // Test hook: the first K tile is never copied, so its consumer's wait runs out.
        if (p.fault == FAULT_SKIP_FIRST_K && it == 0) continue;
        mbar_arrive_expect_tx(BAR(CF::B_KFULL + ks), CF::K_TILE);
        for (int kc = 0; kc < D / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::K_OFF + ks * CF::K_TILE + kc * SW_CHUNK_BYTES, &tmK,
                      kc * SW_CHUNK, j * BN, sch.bh, BAR(CF::B_KFULL + ks));
        last[ks] = it;
      }
      // The block the hardware will likely start next, on the first SM to free up, is about
      // one wave ahead: warm L2 with its Q tiles (each unit's own, read from HBM once) so
      // that its first S product does not wait on HBM. (Not in the dense-bias kernel, which
      // is bound by the bias stream and measured slower with it.)
      const unsigned next = blockIdx.x + nsmid();
      if (!CF::DENSE && next < gridDim.x) {
        const Schedule<NQ, CAUSAL> nxt(p, next);
        for (int q = 0; q < nxt.n_exist; ++q)
          for (int kc = 0; kc < D / SW_CHUNK; ++kc)
            tma_prefetch_l2_3d(&tmQ, kc * SW_CHUNK, nxt.q_tile(q) * BM, nxt.bh);
      }
      // Wait for the last copy into each slot to land before the CTA may exit.
      wd.wait1(BAR(CF::B_QFULL), 0, ROLE_DRAIN, CF::B_QFULL, true);
      for (int s = 0; s < CF::KS; ++s)
        if (last[s] >= 0)
          wd.wait1(BAR(CF::B_KFULL + s), (last[s] / CF::KS) & 1, ROLE_DRAIN, CF::B_KFULL + s, true);
    } else if (warp == CF::VLOAD_WARP && lane == 0) {
      // ============================================================== TMA: V
      tma_prefetch_desc(&tmV);
      int last[CF::VS];
      for (int s = 0; s < CF::VS; ++s) last[s] = -1;
      for (int it = 0; it < sch.n_it; ++it) {
        const int j = sch.hi_max - it;
        const int vs = it % CF::VS;
        const bool ok =
            wd.wait1(BAR(CF::B_VEMPTY + vs), ((it / CF::VS) & 1) ^ 1, ROLE_LOAD, CF::B_VEMPTY + vs, false);
        ETA_TRACE(31);
        if (!ok) break;
        mbar_arrive_expect_tx(BAR(CF::B_VFULL + vs), CF::V_TILE);
        for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
          tma_load_3d(sbase + CF::V_OFF + vs * CF::V_TILE + kc * SW_CHUNK_BYTES, &tmV,
                      kc * SW_CHUNK, j * BN, sch.bh, BAR(CF::B_VFULL + vs));
        last[vs] = it;
      }
      for (int s = 0; s < CF::VS; ++s)
        if (last[s] >= 0)
          wd.wait1(BAR(CF::B_VFULL + s), (last[s] / CF::VS) & 1, ROLE_DRAIN, CF::B_VFULL + s, true);
    } else if (warp == CF::CLOAD_WARP) {
      if constexpr (CF::C_RING) {
        // ============================================================ TMA: dense bias
        if (lane == 0) {
          tma_prefetch_desc(&tmC);
          int issued = 0;  // chunks issued, in ring order
          bool ok = true;
          for (int it = 0; ok && it < sch.n_it; ++it) {
            const int j = sch.hi_max - it;
            for (int cc = 0; cc < BN / CCHUNK; ++cc) {
              const int slot = issued % CF::CS;
              ok = wd.wait1(BAR(CF::B_CEMPTY + slot), ((issued / CF::CS) & 1) ^ 1, ROLE_CLOAD,
                            CF::B_CEMPTY + slot, false);
              if (!ok) break;
              mbar_arrive_expect_tx(BAR(CF::B_CFULL + slot), CCHUNK_BYTES);
              tma_load_3d(sbase + CF::C_OFF + slot * CCHUNK_BYTES, &tmC, j * BN + cc * CCHUNK,
                          sch.q_tile(0) * BM, p.c_shared ? 0 : sch.bh, BAR(CF::B_CFULL + slot));
              ++issued;
            }
          }
          // Chunks are issued consecutively: the last fill of each slot follows from the count.
          for (int s = 0; s < CF::CS && s < issued; ++s) {
            const int lastpos = s + ((issued - 1 - s) / CF::CS) * CF::CS;
            wd.wait1(BAR(CF::B_CFULL + s), (lastpos / CF::CS) & 1, ROLE_DRAIN, CF::B_CFULL + s, true);
          }
        }
      } else if constexpr (CF::KEY) {
        // ============================================================ per-key bias
        // The whole warp copies the 128 biases of each K/V tile (4 per lane, zero past
        // the last key) into the next slot of a small ring; every softmax warp that
        // visits the tile releases the slot.
        for (int it = 0; it < sch.n_it; ++it) {
          const int j = sch.hi_max - it;
          const int slot = it % CF::KB;
          if (!wd.wait(BAR(CF::B_KBEMPTY + slot), ((it / CF::KB) & 1) ^ 1, ROLE_CLOAD,
                       CF::B_KBEMPTY + slot))
            break;
          const int k0 = j * BN + 4 * lane;
          const float *src = p.ckey + static_cast<size_t>(sch.bh) * p.Nk;
          float4 v;
          v.x = (k0 + 0 < p.Nk) ? __ldg(src + k0 + 0) : 0.0f;
          v.y = (k0 + 1 < p.Nk) ? __ldg(src + k0 + 1) : 0.0f;
          v.z = (k0 + 2 < p.Nk) ? __ldg(src + k0 + 2) : 0.0f;
          v.w = (k0 + 3 < p.Nk) ? __ldg(src + k0 + 3) : 0.0f;
          // Stored in log2(e) units, the scale of the softmax's exponents.
          v.x *= LOG2E;
          v.y *= LOG2E;
          v.z *= LOG2E;
          v.w *= LOG2E;
          reinterpret_cast<float4 *>(smem + CF::KB_OFF + slot * BN * 4)[lane] = v;
          __syncwarp();
          mbar_arrive_elect(BAR(CF::B_KBFULL + slot));
        }
      }
    }
    __syncwarp();
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
  CUtensorMap tmO;  // O as stored by the CTA-pair kernel: 32-row boxes of 128 bytes
  KernelParams p;
  cudaStream_t stream;
};

// Number of query tiles one CTA owns (the host sizes the grid with it).
constexpr int q_tiles_per_cta(int bias, int d_v) {
  return (bias == BIAS_DENSE_TMA || bias == BIAS_DENSE_DIRECT || (bias == BIAS_NONE && d_v == 128)) ? 1 : 2;
}

template <int D, int DV, bool CAUSAL, int BIAS>
cudaError_t launch_attn(const LaunchArgs &a) {
  using CF = Cfg<D, DV, CAUSAL, BIAS>;
  auto kern = attn_fwd_kernel<D, DV, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  if constexpr (CF::SPLIT_REGS) {
    // The per-warpgroup register budgets are granted out of the registers the block is
    // launched with; refuse to launch if the compiled kernel was given fewer.
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * CF::THREADS < CF::REGS_NEEDED) return cudaErrorLaunchOutOfResources;
  }
  const unsigned grid = static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.ctas_per_head) *
                        static_cast<unsigned>(a.p.n_splits);
  e = launch_pdl(kern, dim3(grid), dim3(CF::THREADS), CF::SMEM_TOTAL, a.stream, a.tmQ, a.tmK, a.tmV, a.tmC, a.p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace eta

// Exact attention backward pass, tile by tile, for sm_103a.
//
// The gradients are those of O = softmax(S) V with S = scale Q K^T + C, for a loss
// gradient dO:
//     dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = dO_i . O_i,
//     dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
// The score and probability tiles are recomputed from Q, K and the forward's kept
// statistic LSE_i (P_ij = exp(S_ij - LSE_i)) instead of being stored, as the pages
// say of the tiled method's backward pass ("Compilers and kernels", section
// "FlashAttention rewrites the algorithm around IO", the paragraph after the
// recurrence).
//
// Three kernels, no atomics (the result is deterministic):
//   prep : a few lanes per query row: Lp_i = -LSE_i log2(e) (-inf for a row with no
//          allowed key and for the padding rows up to a whole tile, so that their p is 0)
//          and D_i = dO_i . O_i, into a caller workspace [BH][nq_tiles * 128] each.
//   dkdv : one CTA per (head, 128-key tile j). Keeps K_j and V_j in shared memory and
//          streams the query tiles i that see tile j (Q_i, dO_i and their Lp, D) through a
//          ring of slots. Per query tile, on the tensor cores with accumulators in tensor
//          memory: S^T = K_j Q_i^T and dP^T = V_j dO_i^T in two 128-column buffers that
//          swap roles every tile; the elementwise warps (thread = key row = tensor-memory
//          lane) form P^T = exp2(S^T scale log2e + Lp) and dS^T = P^T o (dP^T - D) in bf16,
//          packed over S^T; then dV_j += P^T dO_i and dK_j += dS^T Q_i, while S^T of the
//          next tile goes to the buffer dP^T left. At the end dV_j and scale dK_j are
//          written in fp32.
//   dq   : one CTA per (head, 128-query tile i). Keeps Q_i and dO_i, streams the K/V tiles
//          the tile sees: S = Q_i K_t^T, dP = dO_i V_t^T, dS = P o (dP - D) in bf16 over
//          S, dQ_i += dS K_t; at the end scale dQ_i in fp32. S is double-buffered, so
//          the next tile's S and dP run on the tensor cores while dS is formed.
// Warp roles: elementwise warps (16 in dkdv, 32 query columns each; 8 in dq, 64 key
// columns each; each thread owns one tensor-memory lane), the MMA warp (whole warp, one
// elected lane issues) and TMA producer warps. Every wait is bounded (the forward
// kernel's watchdog): a wait that runs out is recorded and the CTA drains and returns.
#pragma once

#include "attn_fwd_kernel.cuh"

namespace eta {

struct BwdParams {
  int BH;
  int Nq, Nk;
  int nq_tiles, nkv_tiles;
  int causal_off;     // Nk - Nq: query i may see keys j <= i + causal_off
  int nqp;            // nq_tiles * 128: row stride of Lp and D
  int head_group;     // heads per scheduling group (unit_of_block)
  float scale_log2;   // scale * log2(e)
  float scale;
  const float *Lp;    // [BH][nqp] -LSE * log2(e), -inf where p must be 0
  const float *Dd;    // [BH][nqp] D_i = dO_i . O_i
  const float *C;     // dense bias [BH][Nq][Nk] or null
  int c_shared;       // 1: C is one [Nq][Nk] array for every head (head index 0)
  const float *ckey;  // per-key bias [BH][Nk] or null
  float *dQ;          // [BH][Nq][d]
  float *dK;          // [BH][Nk][d]
  float *dV;          // [BH][Nk][d_v]
  unsigned int *status;
  unsigned long long timeout_ns;
};

using BwdWatchdog = WatchdogT<BwdParams>;

// ------------------------------------------------------------------------ prep
// O: [rows][DV] bf16 (out_f32 = 0) or fp32; dO: [rows][DV] bf16; LSE: [rows]. DV / 8 lanes
// (16 for d_v = 128, 8 for 64) share a row, each with one 16-byte load of dO (8 bf16)
// and of O (16 or 32 bytes).
template <int DV>
__global__ void __launch_bounds__(256)
    attn_bwd_prep_kernel(const void *__restrict__ O, int out_f32, const uint16_t *__restrict__ dO,
                         const float *__restrict__ LSE, int BH, int Nq, int nqp, float *Lp,
                         float *Dd) {
  constexpr int LPR = DV / 8;  // lanes per row
  grid_dep_wait();  // O and LSE may come from the forward kernel just before
  if (threadIdx.x == 0) grid_dep_launch();
  const long long prow = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / LPR;
  const int sub = threadIdx.x % LPR;
  const bool in = prow < static_cast<long long>(BH) * nqp;
  const int bh = in ? static_cast<int>(prow / nqp) : 0;
  const int i = in ? static_cast<int>(prow % nqp) : Nq;
  float acc = 0.0f;
  float lp = -INFINITY;
  if (i < Nq) {
    const long long row = static_cast<long long>(bh) * Nq + i;
    const uint4 g = __ldg(reinterpret_cast<const uint4 *>(dO + row * DV) + sub);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    float o[8];
    if (out_f32) {
      const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(O) + row * DV) + 2 * sub;
      const float4 a = __ldg(src), b = __ldg(src + 1);
      o[0] = a.x, o[1] = a.y, o[2] = a.z, o[3] = a.w, o[4] = b.x, o[5] = b.y, o[6] = b.z, o[7] = b.w;
    } else {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(O) + row * DV) + sub);
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[2 * k] = __uint_as_float(vw[k] << 16);
        o[2 * k + 1] = __uint_as_float(vw[k] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(gw[k] << 16), o[2 * k], acc);
      acc = fmaf(__uint_as_float(gw[k] & 0xFFFF0000u), o[2 * k + 1], acc);
    }
    const float lse = LSE[row];
    // -LSE log2(e), so that 2^(S scale log2(e) + lp) = exp(S scale - LSE); -inf (every p
    // is 0) for a row with no allowed key, as for a padding row.
    lp = lse == -INFINITY ? -INFINITY : -lse * LOG2E;
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (in && sub == 0) {
    Lp[prow] = lp;
    Dd[prow] = i < Nq ? acc : 0.0f;
  }
}

// ------------------------------------------------------------------------ shared pieces
// Bias sources of the backward kernels.
enum { BWD_BIAS_NONE = 0, BWD_BIAS_DENSE = 1, BWD_BIAS_KEY = 2 };

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int DV, bool CAUSAL, int BIAS>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "d must be 64 or 128");
  static_assert(DV == 64 || DV == 128, "d_v must be 64 or 128");
  static constexpr int Q_TILE = BM * D * 2;   // also a K tile (128 rows x d)
  static constexpr int DO_TILE = BM * DV * 2; // also a V tile (128 rows x d_v)
  static constexpr int LD_BYTES = 2 * BM * 4; // Lp and D of one query tile
  static constexpr int BUDGET = 224 * 1024;
  // dkdv: K_j, V_j resident; ring of (Q_i, dO_i, Lp_i, D_i) slots.
  static constexpr int A_SLOT = Q_TILE + DO_TILE + LD_BYTES;
  static constexpr int A_QS = cmin(3, (BUDGET - Q_TILE - DO_TILE) / A_SLOT);
  static constexpr int A_K_OFF = 0;
  static constexpr int A_V_OFF = Q_TILE;
  static constexpr int A_SLOT_OFF = Q_TILE + DO_TILE;
  static constexpr int A_BAR_OFF = A_SLOT_OFF + A_QS * A_SLOT;
  // dq: Q_i, dO_i resident; a ring of K_j tiles and a ring of V_j tiles. V_j is released
  // as soon as dP(j) is done, K_j only after dQ += dS K_j, so K gets the deeper ring.
  static constexpr int B_REST = BUDGET - Q_TILE - DO_TILE;
  static constexpr int B_KS = cmin(4, (B_REST - 2 * DO_TILE) / Q_TILE);
  static constexpr int B_VS = cmin(4, (B_REST - B_KS * Q_TILE) / DO_TILE);
  static constexpr int B_Q_OFF = 0;
  static constexpr int B_DO_OFF = Q_TILE;
  static constexpr int B_K_OFF = Q_TILE + DO_TILE;
  static constexpr int B_V_OFF = B_K_OFF + B_KS * Q_TILE;
  static constexpr int B_BAR_OFF = B_V_OFF + B_VS * DO_TILE;
  static_assert(A_QS >= 2 && B_KS >= 2 && B_VS >= 2, "need two ring slots");
  // dQ epilogue stages (8 warps x 32 rows x (d / 2 + 4) floats) reuse the K ring.
  static_assert(8 * 32 * (D / 2 + 4) * 4 <= B_KS * Q_TILE,
                "dQ epilogue stage larger than the K ring it reuses");
  static_assert(A_SLOT % 1024 == 0, "slots keep 1024-byte alignment");

  // barriers (the same layout serves both kernels; RING = ring slots; dq's K ring uses
  // FULL/EMPTY, its V ring VFULL/VEMPTY)
  static constexpr int RING = cmin(4, A_QS > B_KS ? A_QS : B_KS);
  static constexpr int BAR_FIXED = 0;               // K_j/V_j (dkdv) or Q_i/dO_i (dq)
  static constexpr int BAR_FULL = 1;                // ring slot filled
  static constexpr int BAR_EMPTY = BAR_FULL + RING; // ring slot released
  static constexpr int BAR_SFULL = BAR_EMPTY + RING;  // [2]: S and dP of a half ready
  static constexpr int BAR_PFULL = BAR_SFULL + 2;     // [2]: its bf16 P and dS written (8 warps)
  static constexpr int BAR_ACC = BAR_PFULL + 2;
  static constexpr int BAR_DRAIN = BAR_ACC + 1;
  static constexpr int BAR_DPFULL = BAR_DRAIN + 1;  // dq: dP of a key tile ready
  static constexpr int BAR_DPFREE = BAR_DPFULL + 1;  // dq: dP read into registers (8 warps)
  static constexpr int BAR_VFULL = BAR_DPFREE + 1;   // dq: [B_VS]
  static constexpr int BAR_VEMPTY = BAR_VFULL + 4;   // dq: [B_VS]
  static constexpr int NUM_BARS = BAR_VEMPTY + 4;
  static constexpr int BAR_BYTES = NUM_BARS * 8;
  static constexpr int TAIL_BYTES = BAR_BYTES + 8;  // + tensor-memory address + abort flag
  static constexpr int A_SMEM = A_BAR_OFF + TAIL_BYTES + 1024;
  static constexpr int B_SMEM = B_BAR_OFF + TAIL_BYTES + 1024;
  static_assert(A_SMEM <= 232448 && B_SMEM <= 232448, "shared memory over the per-CTA limit");
  // At least 120 KB each, so one CTA holds an SM (the CTA allocates all tensor memory).
  static constexpr int A_SMEM_TOTAL = A_SMEM > 120 * 1024 ? A_SMEM : 120 * 1024;
  static constexpr int B_SMEM_TOTAL = B_SMEM > 120 * 1024 ? B_SMEM : 120 * 1024;

  // tensor memory (dkdv): the two score buffers at S_COL and S_COL + 128, then dV and dK
  static constexpr int S_COL = 0;
  static constexpr int ACC0_COL = 256;        // dV (dkdv) or dQ (dq)
  static constexpr int ACC1_COL = 256 + DV;   // dK (dkdv)
  static constexpr int TMEM_COLS = 512;

  static constexpr int NUM_WARPS = 12;  // dq: 8 elementwise warps, MMA, two copy warps
  static constexpr int THREADS = 32 * NUM_WARPS;
  static constexpr int MMA_WARP = 8;
  static constexpr int LOAD_WARP = 9;
  // dkdv: 16 elementwise warps (four per tensor-memory lane quarter, 32 query columns
  // each), the MMA warp and the copy warp.
  static constexpr int A_EW_WARPS = 16;
  static constexpr int A_THREADS = 32 * (A_EW_WARPS + 2);
  static constexpr int A_MMA_WARP = A_EW_WARPS;
  static constexpr int A_LOAD_WARP = A_EW_WARPS + 1;
  // The dK/dV epilogue stages (16 warps x 32 rows x (width / 2 + 4) floats) reuse the K, V
  // and ring memory from offset 0.
  static_assert(16 * 32 * ((D > DV ? D : DV) / 2 + 4) * 4 <= A_SLOT_OFF + A_QS * A_SLOT,
                "dK/dV epilogue stage larger than the memory it reuses");

  static constexpr uint32_t IDESC_SS = idesc_bf16_f32(128, 128, false);     // full-width S, dP
  static constexpr uint32_t IDESC_NV = idesc_bf16_f32(128, DV, true);       // dV += P^T dO
  static constexpr uint32_t IDESC_ND = idesc_bf16_f32(128, D, true);        // dK, dQ
};

// K-major operand step ks (16 elements of the contraction) inside 128-row boxes of 64
// columns: 32 bytes within a 128-byte row, a new box every 4 steps.
__device__ __forceinline__ uint32_t kmajor_step(int ks) {
  return static_cast<uint32_t>(((ks / 4) * SW_CHUNK_BYTES + (ks % 4) * 32) >> 4);
}
// MN-major operand (contraction along rows): step ks of 16 rows.
__device__ __forceinline__ uint32_t mn_step(int ks) { return static_cast<uint32_t>((ks * 16 * 128) >> 4); }
// Loads a 32-column chunk of two tensor-memory matrices.
__device__ __forceinline__ void ld_pair(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                        uint32_t (&b)[32]) {
  tmem_ld32(ta, a);
  tmem_ld32(tb, b);
  tmem_wait_ld(a);
  tmem_wait_ld(b);
}

// Writes accumulator columns [c0, c0 + N) of this warp's 32 rows (its tensor-memory lanes),
// times `mul`, to global memory through a per-warp shared-memory stage of 32 rows x (N + 4)
// floats (the padding puts the rows of a column in different banks). A thread owns a row
// in tensor memory; from the stage, N / 4 lanes write each row, so every store instruction
// writes whole rows instead of one 16-byte piece per row. `grow0` is the global address of
// the warp's first row (column 0), `rows_ok` how many of its rows exist.
template <int N>
__device__ __forceinline__ void store_acc_staged(uint32_t tcol, int c0, float mul, float *grow0,
                                                 size_t row_stride, int rows_ok, float *stage) {
  constexpr int P = N + 4;
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int cc = 0; cc < N; cc += 32) {
    uint32_t r[32];
    tmem_ld32(tcol + c0 + cc, r);
    tmem_wait_ld(r);
    float4 *srow = reinterpret_cast<float4 *>(stage + lane * P + cc);
#pragma unroll
    for (int v = 0; v < 8; ++v)
      srow[v] = make_float4(__uint_as_float(r[4 * v]) * mul, __uint_as_float(r[4 * v + 1]) * mul,
                            __uint_as_float(r[4 * v + 2]) * mul, __uint_as_float(r[4 * v + 3]) * mul);
  }
  __syncwarp();
  constexpr int LPR = N / 4;     // lanes per row
  constexpr int RPS = 32 / LPR;  // rows per store instruction
  const int sub = lane % LPR;
#pragma unroll 4
  for (int r0 = 0; r0 < 32; r0 += RPS) {
    const int row = r0 + lane / LPR;
    if (row < rows_ok)
      *reinterpret_cast<float4 *>(grow0 + static_cast<size_t>(row) * row_stride + c0 + 4 * sub) =
          *reinterpret_cast<const float4 *>(stage + row * P + 4 * sub);
  }
  __syncwarp();
}

__device__ __forceinline__ void store_zero_row(int n, float *dst, bool row_ok) {
  if (!row_ok) return;
  float4 *d4 = reinterpret_cast<float4 *>(dst);
  for (int v = 0; v < n / 4; ++v) d4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------------ dK, dV
template <int D, int DV, bool CAUSAL, int BIAS>
__global__ void __launch_bounds__(BwdCfg<D, DV, CAUSAL, BIAS>::A_THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ BwdParams p) {
  using CF = BwdCfg<D, DV, CAUSAL, BIAS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + CF::A_BAR_OFF;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + CF::A_BAR_OFF + CF::BAR_BYTES);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::A_BAR_OFF + CF::BAR_BYTES + 4);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // This CTA: head bh, key tile j; the query tiles that see it are i_lo .. nq_tiles - 1
  // (tiles t = 0 .. n_it - 1).
  // Units of a head: key tiles from the first (seen by the most queries) on.
  int bh, j;
  unit_of_block(blockIdx.x, p.BH, p.nkv_tiles, p.head_group, &bh, &j);
  int i_lo = 0;
  if (CAUSAL) {
    // The first query that sees key 128 j is q0 = 128 j - (Nk - Nq); none when q0 >= Nq.
    const int q0 = j * BN - p.causal_off;
    i_lo = q0 >= p.Nq ? p.nq_tiles : (q0 <= 0 ? 0 : q0 / BM);
  }
  const int n_it = p.nq_tiles - i_lo;
  BwdWatchdog wd{sbase + CF::A_BAR_OFF + CF::BAR_BYTES + 4, p};
#ifdef ETA_PHASE_TRACE
  int trace_n = 0;
#endif

  if (threadIdx.x == 0) {
    mbar_init(BAR(CF::BAR_FIXED), 1);
    for (int s = 0; s < CF::A_QS; ++s) {
      mbar_init(BAR(CF::BAR_FULL + s), 1);
      mbar_init(BAR(CF::BAR_EMPTY + s), 1);
    }
    mbar_init(BAR(CF::BAR_SFULL), 1);
    mbar_init(BAR(CF::BAR_DPFULL), 1);
    mbar_init(BAR(CF::BAR_DPFREE), CF::A_EW_WARPS);
    mbar_init(BAR(CF::BAR_PFULL), CF::A_EW_WARPS);      // dS^T(t) written
    mbar_init(BAR(CF::BAR_PFULL + 1), CF::A_EW_WARPS);  // P^T(t) written
    mbar_init(BAR(CF::BAR_ACC), 1);
    mbar_init(BAR(CF::BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == CF::A_MMA_WARP) {
    tmem_alloc(smem_u32(tmem_ptr), CF::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;
  // The kernel before this one on the stream is the pre-pass (attn_bwd), which waited for
  // everything before it: Q, K, V, dO and the biases are final, and only the row statistics
  // it writes are not. So the copy warp waits for it (programmatic launch) just before its
  // first copy of the statistics, and only then lets the next kernel start launching (the
  // dQ kernel relies on that order).

  if (warp < CF::A_EW_WARPS) {
    // ============================================================ elementwise
    // Tile t: S^T(t) in buffer t & 1, dP^T(t) in the other. Warp g = warp / 4 owns queries
    // [32 g, 32 g + 32) of the tile (columns of both buffers) for its 32 keys (tensor-memory
    // lanes). It forms P^T from S^T while dP^T is still being computed, then reads dP^T,
    // frees its buffer for S^T(t+1), and writes dS^T. P^T and dS^T go packed (two bf16 per
    // 32-bit column) over the columns of S^T this warp read: P^T at [32 g, 32 g + 16), dS^T
    // at [32 g + 16, 32 g + 32).
    const int g = warp / 4;
    const int r = threadIdx.x % 128;
    const int key = j * BN + r;
    const bool key_ok = key < p.Nk;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const float sl2 = p.scale_log2;
    // Per-key bias of this row, log2-scaled (-inf for a padded key: its p is 0). Rows past
    // the last key need no mask: their K and V rows are zero-filled, so they only produce
    // dK and dV rows that are never stored.
    float kb = 0.0f;
    if (BIAS == BWD_BIAS_KEY) kb = key_ok ? p.ckey[static_cast<size_t>(bh) * p.Nk + key] * LOG2E : 0.0f;
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      const int i = i_lo + t;
      const int slot = t % CF::A_QS;
      const int c0 = 32 * g;  // query offset within the tile
      const uint32_t t_s = tmem + lane_off + CF::S_COL + 128 * (t & 1) + c0;
      const uint32_t t_dp = tmem + lane_off + CF::S_COL + 128 * ((t + 1) & 1) + c0;
      const float *Ls = reinterpret_cast<const float *>(smem + CF::A_SLOT_OFF + slot * CF::A_SLOT +
                                                        CF::Q_TILE + CF::DO_TILE) + c0;
      const float *Ds = Ls + BM;
      ok = wd.wait(BAR(CF::BAR_SFULL), t & 1, ROLE_SOFTMAX, CF::BAR_SFULL);
      if (!ok) break;
      tc_fence_after();
      ETA_TRACE(40);
      // p = 2^x, x = scale S log2(e) + (bias log2(e) - LSE log2(e)) = log2 of exp(S_ij - LSE_i),
      // in pairs of columns.
      float pv[32];
      {
        uint32_t sr[32];
        tmem_ld32(t_s, sr);
        tmem_wait_ld(sr);
        // Keys past the causal limit of this chunk's first query need the elementwise test.
        if (CAUSAL && (j * BN + BN - 1 > i * BM + c0 + p.causal_off)) {
          const int lim = i * BM + c0 + p.causal_off - key;  // column c is forbidden when c < -lim
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c + lim < 0) sr[c] = __float_as_uint(-INFINITY);
        }
        uint32_t pp[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 L4 = *reinterpret_cast<const float4 *>(Ls + c);  // -LSE log2(e)
          float b[4] = {L4.x, L4.y, L4.z, L4.w};
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (BIAS == BWD_BIAS_KEY) b[v] += kb;
            if (BIAS == BWD_BIAS_DENSE) {
              const int q = i * BM + c0 + c + v;
              b[v] += (key_ok && q < p.Nq) ? __ldg(p.C + (static_cast<size_t>(p.c_shared ? 0 : bh) * p.Nq + q) * p.Nk + key) * LOG2E
                                           : 0.0f;
            }
          }
          float x[4];
          fma2(x[0], x[1], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), sl2, sl2, b[0], b[1]);
          fma2(x[2], x[3], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]), sl2, sl2, b[2], b[3]);
#pragma unroll
          for (int v = 0; v < 4; ++v) pv[c + v] = ex2_approx(x[v]);
          pp[c / 2] = pack_bf16(pv[c], pv[c + 1]);
          pp[c / 2 + 1] = pack_bf16(pv[c + 2], pv[c + 3]);
        }
        tmem_st16(t_s, pp);
      }
      // P^T(t) is written: dV += P^T dO may start while dS^T is formed.
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(BAR(CF::BAR_PFULL + 1));
      ETA_TRACE(41);
      ok = wd.wait(BAR(CF::BAR_DPFULL), t & 1, ROLE_SOFTMAX, CF::BAR_DPFULL);
      if (!ok) break;
      tc_fence_after();
      uint32_t dr[32];
      tmem_ld32(t_dp, dr);
      tmem_wait_ld(dr);
      // dP^T(t) is in registers: its buffer may take S^T(t+1).
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(BAR(CF::BAR_DPFREE));
      ETA_TRACE(42);
      uint32_t dd[16];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 D4 = *reinterpret_cast<const float4 *>(Ds + c);
        // dS = p (dP - D), in pairs of columns.
        float tq[4], dv[4];
        sub2(tq[0], tq[1], __uint_as_float(dr[c]), __uint_as_float(dr[c + 1]), D4.x, D4.y);
        sub2(tq[2], tq[3], __uint_as_float(dr[c + 2]), __uint_as_float(dr[c + 3]), D4.z, D4.w);
        mul2(dv[0], dv[1], pv[c], pv[c + 1], tq[0], tq[1]);
        mul2(dv[2], dv[3], pv[c + 2], pv[c + 3], tq[2], tq[3]);
        dd[c / 2] = pack_bf16(dv[0], dv[1]);
        dd[c / 2 + 1] = pack_bf16(dv[2], dv[3]);
      }
      tmem_st16(t_s + 16, dd);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(BAR(CF::BAR_PFULL));
      ETA_TRACE(43);
    }
    // ---------------------------------------------------------- epilogue: dV, scale dK
    // Warps g = 0, 1 store halves of dV, warps g = 2, 3 halves of dK.
    const bool is_dv = g < 2;
    const int half = g & 1;
    if (ok && n_it > 0) {
      ok = wd.wait(BAR(CF::BAR_ACC), 0, ROLE_SOFTMAX, CF::BAR_ACC);
      if (ok) {
        tc_fence_after();
        // Every product has completed and every copy landed: per-warp stages over the K, V
        // and ring memory.
        float *stage = reinterpret_cast<float *>(smem) + warp * 32 * (cmax(D, DV) / 2 + 4);
        const int row0 = j * BN + 32 * (warp % 4);  // the warp's first key
        const int rows_ok = p.Nk - row0 < 32 ? (p.Nk - row0 > 0 ? p.Nk - row0 : 0) : 32;
        const size_t base = static_cast<size_t>(bh) * p.Nk + row0;
        if (is_dv)
          store_acc_staged<DV / 2>(tmem + lane_off + CF::ACC0_COL, half * DV / 2, 1.0f, p.dV + base * DV, DV,
                                   rows_ok, stage);
        else
          store_acc_staged<D / 2>(tmem + lane_off + CF::ACC1_COL, half * D / 2, p.scale, p.dK + base * D, D,
                                  rows_ok, stage);
      }
    } else if (ok) {
      if (is_dv)
        store_zero_row(DV / 2, p.dV + (static_cast<size_t>(bh) * p.Nk + (key_ok ? key : 0)) * DV + half * DV / 2, key_ok);
      else
        store_zero_row(D / 2, p.dK + (static_cast<size_t>(bh) * p.Nk + (key_ok ? key : 0)) * D + half * D / 2, key_ok);
    }
  } else if (warp == CF::A_MMA_WARP) {
    // ============================================================ MMA issue
    // Order on the tensor cores: S^T(0), dP^T(0); then per tile t: S^T(t+1) (once dP^T(t)
    // is in registers), dV += P^T(t) dO_t (once P^T is written), dK += dS^T(t) Q_t (once
    // dS^T is written), dP^T(t+1) into the buffer they came from.
    bool ok = n_it == 0 || wd.wait(BAR(CF::BAR_FIXED), 0, ROLE_MMA, CF::BAR_FIXED);
    const uint64_t k_desc = smem_desc(sbase + CF::A_K_OFF, 16, 1024);
    const uint64_t v_desc = smem_desc(sbase + CF::A_V_OFF, 16, 1024);
    auto slot_addr = [&](int t) -> uint32_t { return sbase + CF::A_SLOT_OFF + (t % CF::A_QS) * CF::A_SLOT; };
    // S^T(t) = K Q_t^T into buffer t & 1, after waiting for tile t's copies.
    auto issue_s = [&](int t) -> bool {
      const int slot = t % CF::A_QS;
      if (!wd.wait(BAR(CF::BAR_FULL + slot), (t / CF::A_QS) & 1, ROLE_MMA, CF::BAR_FULL + slot)) return false;
      tc_fence_after();
      const uint64_t q_desc = smem_desc(slot_addr(t), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss_elect(tmem + CF::S_COL + 128 * (t & 1), k_desc + kmajor_step(ks), q_desc + kmajor_step(ks),
                     CF::IDESC_SS, ks > 0 ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_SFULL));
      return true;
    };
    // dP^T(t) = V dO_t^T into the other buffer (tile t's copies have landed).
    auto issue_dp = [&](int t) {
      const uint64_t do_desc = smem_desc(slot_addr(t) + CF::Q_TILE, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < DV / 16; ++ks)
        mma_ss_elect(tmem + CF::S_COL + 128 * ((t + 1) & 1), v_desc + kmajor_step(ks), do_desc + kmajor_step(ks),
                     CF::IDESC_SS, ks > 0 ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_DPFULL));
    };
    if (ok && n_it > 0 && (ok = issue_s(0))) issue_dp(0);
    for (int t = 0; ok && t < n_it; ++t) {
      ETA_TRACE(50);
      if (t + 1 < n_it) {
        if (!(ok = wd.wait(BAR(CF::BAR_DPFREE), t & 1, ROLE_MMA, CF::BAR_DPFREE))) break;
        tc_fence_after();
        if (!(ok = issue_s(t + 1))) break;
      }
      ETA_TRACE(51);
      // dV_j += P^T dO_t, then dK_j += dS^T Q_t (A from tensor memory: step ks covers
      // queries [16 ks, 16 ks + 16), packed by warp group ks / 2; B MN-major over the
      // tile's rows), each once its operand is written.
      ok = wd.wait(BAR(CF::BAR_PFULL + 1), t & 1, ROLE_MMA, CF::BAR_PFULL + 1);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sb = tmem + CF::S_COL + 128 * (t & 1);
      const uint64_t do_mn = smem_desc(slot_addr(t) + CF::Q_TILE, SW_CHUNK_BYTES, 1024);
      const uint64_t q_mn = smem_desc(slot_addr(t), SW_CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < BM / 16; ++ks)
        mma_ts_elect(tmem + CF::ACC0_COL, sb + 32 * (ks / 2) + 8 * (ks % 2), do_mn + mn_step(ks),
                     CF::IDESC_NV, (t > 0 || ks > 0) ? 1u : 0u);
      ok = wd.wait(BAR(CF::BAR_PFULL), t & 1, ROLE_MMA, CF::BAR_PFULL);
      if (!ok) break;
      tc_fence_after();
      ETA_TRACE(52);
#pragma unroll
      for (int ks = 0; ks < BM / 16; ++ks)
        mma_ts_elect(tmem + CF::ACC1_COL, sb + 16 + 32 * (ks / 2) + 8 * (ks % 2), q_mn + mn_step(ks),
                     CF::IDESC_ND, (t > 0 || ks > 0) ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_EMPTY + (t % CF::A_QS)));
      if (t + 1 < n_it) issue_dp(t + 1);
    }
    if (ok && n_it > 0) mma_commit_elect(BAR(CF::BAR_ACC));
    mma_commit_elect(BAR(CF::BAR_DRAIN));
    wd.drain(BAR(CF::BAR_DRAIN), 0, CF::BAR_DRAIN);
  } else if (warp == CF::A_LOAD_WARP && lane == 0) {
    // ============================================================ TMA producer
    if (n_it > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(BAR(CF::BAR_FIXED), CF::Q_TILE + CF::DO_TILE);
      for (int kc = 0; kc < D / SW_CHUNK; ++kc)
        tma_load_3d(sbase + CF::A_K_OFF + kc * SW_CHUNK_BYTES, &tmK, kc * SW_CHUNK, j * BN, bh,
                    BAR(CF::BAR_FIXED));
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
        tma_load_3d(sbase + CF::A_V_OFF + kc * SW_CHUNK_BYTES, &tmV, kc * SW_CHUNK, j * BN, bh,
                    BAR(CF::BAR_FIXED));
    }
    int issued = 0;
    bool waited = false;
    for (int it = 0; it < n_it; ++it) {
      const int i = i_lo + it;
      const int slot = it % CF::A_QS;
      if (!wd.wait1(BAR(CF::BAR_EMPTY + slot), ((it / CF::A_QS) & 1) ^ 1, ROLE_LOAD,
                    CF::BAR_EMPTY + slot, false))
        break;
      const uint32_t sl = sbase + CF::A_SLOT_OFF + slot * CF::A_SLOT;
      ETA_TRACE(60);
      mbar_arrive_expect_tx(BAR(CF::BAR_FULL + slot), CF::Q_TILE + CF::DO_TILE + CF::LD_BYTES);
      for (int kc = 0; kc < D / SW_CHUNK; ++kc)
        tma_load_3d(sl + kc * SW_CHUNK_BYTES, &tmQ, kc * SW_CHUNK, i * BM, bh, BAR(CF::BAR_FULL + slot));
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
        tma_load_3d(sl + CF::Q_TILE + kc * SW_CHUNK_BYTES, &tmdO, kc * SW_CHUNK, i * BM, bh,
                    BAR(CF::BAR_FULL + slot));
      const size_t lrow = static_cast<size_t>(bh) * p.nqp + static_cast<size_t>(i) * BM;
      if (!waited) {
        grid_dep_wait();
        grid_dep_launch();
        waited = true;
      }
      bulk_load(sl + CF::Q_TILE + CF::DO_TILE, p.Lp + lrow, BM * 4, BAR(CF::BAR_FULL + slot));
      bulk_load(sl + CF::Q_TILE + CF::DO_TILE + BM * 4, p.Dd + lrow, BM * 4, BAR(CF::BAR_FULL + slot));
      ++issued;
    }
    if (!waited) {  // no query tile (or an abort): the block still ends after the pre-pass
      grid_dep_wait();
      grid_dep_launch();
    }
    // The block the hardware will likely start next is about one wave ahead: warm L2 with
    // its K and V tiles (each unit's own) so that its first products do not wait on HBM.
    const unsigned next = blockIdx.x + nsmid();
    if (next < gridDim.x) {
      int nbh, nj;
      unit_of_block(next, p.BH, p.nkv_tiles, p.head_group, &nbh, &nj);
      for (int kc = 0; kc < D / SW_CHUNK; ++kc) tma_prefetch_l2_3d(&tmK, kc * SW_CHUNK, nj * BN, nbh);
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc) tma_prefetch_l2_3d(&tmV, kc * SW_CHUNK, nj * BN, nbh);
    }
    // Copies still in flight land before the CTA exits.
    if (n_it > 0) wd.wait1(BAR(CF::BAR_FIXED), 0, ROLE_DRAIN, CF::BAR_FIXED, true);
    for (int s = 0; s < CF::A_QS && s < issued; ++s) {
      const int lastpos = s + ((issued - 1 - s) / CF::A_QS) * CF::A_QS;
      wd.wait1(BAR(CF::BAR_FULL + s), (lastpos / CF::A_QS) & 1, ROLE_DRAIN, CF::BAR_FULL + s, true);
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == CF::A_MMA_WARP) tmem_dealloc(tmem, CF::TMEM_COLS);
}

// ------------------------------------------------------------------------ dQ
// Tensor memory of the dQ kernel: two full-width score buffers S_0, S_1 (128 columns
// each; dS is packed over the one it came from), one dP buffer and the dQ accumulator.
// While the elementwise warps turn S(t), dP(t) into dS(t), the tensor cores compute
// S(t+1) into the other buffer and, once dP(t) has been read into registers, dP(t+1).
constexpr int DQ_S0_COL = 0;
constexpr int DQ_DP_COL = 256;
constexpr int DQ_ACC_COL = 384;

template <int D, int DV, bool CAUSAL, int BIAS>
__global__ void __launch_bounds__(BwdCfg<D, DV, CAUSAL, BIAS>::THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ BwdParams p) {
  using CF = BwdCfg<D, DV, CAUSAL, BIAS>;
  static_assert(DQ_ACC_COL + D <= CF::TMEM_COLS, "dQ accumulator past the tensor memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + CF::B_BAR_OFF;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + CF::B_BAR_OFF + CF::BAR_BYTES);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + CF::B_BAR_OFF + CF::BAR_BYTES + 4);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Barriers of this kernel: SFULL[2] per score buffer, DSFULL[2] per score buffer (dS(t)
  // written by the 8 elementwise warps), DPFULL, DPFREE (dP(t) read into registers by the
  // 8 elementwise warps). DSFULL is per buffer because warps can finish a tile at
  // different times: a fast warp's arrival for tile t+1 must not complete tile t's phase.
  // A warp cannot get two tiles ahead: S(t+2) is issued only after DSFULL(t).
  const int B_DPFREE = CF::BAR_DPFREE;
  const int B_DSFULL = CF::BAR_PFULL;  // [2]

  // This CTA: head bh, query tile i; it visits key tiles 0 .. hi (none when hi < 0).
  // Units of a head: query tiles from the last (sees the most keys) down.
  int bh, ri;
  unit_of_block(blockIdx.x, p.BH, p.nq_tiles, p.head_group, &bh, &ri);
  const int i = p.nq_tiles - 1 - ri;
  int hi = p.nkv_tiles - 1;
  if (CAUSAL) hi = cmin(floor_div(cmin(i * BM + BM - 1, p.Nq - 1) + p.causal_off, BN), hi);
  const int n_it = hi + 1 > 0 ? hi + 1 : 0;
  BwdWatchdog wd{sbase + CF::B_BAR_OFF + CF::BAR_BYTES + 4, p};
#ifdef ETA_PHASE_TRACE
  int trace_n = 0;
#endif
  ETA_TRACE(90);

  if (threadIdx.x == 0) {
    mbar_init(BAR(CF::BAR_FIXED), 1);
    for (int s = 0; s < CF::B_KS; ++s) {
      mbar_init(BAR(CF::BAR_FULL + s), 1);
      mbar_init(BAR(CF::BAR_EMPTY + s), 1);
    }
    for (int s = 0; s < CF::B_VS; ++s) {
      mbar_init(BAR(CF::BAR_VFULL + s), 1);
      mbar_init(BAR(CF::BAR_VEMPTY + s), 1);
    }
    mbar_init(BAR(CF::BAR_SFULL + 0), 1);
    mbar_init(BAR(CF::BAR_SFULL + 1), 1);
    mbar_init(BAR(B_DSFULL + 0), 8);
    mbar_init(BAR(B_DSFULL + 1), 8);
    mbar_init(BAR(B_DPFREE), 8);
    mbar_init(BAR(CF::BAR_DPFULL), 1);
    mbar_init(BAR(CF::BAR_ACC), 1);
    mbar_init(BAR(CF::BAR_DRAIN), 1);
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
  // Set-up done. The kernel before this one on the stream is the dK/dV kernel (launch_bwd),
  // which writes nothing this kernel reads and lets it launch only once each of its blocks
  // has waited for the pre-pass: the row statistics are complete by now. So blocks start
  // beside the dK/dV kernel's last wave without waiting for it; the grid's last block does
  // wait, so that this kernel completes only after that one (the next kernel on the stream
  // waits for this one alone). The statistics are read through L2 (__ldcg).
  if (blockIdx.x == gridDim.x - 1) grid_dep_wait();
  if (threadIdx.x == 0) grid_dep_launch();

  if (warp < 8) {
    // ============================================================ elementwise
    const int g = warp / 4;  // columns (keys) [64 g, 64 g + 64) of each key tile
    const int r = threadIdx.x % 128;
    const int q = i * BM + r;
    const bool q_ok = q < p.Nq;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp % 4)) << 16;
    const size_t lrow = static_cast<size_t>(bh) * p.nqp + static_cast<size_t>(q);
    const float nL = __ldcg(p.Lp + lrow);  // -LSE log2(e); -inf for padding rows and rows with no allowed key
    const float Dr = __ldcg(p.Dd + lrow);
    const int lim = CAUSAL ? q + p.causal_off : INT_MAX;  // last key this row may see
    bool ok = true;
    for (int t = 0; t < n_it; ++t) {
      const int b = t & 1;
      ok = wd.wait(BAR(CF::BAR_SFULL + b), (t >> 1) & 1, ROLE_SOFTMAX, CF::BAR_SFULL + b) &&
           wd.wait(BAR(CF::BAR_DPFULL), t & 1, ROLE_SOFTMAX, CF::BAR_DPFULL);
      if (!ok) break;
      tc_fence_after();
      ETA_TRACE(70);
      // dP(t) into registers first: its buffer is then free for dP(t+1).
      uint32_t da[32], db[32];
      ld_pair(tmem + lane_off + DQ_DP_COL + 64 * g, tmem + lane_off + DQ_DP_COL + 64 * g + 32, da, db);
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(BAR(B_DPFREE));
      ETA_TRACE(71);
      const uint32_t t_s = tmem + lane_off + DQ_S0_COL + 128 * b + 64 * g;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t sr[32];
        tmem_ld32(t_s + 32 * h, sr);
        tmem_wait_ld(sr);
        const int k0 = t * BN + 64 * g + 32 * h;  // first key of these 32 columns
        if ((CAUSAL && (k0 + 31 > i * BM + p.causal_off)) || (k0 + 31 >= p.Nk)) {
          const int last = cmin(lim, p.Nk - 1) - k0;  // column c is allowed when c <= last
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c > last) sr[c] = __float_as_uint(-INFINITY);
        }
        uint32_t dd[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float dv2[2];
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const int key = k0 + c + v;
            float x = fmaf(__uint_as_float(sr[c + v]), p.scale_log2, nL);
            if (BIAS == BWD_BIAS_KEY)
              x += key < p.Nk ? __ldg(p.ckey + static_cast<size_t>(bh) * p.Nk + key) * LOG2E : 0.0f;
            if (BIAS == BWD_BIAS_DENSE)
              x += (q_ok && key < p.Nk) ? __ldg(p.C + (static_cast<size_t>(p.c_shared ? 0 : bh) * p.Nq + q) * p.Nk + key) * LOG2E
                                        : 0.0f;
            const float pr = ex2_approx(x);
            const float dpv = __uint_as_float(h == 0 ? da[c + v] : db[c + v]);
            dv2[v] = pr * (dpv - Dr);
          }
          dd[c / 2] = pack_bf16(dv2[0], dv2[1]);
        }
        // Packed dS over the S columns this warp has read: keys [64 g + 32 h, +32) at
        // 32-bit columns [64 g + 16 h, +16).
        tmem_st16(t_s + 16 * h, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(BAR(B_DSFULL + b));
      ETA_TRACE(73);
    }
    // ---------------------------------------------------------- epilogue: scale dQ
    float *dq_row = p.dQ + (static_cast<size_t>(bh) * p.Nq + (q_ok ? q : 0)) * D;
    if (ok && n_it > 0) {
      ok = wd.wait(BAR(CF::BAR_ACC), 0, ROLE_SOFTMAX, CF::BAR_ACC);
      if (ok) {
        tc_fence_after();
        // The K ring is idle now (every product has completed): per-warp stages there.
        float *stage = reinterpret_cast<float *>(smem + CF::B_K_OFF) + warp * 32 * (D / 2 + 4);
        const int row0 = i * BM + 32 * (warp % 4);  // the warp's first query
        const int rows_ok = p.Nq - row0 < 32 ? (p.Nq - row0 > 0 ? p.Nq - row0 : 0) : 32;
        store_acc_staged<D / 2>(tmem + lane_off + DQ_ACC_COL, g * D / 2, p.scale,
                                p.dQ + (static_cast<size_t>(bh) * p.Nq + row0) * D, D, rows_ok, stage);
      }
      ETA_TRACE(92);
    } else if (ok) {
      store_zero_row(D / 2, dq_row + g * D / 2, q_ok);
    }
  } else if (warp == CF::MMA_WARP) {
    // ============================================================ MMA issue
    bool ok = n_it == 0 || wd.wait(BAR(CF::BAR_FIXED), 0, ROLE_MMA, CF::BAR_FIXED);
    const uint64_t q_desc = smem_desc(sbase + CF::B_Q_OFF, 16, 1024);
    const uint64_t do_desc = smem_desc(sbase + CF::B_DO_OFF, 16, 1024);
    auto k_addr = [&](int t) -> uint32_t { return sbase + CF::B_K_OFF + (t % CF::B_KS) * CF::Q_TILE; };
    // S(t) = Q_i K_t^T into buffer t & 1, after waiting for the copy of K_t.
    auto issue_s = [&](int t) -> bool {
      const int slot = t % CF::B_KS;
      if (!wd.wait(BAR(CF::BAR_FULL + slot), (t / CF::B_KS) & 1, ROLE_MMA, CF::BAR_FULL + slot)) return false;
      tc_fence_after();
      const uint64_t k_desc = smem_desc(k_addr(t), 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_ss_elect(tmem + DQ_S0_COL + 128 * (t & 1), q_desc + kmajor_step(ks), k_desc + kmajor_step(ks),
                     CF::IDESC_SS, ks > 0 ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_SFULL + (t & 1)));
      return true;
    };
    // dP(t) = dO_i V_t^T after waiting for the copy of V_t; V_t's slot is released when
    // the product is done.
    auto issue_dp = [&](int t) -> bool {
      const int slot = t % CF::B_VS;
      if (!wd.wait(BAR(CF::BAR_VFULL + slot), (t / CF::B_VS) & 1, ROLE_MMA, CF::BAR_VFULL + slot)) return false;
      tc_fence_after();
      const uint64_t v_desc = smem_desc(sbase + CF::B_V_OFF + slot * CF::DO_TILE, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < DV / 16; ++ks)
        mma_ss_elect(tmem + DQ_DP_COL, do_desc + kmajor_step(ks), v_desc + kmajor_step(ks), CF::IDESC_SS,
                     ks > 0 ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_DPFULL));
      mma_commit_elect(BAR(CF::BAR_VEMPTY + slot));
      return true;
    };
    if (ok && n_it > 0) ok = issue_s(0) && issue_dp(0);
    for (int t = 0; ok && t < n_it; ++t) {
      ETA_TRACE(80);
      if (t + 1 < n_it) {
        // S(t+1) into the other buffer (last read by dQ(t-1), issued before it).
        if (!(ok = issue_s(t + 1))) break;
        ETA_TRACE(81);
        // dP(t+1) once the elementwise warps hold dP(t) in registers.
        if (!(ok = wd.wait(BAR(B_DPFREE), t & 1, ROLE_MMA, B_DPFREE))) break;
        tc_fence_after();
        if (!(ok = issue_dp(t + 1))) break;
        ETA_TRACE(82);
      }
      ok = wd.wait(BAR(B_DSFULL + (t & 1)), (t >> 1) & 1, ROLE_MMA, B_DSFULL + (t & 1));
      if (!ok) break;
      tc_fence_after();
      ETA_TRACE(83);
      // dQ_i += dS(t) K_t: A = dS packed in buffer t & 1, B = K_t MN-major over 128 keys.
      const uint64_t k_mn = smem_desc(k_addr(t), SW_CHUNK_BYTES, 1024);
#pragma unroll
      for (int ks = 0; ks < BN / 16; ++ks)
        mma_ts_elect(tmem + DQ_ACC_COL, tmem + DQ_S0_COL + 128 * (t & 1) + 64 * (ks / 4) + 8 * (ks % 4),
                     k_mn + ((ks * 16 * 128) >> 4), CF::IDESC_ND, (t > 0 || ks > 0) ? 1u : 0u);
      mma_commit_elect(BAR(CF::BAR_EMPTY + (t % CF::B_KS)));
    }
    if (ok && n_it > 0) mma_commit_elect(BAR(CF::BAR_ACC));
    mma_commit_elect(BAR(CF::BAR_DRAIN));
    wd.drain(BAR(CF::BAR_DRAIN), 0, CF::BAR_DRAIN);
  } else if (warp == CF::LOAD_WARP && lane == 0) {
    // ============================================================ TMA producer: Q, dO, K
    if (n_it > 0) {
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(BAR(CF::BAR_FIXED), CF::Q_TILE + CF::DO_TILE);
      for (int kc = 0; kc < D / SW_CHUNK; ++kc)
        tma_load_3d(sbase + CF::B_Q_OFF + kc * SW_CHUNK_BYTES, &tmQ, kc * SW_CHUNK, i * BM, bh,
                    BAR(CF::BAR_FIXED));
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
        tma_load_3d(sbase + CF::B_DO_OFF + kc * SW_CHUNK_BYTES, &tmdO, kc * SW_CHUNK, i * BM, bh,
                    BAR(CF::BAR_FIXED));
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int slot = it % CF::B_KS;
      if (!wd.wait1(BAR(CF::BAR_EMPTY + slot), ((it / CF::B_KS) & 1) ^ 1, ROLE_LOAD,
                    CF::BAR_EMPTY + slot, false))
        break;
      const uint32_t sl = sbase + CF::B_K_OFF + slot * CF::Q_TILE;
      mbar_arrive_expect_tx(BAR(CF::BAR_FULL + slot), CF::Q_TILE);
      for (int kc = 0; kc < D / SW_CHUNK; ++kc)
        tma_load_3d(sl + kc * SW_CHUNK_BYTES, &tmK, kc * SW_CHUNK, it * BN, bh, BAR(CF::BAR_FULL + slot));
      ++issued;
    }
    // The block the hardware will likely start next is about one wave ahead: warm L2 with
    // its Q and dO tiles (each unit's own) so that its first products do not wait on HBM.
    const unsigned next = blockIdx.x + nsmid();
    if (next < gridDim.x) {
      int nbh, nri;
      unit_of_block(next, p.BH, p.nq_tiles, p.head_group, &nbh, &nri);
      const int ni = p.nq_tiles - 1 - nri;
      for (int kc = 0; kc < D / SW_CHUNK; ++kc) tma_prefetch_l2_3d(&tmQ, kc * SW_CHUNK, ni * BM, nbh);
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc) tma_prefetch_l2_3d(&tmdO, kc * SW_CHUNK, ni * BM, nbh);
    }
    if (n_it > 0) wd.wait1(BAR(CF::BAR_FIXED), 0, ROLE_DRAIN, CF::BAR_FIXED, true);
    for (int s = 0; s < CF::B_KS && s < issued; ++s) {
      const int lastpos = s + ((issued - 1 - s) / CF::B_KS) * CF::B_KS;
      wd.wait1(BAR(CF::BAR_FULL + s), (lastpos / CF::B_KS) & 1, ROLE_DRAIN, CF::BAR_FULL + s, true);
    }
  } else if (warp == CF::LOAD_WARP + 1 && lane == 0) {
    // ============================================================ TMA producer: V
    if (n_it > 0) tma_prefetch_desc(&tmV);
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int slot = it % CF::B_VS;
      if (!wd.wait1(BAR(CF::BAR_VEMPTY + slot), ((it / CF::B_VS) & 1) ^ 1, ROLE_LOAD,
                    CF::BAR_VEMPTY + slot, false))
        break;
      const uint32_t sl = sbase + CF::B_V_OFF + slot * CF::DO_TILE;
      mbar_arrive_expect_tx(BAR(CF::BAR_VFULL + slot), CF::DO_TILE);
      for (int kc = 0; kc < DV / SW_CHUNK; ++kc)
        tma_load_3d(sl + kc * SW_CHUNK_BYTES, &tmV, kc * SW_CHUNK, it * BN, bh, BAR(CF::BAR_VFULL + slot));
      ++issued;
    }
    for (int s = 0; s < CF::B_VS && s < issued; ++s) {
      const int lastpos = s + ((issued - 1 - s) / CF::B_VS) * CF::B_VS;
      wd.wait1(BAR(CF::BAR_VFULL + s), (lastpos / CF::B_VS) & 1, ROLE_DRAIN, CF::BAR_VFULL + s, true);
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == CF::MMA_WARP) tmem_dealloc(tmem, CF::TMEM_COLS);
}

// ------------------------------------------------------------------------ host side
struct BwdLaunchArgs {
  CUtensorMap tmQ, tmK, tmV, tmdO;
  BwdParams p;
  cudaStream_t stream;
};

template <int D, int DV, bool CAUSAL, int BIAS>
cudaError_t launch_bwd(const BwdLaunchArgs &a) {
  using CF = BwdCfg<D, DV, CAUSAL, BIAS>;
  auto ka = attn_bwd_dkdv_kernel<D, DV, CAUSAL, BIAS>;
  auto kb = attn_bwd_dq_kernel<D, DV, CAUSAL, BIAS>;
  cudaError_t e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::A_SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::B_SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  const unsigned grid_a = static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.nkv_tiles);
  const unsigned grid_b = static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.nq_tiles);
  e = launch_pdl(ka, dim3(grid_a), dim3(CF::A_THREADS), CF::A_SMEM_TOTAL, a.stream, a.tmQ, a.tmK, a.tmV, a.tmdO, a.p);
  if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
  e = launch_pdl(kb, dim3(grid_b), dim3(CF::THREADS), CF::B_SMEM_TOTAL, a.stream, a.tmQ, a.tmK, a.tmV, a.tmdO, a.p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DV>
cudaError_t launch_bwd_prep(const void *O, int out_f32, const uint16_t *dO, const float *LSE,
                            int BH, int Nq, int nqp, float *Lp, float *Dd, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * nqp;
  const long long blocks = (rows * (DV / 8) + 255) / 256;
  const cudaError_t e = launch_pdl(attn_bwd_prep_kernel<DV>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                   stream, O, out_f32, dO, LSE, BH, Nq, nqp, Lp, Dd);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace eta

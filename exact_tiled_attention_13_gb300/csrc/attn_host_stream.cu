// attn_fwd_host, attn_bwd_host: the forward and backward passes on host-resident tensors,
// streamed through the GPU in chunks of heads. Heads are independent, so chunk k's upload,
// chunk k-1's kernels and chunk k-2's download run at the same time on three streams of
// the library, through two slots of a caller-provided device staging buffer. Built on
// attn_fwd_ex, attn_bwd and cudaMemcpyAsync alone.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"

namespace {

// Streams and events of the pipeline, created once per device and kept for the life of
// the process. `start` orders the pipeline after the caller's stream; the per-slot events
// say when a slot's inputs have landed, its kernels have run and its outputs have left.
struct Pipeline {
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in_done[2] = {nullptr, nullptr};
  cudaEvent_t comp_done[2] = {nullptr, nullptr};
  cudaEvent_t out_done[2] = {nullptr, nullptr};
};

constexpr int kMaxDevices = 64;
Pipeline g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;  // held while a call queues its work

int pipeline_for(int dev, Pipeline **out) {
  Pipeline &p = g_pipe[dev];
  if (!p.ready) {
    bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; ok && s < 2; ++s)
      ok = cudaEventCreateWithFlags(&p.in_done[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.comp_done[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&p.out_done[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    p.ready = true;
  }
  *out = &p;
  return ATTN_OK;
}

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// One tensor of a chunk: uploaded from `src`, downloaded to `dst`, or neither (scratch
// space in the slot). `per_head` bytes per head; `off` its offset in a slot.
struct Part {
  const void *src = nullptr;
  void *dst = nullptr;
  size_t per_head = 0;
  size_t off = 0;
};

// Places the parts one after the other in a slot of `h` heads (each 256-byte aligned);
// returns the slot size.
size_t place(Part *parts, int n, int h) {
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    parts[i].off = off;
    off += round_up(parts[i].per_head * static_cast<size_t>(h));
  }
  return off;
}

// Blocks a chunk's launches should carry at least, so that they fill most of the GPU
// (about a wave on a 152-SM part) instead of leaving most SMs idle. Smaller chunks
// overlap better; chunks of much less than a wave waste the SMs they leave idle.
constexpr int kMinChunkBlocks = 128;

// Heads per chunk: the caller's choice, else about eight chunks, but no fewer heads than
// kMinChunkBlocks blocks of `blocks_per_head` need.
int chunk_heads(int BH, int blocks_per_head, int heads_per_chunk) {
  if (heads_per_chunk > 0) return heads_per_chunk < BH ? heads_per_chunk : BH;
  int h = (BH + 7) / 8;
  const int h_fill = blocks_per_head > 0 ? (kMinChunkBlocks + blocks_per_head - 1) / blocks_per_head : 1;
  if (h < h_fill) h = h_fill;
  if (h > BH) h = BH;
  return h > 0 ? h : 1;
}

int slots_for(int BH, int h) { return (BH + h - 1) / h > 1 ? 2 : 1; }

// Host memory (page-locked or pageable) or null; device memory is refused.
bool host_pointer_ok(const void *ptr) {
  if (!ptr) return true;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeUnregistered;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Host checks of a call's parts: outputs overlap no input and no other output (checked
// before any CUDA call), and every pointer is host memory.
int check_host_parts(const Part *parts, int n, int BH) {
  const size_t heads = static_cast<size_t>(BH);
  for (int i = 0; i < n; ++i) {
    if (!parts[i].dst) continue;
    for (int j = 0; j < n; ++j) {
      if (j == i) continue;
      const void *other = parts[j].dst ? parts[j].dst : parts[j].src;
      if (overlaps(parts[i].dst, parts[i].per_head * heads, other, parts[j].per_head * heads))
        return ATTN_ERR_INVALID_ARG;
    }
  }
  for (int i = 0; i < n; ++i)
    if (!host_pointer_ok(parts[i].src) || !host_pointer_ok(parts[i].dst)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Queues the chunks: upload (after the kernels of chunk k - 2, the slot's last reader),
// `compute(slot, heads, stream)` (after chunk k - 2's download, the slot's last user),
// download. Work queued on `user` after the call waits for the last download.
template <class Compute>
int stream_chunks(int BH, int h, const Part *parts, int n, size_t slot_bytes, void *staging,
                  cudaStream_t user, Compute compute) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  Pipeline *pp = nullptr;
  int rc = pipeline_for(dev, &pp);
  if (rc != ATTN_OK) return rc;
  Pipeline &P = *pp;
  char *base = static_cast<char *>(staging);

  cudaError_t e = cudaEventRecord(P.start, user);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.start, 0);
  bool used[2] = {false, false};
  for (int k = 0, h0 = 0; e == cudaSuccess && rc == ATTN_OK && h0 < BH; ++k, h0 += h) {
    const int s = k & 1;
    const int hc = BH - h0 < h ? BH - h0 : h;
    char *slot = base + static_cast<size_t>(s) * slot_bytes;
    if (k >= 2) e = cudaStreamWaitEvent(P.in, P.comp_done[s], 0);
    for (int i = 0; i < n && e == cudaSuccess; ++i)
      if (parts[i].src && parts[i].per_head > 0)
        e = cudaMemcpyAsync(slot + parts[i].off,
                            static_cast<const char *>(parts[i].src) + parts[i].per_head * static_cast<size_t>(h0),
                            parts[i].per_head * hc, cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaEventRecord(P.in_done[s], P.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.in_done[s], 0);
    if (e == cudaSuccess && k >= 2) e = cudaStreamWaitEvent(P.comp, P.out_done[s], 0);
    if (e != cudaSuccess) break;
    rc = compute(slot, hc, P.comp);
    if (rc != ATTN_OK) break;
    e = cudaEventRecord(P.comp_done[s], P.comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.comp_done[s], 0);
    for (int i = 0; i < n && e == cudaSuccess; ++i)
      if (parts[i].dst && parts[i].per_head > 0)
        e = cudaMemcpyAsync(static_cast<char *>(parts[i].dst) + parts[i].per_head * static_cast<size_t>(h0),
                            slot + parts[i].off, parts[i].per_head * hc, cudaMemcpyDeviceToHost, P.out);
    if (e == cudaSuccess) e = cudaEventRecord(P.out_done[s], P.out);
    if (e == cudaSuccess) used[s] = true;
  }
  // The download stream runs in order: waiting for the last record of each slot covers
  // every chunk, also when queueing stopped early.
  for (int s = 0; s < 2; ++s)
    if (used[s] && cudaStreamWaitEvent(user, P.out_done[s], 0) != cudaSuccess) e = cudaErrorUnknown;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return rc != ATTN_OK ? rc : ATTN_ERR_CUDA;
  }
  return rc;
}

// Checks shared by both passes that look at no pointer (mode, sizes, dtype, widths).
int check_sizes(int mode, int BH, int Nq, int Nk, int d, int d_v, int dtype, int heads_per_chunk) {
  if (heads_per_chunk < 0 || BH < 1 || Nq < 0 || Nk < 0 ||
      (dtype != ATTN_OUT_BF16 && dtype != ATTN_OUT_F32) ||
      (mode & ~(ATTN_MASK_CAUSAL | ATTN_BIAS_DENSE | ATTN_BIAS_KEY)) != 0 ||
      ((mode & ATTN_BIAS_DENSE) && (mode & ATTN_BIAS_KEY)))
    return ATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || (d_v != 64 && d_v != 128)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

bool scale_ok(float scale) { return scale > 0.0f && scale < 3.0e38f; }

bool bias_pointers_ok(int mode, const float *C, const float *ckey) {
  return ((mode & ATTN_BIAS_DENSE) != 0) == (C != nullptr) && ((mode & ATTN_BIAS_KEY) != 0) == (ckey != nullptr);
}

// ---- forward: Q, K, V, C, ckey in; O, LSE out
enum { F_Q, F_K, F_V, F_C, F_CK, F_O, F_L, F_N };

int fwd_heads(int mode, int BH, int Nq, int heads_per_chunk) {
  const int q_tiles = (Nq + 127) / 128;
  const int per_block = (mode & ATTN_BIAS_DENSE) ? 1 : 2;  // query tiles per block
  return chunk_heads(BH, (q_tiles + per_block - 1) / per_block, heads_per_chunk);
}

size_t fwd_parts(Part *p, int mode, int Nq, int Nk, int d, int d_v, int out_dtype, int h) {
  p[F_Q].per_head = static_cast<size_t>(Nq) * d * 2;
  p[F_K].per_head = static_cast<size_t>(Nk) * d * 2;
  p[F_V].per_head = static_cast<size_t>(Nk) * d_v * 2;
  p[F_C].per_head = (mode & ATTN_BIAS_DENSE) ? static_cast<size_t>(Nq) * Nk * 4 : 0;
  p[F_CK].per_head = (mode & ATTN_BIAS_KEY) ? static_cast<size_t>(Nk) * 4 : 0;
  p[F_O].per_head = static_cast<size_t>(Nq) * d_v * (out_dtype == ATTN_OUT_F32 ? 4 : 2);
  p[F_L].per_head = static_cast<size_t>(Nq) * 4;
  return place(p, F_N, h);
}

// ---- backward: Q, K, V, O, dO, LSE, C, ckey in; dQ, dK, dV out; the row-statistics
// workspace
enum { B_Q, B_K, B_V, B_O, B_DO, B_L, B_C, B_CK, B_DQ, B_DK, B_DV, B_WS, B_N };

int bwd_heads(int BH, int Nq, int Nk, int heads_per_chunk) {
  const int q_tiles = (Nq + 127) / 128, k_tiles = (Nk + 127) / 128;  // a block per tile
  return chunk_heads(BH, q_tiles > k_tiles ? q_tiles : k_tiles, heads_per_chunk);
}

size_t bwd_parts(Part *p, int mode, int Nq, int Nk, int d, int d_v, int o_dtype, int h) {
  p[B_Q].per_head = static_cast<size_t>(Nq) * d * 2;
  p[B_K].per_head = static_cast<size_t>(Nk) * d * 2;
  p[B_V].per_head = static_cast<size_t>(Nk) * d_v * 2;
  p[B_O].per_head = static_cast<size_t>(Nq) * d_v * (o_dtype == ATTN_OUT_F32 ? 4 : 2);
  p[B_DO].per_head = static_cast<size_t>(Nq) * d_v * 2;
  p[B_L].per_head = static_cast<size_t>(Nq) * 4;
  p[B_C].per_head = (mode & ATTN_BIAS_DENSE) ? static_cast<size_t>(Nq) * Nk * 4 : 0;
  p[B_CK].per_head = (mode & ATTN_BIAS_KEY) ? static_cast<size_t>(Nk) * 4 : 0;
  p[B_DQ].per_head = static_cast<size_t>(Nq) * d * 4;
  p[B_DK].per_head = static_cast<size_t>(Nk) * d * 4;
  p[B_DV].per_head = static_cast<size_t>(Nk) * d_v * 4;
  unsigned long long ws = 0;
  attn_bwd_workspace_bytes(1, Nq, &ws);  // linear in the heads
  p[B_WS].per_head = static_cast<size_t>(ws);
  return place(p, B_N, h);
}

}  // namespace

extern "C" int attn_fwd_host_staging_bytes(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                           int out_dtype, int heads_per_chunk,
                                           unsigned long long *bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  const int rc = check_sizes(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk);
  if (rc != ATTN_OK) return rc;
  const int h = fwd_heads(mode, BH, Nq, heads_per_chunk);
  Part p[F_N];
  *bytes = static_cast<unsigned long long>(slots_for(BH, h)) * fwd_parts(p, mode, Nq, Nk, d, d_v, out_dtype, h);
  return ATTN_OK;
}

extern "C" int attn_fwd_host(const void *Q, const void *K, const void *V, int mode, const float *C,
                             const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                             void *O, int out_dtype, float *LSE, void *staging,
                             unsigned long long staging_bytes, int heads_per_chunk, void *stream) {
  unsigned long long need = 0;
  int rc = attn_fwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk, &need);
  if (rc != ATTN_OK) return rc;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (Nq == 0) return ATTN_OK;               // nothing to compute or to copy
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;  // every row would lack an allowed key
  if (!Q || !K || !V || !O || !staging || !bias_pointers_ok(mode, C, ckey)) return ATTN_ERR_INVALID_ARG;
  if (staging_bytes < need || reinterpret_cast<uintptr_t>(staging) % kAlign != 0) return ATTN_ERR_INVALID_ARG;
  const int h = fwd_heads(mode, BH, Nq, heads_per_chunk);
  Part p[F_N];
  const size_t slot_bytes = fwd_parts(p, mode, Nq, Nk, d, d_v, out_dtype, h);
  p[F_Q].src = Q;
  p[F_K].src = K;
  p[F_V].src = V;
  p[F_C].src = C;
  p[F_CK].src = ckey;
  p[F_O].dst = O;
  p[F_L].dst = LSE;
  if ((rc = check_host_parts(p, F_N, BH)) != ATTN_OK) return rc;
  return stream_chunks(BH, h, p, F_N, slot_bytes, staging, static_cast<cudaStream_t>(stream),
                       [&](char *slot, int hc, cudaStream_t st) {
                         return attn_fwd_ex(slot + p[F_Q].off, slot + p[F_K].off, slot + p[F_V].off, mode,
                                            C ? reinterpret_cast<const float *>(slot + p[F_C].off) : nullptr,
                                            ckey ? reinterpret_cast<const float *>(slot + p[F_CK].off) : nullptr,
                                            hc, Nq, Nk, d, d_v, scale, slot + p[F_O].off, out_dtype,
                                            LSE ? reinterpret_cast<float *>(slot + p[F_L].off) : nullptr, st);
                       });
}

extern "C" int attn_bwd_host_staging_bytes(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                           int o_dtype, int heads_per_chunk,
                                           unsigned long long *bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  const int rc = check_sizes(mode, BH, Nq, Nk, d, d_v, o_dtype, heads_per_chunk);
  if (rc != ATTN_OK) return rc;
  const int h = bwd_heads(BH, Nq, Nk, heads_per_chunk);
  Part p[B_N];
  *bytes = static_cast<unsigned long long>(slots_for(BH, h)) * bwd_parts(p, mode, Nq, Nk, d, d_v, o_dtype, h);
  return ATTN_OK;
}

extern "C" int attn_bwd_host(const void *Q, const void *K, const void *V, const void *O, int o_dtype,
                             const void *dO, const float *LSE, int mode, const float *C,
                             const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                             float *dQ, float *dK, float *dV, void *staging,
                             unsigned long long staging_bytes, int heads_per_chunk, void *stream) {
  unsigned long long need = 0;
  int rc = attn_bwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, o_dtype, heads_per_chunk, &need);
  if (rc != ATTN_OK) return rc;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (Nk == 0) return Nq == 0 ? ATTN_OK : ATTN_ERR_INVALID_ARG;
  const bool q = Nq > 0;
  if (!K || !V || !dK || !dV || !staging || !bias_pointers_ok(mode, C, ckey)) return ATTN_ERR_INVALID_ARG;
  if (q && (!Q || !O || !dO || !LSE || !dQ)) return ATTN_ERR_INVALID_ARG;
  if (staging_bytes < need || reinterpret_cast<uintptr_t>(staging) % kAlign != 0) return ATTN_ERR_INVALID_ARG;
  const int h = bwd_heads(BH, Nq, Nk, heads_per_chunk);
  Part p[B_N];
  const size_t slot_bytes = bwd_parts(p, mode, Nq, Nk, d, d_v, o_dtype, h);
  p[B_Q].src = Q;
  p[B_K].src = K;
  p[B_V].src = V;
  p[B_O].src = O;
  p[B_DO].src = dO;
  p[B_L].src = LSE;
  p[B_C].src = C;
  p[B_CK].src = ckey;
  p[B_DQ].dst = dQ;
  p[B_DK].dst = dK;
  p[B_DV].dst = dV;
  if ((rc = check_host_parts(p, B_N, BH)) != ATTN_OK) return rc;
  return stream_chunks(
      BH, h, p, B_N, slot_bytes, staging, static_cast<cudaStream_t>(stream), [&](char *slot, int hc, cudaStream_t st) {
        auto f = [&](int i) { return reinterpret_cast<float *>(slot + p[i].off); };
        return attn_bwd(q ? slot + p[B_Q].off : nullptr, slot + p[B_K].off, slot + p[B_V].off,
                        q ? slot + p[B_O].off : nullptr, o_dtype, q ? slot + p[B_DO].off : nullptr,
                        q ? f(B_L) : nullptr, mode, C ? f(B_C) : nullptr, ckey ? f(B_CK) : nullptr, hc, Nq, Nk,
                        d, d_v, scale, q ? f(B_DQ) : nullptr, f(B_DK), f(B_DV), q ? slot + p[B_WS].off : nullptr,
                        p[B_WS].per_head * hc, st);
      });
}

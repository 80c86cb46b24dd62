// attn_fwd_host: the forward pass on host-resident tensors, streamed through the GPU in
// chunks of heads. Heads are independent, so chunk k's upload, chunk k-1's attention and
// chunk k-2's download run at the same time on three streams of the library, through two
// slots of a caller-provided device staging buffer. Built on attn_fwd_ex and
// cudaMemcpyAsync alone.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn.h"

namespace {

// Streams and events of the pipeline, created once per device and kept for the life of
// the process. `start` orders the pipeline after the caller's stream; the per-slot events
// say when a slot's inputs have landed, its attention has run and its outputs have left.
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

// Byte sizes of one head's tensors and their offsets in a staging slot of `h` heads.
struct Layout {
  size_t q, k, v, c, ck, o, l;                  // bytes per head
  size_t off_q, off_k, off_v, off_c, off_ck, off_o, off_l, slot;
  Layout(int mode, int Nq, int Nk, int d, int d_v, int out_dtype, int h) {
    q = static_cast<size_t>(Nq) * d * 2;
    k = static_cast<size_t>(Nk) * d * 2;
    v = static_cast<size_t>(Nk) * d_v * 2;
    c = (mode & ATTN_BIAS_DENSE) ? static_cast<size_t>(Nq) * Nk * 4 : 0;
    ck = (mode & ATTN_BIAS_KEY) ? static_cast<size_t>(Nk) * 4 : 0;
    o = static_cast<size_t>(Nq) * d_v * (out_dtype == ATTN_OUT_F32 ? 4 : 2);
    l = static_cast<size_t>(Nq) * 4;
    off_q = 0;
    off_k = off_q + round_up(q * h);
    off_v = off_k + round_up(k * h);
    off_c = off_v + round_up(v * h);
    off_ck = off_c + round_up(c * h);
    off_o = off_ck + round_up(ck * h);
    off_l = off_o + round_up(o * h);
    slot = off_l + round_up(l * h);
  }
};

// Blocks a chunk's attention launch should carry at least, so that it fills most of the
// GPU (about a wave on a 152-SM part) instead of leaving most SMs idle. Smaller chunks
// overlap better; chunks of much less than a wave waste the SMs they leave idle.
constexpr int kMinChunkBlocks = 128;

// Heads per chunk: the caller's choice, else about eight chunks, but no fewer heads than
// kMinChunkBlocks blocks need (one block per 128-query tile with a dense bias, per two
// tiles otherwise).
int chunk_heads(int mode, int BH, int Nq, int heads_per_chunk) {
  if (heads_per_chunk > 0) return heads_per_chunk < BH ? heads_per_chunk : BH;
  const int q_tiles = (Nq + 127) / 128;
  const int per_block = (mode & ATTN_BIAS_DENSE) ? 1 : 2;
  const int blocks_per_head = (q_tiles + per_block - 1) / per_block;
  int h = (BH + 7) / 8;
  const int h_fill = blocks_per_head > 0 ? (kMinChunkBlocks + blocks_per_head - 1) / blocks_per_head : 1;
  if (h < h_fill) h = h_fill;
  if (h > BH) h = BH;
  return h > 0 ? h : 1;
}

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

const char *at(const void *base, size_t bytes_per_head, int h0) {
  return static_cast<const char *>(base) + bytes_per_head * static_cast<size_t>(h0);
}

}  // namespace

extern "C" int attn_fwd_host_staging_bytes(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                           int out_dtype, int heads_per_chunk,
                                           unsigned long long *bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (heads_per_chunk < 0 || BH < 1 || Nq < 0 || Nk < 0 ||
      (out_dtype != ATTN_OUT_BF16 && out_dtype != ATTN_OUT_F32) ||
      (mode & ~(ATTN_MASK_CAUSAL | ATTN_BIAS_DENSE | ATTN_BIAS_KEY)) != 0 ||
      ((mode & ATTN_BIAS_DENSE) && (mode & ATTN_BIAS_KEY)))
    return ATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || (d_v != 64 && d_v != 128)) return ATTN_ERR_UNSUPPORTED;
  const int h = chunk_heads(mode, BH, Nq, heads_per_chunk);
  const int slots = (BH + h - 1) / h > 1 ? 2 : 1;
  *bytes = static_cast<unsigned long long>(slots) * Layout(mode, Nq, Nk, d, d_v, out_dtype, h).slot;
  return ATTN_OK;
}

extern "C" int attn_fwd_host(const void *Q, const void *K, const void *V, int mode, const float *C,
                             const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                             void *O, int out_dtype, float *LSE, void *staging,
                             unsigned long long staging_bytes, int heads_per_chunk, void *stream) {
  unsigned long long need = 0;
  int rc = attn_fwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk, &need);
  if (rc != ATTN_OK) return rc;
  if (!(scale > 0.0f) || !(scale < 3.0e38f)) return ATTN_ERR_INVALID_ARG;
  if (Nq == 0) return ATTN_OK;  // nothing to compute or to copy
  if (Nk == 0) return ATTN_ERR_INVALID_ARG;  // every row would lack an allowed key
  if (!Q || !K || !V || !O || !staging) return ATTN_ERR_INVALID_ARG;
  if (((mode & ATTN_BIAS_DENSE) != 0) != (C != nullptr) || ((mode & ATTN_BIAS_KEY) != 0) != (ckey != nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (staging_bytes < need || reinterpret_cast<uintptr_t>(staging) % kAlign != 0) return ATTN_ERR_INVALID_ARG;
  const int h = chunk_heads(mode, BH, Nq, heads_per_chunk);
  const Layout lay(mode, Nq, Nk, d, d_v, out_dtype, h);
  const size_t n = static_cast<size_t>(BH);
  const void *ins[5] = {Q, K, V, C, ckey};
  const size_t in_bytes[5] = {lay.q * n, lay.k * n, lay.v * n, C ? lay.c * n : 0, ckey ? lay.ck * n : 0};
  for (int i = 0; i < 5; ++i)
    if (overlaps(O, lay.o * n, ins[i], in_bytes[i]) || overlaps(LSE, LSE ? lay.l * n : 0, ins[i], in_bytes[i]))
      return ATTN_ERR_INVALID_ARG;
  if (overlaps(O, lay.o * n, LSE, LSE ? lay.l * n : 0)) return ATTN_ERR_INVALID_ARG;
  const void *hosts[7] = {Q, K, V, C, ckey, O, LSE};
  for (const void *ptr : hosts)
    if (!host_pointer_ok(ptr)) return ATTN_ERR_INVALID_ARG;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  Pipeline *pp = nullptr;
  if ((rc = pipeline_for(dev, &pp)) != ATTN_OK) return rc;
  Pipeline &P = *pp;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(staging);

  cudaError_t e = cudaEventRecord(P.start, user);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.start, 0);
  int last_slot_used[2] = {0, 0};
  for (int k = 0, h0 = 0; e == cudaSuccess && rc == ATTN_OK && h0 < BH; ++k, h0 += h) {
    const int s = k & 1;
    const int hc = BH - h0 < h ? BH - h0 : h;
    char *slot = base + static_cast<size_t>(s) * lay.slot;
    // Upload chunk k once the attention of chunk k - 2 (the slot's last reader) has run.
    if (k >= 2) e = cudaStreamWaitEvent(P.in, P.comp_done[s], 0);
    const struct {
      const void *src;
      size_t per_head, off;
    } up[5] = {{Q, lay.q, lay.off_q}, {K, lay.k, lay.off_k}, {V, lay.v, lay.off_v},
               {C, lay.c, lay.off_c}, {ckey, lay.ck, lay.off_ck}};
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
      if (up[i].src && up[i].per_head > 0)
        e = cudaMemcpyAsync(slot + up[i].off, at(up[i].src, up[i].per_head, h0), up[i].per_head * hc,
                            cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaEventRecord(P.in_done[s], P.in);
    // Attention of chunk k once its inputs have landed and chunk k - 2's outputs have left.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.comp, P.in_done[s], 0);
    if (e == cudaSuccess && k >= 2) e = cudaStreamWaitEvent(P.comp, P.out_done[s], 0);
    if (e != cudaSuccess) break;
    rc = attn_fwd_ex(slot + lay.off_q, slot + lay.off_k, slot + lay.off_v, mode,
                     C ? reinterpret_cast<const float *>(slot + lay.off_c) : nullptr,
                     ckey ? reinterpret_cast<const float *>(slot + lay.off_ck) : nullptr, hc, Nq, Nk, d,
                     d_v, scale, slot + lay.off_o, out_dtype,
                     LSE ? reinterpret_cast<float *>(slot + lay.off_l) : nullptr, P.comp);
    if (rc != ATTN_OK) break;
    e = cudaEventRecord(P.comp_done[s], P.comp);
    // Download chunk k's outputs.
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.comp_done[s], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char *>(O) + lay.o * static_cast<size_t>(h0), slot + lay.off_o,
                          lay.o * hc, cudaMemcpyDeviceToHost, P.out);
    if (e == cudaSuccess && LSE)
      e = cudaMemcpyAsync(reinterpret_cast<char *>(LSE) + lay.l * static_cast<size_t>(h0), slot + lay.off_l,
                          lay.l * hc, cudaMemcpyDeviceToHost, P.out);
    if (e == cudaSuccess) e = cudaEventRecord(P.out_done[s], P.out);
    if (e == cudaSuccess) last_slot_used[s] = 1;
  }
  // Work queued on the caller's stream after this call waits for every download (the
  // download stream runs them in order), also when queueing stopped early.
  for (int s = 0; s < 2; ++s)
    if (last_slot_used[s] && cudaStreamWaitEvent(user, P.out_done[s], 0) != cudaSuccess) e = cudaErrorUnknown;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return rc != ATTN_OK ? rc : ATTN_ERR_CUDA;
  }
  return rc;
}

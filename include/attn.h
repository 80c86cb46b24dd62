/*
 * attn.h -- C ABI of the exact tiled attention forward pass for NVIDIA GB300 (sm_103a).
 *
 * The operation is exact scaled dot-product attention for B*H independent heads,
 * as defined in "Compilers and kernels", section "FlashAttention rewrites the algorithm
 * around IO",
 * first display and its symbol list:
 *
 *     S = Q K^T * scale + C,  m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i),
 *     P_ij = exp(S_ij - m_i) / l_i,  O = P V,
 *
 * with C an additive bias or mask (-inf forbids a key) and at least one allowed key
 * per query row. The library evaluates it tile by tile with the online recurrence of
 * the same section (b_t, m_t = max(m_{t-1}, b_t), alpha_t = exp(m_{t-1} - m_t), l_t,
 * o_t, O_i = o_T / l_T), so S and P never reach device memory. "Exact" means the same
 * function, not the same bits: tiling changes the floating-point evaluation order
 * (same section, the paragraph after the recurrence).
 *
 * Numeric contract of this implementation: Q K^T and P V run on the tensor cores with
 * bf16 operands and fp32 accumulation; scores, the running max and sum, and O are fp32;
 * P is rounded to bf16 before it multiplies V; LSE_i = m_i + ln l_i (natural log, in the
 * units of S, bias included) uses the sum of the unrounded fp32 p, and O_i = o_i / l_i
 * uses that sum with each tile's largest p taken as rounded. The exponent reference
 * m_t of the recurrence is moved only when a tile's maximum exceeds it by more than a
 * factor 2^8 (any reference used consistently gives the same o_T / l_T), so o is
 * rescaled only then.
 *
 * All entry points are plain C, take device pointers and sizes (attn_fwd_host and
 * attn_bwd_host: host tensors and a device staging buffer), and never allocate device
 * memory (the host-streaming calls create three streams and seven events per device on
 * their first call). They are thread-safe:
 * calls from several host threads or on several streams may overlap.
 *
 * Device reset: the library caches, per device, the device addresses of its own
 * __device__ variables (the watchdog word, the fixed scratch array of
 * attn_fwd_splitkv_static). cudaDeviceReset or cuDevicePrimaryCtxReset unloads the
 * library's device code with the context and leaves those addresses stale: do not reset
 * a device and then call this library on it again in the same process.
 */
#ifndef EXACT_TILED_ATTENTION_13_ATTN_H
#define EXACT_TILED_ATTENTION_13_ATTN_H

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Mask / bias terms (argument `mode`, a bit set; C is the sum of the selected terms). */
#define ATTN_MASK_NONE 0   /* C = 0 */
#define ATTN_MASK_CAUSAL 1 /* -inf for key j > query i + (Nk - Nq), else 0 (Nq = Nk: j > i) */
#define ATTN_BIAS_DENSE 2  /* a dense fp32 [BH][Nq][Nk] array C */
#define ATTN_BIAS_KEY 4    /* a per-key fp32 [BH][Nk] vector c, the same for every query row
                              (attn_fwd_ex only; key padding is c_j = -inf) */
#define ATTN_BIAS_SHARED 8 /* with ATTN_BIAS_DENSE only: C is one fp32 [Nq][Nk] array that
                              every head adds (a bias broadcast over the heads), instead of
                              [BH][Nq][Nk]; rejected by the host-streaming calls */

/* Output element types (argument `out_dtype`). */
#define ATTN_OUT_BF16 0
#define ATTN_OUT_F32 1

/* Return codes. Zero is success; every error is negative. */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG (-1)        /* null/misaligned/overlapping pointer, bad size, mode or scale */
#define ATTN_ERR_UNSUPPORTED (-2)        /* a head width d or d_v the library has no kernel for */
#define ATTN_ERR_NO_DEVICE (-3)          /* no CUDA device, or no CUDA driver */
#define ATTN_ERR_UNSUPPORTED_DEVICE (-4) /* the current device is not compute capability 10.3 */
#define ATTN_ERR_LAUNCH (-5)             /* the kernel launch was rejected by the CUDA runtime */
#define ATTN_ERR_DEVICE_TIMEOUT (-6)     /* a kernel gave up on a pipeline wait (see attn_device_status) */
#define ATTN_ERR_CUDA (-7)               /* another CUDA runtime or driver call failed */
#define ATTN_ERR_SCRATCH_LIMIT (-8)      /* attn_fwd_splitkv_static: the problem needs more scratch
                                            than ATTN_STATIC_SCRATCH_BYTES */

/*
 * attn_fwd -- O = softmax(Q K^T * scale + C) V and LSE for BH heads, on `stream`.
 *
 * Arguments (all pointers are device pointers, or managed memory):
 *   Q     bf16, contiguous row-major [BH][N][d]      queries
 *   K     bf16, contiguous row-major [BH][N][d]      keys
 *   V     bf16, contiguous row-major [BH][N][d_v]    values
 *   mode  ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_BIAS_DENSE, or
 *         ATTN_MASK_CAUSAL | ATTN_BIAS_DENSE (causal mask and dense bias together); with
 *         ATTN_BIAS_DENSE also ATTN_BIAS_SHARED (one C for all heads)
 *   C     fp32, contiguous row-major [BH][N][N] when mode has ATTN_BIAS_DENSE ([N][N] with
 *         ATTN_BIAS_SHARED: the same bias for every head), else NULL.
 *         Entries are finite or -inf; C is added after the scaling and is not scaled.
 *   BH    number of heads (batch times heads), >= 1
 *   N     sequence length (queries = keys), >= 0; N == 0 is a successful no-op in which
 *         the pointers are not inspected (empty buffers may be NULL)
 *   d     query/key width, 64 or 128
 *   d_v   value width, 64 or 128
 *   scale score scale, finite and > 0 (the pages use 1/sqrt(d))
 *   O     [BH][N][d_v] output, bf16 (out_dtype ATTN_OUT_BF16) or fp32 (ATTN_OUT_F32)
 *   LSE   fp32 [BH][N] output, ln sum_j exp(S_ij); may be NULL to skip it
 *   stream cudaStream_t to launch on; NULL means the legacy default stream
 *
 * Alignment: Q, K, V, C and O must be 16-byte aligned; LSE 4-byte aligned.
 * Aliasing: O and LSE must not overlap each other or any input. Inputs are not
 * modified.
 * Ownership: the caller owns every buffer and must keep it alive until the work on
 * `stream` completes. The library keeps no pointer after the call returns.
 * Asynchrony: the call validates its arguments, launches one kernel and returns; the
 * results are ready when `stream` reaches that point.
 * Determinism: the same inputs give bit-identical outputs (no atomics, fixed order).
 * Precondition (the pages' assumption): every query row has at least one allowed
 * key. A row with none gets O_i = 0 and LSE_i = -inf.
 *
 * Returns ATTN_OK or one of the negative codes above. Argument errors are reported
 * before anything is launched. A wait that times out inside the kernel is reported
 * by attn_device_status, not here.
 */
ATTN_API int attn_fwd(const void *Q, const void *K, const void *V, int mode, const float *C, int BH, int N,
             int d, int d_v, float scale, void *O, int out_dtype, float *LSE, void *stream);

/*
 * attn_fwd_ex -- the same operation with Nq queries and Nk keys per head, and the
 * per-key bias term. Everything not listed here is as for attn_fwd.
 *   Q     bf16 [BH][Nq][d];  K bf16 [BH][Nk][d];  V bf16 [BH][Nk][d_v]
 *   mode  bit set of ATTN_MASK_CAUSAL, ATTN_BIAS_DENSE, ATTN_BIAS_KEY, ATTN_BIAS_SHARED
 *         (DENSE and KEY together are rejected: add the vector into C instead; SHARED needs
 *         DENSE)
 *   C     fp32 [BH][Nq][Nk] with ATTN_BIAS_DENSE ([Nq][Nk] with ATTN_BIAS_SHARED), else NULL
 *   ckey  fp32 [BH][Nk] with ATTN_BIAS_KEY, else NULL; 4-byte aligned; finite or -inf.
 *         At d = 64, d_v = 128 (one key range) the bias enters the score product as
 *         c_j / scale in two bf16 parts, carried to about 2^-17 relative; finite values
 *         need |c_j| < 3.3e38 * scale there (4.1e37 at scale 1/8), as they need
 *         |c_j| < 2.3e38 on the other paths, which scale them by log2(e).
 *   Nq    >= 0 (0: no-op); Nk >= 1 when Nq >= 1
 *   O     [BH][Nq][d_v];  LSE fp32 [BH][Nq] or NULL
 * The causal mask aligns the last query with the last key: query i may see keys
 * j <= i + (Nk - Nq). With Nq > Nk the first Nq - Nk queries see no key and get the
 * defined result O_i = 0, LSE_i = -inf.
 */
ATTN_API int attn_fwd_ex(const void *Q, const void *K, const void *V, int mode, const float *C,
                         const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                         void *O, int out_dtype, float *LSE, void *stream);

/*
 * attn_fwd_splitkv -- the attn_fwd_ex operation with each head's keys cut into ranges of
 * whole 128-key tiles that run as separate thread blocks, for shapes with few query
 * tiles and many keys (decoding, a short query block against a long key cache), where
 * one block per query tile would leave most of the GPU idle. Each range stores its
 * normalised partial output and log-sum-exp in `workspace`; a second kernel merges the
 * ranges in increasing order by rescaling them to the common maximum (the blockwise
 * softmax statistics of "AI Infra ch. 5", section 5.4, and the alpha rescaling of
 * "Compilers and kernels", section "FlashAttention rewrites the algorithm around IO").
 * Arguments as for attn_fwd_ex, plus:
 *   n_splits  requested number of key ranges, >= 0. It is rounded to whole tiles
 *             (ceil(Nk/128) / ceil(ceil(Nk/128) / n_splits) ranges) and capped at the
 *             number of key tiles. 0 lets the library choose for the current device.
 *   workspace device memory of at least the size attn_fwd_splitkv_plan reports for the
 *             same arguments, 16-byte aligned, overlapping no input or output. The
 *             caller owns it; its contents on entry do not matter and are overwritten.
 *             It must stay untouched until the work on `stream` completes. When the
 *             plan has one range the kernel writes O directly and the workspace is
 *             not used (it may then be NULL).
 *   workspace_bytes its size in bytes.
 * Two kernels are launched on `stream` (one when the plan has one range). The result
 * is deterministic for a given number of ranges (fixed merge order, no atomics); a
 * different number of ranges may differ in rounding, within the tolerance of the
 * method. Errors as for attn_fwd_ex; a missing, misaligned, too small or overlapping
 * workspace is ATTN_ERR_INVALID_ARG.
 */
ATTN_API int attn_fwd_splitkv(const void *Q, const void *K, const void *V, int mode,
                              const float *C, const float *ckey, int BH, int Nq, int Nk, int d,
                              int d_v, float scale, int n_splits, void *workspace,
                              unsigned long long workspace_bytes, void *O, int out_dtype,
                              float *LSE, void *stream);

/*
 * attn_fwd_splitkv_plan -- the number of key ranges attn_fwd_splitkv will use for
 * these arguments (`*splits`) and the workspace bytes it needs (`*workspace_bytes`,
 * splits x BH x Nq x (d_v + 1) x 4 bytes: fp32 partial O and LSE per range; 0 when
 * splits is 1). n_splits == 0 (automatic) reads the current device's multiprocessor
 * count; any other value involves no CUDA call. Returns ATTN_OK, or the argument
 * error attn_fwd_splitkv would return for the same shape, mode and n_splits
 * (ATTN_ERR_INVALID_ARG also for NULL out-pointers).
 */
ATTN_API int attn_fwd_splitkv_plan(int mode, int BH, int Nq, int Nk, int d, int d_v, int n_splits,
                                   int *splits, unsigned long long *workspace_bytes);

/*
 * attn_fwd_splitkv_static -- attn_fwd_splitkv for callers that cannot allocate device
 * memory (the pages have no counterpart: this is a deployment variant of the split
 * forward pass, not a step of the method). It takes the arguments of attn_fwd_splitkv
 * without the workspace and keeps its partials in a fixed array inside the library,
 * ATTN_STATIC_SCRATCH_BYTES (32 MiB) per device. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   - A problem whose plan (attn_fwd_splitkv_plan with the same arguments) needs more
 *     than ATTN_STATIC_SCRATCH_BYTES is rejected with ATTN_ERR_SCRATCH_LIMIT before any
 *     CUDA call (n_splits > 0) or after reading the device's multiprocessor count
 *     (n_splits == 0). Pass a smaller n_splits to fit; one range needs no scratch.
 *   - Every call on a device shares the one array. Nothing in it needs to start at
 *     zero (each call writes every partial it reads), but two calls whose work may
 *     overlap on the GPU (different streams, or host threads without ordering between
 *     them) race on it and may return wrong results: order such calls on one stream.
 *   - The first call on each device looks up the array's address (cudaGetSymbolAddress),
 *     which loads the library's device code on that device; make that first call with
 *     the device current and before any stream capture begins.
 * Returns what attn_fwd_splitkv returns, or ATTN_ERR_SCRATCH_LIMIT.
 */
#define ATTN_STATIC_SCRATCH_BYTES 33554432
ATTN_API int attn_fwd_splitkv_static(const void *Q, const void *K, const void *V, int mode,
                                     const float *C, const float *ckey, int BH, int Nq, int Nk,
                                     int d, int d_v, float scale, int n_splits, void *O,
                                     int out_dtype, float *LSE, void *stream);

/*
 * attn_fwd_host -- attn_fwd_ex on tensors that live in host memory (the pages have no
 * counterpart: this is a way of feeding the forward pass, not a step of the method).
 * Heads are independent, so the call cuts the BH heads into chunks and streams them:
 * the upload of one chunk, the attention of the previous one and the download of the
 * one before run at the same time, on three streams the library creates once per device,
 * through two slots of a caller-provided device staging buffer.
 *   Q, K, V, C, ckey  HOST pointers, the layouts and dtypes of attn_fwd_ex (C, ckey as the
 *                     mode requires, else NULL). Page-locked memory lets the copies overlap
 *                     the kernels; pageable memory works but the copies then serialise.
 *   O, LSE            HOST pointers for the outputs (LSE may be NULL).
 *   staging           device memory of the current device, 256-byte aligned, at least
 *                     attn_fwd_host_staging_bytes(...) bytes, owned by the caller; its
 *                     contents do not matter and are overwritten. It must not be used by
 *                     anything else until the work of this call on `stream` completes.
 *   staging_bytes     its size.
 *   heads_per_chunk   heads per chunk, >= 0; 0 lets the library choose: about eight chunks,
 *                     but at least as many heads as 128 blocks need (one block per 128
 *                     queries with a dense bias, per 256 otherwise), so each launch fills
 *                     the GPU.
 *   stream            the caller's stream: the call's work starts after work already queued
 *                     on it, and work queued on it afterwards waits for the last download.
 * The call queues the work and returns (asynchronous, like attn_fwd_ex); the host outputs
 * are complete when `stream` has reached the point after the call. The results are
 * bit-identical to attn_fwd_ex on the same data (the same kernel per head). Host buffers
 * must not be written, nor outputs read, until then. Calls are serialised on a mutex
 * while they queue their work.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG (a device pointer where a host pointer belongs,
 * overlapping host buffers, staging too small or misaligned, bad sizes or mode), or what
 * attn_fwd_ex or the CUDA runtime returns; after an error some chunks may already have
 * been queued and the outputs are unspecified.
 */
ATTN_API int attn_fwd_host(const void *Q, const void *K, const void *V, int mode, const float *C,
                           const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                           void *O, int out_dtype, float *LSE, void *staging,
                           unsigned long long staging_bytes, int heads_per_chunk, void *stream);

/*
 * attn_fwd_host_staging_bytes -- the staging size attn_fwd_host needs for these
 * arguments (two chunk slots of Q, K, V, the bias, O and LSE, each 256-byte aligned; one
 * slot when everything fits one chunk). Makes no CUDA call. Returns ATTN_OK, or
 * ATTN_ERR_INVALID_ARG (NULL bytes, bad sizes, mode or dtype, negative heads_per_chunk).
 */
ATTN_API int attn_fwd_host_staging_bytes(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                         int out_dtype, int heads_per_chunk,
                                         unsigned long long *bytes);

/*
 * attn_bwd -- gradients dQ, dK, dV of O = softmax(Q K^T * scale + C) V for a loss
 * gradient dO, on `stream`. They are the derivatives of the attn_fwd_ex operation:
 *     dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = dO_i . O_i,
 *     dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
 * with P recomputed tile by tile from Q, K, the bias and the forward's LSE instead of
 * being stored ("Compilers and kernels", section "FlashAttention rewrites the algorithm
 * around IO", the remark after the recurrence that the backward pass recomputes the
 * score and probability blocks). The bias C itself gets no gradient.
 * Arguments (device pointers):
 *   Q, K, V, mode, C, ckey, BH, Nq, Nk, d, d_v, scale
 *            exactly as given to attn_fwd_ex for the forward pass
 *   O        that forward pass's output [BH][Nq][d_v], element type o_dtype
 *            (ATTN_OUT_BF16 or ATTN_OUT_F32)
 *   dO       bf16 [BH][Nq][d_v], the gradient of the loss with respect to O
 *   LSE      fp32 [BH][Nq], the forward pass's LSE (required here)
 *   dQ       fp32 [BH][Nq][d];  dK fp32 [BH][Nk][d];  dV fp32 [BH][Nk][d_v]  (outputs)
 *   workspace device memory of attn_bwd_workspace_bytes(BH, Nq) bytes, 16-byte aligned,
 *            for the per-row statistics (-LSE in log2 units and D); overwritten
 * Alignment: Q, K, V, O, dO, C, dQ, dK, dV 16 bytes; LSE, ckey 4 bytes.
 * Aliasing: dQ, dK, dV and the workspace overlap no input and no other output.
 * Nq == 0 writes zeros to dK and dV; Nk == 0 with Nq >= 1 is rejected.
 * Rows whose LSE is -inf (no allowed key) contribute nothing and get dQ_i = 0.
 * Three kernels run on `stream` (row statistics, then dK/dV, then dQ); no atomics, so
 * the result is deterministic. Errors as for attn_fwd_ex.
 */
ATTN_API int attn_bwd(const void *Q, const void *K, const void *V, const void *O, int o_dtype,
                      const void *dO, const float *LSE, int mode, const float *C, const float *ckey,
                      int BH, int Nq, int Nk, int d, int d_v, float scale, float *dQ, float *dK,
                      float *dV, void *workspace, unsigned long long workspace_bytes, void *stream);

/* attn_bwd_workspace_bytes -- the workspace attn_bwd needs: 2 x BH x ceil(Nq/128) x 128
 * x 4 bytes. Returns ATTN_OK, or ATTN_ERR_INVALID_ARG (BH < 1, Nq < 0, NULL bytes). */
ATTN_API int attn_bwd_workspace_bytes(int BH, int Nq, unsigned long long *bytes);

/*
 * attn_bwd_host -- attn_bwd on tensors that live in host memory, streamed through the GPU
 * in chunks of heads like attn_fwd_host (no counterpart on the pages either).
 *   Q, K, V, O, dO, LSE, C, ckey  HOST pointers, the layouts and dtypes of attn_bwd.
 *   dQ, dK, dV        HOST pointers for the fp32 gradients.
 *   staging, staging_bytes, heads_per_chunk, stream  as for attn_fwd_host, with the size
 *                     from attn_bwd_host_staging_bytes (the chunks also hold each one's
 *                     row-statistics workspace). By default a chunk holds about an eighth
 *                     of the heads, but at least as many as 128 blocks need (one block per
 *                     128-query or 128-key tile, whichever count is larger).
 * Asynchronous on `stream` like attn_bwd; the gradients are bit-identical to attn_bwd's.
 * Returns what attn_fwd_host returns for the same kinds of error, or what attn_bwd returns.
 */
ATTN_API int attn_bwd_host(const void *Q, const void *K, const void *V, const void *O, int o_dtype,
                           const void *dO, const float *LSE, int mode, const float *C,
                           const float *ckey, int BH, int Nq, int Nk, int d, int d_v, float scale,
                           float *dQ, float *dK, float *dV, void *staging,
                           unsigned long long staging_bytes, int heads_per_chunk, void *stream);

/* attn_bwd_host_staging_bytes -- the staging size attn_bwd_host needs; no CUDA call. */
ATTN_API int attn_bwd_host_staging_bytes(int mode, int BH, int Nq, int Nk, int d, int d_v,
                                         int o_dtype, int heads_per_chunk,
                                         unsigned long long *bytes);

/* Static English text for a return code (never NULL). The pages have no counterpart: it
 * spells out the error part of the kernel contract (shapes, layout, aliasing, errors) that
 * "AI compiler engineer: how a compute graph becomes a GPU kernel" asks every kernel
 * interface to state. */
ATTN_API const char *attn_strerror(int code);

/*
 * attn_device_status -- synchronizes `stream` (NULL: the legacy default stream),
 * then reads and clears the current device's watchdog word. Every pipeline wait in
 * the kernels is bounded; a wait that runs out records where it stopped in that
 * word and the kernel returns without hanging the device. This is the pages' advice
 * for a program that stops making progress ("AI Infra ch. 5", section 5.1, the passage
 * on telling a slow program from a stuck one: every wait names the event it waits for,
 * and a wait is given a timeout after which it reports what was still outstanding).
 * Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT, or ATTN_ERR_CUDA / ATTN_ERR_NO_DEVICE
 * when the synchronization or the read itself fails.
 * If `detail` is not NULL it receives the raw watchdog word (0 when clear).
 */
ATTN_API int attn_device_status(void *stream, unsigned int *detail);

/*
 * attn_set_wait_timeout_ns -- the bound on each pipeline wait inside the kernels,
 * in nanoseconds, for launches that follow (process-wide). 0 restores the default
 * of 2 seconds. Returns the previous value.
 */
ATTN_API unsigned long long attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * attn_set_fault_injection -- test hook for the watchdog (process-wide, for launches
 * that follow). ATTN_FAULT_SKIP_FIRST_K makes each CTA's first K tile never be
 * copied, so the wait on it runs out after the wait timeout: the kernel records the
 * timeout in the watchdog word, every warp of the CTA stops waiting, copies already
 * issued are drained, tensor memory is freed and the kernel returns. Outputs of such a
 * launch are undefined. ATTN_FAULT_NONE (the default) turns it off.
 * Returns ATTN_OK, or ATTN_ERR_INVALID_ARG for an unknown value.
 */
#define ATTN_FAULT_NONE 0
#define ATTN_FAULT_SKIP_FIRST_K 1
ATTN_API int attn_set_fault_injection(int fault);

/* ABI version of this header (major * 100 + minor): 1.00 attn_fwd; 1.01 attn_fwd_ex;
 * 1.02 attn_fwd_splitkv, attn_fwd_splitkv_plan; 1.03 attn_fwd_splitkv_static;
 * 1.04 attn_bwd, attn_bwd_workspace_bytes; 1.05 attn_fwd_host, attn_fwd_host_staging_bytes;
 * 1.06 attn_bwd_host, attn_bwd_host_staging_bytes; 1.07 ATTN_BIAS_SHARED (one dense bias for
 * all heads). attn_version() returns the library's. */
#define ATTN_ABI_VERSION 107
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TILED_ATTENTION_13_ATTN_H */

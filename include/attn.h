/*
 * attn.h -- C ABI of libattn: the tiled (FlashAttention) forward pass on
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (lynx-cortex phase-27 lab 02 "Forward de flash attention en
 * Triton", kernel skeleton and "Bloque C"; cruxr.ai "Optimizaciones de
 * Atencion", section "FlashAttention: Nunca materializar la matriz de
 * atencion"): for every batch b, query head h and query row i,
 *
 *   O[b,h,i,:] = sum_j softmax_j(sm_scale * Q[b,h,i,:] . K[b,kvh,j,:] + mask) V[b,kvh,j,:]
 *   LSE[b,h,i] = ln sum_j exp(sm_scale * Q[b,h,i,:] . K[b,kvh,j,:] + mask)
 *
 * computed tile by tile with the online-softmax recurrence so that the score
 * matrix never reaches device memory.
 *   - GQA/MQA: Hq query heads share Hkv K/V heads, kvh = h / (Hq / Hkv)
 *     (consecutive groups; cruxr.ai "Multi-Head Latent Attention" recap of
 *     GQA and the motivation page's "Grouped/Multi-Query Attention").
 *   - causal: key j is visible to query i iff j <= Nk - Nq + i (the square
 *     case Nq == Nk keeps j <= i, "position i attends to itself", lab 02
 *     "Errores tipicos"; for Nq < Nk the queries are the last Nq positions).
 *   - window > 0 (requires causal): additionally Nk - Nq + i - j < window,
 *     i.e. the last `window` tokens including itself (motivation page,
 *     "Sliding window attention").
 *   - LSE is the natural-log log-sum-exp of the scaled, masked scores (the
 *     lab 02 skeleton stores m + log(l)).
 *
 * Layout: Q, O are (B, Hq, Nq, d) and K, V are (B, Hkv, Nk, d), dense
 * row-major (d fastest), elements fp16 or bf16; LSE is (B, Hq, Nq) fp32.
 * All pointers are DEVICE pointers on the current device, 16-byte aligned,
 * except where a function says HOST.
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory on any call, never synchronises, and only enqueues work on `stream`;
 * results are complete when the stream reaches that point.  O and LSE are
 * fully overwritten; LSE may be NULL (then it is not written).  Q, K, V are
 * read only.  Outputs must not alias inputs.
 *
 * Errors: every call validates its arguments on the host and returns a status
 * without launching anything when they are bad.  No C++ exception crosses the
 * ABI.  Launch failures return ATTN_ERR_CUDA.  Kernels bound every internal
 * wait; a wait that runs out records ATTN_ERR_TIMEOUT in a per-device status
 * word that attn_device_status() reads back.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 1

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, size <= 0, Hq % Hkv != 0,
                               window < 0, window > 0 without causal, causal with
                               Nq > Nk, sm_scale not finite or <= 0, bad dtype,
                               workspace too small */
  ATTN_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, or no sm_100-family GPU */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a kernel's bounded internal wait ran out */
  ATTN_ERR_SCRATCH_LIMIT = 5, /* attn_fwd_decode_noalloc: the shape needs more than the
                                 library's built-in scratch, or does not take the
                                 split-KV path at all */
  ATTN_ERR_DEVICE_ARG = 6     /* reported by attn_device_status(): a kernel found a
                                 device-side argument out of range (attn_fwd_paged:
                                 a page index or a sequence length) */
} attn_status_t;

typedef enum { ATTN_DTYPE_FP16 = 0, ATTN_DTYPE_BF16 = 1 } attn_dtype_t;

/* The kernels a call runs (see attn_fwd_ex). */
typedef enum {
  ATTN_PATH_PREFILL = 0,       /* tiled tcgen05 kernel: one launch */
  ATTN_PATH_SPLIT_KV = 1,      /* split-KV kernel + merge kernel: two launches */
  ATTN_PATH_SHORT = 2,         /* short-key kernel (Nk <= 128): one launch */
  ATTN_PATH_PREFILL_SPLIT = 3, /* tiled tcgen05 kernel, work split evenly over the
                                  SMs by K/V tiles (stream-K): one launch */
  ATTN_PATH_SPLIT_KV_FUSED = 4 /* split-KV kernel whose last CTA to finish in each
                                  query group merges the group (small merges): one
                                  launch */
} attn_path_t;

/* Square attention, Nq = Nk = N.  Equivalent to attn_fwd_ex with Nq = Nk = N
 * and no workspace. */
attn_status_t attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int Hq,
                       int Hkv, int N, int d, int causal, int window, float sm_scale, attn_dtype_t dtype,
                       cudaStream_t stream);

/* General call with Nq query rows against Nk keys (Nq <= Nk when causal; a
 * decode step is Nq = 1 against an Nk-token cache).
 *
 * Paths: a call with Nk <= 128 runs the short-key kernel (every head's keys
 * fit one tile; the workspace, if any, is not used).  Otherwise, with a
 * workspace: the split-KV path for small query groups (decode); else, for a
 * d = 128 call without a window whose 128-row tile pairs fill less than two
 * waves of CTAs, the prefill kernel with its work split evenly over the SMs
 * by K/V tiles.  Otherwise the tiled prefill kernel.  attn_fwd_path() says
 * which.
 *
 * workspace/workspace_bytes: optional DEVICE scratch for the split paths.
 * Both keep, for keys processed apart, a partial max, sum and output per
 * query row and combine them by rescaling with exp(m_p - m) (cruxr.ai
 * "FlashDecoding"): the split-KV path in a second kernel, the prefill split
 * in the CTA that holds the first keys of the rows.  When workspace is NULL
 * the non-split paths run.  When it is given it must hold at least
 * attn_fwd_workspace_bytes(...) bytes, 16-byte aligned, and must not be used
 * by another call that overlaps on the GPU.  Its contents need no
 * initialisation: the split kernels' cross-CTA handshake words carry a tag
 * of the enqueued call, and every launch leaves them cleared, so a CUDA
 * graph that captured the call may replay it with new inputs written in
 * place.  A launch that ends with ATTN_ERR_TIMEOUT may leave a prefill-split
 * handshake word set: clear the workspace (all zero bytes) before a graph
 * replays onto it again.  The prefill split has the CTAs
 * of one launch wait (bounded) for each other, so it expects its CTAs (one
 * per SM, at most the SM count) to be resident together; a concurrent
 * kernel that holds SMs for longer than the wait limit ends the call with
 * ATTN_ERR_TIMEOUT. */
attn_status_t attn_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int Hq,
                          int Hkv, int Nq, int Nk, int d, int causal, int window, float sm_scale,
                          attn_dtype_t dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Scratch bytes the split paths want for this shape on the current device:
 * the split-KV path's when the shape takes it (GQA groups of at most 32
 * query rows, i.e. (Hq / Hkv) * Nq <= 32, such as a decode step), else the
 * prefill split's when the shape takes it (d = 128, no window, fewer 128-row
 * tile pairs than twice the SM count), else 0.  The size depends on the device's
 * SM count. */
size_t attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/* The path (attn_path_t) that attn_fwd_ex takes for these sizes on the
 * current device, with (with_workspace != 0) or without a workspace of
 * attn_fwd_workspace_bytes(...) bytes, for a call without a window; -1 when
 * the sizes are invalid.  A window turns ATTN_PATH_PREFILL_SPLIT into
 * ATTN_PATH_PREFILL; the causal flag, dtype and scale do not change the
 * path.  No device work. */
int attn_fwd_path(int B, int Hq, int Hkv, int Nq, int Nk, int d, int with_workspace);

/* The split-KV plan for these sizes on a device of `sms` SMs holding
 * `ctas_per_sm` split CTAs each (the occupancy of the split kernel), without
 * device work (cruxr.ai "FlashDecoding": the keys are cut into chunks that
 * are processed in parallel, then merged).  `paged` selects the call:
 * 0 attn_fwd_ex on a flat 16-bit cache (chunks minimise CTAs per SM x
 * (tiles per CTA + 6)), 1 attn_fwd_paged (waves of resident CTAs x (tiles
 * per CTA + 2), then at most 2048 keys a chunk; max_seq_len = Nk), 2
 * attn_fwd_kv_int8 (the waves model, no cap).  info (HOST, 5 values,
 * written): chunks per GQA group, keys per chunk (a multiple of 64; the last
 * chunk may be shorter), 1 when each group's last CTA to finish merges (one
 * launch) else 0, byte offset of the per-group arrival counters (8 bytes
 * each) in the workspace, and the workspace bytes.  Returns 0, or -1 when
 * the shape does not take the split-KV path ((Hq / Hkv) * Nq > 32,
 * B * Hkv > 65535, bad sizes) or `paged` is not 0, 1 or 2. */
int attn_fwd_decode_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int paged, int sms, int ctas_per_sm,
                         long long *info);

/* The prefill kernel's schedule for these sizes, without device work: what
 * attn_fwd_ex would launch on a device of `sms` SMs (lab 02, "La estructura
 * del kernel": one program per batch x head and query tile, here query tiles
 * of 128 rows as independent units, each walking its live K/V tiles of 128
 * keys).  Only for shapes that take a prefill path
 * (ATTN_PATH_PREFILL or ATTN_PATH_PREFILL_SPLIT); returns -1 for invalid
 * sizes, a shape of another path or sms <= 0.
 *   info (HOST, 4 ints, written): grid (CTAs), schedule (0 one tile pass per
 *     item, 1 work split by K/V tiles, 2 two warpgroups on one tile's
 *     halves), item shape (0 consecutive row tiles, 1 two heads of a group,
 *     2 one tile, 3 one tile in halves), item count.
 *   visits (HOST, 6 ints per visit, written up to max_visits visits): one
 *     visit per (query tile, K/V tile) product that a softmax warpgroup
 *     computes, in each CTA's order and, within a piece of work, in the
 *     order the K/V ring is loaded: {cta, item, tile slot (0 or 1), b * Hq +
 *     h, first query row, K/V tile index}.
 * Returns the number of visits (it may exceed max_visits: then only the
 * first max_visits are written). */
int attn_fwd_prefill_visits(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window,
                            int with_workspace, int sms, int *info, int *visits, int max_visits);

/* Attention over a paged K/V cache (the motivation page, "PagedAttention es
 * un problema distinto": the cache is a pool of fixed-size pages, each
 * request has a page table listing the pages that hold its tokens in order,
 * and the attention kernel follows the table instead of reading a flat K and
 * V).  Same result as attn_fwd_ex on each request's K and V gathered into
 * order, with that request's own key count.  GQA groups of at most 32 query
 * rows ((Hq / Hkv) * Nq <= 32: a decode step, or a few speculative tokens)
 * run the split-KV kernel; larger groups (a prefill, or chunks of one,
 * against a paged cache) run the tiled tcgen05 prefill kernel, whose TMA
 * producer follows the page table, one copy per page.
 *
 * Q (DEVICE, B x Hq x Nq x d), O (DEVICE, same), LSE (DEVICE fp32, B x Hq x
 *   Nq, or NULL): as attn_fwd_ex.  Query row i of request b sits at key
 *   position seq_lens[b] - Nq + i (the causal mask is bottom-right aligned).
 * K_pages, V_pages (DEVICE, 16-byte aligned): the pools, num_pages x Hkv x
 *   page_size x d, 16-bit; page p of head h holds page_size consecutive
 *   tokens of whichever request's table lists p.
 * block_table (DEVICE int32, B x max_pages_per_seq, row-major): entry
 *   [b][j] is the pool page holding tokens [j * page_size, (j + 1) *
 *   page_size) of request b.  Entries past ceil(seq_lens[b] / page_size) are
 *   not read.
 * seq_lens (DEVICE int32, B): tokens in each request's cache, 1 <=
 *   seq_lens[b] <= max_seq_len, and >= Nq when causal.  Pool slots past a
 *   request's length may hold anything (NaN included): they are not used.
 * page_size: a power of two from 8 to 256.  max_pages_per_seq * page_size
 *   must cover max_seq_len; num_pages * Hkv must stay below 2^31 - 1.
 * workspace (DEVICE, 16-byte aligned): at least
 *   attn_fwd_paged_workspace_bytes(...) bytes, not used by an overlapping
 *   call; required by the split-KV path, not used (may be NULL) by the
 *   prefill path, whose workspace size is 0.
 * The host checks everything it can see; a page index outside [0,
 * num_pages) or a length out of range is found by the kernel, which reads
 * zeros for that page (or clamps the length), finishes the call and records
 * ATTN_ERR_DEVICE_ARG for attn_device_status().  Enqueued on `stream`;
 * nothing is allocated; the call does not synchronise. */
attn_status_t attn_fwd_paged(const void *Q, const void *K_pages, const void *V_pages, const int *block_table,
                             const int *seq_lens, void *O, float *LSE, int B, int Hq, int Hkv, int Nq,
                             int max_seq_len, int d, int page_size, int num_pages, int max_pages_per_seq,
                             int causal, int window, float sm_scale, attn_dtype_t dtype, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_fwd_paged wants for these sizes on the current device
 * (the split-KV scratch for max_seq_len keys); 0 when the sizes are invalid
 * or the call takes the prefill path (query groups of more than 32 rows). */
size_t attn_fwd_paged_workspace_bytes(int B, int Hq, int Hkv, int Nq, int max_seq_len, int d);

/* The path attn_fwd_paged takes for these sizes on the current device:
 * ATTN_PATH_SPLIT_KV_FUSED (each group's last CTA to finish merges the
 * chunks: one launch), ATTN_PATH_SPLIT_KV (a second, merge kernel), or
 * ATTN_PATH_PREFILL (query groups of more than 32 rows: the tiled kernel,
 * one launch); -1 when the sizes are invalid.  The paged split plan caps
 * the keys per chunk, since request lengths are known only on the device,
 * so it can split more finely than the flat call of max_seq_len keys.  No
 * device work. */
int attn_fwd_paged_path(int B, int Hq, int Hkv, int Nq, int max_seq_len, int d);

/* Decode over an INT8 K/V cache (cruxr.ai "Optimizaciones de Atencion",
 * section "Elegir optimizaciones de atencion": INT8 quantisation of the KV
 * cache is among the optimisations that compose with the others; the page
 * gives no scheme, so this is the plainest one).  K = k_scale * K_codes and
 * V = v_scale * V_codes with symmetric int8 codes (-127..127) and one fp32
 * scale per tensor; otherwise the same result as attn_fwd_ex on the
 * dequantised K and V.  The kernel loads the codes (half the bytes of a
 * 16-bit cache), widens them exactly to the dtype of Q, folds k_scale into
 * the softmax scale and v_scale into O.
 *
 * K_codes, V_codes (DEVICE, int8, B x Hkv x Nk x d, dense, 16-byte aligned);
 *   every other argument as attn_fwd_ex.  Only shapes that take the split-KV
 *   path (query groups of at most 32 rows: (Hq / Hkv) * Nq <= 32) are served;
 *   others return ATTN_ERR_UNSUPPORTED.  workspace (DEVICE, required, 16-byte
 *   aligned): at least attn_fwd_kv_int8_workspace_bytes(...) bytes, laid
 *   out as attn_fwd_ex's split-KV workspace (its chunk plan differs: two
 *   resident CTAs per SM pay for the widening work).
 *   k_scale, v_scale: finite and > 0, else ATTN_ERR_INVALID_ARG. */
attn_status_t attn_fwd_kv_int8(const void *Q, const void *K_codes, const void *V_codes, float k_scale,
                               float v_scale, void *O, float *LSE, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                               int causal, int window, float sm_scale, attn_dtype_t dtype, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_fwd_kv_int8 wants for these sizes on the current
 * device; 0 when the shape takes no split-KV path.  No device work. */
size_t attn_fwd_kv_int8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/* Backward pass: the gradients of the forward definition for an upstream
 * gradient dO (the pages store the log-sum-exp "for the backward pass":
 * cruxr.ai "FlashAttention: Nunca materializar la matriz de atencion", lab 02
 * kernel skeleton; the pages defer the backward itself).  With P recomputed
 * tile by tile from Q, K and the forward's LSE, P = exp(sm_scale * Q K^T -
 * LSE) (masked entries 0):
 *   dV = P^T dO,   dS = P o (dO V^T - D) with D = rowsum(dO o O),
 *   dK = sm_scale * dS^T Q,   dQ = sm_scale * dS K,
 * dK and dV summed over the query heads of each K/V head.  P and dS are
 * rounded to the input dtype before their products, as the forward rounds P.
 *
 * Q, K, V, causal, window, sm_scale, dtype: those of the forward call.  O
 *   (B x Hq x Nq x d) and LSE (fp32, B x Hq x Nq, required): its outputs.
 *   dO (B x Hq x Nq x d): the upstream gradient.  dQ (like Q), dK, dV (like
 *   K): outputs, fully written.  All DEVICE, 16-byte aligned.
 * workspace (DEVICE, 16-byte aligned, required): at least
 *   attn_bwd_workspace_bytes(B, Hq, Nq, d) bytes (an fp32 dQ accumulator and
 *   D), not used by an overlapping call; its contents need no
 *   initialisation.  Three kernels are enqueued on `stream` (D and the
 *   accumulator; the gradients; dQ); nothing is allocated; no sync.
 * Errors as attn_fwd_ex; B * Hkv * ceil(Nk / 128) must stay below 2^31. */
attn_status_t attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                       void *dQ, void *dK, void *dV, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                       int window, float sm_scale, attn_dtype_t dtype, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);
size_t attn_bwd_workspace_bytes(int B, int Hq, int Nq, int d);

/* The backward kernel's CTA order for these sizes on a device of `sms` SMs,
 * without device work: one CTA per (K/V group bk = b * Hkv + kvh, key tile
 * kt of 128 keys), in bands of ceil(2 * sms / key tiles) groups (two waves),
 * within a band in key-tile order (under a causal mask the longest first;
 * lab 02, "La estructura del kernel": one program per head and tile).
 * tiles (HOST, 2 ints per CTA, written up to max_ctas CTAs): {bk, kt} in
 * launch order.  Returns the CTA count, or -1 for bad sizes. */
int attn_bwd_cta_order(int B, int Hkv, int Nk, int sms, int *tiles, int max_ctas);

/* Attention over a latent K/V cache with absorbed queries (Multi-Head
 * Latent Attention; cruxr.ai "Optimizaciones de Atencion", section
 * "Multi-Head Latent Attention (MLA)").  Each token caches one latent vector
 * c_t of d_c values; head h's keys and values are c W_K,h and c W_V,h.  With
 * the up-projections absorbed (the same section: the attention is rewritten
 * to work on the compressed form), head h's score for token t is
 * sm_scale * (q~_h . c_t) with q~_h = W_K,h q_h, and its output is o~_h W_V,h
 * with o~_h = sum_t P_t c_t.  This call computes o~ and the log-sum-exp for
 * every head and query: standard attention with one K/V head whose keys and
 * values are both the latent vectors.  The projections themselves (q -> q~,
 * o~ -> o) are ordinary matrix products outside this call.
 *
 * Q_lat (DEVICE, B x n_h x Nq x d_c, dense, dtype): the absorbed queries q~.
 * C_lat (DEVICE, B x Nk x d_c, dense, dtype): the latent cache.
 * O_lat (DEVICE, B x n_h x Nq x d_c, dense, written): o~.
 * LSE (DEVICE fp32 B x n_h x Nq, natural log; may be NULL).
 * d_c: 512 (the width of the page's example); other values return
 *   ATTN_ERR_UNSUPPORTED.  causal / window / sm_scale as attn_fwd_ex, with
 *   query i of every head at position Nk - Nq + i (the last Nq tokens).
 * workspace (DEVICE, required, 16-byte aligned): at least
 *   attn_fwd_mla_workspace_bytes(...) bytes; the partial results of the key
 *   chunks, fully overwritten by every call (no initialisation needed).
 * Pointers 16-byte aligned, else ATTN_ERR_INVALID_ARG.  With at least 17
 * query rows per request (n_h * Nq) the tensor-core kernel runs (pairs of
 * CTAs, one per half of the 512 output columns, per 128 rows and key
 * chunk), otherwise a warp-MMA kernel; either is followed by the merge
 * kernel when the keys are split into more than one chunk.  Enqueued on
 * `stream`; nothing is allocated; the call does not synchronise. */
attn_status_t attn_fwd_mla(const void *Q_lat, const void *C_lat, void *O_lat, float *LSE, int B, int n_h, int Nq,
                           int Nk, int d_c, int causal, int window, float sm_scale, attn_dtype_t dtype,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_fwd_mla wants for these sizes on the current device
 * (at least 256); 0 when the sizes are invalid or d_c is not 512.  No
 * device work. */
size_t attn_fwd_mla_workspace_bytes(int B, int n_h, int Nq, int Nk, int d_c);

/* End-to-end call on HOST buffers: copies Q, K, V (HOST, ideally pinned) into
 * the caller's DEVICE staging buffer `dev_buf`, runs attn_fwd_ex, and copies O
 * (and LSE when non-NULL) back into HOST memory, all enqueued on `stream`.
 * dev_buf must hold attn_fwd_host_staging_bytes(...) bytes (256-byte aligned);
 * that size includes the workspace of a split path when the shape takes one.
 * The host buffers must stay valid until the stream reaches the end of the
 * call; pinned host memory lets the copies run asynchronously.
 *
 * Large calls (Q, K and V of at least 64 MiB, on the plain prefill path) are
 * cut into up to 16 pieces of contiguous (request, K/V head) slabs, so that
 * the copies of one piece overlap the compute of the others: each piece's
 * inputs are copied in on an internal stream, its kernel runs on `stream`
 * after them, and its outputs are copied out on a second internal stream.
 * `stream` is forked to the internal streams at the start of the call and
 * joined at its end, and a piece is computed with the same schedule as the
 * whole call, so the results are the same bits as without pieces.  The
 * internal streams and events are created on the first such call on a
 * device and kept; one pipelined call is enqueued at a time per device (a
 * lock).  A call on a stream that is being captured into a CUDA graph is
 * not cut (copy, compute, copy on `stream`), so a capture never involves
 * the shared internal streams. */
attn_status_t attn_fwd_host(const void *Q_host, const void *K_host, const void *V_host, void *O_host,
                            float *LSE_host, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                            int window, float sm_scale, attn_dtype_t dtype, void *dev_buf, size_t dev_buf_bytes,
                            cudaStream_t stream);
size_t attn_fwd_host_staging_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int with_lse);

/* Synchronises `stream`, then reads and clears the current device's kernel
 * status word: ATTN_OK; ATTN_ERR_TIMEOUT if a kernel gave up a wait since the
 * last call; ATTN_ERR_DEVICE_ARG if a kernel found a device-side argument out
 * of range (the first such event is kept).  Returns ATTN_ERR_CUDA if the
 * synchronisation fails. */
attn_status_t attn_device_status(cudaStream_t stream);

/* Test hook: sets the bound, in nanoseconds, on every internal kernel wait of
 * later launches on any device (default 2e9).  0 restores the default. */
void attn_set_wait_timeout_ns(unsigned long long ns);

/* Test hook: in later launches on any device, the kernels' TMA producers
 * stop loading after `tiles` K/V tiles (per CTA; for the short-key kernel,
 * per unit of work) and wait for nothing more, so that the roles waiting for
 * the missing tiles run into their bounded waits: the call still returns,
 * with ATTN_ERR_TIMEOUT recorded for attn_device_status(), and its outputs
 * are not valid.  A negative value (the default) turns the hook off.  For
 * testing the error path only. */
void attn_set_test_stall(int tiles);

/* Static description of a status code. */
const char *attn_status_string(attn_status_t status);

/* ATTN_ABI_VERSION of the loaded library. */
int attn_abi_version(void);

/* Measurement aid with no counterpart in the pages: launches an empty kernel
 * on `stream` the way every kernel here is launched (programmatic dependent
 * launch, `grid` CTAs of `threads` threads, `smem_bytes` of dynamic shared
 * memory), so that the fixed cost of a launch in a stream or a CUDA graph can
 * be measured next to a call.  ATTN_ERR_INVALID_ARG for grid < 1, threads
 * outside 1..1024 or more than 227 KB of shared memory. */
attn_status_t attn_empty_launch(int grid, int threads, size_t smem_bytes, cudaStream_t stream);

/* Split-KV decode that allocates nothing: the same computation as attn_fwd_ex
 * with a workspace, but its scratch lives in a fixed array inside the
 * library, so the caller passes only inputs and outputs.  The pages have no
 * counterpart; it exists for callers that cannot hand the library any extra
 * device memory, for example a host application whose device memory is all
 * owned by its own pool and that offers plugins no allocation hook, or a
 * serving loop that may not call cudaMalloc (which can synchronise the device)
 * while requests are in flight.
 *
 * Q, K, V, O, LSE, sizes, masks, dtype and stream mean what they mean for
 * attn_fwd_ex.  Only shapes that take the split-KV path qualify
 * ((Hq / Hkv) * Nq <= 32), and their scratch (attn_fwd_workspace_bytes) must
 * fit in the built-in 8 MiB; anything else returns ATTN_ERR_SCRATCH_LIMIT
 * without launching.
 *
 * The scratch array is a single 8 MiB block per GPU, reserved for as long as
 * the library is loaded.  Every call on a device uses the same block and
 * leaves its contents behind; nothing in it needs to start at zero: every
 * value a call reads was written earlier in that call, except the per-group
 * arrival counters of the merge, which carry a tag of the call (a word with
 * another tag counts as zero) and which the call leaves at zero arrivals.
 * Calls whose
 * work overlaps on the GPU (different streams without ordering between them)
 * race on the block and give wrong results: order them on one stream.
 * The first call on a device looks up the block's device address; make that
 * first call before any stream capture begins on that device. */
attn_status_t attn_fwd_decode_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                                      int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window,
                                      float sm_scale, attn_dtype_t dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */

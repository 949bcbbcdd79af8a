// attn_mla.cuh -- attention over a latent K/V cache (Multi-Head Latent
// Attention) for decode, with the up-projections absorbed.
//
// cruxr.ai "Optimizaciones de Atencion", section "Multi-Head Latent Attention
// (MLA)": each token caches one latent vector c_t of d_c values instead of
// per-head keys and values; head h's keys and values are K_h = c W_K,h and
// V_h = c W_V,h.  Absorbing the up-projections, head h's scores are
// q~_h . c_t with q~_h = W_K,h q_h, and its output is o~_h W_V,h with
// o~_h = sum_t P_t c_t.  So the attention itself runs on the latent: every
// head of a request (n_h heads x Nq queries = its query rows) attends to the
// same d_c-wide vectors, which serve as both keys and values.  This kernel
// computes, per query row, the latent output o~ and the log-sum-exp from the
// absorbed queries q~ (d_c = 512); the per-token projections are separate
// products.
//
// GB300 mapping: split-KV, like attn_decode.cuh.  Grid (key chunks, B x row
// blocks of 16): a CTA takes 16 query rows of one request and one chunk of
// its keys.  A producer warp streams 64-key latent tiles (64 keys x 512
// values, 64 KB: eight 128B-swizzled boxes) into a 3-stage ring; four
// consumer warps share each tile:
//   S:  warp w computes the scores of keys 16w..16w+15 for the 16 rows
//       (m16n8k16 MMAs over d_c = 512, fp32)
//   softmax: the warps exchange their row maxima through shared memory, so
//       every warp keeps the same running max per row (lazy rescale when it
//       grew by more than 2^8); each writes its 16 keys' P (16-bit) into a
//       shared 16 x 64 tile and its row sums
//   P V: warp w multiplies all 64 keys' P into its 128 of the 512 output
//       columns (the same latent tile, read as values)
// Each chunk writes its normalised partial output and log2 LSE to a
// workspace; the decode merge kernel (attn_decode_combine_kernel<512>)
// combines the chunks.
#pragma once

#include "attn_decode.cuh"

namespace attn {

constexpr int kMlaD = 512;   // latent width d_c
constexpr int kMlaRows = 16;  // query rows per CTA
constexpr int kMlaWarps = 4;  // consumer warps
constexpr int kMlaThreads = 32 * kMlaWarps + 32;
constexpr float kMlaRescale = 8.0f;  // lazy rescale: only when a row's max grew by more than 2^8

struct MlaParams {
  CUtensorMap tmC;  // (512, Nk, B), box 64 x 64 x 1, 128B swizzle
  const void *Q;    // (B, n_h, Nq, 512) absorbed queries, 16-bit
  float *ws;        // [B*n_h*Nq][nchunks][512]: normalised partial output per chunk
  float *ws_lse;    // [B*n_h*Nq][nchunks]: log2 LSE per chunk (-inf: no live key)
  int *status;
  int B, n_h, Nq, Nk, R;  // R = n_h * Nq query rows per request
  int row_blocks;         // ceil(R / 16)
  int causal, window;
  int nchunks, chunk_keys;
  float scale_log2;
  unsigned long long timeout_ns;
  int stall_after;  // test hook: the producer stops after this many tiles (-1: never)
};

struct MlaCfg {
  static constexpr int kStages = 3;
  static constexpr int kBoxBytes = kDecKeys * 128;       // 64 keys x 64 values x 2 bytes
  static constexpr int kTileBytes = kDecKeys * kMlaD * 2;  // 64 KB
  static constexpr int kOffQ = 0;                          // 16 rows x 512, eight 16-row boxes
  static constexpr int kOffP = kMlaRows * kMlaD * 2;       // [2][16 rows x 64 keys] 16-bit
  static constexpr int kOffRing = kOffP + 2 * kMlaRows * 64 * 2 + 1024 - ((kOffP + 2 * kMlaRows * 64 * 2) % 1024);
  static constexpr int kOffBar = kOffRing + kStages * kTileBytes;  // full[3], empty[3]; abort
  static constexpr int kOffStats = kOffBar + 128;  // [2][4 warps][16 rows] max, then sums
  static constexpr int kSmemBytes = kOffStats + 2 * 2 * kMlaWarps * kMlaRows * 4 + 1024;
  static_assert(kOffRing % 1024 == 0, "swizzled ring alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <bool BF16>
__global__ void __launch_bounds__(kMlaThreads, 1) attn_mla_kernel(const __grid_constant__ MlaParams p) {
  using C = MlaCfg;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  int *abort_flag = reinterpret_cast<int *>(bars + 2 * NS);
  float *smax = reinterpret_cast<float *>(smem + C::kOffStats);  // [buf][warp][row]
  float *ssum = smax + 2 * kMlaWarps * kMlaRows;                 // [buf][warp][row]
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sP0 = smem_u32(smem + C::kOffP);
  const uint32_t sRing = smem_u32(smem + C::kOffRing);
  const uint32_t bar0 = smem_u32(bars);
  auto bFull = [&](int s) { return bar0 + 8u * s; };
  auto bEmpty = [&](int s) { return bar0 + 8u * (NS + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3, jm = lane >> 3;
  const int chunk = blockIdx.x;
  const int b = blockIdx.y / p.row_blocks, rblk = blockIdx.y - b * p.row_blocks;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(bFull(s), 1);
      mbar_init(bEmpty(s), kMlaWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  const int k0 = chunk * p.chunk_keys;
  const int k1 = min(k0 + p.chunk_keys, p.Nk);
  const int ntiles = k1 > k0 ? (k1 - k0 + kDecKeys - 1) / kDecKeys : 0;
  bool ok = true;

  if (warp == kMlaWarps) {
    // ============================================================ TMA producer
    if (elect_one()) tma_prefetch_desc(&p.tmC);
    __syncwarp();
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (p.stall_after >= 0 && i >= p.stall_after) {  // test hook: stop loading
        ok = false;
        break;
      }
      const int s = i % NS;
      if (i >= NS && !mbar_wait_warp(bEmpty(s), ((i / NS) - 1) & 1, wc, kErrDecWaitKV)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(bFull(s), C::kTileBytes);
#pragma unroll
        for (int cc = 0; cc < kMlaD / 64; ++cc)
          tma_load_3d(sRing + s * C::kTileBytes + cc * C::kBoxBytes, &p.tmC, bFull(s), cc * 64, k0 + i * kDecKeys, b);
      }
      __syncwarp();
      issued = i + 1;
    }
    if (!ok && lane == 0)  // never leave with a copy of ours in flight
      for (int i = max(0, issued - NS); i < issued; ++i) mbar_drain_dec(bFull(i % NS), (i / NS) & 1);
  } else {
    // the block's 16 query rows -> shared memory (eight 16-row boxes, swizzled)
    for (int idx = threadIdx.x; idx < kMlaRows * (kMlaD / 8); idx += 32 * kMlaWarps) {
      const int r = idx / (kMlaD / 8), c8 = (idx % (kMlaD / 8)) * 8;
      const int qr = rblk * kMlaRows + r;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (qr < p.R)
        v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.Q) +
                                             (static_cast<size_t>(b) * p.R + qr) * kMlaD + c8);
      *reinterpret_cast<uint4 *>(smem + C::kOffQ + swz(kMlaRows, r, c8)) = v;
    }
    named_bar_and(1, 32 * kMlaWarps, true);  // Q staged
  }

  // rows g (h = 0) and g + 8 (h = 1) of the block
  float m[2], l[2];
  int pos[2];
  bool rowok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int qr = rblk * kMlaRows + g + 8 * h;
    m[h] = -INFINITY;
    l[h] = 0.f;
    rowok[h] = qr < p.R;
    pos[h] = p.Nk - p.Nq + (qr % p.Nq);  // row qr is query qr % Nq of head qr / Nq
  }
  float o[16][4];  // this warp's 128 output columns: 16 n-blocks of 8
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const float sl2 = p.scale_log2;

  for (int i = 0; warp < kMlaWarps && i < ntiles; ++i) {
    const int s = i % NS, buf = i & 1;
    if (!mbar_wait_warp(bFull(s), (i / NS) & 1, wc, kErrDecWaitKV)) ok = false;
    // every consumer warp takes the same decision, so that the barriers below stay matched
    if (!named_bar_and(2, 32 * kMlaWarps, ok)) {
      ok = false;
      break;
    }
    const uint32_t sT = sRing + s * C::kTileBytes;
    const int key_base = k0 + i * kDecKeys + warp * 16;
    // ---- S (16 rows x this warp's 16 keys) = Q~ C^T over 512
    float sc[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
    {
      const int krow = warp * 16 + (jm >> 1) * 8 + (lane & 7);
#pragma unroll 8
      for (int kk = 0; kk < kMlaD / 16; ++kk) {
        uint32_t kb[4], a[4];
        ldsm_x4(sT + swz(kDecKeys, krow, kk * 16 + (jm & 1) * 8), kb[0], kb[1], kb[2], kb[3]);
        ldsm_x4(sQ + swz(kMlaRows, (jm & 1) * 8 + (lane & 7), kk * 16 + (jm >> 1) * 8), a[0], a[1], a[2], a[3]);
        mma16816<BF16>(sc[0], a, kb[0], kb[1]);
        mma16816<BF16>(sc[1], a, kb[2], kb[3]);
      }
    }
    // ---- mask; the warps' row maxima -> the tile's
    float v[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_base + nb * 8 + 2 * tq + e;
          const bool live = rowok[h] && key < k1 && (!p.causal || key <= pos[h]) &&
                            (p.window <= 0 || pos[h] - key < p.window);
          v[h][nb * 2 + e] = live ? sc[nb][2 * h + e] : -INFINITY;
        }
      float tmax = fmaxf(fmaxf(v[h][0], v[h][1]), fmaxf(v[h][2], v[h][3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      if (tq == 0) smax[(buf * kMlaWarps + warp) * kMlaRows + g + 8 * h] = tmax;
    }
    named_bar_sync(3, 32 * kMlaWarps);
    float alpha[2];
    uint32_t pk[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = g + 8 * h;
      float tm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kMlaWarps; ++w) tm = fmaxf(tm, smax[(buf * kMlaWarps + w) * kMlaRows + r]);
      // every warp holds the same m[h]: the same lazy decision everywhere
      const float m_new = fmaxf(m[h], tm * sl2);
      alpha[h] = 1.f;
      if (m_new > m[h] + kMlaRescale) {
        alpha[h] = (m[h] == -INFINITY) ? 0.f : ex2_approx(m[h] - m_new);
        m[h] = m_new;
      }
      const float mref = (m[h] == -INFINITY) ? 0.f : m[h];
      float e4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) e4[q] = ex2_approx(fmaf(v[h][q], sl2, -mref));
      pk[h][0] = pack2<BF16>(e4[0], e4[1]);  // keys nb = 0: 2tq, 2tq + 1
      pk[h][1] = pack2<BF16>(e4[2], e4[3]);  // keys nb = 1
      float sum = (e4[0] + e4[1]) + (e4[2] + e4[3]);
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      if (tq == 0) ssum[(buf * kMlaWarps + warp) * kMlaRows + r] = sum;
    }
    // this warp's P (rows x its 16 keys) into the shared P tile [row][key]
    const uint32_t sP = sP0 + buf * (kMlaRows * 64 * 2);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        const int r = g + 8 * h, key = warp * 16 + nb * 8 + 2 * tq;
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sP + swz(kMlaRows, r, key)), "r"(pk[h][nb]) : "memory");
      }
    named_bar_sync(3, 32 * kMlaWarps);  // the P tile and the warps' sums are complete
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kMlaWarps; ++w) tot += ssum[(buf * kMlaWarps + w) * kMlaRows + g + 8 * h];
      l[h] = l[h] * alpha[h] + tot;
      if (alpha[h] != 1.f) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][2 * h] *= alpha[h];
          o[n][2 * h + 1] *= alpha[h];
        }
      }
    }
    // ---- O[:, 128w:128w+128] += P (16 x 64 keys) V (64 keys x 128)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4];
      ldsm_x4(sP + swz(kMlaRows, (jm & 1) * 8 + (lane & 7), ks * 16 + (jm >> 1) * 8), a[0], a[1], a[2], a[3]);
      const int vrow = ks * 16 + (jm & 1) * 8 + (lane & 7);
#pragma unroll
      for (int nn = 0; nn < 8; ++nn) {
        uint32_t vb[4];
        ldsm_x4_t(sT + swz(kDecKeys, vrow, warp * 128 + nn * 16 + (jm >> 1) * 8), vb[0], vb[1], vb[2], vb[3]);
        mma16816<BF16>(o[2 * nn], a, vb[0], vb[1]);
        mma16816<BF16>(o[2 * nn + 1], a, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bEmpty(s));  // this warp is done with tile i
  }
  if (__syncthreads_or(!ok)) return;
  // ---- this chunk's normalised output and log2 LSE -> workspace
  if (warp < kMlaWarps) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int qr = rblk * kMlaRows + g + 8 * h;
      if (qr >= p.R) continue;
      const size_t grow = static_cast<size_t>(b) * p.R + qr;
      const float inv = (l[h] > 0.f) ? 1.f / l[h] : 0.f;
      float *dst = p.ws + (grow * p.nchunks + chunk) * kMlaD + warp * 128;
#pragma unroll
      for (int n = 0; n < 16; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) = make_float2(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
      if (warp == 0 && tq == 0) p.ws_lse[grow * p.nchunks + chunk] = (l[h] > 0.f) ? m[h] + log2f(l[h]) : -INFINITY;
    }
  }
}

// ============================================================================
// The same attention on the 5th-generation tensor cores, for requests with
// more than a few query rows (n_h x Nq; 128 for one query of DeepSeek-V2's
// 128 heads).
//
// A CTA takes 128 query rows of one request, one chunk of its keys, and one
// half of the 512 output columns: two CTAs (adjacent in the grid, so they
// read the same latent tiles at the same time and the second read hits L2)
// share a row block and a chunk.  Each computes the full scores S = Q~ C^T
// (128 x 64 keys per tile, K = 512), its own softmax (both compute the same
// S bit for bit: the same MMAs in the same order), and O_half += P C_half
// (N = 256).  Tensor memory (512 columns) holds O_half (256), the half of
// Q~ whose columns the CTA does not output (128 columns of packed pairs:
// the A operand of half of the score MMAs) and two S buffers (64 each; P is
// written over S as 16-bit pairs and read from there by the P V MMA).  The
// other half of Q~ sits in shared memory (64 KB): with all of Q~ read from
// shared memory for every tile, the score MMAs would need more operand
// bandwidth than shared memory gives at N = 64.
//
// Latent tiles (64 keys) arrive as two halves of 256 columns (32 KB each,
// four 128B-swizzled boxes): the half this CTA outputs ("own", kept until
// its P V has run: a 3-slot ring) and the other half ("other", needed only
// by the score MMAs: a 2-slot ring, released as soon as they complete).
//
// Roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one lane)
// and TMEM owner, warps 2-5 softmax (one query row per thread; warp w reads
// TMEM lanes 32 (w % 4) ..).  Pipeline per tile i: S(i) is issued before
// P V(i-1), so the softmax of tile i overlaps the P V of tile i-1; S(i)
// reuses the buffer of P(i-2), whose P V was issued before it (the tensor
// pipe completes one CTA's MMAs in order).
constexpr int kMlaTcRows = 128;
constexpr int kMlaTcKeys = 64;
constexpr int kMlaTcThreads = 192;
constexpr int kMlaTcMinRows = 17;  // query rows per request from which this kernel is used

struct MlaTcCfg {
  static constexpr int kOwnSlots = 3, kOthSlots = 2;
  static constexpr int kBoxBytes = kMlaTcKeys * 128;      // 64 keys x 64 columns x 2 bytes
  static constexpr int kHalfBytes = 4 * kBoxBytes;         // 64 keys x 256 columns: 32 KB
  static constexpr int kQBoxBytes = kMlaTcRows * 128;      // 128 rows x 64 columns: 16 KB
  static constexpr int kOffQ = 0;                          // the own half of Q~: four boxes
  static constexpr int kOffOwn = kOffQ + 4 * kQBoxBytes;
  static constexpr int kOffOth = kOffOwn + kOwnSlots * kHalfBytes;
  static constexpr int kOffBar = kOffOth + kOthSlots * kHalfBytes;
  // barriers: own full/empty [3], other full/empty [2], Q, S full [2], P V done, O final, drain
  static constexpr int kNumBars = 2 * kOwnSlots + 2 * kOthSlots + 1 + 2 + 3;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers, TMEM slot, abort flag; alignment
  static_assert(kNumBars * 8 + 8 <= 256, "barriers fit");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM columns
  static constexpr uint32_t kColO = 0, kColQt = 256, kColS = 384, kTmemCols = 512;
};

struct MlaTcParams {
  CUtensorMap tmQ;  // (512, R, B), box 64 x 128 x 1, 128B swizzle
  CUtensorMap tmC;  // (512, Nk, B), box 64 x 64 x 1, 128B swizzle
  const void *Q;    // (B, R, 512): the TMEM half is loaded by the softmax threads
  void *O;          // direct output (nchunks == 1): (B, R, 512) 16-bit
  float *lse;       // direct output: (B, R) natural log, or null
  float *ws;        // nchunks > 1: [B*R][nchunks][512] normalised partials
  float *ws_lse;    // nchunks > 1: [B*R][nchunks] log2 LSE
  int *status;
  int B, Nq, Nk, R, row_blocks;
  int causal, window;
  int nchunks, chunk_keys;
  float scale_log2;
  unsigned long long timeout_ns;
  int stall_after;
};

enum MlaError : int { kErrMlaWait = 0x401 };

// Named barriers between the softmax warps (128, arrive) and the MMA warp
// (32, sync): P(i) written; the TMEM half of Q~ written.
constexpr uint32_t kBarMlaP = 1, kBarMlaQt = 2, kBarMlaThreads = 160;

// Four score MMAs of K = 16 with A from TMEM (column a + 8k) and a K-major B
// (descriptor b + 2k: 32 bytes further in the swizzle row); the first
// accumulates iff `accumulate` != 0.
__device__ __forceinline__ void umma_ts_x4_kmajor(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, p1;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 p1, %4, %4;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, p1;\n\t}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four P V MMAs of K = 16 keys: P at TMEM column a + 8k, B MN-major
// (descriptor b + 128k: 16 key rows = 2048 bytes further).
__device__ __forceinline__ void umma_ts_x4_mnmajor(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                                   uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, p1;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 p1, %4, %4;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, p1;\n\t}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kMlaTcThreads, 1) attn_mla_tc_kernel(const __grid_constant__ MlaTcParams p) {
  using C = MlaTcCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sOwn = smem_u32(smem + C::kOffOwn);
  const uint32_t sOth = smem_u32(smem + C::kOffOth);
  const uint32_t bar0 = smem_u32(bars);
  auto bOwnFull = [&](int s) { return bar0 + 8u * s; };
  auto bOwnEmpty = [&](int s) { return bar0 + 8u * (C::kOwnSlots + s); };
  auto bOthFull = [&](int s) { return bar0 + 8u * (2 * C::kOwnSlots + s); };
  auto bOthEmpty = [&](int s) { return bar0 + 8u * (2 * C::kOwnSlots + C::kOthSlots + s); };
  const uint32_t bX = bar0 + 8u * (2 * C::kOwnSlots + 2 * C::kOthSlots);
  const uint32_t bQ = bX;
  auto bSfull = [&](int t) { return bX + 8u * (1 + t); };
  const uint32_t bPVdone = bX + 24, bOfinal = bX + 32, bDrain = bX + 40;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x & 1, chunk = blockIdx.x >> 1;
  const int b = blockIdx.y / p.row_blocks, rblk = blockIdx.y - b * p.row_blocks;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kOwnSlots; ++s) {
      mbar_init(bOwnFull(s), 1);
      mbar_init(bOwnEmpty(s), 1);
    }
    for (int s = 0; s < C::kOthSlots; ++s) {
      mbar_init(bOthFull(s), 1);
      mbar_init(bOthEmpty(s), 1);
    }
    mbar_init(bQ, 1);
    mbar_init(bSfull(0), 1);
    mbar_init(bSfull(1), 1);
    mbar_init(bPVdone, 1);
    mbar_init(bOfinal, 1);
    mbar_init(bDrain, 1);
    fence_mbar_init();
  }
  if (warp == 0 && elect_one()) {
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  const int k0 = chunk * p.chunk_keys;
  const int k1 = min(k0 + p.chunk_keys, p.Nk);
  const int ntiles = (k1 - k0 + kMlaTcKeys - 1) / kMlaTcKeys;  // >= 1: every chunk holds keys

  if (warp == 0) {
    // ============================================================ TMA producer
    bool ok = true;
    if (elect_one()) {
      mbar_arrive_expect_tx(bQ, 4 * C::kQBoxBytes);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_3d(sQ + c * C::kQBoxBytes, &p.tmQ, bQ, h * 256 + c * 64, rblk * kMlaTcRows, b);
    }
    __syncwarp();
    int nown = 0, noth = 0;  // halves issued
    for (int i = 0; ok && i < ntiles; ++i) {
      if (p.stall_after >= 0 && i >= p.stall_after) {  // test hook: stop loading
        ok = false;
        break;
      }
      // columns 0-255 first: the score MMAs run over the columns in order
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const bool own = part == h;
        uint32_t dst, full;
        if (own) {
          const int s = i % C::kOwnSlots;
          if (i >= C::kOwnSlots && !mbar_wait_warp(bOwnEmpty(s), ((i / C::kOwnSlots) - 1) & 1, wc, kErrMlaWait)) {
            ok = false;
            break;
          }
          dst = sOwn + s * C::kHalfBytes;
          full = bOwnFull(s);
        } else {
          const int s = i % C::kOthSlots;
          if (i >= C::kOthSlots && !mbar_wait_warp(bOthEmpty(s), ((i / C::kOthSlots) - 1) & 1, wc, kErrMlaWait)) {
            ok = false;
            break;
          }
          dst = sOth + s * C::kHalfBytes;
          full = bOthFull(s);
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(full, C::kHalfBytes);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tma_load_3d(dst + c * C::kBoxBytes, &p.tmC, full, part * 256 + c * 64, k0 + i * kMlaTcKeys, b);
        }
        __syncwarp();
        if (own) nown = i + 1;
        else noth = i + 1;
      }
    }
    if (lane == 0) {  // never leave with a copy of ours in flight
      mbar_drain_dec(bQ, 0);
      for (int i = max(0, nown - C::kOwnSlots); i < nown; ++i)
        mbar_drain_dec(bOwnFull(i % C::kOwnSlots), (i / C::kOwnSlots) & 1);
      for (int i = max(0, noth - C::kOthSlots); i < noth; ++i)
        mbar_drain_dec(bOthFull(i % C::kOthSlots), (i / C::kOthSlots) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(kMlaTcRows, kMlaTcKeys, BF16, false, false);
    constexpr uint32_t kIdPV = idesc_f16(kMlaTcRows, 256, BF16, false, true);
    bool ok = mbar_wait_warp(bQ, 0, wc, kErrMlaWait);
    named_bar_sync(kBarMlaQt, kBarMlaThreads);  // the TMEM half of Q~ is written
    // After an abort no MMA is issued, but S full, P V done and O final are
    // still signalled by plain arrivals: the softmax warps wait for them
    // without polling the abort flag, and so never run ahead of this warp
    // at the P barrier.
    auto issue_s = [&](int i) {
      const int so = i % C::kOwnSlots, st = i % C::kOthSlots;
      if (ok) ok = mbar_wait_warp(h == 0 ? bOwnFull(so) : bOthFull(st),
                                  ((h == 0 ? i / C::kOwnSlots : i / C::kOthSlots)) & 1, wc, kErrMlaWait);
      if (ok) ok = mbar_wait_warp(h == 0 ? bOthFull(st) : bOwnFull(so),
                                  ((h == 0 ? i / C::kOthSlots : i / C::kOwnSlots)) & 1, wc, kErrMlaWait);
      if (!ok) {
        if (elect_one()) mbar_arrive(bSfull(i & 1));
        __syncwarp();
        return;
      }
      tc_fence_after();
      if (elect_one()) {
        const uint32_t d = tmem + C::kColS + (i & 1) * kMlaTcKeys;
        const uint32_t own_half = sOwn + so * C::kHalfBytes, oth_half = sOth + st * C::kHalfBytes;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t acc = (part | c) ? 1u : 0u;
            if (part == h) {  // own columns: A = Q~ from shared memory
              const uint64_t ad = sdesc_sw128(sQ + c * C::kQBoxBytes, 16, 1024);
              const uint64_t bd = sdesc_sw128(own_half + c * C::kBoxBytes, 16, 1024);
              umma_ss_x4(d, ad, bd, kIdS, acc);
            } else {  // other columns: A = Q~ from TMEM (8 columns per 16 values)
              const uint64_t bd = sdesc_sw128(oth_half + c * C::kBoxBytes, 16, 1024);
              umma_ts_x4_kmajor(d, tmem + C::kColQt + c * 32, bd, kIdS, acc);
            }
          }
        }
        umma_commit(bOthEmpty(st));  // the other half has served its only use
        umma_commit(bSfull(i & 1));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int j, bool last) {
      named_bar_sync(kBarMlaP, kBarMlaThreads);  // P(j) written (and O rescaled)
      ok = ok && !__any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(abort_flag) != 0);
      if (!ok) {
        if (elect_one()) {
          mbar_arrive(bPVdone);
          if (last) mbar_arrive(bOfinal);
        }
        __syncwarp();
        return;
      }
      tc_fence_after();
      if (elect_one()) {
        const int so = j % C::kOwnSlots;
        const uint64_t vd = sdesc_sw128(sOwn + so * C::kHalfBytes, C::kBoxBytes, 1024);
        umma_ts_x4_mnmajor(tmem + C::kColO, tmem + C::kColS + (j & 1) * kMlaTcKeys, vd, kIdPV, j > 0 ? 1u : 0u);
        umma_commit(bOwnEmpty(so));
        umma_commit(bPVdone);
        if (last) umma_commit(bOfinal);
      }
      __syncwarp();
    };
    for (int i = 0; i < ntiles; ++i) {
      issue_s(i);
      if (i > 0) issue_pv(i - 1, false);
    }
    issue_pv(ntiles - 1, true);
    // every MMA of this warp completes before TMEM is released
    if (elect_one()) {
      umma_commit(bDrain);
      mbar_drain_dec(bDrain, 0);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax (one row per thread)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int qr = rblk * kMlaTcRows + row;
    const bool live_row = qr < p.R;
    const int pos = p.Nk - p.Nq + (qr % p.Nq);  // row qr is query qr % Nq of head qr / Nq
    // the half of Q~ this CTA does not output -> TMEM, as packed pairs
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.Q) +
                                                         (static_cast<size_t>(b) * p.R + (live_row ? qr : 0)) * kMlaD +
                                                         (1 - h) * 256);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 w = live_row ? __ldg(src + cc * 8 + j) : make_uint4(0, 0, 0, 0);
          v[4 * j] = w.x;
          v[4 * j + 1] = w.y;
          v[4 * j + 2] = w.z;
          v[4 * j + 3] = w.w;
        }
        tmem_st32(tmem + lane_off + C::kColQt + cc * 32, v);
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar_arrive(kBarMlaQt, kBarMlaThreads);
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // live keys of this row: one interval [lo, hi)
    const int hi = min(k1, p.causal ? pos + 1 : k1);
    const int lo = (p.window > 0) ? pos - p.window + 1 : k0;
    for (int i = 0; i < ntiles; ++i) {
      ok = mbar_wait_signal(bSfull(i & 1), (i >> 1) & 1, wc, kErrMlaWait) && ok;
      const uint32_t scol = tmem + lane_off + C::kColS + (i & 1) * kMlaTcKeys;
      uint32_t sr[kMlaTcKeys];
      tc_fence_after();
      tmem_ld64(scol, sr);
      const int key0 = k0 + i * kMlaTcKeys;
      if (key0 + kMlaTcKeys > hi || key0 < lo) {
#pragma unroll
        for (int c = 0; c < kMlaTcKeys; ++c)
          if (key0 + c >= hi || key0 + c < lo) sr[c] = 0xff800000u;  // -inf
      }
      float mx = __uint_as_float(sr[0]);
#pragma unroll
      for (int c = 1; c < kMlaTcKeys; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      const float m_new = fmaxf(m, mx * sl2);
      const bool first = i == 0;
      const bool rescale = !first && __any_sync(0xffffffffu, m_new > m + kMlaRescale);
      float alpha = 1.f;
      if (first || rescale) {
        alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
        m = m_new;
      }
      if (rescale) {
        // O holds tiles up to i-1: wait for P V(i-1) (P V(i-2) completed
        // before S(i), so this phase is the only one that can be open)
        ok = mbar_wait_signal(bPVdone, (i - 1) & 1, wc, kErrMlaWait) && ok;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + C::kColO + cc * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tmem + lane_off + C::kColO + cc * 32, r);
        }
      }
      const float negm = (m == -INFINITY) ? 0.f : -m;
      uint32_t pk[kMlaTcKeys / 2];
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int c = 0; c < kMlaTcKeys / 2; ++c) {
        const float e0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), sl2, negm));
        const float e1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, negm));
        pk[c] = pack2<BF16>(e0, e1);
        sum0 += e0;
        sum1 += e1;
      }
      tmem_st32(scol, pk);  // P over the first 32 columns of this S buffer
      l = first ? (sum0 + sum1) : l * alpha + (sum0 + sum1);
      tmem_st_wait();
      tc_fence_before();
      named_bar_arrive(kBarMlaP, kBarMlaThreads);
    }
    // ---- epilogue: O_half / l and the LSE
    ok = mbar_wait_signal(bOfinal, 0, wc, kErrMlaWait) && ok;
    tc_fence_after();
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    const size_t grow = static_cast<size_t>(b) * p.R + (live_row ? qr : 0);
    if (ok) {
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::kColO + cc * 32, r);
        if (!live_row) continue;
        const int col = h * 256 + cc * 32;
        if (p.nchunks == 1) {
          uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.O) + grow * kMlaD + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2<BF16>(__uint_as_float(r[8 * q + 0]) * inv, __uint_as_float(r[8 * q + 1]) * inv);
            w.y = pack2<BF16>(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv);
            w.z = pack2<BF16>(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv);
            w.w = pack2<BF16>(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv);
            dst[q] = w;
          }
        } else {
          float4 *dst = reinterpret_cast<float4 *>(p.ws + (grow * p.nchunks + chunk) * kMlaD + col);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                 __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
        }
      }
      if (live_row && h == 0) {
        const float lse2 = (l > 0.f) ? m + log2f(l) : -INFINITY;
        if (p.nchunks == 1) {
          if (p.lse != nullptr) p.lse[grow] = lse2 * 0.69314718055994530942f;
        } else {
          p.ws_lse[grow * p.nchunks + chunk] = lse2;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn

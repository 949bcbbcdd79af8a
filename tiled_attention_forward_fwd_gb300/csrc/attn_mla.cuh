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

}  // namespace attn

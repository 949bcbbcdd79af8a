// attn_decode.cuh -- split-KV attention for decode and small query counts.
//
// The cruxr.ai "FlashDecoding" section: with few query rows there are too
// few query tiles to occupy the GPU, so the keys are split into chunks that
// are processed in parallel; each chunk yields, per query row, a partial
// maximum, sum and softmax-weighted sum of V rows, and a second step merges
// the chunks by rescaling each one with exp(m_p - m) * l_p and normalising by
// the total.
//
// GB300 mapping.  Kernel 1, grid (chunks, B*Hkv), 128 threads: one CTA takes
// the g*Nq query rows of one GQA group (all query heads that read the same
// K/V head, up to 32 rows; they share every K/V tile) and one chunk of keys.
// K/V tiles of 64 keys stream by TMA into a 3-stage ring (128B-swizzled boxes
// of 64 rows x 64 columns); each of the 4 warps takes 16 keys of every tile
// and keeps its own running max, sum and O for all rows, computed with
// warp-level tensor-core MMAs (m16n8k16, fp32 accumulation); fragments come
// from ldmatrix (transposed for V).  At the end the 4 warps are merged in
// shared memory and the chunk's normalised O and its log2-domain log-sum-exp
// go to the caller's workspace.  Kernel 2 merges the chunks of every row and
// writes O (16-bit) and LSE.
#pragma once

#include <stddef.h>

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kDecKeys = 64;     // keys per K/V tile
constexpr int kDecStages = 3;    // K/V ring depth
constexpr int kDecWarps = 4;     // each warp owns 16 keys of every tile
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecMaxRows = 32;  // query rows of one group handled by one CTA

enum DecodeError : int { kErrDecWaitKV = 0x201 };

struct DecParams {
  CUtensorMap tmK;  // (d, Nk, B*Hkv), box 64 x 64 x 1, 128B swizzle
  CUtensorMap tmV;
  const void *Q;    // (B, Hq, Nq, d), 16-bit
  float *ws;        // [B*Hq*Nq][nchunks][d + 1]: normalised O of the chunk, then its log2 LSE
  int *status;
  int B, Hq, Hkv, Nq, Nk, group, R;  // R = group * Nq query rows per CTA
  int causal, window;
  int nchunks, chunk_keys;
  int kv_lo, kv_hi;  // keys any row of a group can see
  float scale_log2;  // sm_scale * log2(e)
  unsigned long long timeout_ns;
};

template <int D>
struct DecCfg {
  static constexpr int kBoxBytes = kDecKeys * 128;          // 64 rows x 128 B
  static constexpr int kTileBytes = kDecKeys * D * 2;       // one K or V tile
  static constexpr int kQBoxBytes = kDecMaxRows * 128;      // 32 rows x 128 B
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = ((kDecMaxRows * D * 2 + 1023) / 1024) * 1024;
  static constexpr int kStageBytes = 2 * kTileBytes;        // K then V
  static constexpr int kOffBar = kOffKV + kDecStages * kStageBytes;
  static constexpr int kOffStats = kOffBar + 64;            // float wm[4][32], wl[4][32]
  static constexpr int kSmemBytes = kOffStats + 2 * kDecWarps * kDecMaxRows * 4 + 1024;
  static_assert(kDecWarps * kDecMaxRows * D * 4 <= kDecStages * kStageBytes, "O merge slabs fit in the ring");
};

// Byte offset of element (row r, column c) in a stack of 64-column boxes of
// `rows` rows with the 128-byte swizzle (16-byte chunk index ^ row % 8).
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  return static_cast<uint32_t>((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// c (16x8 fp32) += a (16x16, row) * b (16x8, col)
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Partial attention of one GQA group over one key chunk.  RB = row blocks of
// 16 (1: up to 16 rows, 2: up to 32).
template <int D, bool BF16, int RB>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  int *abort_flag = reinterpret_cast<int *>(full + kDecStages);
  float *wm = reinterpret_cast<float *>(smem + C::kOffStats);  // [warp][row] running max (log2 domain)
  float *wl = wm + kDecWarps * kDecMaxRows;                    // [warp][row] running sum
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sKV = smem_u32(smem + C::kOffKV);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int chunk = blockIdx.x;
  const int bk = blockIdx.y;  // b * Hkv + kvh
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int k0 = max(chunk * p.chunk_keys, p.kv_lo);
  const int k1 = min((chunk + 1) * p.chunk_keys, p.kv_hi);
  const int ntiles = (k1 > k0) ? (k1 - k0 + kDecKeys - 1) / kDecKeys : 0;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kDecStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  // the group's query rows -> shared memory (swizzled like a 32-row box); rows >= R are zero
  for (int idx = threadIdx.x; idx < kDecMaxRows * (D / 8); idx += kDecThreads) {
    const int r = idx / (D / 8), c8 = (idx % (D / 8)) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < p.R) {
      const int head = kvh * p.group + r / p.Nq, i = r % p.Nq;
      v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.Q) +
                                           ((static_cast<size_t>(b) * p.Hq + head) * p.Nq + i) * D + c8);
    }
    *reinterpret_cast<uint4 *>(smem + C::kOffQ + swz(kDecMaxRows, r, c8)) = v;
  }
  __syncthreads();

  auto issue = [&](int tile) {
    const int s = tile % kDecStages;
    const uint32_t bar = smem_u32(&full[s]);
    const uint32_t kdst = sKV + s * C::kStageBytes, vdst = kdst + C::kTileBytes;
    mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
      tma_load_3d(kdst + cc * C::kBoxBytes, &p.tmK, bar, cc * 64, k0 + tile * kDecKeys, bk);
      tma_load_3d(vdst + cc * C::kBoxBytes, &p.tmV, bar, cc * 64, k0 + tile * kDecKeys, bk);
    }
  };
  int issued = 0;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
    for (; issued < min(kDecStages, ntiles); ++issued) issue(issued);
  }

  // running state: rows rb*16 + g (h = 0) and rb*16 + g + 8 (h = 1)
  float m[RB][2], l[RB][2];
  float o[RB][D / 8][4];
  int pos[RB][2];
  bool rowok[RB][2];
#pragma unroll
  for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rb * 16 + g + 8 * h;
      m[rb][h] = -INFINITY;
      l[rb][h] = 0.f;
      rowok[rb][h] = r < p.R;
      pos[rb][h] = p.Nk - p.Nq + (r % p.Nq);
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[rb][n][0] = o[rb][n][1] = o[rb][n][2] = o[rb][n][3] = 0.f;
  }
  const float sl2 = p.scale_log2;
  bool aborted = false;

  for (int i = 0; i < ntiles; ++i) {
    const int s = i % kDecStages;
    const bool ok = mbar_wait_warp(smem_u32(&full[s]), (i / kDecStages) & 1, wc, kErrDecWaitKV);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const uint32_t sK = sKV + s * C::kStageBytes, sV = sK + C::kTileBytes;
    const int key_base = k0 + i * kDecKeys + warp * 16;  // this warp's 16 keys
    // ---- S (rows x 16 keys) = Q K^T
    float sc[RB][2][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) sc[rb][nb][0] = sc[rb][nb][1] = sc[rb][nb][2] = sc[rb][nb][3] = 0.f;
    {
      const int j = lane >> 3;
      const int krow = warp * 16 + (j >> 1) * 8 + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t kb[4];
        ldsm_x4(sK + swz(kDecKeys, krow, kk * 16 + (j & 1) * 8), kb[0], kb[1], kb[2], kb[3]);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          uint32_t a[4];
          ldsm_x4(sQ + swz(kDecMaxRows, rb * 16 + (j & 1) * 8 + (lane & 7), kk * 16 + (j >> 1) * 8), a[0], a[1],
                  a[2], a[3]);
          mma16816<BF16>(sc[rb][0], a, kb[0], kb[1]);
          mma16816<BF16>(sc[rb][1], a, kb[2], kb[3]);
        }
      }
    }
    // ---- mask, online softmax (log2 domain), P as A fragments
    uint32_t pa[RB][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = key_base + nb * 8 + 2 * tq + e;
            const bool live = rowok[rb][h] && key < k1 && (!p.causal || key <= pos[rb][h]) &&
                              (p.window <= 0 || pos[rb][h] - key < p.window);
            v[nb * 2 + e] = live ? sc[rb][nb][2 * h + e] : -INFINITY;
          }
        }
        float tmax = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m[rb][h], tmax * sl2);
        const float alpha = (m[rb][h] == -INFINITY) ? 0.f : ex2_approx(m[rb][h] - m_new);
        const float mref = (m_new == -INFINITY) ? 0.f : m_new;
        float e4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) e4[q] = ex2_approx(fmaf(v[q], sl2, -mref));
        l[rb][h] = l[rb][h] * alpha + ((e4[0] + e4[1]) + (e4[2] + e4[3]));
        m[rb][h] = m_new;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[rb][n][2 * h] *= alpha;
          o[rb][n][2 * h + 1] *= alpha;
        }
        // A fragment of P: a0/a2 hold row g (keys 2t, 8+2t), a1/a3 row g+8
        pa[rb][h] = pack2<BF16>(e4[0], e4[1]);
        pa[rb][2 + h] = pack2<BF16>(e4[2], e4[3]);
      }
    }
    // ---- O += P V
    {
      const int j = lane >> 3;
      const int vrow = warp * 16 + (j & 1) * 8 + (lane & 7);
#pragma unroll
      for (int nn = 0; nn < D / 16; ++nn) {
        uint32_t vb[4];
        ldsm_x4_t(sV + swz(kDecKeys, vrow, nn * 16 + (j >> 1) * 8), vb[0], vb[1], vb[2], vb[3]);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          mma16816<BF16>(o[rb][2 * nn], pa[rb], vb[0], vb[1]);
          mma16816<BF16>(o[rb][2 * nn + 1], pa[rb], vb[2], vb[3]);
        }
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (threadIdx.x == 0 && issued < ntiles) issue(issued++);
  }
  if (aborted) {
    // Never leave with one of our copies in flight: wait (bounded) for the
    // last loads issued into each stage.
    if (threadIdx.x == 0) {
      for (int t = max(0, issued - kDecStages); t < issued; ++t) {
        const uint32_t bar = smem_u32(&full[t % kDecStages]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar, (t / kDecStages) & 1))
          if (globaltimer_ns() - t0 > 1000000000ull) break;
      }
    }
    return;
  }

  // ---- merge the 4 warps: row sums over the quad, then max / sums per row in shared memory
#pragma unroll
  for (int rb = 0; rb < RB; ++rb)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[rb][h] += __shfl_xor_sync(0xffffffffu, l[rb][h], 1);
      l[rb][h] += __shfl_xor_sync(0xffffffffu, l[rb][h], 2);
      if (tq == 0) {
        const int r = rb * 16 + g + 8 * h;
        wm[warp * kDecMaxRows + r] = m[rb][h];
        wl[warp * kDecMaxRows + r] = l[rb][h];
      }
    }
  // one slab per warp, summed in a fixed order below (deterministic result)
  float *oacc = reinterpret_cast<float *>(smem + C::kOffKV);  // [warp][32][D], the ring is idle now
  __syncthreads();
#pragma unroll
  for (int rb = 0; rb < RB; ++rb)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = rb * 16 + g + 8 * h;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecMaxRows + r]);
      const float scale = (m[rb][h] == -INFINITY) ? 0.f : ex2_approx(m[rb][h] - M);
      float *slab = oacc + (warp * kDecMaxRows + r) * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2 *>(slab + n * 8 + 2 * tq) =
            make_float2(o[rb][n][2 * h] * scale, o[rb][n][2 * h + 1] * scale);
    }
  __syncthreads();
  // ---- this chunk's normalised O and log2 LSE per row -> workspace
  for (int idx = threadIdx.x; idx < p.R * (D + 1); idx += kDecThreads) {
    const int r = idx / (D + 1), c = idx - r * (D + 1);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecMaxRows + r]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float mw = wm[w * kDecMaxRows + r];
      if (mw != -INFINITY) L += ex2_approx(mw - M) * wl[w * kDecMaxRows + r];
    }
    const int head = kvh * p.group + r / p.Nq, qi = r % p.Nq;
    const size_t grow = (static_cast<size_t>(b) * p.Hq + head) * p.Nq + qi;
    float *dst = p.ws + (grow * p.nchunks + chunk) * (D + 1);
    if (c < D) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) acc += oacc[(w * kDecMaxRows + r) * D + c];
      dst[c] = (L > 0.f) ? acc / L : 0.f;
    }
    else dst[D] = (L > 0.f) ? M + log2f(L) : -INFINITY;
  }
}

// Merge the chunks of every query row: O = sum_c 2^(lse_c - lse) o_c,
// LSE = lse * ln 2 with lse = log2 sum_c 2^(lse_c).  One warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const float *ws, void *O, float *lse, int rows,
                                                                  int nchunks) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float *base = ws + static_cast<size_t>(row) * nchunks * (D + 1);
  float M = -INFINITY;
  for (int c = lane; c < nchunks; c += 32) M = fmaxf(M, base[c * (D + 1) + D]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[D / 32];
#pragma unroll
  for (int k = 0; k < D / 32; ++k) acc[k] = 0.f;
  float L = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const float lc = base[c * (D + 1) + D];
    const float w = (lc == -INFINITY) ? 0.f : ex2_approx(lc - M);
    L += w;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] += w * base[c * (D + 1) + lane + 32 * k];
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  uint16_t *orow = reinterpret_cast<uint16_t *>(O) + static_cast<size_t>(row) * D;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const uint32_t pk = pack2<BF16>(acc[k] * inv, 0.f);
    orow[lane + 32 * k] = static_cast<uint16_t>(pk & 0xFFFFu);
  }
  if (lse != nullptr && lane == 0)
    lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace attn

// attn_short.cuh -- attention for short key sequences (Nk <= 128).
//
// The same computation as the tiled forward pass (the cruxr.ai
// "FlashAttention" section: O = softmax(scale Q K^T + mask) V with the per-row
// log-sum-exp), for the case the pages single out as bandwidth-bound: with
// few keys per head (N = 64) every head is a few kilobytes of Q, K and V,
// the work per byte is tiny, and the prefill kernel's per-tile pipeline
// (TMEM allocation, 128-row tiles, MMA/softmax handoffs) would cost more than
// moving the bytes.  All keys of a head fit in one tile, so the softmax is
// taken over the whole row at once: no running max, no rescaling.
//
// GB300 mapping.  A persistent grid walks units of (batch, query head, 64
// query rows).  A producer warp streams each unit's Q (64 rows), K and V
// (NK = 64 or 128 rows, zero-filled past Nk) by TMA into an NS-stage ring of
// 128B-swizzled boxes; 4 consumer warps take 16 query rows each, compute
// S = Q K^T and O = P V with warp-level tensor-core MMAs (m16n8k16, fp32
// accumulation; fragments by ldmatrix), and write O (16-bit) and LSE straight
// from registers.  A stage is released when all four warps are done with it.
#pragma once

#include "attn_decode.cuh"  // swz, ldsm_x4, ldsm_x4_t, mma16816

namespace attn {

constexpr int kShortRows = 64;  // query rows per unit: 4 consumer warps x 16
constexpr int kShortWarps = 4;
constexpr int kShortThreads = 32 * kShortWarps + 32;  // + one TMA producer warp
constexpr int kShortMaxKeys = 128;

enum ShortError : int { kErrShortWait = 0x301 };

struct ShortParams {
  CUtensorMap tmQ;  // (d, Nq, B*Hq), box 64 x 64 x 1, 128B swizzle
  CUtensorMap tmK;  // (d, Nk, B*Hkv), same boxes
  CUtensorMap tmV;
  void *O;          // (B*Hq*Nq, d) 16-bit
  float *lse;       // (B*Hq*Nq) or null
  int *status;
  int B, Hq, Hkv, Nq, Nk, group;
  int causal, window;
  int n_qblocks;  // ceil(Nq / 64)
  int n_units;    // B * Hq * n_qblocks
  float scale_log2;
  unsigned long long timeout_ns;
  int stall_after;  // test hook: the producer stops after this many K/V tiles (-1: never)
};

// Ring depth and resident CTAs per SM: about 190 KB of loads in flight per SM.
template <int D, int NK>
struct ShortCfg {
  static constexpr int kBox = 64 * 128;  // one TMA box: 64 rows x 64 columns x 2 bytes
  static constexpr int kQBytes = (D / 64) * kBox;
  static constexpr int kKBytes = (NK / 64) * (D / 64) * kBox;  // K or V
  static constexpr int kStageBytes = kQBytes + 2 * kKBytes;
  static constexpr int kMinCtas = (D == 64 && NK == 64) ? 2 : 1;
  static constexpr int kStages = (D == 64 && NK == 64) ? 4 : (D == 64 ? 5 : (NK == 64 ? 4 : 2));
  static constexpr int kOffBar = kStages * kStageBytes;  // full[NS], empty[NS], abort flag
  static constexpr int kSmemBytes = kOffBar + 128 + 1024;  // + alignment slack
  static_assert(2 * kStages * 8 + 4 <= 128, "barriers fit");
  static_assert(kMinCtas * (kSmemBytes + 1024) <= 233472, "shared memory per SM");
};

__device__ __forceinline__ void short_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 1000000000ull) break;
}

template <int D, bool BF16, int NK>
__global__ void __launch_bounds__(kShortThreads, ShortCfg<D, NK>::kMinCtas)
    attn_short_kernel(const __grid_constant__ ShortParams p) {
  using C = ShortCfg<D, NK>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  int *abort_flag = reinterpret_cast<int *>(bars + 2 * NS);
  const uint32_t s0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto bFull = [&](int s) { return bar0 + 8u * s; };
  auto bEmpty = [&](int s) { return bar0 + 8u * (NS + s); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  pdl_launch_dependents();  // the next call's prologue may overlap this one

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(bFull(s), 1);
      mbar_init(bEmpty(s), kShortWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // inputs may come from the previous kernel on the stream
  bool ok = true;

  if (warp == kShortWarps) {
    // ======================================================== TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
    }
    __syncwarp();
    int n = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++n) {
      if (p.stall_after >= 0 && n >= p.stall_after) {  // test hook: stop loading
        ok = false;
        break;
      }
      const int s = n % NS;
      if (n >= NS && !mbar_wait_warp(bEmpty(s), ((n / NS) - 1) & 1, wc, kErrShortWait)) {
        ok = false;
        break;
      }
      const int qb = u % p.n_qblocks, bh = u / p.n_qblocks;
      const int b = bh / p.Hq, h = bh - b * p.Hq;
      const int bkv = b * p.Hkv + h / p.group;
      const uint32_t sq = s0 + s * C::kStageBytes, sk = sq + C::kQBytes, sv = sk + C::kKBytes;
      if (elect_one()) {
        mbar_arrive_expect_tx(bFull(s), C::kStageBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
          tma_load_3d(sq + cb * C::kBox, &p.tmQ, bFull(s), cb * 64, qb * kShortRows, bh);
#pragma unroll
          for (int rb = 0; rb < NK / 64; ++rb) {
            tma_load_3d(sk + (cb * (NK / 64) + rb) * C::kBox, &p.tmK, bFull(s), cb * 64, rb * 64, bkv);
            tma_load_3d(sv + (cb * (NK / 64) + rb) * C::kBox, &p.tmV, bFull(s), cb * 64, rb * 64, bkv);
          }
        }
      }
      __syncwarp();
    }
    if (!ok && lane == 0)  // never leave with one of our copies in flight
      for (int k = max(0, n - NS); k < n; ++k) short_drain(bFull(k % NS), (k / NS) & 1);
  } else {
    // ======================================================== consumer warps
    const int g = lane >> 2, tq = lane & 3, j = lane >> 3;
    const int r0 = warp * 16;  // this warp's rows within the unit
    const float sl2 = p.scale_log2;
    int n = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++n) {
      const int s = n % NS;
      if (!mbar_wait_warp(bFull(s), (n / NS) & 1, wc, kErrShortWait)) {
        ok = false;
        break;
      }
      const int qb = u % p.n_qblocks, bh = u / p.n_qblocks;
      const int row0 = qb * kShortRows + r0;  // first query row of this warp
      const uint32_t sq = s0 + s * C::kStageBytes, sk = sq + C::kQBytes, sv = sk + C::kKBytes;
      if (row0 < p.Nq) {
        // ---- S (16 x NK) = Q K^T
        float sc[NK / 8][4];
#pragma unroll
        for (int t = 0; t < NK / 8; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4];
          ldsm_x4(sq + swz(kShortRows, r0 + (j & 1) * 8 + (lane & 7), kk * 16 + (j >> 1) * 8), a[0], a[1], a[2],
                  a[3]);
#pragma unroll
          for (int kb = 0; kb < NK / 16; ++kb) {
            uint32_t bq[4];
            ldsm_x4(sk + swz(NK, kb * 16 + (j >> 1) * 8 + (lane & 7), kk * 16 + (j & 1) * 8), bq[0], bq[1], bq[2],
                    bq[3]);
            mma16816<BF16>(sc[2 * kb], a, bq[0], bq[1]);
            mma16816<BF16>(sc[2 * kb + 1], a, bq[2], bq[3]);
          }
        }
        // ---- mask and softmax over the whole row (log2 domain)
        float mrow[2], lrow[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int pos = row0 + g + 8 * hh + (p.Nk - p.Nq);  // absolute position of this query row
          float mx = -INFINITY;
#pragma unroll
          for (int t = 0; t < NK / 8; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = t * 8 + 2 * tq + e;
              const bool live = key < p.Nk && (!p.causal || key <= pos) && (p.window <= 0 || pos - key < p.window);
              const float v = live ? sc[t][2 * hh + e] : -INFINITY;
              sc[t][2 * hh + e] = v;
              mx = fmaxf(mx, v);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float m = (mx == -INFINITY) ? -INFINITY : mx * sl2;
          const float mref = (m == -INFINITY) ? 0.f : m;
          float sum = 0.f;
#pragma unroll
          for (int t = 0; t < NK / 8; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float pv = ex2_approx(fmaf(sc[t][2 * hh + e], sl2, -mref));
              sc[t][2 * hh + e] = pv;
              sum += pv;
            }
          sum += __shfl_xor_sync(0xffffffffu, sum, 1);
          sum += __shfl_xor_sync(0xffffffffu, sum, 2);
          mrow[hh] = m;
          lrow[hh] = sum;
        }
        // ---- O (16 x D) = P V; P as A fragments (rows g / g+8, 16 keys per step)
        float o[D / 8][4];
#pragma unroll
        for (int t = 0; t < D / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < NK / 16; ++ks) {
          uint32_t pa[4];
          pa[0] = pack2<BF16>(sc[2 * ks][0], sc[2 * ks][1]);
          pa[1] = pack2<BF16>(sc[2 * ks][2], sc[2 * ks][3]);
          pa[2] = pack2<BF16>(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
          pa[3] = pack2<BF16>(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
#pragma unroll
          for (int nn = 0; nn < D / 16; ++nn) {
            uint32_t vb[4];
            ldsm_x4_t(sv + swz(NK, ks * 16 + (j & 1) * 8 + (lane & 7), nn * 16 + (j >> 1) * 8), vb[0], vb[1], vb[2],
                      vb[3]);
            mma16816<BF16>(o[2 * nn], pa, vb[0], vb[1]);
            mma16816<BF16>(o[2 * nn + 1], pa, vb[2], vb[3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bEmpty(s));  // the stage is no longer read by this warp
        // ---- O / l -> 16-bit, LSE = (m + log2 l) ln 2
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = row0 + g + 8 * hh;
          if (row >= p.Nq) continue;
          const float inv = (lrow[hh] > 0.f) ? 1.f / lrow[hh] : 0.f;
          uint32_t *orow = reinterpret_cast<uint32_t *>(reinterpret_cast<uint16_t *>(p.O) +
                                                        (static_cast<size_t>(bh) * p.Nq + row) * D);
#pragma unroll
          for (int t = 0; t < D / 8; ++t)
            orow[t * 4 + tq] = pack2<BF16>(o[t][2 * hh] * inv, o[t][2 * hh + 1] * inv);
          if (p.lse != nullptr && tq == 0)
            p.lse[static_cast<size_t>(bh) * p.Nq + row] =
                (lrow[hh] > 0.f) ? (mrow[hh] + log2f(lrow[hh])) * 0.69314718055994530942f : -INFINITY;
        }
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(bEmpty(s));  // no rows of this unit for this warp
      }
    }
  }
  // Every thread learns whether some role gave up (the producer has drained
  // its copies by then).
  __syncthreads_or(!ok);
}

}  // namespace attn

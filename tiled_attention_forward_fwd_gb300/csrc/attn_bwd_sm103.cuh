// attn_bwd_sm103.cuh -- tiled attention backward (the gradients of the
// forward definition) for sm_103a.
//
// The forward stores, per query row, the natural-log log-sum-exp LSE "for the
// backward pass" (cruxr.ai "FlashAttention: Nunca materializar la matriz de
// atencion"; lab 02 kernel skeleton).  With it the weights of any (query,
// key) tile can be recomputed without the row's other tiles:
//   P = exp(sm_scale * Q K^T - LSE)           (masked entries 0)
// and the gradients of O = P V for an upstream gradient dO are
//   dV = P^T dO
//   dP = dO V^T,  D = rowsum(dO o O),  dS = P o (dP - D)
//   dK = sm_scale * dS^T Q,   dQ = sm_scale * dS K
// with GQA heads summed into their K/V head.  The score matrix never reaches
// device memory, as in the forward.
//
// GB300 mapping (a synchronous design: each step's MMAs and its elementwise
// work alternate).  One CTA per (K/V group, key tile of 128 keys); one thread per
// TMEM lane r (query row, later key row) at d = 128, two at d = 64 (each
// taking half of the row's columns in the elementwise passes).  A CTA holds K_j and V_j in shared
// memory and walks every query head of the GQA group and every query tile
// that has a live key in the tile:
//   1. TMA Q_i and dO_i (128-row boxes, 128B swizzle).
//   2. tcgen05: S = Q_i K_j^T and dP = dO_i V_j^T into TMEM (fp32).
//   3. The threads of lane r (query row r): P and dS of the row, rounded to
//      the input dtype, into shared memory in the 128B-swizzled layout of a
//      [row][key] tile (two 64-column boxes).
//   4. tcgen05: dV += P^T dO_i and dK += dS^T Q_i (A = P / dS read
//      MN-major, i.e. transposed, from the same tiles; B = dO_i / Q_i
//      MN-major), accumulated in TMEM over the CTA's steps; dQ_part = dS K_j
//      (A K-major, B = K_j MN-major) into TMEM.
//   5. The tile's dQ_part goes from TMEM into an fp32 tile in the (now free)
//      P and dS buffers, and TMA reduce-adds it into an fp32 accumulator in
//      global memory (several CTAs add to one row), while the next step's Q
//      and dO load (their buffers are free once step 4's MMAs, the last to
//      read them, have completed).
// Each group of MMAs is issued in bursts of four from one asm block.
// At the end the CTA writes dK (times sm_scale) and dV for its 128 keys.  A
// pre-pass computes D and zeroes the dQ accumulator; a post-pass writes dQ.
#pragma once

#include "fastdiv.h"
#include "sm103_ptx.cuh"

namespace attn {

enum BwdError : int { kErrBwdWait = 0x301 };

struct BwdParams {
  CUtensorMap tmQ;   // (d, Nq, B*Hq)
  CUtensorMap tmDO;  // (d, Nq, B*Hq)
  CUtensorMap tmK;   // (d, Nk, B*Hkv)
  CUtensorMap tmV;   // (d, Nk, B*Hkv)
  CUtensorMap tmDQ;  // the fp32 dQ accumulator (d, Nq, B*Hq), box 32 x 128 x 1, 128B swizzle
  const float *lse;    // (B*Hq*Nq) natural-log LSE of the forward
  const float *delta;  // (B*Hq*Nq) rowsum(dO o O)
  float *dq_acc;       // (B*Hq*Nq*d) fp32, zeroed by the pre-pass
  void *dK;            // (B*Hkv*Nk*d) 16-bit
  void *dV;            // (B*Hkv*Nk*d) 16-bit
  int *status;
  int B, Hq, Hkv, Nq, Nk, group;
  int causal, window;
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  unsigned long long timeout_ns;
  int band;  // K/V groups (b, kvh) per band of the CTA order
};

// The CTA order: one CTA per (K/V group bk = b * Hkv + kvh, key tile kt), in
// bands of `band` groups; within a band the CTAs go in order of their key
// tile, so under a causal mask the longest (first key tiles, which every
// later query tile reaches) start first and the band ends with its
// shortest, while the CTAs in flight read the Q and dO of one band's groups
// (a few in L2) rather than of all.  Two waves of CTAs per band.
ATTN_HD int bwd_band(long long zk, long long nkt, long long sms) {
  const long long w = (2 * (sms > 0 ? sms : 1) + nkt - 1) / nkt;
  return static_cast<int>(w < 1 ? 1 : (w < zk ? w : zk));
}
// CTA `cta` (launch order) of zk groups x nkt key tiles in bands of `band`.
ATTN_HD void bwd_cta_tile(int cta, int band, int zk, int nkt, int &bk, int &kt) {
  const int per_band = band * nkt;
  const int bd = cta / per_band;
  const int r = cta - bd * per_band;
  const int gb = band < zk - bd * band ? band : zk - bd * band;  // groups in this band (the last may hold fewer)
  kt = r / gb;
  bk = bd * band + (r - kt * gb);
}

template <int D>
struct BwdCfg {
  // threads: one per TMEM lane at d = 128; two at d = 64, each taking half
  // of a row's columns in the elementwise passes (measured: 415 -> 377 us on
  // a d = 64 layer; 7.96 -> 8.22 ms at d = 128, so one there)
  static constexpr int kThreads = D == 64 ? 256 : 128;
  static constexpr int kPerLane = kThreads / 128;
  static constexpr int kBoxBytes = 128 * 128;   // 128 rows x 64 columns x 2 bytes
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffP = kOffDO + kTileBytes;  // [query row][key] 128 x 128, 16-bit
  static constexpr int kOffDS = kOffP + 2 * kBoxBytes;
  static constexpr int kOffBar = kOffDS + 2 * kBoxBytes;  // kv, qdo, s, d, drain; tmem slot; abort
  static constexpr int kSmemBytes = kOffBar + 64 + 1024;  // + alignment slack
  // TMEM columns: S, then dQ_part [0, 128); dP [128, 256); dV [256, 256 + D); dK [256 + D, 256 + 2 D)
  static constexpr uint32_t kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Four MMAs issued back to back in one asm block (a tcgen05.mma issued on
// its own costs about twice the cycles of one in such a burst): D (+)=
// A_k B_k for the four (a_k, b_k) descriptor pairs; the first accumulates
// iff `accumulate` != 0, the others always.
__device__ __forceinline__ void umma_ss_burst4(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2, uint64_t a3,
                                               uint64_t b0, uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred pf, p1;\n\t"
      "setp.ne.b32 pf, %9, 0;\n\tsetp.eq.b32 p1, %9, %9;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, p1;\n\t}\n" ::"r"(d),
      "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(accumulate), "r"(idesc)
      : "memory");
}

// (MN = 128) x N tile product over K = 128 with both operands MN-major (A =
// P or dS stored [K row][M], B = dO or Q stored [K row][N]): 8 K-slices of
// 16 rows, each 2048 bytes (128 descriptor units) further in both.
__device__ __forceinline__ void umma_mn_mn_x8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  umma_ss_burst4(d, a, a + 128, a + 256, a + 384, b, b + 128, b + 256, b + 384, idesc, acc);
  umma_ss_burst4(d, a + 512, a + 640, a + 768, a + 896, b + 512, b + 640, b + 768, b + 896, idesc, 1u);
}
// K = 128 with A K-major (dS stored [M row][K], two 64-column boxes: 32
// bytes per slice within a box, 16 KB to the next box) and B MN-major (K_j
// stored [K row][N]: 2048 bytes per slice).
__device__ __forceinline__ void umma_k_mn_x8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  umma_ss_burst4(d, a, a + 2, a + 4, a + 6, b, b + 128, b + 256, b + 384, idesc, 0u);
  umma_ss_burst4(d, a + 1024, a + 1026, a + 1028, a + 1030, b + 512, b + 640, b + 768, b + 896, idesc, 1u);
}
// S = A B^T with both K-major (Q or dO against K or V): D / 16 K-slices, 32
// bytes per slice within a 64-column box, 16 KB to the next box.
template <int D>
__device__ __forceinline__ void umma_k_k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  umma_ss_burst4(d, a, a + 2, a + 4, a + 6, b, b + 2, b + 4, b + 6, idesc, 0u);
  if constexpr (D == 128)
    umma_ss_burst4(d, a + 1024, a + 1026, a + 1028, a + 1030, b + 1024, b + 1026, b + 1028, b + 1030, idesc, 1u);
}

// Bounded wait that ignores the abort flag: used only to drain our own
// copies and MMAs, which always complete.
__device__ __forceinline__ void mbar_drain_plain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > 3000000000ll) break;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 5);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  const uint32_t bKV = smem_u32(bars), bQ = bKV + 8, bS = bKV + 16, bD = bKV + 24, bDrain = bKV + 32;
  const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sP = smem_u32(smem + C::kOffP), sDS = smem_u32(smem + C::kOffDS);
  const int warp = threadIdx.x >> 5;
  const int row = threadIdx.x & 127;  // TMEM lane: a query row of the tile, later a key row
  const int half = threadIdx.x >> 7;   // which part of the row's columns this thread takes
  // a 1-D grid in the order of bwd_cta_tile
  int kt, bk;  // key tile; K/V group b * Hkv + kvh
  bwd_cta_tile(static_cast<int>(blockIdx.x), p.band, p.B * p.Hkv, (p.Nk + 127) / 128, bk, kt);
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 5; ++i) mbar_init(bKV + 8u * i, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // D and the zeroed dQ accumulator come from the pre-pass
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;  // warp w reads lanes 32 (w % 4) ..

  if (warp == 0) {
    if (elect_one()) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmDO);
      tma_prefetch_desc(&p.tmDQ);
      mbar_arrive_expect_tx(bKV, 2 * C::kTileBytes);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        tma_load_3d(sK + cc * C::kBoxBytes, &p.tmK, bKV, cc * 64, kt * 128, bk);
        tma_load_3d(sV + cc * C::kBoxBytes, &p.tmV, bKV, cc * 64, kt * 128, bk);
      }
    }
    __syncwarp();
  }
  bool ok = mbar_wait_warp(bKV, 0, wc, kErrBwdWait);

  // query tiles with a live key in this key tile: rows at positions >= the
  // tile's first key (causal), and not past its last key by the window
  const int off = p.Nk - p.Nq;
  const int nqt = (p.Nq + 127) / 128;
  int i_lo = 0, i_hi = nqt;
  if (p.causal) {
    const int r0 = kt * 128 - off;  // first row that sees key kt * 128
    i_lo = r0 > 0 ? r0 / 128 : 0;
    if (p.window > 0) {
      const int r1 = kt * 128 + 127 + p.window - 1 - off;  // last row that sees key kt * 128 + 127
      i_hi = r1 < 0 ? 0 : min(nqt, r1 / 128 + 1);
    }
  }
  constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
  constexpr uint32_t kIdT = idesc_f16(128, D, BF16, true, true);   // P^T dO, dS^T Q
  constexpr uint32_t kIdQ = idesc_f16(128, D, BF16, false, true);  // dS K
  const float log2e = 1.4426950408889634074f;
  // The steps: every query head of the group, then every live query tile.
  const int nq_per = i_hi > i_lo ? i_hi - i_lo : 0;
  const int nsteps = p.group * nq_per;
  int issued_q = 0;  // Q / dO loads issued (drained on the way out)
  // Q_i and dO_i of step st into their (single) buffers, by warp 0
  auto issue_load = [&](int st) {
    if (warp != 0) return;
    const int hh = st / nq_per, qt = i_lo + st - hh * nq_per;
    const int zq = b * p.Hq + kvh * p.group + hh;
    if (ok && elect_one()) {
      mbar_arrive_expect_tx(bQ, 2 * C::kTileBytes);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        tma_load_3d(sQ + cc * C::kBoxBytes, &p.tmQ, bQ, cc * 64, qt * 128, zq);
        tma_load_3d(sDO + cc * C::kBoxBytes, &p.tmDO, bQ, cc * 64, qt * 128, zq);
      }
    }
    __syncwarp();
    if (ok) issued_q = st + 1;
  };
  if (nsteps > 0) issue_load(0);
  int step = 0;
  for (; step < nsteps; ++step) {
    {
      const int hh = step / nq_per, qt = i_lo + step - hh * nq_per;
      const int zq = b * p.Hq + kvh * p.group + hh;
      const int qrow = qt * 128 + row;
      const bool live_row = qrow < p.Nq;
      const size_t grow = static_cast<size_t>(zq) * p.Nq + (live_row ? qrow : 0);
      const float lse2 = live_row ? __ldg(p.lse + grow) * log2e : 0.f;
      const float dlt = live_row ? __ldg(p.delta + grow) : 0.f;
      ok = ok && mbar_wait_warp(bQ, step & 1, wc, kErrBwdWait);
      // ---- S = Q K^T and dP = dO V^T
      if (warp == 0) {
        tc_fence_after();
        if (ok && elect_one()) {
          umma_k_k<D>(tmem, sdesc_sw128(sQ, 16, 1024), sdesc_sw128(sK, 16, 1024), kIdS);
          umma_k_k<D>(tmem + C::kColDP, sdesc_sw128(sDO, 16, 1024), sdesc_sw128(sV, 16, 1024), kIdS);
          umma_commit(bS);
        }
        __syncwarp();
      }
      ok = ok && mbar_wait_warp(bS, step & 1, wc, kErrBwdWait);
      tc_fence_after();
      if (step > 0) {  // the previous step's dQ reduce has read its staging tile (the P and dS buffers)
        if (threadIdx.x == 0) tma_store_wait_read0();
        __syncthreads();
      }
      // ---- P and dS of this row -> shared memory, 16-bit, swizzled [row][key]
      const int pos = qrow + off;
      const int key0 = kt * 128;
      // live keys of the row: [lo, hi) relative to key0
      const int hi = live_row ? min(p.Nk, p.causal ? pos + 1 : p.Nk) - key0 : 0;
      const int lo = (p.causal && p.window > 0) ? pos - p.window + 1 - key0 : 0;
      // d = 64 (two chunks a thread): a rolled loop (measured 436 -> 400 us on a
      // gpt_stack layer); d = 128 (four): unrolled (rolled: 7.92 -> 8.25 ms)
#pragma unroll(C::kPerLane == 2 ? 1 : 4)
      for (int c2 = 0; c2 < 4 / C::kPerLane; ++c2) {
        const int cc = half * (4 / C::kPerLane) + c2;  // 32-column chunk of the 128 keys
        uint32_t sr[32], dpr[32];
        tmem_ld32(tmem + lane_off + cc * 32, sr);
        tmem_ld32(tmem + lane_off + C::kColDP + cc * 32, dpr);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float pv[2], ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = cc * 32 + 2 * i + e;
            const bool live = c >= lo && c < hi;
            pv[e] = live ? ex2_approx(fmaf(__uint_as_float(sr[2 * i + e]), p.scale_log2, -lse2)) : 0.f;
            ds[e] = pv[e] * (__uint_as_float(dpr[2 * i + e]) - dlt);
          }
          pk[i] = pack2<BF16>(pv[0], pv[1]);
          dk[i] = pack2<BF16>(ds[0], ds[1]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = cc * 32 + q * 8;
          const uint32_t chunk = static_cast<uint32_t>((col & 63) >> 3) ^ static_cast<uint32_t>(row & 7);
          const uint32_t off_b = (col >> 6) * C::kBoxBytes + row * 128 + chunk * 16;
          st_shared_v4(sP + off_b, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          st_shared_v4(sDS + off_b, dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();  // the tiles are visible to the tensor core
      tc_fence_before();
      __syncthreads();
      // ---- dV += P^T dO, dK += dS^T Q, dQ_part = dS K
      if (warp == 0) {
        tc_fence_after();
        if (ok && elect_one()) {
          const uint32_t acc = step > 0 ? 1u : 0u;
          umma_mn_mn_x8(tmem + C::kColDV, sdesc_sw128(sP, C::kBoxBytes, 1024), sdesc_sw128(sDO, C::kBoxBytes, 1024),
                        kIdT, acc);
          umma_mn_mn_x8(tmem + C::kColDK, sdesc_sw128(sDS, C::kBoxBytes, 1024), sdesc_sw128(sQ, C::kBoxBytes, 1024),
                        kIdT, acc);
          umma_k_mn_x8(tmem, sdesc_sw128(sDS, 16, 1024), sdesc_sw128(sK, C::kBoxBytes, 1024), kIdQ);
          umma_commit(bD);
        }
        __syncwarp();
      }
      ok = ok && mbar_wait_warp(bD, step & 1, wc, kErrBwdWait);
      tc_fence_after();
      // every MMA that reads Q_i and dO_i has completed: the next step's
      // tiles load while this step's dQ_part goes out
      if (step + 1 < nsteps) issue_load(step + 1);
      // ---- dQ_part of the tile into the fp32 accumulator: each row from TMEM
      // into an fp32 staging tile in the P and dS buffers (free: the MMAs
      // that read them have completed), D / 32 boxes of 128 rows x 32
      // columns in the 128-byte swizzle (16-byte chunk q of row r at q ^ (r
      // % 8): no bank conflicts), then one TMA reduce-add per box.  Rows past
      // Nq are clipped by the tensor map.
#pragma unroll 1  // rolled: 7.92 -> 7.83 ms on bwd_gqa (d = 64 takes one box a thread)
      for (int c2 = 0; c2 < D / 32 / C::kPerLane; ++c2) {
        const int cc = half * (D / 32 / C::kPerLane) + c2;  // this thread's 32-column boxes
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + cc * 32, r);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t chunk = static_cast<uint32_t>(q) ^ static_cast<uint32_t>(row & 7);
          st_shared_v4(sP + cc * 16384 + row * 128 + chunk * 16, r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();  // the staged tile is visible to the TMA
      tc_fence_before();
      __syncthreads();  // the tile is staged; TMEM [0, 128) is free for the next step
      if (threadIdx.x == 0 && ok) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tma_reduce_add_3d(&p.tmDQ, sP + cc * 16384, cc * 32, qt * 128, zq);
        tma_store_commit();
      }
    }
  }
  // ---- dK (times sm_scale) and dV of this key tile; zero where no query reached it
  const int key = kt * 128 + row;
  const bool live_key = key < p.Nk;
  uint16_t *dk_out = reinterpret_cast<uint16_t *>(p.dK) + (static_cast<size_t>(bk) * p.Nk + (live_key ? key : 0)) * D;
  uint16_t *dv_out = reinterpret_cast<uint16_t *>(p.dV) + (static_cast<size_t>(bk) * p.Nk + (live_key ? key : 0)) * D;
#pragma unroll
  for (int c2 = 0; c2 < D / 32 / C::kPerLane; ++c2) {
    const int cc = half * (D / 32 / C::kPerLane) + c2;
    uint32_t rk[32], rv[32];
    tmem_ld32(tmem + lane_off + C::kColDK + cc * 32, rk);
    tmem_ld32(tmem + lane_off + C::kColDV + cc * 32, rv);
    if (live_key && ok) {
      const bool any = step > 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 wk, wv;
        float k8[8], v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          k8[e] = any ? __uint_as_float(rk[q * 8 + e]) * p.sm_scale : 0.f;
          v8[e] = any ? __uint_as_float(rv[q * 8 + e]) : 0.f;
        }
        wk.x = pack2<BF16>(k8[0], k8[1]);
        wk.y = pack2<BF16>(k8[2], k8[3]);
        wk.z = pack2<BF16>(k8[4], k8[5]);
        wk.w = pack2<BF16>(k8[6], k8[7]);
        wv.x = pack2<BF16>(v8[0], v8[1]);
        wv.y = pack2<BF16>(v8[2], v8[3]);
        wv.z = pack2<BF16>(v8[4], v8[5]);
        wv.w = pack2<BF16>(v8[6], v8[7]);
        *reinterpret_cast<uint4 *>(dk_out + cc * 32 + q * 8) = wk;
        *reinterpret_cast<uint4 *>(dv_out + cc * 32 + q * 8) = wv;
      }
    }
  }
  // Never leave with a copy or an MMA of ours in flight (the dQ reduces
  // complete before the CTA's shared memory goes).
  if (threadIdx.x == 0) tma_store_wait0();
  if (warp == 0) {
    if (elect_one()) {
      umma_commit(bDrain);
      mbar_drain_plain(bDrain, 0);
      if (issued_q > 0) mbar_drain_plain(bQ, (issued_q - 1) & 1);
      mbar_drain_plain(bKV, 0);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// D = rowsum(dO o O) per query row (fp32), and the row's dQ accumulator
// zeroed.  One warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const void *O, const void *dO, float *delta,
                                                            float *dq_acc, long long rows) {
  pdl_launch_dependents();
  pdl_wait();
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  constexpr int kPer = D / 32;  // elements per lane: 2 or 4
  const uint16_t *o = reinterpret_cast<const uint16_t *>(O) + r * D + lane * kPer;
  const uint16_t *g = reinterpret_cast<const uint16_t *>(dO) + r * D + lane * kPer;
  float s = 0.f;
  if constexpr (kPer == 4) {
    const uint2 ov = *reinterpret_cast<const uint2 *>(o), gv = *reinterpret_cast<const uint2 *>(g);
    const float2 o0 = unpack2<BF16>(ov.x), o1 = unpack2<BF16>(ov.y), g0 = unpack2<BF16>(gv.x), g1 = unpack2<BF16>(gv.y);
    s = o0.x * g0.x + o0.y * g0.y + o1.x * g1.x + o1.y * g1.y;
  } else {
    const float2 o0 = unpack2<BF16>(*reinterpret_cast<const uint32_t *>(o));
    const float2 g0 = unpack2<BF16>(*reinterpret_cast<const uint32_t *>(g));
    s = o0.x * g0.x + o0.y * g0.y;
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) s += __shfl_xor_sync(0xffffffffu, s, sh);
  if (lane == 0) delta[r] = s;
  float *acc = dq_acc + r * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
}

// dQ = sm_scale * accumulator, rounded to 16-bit; four elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const float *dq_acc, void *dQ, long long n4,
                                                          float sm_scale) {
  pdl_launch_dependents();
  pdl_wait();
  for (long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * 256) {
    const float4 v = reinterpret_cast<const float4 *>(dq_acc)[i];
    uint2 w;
    w.x = pack2<BF16>(v.x * sm_scale, v.y * sm_scale);
    w.y = pack2<BF16>(v.z * sm_scale, v.w * sm_scale);
    reinterpret_cast<uint2 *>(dQ)[i] = w;
  }
}

}  // namespace attn

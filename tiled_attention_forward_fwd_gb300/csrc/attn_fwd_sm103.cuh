// attn_fwd_sm103.cuh -- tiled attention forward (prefill) for sm_103a.
//
// One CTA computes one 128-row tile of queries of one (batch, query head)
// against every live 128-key tile of its K/V head: the tiling of the cruxr.ai
// "FlashAttention" section (outer loop over Q blocks, inner loop over K/V
// blocks, online softmax, one write of O) and of the lab 02 kernel skeleton
// (one program per (batch x head, query tile); running max m, running sum l
// and an fp32 accumulator; O / l and LSE = m + log l stored at the end).
//
// GB300 mapping (warp-specialised, 6 warps):
//   warp 0      TMA producer: Q tile once, then K_j / V_j into an NS-stage
//               shared-memory ring (128B-swizzled boxes of 128 rows x 64 cols)
//   warp 1      owns TMEM (512 columns) and issues tcgen05.mma from one lane:
//                 S_j = Q K_j^T      (A, B from shared memory, fp32 in TMEM)
//                 O  += P_j V_j      (A = P from TMEM, B = V from shared memory)
//   warps 2..5  softmax + epilogue: thread r owns query row r (TMEM lane r):
//               loads its S row from TMEM, masks, updates the running max and
//               sum in the log2 domain (sm_scale folded into log2 e), writes P
//               as packed 16-bit pairs back over the S columns, rescales O in
//               TMEM only when the running max grew by more than 2^8, and at
//               the end writes O / l (TMA store) and LSE.
// TMEM columns: S/P double buffer at [0,128) and [128,256), O at [256,256+D).
#pragma once

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kBM = 128;  // query rows per tile (tcgen05 M)
constexpr int kBN = 128;  // keys per K/V tile (MMA N of S, MMA K of P V)
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold: factor 256

enum DeviceError : int {
  kErrWaitQ = 0x101,
  kErrWaitKV = 0x102,
  kErrWaitKVEmpty = 0x103,
  kErrWaitS = 0x104,
  kErrWaitP = 0x105,
  kErrWaitO = 0x106,
  kErrWaitOFinal = 0x107,
};

struct FwdParams {
  CUtensorMap tmQ;  // (d, Nq, B*Hq)
  CUtensorMap tmK;  // (d, Nk, B*Hkv)
  CUtensorMap tmV;  // (d, Nk, B*Hkv)
  CUtensorMap tmO;  // (d, Nq, B*Hq)
  float *lse;       // (B*Hq*Nq) or null
  int *status;      // device status word
  int B, Hq, Hkv, Nq, Nk, group;
  int causal, window;
  int num_q_tiles;
  float scale_log2;  // sm_scale * log2(e)
  unsigned long long timeout_ns;
};

template <int D>
struct FwdCfg {
  static constexpr int kStages = (D == 64) ? 4 : 3;
  static constexpr int kBoxBytes = 128 * 128;  // 128 rows x 64 cols x 2 bytes
  static constexpr int kTileBytes = kBN * D * 2;
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kNumBars = 1 + 3 * kStages + 2 + 2 + 3;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr int kThreads = 192;
  static_assert(kNumBars * 8 + 16 <= 256, "barrier area");
};

__device__ __forceinline__ bool key_live(int key, int pos, int Nk, int causal, int window) {
  return key < Nk && (!causal || key <= pos) && (window <= 0 || pos - key < window);
}

// Bounded wait that ignores the abort flag: used only to drain our own
// asynchronous copies / MMAs, which always complete.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 1000000000ull) break;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t bar0 = smem_u32(bars);
  // barrier addresses
  const uint32_t bQ = bar0;
  auto bKfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bVfull = [&](int s) { return bar0 + 8u * (1 + NS + s); };
  auto bKVempty = [&](int s) { return bar0 + 8u * (1 + 2 * NS + s); };
  auto bSfull = [&](int b) { return bar0 + 8u * (1 + 3 * NS + b); };
  auto bPfull = [&](int b) { return bar0 + 8u * (3 + 3 * NS + b); };
  const uint32_t bOdone = bar0 + 8u * (5 + 3 * NS);
  const uint32_t bOfinal = bar0 + 8u * (6 + 3 * NS);
  const uint32_t bDrain = bar0 + 8u * (7 + 3 * NS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item
  const int bh = blockIdx.x;  // b * Hq + h
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = h / p.group;
  const int q_tile = p.num_q_tiles - 1 - static_cast<int>(blockIdx.y);  // long causal tiles first
  const int i0 = q_tile * kBM;
  const int i1 = min(i0 + kBM, p.Nq);
  const int off = p.Nk - p.Nq;
  const int p0 = i0 + off, p1 = i1 - 1 + off;
  const int nkt = (p.Nk + kBN - 1) / kBN;
  int kv_end = nkt, kv_begin = 0;
  if (p.causal) {
    kv_end = min(nkt, p1 / kBN + 1);
    if (p.window > 0) {
      const int lo = p0 - p.window + 1;
      kv_begin = lo > 0 ? lo / kBN : 0;
    }
  }
  const int n_tiles = kv_end - kv_begin;  // >= 1 (host guarantees Nq <= Nk when causal)

  WaitCtl wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bQ, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKfull(s), 1);
      mbar_init(bVfull(s), 1);
      mbar_init(bKVempty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bSfull(i), 1);
      mbar_init(bPfull(i), 4);
    }
    mbar_init(bOdone, 1);
    mbar_init(bOfinal, 1);
    mbar_init(bDrain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      mbar_arrive_expect_tx(bQ, C::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * C::kBoxBytes, &p.tmQ, bQ, c * 64, i0, bh);
      const int zkv = b * p.Hkv + kvh;
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(bKVempty(s), ((j / NS) - 1) & 1, wc, kErrWaitKVEmpty)) break;
        const int krow = (kv_begin + j) * kBN;
        mbar_arrive_expect_tx(bKfull(s), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sK + s * C::kTileBytes + c * C::kBoxBytes, &p.tmK, bKfull(s), c * 64, krow, zkv);
        mbar_arrive_expect_tx(bVfull(s), C::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sV + s * C::kTileBytes + c * C::kBoxBytes, &p.tmV, bVfull(s), c * 64, krow, zkv);
        issued = j + 1;
      }
      // Never leave the CTA with one of our copies still in flight.
      mbar_drain(bQ, 0);
      for (int t = max(0, issued - NS); t < issued; ++t) {
        mbar_drain(bKfull(t % NS), (t / NS) & 1);
        mbar_drain(bVfull(t % NS), (t / NS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16(kBM, kBN, BF16, false, false);
      constexpr uint32_t kIdescPV = idesc_f16(kBM, D, BF16, false, true);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % NS;
        if (!mbar_wait(bPfull(jj & 1), (jj >> 1) & 1, wc, kErrWaitP)) return false;
        if (!mbar_wait(bVfull(s), (jj / NS) & 1, wc, kErrWaitKV)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + s * C::kTileBytes;
        const uint32_t pcol = tmem + (jj & 1) * 128;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {
          // V: MN-major (d contiguous); 16 keys = two 8-row swizzle atoms.
          const uint64_t bdesc = sdesc_sw128(vbase + k * 2048, C::kBoxBytes, 1024);
          umma_ts(tmem + C::kColO, pcol + k * 8, bdesc, kIdescPV, (jj > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(bKVempty(s));
        umma_commit(bOdone);
        return true;
      };
      bool ok = mbar_wait(bQ, 0, wc, kErrWaitQ);
      int j = 0;
      for (; ok && j < n_tiles; ++j) {
        const int s = j % NS;
        if (!mbar_wait(bKfull(s), (j / NS) & 1, wc, kErrWaitKV)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = sK + s * C::kTileBytes;
        const uint32_t scol = tmem + (j & 1) * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          // Q, K: K-major; 16 elements = 32 bytes inside a 128-byte swizzle row.
          const uint32_t koff = (k / 4) * C::kBoxBytes + (k % 4) * 32;
          const uint64_t adesc = sdesc_sw128(sQ + koff, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(kbase + koff, 16, 1024);
          umma_ss(scol, adesc, bdesc, kIdescQK, k > 0 ? 1u : 0u);
        }
        umma_commit(bSfull(j & 1));
        if (j > 0 && !issue_pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && issue_pv(n_tiles - 1)) umma_commit(bOfinal);
      // Drain every MMA we issued before TMEM can be released.
      umma_commit(bDrain);
      mbar_drain(bDrain, 0);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax + epilogue
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int pos = i0 + row + off;  // absolute position of this query row
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scaled scores, log2 domain (may lag by < 2^8)
    float l = 0.f;        // running sum of exp2(s * sl2 - m) in fp32 (gives LSE)
    float lq = 0.f;       // the same sum over the 16-bit rounded probabilities (normalises O)
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int kt = kv_begin + j;
      const uint32_t scol = tmem + lane_off + (j & 1) * 128;
      if (!mbar_wait_warp(bSfull(j & 1), (j >> 1) & 1, wc, kErrWaitS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(scol + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
      }
      const int key0 = kt * kBN;
      const bool need_mask = (key0 + kBN - 1 >= p.Nk) || (p.causal && key0 + kBN - 1 > p0) ||
                             (p.window > 0 && key0 <= p1 - p.window);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (!key_live(key0 + c, pos, p.Nk, p.causal, p.window)) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sl2);
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, m_new > m + kRescaleLog2)) {
        const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
        // O currently holds P_{j-1} V_{j-1}: wait for that MMA before touching it.
        if (!mbar_wait_warp(bOdone, (j - 1) & 1, wc, kErrWaitO)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          const uint32_t ocol = tmem + lane_off + C::kColO + c * 32;
          tmem_ld32(ocol, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(ocol, r);
        }
        l *= alpha;
        lq *= alpha;
        m = m_new;
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
      float rs = 0.f, rsq = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float e0 = ex2_approx(fmaf(s[c * 32 + 2 * i], sl2, -mref));
          const float e1 = ex2_approx(fmaf(s[c * 32 + 2 * i + 1], sl2, -mref));
          pk[i] = pack2<BF16>(e0, e1);
          rs += e0 + e1;
          // lq sums the 16-bit probabilities the P V contraction really uses,
          // so the weights that normalise O add up to one.
          const float2 r2 = unpack2<BF16>(pk[i]);
          rsq += r2.x + r2.y;
        }
        tmem_st16(scol + c * 16, pk);
      }
      l += rs;
      lq += rsq;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bPfull(j & 1));
    }
    // ---- epilogue: O / l -> 16-bit, staged in the (now idle) Q buffer, TMA store; LSE.
    if (ok) ok = mbar_wait_warp(bOfinal, 0, wc, kErrWaitOFinal);
    if (ok) {
      tc_fence_after();
      const float inv_l = (lq > 0.f) ? 1.f / lq : 0.f;
      uint8_t *stage = smem + C::kOffQ;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::kColO + c * 32, r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col0 = c * 32 + q * 8;
          const int box = col0 / 64, chunk = (col0 % 64) / 8;
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(r[q * 8 + 0]) * inv_l, __uint_as_float(r[q * 8 + 1]) * inv_l);
          w.y = pack2<BF16>(__uint_as_float(r[q * 8 + 2]) * inv_l, __uint_as_float(r[q * 8 + 3]) * inv_l);
          w.z = pack2<BF16>(__uint_as_float(r[q * 8 + 4]) * inv_l, __uint_as_float(r[q * 8 + 5]) * inv_l);
          w.w = pack2<BF16>(__uint_as_float(r[q * 8 + 6]) * inv_l, __uint_as_float(r[q * 8 + 7]) * inv_l);
          *reinterpret_cast<uint4 *>(stage + box * C::kBoxBytes + row * 128 + ((chunk ^ (row & 7)) * 16)) = w;
        }
      }
      if (p.lse != nullptr && i0 + row < p.Nq) {
        const float lse2 = (l > 0.f) ? m + log2f(l) : -INFINITY;
        p.lse[static_cast<size_t>(bh) * p.Nq + i0 + row] = lse2 * 0.69314718055994530942f;
      }
      fence_proxy_async_smem();
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == 2 && lane == 0 && ok && *abort_flag == 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_store_3d(&p.tmO, sQ + c * C::kBoxBytes, c * 64, i0, bh);
      tma_store_commit();
      tma_store_wait0();
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

// attn_fwd_sm103.cuh -- tiled attention forward (prefill) for sm_103a.
//
// The computation is the tiling of the cruxr.ai "FlashAttention" section
// (outer loop over Q blocks, inner loop over K/V blocks, online softmax with a
// running max and running sum, one write of O) and of the lab 02 kernel
// skeleton (running max m, running sum l and an fp32 accumulator per query
// row; O / l and the log-sum-exp m + log l stored at the end).
//
// GB300 mapping.  A persistent grid (one CTA per SM) walks a static list of
// work items, longest first.  An item is two 128-row query tiles that read
// the same K/V rows: two heads of one GQA group at the same rows when the
// group size is even (each K/V tile load then serves both heads), else two
// consecutive row tiles of one head.  12 warps in three warpgroups:
//   WG0  warp 0: TMA producer -- Q tiles, then K_j / V_j into an NS-stage
//                shared-memory ring (128B-swizzled boxes of 128 rows x 64 cols;
//                K_j and V_j complete one barrier)
//        warp 1: owns TMEM (512 columns) and issues tcgen05.mma from one
//                elected lane of the converged warp:
//                  S_t = Q_t K_j^T  (A, B in shared memory, fp32 in TMEM)
//                  O_t += P_t V_j   (A = P_t in TMEM, B = V_j in shared memory)
//                alternating between the two tiles so that one tile's
//                contractions run while the other tile's softmax runs
//   WG1, WG2     softmax of tile 0 / tile 1: thread r owns query row r (TMEM
//                lane r); loads its S row, masks, keeps the running max and
//                sums in the log2 domain (sm_scale folded into log2 e), writes
//                P as packed 16-bit pairs over the S columns, and rescales its
//                O row in TMEM only when the running max grew by more than 2^8;
//                after an item's last tile it reads O_t, frees it for the next
//                item and writes O / l (16-bit) and LSE to global memory
// TMEM columns: S/P of tile t at [128 t, 128 t + 128), O_t at 256 + t*D.
// Every mbarrier wait is bounded (see sm103_ptx.cuh).
#pragma once

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kBM = 128;  // query rows per tile (tcgen05 M)
constexpr int kBN = 128;  // keys per K/V tile (MMA N of S, MMA K of P V)
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold: a factor 256

enum DeviceError : int {
  kErrWaitQ = 0x101,
  kErrWaitKV = 0x102,
  kErrWaitKVEmpty = 0x103,
  kErrWaitS = 0x104,
  kErrWaitOFinal = 0x107,
  kErrWaitQFree = 0x108,
};

struct FwdParams {
  CUtensorMap tmQ;  // (d, Nq, B*Hq)
  CUtensorMap tmK;  // (d, Nk, B*Hkv)
  CUtensorMap tmV;  // (d, Nk, B*Hkv)
  void *O;          // (B*Hq*Nq, d) 16-bit
  float *lse;       // (B*Hq*Nq) or null
  int *status;      // device status word
  int B, Hq, Hkv, Nq, Nk, group;
  int causal, window;
  int heads_mode;    // 1: item = heads (h, h+1) at the same 128 rows; 0: rows (r, r+128) of one head
  int n_row_blocks;  // row blocks per (b, head slot)
  int n_slots;       // heads_mode ? B*Hq/2 : B*Hq
  int n_items;
  float scale_log2;  // sm_scale * log2(e)
  unsigned long long timeout_ns;
};

template <int D>
struct FwdCfg {
  static constexpr int kStages = (D == 64) ? 4 : 2;  // K/V ring depth
  static constexpr int kQBufs = (D == 64) ? 2 : 1;   // Q buffers per tile (2: next item prefetched)
  static constexpr int kBoxBytes = 128 * 128;        // 128 rows x 64 cols x 2 bytes
  static constexpr int kTileBytes = kBN * D * 2;     // one K or V tile
  static constexpr int kQBytes = kBM * D * 2;        // one Q tile
  static constexpr int kOffQ = 0;                    // [tile][buf]
  static constexpr int kOffK = kOffQ + 2 * kQBufs * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // barriers: qfull[2][QB], qfree[2][QB], kvfull[NS], kvempty[NS],
  //           sfull[2], ofinal[2], drain[2]
  static constexpr int kNumBars = 4 * kQBufs + 2 * kStages + 6;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr int kThreads = 384;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Register budget per warpgroup after setmaxnreg.  The kernel is launched
// with 384 threads x 168 registers = 64512; the split must not exceed that.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsWG0 = 72, kRegsSoftmax = 216;
static_assert(128 * kRegsWG0 + 256 * kRegsSoftmax <= 384 * kLaunchRegs, "register split");

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

// S[tmem] = Q K^T for one 128x128 tile: D/16 MMAs of K = 16, issued back to
// back.  qd / kd describe the first K-slice; slice k starts (k/4) 64-column
// boxes plus (k%4)*32 bytes further (16-byte units in the descriptor).
template <int D, bool BF16>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint64_t qd, uint64_t kd) {
  constexpr uint32_t kIdesc = idesc_f16(kBM, kBN, BF16, false, false);
  constexpr uint64_t kBox = (128 * 128) >> 4;
  umma_ss_x4(d_tmem, qd, kd, kIdesc, 0u);
  if constexpr (D == 128) umma_ss_x4(d_tmem, qd + kBox, kd + kBox, kIdesc, 1u);
}

// O[tmem] (+)= P V for one tile: 8 MMAs of K = 16 keys, back to back.  P is
// read from TMEM (8 columns of packed pairs per slice); V is MN-major (d
// contiguous), and 16 keys are two 8-row swizzle atoms, 2048 bytes further
// per slice.
template <int D, bool BF16>
__device__ __forceinline__ void mma_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t vd, uint32_t accumulate) {
  constexpr uint32_t kIdesc = idesc_f16(kBM, D, BF16, false, true);
  umma_ts_x8(o_tmem, p_tmem, vd, kIdesc, accumulate);
}

// One work item: up to two query tiles and the K/V tiles each one needs.
struct Item {
  int b, kvh;
  int bh[2];    // b * Hq + h of each tile
  int row0[2];  // first query row of each tile
  bool valid[2];
  int beg[2], end[2];  // live K/V tile range of each tile
  int ubeg, uend;      // union of the valid tiles' ranges
};

__device__ __forceinline__ void tile_range(const FwdParams &p, int row0, int &beg, int &end) {
  const int i1 = min(row0 + kBM, p.Nq);
  const int off = p.Nk - p.Nq;
  const int p0 = row0 + off, p1 = i1 - 1 + off;
  const int nkt = (p.Nk + kBN - 1) / kBN;
  beg = 0;
  end = nkt;
  if (p.causal) {
    end = min(nkt, p1 / kBN + 1);
    if (p.window > 0) {
      const int lo = p0 - p.window + 1;
      beg = lo > 0 ? lo / kBN : 0;
    }
  }
}

__device__ __forceinline__ Item decode_item(const FwdParams &p, int item) {
  Item it;
  const int rb = p.n_row_blocks - 1 - item / p.n_slots;  // longest (last) row blocks first
  const int slot = item % p.n_slots;
  if (p.heads_mode) {
    const int hp = p.Hq / 2;
    it.b = slot / hp;
    const int h0 = (slot % hp) * 2;
    it.bh[0] = it.b * p.Hq + h0;
    it.bh[1] = it.bh[0] + 1;
    it.kvh = h0 / p.group;
    it.row0[0] = it.row0[1] = rb * kBM;
  } else {
    it.b = slot / p.Hq;
    const int h = slot % p.Hq;
    it.bh[0] = it.bh[1] = slot;
    it.kvh = h / p.group;
    it.row0[0] = rb * 2 * kBM;
    it.row0[1] = rb * 2 * kBM + kBM;
  }
  it.ubeg = 1 << 30;
  it.uend = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.valid[t] = it.row0[t] < p.Nq;
    it.beg[t] = it.end[t] = 0;
    if (it.valid[t]) {
      tile_range(p, it.row0[t], it.beg[t], it.end[t]);
      it.ubeg = min(it.ubeg, it.beg[t]);
      it.uend = max(it.uend, it.end[t]);
    }
  }
  return it;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NS = C::kStages;
  constexpr int QB = C::kQBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t bar0 = smem_u32(bars);
  auto bQfull = [&](int t, int q) { return bar0 + 8u * (t * QB + q); };
  auto bQfree = [&](int t, int q) { return bar0 + 8u * (2 * QB + t * QB + q); };
  auto bKVfull = [&](int s) { return bar0 + 8u * (4 * QB + s); };
  auto bKVempty = [&](int s) { return bar0 + 8u * (4 * QB + NS + s); };
  const uint32_t bX = bar0 + 8u * (4 * QB + 2 * NS);  // per-tile barriers follow
  auto bSfull = [&](int t) { return bX + 8u * (0 + t); };
  auto bOfinal = [&](int t) { return bX + 8u * (2 + t); };
  auto bDrain = [&](int t) { return bX + 8u * (4 + t); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int t = 0; t < 2; ++t) {
      for (int q = 0; q < QB; ++q) {
        mbar_init(bQfull(t, q), 1);
        mbar_init(bQfree(t, q), 1);
      }
      mbar_init(bSfull(t), 1);
      mbar_init(bOfinal(t), 1);
      mbar_init(bDrain(t), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKVfull(s), 1);
      mbar_init(bKVempty(s), 2);  // one arrival per query tile, whether or not it used the slot
    }
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
  const int wg = warp >> 2;

  if (wg == 0) {
    regs_dec<kRegsWG0>();
    if (warp == 0) {
      // ============================================================ TMA producer
      // The loop runs on the whole warp (uniform control flow and addresses);
      // one elected lane issues each copy.
      if (elect_one()) {
        tma_prefetch_desc(&p.tmQ);
        tma_prefetch_desc(&p.tmK);
        tma_prefetch_desc(&p.tmV);
      }
      __syncwarp();
      int nq[2] = {0, 0};
      int ckv = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        const Item it = decode_item(p, item);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || !it.valid[t]) continue;
          const int k = nq[t], q = k % QB;
          if (k >= QB && !mbar_wait_warp(bQfree(t, q), ((k / QB) - 1) & 1, wc, kErrWaitQFree)) {
            ok = false;
            continue;
          }
          const uint32_t dst = sQ + (t * QB + q) * C::kQBytes;
          if (elect_one()) {
            mbar_arrive_expect_tx(bQfull(t, q), C::kQBytes);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(dst + c * C::kBoxBytes, &p.tmQ, bQfull(t, q), c * 64, it.row0[t], it.bh[t]);
          }
          __syncwarp();
          nq[t] = k + 1;
        }
        const int zkv = it.b * p.Hkv + it.kvh;
        for (int j = it.ubeg; ok && j < it.uend; ++j) {
          const int c = ckv, s = c % NS;
          if (c >= NS && !mbar_wait_warp(bKVempty(s), ((c / NS) - 1) & 1, wc, kErrWaitKVEmpty)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(bKVfull(s), 2 * C::kTileBytes);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
              tma_load_3d(sK + s * C::kTileBytes + cc * C::kBoxBytes, &p.tmK, bKVfull(s), cc * 64, j * kBN, zkv);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
              tma_load_3d(sV + s * C::kTileBytes + cc * C::kBoxBytes, &p.tmV, bKVfull(s), cc * 64, j * kBN, zkv);
          }
          __syncwarp();
          ckv = c + 1;
        }
      }
      // Never leave the CTA with one of our copies still in flight.
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
          for (int k = max(0, nq[t] - QB); k < nq[t]; ++k) mbar_drain(bQfull(t, k % QB), (k / QB) & 1);
        for (int c = max(0, ckv - NS); c < ckv; ++c) mbar_drain(bKVfull(c % NS), (c / NS) & 1);
      }
    }
    __syncwarp();
  } else {
    regs_inc<kRegsSoftmax>();
    // ============================================== softmax and MMA issue of tile t
    const int t = wg - 1;
    const int quad = warp & 3;
    const bool issuer = (quad == 0);  // this warp issues the tile's MMAs from one elected lane
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t scol = tmem + lane_off + t * 128;
    const uint32_t ocol = tmem + lane_off + C::kColO + t * D;
    const uint32_t named_bar = 1 + t;  // the 4 warps of this warpgroup
    const float sl2 = p.scale_log2;
    int ns = 0, nfin = 0, nq = 0;
    int ckv = 0;       // ring slots passed (both tiles walk every slot of every item)
    int kv_seen = -1;  // last ring slot whose K/V arrival this warp has waited for
    // `ok` is this thread's view (the issuer warp also fails on its own
    // waits); `wg_ok` is the warpgroup's, agreed at every named barrier, and
    // only it decides whether to leave a loop.
    bool ok = true, wg_ok = true;
    // issuer warp only: wait until ring slot c holds K_j / V_j
    auto wait_kv = [&](int c) -> bool {
      if (c <= kv_seen) return true;
      if (!mbar_wait_warp(bKVfull(c % NS), (c / NS) & 1, wc, kErrWaitKV)) return false;
      kv_seen = c;
      return true;
    };
    // issuer warp only: a slot this tile does not read is released as soon as
    // it is filled (so that the arrival counts towards this fill, not the last)
    auto pass_slot = [&](int c) -> bool {
      if (!wait_kv(c)) return false;
      if (elect_one()) umma_commit(bKVempty(c % NS));
      __syncwarp();
      return true;
    };
    for (int item = blockIdx.x; wg_ok && item < p.n_items; item += gridDim.x) {
      const Item it = decode_item(p, item);
      // this warpgroup's tile, as scalars (t is not a compile-time index)
      const bool tvalid = t ? it.valid[1] : it.valid[0];
      const int trow0 = t ? it.row0[1] : it.row0[0];
      const int tbeg = tvalid ? (t ? it.beg[1] : it.beg[0]) : it.uend;
      const int tend = tvalid ? (t ? it.end[1] : it.end[0]) : it.uend;
      const int tbh = t ? it.bh[1] : it.bh[0];
      const int c0 = ckv - it.ubeg;  // ring slot of K/V tile j is c0 + j
      const int qbuf = nq % QB;
      const uint32_t sQt = sQ + (t * QB + qbuf) * C::kQBytes;  // this tile's Q buffer
      if (issuer) {
        for (int j = it.ubeg; ok && j < tbeg; ++j) ok = pass_slot(c0 + j);
        if (ok && tvalid) {
          // the first S = Q K^T of this tile
          ok = mbar_wait_warp(bQfull(t, qbuf), (nq / QB) & 1, wc, kErrWaitQ) && wait_kv(c0 + tbeg);
          if (ok) {
            tc_fence_after();
            const uint64_t qd = sdesc_sw128(sQt, 16, 1024);
            const uint64_t kd = sdesc_sw128(sK + ((c0 + tbeg) % NS) * C::kTileBytes, 16, 1024);
            if (elect_one()) {
              mma_qk<D, BF16>(tmem + t * 128, qd, kd);
              umma_commit(bSfull(t));
              if (tbeg + 1 == tend) umma_commit(bQfree(t, qbuf));
            }
            __syncwarp();
          }
        }
      }
      ckv = c0 + it.uend;
      wg_ok = named_bar_and(named_bar, 128, ok);
      if (!wg_ok) break;
      if (!tvalid) continue;
      nq++;
      const int pos = trow0 + row + (p.Nk - p.Nq);  // absolute position of this query row
      const int p0 = trow0 + (p.Nk - p.Nq);
      const int p1 = min(trow0 + kBM, p.Nq) - 1 + (p.Nk - p.Nq);
      float m = -INFINITY;  // running max of scaled scores, log2 domain (may lag by < 2^8)
      float l = 0.f;        // running sum of exp2(s * sl2 - m), fp32
      for (int j = tbeg; j < tend; ++j) {
        // A failed wait still goes through this iteration's barrier, so that
        // the whole warpgroup leaves together.
        ok = ok && mbar_wait_warp(bSfull(t), ns & 1, wc, kErrWaitS);
        if (ok) {
          ns++;
          tc_fence_after();
          uint32_t sr[kBN];
          tmem_ld128(scol, sr);
          const int key0 = j * kBN;
          const bool need_mask = (key0 + kBN - 1 >= p.Nk) || (p.causal && key0 + kBN - 1 > p0) ||
                                 (p.window > 0 && key0 <= p1 - p.window);
          if (need_mask) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (!key_live(key0 + c, pos, p.Nk, p.causal, p.window)) sr[c] = 0xff800000u;  // -inf
          }
          // row max: eight independent chains of 3-input max, then a short tree
          float mx[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) mx[c] = __uint_as_float(sr[c]);
#pragma unroll
          for (int c = 8; c < kBN; c += 16) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
          }
          const float mxa = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
          const float m_new = fmaxf(m, mxa * sl2);
          // Lazy rescale: move the reference max only when it grew by more
          // than 2^8 somewhere in the warp (the first tile of an item always
          // sets it).
          float alpha = 1.f;
          const bool first = (j == tbeg);
          const bool rescale = !first && __any_sync(0xffffffffu, m_new > m + kRescaleLog2);
          if (first || rescale) {
            alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
            m = m_new;
          }
          const float mref = (m == -INFINITY) ? 0.f : m;
          // p = 2^(s * sm_scale * log2 e - m), two elements per packed FMA
          const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-mref, -mref);
          float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = ffma2(make_float2(__uint_as_float(sr[c * 32 + 2 * i]),
                                                 __uint_as_float(sr[c * 32 + 2 * i + 1])),
                                     sl2x2, negm);
              const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              pk[i] = pack2<BF16>(e.x, e.y);
              rs[i & 1] = fadd2(rs[i & 1], e);
            }
            tmem_st16(scol + c * 16, pk);
          }
          l = l * alpha + ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y));
          if (rescale) {
            // S_t(j) is complete, so the P V of tile j-1 (issued before the
            // QK of tile j, by the same thread, on the in-order tensor pipe)
            // is too: O_t can be rescaled before the P V of tile j is issued.
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(ocol + c * 32, r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(ocol + c * 32, r);
            }
          }
          tmem_st_wait();
          tc_fence_before();
        }
        wg_ok = named_bar_and(named_bar, 128, ok);  // P_t(j) (and O_t) written by all four warps
        if (!wg_ok) break;
        if (issuer) {
          const int c = c0 + j;
          const bool more = (j + 1 < tend);
          // Wait for the next K/V before issuing anything: with none of our
          // MMAs in flight the check is cheap.
          if (more) ok = wait_kv(c + 1);
          if (ok) {
            tc_fence_after();
            const uint64_t vd = sdesc_sw128(sV + (c % NS) * C::kTileBytes, C::kBoxBytes, 1024);
            const uint64_t qd = sdesc_sw128(sQt, 16, 1024);
            const uint64_t kd = sdesc_sw128(sK + ((c + 1) % NS) * C::kTileBytes, 16, 1024);
            const uint32_t acc = (j > tbeg) ? 1u : 0u;
            if (elect_one()) {
              mma_pv<D, BF16>(tmem + C::kColO + t * D, tmem + t * 128, vd, acc);
              umma_commit(bKVempty(c % NS));
              if (more) {
                mma_qk<D, BF16>(tmem + t * 128, qd, kd);
                umma_commit(bSfull(t));
                if (j + 2 == tend) umma_commit(bQfree(t, qbuf));
              } else {
                umma_commit(bOfinal(t));
              }
            }
            __syncwarp();
          }
        }
      }
      if (!wg_ok) break;
      if (issuer)
        for (int j = tend; ok && j < it.uend; ++j) ok = pass_slot(c0 + j);
      // ---- epilogue of this tile: O / l -> 16-bit, LSE = (m + log2 l) ln 2
      ok = ok && mbar_wait_warp(bOfinal(t), nfin & 1, wc, kErrWaitOFinal);
      wg_ok = named_bar_and(named_bar, 128, ok);
      if (!wg_ok) break;
      nfin++;
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const int grow = trow0 + row;
      const bool live_row = grow < p.Nq;
      uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) +
                      (static_cast<size_t>(tbh) * p.Nq + (live_row ? grow : 0)) * (D * 2);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(ocol + c * 32, r);
        if (live_row) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2<BF16>(__uint_as_float(r[q * 8 + 0]) * inv, __uint_as_float(r[q * 8 + 1]) * inv);
            w.y = pack2<BF16>(__uint_as_float(r[q * 8 + 2]) * inv, __uint_as_float(r[q * 8 + 3]) * inv);
            w.z = pack2<BF16>(__uint_as_float(r[q * 8 + 4]) * inv, __uint_as_float(r[q * 8 + 5]) * inv);
            w.w = pack2<BF16>(__uint_as_float(r[q * 8 + 6]) * inv, __uint_as_float(r[q * 8 + 7]) * inv);
            *reinterpret_cast<uint4 *>(orow + c * 64 + q * 16) = w;
          }
        }
      }
      // The next item's first P V (accumulate = 0) overwrites O_t; it is
      // issued after a named barrier that every warp reaches only after this
      // read has completed (tcgen05.ld waits for its data).
      tc_fence_before();
      if (live_row && p.lse != nullptr)
        p.lse[static_cast<size_t>(tbh) * p.Nq + grow] =
            ((l > 0.f) ? m + log2f(l) : -INFINITY) * 0.69314718055994530942f;
    }
    // Never release TMEM with one of our MMAs in flight: the commit comes from
    // the lane that issued them.
    if (issuer && elect_one()) {
      umma_commit(bDrain(t));
      mbar_drain(bDrain(t), 0);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn

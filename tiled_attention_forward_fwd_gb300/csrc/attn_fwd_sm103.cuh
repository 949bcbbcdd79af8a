// attn_fwd_sm103.cuh -- tiled attention forward (prefill) for sm_103a.
//
// The computation is the tiling of the cruxr.ai "FlashAttention" section
// (outer loop over Q blocks, inner loop over K/V blocks, online softmax with a
// running max and running sum, one write of O) and of the lab 02 kernel
// skeleton (running max m, running sum l and an fp32 accumulator per query
// row; O / l and the log-sum-exp m + log l stored at the end).
//
// GB300 mapping.  A persistent grid (one CTA per SM) walks a static list of
// work items, longest first, in passes that alternate direction.  An item is
// up to two 128-row query tiles that read the same K/V rows (two heads of one
// GQA group at the same rows, or two row tiles of one head; the host picks
// the pairing per call).  12 warps in three warpgroups:
//   WG0  warp 0: TMA producer -- Q tiles, then K_j / V_j into an NS-stage
//                shared-memory ring (128B-swizzled boxes of 128 rows x 64 cols;
//                K_j and V_j complete one barrier)
//        warp 1: owns TMEM (512 columns: allocation and release)
//        warps 2, 3: MMA issuer of tile 0 / tile 1, tcgen05.mma from one
//                elected lane of the converged warp:
//                  S_t = Q_t K_j^T  (A, B in shared memory, fp32 in TMEM)
//                  O_t += P_t V_j   (A = P_t in TMEM, B = V_j in shared memory)
//   WG1, WG2     softmax of tile 0 / tile 1: thread r owns query row r (TMEM
//                lane r); loads its S row, masks, keeps the running max and
//                sum in the log2 domain (sm_scale folded into log2 e), writes
//                P as packed 16-bit pairs to TMEM, and rescales its O row in
//                TMEM only when the running max grew by more than 2^8; after
//                an item's last K/V tile it writes O / l (16-bit) and the LSE.
// The softmax warpgroup hands S-read and P-written to its MMA warp on named
// barriers; the MMA warp signals S ready, P V done and O final on mbarriers
// through tcgen05.commit.  TMEM layout and epilogue per head dim: FwdCfg.
// Every mbarrier wait is bounded (see sm103_ptx.cuh).
#pragma once

#include "fastdiv.h"
#include "sm103_ptx.cuh"

namespace attn {

constexpr int kBM = 128;  // query rows per tile (tcgen05 M)
constexpr int kBN = 128;  // keys per K/V tile (MMA N of S, MMA K of P V)
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold: a factor 256
constexpr float kRescaleSum = 256.0f;  // 2^kRescaleLog2

enum DeviceError : int {
  kErrWaitQ = 0x101,
  kErrWaitKV = 0x102,
  kErrWaitKVEmpty = 0x103,
  kErrWaitS = 0x104,
  kErrWaitOFinal = 0x107,
  kErrWaitQFree = 0x108,
  kErrWaitPartial = 0x109,
};

// Stream-K split of a call's work over at most this many CTAs.
constexpr int kMaxSplitCtas = 256;

struct FwdParams {
  CUtensorMap tmQ;  // (d, Nq, B*Hq)
  CUtensorMap tmK;  // (d, Nk, B*Hkv)
  CUtensorMap tmV;  // (d, Nk, B*Hkv)
  CUtensorMap tmO;  // (d, Nq, B*Hq): tile stores of O (d = 64)
  void *O;          // (B*Hq*Nq, d) 16-bit
  float *lse;       // (B*Hq*Nq) or null
  int *status;      // device status word
  int B, Hq, Hkv, Nq, Nk, group;
  int causal, window;
  int pair_mode;     // how an item's two query tiles are chosen (kPair*)
  int n_row_blocks;  // items per (b, head slot)
  int n_slots;       // pair_mode == kPairHeads ? B*Hq/2 : B*Hq
  int n_items;
  FastDiv fd_slots;  // / n_slots
  FastDiv fd_heads;  // / (pair_mode == kPairHeads ? Hq/2 : Hq): the head slots of one batch
  FastDiv fd_group;  // / group
  float scale_log2;  // sm_scale * log2(e)
  unsigned long long timeout_ns;
  int stall_after;  // test hook: the producer stops after this many K/V tiles (-1: never)
  // Stream-K split (the kSchedSplit kernel): the items, in order, form one
  // sequence of K/V tile steps (each item its union range); CTA c takes the
  // steps from split_at[c] to split_at[c + 1] (x = item, y = step within the
  // item).  An item cut between CTAs is finished by the CTA holding its first
  // steps: the others leave their partial O (fp32, not normalised) and (m, l)
  // per row in the workspace and set their flag to `token` (fresh per
  // enqueued call, so it never matches what other calls left there); the
  // merging CTA clears each flag it consumed, so a graph replay under the
  // same token waits for its own partials.
  unsigned token;
  float *ws_o;        // [CTA][tile][D][128 rows]: a warp's 32 rows of one column are contiguous
  float2 *ws_ml;      // [CTA][tile][128 rows]
  unsigned *ws_flag;  // [CTA][tile]
  int2 split_at[kMaxSplitCtas + 1];
  // Paged K/V (the kPaged kernels; the motivation page's "PagedAttention es
  // un problema distinto"): token t of request b sits in pool page
  // block_table[b * max_pages + t / page_size], slot t % page_size; request b
  // holds seq_lens[b] keys (read on the device; Nk is the largest), and its
  // query rows are its last Nq positions.  tmK / tmV view the pools as (d,
  // page_size, num_pages * Hkv) with boxes of min(page_size, 128) rows.
  const int *block_table;
  const int *seq_lens;
  int page_shift;  // log2(page_size), 3..8
  int max_pages, num_pages;
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
  //           sfull[2], ofinal[2], drain[2], pvdone[2]
  static constexpr int kNumBars = 4 * kQBufs + 2 * kStages + 8;
  static constexpr int kOffMerge = ((kOffBar + kNumBars * 8 + 16) + 15) / 16 * 16;  // float2 (m, l)[128]
  static constexpr int kSmemBytes = kOffMerge + kBM * 8 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns of tile t.  d = 64: S [256t, +128), P [256t + 128, +64) and
  // O [256t + 192, +64): with P apart from S, the Q K^T of the next key block
  // can run while the softmax of this one computes P.  d = 128 has no room
  // for that: P is written over S [128t, +128) and O is [256 + 128t, +128).
  static constexpr bool kSeparateP = (D == 64);
  // d = 64 (softmax-bound): exp2 with the running max first, the row max
  // only when the row sum shows that the max grew past the lazy-rescale
  // threshold; d = 128 (MMA-bound): max first, then exp2.
  static constexpr bool kSpeculativeP = (D == 64);
  // d = 64: the epilogue stages the O tile in the item's Q buffer (free once
  // the tile's last Q K^T is done) and writes it with one TMA store; the
  // softmax warpgroup, not the MMA warp, then releases the Q buffer.  d = 128
  // (one Q buffer per tile, long items) stores rows from registers.
  static constexpr bool kStoreOViaSmem = (D == 64);
  static constexpr uint32_t kColS = kSeparateP ? 256 : 128;  // S column stride per tile
  static constexpr uint32_t kColP = kSeparateP ? 128 : 0;    // P offset within the tile's columns
  static constexpr uint32_t kColO0 = kSeparateP ? 192 : 256; // O_0
  static constexpr uint32_t kColOStride = kSeparateP ? 256 : D;
  static constexpr int kThreads = 384;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Register budget per warpgroup after setmaxnreg.  The kernel is launched
// with 384 threads x 168 registers = 64512; the split must not exceed that.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsWG0 = 72, kRegsSoftmax = 216;
static_assert(128 * kRegsWG0 + 256 * kRegsSoftmax <= 384 * kLaunchRegs, "register split");


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
// Under a stream-K split a CTA may hold only a piece of it: the K/V tiles
// [ubeg, uend) of the item's union range [iubeg, iuend).
struct Item {
  int b, kvh;
  int bh[2];    // b * Hq + h of each tile
  int row0[2];  // first query row of each tile
  bool valid[2];       // the tile has K/V tiles in this piece
  bool exists[2];      // the tile is part of the item
  int beg[2], end[2];  // live K/V tile range of each tile in this piece
  int ubeg, uend;      // union of the valid tiles' ranges in this piece
  int obeg[2], oend[2];  // live K/V tile range of each tile in the whole item
  int iubeg, iuend;      // union range of the whole item
  int item;
  int nk;                // keys of the item's request (Nk unless paged)
};

// Live K/V tiles [beg, end) of the query tile at row0 of a request with nk keys.
ATTN_HD void tile_range(const FwdParams &p, int row0, int nk, int &beg, int &end) {
  const int i1 = min(row0 + kBM, p.Nq);
  const int off = nk - p.Nq;
  const int p0 = row0 + off, p1 = i1 - 1 + off;
  const int nkt = (nk + kBN - 1) / kBN;
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

// Item shapes (the host picks one per call):
//   kPairHeads   two query heads of one GQA group at the same 128 rows: each
//                K/V tile load serves both (group size even)
//   kPairRows    row tiles 2r and 2r+1 of one head (the default otherwise)
//   kPairSingle  one row tile per item: few tiles, each of at most 3 K/V tiles
//   kPairHalves  one row tile per item, its K/V tiles split between the two
//                tiles of the item (tile 0 the first half, tile 1 the rest),
//                loaded into the ring interleaved and merged at the end: both
//                softmax warpgroups work on every item (few, longer tiles)
enum PairMode : int { kPairRows = 0, kPairHeads = 1, kPairSingle = 2, kPairHalves = 3 };

#ifdef __CUDACC__
// Keys of paged request b, read on the device: a length out of range (below
// Nq when causal, below 1, above the largest) is recorded and clamped.
__device__ __forceinline__ int request_keys(const FwdParams &p, int b) {
  int len = __ldg(p.seq_lens + b);
  const int lo = p.causal ? p.Nq : 1;
  if (len < lo || len > p.Nk) {
    atomicCAS(p.status, 0, kErrDeviceArg);
    len = min(max(len, lo), p.Nk);
  }
  return len;
}
#endif

template <bool kPaged = false>
ATTN_HD Item decode_item(const FwdParams &p, int item) {
  Item it;
  it.item = item;
  int idx, slot, hs;
  fastdiv_divmod(p.fd_slots, item, idx, slot);  // idx: longest items first
  fastdiv_divmod(p.fd_heads, slot, it.b, hs);
  it.nk = p.Nk;
  if constexpr (kPaged) {
#ifdef __CUDA_ARCH__
    it.nk = request_keys(p, it.b);
#endif
  }
  if (p.pair_mode == kPairHeads) {
    const int rb = p.n_row_blocks - 1 - idx;
    const int h0 = hs * 2;
    it.bh[0] = it.b * p.Hq + h0;
    it.bh[1] = it.bh[0] + 1;
    it.kvh = static_cast<int>(fastdiv_div(p.fd_group, h0));
    it.row0[0] = it.row0[1] = rb * kBM;
  } else {
    it.bh[0] = it.bh[1] = slot;
    it.kvh = static_cast<int>(fastdiv_div(p.fd_group, hs));
    if (p.pair_mode == kPairRows) {
      const int rb = p.n_row_blocks - 1 - idx;
      it.row0[0] = rb * 2 * kBM;
      it.row0[1] = rb * 2 * kBM + kBM;
    } else {
      it.row0[0] = (p.n_row_blocks - 1 - idx) * kBM;
      // kPairSingle: no second tile; kPairHalves: the same rows
      it.row0[1] = (p.pair_mode == kPairHalves) ? it.row0[0] : p.Nq;
    }
  }
  it.ubeg = 1 << 30;
  it.uend = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.valid[t] = it.row0[t] < p.Nq;
    it.exists[t] = it.valid[t];
    it.beg[t] = it.end[t] = 0;
    if (it.valid[t]) {
      tile_range(p, it.row0[t], it.nk, it.beg[t], it.end[t]);
      it.ubeg = it.ubeg < it.beg[t] ? it.ubeg : it.beg[t];
      it.uend = it.uend > it.end[t] ? it.uend : it.end[t];
    }
    it.obeg[t] = it.beg[t];
    it.oend[t] = it.end[t];
  }
  if (p.pair_mode == kPairHalves && it.valid[0]) {
    // the first half of the K/V tiles (rounded up) to tile 0, the rest to tile 1
    const int mid = it.beg[0] + (it.end[0] - it.beg[0] + 1) / 2;
    it.end[0] = it.oend[0] = mid;
    it.beg[1] = it.obeg[1] = mid;
    it.valid[1] = it.exists[1] = mid < it.end[1];
  }
  it.iubeg = it.ubeg;
  it.iuend = it.uend;
  return it;
}

// K/V tile held by ring position k of an item (k from 0).  The ring is loaded
// in the item's union order, except under kPairHalves, where the two tiles'
// ranges alternate: tile 0's i-th, tile 1's i-th, ..., then the rest of the
// longer one (tile 0's; tile 1 has at most as many).
template <bool kHalves>
ATTN_HD int ring_block(const Item &it, int k) {
  if (!kHalves || !it.valid[1]) return it.ubeg + k;
  const int n1 = it.end[1] - it.beg[1];
  if (k < 2 * n1) return (k & 1) ? it.beg[1] + (k >> 1) : it.beg[0] + (k >> 1);
  return it.beg[0] + (k - n1);
}
// Ring position of tile t's i-th K/V tile of the item.
template <bool kHalves>
ATTN_HD int ring_pos(const Item &it, int t, int i) {
  if (!kHalves || !it.valid[1]) return (t ? it.beg[1] : it.beg[0]) - it.ubeg + i;
  const int n1 = it.end[1] - it.beg[1];
  return (i < n1) ? 2 * i + t : n1 + i;
}

// Restrict an item to the K/V tiles [iubeg + s0, iubeg + s1) of its union
// range; a tile with none of them is not valid in the piece.
ATTN_HD void clip_item(Item &it, int s0, int s1) {
  const int lo = it.iubeg + s0;
  const int hi = (it.iubeg + s1 < it.iuend) ? it.iubeg + s1 : it.iuend;
  it.ubeg = lo;
  it.uend = hi;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.beg[t] = it.obeg[t] > lo ? it.obeg[t] : lo;
    it.end[t] = it.oend[t] < hi ? it.oend[t] : hi;
    it.valid[t] = it.exists[t] && it.beg[t] < it.end[t];
  }
}

// Items are handed to the g persistent CTAs in passes of g, alternating
// direction ("snake"): with items sorted longest first, every CTA gets a
// similar total.  Returns the m-th item of CTA c (>= n_items: none).
ATTN_HD int item_of(int m, int c, int g) { return m * g + ((m & 1) ? (g - 1 - c) : c); }

// Number of work pieces of CTA c of g: passes over the item list, or the
// items that its stream-K range touches.
template <bool kSplit>
ATTN_HD int num_pieces(const FwdParams &p, int c, int g) {
  if constexpr (!kSplit) return (p.n_items + g - 1) / g;
  const int2 s = p.split_at[c], e = p.split_at[c + 1];
  const int last = (e.y > 0) ? e.x : e.x - 1;  // last item touched
  if (s.x > last || (s.x == e.x && s.y >= e.y)) return 0;
  return last - s.x + 1;
}

// The k-th piece of the work of CTA c of g; false when there is none (the
// last pass over the item list may be short).
template <bool kSplit, bool kPaged = false>
ATTN_HD bool piece_at(const FwdParams &p, int c, int g, int k, Item &it) {
  if constexpr (!kSplit) {
    const int item = item_of(k, c, g);
    if (item >= p.n_items) return false;
    it = decode_item<kPaged>(p, item);
    return true;
  }
  const int2 s = p.split_at[c], e = p.split_at[c + 1];
  const int item = s.x + k;
  it = decode_item<kPaged>(p, item);
  clip_item(it, k == 0 ? s.y : 0, item == e.x ? e.y : (1 << 30));
  return true;
}

// Row max of a 128-column S row: eight independent chains, columns 0-15 by
// a 2-input max, then 16 columns per 3-input max step.
__device__ __forceinline__ void softmax_rowmax(const uint32_t (&sr)[kBN], float (&mx)[8]) {
  static_assert(kBN % 16 == 0, "16 columns per step");
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[8 + k]));
#pragma unroll
  for (int c = 16; c < kBN; c += 16) {
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
  }
}
__device__ __forceinline__ float softmax_max8(const float (&mx)[8]) {
  return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
}

// p = 2^(s * sm_scale * log2 e - m) for the 128 columns of a row, two per
// packed FMA, written to TMEM as packed 16-bit pairs (32 columns per chunk);
// rs gets the fp32 sum.  before_store() runs once, after the first chunk's
// exp2 and before its store: a wait for P to be free costs no exp2 latency.
template <bool BF16, typename BeforeStore>
__device__ __forceinline__ void softmax_p(const uint32_t (&sr)[kBN], float2 sl2x2, float m, float2 (&rs)[2],
                                          uint32_t pcol, BeforeStore before_store) {
  const float mref = (m == -INFINITY) ? 0.f : m;
  const float2 negm = make_float2(-mref, -mref);
  rs[0] = rs[1] = make_float2(0.f, 0.f);
#pragma unroll
  for (int cc = 0; cc < kBN / 32; ++cc) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 x = ffma2(make_float2(__uint_as_float(sr[cc * 32 + 2 * i]), __uint_as_float(sr[cc * 32 + 2 * i + 1])),
                             sl2x2, negm);
      const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      pk[i] = pack2<BF16>(e.x, e.y);
      rs[i & 1] = fadd2(rs[i & 1], e);
    }
    if (cc == 0) before_store();
    tmem_st16(pcol + cc * 16, pk);
  }
}

// Named barriers (id 0 is __syncthreads), each between one softmax warpgroup
// (128 threads, which only arrive) and its tile's MMA warp (32, which waits).
constexpr uint32_t kBarP = 1, kBarSRead = 3, kBarHandoffThreads = 128 + 32;
// Named barrier of one softmax warpgroup alone: its O tile is staged.
constexpr uint32_t kBarOStaged = 5;
// kPairHalves merge, both softmax warpgroups (256 threads): tile 0's (m, l)
// and final O are ready (tile 0 arrives, tile 1 syncs); tile 1 has read them
// (tile 1 arrives, tile 0 syncs).
constexpr uint32_t kBarHalfReady = 7, kBarHalfRead = 8, kBarHalvesThreads = 256;


// Schedules, one kernel each: the plain item list, the stream-K split
// (FwdParams::split_at) and the kPairHalves items; each is compiled without
// the others' code.
enum Sched : int { kSchedPlain = 0, kSchedSplit = 1, kSchedHalves = 2 };

template <int D, bool BF16, int kSched, bool kPaged = false>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr bool kSplit = kSched == kSchedSplit;
  constexpr bool kHalves = kSched == kSchedHalves;
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
  auto bPVdone = [&](int t) { return bX + 8u * (6 + t); };  // separate-P layout only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};
  pdl_launch_dependents();  // the next call's prologue may overlap this one

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
      mbar_init(bPVdone(t), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKVfull(s), 1);
      mbar_init(bKVempty(s), 2);  // one arrival per query tile, whether or not it used the slot
    }
    fence_mbar_init();
  }
  if (warp == 0 && elect_one()) {
    // the tensor maps are launch parameters: fetch them while the previous
    // kernel on the stream may still run
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
    if (C::kStoreOViaSmem) tma_prefetch_desc(&p.tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // inputs may come from the previous kernel on the stream
  const uint32_t tmem = *tmem_slot;
  const int wg = warp >> 2;

  if (wg == 0) {
    regs_dec<kRegsWG0>();
    if (warp == 0) {
      // ============================================================ TMA producer
      // The loop runs on the whole warp (uniform control flow and addresses);
      // one elected lane issues each copy.
      int nq[2] = {0, 0};
      int ckv = 0;
      bool ok = true;
      const int npieces = num_pieces<kSplit>(p, blockIdx.x, gridDim.x);
      for (int pk = 0; ok && pk < npieces; ++pk) {
        Item it;
        if (!piece_at<kSplit, kPaged>(p, blockIdx.x, gridDim.x, pk, it)) continue;
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
        for (int k = 0; ok && k < it.uend - it.ubeg; ++k) {
          const int j = ring_block<kHalves>(it, k);  // K/V tile of ring position k
          const int c = ckv, s = c % NS;
          if (p.stall_after >= 0 && c >= p.stall_after) {  // test hook: stop loading
            ok = false;
            break;
          }
          if (c >= NS && !mbar_wait_warp(bKVempty(s), ((c / NS) - 1) & 1, wc, kErrWaitKVEmpty)) {
            ok = false;
            break;
          }
          if constexpr (!kPaged) {
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
          } else {
            // The tile's keys [j * 128, +128) lie in 128 / page_size pages
            // (or in part of one page).  Lane l holds the pool slab (page *
            // Hkv + kv head) of the l-th page and copies its box; a page past
            // the request's end, or an index outside the pool (recorded),
            // becomes the slab one past the pool, which reads as zeros.
            const int sh = p.page_shift;
            const int npg = sh < 7 ? (kBN >> sh) : 1;
            const int lp = ((j * kBN) >> sh) + lane;  // logical page of lane l
            int slab = p.num_pages * p.Hkv;
            if (lane < npg && lp < ((it.nk + (1 << sh) - 1) >> sh)) {
              const int page = __ldg(p.block_table + static_cast<size_t>(it.b) * p.max_pages + lp);
              if (page >= 0 && page < p.num_pages)
                slab = page * p.Hkv + it.kvh;
              else
                atomicCAS(p.status, 0, kErrDeviceArg);
            }
            const int y = sh < 7 ? 0 : (j * kBN) & ((1 << sh) - 1);  // first row within the page
            const uint32_t off = sh < 7 ? static_cast<uint32_t>(lane << sh) * 128u : 0u;
            if (elect_one()) mbar_arrive_expect_tx(bKVfull(s), 2 * C::kTileBytes);
            __syncwarp();
            if (lane < npg) {
#pragma unroll
              for (int cc = 0; cc < D / 64; ++cc)
                tma_load_3d(sK + s * C::kTileBytes + cc * C::kBoxBytes + off, &p.tmK, bKVfull(s), cc * 64, y, slab);
#pragma unroll
              for (int cc = 0; cc < D / 64; ++cc)
                tma_load_3d(sV + s * C::kTileBytes + cc * C::kBoxBytes + off, &p.tmV, bKVfull(s), cc * 64, y, slab);
            }
            __syncwarp();
          }
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
    } else if (warp >= 2) {
      // ====================================================== MMA issuer of tile t
      // One warp per query tile (warps 2 and 3), so that neither tile waits
      // for the other's issue.  The loop runs on the whole warp; one elected
      // lane issues each MMA and commit.  Handoffs from the tile's softmax
      // warpgroup are named barriers that the warpgroup arrives at (without
      // waiting) and this warp syncs on:
      //   kBarP + t       P_t(j) is in TMEM  -> P V of block j may be issued
      //   kBarSRead + t   S_t(j) is in the softmax registers -> the next
      //                   Q K^T may overwrite it (separate-P layout only)
      // An arrival never meets the previous use of its barrier still open:
      // the warpgroup arrives for block j+1 only after waiting for S_t(j+1)
      // (and, with separate P, for P V of block j), which this warp issues
      // after its syncs for block j.  Every barrier of the fixed sequence is
      // taken even after a failed wait, so this warp is never left waiting.
      const int t = warp - 2;
      int nq = 0;        // items of this tile started (Q buffer use)
      int ckv = 0;       // ring slots passed
      int kv_seen = -1;  // last ring slot whose arrival was waited for
      bool ok = true;
      // the pending P V: (stage, accumulate, last) of the previous step, and
      // (paged) the rows of its V tile that hold the request's keys
      bool pending = false;
      int pv_stage = 0;
      uint32_t pv_acc = 0;
      bool pv_last = false;
      int pv_valid = kBN;
      auto wait_kv = [&](int c) {
        if (ok && c > kv_seen) {
          ok = mbar_wait_warp(bKVfull(c % NS), (c / NS) & 1, wc, kErrWaitKV);
          kv_seen = c;
        }
      };
      // a ring slot this tile does not read is released once filled (so that
      // the arrival counts towards this fill, not the last)
      auto pass_slot = [&](int c) {
        wait_kv(c);
        if (ok && elect_one()) umma_commit(bKVempty(c % NS));
        __syncwarp();
      };
      // After an abort (ok false) no MMA is issued, but S full, P V done and
      // O final are still signalled, by a plain arrival: the softmax
      // warpgroup keeps waiting for them, so that it never arrives at a
      // handoff barrier before this warp has passed that barrier's previous
      // phase (an arrive-only side that ran ahead could complete a phase
      // without this warp and leave its next sync waiting forever), and so
      // that no P V done phase is left pending into the next item (O final
      // completes with the item's last one).
      auto issue_qk = [&](int c, int qbuf, bool last) {
        if (!ok) {
          if (elect_one()) mbar_arrive(bSfull(t));
          __syncwarp();
          return;
        }
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(sQ + (t * QB + qbuf) * C::kQBytes, 16, 1024);
        const uint64_t kd = sdesc_sw128(sK + (c % NS) * C::kTileBytes, 16, 1024);
        if (elect_one()) {
          mma_qk<D, BF16>(tmem + t * C::kColS, qd, kd);
          umma_commit(bSfull(t));
          if (last && !C::kStoreOViaSmem) umma_commit(bQfree(t, qbuf));
        }
        __syncwarp();
      };
      auto issue_pv = [&]() {
        named_bar_sync(kBarP + t, kBarHandoffThreads);
        ok = ok && !__any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(abort_flag) != 0);
        if (!ok) {
          if (elect_one()) {
            if constexpr (C::kSeparateP) mbar_arrive(bPVdone(t));
            if (pv_last) mbar_arrive(bOfinal(t));
          }
          __syncwarp();
        }
        if (kPaged && ok && pv_valid < kBN) {
          // Paged: the slots of the request's last page past its end hold
          // whatever the pool held (NaN included); their P is 0, but 0 x NaN
          // is not, so their V rows are zeroed before P V (whole 128-byte
          // rows: the swizzle permutes chunks within a row).  Rows past the
          // last page were read as zeros.
          const int zend = min(kBN, ((pv_valid + (1 << p.page_shift) - 1) >> p.page_shift) << p.page_shift);
          const uint32_t vbase = sV + pv_stage * C::kTileBytes;
          for (int r = pv_valid + lane; r < zend; r += 32)
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc)
#pragma unroll
              for (int q = 0; q < 8; ++q) st_shared_v4(vbase + cc * C::kBoxBytes + r * 128 + q * 16, 0u, 0u, 0u, 0u);
          fence_proxy_async_smem();  // the zeros are visible to the tensor core
          __syncwarp();
        }
        if (ok) {
          tc_fence_after();
          const uint64_t vd = sdesc_sw128(sV + pv_stage * C::kTileBytes, C::kBoxBytes, 1024);
          if (elect_one()) {
            mma_pv<D, BF16>(tmem + C::kColO0 + t * C::kColOStride, tmem + t * C::kColS + C::kColP, vd, pv_acc);
            umma_commit(bKVempty(pv_stage));
            if constexpr (C::kSeparateP) umma_commit(bPVdone(t));
            if (pv_last) umma_commit(bOfinal(t));
          }
          __syncwarp();
        }
        pending = false;
      };
      const int npieces = num_pieces<kSplit>(p, blockIdx.x, gridDim.x);
      for (int pk = 0; pk < npieces; ++pk) {
        Item it;
        if (!piece_at<kSplit, kPaged>(p, blockIdx.x, gridDim.x, pk, it)) continue;
        const bool tvalid = t ? it.valid[1] : it.valid[0];
        const int tbeg = tvalid ? (t ? it.beg[1] : it.beg[0]) : it.uend;
        const int tend = tvalid ? (t ? it.end[1] : it.end[0]) : it.uend;
        const int base = ckv;  // ring slot of the item's first position
        const int npos = it.uend - it.ubeg;
        // positions before this tile's first K/V tile are passed
        const int first_pos = tvalid ? ring_pos<kHalves>(it, t, 0) : npos;
        for (int k = 0; k < first_pos; ++k) pass_slot(base + k);
        int next_pos = first_pos;
        if (tvalid) {
          const int qbuf = nq % QB;
          if (ok) ok = mbar_wait_warp(bQfull(t, qbuf), (nq / QB) & 1, wc, kErrWaitQ);
          for (int j = tbeg; j < tend; ++j) {
            // positions of the other tile between this one's are passed
            const int pos_j = ring_pos<kHalves>(it, t, j - tbeg);
            for (int k = next_pos; k < pos_j; ++k) pass_slot(base + k);
            next_pos = pos_j + 1;
            const int c = base + pos_j;
            if constexpr (C::kSeparateP) {
              // S of the previous block read -> Q K^T of block j; then P V of
              // the previous block once its P is written.
              if (j > tbeg) named_bar_sync(kBarSRead + t, kBarHandoffThreads);
              wait_kv(c);
              issue_qk(c, qbuf, j + 1 == tend);
              if (pending) issue_pv();
            } else {
              // P over S: P V of the previous block must be issued before the
              // Q K^T that overwrites its P.
              if (pending) issue_pv();
              wait_kv(c);
              issue_qk(c, qbuf, j + 1 == tend);
            }
            pending = true;
            pv_stage = c % NS;
            pv_acc = (j > tbeg) ? 1u : 0u;
            pv_last = (j + 1 == tend);
            if constexpr (kPaged) pv_valid = min(kBN, it.nk - j * kBN);
          }
          // The item's last P V goes out now: it releases a K/V stage that a
          // later fill (and this warp's next waits) may need.
          if constexpr (C::kSeparateP) named_bar_sync(kBarSRead + t, kBarHandoffThreads);
          issue_pv();
          nq++;
        }
        for (int k = next_pos; k < npos; ++k) pass_slot(base + k);
        ckv = base + npos;
      }
      // Drain every MMA this warp issued before TMEM can be released (the
      // commit comes from the lane that issued them).
      if (elect_one()) {
        umma_commit(bDrain(t));
        mbar_drain(bDrain(t), 0);
      }
      __syncwarp();
    }
    __syncwarp();
  } else {
    regs_inc<kRegsSoftmax>();
    // ============================================================== softmax of tile t
    const int t = wg - 1;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t scol = tmem + lane_off + t * C::kColS;  // S (and P when shared)
    const uint32_t pcol = scol + C::kColP;                 // P
    const uint32_t ocol = tmem + lane_off + C::kColO0 + t * C::kColOStride;
    const float sl2 = p.scale_log2;
    int ns = 0, nfin = 0;
    int npv = 0;  // P V of this tile issued so far (separate P: P_t is reused once the last one is done)
    bool ok = true;
    // Q buffer whose O tile store may still be reading it; it is handed back
    // to the producer after the next P handoff (or at the end), when the
    // store has long finished reading.
    int o_pending = -1;
    auto release_staging = [&]() {
      if (quad == 0 && lane == 0) {
        tma_store_wait_read0();
        mbar_arrive(bQfree(t, o_pending));  // the producer may load a later item's Q here
      }
      __syncwarp();
      o_pending = -1;
    };
    const int npieces = num_pieces<kSplit>(p, blockIdx.x, gridDim.x);
    for (int pk = 0; pk < npieces; ++pk) {
      Item it;
      if (!piece_at<kSplit, kPaged>(p, blockIdx.x, gridDim.x, pk, it)) continue;
      // this warpgroup's tile, as scalars (t is not a compile-time index)
      const bool tvalid = t ? it.valid[1] : it.valid[0];
      if (!tvalid) continue;
      const int trow0 = t ? it.row0[1] : it.row0[0];
      const int tbeg = t ? it.beg[1] : it.beg[0];
      const int tend = t ? it.end[1] : it.end[0];
      const int tbh = t ? it.bh[1] : it.bh[0];
      const int nk = it.nk;                    // keys of this item's request
      const int pos = trow0 + row + (nk - p.Nq);  // absolute position of this query row
      const int p0 = trow0 + (nk - p.Nq);
      const int p1 = min(trow0 + kBM, p.Nq) - 1 + (nk - p.Nq);
      // kPairHalves with both halves: tile 0 hands its half to tile 1
      const bool half_out = kHalves && t == 0 && it.valid[1];
      const bool half_merge = kHalves && t == 1;
      float m = -INFINITY;  // running max of scaled scores, log2 domain (may lag by < 2^8)
      float l = 0.f;        // running sum of exp2(s * sl2 - m), fp32
      for (int j = tbeg; j < tend; ++j) {
        // The MMA warp signals S full and P V done after an abort too
        // (without MMAs then), so these waits do not poll the abort flag
        // and are always taken, and the block's work always runs (on
        // whatever S holds after an abort): this warpgroup then never
        // arrives at a handoff barrier before the MMA warp has passed that
        // barrier's previous phase.
        ok = mbar_wait_signal(bSfull(t), ns & 1, wc, kErrWaitS) && ok;
        ns++;
        uint32_t sr[kBN];
        tc_fence_after();
        tmem_ld128(scol, sr);
        if constexpr (C::kSeparateP) {
          tc_fence_before();
          named_bar_arrive(kBarSRead + t, kBarHandoffThreads);  // S_t(j) read: the next Q K^T may overwrite it
        }
        {
          const int key0 = j * kBN;
          const bool need_mask = (key0 + kBN - 1 >= nk) || (p.causal && key0 + kBN - 1 > p0) ||
                                 (p.window > 0 && key0 <= p1 - p.window);
          if (need_mask) {
            // The row's live keys are one interval: below Nk, not after the
            // row (causal), within the window.  [lo, hi) relative to key0.
            const int hi = min(nk, p.causal ? pos + 1 : nk) - key0;
            const int lo = (p.window > 0) ? pos - p.window + 1 - key0 : -1;
#pragma unroll
            for (int cc = 0; cc < kBN; ++cc)
              if (cc >= hi || cc < lo) sr[cc] = 0xff800000u;  // -inf
          }
          const bool first = (j == tbeg);
          // Separate P: P_t and O_t are free once the P V of block j-1 has
          // completed (at an item's first block the previous O-final wait
          // covered it).  The wait comes before the first P store; every
          // later access to P_t or O_t (a redo pass, the O rescale) follows.
          bool pv_waited = first;
          auto before_store = [&]() {
            if constexpr (C::kSeparateP) {
              if (!pv_waited) {
                ok = mbar_wait_signal(bPVdone(t), (npv - 1) & 1, wc, kErrWaitS) && ok;
                pv_waited = true;
              }
              tc_fence_after();
            }
          };
          const float2 sl2x2 = make_float2(sl2, sl2);
          float2 rs[2];
          float mx[8];
          float alpha = 1.f;
          bool rescale = false;
          if (first || !C::kSpeculativeP) {
            // max first: the first block of an item sets the reference max;
            // at d = 128 (MMA-bound) every block takes this shorter path
            softmax_rowmax(sr, mx);
            const float m_new = fmaxf(m, softmax_max8(mx) * sl2);
            rescale = !first && __any_sync(0xffffffffu, m_new > m + kRescaleLog2);
            if (first || rescale) {
              alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
              m = m_new;
            }
            softmax_p<BF16>(sr, sl2x2, m, rs, pcol, before_store);
          } else {
            // Speculative pass with the current reference max, no row max.
            // No p exceeds the row sum, so a sum of at most 2^8 shows that
            // the max grew by at most 8 (log2 domain) and the pass stands
            // (lazy rescale).  Otherwise, or while the row has no finite max
            // yet, the row max is taken and the pass redone; after an item's
            // first blocks that is rare.
            softmax_p<BF16>(sr, sl2x2, m, rs, pcol, before_store);
            const float rsum = (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
            rescale = __any_sync(0xffffffffu, !(rsum <= kRescaleSum) || m == -INFINITY);
            if (rescale) {
              softmax_rowmax(sr, mx);
              const float m_new = fmaxf(m, softmax_max8(mx) * sl2);
              alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
              m = m_new;
              softmax_p<BF16>(sr, sl2x2, m, rs, pcol, before_store);
            }
          }
          l = l * alpha + ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y));
          if (rescale) {
            // O_t holds blocks up to j-1 only: with separate P the P V of
            // block j-1 was waited for above; with P over S, S_t(j) completing
            // means that P V (issued before this Q K^T by the same warp, on
            // the in-order tensor pipe) has too.
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t r[32];
              tmem_ld32(ocol + cc * 32, r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(ocol + cc * 32, r);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        named_bar_arrive(kBarP + t, kBarHandoffThreads);  // P_t(j) (and O_t) written: P V of block j may go
        npv++;
        if (C::kStoreOViaSmem && o_pending >= 0) release_staging();
      }
      // ---- epilogue of this tile.  A whole item: O / l -> 16-bit and
      // LSE = (m + log2 l) ln 2.  Under a stream-K split, a piece after the
      // item's first steps hands its partial (O, m, l) on through the
      // workspace; the item's first piece merges the others' partials into its
      // own before O / l.  What does not need O is done while the last P V
      // completes.
      // (the piece is decoded again here, so that its ranges need no
      // registers during the K/V loop)
      Item ie{};
      bool part_out = false, merge_in = false;
      if constexpr (kSplit) {
        piece_at<kSplit, kPaged>(p, blockIdx.x, gridDim.x, pk, ie);
        part_out = ie.ubeg > ie.iubeg;
        merge_in = ie.ubeg == ie.iubeg && ie.uend < ie.iuend;
      }
      const int grow = trow0 + row;
      const bool live_row = grow < p.Nq;
      const int tobeg = t ? ie.obeg[1] : ie.obeg[0];
      const int toend = t ? ie.oend[1] : ie.oend[0];
      // The pieces after this one of the item are the first pieces of the
      // next CTAs; the tile has a partial in those whose steps it reaches.
      auto part_live = [&](int c) {
        const int2 a = p.split_at[c], b = p.split_at[c + 1];
        const int lo = ie.iubeg + a.y, hi = (b.x == ie.item) ? ie.iubeg + b.y : ie.iuend;
        return max(tobeg, lo) < min(toend, hi);
      };
      auto part_ml = [&](int c) {
        return __ldcg(p.ws_ml + (static_cast<size_t>(c) * 2 + t) * kBM + row);
      };
      float mf = m, lf = l;  // merged running max and sum
      if (merge_in) {
        for (int c = blockIdx.x + 1; c < static_cast<int>(gridDim.x) && p.split_at[c].x == ie.item; ++c) {
          if (!part_live(c)) continue;
          ok = ok && flag_wait(p.ws_flag + c * 2 + t, p.token, wc, kErrWaitPartial);
          if (!ok) break;
          const float2 ml = part_ml(c);
          if (ml.y > 0.f) {
            const float mn = fmaxf(mf, ml.x);
            lf = (mf == -INFINITY ? 0.f : lf * ex2_approx(mf - mn)) + ml.y * ex2_approx(ml.x - mn);
            mf = mn;
          }
        }
        // each thread waited on its own: the warp agrees before the
        // warp-collective TMEM loads that ok guards
        ok = __all_sync(0xffffffffu, ok);
      }
      float a_own = (m == -INFINITY) ? 0.f : ex2_approx(m - mf);  // 1 unless merged
      float inv = part_out ? 1.f : ((lf > 0.f) ? 1.f / lf : 0.f);
      if (ok && live_row && p.lse != nullptr && !part_out && !half_out && !half_merge)
        p.lse[static_cast<size_t>(tbh) * p.Nq + grow] =
            ((lf > 0.f) ? mf + log2f(lf) : -INFINITY) * 0.69314718055994530942f;
      const int qbuf = nfin % QB;  // this item's Q buffer (the MMA warp counts items the same way)
      // O final: also a signal wait (given after an abort too); it covers the
      // item's last P V done, which no block of the item waits for
      ok = mbar_wait_signal(bOfinal(t), nfin & 1, wc, kErrWaitOFinal) && ok;
      nfin++;
      // kPairHalves: tile 0's (m, l) go through shared memory, its final O is
      // read by tile 1 straight from TMEM (same lanes: same rows)
      float2 *half_ml = reinterpret_cast<float2 *>(smem + C::kOffMerge);
      float a_half = 0.f;  // weight of tile 0's half in tile 1's merge
      if (half_out) {
        half_ml[row] = make_float2(m, l);
        tc_fence_before();
        named_bar_arrive(kBarHalfReady, kBarHalvesThreads);
        named_bar_sync(kBarHalfRead, kBarHalvesThreads);  // tile 1 has read O_0: it may be overwritten
      }
      if (half_merge) {
        named_bar_sync(kBarHalfReady, kBarHalvesThreads);
        tc_fence_after();
        const float2 h = half_ml[row];
        mf = fmaxf(m, h.x);
        a_own = (m == -INFINITY) ? 0.f : ex2_approx(m - mf);
        a_half = (h.x == -INFINITY) ? 0.f : ex2_approx(h.x - mf);
        lf = l * a_own + h.y * a_half;
        inv = (lf > 0.f) ? 1.f / lf : 0.f;
        if (ok && live_row && p.lse != nullptr)
          p.lse[static_cast<size_t>(tbh) * p.Nq + grow] =
              ((lf > 0.f) ? mf + log2f(lf) : -INFINITY) * 0.69314718055994530942f;
      }
      const uint32_t ocol_half = tmem + lane_off + C::kColO0;  // O of tile 0
      auto half_read_done = [&]() {
        if (half_merge) {
          tc_fence_before();
          named_bar_arrive(kBarHalfRead, kBarHalvesThreads);
        }
      };
      // 32 columns of this row's output before the 1/l: O_t from TMEM, plus
      // the other pieces' partials when merging
      auto out_chunk = [&](int cc, float (&v)[32]) {
        uint32_t r[32];
        tmem_ld32(ocol + cc * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if (half_merge) {
          uint32_t r0[32];
          tmem_ld32(ocol_half + cc * 32, r0);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = fmaf(__uint_as_float(r0[i]), a_half, v[i] * a_own);
        }
        if (merge_in) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= a_own;
          for (int c = blockIdx.x + 1; c < static_cast<int>(gridDim.x) && p.split_at[c].x == ie.item; ++c) {
            if (!part_live(c)) continue;
            const float2 ml = part_ml(c);
            if (!(ml.y > 0.f)) continue;
            const float sp = ex2_approx(ml.x - mf);
            const float *src = p.ws_o + ((static_cast<size_t>(c) * 2 + t) * D + cc * 32) * kBM + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = fmaf(__ldcg(src + i * kBM), sp, v[i]);
          }
        }
      };
      if (half_out) {
        if constexpr (C::kStoreOViaSmem) o_pending = qbuf;  // no store read the Q buffer
      } else if (part_out) {
        // partial O (not normalised) and (m, l) of each row, then the flag:
        // the barrier orders every thread's writes before the one release
        if (ok) {
          tc_fence_after();
          float *dst = p.ws_o + (static_cast<size_t>(blockIdx.x) * 2 + t) * D * kBM + row;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            float v[32];
            out_chunk(cc, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) __stcg(dst + (cc * 32 + i) * kBM, v[i]);
          }
          __stcg(p.ws_ml + (static_cast<size_t>(blockIdx.x) * 2 + t) * kBM + row, make_float2(m, l));
        }
        named_bar_sync(kBarOStaged + t, 128);
        if (ok && quad == 0 && lane == 0) st_release_gpu(p.ws_flag + blockIdx.x * 2 + t, p.token);
        __syncwarp();
        if constexpr (C::kStoreOViaSmem) o_pending = qbuf;  // no store read the Q buffer
      } else if constexpr (C::kStoreOViaSmem) {
        // Each thread writes its row into the Q buffer in the 128-byte
        // swizzled layout of the O tensor map (16-byte chunk c of row r at
        // chunk c ^ (r % 8): no bank conflicts); one TMA store then writes
        // the tile, rows past Nq clipped by the map.  The buffer is free: the
        // tile's last Q K^T completed before its S was seen.
        const uint32_t stage = sQ + (t * QB + qbuf) * C::kQBytes;
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            float v[32];
            out_chunk(cc, v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t chunk = static_cast<uint32_t>(cc * 4 + q) ^ static_cast<uint32_t>(row & 7);
              st_shared_v4(stage + row * 128 + chunk * 16, pack2<BF16>(v[q * 8 + 0] * inv, v[q * 8 + 1] * inv),
                           pack2<BF16>(v[q * 8 + 2] * inv, v[q * 8 + 3] * inv),
                           pack2<BF16>(v[q * 8 + 4] * inv, v[q * 8 + 5] * inv),
                           pack2<BF16>(v[q * 8 + 6] * inv, v[q * 8 + 7] * inv));
            }
          }
          fence_proxy_async_smem();  // the rows are visible to the TMA store
        }
        half_read_done();
        named_bar_sync(kBarOStaged + t, 128);
        if (ok && quad == 0 && lane == 0) {
          tma_store_3d(&p.tmO, stage, 0, trow0, tbh);
          tma_store_commit();
        }
        __syncwarp();
        o_pending = qbuf;
      } else {
        if (ok) {
          tc_fence_after();
          uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) +
                          (static_cast<size_t>(tbh) * p.Nq + (live_row ? grow : 0)) * (D * 2);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            float v[32];
            out_chunk(cc, v);
            if (live_row) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = pack2<BF16>(v[q * 8 + 0] * inv, v[q * 8 + 1] * inv);
                w.y = pack2<BF16>(v[q * 8 + 2] * inv, v[q * 8 + 3] * inv);
                w.z = pack2<BF16>(v[q * 8 + 4] * inv, v[q * 8 + 5] * inv);
                w.w = pack2<BF16>(v[q * 8 + 6] * inv, v[q * 8 + 7] * inv);
                *reinterpret_cast<uint4 *>(orow + cc * 64 + q * 16) = w;
              }
            }
          }
        }
        half_read_done();
      }
      if constexpr (kSplit) {
        if (merge_in) {
          // Every thread of the warpgroup is past its flag waits (and no
          // piece writes its flag twice in a launch): clear the flags read,
          // so that the next launch on this workspace, a CUDA graph replay
          // under the same token included, waits for fresh partials.
          named_bar_sync(kBarOStaged + t, 128);
          if (quad == 0 && lane == 0)
            for (int c = blockIdx.x + 1; c < static_cast<int>(gridDim.x) && p.split_at[c].x == ie.item; ++c)
              if (part_live(c)) st_relaxed_gpu(p.ws_flag + c * 2 + t, 0u);
          __syncwarp();
        }
      }
      // The next item's first P V (accumulate = 0) overwrites O_t; it is
      // issued only after the next P barrier, which these warps reach after
      // this read has completed (tcgen05.ld waits for its data).
      tc_fence_before();
    }
    // the last O tile store has read its staging buffer before the CTA
    // leaves (its global writes complete with the grid)
    if (C::kStoreOViaSmem && o_pending >= 0) release_staging();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn

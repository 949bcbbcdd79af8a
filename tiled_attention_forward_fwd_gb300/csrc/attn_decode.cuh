// attn_decode.cuh -- split-KV attention for decode and small query counts.
//
// The cruxr.ai "FlashDecoding" section: with few query rows there are too
// few query tiles to occupy the GPU, so the keys are split into chunks that
// are processed in parallel; each chunk yields, per query row, a partial
// maximum, sum and softmax-weighted sum of V rows, and a second step merges
// the chunks by rescaling each one with exp(m_p - m) * l_p and normalising by
// the total.
//
// GB300 mapping.  Kernel 1, grid (chunks, B*Hkv), sized by the host to one
// wave of resident CTAs: one CTA takes the g*Nq query rows of one GQA group
// (all query heads that read the same K/V head, up to 32 rows; they share
// every K/V tile) and one chunk of keys.  A producer warp streams K/V tiles of
// 64 keys by TMA into a 3-stage ring (128B-swizzled boxes of 64 rows x 64
// columns) while the query rows are staged; K and V of a stage have their own
// full / empty barriers, so K of tile i+3 is requested as soon as every warp
// has finished Q K^T of tile i.  Each of the 4 consumer warps takes 16 keys
// of every tile and keeps its own running max, sum and O for all rows,
// computed with warp-level tensor-core MMAs (m16n8k16, fp32 accumulation; the
// work is bandwidth-bound, so the legacy MMA is enough); fragments come from
// ldmatrix (transposed for V), and O is rescaled only when a row's max grew
// by more than 2^8.  At the end the 4 warps are merged in shared memory and
// the chunk's normalised O and its log2-domain log-sum-exp go to the
// caller's workspace.  When the merge is small (rows x chunks x d of a group
// at most kDecFusedMerge floats), the last CTA of a group to finish merges
// the group's chunks itself: every CTA counts its arrival on the group's
// tagged counter after writing its partial, and the one that completes the
// count (whichever chunk it holds) merges and clears the counter for the next
// launch, so nothing waits and a CUDA graph can replay the launch.  Otherwise
// kernel 2,
// launched as a programmatic dependent so that its launch overlaps kernel 1,
// merges the chunks of every row (one CTA per row) and writes O (16-bit) and
// LSE.
//
// Paged K/V (kPaged).  The motivation page's "PagedAttention es un problema
// distinto" section: the cache is a pool of fixed-size pages (for example 16
// tokens), each request has a table of the pages that hold its tokens in
// order, and the attention kernel follows that table instead of reading a
// flat K and V.  Here the pool is laid out (num_pages, Hkv, page_size, d), so
// one (page, head) is one contiguous TMA box; a 64-key tile is 64 / page_size
// boxes (or a 64-row part of one page), placed back to back in shared memory,
// where they form the same 128B-swizzled tile as one 64-row box.  The
// producer reads the next tile's page indices while the current tile's copies
// go out.  Each request has its own length (read on the device); slots past
// it in the last page hold whatever the pool held, so their V rows are
// zeroed in shared memory before P V (their P is 0, but 0 x NaN is not).
#pragma once

#include <stddef.h>

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kDecKeys = 64;     // keys per K/V tile
constexpr int kDecWarps = 4;     // consumer warps: each owns 16 keys of every tile
constexpr int kDecThreads = 32 * kDecWarps + 32;  // + one TMA producer warp
constexpr int kDecMaxRows = 32;  // query rows of one group handled by one CTA
constexpr int kDecMaxChunks = 1024;  // key chunks per group (bounds the merge kernel's shared memory)
constexpr int kDecFusedMerge = 8192;  // rows x chunks x d of a group merged by the split kernel itself

enum DecodeError : int { kErrDecWaitKV = 0x201, kErrDecBadIndex = kErrDeviceArg };

struct DecParams {
  // flat: (d, Nk, B*Hkv), box 64 x 64 x 1; paged: (d, page_size,
  // num_pages*Hkv), box 64 x min(page_size, 64) x 1; 128B swizzle
  CUtensorMap tmK;
  CUtensorMap tmV;
  const void *Q;    // (B, Hq, Nq, d), 16-bit
  float *ws;        // [B*Hq*Nq][nchunks][d]: normalised O of each chunk
  float *ws_lse;    // [B*Hq*Nq][nchunks]: log2 LSE of each chunk (-inf: no live key)
  // fused merge (fused != 0): one tagged arrival counter per group
  // [B*Hkv] (tag = `token`, see arrive_tagged); O and LSE written by the
  // group's last CTA to arrive
  int fused;
  unsigned token;
  unsigned long long *counters;
  void *O;
  float *lse;
  int *status;
  int B, Hq, Hkv, Nq, Nk, group, R;  // R = group * Nq query rows per CTA
  int causal, window;
  int nchunks, chunk_keys;
  int kv_lo, kv_hi;  // keys any row of a group can see
  float scale_log2;  // sm_scale * log2(e) (int8 K/V: times the key scale)
  float v_scale;     // int8 K/V: the value scale, applied to each chunk's O (1 otherwise)
  unsigned long long timeout_ns;
  int stall_after;  // test hook: the producer stops after this many K/V tiles (-1: never)
  // paged K/V: token t of request b sits in page block_table[b * max_pages +
  // t / page_size], slot t % page_size; request b holds seq_lens[b] tokens
  // (1..Nk, at least Nq when causal); kv_lo and kv_hi are not used
  const int *block_table;
  const int *seq_lens;
  int page_shift;  // log2(page_size), 3..8
  int max_pages, num_pages;
};

// Ring depth and resident CTAs per SM for (d, row blocks).  Tiles arrive
// about 3 us after they are requested when HBM is busy, so the ring holds as
// many as shared memory allows: 3 stages x 2 CTAs at d = 128 with up to 16
// rows; 6 stages x 1 CTA for 32 rows at d = 128 (whose per-thread O state
// does not fit two CTAs' registers without spilling); 6 stages x 2 CTAs at
// d = 64.
// int8 K/V (kQuant): the ring holds tiles of half the bytes, 4 stages (7 at
// d = 128 with 32 rows, 6 at d = 64), and each warp widens its 16 rows of
// the current K and V tile into a 16-bit staging tile (same layout as a
// 16-bit ring tile), so the rest of the kernel is unchanged.
template <int D, int RB, bool kQuant = false>
struct DecCfg {
  static constexpr int kStages = kQuant ? (D == 64 ? 6 : (RB == 2 ? 7 : 4)) : ((D == 128 && RB == 1) ? 3 : 6);
  static constexpr int kMinCtas = (D == 128 && RB == 2) ? 1 : 2;
  static constexpr int kBoxBytes = kDecKeys * 128;          // 64 rows x 128 B
  static constexpr int kTileBytes = kDecKeys * D * 2;       // one 16-bit K or V tile
  static constexpr int kRingTileBytes = kQuant ? kDecKeys * D : kTileBytes;  // one K or V tile as loaded
  static constexpr int kQBoxBytes = kDecMaxRows * 128;      // 32 rows x 128 B
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = ((kDecMaxRows * D * 2 + 1023) / 1024) * 1024;
  static constexpr int kStageBytes = 2 * kRingTileBytes;    // K then V
  static constexpr int kOffWide = kOffKV + kStages * kStageBytes;  // kQuant: 16-bit K then V staging
  static constexpr int kWideBytes = kQuant ? 2 * kTileBytes : 0;
  // kfull, vfull, kempty, vempty [stages]; abort flag; the group counter as first read
  static constexpr int kOffBar = kOffWide + kWideBytes;
  static constexpr int kOffStats = kOffBar + 256;           // float wm[4][32], wl[4][32], rinv[32]
  static constexpr int kSmemBytes = kOffStats + (2 * kDecWarps + 1) * kDecMaxRows * 4 + 1024;
  static constexpr int kSlabStride = D + 8;                 // floats per merge-slab row (2-way bank conflicts)
  static_assert(kDecWarps * kDecMaxRows * kSlabStride * 4 <= kStages * kStageBytes + kWideBytes,
                "O merge slabs fit in the ring"); 
  static_assert(4 * kStages * 8 + 16 <= 256, "barriers fit");
  static_assert(kMinCtas * (kSmemBytes + 1024) <= 233472, "shared memory per SM");
};

// Byte offset of element (row r, column c) in a stack of 64-column boxes of
// `rows` rows with the 128-byte swizzle (16-byte chunk index ^ row % 8).
__device__ __forceinline__ uint32_t swz(int rows, int r, int c) {
  return static_cast<uint32_t>((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// Four int8 values (a 32-bit word, lowest byte first) widened exactly to two
// packed pairs of 16-bit floats (lower index in the low half).  fp16: the
// byte, offset to unsigned, becomes the low mantissa bits of 1024 + u (an
// fp16 with exponent 10), and 1152 = 1024 + 128 is subtracted; bf16: the same
// with an fp32 of exponent 23 (2^23 + u, minus 2^23 + 128), then rounded to
// bf16, which is exact for |x| <= 127.  Both are exact integer arithmetic.
template <bool BF16>
__device__ __forceinline__ void widen_s8x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t x = w ^ 0x80808080u;
  if constexpr (!BF16) {
    const __half2 bias = __float2half2_rn(1152.f);
    uint32_t a = __byte_perm(x, 0x64646464u, 0x4140), b = __byte_perm(x, 0x64646464u, 0x4342);
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias), hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
  } else {
    const float f0 = __uint_as_float(__byte_perm(x, 0x4B00u, 0x5440)) - 8388736.f;
    const float f1 = __uint_as_float(__byte_perm(x, 0x4B00u, 0x5441)) - 8388736.f;
    const float f2 = __uint_as_float(__byte_perm(x, 0x4B00u, 0x5442)) - 8388736.f;
    const float f3 = __uint_as_float(__byte_perm(x, 0x4B00u, 0x5443)) - 8388736.f;
    lo = pack2<true>(f0, f1);
    hi = pack2<true>(f2, f3);
  }
}

// This warp's 16 rows of an int8 tile (64 rows x D bytes, row-major, as the
// copy left it) widened into the 16-bit staging tile, in the layout of a
// 64-row box stack with the 128-byte swizzle.
template <int D, bool BF16>
__device__ __forceinline__ void widen_rows(uint32_t src, uint32_t dst, int warp, int lane) {
  constexpr int kChunks = D / 16;  // 16-byte pieces of an int8 row
#pragma unroll
  for (int idx = lane; idx < 16 * kChunks; idx += 32) {
    const int r = warp * 16 + idx / kChunks, c = (idx % kChunks) * 16;
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(src + r * D + c));
    uint32_t o[8];
    widen_s8x4<BF16>(w0, o[0], o[1]);
    widen_s8x4<BF16>(w1, o[2], o[3]);
    widen_s8x4<BF16>(w2, o[4], o[5]);
    widen_s8x4<BF16>(w3, o[6], o[7]);
    st_shared_v4(dst + swz(kDecKeys, r, c), o[0], o[1], o[2], o[3]);
    st_shared_v4(dst + swz(kDecKeys, r, c + 8), o[4], o[5], o[6], o[7]);
  }
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

// Bounded wait that ignores the abort flag: used only to drain our own
// copies, which always complete.
__device__ __forceinline__ void mbar_drain_dec(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 1000000000ull) break;
}

// Partial attention of one GQA group over one key chunk.  RB = row blocks of
// 16 (1: up to 16 rows, 2: up to 32); kPaged: K and V come from a page pool.
template <int D, bool BF16, int RB, bool kPaged, bool kQuant = false>
__global__ void __launch_bounds__(kDecThreads, DecCfg<D, RB, kQuant>::kMinCtas)
    attn_decode_kernel(const __grid_constant__ DecParams p) {
  static_assert(!(kPaged && kQuant), "int8 K/V is served from a flat cache");
  using C = DecCfg<D, RB, kQuant>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  int *abort_flag = reinterpret_cast<int *>(bars + 4 * NS);
  unsigned long long *ctr_seen = reinterpret_cast<unsigned long long *>(bars + 4 * NS + 1);
  float *wm = reinterpret_cast<float *>(smem + C::kOffStats);  // [warp][row] running max (log2 domain)
  float *wl = wm + kDecWarps * kDecMaxRows;                    // [warp][row] running sum
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sKV = smem_u32(smem + C::kOffKV);
  const uint32_t bar0 = smem_u32(bars);
  auto bKfull = [&](int s) { return bar0 + 8u * s; };
  auto bVfull = [&](int s) { return bar0 + 8u * (NS + s); };
  auto bKempty = [&](int s) { return bar0 + 8u * (2 * NS + s); };
  auto bVempty = [&](int s) { return bar0 + 8u * (3 * NS + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int chunk = blockIdx.x;
  const int bk = blockIdx.y;  // b * Hkv + kvh
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  WaitCtl wc{abort_flag, p.status, p.timeout_ns};

  // Let the merge kernel launch now; it waits for this grid to finish
  // before it reads anything.
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(bKfull(s), 1);
      mbar_init(bVfull(s), 1);
      mbar_init(bKempty(s), kDecWarps);
      mbar_init(bVempty(s), kDecWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // inputs may come from the previous kernel on the stream
  // the fused merge's group counter, read now (its latency hides behind the
  // keys) by the producer warp
  if (p.fused && threadIdx.x == 32 * kDecWarps) *ctr_seen = ld_relaxed_gpu_u64(p.counters + bk);
  bool ok = true;
  // keys of this request, and the ones this chunk takes
  int nk = p.kv_hi, kv_lo = p.kv_lo;
  if constexpr (kPaged) {
    int len = __ldcg(p.seq_lens + b);
    if (len < (p.causal ? p.Nq : 1) || len > p.Nk) {
      if (threadIdx.x == 0) atomicCAS(p.status, 0, kErrDecBadIndex);
      len = min(max(len, 0), p.Nk);
    }
    nk = len;
    // the first key any row of the group can see, rounded down to a tile
    // boundary so that every tile starts on a page boundary (keys below the
    // window are masked per key)
    kv_lo = (p.causal && p.window > 0) ? max(0, nk - p.Nq - p.window + 1) & ~(kDecKeys - 1) : 0;
  }
  const int k0 = max(chunk * p.chunk_keys, kv_lo);
  const int k1 = min((chunk + 1) * p.chunk_keys, nk);
  const int ntiles = (k1 > k0) ? (k1 - k0 + kDecKeys - 1) / kDecKeys : 0;

  if (warp == kDecWarps) {
    // ======================================================== TMA producer
    // K of tile i goes out as soon as every consumer warp has finished Q K^T
    // of tile i - NS, V as soon as they have finished P V of it.
    if (elect_one()) {
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
    }
    __syncwarp();
    // Paged: lane j < npg reads the pool slab (page * Hkv + kvh) of the j-th
    // page of a tile.  A page past the request's end, or an index outside
    // the pool (recorded as an error), becomes the first slab past the pool,
    // which the copy reads as zeros.
    constexpr int kMaxTilePages = kDecKeys / 8;  // page_size >= 8
    const int pshift = kPaged ? p.page_shift : 0;
    const int npg = (kPaged && pshift < 6) ? (kDecKeys >> pshift) : 1;
    const int req_pages = kPaged ? ((nk + (1 << pshift) - 1) >> pshift) : 0;
    const int past_pool = kPaged ? p.num_pages * p.Hkv : 0;
    auto tile_page = [&](int i) { return ((k0 + i * kDecKeys) >> pshift) + lane; };
    auto read_page = [&](int i) {
      const int lp = tile_page(i);
      return (lane < npg && lp < req_pages) ? __ldcg(p.block_table + static_cast<size_t>(b) * p.max_pages + lp) : 0;
    };
    int page_next = (kPaged && ntiles > 0) ? read_page(0) : 0;
    int kiss = 0, viss = 0;  // K / V tiles issued
    for (int i = 0; i < ntiles; ++i) {
      if (p.stall_after >= 0 && i >= p.stall_after) {  // test hook: stop loading
        ok = false;
        break;
      }
      const int s = i % NS, y = k0 + i * kDecKeys;
      const uint32_t kdst = sKV + s * C::kStageBytes, vdst = kdst + C::kRingTileBytes;
      int slab[kMaxTilePages];
      if constexpr (kPaged) {
        const int page = page_next;
        if (i + 1 < ntiles) page_next = read_page(i + 1);  // in flight during this tile's waits
        int z = past_pool;
        if (lane < npg && tile_page(i) < req_pages) {
          if (page >= 0 && page < p.num_pages)
            z = page * p.Hkv + kvh;
          else
            atomicCAS(p.status, 0, kErrDecBadIndex);
        }
#pragma unroll
        for (int j = 0; j < kMaxTilePages; ++j) slab[j] = __shfl_sync(0xffffffffu, z, j);
      }
      // one K or V tile into dst: a 64-row box per 64 columns (flat), or per
      // page and 64 columns (paged)
      auto load_tile = [&](uint32_t dst, const CUtensorMap *tm, uint32_t bar) {
        if constexpr (kQuant) {
          tma_load_3d(dst, tm, bar, 0, y, bk);  // int8: one box of 64 rows x D bytes
        } else if constexpr (!kPaged) {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) tma_load_3d(dst + cc * C::kBoxBytes, tm, bar, cc * 64, y, bk);
        } else if (pshift >= 6) {
          const int row = y & ((1 << pshift) - 1);  // a multiple of 64
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) tma_load_3d(dst + cc * C::kBoxBytes, tm, bar, cc * 64, row, slab[0]);
        } else {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc)
#pragma unroll
            for (int j = 0; j < kMaxTilePages; ++j)
              if (j < npg) tma_load_3d(dst + cc * C::kBoxBytes + (j << pshift) * 128, tm, bar, cc * 64, 0, slab[j]);
        }
      };
      if (i >= NS && !mbar_wait_warp(bKempty(s), ((i / NS) - 1) & 1, wc, kErrDecWaitKV)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(bKfull(s), C::kRingTileBytes);
        load_tile(kdst, &p.tmK, bKfull(s));
      }
      __syncwarp();
      kiss = i + 1;
      if (i >= NS && !mbar_wait_warp(bVempty(s), ((i / NS) - 1) & 1, wc, kErrDecWaitKV)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        mbar_arrive_expect_tx(bVfull(s), C::kRingTileBytes);
        load_tile(vdst, &p.tmV, bVfull(s));
      }
      __syncwarp();
      viss = i + 1;
    }
    if (!ok && lane == 0) {
      // Never leave with one of our copies in flight: wait (bounded) for the
      // last loads issued into each stage.
      for (int i = max(0, kiss - NS); i < kiss; ++i) mbar_drain_dec(bKfull(i % NS), (i / NS) & 1);
      for (int i = max(0, viss - NS); i < viss; ++i) mbar_drain_dec(bVfull(i % NS), (i / NS) & 1);
    }
  } else {
    // ======================================================== consumer warps
    // the group's query rows -> shared memory (swizzled like a 32-row box); rows >= R are zero
    for (int idx = threadIdx.x; idx < kDecMaxRows * (D / 8); idx += 32 * kDecWarps) {
      const int r = idx / (D / 8), c8 = (idx % (D / 8)) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < p.R) {
        const int head = kvh * p.group + r / p.Nq, i = r % p.Nq;
        v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.Q) +
                                             ((static_cast<size_t>(b) * p.Hq + head) * p.Nq + i) * D + c8);
      }
      *reinterpret_cast<uint4 *>(smem + C::kOffQ + swz(kDecMaxRows, r, c8)) = v;
    }
    named_bar_and(1, 32 * kDecWarps, true);  // Q staged (consumer warps only)
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
      pos[rb][h] = nk - p.Nq + (r % p.Nq);
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[rb][n][0] = o[rb][n][1] = o[rb][n][2] = o[rb][n][3] = 0.f;
  }
  const float sl2 = p.scale_log2;

  for (int i = 0; warp < kDecWarps && i < ntiles; ++i) {
    const int s = i % NS;
    if (!mbar_wait_warp(bKfull(s), (i / NS) & 1, wc, kErrDecWaitKV)) {
      ok = false;
      break;
    }
    uint32_t sK = sKV + s * C::kStageBytes, sV = sK + C::kRingTileBytes;
    if constexpr (kQuant) {
      // widen this warp's rows of the int8 K tile, then hand the stage back
      const uint32_t wide = smem_u32(smem + C::kOffWide);
      __syncwarp();  // this warp's reads of the previous tile's staging are done
      widen_rows<D, BF16>(sK, wide, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bKempty(s));
      sK = wide;
    }
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
    __syncwarp();
    if (!kQuant && lane == 0) mbar_arrive(bKempty(s));  // this warp is done with K of tile i
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
        // Lazy rescale: the reference max moves only when it grew by more
        // than 2^8 for some row of this warp, so O is rarely rescaled.
        const float m_new = fmaxf(m[rb][h], tmax * sl2);
        if (__any_sync(0xffffffffu, m_new > m[rb][h] + 8.0f)) {
          const float alpha = (m[rb][h] == -INFINITY) ? 0.f : ex2_approx(m[rb][h] - m_new);
          l[rb][h] *= alpha;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            o[rb][n][2 * h] *= alpha;
            o[rb][n][2 * h + 1] *= alpha;
          }
          m[rb][h] = m_new;
        }
        const float mref = (m[rb][h] == -INFINITY) ? 0.f : m[rb][h];
        float e4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) e4[q] = ex2_approx(fmaf(v[q], sl2, -mref));
        l[rb][h] += (e4[0] + e4[1]) + (e4[2] + e4[3]);
        // A fragment of P: a0/a2 hold row g (keys 2t, 8+2t), a1/a3 row g+8
        pa[rb][h] = pack2<BF16>(e4[0], e4[1]);
        pa[rb][2 + h] = pack2<BF16>(e4[2], e4[3]);
      }
    }
    // ---- O += P V
    if (!mbar_wait_warp(bVfull(s), (i / NS) & 1, wc, kErrDecWaitKV)) {
      ok = false;
      break;
    }
    if constexpr (kQuant) {
      const uint32_t wide = smem_u32(smem + C::kOffWide) + C::kTileBytes;
      widen_rows<D, BF16>(sV, wide, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bVempty(s));
      sV = wide;
    }
    if (kPaged && key_base + 16 > nk) {
      // this warp's V rows past the request's end: zero them (16-byte
      // pieces; a whole 128-byte row of a box is swizzle-free), then order
      // these writes before the next copy into the stage
      for (int idx = lane; idx < 16 * (D / 64) * 8; idx += 32) {
        const int r = idx / ((D / 64) * 8), cc = (idx / 8) % (D / 64), piece = idx % 8;
        if (key_base + r >= nk)
          st_shared_v4(sV + cc * C::kBoxBytes + (warp * 16 + r) * 128 + piece * 16, 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
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
    __syncwarp();
    if (!kQuant && lane == 0) mbar_arrive(bVempty(s));  // this warp is done with V of tile i
  }
  // Every thread learns whether any role gave up; then nothing is in flight
  // (the producer drained its copies above).  A CTA that gave up writes no
  // partial, but still counts its arrival in a fused merge (below), so that
  // the group's counter is cleared at the end of the launch as always.
  const bool failed = __syncthreads_or(!ok);
  if (failed && !p.fused) return;
  // O slabs, one per warp ([warp][32][kSlabStride]; the ring is idle now)
  float *oacc = reinterpret_cast<float *>(smem + C::kOffKV);
  if (!failed) {
    // ---- merge the 4 warps: row sums over the quad, then max / sums per row in shared memory
    const bool consumer = warp < kDecWarps;
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l[rb][h] += __shfl_xor_sync(0xffffffffu, l[rb][h], 1);
        l[rb][h] += __shfl_xor_sync(0xffffffffu, l[rb][h], 2);
        if (consumer && tq == 0) {
          const int r = rb * 16 + g + 8 * h;
          wm[warp * kDecMaxRows + r] = m[rb][h];
          wl[warp * kDecMaxRows + r] = l[rb][h];
        }
      }
    // each warp's O into its slab, summed in a fixed order below (deterministic result)
    float *rinv = wl + kDecWarps * kDecMaxRows;  // [row] 1 / (chunk sum)
    __syncthreads();
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!consumer) continue;
        const int r = rb * 16 + g + 8 * h;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecMaxRows + r]);
        const float scale = (m[rb][h] == -INFINITY) ? 0.f : ex2_approx(m[rb][h] - M);
        float *slab = oacc + (warp * kDecMaxRows + r) * C::kSlabStride;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
          *reinterpret_cast<float2 *>(slab + n * 8 + 2 * tq) =
              make_float2(o[rb][n][2 * h] * scale, o[rb][n][2 * h + 1] * scale);
      }
    // per-row totals, once per row: the chunk's log2 LSE and 1 / sum
    if (threadIdx.x < p.R) {
      const int r = threadIdx.x;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecMaxRows + r]);
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = wm[w * kDecMaxRows + r];
        if (mw != -INFINITY) L += ex2_approx(mw - M) * wl[w * kDecMaxRows + r];
      }
      rinv[r] = (L > 0.f) ? 1.f / L : 0.f;
      const int head = kvh * p.group + r / p.Nq, qi = r % p.Nq;
      const size_t grow = (static_cast<size_t>(b) * p.Hq + head) * p.Nq + qi;
      p.ws_lse[grow * p.nchunks + chunk] = (L > 0.f) ? M + log2f(L) : -INFINITY;
    }
    __syncthreads();
    // ---- this chunk's normalised O -> workspace, four columns per thread
    for (int idx = threadIdx.x; idx < p.R * (D / 4); idx += kDecThreads) {
      const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
      float4 acc = *reinterpret_cast<const float4 *>(oacc + r * C::kSlabStride + c);
#pragma unroll
      for (int w = 1; w < kDecWarps; ++w) {
        const float4 v = *reinterpret_cast<const float4 *>(oacc + (w * kDecMaxRows + r) * C::kSlabStride + c);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const float inv = rinv[r] * p.v_scale;
      const int head = kvh * p.group + r / p.Nq, qi = r % p.Nq;
      const size_t grow = (static_cast<size_t>(b) * p.Hq + head) * p.Nq + qi;
      *reinterpret_cast<float4 *>(p.ws + (grow * p.nchunks + chunk) * D + c) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
  if (!p.fused) return;
  // ---- fused merge: the group's last CTA to arrive merges (no waiting)
  __syncthreads();  // every thread's partial is written before the one arrival
  bool last = false;
  if (threadIdx.x == 0) {
    unsigned long long *ctr = p.counters + bk;
    last = arrive_tagged(ctr, *ctr_seen, p.token, static_cast<unsigned>(p.nchunks));
    if (last) reset_tagged(ctr, p.token);  // every chunk has arrived: ready for the next launch
  }
  // the last arriver's thread 0 acquired every chunk's partial; the barrier
  // orders its threads' reads (L2, __ldcg) after that
  if (!__syncthreads_or(last) || failed) return;
  // per row: the chunk weights 2^(lse_c - M) and 1 / their sum (shared
  // memory: the ring is idle)
  float *linv = oacc;               // [R]
  float *wts = oacc + kDecMaxRows;  // [R][nchunks]
  if (threadIdx.x < p.R) {
    const int r = threadIdx.x;
    const int head = kvh * p.group + r / p.Nq, qi = r % p.Nq;
    const size_t grow = (static_cast<size_t>(b) * p.Hq + head) * p.Nq + qi;
    const float *lr = p.ws_lse + grow * p.nchunks;
    float M = -INFINITY;
    for (int c = 0; c < p.nchunks; ++c) M = fmaxf(M, __ldcg(lr + c));
    float L = 0.f;
    for (int c = 0; c < p.nchunks; ++c) {
      const float lc = __ldcg(lr + c);
      const float w = (lc == -INFINITY) ? 0.f : ex2_approx(lc - M);
      wts[r * p.nchunks + c] = w;
      L += w;
    }
    linv[r] = (L > 0.f) ? 1.f / L : 0.f;
    if (p.lse != nullptr) p.lse[grow] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < p.R * (D / 4); idx += kDecThreads) {
    const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
    const int head = kvh * p.group + r / p.Nq, qi = r % p.Nq;
    const size_t grow = (static_cast<size_t>(b) * p.Hq + head) * p.Nq + qi;
    const float4 *src = reinterpret_cast<const float4 *>(p.ws + grow * p.nchunks * D + c4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < p.nchunks; ++c) {
      const float w = wts[r * p.nchunks + c];
      const float4 v = __ldcg(src + static_cast<size_t>(c) * (D / 4));
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = linv[r];
    uint2 out;
    out.x = pack2<BF16>(acc.x * inv, acc.y * inv);
    out.y = pack2<BF16>(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(p.O) + grow * D + c4) = out;
  }
}

// Merge the chunks of every query row: O = sum_c 2^(lse_c - lse) o_c,
// LSE = lse * ln 2 with lse = log2 sum_c 2^(lse_c).  One CTA of 128 threads
// per row: the chunk weights go to shared memory, then D/4 threads per chunk
// row read four columns each (float4) and the 128 / (D/4) groups of chunks
// are summed in a fixed order.  D is 64 or 128, or 512 for the latent rows
// of attn_mla.cuh (then the 128 threads are one group of four columns each).
template <int D, bool BF16>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const float *ws, const float *ws_lse, void *O,
                                                                  float *lse, int rows, int nchunks) {
  extern __shared__ float wts[];  // [nchunks] weights, then [groups][D] partial sums
  __shared__ float red[4];
  // Launched as a programmatic dependent of the split kernel: wait until it
  // has finished and its writes are visible; the next call may start its
  // prologue meanwhile.
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  if (row >= rows) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float *lrow = ws_lse + static_cast<size_t>(row) * nchunks;
  float M = -INFINITY;
  for (int c = tid; c < nchunks; c += 128) M = fmaxf(M, lrow[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float Ls = 0.f;
  for (int c = tid; c < nchunks; c += 128) {
    const float lc = lrow[c];
    const float w = (lc == -INFINITY) ? 0.f : ex2_approx(lc - M);
    wts[c] = w;
    Ls += w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  if (lane == 0) red[warp] = Ls;
  __syncthreads();
  const float L = (red[0] + red[1]) + (red[2] + red[3]);
  constexpr int kTpr = D / 4;          // threads per chunk row
  constexpr int kGroups = 128 / kTpr;  // chunk groups
  const int grp = tid / kTpr, col = (tid % kTpr) * 4;
  const float *orow = ws + static_cast<size_t>(row) * nchunks * D + col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = grp; c < nchunks; c += kGroups) {
    const float w = wts[c];
    const float4 v = *reinterpret_cast<const float4 *>(orow + static_cast<size_t>(c) * D);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  float *part = wts + ((nchunks + 3) & ~3);  // 16-byte aligned
  *reinterpret_cast<float4 *>(part + grp * D + col) = acc;
  __syncthreads();
  for (int c2 = tid * 2; c2 < D; c2 += 256) {  // two columns per thread and pass (D up to 512)
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      a0 += part[g * D + c2];
      a1 += part[g * D + c2 + 1];
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    reinterpret_cast<uint32_t *>(O)[(static_cast<size_t>(row) * D + c2) / 2] = pack2<BF16>(a0 * inv, a1 * inv);
  }
  if (lse != nullptr && tid == 0) lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
}

}  // namespace attn

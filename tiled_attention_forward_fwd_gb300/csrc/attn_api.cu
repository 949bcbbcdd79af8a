// attn_api.cu -- the C ABI declared in include/attn.h: argument checks,
// TMA tensor maps, kernel selection and launch.  No allocation, no sync
// (except attn_device_status, whose job is to sync).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/attn.h"
#include "attn_decode.cuh"
#include "attn_mla.cuh"
#include "attn_short.cuh"
#include "attn_bwd_sm103.cuh"
#include "attn_fwd_sm103.cuh"

namespace attn {

// An empty kernel, launched like the others (programmatic dependent launch):
// the fixed cost of one launch, for measurements.
__global__ void attn_empty_kernel() {
  pdl_launch_dependents();
  pdl_wait();
}

// Kernel status word (one per device): first error code wins, 0 = fine.
__device__ int g_status;

static std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
static std::atomic<int> g_stall_after{-1};  // attn_set_test_stall

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D view (d, rows, slabs) of a dense (slabs, rows, d) 16-bit tensor, box
// 64 x 128 x 1 with 128-byte swizzle.  Rows past `rows` read as zero and are
// never written by stores.
static bool make_map(CUtensorMap *m, const void *ptr, int d, int rows, long long slabs, bool bf16,
                     int box_rows = 128) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slabs)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 2 * rows};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (d, rows, slabs) of a dense (slabs, rows, d) fp32 tensor, box 32 x
// 128 x 1 with the 128-byte swizzle (the backward's dQ accumulator, written
// by TMA reduce-adds).
static bool make_map_f32(CUtensorMap *m, void *ptr, int d, int rows, long long slabs) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slabs)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(d) * 4 * rows};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (d, rows, slabs) of a dense (slabs, rows, d) int8 tensor, box d x
// 64 x 1 without swizzle (the decode kernel widens rows itself).
static bool make_map_s8(CUtensorMap *m, const void *ptr, int d, int rows, long long slabs) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slabs)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(d) * rows};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream finishes; it waits (griddepcontrol.wait)
// before touching global memory.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
  int B, Hq, Hkv, Nq, Nk, d, causal, window;
  float sm_scale;
  attn_dtype_t dtype;
};

static attn_status_t validate(const void *Q, const void *K, const void *V, const void *O, const float *LSE,
                              const Shape &s) {
  if (!Q || !K || !V || !O) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return ATTN_ERR_INVALID_ARG;
  if (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (s.B <= 0 || s.Hq <= 0 || s.Hkv <= 0 || s.Nq <= 0 || s.Nk <= 0 || s.d <= 0) return ATTN_ERR_INVALID_ARG;
  if (s.Hq % s.Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (s.window < 0 || (s.window > 0 && !s.causal)) return ATTN_ERR_INVALID_ARG;
  if (s.causal && s.Nq > s.Nk) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(s.sm_scale) || !(s.sm_scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (s.dtype != ATTN_DTYPE_FP16 && s.dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (s.d != 64 && s.d != 128) return ATTN_ERR_UNSUPPORTED;
  // work items are counted in 32-bit integers
  if (static_cast<long long>(s.B) * s.Hq * ((s.Nq + kBM - 1) / kBM) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

static int current_device_sm_major(int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return -1;
  if (dev_out) *dev_out = dev;
  return major;
}

static int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// ---------------------------------------------------------------- stream-K split of the prefill
// A d = 128 call whose items (tile pairs) fill less than two waves of CTAs
// gets an even share of K/V tile steps per CTA instead of whole items, when
// the caller passes a workspace and the call has no window (see FwdParams).
static size_t round_up256(size_t x) { return (x + 255) & ~size_t(255); }

static size_t split_ws_bytes(int d, int ctas) {
  const size_t rows = static_cast<size_t>(ctas) * 2 * kBM;
  return round_up256(rows * d * 4) + round_up256(rows * 8) + round_up256(static_cast<size_t>(ctas) * 2 * 4);
}

// Workspace bytes of the split (0: the shape does not take it), for a call
// without a window on a device with `sms` SMs.  Only d = 128: an item cut
// between CTAs costs its pieces a partial write, a flag and a merge on the
// critical path (a few microseconds), which the better balance of the
// heavier d = 128 tile steps repays and that of d = 64 does not.
static size_t split_plan_bytes(const Shape &s, int sms) {
  if (s.window > 0 || sms <= 0 || s.d != 128) return 0;
  const long long zq = static_cast<long long>(s.B) * s.Hq;
  const long long ntiles = (s.Nq + kBM - 1) / kBM;
  const int group = s.Hq / s.Hkv;
  const long long items = (group % 2 == 0) ? (zq / 2) * ntiles : zq * ((ntiles + 1) / 2);
  if (items >= 2LL * sms) return 0;
  return split_ws_bytes(s.d, std::min(sms, kMaxSplitCtas));
}

// Tags of the split paths' cross-CTA handshakes (a fresh one per enqueued
// call; a captured graph replays its own).  The handshake words are cleared
// by the end of every launch, so a replay under the same tag starts from a
// clean state; a tag never matches what other calls left in the memory.
static std::atomic<unsigned> g_split_token{0};

// One-time set-up of a prefill kernel on a device: its shared-memory size,
// and whether it was built with the register count that the warpgroup
// register split (setmaxnreg) is sized for: kThreads x kLaunchRegs
// registers; any other allocation could stall.
template <int D, bool BF16>
static void (*prefill_kernel(int sched, bool paged))(FwdParams) {
  if (paged) return sched == kSchedHalves ? attn_fwd_kernel<D, BF16, kSchedHalves, true>
                                          : attn_fwd_kernel<D, BF16, kSchedPlain, true>;
  return sched == kSchedSplit    ? attn_fwd_kernel<D, BF16, kSchedSplit>
         : sched == kSchedHalves ? attn_fwd_kernel<D, BF16, kSchedHalves>
                                 : attn_fwd_kernel<D, BF16, kSchedPlain>;
}

template <int D, bool BF16>
static bool prefill_kernel_ready(int dev, int sched, bool paged = false) {
  static std::once_flag once[5][64];
  static bool ok[5][64];
  auto kern = prefill_kernel<D, BF16>(sched, paged);
  const int k = paged ? (sched == kSchedHalves ? 4 : 3) : sched;  // one slot per kernel
  std::call_once(once[k][dev], [&] {
    cudaFuncAttributes fa;
    ok[k][dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      FwdCfg<D>::kSmemBytes) == cudaSuccess &&
                 cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs == kLaunchRegs;
    if (!ok[k][dev]) (void)cudaGetLastError();  // not reported by a later launch check
  });
  return ok[k][dev];
}

// The schedule of a prefill call on `sms_now` SMs: item shape, item count
// and divisors in p, the kernel (kSched*) and its grid; with `split`, the
// stream-K split points too.  Host only, no device work.  False when the
// item count overflows.
static bool prefill_schedule(const Shape &s, bool split, int sms_now, FwdParams &p, int &sched, int &grid) {
  const long long zq = static_cast<long long>(s.B) * s.Hq;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.group = s.Hq / s.Hkv;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  // An item holds up to two query tiles: two heads of one GQA group at the
  // same rows when the group size is even (they share every K/V load);
  // otherwise one tile whose K/V tiles the two softmax warpgroups split, when
  // the tiles are few; consecutive row tiles (2r, 2r+1) of one head
  // otherwise.
  const long long ntiles = (s.Nq + kBM - 1) / kBM;
  if (split) {
    // both tiles of every item busy: heads of a group, else row pairs
    p.pair_mode = (p.group % 2 == 0) ? kPairHeads : kPairRows;
    p.n_row_blocks = static_cast<int>(p.pair_mode == kPairHeads ? ntiles : (ntiles + 1) / 2);
  } else if (p.group % 2 == 0) {
    p.pair_mode = kPairHeads;
    p.n_row_blocks = static_cast<int>(ntiles);
  } else if (zq * ntiles <= sms_now || (s.causal && zq * ((ntiles + 1) / 2) <= sms_now)) {
    // Few tiles (one wave of single tiles, or causal pairs that fit one
    // wave): one tile per item.  When the longest tile has at least 4 K/V
    // tiles, the two softmax warpgroups split them, so that no warpgroup
    // idles while a long tile runs; shorter ones do not repay the merge.
    int beg = 0, end = 0;
    tile_range(p, static_cast<int>((ntiles - 1) * kBM), p.Nk, beg, end);
    p.pair_mode = (end - beg >= 4) ? kPairHalves : kPairSingle;
    p.n_row_blocks = static_cast<int>(ntiles);
  } else {
    p.pair_mode = kPairRows;
    p.n_row_blocks = static_cast<int>((ntiles + 1) / 2);
  }
  const long long slots = (p.pair_mode == kPairHeads) ? zq / 2 : zq;
  const long long items = slots * p.n_row_blocks;
  if (items > 0x7fffffffLL) return false;
  p.n_slots = static_cast<int>(slots);
  p.n_items = static_cast<int>(items);
  p.fd_slots = fastdiv_make(static_cast<uint32_t>(p.n_slots));
  p.fd_heads = fastdiv_make(static_cast<uint32_t>(p.pair_mode == kPairHeads ? s.Hq / 2 : s.Hq));
  p.fd_group = fastdiv_make(static_cast<uint32_t>(p.group));
  int split_ctas = 0;
  if (split) {
    // Items in order, each its union range of K/V tile steps; CTA c starts
    // at step c * W / G of the W steps in all.
    long long total = 0;
    std::vector<int> len(static_cast<size_t>(p.n_items));
    for (int i = 0; i < p.n_items; ++i) {
      const Item it = decode_item(p, i);
      len[static_cast<size_t>(i)] = it.uend - it.ubeg;
      total += len[static_cast<size_t>(i)];
    }
    split_ctas = static_cast<int>(std::min<long long>(std::min(sms_now, kMaxSplitCtas), total));
    int item = 0;
    long long before = 0;  // steps in items [0, item)
    for (int c = 0; c < split_ctas; ++c) {
      const long long target = total * c / split_ctas;
      while (item < p.n_items && before + len[static_cast<size_t>(item)] <= target) {
        before += len[static_cast<size_t>(item)];
        ++item;
      }
      p.split_at[c] = make_int2(item, static_cast<int>(target - before));
    }
    p.split_at[split_ctas] = make_int2(p.n_items, 0);
  }
  sched = split ? kSchedSplit : (p.pair_mode == kPairHalves ? kSchedHalves : kSchedPlain);
  grid = split ? split_ctas : static_cast<int>(std::min<long long>(items, sms_now));
  return true;
}

// A paged K/V cache: the page pool and, per request, its page table and length.
struct PagedKV {
  const int *block_table;
  const int *seq_lens;
  int page_size, num_pages, max_pages;
};

static int log2_pow2(int x) {
  int sh = 0;
  while ((1 << sh) < x) ++sh;
  return sh;
}

// The tiled prefill kernel; with `pg`, on a paged K/V cache (K and V are then
// the pools, s.Nk the largest request length, and there is no split).
template <int D, bool BF16>
static attn_status_t launch_prefill(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                   const Shape &s, void *ws, size_t ws_bytes, cudaStream_t stream,
                                   const PagedKV *pg = nullptr) {
  using Cfg = FwdCfg<D>;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long zq = static_cast<long long>(s.B) * s.Hq;
  const long long zk = static_cast<long long>(s.B) * s.Hkv;
  if (!make_map(&p.tmQ, Q, D, s.Nq, zq, BF16) || (Cfg::kStoreOViaSmem && !make_map(&p.tmO, O, D, s.Nq, zq, BF16)))
    return ATTN_ERR_CUDA;
  if (pg == nullptr) {
    if (!make_map(&p.tmK, K, D, s.Nk, zk, BF16) || !make_map(&p.tmV, V, D, s.Nk, zk, BF16)) return ATTN_ERR_CUDA;
  } else {
    const long long slabs = static_cast<long long>(pg->num_pages) * s.Hkv;
    const int box = std::min(pg->page_size, kBN);
    if (!make_map(&p.tmK, K, D, pg->page_size, slabs, BF16, box) ||
        !make_map(&p.tmV, V, D, pg->page_size, slabs, BF16, box))
      return ATTN_ERR_CUDA;
    p.block_table = pg->block_table;
    p.seq_lens = pg->seq_lens;
    p.page_shift = log2_pow2(pg->page_size);
    p.max_pages = pg->max_pages;
    p.num_pages = pg->num_pages;
  }
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  p.O = O;
  p.lse = LSE;
  p.status = status;
  const int sms = device_sm_count();
  const size_t split_bytes = (ws && pg == nullptr) ? split_plan_bytes(s, sms) : 0;
  if (split_bytes > 0 && (ws_bytes < split_bytes || !aligned16(ws))) return ATTN_ERR_INVALID_ARG;
  int sched = kSchedPlain, grid = 0;
  if (!prefill_schedule(s, split_bytes > 0, sms, p, sched, grid)) return ATTN_ERR_INVALID_ARG;
  if (sched == kSchedSplit) {
    const int split_ctas = grid;
    unsigned tok = ++g_split_token;
    if (tok == 0) tok = ++g_split_token;
    p.token = tok;
    const size_t rows = static_cast<size_t>(split_ctas) * 2 * kBM;
    uint8_t *base = static_cast<uint8_t *>(ws);
    p.ws_o = reinterpret_cast<float *>(base);
    p.ws_ml = reinterpret_cast<float2 *>(base + round_up256(rows * D * 4));
    p.ws_flag = reinterpret_cast<unsigned *>(base + round_up256(rows * D * 4) + round_up256(rows * 8));
  }
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * 1.4426950408889634074);
  p.timeout_ns = g_timeout_ns.load();
  p.stall_after = g_stall_after.load();

  auto kern = prefill_kernel<D, BF16>(sched, pg != nullptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  if (!prefill_kernel_ready<D, BF16>(dev, sched, pg != nullptr)) return ATTN_ERR_UNSUPPORTED;
  if (grid <= 0) return ATTN_ERR_CUDA;
  if (launch_pdl(kern, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t dispatch_prefill(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                      const Shape &s, void *ws, size_t ws_bytes, cudaStream_t stream,
                                      const PagedKV *pg = nullptr) {
  const bool bf16 = s.dtype == ATTN_DTYPE_BF16;
  if (s.d == 64) return bf16 ? launch_prefill<64, true>(Q, K, V, O, LSE, s, ws, ws_bytes, stream, pg)
                             : launch_prefill<64, false>(Q, K, V, O, LSE, s, ws, ws_bytes, stream, pg);
  return bf16 ? launch_prefill<128, true>(Q, K, V, O, LSE, s, ws, ws_bytes, stream, pg)
              : launch_prefill<128, false>(Q, K, V, O, LSE, s, ws, ws_bytes, stream, pg);
}

// ---------------------------------------------------------------- backward
static size_t bwd_ws_bytes(long long rows, int d) {
  return round_up256(static_cast<size_t>(rows) * d * 4) + round_up256(static_cast<size_t>(rows) * 4);
}

template <int D, bool BF16>
static attn_status_t launch_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                const float *LSE, void *dQ, void *dK, void *dV, const Shape &s, void *ws,
                                cudaStream_t stream) {
  using Cfg = BwdCfg<D>;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long zq = static_cast<long long>(s.B) * s.Hq, zk = static_cast<long long>(s.B) * s.Hkv;
  if (!make_map(&p.tmQ, Q, D, s.Nq, zq, BF16) || !make_map(&p.tmDO, dO, D, s.Nq, zq, BF16) ||
      !make_map(&p.tmK, K, D, s.Nk, zk, BF16) || !make_map(&p.tmV, V, D, s.Nk, zk, BF16))
    return ATTN_ERR_CUDA;
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  const long long rows = zq * s.Nq;
  uint8_t *base = static_cast<uint8_t *>(ws);
  p.dq_acc = reinterpret_cast<float *>(base);
  if (!make_map_f32(&p.tmDQ, p.dq_acc, D, s.Nq, zq)) return ATTN_ERR_CUDA;
  p.delta = reinterpret_cast<const float *>(base + round_up256(static_cast<size_t>(rows) * D * 4));
  p.lse = LSE;
  p.dK = dK;
  p.dV = dV;
  p.status = status;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.group = s.Hq / s.Hkv;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * 1.4426950408889634074);
  p.sm_scale = s.sm_scale;
  p.timeout_ns = g_timeout_ns.load();
  const long long nkt = (s.Nk + 127) / 128;
  p.band = bwd_band(zk, nkt, std::max(1, device_sm_count()));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  static std::once_flag once[64];
  static bool ready[64];
  std::call_once(once[dev], [&] {
    ready[dev] = cudaFuncSetAttribute(attn_bwd_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg::kSmemBytes) == cudaSuccess;
    if (!ready[dev]) (void)cudaGetLastError();
  });
  if (!ready[dev]) return ATTN_ERR_UNSUPPORTED;
  float *delta = reinterpret_cast<float *>(base + round_up256(static_cast<size_t>(rows) * D * 4));
  if (launch_pdl(attn_bwd_prep_kernel<D, BF16>, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), 0, stream, O,
                 dO, delta, p.dq_acc, rows) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(zk * nkt));
  if (launch_pdl(attn_bwd_kernel<D, BF16>, grid, dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const long long n4 = rows * D / 4;
  const int sms = std::max(1, device_sm_count());
  const long long blocks = std::min<long long>((n4 + 255) / 256, 8LL * sms);
  if (launch_pdl(attn_bwd_dq_kernel<BF16>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                 static_cast<const float *>(p.dq_acc), dQ, n4, s.sm_scale) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- latent (MLA) decode
struct MlaPlan {
  int nchunks = 0, chunk_keys = 0, row_blocks = 0;
  size_t bytes = 0;  // 0: invalid sizes
};

// Chunks per (request, 16-row block), minimising (waves of one CTA per SM)
// x (tiles per CTA + 2), as for the split-KV decode.
static MlaPlan mla_plan(int B, int n_h, int Nq, int Nk, int sms) {
  MlaPlan pl;
  if (B <= 0 || n_h <= 0 || Nq <= 0 || Nk <= 0 || sms <= 0) return pl;
  const long long R = static_cast<long long>(n_h) * Nq;
  const long long rb = (R + kMlaRows - 1) / kMlaRows;
  const long long units = static_cast<long long>(B) * rb;
  if (units > 65535 || R > 0x7fffffffLL / 4) return pl;
  const long long tiles = (Nk + kDecKeys - 1) / kDecKeys;
  const long long max_n = std::min<long long>(std::min<long long>(tiles, kDecMaxChunks), 4LL * sms / units + 1);
  long long best_n = 1, best_cost = -1;
  for (long long n = 1; n <= max_n; ++n) {
    const long long cost = ((units * n + sms - 1) / sms) * ((tiles + n - 1) / n + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_n = n;
    }
  }
  int ck = static_cast<int>((Nk + best_n - 1) / best_n);
  ck = ((ck + kDecKeys - 1) / kDecKeys) * kDecKeys;
  pl.nchunks = (Nk + ck - 1) / ck;
  pl.chunk_keys = ck;
  pl.row_blocks = static_cast<int>(rb);
  pl.bytes = static_cast<size_t>(B) * R * pl.nchunks * (kMlaD + 1) * sizeof(float);
  return pl;
}

template <bool BF16>
static attn_status_t launch_mla(const void *Q, const void *Cl, void *O, float *LSE, const Shape &s,
                                const MlaPlan &pl, float *ws, cudaStream_t stream) {
  MlaParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.tmC, Cl, kMlaD, s.Nk, s.B, BF16, kDecKeys)) return ATTN_ERR_CUDA;
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  const long long R = static_cast<long long>(s.Hq) * s.Nq;
  p.Q = Q;
  p.ws = ws;
  p.ws_lse = ws + static_cast<size_t>(s.B) * R * pl.nchunks * kMlaD;
  p.status = status;
  p.B = s.B;
  p.n_h = s.Hq;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.R = static_cast<int>(R);
  p.row_blocks = pl.row_blocks;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  p.nchunks = pl.nchunks;
  p.chunk_keys = pl.chunk_keys;
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * 1.4426950408889634074);
  p.timeout_ns = g_timeout_ns.load();
  p.stall_after = g_stall_after.load();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  static std::once_flag once[64];
  static bool ready[64];
  std::call_once(once[dev], [&] {
    ready[dev] = cudaFuncSetAttribute(attn_mla_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      MlaCfg::kSmemBytes) == cudaSuccess &&
                 cudaFuncSetAttribute(attn_mla_kernel<!BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      MlaCfg::kSmemBytes) == cudaSuccess;
    if (!ready[dev]) (void)cudaGetLastError();
  });
  if (!ready[dev]) return ATTN_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(pl.nchunks), static_cast<unsigned>(static_cast<long long>(s.B) * pl.row_blocks));
  if (launch_pdl(attn_mla_kernel<BF16>, grid, dim3(kMlaThreads), MlaCfg::kSmemBytes, stream, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(s.B) * R;
  const size_t merge_smem = static_cast<size_t>(((pl.nchunks + 3) & ~3) + kMlaD) * sizeof(float);
  const float *ws_c = ws, *ws_lse_c = p.ws_lse;
  if (launch_pdl(attn_decode_combine_kernel<kMlaD, BF16>, dim3(static_cast<unsigned>(rows)), dim3(128), merge_smem,
                 stream, ws_c, ws_lse_c, O, LSE, static_cast<int>(rows), pl.nchunks) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Tensor-core latent attention: CTA pairs (one per output half) per
// (request, 128-row block, key chunk), one CTA per SM.  Chunks minimise
// waves x (tiles per chunk + 2, + 4 for the partials' round trip through the
// workspace when there is more than one chunk).
static MlaPlan mla_tc_plan(int B, int n_h, int Nq, int Nk, int sms) {
  MlaPlan pl;
  if (B <= 0 || n_h <= 0 || Nq <= 0 || Nk <= 0 || sms <= 0) return pl;
  const long long R = static_cast<long long>(n_h) * Nq;
  const long long rb = (R + kMlaTcRows - 1) / kMlaTcRows;
  const long long units = static_cast<long long>(B) * rb;
  if (units > 65535 || R > 0x7fffffffLL / 4) return pl;
  const long long tiles = (Nk + kMlaTcKeys - 1) / kMlaTcKeys;
  const long long max_n = std::min<long long>(std::min<long long>(tiles, kDecMaxChunks), 4LL * sms / (2 * units) + 1);
  long long best_n = 1, best_cost = -1;
  for (long long n = 1; n <= max_n; ++n) {
    const long long waves = (2 * units * n + sms - 1) / sms;
    const long long cost = waves * ((tiles + n - 1) / n + 2 + (n > 1 ? 4 : 0));
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_n = n;
    }
  }
  int ck = static_cast<int>((Nk + best_n - 1) / best_n);
  ck = ((ck + kMlaTcKeys - 1) / kMlaTcKeys) * kMlaTcKeys;
  pl.nchunks = (Nk + ck - 1) / ck;
  pl.chunk_keys = ck;
  pl.row_blocks = static_cast<int>(rb);
  pl.bytes = pl.nchunks > 1 ? static_cast<size_t>(B) * R * pl.nchunks * (kMlaD + 1) * sizeof(float) : 0;
  return pl;
}

static bool mla_use_tc(int n_h, int Nq) { return static_cast<long long>(n_h) * Nq >= kMlaTcMinRows; }

template <bool BF16>
static attn_status_t launch_mla_tc(const void *Q, const void *Cl, void *O, float *LSE, const Shape &s,
                                   const MlaPlan &pl, float *ws, cudaStream_t stream) {
  MlaTcParams p;
  std::memset(&p, 0, sizeof(p));
  const long long R = static_cast<long long>(s.Hq) * s.Nq;
  if (!make_map(&p.tmQ, Q, kMlaD, static_cast<int>(R), s.B, BF16, kMlaTcRows) ||
      !make_map(&p.tmC, Cl, kMlaD, s.Nk, s.B, BF16, kMlaTcKeys))
    return ATTN_ERR_CUDA;
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  p.Q = Q;
  p.O = O;
  p.lse = LSE;
  p.ws = ws;
  p.ws_lse = ws + static_cast<size_t>(s.B) * R * pl.nchunks * kMlaD;
  p.status = status;
  p.B = s.B;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.R = static_cast<int>(R);
  p.row_blocks = pl.row_blocks;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  p.nchunks = pl.nchunks;
  p.chunk_keys = pl.chunk_keys;
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * 1.4426950408889634074);
  p.timeout_ns = g_timeout_ns.load();
  p.stall_after = g_stall_after.load();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  static std::once_flag once[64];
  static bool ready[64];
  std::call_once(once[dev], [&] {
    ready[dev] = cudaFuncSetAttribute(attn_mla_tc_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      MlaTcCfg::kSmemBytes) == cudaSuccess &&
                 cudaFuncSetAttribute(attn_mla_tc_kernel<!BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      MlaTcCfg::kSmemBytes) == cudaSuccess;
    if (!ready[dev]) (void)cudaGetLastError();
  });
  if (!ready[dev]) return ATTN_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(2 * pl.nchunks),
                  static_cast<unsigned>(static_cast<long long>(s.B) * pl.row_blocks));
  if (launch_pdl(attn_mla_tc_kernel<BF16>, grid, dim3(kMlaTcThreads), MlaTcCfg::kSmemBytes, stream, p) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  if (pl.nchunks > 1) {
    const long long rows = static_cast<long long>(s.B) * R;
    const size_t merge_smem = static_cast<size_t>(((pl.nchunks + 3) & ~3) + kMlaD) * sizeof(float);
    const float *ws_c = ws, *ws_lse_c = p.ws_lse;
    if (launch_pdl(attn_decode_combine_kernel<kMlaD, BF16>, dim3(static_cast<unsigned>(rows)), dim3(128),
                   merge_smem, stream, ws_c, ws_lse_c, O, LSE, static_cast<int>(rows), pl.nchunks) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- split-KV (decode) path
struct DecPlan {
  int nchunks = 0, chunk_keys = 0;
  bool fused = false;    // the split kernel merges the chunks itself
  size_t flag_off = 0;   // byte offset of the per-group arrival counters (8 bytes each)
  size_t bytes = 0;      // 0: this shape does not take the split-KV path
};


// Resident CTAs per SM of the split kernel for (d, row blocks), from the
// occupancy calculator (shared memory and registers decide it).
template <int D, int RB>
static int decode_ctas_per_sm_t() {
  using Cfg = DecCfg<D, RB>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  static int cache[64];
  static std::once_flag once[64];
  std::call_once(once[dev], [&] {
    bool bad = false;
    for (auto k : {attn_decode_kernel<D, true, RB, false>, attn_decode_kernel<D, false, RB, false>,
                   attn_decode_kernel<D, true, RB, true>, attn_decode_kernel<D, false, RB, true>})
      bad |= cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) != cudaSuccess;
    for (auto k : {attn_decode_kernel<D, true, RB, false, true>, attn_decode_kernel<D, false, RB, false, true>})
      bad |= cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DecCfg<D, RB, true>::kSmemBytes) !=
             cudaSuccess;
    // flat and paged kernels: the smaller residency (the plan sizes one wave)
    int n = 0, n_paged = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<D, true, RB, false>, kDecThreads,
                                                      Cfg::kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n_paged, attn_decode_kernel<D, true, RB, true>, kDecThreads,
                                                      Cfg::kSmemBytes) != cudaSuccess) {
      n = 0;
      bad = true;
    }
    if (bad) (void)cudaGetLastError();  // not reported by a later launch check
    n = std::min(n, n_paged);
    cache[dev] = n;
  });
  return cache[dev];
}

static int decode_ctas_per_sm(int d, int rb) {
  if (d == 64) return rb == 1 ? decode_ctas_per_sm_t<64, 1>() : decode_ctas_per_sm_t<64, 2>();
  return rb == 1 ? decode_ctas_per_sm_t<128, 1>() : decode_ctas_per_sm_t<128, 2>();
}

// Paged calls: each request's length is known only on the device, and the
// lengths of a batch may differ widely.  A plan sized for max_seq_len keys
// in every request can leave the longest requests to single CTAs that
// stream on long after the others have finished, so their chunks hold at
// most this many K/V tiles (chunks past a short request's end are empty and
// end at once).
constexpr int kPagedMaxChunkTiles = 32;
constexpr int kDecCtaCostTiles = 6;  // fixed cost of a flat split-KV CTA, in K/V tiles

// The split-KV path serves shapes whose GQA group holds at most 32 query rows
// (decode: Nq = 1 with up to 32 query heads per K/V head).  The number of
// chunks per group minimises an estimate of the time:
// - flat calls: (CTAs per SM) x (K/V tiles per CTA + 6).  The K/V stream of
//   a CTA is bound by the copies it keeps in flight, and the SM's CTAs
//   share its bandwidth, so what counts is the tiles an SM streams plus a
//   fixed cost per CTA (start, first-tile latency, partial write, merge) of
//   about six tiles: one long chunk per SM beats two CTAs of half the length
//   (on GB300, 4 chunks x 32 groups: 33.0 us against 35.1 us for 9 chunks
//   at two CTAs per SM, for 8192 keys at d = 128);
// - paged calls: (waves of resident CTAs) x (tiles per CTA + 2), then at
//   most 32 tiles per chunk.  Their producer issues one copy per page, so
//   two resident CTAs per SM (two producers) pay;
// - int8 K/V: the same waves model without the cap.  Its consumers widen
//   every tile before the MMAs, so two CTAs per SM (twice the warps) pay
//   (38.1 us against 51.3 us with the flat model's 4 chunks at Hkv = 8).
// The plan for a device of `sms` SMs with `per_sm` resident split CTAs each.
enum DecPlanMode : int { kPlanFlat = 0, kPlanPaged = 1, kPlanQuant = 2 };
static DecPlan decode_plan_for(int B, int Hq, int Hkv, int Nq, int Nk, int d, int mode, int sms, int per_sm) {
  DecPlan pl;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128)) return pl;
  const long long R = static_cast<long long>(Hq / Hkv) * Nq;
  if (R > kDecMaxRows) return pl;
  if (sms <= 0 || per_sm <= 0) return pl;
  const long long units = static_cast<long long>(B) * Hkv;
  if (units > 65535) return pl;  // grid.y limit
  const long long slots = static_cast<long long>(sms) * per_sm;
  const long long tiles = (Nk + kDecKeys - 1) / kDecKeys;
  const long long max_n = std::min<long long>(std::min<long long>(tiles, kDecMaxChunks), 4 * slots / units + 1);
  long long best_n = 1, best_cost = -1;
  for (long long n = 1; n <= max_n; ++n) {
    const long long per_tile = (tiles + n - 1) / n;
    const long long cost = mode != kPlanFlat ? ((units * n + slots - 1) / slots) * (per_tile + 2)
                                             : ((units * n + sms - 1) / sms) * (per_tile + kDecCtaCostTiles);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_n = n;
    }
  }
  if (mode == kPlanPaged) {
    const long long cap_n = (tiles + kPagedMaxChunkTiles - 1) / kPagedMaxChunkTiles;
    best_n = std::max(best_n, std::min<long long>(cap_n, kDecMaxChunks));
  }
  int chunk_keys = static_cast<int>((Nk + best_n - 1) / best_n);
  chunk_keys = ((chunk_keys + kDecKeys - 1) / kDecKeys) * kDecKeys;
  pl.nchunks = (Nk + chunk_keys - 1) / chunk_keys;
  pl.chunk_keys = chunk_keys;
  // A small merge (rows x chunks x d of a group) is done by the split
  // kernel's CTA that finishes last in each group (no CTA waits for
  // another); a large one by the merge kernel, one CTA per row.
  pl.fused = R * pl.nchunks * d <= kDecFusedMerge;
  const size_t part = static_cast<size_t>(B) * Hq * Nq * pl.nchunks * (d + 1) * sizeof(float);
  pl.flag_off = (part + 15) & ~size_t(15);
  pl.bytes = pl.flag_off + static_cast<size_t>(units) * sizeof(unsigned long long);
  return pl;
}

static DecPlan decode_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int mode = kPlanFlat) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128)) return {};
  const long long R = static_cast<long long>(Hq / Hkv) * Nq;
  if (R > kDecMaxRows) return {};
  return decode_plan_for(B, Hq, Hkv, Nq, Nk, d, mode, device_sm_count(), decode_ctas_per_sm(d, R <= 16 ? 1 : 2));
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  return decode_plan(B, Hq, Hkv, Nq, Nk, d).bytes;
}


// Scales of an int8 K/V cache (K = k_scale * codes, V = v_scale * codes).
struct QuantKV {
  float k_scale, v_scale;
};

template <int D, bool BF16>
static attn_status_t launch_decode_t(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                     const Shape &s, const DecPlan &pl, float *ws, int *status,
                                     const PagedKV *pg, cudaStream_t stream, const QuantKV *qk = nullptr) {
  DecParams p;
  std::memset(&p, 0, sizeof(p));
  const long long zk = static_cast<long long>(s.B) * s.Hkv;
  if (qk != nullptr) {
    if (!make_map_s8(&p.tmK, K, D, s.Nk, zk) || !make_map_s8(&p.tmV, V, D, s.Nk, zk)) return ATTN_ERR_CUDA;
  } else if (pg == nullptr) {
    if (!make_map(&p.tmK, K, D, s.Nk, zk, BF16, kDecKeys) || !make_map(&p.tmV, V, D, s.Nk, zk, BF16, kDecKeys))
      return ATTN_ERR_CUDA;
  } else {
    const long long slabs = static_cast<long long>(pg->num_pages) * s.Hkv;
    const int box = std::min(pg->page_size, kDecKeys);
    if (!make_map(&p.tmK, K, D, pg->page_size, slabs, BF16, box) ||
        !make_map(&p.tmV, V, D, pg->page_size, slabs, BF16, box))
      return ATTN_ERR_CUDA;
    p.block_table = pg->block_table;
    p.seq_lens = pg->seq_lens;
    int shift = 0;
    while ((1 << shift) < pg->page_size) ++shift;
    p.page_shift = shift;
    p.max_pages = pg->max_pages;
    p.num_pages = pg->num_pages;
  }
  p.Q = Q;
  p.ws = ws;
  p.ws_lse = ws + static_cast<size_t>(s.B) * s.Hq * s.Nq * pl.nchunks * D;
  p.status = status;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.group = s.Hq / s.Hkv;
  p.R = p.group * s.Nq;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  p.nchunks = pl.nchunks;
  p.chunk_keys = pl.chunk_keys;
  // keys some row of a group can see: all of them, except below the window
  // of the first query row
  p.kv_lo = (s.causal && s.window > 0) ? std::max(0, (s.Nk - s.Nq) - s.window + 1) : 0;
  p.kv_hi = s.Nk;
  // the key scale folds into the softmax scale, the value scale into each chunk's O
  const double ks = qk ? static_cast<double>(qk->k_scale) : 1.0;
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * ks * 1.4426950408889634074);
  p.v_scale = qk ? qk->v_scale : 1.f;
  p.timeout_ns = g_timeout_ns.load();
  p.stall_after = g_stall_after.load();
  if (pl.fused) {
    p.fused = 1;
    unsigned tok = ++g_split_token;
    if (tok == 0) tok = ++g_split_token;
    p.token = tok;
    p.counters = reinterpret_cast<unsigned long long *>(reinterpret_cast<uint8_t *>(ws) + pl.flag_off);
    p.O = O;
    p.lse = LSE;
  }
  // (the plan already set the shared-memory attribute of both kernels)
  if (decode_ctas_per_sm(D, p.R <= 16 ? 1 : 2) <= 0) return ATTN_ERR_CUDA;
  dim3 grid(static_cast<unsigned>(pl.nchunks), static_cast<unsigned>(zk));
  const dim3 block(kDecThreads);
  cudaError_t le;
  if (qk != nullptr)
    le = (p.R <= 16)
             ? launch_pdl(attn_decode_kernel<D, BF16, 1, false, true>, grid, block, DecCfg<D, 1, true>::kSmemBytes, stream, p)
             : launch_pdl(attn_decode_kernel<D, BF16, 2, false, true>, grid, block, DecCfg<D, 2, true>::kSmemBytes, stream, p);
  else if (pg == nullptr)
    le = (p.R <= 16) ? launch_pdl(attn_decode_kernel<D, BF16, 1, false>, grid, block, DecCfg<D, 1>::kSmemBytes, stream, p)
                     : launch_pdl(attn_decode_kernel<D, BF16, 2, false>, grid, block, DecCfg<D, 2>::kSmemBytes, stream, p);
  else
    le = (p.R <= 16) ? launch_pdl(attn_decode_kernel<D, BF16, 1, true>, grid, block, DecCfg<D, 1>::kSmemBytes, stream, p)
                     : launch_pdl(attn_decode_kernel<D, BF16, 2, true>, grid, block, DecCfg<D, 2>::kSmemBytes, stream, p);
  if (le != cudaSuccess || cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  if (pl.fused) return ATTN_OK;
  // The merge kernel is a programmatic dependent: it may launch while the
  // split kernel runs and waits (griddepcontrol.wait) for its results.
  const int rows = s.B * s.Hq * s.Nq;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = static_cast<size_t>(((pl.nchunks + 3) & ~3) + 128 / (D / 4) * D) * sizeof(float);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float *ws_c = ws, *ws_lse_c = p.ws_lse;
  if (cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel<D, BF16>, ws_c, ws_lse_c, O, LSE, rows, pl.nchunks) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t dispatch_decode(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                     const Shape &s, const DecPlan &pl, float *ws, cudaStream_t stream,
                                     const PagedKV *pg = nullptr, const QuantKV *qk = nullptr) {
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  const bool bf16 = s.dtype == ATTN_DTYPE_BF16;
  if (s.d == 64)
    return bf16 ? launch_decode_t<64, true>(Q, K, V, O, LSE, s, pl, ws, status, pg, stream, qk)
                : launch_decode_t<64, false>(Q, K, V, O, LSE, s, pl, ws, status, pg, stream, qk);
  return bf16 ? launch_decode_t<128, true>(Q, K, V, O, LSE, s, pl, ws, status, pg, stream, qk)
              : launch_decode_t<128, false>(Q, K, V, O, LSE, s, pl, ws, status, pg, stream, qk);
}

// ---------------------------------------------------------------- short keys (Nk <= 128)
template <int D, bool BF16, int NK>
static int short_ctas_per_sm() {
  using Cfg = ShortCfg<D, NK>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  static int cache[64];
  static std::once_flag once[64];
  std::call_once(once[dev], [&] {
    bool bad = cudaFuncSetAttribute(attn_short_kernel<D, BF16, NK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg::kSmemBytes) != cudaSuccess;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_short_kernel<D, BF16, NK>, kShortThreads,
                                                      Cfg::kSmemBytes) != cudaSuccess) {
      n = 0;
      bad = true;
    }
    if (bad) (void)cudaGetLastError();  // not reported by a later launch check
    cache[dev] = n;
  });
  return cache[dev];
}

template <int D, bool BF16, int NK>
static attn_status_t launch_short_t(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                    const Shape &s, int *status, cudaStream_t stream) {
  ShortParams p;
  std::memset(&p, 0, sizeof(p));
  const long long zq = static_cast<long long>(s.B) * s.Hq, zk = static_cast<long long>(s.B) * s.Hkv;
  if (!make_map(&p.tmQ, Q, D, s.Nq, zq, BF16, 64) || !make_map(&p.tmK, K, D, s.Nk, zk, BF16, 64) ||
      !make_map(&p.tmV, V, D, s.Nk, zk, BF16, 64))
    return ATTN_ERR_CUDA;
  p.O = O;
  p.lse = LSE;
  p.status = status;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Nq = s.Nq;
  p.Nk = s.Nk;
  p.group = s.Hq / s.Hkv;
  p.causal = s.causal ? 1 : 0;
  p.window = s.window;
  p.n_qblocks = (s.Nq + kShortRows - 1) / kShortRows;
  p.n_units = static_cast<int>(zq * p.n_qblocks);
  p.scale_log2 = static_cast<float>(static_cast<double>(s.sm_scale) * 1.4426950408889634074);
  p.timeout_ns = g_timeout_ns.load();
  p.stall_after = g_stall_after.load();
  const int per_sm = short_ctas_per_sm<D, BF16, NK>(), sms = device_sm_count();
  if (per_sm <= 0 || sms <= 0) return ATTN_ERR_CUDA;
  const int grid = static_cast<int>(std::min<long long>(p.n_units, static_cast<long long>(per_sm) * sms));
  if (launch_pdl(attn_short_kernel<D, BF16, NK>, dim3(grid), dim3(kShortThreads), ShortCfg<D, NK>::kSmemBytes,
                 stream, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Shapes with at most 128 keys take the short-key kernel: every head's K and
// V fit one tile, and the work is bound by moving Q, K, V and O.
static bool short_path(const Shape &s) {
  const long long units = static_cast<long long>(s.B) * s.Hq * ((s.Nq + kShortRows - 1) / kShortRows);
  return s.Nk <= kShortMaxKeys && units <= 0x7fffffffLL;
}

static attn_status_t dispatch_short(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                    const Shape &s, cudaStream_t stream) {
  int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
  const bool bf16 = s.dtype == ATTN_DTYPE_BF16;
  const bool nk64 = s.Nk <= 64;
  if (s.d == 64) {
    if (nk64)
      return bf16 ? launch_short_t<64, true, 64>(Q, K, V, O, LSE, s, status, stream)
                  : launch_short_t<64, false, 64>(Q, K, V, O, LSE, s, status, stream);
    return bf16 ? launch_short_t<64, true, 128>(Q, K, V, O, LSE, s, status, stream)
                : launch_short_t<64, false, 128>(Q, K, V, O, LSE, s, status, stream);
  }
  if (nk64)
    return bf16 ? launch_short_t<128, true, 64>(Q, K, V, O, LSE, s, status, stream)
                : launch_short_t<128, false, 64>(Q, K, V, O, LSE, s, status, stream);
  return bf16 ? launch_short_t<128, true, 128>(Q, K, V, O, LSE, s, status, stream)
              : launch_short_t<128, false, 128>(Q, K, V, O, LSE, s, status, stream);
}

// Workspace of a call (no window): the split-KV decode plan's when the
// shape has one (also for Nk <= 128, which the no-alloc entry runs through
// it), else the stream-K split of the prefill, else none.
static size_t workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  Shape s{B, Hq, Hkv, Nq, Nk, d, 0, 0, 1.f, ATTN_DTYPE_FP16};
  const size_t dec = decode_plan(B, Hq, Hkv, Nq, Nk, d).bytes;
  if (dec > 0) return dec;
  if (short_path(s)) return 0;
  return split_plan_bytes(s, device_sm_count());
}

static attn_status_t run(const void *Q, const void *K, const void *V, void *O, float *LSE, const Shape &s,
                         void *ws, size_t ws_bytes, cudaStream_t stream) {
  attn_status_t st = validate(Q, K, V, O, LSE, s);
  if (st != ATTN_OK) return st;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  if (short_path(s)) return dispatch_short(Q, K, V, O, LSE, s, stream);
  if (ws != nullptr) {
    const DecPlan pl = decode_plan(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d);
    if (pl.bytes > 0) {
      if (ws_bytes < pl.bytes || !aligned16(ws)) return ATTN_ERR_INVALID_ARG;
      return dispatch_decode(Q, K, V, O, LSE, s, pl, static_cast<float *>(ws), stream);
    }
  }
  return dispatch_prefill(Q, K, V, O, LSE, s, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- host-buffer calls, pipelined
// A large call on host buffers is cut into pieces: contiguous ranges of
// (request, K/V head) slabs, each a contiguous byte range of Q, K, V, O and
// LSE and a call of its own.  A piece's inputs are copied in on one internal
// stream, its kernel runs once they have arrived (even pieces on the
// caller's stream, odd ones on an internal compute stream, so that a piece's
// CTAs can start on the SMs the previous piece's last CTAs leave idle), and
// its outputs are copied out on another internal stream: the copies of one
// piece overlap the compute of its neighbours (copy-in and copy-out each go
// in piece order).  Pieces are used only when each is computed with
// the schedule and item shape of the whole call (the plain prefill, the same
// pairing of query tiles), so the results are the same bits.
constexpr int kHostMaxPieces = 16;
constexpr int kHostTargetPieces = 8;
constexpr size_t kHostPipeMinBytes = size_t(64) << 20;  // Q + K + V below this: copy, compute, copy

struct HostPiece {
  int b0, nb;  // requests [b0, b0 + nb)
  int h0, nh;  // K/V heads [h0, h0 + nh) of each (all of them when nb > 1)
};

// Per device: two copy streams, a second compute stream and the events that
// chain the pieces.
struct HostPipe {
  std::mutex mu;  // one pipelined enqueue at a time per device (the events are shared)
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr, s_comp = nullptr;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_comp_end = nullptr;
  cudaEvent_t ev_in[kHostMaxPieces] = {}, ev_comp[kHostMaxPieces] = {};
};

static HostPipe &host_pipe(int dev) {
  static HostPipe pipes[64];
  return pipes[dev];
}

// Creates the streams and events on first use (the caller holds hp.mu and has
// the device current).  A failure is not cached: everything made so far is
// released, the error cleared, and the next call tries again.
static bool host_pipe_init(HostPipe &hp) {
  if (hp.ready) return true;
  bool ok = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.s_comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.ev_start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.ev_end, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.ev_comp_end, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kHostMaxPieces; ++i)
    ok = cudaEventCreateWithFlags(&hp.ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.ev_comp[i], cudaEventDisableTiming) == cudaSuccess;
  if (ok) {
    hp.ready = true;
    return true;
  }
  for (int i = 0; i < kHostMaxPieces; ++i) {
    if (hp.ev_in[i]) cudaEventDestroy(hp.ev_in[i]);
    if (hp.ev_comp[i]) cudaEventDestroy(hp.ev_comp[i]);
    hp.ev_in[i] = hp.ev_comp[i] = nullptr;
  }
  if (hp.ev_start) cudaEventDestroy(hp.ev_start);
  if (hp.ev_end) cudaEventDestroy(hp.ev_end);
  if (hp.ev_comp_end) cudaEventDestroy(hp.ev_comp_end);
  if (hp.s_in) cudaStreamDestroy(hp.s_in);
  if (hp.s_out) cudaStreamDestroy(hp.s_out);
  if (hp.s_comp) cudaStreamDestroy(hp.s_comp);
  hp.ev_start = hp.ev_end = hp.ev_comp_end = nullptr;
  hp.s_in = hp.s_out = hp.s_comp = nullptr;
  cudaGetLastError();
  return false;
}

// The pieces of a host-buffer call, or 0 when it is not cut: small calls,
// one slab, and shapes whose pieces would be scheduled differently from the
// whole call (a split path, few query tiles, another pairing).
static int host_pieces(const Shape &s, HostPiece *out) {
  if (s.d != 64 && s.d != 128) return 0;
  const size_t q = static_cast<size_t>(s.B) * s.Hq * s.Nq * s.d * 2;
  const size_t kv = static_cast<size_t>(s.B) * s.Hkv * s.Nk * s.d * 2;
  if (q + 2 * kv < kHostPipeMinBytes || static_cast<long long>(s.B) * s.Hkv < 2) return 0;
  if (short_path(s) || workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d) > 0) return 0;  // decode or split
  int n = 0;
  if (s.B >= kHostTargetPieces) {
    for (int i = 0; i < kHostTargetPieces; ++i) {
      const int b0 = static_cast<int>(static_cast<long long>(i) * s.B / kHostTargetPieces);
      const int b1 = static_cast<int>(static_cast<long long>(i + 1) * s.B / kHostTargetPieces);
      out[n++] = HostPiece{b0, b1 - b0, 0, s.Hkv};
    }
  } else {
    const int per_b = std::min(s.Hkv, (kHostTargetPieces + s.B - 1) / s.B);
    if (static_cast<long long>(s.B) * per_b > kHostMaxPieces) return 0;
    for (int b = 0; b < s.B; ++b)
      for (int j = 0; j < per_b; ++j) {
        const int h0 = j * s.Hkv / per_b, h1 = (j + 1) * s.Hkv / per_b;
        out[n++] = HostPiece{b, 1, h0, h1 - h0};
      }
  }
  if (n < 2) return 0;
  // every piece on the plain schedule with the whole call's pairing
  const int sms = device_sm_count();
  FwdParams pw, pp;
  int sw = 0, gw = 0, sp = 0, gp = 0;
  if (!prefill_schedule(s, false, sms, pw, sw, gw) || sw != kSchedPlain) return 0;
  const int g = s.Hq / s.Hkv;
  for (int i = 0; i < n; ++i) {
    const Shape ps{out[i].nb, out[i].nh * g, out[i].nh, s.Nq, s.Nk, s.d, s.causal, s.window, s.sm_scale, s.dtype};
    if (!prefill_schedule(ps, false, sms, pp, sp, gp) || sp != kSchedPlain || pp.pair_mode != pw.pair_mode) return 0;
  }
  return n;
}

// Enqueues the pieces of a host-buffer call (device buffers dQ..dL hold the
// whole call; host pointers are its host arrays).  `stream` is forked to the
// two copy streams and the second compute stream at the start and joined at
// the end, so the call as a whole still follows and precedes the work around
// it on `stream`.  On a CUDA error the streams are still joined.
static attn_status_t host_pipelined(const uint8_t *Qh, const uint8_t *Kh, const uint8_t *Vh, uint8_t *Oh,
                                    float *Lh, const Shape &s, const HostPiece *pc, int np, uint8_t *dQ,
                                    uint8_t *dK, uint8_t *dV, uint8_t *dO, float *dL, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  HostPipe &hp = host_pipe(dev);
  std::lock_guard<std::mutex> lock(hp.mu);
  if (!host_pipe_init(hp)) return ATTN_ERR_CUDA;
  const int g = s.Hq / s.Hkv;
  const size_t qh_bytes = static_cast<size_t>(s.Nq) * s.d * 2;   // one query head
  const size_t kvh_bytes = static_cast<size_t>(s.Nk) * s.d * 2;  // one K/V head
  bool ok = cudaEventRecord(hp.ev_start, stream) == cudaSuccess &&
            cudaStreamWaitEvent(hp.s_in, hp.ev_start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.s_out, hp.ev_start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.s_comp, hp.ev_start, 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  attn_status_t st = ATTN_OK;
  for (int i = 0; i < np && ok && st == ATTN_OK; ++i) {
    const HostPiece &p = pc[i];
    // odd pieces compute on the second stream: a piece's kernel can take
    // the SMs that the previous piece's last CTAs leave idle
    cudaStream_t cs = (i & 1) ? hp.s_comp : stream;
    const size_t q0 = static_cast<size_t>(p.b0) * s.Hq + static_cast<size_t>(p.h0) * g;  // first query head
    const size_t nq = static_cast<size_t>(p.nb) * p.nh * g;                                // query heads
    const size_t k0 = static_cast<size_t>(p.b0) * s.Hkv + p.h0;                          // first K/V head
    const size_t nkv = static_cast<size_t>(p.nb) * p.nh;
    ok = cudaMemcpyAsync(dQ + q0 * qh_bytes, Qh + q0 * qh_bytes, nq * qh_bytes, cudaMemcpyHostToDevice,
                         hp.s_in) == cudaSuccess &&
         cudaMemcpyAsync(dK + k0 * kvh_bytes, Kh + k0 * kvh_bytes, nkv * kvh_bytes, cudaMemcpyHostToDevice,
                         hp.s_in) == cudaSuccess &&
         cudaMemcpyAsync(dV + k0 * kvh_bytes, Vh + k0 * kvh_bytes, nkv * kvh_bytes, cudaMemcpyHostToDevice,
                         hp.s_in) == cudaSuccess &&
         cudaEventRecord(hp.ev_in[i], hp.s_in) == cudaSuccess &&
         cudaStreamWaitEvent(cs, hp.ev_in[i], 0) == cudaSuccess;
    if (!ok) break;
    const Shape ps{p.nb, p.nh * g, p.nh, s.Nq, s.Nk, s.d, s.causal, s.window, s.sm_scale, s.dtype};
    float *dLp = dL ? dL + q0 * s.Nq : nullptr;
    st = run(dQ + q0 * qh_bytes, dK + k0 * kvh_bytes, dV + k0 * kvh_bytes, dO + q0 * qh_bytes, dLp, ps, nullptr, 0,
             cs);
    if (st != ATTN_OK) break;
    ok = cudaEventRecord(hp.ev_comp[i], cs) == cudaSuccess &&
         cudaStreamWaitEvent(hp.s_out, hp.ev_comp[i], 0) == cudaSuccess &&
         cudaMemcpyAsync(Oh + q0 * qh_bytes, dO + q0 * qh_bytes, nq * qh_bytes, cudaMemcpyDeviceToHost,
                         hp.s_out) == cudaSuccess &&
         (Lh == nullptr || cudaMemcpyAsync(Lh + q0 * s.Nq, dLp, nq * s.Nq * sizeof(float), cudaMemcpyDeviceToHost,
                                           hp.s_out) == cudaSuccess);
  }
  // join the copy streams and the second compute stream back into
  // `stream`, also after an error
  const bool joined = cudaEventRecord(hp.ev_end, hp.s_out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp.ev_end, 0) == cudaSuccess &&
                      cudaEventRecord(hp.ev_comp_end, hp.s_comp) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp.ev_comp_end, 0) == cudaSuccess &&
                      cudaEventRecord(hp.ev_start, hp.s_in) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp.ev_start, 0) == cudaSuccess;
  if (st != ATTN_OK) return st;
  if (!ok || !joined) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int Hq, int Hkv,
                       int N, int d, int causal, int window, float sm_scale, attn_dtype_t dtype,
                       cudaStream_t stream) {
  Shape s{B, Hq, Hkv, N, N, d, causal, window, sm_scale, dtype};
  return run(Q, K, V, O, LSE, s, nullptr, 0, stream);
}

attn_status_t attn_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int Hq,
                          int Hkv, int Nq, int Nk, int d, int causal, int window, float sm_scale,
                          attn_dtype_t dtype, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype};
  return run(Q, K, V, O, LSE, s, workspace, workspace_bytes, stream);
}

size_t attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128) || Hq % Hkv) return 0;
  return workspace_bytes(B, Hq, Hkv, Nq, Nk, d);
}

attn_status_t attn_fwd_paged(const void *Q, const void *K_pages, const void *V_pages, const int *block_table,
                             const int *seq_lens, void *O, float *LSE, int B, int Hq, int Hkv, int Nq,
                             int max_seq_len, int d, int page_size, int num_pages, int max_pages_per_seq,
                             int causal, int window, float sm_scale, attn_dtype_t dtype, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  Shape s{B, Hq, Hkv, Nq, max_seq_len, d, causal, window, sm_scale, dtype};
  attn_status_t st = validate(Q, K_pages, V_pages, O, LSE, s);
  if (st != ATTN_OK) return st;
  if (block_table == nullptr || seq_lens == nullptr || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (page_size < 8 || page_size > 256 || (page_size & (page_size - 1)) != 0) return ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || max_pages_per_seq <= 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(max_pages_per_seq) * page_size < max_seq_len) return ATTN_ERR_INVALID_ARG;
  // copy coordinates are 32-bit: the pool's slabs and one past them
  if (static_cast<long long>(num_pages) * Hkv >= 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  const PagedKV pg{block_table, seq_lens, page_size, num_pages, max_pages_per_seq};
  const DecPlan pl = decode_plan(B, Hq, Hkv, Nq, max_seq_len, d, kPlanPaged);
  if (pl.bytes == 0) {
    // groups of more than 32 query rows: the tiled prefill kernel on the pages
    if (static_cast<long long>(B) * Hq * ((Nq + kBM - 1) / kBM) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    return dispatch_prefill(Q, K_pages, V_pages, O, LSE, s, nullptr, 0, stream, &pg);
  }
  if (workspace == nullptr || workspace_bytes < pl.bytes || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  return dispatch_decode(Q, K_pages, V_pages, O, LSE, s, pl, static_cast<float *>(workspace), stream, &pg);
}

attn_status_t attn_fwd_kv_int8(const void *Q, const void *K_codes, const void *V_codes, float k_scale,
                               float v_scale, void *O, float *LSE, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                               int causal, int window, float sm_scale, attn_dtype_t dtype, void *workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype};
  attn_status_t st = validate(Q, K_codes, V_codes, O, LSE, s);
  if (st != ATTN_OK) return st;
  if (!std::isfinite(k_scale) || !(k_scale > 0.f) || !std::isfinite(v_scale) || !(v_scale > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  const DecPlan pl = decode_plan(B, Hq, Hkv, Nq, Nk, d, kPlanQuant);
  if (pl.bytes == 0) return ATTN_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < pl.bytes || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  const QuantKV qk{k_scale, v_scale};
  return dispatch_decode(Q, K_codes, V_codes, O, LSE, s, pl, static_cast<float *>(workspace), stream, nullptr, &qk);
}

size_t attn_fwd_kv_int8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  return decode_plan(B, Hq, Hkv, Nq, Nk, d, kPlanQuant).bytes;
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Nq, int d) {
  if (B <= 0 || Hq <= 0 || Nq <= 0 || (d != 64 && d != 128)) return 0;
  return bwd_ws_bytes(static_cast<long long>(B) * Hq * Nq, d);
}

attn_status_t attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                       void *dQ, void *dK, void *dV, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                       int window, float sm_scale, attn_dtype_t dtype, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype};
  attn_status_t st = validate(Q, K, V, O, LSE, s);
  if (st != ATTN_OK) return st;
  if (!dO || !dQ || !dK || !dV || !LSE || !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
    return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hkv * ((static_cast<long long>(Nk) + 127) / 128) > 0x7fffffffLL)
    return ATTN_ERR_INVALID_ARG;  // one CTA per (K/V group, key tile)
  const size_t need = bwd_ws_bytes(static_cast<long long>(B) * Hq * Nq, d);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  if (d == 64)
    return bf16 ? launch_bwd<64, true>(Q, K, V, O, dO, LSE, dQ, dK, dV, s, workspace, stream)
                : launch_bwd<64, false>(Q, K, V, O, dO, LSE, dQ, dK, dV, s, workspace, stream);
  return bf16 ? launch_bwd<128, true>(Q, K, V, O, dO, LSE, dQ, dK, dV, s, workspace, stream)
              : launch_bwd<128, false>(Q, K, V, O, dO, LSE, dQ, dK, dV, s, workspace, stream);
}

size_t attn_fwd_mla_workspace_bytes(int B, int n_h, int Nq, int Nk, int d_c) {
  if (d_c != kMlaD || B <= 0 || n_h <= 0 || Nq <= 0 || Nk <= 0) return 0;
  const int sms = device_sm_count();
  const MlaPlan pl = mla_use_tc(n_h, Nq) ? mla_tc_plan(B, n_h, Nq, Nk, sms) : mla_plan(B, n_h, Nq, Nk, sms);
  if (pl.nchunks == 0) return 0;
  return std::max<size_t>(pl.bytes, 256);
}

attn_status_t attn_fwd_mla(const void *Q_lat, const void *C_lat, void *O_lat, float *LSE, int B, int n_h, int Nq,
                           int Nk, int d_c, int causal, int window, float sm_scale, attn_dtype_t dtype,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (d_c != kMlaD) return d_c > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  Shape s{B, n_h, 1, Nq, Nk, 128, causal, window, sm_scale, dtype};  // d only passes the checks
  attn_status_t st = validate(Q_lat, C_lat, C_lat, O_lat, LSE, s);
  if (st != ATTN_OK) return st;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  const bool tc = mla_use_tc(n_h, Nq);
  const MlaPlan pl = tc ? mla_tc_plan(B, n_h, Nq, Nk, sms) : mla_plan(B, n_h, Nq, Nk, sms);
  if (pl.nchunks == 0) return ATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < std::max<size_t>(pl.bytes, 256) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  float *ws = static_cast<float *>(workspace);
  const bool bf = dtype == ATTN_DTYPE_BF16;
  if (tc)
    return bf ? launch_mla_tc<true>(Q_lat, C_lat, O_lat, LSE, s, pl, ws, stream)
              : launch_mla_tc<false>(Q_lat, C_lat, O_lat, LSE, s, pl, ws, stream);
  return bf ? launch_mla<true>(Q_lat, C_lat, O_lat, LSE, s, pl, ws, stream)
            : launch_mla<false>(Q_lat, C_lat, O_lat, LSE, s, pl, ws, stream);
}

int attn_fwd_paged_path(int B, int Hq, int Hkv, int Nq, int max_seq_len, int d) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || max_seq_len <= 0 || (d != 64 && d != 128) || Hq % Hkv) return -1;
  const DecPlan pl = decode_plan(B, Hq, Hkv, Nq, max_seq_len, d, kPlanPaged);
  if (pl.bytes == 0) return ATTN_PATH_PREFILL;  // larger query groups: the tiled prefill kernel
  return pl.fused ? ATTN_PATH_SPLIT_KV_FUSED : ATTN_PATH_SPLIT_KV;
}

size_t attn_fwd_paged_workspace_bytes(int B, int Hq, int Hkv, int Nq, int max_seq_len, int d) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || max_seq_len <= 0 || (d != 64 && d != 128) || Hq % Hkv) return 0;
  return decode_plan(B, Hq, Hkv, Nq, max_seq_len, d, kPlanPaged).bytes;
}

int attn_fwd_path(int B, int Hq, int Hkv, int Nq, int Nk, int d, int with_workspace) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128)) return -1;
  Shape s{B, Hq, Hkv, Nq, Nk, d, 0, 0, 1.f, ATTN_DTYPE_FP16};
  if (short_path(s)) return ATTN_PATH_SHORT;
  const DecPlan dp = decode_plan(B, Hq, Hkv, Nq, Nk, d);
  if (with_workspace && dp.bytes > 0) return dp.fused ? ATTN_PATH_SPLIT_KV_FUSED : ATTN_PATH_SPLIT_KV;
  if (with_workspace && split_plan_bytes(s, device_sm_count()) > 0) return ATTN_PATH_PREFILL_SPLIT;
  return ATTN_PATH_PREFILL;
}

int attn_fwd_decode_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int paged, int sms, int ctas_per_sm,
                         long long *info) {
  if (info == nullptr) return -1;
  if (paged < 0 || paged > 2) return -1;
  const DecPlan pl = decode_plan_for(B, Hq, Hkv, Nq, Nk, d, paged, sms, ctas_per_sm);
  if (pl.bytes == 0) return -1;
  info[0] = pl.nchunks;
  info[1] = pl.chunk_keys;
  info[2] = pl.fused ? 1 : 0;
  info[3] = static_cast<long long>(pl.flag_off);
  info[4] = static_cast<long long>(pl.bytes);
  return 0;
}

int attn_fwd_prefill_visits(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window,
                            int with_workspace, int sms, int *info, int *visits, int max_visits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128) ||
      sms <= 0 || window < 0 || (window > 0 && !causal) || (causal && Nq > Nk) || info == nullptr ||
      (max_visits > 0 && visits == nullptr))
    return -1;
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, 1.f, ATTN_DTYPE_FP16};
  if (short_path(s)) return -1;
  // with a workspace, small query groups take the split-KV path (on any
  // device where its kernel fits)
  if (with_workspace && static_cast<long long>(Hq / Hkv) * Nq <= kDecMaxRows && static_cast<long long>(B) * Hkv <= 65535)
    return -1;
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  int sched = kSchedPlain, grid = 0;
  if (!prefill_schedule(s, with_workspace && split_plan_bytes(s, sms) > 0, sms, p, sched, grid)) return -1;
  info[0] = grid;
  info[1] = sched;
  info[2] = p.pair_mode;
  info[3] = p.n_items;
  // the kernel's own walk: per CTA its pieces, per piece the ring positions
  // in load order, per position the tiles that take its K/V tile
  long long n = 0;
  for (int c = 0; c < grid; ++c) {
    const int np = sched == kSchedSplit ? num_pieces<true>(p, c, grid) : num_pieces<false>(p, c, grid);
    for (int k = 0; k < np; ++k) {
      Item it;
      const bool got = sched == kSchedSplit ? piece_at<true>(p, c, grid, k, it) : piece_at<false>(p, c, grid, k, it);
      if (!got) continue;
      for (int pos = 0; pos < it.uend - it.ubeg; ++pos) {
        const int j = sched == kSchedHalves ? ring_block<true>(it, pos) : ring_block<false>(it, pos);
        for (int t = 0; t < 2; ++t) {
          if (!it.valid[t] || j < it.beg[t] || j >= it.end[t]) continue;
          if (n < max_visits) {
            int *v = visits + 6 * n;
            v[0] = c;
            v[1] = it.item;
            v[2] = t;
            v[3] = it.bh[t];
            v[4] = it.row0[t];
            v[5] = j;
          }
          ++n;
        }
      }
    }
  }
  return n > 0x7fffffffLL ? -1 : static_cast<int>(n);
}

size_t attn_fwd_host_staging_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int with_lse) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return 0;
  const size_t q = static_cast<size_t>(B) * Hq * Nq * d * 2;
  const size_t kv = static_cast<size_t>(B) * Hkv * Nk * d * 2;
  const size_t lse = with_lse ? static_cast<size_t>(B) * Hq * Nq * 4 : 0;
  const size_t ws = (d == 64 || d == 128) && Hq % Hkv == 0 ? workspace_bytes(B, Hq, Hkv, Nq, Nk, d) : 0;
  return round_up256(q) * 2 + round_up256(kv) * 2 + round_up256(lse) + round_up256(ws);
}

attn_status_t attn_fwd_host(const void *Q_host, const void *K_host, const void *V_host, void *O_host,
                            float *LSE_host, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window,
                            float sm_scale, attn_dtype_t dtype, void *dev_buf, size_t dev_buf_bytes,
                            cudaStream_t stream) {
  if (!Q_host || !K_host || !V_host || !O_host || !dev_buf) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_buf) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype};
  const size_t need = attn_fwd_host_staging_bytes(B, Hq, Hkv, Nq, Nk, d, LSE_host != nullptr);
  if (need == 0 || dev_buf_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t q = static_cast<size_t>(B) * Hq * Nq * d * 2;
  const size_t kv = static_cast<size_t>(B) * Hkv * Nk * d * 2;
  uint8_t *base = static_cast<uint8_t *>(dev_buf);
  void *dQ = base;
  void *dK = base + round_up256(q);
  void *dV = base + round_up256(q) + round_up256(kv);
  void *dO = base + round_up256(q) + 2 * round_up256(kv);
  float *dL = LSE_host ? reinterpret_cast<float *>(base + 2 * round_up256(q) + 2 * round_up256(kv)) : nullptr;
  const size_t lse_bytes = LSE_host ? static_cast<size_t>(B) * Hq * Nq * 4 : 0;
  const size_t ws_bytes = (d == 64 || d == 128) && Hq % Hkv == 0 ? workspace_bytes(B, Hq, Hkv, Nq, Nk, d) : 0;
  void *dW = ws_bytes ? base + 2 * round_up256(q) + 2 * round_up256(kv) + round_up256(lse_bytes) : nullptr;
  attn_status_t st = validate(dQ, dK, dV, dO, dL, s);
  if (st != ATTN_OK) return st;
  if (current_device_sm_major(nullptr) != 10) return ATTN_ERR_UNSUPPORTED;
  // A call captured into a CUDA graph runs unpipelined: the shared copy
  // streams would otherwise stay in the capture until it ends, and another
  // thread's call could be captured with it.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return ATTN_ERR_CUDA;
  HostPiece pieces[kHostMaxPieces];
  const int np = cap == cudaStreamCaptureStatusNone ? host_pieces(s, pieces) : 0;
  if (np > 0)
    return host_pipelined(static_cast<const uint8_t *>(Q_host), static_cast<const uint8_t *>(K_host),
                          static_cast<const uint8_t *>(V_host), static_cast<uint8_t *>(O_host), LSE_host, s, pieces, np,
                          static_cast<uint8_t *>(dQ), static_cast<uint8_t *>(dK), static_cast<uint8_t *>(dV),
                          static_cast<uint8_t *>(dO), dL, stream);
  if (cudaMemcpyAsync(dQ, Q_host, q, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(dK, K_host, kv, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(dV, V_host, kv, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  st = run(dQ, dK, dV, dO, dL, s, dW, ws_bytes, stream);
  if (st != ATTN_OK) return st;
  if (cudaMemcpyAsync(O_host, dO, q, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dL && cudaMemcpyAsync(LSE_host, dL, static_cast<size_t>(B) * Hq * Nq * 4, cudaMemcpyDeviceToHost, stream) !=
                cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    return v == kErrDecBadIndex ? ATTN_ERR_DEVICE_ARG : ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

void attn_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns.store(ns ? ns : 2000000000ull); }

void attn_set_test_stall(int tiles) { g_stall_after.store(tiles < 0 ? -1 : tiles); }

const char *attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "kernel wait timed out";
    case ATTN_ERR_SCRATCH_LIMIT: return "shape exceeds the built-in decode scratch";
    case ATTN_ERR_DEVICE_ARG: return "a kernel found an out-of-range page index or sequence length";
  }
  return "unknown status";
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

int attn_bwd_cta_order(int B, int Hkv, int Nk, int sms, int *tiles, int max_ctas) {
  if (B <= 0 || Hkv <= 0 || Nk <= 0 || sms <= 0 || (max_ctas > 0 && tiles == nullptr)) return -1;
  const long long zk = static_cast<long long>(B) * Hkv, nkt = (static_cast<long long>(Nk) + 127) / 128;
  if (zk * nkt > 0x7fffffffLL) return -1;
  const int band = bwd_band(zk, nkt, sms);
  const int n = static_cast<int>(zk * nkt);
  for (int c = 0; c < n && c < max_ctas; ++c) {
    int bk = 0, kt = 0;
    bwd_cta_tile(c, band, static_cast<int>(zk), static_cast<int>(nkt), bk, kt);
    tiles[2 * c] = bk;
    tiles[2 * c + 1] = kt;
  }
  return n;
}

attn_status_t attn_empty_launch(int grid, int threads, size_t smem_bytes, cudaStream_t stream) {
  if (grid <= 0 || threads <= 0 || threads > 1024 || smem_bytes > 232448) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  static std::once_flag once[64];
  static bool ready[64];
  std::call_once(once[dev], [&] {
    ready[dev] = cudaFuncSetAttribute(attn::attn_empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      232448) == cudaSuccess;
    if (!ready[dev]) (void)cudaGetLastError();
  });
  if (!ready[dev]) return ATTN_ERR_CUDA;
  if (attn::launch_pdl(attn::attn_empty_kernel, dim3(static_cast<unsigned>(grid)), dim3(static_cast<unsigned>(threads)),
                       smem_bytes, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------- decode without allocation
// Scratch for attn_fwd_decode_noalloc: one fixed block per device, reserved
// while the library is loaded.  In host code `g_decode_scratch` only names the
// symbol; its device address comes from cudaGetSymbolAddress below.
namespace attn {
constexpr size_t kNoallocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

// Device address of the scratch block of the current device, looked up with
// that device current and kept once the lookup has succeeded.  nullptr if
// it failed; the failure is not kept (a later call tries again), and its
// error is cleared so that it is not reported by a later launch check.
static float *noalloc_scratch(int dev) {
  static std::mutex mu;
  static float *addr[64];
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) == cudaSuccess) {
      addr[dev] = static_cast<float *>(ptr);
    } else {
      (void)cudaGetLastError();
      return nullptr;
    }
  }
  return addr[dev];
}
}  // namespace attn

extern "C" {

attn_status_t attn_fwd_decode_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                                      int Hq, int Hkv, int Nq, int Nk, int d, int causal, int window,
                                      float sm_scale, attn_dtype_t dtype, cudaStream_t stream) {
  Shape s{B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype};
  attn_status_t st = validate(Q, K, V, O, LSE, s);
  if (st != ATTN_OK) return st;
  int dev = -1;
  if (current_device_sm_major(&dev) != 10) return ATTN_ERR_UNSUPPORTED;
  if (dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  const DecPlan pl = decode_plan(B, Hq, Hkv, Nq, Nk, d);
  if (pl.bytes == 0 || pl.bytes > kNoallocScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
  float *scratch = noalloc_scratch(dev);
  if (scratch == nullptr) return ATTN_ERR_CUDA;
  return dispatch_decode(Q, K, V, O, LSE, s, pl, scratch, stream);
}

}  // extern "C"

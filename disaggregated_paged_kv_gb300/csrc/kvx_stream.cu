// kvx_stream.cu -- layer-streamed, cancellable gather / scatter / transfer (sm_103a).
//
// "DistServe 完全拆解", 一次请求如何穿过 DistServe: prefill writes the prompt's KV layer by
// layer, and decode pulls layer j from prefill's layer j asynchronously, so most of the move
// can run while later layers are still being computed.  "穷人版 PD 分离", 最难的一个问题: a
// transfer the receiver has given up on must not land late in pages that were handed to
// another request, and the sender may only acknowledge the abort once it can prove that no
// write is still in flight.
//
// Items are (layer l, K/V, group of G tokens, m lanes each: the row kernel's shape for the
// row length) in layer-major order: item i has
// l = i / (kv_planes * groups); with one latent plane per layer (MLA) there is no K/V split.
// Two grids move them:
//
// Row grid (the default): one warp per item, one CTA per kWarps consecutive items of one
// layer (each layer's items padded to whole CTAs), as the row kernel of kvx_copy.cu.  Thread 0
// of a CTA waits for the CTA's layer while its warps load their slot indices; the rows are
// loaded once the layer is ready, and stored once the planner's verdict says every index is
// valid (and, with owner epochs, while the row's destination page still belongs to the
// request).  A CTA that gives up on a layer
// (the epoch word changed, or the wait ran past wait_ns) writes a tagged stop word into the
// device-memory mirror, so every CTA that starts later stops at once instead of waiting its
// own wait_ns again; CTAs below the stop layer still move their rows.  A one-thread epilogue
// kernel, launched behind the grid, folds the stop codes into the status and sets the
// "no further write" words once every CTA has finished.
//
// Persistent grid (kvx_stream_ctl::max_ctas > 0): at most max_ctas CTAs, one per SM, so that
// a producer running on the same GPU keeps the rest of it.  Blocks of consecutive items go to
// the CTAs in turn, and a CTA's workers (register warps; by default also TMA bulk-copy
// threads) take its items in order from a shared counter, so every worker reaches the layers
// in increasing order.  A worker entering layer l checks, once per CTA and layer (the first
// to arrive polls, the others read the CTA's shared bit of layer l), the epoch word and the
// ready word of layer l.  A CTA that stops still finishes the layers its workers had already
// entered, so every layer below the smallest stop layer of all CTAs holds every row.  On exit
// each CTA publishes its stop layer and flags its stop code, and the last CTA to finish folds
// the codes into the verdict and sets the "no further write" words.
//
// In both, polling is shared out so that the words of a slow producer (often pinned host
// memory, read over the CPU-GPU link) see few readers: pollers read the device-memory mirror
// of what some CTA has already seen on every round and the producer's words only on their
// first round and every 16th, except in the CTA that owns the layer's first item, which reads
// them on every round and copies what it sees into the mirror.  Every wait is bounded by
// wait_ns of %globaltimer and an iteration cap.  Waits only ever poll memory that the host or
// another engine writes: no CTA waits for another CTA or another kernel.
#include <algorithm>

#include "kvx_bulk_ops.cuh"
#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"
#include "kvx_stream_ops.cuh"

namespace kvx {
namespace {

using namespace ops;
using namespace sops;
using namespace bops;

constexpr int kWarps = kCopyThreads / 32;
// The persistent grid's CTAs: 32 warps, one CTA per SM, so that a grid capped at max_ctas
// CTAs keeps 64 KiB of rows in flight on each of its SMs.
constexpr int kPersistThreads = 1024;
constexpr int kPersistWarps = kPersistThreads / 32;

struct StreamArgs {
  CopyArgs c;   // sides, planes, buffer, status, slot lists (spec_src / spec_dst)
  StreamCtl k;
};

// ---- persistent grid, bulk form ----------------------------------------------------------
// The persistent grid's items with one token each, moved only by TMA bulk copies
// (kvx_bulk_ops.cuh), with kvx_set_copy_engine(KVX_ENGINE_BULK): every thread owns one
// kBulkStage-byte shared-memory stage and one mbarrier and moves whole rows (longer rows in
// pieces), global -> stage -> global, reusing its stage once the previous store has read it.
// A CTA of kBulkThreads threads keeps ~192 KiB in flight, yet it moves less per SM than the
// register form: each bulk operation has a fixed cost on the SM.  Layer waits, stops,
// page-owner checks and the exit protocol are the register form's.

constexpr int kBulkThreads = 96;
constexpr int kBulkStage = 2048;
constexpr size_t kBulkSmem = (size_t)kBulkThreads * kBulkStage + 8 * kBulkThreads;

// Bulk operations for bytes [x0, x0 + n) of a row of side s at `row` (row_base): one per
// contiguous piece, i.e. the whole range, or on an HND pool side the part of each head vector
// in the range.  Loads complete on bar; stores join the thread's open bulk async-group.
template <bool kHnd, bool kLoad>
__device__ __forceinline__ void bulk_row_range(const Side &s, bool pool, const char *row,
                                               int32_t x0, int32_t n, unsigned char *stage,
                                               uint64_t *bar) {
  if (!kHnd || !pool) {
    if constexpr (kLoad) bulk_load(stage, row + x0, (uint32_t)n, bar);
    else bulk_store(const_cast<char *>(row) + x0, stage, (uint32_t)n);
    return;
  }
  const int32_t seg = s.seg_bytes, end = x0 + n;
  for (int32_t x = x0; x < end;) {
    const int32_t h = x / seg, off = x - h * seg;
    const int32_t len = min(seg - off, end - x);
    const char *g = row + (int64_t)h * s.page_size * seg + off;
    if constexpr (kLoad) bulk_load(stage + (x - x0), g, (uint32_t)len, bar);
    else bulk_store(const_cast<char *>(g), stage + (x - x0), (uint32_t)len);
    x += len;
  }
}

template <bool kSrcHnd, bool kDstHnd>
__global__ void __launch_bounds__(kBulkThreads, 1)
    stream_bulk_kernel(const __grid_constant__ StreamArgs s) {
  extern __shared__ __align__(128) unsigned char smem[];  // stages | mbarriers
  __shared__ CtaState cs;
  const CopyArgs &a = s.c;
  const StreamCtl &k = s.k;
  const int32_t layers = k.layers;
  unsigned char *stage = smem + threadIdx.x * kBulkStage;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)kBulkThreads * kBulkStage) + threadIdx.x;
  if (threadIdx.x < kReadyWords) {
    cs.ready[threadIdx.x] = 0;
    cs.polling[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) {
    cs.stop = layers;
    cs.code = 0;
  }
  mbar_init(bar);
  __syncthreads();

  const int32_t R = a.row_bytes;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  // Blocks of kBulkThreads * k.block consecutive items go to the CTAs in turn; thread x of a
  // CTA takes items x, x + kBulkThreads, ... of each of its blocks, so its layers increase.
  const uint32_t bs = kBulkThreads * k.block;
  const uint32_t stride = gridDim.x * bs;
  int32_t lcur = -1;
  bool verdict_ok = false;  // this thread has seen the planner's verdict (every index valid)
  bool stuck = false;       // a bulk load did not complete in time (never expected)
  uint32_t parity = 0;
  // The token of item i: the row of layer i / per_layer, K or V, token r mod groups.
  auto token_of = [&](uint32_t i) -> int64_t {
    const uint32_t r = i % k.per_layer;
    return (int64_t)(r >= k.groups ? r - k.groups : r);
  };
  // Each item's slot indices are loaded one item ahead, while the previous row's bulk load is
  // in flight, so that a thread's rows follow each other without an index round trip between.
  uint32_t base = blockIdx.x * bs, j = 0;
  uint32_t i = base + threadIdx.x;
  int32_t si = 0, di = 0;
  if (i < k.items) {
    const int64_t t = token_of(i);
    si = sp ? a.spec_src[t] : (int32_t)t;
    di = dp ? a.spec_dst[t] : (int32_t)t;
  }
  while (i < k.items) {
    if (++j == k.block) {
      j = 0;
      base += stride;
    }
    const uint32_t inext = base + j * kBulkThreads + threadIdx.x;
    const int32_t l = (int32_t)(i / k.per_layer);
    if (l != lcur) {
      const bool owner = blockIdx.x == ((uint64_t)l * k.per_layer / bs) % gridDim.x;
      if (!wait_layer(k, l, owner, &cs)) break;
      fence_proxy_async_global();  // the layer's rows, seen by the acquire, reach the bulk loads
      lcur = l;
    }
    const uint32_t r = i - (uint32_t)l * k.per_layer;
    const int32_t p = k.kv_planes * l + (r >= k.groups ? 1 : 0);  // K or V (0 with MLA)
    const bool ok = (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
                    (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
    if (!ok) {  // the planner refuses the request: nothing may be stored
      pdl_wait();
      atomicMin(&cs.stop, 0);
      break;
    }
    const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
    const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
    char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
    const int32_t di_row = di;
    bool drop = false, stop = false;
    for (int32_t x0 = 0; x0 < R; x0 += kBulkStage) {
      const int32_t n = min(kBulkStage, R - x0);
      bulk_wait_read_all();  // the previous store has finished reading the stage
      mbar_expect_tx(bar, (uint32_t)n);
      bulk_row_range<kSrcHnd, true>(a.src, sp, srow, x0, n, stage, bar);
      if (x0 == 0 && inext < k.items) {  // the next item's indices, under this load
        const int64_t tn = token_of(inext);
        si = sp ? a.spec_src[tn] : (int32_t)tn;
        di = dp ? a.spec_dst[tn] : (int32_t)tn;
      }
      if (!verdict_ok) {  // the first row's load goes out before the planner's verdict
        pdl_wait();       // the planner has checked every index and written status[0]
        if (a.status[0] != KVX_OK) {
          atomicMin(&cs.stop, 0);
          stop = true;
        }
        verdict_ok = !stop;
      }
      if (!mbar_wait_bounded(bar, parity)) {
        stuck = true;
        give_up(&cs, l, KVX_ERR_TIMEOUT);
        break;
      }
      parity ^= 1u;
      if (stop) break;
      if (x0 == 0 && dp && k.page_epochs && !page_owned(k, di_row)) {
        // the page went to another request: the row is dropped and reported
        drop = true;
        atomicMax(&cs.code, (int32_t)KVX_ERR_CANCELLED);
        atomicMax(&a.status[1], layers - l);
      }
      if (drop) break;
      bulk_row_range<kDstHnd, false>(a.dst, dp, drow, x0, n, stage, bar);
      bulk_commit();
    }
    if (stuck || stop) break;
    i = inext;
  }
  if (stuck) (void)mbar_wait_bounded(bar, parity);  // let the late load land before leaving
  bulk_wait_all();             // every store of this thread is complete
  fence_proxy_async_global();  // ... and ordered before the generic-proxy release below

  // every thread's writes before this CTA's report; the last CTA's release covers all CTAs
  pdl_wait();  // the planner's status words are written before any CTA reports
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) persistent_cta_exit(a.status, k, cs, layers);
}

// ---- persistent grid ---------------------------------------------------------------------
// One 1024-thread CTA per SM (32 warps, 64 KiB of rows in flight per SM: a grid capped at
// max_ctas CTAs is bound by what each of its SMs keeps in flight).  Workers -- a warp moving a
// row group through registers, or with kTma one thread of the first kTmaWarps warps moving it
// by TMA bulk copies through its own 2 KiB shared-memory stage and mbarrier -- take the CTA's
// items from a shared counter, so the faster kind takes more while every worker's items (and
// so its layers) increase.  The two kinds are bound by different limits of an SM (rows in
// flight; a cost per bulk operation), so mixing them moves a little more per SM than either.
// kTma only for row groups of at most kBulkStage bytes moved in one register pass.

constexpr int kTmaWarps = 3;
constexpr int kTmaThreads = kTmaWarps * 32;
constexpr size_t kTmaSmem = (size_t)kTmaThreads * kBulkStage + 8 * kTmaThreads;

template <bool kSrcHnd, bool kDstHnd, bool kTma>
__global__ void __launch_bounds__(kPersistThreads, 1)
    stream_kernel(const __grid_constant__ StreamArgs s) {
  extern __shared__ __align__(128) unsigned char smem[];  // kTma: stages | mbarriers
  __shared__ CtaState cs;
  __shared__ uint32_t next;  // the CTA's next item (in its own order)
  const CopyArgs &a = s.c;
  const StreamCtl &k = s.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool tma = kTma && warp < kTmaWarps;
  const int32_t layers = k.layers;
  unsigned char *stage = smem + threadIdx.x * kBulkStage;  // TMA threads only
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)kTmaThreads * kBulkStage) + threadIdx.x;
  if (threadIdx.x < kReadyWords) {
    cs.ready[threadIdx.x] = 0;
    cs.polling[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) {
    cs.stop = layers;
    cs.code = 0;
    next = 0;
  }
  if (tma) mbar_init(bar);  // (never with !kTma)
  __syncthreads();

  const int32_t m = a.row_lanes, G = a.rows_per_warp;  // lanes per token, tokens per group
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  // Item q of this CTA: blocks of bs consecutive items go to the CTAs in turn.
  const uint32_t bs = kPersistWarps * k.block;
  auto item_of = [&](uint32_t q) -> uint32_t {
    return ((q / bs) * gridDim.x + blockIdx.x) * bs + q % bs;
  };
  int32_t lcur = -1;
  bool verdict_ok = false;  // this worker has seen the planner's verdict (every index valid)

  if (tma) {
    if constexpr (kTma) {  // (tma is false without kTma)
      bool stuck = false;  // a bulk load did not complete in time (never expected)
      uint32_t parity = 0;
      for (;;) {
        const uint32_t i = item_of(atomicAdd(&next, 1u));
        if (i >= k.items) break;
        const int32_t l = (int32_t)(i / k.per_layer);
        if (l != lcur) {
          const bool owner = blockIdx.x == ((uint64_t)l * k.per_layer / bs) % gridDim.x;
          if (!wait_layer(k, l, owner, &cs)) break;
          fence_proxy_async_global();  // the layer's rows, seen by the acquire, reach the loads
          lcur = l;
        }
        const uint32_t r = i - (uint32_t)l * k.per_layer;
        const int32_t kv = r >= k.groups ? 1 : 0;
        const int32_t p = k.kv_planes * l + kv;
        const int64_t t0 = (int64_t)(r - kv * k.groups) * G;
        const int32_t gn = (int32_t)min((int64_t)G, a.n_tokens - t0);  // tokens in this group
        const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
        bool bad = false;
        for (int32_t g = 0; g < gn; ++g) {
          const int32_t si = sp ? a.spec_src[t0 + g] : (int32_t)(t0 + g);
          const int32_t di = dp ? a.spec_dst[t0 + g] : (int32_t)(t0 + g);
          bad |= (sp && (si < 0 || (int64_t)si >= a.src.num_slots)) ||
                 (dp && (di < 0 || (int64_t)di >= a.dst.num_slots));
        }
        if (bad) {  // the planner refuses the request: nothing may be stored
          pdl_wait();
          atomicMin(&cs.stop, 0);
          break;
        }
        bulk_wait_read_all();  // the previous stores have finished reading the stage
        mbar_expect_tx(bar, (uint32_t)(gn * R));
        for (int32_t g = 0; g < gn; ++g) {
          const int32_t si = sp ? a.spec_src[t0 + g] : (int32_t)(t0 + g);
          const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
          bulk_row_range<kSrcHnd, true>(a.src, sp, srow, 0, R, stage + g * R, bar);
        }
        bool stop = false;
        if (!verdict_ok) {  // the first group's loads go out before the planner's verdict
          pdl_wait();
          if (a.status[0] != KVX_OK) {
            atomicMin(&cs.stop, 0);
            stop = true;
          }
          verdict_ok = !stop;
        }
        if (!mbar_wait_bounded(bar, parity)) {
          stuck = true;
          give_up(&cs, l, KVX_ERR_TIMEOUT);
          break;
        }
        parity ^= 1u;
        if (stop) break;
        for (int32_t g = 0; g < gn; ++g) {
          const int32_t di = dp ? a.spec_dst[t0 + g] : (int32_t)(t0 + g);
          if (dp && k.page_epochs && !page_owned(k, di)) {
            // the page went to another request: the row is dropped and reported
            atomicMax(&cs.code, (int32_t)KVX_ERR_CANCELLED);
            atomicMax(&a.status[1], layers - l);
            continue;
          }
          char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
          bulk_row_range<kDstHnd, false>(a.dst, dp, drow, 0, R, stage + g * R, bar);
        }
        bulk_commit();
      }
      if (stuck) (void)mbar_wait_bounded(bar, parity);  // let the late load land before leaving
      bulk_wait_all();             // every store of this thread is complete
      fence_proxy_async_global();  // ... and ordered before the generic-proxy release below
    }
  } else {
    const int32_t rl = lane / m, li = lane - rl * m;
    for (;;) {
      uint32_t q = 0;
      if (lane == 0) q = atomicAdd(&next, 1u);
      const uint32_t i = item_of(__shfl_sync(0xffffffffu, q, 0));
      if (i >= k.items) break;
      const int32_t l = (int32_t)(i / k.per_layer);
      if (l != lcur) {
        const bool owner = blockIdx.x == ((uint64_t)l * k.per_layer / bs) % gridDim.x;
        int32_t go = lane == 0 ? wait_layer(k, l, owner, &cs) : 0;
        go = __shfl_sync(0xffffffffu, go, 0);
        __syncwarp();  // lane 0's acquire orders every lane's loads of the layer
        if (!go) break;
        lcur = l;
      }
      const uint32_t r = i - (uint32_t)l * k.per_layer;
      const int32_t kv = r >= k.groups ? 1 : 0;
      const int64_t t = (int64_t)(r - kv * k.groups) * G + rl;
      const int32_t p = k.kv_planes * l + kv;
      bool ok = rl < G && t < a.n_tokens;
      const int64_t tt = ok ? t : 0;
      const int32_t si = sp ? a.spec_src[tt] : (int32_t)tt;
      const int32_t di = dp ? a.spec_dst[tt] : (int32_t)tt;
      ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
           (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
      const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
      const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
      char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
      // The first item's loads go out before the planner's verdict, like the row kernel's; a
      // lane range-checked its own indices above, so it never reads outside a pool.
#pragma unroll 1
      for (int32_t x0 = 0; x0 < vpr; x0 += kUnroll * m) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int32_t xv = x0 + li + u * m;
          if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
        }
        if (!verdict_ok) {
          pdl_wait();  // the planner has checked every index and written status[0]
          if (a.status[0] != KVX_OK) {
            if (lane == 0) atomicMin(&cs.stop, 0);
            break;
          }
          verdict_ok = true;
        }
        if (x0 == 0 && ok && dp && k.page_epochs && !page_owned(k, di)) {
          // the page went to another request: the row is dropped and reported
          ok = false;
          atomicMax(&cs.code, (int32_t)KVX_ERR_CANCELLED);
          atomicMax(&a.status[1], layers - l);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int32_t xv = x0 + li + u * m;
          if (ok && xv < vpr) st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, xv << 4)), v[u]);
        }
      }
      if (!verdict_ok) break;
    }
  }

  // every thread's writes before this CTA's report; the last CTA's release covers all CTAs
  pdl_wait();  // the planner's status words are written before any CTA reports
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) persistent_cta_exit(a.status, k, cs, layers);
}

// ---- row grid ------------------------------------------------------------------------

// kTail: rows of more than kUnroll * m vectors (more than one pass of the warp), a separate
// instance as in the row kernel so that the one-pass instances keep every value in registers.
template <bool kSrcHnd, bool kDstHnd, bool kTail>
__global__ void __launch_bounds__(kCopyThreads, kTail && (kSrcHnd || kDstHnd) ? 6 : 8)
    stream_row_kernel(const __grid_constant__ StreamArgs s) {
  __shared__ int32_t s_stop;  // 1: the CTA's layer moves, 0: it stopped
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the epilogue may queue
  const CopyArgs &a = s.c;
  const StreamCtl &k = s.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Each layer's items are padded to a multiple of kWarps, so the CTA's items all belong to
  // one layer: a layer that is late never holds back rows of an earlier one.
  const uint32_t i0 = blockIdx.x * kWarps;  // the CTA's first (padded) item
  const int32_t l = (int32_t)(i0 / k.per_layer_pad);
  const uint32_t r = i0 - (uint32_t)l * k.per_layer_pad + warp;
  const bool has = r < k.per_layer;
  const uint32_t rc = has ? r : 0;
  const int32_t m = a.row_lanes, G = a.rows_per_warp;  // lanes per token, tokens per warp
  const int32_t rl = lane / m;
  const int32_t kv = rc >= k.groups ? 1 : 0;  // K or V (always 0 with one latent plane)
  const int64_t t = (int64_t)(rc - kv * k.groups) * G + rl;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  // slot indices and their range checks go out before the wait
  bool ok = has && rl < G && t < a.n_tokens;
  const int64_t tt = ok ? t : 0;
  const int32_t si = sp ? a.spec_src[tt] : (int32_t)tt;
  const int32_t di = dp ? a.spec_dst[tt] : (int32_t)tt;
  ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
       (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
  if (threadIdx.x == 0) {
    int32_t go = 1;
    if (k.layer_ready || k.epoch_word) {
      // the CTA holding the layer's first items polls the producer on every round
      const bool owner = blockIdx.x == (uint32_t)((uint64_t)l * k.per_layer_pad / kWarps);
      const int32_t code = row_wait(k, l, owner);
      if (code) {
        go = 0;
        // The stop is recorded only once the planner has finished: a one-CTA validation
        // stores all four status words and would otherwise overwrite it.  This also keeps the
        // grid from completing before the planner, so the epilogue reads the final verdict.
        pdl_wait();
        atomicMax(&a.status[2], code);
        atomicMax(&a.status[1], k.layers - l);
      }
    }
    s_stop = go;
  }
  __syncthreads();  // thread 0's acquire of the layer orders every thread's row loads
  if (!s_stop) return;  // stopped: this CTA writes no row
  const int32_t p = k.kv_planes * l + kv;
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const int32_t li = lane - rl * m;
  const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
  const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
  char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int32_t xv = li + u * m;
    if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
  }
  pdl_wait();  // the planner has checked every index and written status[0]
  if (a.status[0] != KVX_OK || !ok) return;
  if (dp && k.page_epochs && !page_owned(k, di)) {
    // the page went to another request: the row is dropped and reported
    atomicMax(&a.status[2], (int32_t)KVX_ERR_CANCELLED);
    atomicMax(&a.status[1], k.layers - l);
    return;
  }
  // the stores of each pass, then (kTail) the next pass's loads
  const int32_t step = kUnroll * m;
#pragma unroll 1
  for (int32_t x0 = 0;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, xv << 4)), v[u]);
    }
    if constexpr (!kTail) break;
    x0 += step;
    if (x0 >= vpr) break;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
    }
  }
}

// Behind the row grid: once every CTA has finished (griddepcontrol.wait), the stop code joins
// the verdict and the "no further write" words are set.
__global__ void stream_done_kernel(int32_t *status, int32_t *host_done, int32_t layers) {
  pdl_wait();
  if (status[0] != KVX_OK) status[1] = layers;  // refused by the planner: nothing moved
  const int32_t code = status[2];
  if (code) atomicMax(&status[0], code);
  status[2] = 0;
  publish_done(&status[3], host_done);
}

template <bool kTail>
const void *stream_row_fn_of(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(stream_row_kernel<true, true, kTail>);
  if (sh) return reinterpret_cast<const void *>(stream_row_kernel<true, false, kTail>);
  if (dh) return reinterpret_cast<const void *>(stream_row_kernel<false, true, kTail>);
  return reinterpret_cast<const void *>(stream_row_kernel<false, false, kTail>);
}


template <bool kTma>
const void *stream_fn_of(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(stream_kernel<true, true, kTma>);
  if (sh) return reinterpret_cast<const void *>(stream_kernel<true, false, kTma>);
  if (dh) return reinterpret_cast<const void *>(stream_kernel<false, true, kTma>);
  return reinterpret_cast<const void *>(stream_kernel<false, false, kTma>);
}

const void *stream_fn(bool sh, bool dh, bool tma) {
  return tma ? stream_fn_of<true>(sh, dh) : stream_fn_of<false>(sh, dh);
}

const void *stream_bulk_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(stream_bulk_kernel<true, true>);
  if (sh) return reinterpret_cast<const void *>(stream_bulk_kernel<true, false>);
  if (dh) return reinterpret_cast<const void *>(stream_bulk_kernel<false, true>);
  return reinterpret_cast<const void *>(stream_bulk_kernel<false, false>);
}

}  // namespace

bool stream_tma_fits(const CopyArgs &c) {
  return (int64_t)c.rows_per_warp * c.row_bytes <= kBulkStage &&
         (c.row_bytes >> 4) <= kUnroll * c.row_lanes;  // one register pass per row
}

int stream_bulk_blocks_per_sm() {
  for (int v = 0; v < 4; ++v)
    if (cudaFuncSetAttribute(stream_bulk_fn(v & 1, v & 2), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kBulkSmem) != cudaSuccess)
      return 0;
  int nb = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &nb, stream_bulk_fn(false, false), kBulkThreads, kBulkSmem);
  return e == cudaSuccess ? nb : 0;
}

int stream_bulk_threads() { return kBulkThreads; }
int stream_threads() { return kPersistThreads; }

cudaError_t launch_stream_bulk(const CopyArgs &c, const StreamCtl &k, int grid, cudaStream_t s) {
  static thread_local StreamArgs args;  // ~4 KiB of plane pointers: keep it off the stack
  args.c = c;
  args.k = k;
  const bool sh = c.src.hnd && c.src.is_pool, dh = c.dst.hnd && c.dst.is_pool;
  void *params[] = {&args};
  return launch_pdl(stream_bulk_fn(sh, dh), dim3((unsigned)grid), dim3(kBulkThreads), params, s,
                    kBulkSmem);
}

int stream_blocks_per_sm() {
  for (int v = 0; v < 4; ++v)
    if (cudaFuncSetAttribute(stream_fn(v & 1, v & 2, true),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmaSmem) != cudaSuccess)
      return 0;
  int nb = 0, nb_tma = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, stream_fn(false, false, false),
                                                    kPersistThreads, 0) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb_tma, stream_fn(false, false, true),
                                                    kPersistThreads, kTmaSmem) != cudaSuccess)
    return 0;
  return std::min(nb, nb_tma);
}

void stream_sizes(StreamCtl &k, int64_t n_tokens, int32_t rows_per_warp) {
  const int64_t groups = (n_tokens + rows_per_warp - 1) / rows_per_warp;
  k.groups = (uint32_t)groups;
  k.per_layer = (uint32_t)(k.kv_planes * groups);
  k.items = (uint32_t)(k.kv_planes * groups * k.layers);
  k.per_layer_pad = (k.per_layer + kWarps - 1) / kWarps * kWarps;
}

cudaError_t launch_stream(const CopyArgs &c, const StreamCtl &k, int grid, bool tma,
                          cudaStream_t s) {
  static thread_local StreamArgs args;  // ~4 KiB of plane pointers: keep it off the stack
  args.c = c;
  args.k = k;
  const bool sh = c.src.hnd && c.src.is_pool, dh = c.dst.hnd && c.dst.is_pool;
  void *params[] = {&args};
  return launch_pdl(stream_fn(sh, dh, tma), dim3((unsigned)grid), dim3(kPersistThreads), params,
                    s, tma ? kTmaSmem : 0);
}

cudaError_t launch_stream_rows(const CopyArgs &c, const StreamCtl &k, cudaStream_t s) {
  static thread_local StreamArgs args;
  args.c = c;
  args.k = k;
  const bool sh = c.src.hnd && c.src.is_pool, dh = c.dst.hnd && c.dst.is_pool;
  const bool tail = (c.row_bytes >> 4) > kUnroll * c.row_lanes;  // more than one pass
  const void *fn = tail ? stream_row_fn_of<true>(sh, dh) : stream_row_fn_of<false>(sh, dh);
  void *params[] = {&args};
  cudaError_t e = cudaSuccess;
  if (k.items > 0) {
    e = launch_pdl(fn, dim3(k.per_layer_pad / kWarps * k.layers), dim3(kCopyThreads), params, s);
    if (e != cudaSuccess) return e;
  }
  return launch_stream_done(c.status, k.host_done, k.layers, s);
}

cudaError_t launch_stream_done(int32_t *status, int32_t *host_done, int32_t layers,
                               cudaStream_t s) {
  void *dparams[] = {&status, &host_done, &layers};
  return launch_pdl(reinterpret_cast<const void *>(stream_done_kernel), dim3(1), dim3(1), dparams, s);
}

}  // namespace kvx

// kvx_copy.cu -- the data movement of gather / scatter / transfer / batch (sm_103a).
//
// "穷人版 PD 分离", section "B300：让 P 直接写 D 的显存": one gather kernel moves every
// scattered source row straight into the destination's pages.  Here both pools live in one
// GB300's HBM, so the move is HBM-bound: every byte is read once and written once.
//
// Persistent grid (SM count x resident CTAs).  Work item w = (chunk c, plane p) with
// c = w / P, p = w % P, so the P planes of one chunk go to neighbouring warps and share the
// chunk record through L1.  One warp moves one work item: rows x R bytes as 16-byte vectors,
// kUnroll independent loads in flight per lane before the matching stores.  Loads bypass L1
// (each byte is read once); stores are streaming so the written rows do not evict the
// chunk table from L2.
//
// A chunk is "linear" when its rows are contiguous on both sides (token-row pools whose slot
// stride is the row size, and every transfer buffer): the warp copies one flat byte range.
// Otherwise (slot-major pools, HND pages) each 16-byte vector v is placed at
// (row j, head h, piece w) = (v / vps / H, v / vps % H, v % vps) on each side, vps = 16-byte
// pieces per head vector; on an HND side that turns [head][token] into [token][head], which
// is the fused permute of "mini-infer系统实战-18-PD 解耦" (KV 序列化格式选择).
#include <atomic>

#include "kvx_bulk_ops.cuh"
#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"

namespace kvx {
namespace {

using namespace ops;


// Common start of every copy kernel: checks the plan header (and, for single calls, the
// status word) and turns the per-tile chunk counts into each tile's first chunk in shared
// memory.  Returns the plan's chunk count, or -1 if this CTA must not move anything.
template <int THREADS>
__device__ __forceinline__ int32_t copy_prologue(const CopyArgs &a, int32_t *s_tile_base,
                                                 int32_t *s_warp, int32_t *s_ok) {
  constexpr int kWarps = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    int32_t ok = header_matches(a) ? 1 : 0;
    if (!ok && blockIdx.x == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_INVALID_ARG);
    if (ok && a.mode != kModeBatch && a.status[0] != KVX_OK) ok = 0;
    *s_ok = ok;
  }
  __syncthreads();
  if (!*s_ok) return -1;
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const int32_t *tiles = reinterpret_cast<const int32_t *>(a.ws + a.L.tiles_off);
  int32_t carry = 0;
  for (int32_t base = 0; base < nt; base += THREADS) {
    const int32_t t = base + tid;
    int32_t v = t < nt ? tiles[t] : 0;
    v = v < 0 ? 0 : (v > kTile ? kTile : v);  // never index past a tile's table
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int32_t wex = 0, tot = 0;
    for (int i = 0; i < kWarps; ++i) {
      if (i < warp) wex += s_warp[i];
      tot += s_warp[i];
    }
    if (t < nt) s_tile_base[t] = carry + wex + x - v;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) s_tile_base[nt] = carry;
  __syncthreads();
  return carry;
}

// Work item w = (chunk w / P, plane w % P): both sides' addresses and the row count.  False
// if the item belongs to a failed request of a batch.
__device__ __forceinline__ bool decode_item(const CopyArgs &a, uint32_t w,
                                            const int32_t *s_tile_base, int32_t nt, Addr &sa,
                                            Addr &da, int32_t &rows) {
  const uint32_t c = w / (uint32_t)a.planes;
  const int32_t p = (int32_t)(w - c * (uint32_t)a.planes);
  int32_t lo = 0, hi = nt;  // tile holding chunk c
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if ((uint32_t)s_tile_base[mid] <= c) lo = mid; else hi = mid;
  }
  const Chunk *chunks = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off);
  const Chunk ch = chunks[(int64_t)lo * kTile + (c - (uint32_t)s_tile_base[lo])];
  int32_t op = a.op;
  const char *bufp = a.buf;
  int64_t nreq = a.n_tokens;
  bool src_pool = a.src.is_pool, dst_pool = a.dst.is_pool;
  if (a.mode == kModeBatch) {
    if (a.status[1 + ch.req] != KVX_OK) return false;
    const kvx_request rq = a.reqs[ch.req];
    op = rq.op;
    bufp = a.buf + rq.buf_off;
    nreq = rq.n_tokens;
    src_pool = (op == KVX_OP_GATHER || op == KVX_OP_TRANSFER);
    dst_pool = (op == KVX_OP_SCATTER || op == KVX_OP_TRANSFER);
  }
  const int32_t R = a.row_bytes;
  const char *buf_plane = bufp + (int64_t)p * nreq * R;
  sa = side_addr(a.src, src_pool, a.src_planes[p], ch.src, buf_plane, R);
  da = side_addr(a.dst, dst_pool, a.dst_planes[p], ch.dst, buf_plane, R);
  rows = ch.rows;
  return true;
}

// Register path: one warp per work item.  kLinear: the host has seen that every chunk is
// linear on both sides (token-row pools with dense rows, and buffers), so the per-vector
// placement path is compiled out.
template <bool kLinear>
__global__ void __launch_bounds__(kCopyThreads, 4) copy_kernel(const __grid_constant__ CopyArgs a) {
  extern __shared__ int32_t s_tile_base[];  // n_tiles + 1 entries
  __shared__ int32_t s_warp[kCopyThreads / 32];
  __shared__ int32_t s_ok;

  pdl_wait();  // the planner's tables must be complete
  const int32_t C = copy_prologue<kCopyThreads>(a, s_tile_base, s_warp, &s_ok);
  if (C < 0) return;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const uint32_t total = (uint32_t)C * (uint32_t)a.planes;
  const int32_t R = a.row_bytes;
  const uint32_t nwarps = gridDim.x * (kCopyThreads / 32);
  for (uint32_t w = blockIdx.x * (kCopyThreads / 32) + warp; w < total; w += nwarps) {
    Addr sa, da;
    int32_t rows;
    if (!decode_item(a, w, s_tile_base, nt, sa, da, rows)) continue;
    const int32_t nvec = rows * (R >> 4);
    if (kLinear) {
      copy_linear(sa.base, const_cast<char *>(da.base), nvec, lane);
    } else {
      const bool linear = sa.head == a.seg_bytes && da.head == a.seg_bytes &&
                          (rows == 1 || (sa.row == R && da.row == R));
      if (linear)
        copy_linear(sa.base, const_cast<char *>(da.base), nvec, lane);
      else
        copy_pieces(sa, da, nvec, a.seg_bytes >> 4, a.heads, lane);
    }
  }
}

// Lean register path for the common case: one request (gather, scatter or transfer, from a
// slot list or a run list) whose chunks are all linear.  Only base pointers are kept per side
// (no row / head strides, no batch records), so the kernel fits in 32 registers and an SM holds
// 8 CTAs = 64 warps: twice the 16-byte loads in flight of the general kernel.
__device__ __forceinline__ const char *lin_addr(const Side &s, bool pool, const char *plane,
                                                int32_t idx, const char *buf_plane,
                                                int32_t row_bytes) {
  return pool ? plane + (int64_t)idx * s.slot_stride : buf_plane + (int64_t)idx * row_bytes;
}

__global__ void __launch_bounds__(kCopyThreads, 8)
    copy_lean_kernel(const __grid_constant__ CopyArgs a) {
  extern __shared__ int32_t s_tile_base[];  // n_tiles + 1 entries
  __shared__ int32_t s_warp[kCopyThreads / 32];
  __shared__ int32_t s_ok;

  pdl_wait();
  const int32_t C = copy_prologue<kCopyThreads>(a, s_tile_base, s_warp, &s_ok);
  if (C < 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const uint32_t P = (uint32_t)a.planes;
  const uint32_t total = (uint32_t)C * P;
  const int32_t R = a.row_bytes;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const Chunk *chunks = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off);
  const uint32_t nwarps = gridDim.x * (kCopyThreads / 32);
  for (uint32_t w = blockIdx.x * (kCopyThreads / 32) + warp; w < total; w += nwarps) {
    const uint32_t c = w / P;
    const int32_t p = (int32_t)(w - c * P);
    int32_t lo = 0, hi = nt;
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if ((uint32_t)s_tile_base[mid] <= c) lo = mid; else hi = mid;
    }
    const Chunk ch = chunks[(int64_t)lo * kTile + (c - (uint32_t)s_tile_base[lo])];
    const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
    const char *src = lin_addr(a.src, sp, a.src_planes[p], ch.src, buf_plane, R);
    char *dst = const_cast<char *>(lin_addr(a.dst, dp, a.dst_planes[p], ch.dst, buf_plane, R));
    copy_linear(src, dst, ch.rows * (R >> 4), lane);
  }
}

// Row path.  Non-persistent grid: one warp per (group of G consecutive tokens, plane), plane
// major -- a CTA's warps take consecutive token groups of one plane and neighbouring CTAs the
// next ones, so the grid streams through one plane's rows at a time (a buffer side is read or
// written front to back; page runs of an HND side stay within one CTA) -- with m lanes per
// token (m * G <= 32; lanes past m * G idle).  Each lane moves vectors
// li, li + m, li + 2m, ... of its token's row, kUnroll of them in flight per pass.  The host
// picks (m, G) for the row length (row_shape): as many row bytes in flight per pass as the
// lanes allow, in as few passes as possible -- a 2 KiB row takes a whole warp (m = 32, one
// pass), 576-byte rows go three to a warp with nine lanes each (one pass; sixteen lanes for
// two rows would leave 44 % of the slots empty).  The hardware keeps every SM full of
// short-lived 32-register warps (64 per SM).  Two sources of indices:
//  - speculative (one-shot calls, slot lists at hand): a lane range-checks its token and issues
//    its loads before griddepcontrol.wait, so the planner runs under the first wave of loads;
//    the stores wait for the planner's verdict, so the move stays all-or-nothing;
//  - plan (G == 1, one-row chunks): after griddepcontrol.wait a warp reads chunk t of the plan
//    (one chunk per token), including the request record of a batch.
// Byte x of a token's row: on a token-row side the row is contiguous; on an HND side it sits at
// head x / seg, offset x % seg of the token's page -- the fused [heads, tokens, dim] <->
// [tokens, heads, dim] permute (row_base / row_byte).

// The final status into the caller's pinned host word (kvx_submit), visible to the host once
// the stream has reached the end of the call.
__device__ __forceinline__ void report_host_status(int32_t *host_status, int32_t v) {
  *reinterpret_cast<volatile int32_t *>(host_status) = v;
  __threadfence_system();
}

// Whether this thread (the first of the grid) reports to the host status word.
__device__ __forceinline__ bool reports(const CopyArgs &a) {
  return a.host_status != nullptr && blockIdx.x == 0 && threadIdx.x == 0;
}

// kSpec: indices from the slot lists (one-shot, single request); otherwise from the plan.
// kTail: rows of more than kUnroll * m vectors, moved in further passes; a separate instance so
// that the one-pass kernels keep every value in registers.
template <bool kSrcHnd, bool kDstHnd, bool kSpec, bool kTail>
__global__ void __launch_bounds__(kCopyThreads, kTail && (kSrcHnd || kDstHnd) ? 6 : 8)
    copy_row_kernel(const __grid_constant__ CopyArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t pc = blockIdx.x / a.row_blocks;  // plane-major (CopyArgs::row_blocks)
  const int32_t p = (int32_t)pc;
  const uint32_t q = (blockIdx.x - pc * a.row_blocks) * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const int32_t m = a.row_lanes;      // lanes per token
  const int32_t G = a.rows_per_warp;  // tokens per warp
  const int64_t t0 = (int64_t)q * G;
  if (t0 >= a.n_tokens) return;
  const int32_t rl = lane / m;        // this lane's token within the group
  const int32_t li = lane - rl * m;
  const int64_t t = t0 + rl;
  const int32_t R = a.row_bytes, vpr = R >> 4;
  bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const char *bufp = a.buf;
  int64_t nreq = a.n_tokens;
  int32_t si, di;
  bool ok = rl < G && t < a.n_tokens;
  if constexpr (kSpec) {
    const int64_t tt = ok ? t : t0;
    si = sp ? a.spec_src[tt] : (int32_t)tt;
    di = dp ? a.spec_dst[tt] : (int32_t)tt;
    ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
         (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
  } else {
    pdl_wait();
    if (!header_matches(a)) {
      if (q == 0 && p == 0 && lane == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_INVALID_ARG);
      return;
    }
    const Chunk ch = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off)[t0];  // G == 1
    if (a.mode == kModeBatch) {
      if (a.status[1 + ch.req] != KVX_OK) return;
      const kvx_request rq = a.reqs[ch.req];
      sp = (rq.op == KVX_OP_GATHER || rq.op == KVX_OP_TRANSFER);
      dp = (rq.op == KVX_OP_SCATTER || rq.op == KVX_OP_TRANSFER);
      bufp = a.buf + rq.buf_off;
      nreq = rq.n_tokens;
    } else if (a.status[0] != KVX_OK) {
      return;
    }
    si = ch.src;
    di = ch.dst;
  }
  const char *buf_plane = bufp + (int64_t)p * nreq * R;
  const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
  char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
  uint4 r[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int32_t xv = li + u * m;
    if (ok && xv < vpr) r[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
  }
  if constexpr (kSpec) {
    pdl_wait();  // the planner has checked every index of the request
    const int32_t verdict = a.status[0];
    if (verdict != KVX_OK) {
      if (reports(a)) report_host_status(a.host_status, verdict);
      return;
    }
  }
  if (kSpec && reports(a) && !ok) report_host_status(a.host_status, KVX_OK);
  if (!ok) return;
  // the stores of each pass, then (kTail) the next pass's loads
  const int32_t step = kUnroll * m;
#pragma unroll 1
  for (int32_t x0 = 0;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, xv << 4)), r[u]);
    }
    if constexpr (!kTail) break;
    x0 += step;
    if (x0 >= vpr) break;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) r[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
    }
  }
  if (kSpec && reports(a)) report_host_status(a.host_status, KVX_OK);
}

// ---- bulk (TMA) path ----------------------------------------------------------------------
// For linear chunks only.  Every thread owns one kBulkStage-byte shared-memory stage and one
// mbarrier: cp.async.bulk global -> shared, then shared -> global, and the stage is reused once
// that store has read it (kvx_bulk_ops.cuh).  A wait that exceeds kBulkWaitLimitNs (never
// expected) sets KVX_ERR_TIMEOUT, drains this thread's transfers and ends the thread.

using namespace bops;

template <int kThreads, int kStage>
__global__ void __launch_bounds__(kThreads) copy_bulk_kernel(const __grid_constant__ CopyArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];  // stages | mbarriers | tile bases
  __shared__ int32_t s_warp[kThreads / 32];
  __shared__ int32_t s_ok;
  unsigned char *stage = smem + threadIdx.x * kStage;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kThreads * kStage) + threadIdx.x;
  int32_t *s_tile_base = reinterpret_cast<int32_t *>(smem + kThreads * kStage + 8 * kThreads);

  pdl_wait();
  const int32_t C = copy_prologue<kThreads>(a, s_tile_base, s_warp, &s_ok);
  if (C < 0) return;
  mbar_init(bar);

  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const uint32_t total = (uint32_t)C * (uint32_t)a.planes;
  const uint32_t R = (uint32_t)a.row_bytes;
  uint32_t parity = 0;
  bool failed = false;
  for (uint32_t w = blockIdx.x * kThreads + threadIdx.x; w < total && !failed;
       w += gridDim.x * kThreads) {
    Addr sa, da;
    int32_t rows;
    if (!decode_item(a, w, s_tile_base, nt, sa, da, rows)) continue;
    const uint32_t bytes = (uint32_t)rows * R;
    for (uint32_t off = 0; off < bytes; off += kStage) {
      const uint32_t n = bytes - off < (uint32_t)kStage ? bytes - off : (uint32_t)kStage;
      bulk_wait_read_all();  // the previous store has finished reading this stage
      mbar_expect_tx(bar, n);
      bulk_load(stage, sa.base + off, n, bar);
      if (!mbar_wait_bounded(bar, parity)) {
        failed = true;
        break;
      }
      parity ^= 1u;
      bulk_store(const_cast<char *>(da.base) + off, stage, n);
      bulk_commit();
    }
  }
  if (failed) {
    atomicMax(&a.status[0], (int32_t)KVX_ERR_TIMEOUT);
    (void)mbar_wait_bounded(bar, parity);  // let the outstanding load land before leaving
  }
  bulk_wait_all();  // every store complete before the kernel ends
}

constexpr int kBulkThreads = kBulkThreadsPerCta;
constexpr int kBulkStage = 2048;

size_t bulk_smem_bytes(int32_t n_tiles) {
  return (size_t)kBulkThreads * kBulkStage + 8 * kBulkThreads + 4 * (size_t)(n_tiles + 1);
}

}  // namespace

std::atomic<int32_t> g_engine{KVX_ENGINE_AUTO};

bool side_is_linear(const Side &s, int32_t row_bytes) {
  return !s.is_pool || (!s.hnd && s.slot_stride == row_bytes);
}

bool copy_is_linear(const CopyArgs &a) {
  // in a batch either side may be a pool or the buffer; both must then be linear as a pool
  if (a.mode == kModeBatch)
    return !a.src.hnd && a.src.slot_stride == a.row_bytes && !a.dst.hnd &&
           a.dst.slot_stride == a.row_bytes;
  return side_is_linear(a.src, a.row_bytes) && side_is_linear(a.dst, a.row_bytes);
}

CopyVariant copy_variant(const CopyArgs &a, int32_t engine) {
  const bool linear = copy_is_linear(a);
  if (linear && engine == KVX_ENGINE_BULK) return kVariantBulk;
  // the row kernel takes every one-shot request (slot lists at hand) and every plan with
  // one-row chunks; multi-row plans keep the persistent kernels
  const bool spec = a.spec_src != nullptr || a.spec_dst != nullptr;
  if ((spec && a.mode == kModeSlots) || a.chunk_rows == 1) return kVariantRow;
  if (!linear) return kVariantGeneral;
  return a.mode == kModeBatch ? kVariantLinear : kVariantLean;
}

// Most passes row_shape lets a warp make over its rows.  Measured on 16,384 random tokens x 27
// planes: 1152-byte rows move at 80 % of the copy peak in one pass of a whole warp and at 90 %
// three to a warp with ten lanes each in two passes; three or more passes (fewer lanes, more
// rows) fell to 71 % and below, as did 576-byte rows (76 % in one pass, 45 % in three).
constexpr int32_t kMaxRowPasses = 2;

void row_shape(const CopyArgs &a, int32_t *lanes, int32_t *rows) {
  *lanes = 32;
  *rows = 1;
  // plans are read one chunk (= one token) per warp
  if (!(a.spec_src != nullptr || a.spec_dst != nullptr)) return;
  row_shape_for(a.row_bytes, lanes, rows);
}

void row_shape_for(int64_t row_bytes, int32_t *lanes, int32_t *rows) {
  *lanes = 32;
  *rows = 1;
  // m lanes per token, G = 32 / m tokens per warp, passes = ceil(vpr / (kUnroll m)): the most
  // row vectors per pass (G vpr / passes), then the fewest passes, then the most lanes.  A
  // shape of several passes needs m >= 8 (each pass takes at least 128 bytes of every row).
  const int64_t vpr = row_bytes >> 4;
  int64_t best_num = 0, best_den = 1, best_passes = 0;
  for (int32_t m = 32; m >= 1; --m) {
    const int64_t G = 32 / m;
    const int64_t passes = (vpr + (int64_t)kUnroll * m - 1) / ((int64_t)kUnroll * m);
    if (m < 32 && (passes > kMaxRowPasses || (passes > 1 && m < 8))) continue;
    const int64_t num = G * vpr;  // vectors per pass = num / passes
    const bool better = num * best_den > best_num * passes ||
                        (num * best_den == best_num * passes && passes < best_passes);
    if (best_passes == 0 || better) {
      best_num = num;
      best_den = passes;
      best_passes = passes;
      *lanes = m;
      *rows = (int32_t)G;
    }
  }
}

int64_t row_grid(CopyArgs &a) {
  const int64_t groups = (a.n_tokens + a.rows_per_warp - 1) / a.rows_per_warp;
  const int64_t wpb = kCopyThreads / 32;
  a.row_blocks = (uint32_t)((groups + wpb - 1) / wpb);
  return (int64_t)a.row_blocks * a.planes;
}

template <bool kSpec, bool kTail>
const void *row_fn_of(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(copy_row_kernel<true, true, kSpec, kTail>);
  if (sh) return reinterpret_cast<const void *>(copy_row_kernel<true, false, kSpec, kTail>);
  if (dh) return reinterpret_cast<const void *>(copy_row_kernel<false, true, kSpec, kTail>);
  return reinterpret_cast<const void *>(copy_row_kernel<false, false, kSpec, kTail>);
}

const void *row_fn(const CopyArgs &a) {
  // an HND side only matters where the request uses it as a pool
  const bool sh = a.src.hnd && (a.src.is_pool || a.mode == kModeBatch);
  const bool dh = a.dst.hnd && (a.dst.is_pool || a.mode == kModeBatch);
  const bool spec = a.spec_src != nullptr || a.spec_dst != nullptr;
  const bool tail = (a.row_bytes >> 4) > kUnroll * a.row_lanes;  // more than one pass
  if (spec) return tail ? row_fn_of<true, true>(sh, dh) : row_fn_of<true, false>(sh, dh);
  return tail ? row_fn_of<false, true>(sh, dh) : row_fn_of<false, false>(sh, dh);
}

int variant_threads(CopyVariant v) { return v == kVariantBulk ? kBulkThreads : kCopyThreads; }

size_t variant_smem(CopyVariant v, int32_t n_tiles) {
  if (v == kVariantRow) return 0;
  return v == kVariantBulk ? bulk_smem_bytes(n_tiles) : sizeof(int32_t) * (size_t)(n_tiles + 1);
}

const void *variant_fn(CopyVariant v) {
  switch (v) {
    case kVariantLean: return reinterpret_cast<const void *>(copy_lean_kernel);
    case kVariantLinear: return reinterpret_cast<const void *>(copy_kernel<true>);
    case kVariantGeneral: return reinterpret_cast<const void *>(copy_kernel<false>);
    case kVariantRow: return reinterpret_cast<const void *>(copy_row_kernel<false, false, true, false>);
    default: return reinterpret_cast<const void *>(copy_bulk_kernel<kBulkThreads, kBulkStage>);
  }
}

int variant_blocks_per_sm(CopyVariant v, int32_t n_tiles) {
  const void *fn = variant_fn(v);
  if (v == kVariantBulk &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bulk_smem_bytes(kMaxTiles)) != cudaSuccess)
    return 0;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, variant_threads(v),
                                                    variant_smem(v, n_tiles)) != cudaSuccess)
    return 0;
  return nb;
}

int copy_kernel_list(const void **out, int max) {
  const void *k[20];
  int n = 0;
  for (int sh = 0; sh < 2; ++sh)
    for (int dh = 0; dh < 2; ++dh) {
      k[n++] = row_fn_of<true, false>(sh, dh);
      k[n++] = row_fn_of<true, true>(sh, dh);
      k[n++] = row_fn_of<false, false>(sh, dh);
      k[n++] = row_fn_of<false, true>(sh, dh);
    }
  k[n++] = variant_fn(kVariantLean);
  k[n++] = variant_fn(kVariantLinear);
  k[n++] = variant_fn(kVariantGeneral);
  k[n++] = variant_fn(kVariantBulk);
  return kernel_list_out(k, n, out, max);
}

cudaError_t launch_copy(const CopyArgs &a, CopyVariant v, int grid, cudaStream_t s) {
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  void *args[] = {const_cast<CopyArgs *>(&a)};
  const void *fn = v == kVariantRow ? row_fn(a) : variant_fn(v);
  return launch_pdl(fn, dim3((unsigned)grid), dim3(variant_threads(v)), args, s,
                    variant_smem(v, nt));
}

}  // namespace kvx

extern "C" kvx_status kvx_set_copy_engine(int32_t engine) {
  if (engine < KVX_ENGINE_AUTO || engine > KVX_ENGINE_BULK) return KVX_ERR_INVALID_ARG;
  kvx::g_engine.store(engine, std::memory_order_relaxed);
  return KVX_OK;
}

extern "C" int32_t kvx_get_copy_engine(void) {
  return kvx::g_engine.load(std::memory_order_relaxed);
}

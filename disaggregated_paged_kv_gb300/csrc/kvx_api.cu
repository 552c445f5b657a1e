// kvx_api.cu -- libkvx's C ABI: layout handles, host-side validation, and the launches.
//
// Every entry point checks what the host can see (pointers, alignment, sizes, layout
// agreement, overlapping memory, workspace size) and returns at once with nothing enqueued
// if it fails; data-dependent checks happen in the planner and end up in the device status
// word ("穷人版 PD 分离", section "最难的一个问题": the client learns of a failure right away
// and no half-written KV is left behind).
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "kvx_internal.cuh"
#include "kvx_reshard.cuh"

struct kvx_layout {
  int32_t num_layers, kv_heads, head_dim, elem, kind, page_size;
  int32_t kv_planes;  // planes per layer: 2 (K, V) or 1 (MLA latent)
  int32_t vec;        // widest access (16, 8, 4, 2, 1 bytes) every row and head vector allows
  int32_t planes;
  int64_t num_slots;
  int64_t row_bytes, seg_bytes;
  int64_t slot_stride;  // NHD
  int64_t page_bytes;   // HND
  int64_t extent;       // bytes one plane spans from its start
  uintptr_t lo, hi;     // envelope of all planes
  uintptr_t plane[KVX_MAX_PLANES];
};

namespace {

thread_local int32_t g_last_cuda = 0;

kvx_status cuda_fail(cudaError_t e) {
  g_last_cuda = (int32_t)e;
  return KVX_ERR_CUDA;
}

int elem_bytes_of(int32_t dtype) {
  switch (dtype) {
    case KVX_F16:
    case KVX_BF16:
      return 2;
    case KVX_F32:
      return 4;
    case KVX_FP8:
      return 1;
    default:
      return 0;
  }
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
  return a0 < b1 && b0 < a1;
}

bool layout_overlaps_range(const kvx_layout *l, uintptr_t b0, uintptr_t b1) {
  if (!ranges_overlap(l->lo, l->hi, b0, b1)) return false;
  for (int p = 0; p < l->planes; ++p)
    if (ranges_overlap(l->plane[p], l->plane[p] + l->extent, b0, b1)) return true;
  return false;
}

bool layouts_overlap(const kvx_layout *a, const kvx_layout *b) {
  if (!ranges_overlap(a->lo, a->hi, b->lo, b->hi)) return false;
  for (int p = 0; p < a->planes; ++p)
    if (layout_overlaps_range(b, a->plane[p], a->plane[p] + a->extent)) return true;
  return false;
}

bool same_rows(const kvx_layout *a, const kvx_layout *b) {
  return a->num_layers == b->num_layers && a->kv_planes == b->kv_planes &&
         a->kv_heads == b->kv_heads && a->head_dim == b->head_dim && a->elem == b->elem;
}

int32_t log2_exact(int64_t v) {
  if (v <= 0 || (v & (v - 1)) != 0) return -1;
  int32_t sh = 0;
  while ((int64_t)1 << sh < v) ++sh;
  return sh;
}

// Largest power of two, at most 16, that divides x (x > 0).
int32_t pow2_align(int64_t x) {
  int32_t a = 16;
  while (a > 1 && x % a != 0) a >>= 1;
  return a;
}

kvx::Side pool_side(const kvx_layout *l) {
  kvx::Side s = {};
  s.is_pool = 1;
  s.hnd = l->kind == KVX_HND_PAGED ? 1 : 0;
  s.page_size = s.hnd ? l->page_size : 1;
  s.seg_bytes = (int32_t)l->seg_bytes;
  s.num_slots = l->num_slots;
  s.slot_stride = l->slot_stride;
  s.page_bytes = l->page_bytes;
  s.seg_shift = log2_exact(s.seg_bytes);
  s.ps_shift = log2_exact(s.page_size);
  return s;
}

kvx::Side buffer_side(int64_t seg_bytes) {
  kvx::Side s = {};
  s.is_pool = 0;
  s.hnd = 0;
  s.page_size = 1;
  s.seg_bytes = (int32_t)seg_bytes;
  s.seg_shift = log2_exact(seg_bytes);
  s.ps_shift = 0;
  return s;
}

int32_t chunk_rows_for(int64_t row_bytes) {
  int64_t m = kvx::kDefaultChunkBytes / row_bytes;
  if (m < 1) m = 1;
  if (m > kvx::kTile) m = kvx::kTile;
  return (int32_t)m;
}

struct DeviceInfo {
  int sms = 0;
  int bps[kvx::kNumVariants] = {};        // resident CTAs per SM per copy variant (largest plan)
  int bps_small[kvx::kNumVariants] = {};  // the same for plans of <= kBulkSmallTiles tiles
  int bps_fused_linear = 0;               // one-launch path, linear rows
  int bps_fused_general = 0;              // one-launch path, general placement
  int bps_stream = 0;                     // layer-streamed copy
  int bps_stream_bulk = 0;                // layer-streamed copy, bulk (TMA) form
  int bps_reshard_persist = 0;            // layer-streamed reshard, capped persistent grid
};

std::atomic<int32_t> g_fused_max{0};  // measured: planner + row kernel is faster
std::atomic<int32_t> g_check_dup{0};  // kvx_set_check_duplicates

kvx_status device_info(DeviceInfo *out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return KVX_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].sms == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo d;
    d.sms = sms;
    for (int v = 0; v < kvx::kNumVariants; ++v) {
      d.bps[v] = kvx::variant_blocks_per_sm((kvx::CopyVariant)v, kvx::kMaxTiles);
      d.bps_small[v] = kvx::variant_blocks_per_sm((kvx::CopyVariant)v, kvx::kBulkSmallTiles);
      if (d.bps[v] <= 0 || d.bps_small[v] <= 0) {
        e = cudaGetLastError();
        return cuda_fail(e != cudaSuccess ? e : cudaErrorUnknown);
      }
    }
    d.bps_fused_linear = kvx::fused_blocks_per_sm(true);
    d.bps_fused_general = kvx::fused_blocks_per_sm(false);
    d.bps_stream = kvx::stream_blocks_per_sm();
    d.bps_stream_bulk = kvx::stream_bulk_blocks_per_sm();
    d.bps_reshard_persist = kvx::reshard_persist_blocks_per_sm();
    if (d.bps_fused_linear <= 0 || d.bps_fused_general <= 0 || d.bps_stream <= 0 ||
        d.bps_stream_bulk <= 0 || d.bps_reshard_persist <= 0) {
      e = cudaGetLastError();
      return cuda_fail(e != cudaSuccess ? e : cudaErrorUnknown);
    }
    cache[dev] = d;
  }
  *out = cache[dev];
  return KVX_OK;
}

// What a plan or a copy is about: the two sides and the token space.
struct Call {
  int32_t mode = kvx::kModeSlots;
  int32_t op = KVX_OP_GATHER;
  const kvx_layout *src = nullptr, *dst = nullptr;  // pools (nullptr = buffer side)
  const kvx_layout *shape = nullptr;                // the layout that fixes P and R
  int64_t n_tokens = 0;
  int32_t n_segs = 0;
  int32_t n_status = 1;
  // Geometry of the rows moved: the shape layout's whole rows, or (kvx_move_heads) a range of
  // heads of each side, reached by offsetting every plane base of that side.
  int32_t planes = 0;
  int32_t heads = 0;
  int64_t row_bytes = 0, seg_bytes = 0;
  int64_t src_head_off = 0, dst_head_off = 0;
  // Widest access every row, head vector and plane of the call allows.  Below 16 bytes the
  // call takes the narrow row kernel with one row per plan chunk.
  int32_t vec = 16;
  // The call's options (its flags word, or the process-wide settings for KVX_DEFAULTS).
  bool check_dup = false;
  int32_t engine = KVX_ENGINE_AUTO;
  int32_t fused_max = 0;
};

// Resolves a call's flags word into c's options.  KVX_ERR_INVALID_ARG for unknown bits or both
// engines at once.
kvx_status apply_flags(Call &c, uint32_t flags) {
  if (flags == KVX_DEFAULTS) {
    c.check_dup = g_check_dup.load(std::memory_order_relaxed) != 0;
    c.engine = kvx_get_copy_engine();
    c.fused_max = g_fused_max.load(std::memory_order_relaxed);
    return KVX_OK;
  }
  const uint32_t known = KVX_CHECK_DUP | KVX_USE_REGISTERS | KVX_USE_BULK | KVX_ONE_LAUNCH;
  if ((flags & ~known) != 0 || ((flags & KVX_USE_REGISTERS) && (flags & KVX_USE_BULK)))
    return KVX_ERR_INVALID_ARG;
  c.check_dup = (flags & KVX_CHECK_DUP) != 0;
  c.engine = (flags & KVX_USE_BULK) ? KVX_ENGINE_BULK
             : (flags & KVX_USE_REGISTERS) ? KVX_ENGINE_REGISTERS : KVX_ENGINE_AUTO;
  c.fused_max = (flags & KVX_ONE_LAUNCH) ? KVX_FUSED_MAX_TOKENS : 0;
  return KVX_OK;
}

// The access width a pool side allows: its own, and its head vectors' (the per-head
// placement of the fast kernels moves 16-byte pieces of head vectors).
int32_t side_vec(const kvx_layout *l) {
  return l ? std::min(l->vec, pow2_align(l->seg_bytes)) : 16;
}

void set_whole_rows(Call &c) {
  c.planes = c.shape->planes;
  c.heads = c.shape->kv_heads;
  c.row_bytes = c.shape->row_bytes;
  c.seg_bytes = c.shape->seg_bytes;
  c.src_head_off = c.dst_head_off = 0;
  c.vec = std::min(std::min(side_vec(c.src), side_vec(c.dst)), pow2_align(c.row_bytes));
}

// Rows per plan chunk: runs cut into chunks of up to KVX_CHUNK_BYTES, one row for narrow rows.
int32_t call_chunk_rows(const Call &c) {
  return c.vec < 16 ? 1 : chunk_rows_for(c.row_bytes);
}

// Whether the planner checks this call's destination slots for repeats: calls that write
// into a pool, with KVX_CHECK_DUP.
bool dup_check(const Call &c) { return c.check_dup && c.dst != nullptr && c.n_tokens > 0; }

// The workspace a slot-list call needs (the duplicate table included when it is checked).
kvx::WsLayout slots_ws(const Call &c) { return kvx::ws_layout(c.n_tokens, 0, false, dup_check(c)); }

// Checks the layouts an op needs and fills call.src / call.dst / call.shape.
kvx_status bind_layouts(Call &c, kvx_layout_t src, kvx_layout_t dst) {
  switch (c.op) {
    case KVX_OP_GATHER:
      if (!src) return KVX_ERR_INVALID_ARG;
      c.src = src;
      c.shape = src;
      set_whole_rows(c);
      return KVX_OK;
    case KVX_OP_SCATTER:
      if (!dst) return KVX_ERR_INVALID_ARG;
      c.dst = dst;
      c.shape = dst;
      set_whole_rows(c);
      return KVX_OK;
    case KVX_OP_TRANSFER:
    case KVX_OP_BATCH:
      if (c.op == KVX_OP_TRANSFER && (!src || !dst)) return KVX_ERR_INVALID_ARG;
      if (!src && !dst) return KVX_ERR_INVALID_ARG;
      if (src && dst && !same_rows(src, dst)) return KVX_ERR_INVALID_ARG;
      if (src && dst && layouts_overlap(src, dst)) return KVX_ERR_OVERLAP;
      c.src = src;
      c.dst = dst;
      c.shape = src ? src : dst;
      set_whole_rows(c);
      return KVX_OK;
    default:
      return KVX_ERR_INVALID_ARG;
  }
}

kvx::Side src_side(const Call &c) {
  if (c.mode == kvx::kModeBatch) {
    if (c.src) return pool_side(c.src);
    kvx::Side s = pool_side(c.shape);
    s.num_slots = 0;
    return s;
  }
  return c.src ? pool_side(c.src) : buffer_side(c.seg_bytes);
}

kvx::Side dst_side(const Call &c) {
  if (c.mode == kvx::kModeBatch) {
    if (c.dst) return pool_side(c.dst);
    kvx::Side s = pool_side(c.shape);
    s.num_slots = 0;
    return s;
  }
  return c.dst ? pool_side(c.dst) : buffer_side(c.seg_bytes);
}

kvx_status check_ws(const void *d_ws, size_t ws_bytes, const kvx::WsLayout &L) {
  if (!d_ws || !aligned(d_ws, 256)) return KVX_ERR_NO_WORKSPACE;
  if ((int64_t)ws_bytes < L.total) return KVX_ERR_NO_WORKSPACE;
  return KVX_OK;
}

kvx_status check_buffer(const Call &c, const void *d_buf, size_t buf_bytes) {
  if (c.mode == kvx::kModeBatch) {
    if (buf_bytes > 0 && (!d_buf || !aligned(d_buf, 16))) return KVX_ERR_ALIGNMENT;
  } else if (c.op == KVX_OP_GATHER || c.op == KVX_OP_SCATTER) {
    const int64_t need = (int64_t)c.planes * c.n_tokens * c.row_bytes;
    if (!d_buf) return KVX_ERR_INVALID_ARG;
    if (!aligned(d_buf, 16)) return KVX_ERR_ALIGNMENT;
    if ((int64_t)buf_bytes < need) return KVX_ERR_INVALID_ARG;
    buf_bytes = (size_t)need;
  } else {
    return KVX_OK;
  }
  if (buf_bytes == 0) return KVX_OK;
  const uintptr_t b0 = (uintptr_t)d_buf, b1 = b0 + buf_bytes;
  if (c.src && layout_overlaps_range(c.src, b0, b1)) return KVX_ERR_OVERLAP;
  if (c.dst && layout_overlaps_range(c.dst, b0, b1)) return KVX_ERR_OVERLAP;
  return KVX_OK;
}

kvx::PlanArgs plan_args(const Call &c, void *d_ws, int32_t *d_status) {
  kvx::PlanArgs a;
  std::memset(&a, 0, sizeof(a));
  a.mode = c.mode;
  a.op = c.op;
  a.n_tokens = c.n_tokens;
  a.n_segs = c.n_segs;
  a.chunk_rows = call_chunk_rows(c);
  a.planes = c.planes;
  a.row_bytes = (int32_t)c.row_bytes;
  a.src = src_side(c);
  a.dst = dst_side(c);
  a.has_src = c.src != nullptr;
  a.has_dst = c.dst != nullptr;
  a.ws = static_cast<char *>(d_ws);
  a.L = kvx::ws_layout(c.n_tokens, c.n_segs, false, dup_check(c));
  a.status = d_status;
  if (dup_check(c)) {
    a.dup_table =
        reinterpret_cast<unsigned long long *>(static_cast<char *>(d_ws) + a.L.dup_off);
    a.dup_mask = (uint32_t)(a.L.dup_slots - 1);
    int32_t bits = 0;
    while (((int64_t)1 << bits) < a.L.dup_slots) ++bits;
    a.dup_bits = bits;
  }
  return a;
}

kvx_status enqueue_plan(const Call &c, kvx::PlanArgs &a, cudaStream_t s) {
  cudaError_t e;
  if (c.n_tokens == 0) {
    e = cudaMemsetAsync(a.status, 0, sizeof(int32_t) * (size_t)c.n_status, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  if (a.dup_table) {  // an empty duplicate table
    e = cudaMemsetAsync(a.dup_table, 0, sizeof(unsigned long long) * ((size_t)a.dup_mask + 1), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (c.mode == kvx::kModeSlots) {
    if (kvx::validates_direct(c.n_tokens, a.validate_only != 0)) {
      a.status_direct = 1;
    } else {
      e = cudaMemsetAsync(a.status, 0, sizeof(int32_t), s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  } else {
    e = kvx::launch_prefix(a, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = kvx::launch_plan(a, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

void fill_copy_args(kvx::CopyArgs &a, const Call &c, const kvx_request *d_reqs, void *d_buf,
                    const void *d_ws, int32_t *d_status) {
  std::memset(&a, 0, sizeof(a));
  a.mode = c.mode;
  a.op = c.op;
  a.n_tokens = c.n_tokens;
  a.n_segs = c.n_segs;
  a.chunk_rows = call_chunk_rows(c);
  a.planes = c.planes;
  a.row_bytes = (int32_t)c.row_bytes;
  a.seg_bytes = (int32_t)c.seg_bytes;
  a.heads = c.heads;
  a.vec_bytes = c.vec;
  a.src = src_side(c);
  a.dst = dst_side(c);
  a.buf = static_cast<char *>(d_buf);
  a.reqs = d_reqs;
  a.ws = static_cast<const char *>(d_ws);
  a.L = kvx::ws_layout(c.n_tokens, c.n_segs, false);
  a.status = d_status;
  a.row_lanes = 32;  // one token per warp unless the call's row shape says otherwise
  a.rows_per_warp = 1;
  for (int p = 0; p < c.planes; ++p) {
    a.src_planes[p] = c.src ? reinterpret_cast<const char *>(c.src->plane[p]) + c.src_head_off
                            : nullptr;
    a.dst_planes[p] = c.dst ? reinterpret_cast<char *>(c.dst->plane[p]) + c.dst_head_off : nullptr;
  }
}

// engine: the call's KVX_ENGINE_* (read once per call, so that it matches what the planner
// was told).
kvx_status enqueue_copy(const Call &c, const kvx_request *d_reqs, void *d_buf, const void *d_ws,
                        int32_t *d_status, cudaStream_t s, int32_t engine,
                        const int32_t *spec_src = nullptr,
                        const int32_t *spec_dst = nullptr, int32_t *host_status = nullptr,
                        bool *host_status_written = nullptr) {
  if (host_status_written) *host_status_written = false;
  if (c.n_tokens == 0) return KVX_OK;
  DeviceInfo di;
  kvx_status st = device_info(&di);
  if (st != KVX_OK) return st;
  static thread_local kvx::CopyArgs a;  // ~4 KiB of plane pointers: keep it off the stack
  fill_copy_args(a, c, d_reqs, d_buf, d_ws, d_status);
  a.spec_src = spec_src;
  a.spec_dst = spec_dst;
  if (c.vec < 16) {  // narrow rows: read after the planner, several rows per warp
    a.row_group_shift = kvx::narrow_group_shift(a.row_bytes, a.vec_bytes);
    const cudaError_t e = kvx::launch_narrow(a, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  const kvx::CopyVariant v = kvx::copy_variant(a, engine);
  if (v == kvx::kVariantRow) {
    a.host_status = host_status;
    if (host_status_written) *host_status_written = host_status != nullptr;
    kvx::row_shape(a, &a.row_lanes, &a.rows_per_warp);
    const int64_t grid = kvx::row_grid(a);
    const cudaError_t e = kvx::launch_copy(a, v, (int)grid, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  a.spec_src = a.spec_dst = nullptr;  // the other kernels read the plan
  // one warp (register paths) or one thread (bulk path) per work item; at most n*P items
  const int64_t items = (int64_t)c.planes * c.n_tokens;
  const int64_t per_cta = v == kvx::kVariantBulk ? kvx::variant_threads(v) : kvx::kCopyThreads / 32;
  const bool small = kvx::num_tiles(c.n_tokens) <= kvx::kBulkSmallTiles;
  int64_t grid = (int64_t)di.sms * (small ? di.bps_small[v] : di.bps[v]);
  const int64_t need = (items + per_cta - 1) / per_cta;
  if (need < grid) grid = need;
  if (grid < 1) grid = 1;
  cudaError_t e = kvx::launch_copy(a, v, (int)grid, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

// The one-launch path of a single request (see kvx_set_fused_max_tokens).
kvx_status enqueue_fused(const Call &c, const int32_t *d_src, const int32_t *d_dst, void *d_buf,
                         int32_t *d_status, cudaStream_t s) {
  DeviceInfo di;
  kvx_status st = device_info(&di);
  if (st != KVX_OK) return st;
  static thread_local kvx::CopyArgs a;
  fill_copy_args(a, c, nullptr, d_buf, nullptr, d_status);
  const int bps = kvx::copy_is_linear(a) ? di.bps_fused_linear : di.bps_fused_general;
  cudaError_t e = kvx::launch_fused(a, d_src, d_dst, (int32_t)c.n_tokens,
                                    chunk_rows_for(c.row_bytes), di.sms, bps, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

bool valid_n(int64_t n) { return n >= 0 && n <= KVX_MAX_TOKENS; }

}  // namespace

void kvx::record_cuda_error(cudaError_t e) { g_last_cuda = (int32_t)e; }

extern "C" {

kvx_status kvx_layout_create(const kvx_layout_desc *d, kvx_layout_t *out) {
  if (!d || !out) return KVX_ERR_INVALID_ARG;
  *out = nullptr;
  const int eb = elem_bytes_of(d->dtype);
  const int32_t kvp = d->kv_planes == 0 ? 2 : d->kv_planes;
  if ((kvp != 1 && kvp != 2) || d->reserved != 0) return KVX_ERR_INVALID_ARG;
  if (d->num_layers < 1 || kvp * (int64_t)d->num_layers > KVX_MAX_PLANES || d->kv_heads < 1 ||
      d->head_dim < 1 || eb == 0 || d->num_slots < 1 || d->num_slots > INT32_MAX)
    return KVX_ERR_INVALID_ARG;
  if (d->kind != KVX_NHD && d->kind != KVX_HND_PAGED) return KVX_ERR_INVALID_ARG;
  const int64_t seg = (int64_t)d->head_dim * eb;
  const int64_t R = seg * d->kv_heads;
  if (R > (int64_t)1 << 30) return KVX_ERR_INVALID_ARG;
  kvx_layout *l = new (std::nothrow) kvx_layout;
  if (!l) return KVX_ERR_INVALID_ARG;
  std::memset(l, 0, sizeof(*l));
  l->num_layers = d->num_layers;
  l->kv_heads = d->kv_heads;
  l->head_dim = d->head_dim;
  l->elem = eb;
  l->kind = d->kind;
  l->kv_planes = kvp;
  l->planes = kvp * d->num_layers;
  l->num_slots = d->num_slots;
  l->row_bytes = R;
  l->seg_bytes = seg;
  kvx_status st = KVX_OK;
  // Rows move in the widest accesses that every row start, head vector and plane allows:
  // 16 bytes for the usual shapes, narrower for rows that are not 16-byte multiples.
  l->vec = pow2_align(R);
  if (d->kind == KVX_HND_PAGED) {
    if (d->page_size < 1 || d->num_slots % d->page_size != 0 || d->slot_stride != 0)
      st = KVX_ERR_INVALID_ARG;
    l->vec = std::min(l->vec, pow2_align(seg));  // a head vector is contiguous, not a row
    l->page_size = d->page_size;
    l->page_bytes = R * d->page_size;
    l->extent = l->page_bytes * (d->num_slots / (d->page_size > 0 ? d->page_size : 1));
  } else {
    l->page_size = 1;
    l->slot_stride = d->slot_stride == 0 ? R : d->slot_stride;
    if (l->slot_stride < R) st = KVX_ERR_INVALID_ARG;
    else if (l->slot_stride > ((int64_t)1 << 62) / d->num_slots) st = KVX_ERR_INVALID_ARG;
    l->vec = std::min(l->vec, pow2_align(l->slot_stride));
    l->extent = (d->num_slots - 1) * l->slot_stride + R;
  }
  if (st == KVX_OK) {
    l->lo = UINTPTR_MAX;
    l->hi = 0;
    for (int p = 0; p < l->planes; ++p) {
      uintptr_t a;
      if (d->plane_ptrs) {
        a = (uintptr_t)d->plane_ptrs[p];
      } else {
        if (!d->base) { st = KVX_ERR_INVALID_ARG; break; }
        a = (uintptr_t)d->base + (uintptr_t)(d->plane_stride * p);
      }
      if (a == 0) { st = KVX_ERR_INVALID_ARG; break; }
      if (a % l->elem != 0) { st = KVX_ERR_ALIGNMENT; break; }  // elements stay aligned
      l->vec = std::min(l->vec, pow2_align((int64_t)a));
      l->plane[p] = a;
      if (a < l->lo) l->lo = a;
      if (a + l->extent > l->hi) l->hi = a + l->extent;
    }
  }
  if (st != KVX_OK) {
    delete l;
    return st;
  }
  *out = l;
  return KVX_OK;
}

kvx_status kvx_layout_destroy(kvx_layout_t layout) {
  delete layout;
  return KVX_OK;
}

int64_t kvx_layout_row_bytes(kvx_layout_t l) { return l ? l->row_bytes : -1; }

int32_t kvx_layout_num_planes(kvx_layout_t l) { return l ? l->planes : -1; }

size_t kvx_workspace_size(int64_t max_tokens, int32_t max_requests) {
  if (!valid_n(max_tokens) || max_requests < 0 || max_requests > kvx::kMaxSegs) return 0;
  return (size_t)kvx::ws_layout(max_tokens, max_requests, true, true).total;
}

kvx_status kvx_plan(int32_t op, kvx_layout_t src, const int32_t *d_src_slots, kvx_layout_t dst,
                    const int32_t *d_dst_slots, int32_t n, void *d_ws, size_t ws_bytes,
                    int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_TRANSFER || !valid_n(n)) return KVX_ERR_INVALID_ARG;
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  Call c;
  c.mode = kvx::kModeSlots;
  c.op = op;
  c.n_tokens = n;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st != KVX_OK) return st;
  if (n > 0) {
    if (c.src && (!d_src_slots || !aligned(d_src_slots, 4))) return KVX_ERR_INVALID_ARG;
    if (c.dst && (!d_dst_slots || !aligned(d_dst_slots, 4))) return KVX_ERR_INVALID_ARG;
  }
  const kvx::WsLayout L = slots_ws(c);
  if (n > 0 && (st = check_ws(d_ws, ws_bytes, L)) != KVX_OK) return st;
  kvx::PlanArgs a = plan_args(c, d_ws, d_status);
  a.src_idx = d_src_slots;
  a.dst_idx = d_dst_slots;
  return enqueue_plan(c, a, reinterpret_cast<cudaStream_t>(stream));
}

kvx_status kvx_plan_runs(int32_t op, kvx_layout_t src, kvx_layout_t dst, const int32_t *d_runs,
                         int32_t n_runs, int32_t n_tokens, void *d_ws, size_t ws_bytes,
                         int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_TRANSFER || !valid_n(n_tokens) || n_runs < 0 ||
      n_runs > kvx::kMaxSegs)
    return KVX_ERR_INVALID_ARG;
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  if (n_runs > 0 && (!d_runs || !aligned(d_runs, 4))) return KVX_ERR_INVALID_ARG;
  Call c;
  c.mode = kvx::kModeRuns;
  c.op = op;
  c.n_tokens = n_tokens;
  c.n_segs = n_runs;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st != KVX_OK) return st;
  if (n_runs == 0 && n_tokens > 0) return KVX_ERR_INVALID_ARG;
  const kvx::WsLayout L = kvx::ws_layout(n_tokens, n_runs, false, dup_check(c));
  if ((n_tokens > 0 || n_runs > 0) && (st = check_ws(d_ws, ws_bytes, L)) != KVX_OK) return st;
  kvx::PlanArgs a = plan_args(c, d_ws, d_status);
  a.runs = d_runs;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n_tokens == 0 && n_runs > 0) {
    // nothing to move, but the runs must still add up to zero
    cudaError_t e = kvx::launch_prefix(a, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  return enqueue_plan(c, a, s);
}

kvx_status kvx_plan_batch(kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                          int32_t n_reqs, int64_t total_tokens, const int32_t *d_src_slots,
                          int64_t n_src_slots, const int32_t *d_dst_slots, int64_t n_dst_slots,
                          size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                          uint32_t flags, kvx_stream_t stream) {
  if (!valid_n(total_tokens) || n_reqs < 0 || n_reqs > kvx::kMaxSegs || n_src_slots < 0 ||
      n_dst_slots < 0)
    return KVX_ERR_INVALID_ARG;
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  if (n_reqs > 0 && (!d_reqs || !aligned(d_reqs, 8))) return KVX_ERR_INVALID_ARG;
  if (n_src_slots > 0 && (!d_src_slots || !aligned(d_src_slots, 4))) return KVX_ERR_INVALID_ARG;
  if (n_dst_slots > 0 && (!d_dst_slots || !aligned(d_dst_slots, 4))) return KVX_ERR_INVALID_ARG;
  Call c;
  c.mode = kvx::kModeBatch;
  c.op = KVX_OP_BATCH;
  c.n_tokens = total_tokens;
  c.n_segs = n_reqs;
  c.n_status = n_reqs + 1;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st != KVX_OK) return st;
  const kvx::WsLayout L = kvx::ws_layout(total_tokens, n_reqs, false, dup_check(c));
  if (n_reqs > 0 && (st = check_ws(d_ws, ws_bytes, L)) != KVX_OK) return st;
  kvx::PlanArgs a = plan_args(c, d_ws, d_status);
  a.src_idx = d_src_slots;
  a.dst_idx = d_dst_slots;
  a.n_src_idx = n_src_slots;
  a.n_dst_idx = n_dst_slots;
  a.reqs = d_reqs;
  a.buf_bytes = (int64_t)buf_bytes;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n_reqs == 0) {
    if (total_tokens != 0) return KVX_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int32_t), s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  cudaError_t e;
  if (a.dup_table) {  // an empty duplicate table
    e = cudaMemsetAsync(a.dup_table, 0, sizeof(unsigned long long) * ((size_t)a.dup_mask + 1), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = kvx::launch_prefix(a, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (total_tokens == 0) return KVX_OK;
  e = kvx::launch_plan(a, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

kvx_status kvx_execute(int32_t op, kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                       int32_t n_reqs, int64_t n_tokens, void *d_buf, size_t buf_bytes,
                       const void *d_ws, size_t ws_bytes, int32_t *d_status, uint32_t flags,
                       kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_BATCH || !valid_n(n_tokens)) return KVX_ERR_INVALID_ARG;
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  Call c;
  c.op = op;
  c.mode = op == KVX_OP_BATCH ? kvx::kModeBatch : kvx::kModeSlots;
  c.n_tokens = n_tokens;
  if (op == KVX_OP_BATCH) {
    if (n_reqs < 0 || n_reqs > kvx::kMaxSegs || (n_reqs > 0 && !d_reqs)) return KVX_ERR_INVALID_ARG;
    c.n_segs = n_reqs;
  }
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st != KVX_OK) return st;
  if ((st = check_buffer(c, d_buf, buf_bytes)) != KVX_OK) return st;
  if (n_tokens == 0) return KVX_OK;
  if ((st = check_ws(d_ws, ws_bytes, kvx::ws_layout(n_tokens, c.n_segs, false))) != KVX_OK)
    return st;
  return enqueue_copy(c, d_reqs, d_buf, d_ws, d_status, reinterpret_cast<cudaStream_t>(stream),
                      c.engine);
}

// gather / scatter / transfer of one slot-list request: one launch up to the fused limit,
// otherwise the planner + copy launches.
// The one-shot path of a bound call: planner + copy (the copy reading the slot lists itself),
// or the one-launch fused path.
static kvx_status run_call(const Call &c, const int32_t *d_src_slots, const int32_t *d_dst_slots,
                           void *d_buf, void *d_ws, size_t ws_bytes, int32_t *d_status,
                           kvx_stream_t stream, int32_t *host_status = nullptr,
                           bool *host_status_written = nullptr) {
  if (host_status_written) *host_status_written = false;
  const int64_t n = c.n_tokens;
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  if (n > 0) {
    if (c.src && (!d_src_slots || !aligned(d_src_slots, 4))) return KVX_ERR_INVALID_ARG;
    if (c.dst && (!d_dst_slots || !aligned(d_dst_slots, 4))) return KVX_ERR_INVALID_ARG;
  }
  const kvx::WsLayout L = slots_ws(c);
  kvx_status st;
  if (n > 0 && (st = check_ws(d_ws, ws_bytes, L)) != KVX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int32_t engine = c.engine;
  // Requests of up to the fused limit with rows under KVX_CHUNK_BYTES take the one-launch
  // path; the rest take the planner + row kernel (the row kernel overlaps the planner).
  const bool fused = call_chunk_rows(c) > 1 && !dup_check(c) && n <= c.fused_max;
  // small requests: one launch whose every CTA checks every index (no planner), unless the
  // duplicate check or the bulk engine was asked for
  const bool small = n > 0 && n <= kvx::kSmallMaxTokens && !fused && !dup_check(c) &&
                     c.vec == 16 && engine != KVX_ENGINE_BULK;
  if (small) {
    static thread_local kvx::CopyArgs a;  // ~4 KiB of plane pointers: keep it off the stack
    fill_copy_args(a, c, nullptr, d_buf, d_ws, d_status);
    a.spec_src = c.src ? d_src_slots : nullptr;
    a.spec_dst = c.dst ? d_dst_slots : nullptr;
    a.host_status = host_status;
    if (host_status_written) *host_status_written = host_status != nullptr;
    kvx::row_shape(a, &a.row_lanes, &a.rows_per_warp);
    const cudaError_t e = kvx::launch_small(a, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  if (n == 0 || !fused) {
    kvx::PlanArgs a = plan_args(c, d_ws, d_status);
    a.src_idx = d_src_slots;
    a.dst_idx = d_dst_slots;
    // The copy reads the slot lists itself (see CopyArgs::spec_src) and needs only the
    // planner's verdict, except the TMA bulk kernel, which walks the plan's chunks.
    a.validate_only = c.vec < 16 || engine != KVX_ENGINE_BULK;
    st = enqueue_plan(c, a, s);
    if (st != KVX_OK || n == 0) return st;
    return enqueue_copy(c, nullptr, d_buf, d_ws, d_status, s, engine,
                        c.src ? d_src_slots : nullptr, c.dst ? d_dst_slots : nullptr,
                        host_status, host_status_written);
  }
  return enqueue_fused(c, c.src ? d_src_slots : nullptr, c.dst ? d_dst_slots : nullptr, d_buf,
                       d_status, s);
}

static kvx_status run_slots(int32_t op, kvx_layout_t src, const int32_t *d_src_slots,
                            kvx_layout_t dst, const int32_t *d_dst_slots, int32_t n, void *d_buf,
                            size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                            uint32_t flags, kvx_stream_t stream, int32_t *host_status = nullptr,
                            bool *host_status_written = nullptr) {
  if (host_status_written) *host_status_written = false;
  if (!valid_n(n)) return KVX_ERR_INVALID_ARG;
  Call c;
  c.op = op;
  c.n_tokens = n;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st == KVX_OK) st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  return run_call(c, d_src_slots, d_dst_slots, d_buf, d_ws, ws_bytes, d_status, stream,
                  host_status, host_status_written);
}

kvx_status kvx_gather(kvx_layout_t src, const int32_t *d_src_slots, int32_t n, void *d_buf,
                      size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                      uint32_t flags, kvx_stream_t stream) {
  return run_slots(KVX_OP_GATHER, src, d_src_slots, nullptr, nullptr, n, d_buf, buf_bytes, d_ws,
                   ws_bytes, d_status, flags, stream);
}

kvx_status kvx_scatter(kvx_layout_t dst, const int32_t *d_dst_slots, int32_t n,
                       const void *d_buf, size_t buf_bytes, void *d_ws, size_t ws_bytes,
                       int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  return run_slots(KVX_OP_SCATTER, nullptr, nullptr, dst, d_dst_slots, n,
                   const_cast<void *>(d_buf), buf_bytes, d_ws, ws_bytes, d_status, flags, stream);
}

kvx_status kvx_transfer(kvx_layout_t src, const int32_t *d_src_slots, kvx_layout_t dst,
                        const int32_t *d_dst_slots, int32_t n, void *d_ws, size_t ws_bytes,
                        int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  return run_slots(KVX_OP_TRANSFER, src, d_src_slots, dst, d_dst_slots, n, nullptr, 0, d_ws,
                   ws_bytes, d_status, flags, stream);
}

kvx_status kvx_gather_runs(kvx_layout_t src, const int32_t *d_runs, int32_t n_runs,
                           int32_t n_tokens, void *d_buf, size_t buf_bytes, void *d_ws,
                           size_t ws_bytes, int32_t *d_status, uint32_t flags,
                           kvx_stream_t stream) {
  Call c;
  c.op = KVX_OP_GATHER;
  c.n_tokens = n_tokens;
  kvx_status st = bind_layouts(c, src, nullptr);
  if (st == KVX_OK && valid_n(n_tokens)) st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  st = kvx_plan_runs(KVX_OP_GATHER, src, nullptr, d_runs, n_runs, n_tokens, d_ws, ws_bytes,
                     d_status, flags, stream);
  if (st != KVX_OK) return st;
  return kvx_execute(KVX_OP_GATHER, src, nullptr, nullptr, 0, n_tokens, d_buf, buf_bytes, d_ws,
                     ws_bytes, d_status, flags, stream);
}

kvx_status kvx_scatter_runs(kvx_layout_t dst, const int32_t *d_runs, int32_t n_runs,
                            int32_t n_tokens, const void *d_buf, size_t buf_bytes, void *d_ws,
                            size_t ws_bytes, int32_t *d_status, uint32_t flags,
                            kvx_stream_t stream) {
  Call c;
  c.op = KVX_OP_SCATTER;
  c.n_tokens = n_tokens;
  kvx_status st = bind_layouts(c, nullptr, dst);
  if (st == KVX_OK && valid_n(n_tokens)) st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  st = kvx_plan_runs(KVX_OP_SCATTER, nullptr, dst, d_runs, n_runs, n_tokens, d_ws, ws_bytes,
                     d_status, flags, stream);
  if (st != KVX_OK) return st;
  return kvx_execute(KVX_OP_SCATTER, nullptr, dst, nullptr, 0, n_tokens,
                     const_cast<void *>(d_buf), buf_bytes, d_ws, ws_bytes, d_status, flags,
                     stream);
}

kvx_status kvx_transfer_runs(kvx_layout_t src, kvx_layout_t dst, const int32_t *d_runs,
                             int32_t n_runs, int32_t n_tokens, void *d_ws, size_t ws_bytes,
                             int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  kvx_status st = kvx_plan_runs(KVX_OP_TRANSFER, src, dst, d_runs, n_runs, n_tokens, d_ws,
                                ws_bytes, d_status, flags, stream);
  if (st != KVX_OK) return st;
  return kvx_execute(KVX_OP_TRANSFER, src, dst, nullptr, 0, n_tokens, nullptr, 0, d_ws, ws_bytes,
                     d_status, flags, stream);
}

kvx_status kvx_batch(kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                     int32_t n_reqs, int64_t total_tokens, const int32_t *d_src_slots,
                     int64_t n_src_slots, const int32_t *d_dst_slots, int64_t n_dst_slots,
                     void *d_buf, size_t buf_bytes, void *d_ws, size_t ws_bytes,
                     int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  Call c;
  c.op = KVX_OP_BATCH;
  c.mode = kvx::kModeBatch;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st == KVX_OK) st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  st = kvx_plan_batch(src, dst, d_reqs, n_reqs, total_tokens, d_src_slots, n_src_slots,
                      d_dst_slots, n_dst_slots, buf_bytes, d_ws, ws_bytes, d_status, flags,
                      stream);
  if (st != KVX_OK) return st;
  return kvx_execute(KVX_OP_BATCH, src, dst, d_reqs, n_reqs, total_tokens, d_buf, buf_bytes,
                     d_ws, ws_bytes, d_status, flags, stream);
}

// Device address of a pinned (page-locked) host buffer, or nullptr for pageable memory.
static const void *pinned_alias(const void *h) {
  if (!h) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

kvx_status kvx_submit(int32_t op, kvx_layout_t src, const int32_t *h_src_slots,
                      kvx_layout_t dst, const int32_t *h_dst_slots, int32_t n, void *d_buf,
                      size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *h_status,
                      uint32_t flags, kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_TRANSFER || !valid_n(n) || !h_status)
    return KVX_ERR_INVALID_ARG;
  Call c;
  c.op = op;
  c.n_tokens = n;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st != KVX_OK) return st;
  if ((st = check_buffer(c, d_buf, buf_bytes)) != KVX_OK) return st;
  if (n > 0 && ((c.src && !h_src_slots) || (c.dst && !h_dst_slots))) return KVX_ERR_INVALID_ARG;
  const kvx::WsLayout L = kvx::ws_layout(n, 0, true, dup_check(c));
  if ((st = check_ws(d_ws, ws_bytes, L)) != KVX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *stage = static_cast<char *>(d_ws) + L.stage_off;
  int32_t *d_st = reinterpret_cast<int32_t *>(stage + kvx::align_up(8 * (int64_t)n, 16));
  cudaError_t e;
  // Pinned host memory is reachable from the GPU (over NVLink-C2C on GB300): the kernels then
  // read the slot lists and write the status word in place.  Pageable memory is staged with
  // copies into the workspace.
  const int32_t *z_src = static_cast<const int32_t *>(pinned_alias(h_src_slots));
  const int32_t *z_dst = static_cast<const int32_t *>(pinned_alias(h_dst_slots));
  int32_t *z_status = static_cast<int32_t *>(const_cast<void *>(pinned_alias(h_status)));
  const int32_t *use_src = z_src, *use_dst = z_dst;
  if (n > 0 && c.src && !z_src) {
    int32_t *d_src = reinterpret_cast<int32_t *>(stage);
    e = cudaMemcpyAsync(d_src, h_src_slots, sizeof(int32_t) * (size_t)n, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    use_src = d_src;
  }
  if (n > 0 && c.dst && !z_dst) {
    int32_t *d_dst = reinterpret_cast<int32_t *>(stage) + n;
    e = cudaMemcpyAsync(d_dst, h_dst_slots, sizeof(int32_t) * (size_t)n, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    use_dst = d_dst;
  }
  bool written = false;
  st = run_slots(op, src, c.src ? use_src : nullptr, dst, c.dst ? use_dst : nullptr, n, d_buf,
                 buf_bytes, d_ws, ws_bytes, d_st, flags, stream, z_status, &written);
  if (st != KVX_OK || written) return st;
  e = cudaMemcpyAsync(h_status, d_st, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

// Tags the mirror words of each streamed call: a Weyl sequence (odd step), so tags of nearby
// calls differ in every bit range.
std::atomic<uint64_t> g_stream_gen{0xD1B54A32D192ED03ull};

// The streamed kernels' device-memory mirror (in the workspace, where a plan's chunk table
// would be) and the call's tag.  Words of earlier calls never match a new tag, so an eager call
// needs no reset; a call being captured into a CUDA graph replays with the tag it was captured
// with, so its mirror is cleared at the start of every replay (a zero word never matches a tag:
// tags are non-zero with non-zero low 40 bits, which also keeps zero from reading as a stop).
static kvx_status stream_mirror(void *d_ws, int64_t n, cudaStream_t s, kvx::StreamCtl *k) {
  uint64_t gen;
  do {
    gen = g_stream_gen.fetch_add(0x9E3779B97F4A7C15ull, std::memory_order_relaxed);
  } while ((gen & 0xFFFFFFFFFFull) == 0);
  k->gen = gen;
  k->mirror = nullptr;
  if (n == 0) return KVX_OK;
  k->mirror = reinterpret_cast<uint64_t *>(static_cast<char *>(d_ws) +
                                           kvx::ws_layout(n, 0, false).chunks_off);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return cuda_fail(e);
  if (cs != cudaStreamCaptureStatusNone) {
    e = cudaMemsetAsync(k->mirror, 0, sizeof(uint64_t) * kvx::kMirrorWords, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return KVX_OK;
}
static_assert(sizeof(kvx::Chunk) * kvx::kTile >= sizeof(uint64_t) * kvx::kMirrorWords,
              "the stream mirror fits in one tile's chunk table");

// Device address of a control word: device memory as is, pinned host memory through its
// device mapping; anything else (pageable memory, unknown pointers) gives nullptr.
static const void *device_word(const void *p, bool *in_device_memory = nullptr) {
  if (in_device_memory) *in_device_memory = false;
  if (!p) return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice) {
    if (in_device_memory) *in_device_memory = true;
    return at.devicePointer;
  }
  if (at.type == cudaMemoryTypeManaged || at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

// The device form of a kvx_stream_ctl for a move of op over layouts shaped like shape (the
// fields every streamed move shares); KVX_ERR_INVALID_ARG for a malformed control block.
static kvx_status stream_ctl_of(const kvx_stream_ctl *ctl, int32_t op, const kvx_layout *shape,
                                kvx::StreamCtl *out) {
  if (!ctl || ctl->wait_ns < 1 || ctl->wait_ns > KVX_MAX_WAIT_NS || ctl->max_ctas < 0 ||
      ctl->reserved != 0 || ctl->reserved2 != 0)
    return KVX_ERR_INVALID_ARG;
  if (ctl->dst_page_epochs && (op == KVX_OP_GATHER || ctl->epoch_page < 1))
    return KVX_ERR_INVALID_ARG;
  kvx::StreamCtl k = {};
  bool ready_local = false, epoch_local = false;
  k.layer_ready = static_cast<const int32_t *>(device_word(ctl->layer_ready, &ready_local));
  k.epoch_word = static_cast<const int32_t *>(device_word(ctl->epoch_word, &epoch_local));
  k.words_local = (!ctl->layer_ready || ready_local) && (!ctl->epoch_word || epoch_local);
  k.host_done = static_cast<int32_t *>(const_cast<void *>(pinned_alias(ctl->host_done)));
  k.page_epochs = static_cast<const int32_t *>(device_word(ctl->dst_page_epochs));
  k.epoch_page = ctl->epoch_page;
  if ((ctl->dst_page_epochs && (!k.page_epochs || !aligned(ctl->dst_page_epochs, 4))) ||
      (ctl->layer_ready && (!k.layer_ready || !aligned(ctl->layer_ready, 4))) ||
      (ctl->epoch_word && (!k.epoch_word || !aligned(ctl->epoch_word, 4))) ||
      (ctl->host_done && (!k.host_done || !aligned(ctl->host_done, 4))))
    return KVX_ERR_INVALID_ARG;
  k.wait_ns = ctl->wait_ns;
  k.ready_value = ctl->ready_value;
  k.epoch = ctl->epoch;
  k.layers = shape->num_layers;
  k.kv_planes = shape->kv_planes;
  *out = k;
  return KVX_OK;
}

kvx_status kvx_stream(int32_t op, kvx_layout_t src, const int32_t *d_src_slots, kvx_layout_t dst,
                      const int32_t *d_dst_slots, int32_t n, void *d_buf, size_t buf_bytes,
                      const kvx_stream_ctl *ctl, void *d_ws, size_t ws_bytes, int32_t *d_status,
                      uint32_t flags, kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_TRANSFER || !valid_n(n)) return KVX_ERR_INVALID_ARG;
  if (!d_status || !aligned(d_status, 16)) return KVX_ERR_INVALID_ARG;
  Call c;
  c.op = op;
  c.n_tokens = n;
  kvx_status st = apply_flags(c, flags);
  if (st == KVX_OK) st = bind_layouts(c, src, dst);
  if (st == KVX_OK) st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  if (c.vec < 16) return KVX_ERR_ALIGNMENT;  // the streamed kernels move 16-byte vectors
  kvx::StreamCtl k = {};
  if ((st = stream_ctl_of(ctl, op, c.shape, &k)) != KVX_OK) return st;
  if (n > 0) {
    if (c.src && (!d_src_slots || !aligned(d_src_slots, 4))) return KVX_ERR_INVALID_ARG;
    if (c.dst && (!d_dst_slots || !aligned(d_dst_slots, 4))) return KVX_ERR_INVALID_ARG;
    if ((st = check_ws(d_ws, ws_bytes, slots_ws(c))) != KVX_OK) return st;
  }
  DeviceInfo di;
  if ((st = device_info(&di)) != KVX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((st = stream_mirror(d_ws, n, s, &k)) != KVX_OK) return st;
  // status[0..3]: verdict, layers pending, CTAs finished, done.  A one-CTA validation
  // writes all four itself; otherwise they are zeroed first and the planner's tiles raise [0].
  const bool direct = kvx::validates_direct(n, true);
  if (!direct) {
    e = cudaMemsetAsync(d_status, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (n > 0) {
    kvx::PlanArgs pa = plan_args(c, d_ws, d_status);
    pa.src_idx = d_src_slots;
    pa.dst_idx = d_dst_slots;
    pa.validate_only = 1;  // the streamed copy reads the slot lists itself
    if (direct) pa.status_direct = 4;
    if (pa.dup_table) {
      e = cudaMemsetAsync(pa.dup_table, 0, sizeof(unsigned long long) * ((size_t)pa.dup_mask + 1), s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    e = kvx::launch_plan(pa, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  static thread_local kvx::CopyArgs a;  // ~4 KiB of plane pointers: keep it off the stack
  fill_copy_args(a, c, nullptr, d_buf, d_ws, d_status);
  a.spec_src = c.src ? d_src_slots : nullptr;
  a.spec_dst = c.dst ? d_dst_slots : nullptr;
  kvx::row_shape(a, &a.row_lanes, &a.rows_per_warp);
  kvx::stream_sizes(k, n, a.rows_per_warp);
  if (ctl->max_ctas == 0) {  // one warp per item, then the epilogue
    e = kvx::launch_stream_rows(a, k, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  // persistent grid of at most max_ctas CTAs (at least one: it also runs the exit protocol)
  if (c.engine == KVX_ENGINE_BULK) {
    // bulk form: one thread per one-token item, a 2 KiB shared-memory stage each
    kvx::stream_sizes(k, n, 1);
    const int64_t per_cta = kvx::stream_bulk_threads();
    int64_t grid = (int64_t)di.sms * di.bps_stream_bulk;
    if (ctl->max_ctas < grid) grid = ctl->max_ctas;
    const int64_t need = ((int64_t)k.items + per_cta - 1) / per_cta;
    if (need < grid) grid = need;
    if (grid < 1) grid = 1;
    const int64_t per_thread = ((int64_t)k.items + grid * per_cta - 1) / (grid * per_cta);
    k.block = (uint32_t)std::min<int64_t>(std::max<int64_t>(per_thread / 4, 1), 8);
    e = kvx::launch_stream_bulk(a, k, (int)grid, s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  // register CTAs of 32 warps; with the default engine, three of the warps move their rows by
  // TMA bulk copies where a row group fits one stage
  const bool tma = c.engine == KVX_ENGINE_AUTO && kvx::stream_tma_fits(a);
  const int64_t warps = k.items;
  int64_t grid = (int64_t)di.sms * di.bps_stream;
  if (ctl->max_ctas < grid) grid = ctl->max_ctas;
  const int64_t wpc = kvx::stream_threads() / 32;  // warps per CTA
  const int64_t need = (warps + wpc - 1) / wpc;
  if (need < grid) grid = need;
  if (grid < 1) grid = 1;
  // about four blocks per warp: few layer entries per warp, yet each layer's items spread
  // over many warps (a late layer moves in a few row latencies)
  const int64_t per_warp = (warps + grid * wpc - 1) / (grid * wpc);
  k.block = (uint32_t)std::min<int64_t>(std::max<int64_t>(per_warp / 4, 1), 8);
  e = kvx::launch_stream(a, k, (int)grid, tma, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

// Heads [*first, *first + *count) held by rank r of a tensor-parallel group of size t.
static kvx_status tp_heads(int32_t heads, int32_t t, int32_t r, int32_t *first, int32_t *count) {
  if (heads < 1 || t < 1 || r < 0 || r >= t) return KVX_ERR_INVALID_ARG;
  if (t <= heads) {
    if (heads % t != 0) return KVX_ERR_INVALID_ARG;
    *first = r * (heads / t);
    *count = heads / t;
  } else {
    if (t % heads != 0) return KVX_ERR_INVALID_ARG;
    *first = r / (t / heads);  // t / heads ranks hold the same head
    *count = 1;
  }
  return KVX_OK;
}

kvx_status kvx_tp_slice(int32_t kv_heads, int32_t src_tp, int32_t src_rank, int32_t dst_tp,
                        int32_t dst_rank, int32_t *src_head0, int32_t *dst_head0,
                        int32_t *n_heads) {
  if (!src_head0 || !dst_head0 || !n_heads) return KVX_ERR_INVALID_ARG;
  int32_t sf, sc, df, dc;
  kvx_status st = tp_heads(kv_heads, src_tp, src_rank, &sf, &sc);
  if (st == KVX_OK) st = tp_heads(kv_heads, dst_tp, dst_rank, &df, &dc);
  if (st != KVX_OK) return st;
  *src_head0 = *dst_head0 = *n_heads = 0;
  const int32_t lo = std::max(sf, df), hi = std::min(sf + sc, df + dc);
  if (hi <= lo) return KVX_OK;
  if (src_tp > kv_heads && src_rank % (src_tp / kv_heads) != 0) return KVX_OK;  // a replica
  *src_head0 = lo - sf;
  *dst_head0 = lo - df;
  *n_heads = hi - lo;
  return KVX_OK;
}

// Byte offset of head h within a plane's token row (token-row pool) or page (HND pool).
static int64_t head_offset(const kvx_layout *l, int32_t h) {
  return l->kind == KVX_HND_PAGED ? (int64_t)h * l->page_size * l->seg_bytes
                                  : (int64_t)h * l->seg_bytes;
}

kvx_status kvx_move_heads(int32_t op, kvx_layout_t src, const int32_t *d_src_slots,
                          int32_t src_head0, kvx_layout_t dst, const int32_t *d_dst_slots,
                          int32_t dst_head0, int32_t n_heads, int32_t n, void *d_buf,
                          size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                          uint32_t flags, kvx_stream_t stream) {
  if (op < KVX_OP_GATHER || op > KVX_OP_TRANSFER || !valid_n(n) || n_heads < 1)
    return KVX_ERR_INVALID_ARG;
  const bool uses_src = op != KVX_OP_SCATTER, uses_dst = op != KVX_OP_GATHER;
  if ((uses_src && !src) || (uses_dst && !dst)) return KVX_ERR_INVALID_ARG;
  Call c;
  if (apply_flags(c, flags) != KVX_OK) return KVX_ERR_INVALID_ARG;
  c.op = op;
  c.n_tokens = n;
  c.src = uses_src ? src : nullptr;
  c.dst = uses_dst ? dst : nullptr;
  c.shape = uses_src ? src : dst;
  if (c.src && c.dst) {
    if (src->num_layers != dst->num_layers || src->kv_planes != dst->kv_planes ||
        src->head_dim != dst->head_dim || src->elem != dst->elem)
      return KVX_ERR_INVALID_ARG;
    if (layouts_overlap(src, dst)) return KVX_ERR_OVERLAP;
  }
  if (c.src && (src_head0 < 0 || (int64_t)src_head0 + n_heads > src->kv_heads))
    return KVX_ERR_INVALID_ARG;
  if (c.dst && (dst_head0 < 0 || (int64_t)dst_head0 + n_heads > dst->kv_heads))
    return KVX_ERR_INVALID_ARG;
  c.planes = c.shape->planes;
  c.heads = n_heads;
  c.seg_bytes = c.shape->seg_bytes;
  c.row_bytes = (int64_t)n_heads * c.seg_bytes;
  c.src_head_off = c.src ? head_offset(src, src_head0) : 0;
  c.dst_head_off = c.dst ? head_offset(dst, dst_head0) : 0;
  // accesses no wider than the slice's length and start on either side allow
  c.vec = std::min(std::min(side_vec(c.src), side_vec(c.dst)), pow2_align(c.row_bytes));
  if (c.src_head_off) c.vec = std::min(c.vec, pow2_align(c.src_head_off));
  if (c.dst_head_off) c.vec = std::min(c.vec, pow2_align(c.dst_head_off));
  kvx_status st = check_buffer(c, d_buf, buf_bytes);
  if (st != KVX_OK) return st;
  return run_call(c, d_src_slots, d_dst_slots, d_buf, d_ws, ws_bytes, d_status, stream);
}

kvx_status kvx_tp_plan(int32_t kv_heads, int32_t src_tp, int32_t dst_tp, kvx_head_part *parts,
                       int32_t max_parts, int32_t *n_parts) {
  if (!n_parts || max_parts < 0 || (max_parts > 0 && !parts)) return KVX_ERR_INVALID_ARG;
  if (src_tp < 1 || dst_tp < 1 || src_tp > 1024 || dst_tp > 1024) return KVX_ERR_INVALID_ARG;
  int32_t count = 0;
  for (int32_t dr = 0; dr < dst_tp; ++dr)
    for (int32_t sr = 0; sr < src_tp; ++sr) {
      int32_t h0 = 0, g0 = 0, nh = 0;
      const kvx_status st = kvx_tp_slice(kv_heads, src_tp, sr, dst_tp, dr, &h0, &g0, &nh);
      if (st != KVX_OK) return st;
      if (nh == 0) continue;
      if (count < max_parts) parts[count] = kvx_head_part{sr, dr, h0, g0, nh, 0};
      ++count;
    }
  *n_parts = count;
  return count > max_parts ? KVX_ERR_INVALID_ARG : KVX_OK;
}

// The same pool apart from its plane addresses: the ranks of one tensor-parallel group.
static bool same_pool(const kvx_layout *a, const kvx_layout *b) {
  return same_rows(a, b) && a->kind == b->kind && a->page_size == b->page_size &&
         a->num_slots == b->num_slots && a->slot_stride == b->slot_stride &&
         a->page_bytes == b->page_bytes;
}

// Layout l of a reshard in device terms: first plane and stride, or (planes not evenly
// spaced) a run of the call's plane table.  False if the table is full.
static bool reshard_layout(kvx::ReshardCall &rc, int32_t idx, const kvx_layout *l) {
  const int64_t stride = l->planes > 1 ? (int64_t)(l->plane[1] - l->plane[0]) : 0;
  bool even = true;
  for (int p = 2; p < l->planes && even; ++p)
    even = l->plane[p] == l->plane[0] + (uintptr_t)((int64_t)p * stride);
  rc.base[idx] = reinterpret_cast<const char *>(l->plane[0]);
  rc.stride[idx] = stride;
  rc.tab[idx] = -1;
  if (even) return true;
  if (rc.n_ptrs + l->planes > kvx::kReshardMaxPtrs) return false;
  rc.tab[idx] = rc.n_ptrs;
  for (int p = 0; p < l->planes; ++p)
    rc.ptrs[rc.n_ptrs++] = reinterpret_cast<const char *>(l->plane[p]);
  return true;
}

// Every host-side check of a reshard, and its device form in rc (the call's Call in c); the
// planner and the copy are not enqueued.
static kvx_status prepare_reshard(const kvx_layout_t *srcs, int32_t n_srcs,
                                  const int32_t *d_src_slots, const kvx_layout_t *dsts,
                                  int32_t n_dsts, const int32_t *d_dst_slots,
                                  const kvx_head_part *parts, int32_t n_parts, int32_t n,
                                  void *d_ws, size_t ws_bytes, Call &c, kvx::ReshardCall &rc) {
  if (!srcs || !dsts || !parts || n_srcs < 1 || n_dsts < 1 ||
      n_srcs + n_dsts > KVX_RESHARD_MAX_LAYOUTS || n_parts < 1 ||
      n_parts > KVX_RESHARD_MAX_PARTS || !valid_n(n))
    return KVX_ERR_INVALID_ARG;
  const kvx_layout *s0 = srcs[0], *d0 = dsts[0];
  if (!s0 || !d0) return KVX_ERR_INVALID_ARG;
  for (int32_t k = 1; k < n_srcs; ++k)
    if (!srcs[k] || !same_pool(srcs[k], s0)) return KVX_ERR_INVALID_ARG;
  for (int32_t k = 1; k < n_dsts; ++k)
    if (!dsts[k] || !same_pool(dsts[k], d0)) return KVX_ERR_INVALID_ARG;
  if (s0->num_layers != d0->num_layers || s0->kv_planes != d0->kv_planes ||
      s0->head_dim != d0->head_dim || s0->elem != d0->elem)
    return KVX_ERR_INVALID_ARG;
  const int32_t nh = parts[0].n_heads;
  for (int32_t k = 0; k < n_parts; ++k) {
    const kvx_head_part &q = parts[k];
    if (q.reserved != 0 || q.n_heads != nh || nh < 1 || q.src < 0 || q.src >= n_srcs ||
        q.dst < 0 || q.dst >= n_dsts)
      return KVX_ERR_INVALID_ARG;
    if (q.src_head0 < 0 || (int64_t)q.src_head0 + nh > s0->kv_heads || q.dst_head0 < 0 ||
        (int64_t)q.dst_head0 + nh > d0->kv_heads)
      return KVX_ERR_INVALID_ARG;
    for (int32_t m = 0; m < k; ++m)  // one writer per destination head
      if (parts[m].dst == q.dst && parts[m].dst_head0 < q.dst_head0 + nh &&
          q.dst_head0 < parts[m].dst_head0 + nh)
        return KVX_ERR_INVALID_ARG;
  }
  for (int32_t k = 0; k < n_dsts; ++k) {
    for (int32_t m = 0; m < n_srcs; ++m)
      if (layouts_overlap(srcs[m], dsts[k])) return KVX_ERR_OVERLAP;
    for (int32_t m = 0; m < k; ++m)
      if (layouts_overlap(dsts[m], dsts[k])) return KVX_ERR_OVERLAP;
  }
  c.op = KVX_OP_TRANSFER;
  c.n_tokens = n;
  c.src = s0;
  c.dst = d0;
  c.shape = s0;
  c.planes = s0->planes;
  c.heads = nh;
  c.seg_bytes = s0->seg_bytes;
  c.row_bytes = (int64_t)nh * c.seg_bytes;
  // the reshard kernel moves 16-byte vectors: every piece must start and end on 16 bytes
  int32_t vec = std::min(std::min(side_vec(s0), side_vec(d0)), pow2_align(c.row_bytes));
  for (int32_t k = 0; k < n_parts; ++k) {
    const int64_t so = head_offset(s0, parts[k].src_head0), dof = head_offset(d0, parts[k].dst_head0);
    if (so) vec = std::min(vec, pow2_align(so));
    if (dof) vec = std::min(vec, pow2_align(dof));
  }
  if (vec < 16) return KVX_ERR_ALIGNMENT;
  c.vec = 16;
  std::memset(&rc, 0, sizeof(rc));
  for (int32_t k = 0; k < n_srcs; ++k)
    if (!reshard_layout(rc, k, srcs[k])) return KVX_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_dsts; ++k)
    if (!reshard_layout(rc, n_srcs + k, dsts[k])) return KVX_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_parts; ++k)
    rc.parts[k] = kvx::ReshardPart{parts[k].src, n_srcs + parts[k].dst,
                                   head_offset(s0, parts[k].src_head0),
                                   head_offset(d0, parts[k].dst_head0)};
  kvx_status st;
  if (n > 0) {
    if (!d_src_slots || !aligned(d_src_slots, 4) || !d_dst_slots || !aligned(d_dst_slots, 4))
      return KVX_ERR_INVALID_ARG;
    if ((st = check_ws(d_ws, ws_bytes, slots_ws(c))) != KVX_OK) return st;
  }
  rc.n_tokens = n;
  rc.planes = c.planes;
  rc.n_parts = n_parts;
  rc.row_bytes = (int32_t)c.row_bytes;
  rc.src = pool_side(s0);
  rc.dst = pool_side(d0);
  rc.src_slots = d_src_slots;
  rc.dst_slots = d_dst_slots;
  return KVX_OK;
}

kvx_status kvx_reshard(const kvx_layout_t *srcs, int32_t n_srcs, const int32_t *d_src_slots,
                       const kvx_layout_t *dsts, int32_t n_dsts, const int32_t *d_dst_slots,
                       const kvx_head_part *parts, int32_t n_parts, int32_t n, void *d_ws,
                       size_t ws_bytes, int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  if (!d_status || !aligned(d_status, 4)) return KVX_ERR_INVALID_ARG;
  Call c;
  if (apply_flags(c, flags) != KVX_OK) return KVX_ERR_INVALID_ARG;
  static thread_local kvx::ReshardCall rc;  // ~30 KB: keep it off the stack
  kvx_status st = prepare_reshard(srcs, n_srcs, d_src_slots, dsts, n_dsts, d_dst_slots, parts,
                                  n_parts, n, d_ws, ws_bytes, c, rc);
  if (st != KVX_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (n == 0) {
    e = cudaMemsetAsync(d_status, 0, sizeof(int32_t), s);
    return e == cudaSuccess ? KVX_OK : cuda_fail(e);
  }
  // the validation: one CTA writes the verdict itself, a multi-tile planner raises it
  const bool direct = kvx::validates_direct(n, true);
  if (!direct) {
    e = cudaMemsetAsync(d_status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  kvx::PlanArgs pa = plan_args(c, d_ws, d_status);
  pa.src_idx = d_src_slots;
  pa.dst_idx = d_dst_slots;
  pa.validate_only = 1;
  if (direct) pa.status_direct = 1;
  if (pa.dup_table) {
    e = cudaMemsetAsync(pa.dup_table, 0, sizeof(unsigned long long) * ((size_t)pa.dup_mask + 1), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = kvx::launch_plan(pa, s);
  if (e != cudaSuccess) return cuda_fail(e);
  rc.status = d_status;
  e = kvx::launch_reshard(rc, s);
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

kvx_status kvx_stream_reshard(const kvx_layout_t *srcs, int32_t n_srcs,
                              const int32_t *d_src_slots, const kvx_layout_t *dsts,
                              int32_t n_dsts, const int32_t *d_dst_slots,
                              const kvx_head_part *parts, int32_t n_parts, int32_t n,
                              const kvx_stream_ctl *ctl, void *d_ws, size_t ws_bytes,
                              int32_t *d_status, uint32_t flags, kvx_stream_t stream) {
  if (!d_status || !aligned(d_status, 16)) return KVX_ERR_INVALID_ARG;
  Call c;
  if (apply_flags(c, flags) != KVX_OK) return KVX_ERR_INVALID_ARG;
  static thread_local kvx::ReshardCall rc;  // ~30 KB: keep it off the stack
  kvx_status st = prepare_reshard(srcs, n_srcs, d_src_slots, dsts, n_dsts, d_dst_slots, parts,
                                  n_parts, n, d_ws, ws_bytes, c, rc);
  if (st != KVX_OK) return st;
  kvx::StreamCtl k = {};
  if ((st = stream_ctl_of(ctl, KVX_OP_TRANSFER, c.shape, &k)) != KVX_OK) return st;
  if (!kvx::reshard_stream_fits(rc, k)) return KVX_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((st = stream_mirror(d_ws, n, s, &k)) != KVX_OK) return st;
  // status[0..3]: verdict, layers pending, stop code, done; as kvx_stream
  const bool direct = kvx::validates_direct(n, true);
  if (!direct) {
    e = cudaMemsetAsync(d_status, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (n > 0) {
    kvx::PlanArgs pa = plan_args(c, d_ws, d_status);
    pa.src_idx = d_src_slots;
    pa.dst_idx = d_dst_slots;
    pa.validate_only = 1;
    if (direct) pa.status_direct = 4;
    if (pa.dup_table) {
      e = cudaMemsetAsync(pa.dup_table, 0, sizeof(unsigned long long) * ((size_t)pa.dup_mask + 1), s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    e = kvx::launch_plan(pa, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  rc.status = d_status;
  if (ctl && ctl->max_ctas > 0) {  // capped persistent grid, one CTA per SM at most
    DeviceInfo di;
    if ((st = device_info(&di)) != KVX_OK) return st;
    const int64_t cap = (int64_t)di.sms * di.bps_reshard_persist;
    e = kvx::launch_reshard_stream_capped(rc, k, (int)std::min<int64_t>(ctl->max_ctas, cap), s);
  } else {
    e = kvx::launch_reshard_stream(rc, k, s);
  }
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

kvx_status kvx_plan_export(const void *d_ws, size_t ws_bytes, int64_t n_tokens,
                           int32_t *d_chunks, int64_t max_chunks, int64_t *d_count,
                           kvx_stream_t stream) {
  if (!valid_n(n_tokens) || max_chunks < 0 || !d_count) return KVX_ERR_INVALID_ARG;
  if (max_chunks > 0 && (!d_chunks || !aligned(d_chunks, 4))) return KVX_ERR_INVALID_ARG;
  const kvx::WsLayout L = kvx::ws_layout(n_tokens, 0, false);
  // the export reads only the header, tile and chunk sections, which do not depend on n_segs
  if (!d_ws || !aligned(d_ws, 256) || (int64_t)ws_bytes < L.prefix_off) return KVX_ERR_NO_WORKSPACE;
  cudaError_t e = kvx::launch_export(static_cast<const char *>(d_ws), L, n_tokens, d_chunks,
                                     max_chunks, d_count, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVX_OK : cuda_fail(e);
}

const char *kvx_status_str(kvx_status s) {
  switch (s) {
    case KVX_OK: return "ok";
    case KVX_ERR_INVALID_ARG: return "invalid argument";
    case KVX_ERR_ALIGNMENT: return "misaligned pointer or row size";
    case KVX_ERR_OUT_OF_RANGE: return "index out of range";
    case KVX_ERR_DUPLICATE_DST: return "duplicate destination";
    case KVX_ERR_OVERLAP: return "source and destination memory overlap";
    case KVX_ERR_CUDA: return "CUDA error";
    case KVX_ERR_NO_WORKSPACE: return "workspace too small or misaligned";
    case KVX_ERR_TIMEOUT: return "timeout";
    case KVX_ERR_CANCELLED: return "cancelled";
    default: return "unknown status";
  }
}

int32_t kvx_last_cuda_error(void) { return g_last_cuda; }

kvx_status kvx_set_fused_max_tokens(int32_t max_tokens) {
  if (max_tokens < 0 || max_tokens > KVX_FUSED_MAX_TOKENS) return KVX_ERR_INVALID_ARG;
  g_fused_max.store(max_tokens, std::memory_order_relaxed);
  return KVX_OK;
}

int32_t kvx_get_fused_max_tokens(void) { return g_fused_max.load(std::memory_order_relaxed); }

kvx_status kvx_set_check_duplicates(int32_t on) {
  if (on != 0 && on != 1) return KVX_ERR_INVALID_ARG;
  g_check_dup.store(on, std::memory_order_relaxed);
  return KVX_OK;
}

int32_t kvx_get_check_duplicates(void) { return g_check_dup.load(std::memory_order_relaxed); }

int32_t kvx_version(void) { return 300; }

}  // extern "C"

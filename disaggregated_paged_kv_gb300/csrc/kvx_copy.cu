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
#include "kvx_internal.cuh"

namespace kvx {
namespace {

constexpr int kUnroll = 4;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

struct Addr {
  const char *base;  // row 0, head 0
  int64_t row;       // bytes between consecutive rows of the chunk
  int64_t head;      // bytes between consecutive head vectors of a row
};

// Address of the chunk's first row on one side.  idx: slot (pool) or row (buffer).  The
// side's geometry stays in the kernel's parameter space (read by reference, not copied).
__device__ __forceinline__ Addr side_addr(const Side &s, bool is_pool, const char *plane,
                                          int64_t idx, const char *buf_plane, int32_t row_bytes) {
  Addr a;
  if (!is_pool) {
    a.base = buf_plane + idx * row_bytes;
    a.row = row_bytes;
    a.head = s.seg_bytes;
  } else if (s.hnd) {
    const int64_t page = idx / s.page_size, off = idx - page * s.page_size;
    a.base = plane + page * s.page_bytes + off * s.seg_bytes;
    a.row = s.seg_bytes;
    a.head = (int64_t)s.page_size * s.seg_bytes;
  } else {
    a.base = plane + idx * s.slot_stride;
    a.row = s.slot_stride;
    a.head = s.seg_bytes;
  }
  return a;
}

__device__ __forceinline__ void copy_linear(const char *src, char *dst, int32_t nvec, int lane) {
  const uint4 *s = reinterpret_cast<const uint4 *>(src);
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  for (int32_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + 32 * u < nvec) r[u] = ld_stream(s + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + 32 * u < nvec) st_stream(d + v0 + 32 * u, r[u]);
  }
}

__device__ __forceinline__ int64_t vec_off(const Addr &a, int32_t v, int32_t vps, int32_t heads) {
  const int32_t q = v / vps, w = v - q * vps;
  const int32_t j = q / heads, h = q - j * heads;
  return j * a.row + h * a.head + (int64_t)w * 16;
}

__device__ __forceinline__ void copy_pieces(const Addr &s, const Addr &d, int32_t nvec,
                                            int32_t vps, int32_t heads, int lane) {
  for (int32_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nvec) r[u] = ld_stream(s.base + vec_off(s, v, vps, heads));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nvec) st_stream(const_cast<char *>(d.base) + vec_off(d, v, vps, heads), r[u]);
    }
  }
}

__device__ __forceinline__ bool header_matches(const CopyArgs &a) {
  const PlanHeader *h = reinterpret_cast<const PlanHeader *>(a.ws + a.L.header_off);
  // slot-list and run-list plans share one chunk format; a batch plan must be run as a batch
  const bool batch = a.mode == kModeBatch;
  return h->magic == kPlanMagic && (h->mode == kModeBatch) == batch && h->op == a.op &&
         (!batch || h->n_segs == a.n_segs) && h->n_tokens == a.n_tokens &&
         h->chunk_rows == a.chunk_rows &&
         h->planes == a.planes && h->row_bytes == a.row_bytes &&
         h->src_is_pool == a.src.is_pool && h->src_hnd == a.src.hnd &&
         h->src_page_size == a.src.page_size && h->dst_is_pool == a.dst.is_pool &&
         h->dst_hnd == a.dst.hnd && h->dst_page_size == a.dst.page_size &&
         h->src_num_slots == a.src.num_slots && h->dst_num_slots == a.dst.num_slots;
}

// kLinear: the host has seen that every chunk is linear on both sides (token-row pools with
// dense rows, and buffers), so the per-vector placement path is compiled out.
template <bool kLinear>
__global__ void __launch_bounds__(kCopyThreads, 4) copy_kernel(const __grid_constant__ CopyArgs a) {
  extern __shared__ int32_t s_tile_base[];  // n_tiles + 1 entries
  __shared__ int32_t s_warp[kCopyThreads / 32];
  __shared__ int32_t s_ok;

  pdl_wait();  // the planner's tables must be complete

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    int32_t ok = header_matches(a) ? 1 : 0;
    if (!ok && blockIdx.x == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_INVALID_ARG);
    if (ok && a.mode != kModeBatch && a.status[0] != KVX_OK) ok = 0;
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;

  // chunk counts of every tile -> first chunk of every tile
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const int32_t *tiles = reinterpret_cast<const int32_t *>(a.ws + a.L.tiles_off);
  int32_t carry = 0;
  for (int32_t base = 0; base < nt; base += kCopyThreads) {
    const int32_t t = base + tid;
    int32_t v = t < nt ? tiles[t] : 0;
    v = v < 0 ? 0 : (v > kTile ? kTile : v);  // never index past a tile's table
    // block exclusive scan
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int32_t wex = 0, tot = 0;
    for (int i = 0; i < kCopyThreads / 32; ++i) {
      if (i < warp) wex += s_warp[i];
      tot += s_warp[i];
    }
    if (t < nt) s_tile_base[t] = carry + wex + x - v;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) s_tile_base[nt] = carry;
  __syncthreads();

  const uint32_t total = (uint32_t)carry * (uint32_t)a.planes;
  const Chunk *chunks = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off);
  const int32_t R = a.row_bytes;
  const int32_t vps = a.seg_bytes >> 4;
  const int32_t *st = a.status;
  const uint32_t nwarps = gridDim.x * (kCopyThreads / 32);

  for (uint32_t w = blockIdx.x * (kCopyThreads / 32) + warp; w < total; w += nwarps) {
    const uint32_t c = w / (uint32_t)a.planes;
    const int32_t p = (int32_t)(w - c * (uint32_t)a.planes);
    int32_t lo = 0, hi = nt;  // tile holding chunk c
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if ((uint32_t)s_tile_base[mid] <= c) lo = mid; else hi = mid;
    }
    const Chunk ch = chunks[(int64_t)lo * kTile + (c - (uint32_t)s_tile_base[lo])];

    int32_t op = a.op;
    const char *bufp = a.buf;
    int64_t nreq = a.n_tokens;
    if (a.mode == kModeBatch) {
      if (st[1 + ch.req] != KVX_OK) continue;
      const kvx_request rq = a.reqs[ch.req];
      op = rq.op;
      bufp = a.buf + rq.buf_off;
      nreq = rq.n_tokens;
    }
    bool src_pool = a.src.is_pool, dst_pool = a.dst.is_pool;
    if (a.mode == kModeBatch) {
      src_pool = (op == KVX_OP_GATHER || op == KVX_OP_TRANSFER);
      dst_pool = (op == KVX_OP_SCATTER || op == KVX_OP_TRANSFER);
    }
    const char *buf_plane = bufp + (int64_t)p * nreq * R;
    const Addr sa = side_addr(a.src, src_pool, a.src_planes[p], ch.src, buf_plane, R);
    const Addr da = side_addr(a.dst, dst_pool, a.dst_planes[p], ch.dst, buf_plane, R);
    const int32_t nvec = ch.rows * (R >> 4);
    if (kLinear) {
      copy_linear(sa.base, const_cast<char *>(da.base), nvec, lane);
    } else {
      const bool linear = sa.head == a.seg_bytes && da.head == a.seg_bytes &&
                          (ch.rows == 1 || (sa.row == R && da.row == R));
      if (linear)
        copy_linear(sa.base, const_cast<char *>(da.base), nvec, lane);
      else
        copy_pieces(sa, da, nvec, vps, a.heads, lane);
    }
  }
}

}  // namespace

int copy_blocks_per_sm(bool linear, int n_tiles) {
  int nb = 0;
  const size_t smem = sizeof(int32_t) * (size_t)(n_tiles + 1);
  const cudaError_t e =
      linear ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, copy_kernel<true>, kCopyThreads, smem)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, copy_kernel<false>, kCopyThreads, smem);
  return e == cudaSuccess ? nb : 0;
}

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

cudaError_t launch_copy(const CopyArgs &a, int grid, cudaStream_t s) {
  const int32_t nt = (int32_t)num_tiles(a.n_tokens);
  const bool lin = copy_is_linear(a);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.dynamicSmemBytes = sizeof(int32_t) * (size_t)(nt + 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {const_cast<CopyArgs *>(&a)};
  const void *fn = lin ? reinterpret_cast<const void *>(copy_kernel<true>)
                       : reinterpret_cast<const void *>(copy_kernel<false>);
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
    // programmatic dependent launch refused on this stream: launch in plain stream order
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  return e;
}

}  // namespace kvx

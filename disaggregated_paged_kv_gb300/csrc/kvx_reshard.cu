// kvx_reshard.cu -- a whole tensor-parallel reshard in one copy launch (sm_103a).
//
// "PD分离调研：从推理阶段拆分到Mooncake的KVCache中心架构", section 7.7 异构TP: when P and D
// run different tensor-parallel sizes, a D rank's shard is put together from head ranges of
// several P ranks' shards (or one P shard is cut up for several D ranks).  kvx_move_heads
// moves one such range; done pair by pair, a reshard from TP 8 to TP 1 is eight planner + copy
// launch pairs over 256-byte pieces, each with its own ramp and tail.  Here one validating
// planner checks the two slot lists once and one row grid moves every part of the plan.
//
// Warp w of grid row y moves G tokens of one (plane, part) pair with m lanes per token (the
// row kernel's shape for the piece length, row_shape_for), parts fastest and planes slowest:
// w = (p * Q + q) * J + j for plane p, token group q of the row's Q, part j.  The J parts
// that fill one destination row run in neighbouring warps of one CTA, so the pieces of a row
// reach L2 together, and the warps in flight at any time cover few planes (measured on a
// TP 8 -> 1 reshard of 2048 tokens x 72 planes: 107.2 us against 111.5 us token-major).
// Grid rows (blockIdx.y) of 4096 token groups keep w small.
// As in the row kernel of kvx_copy.cu, each lane range-checks its token and issues its loads
// before the planner's verdict, and stores only after it (all-or-nothing).
#include <algorithm>

#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"
#include "kvx_reshard.cuh"
#include "kvx_stream_ops.cuh"

namespace kvx {
namespace {

using namespace ops;

constexpr int64_t kGroupsPerRow = 4096;  // token groups per grid row (blockIdx.y)

// The device copy of ReshardCall; kPtrs == 0 drops the table of uneven plane addresses, so a
// call whose layouts are all evenly spaced passes ~5 KB of parameters instead of ~29 KB.
template <int kPtrs>
struct ReshardArgs {
  int64_t n_tokens;
  int32_t planes;
  int32_t n_parts;
  int32_t row_bytes;
  int32_t lanes;        // m lanes per token
  int32_t rows;         // G tokens per warp
  uint32_t groups_per_y;
  Side src, dst;
  int32_t *status;
  const int32_t *src_slots;
  const int32_t *dst_slots;
  const char *base[KVX_RESHARD_MAX_LAYOUTS];
  int64_t stride[KVX_RESHARD_MAX_LAYOUTS];
  int32_t tab[KVX_RESHARD_MAX_LAYOUTS];
  ReshardPart parts[KVX_RESHARD_MAX_PARTS];
  const char *ptrs[kPtrs > 0 ? kPtrs : 1];
};
// kernel parameters are limited to 32,764 bytes
static_assert(sizeof(ReshardArgs<kReshardMaxPtrs>) <= 32764, "reshard parameters too large");

template <int kPtrs>
__device__ __forceinline__ const char *plane_addr(const ReshardArgs<kPtrs> &a, int32_t l,
                                                  int32_t p) {
  if constexpr (kPtrs > 0) {
    const int32_t t = a.tab[l];
    if (t >= 0) return a.ptrs[t + p];
  }
  return a.base[l] + (int64_t)p * a.stride[l];
}

// kTail: rows of more than kUnroll * m vectors, moved in further passes.
template <bool kSrcHnd, bool kDstHnd, bool kTail, int kPtrs>
__global__ void __launch_bounds__(kCopyThreads, kTail && (kSrcHnd || kDstHnd) ? 6 : 8)
    reshard_kernel(const __grid_constant__ ReshardArgs<kPtrs> a) {
  const int lane = threadIdx.x & 31;
  const uint32_t w = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const uint32_t J = (uint32_t)a.n_parts, P = (uint32_t)a.planes;
  const uint32_t r = w / J;
  const int32_t j = (int32_t)(w - r * J);
  const int32_t p = (int32_t)(r / a.groups_per_y);
  const uint32_t qy = r - (uint32_t)p * a.groups_per_y;
  if ((uint32_t)p >= P || qy >= a.groups_per_y) return;
  const int32_t m = a.lanes, G = a.rows;
  // n_tokens <= KVX_MAX_TOKENS (2^23): token indices fit in 32 bits
  const int32_t nt = (int32_t)a.n_tokens;
  const int32_t t0 = (int32_t)((blockIdx.y * a.groups_per_y + qy) * G);
  if (t0 >= nt) return;
  const int32_t rl = lane / m;
  const int32_t li = lane - rl * m;
  const int32_t t = t0 + rl;
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const bool in = rl < G && t < nt;
  const int32_t tt = in ? t : t0;
  const int32_t si = a.src_slots[tt], di = a.dst_slots[tt];
  const bool ok = in && si >= 0 && (int64_t)si < a.src.num_slots && di >= 0 &&
                  (int64_t)di < a.dst.num_slots;
  const ReshardPart &pt = a.parts[j];
  const char *srow =
      row_base<kSrcHnd>(a.src, true, plane_addr(a, pt.src, p) + pt.src_off, nullptr, si, R);
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int32_t xv = li + u * m;
    if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, true, srow, xv << 4));
  }
  pdl_wait();  // the planner has checked both slot lists
  if (a.status[0] != KVX_OK) return;
  if (!ok) return;
  char *drow = const_cast<char *>(row_base<kDstHnd>(
      a.dst, true, plane_addr(a, a.parts[j].dst, p) + a.parts[j].dst_off, nullptr, di, R));
  const int32_t step = kUnroll * m;
#pragma unroll 1
  for (int32_t x0 = 0;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr)
        st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, true, drow, xv << 4)), v[u]);
    }
    if constexpr (!kTail) break;
    x0 += step;
    if (x0 >= vpr) break;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, true, srow, xv << 4));
    }
  }
}

// ---- layer-streamed reshard ---------------------------------------------------------------
// The grid of kvx_stream's row grid over (layer, K/V, token group, part): each layer's items
// padded to whole CTAs, parts fastest within a layer; thread 0 of a CTA waits for the CTA's
// layer (sops::row_wait: the producer's ready word, the request's epoch word, the tagged stop
// word), the rows load once it may go on and store once the planner's verdict is in and, with
// owner epochs, while the destination page still belongs to the request.  The epilogue of
// kvx_stream follows the grid.

template <int kPtrs>
struct ReshardStreamArgs {
  ReshardArgs<kPtrs> r;
  StreamCtl k;
};
static_assert(sizeof(ReshardStreamArgs<kReshardMaxPtrs>) <= 32764, "parameters too large");

constexpr int kRsWarps = kCopyThreads / 32;

template <bool kSrcHnd, bool kDstHnd, bool kTail, int kPtrs>
__global__ void __launch_bounds__(kCopyThreads, kTail && (kSrcHnd || kDstHnd) ? 6 : 8)
    reshard_stream_kernel(const __grid_constant__ ReshardStreamArgs<kPtrs> s) {
  __shared__ int32_t s_go;  // 1: the CTA's layer moves, 0: it stopped
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the epilogue may queue
  const ReshardArgs<kPtrs> &a = s.r;
  const StreamCtl &k = s.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t i0 = blockIdx.x * kRsWarps;  // the CTA's first (padded) item
  const int32_t l = (int32_t)(i0 / k.per_layer_pad);
  const uint32_t r = i0 - (uint32_t)l * k.per_layer_pad + warp;
  const bool has = r < k.per_layer;
  const uint32_t rc = has ? r : 0;
  const uint32_t J = (uint32_t)a.n_parts;
  const uint32_t qq = rc / J;
  const int32_t j = (int32_t)(rc - qq * J);
  const int32_t kv = qq >= k.groups ? 1 : 0;  // K or V (always 0 with one latent plane)
  const int32_t q = (int32_t)(qq - (uint32_t)kv * k.groups);
  const int32_t m = a.lanes, G = a.rows;
  const int32_t rl = lane / m, li = lane - rl * m;
  const int32_t nt = (int32_t)a.n_tokens;
  const int32_t t = q * G + rl;
  bool ok = has && rl < G && t < nt;
  const int32_t tt = ok ? t : 0;
  const int32_t si = a.src_slots[tt], di = a.dst_slots[tt];
  ok = ok && si >= 0 && (int64_t)si < a.src.num_slots && di >= 0 && (int64_t)di < a.dst.num_slots;
  if (threadIdx.x == 0) {
    int32_t go = 1;
    if (k.layer_ready || k.epoch_word) {
      const bool owner = blockIdx.x == (uint32_t)((uint64_t)l * k.per_layer_pad / kRsWarps);
      const int32_t code = sops::row_wait(k, l, owner);
      if (code) {
        go = 0;
        pdl_wait();  // after the planner's status words (as kvx_stream's row grid)
        atomicMax(&a.status[2], code);
        atomicMax(&a.status[1], k.layers - l);
      }
    }
    s_go = go;
  }
  __syncthreads();  // thread 0's acquire of the layer orders every thread's row loads
  if (!s_go) return;  // stopped: this CTA writes nothing
  const int32_t p = k.kv_planes * l + kv;
  const ReshardPart &pt = a.parts[j];
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const char *srow =
      row_base<kSrcHnd>(a.src, true, plane_addr(a, pt.src, p) + pt.src_off, nullptr, si, R);
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int32_t xv = li + u * m;
    if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, true, srow, xv << 4));
  }
  pdl_wait();  // the planner has checked both slot lists and written status[0]
  if (a.status[0] != KVX_OK || !ok) return;
  if (k.page_epochs && !sops::page_owned(k, di)) {
    // the page went to another request: the row is dropped and reported
    atomicMax(&a.status[2], (int32_t)KVX_ERR_CANCELLED);
    atomicMax(&a.status[1], k.layers - l);
    return;
  }
  char *drow = const_cast<char *>(row_base<kDstHnd>(
      a.dst, true, plane_addr(a, a.parts[j].dst, p) + a.parts[j].dst_off, nullptr, di, R));
  const int32_t step = kUnroll * m;
#pragma unroll 1
  for (int32_t x0 = 0;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr)
        st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, true, drow, xv << 4)), v[u]);
    }
    if constexpr (!kTail) break;
    x0 += step;
    if (x0 >= vpr) break;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t xv = x0 + li + u * m;
      if (xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, true, srow, xv << 4));
    }
  }
}

// ---- layer-streamed reshard on a capped persistent grid -----------------------------------
// kvx_stream's capped persistent grid over the streamed reshard's items (layer-major, parts
// fastest within a layer, unpadded): at most max_ctas CTAs of 1024 threads, one per SM, whose
// warps take the CTA's items from a shared counter, one poller per CTA and layer
// (sops::wait_layer), and the last CTA to finish folds the stop codes into the verdict and
// sets the "no further write" words (sops::persistent_cta_exit); no epilogue kernel.

constexpr int kRsPersistThreads = 1024;
constexpr int kRsPersistWarps = kRsPersistThreads / 32;

template <bool kSrcHnd, bool kDstHnd, int kPtrs>
__global__ void __launch_bounds__(kRsPersistThreads, 1)
    reshard_persist_kernel(const __grid_constant__ ReshardStreamArgs<kPtrs> s) {
  __shared__ sops::CtaState cs;
  __shared__ uint32_t next;  // the CTA's next item (in its own order)
  const ReshardArgs<kPtrs> &a = s.r;
  const StreamCtl &k = s.k;
  const int lane = threadIdx.x & 31;
  const int32_t layers = k.layers;
  if (threadIdx.x < sops::kReadyWords) {
    cs.ready[threadIdx.x] = 0;
    cs.polling[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) {
    cs.stop = layers;
    cs.code = 0;
    next = 0;
  }
  __syncthreads();

  const uint32_t J = (uint32_t)a.n_parts;
  const int32_t m = a.lanes, G = a.rows;
  const int32_t rl = lane / m, li = lane - rl * m;
  const int32_t nt = (int32_t)a.n_tokens, R = a.row_bytes, vpr = R >> 4;
  // Item q of this CTA: blocks of bs consecutive items go to the CTAs in turn.
  const uint32_t bs = kRsPersistWarps * k.block;
  auto item_of = [&](uint32_t q) -> uint32_t {
    return ((q / bs) * gridDim.x + blockIdx.x) * bs + q % bs;
  };
  int32_t lcur = -1;
  bool verdict_ok = false;  // this warp has seen the planner's verdict (both lists valid)
  for (;;) {
    uint32_t q = 0;
    if (lane == 0) q = atomicAdd(&next, 1u);
    const uint32_t i = item_of(__shfl_sync(0xffffffffu, q, 0));
    if (i >= k.items) break;
    const int32_t l = (int32_t)(i / k.per_layer);
    if (l != lcur) {
      const bool owner = blockIdx.x == ((uint64_t)l * k.per_layer / bs) % gridDim.x;
      int32_t go = lane == 0 ? sops::wait_layer(k, l, owner, &cs) : 0;
      go = __shfl_sync(0xffffffffu, go, 0);
      __syncwarp();  // lane 0's acquire orders every lane's loads of the layer
      if (!go) break;
      lcur = l;
    }
    const uint32_t r = i - (uint32_t)l * k.per_layer;
    const uint32_t qq = r / J;
    const int32_t j = (int32_t)(r - qq * J);
    const int32_t kv = qq >= k.groups ? 1 : 0;  // K or V (always 0 with one latent plane)
    const int32_t t = (int32_t)(qq - (uint32_t)kv * k.groups) * G + rl;
    bool ok = rl < G && t < nt;
    const int32_t tt = ok ? t : 0;
    const int32_t si = a.src_slots[tt], di = a.dst_slots[tt];
    ok = ok && si >= 0 && (int64_t)si < a.src.num_slots && di >= 0 && (int64_t)di < a.dst.num_slots;
    const int32_t p = k.kv_planes * l + kv;
    const ReshardPart &pt = a.parts[j];
    const char *srow =
        row_base<kSrcHnd>(a.src, true, plane_addr(a, pt.src, p) + pt.src_off, nullptr, si, R);
    char *drow = const_cast<char *>(
        row_base<kDstHnd>(a.dst, true, plane_addr(a, pt.dst, p) + pt.dst_off, nullptr, di, R));
#pragma unroll 1
    for (int32_t x0 = 0; x0 < vpr; x0 += kUnroll * m) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t xv = x0 + li + u * m;
        if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, true, srow, xv << 4));
      }
      if (!verdict_ok) {
        pdl_wait();  // the planner has checked both slot lists and written status[0]
        if (a.status[0] != KVX_OK) {
          if (lane == 0) atomicMin(&cs.stop, 0);
          break;
        }
        verdict_ok = true;
      }
      if (x0 == 0 && ok && k.page_epochs && !sops::page_owned(k, di)) {
        // the page went to another request: the piece is dropped and reported
        ok = false;
        atomicMax(&cs.code, (int32_t)KVX_ERR_CANCELLED);
        atomicMax(&a.status[1], layers - l);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t xv = x0 + li + u * m;
        if (ok && xv < vpr)
          st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, true, drow, xv << 4)), v[u]);
      }
    }
    if (!verdict_ok) break;
  }

  // every thread's writes before this CTA's report; the last CTA's release covers all CTAs
  pdl_wait();  // the planner's status words are written before any CTA reports
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) sops::persistent_cta_exit(a.status, k, cs, layers);
}

template <int kPtrs>
const void *reshard_persist_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(reshard_persist_kernel<true, true, kPtrs>);
  if (sh) return reinterpret_cast<const void *>(reshard_persist_kernel<true, false, kPtrs>);
  if (dh) return reinterpret_cast<const void *>(reshard_persist_kernel<false, true, kPtrs>);
  return reinterpret_cast<const void *>(reshard_persist_kernel<false, false, kPtrs>);
}

template <bool kTail, int kPtrs>
const void *reshard_stream_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(reshard_stream_kernel<true, true, kTail, kPtrs>);
  if (sh) return reinterpret_cast<const void *>(reshard_stream_kernel<true, false, kTail, kPtrs>);
  if (dh) return reinterpret_cast<const void *>(reshard_stream_kernel<false, true, kTail, kPtrs>);
  return reinterpret_cast<const void *>(reshard_stream_kernel<false, false, kTail, kPtrs>);
}

// Items of one layer of a streamed reshard (padded to whole CTAs), and the row shape.
struct RsSizes {
  int32_t m, G;
  int64_t groups, per_layer, per_layer_pad;
};

RsSizes rs_sizes(const ReshardCall &c, const StreamCtl &k) {
  RsSizes z;
  row_shape_for(c.row_bytes, &z.m, &z.G);
  z.groups = (c.n_tokens + z.G - 1) / z.G;
  z.per_layer = (int64_t)k.kv_planes * z.groups * c.n_parts;
  z.per_layer_pad = (z.per_layer + kRsWarps - 1) / kRsWarps * kRsWarps;
  return z;
}

template <int kPtrs>
cudaError_t launch_persist_with(const ReshardCall &c, const StreamCtl &k, const RsSizes &z,
                                int grid, cudaStream_t s) {
  static thread_local ReshardStreamArgs<kPtrs> args;  // up to ~29 KB: keep it off the stack
  fill_args(args.r, c, z.m, z.G, 0);
  args.k = k;
  void *params[] = {&args};
  return launch_pdl(reshard_persist_fn<kPtrs>(c.src.hnd != 0, c.dst.hnd != 0),
                    dim3((unsigned)grid), dim3(kRsPersistThreads), params, s);
}

template <int kPtrs>
cudaError_t launch_stream_with(const ReshardCall &c, const StreamCtl &k, const RsSizes &z,
                               cudaStream_t s) {
  static thread_local ReshardStreamArgs<kPtrs> args;  // up to ~29 KB: keep it off the stack
  fill_args(args.r, c, z.m, z.G, 0);
  args.k = k;
  const bool sh = c.src.hnd != 0, dh = c.dst.hnd != 0;
  const bool tail = (c.row_bytes >> 4) > kUnroll * z.m;
  const void *fn = tail ? reshard_stream_fn<true, kPtrs>(sh, dh)
                        : reshard_stream_fn<false, kPtrs>(sh, dh);
  void *params[] = {&args};
  return launch_pdl(fn, dim3((unsigned)(k.per_layer_pad / kRsWarps * k.layers)),
                    dim3(kCopyThreads), params, s);
}

template <bool kTail, int kPtrs>
const void *reshard_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(reshard_kernel<true, true, kTail, kPtrs>);
  if (sh) return reinterpret_cast<const void *>(reshard_kernel<true, false, kTail, kPtrs>);
  if (dh) return reinterpret_cast<const void *>(reshard_kernel<false, true, kTail, kPtrs>);
  return reinterpret_cast<const void *>(reshard_kernel<false, false, kTail, kPtrs>);
}

template <int kPtrs>
void fill_args(ReshardArgs<kPtrs> &a, const ReshardCall &c, int32_t m, int32_t G, uint32_t per_y) {
  a.n_tokens = c.n_tokens;
  a.planes = c.planes;
  a.n_parts = c.n_parts;
  a.row_bytes = c.row_bytes;
  a.lanes = m;
  a.rows = G;
  a.groups_per_y = per_y;
  a.src = c.src;
  a.dst = c.dst;
  a.status = c.status;
  a.src_slots = c.src_slots;
  a.dst_slots = c.dst_slots;
  for (int l = 0; l < KVX_RESHARD_MAX_LAYOUTS; ++l) {
    a.base[l] = c.base[l];
    a.stride[l] = c.stride[l];
    a.tab[l] = kPtrs > 0 ? c.tab[l] : -1;
  }
  for (int k = 0; k < KVX_RESHARD_MAX_PARTS; ++k) a.parts[k] = c.parts[k];
  for (int k = 0; k < kPtrs; ++k) a.ptrs[k] = k < c.n_ptrs ? c.ptrs[k] : nullptr;
}

template <int kPtrs>
cudaError_t launch_with(const ReshardCall &c, int32_t m, int32_t G, uint32_t per_y, dim3 grid,
                        cudaStream_t s) {
  static thread_local ReshardArgs<kPtrs> a;  // up to ~29 KB: keep it off the stack
  fill_args(a, c, m, G, per_y);
  const bool sh = c.src.hnd != 0, dh = c.dst.hnd != 0;
  const bool tail = (c.row_bytes >> 4) > kUnroll * m;  // more than one pass
  const void *fn = tail ? reshard_fn<true, kPtrs>(sh, dh) : reshard_fn<false, kPtrs>(sh, dh);
  void *params[] = {&a};
  return launch_pdl(fn, grid, dim3(kCopyThreads), params, s);
}

}  // namespace

bool reshard_stream_fits(const ReshardCall &c, const StreamCtl &k) {
  const RsSizes z = rs_sizes(c, k);
  return z.per_layer_pad * k.layers <= (int64_t)0x7fffffff;  // 32-bit item indices
}

cudaError_t launch_reshard_stream(const ReshardCall &c, StreamCtl k, cudaStream_t s) {
  const RsSizes z = rs_sizes(c, k);
  k.groups = (uint32_t)z.groups;
  k.per_layer = (uint32_t)z.per_layer;
  k.per_layer_pad = (uint32_t)z.per_layer_pad;
  k.items = (uint32_t)(z.per_layer * k.layers);
  cudaError_t e = cudaSuccess;
  if (c.n_tokens > 0)
    e = c.n_ptrs > 0 ? launch_stream_with<kReshardMaxPtrs>(c, k, z, s)
                     : launch_stream_with<0>(c, k, z, s);
  if (e != cudaSuccess) return e;
  return launch_stream_done(c.status, k.host_done, k.layers, s);
}

int reshard_persist_blocks_per_sm() {
  int nb = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &nb, reshard_persist_fn<kReshardMaxPtrs>(false, false), kRsPersistThreads, 0);
  return e == cudaSuccess ? nb : 0;
}

cudaError_t launch_reshard_stream_capped(const ReshardCall &c, StreamCtl k, int max_grid,
                                         cudaStream_t s) {
  const RsSizes z = rs_sizes(c, k);
  k.groups = (uint32_t)z.groups;
  k.per_layer = (uint32_t)z.per_layer;
  k.items = (uint32_t)(z.per_layer * k.layers);
  if (k.items == 0)  // nothing to move: the epilogue alone writes the status words
    return launch_stream_done(c.status, k.host_done, k.layers, s);
  const int64_t warps = k.items;
  int64_t grid = std::min<int64_t>(max_grid, (warps + kRsPersistWarps - 1) / kRsPersistWarps);
  if (grid < 1) grid = 1;
  // about four blocks per warp: few layer entries per warp, each layer spread over many warps
  const int64_t per_warp = (warps + grid * kRsPersistWarps - 1) / (grid * kRsPersistWarps);
  k.block = (uint32_t)std::min<int64_t>(std::max<int64_t>(per_warp / 4, 1), 8);
  return c.n_ptrs > 0 ? launch_persist_with<kReshardMaxPtrs>(c, k, z, (int)grid, s)
                      : launch_persist_with<0>(c, k, z, (int)grid, s);
}

cudaError_t launch_reshard(const ReshardCall &c, cudaStream_t s) {
  // lanes per token and tokens per warp: the row kernel's shape for this piece length
  int32_t m = 32, G = 1;
  row_shape_for(c.row_bytes, &m, &G);
  const int64_t groups = (c.n_tokens + G - 1) / G;
  const int64_t pj = (int64_t)c.planes * c.n_parts;  // at most 256 x 128 = 2^15
  // grid rows of at most 4096 token groups: warp indices of a row stay below 2^27, and the
  // rows number at most 2^23 / 4096 = 2048
  const int64_t per_y = groups < kGroupsPerRow ? groups : kGroupsPerRow;
  const int64_t warps = per_y * pj;
  const int64_t gx = (warps + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int64_t gy = (groups + per_y - 1) / per_y;
  const dim3 grid((unsigned)gx, (unsigned)gy);
  return c.n_ptrs > 0 ? launch_with<kReshardMaxPtrs>(c, m, G, (uint32_t)per_y, grid, s)
                      : launch_with<0>(c, m, G, (uint32_t)per_y, grid, s);
}

}  // namespace kvx

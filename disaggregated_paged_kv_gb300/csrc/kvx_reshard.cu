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
// row kernel's shape for the piece length, row_shape_for), parts fastest:
// w = (q * P + p) * J + j for token group q, plane p, part j.  The J parts that fill one
// destination row therefore run in neighbouring warps of one CTA, and the pieces of a row
// reach L2 together.  Grid rows (blockIdx.y) of 4096 token groups keep w small.
// As in the row kernel of kvx_copy.cu, each lane range-checks its token and issues its loads
// before the planner's verdict, and stores only after it (all-or-nothing).
#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"
#include "kvx_reshard.cuh"

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
  const uint32_t qy = r / P;
  const int32_t p = (int32_t)(r - qy * P);
  if (qy >= a.groups_per_y) return;
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
  if (*reinterpret_cast<volatile const int32_t *>(a.status) != KVX_OK) return;
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

template <bool kTail, int kPtrs>
const void *reshard_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(reshard_kernel<true, true, kTail, kPtrs>);
  if (sh) return reinterpret_cast<const void *>(reshard_kernel<true, false, kTail, kPtrs>);
  if (dh) return reinterpret_cast<const void *>(reshard_kernel<false, true, kTail, kPtrs>);
  return reinterpret_cast<const void *>(reshard_kernel<false, false, kTail, kPtrs>);
}

template <int kPtrs>
cudaError_t launch_with(const ReshardCall &c, int32_t m, int32_t G, uint32_t per_y, dim3 grid,
                        cudaStream_t s) {
  static thread_local ReshardArgs<kPtrs> a;  // up to ~29 KB: keep it off the stack
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
  const bool sh = c.src.hnd != 0, dh = c.dst.hnd != 0;
  const bool tail = (c.row_bytes >> 4) > kUnroll * m;  // more than one pass
  const void *fn = tail ? reshard_fn<true, kPtrs>(sh, dh) : reshard_fn<false, kPtrs>(sh, dh);
  void *params[] = {&a};
  return launch_pdl(fn, grid, dim3(kCopyThreads), params, s);
}

}  // namespace

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

// kvx_narrow.cu -- moves of rows that do not allow 16-byte accesses (sm_103a).
//
// The fast kernels move 16-byte vectors, which needs every row start, row length and (on an
// HND side) head vector to be a multiple of 16 bytes.  Rows of other shapes -- a head_dim of
// 100 fp16 (200-byte rows), 72 fp8 elements, a plane base on an 8-byte boundary -- move here
// in the widest access V (8, 4, 2 or 1 bytes; 16 when only the head vectors are narrow) that
// every address of the call allows, which the host works out from the layouts.
//
// One warp per group of 1 << g tokens of one plane (a power of two, unlike the row kernel of
// kvx_copy.cu, which may give a token any number of lanes), CTAs in plane-major order as the
// row kernel's (measured on 200-byte rows of 16,384 random tokens: 159.3 -> 132.9 us; with all
// writes in flight inside one plane, neighbouring rows' partial sectors meet in L2): 32 >> g
// lanes per row, enough for the lane's kUnroll independent loads to cover the row
// (narrow_group_shift).  One-shot calls read the slot lists, range-check them and load
// before the planner's verdict; plans (one row per chunk, including a batch's request
// records, lane by lane) are read after the planner.
#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"

namespace kvx {
namespace {

using namespace ops;

template <int V> struct Word;
template <> struct Word<16> { using T = uint4; };
template <> struct Word<8> { using T = unsigned long long; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<2> { using T = uint16_t; };
template <> struct Word<1> { using T = uint8_t; };

// Independent loads in flight per lane (measured on 200-byte rows: 4 beats 8, which halves the
// warps for the same rows).
__host__ __device__ constexpr int unroll_for(int) { return kUnroll; }

// The lanes of one row (1 << lsh of them, lane li among them) move its nv V-byte words.  In a
// one-shot call (spec) the first pass's loads go out before the planner's verdict and the
// stores wait for it; the range checks already done by the lane keep every load in bounds.
template <int V, bool kSrcHnd, bool kDstHnd>
__device__ __forceinline__ void move_rows(const CopyArgs &a, bool sp, const char *srow, bool dp,
                                          char *drow, int32_t li, int32_t lsh, bool ok,
                                          bool spec) {
  using T = typename Word<V>::T;
  constexpr int U = unroll_for(V);
  const int32_t nv = a.row_bytes / V;
  T r[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int32_t v = li + (u << lsh);
    if (ok && v < nv) r[u] = *reinterpret_cast<const T *>(row_byte<kSrcHnd>(a.src, sp, srow, v * V));
  }
  if (spec) {
    pdl_wait();  // the planner has checked every index of the request
    if (a.status[0] != KVX_OK) return;
  }
  if (!ok) return;
  for (int32_t v0 = li;;) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t v = v0 + (u << lsh);
      if (v < nv)
        *reinterpret_cast<T *>(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, v * V))) = r[u];
    }
    v0 += U << lsh;
    if (v0 >= nv) break;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t v = v0 + (u << lsh);
      if (v < nv) r[u] = *reinterpret_cast<const T *>(row_byte<kSrcHnd>(a.src, sp, srow, v * V));
    }
  }
}

template <bool kSrcHnd, bool kDstHnd>
__global__ void __launch_bounds__(kCopyThreads) copy_narrow_kernel(const __grid_constant__ CopyArgs a) {
  const int lane = threadIdx.x & 31;
  // plane-major CTAs, as the row kernel: CTA c works on plane c / row_blocks
  const uint32_t pc = blockIdx.x / a.row_blocks;
  const int32_t p = (int32_t)pc;
  const uint32_t q = (blockIdx.x - pc * a.row_blocks) * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const int32_t gsh = a.row_group_shift;  // 1 << gsh tokens per warp
  const int32_t lsh = 5 - gsh;            // 1 << lsh lanes per token
  const int64_t t0 = (int64_t)q << gsh;
  if (t0 >= a.n_tokens) return;
  const int64_t t = t0 + (lane >> lsh);
  const int32_t li = lane & ((1 << lsh) - 1);
  bool ok = t < a.n_tokens;
  const int64_t tt = ok ? t : t0;
  bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const char *bufp = a.buf;
  int64_t nreq = a.n_tokens;
  int32_t si, di;
  const bool spec = a.spec_src || a.spec_dst;
  if (spec) {
    si = sp ? a.spec_src[tt] : (int32_t)tt;
    di = dp ? a.spec_dst[tt] : (int32_t)tt;
    ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
         (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
  } else {
    pdl_wait();  // the plan is complete
    const bool batch = a.mode == kModeBatch;
    if (!header_matches(a)) {
      if (q == 0 && p == 0 && lane == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_INVALID_ARG);
      return;
    }
    const Chunk ch = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off)[tt];  // one row each
    if (batch) {
      // tokens of one warp may belong to different requests: each lane follows its own
      if (a.status[1 + ch.req] != KVX_OK) ok = false;
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
  const int32_t R = a.row_bytes;
  const char *buf_plane = bufp + (int64_t)p * nreq * R;
  const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
  char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
  switch (a.vec_bytes) {
    case 16: move_rows<16, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, li, lsh, ok, spec); break;
    case 8: move_rows<8, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, li, lsh, ok, spec); break;
    case 4: move_rows<4, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, li, lsh, ok, spec); break;
    case 2: move_rows<2, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, li, lsh, ok, spec); break;
    default: move_rows<1, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, li, lsh, ok, spec); break;
  }
}

}  // namespace

int32_t narrow_group_shift(int32_t row_bytes, int32_t vec_bytes) {
  // lanes per row: a power of two >= the row's words / kUnroll, at most 32
  const int32_t nv = row_bytes / vec_bytes;
  int32_t lanes = 1;
  while (lanes < 32 && lanes * unroll_for(vec_bytes) < nv) lanes <<= 1;
  int32_t g = 0;
  while ((32 >> g) > lanes) ++g;
  return g;
}

int narrow_kernel_list(const void **out, int max) {
  const void *k[] = {reinterpret_cast<const void *>(copy_narrow_kernel<true, true>),
                     reinterpret_cast<const void *>(copy_narrow_kernel<true, false>),
                     reinterpret_cast<const void *>(copy_narrow_kernel<false, true>),
                     reinterpret_cast<const void *>(copy_narrow_kernel<false, false>)};
  return kernel_list_out(k, 4, out, max);
}

cudaError_t launch_narrow(CopyArgs &a, cudaStream_t s) {
  // an HND side only matters where the request uses it as a pool
  const bool sh = a.src.hnd && (a.src.is_pool || a.mode == kModeBatch);
  const bool dh = a.dst.hnd && (a.dst.is_pool || a.mode == kModeBatch);
  const void *fn = sh && dh ? reinterpret_cast<const void *>(copy_narrow_kernel<true, true>)
                 : sh       ? reinterpret_cast<const void *>(copy_narrow_kernel<true, false>)
                 : dh       ? reinterpret_cast<const void *>(copy_narrow_kernel<false, true>)
                            : reinterpret_cast<const void *>(copy_narrow_kernel<false, false>);
  const int64_t groups = (a.n_tokens + (1 << a.row_group_shift) - 1) >> a.row_group_shift;
  const int64_t wpb = kCopyThreads / 32;
  a.row_blocks = (uint32_t)((groups + wpb - 1) / wpb);
  const int64_t grid = (int64_t)a.row_blocks * a.planes;
  void *args[] = {const_cast<CopyArgs *>(&a)};
  return launch_pdl(fn, dim3((unsigned)grid), dim3(kCopyThreads), args, s);
}

}  // namespace kvx

// kvx_narrow.cu -- moves of rows that do not allow 16-byte accesses (sm_103a).
//
// The fast kernels move 16-byte vectors, which needs every row start, row length and (on an
// HND side) head vector to be a multiple of 16 bytes.  Rows of other shapes -- a head_dim of
// 100 fp16 (200-byte rows), 72 fp8 elements, a plane base on an 8-byte boundary -- move here
// in the widest access V (8, 4, 2 or 1 bytes; 16 when only the head vectors are narrow) that
// every address of the call allows, which the host works out from the layouts.
//
// One warp per (token, plane) row, as the row kernel of kvx_copy.cu but without its
// speculation: the warp waits for the planner, then reads its token's indices (one-shot calls:
// the slot lists; otherwise chunk t of a one-row-per-chunk plan, including a batch's request
// record) and moves the row with kUnroll independent V-byte loads in flight per lane.
#include "kvx_copy_ops.cuh"

namespace kvx {
namespace {

using namespace ops;

template <int V> struct Word;
template <> struct Word<16> { using T = uint4; };
template <> struct Word<8> { using T = unsigned long long; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<2> { using T = uint16_t; };
template <> struct Word<1> { using T = uint8_t; };

template <int V, bool kSrcHnd, bool kDstHnd>
__device__ __forceinline__ void move_row(const CopyArgs &a, bool sp, const char *srow, bool dp,
                                         char *drow, int lane) {
  using T = typename Word<V>::T;
  const int32_t nv = a.row_bytes / V;
  for (int32_t v0 = lane; v0 < nv; v0 += 32 * kUnroll) {
    T r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nv) r[u] = *reinterpret_cast<const T *>(row_byte<kSrcHnd>(a.src, sp, srow, v * V));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nv)
        *reinterpret_cast<T *>(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, v * V))) = r[u];
    }
  }
}

template <bool kSrcHnd, bool kDstHnd>
__global__ void __launch_bounds__(kCopyThreads) copy_narrow_kernel(const __grid_constant__ CopyArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t w = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const uint32_t P = (uint32_t)a.planes;
  const uint32_t t = w / P;
  const int32_t p = (int32_t)(w - t * P);
  if (t >= a.n_tokens) return;
  bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const char *bufp = a.buf;
  int64_t nreq = a.n_tokens;
  int32_t si, di;
  pdl_wait();  // the planner has checked every index (and written the plan)
  if (a.spec_src || a.spec_dst) {
    if (*reinterpret_cast<volatile const int32_t *>(a.status) != KVX_OK) return;
    si = sp ? a.spec_src[t] : (int32_t)t;
    di = dp ? a.spec_dst[t] : (int32_t)t;
  } else {
    const bool batch = a.mode == kModeBatch;
    if (!header_matches(a)) {
      if (w == 0 && lane == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_INVALID_ARG);
      return;
    }
    const Chunk ch = reinterpret_cast<const Chunk *>(a.ws + a.L.chunks_off)[t];  // one row each
    if (batch) {
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
  const int32_t R = a.row_bytes;
  const char *buf_plane = bufp + (int64_t)p * nreq * R;
  const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
  char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
  switch (a.vec_bytes) {
    case 16: move_row<16, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, lane); break;
    case 8: move_row<8, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, lane); break;
    case 4: move_row<4, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, lane); break;
    case 2: move_row<2, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, lane); break;
    default: move_row<1, kSrcHnd, kDstHnd>(a, sp, srow, dp, drow, lane); break;
  }
}

}  // namespace

cudaError_t launch_narrow(const CopyArgs &a, cudaStream_t s) {
  // an HND side only matters where the request uses it as a pool
  const bool sh = a.src.hnd && (a.src.is_pool || a.mode == kModeBatch);
  const bool dh = a.dst.hnd && (a.dst.is_pool || a.mode == kModeBatch);
  const void *fn = sh && dh ? reinterpret_cast<const void *>(copy_narrow_kernel<true, true>)
                 : sh       ? reinterpret_cast<const void *>(copy_narrow_kernel<true, false>)
                 : dh       ? reinterpret_cast<const void *>(copy_narrow_kernel<false, true>)
                            : reinterpret_cast<const void *>(copy_narrow_kernel<false, false>);
  const int64_t warps = a.n_tokens * (int64_t)a.planes;
  const int64_t grid = (warps + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  void *args[] = {const_cast<CopyArgs *>(&a)};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
    (void)cudaGetLastError();  // no programmatic dependent launch here: plain stream order
    cfg.numAttrs = 0;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  return e;
}

}  // namespace kvx

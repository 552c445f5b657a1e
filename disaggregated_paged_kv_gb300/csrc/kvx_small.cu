// kvx_small.cu -- one-launch gather / scatter / transfer of a small request (sm_103a).
//
// "穷人版 PD 分离", section "5090：一个看得见所有卡的代理": a request's cost is set by its
// fragments and fixed overheads, not its bytes, once it is small.  A request of a few hundred
// tokens (a decode-time handoff, a short prompt) moves a few MB: the planner launch and the
// copy's wait for it then take as long as the data.  Here the row kernel's warps (m lanes per
// token, G tokens per warp, loads issued first) do without the planner: every CTA reads and
// range-checks every index of the request itself -- at most kSmallMaxTokens per list, one or
// two coalesced loads per thread -- so all CTAs reach the same verdict and the move stays
// all-or-nothing without any wait between CTAs.  CTA 0 writes the status word.
#include "kvx_copy_ops.cuh"
#include "kvx_launch.cuh"

namespace kvx {
namespace {

using namespace ops;

constexpr int kIdxPerThread = kSmallMaxTokens / kCopyThreads;
static_assert(kIdxPerThread * kCopyThreads == kSmallMaxTokens, "whole index loads per thread");

template <bool kSrcHnd, bool kDstHnd, bool kTail>
__global__ void __launch_bounds__(kCopyThreads, kTail && (kSrcHnd || kDstHnd) ? 6 : 8)
    copy_small_kernel(const __grid_constant__ CopyArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t w = blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const uint32_t P = (uint32_t)a.planes;
  const uint32_t q = w / P;
  const int32_t p = (int32_t)(w - q * P);
  pdl_wait();  // whatever ran before on the stream is complete: its writes are visible
  const int32_t m = a.row_lanes, G = a.rows_per_warp;
  const int32_t n = (int32_t)a.n_tokens;  // <= kSmallMaxTokens
  const int32_t t0 = (int32_t)q * G;
  const int32_t rl = lane / m, li = lane - rl * m;
  const int32_t t = t0 + rl;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  bool ok = t0 < n && rl < G && t < n;  // no early exit: every thread takes the barrier
  const int32_t tt = ok ? t : 0;
  const int32_t si = sp ? a.spec_src[tt] : tt;
  const int32_t di = dp ? a.spec_dst[tt] : tt;
  ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
       (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const char *buf_plane = a.buf + (int64_t)p * n * R;
  const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
  char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int32_t xv = li + u * m;
    if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
  }
  // every index of the request, all loads issued before any is tested
  int32_t sv[kIdxPerThread], dv[kIdxPerThread];
#pragma unroll
  for (int k = 0; k < kIdxPerThread; ++k) {
    const int32_t i = threadIdx.x + k * kCopyThreads;
    sv[k] = sp && i < n ? a.spec_src[i] : 0;
    dv[k] = dp && i < n ? a.spec_dst[i] : 0;
  }
  int bad = 0;
#pragma unroll
  for (int k = 0; k < kIdxPerThread; ++k)
    bad |= (sv[k] < 0 || (int64_t)sv[k] >= (sp ? a.src.num_slots : 1)) |
           (dv[k] < 0 || (int64_t)dv[k] >= (dp ? a.dst.num_slots : 1));
  bad = __syncthreads_or(bad);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int32_t verdict = bad ? (int32_t)KVX_ERR_OUT_OF_RANGE : (int32_t)KVX_OK;
    *a.status = verdict;
    if (a.host_status) {  // kvx_submit: the caller's pinned word, through its device mapping
      *reinterpret_cast<volatile int32_t *>(a.host_status) = verdict;
      __threadfence_system();
    }
  }
  if (bad || !ok) return;
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

template <bool kTail>
const void *small_fn_of(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(copy_small_kernel<true, true, kTail>);
  if (sh) return reinterpret_cast<const void *>(copy_small_kernel<true, false, kTail>);
  if (dh) return reinterpret_cast<const void *>(copy_small_kernel<false, true, kTail>);
  return reinterpret_cast<const void *>(copy_small_kernel<false, false, kTail>);
}

}  // namespace

int small_kernel_list(const void **out, int max) {
  const void *k[8];
  int n = 0;
  for (int sh = 0; sh < 2; ++sh)
    for (int dh = 0; dh < 2; ++dh) {
      k[n++] = small_fn_of<false>(sh, dh);
      k[n++] = small_fn_of<true>(sh, dh);
    }
  return kernel_list_out(k, n, out, max);
}

cudaError_t launch_small(const CopyArgs &a, cudaStream_t s) {
  const bool sh = a.src.hnd && a.src.is_pool, dh = a.dst.hnd && a.dst.is_pool;
  const bool tail = (a.row_bytes >> 4) > kUnroll * a.row_lanes;  // more than one pass
  const void *fn = tail ? small_fn_of<true>(sh, dh) : small_fn_of<false>(sh, dh);
  const int64_t warps = (a.n_tokens + a.rows_per_warp - 1) / a.rows_per_warp * a.planes;
  const int64_t grid = (warps + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  void *args[] = {const_cast<CopyArgs *>(&a)};
  return launch_pdl(fn, dim3((unsigned)grid), dim3(kCopyThreads), args, s);
}

}  // namespace kvx

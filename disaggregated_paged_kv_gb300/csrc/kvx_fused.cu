// kvx_fused.cu -- gather / scatter / transfer of one request in a single launch (sm_103a).
//
// For a request of up to kFusedMaxTokens tokens the separate planner launch, the plan
// header / tile reads and the status reset cost more than the planning itself ("DistServe
// 完全拆解", KV Cache 跨实例传输: T = B_KV / BW_eff + T_setup; for a 288 MiB request the
// setup term was ~8 us of ~110).  So every CTA of one persistent grid:
//   1. reads and range-checks every index of the request (all CTAs see the same verdict, so
//      the move stays all-or-nothing without any inter-CTA wait), staging the indices in
//      shared memory when they fit; CTA 0 writes the status word;
//   2. takes an equal slice of the plane-major work space (plane p, token t) -> p * n + t;
//   3. for each (plane, token range) segment of its slice, finds the runs of consecutive
//      source and destination indices with block-wide scans (the same break rules as the
//      planner, with the segment as the tile) and cuts them into chunks of <= chunk_rows rows;
//   4. moves the chunks with the same warp copy as the two-launch path.
#include "kvx_copy_ops.cuh"

namespace kvx {
namespace {

using namespace ops;

constexpr int kFThreads = 256;
constexpr int kFItems = 2;                     // tokens per thread when planning a segment
constexpr int kFSeg = kFThreads * kFItems;     // most tokens planned at once
constexpr int kFStage = 1024;                  // indices staged in shared memory up to this n

struct FusedArgs {
  CopyArgs c;  // mode = slots; sides, planes, buffer, status
  const int32_t *src_idx;
  const int32_t *dst_idx;
  int32_t n;
  int32_t chunk_rows;
};

template <int THREADS>
__device__ __forceinline__ int32_t block_scan_excl(int32_t v, int32_t *total, int32_t *s_warp) {
  constexpr int kWarps = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int32_t wex = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    const int32_t w = s_warp[i];
    wex += i < warp ? w : 0;
    tot += w;
  }
  *total = tot;
  __syncthreads();
  return wex + x - v;
}

template <bool kLinear>
__global__ void __launch_bounds__(kFThreads, kLinear ? 8 : 4)
    fused_kernel(const __grid_constant__ FusedArgs f) {
  __shared__ int32_t s_si[kFStage];      // staged source indices
  __shared__ int32_t s_di[kFStage];      // staged destination indices
  __shared__ int32_t s_tok[kFSeg];       // segment-relative first token of run r
  __shared__ int32_t s_rs[kFSeg];        // first source index of run r
  __shared__ int32_t s_rd[kFSeg];        // first destination index of run r
  __shared__ int32_t s_coff[kFSeg + 1];  // first chunk of run r
  __shared__ int32_t s_warp[kFThreads / 32];

  const CopyArgs &a = f.c;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const int32_t n = f.n;
  const bool staged = n <= kFStage;

  // 1. every index, checked by every CTA; the loads of a batch of 4 per thread are all
  //    issued before any of them is used
  int bad = 0;
  for (int32_t base = 0; base < n; base += 4 * kFThreads) {
    int32_t sv4[4], dv4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int32_t i = base + k * kFThreads + tid;
      sv4[k] = (sp && i < n) ? __ldg(f.src_idx + i) : 0;
      dv4[k] = (dp && i < n) ? __ldg(f.dst_idx + i) : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int32_t i = base + k * kFThreads + tid;
      if (i < n) {
        bad |= (sp && (sv4[k] < 0 || (int64_t)sv4[k] >= a.src.num_slots)) ? 1 : 0;
        bad |= (dp && (dv4[k] < 0 || (int64_t)dv4[k] >= a.dst.num_slots)) ? 1 : 0;
        if (staged) {
          s_si[i] = sv4[k];
          s_di[i] = dv4[k];
        }
      }
    }
  }
  bad = __syncthreads_or(bad);
  if (blockIdx.x == 0 && tid == 0) a.status[0] = bad ? KVX_ERR_OUT_OF_RANGE : KVX_OK;
  if (bad) return;

  // source / destination index of token t (a buffer side's index is the token itself)
  auto src_of = [&](int32_t t) -> int32_t { return !sp ? t : staged ? s_si[t] : f.src_idx[t]; };
  auto dst_of = [&](int32_t t) -> int32_t { return !dp ? t : staged ? s_di[t] : f.dst_idx[t]; };

  // 2. this CTA's slice of the plane-major work space
  const int64_t T = (int64_t)n * a.planes;
  const int64_t i0 = T * blockIdx.x / gridDim.x, i1 = T * (blockIdx.x + 1) / gridDim.x;
  const int32_t R = a.row_bytes, m = f.chunk_rows;
  for (int64_t i = i0; i < i1;) {
    const int32_t p = (int32_t)(i / n);
    const int32_t ta = (int32_t)(i - (int64_t)p * n);
    int64_t tb = ta + (i1 - i);
    if (tb > n) tb = n;
    if (tb > ta + kFSeg) tb = ta + kFSeg;
    const int32_t cnt = (int32_t)tb - ta;
    i += cnt;

    // 3. runs of this segment
    int32_t sv[kFItems], dv[kFItems];
    bool brk[kFItems];
    int32_t nb = 0;
    const int32_t j0 = tid * kFItems;
    int32_t ps = 0, pd = 0;
    if (j0 > 0 && j0 < cnt) {
      ps = src_of(ta + j0 - 1);
      pd = dst_of(ta + j0 - 1);
    }
#pragma unroll
    for (int k = 0; k < kFItems; ++k) {
      const int32_t j = j0 + k;
      brk[k] = false;
      if (j < cnt) {
        sv[k] = src_of(ta + j);
        dv[k] = dst_of(ta + j);
        brk[k] = j == 0 || (int64_t)sv[k] != (int64_t)ps + 1 || (int64_t)dv[k] != (int64_t)pd + 1 ||
                 (sp && a.src.hnd && sv[k] % a.src.page_size == 0) ||
                 (dp && a.dst.hnd && dv[k] % a.dst.page_size == 0);
        ps = sv[k];
        pd = dv[k];
        nb += brk[k] ? 1 : 0;
      }
    }
    int32_t n_runs;
    int32_t r = block_scan_excl<kFThreads>(nb, &n_runs, s_warp);
#pragma unroll
    for (int k = 0; k < kFItems; ++k) {
      if (brk[k]) {
        s_tok[r] = j0 + k;
        s_rs[r] = sv[k];
        s_rd[r] = dv[k];
        ++r;
      }
    }
    __syncthreads();
    int32_t nch[kFItems], mine = 0;
#pragma unroll
    for (int k = 0; k < kFItems; ++k) {
      const int32_t rr = j0 + k;
      nch[k] = 0;
      if (rr < n_runs) {
        const int32_t len = (rr + 1 < n_runs ? s_tok[rr + 1] : cnt) - s_tok[rr];
        nch[k] = (len + m - 1) / m;
      }
      mine += nch[k];
    }
    int32_t n_chunks;
    int32_t c0 = block_scan_excl<kFThreads>(mine, &n_chunks, s_warp);
#pragma unroll
    for (int k = 0; k < kFItems; ++k) {
      if (j0 + k < n_runs) s_coff[j0 + k] = c0;
      c0 += nch[k];
    }
    __syncthreads();

    // 4. one warp per chunk of plane p
    const char *buf_plane = a.buf + (int64_t)p * n * R;
    if (kLinear) {
      // rows are contiguous on both sides: base pointer and row stride per side are enough
      const char *sbase = sp ? a.src_planes[p] : buf_plane;
      const char *dbase = dp ? a.dst_planes[p] : buf_plane;
      const int64_t sstr = sp ? a.src.slot_stride : R, dstr = dp ? a.dst.slot_stride : R;
      for (int32_t ci = warp; ci < n_chunks; ci += kFThreads / 32) {
        int32_t lo = 0, hi = n_runs;
        while (hi - lo > 1) {
          const int32_t mid = (lo + hi) >> 1;
          if (s_coff[mid] <= ci) lo = mid; else hi = mid;
        }
        const int32_t len = (lo + 1 < n_runs ? s_tok[lo + 1] : cnt) - s_tok[lo];
        const int32_t off = (ci - s_coff[lo]) * m;
        const int32_t rows = len - off < m ? len - off : m;
        copy_linear(sbase + (int64_t)(s_rs[lo] + off) * sstr,
                    const_cast<char *>(dbase) + (int64_t)(s_rd[lo] + off) * dstr,
                    rows * (R >> 4), lane);
      }
    } else {
      for (int32_t ci = warp; ci < n_chunks; ci += kFThreads / 32) {
        int32_t lo = 0, hi = n_runs;
        while (hi - lo > 1) {
          const int32_t mid = (lo + hi) >> 1;
          if (s_coff[mid] <= ci) lo = mid; else hi = mid;
        }
        const int32_t len = (lo + 1 < n_runs ? s_tok[lo + 1] : cnt) - s_tok[lo];
        const int32_t off = (ci - s_coff[lo]) * m;
        const int32_t rows = len - off < m ? len - off : m;
        const Addr sa = side_addr(a.src, sp, a.src_planes[p], (int64_t)s_rs[lo] + off, buf_plane, R);
        const Addr da = side_addr(a.dst, dp, a.dst_planes[p], (int64_t)s_rd[lo] + off, buf_plane, R);
        const int32_t nvec = rows * (R >> 4);
        const bool linear = sa.head == a.seg_bytes && da.head == a.seg_bytes &&
                            (rows == 1 || (sa.row == R && da.row == R));
        if (linear)
          copy_linear(sa.base, const_cast<char *>(da.base), nvec, lane);
        else
          copy_pieces(sa, da, nvec, a.seg_bytes >> 4, a.heads, lane);
      }
    }
    __syncthreads();  // the next segment reuses the run tables
  }
}

}  // namespace

int fused_blocks_per_sm(bool linear) {
  int nb = 0;
  const cudaError_t e =
      linear ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_kernel<true>, kFThreads, 0)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fused_kernel<false>, kFThreads, 0);
  return e == cudaSuccess ? nb : 0;
}

int fused_kernel_list(const void **out, int max) {
  const void *k[] = {reinterpret_cast<const void *>(fused_kernel<true>),
                     reinterpret_cast<const void *>(fused_kernel<false>)};
  return kernel_list_out(k, 2, out, max);
}

cudaError_t launch_fused(const CopyArgs &c, const int32_t *src_idx, const int32_t *dst_idx,
                         int32_t n, int32_t chunk_rows, int sms, int bps, cudaStream_t s) {
  static thread_local FusedArgs f;  // ~4 KiB of plane pointers: keep it off the stack
  f.c = c;
  f.src_idx = src_idx;
  f.dst_idx = dst_idx;
  f.n = n;
  f.chunk_rows = chunk_rows;
  // one warp per chunk of a CTA's slice; at least one item per warp
  const int64_t items = (int64_t)n * c.planes;
  int64_t grid = (int64_t)sms * bps;
  const int64_t cap = (items + kFThreads / 32 - 1) / (kFThreads / 32);
  if (cap < grid) grid = cap;
  if (grid < 1) grid = 1;
  void *args[] = {&f};
  const void *fn = copy_is_linear(c) ? reinterpret_cast<const void *>(fused_kernel<true>)
                                     : reinterpret_cast<const void *>(fused_kernel<false>);
  return cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kFThreads), args, 0, s);
}

}  // namespace kvx

// kvx_plan.cu -- index validation and run-length planning on the device (sm_103a).
//
// "PD分离调研" (Mooncake survey) 7.6: the sender merges contiguous blocks into fewer transfer
// descriptors.  "穷人版 PD 分离", section "5090：一个看得见所有卡的代理": the cost of a KV move
// is set by the number of fragments (72 blocks on a fresh pool, 105,660 once it fragments),
// so fragments are found and merged on the GPU, next to the data, without a host round trip.
//
// Planner CTA (one per tile of kTile tokens), three phases, all in shared memory:
//   1. each thread takes kPlanItems consecutive tokens, fetches their source and destination
//      index, range-checks it and sets brk = "a new run starts here";
//   2. a block-wide exclusive scan of brk numbers the runs; each run start records its token
//      offset and first indices; run r's length is start[r+1] - start[r];
//   3. a second scan of ceil(len / chunk_rows) gives each run's first chunk; every chunk is
//      then written with one binary search over those chunk offsets.
#include "kvx_internal.cuh"
#include "kvx_launch.cuh"

namespace kvx {
namespace {

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Exclusive scan of one value per thread across the block; *total gets the block sum.
// s_warp must hold THREADS / 32 elements.  Ends with a barrier, so s_warp is reusable.
template <int THREADS, typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T *total, T *s_warp) {
  constexpr int kWarps = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = lane < kWarps ? s_warp[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) s_warp[lane] = w;
  }
  __syncthreads();
  T res = (warp > 0 ? s_warp[warp - 1] : T(0)) + x - v;
  *total = s_warp[kWarps - 1];
  __syncthreads();
  return res;
}

template <int THREADS>
__device__ __forceinline__ int32_t block_max(int32_t v, int32_t *s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_max_sync(0xffffffffu, v);
  if (lane == 0) s_warp[warp] = v;
  __syncthreads();
  int32_t r = 0;
  for (int i = 0; i < THREADS / 32; ++i) r = max(r, s_warp[i]);
  __syncthreads();
  return r;
}

// Largest q in [0, n) with pre[q] <= g (pre[0] = 0 <= g).
__device__ __forceinline__ int32_t seg_of(const int64_t *pre, int32_t n, int64_t g) {
  int32_t lo = 0, hi = n;  // invariant: pre[lo] <= g, answer in [lo, hi)
  while (hi - lo > 1) {
    int32_t mid = (lo + hi) >> 1;
    if (pre[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ bool uses_src_pool(int32_t op) {
  return op == KVX_OP_GATHER || op == KVX_OP_TRANSFER;
}
__device__ __forceinline__ bool uses_dst_pool(int32_t op) {
  return op == KVX_OP_SCATTER || op == KVX_OP_TRANSFER;
}

struct Tok {
  int64_t s, d;     // source / destination index
  int32_t req;      // request (batch) or 0
  int32_t err;      // kvx_status of this token's indices
  int32_t op;       // operation of the token's request
  bool start;       // first token of a request
  bool live;        // false: token of a failed request or past the planned range
};

// Indices of token g.  hint: a segment known to start at or before g (batch / runs).
__device__ __forceinline__ Tok fetch(const PlanArgs &a, int64_t g, int32_t &seg) {
  Tok t;
  t.req = 0;
  t.err = 0;
  t.op = a.op;
  t.start = (g == 0);
  t.live = true;
  if (a.mode == kModeSlots) {
    t.s = a.src.is_pool ? (int64_t)a.src_idx[g] : g;
    t.d = a.dst.is_pool ? (int64_t)a.dst_idx[g] : g;
  } else {
    const int64_t *pre = reinterpret_cast<const int64_t *>(a.ws + a.L.prefix_off);
    if (g >= pre[a.n_segs]) {  // fewer tokens than promised: already a fatal status
      t.s = t.d = 0;
      t.live = false;
      return t;
    }
    while (seg + 1 < a.n_segs && pre[seg + 1] <= g) ++seg;
    const int64_t off = g - pre[seg];
    if (a.mode == kModeRuns) {
      t.s = a.src.is_pool ? (int64_t)a.runs[3 * (int64_t)seg] + off : g;
      t.d = a.dst.is_pool ? (int64_t)a.runs[3 * (int64_t)seg + 1] + off : g;
    } else {
      t.req = seg;
      t.start = (off == 0);
      if (a.status[1 + seg] != KVX_OK) {  // bad record: never read its indices
        t.s = t.d = off;
        t.live = false;
        return t;
      }
      const kvx_request r = a.reqs[seg];
      t.op = r.op;
      t.s = uses_src_pool(r.op) ? (int64_t)a.src_idx[r.src_off + off] : off;
      t.d = uses_dst_pool(r.op) ? (int64_t)a.dst_idx[r.dst_off + off] : off;
    }
  }
  const bool sp = (a.mode == kModeBatch) ? uses_src_pool(t.op) : (bool)a.src.is_pool;
  const bool dp = (a.mode == kModeBatch) ? uses_dst_pool(t.op) : (bool)a.dst.is_pool;
  if ((sp && (t.s < 0 || t.s >= a.src.num_slots)) || (dp && (t.d < 0 || t.d >= a.dst.num_slots)))
    t.err = KVX_ERR_OUT_OF_RANGE;
  return t;
}

__device__ __forceinline__ bool starts_run(const PlanArgs &a, const Tok &t, const Tok &prev,
                                           bool first_in_tile) {
  if (first_in_tile || t.start || t.req != prev.req) return true;
  // 64-bit steps: an index list may hold INT32_MAX (refused later, but never overflowed here)
  if ((int64_t)t.s != (int64_t)prev.s + 1 || (int64_t)t.d != (int64_t)prev.d + 1) return true;
  const bool sp = (a.mode == kModeBatch) ? uses_src_pool(t.op) : (bool)a.src.is_pool;
  const bool dp = (a.mode == kModeBatch) ? uses_dst_pool(t.op) : (bool)a.dst.is_pool;
  if (sp && a.src.hnd && t.s % a.src.page_size == 0) return true;
  if (dp && a.dst.hnd && t.d % a.dst.page_size == 0) return true;
  return false;
}

__device__ __forceinline__ void write_header(const PlanArgs &a) {
  PlanHeader *h = reinterpret_cast<PlanHeader *>(a.ws + a.L.header_off);
  h->mode = a.mode;
  h->op = a.op;
  h->n_segs = a.n_segs;
  h->n_tokens = a.n_tokens;
  h->chunk_rows = a.chunk_rows;
  h->planes = a.planes;
  h->row_bytes = a.row_bytes;
  h->src_is_pool = a.src.is_pool;
  h->src_hnd = a.src.hnd;
  h->src_page_size = a.src.page_size;
  h->dst_is_pool = a.dst.is_pool;
  h->dst_hnd = a.dst.hnd;
  h->dst_page_size = a.dst.page_size;
  h->pad = 0;
  h->src_num_slots = a.src.num_slots;
  h->dst_num_slots = a.dst.num_slots;
  h->magic = kPlanMagic;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanArgs a) {
  __shared__ int32_t s_tok[kTile];   // token offset (in tile) of run r
  __shared__ int32_t s_src[kTile];   // first source index of run r
  __shared__ int32_t s_dst[kTile];   // first destination index of run r
  __shared__ int32_t s_req[kTile];   // request of run r
  __shared__ int32_t s_coff[kTile + 1];
  __shared__ int32_t s_warp[kPlanThreads / 32];

  // the kernel before (the prefix kernel, or whatever the caller ran last) must be complete
  // before the kernels behind may start: they read slot lists and rows before they wait
  pdl_wait();
  pdl_trigger();

  const int tile = blockIdx.x;
  const int64_t t0 = (int64_t)tile * kTile;
  const int64_t rem = a.n_tokens - t0;
  const int32_t cnt = (int32_t)(rem < kTile ? rem : kTile);
  const int tid = threadIdx.x;

  // phase 1: indices, checks and run starts of this thread's tokens
  Tok tk[kPlanItems];
  bool brk[kPlanItems];
  int32_t nbrk = 0, err = 0;
  const int32_t i0 = tid * kPlanItems;
  int32_t seg = 0;
  if ((a.mode != kModeSlots) && i0 < cnt) {
    const int64_t *pre = reinterpret_cast<const int64_t *>(a.ws + a.L.prefix_off);
    const int64_t g = t0 + i0 - (i0 > 0 ? 1 : 0);
    seg = (g < pre[a.n_segs]) ? seg_of(pre, a.n_segs, g) : 0;
  }
  Tok prev;
  if (a.mode == kModeSlots) {
    // Slot lists: issue every index load of this thread (and its predecessor token) before
    // using any of them, so they cost one memory round trip instead of one per token.
    int32_t sraw[kPlanItems + 1], draw[kPlanItems + 1];
#pragma unroll
    for (int k = 0; k <= kPlanItems; ++k) {
      const int32_t i = i0 + k - 1;
      const bool in = i >= 0 && i < cnt;
      sraw[k] = (in && a.src.is_pool) ? __ldg(a.src_idx + t0 + i) : (int32_t)(t0 + i);
      draw[k] = (in && a.dst.is_pool) ? __ldg(a.dst_idx + t0 + i) : (int32_t)(t0 + i);
    }
    prev.s = sraw[0];
    prev.d = draw[0];
    prev.req = 0;
    prev.op = a.op;
#pragma unroll
    for (int k = 0; k < kPlanItems; ++k) {
      const int32_t i = i0 + k;
      brk[k] = false;
      if (i < cnt) {
        Tok &t = tk[k];
        t.s = sraw[k + 1];
        t.d = draw[k + 1];
        t.req = 0;
        t.op = a.op;
        t.start = (t0 + i == 0);
        t.live = true;
        t.err = ((a.src.is_pool && (t.s < 0 || t.s >= a.src.num_slots)) ||
                 (a.dst.is_pool && (t.d < 0 || t.d >= a.dst.num_slots)))
                    ? KVX_ERR_OUT_OF_RANGE
                    : KVX_OK;

        err = max(err, t.err);
        brk[k] = starts_run(a, t, prev, i == 0);
        prev = t;
        nbrk += brk[k] ? 1 : 0;
      }
    }
  } else {
    if (i0 > 0 && i0 < cnt) prev = fetch(a, t0 + i0 - 1, seg);
#pragma unroll
    for (int k = 0; k < kPlanItems; ++k) {
      const int32_t i = i0 + k;
      brk[k] = false;
      if (i < cnt) {
        tk[k] = fetch(a, t0 + i, seg);
        err = max(err, tk[k].err);
        brk[k] = starts_run(a, tk[k], prev, i == 0);
        prev = tk[k];
        nbrk += brk[k] ? 1 : 0;
        if (tk[k].err != KVX_OK && a.mode == kModeBatch)
          atomicMax(&a.status[1 + tk[k].req], tk[k].err);
      }
    }
  }
  err = block_max<kPlanThreads>(err, s_warp);
  if (tid == 0) {
    if (a.status_direct) {
      a.status[0] = err;
      for (int k = 1; k < a.status_direct; ++k) a.status[k] = 0;
    } else if (err != KVX_OK) {
      atomicMax(&a.status[0], err);
    }
  }
  if (a.validate_only) return;
  Chunk *out = reinterpret_cast<Chunk *>(a.ws + a.L.chunks_off) + (int64_t)tile * kTile;

  if (a.chunk_rows == 1) {
    // Every chunk is one row, so the plan is one chunk per token in token order whatever the
    // runs are: no scans needed.
#pragma unroll
    for (int k = 0; k < kPlanItems; ++k) {
      if (i0 + k < cnt) {
        Chunk ch;
        ch.req = tk[k].req;
        ch.src = (int32_t)tk[k].s;
        ch.dst = (int32_t)tk[k].d;
        ch.rows = 1;
        out[i0 + k] = ch;
      }
    }
    if (tid == 0) {
      reinterpret_cast<int32_t *>(a.ws + a.L.tiles_off)[tile] = cnt;
      if (tile == 0) write_header(a);
    }
    return;
  }

  int32_t n_runs;
  int32_t r = block_exclusive_scan<kPlanThreads>(nbrk, &n_runs, s_warp);
#pragma unroll
  for (int k = 0; k < kPlanItems; ++k) {
    if (brk[k]) {
      s_tok[r] = i0 + k;
      s_src[r] = (int32_t)tk[k].s;
      s_dst[r] = (int32_t)tk[k].d;
      s_req[r] = tk[k].req;
      ++r;
    }
  }
  __syncthreads();

  // phase 2: chunks per run, scanned into each run's first chunk
  const int32_t m = a.chunk_rows;
  int32_t nch[kPlanItems];
  int32_t my_chunks = 0;
#pragma unroll
  for (int k = 0; k < kPlanItems; ++k) {
    const int32_t rr = i0 + k;
    nch[k] = 0;
    if (rr < n_runs) {
      const int32_t len = (rr + 1 < n_runs ? s_tok[rr + 1] : cnt) - s_tok[rr];
      nch[k] = (len + m - 1) / m;
    }
    my_chunks += nch[k];
  }
  int32_t n_chunks;
  int32_t c = block_exclusive_scan<kPlanThreads>(my_chunks, &n_chunks, s_warp);
#pragma unroll
  for (int k = 0; k < kPlanItems; ++k) {
    if (i0 + k < n_runs) s_coff[i0 + k] = c;
    c += nch[k];
  }
  if (tid == 0) s_coff[n_runs] = n_chunks;
  __syncthreads();

  if (tid == 0) {
    reinterpret_cast<int32_t *>(a.ws + a.L.tiles_off)[tile] = n_chunks;
    if (tile == 0) write_header(a);
  }

  // phase 3: write the chunks
  for (int32_t ci = tid; ci < n_chunks; ci += kPlanThreads) {
    int32_t lo = 0, hi = n_runs;  // largest run with s_coff[run] <= ci
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (s_coff[mid] <= ci) lo = mid; else hi = mid;
    }
    const int32_t len = (lo + 1 < n_runs ? s_tok[lo + 1] : cnt) - s_tok[lo];
    const int32_t j0 = (ci - s_coff[lo]) * m;
    Chunk ch;
    ch.req = s_req[lo];
    ch.src = s_src[lo] + j0;
    ch.dst = s_dst[lo] + j0;
    ch.rows = min(m, len - j0);
    out[ci] = ch;
  }
}

// Checks one batch record; returns its status.
__device__ __forceinline__ int32_t check_request(const PlanArgs &a, const kvx_request &r) {
  if (r.op < KVX_OP_GATHER || r.op > KVX_OP_TRANSFER) return KVX_ERR_INVALID_ARG;
  if (r.n_tokens < 0 || r.n_tokens > KVX_MAX_TOKENS) return KVX_ERR_INVALID_ARG;
  const bool us = uses_src_pool(r.op), ud = uses_dst_pool(r.op);
  if (us && (!a.has_src || r.src_off < 0 || r.src_off + r.n_tokens > a.n_src_idx))
    return KVX_ERR_INVALID_ARG;
  if (ud && (!a.has_dst || r.dst_off < 0 || r.dst_off + r.n_tokens > a.n_dst_idx))
    return KVX_ERR_INVALID_ARG;
  if (r.op != KVX_OP_TRANSFER) {
    const int64_t need = (int64_t)a.planes * r.n_tokens * a.row_bytes;
    if (r.buf_off < 0 || (r.buf_off & 15) != 0 || r.buf_off + need > a.buf_bytes)
      return KVX_ERR_INVALID_ARG;
  }
  return KVX_OK;
}

// One CTA: token offset of every run / request, their checks, and status words.
__global__ void __launch_bounds__(kPrefixThreads) prefix_kernel(const __grid_constant__ PlanArgs a) {
  __shared__ int64_t s_warp64[kPrefixThreads / 32];
  __shared__ int32_t s_warp32[kPrefixThreads / 32];
  pdl_wait();  // the caller's last kernel is complete before the planner behind may start
  pdl_trigger();
  int64_t *pre = reinterpret_cast<int64_t *>(a.ws + a.L.prefix_off);
  const int tid = threadIdx.x;
  int64_t carry = 0;
  int32_t err = 0;
  for (int64_t base = 0; base < a.n_segs; base += (int64_t)kPrefixThreads * kPrefixItems) {
    int64_t len[kPrefixItems];
    int64_t sum = 0;
#pragma unroll
    for (int k = 0; k < kPrefixItems; ++k) {
      const int64_t q = base + (int64_t)tid * kPrefixItems + k;
      len[k] = 0;
      if (q < a.n_segs) {
        int32_t e = KVX_OK;
        if (a.mode == kModeRuns) {
          len[k] = a.runs[3 * q + 2];
          if (len[k] < 0) { e = KVX_ERR_INVALID_ARG; len[k] = 0; }
        } else {
          const kvx_request r = a.reqs[q];
          e = check_request(a, r);
          len[k] = r.n_tokens > 0 && r.n_tokens <= KVX_MAX_TOKENS ? r.n_tokens : 0;
          a.status[1 + q] = e;
        }
        err = max(err, e);
      }
      sum += len[k];
    }
    int64_t total;
    int64_t run = carry + block_exclusive_scan<kPrefixThreads>(sum, &total, s_warp64);
#pragma unroll
    for (int k = 0; k < kPrefixItems; ++k) {
      const int64_t q = base + (int64_t)tid * kPrefixItems + k;
      if (q < a.n_segs) pre[q] = run;
      run += len[k];
    }
    carry += total;
  }
  if (tid == 0) pre[a.n_segs] = carry;
  const int32_t fatal = (carry != a.n_tokens) ? KVX_ERR_INVALID_ARG : KVX_OK;
  err = block_max<kPrefixThreads>(err, s_warp32);
  if (fatal != KVX_OK && a.mode == kModeBatch) {
    for (int64_t q = tid; q < a.n_segs; q += kPrefixThreads) a.status[1 + q] = fatal;
  }
  if (tid == 0) a.status[0] = max(err, fatal);
}

// Flattens the per-tile chunk tables (one CTA).
__global__ void __launch_bounds__(1024) export_kernel(const char *ws, WsLayout L, int64_t n_tokens,
                                                      int32_t *out, int64_t max_chunks,
                                                      int64_t *count) {
  __shared__ int64_t s_warp[32];
  const int32_t *tiles = reinterpret_cast<const int32_t *>(ws + L.tiles_off);
  const Chunk *chunks = reinterpret_cast<const Chunk *>(ws + L.chunks_off);
  const int64_t nt = num_tiles(n_tokens);
  int64_t carry = 0;
  for (int64_t base = 0; base < nt; base += 1024) {
    const int64_t t = base + threadIdx.x;
    int64_t mine = t < nt ? tiles[t] : 0;
    mine = mine < 0 ? 0 : (mine > kTile ? kTile : mine);  // never read past a tile's table
    int64_t total;
    const int64_t at = carry + block_exclusive_scan<1024>(mine, &total, s_warp);
    carry += total;
    if (t < nt) {
      for (int64_t k = 0; k < mine; ++k) {
        if (at + k < max_chunks) {
          const Chunk c = chunks[t * kTile + k];
          int32_t *o = out + 4 * (at + k);
          o[0] = c.req;
          o[1] = c.src;
          o[2] = c.dst;
          o[3] = c.rows;
        }
      }
    }
  }
  if (threadIdx.x == 0) *count = carry;
}

}  // namespace

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, cudaStream_t s,
                       size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
    // programmatic dependent launch refused on this stream: launch in plain stream order
    (void)cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  return e;
}

namespace {

// Duplicate-destination check (KVX_CHECK_DUP), behind the planner: one thread per token
// inserts the token's destination slot into an open-addressing table in the workspace
// (entry = (slot + 1) << 32 | request, home bucket from a multiplicative hash, linear probing
// bounded by the table size; entries only ever go from empty to a slot, and the table holds at
// most n < size of them).  Spread over many CTAs because one SM keeps only a limited number of
// atomics in flight.  Slot lists: the inserts go out before griddepcontrol.wait and the verdict
// is raised once the planner, which writes the status word, has finished.  Runs and batches:
// a token's run or request comes from the prefix kernel's offsets, and a batch request whose
// record or indices the planner refused writes nothing, so its slots are not inserted; both
// wait for the planner first.  A repeated slot in a batch fails every request naming it (the
// one found in the table and the inserting one), each in its own status word.
constexpr int kDupThreads = 128;

__global__ void __launch_bounds__(kDupThreads) dup_kernel(const __grid_constant__ PlanArgs a) {
  pdl_trigger();
  if (a.mode != kModeSlots) pdl_wait();
  const int64_t g = (int64_t)blockIdx.x * kDupThreads + threadIdx.x;
  int64_t slot = -1;
  uint32_t req = 0;
  if (g < a.n_tokens) {
    if (a.mode == kModeSlots) {
      slot = __ldg(a.dst_idx + g);
    } else {
      const int64_t *pre = reinterpret_cast<const int64_t *>(a.ws + a.L.prefix_off);
      if (g < pre[a.n_segs]) {
        const int32_t seg = seg_of(pre, a.n_segs, g);
        const int64_t off = g - pre[seg];
        if (a.mode == kModeRuns) {
          slot = (int64_t)a.runs[3 * (int64_t)seg + 1] + off;
        } else if (const int32_t st = a.status[1 + seg];
                   st == KVX_OK || st == KVX_ERR_DUPLICATE_DST) {
          // accepted by the planner (a duplicate raised by this kernel meanwhile does not
          // take a request's slots out of the check: the other requests naming them still fail)
          const kvx_request r = a.reqs[seg];
          if (uses_dst_pool(r.op)) {
            slot = a.dst_idx[r.dst_off + off];
            req = (uint32_t)seg;
          }
        }
      }
    }
  }
  bool dup = false;
  uint32_t other = 0;
  if (slot >= 0 && slot < a.dst.num_slots) {  // the planner reports the others
    const unsigned long long key = (unsigned long long)(slot + 1) << 32;
    uint32_t h = ((uint32_t)slot * 2654435761u) >> (32 - a.dup_bits);
    for (uint32_t probe = 0; probe <= a.dup_mask; ++probe, h = (h + 1) & a.dup_mask) {
      const unsigned long long cur = atomicCAS(a.dup_table + h, 0ull, key | req);
      if (cur == 0) break;  // claimed
      if ((cur & 0xFFFFFFFF00000000ull) == key) {
        dup = true;
        other = (uint32_t)cur;
        break;
      }
    }
  }
  if (a.mode == kModeBatch) {
    if (dup) {
      atomicMax(&a.status[1 + req], (int32_t)KVX_ERR_DUPLICATE_DST);
      atomicMax(&a.status[1 + other], (int32_t)KVX_ERR_DUPLICATE_DST);
      atomicMax(&a.status[0], (int32_t)KVX_ERR_DUPLICATE_DST);
    }
    return;
  }
  dup = __syncthreads_or(dup);
  pdl_wait();  // the planner's status words are written
  if (dup && threadIdx.x == 0) atomicMax(&a.status[0], (int32_t)KVX_ERR_DUPLICATE_DST);
}

}  // namespace

// Validate-only check of one request's slot lists by a single CTA (validates_direct): every
// index of both lists range-checked, the loads of both lists in flight together (16-byte loads
// over each list's aligned body, four per list and thread per round, plus scalar loads of the
// up to three elements before and after it) before any is tested, and the verdict stored
// straight into the status words.  Ordered like the planner: it waits for the kernel before it
// and only then lets the copy behind it start.
constexpr int kValidateThreads = 1024;
constexpr int kValidateIn = 4;

__device__ __forceinline__ int32_t out_of_range(int32_t v, int64_t num) {
  return (v < 0 || (int64_t)v >= num) ? 1 : 0;
}

__device__ __forceinline__ int32_t out_of_range4(int4 v, int64_t num) {
  return out_of_range(v.x, num) | out_of_range(v.y, num) | out_of_range(v.z, num) |
         out_of_range(v.w, num);
}

// One list: elements [0, head) and [tail0, n) are read one by one, [head, tail0) as int4s.
struct ListSpan {
  const int32_t *idx;  // nullptr: the side is a buffer (nothing to check)
  int64_t num, head, body, tail0;
};

__device__ __forceinline__ ListSpan list_span(const int32_t *idx, int64_t n, int64_t num) {
  ListSpan l{idx, num, 0, 0, 0};
  if (idx == nullptr) {  // no list: its placeholder zeros must pass every check
    l.num = INT64_MAX;
    return l;
  }
  const int64_t mis = (int64_t)(((uintptr_t)idx & 15) >> 2);
  l.head = mis ? (4 - mis < n ? 4 - mis : n) : 0;
  l.body = (n - l.head) >> 2;
  l.tail0 = l.head + 4 * l.body;
  return l;
}

__global__ void __launch_bounds__(kValidateThreads) validate_kernel(const __grid_constant__ PlanArgs a) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = a.n_tokens;
  const int tid = threadIdx.x;
  const ListSpan ls = list_span(a.src.is_pool ? a.src_idx : nullptr, n, a.src.num_slots);
  const ListSpan ld = list_span(a.dst.is_pool ? a.dst_idx : nullptr, n, a.dst.num_slots);
  // the scalar ends of both lists (threads 0..3: head, 4..7: tail)
  int32_t end_s = 0, end_d = 0;
  bool has_s = false, has_d = false;
  if (tid < 8) {
    const int64_t i_s = tid < 4 ? tid : ls.tail0 + (tid - 4);
    const int64_t i_d = tid < 4 ? tid : ld.tail0 + (tid - 4);
    has_s = ls.idx && (tid < 4 ? i_s < ls.head : i_s < n);
    has_d = ld.idx && (tid < 4 ? i_d < ld.head : i_d < n);
    if (has_s) end_s = __ldg(ls.idx + i_s);
    if (has_d) end_d = __ldg(ld.idx + i_d);
  }
  const int4 *vs = reinterpret_cast<const int4 *>(ls.idx + ls.head);
  const int4 *vd = reinterpret_cast<const int4 *>(ld.idx + ld.head);
  const int64_t body = ls.body > ld.body ? ls.body : ld.body;
  int32_t bad = 0;
  for (int64_t base = 0; base < body; base += (int64_t)kValidateIn * kValidateThreads) {
    int4 xs[kValidateIn], xd[kValidateIn];
#pragma unroll
    for (int k = 0; k < kValidateIn; ++k) {
      const int64_t i = base + (int64_t)k * kValidateThreads + tid;
      xs[k] = i < ls.body ? __ldg(vs + i) : make_int4(0, 0, 0, 0);
      xd[k] = i < ld.body ? __ldg(vd + i) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kValidateIn; ++k)
      bad |= out_of_range4(xs[k], ls.num) | out_of_range4(xd[k], ld.num);
  }
  if (has_s) bad |= out_of_range(end_s, ls.num);
  if (has_d) bad |= out_of_range(end_d, ld.num);
  bad = __syncthreads_or(bad);
  if (tid == 0) {
    a.status[0] = bad ? (int32_t)KVX_ERR_OUT_OF_RANGE : (int32_t)KVX_OK;
    for (int k = 1; k < a.status_direct; ++k) a.status[k] = 0;
  }
}

cudaError_t launch_prefix(const PlanArgs &a, cudaStream_t s) {
  void *args[] = {const_cast<PlanArgs *>(&a)};
  return launch_pdl(reinterpret_cast<const void *>(prefix_kernel), dim3(1), dim3(kPrefixThreads),
                    args, s);
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s) {
  void *args[] = {const_cast<PlanArgs *>(&a)};
  // one tile: the planner's own validate-only pass (measured 0.3 us faster than the one-CTA
  // kernel at 2048 tokens); more tiles up to kValidateMaxTokens: the one-CTA kernel, which
  // spares the status memset a multi-tile planner needs
  const bool one_cta = a.validate_only && a.mode == kModeSlots && a.status_direct &&
                       num_tiles(a.n_tokens) > 1 && a.n_tokens <= kValidateMaxTokens;
  cudaError_t e =
      one_cta ? launch_pdl(reinterpret_cast<const void *>(validate_kernel), dim3(1),
                           dim3(kValidateThreads), args, s)
              : launch_pdl(reinterpret_cast<const void *>(plan_kernel),
                           dim3((unsigned)num_tiles(a.n_tokens)), dim3(kPlanThreads), args, s);
  if (e != cudaSuccess || !a.dup_table) return e;
  const int64_t grid = (a.n_tokens + kDupThreads - 1) / kDupThreads;
  return launch_pdl(reinterpret_cast<const void *>(dup_kernel), dim3((unsigned)grid),
                    dim3(kDupThreads), args, s);
}

int plan_kernel_list(const void **out, int max) {
  const void *k[] = {reinterpret_cast<const void *>(plan_kernel),
                     reinterpret_cast<const void *>(validate_kernel),
                     reinterpret_cast<const void *>(dup_kernel),
                     reinterpret_cast<const void *>(prefix_kernel)};
  return kernel_list_out(k, 4, out, max);
}

cudaError_t launch_export(const char *ws, WsLayout L, int64_t n_tokens, int32_t *out,
                          int64_t max_chunks, int64_t *count, cudaStream_t s) {
  export_kernel<<<1, 1024, 0, s>>>(ws, L, n_tokens, out, max_chunks, count);
  return cudaGetLastError();
}

}  // namespace kvx

// kvx_stream.cu -- layer-streamed, cancellable gather / scatter / transfer (sm_103a).
//
// "DistServe 完全拆解", 一次请求如何穿过 DistServe: prefill writes the prompt's KV layer by
// layer, and decode pulls layer j from prefill's layer j asynchronously, so most of the move
// can run while later layers are still being computed.  "穷人版 PD 分离", 最难的一个问题: a
// transfer the receiver has given up on must not land late in pages that were handed to
// another request, and the sender may only acknowledge the abort once it can prove that no
// write is still in flight.
//
// One persistent grid walks the request's rows in layer-major order: item i is
// (layer l, K/V, group of g tokens) with l = i / (2 * groups); warp w takes items w, w + W,
// w + 2W, ... (W warps in the grid), so every warp reaches the layers in increasing order and
// all warps stay busy however few tokens a layer has.  A warp entering layer l checks, once
// per CTA and layer (the first warp to arrive polls, the others read the CTA's shared bit of
// layer l):
//   - the request's epoch word: changed -> the CTA stops before layer l (KVX_ERR_CANCELLED);
//   - the producer's ready word of layer l: below ready_value -> poll with back-off, bounded
//     by wait_ns of %globaltimer and an iteration cap -> the CTA stops before layer l
//     (KVX_ERR_TIMEOUT).
// A CTA that stops still finishes the layers its warps had already entered, so every layer
// below the smallest stop layer of all CTAs holds every row.  On exit each CTA publishes its
// stop layer and code, and the last CTA to finish sets the "no further write" word with a
// system-scope release after all CTAs' writes.
//
// Waits only ever poll memory that the host or another engine writes; the kernel never waits
// for another CTA or another kernel.
#include "kvx_copy_ops.cuh"

namespace kvx {
namespace {

using namespace ops;

constexpr int kWarps = kCopyThreads / 32;
constexpr uint32_t kMaxPolls = 1u << 24;  // backstop behind the %globaltimer bound
constexpr uint32_t kMaxSleepNs = 1024;

struct StreamArgs {
  CopyArgs c;   // sides, planes, buffer, status, slot lists (spec_src / spec_dst)
  StreamCtl k;
};

__device__ __forceinline__ int32_t ld_acquire_sys(const int32_t *p) {
  int32_t v;
  asm volatile("ld.acquire.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_sys(int32_t *p, int32_t v) {
  asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t ld_acquire_cta(const int32_t *smem) {
  int32_t v;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void or_release_cta(uint32_t *smem, uint32_t v) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("red.release.cta.shared::cta.or.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

constexpr int kReadyWords = KVX_MAX_PLANES / 2 / 32;
static_assert(kReadyWords * 32 * 2 == KVX_MAX_PLANES, "one ready bit per layer");

struct CtaState {
  uint32_t ready[kReadyWords];    // bit l: layer l is known ready in this CTA
  uint32_t polling[kReadyWords];  // bit l: one warp of this CTA polls for layer l
  int32_t stop;                   // first layer this CTA does not start (num_layers: none)
  int32_t code;                   // KVX_ERR_TIMEOUT / KVX_ERR_CANCELLED, or 0
};

__device__ __forceinline__ bool known_ready(CtaState *cs, int32_t l) {
  return (ld_acquire_cta(reinterpret_cast<const int32_t *>(&cs->ready[l >> 5])) >> (l & 31)) & 1;
}

__device__ __forceinline__ int32_t stopped_before(CtaState *cs, int32_t l) {
  return *reinterpret_cast<volatile int32_t *>(&cs->stop) <= l;
}

__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int32_t give_up(CtaState *cs, int32_t l, int32_t code) {
  atomicMin(&cs->stop, l);
  atomicMax(&cs->code, code);
  return 0;
}

// Lane 0 of a warp entering layer l: 1 to go on, 0 to stop.  Polling is shared out so that
// the words of a slow producer (often pinned host memory, read over the CPU-GPU link) see
// few readers: in each CTA one warp polls and the others watch the CTA's shared bit; the
// polling warp reads the device-memory mirror on every round and the producer's words only
// on its first round and every 16th, except in the CTA that owns the layer's first item,
// which reads them on every round and copies what it sees into the mirror.
__device__ int32_t wait_layer(const StreamCtl &k, int32_t l, bool owner, CtaState *cs) {
  if (stopped_before(cs, l)) return 0;
  if (known_ready(cs, l)) return 1;
  const uint32_t bit = 1u << (l & 31);
  if (!k.layer_ready && !k.epoch_word) {  // nothing to wait for
    or_release_cta(&cs->ready[l >> 5], bit);
    return 1;
  }
  const bool poller = !(atomicOr(&cs->polling[l >> 5], bit) & bit);
  const uint64_t t0 = globaltimer_ns();
  uint32_t sleep_ns = 32;
  for (uint32_t it = 0;; ++it) {
    if (poller) {
      if (ld_acquire_gpu(k.mirror) == k.gen) return give_up(cs, l, KVX_ERR_CANCELLED);
      if (ld_acquire_gpu(k.mirror + 1 + l) == k.gen) {
        or_release_cta(&cs->ready[l >> 5], bit);
        return 1;
      }
      if (owner || it == 0 || (it & 15) == 15) {
        if (k.epoch_word && ld_acquire_sys(k.epoch_word) != k.epoch) {
          st_release_gpu(k.mirror, k.gen);
          return give_up(cs, l, KVX_ERR_CANCELLED);
        }
        if (!k.layer_ready || ld_acquire_sys(k.layer_ready + l) >= k.ready_value) {
          st_release_gpu(k.mirror + 1 + l, k.gen);
          or_release_cta(&cs->ready[l >> 5], bit);
          return 1;
        }
      }
    }
    if (globaltimer_ns() - t0 >= (uint64_t)k.wait_ns || it >= kMaxPolls)
      return give_up(cs, l, KVX_ERR_TIMEOUT);
    __nanosleep(sleep_ns);
    if (sleep_ns < kMaxSleepNs) sleep_ns <<= 1;
    if (stopped_before(cs, l)) return 0;
    if (known_ready(cs, l)) return 1;
  }
}

template <bool kSrcHnd, bool kDstHnd>
__global__ void __launch_bounds__(kCopyThreads, 6) stream_kernel(const __grid_constant__ StreamArgs s) {
  __shared__ CtaState cs;
  const CopyArgs &a = s.c;
  const StreamCtl &k = s.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t layers = k.layers;
  if (threadIdx.x < kReadyWords) {
    cs.ready[threadIdx.x] = 0;
    cs.polling[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) {
    cs.stop = layers;
    cs.code = 0;
  }
  __syncthreads();

  const int32_t gsh = a.row_group_shift, lsh = 5 - gsh;
  const int32_t li = lane & ((1 << lsh) - 1);
  const int32_t R = a.row_bytes, vpr = R >> 4;
  const bool sp = a.src.is_pool != 0, dp = a.dst.is_pool != 0;
  const uint32_t W = gridDim.x * kWarps;
  int32_t lcur = -1;
  bool verdict_ok = false;  // this warp has seen the planner's verdict (every index valid)
  for (uint32_t i = blockIdx.x * kWarps + warp; i < k.items; i += W) {
    const int32_t l = (int32_t)(i / k.per_layer);
    if (l != lcur) {
      const bool owner = blockIdx.x == ((uint64_t)l * k.per_layer % W) / kWarps;
      int32_t go = lane == 0 ? wait_layer(k, l, owner, &cs) : 0;
      go = __shfl_sync(0xffffffffu, go, 0);
      __syncwarp();  // lane 0's acquire orders every lane's loads of the layer
      if (!go) break;
      lcur = l;
    }
    const uint32_t r = i - (uint32_t)l * k.per_layer;
    const int32_t kv = r >= k.groups ? 1 : 0;
    const int64_t t = ((int64_t)(r - kv * k.groups) << gsh) + (lane >> lsh);
    const int32_t p = 2 * l + kv;
    // The first item's loads go out before the planner's verdict, like the row kernel's; a
    // lane range-checks its own indices first so that it never reads outside a pool.
    bool ok = t < a.n_tokens;
    const int64_t tt = ok ? t : 0;
    const int32_t si = sp ? a.spec_src[tt] : (int32_t)tt;
    const int32_t di = dp ? a.spec_dst[tt] : (int32_t)tt;
    ok = ok && (!sp || (si >= 0 && (int64_t)si < a.src.num_slots)) &&
         (!dp || (di >= 0 && (int64_t)di < a.dst.num_slots));
    const char *buf_plane = a.buf + (int64_t)p * a.n_tokens * R;
    const char *srow = row_base<kSrcHnd>(a.src, sp, a.src_planes[p], buf_plane, si, R);
    char *drow = const_cast<char *>(row_base<kDstHnd>(a.dst, dp, a.dst_planes[p], buf_plane, di, R));
#pragma unroll 1
    for (int32_t x0 = 0; x0 < vpr; x0 += kUnroll << lsh) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t xv = x0 + li + (u << lsh);
        if (ok && xv < vpr) v[u] = ld_stream(row_byte<kSrcHnd>(a.src, sp, srow, xv << 4));
      }
      if (!verdict_ok) {
        pdl_wait();  // the planner has checked every index and written status[0]
        if (*reinterpret_cast<volatile const int32_t *>(a.status) != KVX_OK) {
          if (lane == 0) atomicMin(&cs.stop, 0);
          break;
        }
        verdict_ok = true;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t xv = x0 + li + (u << lsh);
        if (ok && xv < vpr) st_stream(const_cast<char *>(row_byte<kDstHnd>(a.dst, dp, drow, xv << 4)), v[u]);
      }
    }
    if (!verdict_ok) break;
  }

  // every thread's writes before this CTA's report; the last CTA's release covers all CTAs
  pdl_wait();  // the planner's status words are written before any CTA reports
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (cs.code) atomicMax(&a.status[0], cs.code);
    if (cs.stop < layers) atomicMax(&a.status[1], layers - cs.stop);
    __threadfence_system();
    if (atomicAdd(&a.status[2], 1) == (int32_t)gridDim.x - 1) {
      __threadfence_system();
      st_release_sys(&a.status[3], 1);
      if (k.host_done) st_release_sys(k.host_done, 1);
    }
  }
}

const void *stream_fn(bool sh, bool dh) {
  if (sh && dh) return reinterpret_cast<const void *>(stream_kernel<true, true>);
  if (sh) return reinterpret_cast<const void *>(stream_kernel<true, false>);
  if (dh) return reinterpret_cast<const void *>(stream_kernel<false, true>);
  return reinterpret_cast<const void *>(stream_kernel<false, false>);
}

}  // namespace

int stream_blocks_per_sm() {
  int nb = 0;
  const cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, stream_kernel<false, false>, kCopyThreads, 0);
  return e == cudaSuccess ? nb : 0;
}

void stream_sizes(StreamCtl &k, int64_t n_tokens, int32_t group_shift) {
  const int64_t groups = (n_tokens + (1 << group_shift) - 1) >> group_shift;
  k.groups = (uint32_t)groups;
  k.per_layer = (uint32_t)(2 * groups);
  k.items = (uint32_t)(2 * groups * k.layers);
}

cudaError_t launch_stream(const CopyArgs &c, const StreamCtl &k, int grid, cudaStream_t s) {
  static thread_local StreamArgs args;  // ~4 KiB of plane pointers: keep it off the stack
  args.c = c;
  args.k = k;
  const bool sh = c.src.hnd && c.src.is_pool, dh = c.dst.hnd && c.dst.is_pool;
  const void *fn = stream_fn(sh, dh);
  void *params[] = {&args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, params);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
    (void)cudaGetLastError();  // no programmatic dependent launch here: plain stream order
    cfg.numAttrs = 0;
    e = cudaLaunchKernelExC(&cfg, fn, params);
  }
  return e;
}

}  // namespace kvx

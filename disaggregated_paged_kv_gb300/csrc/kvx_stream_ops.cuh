// kvx_stream_ops.cuh -- the per-layer waits of the layer-streamed grids (sm_103a): memory
// ordering helpers, the owner-epoch check of a destination page, the tagged stop word, the
// bounded wait of a row-grid CTA's thread 0 for its layer, and the per-CTA layer state, wait
// and exit protocol of the persistent grids.  Shared by kvx_stream.cu and kvx_reshard.cu.
#pragma once

#include "kvx_copy_ops.cuh"

namespace kvx {
namespace sops {

using ops::globaltimer_ns;

constexpr uint32_t kMaxPolls = 1u << 24;  // backstop behind the %globaltimer bound
constexpr uint32_t kMaxSleepNs = 1024;

__device__ __forceinline__ int32_t ld_acquire_sys(const int32_t *p) {
  int32_t v;
  asm volatile("ld.acquire.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ld_relaxed_sys(const int32_t *p) {
  int32_t v;
  asm volatile("ld.relaxed.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Whether destination slot di still belongs to the request (its page's owner epoch).
__device__ __forceinline__ bool page_owned(const StreamCtl &k, int32_t di) {
  return ld_relaxed_sys(k.page_epochs + di / k.epoch_page) == k.epoch;
}

// The "no further write" words of a finished move: one release fence at system scope, then the
// status word and (if any) the caller's pinned word as plain strong stores.  The fence orders
// every write before it -- the thread's own, and through cumulativity the whole grid's writes
// it has synchronised with -- before both stores, so a reader that sees either word set sees
// every row the move wrote; one fence instead of one per store (measured: 0.5-0.8 us less per
// streamed call).
__device__ __forceinline__ void publish_done(int32_t *status_done, int32_t *host_done) {
  asm volatile("fence.acq_rel.sys;" ::: "memory");
  asm volatile("st.relaxed.sys.global.b32 [%0], %1;" ::"l"(status_done), "r"(1) : "memory");
  if (host_done)
    asm volatile("st.relaxed.sys.global.b32 [%0], %1;" ::"l"(host_done), "r"(1) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The stop word (mirror[kStopWord]) of the row grid: gen ^ (code << 56 | layer << 40).  Any
// value whose low 40 bits differ from gen's -- stale words of earlier calls, never-written
// workspace -- decodes as "no stop".
constexpr int kStopWord = 1 + KVX_MAX_PLANES / 2;

struct Stop {
  int32_t layer;  // first layer not to move
  int32_t code;   // KVX_ERR_TIMEOUT / KVX_ERR_CANCELLED; 0: no stop
};

__device__ __forceinline__ Stop decode_stop(uint64_t v, uint64_t gen) {
  const uint64_t d = v ^ gen;
  Stop st = {0, 0};
  if (d != 0 && (d & ((1ull << 40) - 1)) == 0) {
    st.code = (int32_t)(d >> 56);
    st.layer = (int32_t)((d >> 40) & 0xFFFF);
  }
  return st;
}

// Records a stop unless one is recorded already (the first one stays).
__device__ __forceinline__ void publish_stop(const StreamCtl &k, uint64_t seen, int32_t layer,
                                             int32_t code) {
  const uint64_t v = k.gen ^ (((uint64_t)code << 56) | ((uint64_t)layer << 40));
  atomicCAS(reinterpret_cast<unsigned long long *>(k.mirror + kStopWord),
            (unsigned long long)seen, (unsigned long long)v);
}

// Thread 0 of a CTA: waits until layer l may move.  Returns 0 to go on, else the stop code.
__device__ inline int32_t row_wait(const StreamCtl &k, int32_t l, bool owner) {
  if (k.words_local) {  // one round trip: the epoch and the ready word together
    const int32_t e = k.epoch_word ? ld_relaxed_sys(k.epoch_word) : k.epoch;
    const bool ready = !k.layer_ready || ld_acquire_sys(k.layer_ready + l) >= k.ready_value;
    if (e == k.epoch && ready) return 0;
  }
  const uint64_t t0 = globaltimer_ns();
  uint32_t sleep_ns = 32;
  for (uint32_t it = 0;; ++it) {
    const uint64_t sw = ld_relaxed_gpu(k.mirror + kStopWord);
    const uint64_t m = ld_acquire_gpu(k.mirror + 1 + l);
    const Stop st = decode_stop(sw, k.gen);
    if (st.code && l >= st.layer) return st.code;
    if (m == k.gen) return 0;
    if (owner || it == 0 || (it & 15) == 15) {
      const int32_t e = k.epoch_word ? ld_relaxed_sys(k.epoch_word) : k.epoch;
      if (e != k.epoch) {  // cancelled: every layer not started is dropped
        publish_stop(k, sw, 0, KVX_ERR_CANCELLED);
        return KVX_ERR_CANCELLED;
      }
      if (!k.layer_ready || ld_acquire_sys(k.layer_ready + l) >= k.ready_value) {
        st_release_gpu(k.mirror + 1 + l, k.gen);
        return 0;
      }
    }
    if (globaltimer_ns() - t0 >= (uint64_t)k.wait_ns || it >= kMaxPolls) {
      publish_stop(k, sw, l, KVX_ERR_TIMEOUT);
      return KVX_ERR_TIMEOUT;
    }
    __nanosleep(sleep_ns);
    if (sleep_ns < kMaxSleepNs) sleep_ns <<= 1;
  }
}

// ---- persistent grids: per-CTA layer state, the shared wait, the exit protocol ------------
// Used by the capped persistent grids of kvx_stream (kvx_stream.cu) and kvx_stream_reshard
// (kvx_reshard.cu): a CTA's workers enter the layers in increasing order, one of them polls
// per CTA and layer, the others read the CTA's shared bits.

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
__device__ inline int32_t wait_layer(const StreamCtl &k, int32_t l, bool owner, CtaState *cs) {
  if (stopped_before(cs, l)) return 0;
  if (known_ready(cs, l)) return 1;
  const uint32_t bit = 1u << (l & 31);
  if (!k.layer_ready && !k.epoch_word) {  // nothing to wait for
    or_release_cta(&cs->ready[l >> 5], bit);
    return 1;
  }
  if (k.words_local) {  // one round trip: the epoch and the ready word together
    const int32_t e = k.epoch_word ? ld_relaxed_sys(k.epoch_word) : k.epoch;
    const bool ready = !k.layer_ready || ld_acquire_sys(k.layer_ready + l) >= k.ready_value;
    if (e == k.epoch && ready) {
      or_release_cta(&cs->ready[l >> 5], bit);
      return 1;
    }
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

// Exit of a persistent grid's CTA (thread 0, once every thread of the CTA has made its last
// write).  Warps of CTAs that started late may still be about to read the planner's verdict in
// status[0], so no CTA writes its stop code there: the code goes into status[2] as a flag above
// the count of finished CTAs, and the last CTA to finish folds the flags into status[0]
// (CANCELLED over TIMEOUT) and sets the "no further write" words.
constexpr int32_t kFinishedMask = (1 << 24) - 1;
constexpr int32_t kTimeoutFlag = 1 << 24;
constexpr int32_t kCancelledFlag = 1 << 25;

__device__ inline void persistent_cta_exit(int32_t *status, const StreamCtl &k, const CtaState &cs,
                                           int32_t layers) {
  if (cs.code) atomicOr(&status[2], cs.code == KVX_ERR_CANCELLED ? kCancelledFlag : kTimeoutFlag);
  if (cs.stop < layers) atomicMax(&status[1], layers - cs.stop);
  __threadfence_system();
  const int32_t before = atomicAdd(&status[2], 1);
  if ((before & kFinishedMask) == (int32_t)gridDim.x - 1) {
    __threadfence_system();
    const int32_t flags = atomicOr(&status[2], 0);  // every CTA set its flag before counting
    if (flags & kCancelledFlag) atomicMax(&status[0], (int32_t)KVX_ERR_CANCELLED);
    else if (flags & kTimeoutFlag) atomicMax(&status[0], (int32_t)KVX_ERR_TIMEOUT);
    publish_done(&status[3], k.host_done);
  }
}

}  // namespace sops

// The one-thread epilogue behind a streamed row grid: once every CTA has finished, the stop code
// joins the verdict and the "no further write" words (status[3], host_done) are set.
cudaError_t launch_stream_done(int32_t *status, int32_t *host_done, int32_t layers,
                               cudaStream_t s);

}  // namespace kvx

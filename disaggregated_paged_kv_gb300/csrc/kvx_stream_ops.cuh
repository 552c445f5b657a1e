// kvx_stream_ops.cuh -- the per-layer wait of the layer-streamed row grids (sm_103a): memory
// ordering helpers, the owner-epoch check of a destination page, the tagged stop word and the
// bounded wait of a CTA's thread 0 for its layer.  Shared by kvx_stream.cu and kvx_reshard.cu.
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

__device__ __forceinline__ void st_release_sys(int32_t *p, int32_t v) {
  asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

}  // namespace sops

// The one-thread epilogue behind a streamed row grid: once every CTA has finished, the stop code
// joins the verdict and the "no further write" words (status[3], host_done) are set.
cudaError_t launch_stream_done(int32_t *status, int32_t *host_done, int32_t layers,
                               cudaStream_t s);

}  // namespace kvx

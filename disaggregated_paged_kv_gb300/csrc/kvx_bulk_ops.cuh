// kvx_bulk_ops.cuh -- TMA bulk copies (cp.async.bulk) and mbarriers for libkvx's kernels
// (sm_103a).  Shared by the bulk copy kernel (kvx_copy.cu) and the bulk form of the
// persistent streamed grid (kvx_stream.cu).
//
// A move is global -> shared (cp.async.bulk, completion counted in bytes on an mbarrier),
// then shared -> global (cp.async.bulk in a bulk async-group).  Data never passes through
// registers, so an SM keeps as many bytes in flight as it has shared-memory stages.  Every
// mbarrier wait is bounded by %globaltimer (kBulkWaitLimitNs) and an iteration cap.
#pragma once

#include <cstdint>

#include "kvx_copy_ops.cuh"

namespace kvx {
namespace bops {

// Bound on one mbarrier wait for a bulk load (never expected to run out).
constexpr uint64_t kBulkWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// The phase's one arrival, and `bytes` more bytes that bulk loads will complete on it.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// false: the phase did not complete within kBulkWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ops::globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ops::globaltimer_ns() - t0 > kBulkWaitLimitNs) return false;
  }
  return false;
}
// bytes (a multiple of 16) from gsrc (16-byte aligned) into shared memory at smem_dst.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// bytes from shared memory to gdst, in the current bulk async-group (see bulk_commit).
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy accesses of global memory with its async-proxy (bulk)
// accesses, in both directions.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

}  // namespace bops
}  // namespace kvx

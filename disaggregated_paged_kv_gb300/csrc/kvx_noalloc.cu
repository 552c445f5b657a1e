// kvx_noalloc.cu -- kvx_transfer_noalloc: a pool-to-pool transfer that needs no workspace from
// the caller, because its planner scratch is a fixed device array compiled into libkvx.
//
// Who needs it: callers that cannot allocate device memory at the moment they move KV.  A
// decode engine usually reserves nearly all free HBM for its KV pool when it starts, so when a
// request's KV has to move there may be nothing left to allocate a workspace from; and
// cudaMalloc / cudaFree synchronise the whole device, which a transfer issued between decode
// steps cannot afford.  Such callers still own the pools, the slot lists and the status word;
// only the plan's scratch lives here.
//
// Rules of the shared scratch:
//  - one array per device, kNoallocScratchBytes long; every GPU that loads libkvx keeps it
//    until the process exits;
//  - its device address is looked up with cudaGetSymbolAddress the first time the entry point
//    runs while a given device is current, and cached; make that first call on each device
//    before any stream capture;
//  - all calls share it and it keeps the last call's contents.  Nothing in it has to start at
//    zero: every byte a call reads was written earlier in that same call.  Two calls whose
//    work overlaps on the GPU (other streams, or other host threads without ordering between
//    them) race on it and may corrupt each other's plan.
#include <cstdint>
#include <mutex>

#include "kvx_internal.cuh"

namespace {

constexpr int64_t cx_align(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
constexpr int64_t kNoallocTiles = (KVX_NOALLOC_MAX_TOKENS + kvx::kTile - 1) / kvx::kTile;
// header | per-tile chunk counts | per-tile chunk tables | one prefix entry (unused here)
constexpr int64_t kNoallocScratchBytes =
    cx_align(cx_align(cx_align(256 + 4 * kNoallocTiles, 256) +
                          (int64_t)sizeof(kvx::Chunk) * kvx::kTile * kNoallocTiles,
                      256) +
                 8,
             256);

static __device__ __align__(256) char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch (set up on first use per device).
kvx_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    kvx::record_cuda_error(e);
    return KVX_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return KVX_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      kvx::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return KVX_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVX_OK;
}

}  // namespace

extern "C" kvx_status kvx_transfer_noalloc(kvx_layout_t src, const int32_t *d_src_slots,
                                           kvx_layout_t dst, const int32_t *d_dst_slots,
                                           int32_t n, int32_t *d_status, kvx_stream_t stream) {
  if (n < 0) return KVX_ERR_INVALID_ARG;
  if (n > KVX_NOALLOC_MAX_TOKENS) return KVX_ERR_NO_WORKSPACE;  // larger than the fixed scratch
  if (kvx::ws_layout(n, 0, false).total > kNoallocScratchBytes) return KVX_ERR_NO_WORKSPACE;
  void *scratch = nullptr;
  const kvx_status st = scratch_address(&scratch);
  if (st != KVX_OK) return st;
  return kvx_transfer(src, d_src_slots, dst, d_dst_slots, n, scratch,
                      (size_t)kNoallocScratchBytes, d_status, stream);
}

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
//  - CUDA loads a module, and the device memory of its arrays and kernels, when the module is
//    first used.  The first call on a device (n = 0 is enough) therefore sets up that device:
//    it looks up the array (loading it) and loads every kernel a transfer can launch, so that
//    later calls load nothing.  Make it before the pool takes the device's free memory, and
//    before any stream capture.  After a device reset the array's address changes and the
//    next call sets the device up again;
//  - the array's address is looked up on every call (cudaGetSymbolAddress, cheap once loaded)
//    and passed to the kernels: in host code the array's name is only a host-side stand-in;
//  - all calls share it and it keeps the last call's contents.  Nothing in it has to start at
//    zero: every byte a call reads was written earlier in that same call (the duplicate table
//    is cleared by the call itself).  Two calls whose work overlaps on the GPU (other streams,
//    or other host threads without ordering between them) race on it and may corrupt each
//    other's plan.
#include <cstdint>
#include <mutex>

#include "kvx_internal.cuh"

namespace {

// Room for a plan of KVX_NOALLOC_MAX_TOKENS tokens, or of KVX_NOALLOC_MAX_DUP_TOKENS tokens
// with the duplicate-destination table: the workspace layout every call computes.
constexpr int64_t kPlainBytes = kvx::ws_layout(KVX_NOALLOC_MAX_TOKENS, 0, false).total;
constexpr int64_t kDupBytes = kvx::ws_layout(KVX_NOALLOC_MAX_DUP_TOKENS, 0, false, true).total;
constexpr int64_t kNoallocScratchBytes = kPlainBytes > kDupBytes ? kPlainBytes : kDupBytes;
static_assert(kvx::ws_layout(KVX_NOALLOC_MAX_DUP_TOKENS + 1, 0, false, true).total >
                  kNoallocScratchBytes,
              "with the duplicate check the limit is exactly KVX_NOALLOC_MAX_DUP_TOKENS");

static __device__ __align__(256) char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_set_up_for[kMaxDevices] = {};  // the scratch address each device was last set up with

// Loads every kernel kvx_transfer (and so this entry point) can launch.
cudaError_t load_transfer_kernels() {
  const void *k[64];
  int n = 0;
  n += kvx::plan_kernel_list(k + n, 64 - n);
  n += kvx::copy_kernel_list(k + n, 64 - n);
  n += kvx::small_kernel_list(k + n, 64 - n);
  n += kvx::narrow_kernel_list(k + n, 64 - n);
  n += kvx::fused_kernel_list(k + n, 64 - n);
  for (int i = 0; i < n; ++i) {
    cudaFuncAttributes at;
    const cudaError_t e = cudaFuncGetAttributes(&at, k[i]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Device address of the current device's scratch; sets the device up on its first call.
kvx_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    kvx::record_cuda_error(e);
    return KVX_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return KVX_ERR_INVALID_ARG;
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    kvx::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    return KVX_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_set_up_for[dev] != p) {
    if ((e = load_transfer_kernels()) != cudaSuccess) {
      kvx::record_cuda_error(e);
      return KVX_ERR_CUDA;
    }
    g_set_up_for[dev] = p;
  }
  *out = p;
  return KVX_OK;
}

}  // namespace

extern "C" kvx_status kvx_transfer_noalloc(kvx_layout_t src, const int32_t *d_src_slots,
                                           kvx_layout_t dst, const int32_t *d_dst_slots,
                                           int32_t n, int32_t *d_status, uint32_t flags,
                                           kvx_stream_t stream) {
  if (n < 0) return KVX_ERR_INVALID_ARG;
  if (n > KVX_NOALLOC_MAX_TOKENS) return KVX_ERR_NO_WORKSPACE;  // larger than the fixed scratch
  void *scratch = nullptr;
  const kvx_status st = scratch_address(&scratch);
  if (st != KVX_OK) return st;
  // kvx_transfer checks the plan (and, with KVX_CHECK_DUP, its table) against the scratch size
  return kvx_transfer(src, d_src_slots, dst, d_dst_slots, n, scratch,
                      (size_t)kNoallocScratchBytes, d_status, flags, stream);
}

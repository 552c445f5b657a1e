// kvx_reshard.cuh -- what the host hands the one-launch reshard of kvx_reshard.cu.
#pragma once

#include "kvx_internal.cuh"

namespace kvx {

// Plane addresses of one call: up to this many for layouts whose planes are not evenly
// spaced (every other layout is its first plane and a stride).
constexpr int kReshardMaxPtrs = KVX_RESHARD_MAX_PLANE_TABLE;

// One part, in device terms: layout indices (sources first, then destinations) and the byte
// offset of the first moved head within a row (token rows) or a page (HND) of each side.
struct ReshardPart {
  int32_t src;
  int32_t dst;
  int64_t src_off;
  int64_t dst_off;
};

struct ReshardCall {
  int64_t n_tokens;
  int32_t planes;
  int32_t n_parts;
  int32_t row_bytes;    // n_heads * head bytes, a multiple of 16
  int32_t n_ptrs;       // entries of ptrs in use
  Side src, dst;        // every source and every destination share these
  int32_t *status;      // the validating planner's verdict
  const int32_t *src_slots, *dst_slots;
  // plane p of layout l: tab[l] < 0 ? base[l] + p * stride[l] : ptrs[tab[l] + p]
  const char *base[KVX_RESHARD_MAX_LAYOUTS];
  int64_t stride[KVX_RESHARD_MAX_LAYOUTS];
  int32_t tab[KVX_RESHARD_MAX_LAYOUTS];
  ReshardPart parts[KVX_RESHARD_MAX_PARTS];
  const char *ptrs[kReshardMaxPtrs];
};

// Enqueues the copy of a validated reshard behind its planner (programmatic dependent launch).
cudaError_t launch_reshard(const ReshardCall &c, cudaStream_t s);

// Layer-streamed reshard (kvx_stream_reshard): whether its layer-major grid fits 32-bit item
// indices, and the grid plus its epilogue behind the validating planner.  k holds the parsed
// control block, the mirror and its tag; the item counts are filled in here.
bool reshard_stream_fits(const ReshardCall &c, const StreamCtl &k);
cudaError_t launch_reshard_stream(const ReshardCall &c, StreamCtl k, cudaStream_t s);
// The same on a capped persistent grid of at most max_grid CTAs (1024 threads, one per SM):
// kvx_stream_ctl::max_ctas > 0.  Writes the status words itself (no epilogue kernel).
int reshard_persist_blocks_per_sm();
cudaError_t launch_reshard_stream_capped(const ReshardCall &c, StreamCtl k, int max_grid,
                                         cudaStream_t s);

}  // namespace kvx

// kvx_copy_ops.cuh -- device helpers shared by libkvx's copy kernels (sm_103a): 16-byte
// streaming loads and stores, the address of a chunk's first row (or of byte x of one token's
// row) on either side of a move, and the two ways a warp moves a chunk (flat byte range, or
// 16-byte pieces placed by row / head).
#pragma once

#include "kvx_internal.cuh"

namespace kvx {
namespace ops {

constexpr int kUnroll = 4;  // independent 16-byte loads in flight per lane

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Whether the plan in the workspace was made for this call's sizes and sides.
__device__ __forceinline__ bool header_matches(const CopyArgs &a) {
  const PlanHeader *h = reinterpret_cast<const PlanHeader *>(a.ws + a.L.header_off);
  // slot-list and run-list plans share one chunk format; a batch plan must be run as a batch
  const bool batch = a.mode == kModeBatch;
  return h->magic == kPlanMagic && (h->mode == kModeBatch) == batch && h->op == a.op &&
         (!batch || h->n_segs == a.n_segs) && h->n_tokens == a.n_tokens &&
         h->chunk_rows == a.chunk_rows &&
         h->planes == a.planes && h->row_bytes == a.row_bytes &&
         h->src_is_pool == a.src.is_pool && h->src_hnd == a.src.hnd &&
         h->src_page_size == a.src.page_size && h->dst_is_pool == a.dst.is_pool &&
         h->dst_hnd == a.dst.hnd && h->dst_page_size == a.dst.page_size &&
         h->src_num_slots == a.src.num_slots && h->dst_num_slots == a.dst.num_slots;
}

// Nanoseconds of the GPU's global timer (bounds every wait in libkvx's kernels).
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Plain 16-byte global load.  Measured on the 288 MiB transfer: 1.7 us per step faster than the
// read-only path (ld.global.nc with L1::no_allocate), and .L2::256B prefetch hints only added
// L2 traffic past the end of every row.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

struct Addr {
  const char *base;  // row 0, head 0
  int64_t row;       // bytes between consecutive rows of the chunk
  int64_t head;      // bytes between consecutive head vectors of a row
};

// Address of the chunk's first row on one side.  idx: slot (pool) or row (buffer).  The
// side's geometry stays in the kernel's parameter space (read by reference, not copied).
__device__ __forceinline__ Addr side_addr(const Side &s, bool is_pool, const char *plane,
                                          int64_t idx, const char *buf_plane, int32_t row_bytes) {
  Addr a;
  if (!is_pool) {
    a.base = buf_plane + idx * row_bytes;
    a.row = row_bytes;
    a.head = s.seg_bytes;
  } else if (s.hnd) {
    const int64_t page = idx / s.page_size, off = idx - page * s.page_size;
    a.base = plane + page * s.page_bytes + off * s.seg_bytes;
    a.row = s.seg_bytes;
    a.head = (int64_t)s.page_size * s.seg_bytes;
  } else {
    a.base = plane + idx * s.slot_stride;
    a.row = s.slot_stride;
    a.head = s.seg_bytes;
  }
  return a;
}

// v / d, by a shift where d is a power of two (shift >= 0).
__device__ __forceinline__ int32_t div_p2(int32_t v, int32_t d, int32_t shift) {
  return shift >= 0 ? v >> shift : v / d;
}

// Start of a token's row (head 0) on one side.
template <bool kHnd>
__device__ __forceinline__ const char *row_base(const Side &s, bool pool, const char *plane,
                                                const char *buf_plane, int32_t idx, int32_t R) {
  if (!pool) return buf_plane + (int64_t)idx * R;
  if (!kHnd) return plane + (int64_t)idx * s.slot_stride;
  const int32_t page = div_p2(idx, s.page_size, s.ps_shift), off = idx - page * s.page_size;
  return plane + (int64_t)page * s.page_bytes + (int64_t)off * s.seg_bytes;
}

// Byte x of the row: contiguous, except on an HND pool side where head h = x / seg sits
// page_size * seg bytes after head h - 1.
template <bool kHnd>
__device__ __forceinline__ const char *row_byte(const Side &s, bool pool, const char *row,
                                                int32_t x) {
  if (!kHnd || !pool) return row + x;
  const int32_t h = div_p2(x, s.seg_bytes, s.seg_shift);
  return row + (int64_t)h * s.page_size * s.seg_bytes + (x - h * s.seg_bytes);
}

__device__ __forceinline__ void copy_linear(const char *src, char *dst, int32_t nvec, int lane) {
  const uint4 *s = reinterpret_cast<const uint4 *>(src);
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  for (int32_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + 32 * u < nvec) r[u] = ld_stream(s + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + 32 * u < nvec) st_stream(d + v0 + 32 * u, r[u]);
  }
}

__device__ __forceinline__ int64_t vec_off(const Addr &a, int32_t v, int32_t vps, int32_t heads) {
  const int32_t q = v / vps, w = v - q * vps;
  const int32_t j = q / heads, h = q - j * heads;
  return j * a.row + h * a.head + (int64_t)w * 16;
}

__device__ __forceinline__ void copy_pieces(const Addr &s, const Addr &d, int32_t nvec,
                                            int32_t vps, int32_t heads, int lane) {
  for (int32_t v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nvec) r[u] = ld_stream(s.base + vec_off(s, v, vps, heads));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t v = v0 + 32 * u;
      if (v < nvec) st_stream(const_cast<char *>(d.base) + vec_off(d, v, vps, heads), r[u]);
    }
  }
}

}  // namespace ops
}  // namespace kvx

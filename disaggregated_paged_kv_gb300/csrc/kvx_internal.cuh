// kvx_internal.cuh -- structures shared by libkvx's host code and its sm_103a kernels.
//
// The hot path is two kernels on the caller's stream:
//   planner  one CTA per tile of KVX_PLAN_TILE consecutive tokens: checks every index, marks
//            where a run of consecutive source and destination rows breaks, compacts the runs
//            with block-wide prefix sums and cuts them into chunks of at most chunk_rows rows
//            ("Mooncake" survey 7.6: contiguous blocks merged into fewer descriptors).  The
//            chunk table of each tile goes into the workspace.
//   copy     a persistent grid of warps; work item w is (chunk w / P, plane w % P).  A warp
//            moves the chunk's rows for one plane with 16-byte vector loads and stores
//            ("DistServe" 第三步: plane p only ever goes to plane p).
// Runs and batches add a one-CTA prefix kernel in front of the planner that turns run lengths
// or request token counts into token offsets.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvx.h"

namespace kvx {

constexpr int kTile = KVX_PLAN_TILE;           // tokens per planner CTA
constexpr int kPlanThreads = 512;
constexpr int kPlanItems = kTile / kPlanThreads;  // consecutive tokens per planner thread
constexpr int kMaxTiles = KVX_MAX_TOKENS / KVX_PLAN_TILE;
constexpr int kCopyThreads = 256;
constexpr int kPrefixThreads = 1024;
constexpr int kPrefixItems = 4;
constexpr int kMaxSegs = 1 << 24;              // most runs / requests per call
constexpr uint32_t kPlanMagic = 0x4B565831u;   // "KVX1"
constexpr int kDefaultChunkBytes = KVX_CHUNK_BYTES;  // target bytes per chunk (per plane)

static_assert(kTile % kPlanThreads == 0, "tile must split evenly over planner threads");
static_assert(kPlanItems * kPlanThreads == kTile, "one planner item per token");

enum Mode : int32_t { kModeSlots = 0, kModeRuns = 1, kModeBatch = 2 };

// Geometry of one side of a move.
struct Side {
  int32_t is_pool;     // 1: a pool (index = slot); 0: a transfer buffer (index = row)
  int32_t hnd;         // 1: HND pages; runs break at every page start
  int32_t page_size;   // HND tokens per page (1 otherwise)
  int32_t seg_bytes;   // bytes of one head vector (head_dim * elem)
  int64_t num_slots;   // pool: valid slots [0, num_slots)
  int64_t slot_stride; // NHD pool: bytes from slot s to s+1
  int64_t page_bytes;  // HND pool: bytes of one page of one plane (= H * page_size * seg)
  int32_t seg_shift;   // log2(seg_bytes) if a power of two, else -1
  int32_t ps_shift;    // log2(page_size) if a power of two, else -1
};

// One chunk of the plan: rows consecutive rows starting at (src, dst) of request req.
struct __align__(16) Chunk {
  int32_t req;
  int32_t src;
  int32_t dst;
  int32_t rows;
};

// Byte offsets of the workspace sections; a pure function of the call's sizes, so the host
// and every kernel agree on it.
struct WsLayout {
  int64_t header_off;  // PlanHeader
  int64_t tiles_off;   // int32[n_tiles]: chunks per tile
  int64_t chunks_off;  // Chunk[n_tiles][kTile]
  int64_t prefix_off;  // int64[n_segs + 1]: token offset of each run / request
  int64_t stage_off;   // kvx_submit: int32 src[n], int32 dst[n], int32 status
  int64_t dup_off;     // duplicate-destination check: uint64[dup_slots] hash table
  int64_t dup_slots;   // power of two >= 2n
  int64_t total;       // bytes required
};

__host__ __device__ constexpr int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

__host__ __device__ constexpr int64_t num_tiles(int64_t n_tokens) {
  return (n_tokens + kTile - 1) / kTile;
}

// staging: kvx_submit's copies of host slot lists; dup: the duplicate-destination table
// (after the staging area whether or not that is used, so every call agrees on its place).
__host__ __device__ constexpr WsLayout ws_layout(int64_t n_tokens, int64_t n_segs, bool staging,
                                                 bool dup = false) {
  WsLayout L{};
  int64_t tiles = num_tiles(n_tokens);
  L.header_off = 0;
  L.tiles_off = 256;
  L.chunks_off = align_up(L.tiles_off + 4 * (tiles > 0 ? tiles : 1), 256);
  L.prefix_off = align_up(L.chunks_off + (int64_t)sizeof(Chunk) * kTile * tiles, 256);
  L.stage_off = align_up(L.prefix_off + 8 * (n_segs + 1), 256);
  L.dup_off = align_up(L.stage_off + 8 * n_tokens + 16, 256);
  L.dup_slots = 64;
  while (L.dup_slots < 2 * n_tokens) L.dup_slots <<= 1;
  if (dup) L.total = L.dup_off + 8 * L.dup_slots;
  else L.total = staging ? L.dup_off : L.stage_off;
  return L;
}

// Written by the planner (or the prefix kernel) into the workspace; the copy kernel compares
// it with its own arguments before it moves anything.
struct PlanHeader {
  uint32_t magic;
  int32_t mode;
  int32_t op;
  int32_t n_segs;
  int64_t n_tokens;
  int32_t chunk_rows;
  int32_t planes;
  int32_t row_bytes;
  int32_t src_is_pool, src_hnd, src_page_size;
  int32_t dst_is_pool, dst_hnd, dst_page_size;
  int32_t pad;
  int64_t src_num_slots;
  int64_t dst_num_slots;
};

struct PlanArgs {
  int32_t mode;
  int32_t op;          // slots / runs modes
  int64_t n_tokens;    // size of the planned token space
  int32_t n_segs;      // runs: n_runs; batch: n_reqs
  int32_t chunk_rows;
  int32_t planes;
  int32_t row_bytes;
  const int32_t *src_idx;  // slots / batch: source slot list
  const int32_t *dst_idx;  // slots / batch: destination slot list
  int64_t n_src_idx;       // batch: elements in src_idx
  int64_t n_dst_idx;       // batch: elements in dst_idx
  const int32_t *runs;     // runs: [n_segs][3]
  const kvx_request *reqs; // batch
  int64_t buf_bytes;       // batch: capacity of the buffer for request checks
  int32_t has_src, has_dst;
  int32_t status_direct;   // slots mode with one validating CTA (validates_direct): that CTA
                           // stores status[0] itself and zeroes status[1 .. status_direct - 1]
  int32_t validate_only;   // check the indices and write the status only (no chunk table:
                           // streamed calls, and one-shot calls whose copy reads the slot lists)
  // Duplicate-destination check (destination pool; slots, runs and batch modes): open-
  // addressing table of dup_mask + 1 words in the workspace, zeroed before the planner;
  // entry = (slot + 1) << 32 | request, so a batch knows both requests of a repeated slot.
  unsigned long long *dup_table;  // nullptr: no check
  uint32_t dup_mask;
  int32_t dup_bits;        // log2 of the table size
  Side src, dst;           // batch: pool geometry of the two layouts (is_pool = 1)
  char *ws;
  WsLayout L;
  int32_t *status;
};

struct CopyArgs {
  int32_t mode;
  int32_t op;
  int64_t n_tokens;
  int32_t n_segs;
  int32_t chunk_rows;
  int32_t planes;
  int32_t row_bytes;
  int32_t seg_bytes;
  int32_t heads;
  Side src, dst;           // single modes: the two sides; batch: the two pools
  char *buf;               // single modes: the transfer buffer
  const kvx_request *reqs; // batch
  const char *ws;
  WsLayout L;
  int32_t *status;
  // One-shot calls with one-row chunks also pass the slot lists themselves: the row kernel
  // then range-checks and loads its row before the planner has finished, and stores only
  // once the planner's status word says every index is valid.  nullptr: read the plan.
  const int32_t *spec_src;
  const int32_t *spec_dst;
  int32_t row_group_shift;  // narrow kernel: log2 of the tokens one warp moves
  int32_t row_lanes;        // row and streamed kernels: lanes per token (1 .. 32)
  int32_t rows_per_warp;    // tokens per warp (row_lanes * rows_per_warp <= 32)
  // Row and narrow kernel order (plane-major): CTA c works on plane c / row_blocks, its warps on the
  // consecutive token groups (c % row_blocks) * (kCopyThreads / 32) + warp, so neighbouring
  // CTAs stream through one plane's rows and a buffer side is read or written front to back.
  uint32_t row_blocks;      // CTAs per plane
  int32_t vec_bytes;        // widest access the call's rows allow: 16, or 8/4/2/1 (kvx_narrow.cu)
  // kvx_submit with a pinned host status word: the row kernel stores the final status there
  // itself (through its device mapping) instead of a device-to-host copy.  nullptr: none.
  int32_t *host_status;
  const char *src_planes[KVX_MAX_PLANES];
  char *dst_planes[KVX_MAX_PLANES];
};

// Words of the streamed kernels' mirror: the cancel word, one word per layer, the stop word.
constexpr int kMirrorWords = 2 + KVX_MAX_PLANES / 2;

// kvx_stream's control words, as device addresses (pinned host words through their device
// mapping).
struct StreamCtl {
  const int32_t *layer_ready;  // [layers] or nullptr (all ready)
  const int32_t *epoch_word;   // nullptr: never cancelled
  int32_t *host_done;          // nullptr: none
  // Device-memory copy of what some CTA has seen in the words above, in the workspace:
  // [0] == gen: cancelled (persistent grid); [1 + l] == gen: layer l ready;
  // [1 + KVX_MAX_PLANES / 2]: the row grid's stop word.  gen is a 64-bit tag new for every
  // eager call, so words left by earlier calls (or any stale workspace bytes) do not match it;
  // a call captured into a CUDA graph keeps its tag, so its mirror is zeroed on each replay.
  uint64_t *mirror;  // kMirrorWords words
  uint64_t gen;
  int64_t wait_ns;
  int32_t ready_value;
  int32_t epoch;
  int32_t layers;
  uint32_t groups;     // row groups of rows_per_warp tokens per plane
  uint32_t per_layer;  // items per layer: kv_planes * groups
  uint32_t items;      // per_layer * layers (< 2^32 for every legal size)
  uint32_t per_layer_pad;  // row grid: per_layer rounded up to whole CTAs
  uint32_t block;      // consecutive items a warp takes per block (see kvx_stream.cu)
  int32_t kv_planes;   // planes per layer: 2 (K, V) or 1 (MLA latent); plane = kv_planes*l + kv
  // The producer's words all live in this GPU's memory (or are absent): a direct read costs
  // what a mirror read costs, so the waits read them first and skip the mirror.
  int32_t words_local;
  // Owner epoch of every destination page (page = slot / epoch_page), or nullptr: a row is
  // stored only while its page's word holds `epoch`.
  int32_t epoch_page;
  const int32_t *page_epochs;
};

// Copy kernel variants: row (non-persistent, one warp per group of tokens of one plane: every
// one-shot request, and every plan with one-row chunks), lean (one request, linear multi-row
// chunks, persistent, 32 registers), linear (batches of linear multi-row chunks), general
// (per-16-byte placement of multi-row chunks: HND pages, slot-major pools) and bulk (TMA,
// linear chunks, chosen with kvx_set_copy_engine).
enum CopyVariant : int {
  kVariantLean = 0,
  kVariantLinear,
  kVariantGeneral,
  kVariantBulk,
  kVariantRow,
  kNumVariants
};

// Launchers (enqueue only; return the launch's cudaError_t).
cudaError_t launch_prefix(const PlanArgs &a, cudaStream_t s);
cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s);
// Every kernel of one translation unit that a gather / scatter / transfer may launch: writes
// at most max function pointers into out and returns how many it wrote (for loading them all
// ahead of time, kvx_transfer_noalloc).
int plan_kernel_list(const void **out, int max);
int copy_kernel_list(const void **out, int max);
int small_kernel_list(const void **out, int max);
int narrow_kernel_list(const void **out, int max);
int fused_kernel_list(const void **out, int max);
inline int kernel_list_out(const void *const *k, int n, const void **out, int max) {
  int c = 0;
  for (; c < n && c < max; ++c) out[c] = k[c];
  return c;
}
// Validate-only calls of up to this many tokens are checked by a single CTA (validate_kernel),
// which stores the status words itself (status_direct), so no status memset is needed first.
// Measured on GB300: 0.8-1.2 us faster than memset + multi-tile planner at 4096 and 8192
// tokens, 1.7-2.2 us slower at 16384 and 32768 (one SM then reads 64-128 KB of indices).
constexpr int64_t kValidateMaxTokens = 8192;
inline bool validates_direct(int64_t n_tokens, bool validate_only) {
  return n_tokens > 0 && (num_tiles(n_tokens) == 1 || (validate_only && n_tokens <= kValidateMaxTokens));
}
// v: the variant copy_variant chose for these arguments and the call's engine.
cudaError_t launch_copy(const CopyArgs &a, CopyVariant v, int grid, cudaStream_t s);
cudaError_t launch_export(const char *ws, WsLayout L, int64_t n_tokens, int32_t *out,
                          int64_t max_chunks, int64_t *count, cudaStream_t s);
// engine: KVX_ENGINE_*, read once per call (kvx_get_copy_engine) so that the planner and the
// copy of one call agree on it.
CopyVariant copy_variant(const CopyArgs &a, int32_t engine);
bool copy_is_linear(const CopyArgs &a);
int variant_threads(CopyVariant v);
int variant_blocks_per_sm(CopyVariant v, int32_t n_tiles);
// Grid of the row variant: one warp per (group of rows_per_warp tokens, plane), plane-major
// (sets CopyArgs::row_blocks).
int64_t row_grid(CopyArgs &a);
// Lanes per token and tokens per warp of the row variant (CopyArgs::row_lanes, rows_per_warp).
void row_shape(const CopyArgs &a, int32_t *lanes, int32_t *rows);
// The same for any kernel whose warps each move whole rows of row_bytes (a multiple of 16).
void row_shape_for(int64_t row_bytes, int32_t *lanes, int32_t *rows);
constexpr int kBulkThreadsPerCta = 32;
constexpr int kBulkSmallTiles = 256;  // occupancy is cached for <= this many tiles and for the max
// Records e as this thread's kvx_last_cuda_error().
void record_cuda_error(cudaError_t e);
// Rows that do not allow 16-byte accesses (kvx_narrow.cu): one warp per (token, plane) row.
cudaError_t launch_narrow(CopyArgs &a, cudaStream_t s);  // sets a.row_blocks
// log2 of the tokens one warp of the narrow kernel moves (CopyArgs::row_group_shift).
int32_t narrow_group_shift(int32_t row_bytes, int32_t vec_bytes);
// One-launch path of small one-shot requests (kvx_small.cu): every CTA checks every index.
constexpr int32_t kSmallMaxTokens = 512;
cudaError_t launch_small(const CopyArgs &a, cudaStream_t s);
// Layer-streamed copy (kvx_stream.cu): persistent grid over layer-major row groups, one
// 1024-thread CTA per SM; tma: three of its warps move row groups by TMA bulk copies (only
// where stream_tma_fits).  stream_blocks_per_sm also sets the kernels' shared-memory limit.
int stream_blocks_per_sm();
int stream_threads();  // threads per CTA of the persistent grid
bool stream_tma_fits(const CopyArgs &c);
void stream_sizes(StreamCtl &k, int64_t n_tokens, int32_t rows_per_warp);
cudaError_t launch_stream(const CopyArgs &c, const StreamCtl &k, int grid, bool tma,
                          cudaStream_t s);
// The same walk with one-token rows moved only by TMA bulk copies (one shared-memory stage per
// thread, rows of any length in pieces); sizes from stream_sizes(k, n, 1).
// stream_bulk_blocks_per_sm also sets the kernels' shared-memory limit.
int stream_bulk_blocks_per_sm();
int stream_bulk_threads();
cudaError_t launch_stream_bulk(const CopyArgs &c, const StreamCtl &k, int grid, cudaStream_t s);
// Row grid (one warp per item) and the epilogue that sets the "no further write" words.
cudaError_t launch_stream_rows(const CopyArgs &c, const StreamCtl &k, cudaStream_t s);
// One-launch path for single requests of up to KVX_FUSED_MAX_TOKENS tokens (kvx_fused.cu).
int fused_blocks_per_sm(bool linear);
cudaError_t launch_fused(const CopyArgs &c, const int32_t *src_idx, const int32_t *dst_idx,
                         int32_t n, int32_t chunk_rows, int sms, int bps, cudaStream_t s);

}  // namespace kvx

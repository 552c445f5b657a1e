/*
 * kvx.h -- libkvx: move a finished prefill's KV cache out of a token-paged KV pool on one
 * GB300 (sm_103a).
 *
 * A request's K/V rows sit scattered across a paged pool, often as thousands of few-KB
 * fragments.  libkvx gathers them by slot index into a contiguous transfer buffer (optionally
 * turning per-page [heads][tokens][dim] into [tokens][heads][dim]), scatters a buffer back into
 * a pool, or moves rows straight from one pool into another pool in the same HBM.
 *
 * Sources (web pages, cited by title and section):
 *  [PD-budget]  "穷人版 PD 分离：在消费级显卡上把 TTS 推理拆成两半" (kilerd.me/pd-on-a-budget):
 *               "B300：让 P 直接写 D 的显存" (a gather kernel writes scattered source rows
 *               straight into the decode side's pages), "5090：一个看得见所有卡的代理" (token-paged
 *               pool, ~7,660 few-KB fragments per request, gather into a contiguous staging
 *               region then scatter back; fragment count, not bytes, sets the cost), "最难的一个
 *               问题" (a failed transfer must be reported to the client at once).
 *  [DistServe]  "DistServe 完全拆解": "KV Cache 跨实例传输" (B_KV = 2 L n_layer n_kvhead d_head b,
 *               T = B_KV / BW_eff + T_setup), "一次请求如何穿过 DistServe" (per-layer pulls, no
 *               contiguous buffer needed).
 *  [mini-infer] "mini-infer系统实战-18-PD 解耦": "KV 序列化格式选择" (per-layer (k, v), each
 *               [seq, kv_heads, head_dim]; permute(1,0,2) on extract and on rebuild).
 *  [Mooncake]   "PD分离调研：从推理阶段拆分到Mooncake的KVCache中心架构": 6.1 (TransferEngine:
 *               registered memory, batches of non-contiguous src/dst, asynchronous status),
 *               7.4 (per-layer KV tensors registered as base address + block length),
 *               7.6 (src_ptrs/dst_ptrs/lengths, contiguous blocks coalesced),
 *               7.7 (HND layout for non-MLA KV).
 *
 * Conventions used by every call:
 *  - A layout has P = 2 * num_layers planes, plane p = 2*layer + kv with K = 0, V = 1 (or, with
 *    kv_planes = 1 for MLA, P = num_layers latent planes, plane p = layer).
 *  - A row is one (plane, token): kv_heads * head_dim elements, R bytes (any R; rows that are
 *    not 16-byte multiples move in narrower accesses, see kvx_layout_desc).  Values are never
 *    interpreted: every operation is an exact byte copy, so NaN payloads and any bit pattern
 *    survive.
 *  - A contiguous transfer buffer holding n tokens is [plane][n][kv_heads][head_dim], i.e.
 *    [layer][K/V][seq][head][dim]: row (p, i) starts at byte (p * n + i) * R.
 *  - Slots and page-table entries are int32.  Byte offsets are 64-bit.
 *
 * Ownership: the caller owns every device buffer (pools, index arrays, transfer buffers,
 * workspace, status words).  The library owns only the host-side layout handle.  No call
 * allocates memory or synchronises the host; work is enqueued on the caller's stream and the
 * call returns.
 *
 * Errors come in two kinds ([PD-budget] "最难的一个问题": the client learns of a failure at
 * once, and nothing is half-written):
 *  - Problems visible on the host (null or misaligned pointers, bad sizes, mismatched
 *    layouts, overlapping memory, short workspace) return a kvx_status immediately and enqueue
 *    nothing.
 *  - Problems in device-resident data (an index out of range, a bad request record) are
 *    written by the planner into the device status word(s).  The copy then moves nothing for
 *    the affected call (or, in kvx_batch, the affected request): all or nothing.  Read the
 *    status after synchronising the stream.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVX_API __attribute__((visibility("default")))
#else
#define KVX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *kvx_stream_t;

typedef enum kvx_status {
  KVX_OK = 0,
  KVX_ERR_INVALID_ARG = 1,   /* bad size, null pointer, inconsistent layouts or request */
  KVX_ERR_ALIGNMENT = 2,     /* a pointer or size not aligned as the call needs */
  KVX_ERR_OUT_OF_RANGE = 3,  /* a slot / page index outside the pool (device status) */
  KVX_ERR_DUPLICATE_DST = 4, /* a destination slot named twice (device status; only checked
                                with KVX_CHECK_DUP) */
  KVX_ERR_OVERLAP = 5,       /* source and destination memory overlap */
  KVX_ERR_CUDA = 6,          /* a CUDA runtime call failed; see kvx_last_cuda_error() */
  KVX_ERR_NO_WORKSPACE = 7,  /* workspace too small or misaligned */
  KVX_ERR_TIMEOUT = 8,       /* a bounded device wait ran out: kvx_stream's wait for a layer
                                (ctl->wait_ns), or the bulk engine's wait on its own transfer
                                (200 ms, never expected); the kernel stopped instead of hanging */
  KVX_ERR_CANCELLED = 9      /* kvx_stream: the request's epoch word changed; the rest of the
                                request was dropped */
} kvx_status;

typedef enum kvx_dtype {
  KVX_F16 = 1,  /* 2-byte elements */
  KVX_BF16 = 2, /* 2-byte elements */
  KVX_F32 = 3,  /* 4-byte elements */
  KVX_FP8 = 4   /* 1-byte elements */
} kvx_dtype;

typedef enum kvx_kind {
  /* Token rows: each plane is [num_slots][kv_heads][head_dim]; slot s starts at
   * plane + s * slot_stride.  Covers per-plane pools ([Mooncake] 7.4: one tensor per layer,
   * block length = row bytes) and slot-major pools [slot][layer][K/V][head][dim]
   * (plane_stride = R, slot_stride = P * R). */
  KVX_NHD = 0,
  /* HND pages ([Mooncake] 7.7): each plane is [num_slots / page_size][kv_heads][page_size]
   * [head_dim].  Slot s is token s % page_size of page s / page_size. */
  KVX_HND_PAGED = 1
} kvx_kind;

typedef enum kvx_op {
  KVX_OP_GATHER = 0,   /* pool rows -> contiguous buffer */
  KVX_OP_SCATTER = 1,  /* contiguous buffer -> pool rows */
  KVX_OP_TRANSFER = 2, /* pool rows -> pool rows */
  KVX_OP_BATCH = 3     /* kvx_execute only: the plan came from kvx_plan_batch */
} kvx_op;

/* Per-call options: the `flags` argument of every call that moves rows (the one before the
 * stream).  KVX_DEFAULTS takes the process-wide settings (kvx_set_check_duplicates,
 * kvx_set_copy_engine, kvx_set_fused_max_tokens).  Any other value is the call's complete
 * option set, a combination of the bits below (0: no duplicate check, the automatic engine,
 * the planner path): two threads may then move KV on two streams with different options
 * without touching each other's.  Unknown bits, or both engines, are KVX_ERR_INVALID_ARG.
 *  KVX_CHECK_DUP      also check that no destination slot is named twice: the planner inserts
 *                     every destination slot into a hash table in the workspace (8 bytes per
 *                     slot of a power of two >= 2n, beyond the plan: kvx_workspace_size
 *                     covers it, plus a memset per call).  A repeat gives
 *                     KVX_ERR_DUPLICATE_DST with nothing moved.  A list with both a repeated
 *                     and an out-of-range slot may report either error.  In a batch the check
 *                     covers the destination slots of every scatter and transfer request the
 *                     planner accepted (requests refused for a bad record or index write
 *                     nothing and keep their own error): every request naming a slot that
 *                     appears twice among them fails with KVX_ERR_DUPLICATE_DST and moves
 *                     nothing, the others move.  Without the check a repeated destination ends
 *                     up holding one of its source rows, which one unspecified.
 *  KVX_USE_REGISTERS  linear chunks moved by 16-byte register loads and stores (what the
 *                     automatic choice does too); KVX_USE_BULK: by the TMA bulk-copy kernel
 *                     (see kvx_set_copy_engine).  Also the form of a capped kvx_stream grid.
 *  KVX_ONE_LAUNCH     the one-launch path of kvx_set_fused_max_tokens for requests of up to
 *                     KVX_FUSED_MAX_TOKENS tokens whose rows are shorter than KVX_CHUNK_BYTES
 *                     (not with KVX_CHECK_DUP). */
#define KVX_DEFAULTS 0xFFFFFFFFu
#define KVX_CHECK_DUP 0x1u
#define KVX_USE_REGISTERS 0x2u
#define KVX_USE_BULK 0x4u
#define KVX_ONE_LAUNCH 0x8u

/* Most planes a layout may have (128 layers x K/V). */
#define KVX_MAX_PLANES 256
/* The planner works on tiles of this many consecutive tokens; a run never crosses a multiple
 * of it. */
#define KVX_PLAN_TILE 2048
/* Most tokens (or rows) one call may move per plane. */
#define KVX_MAX_TOKENS (KVX_PLAN_TILE * 4096)
/* The planner cuts every run into chunks of at most max(1, KVX_CHUNK_BYTES / R) rows; one
 * warp moves one chunk of one plane. */
#define KVX_CHUNK_BYTES 2048

typedef struct kvx_layout_desc {
  int32_t num_layers; /* L >= 1, kv_planes * L <= KVX_MAX_PLANES */
  int32_t kv_heads;   /* H >= 1 */
  int32_t head_dim;   /* D >= 1 (elements) */
  int32_t dtype;      /* kvx_dtype; only its byte width is used */
  int32_t kind;       /* kvx_kind */
  int32_t page_size;  /* KVX_HND_PAGED: tokens per page (>= 1).  KVX_NHD: ignored. */
  int64_t num_slots;  /* token slots per plane; HND: a multiple of page_size */
  /* Plane addresses: either plane_ptrs (host array of P = kv_planes * L device pointers, read
   * during kvx_layout_create and not kept) or, when plane_ptrs is NULL, plane p at
   * base + p * plane_stride.  Every plane address must be a multiple of the element size.
   * Rows move in the widest access (16, 8, 4, 2 or 1 bytes) that divides R, every plane
   * address, the slot stride (KVX_NHD) and the head vector (KVX_HND_PAGED): 16 for the usual
   * shapes; kvx_stream, kvx_reshard and kvx_stream_reshard need 16. */
  void *const *plane_ptrs;
  void *base;
  int64_t plane_stride;
  /* KVX_NHD: bytes from slot s to slot s+1 within a plane; 0 means R (dense rows).  Must be
   * >= R.  KVX_HND_PAGED: must be 0. */
  int64_t slot_stride;
  /* Planes per layer: 2 (K and V; 0 also means 2) or 1 -- one latent vector per layer and
   * token (MLA: [mini-infer] "KV 传输大小", latent + rope in a single plane).  With 1, plane p
   * is layer p and a transfer buffer is [layer][seq][head][dim]. */
  int32_t kv_planes;
  int32_t reserved; /* must be 0 */
} kvx_layout_desc;

typedef struct kvx_layout *kvx_layout_t;

/* One request of a batch ([Mooncake] 6.1 BatchTransfer entry).  32 bytes, device-resident.
 *  op        KVX_OP_GATHER, KVX_OP_SCATTER or KVX_OP_TRANSFER
 *  n_tokens  rows per plane moved by this request (>= 0)
 *  src_off   first element of this request's source slots in the batch's source slot list
 *            (GATHER, TRANSFER)
 *  dst_off   first element of its destination slots in the destination slot list
 *            (SCATTER, TRANSFER)
 *  buf_off   byte offset (multiple of 16) of its buffer region, laid out
 *            [plane][n_tokens][head][dim] (GATHER, SCATTER) */
typedef struct kvx_request {
  int32_t op;
  int32_t n_tokens;
  int64_t src_off;
  int64_t dst_off;
  int64_t buf_off;
} kvx_request;

/* ---- layouts ------------------------------------------------------------------------ */

/* Validates desc and creates a host-only handle (no device memory).  Errors:
 * KVX_ERR_INVALID_ARG (bad field), KVX_ERR_ALIGNMENT (a plane address not a multiple of the
 * element size). */
KVX_API kvx_status kvx_layout_create(const kvx_layout_desc *desc, kvx_layout_t *out);
KVX_API kvx_status kvx_layout_destroy(kvx_layout_t layout);
/* R, the bytes of one (plane, token) row; -1 for a NULL handle. */
KVX_API int64_t kvx_layout_row_bytes(kvx_layout_t layout);
/* P = 2 * num_layers; -1 for a NULL handle. */
KVX_API int32_t kvx_layout_num_planes(kvx_layout_t layout);

/* ---- workspace ---------------------------------------------------------------------- */

/* Bytes of device workspace (256-byte aligned) that any call moving up to max_tokens rows per
 * plane, with up to max_requests requests (kvx_batch) or runs (kvx_*_runs), needs.  The
 * workspace holds the plan between the planner and the copy; its contents need no
 * initialisation.  Returns 0 if the arguments are out of range. */
KVX_API size_t kvx_workspace_size(int64_t max_tokens, int32_t max_requests);

/* ---- one-shot calls: plan + copy on `stream` ----------------------------------------- */

/* Gather ([PD-budget] 5090 section; [mini-infer] KV 序列化格式选择):
 *   buf[p][i] = row(src, p, src_slots[i]) for every plane p and i < n.
 * d_src_slots: device int32[n].  d_buf: device, 16-byte aligned, >= P*n*R bytes.
 * With a KVX_HND_PAGED source the buffer row is [head][dim], so the call is the fused
 * [heads,tokens,dim] -> [tokens,heads,dim] permute.
 * d_status: device int32[1]; KVX_OK or KVX_ERR_OUT_OF_RANGE after the stream reaches it. */
KVX_API kvx_status kvx_gather(kvx_layout_t src, const int32_t *d_src_slots, int32_t n, void *d_buf,
                      size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                      uint32_t flags, kvx_stream_t stream);

/* Scatter ([PD-budget] 5090 section: D scatters the staged rows into its own pages):
 *   row(dst, p, dst_slots[i]) = buf[p][i].  Slots not named keep their bytes.  Naming a slot
 * twice leaves either of the two rows there (unspecified which). */
KVX_API kvx_status kvx_scatter(kvx_layout_t dst, const int32_t *d_dst_slots, int32_t n,
                       const void *d_buf, size_t buf_bytes, void *d_ws, size_t ws_bytes,
                       int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* Pool-to-pool transfer ([PD-budget] B300 section; [Mooncake] 7.6):
 *   row(dst, p, dst_slots[i]) = row(src, p, src_slots[i]).
 * src and dst must have the same num_layers, kv_heads, head_dim and element size and must
 * not share memory (KVX_ERR_OVERLAP). */
KVX_API kvx_status kvx_transfer(kvx_layout_t src, const int32_t *d_src_slots, kvx_layout_t dst,
                        const int32_t *d_dst_slots, int32_t n, void *d_ws, size_t ws_bytes,
                        int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* Run-list forms ([Mooncake] 7.6 src/dst/length descriptors).  d_runs: device int32[n_runs][3]
 * = {src_start, dst_start, len}; run r names rows src_start .. src_start+len-1 and
 * dst_start .. dst_start+len-1.  A buffer side ignores its start field: runs fill (or drain)
 * consecutive buffer rows in run order.  n_tokens must equal the sum of len (checked on the
 * device: KVX_ERR_INVALID_ARG in the status word). */
KVX_API kvx_status kvx_gather_runs(kvx_layout_t src, const int32_t *d_runs, int32_t n_runs,
                           int32_t n_tokens, void *d_buf, size_t buf_bytes, void *d_ws,
                           size_t ws_bytes, int32_t *d_status, uint32_t flags, kvx_stream_t stream);
KVX_API kvx_status kvx_scatter_runs(kvx_layout_t dst, const int32_t *d_runs, int32_t n_runs,
                            int32_t n_tokens, const void *d_buf, size_t buf_bytes, void *d_ws,
                            size_t ws_bytes, int32_t *d_status, uint32_t flags, kvx_stream_t stream);
KVX_API kvx_status kvx_transfer_runs(kvx_layout_t src, kvx_layout_t dst, const int32_t *d_runs,
                             int32_t n_runs, int32_t n_tokens, void *d_ws, size_t ws_bytes,
                             int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* Batch of requests in one plan + one copy launch ([Mooncake] 6.1).  d_reqs: device
 * kvx_request[n_reqs].  total_tokens must equal the sum of n_tokens.  src / dst may be NULL
 * if no request uses them.  d_src_slots / d_dst_slots: device int32 arrays of n_src_slots /
 * n_dst_slots elements.  d_status: device int32[n_reqs + 1]: [1 + q] is request q's code,
 * [0] the largest of all.  A failing request moves nothing; the others still run. */
KVX_API kvx_status kvx_batch(kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                     int32_t n_reqs, int64_t total_tokens, const int32_t *d_src_slots,
                     int64_t n_src_slots, const int32_t *d_dst_slots, int64_t n_dst_slots,
                     void *d_buf, size_t buf_bytes, void *d_ws, size_t ws_bytes,
                     int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* Host-index submission ([Mooncake] 6.1 submitTransfer + getTransferStatus): like
 * kvx_gather / kvx_scatter / kvx_transfer, but the slot lists and the status word are host
 * memory.  Pinned (page-locked) host memory is read and written by the kernels in place, over
 * the CPU-GPU link; pageable memory is staged through the workspace with copies on the
 * stream.  *h_status is valid once the stream has reached the end of this call, not before
 * (it may show KVX_OK while rows are still moving). */
KVX_API kvx_status kvx_submit(int32_t op, kvx_layout_t src, const int32_t *h_src_slots,
                      kvx_layout_t dst, const int32_t *h_dst_slots, int32_t n, void *d_buf,
                      size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *h_status,
                      uint32_t flags, kvx_stream_t stream);

/* Pool-to-pool transfer without a workspace argument.  The pages have no counterpart to this
 * call: it exists for callers that cannot allocate device memory when KV has to move -- an
 * engine that reserved nearly all HBM for its KV pool at start-up has none left for a
 * workspace, and cudaMalloc would synchronise the device between decode steps.  Same
 * arguments, results and errors as kvx_transfer, except that the planner's scratch is one
 * fixed array per device inside libkvx (about 321 KiB, held by every GPU that loads the
 * library until the process exits):
 *  - n may be at most KVX_NOALLOC_MAX_TOKENS, and with the duplicate check (KVX_CHECK_DUP, or
 *    the process default) at most KVX_NOALLOC_MAX_DUP_TOKENS; a larger n returns
 *    KVX_ERR_NO_WORKSPACE with nothing enqueued;
 *  - CUDA loads the array, and each of libkvx's kernels, into device memory when it is first
 *    used.  The first call on a device -- n = 0 is enough -- loads the array and every kernel
 *    this call can launch, so that no later call needs device memory.  Make that first call on
 *    each device before the KV pool takes the device's free memory and before any stream
 *    capture (after a device reset, make it again);
 *  - all calls share the array, so calls whose work overlaps on the GPU (other streams, other
 *    host threads without ordering) race and may corrupt each other; calls in one stream are
 *    safe.  Nothing in it needs to be cleared between calls.
 * After the first call per device it allocates nothing and calls no allocating library
 * routine. */
#define KVX_NOALLOC_MAX_TOKENS 16384
#define KVX_NOALLOC_MAX_DUP_TOKENS 8192
KVX_API kvx_status kvx_transfer_noalloc(kvx_layout_t src, const int32_t *d_src_slots,
                                        kvx_layout_t dst, const int32_t *d_dst_slots, int32_t n,
                                        int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* ---- two-phase form: the plan (validation + run-length planning) and the copy -------- */

/* Validates the indices and writes the plan into d_ws; the status word(s) get the result.
 * op is KVX_OP_GATHER, KVX_OP_SCATTER or KVX_OP_TRANSFER; unused side arguments are NULL. */
KVX_API kvx_status kvx_plan(int32_t op, kvx_layout_t src, const int32_t *d_src_slots, kvx_layout_t dst,
                    const int32_t *d_dst_slots, int32_t n, void *d_ws, size_t ws_bytes,
                    int32_t *d_status, uint32_t flags, kvx_stream_t stream);
KVX_API kvx_status kvx_plan_runs(int32_t op, kvx_layout_t src, kvx_layout_t dst, const int32_t *d_runs,
                         int32_t n_runs, int32_t n_tokens, void *d_ws, size_t ws_bytes,
                         int32_t *d_status, uint32_t flags, kvx_stream_t stream);
KVX_API kvx_status kvx_plan_batch(kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                          int32_t n_reqs, int64_t total_tokens, const int32_t *d_src_slots,
                          int64_t n_src_slots, const int32_t *d_dst_slots, int64_t n_dst_slots,
                          size_t buf_bytes, void *d_ws, size_t ws_bytes, int32_t *d_status,
                          uint32_t flags, kvx_stream_t stream);

/* Runs the copy the plan in d_ws describes.  op, layouts, n_tokens (the planned token count:
 * n, the runs' total, or total_tokens) and, for KVX_OP_BATCH, d_reqs / n_reqs must be those
 * the plan was made with; the device checks them against the plan and writes
 * KVX_ERR_INVALID_ARG on a mismatch.  d_status is the array given to the planner; nothing
 * moves where it holds an error.  A plan may be executed more than once (for instance with
 * other layouts of the same geometry). */
KVX_API kvx_status kvx_execute(int32_t op, kvx_layout_t src, kvx_layout_t dst, const kvx_request *d_reqs,
                       int32_t n_reqs, int64_t n_tokens, void *d_buf, size_t buf_bytes,
                       const void *d_ws, size_t ws_bytes, int32_t *d_status,
                       uint32_t flags, kvx_stream_t stream);

/* Copies the plan's chunks out of the workspace, in plan order, as device int32[4] records
 * {request, src_index, dst_index, rows}; *d_count (device int64) gets the total, and at most
 * max_chunks records are written.  n_tokens as for kvx_execute.  For tests and inspection. */
KVX_API kvx_status kvx_plan_export(const void *d_ws, size_t ws_bytes, int64_t n_tokens,
                           int32_t *d_chunks, int64_t max_chunks, int64_t *d_count,
                           kvx_stream_t stream);

/* ---- head ranges: heterogeneous tensor parallelism ------------------------------------- */

/* Which kv heads a rank of one tensor-parallel group sends to a rank of another ([Mooncake] 7.7
 * 异构TP: with different TP sizes on the two sides, one D rank may merge the shards of several
 * P ranks, or one P rank's shard is split over several D ranks; the sender computes whether it
 * sends, the source offset, the destination offset and the length).  A model has kv_heads kv
 * heads; rank r of a group of size t holds heads [r*kv_heads/t, (r+1)*kv_heads/t) when
 * t <= kv_heads (t must divide kv_heads), and the single head r/(t/kv_heads) when
 * t > kv_heads (kv_heads must divide t; the head is replicated over t/kv_heads ranks).
 * Outputs (host memory): the first head to send in the source rank's own shard, the first head
 * it lands on in the destination rank's shard, and the count; *n_heads = 0 when the pair
 * exchanges nothing.  Of source ranks holding the same replicated head, only the
 * lowest-numbered sends it.  Host-only arithmetic; KVX_ERR_INVALID_ARG for sizes that do not
 * divide, ranks out of range or null outputs. */
KVX_API kvx_status kvx_tp_slice(int32_t kv_heads, int32_t src_tp, int32_t src_rank,
                                int32_t dst_tp, int32_t dst_rank, int32_t *src_head0,
                                int32_t *dst_head0, int32_t *n_heads);

/* Gather / scatter / transfer of a range of kv heads between layouts whose kv_heads differ
 * ([Mooncake] 7.7 异构TP).  For every plane and token i, heads src_head0 .. src_head0 +
 * n_heads - 1 of source row i go to heads dst_head0 .. dst_head0 + n_heads - 1 of destination
 * row i.  Both layouts (where the op uses them) have the same num_layers, head_dim and dtype;
 * kv_heads may differ.  A gather's buffer holds the moved heads only: [plane][n][n_heads]
 * [head_dim] (buf_bytes >= P * n * n_heads * head_dim * elem); a scatter reads that form.
 * Arguments, workspace, status and errors otherwise as kvx_gather / kvx_scatter /
 * kvx_transfer (src_head0 is ignored by a scatter, dst_head0 by a gather); a head range outside
 * a layout's kv_heads is KVX_ERR_INVALID_ARG.  A range whose bytes do not start and end on
 * 16-byte boundaries within a row moves in the widest access its offsets and length allow. */
KVX_API kvx_status kvx_move_heads(int32_t op, kvx_layout_t src, const int32_t *d_src_slots,
                                  int32_t src_head0, kvx_layout_t dst,
                                  const int32_t *d_dst_slots, int32_t dst_head0,
                                  int32_t n_heads, int32_t n, void *d_buf, size_t buf_bytes,
                                  void *d_ws, size_t ws_bytes, int32_t *d_status,
                                  uint32_t flags, kvx_stream_t stream);

/* One part of a reshard (kvx_reshard): heads src_head0 .. src_head0 + n_heads - 1 of layout
 * srcs[src] go to heads dst_head0 .. dst_head0 + n_heads - 1 of layout dsts[dst].  Host
 * memory, 24 bytes. */
typedef struct kvx_head_part {
  int32_t src;
  int32_t dst;
  int32_t src_head0;
  int32_t dst_head0;
  int32_t n_heads;
  int32_t reserved; /* must be 0 */
} kvx_head_part;

/* Most layouts (sources plus destinations) and most parts of one kvx_reshard, and most plane
 * addresses its layouts whose planes are not evenly spaced (plane_ptrs not a constant stride
 * apart) may bring together; evenly spaced layouts count nothing towards the last. */
#define KVX_RESHARD_MAX_LAYOUTS 64
#define KVX_RESHARD_MAX_PARTS 128
#define KVX_RESHARD_MAX_PLANE_TABLE 3072

/* The whole transfer plan between a tensor-parallel group of size src_tp and one of size
 * dst_tp ([Mooncake] 7.7 异构TP): kvx_tp_slice for every (source rank, destination rank)
 * pair, the pairs that exchange nothing left out, destination rank major and source rank
 * minor, with part.src = the source rank and part.dst = the destination rank.  Writes at most
 * max_parts parts (host memory; parts may be NULL when max_parts is 0) and sets *n_parts to
 * the plan's count.  KVX_ERR_INVALID_ARG for sizes kvx_tp_slice refuses, a group size above
 * 1024, a null n_parts, or a plan of more than max_parts parts (*n_parts still says how many
 * it needs).  Host-only. */
KVX_API kvx_status kvx_tp_plan(int32_t kv_heads, int32_t src_tp, int32_t dst_tp,
                               kvx_head_part *parts, int32_t max_parts, int32_t *n_parts);

/* A whole reshard between two tensor-parallel groups in one call ([Mooncake] 7.7 异构TP: a D
 * rank merges the shards of several P ranks; a P rank's shard is split over several D ranks).
 * For every part, plane p and token i < n, heads part.src_head0 .. + n_heads - 1 of
 * row(srcs[part.src], p, d_src_slots[i]) go to heads part.dst_head0 .. + n_heads - 1 of
 * row(dsts[part.dst], p, d_dst_slots[i]): the result of the parts' kvx_move_heads transfers,
 * done by one planner and one copy launch.  The ranks of one instance share its block table,
 * so one slot list (device int32[n]) serves every source and one every destination.
 *  - srcs: host array of n_srcs >= 1 layouts, the pools of one group's ranks: identical
 *    descriptors apart from their plane addresses.  dsts likewise (n_dsts >= 1), with
 *    n_srcs + n_dsts <= KVX_RESHARD_MAX_LAYOUTS.  Both sides share num_layers, kv_planes,
 *    head_dim and dtype; kv_heads may differ between the sides.
 *  - parts: host array of 1 .. KVX_RESHARD_MAX_PARTS parts, all with the same n_heads (every
 *    plan kvx_tp_plan makes has this form), head ranges inside their layouts, and no two parts
 *    writing the same head of the same destination.
 *  - layouts given by uneven plane_ptrs bring at most KVX_RESHARD_MAX_PLANE_TABLE plane
 *    addresses together.
 * Errors before anything is enqueued: KVX_ERR_INVALID_ARG (the conditions above, null
 * pointers); KVX_ERR_OVERLAP (a source's memory overlaps a destination's, or two
 * destinations' memory overlaps, the same layout listed twice included); KVX_ERR_ALIGNMENT
 * (a part's bytes do not start and end on 16-byte boundaries within rows); KVX_ERR_NO_WORKSPACE
 * (d_ws as kvx_transfer: kvx_workspace_size(n, 0) bytes).  On the stream: *d_status = KVX_OK,
 * or KVX_ERR_OUT_OF_RANGE (a slot outside [0, num_slots)) or KVX_ERR_DUPLICATE_DST (with
 * KVX_CHECK_DUP), with nothing written. */
KVX_API kvx_status kvx_reshard(const kvx_layout_t *srcs, int32_t n_srcs,
                               const int32_t *d_src_slots, const kvx_layout_t *dsts,
                               int32_t n_dsts, const int32_t *d_dst_slots,
                               const kvx_head_part *parts, int32_t n_parts, int32_t n,
                               void *d_ws, size_t ws_bytes, int32_t *d_status,
                               uint32_t flags, kvx_stream_t stream);

/* ---- layer-streamed, cancellable copy ------------------------------------------------- */

/* Longest a kvx_stream wait for one layer may be bounded to (ctl->wait_ns): 10 s. */
#define KVX_MAX_WAIT_NS 10000000000LL

/* Control block of kvx_stream (read on the host at the call; the words it points to are read
 * by the kernel while it runs).  Pointers may be device memory or pinned (page-locked) host
 * memory; pageable host memory is rejected (KVX_ERR_INVALID_ARG). */
typedef struct kvx_stream_ctl {
  /* int32[num_layers] or NULL.  Layer l (planes 2l and 2l+1) is moved once
   * layer_ready[l] >= ready_value; the producer raises the word after the layer's rows are
   * written ([DistServe] "一次请求如何穿过 DistServe": prefill writes the prompt's KV layer by
   * layer, decode pulls layer j as soon as it exists).  NULL: every layer is ready. */
  const int32_t *layer_ready;
  int32_t ready_value;
  /* int32 or NULL.  The request is live while *epoch_word == epoch.  The receiving side
   * cancels it (gives up on the transfer, reassigns its pages) by changing the word; the copy
   * then drops every layer it has not started ([PD-budget] "最难的一个问题": each request
   * carries an identity, late data for a dead request is discarded). */
  const int32_t *epoch_word;
  int32_t epoch;
  /* Bound on each wait for one layer, 1 .. KVX_MAX_WAIT_NS nanoseconds.  A layer not ready in
   * time ends the copy with KVX_ERR_TIMEOUT ([DistServe] "一次请求如何穿过 DistServe": every
   * abnormal path needs a lease or a timeout). */
  int64_t wait_ns;
  /* 0: one warp per row (group) on as many CTAs as the request needs; CTAs waiting for a
   * layer hold their SM slots.  > 0: a persistent grid of at most max_ctas CTAs, at most one
   * per SM, for the whole move, leaving the rest of the GPU to a producer running on the same
   * GPU, which needs SMs to make progress.  Its CTAs (see kvx_set_copy_engine): by default
   * 1024 threads moving rows through registers, three of their warps by TMA bulk copies where
   * a row group fits one 2 KiB stage; KVX_ENGINE_REGISTERS: registers only; KVX_ENGINE_BULK:
   * 96 threads moving rows by TMA bulk copies only.  Every SM moves at most ~89 GB/s
   * (read + write) in any form, so the HBM peak takes about half the SMs. */
  int32_t max_ctas;
  int32_t reserved;  /* must be 0 */
  /* Pinned host int32 or NULL: set to 1 when d_status[3] is (see kvx_stream). */
  int32_t *host_done;
  /* int32[ceil(num_slots / epoch_page)] or NULL: the owner epoch of every destination page
   * (page = slot / epoch_page).  A row is stored only while its page's word holds `epoch`;
   * rows of pages the receiver has handed to another request are dropped and reported
   * (KVX_ERR_CANCELLED), the rest of the request still moves ([PD-budget] "最难的一个问题":
   * late data must not land in reassigned pages).  Needs a destination pool (not a gather).
   * Device memory keeps the per-row check cheap; pinned host memory is read over the link. */
  const int32_t *dst_page_epochs;
  int32_t epoch_page; /* slots per epoch page, >= 1 when dst_page_epochs is set */
  int32_t reserved2;  /* must be 0 */
} kvx_stream_ctl;

/* Gather / scatter / transfer of one request (op and arguments as kvx_gather / kvx_scatter /
 * kvx_transfer; d_buf / buf_bytes are ignored by a transfer) that moves layer by layer as the
 * producer marks layers ready, and stops early on cancellation or a wait running out.
 *
 * d_status: device int32[4], written by the call (no initialisation needed):
 *   [0] KVX_OK, or the first error: KVX_ERR_OUT_OF_RANGE (nothing moved, as kvx_transfer),
 *       KVX_ERR_TIMEOUT or KVX_ERR_CANCELLED (the larger code if both happened; CANCELLED
 *       also when rows were dropped for pages that changed owner).
 *   [1] layers pending: the trailing layers not guaranteed moved.  Layers
 *       0 .. num_layers - [1] - 1 hold every row of the request; rows of later layers may or
 *       may not have been written (except rows dropped for a changed page owner, never
 *       written once the change was seen).  0 when [0] is KVX_OK.
 *   [2] internal.
 *   [3] 1 once every CTA of the copy has finished and its writes are visible system-wide: no
 *       further write of this call can land ([PD-budget] "最难的一个问题": the sender may only
 *       acknowledge an aborted transfer once it can prove no late write is still in flight).
 *       The receiving side may reuse cancelled pages after seeing it (or after the stream has
 *       passed the call).
 * The copy occupies up to ctl->max_ctas CTAs while it waits; every wait polls with back-off
 * and ends by ctl->wait_ns, so the kernel always finishes.
 * May be captured into a CUDA graph: every replay is a new call (it reads the slot lists,
 * the control words and the workspace afresh and keeps nothing from an earlier replay); the
 * host-side checks and the control block's values are those of the captured call.
 * Layouts whose rows do not move in 16-byte accesses (see kvx_layout_desc) are
 * KVX_ERR_ALIGNMENT. */
KVX_API kvx_status kvx_stream(int32_t op, kvx_layout_t src, const int32_t *d_src_slots,
                              kvx_layout_t dst, const int32_t *d_dst_slots, int32_t n,
                              void *d_buf, size_t buf_bytes, const kvx_stream_ctl *ctl,
                              void *d_ws, size_t ws_bytes, int32_t *d_status,
                              uint32_t flags, kvx_stream_t stream);

/* kvx_reshard, layer-streamed and cancellable as kvx_stream ("DistServe 完全拆解", layer j
 * pulled as soon as prefill has written it; [Mooncake] 7.7 异构TP for the parts): layer l of
 * every part moves once ctl->layer_ready[l] >= ctl->ready_value (one word per layer for the
 * whole source group: its ranks finish a layer together), the move stops when ctl->epoch_word
 * no longer holds ctl->epoch or a wait runs past ctl->wait_ns, and with ctl->dst_page_epochs
 * a row is written only while its destination page (slot / epoch_page, the same slot list for
 * every destination) still holds ctl->epoch.  Arguments and host-side errors as kvx_reshard
 * and kvx_stream.  ctl->max_ctas == 0: one CTA per padded group of items, as kvx_stream's
 * default grid; > 0: a persistent grid of at most max_ctas CTAs of 1024 threads, one per SM,
 * leaving the rest of the GPU to a producer (as kvx_stream's, with registers only).  A reshard
 * whose padded items exceed 2^31 - 1 is KVX_ERR_INVALID_ARG.
 * d_status: device int32[4], 16-byte aligned, with kvx_stream's meaning (verdict, layers
 * pending, internal, "no further write").  May be captured into a CUDA graph, as kvx_stream. */
KVX_API kvx_status kvx_stream_reshard(const kvx_layout_t *srcs, int32_t n_srcs,
                                      const int32_t *d_src_slots, const kvx_layout_t *dsts,
                                      int32_t n_dsts, const int32_t *d_dst_slots,
                                      const kvx_head_part *parts, int32_t n_parts, int32_t n,
                                      const kvx_stream_ctl *ctl, void *d_ws, size_t ws_bytes,
                                      int32_t *d_status, uint32_t flags, kvx_stream_t stream);

/* ---- misc ---------------------------------------------------------------------------- */

/* Which kernel moves linear chunks (rows contiguous on both sides).  KVX_ENGINE_BULK uses the
 * TMA bulk-copy kernel (cp.async.bulk through shared memory); KVX_ENGINE_AUTO (default) and
 * KVX_ENGINE_REGISTERS use 16-byte register loads and stores.  Both move the same bytes;
 * chunks that are not linear always take the register path.  It also picks the form of
 * kvx_stream's capped persistent grid (kvx_stream_ctl::max_ctas).  A process-wide default read
 * once per call made with flags = KVX_DEFAULTS (KVX_USE_REGISTERS / KVX_USE_BULK choose it per
 * call); returns KVX_ERR_INVALID_ARG for an unknown value. */
#define KVX_ENGINE_AUTO 0
#define KVX_ENGINE_REGISTERS 1
#define KVX_ENGINE_BULK 2
KVX_API kvx_status kvx_set_copy_engine(int32_t engine);
KVX_API int32_t kvx_get_copy_engine(void);

/* Optional one-launch path for kvx_gather, kvx_scatter and kvx_transfer (and kvx_submit,
 * kvx_transfer_noalloc): a request whose rows are shorter than KVX_CHUNK_BYTES and whose n is
 * at most this limit moves in one launch, every CTA checking all n indices itself (the move
 * stays all-or-nothing), planning the runs of its own slice and copying it.  Otherwise the
 * planner launch and the row copy kernel run (the copy overlaps the planner).  Both reach the
 * same bytes.  The default is 0 (off: on GB300 the two launches measured faster at every size);
 * the most is KVX_FUSED_MAX_TOKENS.  A process-wide default for calls made with flags =
 * KVX_DEFAULTS; a call's own flags choose it with KVX_ONE_LAUNCH (limit KVX_FUSED_MAX_TOKENS). */
#define KVX_FUSED_MAX_TOKENS 8192
KVX_API kvx_status kvx_set_fused_max_tokens(int32_t max_tokens);
KVX_API int32_t kvx_get_fused_max_tokens(void);

/* Process-wide default of the duplicate-destination check (KVX_CHECK_DUP), off at start: calls
 * made with flags = KVX_DEFAULTS check for repeats while it is 1.  Calls with their own flags
 * word are not affected.  KVX_ERR_INVALID_ARG for values other than 0 / 1. */
KVX_API kvx_status kvx_set_check_duplicates(int32_t on);
KVX_API int32_t kvx_get_check_duplicates(void);

KVX_API const char *kvx_status_str(kvx_status status);
/* The cudaError_t of the last failing CUDA call made by this thread inside libkvx. */
KVX_API int32_t kvx_last_cuda_error(void);
/* Library version, major * 10000 + minor * 100 + patch. */
KVX_API int32_t kvx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVX_H */

/*
 * kvx_oracle.h -- CPU oracle for moving a finished prefill's KV cache out of a
 * token-paged KV pool.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the plain, slow, single-threaded
 * definition of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path never
 * calls, links or imports it.  It shares no code, header, helper or constant
 * table with the CUDA library: every address below is computed here, from the
 * pages' definitions, independently.
 *
 * Sources (web pages, cited by title and section):
 *  [PD-budget]  "穷人版 PD 分离：在消费级显卡上把 TTS 推理拆成两半" (kilerd.me/pd-on-a-budget)
 *               sections "第一堵墙" (144 KiB/token x 2048 = 288 MiB), "B300：让 P 直接写 D 的显存"
 *               (gather kernel writes scattered source rows straight into D's pages),
 *               "5090：一个看得见所有卡的代理" (token-paged pool, few-KB fragments, gather to a
 *               contiguous staging region, then scatter back into D's pages).
 *  [DistServe]  "DistServe 完全拆解" section "KV Cache 跨实例传输" (B_KV = 2 L n_layer n_kvhead
 *               d_head b) and "第三步：根据网络亲和性映射 stage" (layer j goes only to layer j).
 *  [mini-infer] "mini-infer系统实战-18-PD 解耦" sections "KV 序列化格式选择" (list of per-layer
 *               (k, v), each [seq, kv_heads, head_dim], via permute(1,0,2) of [heads, seq, dim])
 *               and "KV 传输大小" (the KV size table).
 *  [Mooncake]   "PD分离调研：从推理阶段拆分到Mooncake的KVCache中心架构" sections 6.1 (batch of
 *               non-contiguous src/dst transfers), 7.4 (per-layer KV tensors registered by base
 *               address and block length), 7.6 (contiguous blocks coalesced into fewer transfer
 *               descriptors), 7.7 (HND layout for non-MLA KV).
 *
 * Conventions:
 *  - A pool has P = 2 * num_layers planes; plane p = 2*layer + kv with K = 0, V = 1
 *    (the (k, v) tuple order of [mini-infer] "KV 序列化格式选择").
 *  - A row is one (plane, token): kv_heads head vectors of head_dim elements, R bytes.
 *  - A contiguous transfer buffer is [plane][token][head][dim]
 *    = [layer][K/V][seq][kv_heads][head_dim] ([mini-infer] transfer format).
 *  - Values are never interpreted: every operation is a byte copy.
 */
#ifndef KVX_ORACLE_H
#define KVX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Result codes (numerically equal to the library's, written out here on their own). */
#define KVXO_OK 0
#define KVXO_ERR_INVALID_ARG 1
#define KVXO_ERR_OUT_OF_RANGE 3
#define KVXO_ERR_DUPLICATE_DST 4

/* Pool kinds. */
#define KVXO_TOKEN_ROWS 0 /* plane = [slot][head][dim]; slot rows slot_stride bytes apart */
#define KVXO_HND_PAGES 1  /* plane = [page][head][page_size][dim]  ([Mooncake] 7.7 HND) */

/* Batch request kinds. */
#define KVXO_OP_GATHER 0
#define KVXO_OP_SCATTER 1
#define KVXO_OP_TRANSFER 2

typedef struct kvxo_pool {
  int32_t num_layers;
  int32_t kv_heads;
  int32_t head_dim;
  int32_t elem_bytes;
  int32_t kind;
  int32_t page_size; /* HND pages only */
  int64_t num_slots; /* token slots per plane (HND: pages * page_size) */
  uint8_t **planes;  /* 2*num_layers plane base addresses, plane 2*layer + kv */
  int64_t slot_stride; /* token rows only: bytes from slot s to slot s+1 */
  int32_t kv_planes;   /* planes per layer: 2 (K then V; 0 also means 2) or 1 (one latent
                        * vector per layer, MLA: [mini-infer] "KV 传输大小") */
} kvxo_pool;

typedef struct kvxo_request {
  int32_t op;
  int32_t n_tokens;
  int64_t src_off; /* element offset into the batch's source slot list */
  int64_t dst_off; /* element offset into the batch's destination slot list */
  int64_t buf_off; /* byte offset of this request's [plane][token][head][dim] region */
} kvxo_request;

typedef struct kvxo_run {
  int32_t req; /* request the rows belong to */
  int32_t src; /* first source index (slot, or token for a buffer side) */
  int32_t dst; /* first destination index */
  int32_t len; /* consecutive tokens covered */
} kvxo_run;

/* B_KV per token = 2 * n_layer * n_kvhead * d_head * b   ([DistServe] KV Cache 跨实例传输). */
int64_t kvxo_bytes_per_token(int32_t num_layers, int32_t kv_heads, int32_t head_dim,
                             int32_t elem_bytes);

/* MLA bytes per token ([mini-infer] "KV 传输大小": MLA keeps one compressed vector per layer,
 * latent + rope, so there is no factor 2): num_layers * (latent_dim + rope_dim) * elem_bytes. */
int64_t kvxo_mla_bytes_per_token(int32_t num_layers, int32_t latent_dim, int32_t rope_dim,
                                 int32_t elem_bytes);

/* Bytes of one (plane, token) row: kv_heads * head_dim * elem_bytes. */
int64_t kvxo_row_bytes(const kvxo_pool *pool);

/* Validation shared by every operation below: every index in [0, num_slots). */
int kvxo_check_slots(const kvxo_pool *pool, const int32_t *slots, int64_t n);

/* Same slot twice among the destinations. */
int kvxo_has_duplicate(const int32_t *slots, int64_t n, int64_t num_slots);

/* Gather: buf[p][i] = row(src, p, slots[i]).  Returns a status code; nothing is written on
 * error.  *bytes_written (may be NULL) receives n * P * R. */
int kvxo_gather(const kvxo_pool *src, const int32_t *slots, int64_t n, uint8_t *buf,
                int64_t *bytes_written);

/* Scatter: row(dst, p, slots[i]) = buf[p][i].  check_dup != 0 rejects repeated slots. */
int kvxo_scatter(const kvxo_pool *dst, const int32_t *slots, int64_t n, const uint8_t *buf,
                 int check_dup, int64_t *bytes_written);

/* Pool-to-pool transfer: row(dst, p, dst_slots[i]) = row(src, p, src_slots[i]). */
int kvxo_transfer(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                  const int32_t *dst_slots, int64_t n, int check_dup, int64_t *bytes_written);

/* kvxo_transfer restricted to the layers before `stop` (0 <= stop <= num_layers): what a
 * layer-streamed move that stopped before layer `stop` has written.  Planes 2l and 2l+1 of
 * every layer l < stop are moved; later planes are untouched.  Written bytes: n * 2 * stop * R. */
int kvxo_transfer_layers(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                         const int32_t *dst_slots, int64_t n, int32_t stop,
                         int64_t *bytes_written);

/* kvxo_transfer_layers restricted to rows whose destination page is still owned by the
 * request: page_epochs[slot / epoch_page] must equal epoch for row (slot) to be written.
 * Bytes written: the rows written * R. */
int kvxo_transfer_owned(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                        const int32_t *dst_slots, int64_t n, int32_t stop,
                        const int32_t *page_epochs, int32_t epoch_page, int32_t epoch,
                        int64_t *bytes_written);

/* Head-range move between pools whose kv_heads differ ([Mooncake] 7.7 异构TP).  op: 0 gather
 * (src -> buf [plane][n][n_heads][head_dim]), 1 scatter (buf -> dst), 2 transfer (src ->
 * dst).  For every plane and token i, heads src_head0 .. src_head0 + n_heads - 1 of source
 * row i go to heads dst_head0 .. of destination row i.  The pools share num_layers, head_dim
 * and elem_bytes.  Errors: KVXO_ERR_INVALID_ARG (bad op, geometry or head range),
 * KVXO_ERR_OUT_OF_RANGE; nothing written on error. */
int kvxo_move_heads(int32_t op, const kvxo_pool *src, const int32_t *src_slots,
                    int32_t src_head0, const kvxo_pool *dst, const int32_t *dst_slots,
                    int32_t dst_head0, int32_t n_heads, int64_t n, uint8_t *buf,
                    int64_t *bytes_written);

/* One part of a reshard: heads src_head0 .. src_head0 + n_heads - 1 of source pool `src`
 * go to heads dst_head0 .. dst_head0 + n_heads - 1 of destination pool `dst` (indices into
 * the srcs / dsts arrays of kvxo_reshard). */
typedef struct kvxo_part {
  int32_t src;
  int32_t dst;
  int32_t src_head0;
  int32_t dst_head0;
  int32_t n_heads;
} kvxo_part;

/* A whole reshard between two tensor-parallel groups ([Mooncake] 7.7 异构TP: one D rank may
 * merge the shards of several P ranks; one P rank's shard may be split over several D ranks).
 * Every part is a head-range transfer (kvxo_move_heads, op 2) from srcs[part.src] to
 * dsts[part.dst] with the one source slot list and the one destination slot list (the ranks
 * of one instance share its block table).  The result is that of the parts' transfers done
 * one after another; no two parts may write the same head of the same destination pool, so
 * their order does not matter.  Every pool listed shares num_layers, kv_planes, head_dim
 * and elem_bytes, and every slot is checked against every pool of its side.  Errors:
 * KVXO_ERR_INVALID_ARG (no part, a pool index or head range outside its pool, differing
 * geometry, two parts writing one destination head), then KVXO_ERR_OUT_OF_RANGE; nothing
 * written on error.  Bytes written: the sum over parts of n * P * n_heads * head bytes. */
int kvxo_reshard(const kvxo_pool *const *srcs, int32_t n_srcs, const int32_t *src_slots,
                 const kvxo_pool *const *dsts, int32_t n_dsts, const int32_t *dst_slots,
                 const kvxo_part *parts, int32_t n_parts, int64_t n, int64_t *bytes_written);

/* The transfer plan between P rank p_rank of a tensor-parallel group of size p_tp and D rank
 * d_rank of a group of size d_tp, for a model with `heads` kv heads ([Mooncake] 7.7 异构TP).
 * Rank r of a group of size t holds heads [r*heads/t, (r+1)*heads/t) (t <= heads, t divides
 * heads) or the single head r/(t/heads) (t > heads, heads divides t).  Output: the first
 * head to send in the P rank's shard, the first head in the D rank's shard, and the count
 * (0: nothing to send; of P ranks holding the same head only the lowest-numbered sends). */
int kvxo_tp_slice(int32_t heads, int32_t p_tp, int32_t p_rank, int32_t d_tp, int32_t d_rank,
                  int32_t *src_head0, int32_t *dst_head0, int32_t *n_heads);

/* HND gather by page table, through the logical per-plane [heads][seq][dim] view, then the
 * [heads,seq,dim] -> [seq,heads,dim] permute of [mini-infer] "KV 序列化格式选择".
 * Token s lives in page page_table[s / page_size] at offset s % page_size. */
int kvxo_hnd_gather(const kvxo_pool *src, const int32_t *page_table, int64_t seq_len,
                    uint8_t *buf);

/* Inverse rebuild: [seq,heads,dim] -> [heads,seq,dim] permute, then written into the pages. */
int kvxo_hnd_rebuild(const kvxo_pool *dst, const int32_t *page_table, int64_t seq_len,
                     const uint8_t *buf);

/* Batch: every request applied in index order ([Mooncake] 6.1 BatchTransfer).
 * status[0] = largest code of any request, status[1 + q] = code of request q.  A failing
 * request writes nothing; the others still run.  The buffer region of request q is
 * buf + buf_off laid out [plane][n_tokens][head][dim].  With check_dup, a destination slot
 * named more than once among the scatter and transfer requests that passed their own checks
 * fails every such request naming it (KVXO_ERR_DUPLICATE_DST). */
int kvxo_batch(const kvxo_pool *src, const kvxo_pool *dst, const kvxo_request *reqs,
               int32_t n_reqs, const int32_t *src_slots, int64_t n_src_slots,
               const int32_t *dst_slots, int64_t n_dst_slots, uint8_t *buf, int64_t buf_bytes,
               int check_dup, int32_t *status);

/* Run-length coalescing ([Mooncake] 7.6: blocks at consecutive addresses are merged into one
 * (source, destination, length) descriptor).  src_idx / dst_idx give each token's source and
 * destination index (slot, or the token's own position for a buffer side).  req_start lists
 * the first token of every request (ascending, req_start[0] = 0).  A run is a longest stretch
 * of tokens of one request over which both index sequences step up by exactly one: it ends
 * where either sequence does not, and at a request start; nothing else ends it.
 * Writes up to max_runs runs in token order and returns the number of runs. */
int64_t kvxo_runs(const int32_t *src_idx, const int32_t *dst_idx, int64_t n,
                  const int64_t *req_start, int32_t n_reqs, kvxo_run *out, int64_t max_runs);

#ifdef __cplusplus
}
#endif

#endif /* KVX_ORACLE_H */

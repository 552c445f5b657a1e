/*
 * kvx_oracle.c -- the plain CPU definition of paged-KV gather / scatter / transfer.
 *
 * TEST INFRASTRUCTURE ONLY (see kvx_oracle.h): single-threaded, one head vector at a time,
 * no blocking, no fusion, no reordering.  Each function says which passage it follows.
 */
#include "kvx_oracle.h"

#include <stdlib.h>
#include <string.h>

int64_t kvxo_bytes_per_token(int32_t num_layers, int32_t kv_heads, int32_t head_dim,
                             int32_t elem_bytes) {
  /* [DistServe] KV Cache 跨实例传输: B_KV = 2 x L x n_layer x n_kvhead x d_head x b, here
   * for L = 1 token.  The 2 is K and V. */
  return (int64_t)2 * num_layers * kv_heads * head_dim * elem_bytes;
}

static int64_t head_bytes(const kvxo_pool *pool) {
  return (int64_t)pool->head_dim * pool->elem_bytes;
}

int64_t kvxo_row_bytes(const kvxo_pool *pool) { return pool->kv_heads * head_bytes(pool); }

int64_t kvxo_mla_bytes_per_token(int32_t num_layers, int32_t latent_dim, int32_t rope_dim,
                                 int32_t elem_bytes) {
  /* [mini-infer] KV 传输大小: MLA stores a single compressed vector (latent + rope) per layer
   * and token instead of a K and a V row. */
  return (int64_t)num_layers * (latent_dim + rope_dim) * elem_bytes;
}

/* Planes per layer: K and V, or (MLA) one latent plane. */
static int32_t planes_per_layer(const kvxo_pool *pool) { return pool->kv_planes == 1 ? 1 : 2; }

static int32_t num_planes(const kvxo_pool *pool) {
  return planes_per_layer(pool) * pool->num_layers;
}

/* Address of head vector (plane, slot, head). */
static uint8_t *head_vec(const kvxo_pool *pool, int32_t plane, int64_t slot, int32_t head) {
  uint8_t *base = pool->planes[plane];
  int64_t hb = head_bytes(pool);
  if (pool->kind == KVXO_HND_PAGES) {
    /* [Mooncake] 7.7: HND page = [head][page_size][dim]. */
    int64_t page = slot / pool->page_size;
    int64_t off = slot % pool->page_size;
    return base + ((page * pool->kv_heads + head) * pool->page_size + off) * hb;
  }
  /* Token rows: one slot holds every head of one token ([PD-budget] 5090 section: the pool is
   * paged per token). */
  return base + slot * pool->slot_stride + head * hb;
}

/* Address of head vector (plane, token, head) in a [plane][n][head][dim] buffer. */
static uint8_t *buf_vec(uint8_t *buf, const kvxo_pool *pool, int32_t plane, int64_t n,
                        int64_t token, int32_t head) {
  return buf + (((int64_t)plane * n + token) * pool->kv_heads + head) * head_bytes(pool);
}

int kvxo_check_slots(const kvxo_pool *pool, const int32_t *slots, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    if (slots[i] < 0 || (int64_t)slots[i] >= pool->num_slots) return KVXO_ERR_OUT_OF_RANGE;
  return KVXO_OK;
}

int kvxo_has_duplicate(const int32_t *slots, int64_t n, int64_t num_slots) {
  unsigned char *seen = (unsigned char *)calloc((size_t)num_slots, 1);
  int dup = 0;
  if (!seen) return 1;
  for (int64_t i = 0; i < n && !dup; ++i) {
    if (slots[i] < 0 || slots[i] >= num_slots) continue;
    if (seen[slots[i]]) dup = 1;
    seen[slots[i]] = 1;
  }
  free(seen);
  return dup;
}

int kvxo_gather(const kvxo_pool *src, const int32_t *slots, int64_t n, uint8_t *buf,
                int64_t *bytes_written) {
  /* [PD-budget] 5090 section: P gathers the rows to send into one contiguous staging region.
   * [mini-infer] KV 序列化格式选择: per layer (k, v), each [seq, kv_heads, head_dim]. */
  int64_t hb = head_bytes(src);
  int rc = kvxo_check_slots(src, slots, n);
  if (rc != KVXO_OK) return rc;
  for (int32_t p = 0; p < num_planes(src); ++p)
    for (int64_t i = 0; i < n; ++i)
      for (int32_t h = 0; h < src->kv_heads; ++h)
        memcpy(buf_vec(buf, src, p, n, i, h), head_vec(src, p, slots[i], h), (size_t)hb);
  if (bytes_written) *bytes_written = n * num_planes(src) * kvxo_row_bytes(src);
  return KVXO_OK;
}

int kvxo_scatter(const kvxo_pool *dst, const int32_t *slots, int64_t n, const uint8_t *buf,
                 int check_dup, int64_t *bytes_written) {
  /* [PD-budget] 5090 section: D scatters the staged rows back into its own pages. */
  int64_t hb = head_bytes(dst);
  int rc = kvxo_check_slots(dst, slots, n);
  if (rc != KVXO_OK) return rc;
  if (check_dup && kvxo_has_duplicate(slots, n, dst->num_slots)) return KVXO_ERR_DUPLICATE_DST;
  for (int32_t p = 0; p < num_planes(dst); ++p)
    for (int64_t i = 0; i < n; ++i)
      for (int32_t h = 0; h < dst->kv_heads; ++h)
        memcpy(head_vec(dst, p, slots[i], h), buf_vec((uint8_t *)buf, dst, p, n, i, h),
               (size_t)hb);
  if (bytes_written) *bytes_written = n * num_planes(dst) * kvxo_row_bytes(dst);
  return KVXO_OK;
}

static int same_row_shape(const kvxo_pool *a, const kvxo_pool *b) {
  return a->num_layers == b->num_layers && a->kv_heads == b->kv_heads &&
         a->head_dim == b->head_dim && a->elem_bytes == b->elem_bytes &&
         planes_per_layer(a) == planes_per_layer(b);
}

int kvxo_transfer(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                  const int32_t *dst_slots, int64_t n, int check_dup, int64_t *bytes_written) {
  /* [PD-budget] B300 section: a gather kernel on P writes the scattered source rows straight
   * into D's pages.  [DistServe] 第三步: layer j of P goes only to layer j of D, so plane p
   * maps to plane p. */
  int64_t hb = head_bytes(src);
  int rc;
  if (!same_row_shape(src, dst)) return KVXO_ERR_INVALID_ARG;
  rc = kvxo_check_slots(src, src_slots, n);
  if (rc == KVXO_OK) rc = kvxo_check_slots(dst, dst_slots, n);
  if (rc != KVXO_OK) return rc;
  if (check_dup && kvxo_has_duplicate(dst_slots, n, dst->num_slots))
    return KVXO_ERR_DUPLICATE_DST;
  for (int32_t p = 0; p < num_planes(src); ++p)
    for (int64_t i = 0; i < n; ++i)
      for (int32_t h = 0; h < src->kv_heads; ++h)
        memcpy(head_vec(dst, p, dst_slots[i], h), head_vec(src, p, src_slots[i], h),
               (size_t)hb);
  if (bytes_written) *bytes_written = n * num_planes(src) * kvxo_row_bytes(src);
  return KVXO_OK;
}

static int check_page_table(const kvxo_pool *pool, const int32_t *page_table, int64_t seq_len) {
  int64_t num_pages, n_pt;
  if (pool->kind != KVXO_HND_PAGES || pool->page_size <= 0) return KVXO_ERR_INVALID_ARG;
  num_pages = pool->num_slots / pool->page_size;
  n_pt = (seq_len + pool->page_size - 1) / pool->page_size;
  for (int64_t j = 0; j < n_pt; ++j)
    if (page_table[j] < 0 || page_table[j] >= num_pages) return KVXO_ERR_OUT_OF_RANGE;
  return KVXO_OK;
}

int kvxo_transfer_layers(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                         const int32_t *dst_slots, int64_t n, int32_t stop,
                         int64_t *bytes_written) {
  /* [DistServe] 一次请求如何穿过 DistServe: prefill writes the prompt's KV layer by layer and
   * decode pulls layer j once it exists.  A layer-streamed move that stopped before layer
   * `stop` has moved exactly the rows of layers 0 .. stop-1 (planes 2l and 2l+1; plane l for
   * one latent plane per layer), as kvxo_transfer moves them; later planes are untouched. */
  const int32_t ppl = planes_per_layer(src);
  int64_t hb = head_bytes(src);
  int rc;
  if (!same_row_shape(src, dst) || stop < 0 || stop > src->num_layers)
    return KVXO_ERR_INVALID_ARG;
  rc = kvxo_check_slots(src, src_slots, n);
  if (rc == KVXO_OK) rc = kvxo_check_slots(dst, dst_slots, n);
  if (rc != KVXO_OK) return rc;
  for (int32_t layer = 0; layer < stop; ++layer)
    for (int32_t kv = 0; kv < ppl; ++kv)
      for (int64_t i = 0; i < n; ++i)
        for (int32_t h = 0; h < src->kv_heads; ++h)
          memcpy(head_vec(dst, ppl * layer + kv, dst_slots[i], h),
                 head_vec(src, ppl * layer + kv, src_slots[i], h), (size_t)hb);
  if (bytes_written) *bytes_written = n * ppl * (int64_t)stop * kvxo_row_bytes(src);
  return KVXO_OK;
}

int kvxo_transfer_owned(const kvxo_pool *src, const int32_t *src_slots, const kvxo_pool *dst,
                        const int32_t *dst_slots, int64_t n, int32_t stop,
                        const int32_t *page_epochs, int32_t epoch_page, int32_t epoch,
                        int64_t *bytes_written) {
  /* [PD-budget] 最难的一个问题: once the receiver hands a page to another request, late data
   * of the old request must not land in it.  Every destination page (epoch_page consecutive
   * slots) carries the epoch of the request that owns it; a row is written only while its
   * page still holds this request's epoch.  With the layer-streamed stop as in
   * kvxo_transfer_layers. */
  const int32_t ppl = planes_per_layer(src);
  int64_t hb = head_bytes(src), rows = 0;
  int rc;
  if (!same_row_shape(src, dst) || stop < 0 || stop > src->num_layers || epoch_page < 1 ||
      !page_epochs)
    return KVXO_ERR_INVALID_ARG;
  rc = kvxo_check_slots(src, src_slots, n);
  if (rc == KVXO_OK) rc = kvxo_check_slots(dst, dst_slots, n);
  if (rc != KVXO_OK) return rc;
  for (int32_t layer = 0; layer < stop; ++layer)
    for (int32_t kv = 0; kv < ppl; ++kv)
      for (int64_t i = 0; i < n; ++i) {
        if (page_epochs[dst_slots[i] / epoch_page] != epoch) continue; /* page reassigned */
        for (int32_t h = 0; h < src->kv_heads; ++h)
          memcpy(head_vec(dst, ppl * layer + kv, dst_slots[i], h),
                 head_vec(src, ppl * layer + kv, src_slots[i], h), (size_t)hb);
        ++rows;
      }
  if (bytes_written) *bytes_written = rows * kvxo_row_bytes(src);
  return KVXO_OK;
}

int kvxo_move_heads(int32_t op, const kvxo_pool *src, const int32_t *src_slots,
                    int32_t src_head0, const kvxo_pool *dst, const int32_t *dst_slots,
                    int32_t dst_head0, int32_t n_heads, int64_t n, uint8_t *buf,
                    int64_t *bytes_written) {
  /* [Mooncake] 7.7 异构TP: with different tensor-parallel sizes on the two sides, one rank's
   * KV shard is a range of kv heads of the other side's shard; the move takes, for every plane
   * and token, head vectors src_head0 .. src_head0 + n_heads - 1 of the source row to head
   * vectors dst_head0 .. dst_head0 + n_heads - 1 of the destination row. */
  const kvxo_pool *shape = op == 1 ? dst : src;
  int64_t hb;
  int rc;
  if (op < 0 || op > 2 || n_heads < 1 || !shape) return KVXO_ERR_INVALID_ARG;
  if (op == 2 && (src->num_layers != dst->num_layers || src->head_dim != dst->head_dim ||
                  src->elem_bytes != dst->elem_bytes ||
                  planes_per_layer(src) != planes_per_layer(dst)))
    return KVXO_ERR_INVALID_ARG;
  if (op != 1 && (src_head0 < 0 || src_head0 + n_heads > src->kv_heads))
    return KVXO_ERR_INVALID_ARG;
  if (op != 0 && (dst_head0 < 0 || dst_head0 + n_heads > dst->kv_heads))
    return KVXO_ERR_INVALID_ARG;
  rc = op != 1 ? kvxo_check_slots(src, src_slots, n) : KVXO_OK;
  if (rc == KVXO_OK && op != 0) rc = kvxo_check_slots(dst, dst_slots, n);
  if (rc != KVXO_OK) return rc;
  hb = head_bytes(shape);
  for (int32_t p = 0; p < num_planes(shape); ++p)
    for (int64_t i = 0; i < n; ++i)
      for (int32_t j = 0; j < n_heads; ++j) {
        /* the buffer holds the n_heads moved heads: [plane][n][n_heads][dim] */
        uint8_t *b = buf + (((int64_t)p * n + i) * n_heads + j) * hb;
        if (op == 0)
          memcpy(b, head_vec(src, p, src_slots[i], src_head0 + j), (size_t)hb);
        else if (op == 1)
          memcpy(head_vec(dst, p, dst_slots[i], dst_head0 + j), b, (size_t)hb);
        else
          memcpy(head_vec(dst, p, dst_slots[i], dst_head0 + j),
                 head_vec(src, p, src_slots[i], src_head0 + j), (size_t)hb);
      }
  if (bytes_written) *bytes_written = n * num_planes(shape) * n_heads * hb;
  return KVXO_OK;
}

/* Same planes and head vectors (kv_heads may differ): what a head-range transfer between a
 * and b needs. */
static int same_geometry(const kvxo_pool *a, const kvxo_pool *b) {
  return a->num_layers == b->num_layers && a->head_dim == b->head_dim &&
         a->elem_bytes == b->elem_bytes && planes_per_layer(a) == planes_per_layer(b);
}

int kvxo_reshard(const kvxo_pool *const *srcs, int32_t n_srcs, const int32_t *src_slots,
                 const kvxo_pool *const *dsts, int32_t n_dsts, const int32_t *dst_slots,
                 const kvxo_part *parts, int32_t n_parts, int64_t n, int64_t *bytes_written) {
  /* [Mooncake] 7.7 异构TP: when the two tensor-parallel sizes differ, a D rank assembles its
   * shard from pieces of several P ranks (or a P rank's shard goes out in pieces to several
   * D ranks).  Each piece is one head-range transfer; a reshard is all of them. */
  int64_t total = 0, w;
  int rc;
  if (n_srcs < 1 || n_dsts < 1 || n_parts < 1 || !srcs || !dsts || !parts)
    return KVXO_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_srcs; ++k)
    if (!srcs[k] || !same_geometry(srcs[k], srcs[0])) return KVXO_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_dsts; ++k)
    if (!dsts[k] || !same_geometry(dsts[k], srcs[0])) return KVXO_ERR_INVALID_ARG;
  for (int32_t k = 0; k < n_parts; ++k) {
    const kvxo_part *q = &parts[k];
    if (q->src < 0 || q->src >= n_srcs || q->dst < 0 || q->dst >= n_dsts || q->n_heads < 1)
      return KVXO_ERR_INVALID_ARG;
    if (q->src_head0 < 0 || q->src_head0 + q->n_heads > srcs[q->src]->kv_heads)
      return KVXO_ERR_INVALID_ARG;
    if (q->dst_head0 < 0 || q->dst_head0 + q->n_heads > dsts[q->dst]->kv_heads)
      return KVXO_ERR_INVALID_ARG;
    for (int32_t m = 0; m < k; ++m) /* one writer per destination head */
      if (parts[m].dst == q->dst && parts[m].dst_head0 < q->dst_head0 + q->n_heads &&
          q->dst_head0 < parts[m].dst_head0 + parts[m].n_heads)
        return KVXO_ERR_INVALID_ARG;
  }
  for (int32_t k = 0; k < n_srcs; ++k)
    if ((rc = kvxo_check_slots(srcs[k], src_slots, n)) != KVXO_OK) return rc;
  for (int32_t k = 0; k < n_dsts; ++k)
    if ((rc = kvxo_check_slots(dsts[k], dst_slots, n)) != KVXO_OK) return rc;
  for (int32_t k = 0; k < n_parts; ++k) {
    const kvxo_part *q = &parts[k];
    rc = kvxo_move_heads(2, srcs[q->src], src_slots, q->src_head0, dsts[q->dst], dst_slots,
                         q->dst_head0, q->n_heads, n, NULL, &w);
    if (rc != KVXO_OK) return rc; /* not reached: every check above has passed */
    total += w;
  }
  if (bytes_written) *bytes_written = total;
  return KVXO_OK;
}

/* Heads [*first, *first + *count) held by rank r of a tensor-parallel group of size t. */
static int tp_heads(int32_t heads, int32_t t, int32_t r, int32_t *first, int32_t *count) {
  if (heads < 1 || t < 1 || r < 0 || r >= t) return KVXO_ERR_INVALID_ARG;
  if (t <= heads) {
    if (heads % t != 0) return KVXO_ERR_INVALID_ARG;
    *first = r * (heads / t);
    *count = heads / t;
  } else {
    if (t % heads != 0) return KVXO_ERR_INVALID_ARG;
    *first = r / (t / heads); /* replicated: t / heads ranks hold the same head */
    *count = 1;
  }
  return KVXO_OK;
}

int kvxo_tp_slice(int32_t heads, int32_t p_tp, int32_t p_rank, int32_t d_tp, int32_t d_rank,
                  int32_t *src_head0, int32_t *dst_head0, int32_t *n_heads) {
  /* [Mooncake] 7.7 异构TP: the sender's transfer plan -- whether this P rank sends to this D
   * rank, where in its own shard the heads start, where they start in the D rank's shard and
   * how many.  Of the P ranks holding the same (replicated) head, the lowest-numbered sends. */
  int32_t pf, pc, df, dc, lo, hi;
  int rc = tp_heads(heads, p_tp, p_rank, &pf, &pc);
  if (rc == KVXO_OK) rc = tp_heads(heads, d_tp, d_rank, &df, &dc);
  if (rc != KVXO_OK) return rc;
  lo = pf > df ? pf : df;
  hi = (pf + pc) < (df + dc) ? (pf + pc) : (df + dc);
  *src_head0 = 0;
  *dst_head0 = 0;
  *n_heads = 0;
  if (hi <= lo) return KVXO_OK;
  if (p_tp > heads && p_rank % (p_tp / heads) != 0) return KVXO_OK; /* another replica sends */
  *src_head0 = lo - pf;
  *dst_head0 = lo - df;
  *n_heads = hi - lo;
  return KVXO_OK;
}

int kvxo_hnd_gather(const kvxo_pool *src, const int32_t *page_table, int64_t seq_len,
                    uint8_t *buf) {
  /* [mini-infer] KV 序列化格式选择: take the per-layer [heads, seq, dim] cache and permute
   * (1, 0, 2) to [seq, heads, dim].  Here the [heads, seq, dim] view is read through the page
   * table of an HND pool ([Mooncake] 7.7), materialised per plane, then permuted. */
  int32_t H = src->kv_heads, ps = src->page_size;
  int64_t hb = head_bytes(src);
  uint8_t *logical;
  int rc = check_page_table(src, page_table, seq_len);
  if (rc != KVXO_OK) return rc;
  logical = (uint8_t *)malloc((size_t)(H * seq_len * hb > 0 ? H * seq_len * hb : 1));
  if (!logical) return KVXO_ERR_INVALID_ARG;
  for (int32_t p = 0; p < num_planes(src); ++p) {
    /* logical[h][s][:] = page page_table[s / ps], head h, offset s % ps */
    for (int32_t h = 0; h < H; ++h)
      for (int64_t s = 0; s < seq_len; ++s) {
        int64_t slot = (int64_t)page_table[s / ps] * ps + s % ps;
        memcpy(logical + ((int64_t)h * seq_len + s) * hb, head_vec(src, p, slot, h),
               (size_t)hb);
      }
    /* buf[p][s][h][:] = logical[h][s][:]   (permute(1, 0, 2)) */
    for (int64_t s = 0; s < seq_len; ++s)
      for (int32_t h = 0; h < H; ++h)
        memcpy(buf_vec(buf, src, p, seq_len, s, h), logical + ((int64_t)h * seq_len + s) * hb,
               (size_t)hb);
  }
  free(logical);
  return KVXO_OK;
}

int kvxo_hnd_rebuild(const kvxo_pool *dst, const int32_t *page_table, int64_t seq_len,
                     const uint8_t *buf) {
  /* [mini-infer] KV 序列化格式选择, rebuild direction: [seq, heads, dim] -> permute(1, 0, 2)
   * -> [heads, seq, dim], then stored into the pages named by the page table. */
  int32_t H = dst->kv_heads, ps = dst->page_size;
  int64_t hb = head_bytes(dst);
  uint8_t *logical;
  int rc = check_page_table(dst, page_table, seq_len);
  if (rc != KVXO_OK) return rc;
  logical = (uint8_t *)malloc((size_t)(H * seq_len * hb > 0 ? H * seq_len * hb : 1));
  if (!logical) return KVXO_ERR_INVALID_ARG;
  for (int32_t p = 0; p < num_planes(dst); ++p) {
    for (int64_t s = 0; s < seq_len; ++s)
      for (int32_t h = 0; h < H; ++h)
        memcpy(logical + ((int64_t)h * seq_len + s) * hb,
               buf_vec((uint8_t *)buf, dst, p, seq_len, s, h), (size_t)hb);
    for (int32_t h = 0; h < H; ++h)
      for (int64_t s = 0; s < seq_len; ++s) {
        int64_t slot = (int64_t)page_table[s / ps] * ps + s % ps;
        memcpy(head_vec(dst, p, slot, h), logical + ((int64_t)h * seq_len + s) * hb,
               (size_t)hb);
      }
  }
  free(logical);
  return KVXO_OK;
}

static int check_request(const kvxo_pool *src, const kvxo_pool *dst, const kvxo_request *r,
                         int64_t n_src_slots, int64_t n_dst_slots, int64_t buf_bytes,
                         const int32_t *src_slots, const int32_t *dst_slots) {
  int uses_src = r->op == KVXO_OP_GATHER || r->op == KVXO_OP_TRANSFER;
  int uses_dst = r->op == KVXO_OP_SCATTER || r->op == KVXO_OP_TRANSFER;
  int uses_buf = r->op == KVXO_OP_GATHER || r->op == KVXO_OP_SCATTER;
  int rc;
  if (r->op < KVXO_OP_GATHER || r->op > KVXO_OP_TRANSFER || r->n_tokens < 0)
    return KVXO_ERR_INVALID_ARG;
  if (uses_src && (r->src_off < 0 || r->src_off + r->n_tokens > n_src_slots))
    return KVXO_ERR_INVALID_ARG;
  if (uses_dst && (r->dst_off < 0 || r->dst_off + r->n_tokens > n_dst_slots))
    return KVXO_ERR_INVALID_ARG;
  if (uses_buf) {
    const kvxo_pool *pool = uses_src ? src : dst;
    int64_t need = (int64_t)r->n_tokens * num_planes(pool) * kvxo_row_bytes(pool);
    if (r->buf_off < 0 || r->buf_off % 16 != 0 || r->buf_off + need > buf_bytes)
      return KVXO_ERR_INVALID_ARG;
  }
  if (uses_src && (rc = kvxo_check_slots(src, src_slots + r->src_off, r->n_tokens)) != KVXO_OK)
    return rc;
  if (uses_dst && (rc = kvxo_check_slots(dst, dst_slots + r->dst_off, r->n_tokens)) != KVXO_OK)
    return rc;
  return KVXO_OK;
}

int kvxo_batch(const kvxo_pool *src, const kvxo_pool *dst, const kvxo_request *reqs,
               int32_t n_reqs, const int32_t *src_slots, int64_t n_src_slots,
               const int32_t *dst_slots, int64_t n_dst_slots, uint8_t *buf, int64_t buf_bytes,
               int check_dup, int32_t *status) {
  /* [Mooncake] 6.1: a batch of non-contiguous transfers submitted together; each is its own
   * request with its own status. */
  status[0] = KVXO_OK;
  if (src && dst && !same_row_shape(src, dst)) {
    for (int32_t q = 0; q <= n_reqs; ++q) status[q] = KVXO_ERR_INVALID_ARG;
    return KVXO_ERR_INVALID_ARG;
  }
  /* each request's own checks: its record and its indices */
  for (int32_t q = 0; q < n_reqs; ++q)
    status[1 + q] = check_request(src, dst, &reqs[q], n_src_slots, n_dst_slots, buf_bytes,
                                  src_slots, dst_slots);
  /* the duplicate check (asked for by the caller; the pages are silent on repeats): count
   * every destination slot of the accepted requests that write into the pool; a request
   * naming a slot counted more than once fails and writes nothing */
  if (check_dup && dst) {
    int32_t *count = (int32_t *)calloc((size_t)dst->num_slots, sizeof(int32_t));
    if (!count) return KVXO_ERR_INVALID_ARG;
    for (int32_t q = 0; q < n_reqs; ++q) {
      const kvxo_request *r = &reqs[q];
      const int counted = status[1 + q] == KVXO_OK && r->op != KVXO_OP_GATHER;
      if (counted)
        for (int32_t i = 0; i < r->n_tokens; ++i) ++count[dst_slots[r->dst_off + i]];
    }
    for (int32_t q = 0; q < n_reqs; ++q) {
      const kvxo_request *r = &reqs[q];
      if (status[1 + q] != KVXO_OK || r->op == KVXO_OP_GATHER) continue;
      for (int32_t i = 0; i < r->n_tokens; ++i)
        if (count[dst_slots[r->dst_off + i]] > 1) {
          status[1 + q] = KVXO_ERR_DUPLICATE_DST;
          break;
        }
    }
    free(count);
  }
  /* the accepted requests, one by one in index order */
  for (int32_t q = 0; q < n_reqs; ++q) {
    const kvxo_request *r = &reqs[q];
    int rc = status[1 + q];
    if (rc == KVXO_OK) {
      if (r->op == KVXO_OP_GATHER)
        rc = kvxo_gather(src, src_slots + r->src_off, r->n_tokens, buf + r->buf_off, NULL);
      else if (r->op == KVXO_OP_SCATTER)
        rc = kvxo_scatter(dst, dst_slots + r->dst_off, r->n_tokens, buf + r->buf_off, 0, NULL);
      else
        rc = kvxo_transfer(src, src_slots + r->src_off, dst, dst_slots + r->dst_off,
                           r->n_tokens, 0, NULL);
    }
    status[1 + q] = rc;
    if (rc > status[0]) status[0] = rc;
  }
  return status[0];
}

int64_t kvxo_runs(const int32_t *src_idx, const int32_t *dst_idx, int64_t n,
                  const int64_t *req_start, int32_t n_reqs, kvxo_run *out, int64_t max_runs) {
  /* [Mooncake] 7.6 (_build_transfer_params): blocks whose addresses follow one another are
   * merged into one descriptor (source start, destination start, length).  A run therefore
   * goes on while both index sequences step up by exactly one; it ends where either one does
   * not, and (a batch being a list of separate requests, [Mooncake] 6.1) where a new request
   * starts.  Nothing else ends a run. */
  int64_t count = 0;
  int32_t q = 0;
  if (n <= 0) return 0;
  for (int64_t a = 0; a < n;) {
    while (q + 1 < n_reqs && req_start[q + 1] <= a) ++q; /* request of token a */
    const int64_t req_end = (q + 1 < n_reqs) ? req_start[q + 1] : n;
    int64_t b = a + 1;
    /* the step test in 64 bits: an index list may hold INT32_MAX */
    while (b < req_end && (int64_t)src_idx[b] == (int64_t)src_idx[b - 1] + 1 &&
           (int64_t)dst_idx[b] == (int64_t)dst_idx[b - 1] + 1)
      ++b;
    if (count < max_runs) {
      out[count].req = q;
      out[count].src = src_idx[a];
      out[count].dst = dst_idx[a];
      out[count].len = (int32_t)(b - a);
    }
    ++count;
    a = b;
  }
  return count;
}
